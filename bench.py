#!/usr/bin/env python
"""Decode-step benchmark of the paged KV cache library on GB300.

A step is one pass of the whole hot path over one synthetic batch: the cache
write of one new token per sequence (paged_kv_write) followed by paged decode
attention over every sequence's context (paged_attention_decode: the decode
kernel, plus the log-sum-exp reduce when a context spans several partitions).

Default workload: the LLaMA-2-13B-shaped decode batch (64 sequences, 40 MHA
heads x 128, fp16, block 16, contexts U[128, 2048]). The pool (1.7 GB) is
larger than L2, so no flush runs between steps.

One JSON line on rank 0:
  value         KV bytes read per step / step time (GB/s), inputs resident in HBM
  tokens_per_s  sequences decoded per second (one layer)
  roofline      the decode call's algorithmic bytes / its event-timed duration
                against the measured HBM copy bandwidth
  e2e           the same metric through the public API with the step's inputs
                copied from pinned host memory and the output read back
  cpu_baseline  the CPU oracle (fp64, all host cores) on a bounded sample

--impl reference times the CPU oracle alone (the only other implementation of
this path) on the same workload and prints the same line with "impl".
Multi-GPU (torchrun): every rank decodes its own batch (weak scaling); the
timed region is bracketed by barriers and the max over ranks is reported.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode attention: KV-read HBM GB/s (% of peak) and decode tokens/s"
FALLBACK_HBM_GBS = 6800.0
FP8_SCALE = 2.0 ** -6  # k_scale = v_scale of the FP8 runs: N(0,1) values up to 7 are not saturated


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--op", choices=["decode-step", "copy-blocks"], default="decode-step",
                    help="decode-step: the hot path (default); copy-blocks: the copy-on-write block copy alone")
    ap.add_argument("--config", type=int, default=2, help="workload 1..5 (default 2: LLaMA-2-13B-shaped)")
    ap.add_argument("--partition-size", type=int, default=0)
    ap.add_argument("--max-seqs", type=int, default=None, help="use only the workload's first N sequences")
    ap.add_argument("--block-size", type=int, default=16, choices=[8, 16, 32],
                    help="tokens per KV block (the pages' block-size ablation)")
    ap.add_argument("--kv-dtype", choices=["auto", "fp8_e4m3"], default="auto",
                    help="auto: the cache holds the workload's fp16/bf16 values; fp8_e4m3: E4M3 codes "
                         "(paged_kv_write_fp8 / paged_attention_decode_fp8, or paged_attention_multi_query_fp8 "
                         "with --query-len; k_scale = v_scale = FP8_SCALE)")
    ap.add_argument("--query-len", type=int, default=None,
                    help="multi-query step: each sequence's last N context tokens are written and attend causally "
                         "(paged_attention_multi_query; speculative verification / chunked prefill)")
    ap.add_argument("--mq-tile", choices=["auto", "columns", "rows", "tensor", "pairs"], default="auto",
                    help="multi-query tile (default: the library's choice by rows per kv head)")
    ap.add_argument("--shared-prefix", action="store_true",
                    help="workload 4 through paged_attention_decode_shared_prefix: the 1024-token prefix is "
                         "attended once for the whole batch, then each tail, then a merge")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="wall-time budget of the CPU baseline on all host cores (half of it again single-threaded)")
    ap.add_argument("--no-suite", action="store_true",
                    help="skip the other workloads (the default run also times workloads 1, 3, 4, 5, the FP8 cache "
                         "and multi-query steps, each in its own timed region, into the line's workloads object)")
    ap.add_argument("--suite-steps", type=int, default=200, help="timed steps of each suite entry")
    ap.add_argument("--suite-cpu-seconds", type=float, default=1.5, help="CPU oracle budget of each suite entry")
    return ap.parse_args()


# ----------------------------------------------------------------------------
# process group (weak scaling: one independent batch per rank)


class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist

            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group("gloo", rank=self.rank, world_size=self.world)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch

        t = torch.tensor([x], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x: float) -> float:
        if not self.pg:
            return x
        import torch

        t = torch.tensor([x], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ----------------------------------------------------------------------------
# byte accounting


def default_partition(fp8: bool, mq: bool = False, block_size: int = 16, max_context_len: int = 0) -> int:
    """The library's partition size when the call passes 0 (longer for multi-query and for contexts that may
    exceed 8192 tokens; at most 128 blocks)."""
    if mq:
        return min(2048, 128 * block_size)
    return min(2048 if max_context_len > 8192 else 1024, 128 * block_size)


SHARED_PREFIX_TOKENS = 1024  # workload 4's common prefix


def shared_prefix_call_bytes(batch, prefix_tokens: int, ws_bytes: int, cache_bytes: int = 2):
    """Bytes the shared-prefix call must move: the prefix's K/V once, every tail's K/V, q and out, the
    tables, and the two stages' partials (written, then read by the merge). cache_bytes: per cached
    K/V element (1 for an FP8 cache)."""
    from paged_kv_cache_91_gb300 import workloads as W

    S, H, D, B, e = batch.num_seqs, batch.num_heads, batch.head_dim, batch.block_size, batch.elem_bytes
    kv = W.unique_kv_bytes(batch) * cache_bytes // e
    tail_blocks = int(((batch.context_lens - prefix_tokens + B - 1) // B).sum())
    tables = (prefix_tokens // B + tail_blocks) * 4 + S * 4
    return kv + 2 * S * H * D * e + tables + 2 * ws_bytes


def step_bytes(batch, partition_size: int, cache_bytes: int = 2):
    """Algorithmic bytes of one decode call: KV reads plus q, out, tables and split-K partials.
    cache_bytes: bytes per cached K/V element (2, or 1 for an FP8 cache)."""
    import numpy as np

    from paged_kv_cache_91_gb300 import workloads as W

    P = partition_size or default_partition(cache_bytes == 1, batch.query_start_loc is not None, batch.block_size,
                                            batch.max_context_len)
    ctx = batch.context_lens.astype(np.int64)
    kv = W.algorithmic_kv_bytes(batch) * cache_bytes // batch.elem_bytes
    S, H, D, B = batch.num_seqs, batch.num_heads, batch.head_dim, batch.block_size
    # query rows per sequence: 1 in decode, q_len in the multi-query form
    qlen = np.ones(S, np.int64) if batch.query_start_loc is None else np.diff(batch.query_start_loc).astype(np.int64)
    qo = 2 * int(qlen.sum()) * H * D * batch.elem_bytes
    tables = int(((ctx + B - 1) // B).sum()) * 4 + S * 4
    nparts = (ctx + P - 1) // P
    split = nparts > 1
    partials = int((nparts[split] * qlen[split] * H).sum()) * (D + 2) * 4 * 2
    return kv, kv + qo + tables + partials


KERNEL_SOURCES = {
    "simt": ("pkv_common.cuh", "pkv_decode_simt.cuh", "pkv_decode_simt_f16.cu", "pkv_decode_simt_bf16.cu"),
    "mma": ("pkv_common.cuh", "pkv_decode_mma.cuh", "pkv_decode_mma_f16.cu", "pkv_decode_mma_bf16.cu"),
    "simt_fp8": ("pkv_common.cuh", "pkv_decode_simt.cuh", "pkv_decode_simt_fp8.cu"),
    "mma_fp8": ("pkv_common.cuh", "pkv_decode_mma.cuh", "pkv_decode_mma_fp8.cuh", "pkv_decode_mma_fp8.cu"),
    "mq": ("pkv_common.cuh", "pkv_decode_mma.cuh", "pkv_decode_mq.cuh", "pkv_mq_wide.cuh", "pkv_mq_tc.cuh",
           "pkv_tcgen05.cuh", "pkv_decode_mq.cu"),
    "mq_fp8": ("pkv_common.cuh", "pkv_decode_mma.cuh", "pkv_decode_mma_fp8.cuh", "pkv_decode_mq.cuh",
               "pkv_mq_tc.cuh", "pkv_tcgen05.cuh", "pkv_decode_mq_fp8.cu"),
    "mq_fp8_pairs": ("pkv_common.cuh", "pkv_decode_mma.cuh", "pkv_decode_mma_fp8.cuh", "pkv_decode_mq.cuh",
                     "pkv_mq_pairs.cuh", "pkv_decode_mq_pairs.cu"),
}


def kernel_hash(kind: str) -> str:
    """Hash of the sources that define one decode kernel (ties an ncu capture to the code it measured)."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, "paged_kv_cache_91_gb300", "csrc", name), "rb") as fh:
            h.update(name.encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str, kind: str):
    """DRAM bytes per decode launch from the committed ncu summary, if it matches the kernel's sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    entry = rec.get(workload)
    if not entry or entry.get("kernel_hash") != kernel_hash(kind):
        return None
    return entry.get("dram_bytes_per_call")


# Layers of the models the workloads are shaped after ("KV Cache와 PagedAttention 완전 해부": Qwen3-4B has 36
# layers (§2단계); the LLaMA-2-13B example has 40 (§3단계)).
MODEL_LAYERS = {2: ("LLaMA-2-13B", 40), 3: ("Qwen3-4B", 36), 4: ("Qwen3-4B-shaped heads", 36),
                5: ("LLaMA-2-13B", 40)}


def model_extrapolation(config: int, tokens_per_s_one_layer: float):
    """Tokens/s of a model of L such layers if attention were the whole step (labelled as such)."""
    if config not in MODEL_LAYERS:
        return None
    name, layers = MODEL_LAYERS[config]
    return {"model": name, "layers": layers, "value": round(tokens_per_s_one_layer / layers, 1),
            "note": "attention only: one layer's measured step time x layers; no projections, MLP or sampling"}


def hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return FALLBACK_HBM_GBS, "fallback"


# ----------------------------------------------------------------------------
# clocks during the timed region


class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    PERIOD_MS = 20

    def __init__(self, gpu_id: str):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_id}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.PERIOD_MS)], stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        self.windows = []

    def mark(self):
        return time.time()

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = []
        for line in self.file.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append(dict(ts=ts, sm=float(parts[2]), smax=float(parts[3]),
                                 reasons=[r for r, v in zip(self.REASONS, parts[6:10]) if v.lower() == "active"]))
            except (ValueError, IndexError):
                continue
        self.file.close()
        os.unlink(self.file.name)
        return rows

    @staticmethod
    def summarise(rows, t0, t1, margin: float = 0.25):
        """Clocks of a timed region: the samples taken inside it, or, when fewer than 3 fall inside (a region
        of a few ms), every sample within ``margin`` seconds of it, labelled so."""
        inside = [r for r in rows if t0 <= r["ts"] <= t1]
        near = [r for r in rows if t0 - margin <= r["ts"] <= t1 + margin]
        used, window = (inside, "timed region") if len(inside) >= 3 else (near, f"timed region +- {margin} s")
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": window}
        reasons = sorted({x for r in used for x in r["reasons"]})
        return {"sm_mhz": statistics.median(r["sm"] for r in used), "sm_max_mhz": max(r["smax"] for r in used),
                "sm_mhz_min": min(r["sm"] for r in used), "reasons": reasons, "samples": len(used),
                "samples_inside": len(inside), "window": window}


def gpu_id_for(device) -> str:
    import torch

    try:
        u = str(torch.cuda.get_device_properties(device).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:  # noqa: BLE001
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        idx = torch.cuda.current_device() if device is None else torch.device(device).index or 0
        return vis.split(",")[idx] if vis else str(idx)


# ----------------------------------------------------------------------------
# CPU oracle timing (baseline leg and reference arm)


def oracle_fp8_pools(batch, scale: float):
    """The batch's pools as E4M3 codes from the oracle's encoder: E4M3(fp32(x) / scale) per element."""
    import numpy as np

    import oracle

    with np.errstate(invalid="ignore", over="ignore"):
        vals = oracle.widen_np(np.arange(65536, dtype=np.uint32).astype(np.uint16), batch.dtype).astype(np.float32)
        lut = oracle.e4m3_encode_np(vals / np.float32(scale))
    return lut[batch.key_cache], lut[batch.value_cache]


def time_oracle(batch, seqs, budget_s: float, min_reps: int = 1, fp8_pools=None):
    """Run the oracle over the given sequences (all heads) until budget_s; returns (seconds, reps).
    fp8_pools: (key codes, value codes) of an FP8 cache with k_scale = v_scale = FP8_SCALE."""
    import numpy as np

    import oracle

    pairs = np.array([(s, h) for s in seqs for h in range(batch.num_heads)], dtype=np.int32)
    kc, vc = fp8_pools if fp8_pools is not None else (batch.key_cache, batch.value_cache)
    sc = FP8_SCALE if fp8_pools is not None else 1.0
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.decode_c(batch.query, kc, vc, batch.block_tables, batch.context_lens,
                        batch.scale, batch.dtype, pairs=pairs, k_scale=sc, v_scale=sc)
        reps += 1
        el = time.perf_counter() - t0
        if reps >= min_reps and el >= budget_s:
            return el, reps


def sample_kv_bytes(batch, seqs, cache_bytes: int = 2):
    ctx = batch.context_lens[list(seqs)].astype("int64").sum()
    return int(ctx) * batch.num_kv_heads * batch.head_dim * 2 * cache_bytes


# ----------------------------------------------------------------------------


def mq_summary(batch, tile_arg, call_ms, fp8=False):
    """The multi-query tile that ran and the rate of its attention arithmetic (causal QK and PV, 4 flops per
    (row, visible position, dim))."""
    import numpy as np

    ql = np.diff(batch.query_start_loc).astype(np.int64)
    ctx = batch.context_lens.astype(np.int64)
    vis = (ql * (ctx - ql) + ql * (ql + 1) // 2).sum()  # positions seen, summed over query tokens
    flops = 4.0 * batch.head_dim * batch.num_heads * float(vis)
    rows_per_kv_head = int(ql.max()) * (batch.num_heads // batch.num_kv_heads)
    if tile_arg != "auto":
        tile = tile_arg
    elif rows_per_kv_head > (32 if fp8 else 16):
        tile = "tensor"
    else:
        tile = "pairs" if fp8 and rows_per_kv_head > 8 else "columns"
    if fp8 and tile == "rows":
        tile = "columns"  # no FP8 form of the 64-row tile
    if not fp8 and tile == "pairs":
        tile = "columns"  # the 16-row pairs exist for FP8 pools only
    return {"tile": tile, "rows_per_kv_head": rows_per_kv_head, "attention_gflop_per_call": round(flops / 1e9, 2),
            "attention_tflops": round(flops / (call_ms * 1e-3) / 1e12, 1)}


def workload_config(batch, n, partition_size, pool_bytes, fp8=False):
    import numpy as np

    from paged_kv_cache_91_gb300 import workloads as W

    extra = {"query_dtype": batch.dtype, "k_scale": FP8_SCALE, "v_scale": FP8_SCALE} if fp8 else {}
    if batch.query_start_loc is not None:
        ql = np.diff(batch.query_start_loc)
        extra.update({"query_tokens_per_step": int(ql.sum()), "query_len": {"min": int(ql.min()), "max": int(ql.max())},
                      "attention": "multi-query, causal within each sequence's last query_len positions"})
    return {
        "workload": W.CONFIG_NAMES[n] + (" with an FP8 (E4M3) KV cache" if fp8 else "")
        + ("" if batch.query_start_loc is None else
           f", {int(np.diff(batch.query_start_loc).max())} query tokens per sequence"),
        "num_seqs": batch.num_seqs, "num_heads": batch.num_heads, "num_kv_heads": batch.num_kv_heads,
        "head_dim": batch.head_dim, "block_size": batch.block_size, "cache_dtype": "e4m3" if fp8 else batch.dtype,
        **extra,
        "context_lens": {"min": int(batch.context_lens.min()), "mean": float(batch.context_lens.mean()),
                         "max": int(batch.context_lens.max())},
        "partition_size": partition_size or default_partition(fp8, batch.query_start_loc is not None,
                                                              batch.block_size, batch.max_context_len),
        "new_tokens_per_step": int((batch.slot_mapping >= 0).sum()),
        "pool_bytes": pool_bytes,
        "l2": "inputs larger than L2 (KV pool > 129 MB); no flush between steps",
    }


def run_reference(args, dist):
    if dist.rank != 0:
        return
    import numpy as np

    import oracle
    from paged_kv_cache_91_gb300 import workloads as W

    batch = W.make_config(args.config)
    S = batch.num_seqs
    fp8 = args.kv_dtype == "fp8_e4m3"
    pools = oracle_fp8_pools(batch, FP8_SCALE) if fp8 else None
    cb = 1 if fp8 else 2
    # size each step's sample so warm-up + timed steps take about two minutes
    t_one, _ = time_oracle(batch, [0], 0.0, fp8_pools=pools)
    per_seq = max(t_one, 1e-4)
    total_steps = args.steps + args.warmup
    nseq = int(max(1, min(S, 120.0 / (total_steps * per_seq))))
    rng = np.random.default_rng(7)
    times = []
    kv_total = 0
    for k in range(total_steps):
        seqs = sorted(rng.choice(S, size=nseq, replace=False).tolist())
        t0 = time.perf_counter()
        time_oracle(batch, seqs, 0.0, fp8_pools=pools)
        dt = time.perf_counter() - t0
        if k >= args.warmup:
            times.append(dt)
            kv_total += sample_kv_bytes(batch, seqs, cb)
    total = sum(times)
    value = kv_total / total / 1e9
    cores = oracle.max_threads()
    sample = f"{nseq} of {S} sequences (all {batch.num_heads} heads) per step, drawn at random"
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "impl": "reference", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total / len(times), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(batch, args.config, args.partition_size, int(batch.key_cache.nbytes * cb), fp8),
        "tokens_per_s": round(nseq * len(times) / total, 3),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


class Case:
    """One timed configuration: a batch resident on the device and the library calls of its step (the
    cache write of the step's new tokens, then the attention call)."""

    def __init__(self, batch, config: int, dev, *, fp8=False, shared=False, partition_size=0, mq_tile="auto"):
        import numpy as np
        import torch

        from paged_kv_cache_91_gb300 import binding
        from paged_kv_cache_91_gb300 import workloads as W

        self.binding = binding
        self.batch, self.config, self.dev = batch, config, dev
        self.fp8, self.shared, self.P = fp8, shared, partition_size
        self.mq = batch.query_start_loc is not None
        self.mq_tile = mq_tile
        if shared and (self.mq or config != 4):
            raise SystemExit("--shared-prefix runs workload 4 (one query token per sequence)")
        self.apply_settings()
        t = W.as_torch(batch, dev)
        self.t = t
        self.max_query_len = int(np.diff(batch.query_start_loc).max()) if self.mq else 1
        self.n_query_rows = int(batch.query_start_loc[-1]) if self.mq else batch.num_seqs
        self.out = torch.empty_like(t["query"])
        self.mcl = batch.max_context_len
        if shared:
            # the call's own inputs: the common prefix's blocks, then each sequence's tail table and length
            pb, tails, tail_lens = W.split_shared_prefix(batch, SHARED_PREFIX_TOKENS)
            self.prefix_dev = torch.from_numpy(pb).to(dev)
            t["block_tables"] = torch.from_numpy(tails).to(dev)
            t["context_lens"] = torch.from_numpy(tail_lens).to(dev)
            self.max_tail = int(tail_lens.max())
            ws_bytes = binding.paged_attention_shared_prefix_workspace_size(
                batch.num_seqs, batch.num_heads, batch.num_kv_heads, batch.head_dim, batch.block_size,
                SHARED_PREFIX_TOKENS, self.max_tail)
        elif self.mq:
            ws_bytes = binding.paged_attention_multi_query_workspace_size(
                self.n_query_rows, batch.num_heads, batch.num_kv_heads, batch.head_dim, batch.block_size,
                self.mcl, partition_size)
        else:
            wsize = binding.paged_attention_workspace_size_fp8 if fp8 else binding.paged_attention_workspace_size
            ws_bytes = wsize(batch.num_seqs, batch.num_heads, batch.num_kv_heads, batch.head_dim, batch.block_size,
                             self.mcl, partition_size)
        self.ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
        self.stream = torch.cuda.current_stream(dev)
        self.nparts = -(-self.mcl // (partition_size or default_partition(fp8, self.mq, batch.block_size, self.mcl)))
        self.launches_per_step = 2 + (1 if self.nparts > 1 else 0)
        self.cache_bytes = 1 if fp8 else 2
        self.kv_bytes, self.call_bytes = step_bytes(batch, partition_size, self.cache_bytes)
        if shared:
            self.launches_per_step = 4  # write, prefix, tails, merge
            self.call_bytes = shared_prefix_call_bytes(batch, SHARED_PREFIX_TOKENS, ws_bytes, self.cache_bytes)
        self.unique_kv_bytes = (W.unique_kv_bytes(batch) * self.cache_bytes // batch.elem_bytes
                                if batch.meta.get("shared_prefix_tokens") else self.kv_bytes)
        if fp8:
            # the FP8 pool: every slot of the 16-bit pool quantized by the library's own write (setup, untimed)
            NB, Hkv, B, D = t["key_cache"].shape
            kc, vc = (torch.empty((NB, Hkv, B, D), dtype=torch.uint8, device=dev) for _ in range(2))
            all_slots = torch.arange(NB * B, dtype=torch.int64, device=dev)
            binding.paged_kv_write_fp8(t["key_cache"].permute(0, 2, 1, 3).reshape(NB * B, Hkv, D),
                                       t["value_cache"].permute(0, 2, 1, 3).reshape(NB * B, Hkv, D), kc, vc,
                                       all_slots, FP8_SCALE, FP8_SCALE, stream=self.stream)
            torch.cuda.synchronize()
            del all_slots
            t["key_cache"], t["value_cache"] = kc, vc

    def apply_settings(self):
        b = self.binding
        b.set_multi_query_tile({"auto": b.MQ_TILE_AUTO, "columns": b.MQ_TILE_COLUMNS, "rows": b.MQ_TILE_ROWS,
                                "tensor": b.MQ_TILE_TENSOR, "pairs": b.MQ_TILE_PAIRS}[self.mq_tile])

    def write(self, nk, nv, sm):
        b, t = self.binding, self.t
        if self.fp8:
            b.paged_kv_write_fp8(nk, nv, t["key_cache"], t["value_cache"], sm, FP8_SCALE, FP8_SCALE,
                                 stream=self.stream)
        else:
            b.paged_kv_write(nk, nv, t["key_cache"], t["value_cache"], sm, stream=self.stream)

    def decode(self, q, bt, cl, o, qsl=None):
        b, t, batch, P, ws, st = self.binding, self.t, self.batch, self.P, self.ws, self.stream
        kc, vc = t["key_cache"], t["value_cache"]
        if self.shared and self.fp8:  # bt, cl: the tail tables and lengths
            b.paged_attention_decode_shared_prefix_fp8(o, q, kc, vc, self.prefix_dev, SHARED_PREFIX_TOKENS, bt, cl,
                                                       batch.scale, FP8_SCALE, FP8_SCALE,
                                                       max_tail_len=self.max_tail, workspace=ws, stream=st)
        elif self.shared:
            b.paged_attention_decode_shared_prefix(o, q, kc, vc, self.prefix_dev, SHARED_PREFIX_TOKENS, bt, cl,
                                                   batch.scale, max_tail_len=self.max_tail, workspace=ws, stream=st)
        elif self.mq and self.fp8:
            b.paged_attention_multi_query_fp8(o, q, kc, vc, bt, cl, qsl, batch.scale, FP8_SCALE, FP8_SCALE,
                                              max_query_len=self.max_query_len, max_context_len=self.mcl,
                                              partition_size=P, workspace=ws, stream=st)
        elif self.mq:
            b.paged_attention_multi_query(o, q, kc, vc, bt, cl, qsl, batch.scale, max_query_len=self.max_query_len,
                                          max_context_len=self.mcl, partition_size=P, workspace=ws, stream=st)
        elif self.fp8:
            b.paged_attention_decode_fp8(o, q, kc, vc, bt, cl, batch.scale, FP8_SCALE, FP8_SCALE,
                                         max_context_len=self.mcl, partition_size=P, workspace=ws, stream=st)
        else:
            b.paged_attention_decode(o, q, kc, vc, bt, cl, batch.scale, max_context_len=self.mcl, partition_size=P,
                                     workspace=ws, stream=st)

    def step(self, q, nk, nv, sm, bt, cl, o, qsl=None):
        self.write(nk, nv, sm)
        self.decode(q, bt, cl, o, qsl)

    def device_args(self):
        t = self.t
        return (t["query"], t["new_key"], t["new_value"], t["slot_mapping"], t["block_tables"], t["context_lens"],
                self.out, t.get("query_start_loc"))

    def time_device(self, K: int, warmup: int, dist):
        """K steps with every input resident in HBM, timed twice on the launching stream: first with events
        around the whole region only (the step time: value and ms_per_step), then with events around each
        attention call and before each write as well (the call's own time, for the roofline; events between
        the launches cost the step a little)."""
        import torch

        self.apply_settings()
        t, st = self.t, self.stream
        for _ in range(warmup):
            self.step(*self.device_args())
        torch.cuda.synchronize()
        self.binding.device_errors(clear=True)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        dist.barrier()
        t_wall0 = time.time()
        start.record(st)
        for _ in range(K):
            self.write(t["new_key"], t["new_value"], t["slot_mapping"])
            self.decode(t["query"], t["block_tables"], t["context_lens"], self.out, t.get("query_start_loc"))
        end.record(st)
        torch.cuda.synchronize()
        dist.barrier()
        total_ms = dist.max(start.elapsed_time(end))
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        ev_w = [torch.cuda.Event(enable_timing=True) for _ in range(K)]  # before each step's write
        for k in range(K):
            ev_w[k].record(st)
            self.write(t["new_key"], t["new_value"], t["slot_mapping"])
            ev[k][0].record(st)
            self.decode(t["query"], t["block_tables"], t["context_lens"], self.out, t.get("query_start_loc"))
            ev[k][1].record(st)
        torch.cuda.synchronize()
        t_wall1 = time.time()
        return dict(total_ms=total_ms, call_ms=statistics.fmean(a.elapsed_time(b) for a, b in ev),
                    write_ms=statistics.fmean(w.elapsed_time(a) for w, (a, _) in zip(ev_w, ev)),
                    t0=t_wall0, t1=t_wall1, errors=self.binding.device_errors(clear=True))

    def time_e2e(self, K: int, warmup: int, dist):
        """The same step through the public API with the step's inputs copied from pinned host memory and
        the output read back, every step. The pool stays resident: it is the cache. The uploads and the
        downloads run on two more streams, into and out of two alternating sets of device buffers, so that
        step k + 1's inputs upload (and step k - 1's output downloads) while step k computes; events order
        every copy against the steps that use its buffers. (With one stream for both, step k + 1's uploads
        queued behind step k's download, which waits for step k.)"""
        import torch

        self.apply_settings()
        t, st = self.t, self.stream
        names = ("query", "new_key", "new_value", "slot_mapping", "block_tables", "context_lens") + \
            (("query_start_loc",) if self.mq else ())
        host = {k: t[k].cpu().pin_memory() for k in names}
        dbuf = [{k: torch.empty_like(t[k]) for k in names} for _ in range(2)]
        outs = [torch.empty_like(self.out) for _ in range(2)]
        out_h = [torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory() for _ in range(2)]
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        d2h = out_h[0].numel() * out_h[0].element_size()
        cs = torch.cuda.Stream(self.dev)  # uploads
        ds = torch.cuda.Stream(self.dev)  # downloads
        ev = lambda: torch.cuda.Event()  # noqa: E731
        uploaded = [ev(), ev()]   # inputs of the set are on the device
        consumed = [ev(), ev()]   # the step that read the set (and wrote its output) has run
        downloaded = [ev(), ev()]  # the set's output is back on the host

        def run(n):
            for k in range(n):
                i = k & 1
                with torch.cuda.stream(cs):
                    if k >= 2:
                        cs.wait_event(consumed[i])  # step k - 2 has finished with this set
                    for name in names:
                        dbuf[i][name].copy_(host[name], non_blocking=True)
                    uploaded[i].record(cs)
                st.wait_event(uploaded[i])
                if k >= 2:
                    st.wait_event(downloaded[i])  # step k - 2's output is read out before this one overwrites it
                b = dbuf[i]
                self.step(b["query"], b["new_key"], b["new_value"], b["slot_mapping"], b["block_tables"],
                          b["context_lens"], outs[i], b.get("query_start_loc"))
                consumed[i].record(st)
                with torch.cuda.stream(ds):
                    ds.wait_event(consumed[i])
                    out_h[i].copy_(outs[i], non_blocking=True)
                    downloaded[i].record(ds)
            st.wait_stream(ds)  # the last output is on the host before the region ends

        run(warmup)
        torch.cuda.synchronize()
        dist.barrier()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(st)
        cs.wait_event(s0)  # no copy of the timed steps starts before the region
        ds.wait_event(s0)
        run(K)
        s1.record(st)
        torch.cuda.synchronize()
        dist.barrier()
        e2e_ms = dist.max(s0.elapsed_time(s1))
        return dict(ms=e2e_ms / K, h2d=int(h2d), d2h=int(d2h))

    def time_graph(self, K: int, replays: int = 20):
        """us per step with K steps captured in one CUDA graph and replayed: the device-side latency of the
        step, without the per-call host work (for the launch-bound tiny batch)."""
        import torch

        self.apply_settings()
        t = self.t
        side = torch.cuda.Stream(self.dev)
        side.wait_stream(torch.cuda.current_stream(self.dev))
        main, self.stream = self.stream, side  # the calls take the capturing stream
        try:
            with torch.cuda.stream(side):
                self.step(*self.device_args())  # warm the calls on the capturing stream
            torch.cuda.current_stream(self.dev).wait_stream(side)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                for _ in range(K):
                    self.write(t["new_key"], t["new_value"], t["slot_mapping"])
                    self.decode(t["query"], t["block_tables"], t["context_lens"], self.out, t.get("query_start_loc"))
        finally:
            self.stream = main
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(replays):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        return 1e3 * a.elapsed_time(b) / (replays * K)

    def kernel_kind(self) -> str:
        G = self.batch.num_heads // self.batch.num_kv_heads
        if self.mq:
            kind = "mq_fp8" if self.fp8 else "mq"
            if mq_summary(self.batch, self.mq_tile, 1.0, self.fp8)["tile"] == "pairs":
                kind = "mq_fp8_pairs"
            return kind
        if self.fp8:
            return "mma_fp8" if G <= 8 and self.batch.head_dim == 128 else "simt_fp8"
        return "mma" if 2 <= G <= 8 else "simt"

    def workload_key(self) -> str:
        return (f"cfg{self.config}" + ("-fp8" if self.fp8 else "")
                + (f"-q{self.max_query_len}" if self.mq else "") + ("-shared" if self.shared else ""))

    def call_name(self) -> str:
        if self.shared:
            return "paged_attention_decode_shared_prefix" + ("_fp8" if self.fp8 else "")
        if self.mq:
            return "paged_attention_multi_query" + ("_fp8" if self.fp8 else "")
        return "paged_attention_decode" + ("_fp8" if self.fp8 else "")

    def roofline(self, call_ms: float):
        peak, peak_kind = hbm_peak()
        # a shared-prefix batch must bring each shared block from HBM once: its roofline counts unique bytes
        hbm_bytes = self.call_bytes - (self.kv_bytes - self.unique_kv_bytes) if not self.shared else self.call_bytes
        achieved = hbm_bytes / (call_ms / 1e3) / 1e9
        what = ("prefix, tail and merge kernels; bytes: the prefix once, the tails, q, out, partials" if self.shared
                else ("multi-query kernel" if self.mq else "decode kernel")
                + (" + log-sum-exp reduce" if self.nparts > 1 else ""))
        traffic = None if self.shared else ncu_traffic(self.workload_key(), self.kernel_kind())
        tile = self.batch.block_size * self.batch.head_dim * self.cache_bytes  # bytes of one (block, kv head) tile
        ceil = read_ceiling(self.dev, tile)
        return {"bound": "hbm", "kernel": f"{self.call_name()} ({what})", "achieved": round(achieved, 2),
                "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                "frac_of_spec_8tbs": round(achieved / SPEC_HBM_GBS, 4), "traffic": traffic,
                "algorithmic_bytes_per_call": int(hbm_bytes), "avg_call_ms": round(call_ms, 4),
                "kernel_hash": kernel_hash(self.kernel_kind()),
                "read_ceiling": None if ceil is None else {
                    "gbs": ceil, "frac": round(achieved / ceil, 4), "chunk_bytes": tile,
                    "what": "pkv_read_chunks over random whole tiles of a 2 GiB buffer (read only, no arithmetic)"}}

    def close(self):
        import torch

        self.t.clear()
        self.out = self.ws = None
        torch.cuda.empty_cache()


SPEC_HBM_GBS = 8000.0  # GB300's nominal HBM3e bandwidth

_CEILING = {}


def read_ceiling(dev, chunk_bytes: int, buf_bytes: int = 2 << 30, reps: int = 5):
    """GB/s of the library's read helper over a random order of whole chunk_bytes chunks of a 2 GiB buffer
    (larger than L2): the read ceiling of the decode's access pattern, where every (block, kv head) tile is
    such a chunk at a random place in the pool. Measured once per chunk size and process."""
    if chunk_bytes not in (1024, 2048, 4096, 8192):
        return None
    if chunk_bytes in _CEILING:
        return _CEILING[chunk_bytes]
    import torch

    from paged_kv_cache_91_gb300 import binding

    buf = torch.empty(buf_bytes, dtype=torch.uint8, device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(11)
    order = torch.randperm(buf_bytes // chunk_bytes, device=dev, dtype=torch.int32, generator=gen)
    st = torch.cuda.current_stream(dev)
    for _ in range(2):
        binding.read_chunks(buf, order, chunk_bytes, stream=st)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(st)
    for _ in range(reps):
        binding.read_chunks(buf, order, chunk_bytes, stream=st)
    b.record(st)
    torch.cuda.synchronize()
    gbs = round(order.numel() * chunk_bytes * reps / (a.elapsed_time(b) / 1e3) / 1e9, 1)
    del buf, order
    torch.cuda.empty_cache()
    _CEILING[chunk_bytes] = gbs
    return gbs


def cpu_oracle(batch, budget_s: float, threads: int, fp8: bool, seed: int = 7):
    """The oracle, as it stands, on a seeded random sample of the batch's sequences (compact pool, all heads,
    every query row), repeated until budget_s. Returns a cpu_baseline dict: KV GB/s of the sample's contexts,
    the threads used and what the sample was."""
    import numpy as np

    import oracle
    from paged_kv_cache_91_gb300 import workloads as W

    S = batch.num_seqs
    order = np.random.default_rng(seed).permutation(S).tolist()
    cb = 1 if fp8 else 2

    def run(sb):
        kc, vc, sc = sb.key_cache, sb.value_cache, 1.0
        if fp8:
            kc, vc = oracle_fp8_pools(sb, FP8_SCALE)
            sc = FP8_SCALE
        t0 = time.perf_counter()
        if sb.query_start_loc is None:
            oracle.decode_c(sb.query, kc, vc, sb.block_tables, sb.context_lens, sb.scale, sb.dtype,
                            num_threads=threads, k_scale=sc, v_scale=sc)
        else:
            oracle.multi_query_c(sb.query, kc, vc, sb.block_tables, sb.context_lens, sb.query_start_loc, sb.scale,
                                 sb.dtype, num_threads=threads, k_scale=sc, v_scale=sc)
        return time.perf_counter() - t0

    # size the sample from one sequence's time, so that one pass takes about a third of the budget
    one = W.sub_batch(batch, order[:1])
    t_one = max(run(one), 1e-4) / max(1, sample_kv_bytes(one, [0], cb))
    n = 1
    while n < S and sample_kv_bytes(batch, order[:n + 1], cb) * t_one < budget_s / 3:
        n += 1
    seqs = sorted(order[:n])
    sb = W.sub_batch(batch, seqs)
    el, reps = 0.0, 0
    while reps == 0 or el < budget_s:
        el += run(sb)
        reps += 1
    kv = sample_kv_bytes(batch, seqs, cb)
    rows = int(sb.query_start_loc[-1]) if sb.query_start_loc is not None else n
    return {"value": round(kv * reps / el / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} of {S} sequences ({rows} query rows x {batch.num_heads} heads), drawn at random, "
                      f"{reps} pass(es), fp64, {el:.1f} s"}


def entry_summary(case: Case, dev_t, e2e_t, clocks, cpu, steps: int):
    """One workload's figures: per-call and per-step times, KV GB/s, roofline, e2e, clocks, CPU oracle."""
    b = case.batch
    step_s = dev_t["total_ms"] / steps / 1e3
    e = {
        "workload": workload_config(b, case.config, case.P, int(b.key_cache.nbytes * case.cache_bytes // 2),
                                    case.fp8)["workload"],
        "call": case.call_name(), "cache_dtype": "e4m3" if case.fp8 else b.dtype, "steps": steps,
        "ms_per_step": round(dev_t["total_ms"] / steps, 4), "call_ms": round(dev_t["call_ms"], 4),
        "write_call_ms": round(dev_t["write_ms"], 4), "new_tokens_per_step": int((b.slot_mapping >= 0).sum()),
        "kv_gbs": round(case.kv_bytes / step_s / 1e9, 2), "kv_bytes_per_step": int(case.kv_bytes),
        "tokens_per_s": round(case.n_query_rows / step_s, 1),
        "roofline": case.roofline(dev_t["call_ms"]),
        "e2e": None if e2e_t is None else {
            "value": round(case.kv_bytes / (e2e_t["ms"] / 1e3) / 1e9, 2), "unit": "GB/s",
            "ms_per_step": round(e2e_t["ms"], 4), "h2d_bytes_per_step": e2e_t["h2d"],
            "d2h_bytes_per_step": e2e_t["d2h"]},
        "gpu_launches_per_step": case.launches_per_step, "clocks": clocks, "device_errors": dev_t["errors"],
        "cpu_baseline": cpu,
    }
    if case.unique_kv_bytes != case.kv_bytes:
        e["unique_kv_bytes_per_step"] = int(case.unique_kv_bytes)
        e["kv_gbs_note"] = "kv_gbs counts every sequence's prefix (logical bytes; repeats come from L2)"
    if case.mq:
        e["multi_query"] = mq_summary(b, case.mq_tile, dev_t["call_ms"], case.fp8)
    if b.num_seqs <= 4:  # the tiny batch is launch-bound: its figures are latencies
        e["us_per_step"] = round(1e3 * dev_t["total_ms"] / steps, 2)
        e["call_us"] = round(1e3 * dev_t["call_ms"], 2)
        e["write_us"] = round(1e3 * dev_t["write_ms"], 2)
        if e2e_t is not None:
            e["e2e"]["us_per_step"] = round(1e3 * e2e_t["ms"], 2)
    return e


# The workloads the default run measures beside the headline: (key, config, options). Each is timed with
# its own events; multi-query batches reuse the pool of their workload.
SUITE = [
    ("w2_fp8", 2, {"fp8": True}),
    ("w2_q4", 2, {"query_len": 4}),
    ("w2_q128", 2, {"query_len": 128}),
    ("w2_q128_fp8", 2, {"query_len": 128, "fp8": True}),
    ("w1_tiny", 1, {}),
    ("w3_gqa_bf16", 3, {}),
    ("w3_fp8", 3, {"fp8": True}),
    ("w3_q32", 3, {"query_len": 32}),
    ("w3_q4_fp8", 3, {"query_len": 4, "fp8": True}),
    ("w3_q32_fp8", 3, {"query_len": 32, "fp8": True}),
    ("w4_shared_prefix", 4, {}),
    ("w4_shared_prefix_call", 4, {"shared": True}),
    ("w4_fp8", 4, {"fp8": True}),
    ("w4_shared_prefix_call_fp8", 4, {"shared": True, "fp8": True}),
    ("w5_long_split_k", 5, {}),
    ("w5_fp8", 5, {"fp8": True}),
]


def run_suite(args, dist, dev, base_batch):
    """Every other workload, one after another, each with its own timed region (args.suite_steps steps)."""
    import numpy as np

    from paged_kv_cache_91_gb300 import workloads as W

    results = {}
    # one workload's pool at a time in host memory; the headline's batch serves the suite's entries of its
    # workload, which come first
    batches = {args.config: base_batch} if args.max_seqs is None and args.block_size == 16 else {}
    cpu_on = dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline
    for key, n, opt in SUITE:
        if n not in batches:
            batches = {n: W.make_config(n)}
        batch = batches[n]
        if opt.get("query_len"):
            batch = W.with_query_lens(batch, np.minimum(batch.context_lens, opt["query_len"]))
        case = Case(batch, n, dev, fp8=opt.get("fp8", False), shared=opt.get("shared", False))
        K = args.suite_steps
        dev_t = case.time_device(K, args.warmup, dist)
        e2e_t = None if args.no_e2e else case.time_e2e(K, args.warmup, dist)
        cpu = cpu_oracle(batch, args.suite_cpu_seconds, _all_cores(), case.fp8) if cpu_on else None
        results[key] = entry_summary(case, dev_t, e2e_t, None, cpu, K)
        if batch.num_seqs <= 4:  # launch-bound: the step also from a CUDA graph
            results[key]["graph_us_per_step"] = round(case.time_graph(100), 2)
        results[key]["_window"] = (dev_t["t0"], dev_t["t1"])
        case.close()
    return results


def _all_cores() -> int:
    import oracle

    try:
        n = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        n = os.cpu_count() or 1
    return max(1, min(n, oracle.max_threads()))


def run_ours(args, dist):
    import torch

    from paged_kv_cache_91_gb300 import binding
    from paged_kv_cache_91_gb300 import workloads as W

    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    binding.load()
    batch = W.make_config(args.config, max_seqs=args.max_seqs, block_size=args.block_size,
                          query_len=args.query_len)
    case = Case(batch, args.config, dev, fp8=args.kv_dtype == "fp8_e4m3", shared=args.shared_prefix,
                partition_size=args.partition_size, mq_tile=args.mq_tile)
    sampler = ClockSampler(gpu_id_for(dev))
    K = args.steps
    dev_t = case.time_device(K, args.warmup, dist)
    e2e_t = None if args.no_e2e else case.time_e2e(K, args.warmup, dist)
    total_ms = dev_t["total_ms"]

    cpu = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        cores = _all_cores()
        cpu = cpu_oracle(batch, args.cpu_seconds, cores, case.fp8)
        single = cpu_oracle(batch, args.cpu_seconds / 2, 1, case.fp8)
        cpu["single_thread"] = {"value": single["value"], "unit": "GB/s", "cores": 1, "sample": single["sample"]}
    case.close()

    suite = None
    if not args.no_suite and dist.world == 1 and args.query_len is None and not args.shared_prefix \
            and args.kv_dtype == "auto":
        suite = run_suite(args, dist, dev, batch)

    rows = sampler.stop()
    clocks = ClockSampler.summarise(rows, dev_t["t0"], dev_t["t1"])
    if suite:
        for e in suite.values():
            e["clocks"] = ClockSampler.summarise(rows, *e.pop("_window"))

    value = dist.sum(case.kv_bytes) * K / (total_ms / 1e3) / 1e9
    peak, _ = hbm_peak()
    if dist.rank == 0:
        b = case.batch
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": dist.world, "steps": K,
            "warmup": args.warmup, "ms_per_step": round(total_ms / K, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3" if case.fp8 else ("f16" if b.dtype == "f16" else "bf16"),
            "accumulate": "f32", "data": "synthetic (seeded N(0,1) K/V/q, block tables from a shuffled free list)",
            "config": workload_config(b, args.config, args.partition_size, int(b.key_cache.nbytes * case.cache_bytes
                                                                               // 2), case.fp8),
            "tokens_per_s": round(case.n_query_rows * dist.world * K / (total_ms / 1e3), 1),
            "pct_of_peak": {"measured_hbm": round(100 * value / dist.world / peak, 2),
                            "spec_8tbs": round(100 * value / dist.world / SPEC_HBM_GBS, 2)},
            "roofline": case.roofline(dev_t["call_ms"]),
            "write_call_ms": round(dev_t["write_ms"], 4),
            "attention_only_model_tokens_per_s": model_extrapolation(args.config, case.n_query_rows * dist.world * K
                                                                     / (total_ms / 1e3)),
            "gpu_launches": K * case.launches_per_step,
            "clocks": clocks,
            "device_errors": dev_t["errors"],
            "e2e": None if e2e_t is None else {
                "value": round(dist.sum(case.kv_bytes) / (e2e_t["ms"] / 1e3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": e2e_t["h2d"], "d2h_bytes_per_step": e2e_t["d2h"],
                "ms_per_step": round(e2e_t["ms"], 4)},
            "cpu_baseline": cpu,
        }
        if case.mq:
            line["multi_query"] = mq_summary(b, args.mq_tile, dev_t["call_ms"], case.fp8)
        if case.shared:
            line["config"]["call"] = (f"paged_attention_decode_shared_prefix: the {SHARED_PREFIX_TOKENS}-token "
                                      "prefix attended once for the whole batch, then each tail, then a merge")
        if suite:
            line["workloads"] = suite
            line["workloads_note"] = (f"each entry: {args.suite_steps} steps of its own after {args.warmup} warm-up "
                                      "steps, events on the launching stream; inputs larger than L2 except w1 "
                                      "(a latency case); cpu_baseline: the oracle on all host cores over a "
                                      "random sample of the workload's sequences")
        print(json.dumps(line), flush=True)


def run_copy_blocks(args, dist):
    """Time paged_kv_copy_blocks: 256 disjoint (src, dst) block pairs of the workload's pool per call."""
    import numpy as np
    import torch

    from paged_kv_cache_91_gb300 import binding
    from paged_kv_cache_91_gb300 import workloads as W

    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    batch = W.make_config(args.config, max_seqs=args.max_seqs, block_size=args.block_size)
    t = W.as_torch(batch, dev)
    NB = batch.num_blocks
    npairs = min(256, NB // 2)
    perm = np.random.default_rng(9).permutation(NB)
    mapping = torch.from_numpy(np.stack([perm[:npairs], perm[npairs:2 * npairs]], axis=1).astype(np.int64)).to(dev)
    block_bytes = batch.num_kv_heads * batch.block_size * batch.head_dim * 2
    moved = 2 * 2 * npairs * block_bytes  # K and V, read and written
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        binding.paged_kv_copy_blocks(t["key_cache"], t["value_cache"], mapping, stream=stream)
    K = args.steps
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    dist.barrier()
    a.record(stream)
    for _ in range(K):
        binding.paged_kv_copy_blocks(t["key_cache"], t["value_cache"], mapping, stream=stream)
    b.record(stream)
    torch.cuda.synchronize()
    ms = dist.max(a.elapsed_time(b))
    peak, peak_kind = hbm_peak()
    gbs = dist.sum(moved) * K / (ms / 1e3) / 1e9
    if dist.rank == 0:
        print(json.dumps({
            "metric": "copy-on-write block copy: HBM GB/s (read + write)", "op": "copy_blocks", "value": round(gbs, 2),
            "unit": "GB/s", "n_gpus": dist.world, "steps": K, "warmup": args.warmup,
            "ms_per_step": round(ms / K, 4), "higher_is_better": True, "scaling": "weak",
            "config": {"workload": W.CONFIG_NAMES[args.config], "pairs_per_call": npairs,
                       "block_bytes_per_cache": block_bytes},
            "roofline": {"bound": "hbm", "achieved": round(gbs / dist.world, 2), "peak": peak, "peak_kind": peak_kind,
                         "unit": "GB/s", "frac": round(gbs / dist.world / peak, 4)},
            "gpu_launches": K, "device_errors": binding.device_errors()}), flush=True)


def main():
    args = parse_args()
    dist = Dist()
    try:
        if args.impl == "reference":
            run_reference(args, dist)
        elif args.op == "copy-blocks":
            run_copy_blocks(args, dist)
        else:
            run_ours(args, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
