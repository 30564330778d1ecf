/*
 * paged_kv.h -- C ABI of the GB300 (sm_103a) paged KV cache library.
 *
 * Two operations make up the decode-step hot path of PagedAttention:
 *
 *   paged_kv_write          the reshape_and_cache scatter: each new token's key and
 *                           value rows go into the physical slot that slot_mapping
 *                           names.
 *   paged_attention_decode  decode-phase attention of one query token per sequence
 *                           over that sequence's cached tokens, found through its
 *                           block table.
 *
 * Conventions shared by every call:
 *   - Every array pointer is a DEVICE pointer owned by the caller. The library
 *     allocates nothing and keeps no pointer after a call returns.
 *   - Calls are asynchronous on `stream` (0 = the legacy default stream) and never
 *     synchronise, except paged_kv_device_errors.
 *   - Arguments are validated on the host before any CUDA call. A rejected call
 *     launches nothing and returns a negative pkv_status_t;
 *     pkv_last_error_message() then describes the problem.
 *   - Kernels check every block-table entry, slot and context length they read.
 *     A bad one is skipped or clamped (never dereferenced), and a bit is set in
 *     a per-device error word that paged_kv_device_errors reads.
 *   - fp16 and bf16 are supported. Query, caches and output share one dtype,
 *     except in the *_fp8 calls, whose caches hold FP8 (E4M3) codes.
 *
 * KV pool layout (both key_cache and value_cache):
 *     [num_blocks][num_kv_heads][block_size][head_dim], row-major,
 * so the block_size x head_dim tile of one (physical block, kv head) is one
 * contiguous run of block_size * head_dim * 2 bytes. Token j of a sequence lives
 * in physical block block_tables[s][j / block_size] at offset j % block_size.
 * The pages fix the block / block table / slot vocabulary but not the byte
 * layout; it is chosen so a whole tile moves with one bulk copy.
 */
#ifndef PAGED_KV_H_
#define PAGED_KV_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* PKV_FP8_E4M3 names an FP8 cache; it is accepted only where a call says so. */
typedef enum { PKV_F16 = 0, PKV_BF16 = 1, PKV_FP8_E4M3 = 2 } pkv_dtype_t;

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = -1, /* a null pointer, a negative size, inconsistent shapes */
  PKV_ERR_UNSUPPORTED = -2, /* valid, but outside what the kernels are built for    */
  PKV_ERR_WORKSPACE = -3,   /* split-K workspace missing, too small or misaligned   */
  PKV_ERR_CUDA = -4,        /* a CUDA runtime call or a kernel launch failed        */
  PKV_ERR_DEVICE_CHECK = -5 /* paged_kv_device_errors found a device-side error bit */
} pkv_status_t;

/* Bits of the per-device error word (see paged_kv_device_errors). */
#define PKV_DEVERR_BLOCK_ID 1u /* a block-table entry outside [0, num_blocks)            */
#define PKV_DEVERR_CONTEXT 2u  /* a context length < 0 or above max_context_len or
                                  max_blocks_per_seq * block_size (clamped)               */
#define PKV_DEVERR_SLOT 4u     /* a slot_mapping entry >= num_blocks * block_size        */
#define PKV_DEVERR_TIMEOUT 8u  /* a wait for a bulk copy gave up after its time limit   */
#define PKV_DEVERR_QUERY 16u   /* query_start_loc gives a sequence a negative number of
                                  query tokens, more than max_query_len or its context,
                                  or rows outside [0, num_query_tokens)                  */
#define PKV_DEVERR_LAYOUT 32u  /* a kernel found its shared memory misaligned for the
                                  tensor-core operand layout and wrote nothing           */

/*
 * paged_kv_write -- store the step's new keys and values in the paged pool.
 *
 * Source: "[vLLM] PagedAttention: OS 페이징 기법으로 KV 캐시를 관리하는 방법",
 * section "PagedAttention 커널" (write_to_paged_cache -> ops.reshape_and_cache with
 * slot_mapping); slot arithmetic as in "KV Cache와 PagedAttention 완전 해부",
 * §5단계 and §6단계 (the 7th token of a request whose block is 42 goes to slot 6).
 *
 * For every token t with slot = slot_mapping[t] >= 0 and every kv head h:
 *     key_cache  [slot / block_size][h][slot % block_size][:] = key  [t][h][:]
 *     value_cache[slot / block_size][h][slot % block_size][:] = value[t][h][:]
 * as a bit copy. Tokens with a negative slot are padding and are skipped.
 *
 *   key, value          [num_tokens][num_kv_heads][head_dim], contiguous
 *   key_cache, value_cache  the pool, layout above; 16-byte aligned
 *   slot_mapping        [num_tokens] int64
 *   head_dim            64 or 128; block_size 8, 16 or 32
 *
 * Two tokens naming the same slot give an undefined winner. A slot at or past
 * num_blocks * block_size is skipped and sets PKV_DEVERR_SLOT.
 * num_tokens == 0 is a no-op that returns PKV_OK.
 */
pkv_status_t paged_kv_write(const void* key, const void* value, void* key_cache,
                            void* value_cache, const int64_t* slot_mapping, int32_t num_tokens,
                            int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                            int32_t num_blocks, pkv_dtype_t dtype, cudaStream_t stream);

/*
 * paged_kv_copy_blocks -- the copy of copy-on-write: whole physical blocks,
 * every kv head's K and V rows, copied bit for bit.
 *
 * Source: "Sparse Computation and Memory Management for Efficient LLM
 * Inference", Copy-on-Write (append_kv_with_cow copies a shared block to a new
 * one with fused_block_copy before writing into it); "KV Cache와 PagedAttention
 * 완전 해부", §9단계 (shared blocks with reference counts; a write into a shared
 * block copies it first).
 *
 * For each pair i: block block_mapping[2i + 1] (dst) of key_cache and
 * value_cache receives the contents of block block_mapping[2i] (src).
 *
 *   block_mapping   [num_pairs][2] int64 (src, dst), device memory
 *   key_cache, value_cache  the pool, layout above; 16-byte aligned
 *   dtype           the cache's element type: PKV_F16, PKV_BF16 or PKV_FP8_E4M3
 *
 * No block may be both a source and a destination in one call, and
 * destinations must be distinct (the result is otherwise undefined). A pair
 * naming a block outside [0, num_blocks) is skipped and sets
 * PKV_DEVERR_BLOCK_ID. num_pairs == 0 is a no-op; at most 65535 pairs per call.
 */
pkv_status_t paged_kv_copy_blocks(void* key_cache, void* value_cache, const int64_t* block_mapping,
                                  int32_t num_pairs, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t block_size, int32_t num_blocks, pkv_dtype_t dtype,
                                  cudaStream_t stream);

/*
 * paged_attention_workspace_size -- bytes of device workspace that
 * paged_attention_decode needs for its split-K partial results:
 * ceil(max_context_len / partition_size) partitions of num_heads *
 * (head_dim + 2) fp32 per sequence. The size is 0 when max_context_len <=
 * partition_size (no split).
 *
 * partition_size 0 selects the default: 1024, or 2048 when max_context_len >
 * 8192 (at most 128 blocks either way). Returns 0 for invalid arguments,
 * which paged_attention_decode then rejects.
 */
size_t paged_attention_workspace_size(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                      int32_t head_dim, int32_t block_size, int32_t max_context_len,
                                      int32_t partition_size);

/*
 * paged_attention_decode -- one decode step of attention over the paged pool.
 *
 * Source: "KV Cache와 PagedAttention 완전 해부", 부록 (softmax(Q K^T / sqrt d) V,
 * computed block by block through the block table with a running softmax) and
 * §6단계 (decode is matrix-vector and memory-bound); "vLLM: LLM 서빙 메모리 최적화의
 * 교과서", 01 Problem Definition (a_ij, o_i) and eq. (4) (the block-wise form, equal
 * to ordinary attention); "Sparse Computation and Memory Management for Efficient
 * LLM Inference", Block-level Attention Formulation.
 *
 * For every sequence s, query head h, kv head g = h / (num_heads / num_kv_heads)
 * and the first n = context_lens[s] cached tokens:
 *     x_j = scale * dot(query[s][h][:], K_j)        j = 0 .. n-1
 *     out[s][h][:] = sum_j softmax(x)_j * V_j
 * where K_j, V_j are row j % block_size of the (block_tables[s][j / block_size], g)
 * tile. n == 0 gives zeros. Accumulation is fp32; out is rounded to nearest-even
 * into the query dtype.
 *
 *   out, query           [num_seqs][num_heads][head_dim], contiguous, 16-byte aligned
 *   key_cache, value_cache  the pool, layout above; 16-byte aligned
 *   block_tables         [num_seqs][max_blocks_per_seq] int32; entries at or past
 *                        ceil(n / block_size) are never read
 *   context_lens         [num_seqs] int32
 *   max_context_len      host-side upper bound on every context_lens entry; sizes
 *                        the launch (longer contexts are clamped, PKV_DEVERR_CONTEXT)
 *   scale                usually 1 / sqrt(head_dim)
 *   head_dim             64 or 128; block_size 8, 16 or 32
 *   num_heads            a multiple of num_kv_heads (GQA when larger)
 *   partition_size       0 = the default (see paged_attention_workspace_size);
 *                        else a multiple of block_size in
 *                        [block_size, 128 * block_size]: the tokens of one
 *                        CTA's share of a context (contexts longer than this
 *                        are split and merged by log-sum-exp)
 *   workspace            paged_attention_workspace_size(...) bytes, 16-byte aligned;
 *                        may be NULL when that size is 0
 *
 * Rows of out for every (s, h) are written by this call. The workspace is
 * scratch: its contents need no initialisation and are not meaningful after the
 * call. Concurrent calls must not share a workspace.
 */
pkv_status_t paged_attention_decode(void* out, const void* query, const void* key_cache,
                                    const void* value_cache, const int32_t* block_tables,
                                    int32_t max_blocks_per_seq, const int32_t* context_lens,
                                    int32_t num_seqs, int32_t max_context_len, float scale,
                                    int32_t block_size, int32_t num_heads, int32_t num_kv_heads,
                                    int32_t head_dim, int32_t num_blocks, pkv_dtype_t dtype,
                                    int32_t partition_size, void* workspace,
                                    size_t workspace_bytes, cudaStream_t stream);

/* Size of the library-owned split-K scratch of
 * paged_attention_decode_static_workspace: 32 MiB per device. It covers, for
 * example, 16 sequences x 40 heads x 32768-token contexts at partition_size 512
 * (about 5 MiB at the default, 2048 for such contexts). */
#define PKV_STATIC_WORKSPACE_BYTES (32u * 1024u * 1024u)

/*
 * paged_attention_decode_static_workspace -- paged_attention_decode for callers
 * that cannot allocate device memory at call time.
 *
 * The pages have no counterpart to this call; it exists for users of this
 * library. Some callers cannot hand paged_attention_decode a workspace: a plain
 * C host with no device allocator of its own, a process whose device memory is
 * already fully reserved by another allocator (a new cudaMalloc would fail), or
 * a latency-bound decode loop that must not call cudaMalloc (it can synchronise
 * the device). This call takes the same arguments minus the workspace and uses
 * a scratch array compiled into the library instead. It allocates nothing:
 * no cudaMalloc, no cudaFree, no allocating library routine.
 *
 *   - The scratch is PKV_STATIC_WORKSPACE_BYTES of device memory per GPU that
 *     loads the library, held until the process exits.
 *   - The first call on each device (with that device current) looks up the
 *     scratch array's device address with cudaGetSymbolAddress; make that first
 *     call before any stream capture on that device. The address is kept per
 *     device ordinal for the life of the process (the device's primary
 *     context): do not call this entry point on a device after
 *     cudaDeviceReset there.
 *   - A call whose split-K scratch (paged_attention_workspace_size) exceeds
 *     PKV_STATIC_WORKSPACE_BYTES launches nothing and returns PKV_ERR_WORKSPACE,
 *     with the sizes in pkv_last_error_message(). The other arguments are
 *     checked first: a bad one returns its own error, as in
 *     paged_attention_decode.
 *   - Every call on a device shares the one scratch array, which keeps the last
 *     call's contents. Nothing in it needs clearing: each call writes every
 *     partial before reading it. Calls whose kernels overlap on the GPU (other
 *     streams, other host threads) race on the scratch and give wrong results;
 *     keep such calls on one stream, or use paged_attention_decode with
 *     separate workspaces.
 *
 * Results, arguments and every other error behaviour are those of
 * paged_attention_decode.
 */
pkv_status_t paged_attention_decode_static_workspace(
    void* out, const void* query, const void* key_cache, const void* value_cache, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs, int32_t max_context_len,
    float scale, int32_t block_size, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t num_blocks, pkv_dtype_t dtype, int32_t partition_size, cudaStream_t stream);

/*
 * pkv_read_chunks -- a measurement helper with no counterpart on the pages (it
 * is not a step of the method). Reads num_reads chunks of chunk_bytes from
 * `buffer`: read i is chunk order[i], the bytes [order[i] * chunk_bytes,
 * (order[i] + 1) * chunk_bytes). Each chunk is one bulk copy into a per-warp
 * shared-memory ring; nothing is written to global memory. Timed over a random
 * order of whole chunks the size of one (block, kv head) tile, in a buffer
 * larger than L2, it measures the read ceiling of the decode's access pattern
 * (the decode reads every tile as such a chunk at a random place in the pool).
 *
 *   buffer       device memory, 16-byte aligned, buffer_bytes long (caller-owned)
 *   order        [num_reads] int32 chunk indices on the device; an index outside
 *                [0, buffer_bytes / chunk_bytes) is skipped and sets
 *                PKV_DEVERR_BLOCK_ID
 *   chunk_bytes  1024, 2048, 4096 or 8192
 *
 * Asynchronous on `stream`. Returns PKV_OK, PKV_ERR_INVALID_ARG (null or
 * unaligned pointer, negative size), PKV_ERR_UNSUPPORTED (chunk size) or
 * PKV_ERR_CUDA (launch).
 */
pkv_status_t pkv_read_chunks(const void* buffer, int64_t buffer_bytes, const int32_t* order,
                             int64_t num_reads, int32_t chunk_bytes, cudaStream_t stream);

/*
 * paged_kv_device_errors -- read the current device's error word (PKV_DEVERR_* bits
 * set by kernels since it was last cleared) into *flags, and clear it if `clear`
 * is non-zero. Synchronises the current device first. Returns PKV_OK, or
 * PKV_ERR_CUDA if a CUDA call fails. The library sets *flags; callers compare
 * against 0.
 */
pkv_status_t paged_kv_device_errors(uint32_t* flags, int32_t clear);

/*
 * pkv_selftest_wait_timeout -- check the kernels' bounded wait on this GPU.
 * Launches one warp that waits on a shared-memory barrier for 16 bytes that no
 * copy will deliver. After limit_cycles SM cycles (at most about 1 s) the wait
 * gives up and sets PKV_DEVERR_TIMEOUT in the error word, exactly as a decode
 * kernel does when a tile copy never lands. The context stays usable. The
 * pages have no counterpart; this exists to test failure reporting without a
 * GPU fault.
 */
pkv_status_t pkv_selftest_wait_timeout(int64_t limit_cycles, cudaStream_t stream);

/*
 * paged_attention_multi_query -- attention of several query tokens per
 * sequence over the paged pool: a chunked-prefill chunk batched with decode
 * tokens, or the tokens a speculative step verifies.
 *
 * Source: "Sparse Computation and Memory Management for Efficient LLM
 * Inference", the chunked prefill paragraph (prefill chunks share a step with
 * decode tokens) and Speculative Decoding; the causal rule is a_ij and o_i
 * over j <= i, "vLLM: LLM 서빙 메모리 최적화의 교과서", 01 Problem Definition.
 *
 * Sequence s has q_len = query_start_loc[s+1] - query_start_loc[s] query
 * tokens, rows query_start_loc[s] .. + q_len - 1 of query and out. They are its
 * last q_len context positions (their keys and values are already in the pool,
 * written by paged_kv_write), so query token i sits at position
 * p = context_lens[s] - q_len + i and, for every query head h,
 *     out[query_start_loc[s] + i][h][:] = sum_{j <= p} softmax_j(x) * V_j,
 *     x_j = scale * dot(query[query_start_loc[s] + i][h][:], K_j)
 * with K_j, V_j as in paged_attention_decode. q_len = 1 everywhere is exactly
 * paged_attention_decode; q_len = context_lens[s] is causal self-attention over
 * the whole prompt.
 *
 *   out, query        [num_query_tokens][num_heads][head_dim], contiguous, 16-byte aligned
 *   query_start_loc   [num_seqs + 1] int32, device memory: 0, then non-decreasing
 *   num_query_tokens  host-side: query_start_loc[num_seqs] (rows of query and out)
 *   max_query_len     host-side bound on every q_len; sizes the launch; <= max_context_len
 *   partition_size    0 = 2048 tokens, capped at 128 blocks (every query row
 *                     writes a partial per partition, so long partitions are
 *                     fastest here); else as in paged_attention_decode
 *   workspace         paged_attention_multi_query_workspace_size(...) bytes: the
 *                     split-K partials (required when a context spans several
 *                     partitions), then room for one int32 per sequence that
 *                     the 8-column and 128-row tiles fill with the sequences
 *                     ordered by context length, longest first, and dispatch
 *                     their grids in that order (its long items start first, which
 *                     shortens the grid's end). A workspace of only the
 *                     partials' size, or none when there are no partials, is
 *                     accepted: the sequences then run in index order. The
 *                     order changes no result.
 * Everything else is as in paged_attention_decode (the decode-path choice does
 * not apply: this call always runs partitioned, on the tensor cores, for every
 * group size). A sequence whose query_start_loc entries are out of order,
 * give it more than max_query_len or context_lens[s] tokens, or reach past
 * num_query_tokens is skipped (its rows are not written), and the call sets
 * PKV_DEVERR_QUERY.
 */
/*
 * Multi-query tiles (pkv_set_multi_query_tile). All compute the same result,
 * up to rounding order.
 *   PKV_MQ_TILE_COLUMNS  8 (query token, head) rows of one kv head per CTA, in
 *                        the n = 8 dimension of the MMA, the CTA's warps
 *                        splitting the context's blocks. Reads no padding rows
 *                        when a kv head has few rows (e.g. speculative
 *                        verification of a few tokens).
 *   PKV_MQ_TILE_ROWS     64 rows per CTA, 16 per warp in the MMA's M dimension,
 *                        the warps sharing each K/V tile. Reads the context
 *                        8 times less often for long chunks.
 *   PKV_MQ_TILE_TENSOR   128 rows per CTA on the fifth-generation tensor cores
 *                        (tcgen05): scores and outputs accumulate in tensor
 *                        memory, one thread per row runs the softmax.
 *   PKV_MQ_TILE_PAIRS    FP8 pools only (COLUMNS over a 16-bit pool): 16 rows
 *                        per CTA as two 8-column groups over one K/V ring,
 *                        each K/V code widened once for both groups.
 *   PKV_MQ_TILE_AUTO     TENSOR when max_query_len * (num_heads / num_kv_heads)
 *                        > 16 (more than two 8-column CTAs per kv head), else
 *                        COLUMNS (default). Over an FP8 pool: TENSOR above 32
 *                        rows, PAIRS from 9 to 32, COLUMNS up to 8
 *                        (paged_attention_multi_query_fp8).
 */
#define PKV_MQ_TILE_AUTO 0
#define PKV_MQ_TILE_COLUMNS 1
#define PKV_MQ_TILE_ROWS 2
#define PKV_MQ_TILE_TENSOR 3
#define PKV_MQ_TILE_PAIRS 4

/* Choose the multi-query tile for later calls in this process (PKV_MQ_TILE_*).
 * Returns the previous choice, or -1 for an unknown value (nothing changes). */
int32_t pkv_set_multi_query_tile(int32_t tile);

size_t paged_attention_multi_query_workspace_size(int32_t num_query_tokens, int32_t num_heads,
                                                  int32_t num_kv_heads, int32_t head_dim,
                                                  int32_t block_size, int32_t max_context_len,
                                                  int32_t partition_size);

pkv_status_t paged_attention_multi_query(void* out, const void* query, const void* key_cache,
                                         const void* value_cache, const int32_t* block_tables,
                                         int32_t max_blocks_per_seq, const int32_t* context_lens,
                                         const int32_t* query_start_loc, int32_t num_seqs,
                                         int32_t num_query_tokens, int32_t max_query_len,
                                         int32_t max_context_len, float scale, int32_t block_size,
                                         int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                                         int32_t num_blocks, pkv_dtype_t dtype,
                                         int32_t partition_size, void* workspace,
                                         size_t workspace_bytes, cudaStream_t stream);

/*
 * paged_attention_multi_query_fp8 -- paged_attention_multi_query over an FP8
 * (E4M3) pool ("vLLM PagedAttention Kernel", the kv_cache_dtype, k_scale and
 * v_scale of reshape_and_cache; the scales as in paged_attention_decode_fp8:
 * a cached code c stands for c * k_scale in K and c * v_scale in V).
 *
 *   key_cache,        [num_blocks][num_kv_heads][block_size][head_dim] uint8
 *   value_cache       E4M3 codes, as written by paged_kv_write_fp8
 *   dtype             of query and out (PKV_F16 or PKV_BF16)
 *   k_scale, v_scale  finite and > 0
 * head_dim must be 128 (PKV_ERR_UNSUPPORTED otherwise). Every other argument,
 * the workspace (paged_attention_multi_query_workspace_size) and the results'
 * meaning are those of paged_attention_multi_query. Tiles: the 8-column tile
 * multiplies the codes widened in registers (f16 MMAs); the tensor-memory tile
 * widens each K/V tile's codes to f16 in shared memory, and a bf16 query is
 * scaled per row by a power of two into f16, so that both MMAs multiply f16.
 * PKV_MQ_TILE_AUTO takes the tensor-memory tile above 32 rows per kv head (the
 * 8-column forms are relatively faster over an FP8 pool), PKV_MQ_TILE_PAIRS
 * from 9 to 32 rows and the 8-column tile up to 8; PKV_MQ_TILE_ROWS runs the
 * 8-column tile.
 */
pkv_status_t paged_attention_multi_query_fp8(void* out, const void* query, const void* key_cache,
                                             const void* value_cache, const int32_t* block_tables,
                                             int32_t max_blocks_per_seq, const int32_t* context_lens,
                                             const int32_t* query_start_loc, int32_t num_seqs,
                                             int32_t num_query_tokens, int32_t max_query_len,
                                             int32_t max_context_len, float scale, int32_t block_size,
                                             int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                                             int32_t num_blocks, pkv_dtype_t dtype, float k_scale,
                                             float v_scale, int32_t partition_size, void* workspace,
                                             size_t workspace_bytes, cudaStream_t stream);

/*
 * paged_attention_decode_shared_prefix -- the decode step of a batch whose
 * sequences all begin with the same prefix blocks (one prompt with several
 * continuations, as in parallel sampling or beam search). Copy-on-write keeps
 * those full blocks shared in the pool ("'안녕하세요 반갑습니다'로 배우는 vLLM
 * — KV Cache와 PagedAttention 완전 해부", §9단계; "Sparse Computation and
 * Memory Management for Efficient LLM Inference", Copy-on-Write). The result
 * is paged_attention_decode's, up to rounding order, with block table
 * prefix_blocks ++ block_tables[s] and context length prefix_len +
 * tail_lens[s], but the prefix's K/V tiles are read and multiplied once for
 * all sequences. All num_seqs * num_heads query rows of the batch attend the
 * prefix as one multi-query problem on the tensor-memory tile (the 8-column
 * tile at 16 or fewer rows per kv head, num_seqs * group; the FP8 form
 * switches at the same 16 rows, so both forms share one workspace size). Each
 * sequence's tail is one decode token over its own blocks. The two parts'
 * (m, l, o) partials are merged by the log-sum-exp rule of the split-K reduce.
 *
 *   out, query         [num_seqs][num_heads][head_dim], dtype
 *   key_cache, value_cache   the pool, [num_blocks][num_kv_heads][block_size][head_dim]
 *   prefix_blocks      [prefix_len / block_size] int32 physical ids of the shared
 *                      prefix, in logical order; prefix_len must be a whole
 *                      number of blocks (0: no prefix; then every sequence is
 *                      its tail)
 *   block_tables       [num_seqs][max_blocks_per_seq] int32: sequence s's blocks
 *                      after the prefix (its logical blocks prefix_len / block_size ...)
 *   tail_lens          [num_seqs] int32 tokens after the prefix (0 allowed); values
 *                      outside [0, max_tail_len] are clamped and set PKV_DEVERR_CONTEXT
 *   max_tail_len       host bound on tail_lens, <= max_blocks_per_seq * block_size
 *   workspace          >= paged_attention_shared_prefix_workspace_size(...) bytes,
 *                      16-byte aligned (always needed: both parts leave partials)
 *
 * 16-bit caches (PKV_F16, PKV_BF16; an FP8 pool: the _fp8 form below); head_dim
 * 64 or 128; block_size 8, 16 or 32. Errors as in paged_attention_decode: bad block ids are skipped with
 * PKV_DEVERR_BLOCK_ID. Asynchronous on `stream`; three kernels (prefix, tails,
 * merge). The prefix kernel runs on a second stream beside the tails: event
 * waits order it after the work already queued on `stream` and the merge after
 * it, so the call is ordered on `stream` as a whole and can be captured into a
 * CUDA graph. That stream and its two events are created on first use, one
 * set per host thread and device, and kept until the process exits.
 */
size_t paged_attention_shared_prefix_workspace_size(int32_t num_seqs, int32_t num_heads,
                                                    int32_t num_kv_heads, int32_t head_dim,
                                                    int32_t block_size, int32_t prefix_len,
                                                    int32_t max_tail_len);

pkv_status_t paged_attention_decode_shared_prefix(void* out, const void* query, const void* key_cache,
                                                  const void* value_cache, const int32_t* prefix_blocks,
                                                  int32_t prefix_len, const int32_t* block_tables,
                                                  int32_t max_blocks_per_seq, const int32_t* tail_lens,
                                                  int32_t num_seqs, int32_t max_tail_len, float scale,
                                                  int32_t block_size, int32_t num_heads,
                                                  int32_t num_kv_heads, int32_t head_dim,
                                                  int32_t num_blocks, pkv_dtype_t dtype, void* workspace,
                                                  size_t workspace_bytes, cudaStream_t stream);

/*
 * paged_attention_decode_shared_prefix_fp8 -- paged_attention_decode_shared_prefix
 * over an FP8 (E4M3) pool: key_cache and value_cache hold uint8 codes standing
 * for code * k_scale and code * v_scale (as in paged_attention_decode_fp8; both
 * scales finite and > 0), head_dim 128, dtype the query's and out's (PKV_F16 or
 * PKV_BF16). The stages run the FP8 forms of the multi-query tiles; the
 * workspace and every other argument are those of the 16-bit call.
 */
pkv_status_t paged_attention_decode_shared_prefix_fp8(void* out, const void* query, const void* key_cache,
                                                      const void* value_cache, const int32_t* prefix_blocks,
                                                      int32_t prefix_len, const int32_t* block_tables,
                                                      int32_t max_blocks_per_seq, const int32_t* tail_lens,
                                                      int32_t num_seqs, int32_t max_tail_len, float scale,
                                                      int32_t block_size, int32_t num_heads, int32_t num_kv_heads,
                                                      int32_t head_dim, int32_t num_blocks, pkv_dtype_t dtype,
                                                      float k_scale, float v_scale, void* workspace,
                                                      size_t workspace_bytes, cudaStream_t stream);

/*
 * FP8 KV cache. The pages pass kv_cache_dtype, k_scale and v_scale to the cache
 * write ("[vLLM] PagedAttention: OS 페이징 기법으로 KV 캐시를 관리하는 방법",
 * section "PagedAttention 커널", write_to_paged_cache) without fixing the format.
 * Here the format is OCP FP8 E4M3 (1 sign, 4 exponent bits with bias 7, 3
 * mantissa bits; largest finite value 448; S.1111.111 is NaN; no infinities).
 * A cache element holds the code of value / scale, so its value is
 * code * scale: k_scale for key_cache, v_scale for value_cache. Both are host
 * floats, finite and > 0; others are rejected with PKV_ERR_INVALID_ARG.
 * The pool layout is the one above with 1-byte elements: a (block, kv head)
 * tile is block_size * head_dim bytes. paged_kv_copy_blocks copies such a
 * pool with dtype PKV_FP8_E4M3.
 */

/*
 * paged_kv_write_fp8 -- paged_kv_write into an FP8 pool (quantizing).
 *
 * For every token t with slot = slot_mapping[t] >= 0 and every kv head h:
 *     key_cache[slot / block_size][h][slot % block_size][d] = E4M3(key[t][h][d] / k_scale)
 *     (value_cache likewise with v_scale)
 * key and value are fp16 or bf16 (dtype). The division is the correctly
 * rounded fp32 quotient; E4M3() rounds it to the nearest E4M3 value, ties to
 * the even code, and saturates magnitudes above 448 (infinities included) to
 * +-448. A NaN gives a NaN code (0x7F or 0xFF). Padding, bad slots, alignment
 * and the other arguments are as in paged_kv_write.
 */
pkv_status_t paged_kv_write_fp8(const void* key, const void* value, void* key_cache,
                                void* value_cache, const int64_t* slot_mapping, int32_t num_tokens,
                                int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                int32_t num_blocks, pkv_dtype_t dtype, float k_scale, float v_scale,
                                cudaStream_t stream);

/*
 * paged_attention_workspace_size_fp8 -- workspace bytes of
 * paged_attention_decode_fp8: the size paged_attention_workspace_size gives
 * (partition_size 0 selects the same default for both).
 */
size_t paged_attention_workspace_size_fp8(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                          int32_t head_dim, int32_t block_size,
                                          int32_t max_context_len, int32_t partition_size);

/*
 * paged_attention_decode_fp8 -- paged_attention_decode over an FP8 pool.
 *
 * The result is that of paged_attention_decode with K_j and V_j replaced by
 * their values code * k_scale and code * v_scale:
 *     x_j = scale * k_scale * dot(query[s][h][:], codes of K_j)
 *     out[s][h][:] = v_scale * sum_j softmax(x)_j * (codes of V_j)
 * query and out are fp16 or bf16 (dtype). With head_dim 128 and up to 8 query
 * heads per kv head (MHA included) the tensor cores compute both products in
 * f16 with fp32 accumulation: the codes widen exactly to f16, a bf16 query is
 * scaled per head by a power of two into f16 range, and the softmax weights are
 * rounded to f16 (the normaliser sums the rounded weights). Other shapes run on
 * the CUDA cores in fp32. All other
 * arguments, the split-K workspace (paged_attention_workspace_size_fp8) and the
 * error behaviour are those of paged_attention_decode.
 */
pkv_status_t paged_attention_decode_fp8(void* out, const void* query, const void* key_cache,
                                        const void* value_cache, const int32_t* block_tables,
                                        int32_t max_blocks_per_seq, const int32_t* context_lens,
                                        int32_t num_seqs, int32_t max_context_len, float scale,
                                        int32_t block_size, int32_t num_heads, int32_t num_kv_heads,
                                        int32_t head_dim, int32_t num_blocks, pkv_dtype_t dtype,
                                        float k_scale, float v_scale, int32_t partition_size,
                                        void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Static string naming a status code. */
const char* pkv_status_string(pkv_status_t status);

/* Description of the last failed call on the calling thread ("" if none). */
const char* pkv_last_error_message(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_KV_H_ */
