/*
 * pa.h -- C ABI of the GB300 (sm_103a) paged decode-attention library.
 *
 * The library computes single-query (decode) attention over a KV cache that
 * is stored in fixed-size physical blocks, together with the two kernels that
 * feed that cache and a host-side block manager.  Sources for the method:
 *   [P1] "PagedAttention: Virtual Memory for the KV Cache" (int8ai.pages.dev)
 *   [P2] "PagedAttention in vLLM: scattered memory, exact attention"
 *        (abhiram1809.github.io)
 *   [P3] "PagedAttention and KV Memory" (blog.michaelsam94.com)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensors are caller-owned.  Device pointers point to CUDA device
 *    memory of the current device; the library never allocates or frees
 *    device memory and keeps no pointer to caller memory after a call
 *    returns.  The only device memory the library owns is the static array
 *    of pa_decode_static_scratch (PA_STATIC_SCRATCH_BYTES on every device
 *    that loads the library, held until the process exits).  Host pointers
 *    are only read during the call.
 *  - Element types: K/V caches, q, new keys/values are bf16 (2 bytes);
 *    attention output is bf16 or fp32 (see PA_DTYPE_*).  Integers are the
 *    fixed-width types named in each signature.
 *  - Cache layout (one pair of tensors per layer): k_cache and v_cache are
 *    contiguous [num_blocks][n_kv_heads][block_size][d_head].  The keys of one
 *    (block, kv head) are one contiguous block_size * d_head * 2 byte run.
 *  - Supported shapes: block_size in {8, 16, 32}; d_head in {64, 128};
 *    n_q_heads a multiple of n_kv_heads with G = n_q_heads / n_kv_heads in
 *    {1, 2, 4, 8, 16}.  Other shapes return PA_ERR_UNSUPPORTED.
 *  - Device pointers must be 16-byte aligned (PA_ERR_MISALIGNED otherwise).
 *  - GPU work is enqueued asynchronously on `stream` (a cudaStream_t passed
 *    as void*; NULL is the legacy default stream).  A return of PA_OK means
 *    the launch was enqueued; errors detected on the host are returned before
 *    anything is enqueued.
 *  - Errors that only the device can see (a block id outside
 *    [0, num_blocks), a slot outside [0, num_blocks * block_size), a context
 *    length above max_blocks_per_seq * block_size or max_context_len) never
 *    trap: the offending access is skipped or clamped and a PA_DEV_* bit is
 *    OR-ed into *status_dev, if status_dev is not NULL (a device int32 the
 *    caller zeroes and reads back).  Outputs touched by such an error are
 *    unspecified.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes (returned) ---------------------------------------------- */
#define PA_OK                 0
#define PA_FAIL_NO_BLOCKS     1   /* pool exhausted; nothing was changed        */
#define PA_ERR_INVALID_ARG   -1
#define PA_ERR_UNSUPPORTED   -2
#define PA_ERR_MISALIGNED    -3
#define PA_ERR_CUDA          -4   /* a CUDA runtime call failed                 */
#define PA_ERR_WORKSPACE     -5   /* workspace missing or too small             */
#define PA_ERR_UNKNOWN_SEQ   -6
#define PA_ERR_DUPLICATE_SEQ -7
#define PA_ERR_SWAPPED       -8   /* the sequence's blocks are in host memory  */

/* ---- device-side status bits (OR-ed into *status_dev) ---------------------- */
#define PA_DEV_BAD_BLOCK_ID   1   /* table entry or copy pair outside the pool  */
#define PA_DEV_BAD_SLOT       2   /* slot_mapping entry outside the pool        */
#define PA_DEV_BAD_CONTEXT    4   /* context length above the stated maximum    */
#define PA_DEV_WAIT_TIMEOUT   8   /* a bounded wait for a bulk copy gave up     */

/* ---- output element types ------------------------------------------------- */
#define PA_DTYPE_BF16 0
#define PA_DTYPE_F32  1

/* Library version string and a short text for a status code. */
const char* pa_version(void);
const char* pa_status_string(int status);

/* ===========================================================================
 * Decode attention
 * ===========================================================================
 * Operation ([P1] section 1; [P2] section 10; [P1] sections 7 and 13):
 * for every sequence s and query head g, with G = n_q_heads / n_kv_heads and
 * KV head h = g / G (contiguous groups; [P1] section 1 and [P2] section 7 fix
 * that G query heads share a KV head, not which ones),
 *
 *   out[s][g][:] = sum_j a_j V_j,   a = softmax(scale * q[s][g] . K_j),
 *
 * over positions j = 0 .. context_lens[s]-1, where position j of sequence s
 * is read from physical block block_tables[s][j / block_size] at offset
 * j % block_size ([P1] section 7).  Positions at and beyond the context
 * length are never read into the result ([P1] section 13, item 4).  The
 * softmax is computed online in fp32 with a running maximum and sum
 * ([P1] section 13; [P2] section 11).  A context length of 0 gives a zero
 * row.  The token this step appended is part of the context: context_lens
 * counts it.
 *
 * Each sequence is split into partitions of partition_size positions, one
 * thread block per (sequence, group of up to 8 query heads, partition).  A
 * sequence that fits one partition is finished by its block.  When the batch
 * has many head groups (at least two waves of resident blocks) and
 * max_context_len spans four partitions or more, the resident blocks
 * instead claim the (sequence, head group, partition) items that exist, so
 * that no block is spent on the partitions past a short sequence's end.  Otherwise
 * every block leaves its partition's maximum m, weight sum z and
 * unnormalised weighted value sum u (the statistics of [P2] section 11) in
 * `workspace`, and a second kernel merges them exactly (the "secondary
 * reduction" of [P1] section 13).
 *
 * Arguments
 *   out           device [num_seqs][n_q_heads][d_head], PA_DTYPE_BF16 (round
 *                 to nearest even) or PA_DTYPE_F32, per out_dtype.
 *   q             device bf16 [num_seqs][n_q_heads][d_head].
 *   k_cache,
 *   v_cache       device bf16 [num_blocks][n_kv_heads][block_size][d_head].
 *   block_tables  device int32 [num_seqs][max_blocks_per_seq], row-major;
 *                 only the first ceil(context_lens[s] / block_size) entries of
 *                 row s are read.
 *   context_lens  device int32 [num_seqs].
 *   scale         score scale, normally 1 / sqrt(d_head).
 *   max_context_len  host upper bound on every context_lens[s].  Larger
 *                 device values are clamped to it and flagged with
 *                 PA_DEV_BAD_CONTEXT.
 *   partition_size   positions per partition: 0 lets the library choose
 *                 from the batch shape, the device and the cache type (256
 *                 to 1536), else a multiple of 64 in [64, 8192].
 *   workspace     device scratch of at least pa_decode_workspace_size(...)
 *                 bytes (same arguments, same current device), 256-byte
 *                 aligned; may be NULL (bytes 0) when that size is 0 (every
 *                 sequence fits one partition).  Its first 8 bytes are two
 *                 int32 counters through which blocks claim work: they must
 *                 be zero before the workspace's first use, and every call
 *                 leaves them zero (the last block to finish resets them).
 *                 Nothing else in it needs to be initialised; its contents
 *                 are not preserved across calls, and calls that share a
 *                 workspace must be stream-ordered.
 *   status_dev    optional device int32, see PA_DEV_* above.
 * Returns PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_MISALIGNED,
 * PA_ERR_WORKSPACE or PA_ERR_CUDA (launch failure).
 */
/* FP8 caches ([P3] "Alternatives and ecosystem": quantised KV cuts the bytes
 * per token; [P2] section 11: exactness is judged at the same KV precision).
 * k_cache / v_cache hold E4M3 codes (1 byte per element, same
 * [num_blocks][n_kv_heads][block_size][d_head] layout) written by
 * pa_reshape_and_cache_fp8; element = E4M3(code) * k_scale (or v_scale).  The
 * result is the attention over those dequantised keys and values, computed
 * as pa_decode computes it (fp32 softmax and accumulation; f16 operands,
 * which hold every E4M3 value exactly; q is rounded to f16 after a per-head
 * power-of-two scaling, the softmax weights to f16 after a 2^15 scaling, a
 * relative error of at most 2^-11).  Same arguments and
 * workspace as pa_decode, plus the two scales (finite, > 0).  d_head must be
 * 128 (PA_ERR_UNSUPPORTED otherwise).  With G = 4 and an even n_kv_heads a
 * thread block covers two adjacent KV heads (their 8 query heads fill the
 * products' columns), so the grid has n_kv_heads / 2 head groups. */
int pa_decode_fp8(void* out, int out_dtype, const void* q,
                  const void* k_cache, const void* v_cache,
                  const int32_t* block_tables, const int32_t* context_lens,
                  int block_size, float scale, float k_scale, float v_scale,
                  int n_q_heads, int n_kv_heads, int d_head, int num_seqs,
                  int max_blocks_per_seq, int num_blocks, int max_context_len,
                  int partition_size, void* workspace, size_t workspace_bytes,
                  int32_t* status_dev, void* stream);

/* Workspace bytes pa_decode or pa_decode_fp8 needs for these sizes on the
 * current device (the default partition size depends on the device's SM
 * count and, with partition_size 0, on the call: the size returned serves
 * both); 0 when no sequence can span more than one partition. */
size_t pa_decode_workspace_size(int num_seqs, int n_q_heads, int d_head,
                                int max_context_len, int partition_size);

/* Decode attention over a bf16 cache: the operation, the arguments and the
 * return codes are those of the "Decode attention" block above. */
int pa_decode(void* out, int out_dtype, const void* q,
              const void* k_cache, const void* v_cache,
              const int32_t* block_tables, const int32_t* context_lens,
              int block_size, float scale, int n_q_heads, int n_kv_heads,
              int d_head, int num_seqs, int max_blocks_per_seq, int num_blocks,
              int max_context_len, int partition_size,
              void* workspace, size_t workspace_bytes,
              int32_t* status_dev, void* stream);

/* One decode step's cache write and attention in one call: the token each
 * sequence appended this step (its keys and values join the cache when it is
 * fed back for the next decode pass, [P1] section 16; the decode kernel
 * reading the blocks, section 13) is written into the cache and attended to,
 * with the result, the
 * cache contents and the status bits equal, bit for bit, to
 * pa_reshape_and_cache of those rows followed by pa_decode.
 *   k_cache, v_cache   as pa_decode, written at one slot per sequence.
 *   k_new, v_new       device bf16 [num_seqs][n_kv_heads][d_head], 16-byte
 *                      aligned: the keys and values of position
 *                      context_lens[s] - 1 of sequence s (the position just
 *                      appended; context_lens counts it).  Its slot is the
 *                      one the block table gives for that position:
 *                      block_tables[s][(ctx - 1) / block_size] at offset
 *                      (ctx - 1) % block_size.
 * The thread block that reads that position's tile writes the rows into the
 * cache and into its own copy of the tile, so the step needs no separate
 * cache-write kernel before the attention.  Sequences with context length 0
 * append nothing; a context above its stated maximum is clamped and flagged
 * (PA_DEV_BAD_CONTEXT) and appends nothing; a bad block id is flagged
 * (PA_DEV_BAD_BLOCK_ID) and nothing is written.  Other arguments, the
 * workspace and the return codes are those of pa_decode (PA_ERR_INVALID_ARG
 * if k_new or v_new is NULL). */
int pa_decode_append(void* out, int out_dtype, const void* q,
                     void* k_cache, void* v_cache,
                     const void* k_new, const void* v_new,
                     const int32_t* block_tables, const int32_t* context_lens,
                     int block_size, float scale, int n_q_heads,
                     int n_kv_heads, int d_head, int num_seqs,
                     int max_blocks_per_seq, int num_blocks,
                     int max_context_len, int partition_size,
                     void* workspace, size_t workspace_bytes,
                     int32_t* status_dev, void* stream);

/* pa_decode_append for FP8 caches: the appended rows are quantised exactly
 * as pa_reshape_and_cache_fp8 quantises them (code = E4M3(float(x) / scale),
 * IEEE division, round to nearest even, saturating), then attended to as by
 * pa_decode_fp8; bit-equal to those two calls. */
int pa_decode_append_fp8(void* out, int out_dtype, const void* q,
                         void* k_cache, void* v_cache,
                         const void* k_new, const void* v_new,
                         const int32_t* block_tables,
                         const int32_t* context_lens, int block_size,
                         float scale, float k_scale, float v_scale,
                         int n_q_heads, int n_kv_heads, int d_head,
                         int num_seqs, int max_blocks_per_seq, int num_blocks,
                         int max_context_len, int partition_size,
                         void* workspace, size_t workspace_bytes,
                         int32_t* status_dev, void* stream);

/* Exact merge of partition statistics ([P2] section 11):
 *   M = max_p m_p,  Z = sum_p exp(m_p - M) z_p,  U = sum_p exp(m_p - M) u_p,
 *   out = U / Z,
 * over partitions p = 0 .. ceil(context_lens[s] / partition_size) - 1 of each
 * (sequence s, query head g).  m is in the units of the scores themselves
 * (natural-log domain).  This is the second kernel of pa_decode, exposed so
 * that partition statistics from any source can be merged; d_head <= 1024.
 *   part_max, part_sum  device f32 [num_seqs][n_q_heads][max_parts]
 *   part_acc            device f32 [num_seqs][n_q_heads][max_parts][d_head]
 *   context_lens        device int32 [num_seqs]; partitions counted as above,
 *                       capped at max_parts; a count of 0 writes zeros.
 *   partition_size      any value >= 1.
 * Returns PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_MISALIGNED
 * or PA_ERR_CUDA. */
int pa_lse_merge(void* out, int out_dtype, const float* part_max,
                 const float* part_sum, const float* part_acc,
                 const int32_t* context_lens, int partition_size, int max_parts,
                 int num_seqs, int n_q_heads, int d_head, void* stream);

/* pa_decode without a caller-supplied workspace.  The pages have no
 * counterpart of this entry point; it exists for callers that cannot hand the
 * library device memory: code that runs where cudaMalloc is not allowed or
 * not wanted (inside an allocator callback, in a process whose memory pool is
 * fixed up front, or in a host framework that owns every device allocation
 * and offers no scratch buffer).  Arguments and results are those of
 * pa_decode minus workspace/workspace_bytes; the split path keeps its
 * partition statistics in a static device array of PA_STATIC_SCRATCH_BYTES
 * bytes that the library itself declares, so this call never allocates.
 *  - The array is part of the library's device image: every GPU that loads
 *    the library holds PA_STATIC_SCRATCH_BYTES of it until the process exits.
 *  - Problems whose pa_decode_workspace_size(...) exceeds
 *    PA_STATIC_SCRATCH_BYTES are rejected with PA_ERR_WORKSPACE before
 *    anything is launched.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before any stream capture.  The address is cached per CUDA context: a
 *    context created anew on the device (after cudaDeviceReset, say) holds
 *    its own copy of the array, and the first call in it looks the address
 *    up again.
 *  - All calls share the one array and it keeps whatever the last call left
 *    there.  Its first 8 bytes are pa_decode's claim counters, zero when the
 *    library is loaded and left zero by every call; every value the merge
 *    reads was written earlier in the same call.  Calls whose kernels
 *    overlap on the GPU (other streams, other host threads) race on it; order
 *    them on one stream.
 */
#define PA_STATIC_SCRATCH_BYTES (16u << 20)

int pa_decode_static_scratch(void* out, int out_dtype, const void* q,
                             const void* k_cache, const void* v_cache,
                             const int32_t* block_tables,
                             const int32_t* context_lens, int block_size,
                             float scale, int n_q_heads, int n_kv_heads,
                             int d_head, int num_seqs, int max_blocks_per_seq,
                             int num_blocks, int max_context_len,
                             int partition_size, int32_t* status_dev,
                             void* stream);

/* ===========================================================================
 * Prefill attention (causal, many query positions per sequence)
 * ===========================================================================
 * Operation ([P2] sections 4 and 8; [P1] sections 7 and 13): sequence s has
 * context length C = context_lens[s], of which the last n = query_start[s+1]
 * - query_start[s] positions are new; their keys and values must already be
 * in the cache (pa_reshape_and_cache, earlier on the stream).  New position
 * p = C - n + i (i = 0 .. n-1) is query row query_start[s] + i, and for each
 * query head g (KV head g / G, as for decode)
 *
 *   out[row][g][:] = sum_{j <= p} a_j V_j,   a = softmax(scale * q[row][g] . K_j)
 *
 * over positions 0 .. p only (causal).  A whole prompt is n = C; a later
 * chunk of a prompt, or the part of a prompt after a prefix-cache hit, is
 * n < C.  Positions are read through block_tables as for decode.
 *
 * Scores and sums are fp32 (tensor cores; bf16 q and K).  The weighted sum
 * of values takes fp16 operands: first, V is gathered through the block
 * table into the caller's workspace (each 128-position tile of each
 * sequence and KV head contiguous), as fp16, which holds every bf16
 * magnitude in [2^-14, 2^16) exactly and is within 2^-25 below it; the
 * softmax weights are rounded to fp16 (a relative 2^-11; the normaliser
 * sums them unrounded), so an output element can differ from the exact
 * value by up to about 2^-11 * sum_j a_j |V_j| besides fp32 rounding.  A
 * tile holding a value of magnitude 2^16 or more, or a non-finite one,
 * stays bf16, and its weights go as two bf16 terms (hi + lo, a relative
 * 2^-16).
 *
 * Arguments
 *   out           device [num_tokens][n_q_heads][d_head], bf16 or fp32 per
 *                 out_dtype, 16-byte aligned.  Rows of tokens not covered by
 *                 any sequence are not written.
 *   q             device bf16 [num_tokens][n_q_heads][d_head], 16-byte aligned.
 *   k_cache,
 *   v_cache       device bf16 [num_blocks][n_kv_heads][block_size][d_head].
 *   block_tables  device int32 [num_seqs][max_blocks_per_seq].
 *   query_start   device int32 [num_seqs + 1], non-decreasing, query_start[0]
 *                 >= 0 and query_start[num_seqs] <= num_tokens.
 *   context_lens  device int32 [num_seqs], each >= its n.  A sequence with
 *                 C < n, or C above max_blocks_per_seq * block_size, is
 *                 flagged PA_DEV_BAD_CONTEXT (the first is skipped, the
 *                 second clamped).
 *   max_query_len host upper bound on every n (query rows beyond it are not
 *                 computed).
 *   n_q_heads / n_kv_heads must be a power of two <= 128; d_head 64 or 128;
 *   block_size 8, 16 or 32.
 *   workspace     device, 16-byte aligned, at least
 *                 pa_prefill_workspace_size(num_seqs, max_blocks_per_seq,
 *                 block_size, n_kv_heads, d_head) bytes (workspace_bytes):
 *                 the V staging (n_kv_heads x num_seqs x L positions x
 *                 d_head x 2 bytes, L = max_blocks_per_seq * block_size
 *                 rounded up to 128) and one format byte per 128 positions.
 *                 Caller-owned; overwritten by each call, so calls that
 *                 share one must be ordered (one stream).  Missing or too
 *                 small: PA_ERR_WORKSPACE.  num_seqs at most 65535.
 *   sched_dev     optional device int32 [2], zero before the first call; the
 *                 kernel's blocks claim work items from it (KV head by KV
 *                 head, within a head the latest query rows, which see the
 *                 most keys, first) and the last block to finish zeroes it
 *                 again.  Calls that share one pair must be ordered (one
 *                 stream).  NULL: a fixed round-robin assignment, slower when
 *                 sequences differ in length.  Caller-owned.
 *   status_dev    optional device int32, see PA_DEV_* above.
 * Returns PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_MISALIGNED,
 * PA_ERR_WORKSPACE or PA_ERR_CUDA.
 */
int pa_prefill(void* out, int out_dtype, const void* q,
               const void* k_cache, const void* v_cache,
               const int32_t* block_tables, int max_blocks_per_seq,
               const int32_t* query_start, const int32_t* context_lens,
               int num_seqs, int num_tokens, int max_query_len, int num_blocks,
               int block_size, float scale, int n_q_heads, int n_kv_heads,
               int d_head, void* workspace, size_t workspace_bytes,
               int32_t* sched_dev, int32_t* status_dev, void* stream);

/* Bytes of workspace pa_prefill needs (0 for a non-positive argument). */
size_t pa_prefill_workspace_size(int num_seqs, int max_blocks_per_seq,
                                 int block_size, int n_kv_heads, int d_head);

/* pa_prefill over FP8 caches (E4M3 codes written by pa_reshape_and_cache_fp8,
 * element = E4M3(code) * k_scale or v_scale, the layout of pa_decode_fp8).
 * The result is the causal attention over those dequantised keys and values,
 * computed as pa_prefill computes it: the codes are staged in the workspace,
 * K as bf16 (the score products take q as given) and V as fp16 (the value
 * products take fp16 weights), both of which hold every E4M3 value exactly;
 * k_scale joins the score scale and v_scale the output's.  Arguments as
 * pa_prefill plus the two scales (finite, > 0); d_head must be 128
 * (PA_ERR_UNSUPPORTED otherwise); workspace of at least
 * pa_prefill_fp8_workspace_size(...) bytes (the V staging and its format
 * bytes, then the K staging).  A table entry outside the pool reads zeros and
 * is flagged PA_DEV_BAD_BLOCK_ID. */
int pa_prefill_fp8(void* out, int out_dtype, const void* q,
                   const void* k_cache, const void* v_cache,
                   const int32_t* block_tables, int max_blocks_per_seq,
                   const int32_t* query_start, const int32_t* context_lens,
                   int num_seqs, int num_tokens, int max_query_len,
                   int num_blocks, int block_size, float scale, float k_scale,
                   float v_scale, int n_q_heads, int n_kv_heads, int d_head,
                   void* workspace, size_t workspace_bytes, int32_t* sched_dev,
                   int32_t* status_dev, void* stream);

/* Bytes of workspace pa_prefill_fp8 needs (0 for a non-positive argument). */
size_t pa_prefill_fp8_workspace_size(int num_seqs, int max_blocks_per_seq,
                                     int block_size, int n_kv_heads,
                                     int d_head);

/* ===========================================================================
 * Cache writes
 * ===========================================================================
 * reshape_and_cache ([P1] section 16 item 3 and section 20: each newly
 * computed position's key and value are written to its place in the pool):
 * for every token t with slot = slot_mapping[t] >= 0, and every KV head h,
 *   k_cache[slot / block_size][h][slot % block_size][:] = k[t][h][:]
 *   v_cache[slot / block_size][h][slot % block_size][:] = v[t][h][:]
 * The slot number is physical_block * block_size + offset, the
 * frame * size + offset form of [P2] section 2.  Negative slots are skipped
 * (padding); slots >= num_blocks * block_size are skipped and flagged
 * PA_DEV_BAD_SLOT.  The copy is bit-exact.  Two tokens with the same slot in
 * one call race (one of them wins).
 *   k, v          device bf16 [num_tokens][n_kv_heads][d_head], contiguous.
 *   slot_mapping  device int64 [num_tokens].
 * num_tokens == 0 is a no-op returning PA_OK.
 */
int pa_reshape_and_cache(void* k_cache, void* v_cache, const void* k,
                         const void* v, const int64_t* slot_mapping,
                         int num_tokens, int n_kv_heads, int d_head,
                         int block_size, int num_blocks, int32_t* status_dev,
                         void* stream);

/* pa_reshape_and_cache for FP8 caches: each element x of k (v) is stored as
 * the E4M3 code of float32(x) / k_scale (v_scale): IEEE float32 division,
 * then round to nearest even, saturating at +-448, NaN kept.  k, v are bf16
 * [num_tokens][n_kv_heads][d_head] as for pa_reshape_and_cache; the caches
 * are bytes [num_blocks][n_kv_heads][block_size][d_head].  Scales must be
 * finite and > 0 (PA_ERR_INVALID_ARG). */
int pa_reshape_and_cache_fp8(void* k_cache, void* v_cache, const void* k,
                             const void* v, const int64_t* slot_mapping,
                             int num_tokens, int n_kv_heads, int d_head,
                             int block_size, int num_blocks, float k_scale,
                             float v_scale, int32_t* status_dev, void* stream);

/* copy_blocks: the copy-on-write clone of a shared tail block ([P1]
 * sections 15 and 16): for every pair (src, dst) = (block_pairs[2i],
 * block_pairs[2i+1]) and every layer l, block dst of k_caches[l] and
 * v_caches[l] becomes a bit-exact copy of block src (all heads, all
 * block_size slots).  Pairs are copied concurrently, so no dst may repeat
 * and no dst may be another pair's src (the block manager never emits
 * such pairs: dst is always a freshly taken block).  Ids outside
 * [0, num_blocks) are skipped and flagged PA_DEV_BAD_BLOCK_ID.
 *   k_caches, v_caches  HOST arrays of num_layers device pointers, each a
 *                       cache laid out as above (same shape for all layers).
 *   block_pairs         device int32 [num_pairs][2].
 * num_pairs == 0 or num_layers == 0 is a no-op returning PA_OK.
 * Must be ordered before the reshape_and_cache that writes into dst in the
 * same step (same stream, earlier launch). */
int pa_copy_blocks(void* const* k_caches, void* const* v_caches,
                   int num_layers, const int32_t* block_pairs, int num_pairs,
                   int n_kv_heads, int d_head, int block_size, int num_blocks,
                   int32_t* status_dev, void* stream);

/* pa_copy_blocks for FP8 caches: the same copy of whole blocks, each cache
 * bytes [num_blocks][n_kv_heads][block_size][d_head] (E4M3 codes; the copy
 * is of bits, so any one-byte element type serves). */
int pa_copy_blocks_fp8(void* const* k_caches, void* const* v_caches,
                       int num_layers, const int32_t* block_pairs,
                       int num_pairs, int n_kv_heads, int d_head,
                       int block_size, int num_blocks, int32_t* status_dev,
                       void* stream);

/* Copy whole blocks between two pools with the cache layout: for every pair
 * (src, dst) in block_pairs and every layer, the K block src of src_k[l] goes
 * to block dst of dst_k[l], and likewise for V.  Either side may be device
 * memory or page-locked host memory (cudaHostAlloc / cudaHostRegister), which
 * the kernel reads or writes directly (over NVLink-C2C on Grace hosts): this
 * is the payload move of swapping ([P1] section 19, item 4).
 *   dst_k, dst_v, src_k, src_v  HOST arrays of num_layers pointers; each pool
 *                 [num_blocks][n_kv_heads][block_size][d_head] bf16, 16-byte
 *                 aligned.  Host pools are translated with
 *                 cudaPointerGetAttributes; pageable memory is rejected.
 *   block_pairs   int32 [num_pairs][2] (src, dst), device or page-locked host;
 *                 read by the kernel, so it must stay unchanged until the copy
 *                 has run (stream order), like every input of an async call.
 * Ids outside [0, src_num_blocks) or [0, dst_num_blocks) are skipped and
 * flagged PA_DEV_BAD_BLOCK_ID.  Destinations must be distinct.
 * PA_ERR_INVALID_ARG (NULL, pageable or unknown pointer), PA_ERR_UNSUPPORTED,
 * PA_ERR_MISALIGNED, PA_ERR_CUDA. */
int pa_swap_blocks(void* const* dst_k, void* const* dst_v,
                   const void* const* src_k, const void* const* src_v,
                   int num_layers, const int32_t* block_pairs, int num_pairs,
                   int n_kv_heads, int d_head, int block_size,
                   int src_num_blocks, int dst_num_blocks,
                   int32_t* status_dev, void* stream);

/* pa_swap_blocks for FP8 caches: pools of bytes
 * [num_blocks][n_kv_heads][block_size][d_head] (E4M3 codes) on either side;
 * everything else as for pa_swap_blocks. */
int pa_swap_blocks_fp8(void* const* dst_k, void* const* dst_v,
                       const void* const* src_k, const void* const* src_v,
                       int num_layers, const int32_t* block_pairs,
                       int num_pairs, int n_kv_heads, int d_head,
                       int block_size, int src_num_blocks, int dst_num_blocks,
                       int32_t* status_dev, void* stream);

/* Self-test of the failure path of every kernel: one thread block waits on
 * an mbarrier that nothing ever arrives on, with the bounded wait routine the
 * decode pipeline uses (max_probes probes of at most ~1 us each), then
 * records PA_DEV_WAIT_TIMEOUT in *status_dev and returns.  No fault and no
 * hang: the context stays usable.  max_probes in [1, 10^7]; status_dev
 * required (device int32).  Returns PA_OK, PA_ERR_INVALID_ARG or PA_ERR_CUDA. */
int pa_check_bounded_wait(int max_probes, int32_t* status_dev, void* stream);

/* ===========================================================================
 * Host block manager ([P1] sections 14-17 and 20)
 * ===========================================================================
 * A pool of num_blocks blocks of block_size positions.  The free list is a
 * stack: a fresh manager hands out blocks 0, 1, 2, ... and released blocks
 * are reused last-released-first ([P1] section 20).  Every block carries a
 * reference count; sequences are named by caller-chosen int64 ids.
 * Appending only plans a step: it returns the slot for the new position and,
 * when the tail block was shared, the (src, dst) block pair that the caller
 * must pass to pa_copy_blocks before writing with pa_reshape_and_cache.
 * Every call that can fail for lack of blocks is transactional: on
 * PA_FAIL_NO_BLOCKS nothing changes ([P1] section 20, test 4).
 * A handle is not thread-safe; use one per thread or lock around it. */
typedef struct pa_alloc pa_alloc_t;

/* Pool counters, filled by pa_alloc_get_stats.  They give the operational
 * metrics of [P3] "Operational metrics": block-pool usage (num_used /
 * num_blocks), preemptions by swapping (num_swap_outs), the prefix-cache hit
 * rate (num_cached_tokens / num_prompt_tokens) and the mean sequence length
 * (num_context_tokens / num_seqs). */
typedef struct pa_alloc_stats {
    int32_t num_blocks;
    int32_t num_free;           /* on the free list                        */
    int32_t num_used;           /* count >= 1                              */
    int32_t num_seqs;
    int64_t num_cow_copies;     /* CoW pairs emitted since creation        */
    int32_t num_cached;         /* count 0, kept for prefix reuse          */
    int32_t num_swapped;        /* sequences whose blocks are in host memory */
    int64_t num_prompt_tokens;  /* prompt positions admitted since creation */
    int64_t num_cached_tokens;  /* of those, found in the prefix cache     */
    int64_t num_swap_outs;      /* sequences swapped out since creation    */
    int64_t num_context_tokens; /* sum of every live sequence's length     */
} pa_alloc_stats_t;

/* NULL if num_blocks <= 0 or block_size <= 0 or on allocation failure. */
pa_alloc_t* pa_alloc_create(int num_blocks, int block_size);
/* Frees the manager and everything it holds; NULL is ignored. */
void pa_alloc_destroy(pa_alloc_t* a);

/* Replace the free list by order[0 .. n-1] (blocks leave from the end), e.g.
 * to place sequences at seeded random physical blocks.  Only while no block
 * is in use; order must be a permutation of 0 .. num_blocks-1.
 * PA_ERR_INVALID_ARG otherwise. */
int pa_alloc_set_free_order(pa_alloc_t* a, const int32_t* order, int n);

/* Take ceil(num_tokens / block_size) blocks (ref 1) for a new sequence of
 * num_tokens prompt positions.  PA_ERR_DUPLICATE_SEQ if seq exists,
 * PA_ERR_INVALID_ARG if num_tokens <= 0, PA_FAIL_NO_BLOCKS if too few free.
 * Its token ids are unknown, so none of its blocks is ever cached. */
int pa_alloc_sequence(pa_alloc_t* a, int64_t seq, int num_tokens);

/* ---------------------------------------------------------------------------
 * Automatic prefix caching ([P1] section 18; [P2] section 6; [P3] "Prefix
 * caching").  Off by default.  When on, a FULL block whose token ids are
 * known is registered under a key made of its block_size token ids and the
 * key of the block before it (the root key for block 0), so two blocks match
 * only when the whole prefix up to and including them is identical.  A
 * registered block whose count falls to 0 is not put on the free list but
 * queued for eviction (least recently released first; within one release,
 * the deepest block of the table is queued first).  Fresh blocks come from
 * the free list first and only when it is empty from the front of the
 * eviction queue, which drops that block's key.  Partly filled blocks are
 * never registered; when a block fills under a key that another block
 * already holds, it is left unregistered and returns to the free list when
 * released.  Keys are exact: each distinct token prefix ending on a block
 * boundary is interned once (its parent prefix and its block's token ids),
 * and a 64-bit chained hash serves only to find candidates, every one of
 * which is compared in full, so a hash collision can never match the wrong
 * prefix.
 * ------------------------------------------------------------------------- */

/* Switch caching on (enable != 0) or off.  Only while no sequence exists;
 * switching off forgets every key and moves the queued blocks to the free
 * list (oldest first, so the newest is handed out first).
 * PA_ERR_INVALID_ARG otherwise. */
int pa_alloc_enable_prefix_caching(pa_alloc_t* a, int enable);

/* Testing hook: the 64-bit hash that buckets the interned prefixes is ANDed
 * with mask (all bits by default); mask = 0 puts every prefix in one bucket,
 * so every lookup meets colliding candidates and must tell them apart by
 * content.  Only while no sequence exists and no prefix is interned
 * (PA_ERR_INVALID_ARG otherwise).  Results never depend on the mask. */
int pa_alloc_set_key_mask(pa_alloc_t* a, uint64_t mask);

/* Number of interned prefixes (held by registered blocks, sequences, or
 * longer prefixes); -1 if a is NULL. */
int pa_alloc_num_prefix_nodes(const pa_alloc_t* a);

/* New sequence with known prompt token ids tokens[0 .. num_tokens-1].
 * With caching on, its leading full blocks are looked up in order and the
 * search stops at the first miss; each hit is shared (count + 1; a queued
 * block leaves the queue and goes from 0 back to 1) and its positions need
 * no prefill: *num_cached_tokens = hits * block_size.  The rest are fresh
 * blocks; the full ones among them are registered at once (the caller must
 * write their KV before any other sequence can read it, i.e. before the next
 * decode on the same stream).  With caching off it behaves as
 * pa_alloc_sequence and *num_cached_tokens = 0.
 * PA_ERR_DUPLICATE_SEQ, PA_ERR_INVALID_ARG, PA_FAIL_NO_BLOCKS when the free
 * list plus the queue (less the hits taken from it) is short: no change. */
int pa_alloc_sequence_tokens(pa_alloc_t* a, int64_t seq, const int32_t* tokens,
                             int num_tokens, int* num_cached_tokens);

/* pa_alloc_append_slot for a position whose token id is known.  When that
 * position fills the block and caching is on, the block is registered.  A
 * sequence extended with pa_alloc_append_slot loses its token ids and is
 * not registered from then on. */
int pa_alloc_append_token(pa_alloc_t* a, int64_t seq, int32_t token,
                          int64_t* slot_out, int32_t* cow_src, int32_t* cow_dst);

/* Blocks with count 0 held for reuse (-1 for a NULL handle). */
int pa_alloc_num_cached(const pa_alloc_t* a);

/* ---------------------------------------------------------------------------
 * Swap space ([P1] section 19, item 4: preemption by moving a request's
 * blocks to host memory and back; item 3, preemption by recomputation, is
 * pa_alloc_free now and pa_alloc_sequence_tokens later, which finds whatever
 * the prefix cache still holds).  A pool of host blocks, numbered
 * 0 .. num_host_blocks-1 and handed out like device blocks (a stack that
 * starts with 0, 1, 2, ...).  The payload lives in caller-owned host pools
 * laid out like the device caches; pa_swap_blocks moves it.
 * ------------------------------------------------------------------------- */

/* Size the host pool (0 disables swapping).  Only while no sequence is
 * swapped out; PA_ERR_INVALID_ARG otherwise. */
int pa_alloc_enable_swap(pa_alloc_t* a, int num_host_blocks);

/* Swap out the running sequences seqs[0..n-1] (distinct).  Every distinct
 * device block in their tables gets one host block, whose reference count
 * is the number of these sequences that use it; the device blocks lose those
 * references (freed, or queued by the prefix cache, at 0; blocks shared with
 * other running sequences stay).  The sequences keep their lengths and token
 * ids; until swapped in, only pa_alloc_free, pa_alloc_block_table (which then
 * returns host block ids) and pa_alloc_seq_len accept them, the rest return
 * PA_ERR_SWAPPED.  Writes the (device block, host block) pairs, first
 * appearance order, to pairs_out[2i], [2i+1] and their count to *num_pairs;
 * the caller copies them with pa_swap_blocks before the freed device blocks
 * are written again (same stream).
 * PA_ERR_UNKNOWN_SEQ, PA_ERR_SWAPPED (a sequence is already out),
 * PA_ERR_INVALID_ARG (duplicates, or pair_capacity < *num_pairs: nothing
 * changes, *num_pairs says how many are needed), PA_FAIL_NO_BLOCKS (too few
 * free host blocks: nothing changes). */
int pa_alloc_swap_out(pa_alloc_t* a, const int64_t* seqs, int n,
                      int32_t* pairs_out, int pair_capacity, int* num_pairs);

/* Swap in the swapped-out sequences seqs[0..n-1]: the mirror image.  Every
 * distinct host block gets a fresh device block (free list first, then the
 * prefix cache's eviction queue) with as many references as sequences of
 * the batch use it; the host blocks lose those references.  Pairs are
 * (host block, device block).  PA_ERR_INVALID_ARG also when a sequence is
 * not swapped out; PA_FAIL_NO_BLOCKS when too few device blocks: nothing
 * changes. */
int pa_alloc_swap_in(pa_alloc_t* a, const int64_t* seqs, int n,
                     int32_t* pairs_out, int pair_capacity, int* num_pairs);

int pa_alloc_num_free_host(const pa_alloc_t* a);        /* -1 for NULL */
int pa_alloc_is_swapped(const pa_alloc_t* a, int64_t seq); /* 1 out, 0 in, -1 unknown */
/* Copy the eviction queue front (next evicted) to back into out (cap
 * entries); returns its size. */
int pa_alloc_cached_list(const pa_alloc_t* a, int32_t* out, int cap);

/* child gets a copy of parent's table and length; every block's count +1
 * ([P1] section 16, step 2).  PA_ERR_UNKNOWN_SEQ / PA_ERR_DUPLICATE_SEQ. */
int pa_alloc_fork(pa_alloc_t* a, int64_t parent, int64_t child);

/* Plan one appended position at index L = current length ([P1] sections
 * 15, 16): tail shared and partly filled -> new block, *cow_src = old tail,
 * *cow_dst = new block; tail private with room -> in place; tail full ->
 * new block.  *slot_out = block * block_size + (L % block_size); the length
 * becomes L + 1.  *cow_src = *cow_dst = -1 when no copy is needed.
 * PA_ERR_UNKNOWN_SEQ, PA_FAIL_NO_BLOCKS (no change). */
int pa_alloc_append_slot(pa_alloc_t* a, int64_t seq, int64_t* slot_out,
                         int32_t* cow_src, int32_t* cow_dst);

/* Batch form: plans one position for each of seqs[0..n-1] in order.  Writes
 * slots_out[i]; CoW pairs go to cow_pairs_out[2k], [2k+1] (capacity
 * cow_capacity pairs, n is always enough) and their count to *num_cow.
 * Stops at the first failure: *num_done (if not NULL) tells how many
 * sequences were planned; their changes stay.  Returns the first failure's
 * status or PA_OK. */
int pa_alloc_append_slots(pa_alloc_t* a, const int64_t* seqs, int n,
                          int64_t* slots_out, int32_t* cow_pairs_out,
                          int cow_capacity, int* num_cow, int* num_done);

/* Release: every block in seq's table loses one reference and returns to
 * the free list at 0, in table order ([P1] section 17); with caching on, a
 * registered block at 0 is queued for eviction instead (see above).  Unknown seq: no-op,
 * PA_OK.  Blocks are reusable only after GPU work that reads or writes them
 * has completed; the caller orders that (same stream). */
int pa_alloc_free(pa_alloc_t* a, int64_t seq);

/* Copy seq's block table into out[0 .. cap-1]; *n_out = its length.
 * PA_ERR_UNKNOWN_SEQ; PA_ERR_INVALID_ARG if cap is too small. */
int pa_alloc_block_table(const pa_alloc_t* a, int64_t seq, int32_t* out,
                         int cap, int* n_out);

/* Decode metadata for a batch: row i of tables (row stride max_blocks) gets
 * seqs[i]'s table, padded with -1; context_lens[i] its length.
 * PA_ERR_UNKNOWN_SEQ, PA_ERR_INVALID_ARG if a table is longer than
 * max_blocks. */
int pa_alloc_build_tables(const pa_alloc_t* a, const int64_t* seqs, int n,
                          int32_t* tables, int max_blocks, int32_t* context_lens);

/* Slots of positions start .. start+n-1 of seq ([P1] section 7):
 * table[i / B] * B + i % B.  PA_ERR_INVALID_ARG if the range is outside
 * [0, length). */
int pa_alloc_slot_mapping(const pa_alloc_t* a, int64_t seq, int start, int n,
                          int64_t* out);

int pa_alloc_seq_len(const pa_alloc_t* a, int64_t seq);      /* -1 if unknown */
int pa_alloc_ref_count(const pa_alloc_t* a, int32_t block);  /* -1 if out of range */
/* Blocks on the free list, not counting zero-count cached blocks (-1 for NULL). */
int pa_alloc_num_free(const pa_alloc_t* a);
/* Copy the free stack bottom-to-top into out (cap entries); returns its size. */
int pa_alloc_free_list(const pa_alloc_t* a, int32_t* out, int cap);
/* Fill *out with the counts above; PA_ERR_INVALID_ARG if a or out is NULL. */
int pa_alloc_get_stats(const pa_alloc_t* a, pa_alloc_stats_t* out);

#ifdef __cplusplus
}
#endif
#endif /* PA_H_ */
