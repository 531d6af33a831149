// Paged prefill attention for sm_103a on the 5th-generation tensor cores.
//
// Operation ("PagedAttention in vLLM: scattered memory, exact attention",
// sections 4 and 8; "PagedAttention: Virtual Memory for the KV Cache",
// sections 7 and 13): a sequence with context length ctx whose last n
// positions are new (their keys and values already written to the paged
// cache) gets, for each new position p = ctx - n + i and each query head,
//     o = softmax(scale * q . K[0..p]) V[0..p]
// with K and V read through the block table (causal: a query sees only the
// positions up to its own).  The whole prompt (n = ctx), a later chunk of it
// (chunked prefill), or the suffix after a prefix-cache hit are all this
// same call.
//
// Design (a staging pass, then a persistent CTA per SM; a work item is two
// tiles of 128 query rows of one KV head):
//   * stage_v_kernel gathers V through the block table into the caller's
//     workspace, each (KV head, sequence) owning consecutive rows, so that a
//     128-position V tile is contiguous.  It stores a tile as fp16, which
//     holds every bf16 magnitude in [2^-14, 2^16) exactly and is off by at
//     most 2^-25 below that range, with the rows past the context zeroed; a
//     tile holding a magnitude of 2^16 or more (or a non-finite value)
//     stays bf16, and a format byte per tile says which.
//   * Rows are (token, grouped query head) pairs: 128 / G consecutive new
//     tokens times the G query heads that share KV head h, so every K/V tile
//     is read once for all G heads (GQA).  Each Q tile is one 3-D TMA box;
//     an item's two tiles (A, B) are consecutive token ranges and share every
//     K/V tile.
//   * Items are claimed from a counter shared by all CTAs, by group of KV
//     heads and heaviest first within a group (the group's K/V stays in L2);
//     the claiming warp decodes each item once and posts it to a ring in
//     shared memory for the other warps.  Barrier phases run on across
//     items, so the next item's loads and first products overlap the
//     current item's last products and output.
//   * K tiles of 128 positions are gathered through the block table with
//     one 2-D TMA box (64 columns x B rows, 128-byte swizzle) per block and
//     64-column half; a warp issues its boxes one lane after another, so K
//     and V have a producer warp each, and table entries are fetched four
//     tiles ahead.  Blocks past the needed range, and bad table entries, are
//     loaded from outside the tensor, which fills zeros and reads no HBM.  A
//     staged V tile is one box of 128 rows per 64 columns.
//   * S = Q K^T (M 128, N 128, K d) and O += P V (M 128, N d, K 128) are
//     tcgen05.mma kind::f16 (fp32 accumulate), one issuing thread per Q
//     tile (two issuers hide most of the pipe drain between groups of
//     products of different kinds).  Tensor memory holds S_A, S_B (128
//     columns each) and O_A, O_B (d columns each).  S takes bf16 Q and K.
//     P V takes fp16 weights (written over the first 64 columns of their
//     own S and read from there as the A operand) and the staged fp16
//     values: fp16 carries each weight to a relative 2^-11 where bf16 would
//     give 2^-8.  For a V tile that stayed bf16 each weight is split into
//     two bf16 terms, hi = bf16(p) and lo = bf16(p - hi), written over the
//     first and the second 64 columns of S (O += P_hi V + P_lo V, a relative
//     2^-16).  An item learns once whether any of its V tiles stayed bf16,
//     and the softmax and MMA warps run one of two compiled forms of their
//     tile loop (the fp16-only form checks no formats).  V is an MN-major
//     operand read straight from the TMA layout.
//   * Eight softmax warps work on tile A, then on tile B, then on tile A of
//     the next K/V tile, ...: warps w and w + 4 share the 32 rows of lane
//     quarter w (tensor-memory lane = row), each taking 64 of the 128
//     columns; the two halves of a row exchange their maxima (and, at the
//     end, their sums) through shared memory.  Per row: mask, online maximum
//     in the log2 domain, exp2, running sum, P; the scale-and-subtract and
//     the running sums use packed f32x2 arithmetic (one instruction for two
//     columns), which the softmax's instruction issue is bound by.  O is
//     rescaled in tensor memory only when a row's maximum grows by more than
//     2^8 (the weights, which carry a factor 2^7, stay below 2^15 otherwise),
//     which is rare after the first tiles.  At the end of an item each
//     thread writes its half row with 32-byte stores.
//   * Every wait is bounded; on a timeout the CTA flags PA_DEV_WAIT_TIMEOUT,
//     waits (bounded) for its own copies and products in flight, frees its
//     tensor memory and returns.

#include <cuda.h>
#include <cudaTypedefs.h>

#include <climits>
#include <type_traits>
#include <mutex>

#include "pa_common.cuh"

namespace {

constexpr int kRows = 128;                 // MMA M: query rows per tile
constexpr int kKv = 128;                   // positions per K/V tile
constexpr int kProducerWarp = 8;           // claims work items, loads Q and K
constexpr int kVProducerWarp = 9;          // loads V
constexpr int kMmaWarp0 = 10;              // MMA warps 10 (tile A) and 11 (tile B); 10 owns the tensor memory
constexpr int kThreads = 384;              // 8 softmax warps, 2 producers, 2 MMA warps
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS0 = 0;            // S_A; S_B at +128
constexpr uint32_t kTmemO0 = 256;          // O_A; O_B at +128
constexpr int kMaxProbes = 2000000;        // x <= ~1 us per probe
constexpr float kRescaleThreshold = 8.0f;  // log2 of the largest weight allowed before a rescale
constexpr float kWeightShift = 7.0f;       // weights carry 2^7: at most 2^15, within fp16's range
// Two stages each for K and V: a third K stage (the shared memory allows one)
// measured no faster.
constexpr int kKStages = 2;
constexpr int kVStages = 2;
constexpr int kSoftmaxThreads = 256;
constexpr int kRing = 4;              // work items posted ahead by the producer
constexpr int kItemReaders = 11;      // warps that read each posted item: V producer, 2 MMA, 8 softmax

template <int D>
struct PGeo {
    static constexpr int kHalves = D / 64;
    static constexpr int kHalfBytes = kRows * 128;            // 128 rows of 64 bf16
    static constexpr int kQBytes = kHalves * kHalfBytes;      // one Q tile
    static constexpr int kKVBytes = kHalves * kHalfBytes;     // one K (or V) tile of 128 positions
    static constexpr int kQ = 0;                              // Q_A, then Q_B
    static constexpr int kK0 = 2 * kQBytes;                   // K stages (kKStages)
    static constexpr int kV0 = kK0 + kKStages * kKVBytes;     // V stages (kVStages)
    static constexpr int kRed = kV0 + kVStages * kKVBytes;     // row-half exchange: [tile][parity][half][row] fp32
    static constexpr int kBars = kRed + 2 * 2 * 2 * kRows * 4;
    // barriers, slots and alignment slack; at least 120 KiB so that two CTAs
    // never share an SM (each holds 512 tensor-memory columns)
    static constexpr int kSmem = kBars + 512 + 1024 > 120 * 1024 ? kBars + 512 + 1024 : 120 * 1024;
};

struct PrefillArgs {
    void* out;
    int out_f32;
    int out_al32;         // out is 32-byte aligned: 256-bit stores
    const int32_t* block_tables;
    int max_blocks;
    const int32_t* query_start;
    const int32_t* context_lens;
    int num_seqs;
    int num_tokens;
    int tiles_per_seq;    // work items per sequence and KV head (each covers 2 * tq tokens)
    int heads_per_group;  // KV heads whose items are claimed together
    int block_size;
    int n_kv_heads;
    int group;            // query heads per KV head
    int tq;               // tokens per Q tile = 128 / group
    int n_q_heads;
    int num_blocks;
    int oob_row;          // a row coordinate past the end of the cache view
    float scale_log2;     // scale * log2(e)
    const uint8_t* v_fmt; // per (KV head, sequence, 128-position tile) of the V staging: 0 fp16, 1 bf16
    float k_scale;        // FP8: dequantisation scales of K and V
    float v_scale;
    int l_slot;           // positions per (KV head, sequence) in the V staging, a multiple of 128
    int t_slot;           // l_slot / 128
    int32_t* status;
    int* sched;           // {next item, CTAs done} claimed with atomics, or null: fixed order
};

// One work item: query rows [t0, t0 + 2 tq) of sequence seq's n new tokens
// (Q tiles A and B; has_b = 0: A only) and KV head h; tile x sees keys
// [0, kv_end_x), nt_x tiles of them, n_tiles in all.  The producer decodes
// it once and posts it; seq < 0 ends the stream.
struct Item {
    int seq, h, q0, n, ctx, t0;
    int kv_end0, kv_end1, nt0, nt1, n_tiles, has_b;
    int wide;             // some V tile of the item is staged as bf16
};

struct Bars {
    uint64_t q_full;
    uint64_t k_full[kKStages];
    uint64_t v_full[kVStages];
    uint64_t k_empty[2][kKStages];  // per Q tile and stage: its score products reading K are done
    uint64_t v_empty[2][kVStages];  // per Q tile and stage: its value products reading V are done
    uint64_t s_full[2];   // per Q tile: its scores are in tensor memory
    uint64_t p_full[2];   // per Q tile: its weights (fp16, or the bf16 hi terms) are in tensor memory (and O rescaled)
    uint64_t plo_full[2]; // per Q tile: the bf16 lo terms of a wide tile's weights are in tensor memory
    uint64_t o_done[2];   // per Q tile: its last product of an item has finished
    uint64_t o_free[2];   // per Q tile: the softmax warps have read O out
    uint64_t q_empty[2];  // per Q tile: its last score product of an item has finished
    uint64_t red[2];      // per Q tile: both halves of every row posted their value
    uint64_t item_full[kRing];    // the producer posted the next work item
    uint64_t item_empty[kRing];   // every consumer warp has read it
    Item item[kRing];
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(Bars) <= 512, "barrier block overflows its reserved space");

// --- tcgen05 / TMA wrappers --------------------------------------------------

__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    // start address, leading and stride byte offsets (all >> 4), descriptor
    // version 1, 128-byte swizzle
    return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)((lbo & 0x3FFFF) >> 4) << 16) |
           ((uint64_t)((sbo & 0x3FFFF) >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// kind::f16 instruction descriptor: fp32 accumulator, A and B both bf16 (bf = 1)
// or both fp16 (bf = 0), A K-major, B K-major (b_mn = 0) or MN-major
// (b_mn = 1), shape M x N.
__host__ __device__ constexpr uint32_t idesc_f16(int m, int n, int b_mn, int bf) {
    return (1u << 4) | ((uint32_t)bf << 7) | ((uint32_t)bf << 10) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     pa::smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31])));
}

__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t* w) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]), "r"(w[8]),
        "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15]));
}

// A operand from tensor memory (M rows in lanes, two 16-bit values per column).
__device__ __forceinline__ void mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                            uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}

// One 32-byte store (address 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t (&w)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                 "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(pa::smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tma_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(pa::smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two fp32 values in one 64-bit register pair, for the packed f32x2
// arithmetic (one instruction for both lanes of the pair).
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void f32x2_split(uint64_t r, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}

__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// v[0 .. n) *= k, two at a time
template <int n>
__device__ __forceinline__ void scale_f32x2(float* v, float k) {
    const uint64_t kk = f32x2(k, k);
#pragma unroll
    for (int i = 0; i < n; i += 2) f32x2_split(mul_f32x2(f32x2(v[i], v[i + 1]), kk), v[i], v[i + 1]);
}

__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t sub_f32x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint32_t pack_bf16_rn(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_f16_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two bf16 values to two fp16 values (each bf16 value is exact in fp32; the
// fp16 rounding is exact for magnitudes in [2^-14, 65536)).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
    return pack_f16_rn(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// The smallest bf16 magnitude pattern (sign cleared) that fp16 cannot
// hold: 0x4780 is 2^16, which fp16 rounds to infinity (the bf16 value below
// it, 65280, is exact in fp16); patterns above it also cover infinities and
// NaNs.
constexpr uint32_t kF16Wide = 0x4780u;

// The weights of one thread's kHalfCols scores s (in place: s becomes the
// fp32 weights p = 2^(s * c2 + neg)), their sums (into lp) and, at t_p in
// tensor memory, their kHalfCols / 2 columns of packed pairs: fp16, or the
// bf16 hi terms (kBf16) whose lo terms the caller writes next.
template <int kHalfCols, bool kBf16>
__device__ __forceinline__ void write_weights(float (&s)[kHalfCols], uint64_t c2x2, uint64_t negx2, uint64_t (&lp)[2],
                                              uint32_t t_p) {
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
        uint32_t w[kHalfCols / 4];
#pragma unroll
        for (int qq = 0; qq < kHalfCols / 4; ++qq) {
            const int q = h2 * (kHalfCols / 4) + qq;
            float x0, x1;
            f32x2_split(fma_f32x2(f32x2(s[2 * q], s[2 * q + 1]), c2x2, negx2), x0, x1);
            s[2 * q] = fast_exp2(x0);
            s[2 * q + 1] = fast_exp2(x1);
            lp[q & 1] = add_f32x2(lp[q & 1], f32x2(s[2 * q], s[2 * q + 1]));
            w[qq] = kBf16 ? pack_bf16_rn(s[2 * q], s[2 * q + 1]) : pack_f16_rn(s[2 * q], s[2 * q + 1]);
        }
        tmem_st16u(t_p + h2 * (kHalfCols / 4), w);
    }
}

// --- bounded waits -------------------------------------------------------------

// One thread.  Gives up when another role has aborted or after kMaxProbes
// probes (then aborts the CTA and flags the timeout).
__device__ bool wait1(uint64_t* bar, uint32_t parity, Bars* b, int32_t* status) {
#pragma unroll 1
    for (int i = 0; i < kMaxProbes; ++i) {
        if (pa::mbar_try_wait(bar, parity)) return true;
        if ((i & 63) == 63 && *reinterpret_cast<volatile int*>(&b->abort)) return false;
    }
    *reinterpret_cast<volatile int*>(&b->abort) = 1;
    pa::set_status(status, PA_DEV_WAIT_TIMEOUT);
    return false;
}

// Whole warp, warp-uniform result.
__device__ bool wait_warp(uint64_t* bar, uint32_t parity, Bars* b, int32_t* status) {
#pragma unroll 1
    for (int i = 0; i < kMaxProbes; ++i) {
        const bool done = pa::mbar_try_wait(bar, parity);
        if (__all_sync(0xffffffffu, done)) return true;
        if ((i & 63) == 63 && __any_sync(0xffffffffu, *reinterpret_cast<volatile int*>(&b->abort) != 0))
            return false;
    }
    if ((threadIdx.x & 31) == 0) {
        *reinterpret_cast<volatile int*>(&b->abort) = 1;
        pa::set_status(status, PA_DEV_WAIT_TIMEOUT);
    }
    __syncwarp();
    return false;
}

// --- the kernel ------------------------------------------------------------------

// One work item: 2 x 128 query rows (Q tiles A, B) of one KV head of one
// sequence.  Every role of a CTA decodes the same items in the same order.

// Item i of the claim order: by group of KV heads, and within a group the
// latest token tiles (the most keys) first.  The CTAs then work on a few
// heads' K/V at a time, which stays in L2 while every tile of it is read; a
// group holds at least two items per CTA, so that its lightest items, not
// heavy ones, end each group.  False when the item holds no query row (past
// the sequence's new tokens) or is invalid.
// Item i's sequence, KV head and query tile pair (arithmetic only).
__device__ __forceinline__ void item_coords(int i, const PrefillArgs& a, int& seq, int& h, int& tile) {
    const int per_group = a.tiles_per_seq * a.num_seqs * a.heads_per_group;
    const int grp = i / per_group;
    const int r = i - grp * per_group;
    const int per_tile = a.num_seqs * min(a.heads_per_group, a.n_kv_heads - grp * a.heads_per_group);
    tile = a.tiles_per_seq - 1 - r / per_tile;
    const int r2 = r % per_tile;
    seq = r2 % a.num_seqs;
    h = grp * a.heads_per_group + r2 / a.num_seqs;
}

__device__ __forceinline__ bool decode_item(int i, const PrefillArgs& a, Item& it, bool flag) {
    int tile;
    item_coords(i, a, it.seq, it.h, tile);
    it.q0 = a.query_start[it.seq];
    it.n = a.query_start[it.seq + 1] - it.q0;
    it.ctx = a.context_lens[it.seq];
    it.t0 = tile * 2 * a.tq;
    if (it.t0 >= it.n || it.q0 < 0) return false;
    if (it.ctx > a.max_blocks * a.block_size) {
        if (flag) pa::set_status(a.status, PA_DEV_BAD_CONTEXT);
        it.ctx = a.max_blocks * a.block_size;
    }
    if (it.ctx < it.n) {
        if (flag) pa::set_status(a.status, PA_DEV_BAD_CONTEXT);
        return false;
    }
    it.has_b = it.t0 + a.tq < it.n ? 1 : 0;
    it.kv_end0 = it.ctx - it.n + min(it.n, it.t0 + a.tq);
    it.kv_end1 = it.ctx - it.n + min(it.n, it.t0 + 2 * a.tq);
    it.nt0 = (it.kv_end0 + kKv - 1) / kKv;
    it.nt1 = it.has_b ? (it.kv_end1 + kKv - 1) / kKv : 0;
    it.n_tiles = it.has_b ? it.nt1 : it.nt0;
    return true;
}

// A posted ring entry, read once its item_full phase has completed.
__device__ __forceinline__ Item read_item(const Item* src) {
    const volatile int* p = reinterpret_cast<const volatile int*>(src);
    Item it;
    int* d = reinterpret_cast<int*>(&it);
#pragma unroll
    for (int k = 0; k < (int)(sizeof(Item) / sizeof(int)); ++k) d[k] = p[k];
    return it;
}

// Twelve warps on four SM sub-partitions: three share one 16K-register file,
// so at most 168 registers per thread.
//
// Persistent: one CTA per SM walks items blockIdx.x, blockIdx.x + gridDim.x,
// ...; every barrier's phase runs on across items, so the next item's Q and
// K/V copies and score products overlap the current item's last products and
// output.
// kF8: the caches hold E4M3 codes; K comes staged as bf16 and V as fp16 (both
// exact), the K scale joins the score scale and the V scale the output's.
template <int D, bool kF8 = false>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                   const __grid_constant__ CUtensorMap mv, const PrefillArgs a) {
    using G = PGeo<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars* bars = reinterpret_cast<Bars*>(sm + G::kBars);
    const uint32_t s_q = pa::smem_addr(sm + G::kQ);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_items = a.tiles_per_seq * a.num_seqs * a.n_kv_heads;

    if (threadIdx.x == 0) {
        pa::mbar_init(&bars->q_full, 1);
        for (int i = 0; i < kKStages; ++i) {
            pa::mbar_init(&bars->k_full[i], 1);
            pa::mbar_init(&bars->k_empty[0][i], 1);
            pa::mbar_init(&bars->k_empty[1][i], 1);
        }
        for (int i = 0; i < kVStages; ++i) {
            pa::mbar_init(&bars->v_full[i], 1);
            pa::mbar_init(&bars->v_empty[0][i], 1);
            pa::mbar_init(&bars->v_empty[1][i], 1);
        }
        for (int i = 0; i < kRing; ++i) {
            pa::mbar_init(&bars->item_full[i], 1);
            pa::mbar_init(&bars->item_empty[i], kItemReaders);
        }
        for (int i = 0; i < 2; ++i) {
            pa::mbar_init(&bars->q_empty[i], 1);
            pa::mbar_init(&bars->s_full[i], 1);
            pa::mbar_init(&bars->p_full[i], kSoftmaxThreads);
            pa::mbar_init(&bars->plo_full[i], kSoftmaxThreads);
            pa::mbar_init(&bars->o_done[i], 1);
            pa::mbar_init(&bars->o_free[i], kSoftmaxThreads);
            pa::mbar_init(&bars->red[i], kSoftmaxThreads);
        }
        bars->abort = 0;
        pa::fence_mbar_init();
    }
    if (warp == kMmaWarp0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         pa::smem_addr(&bars->tmem_base)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    // Launched as a programmatic dependent of the V staging: everything above
    // (barriers, tensor memory) overlaps its end; every input is read below.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp == kProducerWarp || warp == kVProducerWarp) {
        // ------------------------------------------------------------ TMA producers
        // A warp issues its copies one lane after another (tens of cycles
        // each), so K and V have a producer warp each.  The K warp claims work
        // items, posts them to the other warps and loads Q and K; the V warp
        // follows the posted items.  Lane i handles block i of each tile.
        const bool is_k = warp == kProducerWarp;
        const int bpt = kKv / a.block_size;              // blocks per tile
        int g = 0, c = 0;                                 // K/V tiles and items so far
        int nq = 0, np = 0;                               // Q copies issued, ring entries posted (K) or read (V)
        bool ok = true;
        // post an item (seq < 0: no more) to the other warps
        auto post = [&](const Item& it) {
            const int slot = np % kRing;
            if (np >= kRing && !wait_warp(&bars->item_empty[slot], (np / kRing - 1) & 1, bars, a.status))
                return false;
            if (lane == 0) {
                volatile int* d = reinterpret_cast<volatile int*>(&bars->item[slot]);
                const int* s_ = reinterpret_cast<const int*>(&it);
#pragma unroll
                for (int k = 0; k < (int)(sizeof(Item) / sizeof(int)); ++k) d[k] = s_[k];
                pa::mbar_arrive(&bars->item_full[slot]);
            }
            ++np;
            return true;
        };
        // Items are claimed in decode_item's order, from a counter shared by
        // all CTAs (the next free CTA takes the next item) or, without one,
        // round-robin.
        for (int k = 0; ok; ++k) {
            Item it;
            if (is_k) {
                int i = 0;
                if (lane == 0) i = a.sched ? atomicAdd(a.sched, 1) : (int)blockIdx.x + k * (int)gridDim.x;
                i = __shfl_sync(0xffffffffu, i, 0);
                if (i >= n_items) {
                    it.seq = -1;
                    post(it);
                    break;
                }
                if constexpr (kF8) {
                    // E4M3 values are all exact in fp16: no tile stays bf16
                    if (!decode_item(i, a, it, lane == 0)) continue;
                    it.wide = 0;
                } else {
                    // Do any of the item's V tiles stay bf16?  (The other
                    // warps then check tile by tile.)  The first 32 format
                    // bytes are loaded alongside the item's own loads.
                    int fseq, fh, ftile;
                    item_coords(i, a, fseq, fh, ftile);
                    const uint8_t* fmt = a.v_fmt + (size_t)(fh * a.num_seqs + fseq) * a.t_slot;
                    int w = lane < a.t_slot ? fmt[lane] : 0;
                    if (!decode_item(i, a, it, lane == 0)) continue;
                    w = lane < it.n_tiles ? w : 0;
                    for (int jj = lane + 32; jj < it.n_tiles; jj += 32) w |= fmt[jj];
                    it.wide = __any_sync(0xffffffffu, w != 0) ? 1 : 0;
                }
                ok = post(it);
                if (!ok) break;
                // Q of this item replaces the previous item's once both tiles'
                // last score products are done
                if (c >= 1)
                    ok = wait_warp(&bars->q_empty[0], (c - 1) & 1, bars, a.status) &&
                         wait_warp(&bars->q_empty[1], (c - 1) & 1, bars, a.status);
                if (!ok) break;
                if (lane == 0) {
                    pa::mbar_arrive_expect_tx(&bars->q_full, (it.has_b ? 2 : 1) * G::kQBytes);
                    for (int x = 0; x < (it.has_b ? 2 : 1); ++x)
#pragma unroll
                        for (int hh = 0; hh < G::kHalves; ++hh)
                            tma_3d(s_q + x * G::kQBytes + hh * G::kHalfBytes, &mq, hh * 64, it.h * a.group,
                                   it.q0 + it.t0 + x * a.tq, &bars->q_full);
                }
                ++nq;
            } else {
                const int slot = np % kRing;
                ok = wait_warp(&bars->item_full[slot], (np / kRing) & 1, bars, a.status);
                if (!ok) break;
                it = read_item(&bars->item[slot]);
                __syncwarp();
                if (lane == 0) pa::mbar_arrive(&bars->item_empty[slot]);
                ++np;
                if (it.seq < 0) break;
            }
            const int kv_all = it.has_b ? it.kv_end1 : it.kv_end0;
            const int32_t* table = a.block_tables + (size_t)it.seq * a.max_blocks;
            // K: block-table entries are fetched kAhead tiles before their
            // copies and checked only when used, so no copy waits on a table
            // load.  V comes from the staging buffer, whose tiles are
            // contiguous (one box of 128 rows per 64 columns).
            constexpr int kAhead = 4;
            constexpr int kNoBlock = INT_MIN;             // past the needed range: nothing loaded
            const int vrow0 = (it.h * a.num_seqs + it.seq) * a.l_slot;
            const bool gather = is_k && !kF8;              // FP8: K is staged like V
            auto fetch = [&](int j) {
                const int pos = j * kKv + lane * a.block_size;
                return (gather && lane < bpt && pos < kv_all) ? __ldg(table + pos / a.block_size) : kNoBlock;
            };
            auto to_row = [&](int blk) {
                if (blk == kNoBlock) return a.oob_row;
                if (blk < 0 || blk >= a.num_blocks) {
                    if (is_k) pa::set_status(a.status, PA_DEV_BAD_BLOCK_ID);
                    return a.oob_row;
                }
                return (blk * a.n_kv_heads + it.h) * a.block_size;
            };
            int blks[kAhead];
#pragma unroll
            for (int u = 0; u < kAhead; ++u) blks[u] = fetch(u);
            uint64_t* full = is_k ? bars->k_full : bars->v_full;
            uint64_t* empty0 = is_k ? bars->k_empty[0] : bars->v_empty[0];
            uint64_t* empty1 = is_k ? bars->k_empty[1] : bars->v_empty[1];
            const CUtensorMap* map = is_k ? &mk : &mv;
            const int stages = is_k ? kKStages : kVStages;
            const int base = is_k ? G::kK0 : G::kV0;
            for (int j0 = 0; ok && j0 < it.n_tiles; j0 += kAhead) {
#pragma unroll
                for (int u = 0; u < kAhead; ++u) {
                    const int j = j0 + u;
                    if (j >= it.n_tiles) break;
                    const int row = gather ? to_row(blks[u]) : vrow0 + j * kKv;
                    blks[u] = fetch(j + kAhead);
                    const int st = g % stages;
                    const uint32_t s_t =
                        pa::smem_addr(sm + base + st * G::kKVBytes) + (gather ? lane * a.block_size * 128 : 0);
                    // both Q tiles' MMA warps release every K/V tile (used or not)
                    if (g >= stages)
                        ok = wait_warp(&empty0[st], (g / stages - 1) & 1, bars, a.status) &&
                             wait_warp(&empty1[st], (g / stages - 1) & 1, bars, a.status);
                    if (!ok) break;
                    if (lane == 0) pa::mbar_arrive_expect_tx(&full[st], G::kKVBytes);
                    __syncwarp();
                    if (gather ? lane < bpt : lane == 0)
#pragma unroll
                        for (int hh = 0; hh < G::kHalves; ++hh)
                            tma_2d(s_t + hh * G::kHalfBytes, map, hh * 64, row, &full[st]);
                    ++g;
                }
            }
            ++c;
        }
        // the copies this warp started must land before the CTA exits: the
        // last use of each stage (earlier uses completed before it was reused)
        if (lane == 0) {
            if (nq) pa::mbar_wait_bounded(&bars->q_full, (nq - 1) & 1, kMaxProbes);
            uint64_t* full = is_k ? bars->k_full : bars->v_full;
            const int stages = is_k ? kKStages : kVStages;
            for (int i = 0; i < stages && i < g; ++i) {
                const int t = g - 1 - i;
                pa::mbar_wait_bounded(&full[t % stages], (t / stages) & 1, kMaxProbes);
            }
        }
    } else if (warp == kMmaWarp0 || warp == kMmaWarp0 + 1) {
        // ------------------------------------------------------------ MMA issuers
        // One thread per Q tile: a single thread cannot issue N=128 products
        // fast enough to keep the tensor pipe busy, two can.
        const int x = warp - kMmaWarp0;
        if (lane == 0) {
            constexpr uint32_t id_qk = idesc_f16(kRows, kKv, 0, 1);
            constexpr uint32_t id_pv = idesc_f16(kRows, D, 1, 0);      // fp16 weights and values
            constexpr uint32_t id_pv_bf = idesc_f16(kRows, D, 1, 1);   // a wide tile's bf16 hi and lo terms
            const uint32_t t_s = tmem + kTmemS0 + x * 128;
            const uint32_t t_o = tmem + kTmemO0 + x * 128;
            const uint32_t qx = s_q + x * G::kQBytes;
            uint64_t* last = nullptr;
            uint32_t last_par = 0;
            auto commit = [&](uint64_t* bar, uint32_t par) {
                mma_commit(bar);
                last = bar;
                last_par = par;
            };
            auto issue_s = [&](int ks) {
                const uint32_t s_k = pa::smem_addr(sm + G::kK0 + ks * G::kKVBytes);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * G::kHalfBytes + (kk & 3) * 32;
                    mma_f16_ss(t_s, smem_desc(qx + off, 16, 1024), smem_desc(s_k + off, 16, 1024), id_qk, kk > 0);
                }
            };
            // A tile this Q tile does not read is released only once it has
            // landed: the producer has then consumed the stage's previous
            // release, so each barrier moves on by exactly one phase per tile.
            auto skip_tile = [&](int gt) {
                if (!wait1(&bars->k_full[gt % kKStages], (gt / kKStages) & 1, bars, a.status)) return false;
                pa::mbar_arrive(&bars->k_empty[x][gt % kKStages]);
                if (!wait1(&bars->v_full[gt % kVStages], (gt / kVStages) & 1, bars, a.status)) return false;
                pa::mbar_arrive(&bars->v_empty[x][gt % kVStages]);
                return true;
            };
            int g = 0, c = 0, ns = 0, nod = 0, nw = 0;    // K/V tiles, items, S products, outputs, wide tiles so far
            bool ok = true;
            for (int nc = 0;; ++nc) {
                const int slot = nc % kRing;
                ok = wait1(&bars->item_full[slot], (nc / kRing) & 1, bars, a.status);
                if (!ok) break;
                const Item it = read_item(&bars->item[slot]);
                pa::mbar_arrive(&bars->item_empty[slot]);
                if (it.seq < 0) break;
                const int ntx = x ? it.nt1 : it.nt0;
                const int kv_endx = x ? it.kv_end1 : it.kv_end0;
                const size_t fmt0 = (size_t)(it.h * a.num_seqs + it.seq) * a.t_slot;
                if (ntx == 0) {
                    // this Q tile has no rows in the item: release Q and every K/V tile
                    ok = wait1(&bars->q_full, c & 1, bars, a.status);
                    if (!ok) break;
                    pa::mbar_arrive(&bars->q_empty[x]);
                    for (int j = 0; ok && j < it.n_tiles; ++j) ok = skip_tile(g + j);
                    g += it.n_tiles;
                    ++c;
                    continue;
                }
                ok = wait1(&bars->q_full, c & 1, bars, a.status) && wait1(&bars->k_full[g % kKStages],
                                                                            (g / kKStages) & 1, bars, a.status);
                if (!ok) break;
                tc_fence_after();
                issue_s(g % kKStages);
                commit(&bars->s_full[x], ns & 1);
                ++ns;
                commit(&bars->k_empty[x][g % kKStages], (g / kKStages) & 1);
                if (ntx == 1) commit(&bars->q_empty[x], c & 1);
                // The item's tiles, in one of two forms (as the softmax warps):
                // all V tiles fp16, or some bf16, checked tile by tile.
                auto run_tiles = [&](auto may_be_wide) {
                    constexpr bool kMayBeWide = decltype(may_be_wide)::value;
                    for (int j = 0; ok && j < it.n_tiles; ++j) {
                        const int gj = g + j;
                        const int vs = gj % kVStages;
                        if (j >= ntx) {                       // tile beyond this Q tile's keys
                            ok = skip_tile(gj);
                            continue;
                        }
                        // the staged tile's format (loaded before the waits below hide its latency)
                        const bool wide = kMayBeWide && a.v_fmt[fmt0 + j] != 0;
                        ok = wait1(&bars->v_full[vs], (gj / kVStages) & 1, bars, a.status);
                        if (!ok) break;
                        const uint32_t s_v = pa::smem_addr(sm + G::kV0 + vs * G::kKVBytes);
                        const int valid = min(kKv, kv_endx - j * kKv);
                        const int ksteps = (valid + 15) >> 4;
                        const int nks = (gj + 1) % kKStages;
                        if (j + 1 < ntx) ok = wait1(&bars->k_full[nks], ((gj + 1) / kKStages) & 1, bars, a.status);
                        // O must have been read out by the previous item's epilogue
                        if (ok && j == 0 && nod >= 1) ok = wait1(&bars->o_free[x], (nod - 1) & 1, bars, a.status);
                        if (ok) ok = wait1(&bars->p_full[x], (ns - 1) & 1, bars, a.status);
                        if (!ok) break;
                        tc_fence_after();
                        // O += P V with fp16 weights and values; for a wide tile
                        // O += P_hi V as soon as the hi terms are written, then
                        // O += P_lo V (the softmax writes lo meanwhile).  Each
                        // loop keeps its instruction descriptor a constant (a
                        // descriptor chosen at run time slowed the issue by 4 %).
                        if (!wide) {
                            for (int kk = 0; kk < ksteps; ++kk)
                                mma_f16_ta(t_o, t_s + kk * 8, smem_desc(s_v + kk * 2048, G::kHalfBytes, 1024), id_pv,
                                           (j > 0 || kk > 0) ? 1u : 0u);
                        } else {
                            for (int kk = 0; kk < ksteps; ++kk)
                                mma_f16_ta(t_o, t_s + kk * 8, smem_desc(s_v + kk * 2048, G::kHalfBytes, 1024), id_pv_bf,
                                           (j > 0 || kk > 0) ? 1u : 0u);
                            ok = wait1(&bars->plo_full[x], nw & 1, bars, a.status);
                            ++nw;
                            if (!ok) break;
                            tc_fence_after();
                            for (int kk = 0; kk < ksteps; ++kk)
                                mma_f16_ta(t_o, t_s + kKv / 2 + kk * 8,
                                            smem_desc(s_v + kk * 2048, G::kHalfBytes, 1024), id_pv_bf, 1u);
                        }
                        commit(&bars->v_empty[x][vs], (gj / kVStages) & 1);
                        if (j == ntx - 1) {
                            commit(&bars->o_done[x], nod & 1);
                            ++nod;
                        } else {
                            issue_s(nks);
                            commit(&bars->s_full[x], ns & 1);
                            ++ns;
                            commit(&bars->k_empty[x][nks], ((gj + 1) / kKStages) & 1);
                            if (j + 1 == ntx - 1) commit(&bars->q_empty[x], c & 1);
                        }
                    }
                };
                if (!kF8 && it.wide)
                    run_tiles(std::true_type{});
                else
                    run_tiles(std::false_type{});
                g += it.n_tiles;
                ++c;
            }
            // products in flight must finish before the tensor memory is freed
            if (last) pa::mbar_wait_bounded(last, last_par, kMaxProbes);
        }
    } else {
        // ------------------------------------------------------------ softmax warps
        const int quarter = warp & 3, hc = warp >> 2;     // lane quarter, column half
        const int r = quarter * 32 + lane;                // row = tensor-memory lane
        const int t = r / a.group, gq = r - t * a.group;
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        float* red = reinterpret_cast<float*>(sm + G::kRed);
        // score scale (log2 domain; FP8: times the K scale)
        const float c2s = kF8 ? a.scale_log2 * a.k_scale : a.scale_log2;
        const float c2x[2] = {c2s, c2s};
        constexpr int kHalfCols = kKv / 2;                // score columns per thread
        constexpr int kOCols = D / 2;                     // output columns per thread
        int ns[2] = {0, 0}, nred[2] = {0, 0}, nod[2] = {0, 0};
        // Post this half's value for row r of tile x and read the other half's.
        auto exchange = [&](int x, float v, bool& ok_) {
            const int phase = nred[x]++;
            float* slot = red + (((x * 2 + (phase & 1)) * 2) * kRows);
            slot[hc * kRows + r] = v;
            pa::mbar_arrive(&bars->red[x]);
            ok_ = wait_warp(&bars->red[x], phase & 1, bars, a.status);
            return ok_ ? slot[(1 - hc) * kRows + r] : v;
        };
        bool ok = true;
        for (int nc = 0; ok; ++nc) {
            const int slot = nc % kRing;
            ok = wait_warp(&bars->item_full[slot], (nc / kRing) & 1, bars, a.status);
            if (!ok) break;
            const Item it = read_item(&bars->item[slot]);
            __syncwarp();
            if (lane == 0) pa::mbar_arrive(&bars->item_empty[slot]);
            if (it.seq < 0) break;
            const int nt[2] = {it.nt0, it.nt1};
            float m_used[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
            int row_lim[2];
            bool valid_row[2];
            for (int x = 0; x < 2; ++x) {
                const int tok = it.t0 + x * a.tq + t;
                valid_row[x] = tok < it.n && it.q0 + tok < a.num_tokens;
                const int kv_end = x ? it.kv_end1 : it.kv_end0;
                row_lim[x] = valid_row[x] ? min(it.ctx - it.n + tok + 1, kv_end) : kv_end;   // keys [0, row_lim)
            }
            const uint8_t* fmt = a.v_fmt + (size_t)(it.h * a.num_seqs + it.seq) * a.t_slot;
            // The item's tiles, in one of two forms: all V tiles fp16 (the
            // common case, with no per-tile format check) or some bf16.
            auto run_tiles = [&](auto may_be_wide) {
                constexpr bool kMayBeWide = decltype(may_be_wide)::value;
                for (int j = 0; ok && j < it.n_tiles; ++j) {
                    const int wide = kMayBeWide ? fmt[j] : 0;   // V tile j staged as fp16 (0) or bf16 (1)
                    for (int x = 0; x < 2; ++x) {
                        if (j >= nt[x]) continue;
                        ok = wait_warp(&bars->s_full[x], ns[x] & 1, bars, a.status);
                        ++ns[x];
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t t_s = t_lane + kTmemS0 + x * 128;
                        float s[kHalfCols];
#pragma unroll
                        for (int cc = 0; cc < kHalfCols / 32; ++cc)
                            tmem_ld32(t_s + hc * kHalfCols + cc * 32, s + cc * 32);
                        tmem_wait_ld();
                        const int lim = row_lim[x] - j * kKv - hc * kHalfCols;     // valid columns of this half
                        if (lim < kHalfCols) {
#pragma unroll
                            for (int cc = 0; cc < kHalfCols; ++cc) s[cc] = cc < lim ? s[cc] : -INFINITY;
                        }
                        float mp[8];
#pragma unroll
                        for (int k = 0; k < 8; ++k) mp[k] = max3(s[k], s[8 + k], s[16 + k]);
#pragma unroll
                        for (int cc = 24; cc + 16 <= kHalfCols; cc += 16)
#pragma unroll
                            for (int k = 0; k < 8; ++k) mp[k] = max3(mp[k], s[cc + k], s[cc + 8 + k]);
                        if ((kHalfCols - 24) % 16 == 8) {
#pragma unroll
                            for (int k = 0; k < 8; ++k) mp[k] = fmaxf(mp[k], s[kHalfCols - 8 + k]);
                        }
                        float mt = fmaxf(max3(mp[0], mp[1], mp[2]),
                                         fmaxf(max3(mp[3], mp[4], mp[5]), fmaxf(mp[6], mp[7])));
                        mt = fmaxf(mt, exchange(x, mt, ok));
                        if (!ok) break;
                        const float c2 = c2x[x];
                        const float mts = mt * c2;            // scale > 0: the maximum commutes with it
                        const bool rescale = mts > m_used[x] + kRescaleThreshold;
                        const float m_new = rescale ? mts : m_used[x];
                        const float alpha = rescale ? fast_exp2(m_used[x] - m_new) : 1.f;   // exp2(-inf) = 0 at first
                        if (j >= 1 && __any_sync(0xffffffffu, rescale)) {
                            // O holds the products of tiles < j (complete: this tile's
                            // scores were issued after them) and not yet this tile's
                            const uint32_t t_o = t_lane + kTmemO0 + x * 128 + hc * kOCols;
#pragma unroll 1
                            for (int cc = 0; cc < kOCols / 32; ++cc) {
                                float o[32];
                                tmem_ld32(t_o + cc * 32, o);
                                tmem_wait_ld();
                                scale_f32x2<32>(o, alpha);
                                tmem_st32(t_o + cc * 32, o);
                            }
                        }
                        l[x] *= alpha;
                        m_used[x] = m_new;
                        // Weights are p = 2^(s * c2 - m_used + 7): the 2^7 (the sums
                        // carry it too, so it cancels) puts them in [0, 2^15], where
                        // fp16 rounds every weight above 2^-21 of the row maximum to
                        // a relative 2^-11.
                        const float neg = kWeightShift - m_used[x];
                        // Column pairs in packed f32x2 arithmetic: one FMA and one
                        // add per two weights.  The weights go to the tensor cores
                        // as fp16, written over the first 64 columns of S.  For a
                        // wide value tile (bf16) each weight p goes as two bf16
                        // terms instead, hi = bf16(p) and lo = bf16(p - hi) (p - hi
                        // is exact in fp32), so that hi + lo carries p to a relative
                        // 2^-16 instead of bf16's 2^-8.  P_hi is written over the
                        // first 64 columns of S and posted first, so the value
                        // products on it start while lo is computed and written over
                        // the other 64 columns.
                        const uint64_t c2x2 = f32x2(c2, c2), negx2 = f32x2(neg, neg);
                        uint64_t lp[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};   // independent partial sums
                        if (!wide)
                            write_weights<kHalfCols, false>(s, c2x2, negx2, lp, t_s + hc * (kHalfCols / 2));
                        else
                            write_weights<kHalfCols, true>(s, c2x2, negx2, lp, t_s + hc * (kHalfCols / 2));
                        tmem_wait_st();
                        tc_fence_before();
                        pa::mbar_arrive(&bars->p_full[x]);
                        float l0, l1, l2, l3;
                        f32x2_split(lp[0], l0, l1);
                        f32x2_split(lp[1], l2, l3);
                        l[x] += (l0 + l1) + (l2 + l3);
                        if (wide) {
#pragma unroll
                            for (int h2 = 0; h2 < 2; ++h2) {
                                uint32_t wl[kHalfCols / 4];
#pragma unroll
                                for (int qq = 0; qq < kHalfCols / 4; ++qq) {
                                    const int q = h2 * (kHalfCols / 4) + qq;
                                    const uint32_t hi = pack_bf16_rn(s[2 * q], s[2 * q + 1]);
                                    float r0, r1;
                                    f32x2_split(sub_f32x2(f32x2(s[2 * q], s[2 * q + 1]),
                                                          f32x2(__uint_as_float(hi << 16),
                                                                __uint_as_float(hi & 0xffff0000u))),
                                                r0, r1);
                                    wl[qq] = pack_bf16_rn(r0, r1);
                                }
                                tmem_st16u(t_s + kKv / 2 + hc * (kHalfCols / 2) + h2 * (kHalfCols / 4), wl);
                            }
                            tmem_wait_st();
                            tc_fence_before();
                            pa::mbar_arrive(&bars->plo_full[x]);
                        }
                    }
                }
            };
            if (!kF8 && it.wide)
                run_tiles(std::true_type{});
            else
                run_tiles(std::false_type{});
            for (int x = 0; x < 2 && ok; ++x) {
                if (nt[x] == 0) continue;
                const float l_all = l[x] + exchange(x, l[x], ok);
                if (ok) ok = wait_warp(&bars->o_done[x], nod[x] & 1, bars, a.status);
                ++nod[x];
                if (!ok) break;
                tc_fence_after();
                const int tok = it.t0 + x * a.tq + t;
                const float inv = (kF8 ? a.v_scale : 1.f) / l_all;
                const size_t orow = ((size_t)(it.q0 + tok) * a.n_q_heads + (size_t)it.h * a.group + gq) * D + hc * kOCols;
                const uint32_t t_o = t_lane + kTmemO0 + x * 128 + hc * kOCols;
                float o[kOCols];
#pragma unroll
                for (int cc = 0; cc < kOCols / 32; ++cc) tmem_ld32(t_o + cc * 32, o + cc * 32);
                tmem_wait_ld();
                // O is in registers: the next item's products may overwrite it
                tc_fence_before();
                pa::mbar_arrive(&bars->o_free[x]);
                if (valid_row[x]) {
                    scale_f32x2<kOCols>(o, inv);
                    // a thread writes its half row: whole 32-byte sectors when
                    // out allows it (16-byte stores fill half a sector each and
                    // cost as much as a whole one)
                    if (a.out_f32 && a.out_al32) {
                        float* dst = static_cast<float*>(a.out) + orow;
#pragma unroll
                        for (int q = 0; q < kOCols / 8; ++q) {
                            uint32_t w[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) w[e] = __float_as_uint(o[8 * q + e]);
                            st_global_v8(dst + 8 * q, w);
                        }
                    } else if (a.out_f32) {
                        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.out) + orow);
#pragma unroll
                        for (int q = 0; q < kOCols / 4; ++q)
                            dst[q] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
                    } else if (a.out_al32) {
                        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) + orow;
#pragma unroll
                        for (int q = 0; q < kOCols / 16; ++q) {
                            uint32_t w[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) w[e] = pack_bf16_rn(o[16 * q + 2 * e], o[16 * q + 2 * e + 1]);
                            st_global_v8(dst + 16 * q, w);
                        }
                    } else {
                        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + orow);
#pragma unroll
                        for (int q = 0; q < kOCols / 8; ++q)
                            dst[q] = make_uint4(pack_bf16_rn(o[8 * q], o[8 * q + 1]), pack_bf16_rn(o[8 * q + 2], o[8 * q + 3]),
                                                pack_bf16_rn(o[8 * q + 4], o[8 * q + 5]), pack_bf16_rn(o[8 * q + 6], o[8 * q + 7]));
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp0) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
    }
    if (threadIdx.x == 0 && a.sched) {
        // every CTA has made its last claim once all have counted themselves
        // done: the last one leaves both counters at zero for the next launch
        __threadfence();
        if (atomicAdd(a.sched + 1, 1) == (int)gridDim.x - 1) {
            atomicExch(a.sched, 0);
            atomicExch(a.sched + 1, 0);
        }
    }
}

// --- V staging -------------------------------------------------------------------

struct StageArgs {
    const int32_t* block_tables;
    int max_blocks;
    const int32_t* context_lens;
    int num_seqs;
    int block_size;
    int n_kv_heads;
    int num_blocks;
    int l_slot;           // positions per (KV head, sequence)
    int t_slot;
    uint16_t* v_stage;    // [n_kv_heads][num_seqs][l_slot][D]
    uint8_t* v_fmt;       // [n_kv_heads][num_seqs][t_slot]
    int32_t* status;
};

// One thread block per (128-position tile, sequence, KV head): gathers the
// tile's V rows through the block table into the staging buffer, where each
// (KV head, sequence) owns l_slot consecutive rows, so the prefill kernel
// loads a whole tile as one box per 64 columns.  Rows at and past the
// context (anything there, NaN included, would meet weights of 0, and
// 0 * NaN is not 0) become zeros.  The tile is stored as fp16 (exact for
// every bf16 magnitude in [2^-14, 2^16), within 2^-25 below it) unless one
// of its values has a magnitude of 2^16 or more or is not finite; then it
// stays bf16, and its format byte says so.  Tiles at or past the context
// are not read by the prefill kernel and are skipped.  Launched as a
// programmatic dependent: it waits for the work before it on the stream (the
// cache write, or an earlier call still reading this workspace) before it
// reads or writes anything, then lets the prefill kernel begin its launch.
template <int D>
__global__ void __launch_bounds__(256) stage_v_kernel(const uint4* __restrict__ v_cache, const StageArgs a) {
    constexpr int kChunksPerRow = D / 8;                      // 16-byte chunks
    constexpr int kPer = kKv * kChunksPerRow / 256;           // chunks per thread
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int j = blockIdx.x, s = blockIdx.y, h = blockIdx.z;
    int ctx = a.context_lens[s];
    ctx = min(max(ctx, 0), a.max_blocks * a.block_size);     // the prefill kernel flags and clamps the same
    if (j * kKv >= ctx) return;
    const int32_t* table = a.block_tables + (size_t)s * a.max_blocks;
    uint4 v[kPer];
    uint32_t amax = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int c = threadIdx.x + 256 * i;
        const int pos = j * kKv + c / kChunksPerRow;
        v[i] = make_uint4(0, 0, 0, 0);
        if (pos < ctx) {
            const int blk = __ldg(table + pos / a.block_size);
            if (blk >= 0 && blk < a.num_blocks)
                v[i] = __ldg(v_cache + (((size_t)blk * a.n_kv_heads + h) * a.block_size + pos % a.block_size) *
                                           kChunksPerRow + c % kChunksPerRow);
            // a bad entry reads zeros; the prefill kernel's K loads flag it
        }
        amax = max_u16x2(amax, max_u16x2(v[i].x & 0x7fff7fffu, v[i].y & 0x7fff7fffu));
        amax = max_u16x2(amax, max_u16x2(v[i].z & 0x7fff7fffu, v[i].w & 0x7fff7fffu));
    }
    const bool wide = __syncthreads_or((amax & 0xffffu) >= kF16Wide || (amax >> 16) >= kF16Wide) != 0;
    uint4* dst = reinterpret_cast<uint4*>(a.v_stage + ((size_t)(h * a.num_seqs + s) * a.l_slot + (size_t)j * kKv) * D);
#pragma unroll
    for (int i = 0; i < kPer; ++i)
        dst[threadIdx.x + 256 * i] = wide ? v[i]
                                          : make_uint4(bf16x2_to_f16x2(v[i].x), bf16x2_to_f16x2(v[i].y),
                                                       bf16x2_to_f16x2(v[i].z), bf16x2_to_f16x2(v[i].w));
    if (threadIdx.x == 0) a.v_fmt[(size_t)(h * a.num_seqs + s) * a.t_slot + j] = wide ? 1 : 0;
}

// FP8 caches: one thread block per (128-position tile, sequence, KV head)
// gathers the tile's K and V codes (E4M3, one byte each) through the block
// table and stores K as bf16 (for the score products with the caller's bf16
// q) and V as fp16 (for the value products with fp16 weights), in staging
// buffers of the bf16 V staging's layout: both hold every E4M3 value
// exactly.  Rows at and past the context are zeros, and a table entry
// outside the pool reads zeros and is flagged.  The scales are applied by
// the prefill kernel.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t c) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(c));
    return r;
}

template <int D>
__global__ void __launch_bounds__(256) stage_kv_f8_kernel(const uint4* __restrict__ k_cache,
                                                          const uint4* __restrict__ v_cache, uint16_t* k_stage,
                                                          const StageArgs a) {
    constexpr int kChunksPerRow = D / 16;                     // 16 codes per 16-byte chunk
    constexpr int kPer = kKv * kChunksPerRow / 256;           // chunks per thread
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int j = blockIdx.x, s = blockIdx.y, h = blockIdx.z;
    int ctx = a.context_lens[s];
    ctx = min(max(ctx, 0), a.max_blocks * a.block_size);
    if (j * kKv >= ctx) return;
    const int32_t* table = a.block_tables + (size_t)s * a.max_blocks;
    const size_t row0 = ((size_t)(h * a.num_seqs + s) * a.l_slot + (size_t)j * kKv) * D;
#pragma unroll
    for (int kv = 0; kv < 2; ++kv) {
        const uint4* src = kv ? v_cache : k_cache;
        uint4* dst = reinterpret_cast<uint4*>((kv ? a.v_stage : k_stage) + row0);
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int c = threadIdx.x + 256 * i;
            const int pos = j * kKv + c / kChunksPerRow;
            uint4 w = make_uint4(0, 0, 0, 0);
            if (pos < ctx) {
                const int blk = __ldg(table + pos / a.block_size);
                if (blk >= 0 && blk < a.num_blocks)
                    w = __ldg(src + (((size_t)blk * a.n_kv_heads + h) * a.block_size + pos % a.block_size) *
                                        kChunksPerRow + c % kChunksPerRow);
                else if (kv == 0)
                    pa::set_status(a.status, PA_DEV_BAD_BLOCK_ID);
            }
            const uint32_t cw[4] = {w.x, w.y, w.z, w.w};
            uint32_t f[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                f[2 * e] = e4m3x2_to_f16x2((uint16_t)(cw[e] & 0xffffu));
                f[2 * e + 1] = e4m3x2_to_f16x2((uint16_t)(cw[e] >> 16));
            }
            if (kv == 0) {
                // K: fp16 -> fp32 -> bf16, exact at each step for E4M3 values
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const __half2 hv = *reinterpret_cast<const __half2*>(&f[e]);
                    const float2 fv = __half22float2(hv);
                    f[e] = pack_bf16_rn(fv.x, fv.y);
                }
            }
            dst[2 * c] = make_uint4(f[0], f[1], f[2], f[3]);
            dst[2 * c + 1] = make_uint4(f[4], f[5], f[6], f[7]);
        }
    }
}

// Layout of the caller's workspace (each part 256-byte aligned): the V
// staging, then the format bytes; FP8 caches add the K staging.
struct Workspace {
    int l_slot, t_slot;
    size_t stage_bytes, fmt_off, k_off, total;
};

size_t align256(size_t n) { return (n + 255) & ~(size_t)255; }

Workspace workspace_layout(int num_seqs, int max_blocks, int block_size, int n_kv_heads, int d_head, bool f8 = false) {
    Workspace w;
    const long long pos = (long long)max_blocks * block_size;
    w.t_slot = (int)((pos + kKv - 1) / kKv);
    w.l_slot = w.t_slot * kKv;
    w.stage_bytes = (size_t)n_kv_heads * num_seqs * w.l_slot * d_head * 2;
    w.fmt_off = align256(w.stage_bytes);
    w.k_off = w.fmt_off + align256((size_t)n_kv_heads * num_seqs * w.t_slot);
    w.total = w.k_off;
    if (f8) w.total = w.k_off + align256(w.stage_bytes);
    return w;
}

// --- host side -------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

bool encode(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
            const cuuint32_t* box) {
    auto enc = encode_fn();
    if (!enc) return false;
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool kF8>
int g_smem_done[64];   // per kernel instantiation: bytes opted in, by device

int num_sms() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev < 64 && cached[dev]) return cached[dev];
    int n = 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
    if (dev < 64) cached[dev] = n;
    return n;
}

template <int D, bool kF8>
int launch(const PrefillArgs& a, const StageArgs& sa, const void* q, const void* k_cache, const void* v_cache,
           uint16_t* k_stage, int num_tokens, long long cache_rows, dim3 grid, cudaStream_t st) {
    CUtensorMap mq, mk, mv;
    const cuuint64_t qdims[3] = {(cuuint64_t)D, (cuuint64_t)a.n_q_heads, (cuuint64_t)num_tokens};
    const cuuint64_t qstr[2] = {(cuuint64_t)D * 2, (cuuint64_t)a.n_q_heads * D * 2};
    const cuuint32_t qbox[3] = {64u, (cuuint32_t)a.group, (cuuint32_t)a.tq};
    const cuuint64_t cdims[2] = {(cuuint64_t)D, (cuuint64_t)cache_rows};
    const cuuint64_t cstr[1] = {(cuuint64_t)D * 2};
    const cuuint32_t cbox[2] = {64u, (cuuint32_t)a.block_size};
    const cuuint64_t sdims[2] = {(cuuint64_t)D, (cuuint64_t)a.n_kv_heads * a.num_seqs * a.l_slot};
    const cuuint32_t sbox[2] = {64u, (cuuint32_t)kKv};
    // q from the caller; K from the caller's cache (bf16) or from the staging
    // (FP8); V from the staging (the maps only move 16-bit elements)
    if (!encode(&mq, q, 3, qdims, qstr, qbox) ||
        !(kF8 ? encode(&mk, k_stage, 2, sdims, cstr, sbox) : encode(&mk, k_cache, 2, cdims, cstr, cbox)) ||
        !encode(&mv, sa.v_stage, 2, sdims, cstr, sbox))
        return PA_ERR_CUDA;
    if (pa_host::ensure_smem_attr(prefill_kernel<D, kF8>, PGeo<D>::kSmem, g_smem_done<D, kF8>) != cudaSuccess)
        return PA_ERR_CUDA;
    const dim3 sgrid((unsigned)sa.t_slot, (unsigned)sa.num_seqs, (unsigned)sa.n_kv_heads);
    if constexpr (kF8) {
        if (pa_host::launch_dependent(stage_kv_f8_kernel<D>, sgrid, dim3(256), 0, st,
                                      static_cast<const uint4*>(k_cache), static_cast<const uint4*>(v_cache), k_stage,
                                      sa) != cudaSuccess)
            return PA_ERR_CUDA;
    } else {
        if (pa_host::launch_dependent(stage_v_kernel<D>, sgrid, dim3(256), 0, st, static_cast<const uint4*>(v_cache),
                                      sa) != cudaSuccess)
            return PA_ERR_CUDA;
    }
    return pa_host::launch_dependent(prefill_kernel<D, kF8>, grid, dim3(kThreads), PGeo<D>::kSmem, st, mq, mk, mv,
                                     a) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

int prefill_impl(void* out, int out_dtype, const void* q, const void* k_cache, const void* v_cache,
                 const int32_t* block_tables, int max_blocks_per_seq, const int32_t* query_start,
                 const int32_t* context_lens, int num_seqs, int num_tokens, int max_query_len, int num_blocks,
                 int block_size, float scale, int n_q_heads, int n_kv_heads, int d_head, void* workspace,
                 size_t workspace_bytes, int32_t* sched_dev, int32_t* status_dev, void* stream, bool f8,
                 float k_scale, float v_scale) {
    if (num_seqs < 0 || num_tokens < 0 || max_query_len < 0 || num_blocks <= 0 || max_blocks_per_seq < 0 ||
        n_q_heads <= 0 || n_kv_heads <= 0)
        return PA_ERR_INVALID_ARG;
    if (n_q_heads % n_kv_heads != 0) return PA_ERR_UNSUPPORTED;         // as pa_decode
    if (out_dtype != PA_DTYPE_BF16 && out_dtype != PA_DTYPE_F32) return PA_ERR_INVALID_ARG;
    if (f8 && (!(k_scale > 0.f) || !(v_scale > 0.f) || !(k_scale < INFINITY) || !(v_scale < INFINITY)))
        return PA_ERR_INVALID_ARG;
    if (!pa_host::supported_block_size(block_size) || !pa_host::supported_d_head(d_head)) return PA_ERR_UNSUPPORTED;
    if (f8 && d_head != 128) return PA_ERR_UNSUPPORTED;
    const int group = n_q_heads / n_kv_heads;
    if (group > kRows || kRows % group != 0) return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0 || num_tokens == 0 || max_query_len == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !query_start || !context_lens)
        return PA_ERR_INVALID_ARG;
    if (max_blocks_per_seq == 0) return PA_ERR_INVALID_ARG;
    if (num_seqs > 65535) return PA_ERR_UNSUPPORTED;
    const Workspace ws = workspace_layout(num_seqs, max_blocks_per_seq, block_size, n_kv_heads, d_head, f8);
    if ((long long)n_kv_heads * num_seqs * ws.l_slot > INT_MAX - kKv) return PA_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < ws.total) return PA_ERR_WORKSPACE;
    if (!pa_host::aligned16(out) || !pa_host::aligned16(q) || !pa_host::aligned16(k_cache) ||
        !pa_host::aligned16(v_cache) || !pa_host::aligned16(workspace) ||
        (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
        (reinterpret_cast<uintptr_t>(query_start) & 3u) || (reinterpret_cast<uintptr_t>(context_lens) & 3u) ||
        (reinterpret_cast<uintptr_t>(sched_dev) & 3u))
        return PA_ERR_MISALIGNED;
    const long long cache_rows = (long long)num_blocks * n_kv_heads * block_size;
    if (cache_rows > INT_MAX - 64 || (long long)max_blocks_per_seq * block_size > INT_MAX / 2 ||
        n_kv_heads > 65535)
        return PA_ERR_UNSUPPORTED;
    const int tq = kRows / group;
    const long long tiles = (max_query_len + 2 * tq - 1) / (2 * tq);
    if (tiles * num_seqs > INT_MAX) return PA_ERR_UNSUPPORTED;

    uint8_t* w8 = static_cast<uint8_t*>(workspace);
    PrefillArgs a;
    a.out = out;
    a.out_f32 = out_dtype == PA_DTYPE_F32;
    a.out_al32 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0;
    a.block_tables = block_tables;
    a.max_blocks = max_blocks_per_seq;
    a.query_start = query_start;
    a.context_lens = context_lens;
    a.num_seqs = num_seqs;
    a.num_tokens = num_tokens;
    a.tiles_per_seq = (int)tiles;
    a.block_size = block_size;
    a.n_kv_heads = n_kv_heads;
    a.group = group;
    a.tq = tq;
    a.n_q_heads = n_q_heads;
    a.num_blocks = num_blocks;
    a.oob_row = (int)cache_rows;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.v_fmt = w8 + ws.fmt_off;
    a.l_slot = ws.l_slot;
    a.t_slot = ws.t_slot;
    a.k_scale = f8 ? k_scale : 1.f;
    a.v_scale = f8 ? v_scale : 1.f;
    a.status = status_dev;
    a.sched = reinterpret_cast<int*>(sched_dev);
    const long long items = tiles * num_seqs * n_kv_heads;
    if (items > INT_MAX - 4096) return PA_ERR_UNSUPPORTED;    // claims run past the last item by one per CTA
    const int sms = num_sms();
    const dim3 grid((unsigned)(items < sms ? items : sms));
    const long long per_head = tiles * num_seqs;
    long long hpg = (2LL * grid.x + per_head - 1) / per_head;
    a.heads_per_group = (int)(hpg < 1 ? 1 : hpg > n_kv_heads ? n_kv_heads : hpg);
    StageArgs sa;
    sa.block_tables = block_tables;
    sa.max_blocks = max_blocks_per_seq;
    sa.context_lens = context_lens;
    sa.num_seqs = num_seqs;
    sa.block_size = block_size;
    sa.n_kv_heads = n_kv_heads;
    sa.num_blocks = num_blocks;
    sa.l_slot = ws.l_slot;
    sa.t_slot = ws.t_slot;
    sa.v_stage = reinterpret_cast<uint16_t*>(w8);
    sa.v_fmt = w8 + ws.fmt_off;
    sa.status = status_dev;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (f8)
        return launch<128, true>(a, sa, q, k_cache, v_cache, reinterpret_cast<uint16_t*>(w8 + ws.k_off), num_tokens,
                                 cache_rows, grid, st);
    return d_head == 128 ? launch<128, false>(a, sa, q, k_cache, v_cache, nullptr, num_tokens, cache_rows, grid, st)
                         : launch<64, false>(a, sa, q, k_cache, v_cache, nullptr, num_tokens, cache_rows, grid, st);
}

}  // namespace

extern "C" {

size_t pa_prefill_workspace_size(int num_seqs, int max_blocks_per_seq, int block_size, int n_kv_heads,
                                 int d_head) {
    if (num_seqs <= 0 || max_blocks_per_seq <= 0 || block_size <= 0 || n_kv_heads <= 0 || d_head <= 0) return 0;
    return workspace_layout(num_seqs, max_blocks_per_seq, block_size, n_kv_heads, d_head).total;
}

size_t pa_prefill_fp8_workspace_size(int num_seqs, int max_blocks_per_seq, int block_size, int n_kv_heads,
                                     int d_head) {
    if (num_seqs <= 0 || max_blocks_per_seq <= 0 || block_size <= 0 || n_kv_heads <= 0 || d_head <= 0) return 0;
    return workspace_layout(num_seqs, max_blocks_per_seq, block_size, n_kv_heads, d_head, true).total;
}

int pa_prefill(void* out, int out_dtype, const void* q, const void* k_cache, const void* v_cache,
               const int32_t* block_tables, int max_blocks_per_seq, const int32_t* query_start,
               const int32_t* context_lens, int num_seqs, int num_tokens, int max_query_len, int num_blocks,
               int block_size, float scale, int n_q_heads, int n_kv_heads, int d_head, void* workspace,
               size_t workspace_bytes, int32_t* sched_dev, int32_t* status_dev, void* stream) {
    return prefill_impl(out, out_dtype, q, k_cache, v_cache, block_tables, max_blocks_per_seq, query_start,
                        context_lens, num_seqs, num_tokens, max_query_len, num_blocks, block_size, scale, n_q_heads,
                        n_kv_heads, d_head, workspace, workspace_bytes, sched_dev, status_dev, stream, false, 1.f, 1.f);
}

int pa_prefill_fp8(void* out, int out_dtype, const void* q, const void* k_cache, const void* v_cache,
                   const int32_t* block_tables, int max_blocks_per_seq, const int32_t* query_start,
                   const int32_t* context_lens, int num_seqs, int num_tokens, int max_query_len, int num_blocks,
                   int block_size, float scale, float k_scale, float v_scale, int n_q_heads, int n_kv_heads,
                   int d_head, void* workspace, size_t workspace_bytes, int32_t* sched_dev, int32_t* status_dev,
                   void* stream) {
    return prefill_impl(out, out_dtype, q, k_cache, v_cache, block_tables, max_blocks_per_seq, query_start,
                        context_lens, num_seqs, num_tokens, max_query_len, num_blocks, block_size, scale, n_q_heads,
                        n_kv_heads, d_head, workspace, workspace_bytes, sched_dev, status_dev, stream, true, k_scale,
                        v_scale);
}

}  // extern "C"
