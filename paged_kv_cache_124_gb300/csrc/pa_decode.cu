// Paged single-query (decode) attention for sm_103a.
//
// What is computed ("PagedAttention: Virtual Memory for the KV Cache",
// sections 1, 7 and 13; "PagedAttention in vLLM: scattered memory, exact
// attention", sections 10 and 11): for each sequence and query head,
// softmax(scale * q . K^T) . V over the sequence's cached positions, where
// position j lives in physical block block_table[j / B] at offset j % B.
//
// How (GB300 design):
//  * Work is cut into tiles of 16 positions of one (sequence, KV head).  A
//    warp consumes tiles from a ring of shared-memory stages it owns; each
//    stage holds the tile's K and V rows, brought in by TMA tensor copies
//    (cp.async.bulk.tensor over a 2-D view of the cache as rows of d_head,
//    boxes of 64 columns x 16 rows -- 8 rows for 8-position blocks -- with
//    128-byte swizzle) addressed through the block table and counted on an
//    mbarrier.  Lane 0 refills a stage as soon as the warp is done with it.
//  * All query heads of a GQA group (up to 8) are computed from the same K/V
//    bytes: the cache is read once per KV head.
//  * Both contractions of a tile run on the tensor pipe with warp-level
//    mma.m16n8k16 (bf16 in, fp32 accumulate): S[16 x 8 heads] = K . Q^T,
//    then O^T[d_head x 8] += V^T . P^T.  The ncu profile of the CUDA-core
//    form of this kernel showed it issue- and latency-bound (about 800
//    instructions per tile at 48% issue efficiency, DRAM 72% busy); the MMA
//    form needs about 150.
//  * Softmax is online, in fp32, with a running maximum per head in the log2
//    domain.  P enters P.V as two bf16 terms (hi + lo), which keeps its
//    rounding within about 2^-16 relative instead of bf16's 2^-8.
//  * One thread block of 4 warps per (sequence, head group, partition of
//    partition_size positions); the hardware hands blocks to SMs as others
//    finish, which balances ragged batches.  When the head groups alone fill
//    two waves and the longest context spans four partitions or more, most
//    of that grid would be empty partitions of short sequences, so instead
//    the resident blocks claim the (sequence, head group, partition) items
//    that exist from a counter in the workspace.  The 4 warps of a block are
//    merged in shared memory; a sequence that fits one partition is written
//    directly.  Otherwise each block leaves its partition's statistics
//    (m, z, u) in the workspace and lse_merge_kernel -- launched as a
//    programmatic dependent so that its launch overlaps the first kernel's
//    drain -- merges them: the exact block merge of the second page,
//    section 11, as the "secondary reduction kernel" of the first page,
//    section 13.

#include <cuda.h>            // CUtensorMap and its enums (types only)
#include <cudaTypedefs.h>    // PFN_cuTensorMapEncodeTiled
#include <math.h>

#include <mutex>

#include "pa_common.cuh"

namespace {

#ifndef PA_DECODE_STAGES
#define PA_DECODE_STAGES 2         // stages per warp ring
#endif
#ifndef PA_DECODE_MIN_BLOCKS
#define PA_DECODE_MIN_BLOCKS 3     // resident thread blocks per SM the kernels are built for
#endif

#ifndef PA_DECODE_WARPS
#define PA_DECODE_WARPS 4          // warps per thread block
#endif

constexpr int kTile = 16;          // positions per stage
constexpr int kWarps = PA_DECODE_WARPS;
constexpr int kStages = PA_DECODE_STAGES;
constexpr int kThreads = kWarps * 32;
constexpr int kHeads = 8;          // query heads per MMA (the n = 8 of m16n8k16)
constexpr int kMaxProbes = 2000000;   // ~2 s bound on any single wait
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kMaxPartition = 8192;

// Arguments shared by both schedules.
struct DecodeArgs {
    void* out;
    const __nv_bfloat16* q;
    const int32_t* block_tables;
    const int32_t* context_lens;
    float* part_max;
    float* part_sum;
    float* part_acc;
    int32_t* status;
    float scale_log2;        // scale * log2(e): scores live in the log2 domain
    int out_f32;
    int block_size;
    int log2_block;
    int n_q_heads;
    int n_kv_heads;
    int group;               // G = n_q_heads / n_kv_heads
    int heads_per_block;     // hpb = min(G, 8): query heads computed per K/V read
    int n_sub;               // G / hpb
    int max_blocks_per_seq;
    int num_blocks;
    int ctx_cap;             // min(max_blocks_per_seq * B, max_context_len)
    int num_seqs;
    int partition_size;
    int max_parts;
    float k_scale;           // FP8 caches: dequantisation scale of K (folded into the score scale)
    float u_scale;           // factor on the weighted value sums (FP8: V scale / 2^15; else 1)
    float v_scale;           // FP8 caches: V scale (quantises appended values)
    // Fused append (pa_decode_append*): the token at position ctx - 1 of
    // sequence s has keys k_new[s] and values v_new[s] ([S][Hkv][D] bf16);
    // null: plain decode.
    const __nv_bfloat16* k_new;
    const __nv_bfloat16* v_new;
    uint8_t* k_cache;        // the caches, written at the appended positions
    uint8_t* v_cache;
    // Claimed work (many short sequences): {next item, blocks done} in the
    // workspace's header, zero between calls; n_units head groups per
    // sequence.
    int* claim;
    int n_units;
};

// Claimed work: at most this many sequences (their item offsets live in
// shared memory).
constexpr int kClaimMaxSeqs = 1024;

// Shared-memory geometry; F8: one-byte (E4M3) cache elements, rows of d_head
// bytes (d_head 128: one 128-byte box per row).
// NK: KV heads per tile (2: two adjacent KV heads of the same positions, whose
// 2 x 4 query heads fill the 8 columns of the products; FP8 with G = 4).
template <int D, bool F8 = false, int NK = 1>
struct Geo {
    static constexpr int kHalves = F8 ? 1 : D / 64;       // 128-byte boxes per row
    static constexpr int kBoxBytes = kTile * 128;         // one swizzled 16 x 128-byte region
    static constexpr int kHeadBytes = kHalves * kBoxBytes;   // K or V of one KV head's tile
    static constexpr int kTileBytes = NK * kHeadBytes;    // K or V of one tile
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kRingBytes = kWarps * kStages * kStageBytes;
    static constexpr int kSteps = D / 16;                 // k-steps of S, m-tiles of O^T
};

__device__ __forceinline__ void store_out(void* out, int f32, size_t i, float v) {
    if (f32)
        static_cast<float*>(out)[i] = v;
    else
        static_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(v);
}

__device__ __forceinline__ float fast_exp2(float x) {      // 2^x; 2^-inf = +0
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` in a region the
// TMA wrote with 128-byte swizzle (region base 1024-byte aligned): the chunk
// index is XOR-ed with the row index modulo 8.
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

// D[16 x 8] += A[16 x 16] . B[16 x 8], bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;"
        ::"r"(pa::smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1),
        "r"(pa::smem_addr(bar)), "l"(policy)
        : "memory");
}

// Enqueue the TMA copies of one tile (16 positions of one KV head) into a
// stage: K and V rows of block blk0 from offset off0 (and, for 8-position
// blocks, the next 8 rows from block blk1).  Returns nothing; the stage's
// barrier expects exactly the bytes issued.  Boxes are always full: rows
// past the context come along and are masked in the math.
template <int D, bool F8, int NK = 1>
__device__ __forceinline__ void issue_tile(uint8_t* stage, uint64_t* bar, const CUtensorMap* mk,
                                           const CUtensorMap* mv, int blk0, int blk1, int off0, int nv, int kvh,
                                           const DecodeArgs& a, uint64_t policy) {
    using G = Geo<D, F8, NK>;
    const int B = a.block_size;
    const int box_rows = B < kTile ? B : kTile;
    const int n_rows = (nv + box_rows - 1) / box_rows;          // 1, or 2 for 8-position blocks
    pa::mbar_arrive_expect_tx(bar, (uint32_t)(2 * NK * G::kHalves * n_rows * box_rows * 128));
    for (int r = 0; r < n_rows; ++r) {
        int blk = r == 0 ? blk0 : blk1;
        if (blk < 0 || blk >= a.num_blocks) {
            pa::set_status(a.status, PA_DEV_BAD_BLOCK_ID);
            blk = 0;
        }
#pragma unroll
        for (int hh = 0; hh < NK; ++hh) {
            const int row = (blk * a.n_kv_heads + kvh + hh) * B + (r == 0 ? off0 : 0);
#pragma unroll
            for (int h = 0; h < G::kHalves; ++h) {
                uint8_t* dst = stage + hh * G::kHeadBytes + h * G::kBoxBytes + r * box_rows * 128;
                tma_load_2d(dst, mk, h * 64, row, bar, policy);
                tma_load_2d(dst + G::kTileBytes, mv, h * 64, row, bar, policy);
            }
        }
    }
}

// Per-warp running state of one (unit, range): heads h0 = 2 t4, h1 = 2 t4 + 1
// of the 8-head MMA group, lane-local sums, and O^T in the MMA C layout
// (acc[m] = O^T rows 16 m + g and 16 m + g + 8, columns h0 and h1).
template <int D>
struct WarpState {
    float m0, m1, l0, l1;
    float acc[Geo<D>::kSteps][4];

    __device__ __forceinline__ void reset() {
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
#pragma unroll
        for (int m = 0; m < Geo<D>::kSteps; ++m) acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0.f;
    }

    // Sum the lane-local l over the 8 lanes of a column group.
    __device__ __forceinline__ void finish_sums() {
#pragma unroll
        for (int msk = 4; msk <= 16; msk <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, msk);
            l1 += __shfl_xor_sync(0xffffffffu, l1, msk);
        }
    }
};

// Fold one tile (stage at shared addresses ks / vs, nv valid positions) into
// the warp's state.  qb: q as the B operand of S = K . Q^T.
template <int D>
__device__ __forceinline__ void consume_tile(WarpState<D>& st, uint32_t ks, uint32_t vs, int nv,
                                             const uint32_t (&qb)[Geo<D>::kSteps][2], float scale_log2, int lane) {
    using G = Geo<D>;
    const int g = lane >> 2, t4 = lane & 3, mi = lane >> 3;
    // ldmatrix lane addressing (see swz): for S the lanes of matrix mi point at
    // K rows (mi & 1) * 8 + lane % 8, chunk +(mi >> 1); for O^T they point at V
    // rows (mi >> 1) * 8 + lane % 8, chunk +(mi & 1).
    const int k_row = ((mi & 1) << 3) + (lane & 7), k_cadd = mi >> 1;
    const int v_row = ((mi >> 1) << 3) + (lane & 7), v_cadd = mi & 1;

    // ---- S = K . Q^T (two accumulators for a shorter dependency chain) ----
    float s_a[4] = {0.f, 0.f, 0.f, 0.f}, s_b[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < G::kSteps; ++kk) {
        uint32_t af[4];
        ldsm_x4(ks + (kk >> 2) * G::kBoxBytes + swz(k_row, 2 * (kk & 3) + k_cadd), af);
        if (kk & 1)
            mma16816(s_b, af, qb[kk][0], qb[kk][1]);
        else
            mma16816(s_a, af, qb[kk][0], qb[kk][1]);
    }
    // s[0]: (position g, head h0), s[1]: (g, h1), s[2]: (g + 8, h0), s[3]: (g + 8, h1)
    float s[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) s[i] = (s_a[i] + s_b[i]) * scale_log2;
    if (g >= nv) s[0] = s[1] = -INFINITY;          // positions past the context
    if (g + 8 >= nv) s[2] = s[3] = -INFINITY;

    // ---- online softmax -------------------------------------------------------
    float b0 = fmaxf(s[0], s[2]), b1 = fmaxf(s[1], s[3]);
#pragma unroll
    for (int msk = 4; msk <= 16; msk <<= 1) {
        b0 = fmaxf(b0, __shfl_xor_sync(0xffffffffu, b0, msk));
        b1 = fmaxf(b1, __shfl_xor_sync(0xffffffffu, b1, msk));
    }
    const float n0 = fmaxf(st.m0, b0), n1 = fmaxf(st.m1, b1);
    // rescale only when some head's maximum grew (rare after the first tiles)
    if (__any_sync(0xffffffffu, n0 != st.m0 || n1 != st.m1)) {
        const float al0 = fast_exp2(st.m0 - n0), al1 = fast_exp2(st.m1 - n1);
        st.l0 *= al0;
        st.l1 *= al1;
#pragma unroll
        for (int m = 0; m < G::kSteps; ++m) {
            st.acc[m][0] *= al0;
            st.acc[m][1] *= al1;
            st.acc[m][2] *= al0;
            st.acc[m][3] *= al1;
        }
        st.m0 = n0;
        st.m1 = n1;
    }
    const float p0 = fast_exp2(s[0] - n0), p1 = fast_exp2(s[1] - n1);
    const float p2 = fast_exp2(s[2] - n0), p3 = fast_exp2(s[3] - n1);
    st.l0 += p0 + p2;
    st.l1 += p1 + p3;

    // ---- P^T as the B operand, split into bf16 hi + lo -------------------------
    const uint32_t h01 = pack_bf16(p0, p1), h23 = pack_bf16(p2, p3);
    const float2 f01 = pa::bf16x2_to_float2(h01), f23 = pa::bf16x2_to_float2(h23);
    const uint32_t l01 = pack_bf16(p0 - f01.x, p1 - f01.y), l23 = pack_bf16(p2 - f23.x, p3 - f23.y);
    const uint32_t bh0 = movmatrix_trans(h01), bh1 = movmatrix_trans(h23);
    const uint32_t bl0 = movmatrix_trans(l01), bl1 = movmatrix_trans(l23);

    // ---- O^T += V^T . P^T --------------------------------------------------------
    // in the context's last tile the V rows past its end are zeroed (0 * NaN)
    auto pv = [&](uint32_t mlo, uint32_t mhi, bool masked) {
#pragma unroll
        for (int m = 0; m < G::kSteps; ++m) {
            uint32_t af[4];
            ldsm_x4_trans(vs + (m >> 2) * G::kBoxBytes + swz(v_row, 2 * (m & 3) + v_cadd), af);
            if (masked) {
                af[0] &= mlo;
                af[1] &= mlo;
                af[2] &= mhi;
                af[3] &= mhi;
            }
            mma16816(st.acc[m], af, bh0, bh1);
            mma16816(st.acc[m], af, bl0, bl1);
        }
    };
    if (nv < kTile) {
        const int t = 2 * t4;
        pv((t < nv ? 0x0000ffffu : 0u) | (t + 1 < nv ? 0xffff0000u : 0u),
           (t + 8 < nv ? 0x0000ffffu : 0u) | (t + 9 < nv ? 0xffff0000u : 0u), true);
    } else {
        pv(0xffffffffu, 0xffffffffu, false);
    }
}

// q of query heads [qh0, qh0 + hpb) of one sequence as the B operand of
// S = K . Q^T: lane holds q[head g][16 k + 2 t4 + {0,1}] and
// q[head g][16 k + 8 + 2 t4 + {0,1}]; heads past hpb are zero.
template <int D>
__device__ __forceinline__ void load_q(uint32_t (&qb)[Geo<D>::kSteps][2], const __nv_bfloat16* qrow0, int hpb,
                                       int lane) {
    const int g = lane >> 2, t4 = lane & 3;
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(qrow0 + (size_t)(g < hpb ? g : 0) * D);
#pragma unroll
    for (int k = 0; k < Geo<D>::kSteps; ++k) {
        qb[k][0] = g < hpb ? qrow[8 * k + t4] : 0u;
        qb[k][1] = g < hpb ? qrow[8 * k + 4 + t4] : 0u;
    }
}

// ---------------------------------------------------------------------------
// FP8 (E4M3) caches.  Codes are turned into f16 in registers (exact: every
// E4M3 value is an f16) and both products run as f16 MMAs.  The contraction
// index of each product may be permuted freely as long as both operands use
// the same order, and the output rows of O^T may be permuted if the final
// write undoes it; both are used so that ldmatrix, reading 8 x 16-byte
// matrices from the swizzled tiles without bank conflicts, hands every lane
// bytes that go straight into fragments:
//   * S = K . Q^T: an ldmatrix row segment is 16 codes of one position; lane
//     (g, t4) receives codes 4 t4 .. 4 t4 + 3, so k columns 2t4, 2t4+1,
//     2t4+8, 2t4+9 of a 16-wide k-step hold d = 4t4 .. 4t4+3; q's fragments
//     use the same order.  One ldmatrix.x4 covers two k-steps.  q is
//     converted to f16 after scaling each head by a power of two that puts
//     its largest element in [2^14, 2^15); the score scale undoes it,
//     together with the K scale.
//   * O^T += V^T . P^T: ldmatrix.trans on 16-bit elements hands lane (g, t4)
//     codes 2g, 2g+1 of positions 2t4 and 2t4+1; one byte permute pairs them
//     by position, so row g of m-tile m holds d = 16m + 2g and row g + 8 holds
//     d = 16m + 2g + 1.  One ldmatrix.x4.trans covers two m-tiles.  P is
//     scaled by 2^15 before it is rounded to f16 (11-bit significand,
//     weights kept down to 2^-39 of the row maximum); the V scale and 2^-15
//     multiply the final sums.
// ---------------------------------------------------------------------------

__device__ __forceinline__ void mma16816_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four E4M3 codes (bytes 0..3 of x) to two f16x2: bytes 0, 1 -> lo, bytes 2, 3 -> hi.
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t x, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(x));
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// q of query heads [qh0, qh0 + hpb) as f16 B fragments in the permuted order
// (lane holds q[head g][16 k + 4 t4 + 0..3] times the head's power-of-two
// scale); returns that scale for head g.
template <int D>
__device__ __forceinline__ float load_q_f8(uint32_t (&qb)[Geo<D>::kSteps][2], const __nv_bfloat16* qrow0, int hpb,
                                           int lane) {
    constexpr int kSteps = Geo<D>::kSteps;
    const int g = lane >> 2, t4 = lane & 3;
    const uint2* qrow = reinterpret_cast<const uint2*>(qrow0 + (size_t)(g < hpb ? g : 0) * D);
    float v[kSteps][4];
    float mx = 0.f;
#pragma unroll
    for (int k = 0; k < kSteps; ++k) {
        const uint2 w = g < hpb ? qrow[4 * k + t4] : make_uint2(0u, 0u);   // d = 16 k + 4 t4 .. +3
        const float2 f01 = pa::bf16x2_to_float2(w.x), f23 = pa::bf16x2_to_float2(w.y);
        v[k][0] = f01.x;
        v[k][1] = f01.y;
        v[k][2] = f23.x;
        v[k][3] = f23.y;
        mx = fmaxf(mx, fmaxf(fmaxf(fabsf(f01.x), fabsf(f01.y)), fmaxf(fabsf(f23.x), fabsf(f23.y))));
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    int eb = (__float_as_int(mx) >> 23) & 0xff;             // biased exponent of the head's maximum
    eb = eb < 14 ? 14 : (eb > 254 ? 254 : eb);
    const float sh = __int_as_float((268 - eb) << 23);      // 2^(141 - eb): maximum into [2^14, 2^15)
#pragma unroll
    for (int k = 0; k < kSteps; ++k) {
        qb[k][0] = pack_f16(v[k][0] * sh, v[k][1] * sh);
        qb[k][1] = pack_f16(v[k][2] * sh, v[k][3] * sh);
    }
    return sh;
}

// consume_tile for an FP8 stage; c0 / c1: score scale of heads h0 / h1 (the
// log2-domain softmax scale times the K scale over the heads' q scales).
// NK = 2: the stage holds two KV heads (K0, K1, then V0, V1, kHeadBytes
// apart); query heads 0-3 of the 8 product columns read KV head 0 and 4-7 KV
// head 1, so qb[hh] is q with the other head's columns zeroed, and P^T is
// masked the same way for each head's value product.
template <int D, int NK = 1>
__device__ __forceinline__ void consume_tile_f8(WarpState<D>& st, uint32_t ks, uint32_t vs, int nv,
                                                const uint32_t (&qb)[NK][Geo<D>::kSteps][2], float c0, float c1,
                                                int lane) {
    constexpr int kSteps = Geo<D>::kSteps;
    constexpr uint32_t kHeadBytes = Geo<D, true, NK>::kHeadBytes;
    const int g = lane >> 2, t4 = lane & 3, mi = lane >> 3;
    // ldmatrix lane addressing for both tiles: matrix mi covers positions
    // (mi & 1) * 8 .. +7 of 16-byte chunk c + (mi >> 1)
    const int row = ((mi & 1) << 3) + (lane & 7), cadd = mi >> 1;

    float s_a[4] = {0.f, 0.f, 0.f, 0.f}, s_b[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < kSteps / 2; ++j) {
#pragma unroll
        for (int hh = 0; hh < NK; ++hh) {
            uint32_t r[4];
            ldsm_x4(ks + hh * kHeadBytes + swz(row, 2 * j + cadd), r);   // r0, r1: rows g, g+8 of chunk 2j; r2, r3: chunk 2j+1
            uint32_t af[4];
            e4m3x4_to_f16(r[0], af[0], af[2]);
            e4m3x4_to_f16(r[1], af[1], af[3]);
            mma16816_f16(s_a, af, qb[hh][2 * j][0], qb[hh][2 * j][1]);
            e4m3x4_to_f16(r[2], af[0], af[2]);
            e4m3x4_to_f16(r[3], af[1], af[3]);
            mma16816_f16(s_b, af, qb[hh][2 * j + 1][0], qb[hh][2 * j + 1][1]);
        }
    }
    float s[4];
    s[0] = (s_a[0] + s_b[0]) * c0;
    s[1] = (s_a[1] + s_b[1]) * c1;
    s[2] = (s_a[2] + s_b[2]) * c0;
    s[3] = (s_a[3] + s_b[3]) * c1;
    if (g >= nv) s[0] = s[1] = -INFINITY;
    if (g + 8 >= nv) s[2] = s[3] = -INFINITY;

    float b0 = fmaxf(s[0], s[2]), b1 = fmaxf(s[1], s[3]);
#pragma unroll
    for (int msk = 4; msk <= 16; msk <<= 1) {
        b0 = fmaxf(b0, __shfl_xor_sync(0xffffffffu, b0, msk));
        b1 = fmaxf(b1, __shfl_xor_sync(0xffffffffu, b1, msk));
    }
    const float n0 = fmaxf(st.m0, b0), n1 = fmaxf(st.m1, b1);
    // rescale only when some head's maximum grew (rare after the first tiles)
    if (__any_sync(0xffffffffu, n0 != st.m0 || n1 != st.m1)) {
        const float al0 = fast_exp2(st.m0 - n0), al1 = fast_exp2(st.m1 - n1);
        st.l0 *= al0;
        st.l1 *= al1;
#pragma unroll
        for (int m = 0; m < kSteps; ++m) {
            st.acc[m][0] *= al0;
            st.acc[m][1] *= al1;
            st.acc[m][2] *= al0;
            st.acc[m][3] *= al1;
        }
        st.m0 = n0;
        st.m1 = n1;
    }
    const float p0 = fast_exp2(s[0] - n0), p1 = fast_exp2(s[1] - n1);
    const float p2 = fast_exp2(s[2] - n0), p3 = fast_exp2(s[3] - n1);
    st.l0 += p0 + p2;
    st.l1 += p1 + p3;

    constexpr float kP = 32768.f;                                   // 2^15
    const uint32_t bh0 = movmatrix_trans(pack_f16(p0 * kP, p1 * kP));
    const uint32_t bh1 = movmatrix_trans(pack_f16(p2 * kP, p3 * kP));
    // B fragment lane (g, t4) holds column g: query head g reads KV head g / 4
    uint32_t bp[NK][2];
#pragma unroll
    for (int hh = 0; hh < NK; ++hh) {
        const bool mine = NK == 1 || (g >> 2) == hh;
        bp[hh][0] = mine ? bh0 : 0u;
        bp[hh][1] = mine ? bh1 : 0u;
    }

    // P.V over the tile; in the context's last tile the V rows past its end
    // are zeroed (their codes may be NaN, and 0 * NaN is not 0)
    auto pv = [&](uint32_t mlo, uint32_t mhi, bool masked) {
#pragma unroll
        for (int j = 0; j < kSteps / 2; ++j) {
#pragma unroll
            for (int hh = 0; hh < NK; ++hh) {
                uint32_t r[4];
                // r0 / r1: positions 2t4, 2t4+1 / 2t4+8, 2t4+9 of chunk 2j (codes 2g, 2g+1
                // of each); r2 / r3: the same for chunk 2j+1
                ldsm_x4_trans(vs + hh * kHeadBytes + swz(row, 2 * j + cadd), r);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t af[4];
                    e4m3x4_to_f16(prmt(r[2 * h], r[2 * h], 0x3120u), af[0], af[1]);   // [p0 d0, p1 d0 | p0 d1, p1 d1]
                    e4m3x4_to_f16(prmt(r[2 * h + 1], r[2 * h + 1], 0x3120u), af[2], af[3]);
                    if (masked) {
                        af[0] &= mlo;
                        af[1] &= mlo;
                        af[2] &= mhi;
                        af[3] &= mhi;
                    }
                    mma16816_f16(st.acc[2 * j + h], af, bp[hh][0], bp[hh][1]);
                }
            }
        }
    };
    if (nv < kTile) {
        const int t = 2 * t4;
        pv((t < nv ? 0x0000ffffu : 0u) | (t + 1 < nv ? 0xffff0000u : 0u),
           (t + 8 < nv ? 0x0000ffffu : 0u) | (t + 9 < nv ? 0xffff0000u : 0u), true);
    } else {
        pv(0xffffffffu, 0xffffffffu, false);
    }
}

// Every lane waits for the stage itself (visibility of the async copies);
// the decision to give up is warp-uniform.  On a timeout the status is
// flagged and the warp waits again, each with the full bound, for every
// stage it has issued and not consumed (stages k .. issued - 1, this one
// included), so that no copy lands in shared memory after the block has
// moved on; `drained` is cleared if one of them still has not landed.
__device__ __forceinline__ bool wait_stage(uint64_t* bars, int k, int issued, int lane, int32_t* status,
                                           bool& drained) {
    const bool ok = __all_sync(0xffffffffu, pa::mbar_wait_bounded(&bars[k % kStages], (k / kStages) & 1, kMaxProbes));
    if (!ok) {
        if (lane == 0) pa::set_status(status, PA_DEV_WAIT_TIMEOUT);
        bool landed = true;
        for (int kk = k; kk < issued; ++kk)
            landed = pa::mbar_wait_bounded(&bars[kk % kStages], (kk / kStages) & 1, kMaxProbes) && landed;
        drained = __all_sync(0xffffffffu, landed);
    }
    return ok;
}

// ============================================================================
// Fixed partitions: one thread block per (sequence, head group, partition)
// ============================================================================
// FP8 stages are half the size and the kernel is bound by instruction latency,
// not bytes: one more resident block per SM.
#ifndef PA_DECODE_MIN_BLOCKS_F8
#define PA_DECODE_MIN_BLOCKS_F8 4
#endif

// Fused append.  prefetch_row loads this lane's share of the new token's K
// and V rows (position ctx - 1), and for FP8 quantises it, early, so that the
// load's latency and the divisions overlap the pipeline; append_row writes them into the stage the warp has just
// received (row r of the tile, over the stale slot contents the copy
// brought) and, when `to_cache`, into the cache at that position's slot
// (block blk, offset off).  bf16: a row is D / 8 16-byte chunks per K or V,
// chunk c in box c / 8 at swizzled chunk c % 8.  FP8: a row is D / 16 chunks
// of 16 codes, quantised exactly as pa_reshape_and_cache_fp8 does; NK heads.
// The stage holds the block's last tile, so no copy refills it after these
// generic-proxy writes (the warp merge that reuses the ring writes through
// the generic proxy too): no proxy fence is needed.
template <int D, bool F8, int NK>
struct AppendLane {
    static constexpr int kCpr = F8 ? D / 16 : D / 8;      // chunks per K (or V) row
    static constexpr int kLanes = 2 * kCpr * NK;          // lanes with a chunk
    int hh, c;
    bool is_v;
    __device__ __forceinline__ explicit AppendLane(int lane) {
        hh = lane / (2 * kCpr);
        const int rem = lane - hh * 2 * kCpr;
        is_v = rem >= kCpr;
        c = is_v ? rem - kCpr : rem;
    }
};

template <int D, bool F8, int NK>
__device__ __forceinline__ void prefetch_row(const DecodeArgs& a, int seq, int kvh, int lane, uint4& x0) {
    using L = AppendLane<D, F8, NK>;
    if (lane >= L::kLanes) return;
    const L l(lane);
    const uint4* src = reinterpret_cast<const uint4*>((l.is_v ? a.v_new : a.k_new) +
                                                      ((size_t)seq * a.n_kv_heads + kvh + l.hh) * D);
    if constexpr (F8) {
        // quantised here, while the warp waits for its first tiles
        const float sc = l.is_v ? a.v_scale : a.k_scale;
        const uint2 qa = pa::quant8(__ldg(src + 2 * l.c), sc), qb = pa::quant8(__ldg(src + 2 * l.c + 1), sc);
        x0 = make_uint4(qa.x, qa.y, qb.x, qb.y);
    } else {
        x0 = __ldg(src + l.c);
    }
}

template <int D, bool F8, int NK>
__device__ __forceinline__ void append_row(uint8_t* stage, int r, const DecodeArgs& a, int kvh, int blk, int off,
                                           bool to_cache, int lane, uint4 x0) {
    using G = Geo<D, F8, NK>;
    using L = AppendLane<D, F8, NK>;
    if (lane < L::kLanes) {
        const L l(lane);
        const uint4 val = x0;                     // bf16 chunk, or 16 E4M3 codes
        uint8_t* row = stage + (l.is_v ? G::kTileBytes : 0) + l.hh * G::kHeadBytes + (F8 ? 0 : (l.c >> 3) * G::kBoxBytes);
        *reinterpret_cast<uint4*>(row + swz(r, F8 ? l.c : (l.c & 7))) = val;
        if (to_cache) {
            const size_t row_elems = (((size_t)blk * a.n_kv_heads + kvh + l.hh) * a.block_size + off) * D;
            reinterpret_cast<uint4*>((l.is_v ? a.v_cache : a.k_cache) + row_elems * (F8 ? 1 : 2))[l.c] = val;
        }
    }
    __syncwarp();
}

// NK = 2 (FP8, G = 4): a block covers two adjacent KV heads (8 query heads);
// its stages are twice as large, so one block fewer fits an SM.
// kClaim: the grid is the resident blocks, and each claims work items
// (sequence, head group, partition) until none is left, so that no block is
// spent on a partition past its sequence's end; otherwise one block per
// (partition, head group, sequence) of the grid, some of them empty.
template <int D, bool F8, int NK = 1, bool kClaim = false>
__global__ void __launch_bounds__(kThreads, F8 ? (NK == 2 ? PA_DECODE_MIN_BLOCKS_F8 - 1 : PA_DECODE_MIN_BLOCKS_F8)
                                               : PA_DECODE_MIN_BLOCKS)
    decode_partition_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                            const DecodeArgs a) {
    static_assert(NK == 1 || F8, "two KV heads per block are built for FP8 caches only");
    using G = Geo<D, F8, NK>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(ring + G::kRingBytes);
    int32_t* table = reinterpret_cast<int32_t*>(bars + kWarps * kStages);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int B = a.block_size;
    const int P = a.partition_size;
    const int table_ints = (P >> a.log2_block) + 2;
    // claimed work: item offsets per sequence, and the claimed item
    int32_t* pre = table + table_ints;                 // [num_seqs + 1]
    int32_t* claimed = pre + kClaimMaxSeqs + 1;

    // Launched as a programmatic dependent: inputs may come from the kernel
    // before this one on the stream, so nothing is read before this wait.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if constexpr (kClaim) {
        // Items, in order: sequence, head group, partition; sequence s holds
        // n_units * max(1, partitions of s) of them (a context of 0 is one
        // item, which writes zeros).  pre[s] = items before sequence s.
        // (Handing out every sequence's whole partitions before the last,
        // shorter ones measured 2 % slower on a ragged batch.)
        const int S = a.num_seqs;
        constexpr int kPer = (kClaimMaxSeqs + kThreads - 1) / kThreads;
        int cnt[kPer];
        int sum = 0;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int s_ = threadIdx.x * kPer + i;
            int c = 0;
            if (s_ < S) {
                int ctx_ = a.context_lens[s_];
                ctx_ = ctx_ < 0 ? 0 : (ctx_ > a.ctx_cap ? a.ctx_cap : ctx_);
                const int np_ = (ctx_ + P - 1) / P;
                c = a.n_units * (np_ > 0 ? np_ : 1);
            }
            cnt[i] = c;
            sum += c;
        }
        // exclusive scan of the threads' sums: within the warp, then across warps
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) claimed[1 + warp] = incl;
        __syncthreads();
        int base = incl - sum;
        for (int w = 0; w < warp; ++w) base += claimed[1 + w];
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int s_ = threadIdx.x * kPer + i;
            if (s_ < S) pre[s_] = base;
            base += cnt[i];
        }
        if (threadIdx.x == kThreads - 1) pre[S] = base;
        if (threadIdx.x == 0) {
            for (int i = 0; i < kWarps * kStages; ++i) pa::mbar_init(&bars[i], 1);
            pa::fence_mbar_init();
        }
        // the merge kernel may begin its launch (it waits for this grid's
        // results before it reads them)
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }
    int kg = 0;                      // this warp's stages consumed by earlier items
    for (;;) {
        int part, seq, yb;
        if constexpr (kClaim) {
            // claimed once the block is free (claiming the next item while this
            // one runs measured 4-9 % slower: the block holds it back while
            // others run out of work)
            __syncthreads();             // pre is complete, the previous item's readers are done
            if (threadIdx.x == 0) claimed[0] = atomicAdd(a.claim, 1);
            __syncthreads();
            const int v = claimed[0];
            if (v >= pre[a.num_seqs]) break;
            int lo = 0, hi = a.num_seqs - 1;              // the sequence s with pre[s] <= v < pre[s + 1]
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (pre[mid] <= v) lo = mid; else hi = mid - 1;
            }
            seq = lo;
            const int np_ = (pre[seq + 1] - pre[seq]) / a.n_units;
            const int r = v - pre[seq];
            yb = r / np_;
            part = r - yb * np_;
        } else {
            part = blockIdx.x;
            seq = blockIdx.z;
            yb = blockIdx.y;
        }
        const int kvh = NK == 1 ? yb / a.n_sub : yb * NK;
        const int hpb = a.heads_per_block;
        const int qh0 = kvh * a.group + (yb % a.n_sub) * hpb;

        // Independent loads first: the context length, a speculative slice of the
        // block table (this partition's entries, read before the length is known)
        // and q; one memory round trip instead of three.
        const int lb0 = (part * P) >> a.log2_block;
        const int32_t* trow = a.block_tables + (size_t)seq * a.max_blocks_per_seq;
        const int n_spec = max(0, min(P >> a.log2_block, a.max_blocks_per_seq - lb0));
        int ctx = a.context_lens[seq];
        for (int i = threadIdx.x; i < n_spec; i += kThreads) table[i] = trow[lb0 + i];
        const size_t row0 = ((size_t)seq * a.n_q_heads + qh0) * D;   // q / out offset of the block's first head
        uint32_t qb[G::kSteps][2];
        uint32_t qbk[NK][G::kSteps][2];      // FP8: q per KV head of the tile (the other head's columns zero)
        float c0 = 0.f, c1 = 0.f;
        if constexpr (F8) {
            const float sh = load_q_f8<D>(qb, a.q + row0, hpb, lane);
            const int h0_ = 2 * (lane & 3);
            const float sc = a.scale_log2 * a.k_scale;
            c0 = sc / __shfl_sync(0xffffffffu, sh, 4 * h0_);
            c1 = sc / __shfl_sync(0xffffffffu, sh, 4 * h0_ + 4);
#pragma unroll
            for (int hh = 0; hh < NK; ++hh) {
                const bool mine = NK == 1 || ((lane >> 2) >> 2) == hh;     // B column g = query head g
#pragma unroll
                for (int k = 0; k < G::kSteps; ++k) {
                    qbk[hh][k][0] = mine ? qb[k][0] : 0u;
                    qbk[hh][k][1] = mine ? qb[k][1] : 0u;
                }
            }
        } else {
            load_q<D>(qb, a.q + row0, hpb, lane);
        }
        if (!kClaim && threadIdx.x == 0) {
            for (int i = 0; i < kWarps * kStages; ++i) pa::mbar_init(&bars[i], 1);
            pa::fence_mbar_init();
        }

        const bool ctx_ok = ctx >= 0 && ctx <= a.ctx_cap;
        if (!ctx_ok) {
            if (threadIdx.x == 0 && part == 0 && yb == 0) pa::set_status(a.status, PA_DEV_BAD_CONTEXT);
            ctx = ctx < 0 ? 0 : a.ctx_cap;
        }
        const int nparts = (ctx + P - 1) / P;
        if (part >= (nparts > 0 ? nparts : 1)) {
            if constexpr (kClaim) continue;               // not handed out (the offsets use the same clamp)
            else return;
        }
        if (ctx == 0) {
            for (int i = threadIdx.x; i < hpb * D; i += kThreads) store_out(a.out, a.out_f32, row0 + i, 0.f);
            if constexpr (kClaim) continue;
            else return;
        }
        const int t_begin = part * P;
        const int t_end = min(t_begin + P, ctx);
        const int n_tiles = (t_end - t_begin + kTile - 1) / kTile;
        // Once every block has started, the merge kernel may be scheduled onto
        // free SM slots; it waits for this grid's results before reading them.
        if constexpr (!kClaim) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        __syncthreads();

        const uint64_t policy = pa::l2_evict_first_policy();
        uint64_t* wbars = bars + warp * kStages;
        uint8_t* wring = ring + warp * kStages * G::kStageBytes;
        auto issue = [&](int tile, int stage) {
            const int t0 = t_begin + tile * kTile;
            const int nv = min(kTile, t_end - t0);
            const int e0 = (t0 >> a.log2_block) - lb0;
            const int blk1 = (B < kTile && nv > B) ? table[e0 + 1] : 0;
            issue_tile<D, F8, NK>(wring + stage * G::kStageBytes, &wbars[stage], &tmap_k, &tmap_v, table[e0], blk1,
                              t0 & (B - 1), nv, kvh, a, policy);
        };

        WarpState<D> st;
        st.reset();
        // this warp's stages carry on from earlier items: its k-th tile here is
        // stage (kg + k) % kStages
        if (lane == 0) {
#pragma unroll
            for (int k = 0; k < kStages; ++k) {
                const int tile = warp + k * kWarps;
                if (tile < n_tiles) issue(tile, (kg + k) % kStages);
            }
        }
        // this warp's tiles; stages issued before consuming local tile k: min(n_mine, k + kStages)
        const int n_mine = warp < n_tiles ? (n_tiles - warp + kWarps - 1) / kWarps : 0;
        bool drained = true;
        int k = 0;
        // the fused append lands in the tile holding position ctx - 1 (the last
        // tile of the last partition); a clamped context appends nothing
        const bool append = a.k_new != nullptr && ctx_ok && t_end == ctx;
        uint4 app = make_uint4(0, 0, 0, 0);
        if (append && warp == (n_tiles - 1) % kWarps) prefetch_row<D, F8, NK>(a, seq, kvh, lane, app);
        for (int tile = warp; tile < n_tiles; tile += kWarps, ++k) {
            if (!wait_stage(wbars, kg + k, kg + min(n_mine, k + kStages), lane, a.status, drained)) break;
            const int stg = (kg + k) % kStages;
            if (append && tile == n_tiles - 1) {
                const int pos = ctx - 1;
                int blk = table[(pos >> a.log2_block) - lb0];
                const bool blk_ok = blk >= 0 && blk < a.num_blocks;     // a bad id was flagged when the tile was issued
                append_row<D, F8, NK>(wring + stg * G::kStageBytes, pos - (t_begin + tile * kTile), a, kvh,
                                      blk_ok ? blk : 0, pos & (B - 1), blk_ok && (NK == 2 || yb % a.n_sub == 0),
                                      lane, app);
            }
            const uint32_t ks = pa::smem_addr(wring + stg * G::kStageBytes);
            const int nv_ = min(kTile, t_end - (t_begin + tile * kTile));
            if constexpr (F8)
                consume_tile_f8<D, NK>(st, ks, ks + G::kTileBytes, nv_, qbk, c0, c1, lane);
            else
                consume_tile<D>(st, ks, ks + G::kTileBytes, nv_, qb, a.scale_log2, lane);
            __syncwarp();
            if (lane == 0 && tile + kWarps * kStages < n_tiles) issue(tile + kWarps * kStages, stg);
        }
        kg += n_mine;
        st.finish_sums();

        // ---- merge the 4 warps (exact, as in the block merge) ----------------------
        // Ring no longer in use, unless a timed-out copy may still land in it: then
        // the block leaves it alone and stops (outputs unspecified, status set).
        if (!__syncthreads_and(drained ? 1 : 0)) {
            break;
        }
        float* mw = reinterpret_cast<float*>(ring);        // [warp][8]
        float* lw = mw + kWarps * kHeads;                  // [warp][8]
        float* uw = lw + kWarps * kHeads;                  // [warp][8][D]
        const int g = lane >> 2, h0 = 2 * (lane & 3);
        if (g == 0) {
            mw[warp * kHeads + h0] = st.m0;
            mw[warp * kHeads + h0 + 1] = st.m1;
            lw[warp * kHeads + h0] = st.l0;
            lw[warp * kHeads + h0 + 1] = st.l1;
        }
        // rows g and g + 8 of m-tile m are d = 16 m + g and 16 m + g + 8 (FP8:
        // 16 m + 2 g and 16 m + 2 g + 1)
        constexpr int kRow2 = F8 ? 1 : 8;
#pragma unroll
        for (int m = 0; m < G::kSteps; ++m) {
            const int drow = F8 ? 16 * m + 2 * g : 16 * m + g;
            float* u0 = uw + (warp * kHeads + h0) * D + drow;
            float* u1 = u0 + D;
            u0[0] = st.acc[m][0];
            u1[0] = st.acc[m][1];
            u0[kRow2] = st.acc[m][2];
            u1[kRow2] = st.acc[m][3];
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < hpb * D; idx += kThreads) {
            const int h = idx / D;
            const int d = idx % D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mw[w * kHeads + h]);
            float Z = 0.f, U = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float f = fast_exp2(mw[w * kHeads + h] - M);
                Z += f * lw[w * kHeads + h];
                U += f * uw[(w * kHeads + h) * D + d];
            }
            if (nparts == 1) {
                store_out(a.out, a.out_f32, row0 + idx, U * a.u_scale / Z);
            } else {
                const size_t pi = ((size_t)seq * a.n_q_heads + qh0 + h) * a.max_parts + part;
                a.part_acc[pi * D + d] = U * a.u_scale;
                if (d == 0) {
                    a.part_max[pi] = M * kLn2;      // back to natural-log units
                    a.part_sum[pi] = Z;
                }
            }
        }
        if constexpr (!kClaim) break;
        // the next item's copies write the ring, which this one's merge (and
        // append) wrote through the generic proxy
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if constexpr (kClaim) {
        // Every block has made its last claim once all have counted themselves
        // done: the last one leaves both counters at zero for the next call.
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            if (atomicAdd(a.claim + 1, 1) == (int)gridDim.x - 1) {
                atomicExch(a.claim, 0);
                atomicExch(a.claim + 1, 0);
            }
        }
    }
}

// Fold partitions [0, np) of one (sequence, head) row into (M, Z, U) for
// dimension d: kChunk partitions' statistics and values are loaded at once
// (independent loads, one memory round trip per chunk), then merged into the
// running values with the same rule.
template <int kChunk>
__device__ __forceinline__ float merge_row(const float* __restrict__ pmax, const float* __restrict__ psum,
                                           const float* __restrict__ pacc, size_t base, int np, int d_head, int d) {
    float M = -INFINITY, Z = 0.f, U = 0.f;
    for (int c0 = 0; c0 < np; c0 += kChunk) {
        float m[kChunk], z[kChunk], u[kChunk];
#pragma unroll
        for (int r = 0; r < kChunk; ++r) {
            const int p = c0 + r;
            const bool ok = p < np;
            m[r] = ok ? pmax[base + p] : -INFINITY;
            z[r] = ok ? psum[base + p] : 0.f;
            u[r] = ok ? pacc[(base + p) * d_head + d] : 0.f;
        }
        float mc = M;
#pragma unroll
        for (int r = 0; r < kChunk; ++r) mc = fmaxf(mc, m[r]);
        const float sc = fast_exp2((M - mc) * kLog2e);   // 0 on the first chunk (M = -inf)
        Z *= sc;
        U *= sc;
#pragma unroll
        for (int r = 0; r < kChunk; ++r) {
            const float w = fast_exp2((m[r] - mc) * kLog2e);
            Z += w * z[r];
            U += w * u[r];
        }
        M = mc;
    }
    return U / Z;
}

// Exact merge of partition statistics (second page, section 11):
// M = max m_p, Z = sum exp(m_p - M) z_p, U = sum exp(m_p - M) u_p, out = U / Z.
// One thread block per (query head, sequence), one thread per dimension,
// kChunk partitions loaded per memory round trip (4 when no sequence can have
// more than 4 partitions, else 8: wider chunks cost registers that the many
// short rows of a ragged batch do not repay).  When launched as a
// programmatic dependent of the partition kernel, it waits for that grid's
// results before reading them.
template <int kChunk>
__global__ void lse_merge_kernel(void* out, int out_f32, const float* __restrict__ pmax,
                                 const float* __restrict__ psum, const float* __restrict__ pacc,
                                 const int32_t* __restrict__ context_lens, int ctx_cap, int partition_size,
                                 int max_parts, int n_q_heads, int d_head, int skip_single) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int h = blockIdx.x;
    const int seq = blockIdx.y;
    const int d = threadIdx.x;
    int ctx = context_lens[seq];
    ctx = ctx < 0 ? 0 : (ctx > ctx_cap ? ctx_cap : ctx);
    int np = (int)(((long long)ctx + partition_size - 1) / partition_size);
    np = np > max_parts ? max_parts : np;
    if (skip_single && np <= 1) return;             // finished by the partition kernel
    if (d >= d_head) return;
    const size_t orow = ((size_t)seq * n_q_heads + h) * d_head;
    if (np == 0) {
        store_out(out, out_f32, orow + d, 0.f);
        return;
    }
    const size_t base = ((size_t)seq * n_q_heads + h) * max_parts;
    store_out(out, out_f32, orow + d, merge_row<kChunk>(pmax, psum, pacc, base, np, d_head, d));
}

// Launch lse_merge_kernel; as a programmatic dependent launch (its grid may
// be set up while the previous kernel on the stream drains) when pdl is set.
int launch_merge(bool pdl, cudaStream_t st, void* out, int out_f32, const float* pm, const float* ps, const float* pa,
                 const int32_t* ctx, int ctx_cap, int P, int max_parts, int n_q_heads, int num_seqs, int d_head,
                 int skip_single) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n_q_heads, num_seqs);
    cfg.blockDim = dim3((d_head + 31) / 32 * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    auto kernel = max_parts <= 4 ? lse_merge_kernel<4> : lse_merge_kernel<8>;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, out, out_f32, pm, ps, pa, ctx, ctx_cap, P, max_parts,
                                             n_q_heads, d_head, skip_single);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

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

// 2-D view of a cache [num_blocks * n_kv_heads * B rows][d_head] bf16 with
// boxes of 64 columns x box_rows rows and 128-byte swizzle.
bool make_cache_map(CUtensorMap* map, const void* base, long long rows, int d_head, int box_rows) {
    auto enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)d_head, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)d_head * 2};
    const cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1u, 1u};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same view of an FP8 cache [rows][d_head] bytes (d_head 128): boxes of
// 128 columns x box_rows rows, 128-byte swizzle.
bool make_cache_map_f8(CUtensorMap* map, const void* base, long long rows, int d_head, int box_rows) {
    auto enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)d_head, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)d_head};
    const cuuint32_t box[2] = {128u, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1u, 1u};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev < 64 && cached[dev]) return cached[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev < 64) cached[dev] = n;
    return n;
}



size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int ilog2(int x) {
    int r = 0;
    while ((1 << r) < x) ++r;
    return r;
}


// Positions per partition when the caller passes 0.  `units` is the number of
// (sequence, head group) thread blocks per partition index (0: unknown).
// When the units alone fill two waves of resident blocks, sequences are not
// split for parallelism.  If the longest context then spans at least four
// partitions of 1024 positions, the resident blocks claim the items that
// exist (see run()), so no block is spent on an empty partition and smaller
// partitions balance the blocks' loads better: 1024 (on 256 mixed-length
// sequences, 32 layers: FP8 1024 / 768 / 1536 / 2048 positions 3.19 / 3.21 /
// 3.25 / 3.40 ms per step, bf16 5.24 / 5.23 / 5.32 / 5.47 ms).  Otherwise
// 1536, so that most short sequences of a large batch finish in their own
// block without a merge and the one-block-per-partition grid holds few empty
// blocks (4-5 % faster than 1024 on that batch before its blocks claimed
// work).  Otherwise at least
// 256 and at most 1024: enough thread blocks for about two waves of 3 blocks
// per SM (counting 4 query heads per block); for the FP8 kernel that covers
// two KV heads per block (8 query heads, 3 blocks per SM), about three waves,
// which measured best on the 64-sequence batch and on 32K contexts (768
// positions there).
int default_partition(int num_seqs, int n_q_heads, int max_context_len, bool f8_pair = false,
                      long long units = 0) {
    const long long slots = (long long)(f8_pair ? PA_DECODE_MIN_BLOCKS_F8 - 1 : PA_DECODE_MIN_BLOCKS) * sm_count();
    if (units > 0 && slots > 0 && units >= 2 * slots) return max_context_len >= 4 * 1024 ? 1024 : 1536;
    const long long work = (long long)num_seqs * n_q_heads * max_context_len;
    const long long target = f8_pair ? 8LL * 3 * (PA_DECODE_MIN_BLOCKS_F8 - 1) * sm_count()
                                     : 4LL * 2 * PA_DECODE_MIN_BLOCKS * sm_count();
    long long p = target > 0 ? (work + target - 1) / target : 1024;
    p = (p + 63) / 64 * 64;
    p = p < 256 ? 256 : (p > 1024 ? 1024 : p);
    // FP8 pairs: a last wave of blocks that is nearly empty (at most a
    // quarter of the resident slots, from the block count that contexts of
    // max_context_len would give) costs a whole wave's time for a sliver of
    // work, so take the next partition sizes until it is not (8 x 32K
    // contexts: 768 -> 832 positions, 3.02 -> 2.81 waves)
    if (f8_pair && units > 0 && slots > 0) {
        for (int step = 0; step < 8 && p < 1024; ++step) {
            const long long blocks = units * ((max_context_len + p - 1) / p);
            const long long rem = blocks % slots;
            if (rem == 0 || 4 * rem >= slots) break;
            p += 64;
        }
    }
    return (int)p;
}

// Workspace layout for max_parts partitions: a 256-byte header whose first
// two int32 are the claim counters (zero between calls), then part_max and
// part_sum [S][Hq][max_parts] f32, then part_acc [S][Hq][max_parts][D] f32;
// every section 256-byte aligned.
constexpr size_t kWsHeader = 256;
size_t workspace_bytes_for(int num_seqs, int n_q_heads, int d_head, int max_parts) {
    if (max_parts <= 1) return 0;
    const size_t n = (size_t)num_seqs * n_q_heads * max_parts;
    return kWsHeader + 2 * align256(4 * n) + align256(4 * n * d_head);
}

template <typename K>
int launch(K kernel, dim3 grid, int smem, cudaStream_t st, const CUtensorMap& mk, const CUtensorMap& mv,
           const DecodeArgs& a, int* attr_done) {
    if (pa_host::ensure_smem_attr(kernel, smem, attr_done) != cudaSuccess) return PA_ERR_CUDA;
    return pa_host::launch_dependent(kernel, grid, dim3(kThreads), smem, st, mk, mv, a) == cudaSuccess ? PA_OK
                                                                                                      : PA_ERR_CUDA;
}

int run(DecodeArgs a, const CUtensorMap& mk, const CUtensorMap& mv, int d_head, void* workspace,
        size_t workspace_bytes, cudaStream_t st, bool f8 = false, bool pair = false) {
    static int attr128[64] = {0}, attr64[64] = {0}, attr128f8[64] = {0}, attr128f8p[64] = {0};
    static int attr128c[64] = {0}, attr64c[64] = {0}, attr128f8c[64] = {0}, attr128f8pc[64] = {0};
    const int P = a.partition_size;
    a.max_parts = (a.ctx_cap + P - 1) / P;
    if (a.max_parts < 1) a.max_parts = 1;
    if (a.max_parts > 1) {
        if (!workspace || workspace_bytes < workspace_bytes_for(a.num_seqs, a.n_q_heads, d_head, a.max_parts))
            return PA_ERR_WORKSPACE;
        const size_t n = (size_t)a.num_seqs * a.n_q_heads * a.max_parts;
        uint8_t* w = static_cast<uint8_t*>(workspace);
        a.claim = reinterpret_cast<int*>(w);
        w += kWsHeader;
        a.part_max = reinterpret_cast<float*>(w);
        a.part_sum = reinterpret_cast<float*>(w + align256(4 * n));
        a.part_acc = reinterpret_cast<float*>(w + 2 * align256(4 * n));
    }
    const int table_ints = P / a.block_size + 2;
    const int ring = f8 ? (pair ? Geo<128, true, 2>::kRingBytes : Geo<128, true>::kRingBytes)
                        : kWarps * kStages * 2 * kTile * d_head * 2;
    const int merge = kWarps * kHeads * (2 + d_head) * 4;          // the warp merge reuses the ring
    const int smem = 1024 + (ring > merge ? ring : merge) + kWarps * kStages * 8 + table_ints * 4;
    dim3 grid(a.max_parts, a.n_units, a.num_seqs);
    // Many head groups (at least two waves of resident blocks without any
    // split) and contexts of up to four or more partitions: the grid above
    // would hold a block for every partition up to the longest context in
    // every head group, most of them empty when the lengths are ragged, and
    // an empty block still costs a memory round trip.  Instead the resident
    // blocks claim the (sequence, head group, partition) items that exist.
    // (With two or three partitions at most there is little to save: claims
    // cost 6.6 % on 128 sequences of about 2,000 positions, two partitions
    // each and no empty block.)
    const int per_sm = f8 ? (pair ? PA_DECODE_MIN_BLOCKS_F8 - 1 : PA_DECODE_MIN_BLOCKS_F8) : PA_DECODE_MIN_BLOCKS;
    const long long slots = (long long)per_sm * sm_count();
    const long long units = (long long)a.num_seqs * a.n_units;
    // (items and claims are counted in int32)
    const bool claim = a.max_parts >= 4 && a.num_seqs <= kClaimMaxSeqs && units >= 2 * slots &&
                       units * a.max_parts + slots < 0x40000000LL;
    int rc;
    if (claim) {
        const int smem_c = smem + (kClaimMaxSeqs + 2 + kWarps) * 4;
        const long long items = units * a.max_parts;
        const dim3 grid_c((unsigned)(items < slots ? items : slots));
        rc = f8 ? (pair ? launch(decode_partition_kernel<128, true, 2, true>, grid_c, smem_c, st, mk, mv, a, attr128f8pc)
                        : launch(decode_partition_kernel<128, true, 1, true>, grid_c, smem_c, st, mk, mv, a, attr128f8c))
                : d_head == 128 ? launch(decode_partition_kernel<128, false, 1, true>, grid_c, smem_c, st, mk, mv, a, attr128c)
                                : launch(decode_partition_kernel<64, false, 1, true>, grid_c, smem_c, st, mk, mv, a, attr64c);
    } else {
        rc = f8 ? (pair ? launch(decode_partition_kernel<128, true, 2>, grid, smem, st, mk, mv, a, attr128f8p)
                        : launch(decode_partition_kernel<128, true>, grid, smem, st, mk, mv, a, attr128f8))
                : d_head == 128 ? launch(decode_partition_kernel<128, false>, grid, smem, st, mk, mv, a, attr128)
                                : launch(decode_partition_kernel<64, false>, grid, smem, st, mk, mv, a, attr64);
    }
    if (rc != PA_OK || a.max_parts <= 1) return rc;
    return launch_merge(true, st, a.out, a.out_f32, a.part_max, a.part_sum, a.part_acc, a.context_lens, a.ctx_cap, P,
                        a.max_parts, a.n_q_heads, a.num_seqs, d_head, 1);
}

}  // namespace

extern "C" {

size_t pa_decode_workspace_size(int num_seqs, int n_q_heads, int d_head, int max_context_len,
                                int partition_size) {
    if (num_seqs <= 0 || n_q_heads <= 0 || d_head <= 0 || max_context_len < 0 || partition_size < 0) return 0;
    // the library's own choice may differ between pa_decode and pa_decode_fp8
    // and may be larger when the batch has many head groups: size for the
    // smaller work-based partition (more of them), which serves every case
    int P = partition_size;
    if (P == 0) {
        const int p1 = default_partition(num_seqs, n_q_heads, max_context_len);
        const int p2 = default_partition(num_seqs, n_q_heads, max_context_len, true);
        P = p1 < p2 ? p1 : p2;
    }
    return workspace_bytes_for(num_seqs, n_q_heads, d_head, (max_context_len + P - 1) / P);
}

}  // extern "C"

namespace {

// pa_decode and pa_decode_fp8 (f8: E4M3 caches with scales k_scale, v_scale).
int decode_impl(void* out, int out_dtype, const void* q, const void* k_cache, const void* v_cache,
                const int32_t* block_tables, const int32_t* context_lens, int block_size, float scale,
                int n_q_heads, int n_kv_heads, int d_head, int num_seqs, int max_blocks_per_seq, int num_blocks,
                int max_context_len, int partition_size, void* workspace, size_t workspace_bytes,
                int32_t* status_dev, void* stream, bool f8, float k_scale, float v_scale,
                const void* k_new = nullptr, const void* v_new = nullptr) {
    if (num_seqs < 0 || n_q_heads <= 0 || n_kv_heads <= 0 || max_blocks_per_seq <= 0 ||
        num_blocks <= 0 || max_context_len < 0 || !(scale == scale))
        return PA_ERR_INVALID_ARG;
    if (f8 && (!(k_scale > 0.f) || !(v_scale > 0.f) || !(k_scale < INFINITY) || !(v_scale < INFINITY)))
        return PA_ERR_INVALID_ARG;
    if (f8 && d_head != 128) return PA_ERR_UNSUPPORTED;
    if (out_dtype != PA_DTYPE_BF16 && out_dtype != PA_DTYPE_F32) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return PA_ERR_INVALID_ARG;
    if ((k_new == nullptr) != (v_new == nullptr)) return PA_ERR_INVALID_ARG;
    if (k_new && (!pa_host::aligned16(k_new) || !pa_host::aligned16(v_new))) return PA_ERR_MISALIGNED;
    if (!pa_host::supported_block_size(block_size) || !pa_host::supported_d_head(d_head))
        return PA_ERR_UNSUPPORTED;
    if (n_q_heads % n_kv_heads) return PA_ERR_UNSUPPORTED;
    const int group = n_q_heads / n_kv_heads;
    if (group != 1 && group != 2 && group != 4 && group != 8 && group != 16) return PA_ERR_UNSUPPORTED;
    if (!pa_host::aligned16(out) || !pa_host::aligned16(q) || !pa_host::aligned16(k_cache) ||
        !pa_host::aligned16(v_cache))
        return PA_ERR_MISALIGNED;
    if (partition_size < 0 || (partition_size > 0 && (partition_size % 64 || partition_size > kMaxPartition)))
        return PA_ERR_INVALID_ARG;
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return PA_ERR_WORKSPACE;
    // FP8 with G = 4: each block covers two adjacent KV heads (their 8 query
    // heads fill the products' 8 columns)
    const bool pair = f8 && group == 4 && n_kv_heads % 2 == 0;
    const int hpb = pair ? kHeads : (group < kHeads ? group : kHeads);
    const int n_sub = pair ? 1 : group / hpb;
    if ((long long)n_kv_heads * n_sub > 65535 || num_seqs > 65535) return PA_ERR_UNSUPPORTED;
    const long long cache_rows = (long long)num_blocks * n_kv_heads * block_size;
    if (cache_rows > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;

    DecodeArgs a{};
    a.out = out;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.status = status_dev;
    a.scale_log2 = scale * kLog2e;
    a.out_f32 = out_dtype == PA_DTYPE_F32;
    a.block_size = block_size;
    a.log2_block = ilog2(block_size);
    a.n_q_heads = n_q_heads;
    a.n_kv_heads = n_kv_heads;
    a.group = group;
    a.heads_per_block = hpb;
    a.n_sub = n_sub;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    const long long cap_tbl = (long long)max_blocks_per_seq * block_size;
    a.ctx_cap = (int)(cap_tbl < max_context_len ? cap_tbl : max_context_len);
    a.num_seqs = num_seqs;
    a.n_units = pair ? n_kv_heads / 2 : n_kv_heads * n_sub;
    const long long units = (long long)num_seqs * a.n_units;
    a.partition_size = partition_size > 0 ? partition_size
                                          : default_partition(num_seqs, n_q_heads, max_context_len, pair, units);
    a.k_scale = f8 ? k_scale : 1.f;
    a.u_scale = f8 ? v_scale / 32768.f : 1.f;
    a.v_scale = f8 ? v_scale : 1.f;
    a.k_new = static_cast<const __nv_bfloat16*>(k_new);
    a.v_new = static_cast<const __nv_bfloat16*>(v_new);
    a.k_cache = static_cast<uint8_t*>(const_cast<void*>(k_cache));
    a.v_cache = static_cast<uint8_t*>(const_cast<void*>(v_cache));

    const int box_rows = block_size < kTile ? block_size : kTile;
    CUtensorMap mk, mv;
    const bool maps_ok = f8 ? make_cache_map_f8(&mk, k_cache, cache_rows, d_head, box_rows) &&
                                  make_cache_map_f8(&mv, v_cache, cache_rows, d_head, box_rows)
                            : make_cache_map(&mk, k_cache, cache_rows, d_head, box_rows) &&
                                  make_cache_map(&mv, v_cache, cache_rows, d_head, box_rows);
    if (!maps_ok) return PA_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return run(a, mk, mv, d_head, workspace, workspace_bytes, st, f8, pair);
}

}  // namespace

extern "C" {

int pa_decode(void* out, int out_dtype, const void* q, const void* k_cache, const void* v_cache,
              const int32_t* block_tables, const int32_t* context_lens, int block_size, float scale,
              int n_q_heads, int n_kv_heads, int d_head, int num_seqs, int max_blocks_per_seq,
              int num_blocks, int max_context_len, int partition_size, void* workspace,
              size_t workspace_bytes, int32_t* status_dev, void* stream) {
    return decode_impl(out, out_dtype, q, k_cache, v_cache, block_tables, context_lens, block_size, scale, n_q_heads,
                       n_kv_heads, d_head, num_seqs, max_blocks_per_seq, num_blocks, max_context_len, partition_size,
                       workspace, workspace_bytes, status_dev, stream, false, 1.f, 1.f);
}

int pa_decode_fp8(void* out, int out_dtype, const void* q, const void* k_cache, const void* v_cache,
                  const int32_t* block_tables, const int32_t* context_lens, int block_size, float scale,
                  float k_scale, float v_scale, int n_q_heads, int n_kv_heads, int d_head, int num_seqs,
                  int max_blocks_per_seq, int num_blocks, int max_context_len, int partition_size, void* workspace,
                  size_t workspace_bytes, int32_t* status_dev, void* stream) {
    return decode_impl(out, out_dtype, q, k_cache, v_cache, block_tables, context_lens, block_size, scale, n_q_heads,
                       n_kv_heads, d_head, num_seqs, max_blocks_per_seq, num_blocks, max_context_len, partition_size,
                       workspace, workspace_bytes, status_dev, stream, true, k_scale, v_scale);
}

int pa_decode_append(void* out, int out_dtype, const void* q, void* k_cache, void* v_cache, const void* k_new,
                     const void* v_new, const int32_t* block_tables, const int32_t* context_lens, int block_size,
                     float scale, int n_q_heads, int n_kv_heads, int d_head, int num_seqs, int max_blocks_per_seq,
                     int num_blocks, int max_context_len, int partition_size, void* workspace, size_t workspace_bytes,
                     int32_t* status_dev, void* stream) {
    if (!k_new || !v_new) return PA_ERR_INVALID_ARG;
    return decode_impl(out, out_dtype, q, k_cache, v_cache, block_tables, context_lens, block_size, scale, n_q_heads,
                       n_kv_heads, d_head, num_seqs, max_blocks_per_seq, num_blocks, max_context_len, partition_size,
                       workspace, workspace_bytes, status_dev, stream, false, 1.f, 1.f, k_new, v_new);
}

int pa_decode_append_fp8(void* out, int out_dtype, const void* q, void* k_cache, void* v_cache, const void* k_new,
                         const void* v_new, const int32_t* block_tables, const int32_t* context_lens, int block_size,
                         float scale, float k_scale, float v_scale, int n_q_heads, int n_kv_heads, int d_head,
                         int num_seqs, int max_blocks_per_seq, int num_blocks, int max_context_len,
                         int partition_size, void* workspace, size_t workspace_bytes, int32_t* status_dev,
                         void* stream) {
    if (!k_new || !v_new) return PA_ERR_INVALID_ARG;
    return decode_impl(out, out_dtype, q, k_cache, v_cache, block_tables, context_lens, block_size, scale, n_q_heads,
                       n_kv_heads, d_head, num_seqs, max_blocks_per_seq, num_blocks, max_context_len, partition_size,
                       workspace, workspace_bytes, status_dev, stream, true, k_scale, v_scale, k_new, v_new);
}

int pa_lse_merge(void* out, int out_dtype, const float* part_max, const float* part_sum, const float* part_acc,
                 const int32_t* context_lens, int partition_size, int max_parts, int num_seqs, int n_q_heads,
                 int d_head, void* stream) {
    if (num_seqs < 0 || n_q_heads <= 0 || d_head <= 0 || max_parts <= 0 || partition_size <= 0)
        return PA_ERR_INVALID_ARG;
    if (out_dtype != PA_DTYPE_BF16 && out_dtype != PA_DTYPE_F32) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (!out || !part_max || !part_sum || !part_acc || !context_lens) return PA_ERR_INVALID_ARG;
    if (d_head > 1024 || num_seqs > 65535) return PA_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(out) & 3u) || (reinterpret_cast<uintptr_t>(part_max) & 3u) ||
        (reinterpret_cast<uintptr_t>(part_sum) & 3u) || (reinterpret_cast<uintptr_t>(part_acc) & 3u))
        return PA_ERR_MISALIGNED;
    return launch_merge(false, static_cast<cudaStream_t>(stream), out, out_dtype == PA_DTYPE_F32, part_max, part_sum,
                        part_acc, context_lens, 0x7fffffff, partition_size, max_parts, n_q_heads, num_seqs, d_head, 0);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// pa_decode for callers that cannot provide device scratch memory.
//
// The split path's partition statistics live in this file-scope device
// array instead of a caller workspace.  Host code must not use the name
// `g_static_scratch` as an address (on the host it is only a stand-in
// symbol); the device address is looked up with cudaGetSymbolAddress, with
// the device current, once per CUDA context and cached.  The cache is keyed
// by the context's unique id, so a context created anew on the same device
// (after cudaDeviceReset, for instance), whose copy of the array may sit
// elsewhere, gets a fresh lookup instead of a stale address.
// ---------------------------------------------------------------------------
#include <cudaTypedefs.h>

#include <mutex>

static __device__ __align__(256) uint8_t g_static_scratch[PA_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxScratchDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxScratchDevices] = {nullptr};
unsigned long long g_scratch_ctx[kMaxScratchDevices] = {0};

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_ctx_fn_once;

// Unique id of the calling thread's current context (0 if unknown).
unsigned long long current_context_id() {
    std::call_once(g_ctx_fn_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!g_ctx_current || !g_ctx_id || g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx ||
        g_ctx_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of g_static_scratch in the current device's context (looked
// up on the first call in that context).  Returns nullptr on failure.
void* static_scratch_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices) return nullptr;
    const unsigned long long ctx = current_context_id();   // 0 before the runtime has made one current
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev] || ctx == 0 || g_scratch_ctx[dev] != ctx) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr) return nullptr;
        g_scratch_addr[dev] = ptr;
        g_scratch_ctx[dev] = ctx ? ctx : current_context_id();
    }
    return g_scratch_addr[dev];
}

}  // namespace

extern "C" int pa_decode_static_scratch(void* out, int out_dtype, const void* q, const void* k_cache,
                                        const void* v_cache, const int32_t* block_tables,
                                        const int32_t* context_lens, int block_size, float scale, int n_q_heads,
                                        int n_kv_heads, int d_head, int num_seqs, int max_blocks_per_seq,
                                        int num_blocks, int max_context_len, int partition_size,
                                        int32_t* status_dev, void* stream) {
    const size_t need = pa_decode_workspace_size(num_seqs, n_q_heads, d_head, max_context_len, partition_size);
    if (need > PA_STATIC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (need > 0) {
        scratch = static_scratch_address();
        if (!scratch) return PA_ERR_CUDA;
    }
    return pa_decode(out, out_dtype, q, k_cache, v_cache, block_tables, context_lens, block_size, scale, n_q_heads,
                     n_kv_heads, d_head, num_seqs, max_blocks_per_seq, num_blocks, max_context_len, partition_size,
                     scratch, need, status_dev, stream);
}
