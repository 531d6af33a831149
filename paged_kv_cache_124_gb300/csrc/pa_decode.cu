// Paged single-query (decode) attention for sm_103a.
//
// What is computed ("PagedAttention: Virtual Memory for the KV Cache",
// sections 1, 7 and 13; "PagedAttention in vLLM: scattered memory, exact
// attention", sections 10 and 11): for each sequence and query head,
// softmax(scale * q . K^T) . V over the sequence's cached positions, where
// position j lives in physical block block_table[j / B] at offset j % B.
//
// How (GB300 design):
//  * One thread block (4 warps) per (sequence, KV head [, head sub-group],
//    partition of partition_size positions).  All query heads of the GQA
//    group (up to 4 per block) are computed from the same K/V bytes, so the
//    cache is read once per KV head.
//  * Each warp owns a ring of kStages shared-memory stages.  A stage holds
//    16 positions of K and of V (16 x d_head bf16 each), brought in by 1-D
//    bulk async copies (cp.async.bulk, the TMA engine's untiled form) of the
//    contiguous rows of the physical block(s) the block table points to,
//    counted on an mbarrier.  The ring keeps several copies in flight per
//    warp while the warp computes on an earlier stage.
//  * Scores: 8 lanes per position, 4 positions per pass, fp32 products with
//    packed (f32x2) FMAs, reduce-scatter over the 8 lanes with shuffles.
//    Softmax: online, fp32, running maximum per head in the log2 domain,
//    lane-local running sums merged once at the end.
//  * Weighted values: d_head/8 lanes per position row, each lane owns 8
//    dimensions for every head of the group; rows are merged once at the end.
//  * The 4 warps' states are merged exactly in shared memory.  A sequence
//    that fits one partition is normalised and written directly; otherwise
//    (m, z, u) go to the workspace and lse_merge_kernel finishes them
//    ("secondary reduction", section 13 of the first page; statistics of
//    section 11 of the second).

#include <math.h>

#include "pa_common.cuh"

namespace {

constexpr int kTile = 16;          // positions per stage
constexpr int kWarps = 4;          // warps per thread block
constexpr int kStages = 3;         // stages per warp ring
constexpr int kThreads = kWarps * 32;
constexpr int kMaxProbes = 2000000;   // ~2 s bound on any single wait
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kMaxPartition = 8192;

struct DecodeArgs {
    void* out;
    const __nv_bfloat16* q;
    const __nv_bfloat16* k_cache;
    const __nv_bfloat16* v_cache;
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
    int n_sub;               // G / (heads per thread block)
    int max_blocks_per_seq;
    int num_blocks;
    int ctx_cap;             // min(max_blocks_per_seq * B, max_context_len)
    int partition_size;
    int max_parts;
};

template <int D>
struct Geo {
    static constexpr int kRowBytes = D * 2;
    static constexpr int kTileBytes = kTile * kRowBytes;           // K or V
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kRingBytes = kWarps * kStages * kStageBytes;
    static constexpr int kQkChunks = D / 64;      // 16-B chunks per lane per row
    static constexpr int kPvLanes = D / 8;        // lanes per value row
    static constexpr int kPvRows = 32 / kPvLanes; // rows per pass
    static constexpr int kPvPasses = kTile / kPvRows;
};

template <int GP>
struct Own {                                      // scores a lane keeps
    static constexpr int kN = GP >= 2 ? GP / 2 : 1;
};

__device__ __forceinline__ void store_out(void* out, int f32, size_t i, float v) {
    if (f32)
        static_cast<float*>(out)[i] = v;
    else
        static_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(v);
}

__device__ __forceinline__ void unpack8(const uint4& w, float2 (&f)[4]) {
    f[0] = pa::bf16x2_to_float2(w.x);
    f[1] = pa::bf16x2_to_float2(w.y);
    f[2] = pa::bf16x2_to_float2(w.z);
    f[3] = pa::bf16x2_to_float2(w.w);
}

// Sum `v` (N values per lane) over the 8 lanes that share lane >> 3, leaving
// each lane with N/8 of the sums (at least one).  Value index after the call
// for lane bits b2 b1 b0 (of lane & 7): see owned_pass / owned_head.
template <int N>
__device__ __forceinline__ void reduce_scatter8(float (&v)[N], int lane) {
    constexpr int H1 = N / 2 > 0 ? N / 2 : 1;
    constexpr int H2 = H1 / 2 > 0 ? H1 / 2 : 1;
    constexpr int H3 = H2 / 2 > 0 ? H2 / 2 : 1;
    // step xor 4
    if (N >= 2) {
        const bool hi = lane & 4;
#pragma unroll
        for (int k = 0; k < H1; ++k) {
            float send = hi ? v[k] : v[k + H1];
            float keep = hi ? v[k + H1] : v[k];
            v[k] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
        }
    } else {
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], 4);
    }
    // step xor 2
    if (H1 >= 2) {
        const bool hi = lane & 2;
#pragma unroll
        for (int k = 0; k < H2; ++k) {
            float send = hi ? v[k] : v[k + H2];
            float keep = hi ? v[k + H2] : v[k];
            v[k] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
        }
    } else {
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], 2);
    }
    // step xor 1
    if (H2 >= 2) {
        const bool hi = lane & 1;
#pragma unroll
        for (int k = 0; k < H3; ++k) {
            float send = hi ? v[k] : v[k + H3];
            float keep = hi ? v[k + H3] : v[k];
            v[k] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
        }
    } else {
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
    }
}

template <int D, int GP>
__global__ void __launch_bounds__(kThreads, 2) decode_partition_kernel(const DecodeArgs a) {
    using G = Geo<D>;
    constexpr int NO = Own<GP>::kN;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* ring = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + G::kRingBytes);
    float* probs = reinterpret_cast<float*>(bars + kWarps * kStages);    // [warp][pos][GP]
    int32_t* table = reinterpret_cast<int32_t*>(probs + kWarps * kTile * GP);

    const int part = blockIdx.x;
    const int seq = blockIdx.z;
    const int kvh = blockIdx.y / a.n_sub;
    const int qh0 = kvh * a.group + (blockIdx.y % a.n_sub) * GP;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    int ctx = a.context_lens[seq];
    if (ctx < 0 || ctx > a.ctx_cap) {
        if (threadIdx.x == 0 && part == 0 && blockIdx.y == 0) pa::set_status(a.status, PA_DEV_BAD_CONTEXT);
        ctx = ctx < 0 ? 0 : a.ctx_cap;
    }
    const int P = a.partition_size;
    const int nparts = (ctx + P - 1) / P;
    if (part >= (nparts > 0 ? nparts : 1)) return;
    const size_t row0 = ((size_t)seq * a.n_q_heads + qh0) * D;   // q / out offset
    if (ctx == 0) {
        for (int i = threadIdx.x; i < GP * D; i += kThreads) store_out(a.out, a.out_f32, row0 + i, 0.f);
        return;
    }

    const int B = a.block_size;
    const int t_begin = part * P;
    const int t_end = min(t_begin + P, ctx);
    const int n_tiles = (t_end - t_begin + kTile - 1) / kTile;
    const int lb0 = t_begin >> a.log2_block;
    const int n_lb = ((t_end - 1) >> a.log2_block) - lb0 + 1;
    const int32_t* trow = a.block_tables + (size_t)seq * a.max_blocks_per_seq;
    for (int i = threadIdx.x; i < n_lb; i += kThreads) {
        int b = trow[lb0 + i];
        if (b < 0 || b >= a.num_blocks) {
            pa::set_status(a.status, PA_DEV_BAD_BLOCK_ID);
            b = 0;
        }
        table[i] = b;
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < kWarps * kStages; ++i) pa::mbar_init(&bars[i], 1);
        pa::fence_mbar_init();
    }

    // q of the group's heads, fp32, pre-scaled into the log2 domain; lane
    // keeps the 8 (or 16) dimensions it multiplies in the score pass.
    const int j8 = lane & 7;
    float2 qf[GP][G::kQkChunks * 4];
#pragma unroll
    for (int h = 0; h < GP; ++h) {
        const uint4* qrow = reinterpret_cast<const uint4*>(a.q + row0 + (size_t)h * D);
#pragma unroll
        for (int c = 0; c < G::kQkChunks; ++c) {
            float2 f[4];
            unpack8(qrow[j8 + 8 * c], f);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                qf[h][c * 4 + e] = make_float2(f[e].x * a.scale_log2, f[e].y * a.scale_log2);
        }
    }
    __syncthreads();

    const uint64_t policy = pa::l2_evict_first_policy();
    auto issue = [&](int tile, int stage) {
        uint8_t* ks = ring + (warp * kStages + stage) * G::kStageBytes;
        uint8_t* vs = ks + G::kTileBytes;
        const int t0 = t_begin + tile * kTile;
        const int nv = min(kTile, t_end - t0);
        uint64_t* bar = &bars[warp * kStages + stage];
        pa::mbar_arrive_expect_tx(bar, 2u * nv * G::kRowBytes);
        for (int r = 0; r < nv;) {
            const int pos = t0 + r;
            const int off = pos & (B - 1);
            const int rows = min(nv - r, B - off);
            const int blk = table[(pos >> a.log2_block) - lb0];
            const size_t src = (((size_t)blk * a.n_kv_heads + kvh) * B + off) * D;
            pa::bulk_g2s(ks + r * G::kRowBytes, a.k_cache + src, rows * G::kRowBytes, bar, policy);
            pa::bulk_g2s(vs + r * G::kRowBytes, a.v_cache + src, rows * G::kRowBytes, bar, policy);
            r += rows;
        }
    };

    // ---- per-lane state -----------------------------------------------------
    float m_run[GP];
    float l_own[NO];
    float2 acc[GP][4];
#pragma unroll
    for (int h = 0; h < GP; ++h) {
        m_run[h] = -INFINITY;
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[h][e] = make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < NO; ++i) l_own[i] = 0.f;

    const int r4 = lane >> 3;                     // row within a score pass
    const int b1 = lane & 1;
    const int own_pos = (j8 >> 1) * 4 + r4;        // position of the kept scores
    // kept heads: GP=4 -> 2*b1, 2*b1+1; GP=2 -> b1; GP=1 -> 0
    const int pv_row = lane / G::kPvLanes;
    const int pv_col = lane % G::kPvLanes;
    float* pw = probs + warp * kTile * GP;

    if (lane == 0) {
#pragma unroll
        for (int k = 0; k < kStages; ++k) {
            const int tile = warp + k * kWarps;
            if (tile < n_tiles) issue(tile, k);
        }
    }

    int k = 0;
    for (int tile = warp; tile < n_tiles; tile += kWarps, ++k) {
        const int stage = k % kStages;
        uint64_t* bar = &bars[warp * kStages + stage];
        // every lane observes the phase itself (visibility of the async
        // copies); the decision to give up is made warp-uniform
        const bool landed = __all_sync(0xffffffffu, pa::mbar_wait_bounded(bar, (k / kStages) & 1, kMaxProbes));
        if (!landed) {
            if (lane == 0) pa::set_status(a.status, PA_DEV_WAIT_TIMEOUT);
            // drain the other stages this warp may still have in flight
            for (int kk = k + 1; kk < k + kStages; ++kk) {
                const int t2 = warp + kk * kWarps;
                if (t2 < n_tiles) pa::mbar_wait_bounded(&bars[warp * kStages + kk % kStages], (kk / kStages) & 1, 1000);
            }
            break;
        }
        const uint8_t* ks = ring + (warp * kStages + stage) * G::kStageBytes;
        const uint8_t* vs = ks + G::kTileBytes;
        const int nv = min(kTile, t_end - (t_begin + tile * kTile));

        // ---- scores: 4 passes x 4 rows, 8 lanes per row ----------------------
        float sc[4 * GP];
#pragma unroll
        for (int pass = 0; pass < 4; ++pass) {
            const uint8_t* row = ks + (pass * 4 + r4) * G::kRowBytes;
            float2 p2[GP];
#pragma unroll
            for (int h = 0; h < GP; ++h) p2[h] = make_float2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < G::kQkChunks; ++c) {
                const uint4 w = *reinterpret_cast<const uint4*>(row + (j8 + 8 * c) * 16);
                float2 kf[4];
                unpack8(w, kf);
#pragma unroll
                for (int h = 0; h < GP; ++h)
#pragma unroll
                    for (int e = 0; e < 4; ++e) p2[h] = __ffma2_rn(qf[h][c * 4 + e], kf[e], p2[h]);
            }
#pragma unroll
            for (int h = 0; h < GP; ++h) sc[pass * GP + h] = p2[h].x + p2[h].y;
        }
        reduce_scatter8<4 * GP>(sc, lane);

        // ---- online softmax ---------------------------------------------------
        float own[NO], bm[NO];
#pragma unroll
        for (int i = 0; i < NO; ++i) {
            own[i] = own_pos < nv ? sc[i] : -INFINITY;
            bm[i] = own[i];
        }
#pragma unroll
        for (int msk = 2; msk <= 16; msk <<= 1)
#pragma unroll
            for (int i = 0; i < NO; ++i) bm[i] = fmaxf(bm[i], __shfl_xor_sync(0xffffffffu, bm[i], msk));
        float bmax[GP];
        if constexpr (GP == 4) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float other = __shfl_xor_sync(0xffffffffu, bm[i], 1);
                bmax[i] = b1 ? other : bm[i];
                bmax[2 + i] = b1 ? bm[i] : other;
            }
        } else if constexpr (GP == 2) {
            const float other = __shfl_xor_sync(0xffffffffu, bm[0], 1);
            bmax[0] = b1 ? other : bm[0];
            bmax[1] = b1 ? bm[0] : other;
        } else {
            bmax[0] = bm[0];
        }
        float alpha[GP];
#pragma unroll
        for (int h = 0; h < GP; ++h) {
            const float mn = fmaxf(m_run[h], bmax[h]);
            alpha[h] = exp2f(m_run[h] - mn);
            m_run[h] = mn;
        }
#pragma unroll
        for (int i = 0; i < NO; ++i) {
            const float mh = GP == 4 ? (b1 ? m_run[2 + i] : m_run[i]) : (GP == 2 ? (b1 ? m_run[1] : m_run[0]) : m_run[0]);
            const float al = GP == 4 ? (b1 ? alpha[2 + i] : alpha[i]) : (GP == 2 ? (b1 ? alpha[1] : alpha[0]) : alpha[0]);
            const float p = exp2f(own[i] - mh);
            l_own[i] = l_own[i] * al + p;
            own[i] = p;
        }
        if constexpr (GP == 4) {
            *reinterpret_cast<float2*>(pw + own_pos * 4 + 2 * b1) = make_float2(own[0], own[1]);
        } else if constexpr (GP == 2) {
            pw[own_pos * 2 + b1] = own[0];
        } else {
            if (b1 == 0) pw[own_pos] = own[0];
        }
#pragma unroll
        for (int h = 0; h < GP; ++h) {
            const float2 al2 = make_float2(alpha[h], alpha[h]);
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[h][e] = __fmul2_rn(acc[h][e], al2);
        }
        __syncwarp();

        // ---- weighted values ------------------------------------------------
        auto pv_row_step = [&](int pos) {
            const uint4 w = *reinterpret_cast<const uint4*>(vs + pos * G::kRowBytes + pv_col * 16);
            float2 vf[4];
            unpack8(w, vf);
            float pr[GP];
            if constexpr (GP == 4) {
                const float4 t = *reinterpret_cast<const float4*>(pw + pos * 4);
                pr[0] = t.x; pr[1] = t.y; pr[2] = t.z; pr[3] = t.w;
            } else if constexpr (GP == 2) {
                const float2 t = *reinterpret_cast<const float2*>(pw + pos * 2);
                pr[0] = t.x; pr[1] = t.y;
            } else {
                pr[0] = pw[pos];
            }
#pragma unroll
            for (int h = 0; h < GP; ++h) {
                const float2 ph = make_float2(pr[h], pr[h]);
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[h][e] = __ffma2_rn(ph, vf[e], acc[h][e]);
            }
        };
        if (nv == kTile) {
#pragma unroll
            for (int pass = 0; pass < G::kPvPasses; ++pass) pv_row_step(pass * G::kPvRows + pv_row);
        } else {
#pragma unroll
            for (int pass = 0; pass < G::kPvPasses; ++pass) {
                const int pos = pass * G::kPvRows + pv_row;
                if (pos < nv) pv_row_step(pos);    // rows past the context are never read
            }
        }
        __syncwarp();
        if (lane == 0 && tile + kWarps * kStages < n_tiles) issue(tile + kWarps * kStages, stage);
    }

    // ---- finish the warp's state -------------------------------------------
#pragma unroll
    for (int msk = 2; msk <= 16; msk <<= 1)
#pragma unroll
        for (int i = 0; i < NO; ++i) l_own[i] += __shfl_xor_sync(0xffffffffu, l_own[i], msk);
    float l_run[GP];
    if constexpr (GP == 4) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float other = __shfl_xor_sync(0xffffffffu, l_own[i], 1);
            l_run[i] = b1 ? other : l_own[i];
            l_run[2 + i] = b1 ? l_own[i] : other;
        }
    } else if constexpr (GP == 2) {
        const float other = __shfl_xor_sync(0xffffffffu, l_own[0], 1);
        l_run[0] = b1 ? other : l_own[0];
        l_run[1] = b1 ? l_own[0] : other;
    } else {
        l_run[0] = l_own[0];
    }
#pragma unroll
    for (int msk = G::kPvLanes; msk < 32; msk <<= 1)
#pragma unroll
        for (int h = 0; h < GP; ++h)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc[h][e].x += __shfl_xor_sync(0xffffffffu, acc[h][e].x, msk);
                acc[h][e].y += __shfl_xor_sync(0xffffffffu, acc[h][e].y, msk);
            }

    // ---- merge the 4 warps (exact, as in the block merge) --------------------
    __syncthreads();                                   // ring no longer in use
    float* mw = reinterpret_cast<float*>(ring);        // [warp][GP]
    float* lw = mw + kWarps * GP;                      // [warp][GP]
    float* uw = lw + kWarps * GP;                      // [warp][GP][D]
    if (lane == 0) {
#pragma unroll
        for (int h = 0; h < GP; ++h) {
            mw[warp * GP + h] = m_run[h];
            lw[warp * GP + h] = l_run[h];
        }
    }
    if (lane < G::kPvLanes) {
#pragma unroll
        for (int h = 0; h < GP; ++h)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                *reinterpret_cast<float2*>(uw + (warp * GP + h) * D + pv_col * 8 + 2 * e) = acc[h][e];
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < GP * D; idx += kThreads) {
        const int h = idx / D;
        const int d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mw[w * GP + h]);
        float Z = 0.f, U = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float f = exp2f(mw[w * GP + h] - M);
            Z += f * lw[w * GP + h];
            U += f * uw[(w * GP + h) * D + d];
        }
        if (nparts == 1) {
            store_out(a.out, a.out_f32, row0 + idx, U / Z);
        } else {
            const size_t pi = ((size_t)seq * a.n_q_heads + qh0 + h) * a.max_parts + part;
            a.part_acc[pi * D + d] = U;
            if (d == 0) {
                a.part_max[pi] = M * kLn2;      // back to natural-log units
                a.part_sum[pi] = Z;
            }
        }
    }
}

// Exact merge of partition statistics (second page, section 11):
// M = max m_p, Z = sum exp(m_p - M) z_p, U = sum exp(m_p - M) u_p, out = U / Z.
// One thread block per (query head, sequence), one thread per dimension.
__global__ void lse_merge_kernel(void* out, int out_f32, const float* __restrict__ pmax,
                                 const float* __restrict__ psum, const float* __restrict__ pacc,
                                 const int32_t* __restrict__ context_lens, int ctx_cap, int partition_size,
                                 int max_parts, int n_q_heads, int d_head, int skip_single) {
    const int h = blockIdx.x;
    const int seq = blockIdx.y;
    const int d = threadIdx.x;
    int ctx = context_lens[seq];
    ctx = ctx < 0 ? 0 : (ctx > ctx_cap ? ctx_cap : ctx);
    int np = (int)(((long long)ctx + partition_size - 1) / partition_size);
    np = np > max_parts ? max_parts : np;
    if (skip_single && np <= 1) return;             // finished by the partition kernel
    const size_t orow = ((size_t)seq * n_q_heads + h) * d_head;
    if (np == 0) {
        if (d < d_head) store_out(out, out_f32, orow + d, 0.f);
        return;
    }
    const size_t base = ((size_t)seq * n_q_heads + h) * max_parts;
    float M = -INFINITY;
    for (int p = 0; p < np; ++p) M = fmaxf(M, pmax[base + p]);
    float Z = 0.f, U = 0.f;
    for (int p = 0; p < np; ++p) {
        const float w = exp2f((pmax[base + p] - M) * kLog2e);
        Z += w * psum[base + p];
        if (d < d_head) U += w * pacc[(base + p) * d_head + d];
    }
    if (d < d_head) store_out(out, out_f32, orow + d, U / Z);
}

template <int D, int GP>
int launch_decode(const DecodeArgs& a, int num_seqs, int smem_bytes, cudaStream_t stream) {
    static int attr_done[64] = {0};
    auto kernel = decode_partition_kernel<D, GP>;
    if (pa_host::ensure_smem_attr(kernel, smem_bytes, attr_done) != cudaSuccess) return PA_ERR_CUDA;
    dim3 grid(a.max_parts, a.n_kv_heads * a.n_sub, num_seqs);
    kernel<<<grid, kThreads, smem_bytes, stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int ilog2(int x) {
    int r = 0;
    while ((1 << r) < x) ++r;
    return r;
}

}  // namespace

extern "C" {

int pa_decode_default_partition_size(int max_context_len) {
    return max_context_len > 16384 ? 1024 : 512;
}

size_t pa_decode_workspace_size(int num_seqs, int n_q_heads, int d_head, int max_context_len,
                                int partition_size) {
    if (num_seqs <= 0 || n_q_heads <= 0 || d_head <= 0 || max_context_len < 0) return 0;
    const int P = partition_size > 0 ? partition_size : pa_decode_default_partition_size(max_context_len);
    const size_t np = (size_t)((max_context_len + P - 1) / P);
    if (np <= 1) return 0;
    const size_t n = (size_t)num_seqs * n_q_heads * np;
    return 2 * align256(n * sizeof(float)) + align256(n * d_head * sizeof(float));
}

int pa_decode(void* out, int out_dtype, const void* q, const void* k_cache, const void* v_cache,
              const int32_t* block_tables, const int32_t* context_lens, int block_size, float scale,
              int n_q_heads, int n_kv_heads, int d_head, int num_seqs, int max_blocks_per_seq,
              int num_blocks, int max_context_len, int partition_size, void* workspace,
              size_t workspace_bytes, int32_t* status_dev, void* stream) {
    if (num_seqs < 0 || n_q_heads <= 0 || n_kv_heads <= 0 || max_blocks_per_seq <= 0 ||
        num_blocks <= 0 || max_context_len < 0 || !(scale == scale))
        return PA_ERR_INVALID_ARG;
    if (out_dtype != PA_DTYPE_BF16 && out_dtype != PA_DTYPE_F32) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return PA_ERR_INVALID_ARG;
    if (!pa_host::supported_block_size(block_size) || !pa_host::supported_d_head(d_head))
        return PA_ERR_UNSUPPORTED;
    if (n_q_heads % n_kv_heads) return PA_ERR_UNSUPPORTED;
    const int group = n_q_heads / n_kv_heads;
    if (group != 1 && group != 2 && group != 4 && group != 8 && group != 16) return PA_ERR_UNSUPPORTED;
    if (!pa_host::aligned16(out) || !pa_host::aligned16(q) || !pa_host::aligned16(k_cache) ||
        !pa_host::aligned16(v_cache))
        return PA_ERR_MISALIGNED;
    const int P = partition_size > 0 ? partition_size : pa_decode_default_partition_size(max_context_len);
    if (P % 64 || P < 64 || P > kMaxPartition) return PA_ERR_INVALID_ARG;
    const int gp = group < 4 ? group : 4;
    const int n_sub = group / gp;
    if ((long long)n_kv_heads * n_sub > 65535 || num_seqs > 65535) return PA_ERR_UNSUPPORTED;

    DecodeArgs a{};
    a.out = out;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.k_cache = static_cast<const __nv_bfloat16*>(k_cache);
    a.v_cache = static_cast<const __nv_bfloat16*>(v_cache);
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
    a.n_sub = n_sub;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    const long long cap_tbl = (long long)max_blocks_per_seq * block_size;
    a.ctx_cap = (int)(cap_tbl < max_context_len ? cap_tbl : max_context_len);
    a.partition_size = P;
    a.max_parts = (max_context_len + P - 1) / P;
    if (a.max_parts < 1) a.max_parts = 1;

    if (a.max_parts > 1) {
        const size_t need = pa_decode_workspace_size(num_seqs, n_q_heads, d_head, max_context_len, P);
        if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
            return PA_ERR_WORKSPACE;
        const size_t n = (size_t)num_seqs * n_q_heads * a.max_parts;
        uint8_t* w = static_cast<uint8_t*>(workspace);
        a.part_max = reinterpret_cast<float*>(w);
        a.part_sum = reinterpret_cast<float*>(w + align256(n * sizeof(float)));
        a.part_acc = reinterpret_cast<float*>(w + 2 * align256(n * sizeof(float)));
    }

    const int table_ints = P / block_size + 2;
    auto smem_for = [&](int D, int GP) {
        const int ring = kWarps * kStages * 2 * kTile * D * 2;
        return ring + kWarps * kStages * 8 + kWarps * kTile * GP * 4 + table_ints * 4;
    };
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int rc;
    const int smem = smem_for(d_head, gp);
    if (d_head == 128) {
        rc = gp == 4 ? launch_decode<128, 4>(a, num_seqs, smem, st)
           : gp == 2 ? launch_decode<128, 2>(a, num_seqs, smem, st)
                     : launch_decode<128, 1>(a, num_seqs, smem, st);
    } else {
        rc = gp == 4 ? launch_decode<64, 4>(a, num_seqs, smem, st)
           : gp == 2 ? launch_decode<64, 2>(a, num_seqs, smem, st)
                     : launch_decode<64, 1>(a, num_seqs, smem, st);
    }
    if (rc != PA_OK || a.max_parts <= 1) return rc;
    dim3 grid(n_q_heads, num_seqs);
    lse_merge_kernel<<<grid, d_head, 0, st>>>(out, a.out_f32, a.part_max, a.part_sum, a.part_acc, context_lens,
                                              a.ctx_cap, P, a.max_parts, n_q_heads, d_head, 1);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
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
    dim3 grid(n_q_heads, num_seqs);
    const int threads = (d_head + 31) / 32 * 32;
    lse_merge_kernel<<<grid, threads, 0, static_cast<cudaStream_t>(stream)>>>(
        out, out_dtype == PA_DTYPE_F32, part_max, part_sum, part_acc, context_lens, 0x7fffffff, partition_size,
        max_parts, n_q_heads, d_head, 0);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// pa_decode for callers that cannot provide device scratch memory.
//
// The split path's partition statistics live in this file-scope device
// array instead of a caller workspace.  Host code must not use the name
// `g_static_scratch` as an address (on the host it is only a stand-in
// symbol); the device address is looked up once per device with
// cudaGetSymbolAddress and cached.
// ---------------------------------------------------------------------------
#include <mutex>

static __device__ __align__(256) uint8_t g_static_scratch[PA_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxScratchDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxScratchDevices] = {nullptr};

// Device address of g_static_scratch on the current device (looked up on the
// first call for that device).  Returns nullptr on failure.
void* static_scratch_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr) return nullptr;
        g_scratch_addr[dev] = ptr;
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
