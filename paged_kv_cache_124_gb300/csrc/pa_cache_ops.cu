// Cache-feeding kernels for sm_103a: reshape_and_cache (scatter each new
// token's key/value rows into its slot) and copy_blocks (copy-on-write block
// clone).  Both are pure byte copies: 16-byte vector loads and stores, one
// 16-byte chunk per thread per step, coalesced along the d_head rows.
//
// Slot arithmetic ("PagedAttention: Virtual Memory for the KV Cache",
// section 7; "PagedAttention in vLLM: scattered memory, exact attention",
// section 2): slot = physical_block * B + offset.

#include <vector>

#include "pa_common.cuh"

namespace {

constexpr int kCopyThreads = 256;
constexpr int kMaxLayersPerLaunch = 64;

// One warp per token, four tokens per thread block: the token's K rows of
// all heads, then its V rows, as 16-byte chunks.  The slot and the rows are
// loaded together (one memory round trip; at the 8B shape every lane has
// eight chunks in flight), then stored.  Launched as a programmatic
// dependent: it waits for the work before it on the stream before reading
// its inputs, and lets the next kernel start its launch right away.
constexpr int kTokensPerBlock = 4;

__global__ void __launch_bounds__(32 * kTokensPerBlock, 8) reshape_and_cache_kernel(
    uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, const uint4* __restrict__ k,
    const uint4* __restrict__ v, const int64_t* __restrict__ slot_mapping, int num_tokens, int n_kv_heads,
    int chunks_per_row, int block_size, long long num_slots, int32_t* status) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int t = blockIdx.x * kTokensPerBlock + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= num_tokens) return;
    const long long slot = slot_mapping[t];
    const int per_token = n_kv_heads * chunks_per_row;     // 16-B chunks of one token's K
    const int total = 2 * per_token;
    const uint4* ksrc = k + (size_t)t * per_token;
    const uint4* vsrc = v + (size_t)t * per_token;
    constexpr int R = 8;                                    // chunks in flight per lane
    for (int c0 = lane; c0 < total; c0 += R * 32) {
        uint4 r[R];
#pragma unroll
        for (int u = 0; u < R; ++u) {
            const int c = c0 + u * 32;
            if (c < total) r[u] = c < per_token ? ksrc[c] : vsrc[c - per_token];
        }
        if (slot < 0) return;                               // padding token
        if (slot >= num_slots) {
            if (lane == 0) pa::set_status(status, PA_DEV_BAD_SLOT);
            return;
        }
        const long long blk = slot / block_size;
        const int off = (int)(slot - blk * block_size);
#pragma unroll
        for (int u = 0; u < R; ++u) {
            const int c = c0 + u * 32;
            if (c >= total) break;
            const bool is_v = c >= per_token;
            const int cc = is_v ? c - per_token : c;
            const int h = cc / chunks_per_row;
            const int x = cc - h * chunks_per_row;
            const size_t dst = (((size_t)blk * n_kv_heads + h) * block_size + off) * chunks_per_row + x;
            (is_v ? v_cache : k_cache)[dst] = r[u];
        }
    }
}


// FP8 variant of reshape_and_cache: one thread block per token; each thread
// turns 16 bf16 inputs (two 16-byte loads) into 16 codes (one 16-byte store).
__global__ void __launch_bounds__(128) reshape_and_cache_fp8_kernel(
    uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, const uint4* __restrict__ k,
    const uint4* __restrict__ v, const int64_t* __restrict__ slot_mapping, int n_kv_heads, int chunks_per_row,
    int block_size, long long num_slots, float k_scale, float v_scale, int32_t* status) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int t = blockIdx.x;
    const long long slot = slot_mapping[t];
    if (slot < 0) return;                                   // padding token
    if (slot >= num_slots) {
        if (threadIdx.x == 0) pa::set_status(status, PA_DEV_BAD_SLOT);
        return;
    }
    const long long blk = slot / block_size;
    const int off = (int)(slot - blk * block_size);
    const int per_token = n_kv_heads * chunks_per_row;       // 16-element chunks of one token's K
    for (int c = threadIdx.x; c < 2 * per_token; c += blockDim.x) {
        const bool is_v = c >= per_token;
        const int cc = is_v ? c - per_token : c;
        const uint4* src = (is_v ? v : k) + ((size_t)t * per_token + cc) * 2;
        const uint4 a = src[0], b = src[1];
        const float sc = is_v ? v_scale : k_scale;
        const uint2 qa = pa::quant8(a, sc), qb = pa::quant8(b, sc);
        const int h = cc / chunks_per_row;
        const int x = cc - h * chunks_per_row;
        const size_t dst = (((size_t)blk * n_kv_heads + h) * block_size + off) * chunks_per_row + x;
        (is_v ? v_cache : k_cache)[dst] = make_uint4(qa.x, qa.y, qb.x, qb.y);
    }
}

struct LayerPtrs {
    uint4* k[kMaxLayersPerLaunch];
    uint4* v[kMaxLayersPerLaunch];
};

// grid: (pair, layer, 0 = K / 1 = V); each thread block copies one whole
// block (n_kv_heads * B * d_head bf16) with 4 independent 16-B loads in
// flight per thread.
__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(const __grid_constant__ LayerPtrs ptrs,
                                                                   const int32_t* __restrict__ pairs,
                                                                   long long chunks_per_block, int num_blocks,
                                                                   int32_t* status) {
    const int p = blockIdx.x;
    const int layer = blockIdx.y;
    const int src = pairs[2 * p];
    const int dst = pairs[2 * p + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (threadIdx.x == 0) pa::set_status(status, PA_DEV_BAD_BLOCK_ID);
        return;
    }
    uint4* base = blockIdx.z == 0 ? ptrs.k[layer] : ptrs.v[layer];
    const uint4* s = base + (size_t)src * chunks_per_block;
    uint4* d = base + (size_t)dst * chunks_per_block;
    constexpr int U = 4;
    long long i = threadIdx.x;
    for (; i + (U - 1) * kCopyThreads < chunks_per_block; i += U * kCopyThreads) {
        uint4 r[U];
#pragma unroll
        for (int u = 0; u < U; ++u) r[u] = s[i + u * kCopyThreads];
#pragma unroll
        for (int u = 0; u < U; ++u) d[i + u * kCopyThreads] = r[u];
    }
    for (; i < chunks_per_block; i += kCopyThreads) d[i] = s[i];
}

struct SwapPtrs {
    const uint4* src[2][kMaxLayersPerLaunch];   // [K / V][layer]
    uint4* dst[2][kMaxLayersPerLaunch];
};

// grid: (pair, layer, 0 = K / 1 = V); each thread block moves one whole
// block between two pools, either of which may be page-locked host memory:
// 8 independent 16-byte loads in flight per thread to cover the link latency.
__global__ void __launch_bounds__(kCopyThreads) swap_blocks_kernel(const __grid_constant__ SwapPtrs ptrs,
                                                                   const int32_t* __restrict__ pairs,
                                                                   long long chunks_per_block, int src_blocks,
                                                                   int dst_blocks, int32_t* status) {
    const int p = blockIdx.x;
    const int layer = blockIdx.y;
    const int src = pairs[2 * p];
    const int dst = pairs[2 * p + 1];
    if (src < 0 || src >= src_blocks || dst < 0 || dst >= dst_blocks) {
        if (threadIdx.x == 0) pa::set_status(status, PA_DEV_BAD_BLOCK_ID);
        return;
    }
    const uint4* s = ptrs.src[blockIdx.z][layer] + (size_t)src * chunks_per_block;
    uint4* d = ptrs.dst[blockIdx.z][layer] + (size_t)dst * chunks_per_block;
    constexpr int U = 8;
    long long i = threadIdx.x;
    for (; i + (U - 1) * kCopyThreads < chunks_per_block; i += U * kCopyThreads) {
        uint4 r[U];
#pragma unroll
        for (int u = 0; u < U; ++u) r[u] = s[i + u * kCopyThreads];
#pragma unroll
        for (int u = 0; u < U; ++u) d[i + u * kCopyThreads] = r[u];
    }
    for (; i < chunks_per_block; i += kCopyThreads) d[i] = s[i];
}

// Device address of a device, managed or page-locked host pointer; nullptr
// for pageable or unknown memory.
const void* device_address(const void* p) {
    if (!p) return nullptr;
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    switch (attr.type) {
        case cudaMemoryTypeDevice:
        case cudaMemoryTypeManaged:
            return p;
        case cudaMemoryTypeHost:
            return attr.devicePointer;
        default:
            return nullptr;
    }
}

}  // namespace

extern "C" {

int pa_reshape_and_cache(void* k_cache, void* v_cache, const void* k, const void* v,
                         const int64_t* slot_mapping, int num_tokens, int n_kv_heads, int d_head, int block_size,
                         int num_blocks, int32_t* status_dev, void* stream) {
    if (num_tokens < 0 || n_kv_heads <= 0 || num_blocks <= 0) return PA_ERR_INVALID_ARG;
    if (!pa_host::supported_block_size(block_size) || !pa_host::supported_d_head(d_head))
        return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!k_cache || !v_cache || !k || !v || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (!pa_host::aligned16(k_cache) || !pa_host::aligned16(v_cache) || !pa_host::aligned16(k) ||
        !pa_host::aligned16(v) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return PA_ERR_MISALIGNED;
    const cudaError_t e = pa_host::launch_dependent(
        reshape_and_cache_kernel, dim3((num_tokens + kTokensPerBlock - 1) / kTokensPerBlock),
        dim3(32 * kTokensPerBlock), 0, static_cast<cudaStream_t>(stream), static_cast<uint4*>(k_cache),
        static_cast<uint4*>(v_cache), static_cast<const uint4*>(k), static_cast<const uint4*>(v), slot_mapping,
        num_tokens, n_kv_heads, d_head / 8, block_size, (long long)num_blocks * block_size, status_dev);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_reshape_and_cache_fp8(void* k_cache, void* v_cache, const void* k, const void* v,
                             const int64_t* slot_mapping, int num_tokens, int n_kv_heads, int d_head, int block_size,
                             int num_blocks, float k_scale, float v_scale, int32_t* status_dev, void* stream) {
    if (num_tokens < 0 || n_kv_heads <= 0 || num_blocks <= 0) return PA_ERR_INVALID_ARG;
    if (!(k_scale > 0.f) || !(v_scale > 0.f)) return PA_ERR_INVALID_ARG;
    if (!pa_host::supported_block_size(block_size) || !pa_host::supported_d_head(d_head)) return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!k_cache || !v_cache || !k || !v || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (!pa_host::aligned16(k_cache) || !pa_host::aligned16(v_cache) || !pa_host::aligned16(k) ||
        !pa_host::aligned16(v) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return PA_ERR_MISALIGNED;
    const cudaError_t e = pa_host::launch_dependent(
        reshape_and_cache_fp8_kernel, dim3(num_tokens), dim3(128), 0, static_cast<cudaStream_t>(stream),
        static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), static_cast<const uint4*>(k),
        static_cast<const uint4*>(v), slot_mapping, n_kv_heads, d_head / 16, block_size,
        (long long)num_blocks * block_size, k_scale, v_scale, status_dev);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // extern "C"

namespace {

// elem_bytes: 2 for bf16 caches, 1 for E4M3 codes; a block of one head is
// block_size * d_head * elem_bytes bytes, a multiple of 16 for every
// supported shape.
int copy_blocks_impl(void* const* k_caches, void* const* v_caches, int num_layers, const int32_t* block_pairs,
                     int num_pairs, int n_kv_heads, int d_head, int block_size, int num_blocks, int elem_bytes,
                     int32_t* status_dev, void* stream) {
    if (num_layers < 0 || num_pairs < 0 || n_kv_heads <= 0 || num_blocks <= 0) return PA_ERR_INVALID_ARG;
    if (!pa_host::supported_block_size(block_size) || !pa_host::supported_d_head(d_head))
        return PA_ERR_UNSUPPORTED;
    if (num_layers == 0 || num_pairs == 0) return PA_OK;
    if (!k_caches || !v_caches || !block_pairs) return PA_ERR_INVALID_ARG;
    if (num_pairs > 2147483647 / 2) return PA_ERR_UNSUPPORTED;
    for (int l = 0; l < num_layers; ++l) {
        if (!k_caches[l] || !v_caches[l]) return PA_ERR_INVALID_ARG;
        if (!pa_host::aligned16(k_caches[l]) || !pa_host::aligned16(v_caches[l])) return PA_ERR_MISALIGNED;
    }
    if (reinterpret_cast<uintptr_t>(block_pairs) & 3u) return PA_ERR_MISALIGNED;
    const long long chunks = (long long)n_kv_heads * block_size * d_head * elem_bytes / 16;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    for (int l0 = 0; l0 < num_layers; l0 += kMaxLayersPerLaunch) {
        const int nl = num_layers - l0 < kMaxLayersPerLaunch ? num_layers - l0 : kMaxLayersPerLaunch;
        LayerPtrs ptrs{};
        for (int l = 0; l < nl; ++l) {
            ptrs.k[l] = static_cast<uint4*>(k_caches[l0 + l]);
            ptrs.v[l] = static_cast<uint4*>(v_caches[l0 + l]);
        }
        dim3 grid(num_pairs, nl, 2);
        copy_blocks_kernel<<<grid, kCopyThreads, 0, st>>>(ptrs, block_pairs, chunks, num_blocks, status_dev);
        if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
    }
    return PA_OK;
}

int swap_blocks_impl(void* const* dst_k, void* const* dst_v, const void* const* src_k, const void* const* src_v,
                     int num_layers, const int32_t* block_pairs, int num_pairs, int n_kv_heads, int d_head,
                     int block_size, int src_num_blocks, int dst_num_blocks, int elem_bytes, int32_t* status_dev,
                     void* stream) {
    if (num_layers < 0 || num_pairs < 0 || n_kv_heads <= 0 || src_num_blocks <= 0 || dst_num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    if (!pa_host::supported_block_size(block_size) || !pa_host::supported_d_head(d_head)) return PA_ERR_UNSUPPORTED;
    if (num_layers == 0 || num_pairs == 0) return PA_OK;
    if (!dst_k || !dst_v || !src_k || !src_v || !block_pairs) return PA_ERR_INVALID_ARG;
    if (num_pairs > 2147483647 / 2) return PA_ERR_UNSUPPORTED;
    const int32_t* pairs = static_cast<const int32_t*>(device_address(block_pairs));
    if (!pairs) return PA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(pairs) & 3u) return PA_ERR_MISALIGNED;
    const long long chunks = (long long)n_kv_heads * block_size * d_head * elem_bytes / 16;
    // every layer's pools are translated and checked before the first launch,
    // so that a rejected call has enqueued nothing
    std::vector<const void*> dev((size_t)num_layers * 4);      // per layer: src K, src V, dst K, dst V
    for (int l = 0; l < num_layers; ++l) {
        const void** d = dev.data() + (size_t)l * 4;
        d[0] = device_address(src_k[l]);
        d[1] = device_address(src_v[l]);
        d[2] = device_address(dst_k[l]);
        d[3] = device_address(dst_v[l]);
        if (!d[0] || !d[1] || !d[2] || !d[3]) return PA_ERR_INVALID_ARG;
        if (!pa_host::aligned16(d[0]) || !pa_host::aligned16(d[1]) || !pa_host::aligned16(d[2]) ||
            !pa_host::aligned16(d[3]))
            return PA_ERR_MISALIGNED;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    for (int l0 = 0; l0 < num_layers; l0 += kMaxLayersPerLaunch) {
        const int nl = num_layers - l0 < kMaxLayersPerLaunch ? num_layers - l0 : kMaxLayersPerLaunch;
        SwapPtrs ptrs{};
        for (int l = 0; l < nl; ++l) {
            const void* const* d = dev.data() + (size_t)(l0 + l) * 4;
            ptrs.src[0][l] = static_cast<const uint4*>(d[0]);
            ptrs.src[1][l] = static_cast<const uint4*>(d[1]);
            ptrs.dst[0][l] = static_cast<uint4*>(const_cast<void*>(d[2]));
            ptrs.dst[1][l] = static_cast<uint4*>(const_cast<void*>(d[3]));
        }
        dim3 grid(num_pairs, nl, 2);
        swap_blocks_kernel<<<grid, kCopyThreads, 0, st>>>(ptrs, pairs, chunks, src_num_blocks, dst_num_blocks,
                                                          status_dev);
        if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
    }
    return PA_OK;
}

}  // namespace

extern "C" {

int pa_copy_blocks(void* const* k_caches, void* const* v_caches, int num_layers, const int32_t* block_pairs,
                   int num_pairs, int n_kv_heads, int d_head, int block_size, int num_blocks, int32_t* status_dev,
                   void* stream) {
    return copy_blocks_impl(k_caches, v_caches, num_layers, block_pairs, num_pairs, n_kv_heads, d_head, block_size,
                            num_blocks, 2, status_dev, stream);
}

int pa_copy_blocks_fp8(void* const* k_caches, void* const* v_caches, int num_layers, const int32_t* block_pairs,
                       int num_pairs, int n_kv_heads, int d_head, int block_size, int num_blocks, int32_t* status_dev,
                       void* stream) {
    return copy_blocks_impl(k_caches, v_caches, num_layers, block_pairs, num_pairs, n_kv_heads, d_head, block_size,
                            num_blocks, 1, status_dev, stream);
}

int pa_swap_blocks(void* const* dst_k, void* const* dst_v, const void* const* src_k, const void* const* src_v,
                   int num_layers, const int32_t* block_pairs, int num_pairs, int n_kv_heads, int d_head, int block_size,
                   int src_num_blocks, int dst_num_blocks, int32_t* status_dev, void* stream) {
    return swap_blocks_impl(dst_k, dst_v, src_k, src_v, num_layers, block_pairs, num_pairs, n_kv_heads, d_head,
                            block_size, src_num_blocks, dst_num_blocks, 2, status_dev, stream);
}

int pa_swap_blocks_fp8(void* const* dst_k, void* const* dst_v, const void* const* src_k, const void* const* src_v,
                       int num_layers, const int32_t* block_pairs, int num_pairs, int n_kv_heads, int d_head,
                       int block_size, int src_num_blocks, int dst_num_blocks, int32_t* status_dev, void* stream) {
    return swap_blocks_impl(dst_k, dst_v, src_k, src_v, num_layers, block_pairs, num_pairs, n_kv_heads, d_head,
                            block_size, src_num_blocks, dst_num_blocks, 1, status_dev, stream);
}

}  // extern "C"
