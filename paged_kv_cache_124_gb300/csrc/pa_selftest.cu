// Self-test of the kernels' failure path: a bounded wait that runs out.
//
// Every wait of the decode, prefill and copy kernels on an mbarrier (a TMA
// copy landing, a product finishing, a neighbouring warp's result) is
// bounded; when the limit passes, the kernel records PA_DEV_WAIT_TIMEOUT in
// the caller's status word and returns instead of hanging, so the context
// stays usable.  This entry point makes such a wait run out on purpose, on a
// barrier that nothing ever arrives on, with the same wait routine the decode
// pipeline uses, so that a test can check the status and go on using the GPU.

#include "pa_common.cuh"

namespace {

__global__ void bounded_wait_kernel(int max_probes, int32_t* status) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        pa::mbar_init(&bar, 1);                 // one arrival expected; none comes
        pa::fence_mbar_init();
    }
    __syncthreads();
    const bool ok = __all_sync(0xffffffffu, pa::mbar_wait_bounded(&bar, 0, max_probes));
    if (!ok && threadIdx.x == 0) pa::set_status(status, PA_DEV_WAIT_TIMEOUT);
}

}  // namespace

extern "C" {

int pa_check_bounded_wait(int max_probes, int32_t* status_dev, void* stream) {
    if (max_probes <= 0 || max_probes > 10000000 || !status_dev) return PA_ERR_INVALID_ARG;
    bounded_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(max_probes, status_dev);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // extern "C"
