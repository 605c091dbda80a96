// Zero-copy staging for the host-buffer step (hpc_decode_step_host): one
// kernel reads the step's inputs (query, lengths, page table) straight from
// page-locked, device-mapped host memory over the host link and writes them
// into the device workspace, instead of one cudaMemcpyAsync per buffer (a
// copy engine transfer of a few hundred KB to 1 MB measured 110-120 GB/s on
// GB300, with a fixed cost per copy).
#include "hpc_internal.cuh"

namespace hpc {
namespace {

constexpr int kStageThreads = 256;

__device__ __forceinline__ void copy_range(const StageCopy& r, long long tid, long long nthreads) {
    if (r.bytes == 0) return;
    const uintptr_t a = reinterpret_cast<uintptr_t>(r.src) | reinterpret_cast<uintptr_t>(r.dst) | r.bytes;
    if ((a & 15) == 0) {
        const uint4* s = reinterpret_cast<const uint4*>(r.src);
        uint4* d = reinterpret_cast<uint4*>(r.dst);
        for (long long i = tid; i < (long long)(r.bytes / 16); i += nthreads) d[i] = s[i];
    } else if ((a & 3) == 0) {
        const uint32_t* s = reinterpret_cast<const uint32_t*>(r.src);
        uint32_t* d = reinterpret_cast<uint32_t*>(r.dst);
        for (long long i = tid; i < (long long)(r.bytes / 4); i += nthreads) d[i] = s[i];
    } else {
        for (long long i = tid; i < (long long)r.bytes; i += nthreads) r.dst[i] = r.src[i];
    }
}

__global__ void __launch_bounds__(kStageThreads) stage_in_kernel(StageCopy a, StageCopy b, StageCopy c) {
    // the previous step's kernels may still read the workspace this overwrites
    grid_dependency_wait();
    grid_launch_dependents();
    const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long n = (long long)gridDim.x * blockDim.x;
    copy_range(a, tid, n);
    copy_range(b, tid, n);
    copy_range(c, tid, n);
}

}  // namespace

cudaError_t launch_stage_in(const StageCopy& a, const StageCopy& b, const StageCopy& c, cudaStream_t s) {
    const size_t vec = (a.bytes + b.bytes + c.bytes) / 16 + 1;
    const long long blocks = (long long)((vec + kStageThreads - 1) / kStageThreads);
    const unsigned grid = (unsigned)(blocks < 1216 ? blocks : 1216);  // 8 per SM on 152 SMs at most
    return launch_pdl(stage_in_kernel, dim3(grid), dim3(kStageThreads), 0, s, a, b, c);
}

}  // namespace hpc
