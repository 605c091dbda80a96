// Combine stage (HPC-Ops/SGLang blog, "Scheduling around live KV work", the
// paragraph on execution: the combine reads the actual split count of every
// (request, head) and merges the partials under the global softmax
// normalisation; vLLM x HPC-Ops blog, "解决方案：按步负载均衡的 decode 调度器",
// the final combine into the BF16 output).
//
// One warp per output row (request b, new token i, query head qh); lane k
// owns dims [4k, 4k+4). With n partials (o_i, lse_i) of pair (qh / 8, b):
//   M = max lse_i, w_i = exp(lse_i - M), out = sum w_i o_i / sum w_i,
//   out_lse = M + ln sum w_i.
// A long request can leave a pair with ~100 partials, so the weights of a
// tile of splits are staged in shared memory and eight partial rows per lane
// are loaded before they are accumulated (the loop is latency bound).
#include "hpc_internal.cuh"

namespace hpc {
namespace {

constexpr int kCombineWarps = 8;
constexpr int kWTile = 256;  // split weights staged per warp at a time
constexpr int kUnroll = 8;   // split rows in flight per lane
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994530942f;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

__global__ void __launch_bounds__(kCombineWarps * 32)
    combine_kernel(const int32_t* __restrict__ pair_nsplit, const int32_t* __restrict__ pair_split0,
                   const float* __restrict__ split_o, const float* __restrict__ split_lse,
                   __nv_bfloat16* __restrict__ out, float* __restrict__ out_lse, int B, int Hq, int Q) {
    __shared__ float wsh[kCombineWarps][kWTile];
    grid_dependency_wait();  // the partials come from the attention kernel
    grid_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * kCombineWarps + warp;
    if (row >= (long long)B * Q * Hq) return;
    const int b = (int)(row / ((long long)Q * Hq));
    const int r = (int)(row % ((long long)Q * Hq));
    const int qi = r / Hq, qh = r % Hq;
    const int h = qh / kGroup;
    const long long pair = (long long)h * B + b;
    const int n = pair_nsplit[pair];
    // partial rows of split s are [s][Q][8]: this row's partial of split s is
    // s * rs + j with rs = 8 * Q rows per split
    const long long s0 = pair_split0[pair];
    const long long rs = (long long)Q * kGroup;
    const int j = qi * kGroup + qh % kGroup;

    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float lse = -INFINITY;
    if (n == 1) {
        acc = *reinterpret_cast<const float4*>(split_o + (s0 * rs + j) * kHeadDim + 4 * lane);
        lse = split_lse[s0 * rs + j];
    } else if (n > 1) {
        float M = -INFINITY;
        for (int i = lane; i < n; i += 32) M = fmaxf(M, split_lse[(s0 + i) * rs + j]);
        M = warp_max(M);
        if (M != -INFINITY) {
            float wpart = 0.f;
            for (int t0 = 0; t0 < n; t0 += kWTile) {
                const int tn = min(kWTile, n - t0);
                // weights of this tile, one per lane-strided split
                for (int i = lane; i < tn; i += 32) {
                    const float w = exp2f((split_lse[(s0 + t0 + i) * rs + j] - M) * kLog2e);
                    wsh[warp][i] = w;
                    wpart += w;
                }
                __syncwarp();
                // weighted rows, kUnroll independent loads in flight per lane
                const float* base = split_o + ((s0 + t0) * rs + j) * kHeadDim + 4 * lane;
                int i = 0;
                for (; i + kUnroll <= tn; i += kUnroll) {
                    float4 x[kUnroll];
#pragma unroll
                    for (int u = 0; u < kUnroll; ++u)
                        x[u] = *reinterpret_cast<const float4*>(base + (long long)(i + u) * rs * kHeadDim);
#pragma unroll
                    for (int u = 0; u < kUnroll; ++u) {
                        const float w = wsh[warp][i + u];
                        acc.x += w * x[u].x;
                        acc.y += w * x[u].y;
                        acc.z += w * x[u].z;
                        acc.w += w * x[u].w;
                    }
                }
                for (; i < tn; ++i) {
                    const float4 x = *reinterpret_cast<const float4*>(base + (long long)i * rs * kHeadDim);
                    const float w = wsh[warp][i];
                    acc.x += w * x.x;
                    acc.y += w * x.y;
                    acc.z += w * x.z;
                    acc.w += w * x.w;
                }
                __syncwarp();
            }
            const float wsum = warp_sum(wpart);
            const float inv = 1.f / wsum;
            acc.x *= inv;
            acc.y *= inv;
            acc.z *= inv;
            acc.w *= inv;
            lse = M + log2f(wsum) * kLn2;
        }
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 packed;
    packed.x = *reinterpret_cast<uint32_t*>(&lo);
    packed.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(out + row * kHeadDim + 4 * lane) = packed;
    if (out_lse && lane == 0) out_lse[row] = lse;
}

}  // namespace

cudaError_t launch_combine(const int32_t* plan, int C, const float* split_o, const float* split_lse,
                           __nv_bfloat16* out, float* out_lse, int B, int Hq, int Hkv, int q_len, cudaStream_t s) {
    const PlanLayout L = plan_layout(B, Hkv, C);
    const long long rows = (long long)B * q_len * Hq;
    const long long blocks = (rows + kCombineWarps - 1) / kCombineWarps;
    return launch_pdl(combine_kernel, dim3((unsigned)blocks), dim3(kCombineWarps * 32), 0, s,
                      plan + L.pair_nsplit, plan + L.pair_split0, split_o, split_lse, out, out_lse, B, Hq, q_len);
}

}  // namespace hpc
