// Combine stage (HPC-Ops/SGLang blog, "Scheduling around live KV work", the
// paragraph on execution: the combine reads the actual split count of every
// (request, head) and merges the partials under the global softmax
// normalisation; vLLM x HPC-Ops blog, "解决方案：按步负载均衡的 decode 调度器",
// the final combine into the BF16 output).
//
// Two forms, the same sums in the same order per output row (so the same bits):
//  - rows: one warp per output row (request b, new token i, query head qh),
//    lane k owning dims [4k, 4k+4); the weights of a tile of splits are staged
//    in shared memory and eight partial rows per lane are loaded before they
//    are accumulated (a long request can leave a pair with ~100 partials);
//    grids of at most one wave of blocks, whose time is their slowest row,
//    load a row's first 128 LSEs once for its max and its weights and its
//    partials sixteen at a time, the last batch predicated;
//  - pairs: one warp per (KV-head pair, new token): the 8 query heads of the
//    pair share its split range, so one lookup of (n, s0) serves 8 rows and
//    each split contributes 8 independent row loads per lane.
// The launcher takes the pair form when there are enough (pair, token) tasks
// to fill the GPU with it (batches of many short requests), else the row form,
// which spreads a pair's splits over 8 warps. With n partials (o_i, lse_i) of
// a row: M = max lse_i, w_i = exp(lse_i - M), out = sum w_i o_i / sum w_i,
// out_lse = M + ln sum w_i; weights lane-strided then reduced over the warp,
// weighted rows summed split by split.
#include "hpc_internal.cuh"

namespace hpc {
namespace {

constexpr int kCombineWarps = 8;
constexpr int kWTile = 64;     // pair form: splits whose 8 weights are staged per warp at a time
constexpr int kRowTile = 256;  // row form: split weights staged per warp at a time
constexpr int kUnrollShort = 8;  // row form, many rows: split rows in flight per lane
constexpr int kUnrollLong = 16;  // row form, few rows: split rows in flight per lane (last batch predicated)
constexpr int kLsePerLane = 4;   // row form, few rows: LSEs a lane keeps from the max pass for the weights
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

// The 8 LSEs of one split for rows jb .. jb + 7 (32 contiguous, 32-byte aligned bytes).
__device__ __forceinline__ void load_lse8(const float* p, float (&l)[kGroup]) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 c = *reinterpret_cast<const float4*>(p + 4);
    l[0] = a.x, l[1] = a.y, l[2] = a.z, l[3] = a.w, l[4] = c.x, l[5] = c.y, l[6] = c.z, l[7] = c.w;
}

__global__ void __launch_bounds__(kCombineWarps * 32, 2)
    combine_pairs_kernel(const int32_t* __restrict__ pair_nsplit, const int32_t* __restrict__ pair_split0,
                   const float* __restrict__ split_o, const float* __restrict__ split_lse,
                   __nv_bfloat16* __restrict__ out, float* __restrict__ out_lse, int B, int Hq, int Q) {
    __shared__ float wsh[kCombineWarps][kWTile][kGroup];
    grid_dependency_wait();  // the partials come from the attention kernel
    grid_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Hkv = Hq / kGroup;
    const long long task = (long long)blockIdx.x * kCombineWarps + warp;
    if (task >= (long long)Hkv * B * Q) return;
    const long long pair = task / Q;  // h * B + b
    const int qi = (int)(task % Q);
    const int h = (int)(pair / B), b = (int)(pair % B);
    const int n = pair_nsplit[pair];
    // partial rows of split s are [s][Q][8]: head j of new token qi in split s is
    // row s * rs + jb + j
    const long long s0 = pair_split0[pair];
    const long long rs = (long long)Q * kGroup;
    const int jb = qi * kGroup;

    float4 acc[kGroup];
    float lse[kGroup];
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
        acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        lse[j] = -INFINITY;
    }
    if (n == 1) {
        const float* base = split_o + (s0 * rs + jb) * kHeadDim + 4 * lane;
#pragma unroll
        for (int j = 0; j < kGroup; ++j) acc[j] = *reinterpret_cast<const float4*>(base + j * kHeadDim);
        load_lse8(split_lse + s0 * rs + jb, lse);
    } else if (n > 1) {
        float M[kGroup];
#pragma unroll
        for (int j = 0; j < kGroup; ++j) M[j] = -INFINITY;
        for (int i = lane; i < n; i += 32) {
            float l[kGroup];
            load_lse8(split_lse + (s0 + i) * rs + jb, l);
#pragma unroll
            for (int j = 0; j < kGroup; ++j) M[j] = fmaxf(M[j], l[j]);
        }
        float wpart[kGroup];
#pragma unroll
        for (int j = 0; j < kGroup; ++j) {
            M[j] = warp_max(M[j]);
            wpart[j] = 0.f;
        }
        for (int t0 = 0; t0 < n; t0 += kWTile) {
            const int tn = min(kWTile, n - t0);
            for (int i = lane; i < tn; i += 32) {
                float l[kGroup];
                load_lse8(split_lse + (s0 + t0 + i) * rs + jb, l);
#pragma unroll
                for (int j = 0; j < kGroup; ++j) {
                    const float w = M[j] == -INFINITY ? 0.f : exp2f((l[j] - M[j]) * kLog2e);
                    wsh[warp][i][j] = w;
                    wpart[j] += w;
                }
            }
            __syncwarp();
            const float* base = split_o + ((s0 + t0) * rs + jb) * kHeadDim + 4 * lane;
            int i = 0;
            for (; i + 2 <= tn; i += 2) {
                float4 x[2][kGroup];
#pragma unroll
                for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int j = 0; j < kGroup; ++j)
                        x[u][j] = *reinterpret_cast<const float4*>(base + ((i + u) * rs + j) * kHeadDim);
#pragma unroll
                for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int j = 0; j < kGroup; ++j) {
                        if (M[j] == -INFINITY) continue;
                        const float w = wsh[warp][i + u][j];
                        acc[j].x += w * x[u][j].x;
                        acc[j].y += w * x[u][j].y;
                        acc[j].z += w * x[u][j].z;
                        acc[j].w += w * x[u][j].w;
                    }
            }
            for (; i < tn; ++i) {
#pragma unroll
                for (int j = 0; j < kGroup; ++j) {
                    const float4 x = *reinterpret_cast<const float4*>(base + (i * rs + j) * kHeadDim);
                    if (M[j] == -INFINITY) continue;
                    const float w = wsh[warp][i][j];
                    acc[j].x += w * x.x;
                    acc[j].y += w * x.y;
                    acc[j].z += w * x.z;
                    acc[j].w += w * x.w;
                }
            }
            __syncwarp();
        }
#pragma unroll
        for (int j = 0; j < kGroup; ++j) {
            const float wsum = warp_sum(wpart[j]);
            if (M[j] == -INFINITY) continue;
            const float inv = 1.f / wsum;
            acc[j].x *= inv;
            acc[j].y *= inv;
            acc[j].z *= inv;
            acc[j].w *= inv;
            lse[j] = M[j] + log2f(wsum) * kLn2;
        }
    }
    const long long row0 = ((long long)b * Q + qi) * Hq + (long long)h * kGroup;
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc[j].x, acc[j].y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(acc[j].z, acc[j].w);
        uint2 packed;
        packed.x = *reinterpret_cast<uint32_t*>(&lo);
        packed.y = *reinterpret_cast<uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(out + (row0 + j) * kHeadDim + 4 * lane) = packed;
    }
    if (out_lse && lane < kGroup) {
        float v = lse[0];
#pragma unroll
        for (int j = 1; j < kGroup; ++j) v = lane == j ? lse[j] : v;
        out_lse[row0 + lane] = v;
    }
}

template <bool LONG>
__global__ void __launch_bounds__(kCombineWarps * 32)
    combine_rows_kernel(const int32_t* __restrict__ pair_nsplit, const int32_t* __restrict__ pair_split0,
                   const float* __restrict__ split_o, const float* __restrict__ split_lse,
                   __nv_bfloat16* __restrict__ out, float* __restrict__ out_lse, int B, int Hq, int Q) {
    __shared__ float wsh[kCombineWarps][kRowTile];
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
    } else if (n > 1 && !LONG) {
        float M = -INFINITY;
        for (int i = lane; i < n; i += 32) M = fmaxf(M, split_lse[(s0 + i) * rs + j]);
        M = warp_max(M);
        if (M != -INFINITY) {
            float wpart = 0.f;
            for (int t0 = 0; t0 < n; t0 += kRowTile) {
                const int tn = min(kRowTile, n - t0);
                // weights of this tile, one per lane-strided split
                for (int i = lane; i < tn; i += 32) {
                    const float w = exp2f((split_lse[(s0 + t0 + i) * rs + j] - M) * kLog2e);
                    wsh[warp][i] = w;
                    wpart += w;
                }
                __syncwarp();
                // weighted rows, kUnrollShort independent loads in flight per lane
                const float* base = split_o + ((s0 + t0) * rs + j) * kHeadDim + 4 * lane;
                int i = 0;
                for (; i + kUnrollShort <= tn; i += kUnrollShort) {
                    float4 x[kUnrollShort];
#pragma unroll
                    for (int u = 0; u < kUnrollShort; ++u)
                        x[u] = *reinterpret_cast<const float4*>(base + (long long)(i + u) * rs * kHeadDim);
#pragma unroll
                    for (int u = 0; u < kUnrollShort; ++u) {
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
    } else if (n > 1) {
        // the LSEs of the first 32 * kLsePerLane splits load once, all at a time,
        // and serve both the max and the weights
        float lv[kLsePerLane];
#pragma unroll
        for (int t = 0; t < kLsePerLane; ++t) {
            const int i = lane + 32 * t;
            lv[t] = i < n ? split_lse[(s0 + i) * rs + j] : -INFINITY;
        }
        float M = lv[0];
#pragma unroll
        for (int t = 1; t < kLsePerLane; ++t) M = fmaxf(M, lv[t]);
        for (int i = lane + 32 * kLsePerLane; i < n; i += 32) M = fmaxf(M, split_lse[(s0 + i) * rs + j]);
        M = warp_max(M);
        if (M != -INFINITY) {
            float wpart = 0.f;
            for (int t0 = 0; t0 < n; t0 += kRowTile) {
                const int tn = min(kRowTile, n - t0);
                // weights of this tile, one per lane-strided split
                for (int i = lane, t = 0; i < tn; i += 32, ++t) {
                    float l = 0.f;
                    if (t0 == 0 && t < kLsePerLane) {
#pragma unroll
                        for (int k = 0; k < kLsePerLane; ++k) l = t == k ? lv[k] : l;
                    } else {
                        l = split_lse[(s0 + t0 + i) * rs + j];
                    }
                    const float w = exp2f((l - M) * kLog2e);
                    wsh[warp][i] = w;
                    wpart += w;
                }
                __syncwarp();
                // weighted rows, kUnrollLong independent loads in flight per lane; the
                // last batch loads only the splits that exist
                const float* base = split_o + ((s0 + t0) * rs + j) * kHeadDim + 4 * lane;
                for (int i = 0; i < tn; i += kUnrollLong) {
                    float4 x[kUnrollLong];
#pragma unroll
                    for (int u = 0; u < kUnrollLong; ++u)
                        x[u] = i + u < tn ? *reinterpret_cast<const float4*>(base + (long long)(i + u) * rs * kHeadDim)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int u = 0; u < kUnrollLong; ++u) {
                        if (i + u >= tn) break;
                        const float w = wsh[warp][i + u];
                        acc.x += w * x[u].x;
                        acc.y += w * x[u].y;
                        acc.z += w * x[u].z;
                        acc.w += w * x[u].w;
                    }
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
    const long long tasks = (long long)Hkv * B * q_len;  // (pair, new token)
    // one wave of the pair form: 2 blocks of 8 warps per SM (its register bound)
    static const long long full_wave = [] {
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            sms = 0;
        return (long long)(sms > 0 ? sms : 152) * 2 * kCombineWarps;
    }();
    if (tasks >= full_wave) {
        const long long blocks = (tasks + kCombineWarps - 1) / kCombineWarps;
        return launch_pdl(combine_pairs_kernel, dim3((unsigned)blocks), dim3(kCombineWarps * 32), 0, s,
                          plan + L.pair_nsplit, plan + L.pair_split0, split_o, split_lse, out, out_lse, B, Hq, q_len);
    }
    const long long rows = tasks * kGroup;
    const long long blocks = (rows + kCombineWarps - 1) / kCombineWarps;
    // At most one wave of blocks (2 per SM at the long form's registers): the
    // grid's latency is its slowest row, a pair with many partials, so rows
    // load their LSEs once and their partials 16 at a time. More blocks: the
    // lighter form keeps more of them resident.
    if (blocks <= full_wave / kCombineWarps)
        return launch_pdl(combine_rows_kernel<true>, dim3((unsigned)blocks), dim3(kCombineWarps * 32), 0, s,
                          plan + L.pair_nsplit, plan + L.pair_split0, split_o, split_lse, out, out_lse, B, Hq, q_len);
    return launch_pdl(combine_rows_kernel<false>, dim3((unsigned)blocks), dim3(kCombineWarps * 32), 0, s,
                      plan + L.pair_nsplit, plan + L.pair_split0, split_o, split_lse, out, out_lse, B, Hq, q_len);
}

}  // namespace hpc
