// Fused attention prologue (HPC-Ops/SGLang blog, "A fused attention
// prologue"; vLLM x HPC-Ops blog, "融合的注意力前奏", HpcRopeNorm): from the
// fused QKV projection output, RMS QK-norm then rotary embedding on every
// query and key head, the query written out (bf16, or e4m3 with one scale per
// token and head, the form hpc_decode_attn_q8 consumes), and K and V written
// straight into their page slots of the cache (bf16, or e4m3 with one scale
// per token and head). One pass over the QKV output; no intermediate tensors.
//
// One warp per (token, head) row; lane l owns dims [4l, 4l+4). The RMS sum and
// the e4m3 absolute maximum are warp reductions; the rotation partner of dim d
// (d +- 64) lives in lane l ^ 16.
#include "hpc_internal.cuh"

namespace hpc {
namespace {

constexpr int kRowsPerBlock = 8;
constexpr float kE4m3Max = 448.f;

struct PrologueParams {
    const __nv_bfloat16* qkv;
    const int32_t* pos;
    const float* cos_sin;
    int max_pos;
    const float* qw;
    const float* kw;
    float eps;
    const int32_t* slots;
    int T, Hq, Hkv;
    void* q_out;
    float* q_scale;  // non-null: e4m3 query
    void* k_cache;
    void* v_cache;
    float* k_scale;
    float* v_scale;
    int num_pages;
    int kv_fp8;
    int* err;  // nullable
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

// Four floats -> e4m3 with a per-row scale = amax / 448 (1 when the row is 0);
// codes are round-to-nearest-even of x / scale, saturated. Returns the four
// codes (dim 4l in the low byte) and writes the scale.
__device__ __forceinline__ uint32_t quantise_row(const float (&y)[4], float& scale_out) {
    const float amax = warp_max(fmaxf(fmaxf(fabsf(y[0]), fabsf(y[1])), fmaxf(fabsf(y[2]), fabsf(y[3]))));
    const float scale = amax > 0.f ? amax / kE4m3Max : 1.f;
    const __nv_fp8x2_storage_t lo =
        __nv_cvt_float2_to_fp8x2(make_float2(y[0] / scale, y[1] / scale), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi =
        __nv_cvt_float2_to_fp8x2(make_float2(y[2] / scale, y[3] / scale), __NV_SATFINITE, __NV_E4M3);
    scale_out = scale;
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

__device__ __forceinline__ uint2 pack_bf16x4(const float (&y)[4]) {
    uint2 r;
    r.x = pack_bf16x2(y[0], y[1]);
    r.y = pack_bf16x2(y[2], y[3]);
    return r;
}

__global__ void __launch_bounds__(kRowsPerBlock * 32) rope_norm_kernel(const PrologueParams p) {
    grid_dependency_wait();  // the QKV projection may still be finishing
    grid_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int H3 = p.Hq + 2 * p.Hkv;
    const long long r = (long long)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
    if (r >= (long long)p.T * H3) return;
    const int t = (int)(r / H3), j = (int)(r % H3);

    const uint2 raw = *reinterpret_cast<const uint2*>(p.qkv + r * kHeadDim + 4 * lane);
    const float2 x01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
    const float2 x23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
    float y[4] = {x01.x, x01.y, x23.x, x23.y};

    if (j < p.Hq + p.Hkv) {
        // RMS QK-norm
        const float ss = warp_sum(y[0] * y[0] + y[1] * y[1] + y[2] * y[2] + y[3] * y[3]);
        const float inv = rsqrtf(ss * (1.f / kHeadDim) + p.eps);
        const float4 w = *reinterpret_cast<const float4*>((j < p.Hq ? p.qw : p.kw) + 4 * lane);
        y[0] *= inv * w.x;
        y[1] *= inv * w.y;
        y[2] *= inv * w.z;
        y[3] *= inv * w.w;
        // rotary embedding on pairs (i, i + 64)
        const int pos = p.pos[t];
        if (pos >= 0 && pos < p.max_pos) {
            const int i0 = (4 * lane) & 63;
            const float* cs = p.cos_sin + (long long)pos * kHeadDim;
            const float4 c = *reinterpret_cast<const float4*>(cs + i0);
            const float4 s = *reinterpret_cast<const float4*>(cs + 64 + i0);
            const float cv[4] = {c.x, c.y, c.z, c.w}, sv[4] = {s.x, s.y, s.z, s.w};
            const float sign = lane < 16 ? -1.f : 1.f;
            float partner[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) partner[k] = __shfl_xor_sync(0xffffffffu, y[k], 16);
#pragma unroll
            for (int k = 0; k < 4; ++k) y[k] = y[k] * cv[k] + sign * partner[k] * sv[k];
        } else if (lane == 0 && p.err) {
            atomicOr(p.err, (int)HPC_DEVERR_BAD_POSITION);
        }
    }

    if (j < p.Hq) {
        const long long qrow = (long long)t * p.Hq + j;
        if (p.q_scale) {
            float scale;
            const uint32_t codes = quantise_row(y, scale);
            *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(p.q_out) + qrow * kHeadDim + 4 * lane) = codes;
            if (lane == 0) p.q_scale[qrow] = scale;
        } else {
            *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.q_out) + qrow * kHeadDim + 4 * lane) =
                pack_bf16x4(y);
        }
        return;
    }

    // K or V: into the token's page slot
    const int slot = p.slots[t];
    if (slot < 0) return;  // padding token: nothing to write
    const int page = slot / kChunk, off = slot % kChunk;
    if (page >= p.num_pages) {
        if (lane == 0 && p.err) atomicOr(p.err, (int)HPC_DEVERR_PAGE_OUT_OF_RANGE);
        return;
    }
    const bool is_k = j < p.Hq + p.Hkv;
    const int h = is_k ? j - p.Hq : j - p.Hq - p.Hkv;
    const long long elem = (((long long)page * kChunk + off) * p.Hkv + h) * kHeadDim + 4 * lane;
    void* cache = is_k ? p.k_cache : p.v_cache;
    if (p.kv_fp8) {
        float scale;
        const uint32_t codes = quantise_row(y, scale);
        *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(cache) + elem) = codes;
        if (lane == 0) (is_k ? p.k_scale : p.v_scale)[((long long)page * p.Hkv + h) * kChunk + off] = scale;
    } else {
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(cache) + elem) = pack_bf16x4(y);
    }
}

}  // namespace

cudaError_t launch_rope_norm(const RopeNormArgs& a, cudaStream_t s) {
    PrologueParams p;
    p.qkv = static_cast<const __nv_bfloat16*>(a.qkv);
    p.pos = a.positions;
    p.cos_sin = a.cos_sin;
    p.max_pos = a.max_pos;
    p.qw = a.q_weight;
    p.kw = a.k_weight;
    p.eps = a.eps;
    p.slots = a.slots;
    p.T = a.num_tokens;
    p.Hq = a.num_q_heads;
    p.Hkv = a.num_kv_heads;
    p.q_out = a.q_out;
    p.q_scale = a.q_scale;
    p.k_cache = a.k_cache;
    p.v_cache = a.v_cache;
    p.k_scale = a.k_scale;
    p.v_scale = a.v_scale;
    p.num_pages = a.num_pages;
    p.kv_fp8 = a.kv_fp8;
    p.err = a.err;
    const long long rows = (long long)a.num_tokens * (a.num_q_heads + 2 * a.num_kv_heads);
    if (rows == 0) return cudaSuccess;
    const long long blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
    return launch_pdl(rope_norm_kernel, dim3((unsigned)blocks), dim3(kRowsPerBlock * 32), 0, s, p);
}

}  // namespace hpc
