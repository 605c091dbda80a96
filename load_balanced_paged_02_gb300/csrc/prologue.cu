// Fused attention prologue (HPC-Ops/SGLang blog, "A fused attention
// prologue"; vLLM x HPC-Ops blog, "融合的注意力前奏", HpcRopeNorm): from the
// fused QKV projection output, RMS QK-norm then rotary embedding on every
// query and key head, the query written out (bf16, or e4m3 with one scale per
// token and head, the form hpc_decode_attn_q8 consumes), and K and V written
// straight into their page slots of the cache (bf16, or e4m3 with one scale
// per token and head). One pass over the QKV output; no intermediate tensors.
//
// One block per token. A half-warp owns one (token, head) row, lane k of the
// half owning dims [4k, 4k+4) and their rotation partners [64+4k, 64+4k+4)
// (two 8-byte loads and stores, each half-warp-wide access 128 contiguous
// bytes), so the rotary embedding needs no data from other lanes; a warp
// covers two rows per round and the block's 8 warps cover 16 rows per round;
// the five rounds of a Hy3 token (80 rows) are all loaded before any is
// processed, so a block waits on memory once. The token's position, slot and
// rotary row are loaded once per block, the norm weights per row from L1. The
// reductions (norm sum; e4m3 absolute max, only when a call writes e4m3) take
// four xor-shuffle steps inside the half-warp. Row kinds (query, key, value)
// are per-lane predicates, so all lanes run every shuffle. The kernel is bound
// by instruction issue for prefill-sized calls, so per-row work is kept small.
#include "hpc_internal.cuh"

namespace hpc {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kRowsPerRound = 2 * kWarpsPerBlock;  // one row per half-warp
constexpr int kMaxRounds = 5;                        // rounds loaded before any is processed (80 rows)
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
    int rounds_per_block;  // rounds of 16 rows each block of a token takes (gridDim.y splits a token)
};

__device__ __forceinline__ float half_sum(float v) {
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

__device__ __forceinline__ float half_max(float v) {
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

// Dims [4k, 4k+4) and [64+4k, 64+4k+4) of a row that starts at `row` + 4k.
__device__ __forceinline__ uint4 load_pair(const __nv_bfloat16* row) {
    const uint2 a = *reinterpret_cast<const uint2*>(row);
    const uint2 b = *reinterpret_cast<const uint2*>(row + 64);
    return make_uint4(a.x, a.y, b.x, b.y);
}

__device__ __forceinline__ void unpack8(const uint4& r, float (&y)[8]) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
        y[2 * k] = f.x;
        y[2 * k + 1] = f.y;
    }
}

// MINB resident blocks per SM: 3 for decode-size calls (a few blocks, latency
// bound); for many tokens more blocks in flight keep more rows loading: 5 with
// bf16 outputs (8192 tokens at 64/8 heads: 70.2 -> 66.8 us, at the cost of a
// 64-byte spill), 4 when an output is e4m3, whose per-row quantisation gains
// nothing from a fifth block (81.9 -> 82.0 us).
template <int MINB>
__global__ void __launch_bounds__(kWarpsPerBlock * 32, MINB) rope_norm_kernel(const PrologueParams p) {
    grid_dependency_wait();  // the QKV projection may still be finishing
    grid_launch_dependents();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int hl = lane & 15;                 // lane within the half-warp
    const int half = lane >> 4;               // which of the warp's two rows
    const int H3 = p.Hq + 2 * p.Hkv;
    const int t = blockIdx.x;
    // the first rounds' rows load first: they do not depend on the position
    const __nv_bfloat16* src = p.qkv + (size_t)t * H3 * kHeadDim + 4 * hl;
    const int all_rounds = (H3 + kRowsPerRound - 1) / kRowsPerRound;
    const int first = blockIdx.y * p.rounds_per_block;
    const int rounds = min(all_rounds, first + p.rounds_per_block);
    uint4 raw[kMaxRounds];
#pragma unroll
    for (int r = 0; r < kMaxRounds; ++r) {
        const int j = (first + r) * kRowsPerRound + 2 * warp + half;
        raw[r] = make_uint4(0u, 0u, 0u, 0u);
        if (first + r < rounds && j < H3) raw[r] = load_pair(src + (size_t)j * kHeadDim);
    }
    const int pos = p.pos[t];
    const int slot = p.slots[t];
    const bool rotate = pos >= 0 && pos < p.max_pos;
    const bool slot_ok = slot >= 0 && slot / kChunk < p.num_pages;
    if (threadIdx.x == 0 && blockIdx.y == 0 && p.err) {
        if (!rotate) atomicOr(p.err, (int)HPC_DEVERR_BAD_POSITION);
        if (slot >= 0 && !slot_ok) atomicOr(p.err, (int)HPC_DEVERR_PAGE_OUT_OF_RANGE);
    }
    // per-lane constants: rotation cos/sin of pair indices [4*hl, 4*hl+4) (the
    // norm weights are read per row from L1, which keeps the registers for the
    // rows in flight); cos 1, sin 0 without a valid position
    float c[4], sn[4];
    {
        const float* cs = p.cos_sin + (long long)(rotate ? pos : 0) * kHeadDim + 4 * hl;
        const float4 c0 = *reinterpret_cast<const float4*>(cs);
        const float4 s0 = *reinterpret_cast<const float4*>(cs + 64);
        const float cc[4] = {c0.x, c0.y, c0.z, c0.w};
        const float ss[4] = {s0.x, s0.y, s0.z, s0.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            c[k] = rotate ? cc[k] : 1.f;
            sn[k] = rotate ? ss[k] : 0.f;
        }
    }
    const bool any_fp8 = p.q_scale != nullptr || p.kv_fp8 != 0;  // uniform over the grid
    for (int r0 = first; r0 < rounds; r0 += kMaxRounds) {
        if (r0 != first) {
#pragma unroll
            for (int r = 0; r < kMaxRounds; ++r) {
                const int j = (r0 + r) * kRowsPerRound + 2 * warp + half;
                raw[r] = make_uint4(0u, 0u, 0u, 0u);
                if (r0 + r < rounds && j < H3) raw[r] = load_pair(src + (size_t)j * kHeadDim);
            }
        }
#pragma unroll
        for (int r = 0; r < kMaxRounds; ++r) {
            if (r0 + r >= rounds) break;  // uniform across the block
            const int j = (r0 + r) * kRowsPerRound + 2 * warp + half;
            const bool valid = j < H3;
            const bool is_q = j < p.Hq, is_qk = j < p.Hq + p.Hkv;
            float y[8];
            unpack8(raw[r], y);
            // RMS QK-norm (computed for every row, applied to query and key rows)
            float s2 = 0.f;
#pragma unroll
            for (int k = 0; k < 8; ++k) s2 += y[k] * y[k];
            s2 = half_sum(s2);
            const float inv = is_qk ? rsqrtf(s2 * (1.f / kHeadDim) + p.eps) : 1.f;
            if (is_qk) {
                const float* wr = (is_q ? p.qw : p.kw) + 4 * hl;
                const float4 w0 = __ldg(reinterpret_cast<const float4*>(wr));
                const float4 w1 = __ldg(reinterpret_cast<const float4*>(wr + 64));
                const float ww[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                for (int k = 0; k < 8; ++k) y[k] *= inv * ww[k];
            }
            // rotary embedding on pairs (i, i + 64), both in this lane: y[k] and y[k + 4]
            if (is_qk) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float a = y[k], b = y[k + 4];
                    y[k] = a * c[k] + b * -sn[k];
                    y[k + 4] = b * c[k] + a * sn[k];
                }
            }
            // output format of this row
            const bool fp8_row = is_q ? (p.q_scale != nullptr) : (p.kv_fp8 != 0);
            float am = 0.f;
            if (any_fp8) {
#pragma unroll
                for (int k = 0; k < 8; ++k) am = fmaxf(am, fabsf(y[k]));
                am = half_max(am);
            }
            if (!valid || (!is_q && !slot_ok)) continue;
            size_t dst_elem;
            void* dst;
            float* scale_dst = nullptr;
            if (is_q) {
                const size_t qrow = (size_t)t * p.Hq + j;
                dst_elem = qrow * kHeadDim + 4 * hl;
                dst = p.q_out;
                scale_dst = p.q_scale ? p.q_scale + qrow : nullptr;
            } else {
                const int h = is_qk ? j - p.Hq : j - p.Hq - p.Hkv;
                const int page = slot / kChunk, off = slot % kChunk;
                dst_elem = (((size_t)page * kChunk + off) * p.Hkv + h) * kHeadDim + 4 * hl;
                dst = is_qk ? p.k_cache : p.v_cache;
                if (p.kv_fp8) scale_dst = (is_qk ? p.k_scale : p.v_scale) + ((size_t)page * p.Hkv + h) * kChunk + off;
            }
            if (fp8_row) {
                // x / scale correctly rounded: bf16 inputs often land exactly on e4m3
                // rounding midpoints, where a last-bit error would break the tie the
                // other way. Markstein's correction step (P. Markstein, "Computation
                // of elementary functions on the IBM RISC System/6000 processor",
                // IBM J. Res. Dev. 34(1), 1990): with y = RN(1 / scale), q = RN(x y)
                // and the exact residual r = x - scale q (one FMA), RN(q + r y) is
                // the correctly rounded quotient while nothing over- or underflows
                // (|x / scale| <= 448 here).
                const float scale = am > 0.f ? am / kE4m3Max : 1.f;
                const float rcp = __frcp_rn(scale);
                auto qdiv = [scale, rcp](float x) {
                    const float q = x * rcp;
                    return fmaf(fmaf(-q, scale, x), rcp, q);
                };
                uint32_t codes[2];
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
                        make_float2(qdiv(y[4 * k]), qdiv(y[4 * k + 1])), __NV_SATFINITE, __NV_E4M3);
                    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
                        make_float2(qdiv(y[4 * k + 2]), qdiv(y[4 * k + 3])), __NV_SATFINITE, __NV_E4M3);
                    codes[k] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
                }
                uint8_t* d8 = static_cast<uint8_t*>(dst) + dst_elem;
                *reinterpret_cast<uint32_t*>(d8) = codes[0];        // dims [4k, 4k+4)
                *reinterpret_cast<uint32_t*>(d8 + 64) = codes[1];   // dims [64+4k, 64+4k+4)
                if (hl == 0) *scale_dst = scale;
            } else {
                __nv_bfloat16* d16 = static_cast<__nv_bfloat16*>(dst) + dst_elem;
                *reinterpret_cast<uint2*>(d16) = make_uint2(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]));
                *reinterpret_cast<uint2*>(d16 + 64) = make_uint2(pack_bf16x2(y[4], y[5]), pack_bf16x2(y[6], y[7]));
            }
        }
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
    if (a.num_tokens == 0) return cudaSuccess;
    // Few tokens (decode): one round of 16 rows per block, so that a token's
    // rows spread over several blocks; many tokens (prefill): a block per token.
    const int rounds = (a.num_q_heads + 2 * a.num_kv_heads + kRowsPerRound - 1) / kRowsPerRound;
    p.rounds_per_block = (long long)a.num_tokens * rounds < 8LL * 152 ? 1 : rounds;
    const unsigned splits = (unsigned)((rounds + p.rounds_per_block - 1) / p.rounds_per_block);
    const dim3 grid((unsigned)a.num_tokens, splits);
    if ((long long)a.num_tokens * splits >= 4LL * 152 * 4) {
        if (!a.q_scale && !a.kv_fp8)
            return launch_pdl(rope_norm_kernel<5>, grid, dim3(kWarpsPerBlock * 32), 0, s, p);
        return launch_pdl(rope_norm_kernel<4>, grid, dim3(kWarpsPerBlock * 32), 0, s, p);
    }
    return launch_pdl(rope_norm_kernel<3>, grid, dim3(kWarpsPerBlock * 32), 0, s, p);
}

}  // namespace hpc
