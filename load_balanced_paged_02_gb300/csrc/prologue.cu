// Fused attention prologue (HPC-Ops/SGLang blog, "A fused attention
// prologue"; vLLM x HPC-Ops blog, "融合的注意力前奏", HpcRopeNorm): from the
// fused QKV projection output, RMS QK-norm then rotary embedding on every
// query and key head, the query written out (bf16, or e4m3 with one scale per
// token and head, the form hpc_decode_attn_q8 consumes), and K and V written
// straight into their page slots of the cache (bf16, or e4m3 with one scale
// per token and head). One pass over the QKV output; no intermediate tensors.
//
// Two kernels. Prefill-sized calls (at least two ring stages of whole tokens
// per SM, at most 160 rows per token) run the ring-fed persistent kernel
// below (namespace ring). Other calls, decode steps among them, run
// rope_norm_kernel: one block per token, or per round of rows of a token when
// there are few tokens.
//
// In rope_norm_kernel a half-warp owns one (token, head) row, lane k of the
// half owning dims [4k, 4k+4) and their rotation partners [64+4k, 64+4k+4)
// (two 8-byte loads and stores, each half-warp-wide access 128 contiguous
// bytes), so the rotary embedding needs no data from other lanes; a warp
// covers two rows per round and the block's 8 warps cover 16 rows per round;
// the five rounds of a Hy3 token (80 rows) are all loaded before any is
// processed, so a block waits on memory once. The token's position, slot and
// rotary row are loaded once per block, the norm weights per row from L1. The
// reductions (norm sum; e4m3 absolute max, only when a call writes e4m3) take
// four xor-shuffle steps inside the half-warp. Row kinds (query, key, value)
// are per-lane predicates, so all lanes run every shuffle.
#include <algorithm>
#include <atomic>

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

// ------------------------------------------------------------------ prefill-sized calls
//
// A persistent kernel fed by a ring of bulk copies. The QKV output of a token
// is one contiguous run of H3 rows of 256 bytes, so a stage holds G whole
// tokens (G * H3 <= 160 rows) and arrives with one bulk copy, plus each
// token's 512-byte rotary row. One CTA per SM: a producer warp streams the
// stages of its tokens into a 4-deep ring; 24 consumer warps (22 when the
// query is written as e4m3) process them.
// A consumer quarter-warp owns one row (lane k of it: dims [8k, 8k+8) and
// their rotation partners [64+8k, 64+8k+8)); a warp takes units of 4 rows,
// unit u of the CTA's i-th stage going to warp (i * units + u) mod warps, so the
// warps share the rows evenly over the stages. Reductions take three xor
// shuffles inside the quarter-warp. Bound: instruction issue and latency (ncu
// on the 16-warp version: issue slots 60 % busy, short-scoreboard stalls
// first, DRAM well below its peak). Packed f32x2 arithmetic for the norm,
// weights and rotation measured slower: it issues at half rate on GB300.
//
// e4m3 outputs. Query and key rows: the code of element k is the rounding of
// z_k * 448 / max|z|, where z is the weighted, rotated row before the norm
// factor inv is applied, and the stored scale is inv * max|z| / 448; code *
// scale is then inv * z_k, the normalised value, up to float32 rounding
// (these values carry float32 rounding anyway). Value rows are the bf16
// inputs themselves, which often sit exactly on e4m3 rounding midpoints, so
// their scale max|x| / 448 and quotients x / scale are correctly rounded
// (Markstein's correction step, see rope_norm_kernel).
namespace ring {

// Two instances. Calls that write a bf16 query: 24 consumer warps (on GB300
// an 8192-token prefill at 64/8 heads with bf16 outputs took 56.7 us with 16,
// 55.7 with 24, 56.0 with 28). Calls that write an e4m3 query: each lane keeps
// its 16 query norm weights in registers instead of loading them from shared
// memory for every query row (each row needs 128 bytes per lane of weights and
// rotary terms, four times its own data, and shared-memory wavefronts bound the
// e4m3 instance), which leaves room for 22 warps without spills: 59.0 -> 56.5
// us (e4m3 outputs; the bf16 instance lost 1.7 us with the same change).
template <bool QW>
struct RingCfg {
    static constexpr int kConsumerWarps = QW ? 22 : 24;
    static constexpr int kThreads = (kConsumerWarps + 1) * 32;
};
constexpr int kStages = 4;
constexpr int kStageRows = 160;   // QKV rows per stage at most
constexpr int kStageTokens = 16;  // tokens per stage at most
constexpr int kRowBytes = kHeadDim * 2;
constexpr int kRotBytes = kHeadDim * 4;
constexpr int kRowsOff = 0;
constexpr int kRotOff = kStageRows * kRowBytes;                // 40960
constexpr int kMetaOff = kRotOff + kStageTokens * kRotBytes;   // + 8192
constexpr int kStageBytes = kMetaOff + kStageTokens * 8;       // + 128
constexpr int kWeightsOff = kStages * kStageBytes;
constexpr int kBarOff = kWeightsOff + 2 * kHeadDim * 4;
constexpr int kFlagOff = kBarOff + 2 * kStages * 8;
constexpr int kSmemBytes = kFlagOff + 16;
static_assert(kStageBytes % 16 == 0 && kRotOff % 16 == 0 && kWeightsOff % 16 == 0, "bulk-copy alignment");
static_assert(kSmemBytes <= 232448, "over the shared-memory limit of a CTA");
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint64_t kDrainLimitNs = 200000000ull;
constexpr float kInv448 = 1.f / 448.f;  // RN(1/448), the reciprocal Markstein's step needs

struct RingParams {
    PrologueParams p;
    int G;          // tokens per stage
    int H3;         // rows per token
    uint32_t h3_magic;  // ceil(2^32 / H3): r / H3 = umulhi(r, h3_magic) for r < 2^16
    int num_stages;     // ceil(T / G)
};

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                             uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15) == 0) {
            if (abort_flag && *abort_flag) return false;
            if (global_timer_ns() - t0 > limit_ns) return false;
        }
    }
}

// Reductions inside one quarter-warp (mask: its 8 lanes). Each quarter-warp
// owns its own row and may skip it (a padding token's K/V, a row past the
// stage's end) while the others reduce, so the masks name only the quarter.
__device__ __forceinline__ float quarter_sum(float v, uint32_t mask) {
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) v += __shfl_xor_sync(mask, v, off);
    return v;
}

__device__ __forceinline__ float quarter_max(float v, uint32_t mask) {
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(mask, v, off));
    return v;
}

__device__ __forceinline__ void unpack16(const uint4& a, const uint4& b, float (&y)[16]) {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        y[2 * k] = __uint_as_float(w[k] << 16);
        y[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
}

// Packed single precision (two float32 per 64-bit register, one issue slot for
// both; each half rounds as the scalar instruction would): r = a * b and
// r = a * b + c on the pairs (a0, a1), (b0, b1), (c0, c1).
__device__ __forceinline__ void mul2(float& r0, float& r1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "mul.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(r0), "=f"(r1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

__device__ __forceinline__ void fma2(float& r0, float& r1, float a0, float a1, float b0, float b1, float c0,
                                     float c1) {
    asm("{\n\t.reg .b64 a, b, c, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "mov.b64 c, {%6, %7};\n\tfma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(r0), "=f"(r1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

__device__ __forceinline__ float4 lds_f4(uint32_t addr) {
    const uint4 v = lds128(addr);
    return make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z), __uint_as_float(v.w));
}

// Eight e4m3 codes of v[0..7] (rounded to nearest, saturated), packed low byte first.
__device__ __forceinline__ uint2 e4m3x8(const float* v) {
    uint32_t w[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const __nv_fp8x2_storage_t lo =
            __nv_cvt_float2_to_fp8x2(make_float2(v[4 * h], v[4 * h + 1]), __NV_SATFINITE, __NV_E4M3);
        const __nv_fp8x2_storage_t hi =
            __nv_cvt_float2_to_fp8x2(make_float2(v[4 * h + 2], v[4 * h + 3]), __NV_SATFINITE, __NV_E4M3);
        w[h] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
    }
    return make_uint2(w[0], w[1]);
}

template <bool QW>
__global__ void __launch_bounds__(RingCfg<QW>::kThreads, 1) rope_norm_ring_kernel(const RingParams rp) {
    constexpr int kConsumerWarps = RingCfg<QW>::kConsumerWarps;
    const PrologueParams& p = rp.p;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOff);
    uint64_t* empty = full + kStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kFlagOff);
    float* wsm = reinterpret_cast<float*>(smem + kWeightsOff);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    grid_dependency_wait();  // the QKV projection (and any input) may still be finishing
    grid_launch_dependents();
    if (threadIdx.x < 2 * kHeadDim / 4) {  // the norm weights, into shared memory
        const float* src = threadIdx.x < kHeadDim / 4 ? p.qw + 4 * threadIdx.x : p.kw + 4 * (threadIdx.x - 32);
        *reinterpret_cast<float4*>(wsm + 4 * threadIdx.x) = __ldg(reinterpret_cast<const float4*>(src));
    }
    __syncthreads();
    const int H3 = rp.H3, G = rp.G;
    const int rows_per_stage = G * H3;
    const int units = (rows_per_stage + 3) >> 2;

    if (warp == kConsumerWarps) {
        // ================================ producer
        const uint64_t pol = l2_evict_first_policy();
        uint32_t i = 0;
        bool ok = true;
        int k = blockIdx.x;
        // position and slot of this lane's token of stage k, loaded one stage ahead
        int npos = 0, nslot = -1;
        if (k < rp.num_stages && lane < G && k * G + lane < p.T) {
            npos = __ldg(p.pos + k * G + lane);
            nslot = __ldg(p.slots + k * G + lane);
        }
        for (; k < rp.num_stages; k += gridDim.x, ++i) {
            const int t0 = k * G;
            const int n = min(G, p.T - t0);
            const int pos = npos, slot = nslot;
            const int kn = k + gridDim.x;
            if (kn < rp.num_stages && lane < G && kn * G + lane < p.T) {
                npos = __ldg(p.pos + kn * G + lane);
                nslot = __ldg(p.slots + kn * G + lane);
            }
            const int st = (int)(i % kStages);
            if (lane == 0) ok = wait_bounded(&empty[st], ((i / kStages) & 1) ^ 1, abort_flag, kWaitLimitNs);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            uint8_t* stage = smem + (size_t)st * kStageBytes;
            const bool mine = lane < n;
            const bool rotate = mine && pos >= 0 && pos < p.max_pos;
            const bool slot_ok = slot >= 0 && slot / kChunk < p.num_pages;
            if (mine) {
                reinterpret_cast<int2*>(stage + kMetaOff)[lane] = make_int2(rotate ? pos : -1, slot_ok ? slot : -1);
                if (p.err && !rotate) atomicOr(p.err, (int)HPC_DEVERR_BAD_POSITION);
                if (p.err && slot >= 0 && !slot_ok) atomicOr(p.err, (int)HPC_DEVERR_PAGE_OUT_OF_RANGE);
            }
            const uint32_t nrot = __popc(__ballot_sync(0xffffffffu, rotate));
            const uint32_t bytes = (uint32_t)n * H3 * kRowBytes;
            __syncwarp();
            if (lane == 0) {
                mbar_arrive_expect_tx(&full[st], bytes + nrot * kRotBytes);
                bulk_load(stage + kRowsOff, p.qkv + (size_t)t0 * H3 * kHeadDim, bytes, &full[st], pol);
            }
            __syncwarp();
            if (rotate)
                bulk_load_nohint(stage + kRotOff + lane * kRotBytes, p.cos_sin + (size_t)pos * kHeadDim, kRotBytes,
                                 &full[st]);
        }
        if (!ok && lane == 0) {
            *abort_flag = 1;
            if (p.err) atomicOr(p.err, (int)HPC_DEVERR_WAIT_TIMEOUT);
        }
        // every copy lands before the CTA may exit (the consumers may have left)
        if (lane == 0) {
            const uint32_t first = i > (uint32_t)kStages ? i - kStages : 0u;
            for (uint32_t j = first; j < i; ++j)
                wait_bounded(&full[j % kStages], (j / kStages) & 1, nullptr, kDrainLimitNs);
        }
        return;
    }

    // ================================ consumers
    const int q = lane >> 3, hl = lane & 7;
    const uint32_t qmask = 0xffu << (lane & 24);
    const bool q_fp8 = p.q_scale != nullptr, kv_fp8 = p.kv_fp8 != 0;
    float wq[16];
    if constexpr (QW) {
        const uint32_t wb = smem_u32(wsm + 8 * hl);
        const float4 w0 = lds_f4(wb), w1 = lds_f4(wb + 16), w2 = lds_f4(wb + 256), w3 = lds_f4(wb + 272);
        const float ww[16] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w,
                              w2.x, w2.y, w2.z, w2.w, w3.x, w3.y, w3.z, w3.w};
#pragma unroll
        for (int e = 0; e < 16; ++e) wq[e] = ww[e];
    }
    uint32_t i = 0;
    for (int k = blockIdx.x; k < rp.num_stages; k += gridDim.x, ++i) {
        const int st = (int)(i % kStages);
        if (!wait_bounded(&full[st], (i / kStages) & 1, abort_flag, kWaitLimitNs)) {
            if (lane == 0) {
                *abort_flag = 1;
                if (p.err) atomicOr(p.err, (int)HPC_DEVERR_WAIT_TIMEOUT);
            }
            return;
        }
        const uint8_t* stage = smem + (size_t)st * kStageBytes;
        const uint32_t sbase = smem_u32(stage);
        const int t0 = k * G;
        const int n_rows = min(G, p.T - t0) * H3;
        // this warp's first unit of the stage, then every kConsumerWarps-th
        int u = (int)(((uint32_t)warp + kConsumerWarps - (i * (uint32_t)units) % kConsumerWarps) % kConsumerWarps);
        for (; u < units; u += kConsumerWarps) {
            const int r = 4 * u + q;
            if (r >= n_rows) continue;  // quarter-warps of a row past the stage's end
            const int tl = (int)__umulhi((uint32_t)r, rp.h3_magic);
            const int j = r - tl * H3;
            const int t = t0 + tl;
            const int2 meta = reinterpret_cast<const int2*>(stage + kMetaOff)[tl];
            const bool is_q = j < p.Hq, is_qk = j < p.Hq + p.Hkv;
            if (!is_q && meta.y < 0) continue;  // K/V of a padding token (or a bad slot)
            const uint32_t row = sbase + kRowsOff + (uint32_t)r * kRowBytes + 16u * hl;
            float y[16];
            unpack16(lds128(row), lds128(row + 128), y);
            const bool fp8_row = is_q ? q_fp8 : kv_fp8;
            float inv = 1.f;
            if (is_qk) {
                const uint32_t wb = smem_u32(wsm + (is_q ? 0 : kHeadDim) + 8 * hl);
                const uint32_t cb = sbase + kRotOff + (uint32_t)tl * kRotBytes + 32u * hl;
                float s2 = 0.f;
                if constexpr (QW) {
                    // two interleaved partial sums on the packed pipe
                    float sa = 0.f, sb = 0.f;
#pragma unroll
                    for (int e = 0; e < 16; e += 2) fma2(sa, sb, y[e], y[e + 1], y[e], y[e + 1], sa, sb);
                    s2 = sa + sb;
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) s2 = fmaf(y[e], y[e], s2);
                }
                s2 = quarter_sum(s2, qmask);
                inv = rsqrtf(s2 * (1.f / kHeadDim) + p.eps);
                if (QW && is_q) {
#pragma unroll
                    for (int e = 0; e < 16; e += 2) mul2(y[e], y[e + 1], y[e], y[e + 1], wq[e], wq[e + 1]);
                } else {
                    const float4 w0 = lds_f4(wb), w1 = lds_f4(wb + 16), w2 = lds_f4(wb + 256), w3 = lds_f4(wb + 272);
                    const float ww[16] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w,
                                          w2.x, w2.y, w2.z, w2.w, w3.x, w3.y, w3.z, w3.w};
                    if constexpr (QW) {
#pragma unroll
                        for (int e = 0; e < 16; e += 2) mul2(y[e], y[e + 1], y[e], y[e + 1], ww[e], ww[e + 1]);
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e) y[e] *= ww[e];
                    }
                }
                if (meta.x >= 0) {
                    // rotary pairs (i, i + 64), both in this lane: y[e] and y[e + 8]
                    const float4 c0 = lds_f4(cb), c1 = lds_f4(cb + 16), s0 = lds_f4(cb + 256), s1 = lds_f4(cb + 272);
                    const float cc[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                    const float ss[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
                    if constexpr (QW) {
                        // the same roundings as below: a c - RN(b s) and b c + RN(a s)
#pragma unroll
                        for (int e = 0; e < 8; e += 2) {
                            const float a0 = y[e], a1 = y[e + 1], b0 = y[e + 8], b1 = y[e + 9];
                            float ns0, ns1, nbs0, nbs1, as0, as1;
                            mul2(ns0, ns1, ss[e], ss[e + 1], -1.f, -1.f);
                            mul2(nbs0, nbs1, b0, b1, ns0, ns1);
                            mul2(as0, as1, a0, a1, ss[e], ss[e + 1]);
                            fma2(y[e], y[e + 1], a0, a1, cc[e], cc[e + 1], nbs0, nbs1);
                            fma2(y[e + 8], y[e + 9], b0, b1, cc[e], cc[e + 1], as0, as1);
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float a = y[e], b = y[e + 8];
                            y[e] = fmaf(a, cc[e], -b * ss[e]);
                            y[e + 8] = fmaf(b, cc[e], a * ss[e]);
                        }
                    }
                }
            }
            // destination of the row
            size_t dst_elem;
            void* dst;
            float* scale_dst = nullptr;
            if (is_q) {
                const size_t qrow = (size_t)t * p.Hq + j;
                dst_elem = qrow * kHeadDim + 8 * hl;
                dst = p.q_out;
                if (q_fp8) scale_dst = p.q_scale + qrow;
            } else {
                const int h = is_qk ? j - p.Hq : j - p.Hq - p.Hkv;
                const int page = meta.y >> 6, off = meta.y & (kChunk - 1);
                dst_elem = (((size_t)page * kChunk + off) * p.Hkv + h) * kHeadDim + 8 * hl;
                dst = is_qk ? p.k_cache : p.v_cache;
                if (kv_fp8) scale_dst = (is_qk ? p.k_scale : p.v_scale) + ((size_t)page * p.Hkv + h) * kChunk + off;
            }
            if (fp8_row) {
                float am = 0.f;
#pragma unroll
                for (int e = 0; e < 16; ++e) am = fmaxf(am, fabsf(y[e]));
                am = quarter_max(am, qmask);
                float scale;
                if (is_qk) {
                    // z * (448 / max|z|), scale inv * max|z| / 448
                    const float rz = am > 0.f ? __fdividef(448.f, am) : 0.f;
                    scale = am > 0.f ? inv * am * kInv448 : 1.f;
                    if constexpr (QW) {
#pragma unroll
                        for (int e = 0; e < 16; e += 2) mul2(y[e], y[e + 1], y[e], y[e + 1], rz, rz);
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e) y[e] *= rz;
                    }
                } else {
                    // correctly rounded max|x| / 448 and x / scale
                    const float q0 = am * kInv448;
                    scale = am > 0.f ? fmaf(fmaf(-q0, 448.f, am), kInv448, q0) : 1.f;
                    const float rcp = __frcp_rn(scale);
                    if constexpr (QW) {
                        const float ns = -scale;
#pragma unroll
                        for (int e = 0; e < 16; e += 2) {
                            float q0, q1, r0, r1;
                            mul2(q0, q1, y[e], y[e + 1], rcp, rcp);
                            fma2(r0, r1, q0, q1, ns, ns, y[e], y[e + 1]);
                            fma2(y[e], y[e + 1], r0, r1, rcp, rcp, q0, q1);
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const float qq = y[e] * rcp;
                            y[e] = fmaf(fmaf(-qq, scale, y[e]), rcp, qq);
                        }
                    }
                }
                uint8_t* d8 = static_cast<uint8_t*>(dst) + dst_elem;
                *reinterpret_cast<uint2*>(d8) = e4m3x8(y);           // dims [8k, 8k+8)
                *reinterpret_cast<uint2*>(d8 + 64) = e4m3x8(y + 8);  // dims [64+8k, 64+8k+8)
                if (hl == 0) *scale_dst = scale;
            } else {
                __nv_bfloat16* d16 = static_cast<__nv_bfloat16*>(dst) + dst_elem;
                uint32_t w[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) w[e] = pack_bf16x2(y[2 * e] * inv, y[2 * e + 1] * inv);
                *reinterpret_cast<uint4*>(d16) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4*>(d16 + 64) = make_uint4(w[4], w[5], w[6], w[7]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }
}

}  // namespace ring

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
    const int H3 = a.num_q_heads + 2 * a.num_kv_heads;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
        sms = 0;
    // Prefill-sized calls whose tokens fit the ring's stages: the persistent
    // ring kernel, when there are at least two stages per SM.
    if (H3 <= ring::kStageRows && sms > 0) {
        ring::RingParams rp;
        rp.p = p;
        rp.H3 = H3;
        rp.G = std::min(ring::kStageTokens, ring::kStageRows / H3);
        rp.num_stages = (a.num_tokens + rp.G - 1) / rp.G;
        rp.h3_magic = (uint32_t)((0x100000000ull + H3 - 1) / H3);
        if (rp.num_stages >= 2 * sms) {
            // the shared-memory opt-in, once per device (the launch path then makes
            // no extra runtime calls, which keeps it capturable)
            static std::atomic<unsigned long long> attr_set{0};
            const unsigned long long bit = 1ull << (dev & 63);
            if (!(attr_set.load(std::memory_order_acquire) & bit)) {
                for (const void* fn : {(const void*)ring::rope_norm_ring_kernel<false>,
                                       (const void*)ring::rope_norm_ring_kernel<true>}) {
                    cudaError_t e =
                        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, ring::kSmemBytes);
                    if (e != cudaSuccess) return e;
                }
                attr_set.fetch_or(bit, std::memory_order_acq_rel);
            }
            const int grid = std::min(rp.num_stages, sms);
            if (a.q_scale)
                return launch_pdl(ring::rope_norm_ring_kernel<true>, dim3(grid), dim3(ring::RingCfg<true>::kThreads),
                                  ring::kSmemBytes, s, rp);
            return launch_pdl(ring::rope_norm_ring_kernel<false>, dim3(grid), dim3(ring::RingCfg<false>::kThreads),
                              ring::kSmemBytes, s, rp);
        }
    }
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
