// Persistent paged GQA decode attention (compute stage of the load-balanced
// scheduler: HPC-Ops/SGLang blog, "Scheduling around live KV work", the
// paragraph on execution; vLLM x HPC-Ops blog, "解决方案：按步负载均衡的
// decode 调度器", compute-and-combine stage).
//
// CTA j drains its task list: for every descriptor (kv head h, request b,
// chunks [c0, c1), split s) it computes, for the 8 query heads of h, softmax
// attention over tokens [64*c0, min(64*c1, L_b)) and writes the normalised
// partial output and its natural-log LSE to row s of the split buffers.
//
// Block = NG*4 consumer warps + 1 producer warp.
//  * Producer warp: walks the same list; its lanes fetch 32 page ids at a
//    time, lane 0 streams each 64-token chunk (= one page) of K and V into a
//    STAGES-deep shared-memory ring with TMA (3-D tensor maps over
//    [pages*64, Hkv, 128], 128-byte swizzle, L2 evict-first; e4m3 adds the two
//    256-byte scale rows of the page through 2-D maps over [pages*Hkv, 64])
//    and the Q rows of each descriptor (2 KB bulk copy) into a 2-slot ring. mbarrier full/empty
//    pairs hand stages over; a per-stage word carries the chunk's valid token
//    count (0 = skip: page id out of range).
//  * Consumer warps: group gi takes the chunks whose running index is gi mod
//    NG; inside a chunk warp w takes tokens [16w, 16w+16). Tokens are the M
//    dimension of mma.m16n8k16 and the GQA group of 8 query heads is N, so
//    S^T = K Q^T and O^T += V^T P^T need no padding: the S^T accumulator is
//    turned into the P^T operand by movmatrix.trans. Each warp keeps its own
//    online-softmax state (log2 domain) and the warps' states are merged
//    through shared memory at the end of each descriptor.
//  * e4m3 caches: codes are widened exactly to f16 (Q to f16 once per
//    descriptor). K scales multiply the score rows; V scales (x256, undone at
//    the end) fold into P. The k index of S^T and the m index of O^T are
//    permuted so that each thread reads whole 16-byte rows without bank
//    conflicts; the permutation is undone when the merge writes dims back.
// Every wait is bounded (2 s by %globaltimer); on expiry the CTA records
// HPC_DEVERR_WAIT_TIMEOUT, the producer waits (bounded) for its copies in
// flight, and the CTA returns. HPC_ATTN_TEST_WAIT_EXPIRY makes the consumers
// take that path on purpose, for tests of it.
#include <atomic>
#include <cstring>
#include <mutex>

#include "attn_common.cuh"

namespace hpc {
namespace {

using namespace attn;

// one query slot: 8 bf16 rows at the padded pitch (the larger of the two forms;
// e4m3: 8 code rows at their pitch, then 8 float32 scales)
constexpr int kQSlotBytes = kGroup * kQPitchBf16;
static_assert(kQScaleOffE4m3 + kGroup * 4 <= kQSlotBytes, "query slot");
template <bool FP8, int STAGES, int NG>
struct Layout {
    // Chunk k goes to group k % NG and to stage k % STAGES. With STAGES a
    // multiple of NG every stage always belongs to the same group, so a group
    // never waits on a stage lap that another group has not finished (which
    // would alias the mbarrier phase parity).
    static_assert(STAGES % NG == 0, "stage ring must be a multiple of the consumer groups");
    static constexpr int kNCW = NG * 4;
    static constexpr size_t kQ = (size_t)STAGES * KvCfg<FP8>::kStageBytes;
    // merge scratch and (m, l) words, two buffers: descriptor n uses buffer n % 2,
    // so one barrier per descriptor orders the writes of n + 2 after the reads of n
    static constexpr size_t kScratchFloats = (size_t)kNCW * kGroup * kScratchStride;
    static constexpr size_t kScratch = kQ + 2 * kQSlotBytes;
    static constexpr size_t kML = kScratch + 2 * kScratchFloats * 4;
    static constexpr size_t kMeta = kML + 2 * (size_t)kNCW * kGroup * 8;
    static constexpr size_t kSink = kMeta + STAGES * 4;  // one word per consumer warp
    static constexpr size_t kBars = (kSink + kNCW * 4 + 7) / 8 * 8;
    static constexpr int kNumBars = 2 * STAGES + 6;  // full, empty, qfull x2, qempty x2, merge, unset
    static constexpr size_t kFlag = kBars + kNumBars * 8;
    static constexpr size_t kTotal = kFlag + 16;
    static constexpr size_t kAlloc = kTotal + 1024;  // base is rounded up to 1 KB (128B swizzle)
    static constexpr int kThreads = (kNCW + 1) * 32;
    static_assert(kAlloc <= 232448, "over the 227 KB shared-memory limit of a CTA");
};

template <bool FP8, bool QF8>
__device__ __forceinline__ void chunk_compute(uint8_t* stage, int wq, int lane, int nv,
                                              const uint32_t (&qf)[8][2], const float (&qsc)[2],
                                              float (&o)[8][4], float (&m)[2], float (&l)[2],
                                              float scale_log2, int ks_off) {
    const int g = lane >> 2, c = lane & 3;
    const uint32_t sb = smem_u32(stage);
    float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
    float s[4], p[4];
    if (nv < 16) zero_v_tail<FP8>(stage, wq, nv, lane);

    if constexpr (!FP8) {
        // ---- S^T = K Q^T over 8 k-steps of 16 dims (two independent chains)
        const int rr = lane & 7;
        const uint32_t krow = sb + (uint32_t)(16 * wq + ((lane >> 3) & 1) * 8 + rr) * 128u;
        const uint32_t kx = (uint32_t)((lane >> 4) ^ rr);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            uint32_t a[4];
            ldsm_x4(a, krow + (uint32_t)(ks >> 2) * 8192u + (((uint32_t)(2 * (ks & 3)) ^ kx) << 4));
            if (ks & 1)
                mma_bf16(acc1, a, qf[ks][0], qf[ks][1]);
            else
                mma_bf16(acc0, a, qf[ks][0], qf[ks][1]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) s[i] = (acc0[i] + acc1[i]) * scale_log2;
        if (nv < 16) {
            if (g >= nv) s[0] = s[1] = kNegInf;
            if (g + 8 >= nv) s[2] = s[3] = kNegInf;
        }
        softmax_step(s, m, l, o, p);
        const uint32_t pb0 = movmatrix_t(pack_bf16x2(p[0], p[1]));
        const uint32_t pb1 = movmatrix_t(pack_bf16x2(p[2], p[3]));
        // ---- O^T += V^T P^T, 8 m-tiles of 16 dims
        const uint32_t vrow = sb + 16384u + (uint32_t)(16 * wq + (lane >> 4) * 8 + rr) * 128u;
        const uint32_t vx = (uint32_t)(((lane >> 3) & 1) ^ rr);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint32_t a[4];
            ldsm_x4_t(a, vrow + (uint32_t)(i >> 2) * 8192u + (((uint32_t)(2 * (i & 3)) ^ vx) << 4));
            mma_bf16(o[i], a, pb0, pb1);
        }
    } else {
        const float* ksc = reinterpret_cast<const float*>(stage + 16384) + ks_off;
        const float* vsc = reinterpret_cast<const float*>(stage + 16384) + (kChunk - ks_off);
        const int r0 = 16 * wq + g;
        const uint32_t kb = sb;
        // ---- S^T: thread reads dims [32c, 32c+32) of token rows r0 and r0+8
        const uint4 k00 = lds128(kb + (uint32_t)r0 * 128u + ((uint32_t)((2 * c) ^ g) << 4));
        const uint4 k01 = lds128(kb + (uint32_t)r0 * 128u + ((uint32_t)((2 * c + 1) ^ g) << 4));
        const uint4 k10 = lds128(kb + (uint32_t)(r0 + 8) * 128u + ((uint32_t)((2 * c) ^ g) << 4));
        const uint4 k11 = lds128(kb + (uint32_t)(r0 + 8) * 128u + ((uint32_t)((2 * c + 1) ^ g) << 4));
        const uint32_t w0[8] = {k00.x, k00.y, k00.z, k00.w, k01.x, k01.y, k01.z, k01.w};
        const uint32_t w1[8] = {k10.x, k10.y, k10.z, k10.w, k11.x, k11.y, k11.z, k11.w};
        // K widened exactly to f16 (a bf16 query was rounded to f16, an e4m3 one
        // widened exactly, in load_q_frags)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            uint32_t a[4];
            e4m3x4_to_f16x2x2(w0[ks], a[0], a[2]);
            e4m3x4_to_f16x2x2(w1[ks], a[1], a[3]);
            if (ks & 1)
                mma_f16(acc1, a, qf[ks][0], qf[ks][1]);
            else
                mma_f16(acc0, a, qf[ks][0], qf[ks][1]);
        }
        const float ks0 = ksc[r0] * scale_log2, ks1 = ksc[r0 + 8] * scale_log2;
        // score columns 2c and 2c+1 are query heads 2c, 2c+1 (their Q scales)
        s[0] = (acc0[0] + acc1[0]) * ks0 * qsc[0];
        s[1] = (acc0[1] + acc1[1]) * ks0 * qsc[1];
        s[2] = (acc0[2] + acc1[2]) * ks1 * qsc[0];
        s[3] = (acc0[3] + acc1[3]) * ks1 * qsc[1];
        const bool v0 = g < nv, v1 = g + 8 < nv;
        if (!v0) s[0] = s[1] = kNegInf;
        if (!v1) s[2] = s[3] = kNegInf;
        softmax_step(s, m, l, o, p);
        const float vs0 = v0 ? vsc[r0] * KvCfg<true>::kPScale : 0.f;
        const float vs1 = v1 ? vsc[r0 + 8] * KvCfg<true>::kPScale : 0.f;
        const uint32_t pb0 = movmatrix_t(pack_f16x2(v0 ? p[0] * vs0 : 0.f, v0 ? p[1] * vs0 : 0.f));
        const uint32_t pb1 = movmatrix_t(pack_f16x2(v1 ? p[2] * vs1 : 0.f, v1 ? p[3] * vs1 : 0.f));
        // ---- O^T += V^T P^T: thread reads the 16-byte column g of token rows
        // 2c, 2c+1, 2c+8, 2c+9; m-tile i row g is dim 16g+2i, row g+8 is 16g+2i+1
        const uint32_t vb = sb + 8192u;
        const int t0 = 16 * wq + 2 * c;
        const uint4 R0 = lds128(vb + (uint32_t)t0 * 128u + ((uint32_t)(g ^ (2 * c)) << 4));
        const uint4 R1 = lds128(vb + (uint32_t)(t0 + 1) * 128u + ((uint32_t)(g ^ (2 * c + 1)) << 4));
        const uint4 R2 = lds128(vb + (uint32_t)(t0 + 8) * 128u + ((uint32_t)(g ^ (2 * c)) << 4));
        const uint4 R3 = lds128(vb + (uint32_t)(t0 + 9) * 128u + ((uint32_t)(g ^ (2 * c + 1)) << 4));
        const uint32_t x0[4] = {R0.x, R0.y, R0.z, R0.w}, x1[4] = {R1.x, R1.y, R1.z, R1.w};
        const uint32_t x2[4] = {R2.x, R2.y, R2.z, R2.w}, x3[4] = {R3.x, R3.y, R3.z, R3.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t sel = (i & 1) ? 0x7362u : 0x5140u;
            const uint32_t u = prmt(x0[i >> 1], x1[i >> 1], sel);
            const uint32_t v = prmt(x2[i >> 1], x3[i >> 1], sel);
            uint32_t a[4];
            e4m3x4_to_f16x2x2(u, a[0], a[1]);
            e4m3x4_to_f16x2x2(v, a[2], a[3]);
            mma_f16(o[i], a, pb0, pb1);
        }
    }
    if (nv < 16) fence_proxy_async_smem();  // generic zero-fill before the next TMA write
}

// ------------------------------------------------------------------ kernel

template <bool FP8, bool QF8, int STAGES, int NG>
__global__ void __launch_bounds__(Layout<FP8, STAGES, NG>::kThreads, 1)
    decode_attn_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_ks, const __grid_constant__ CUtensorMap tm_vs,
                       const Params p) {
    static_assert(FP8 || !QF8, "an e4m3 query needs the e4m3 cache");
    using LY = Layout<FP8, STAGES, NG>;
    using Cfg = KvCfg<FP8>;
    constexpr int NCW = LY::kNCW;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + LY::kBars);
    uint64_t* empty = full + STAGES;
    uint64_t* qfull = empty + STAGES;
    uint64_t* qempty = qfull + 2;
    uint64_t* merge_bar = qempty + 2;
    uint64_t* unset_bar = merge_bar + 1;  // never completed (failure-path test)
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + LY::kFlag);
    volatile int* meta = reinterpret_cast<volatile int*>(smem + LY::kMeta);
    uint8_t* qbuf = smem + LY::kQ;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 4);  // a stage is consumed by the 4 warps of one group
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&qfull[i], 1);
            mbar_init(&qempty[i], NCW);
        }
        mbar_init(merge_bar, NCW);  // one arrival per consumer warp (lane 0, after __syncwarp)
        mbar_init(unset_bar, 1);    // nothing arrives on it
        *abort_flag = 0;
        fence_mbar_init();
    }
    // Everything above overlaps the predecessor's tail. The task map, lengths
    // and Q may come from earlier kernels: every warp waits for them here but
    // the producer, which waits inside produce() (after its early loads, when
    // the caller allows them). Each thread releases the next kernel only after
    // its own wait.
    __syncthreads();

    if (warp == NCW) {
        produce<FP8, STAGES, QF8 ? QStage::kE4m3 : QStage::kBf16>(p, &tm_k, &tm_v, &tm_ks, &tm_vs, lane, smem,
                                                                  qbuf, kQSlotBytes, full, empty, qfull, qempty,
                                                                  meta, abort_flag);
        return;
    }
    grid_dependency_wait();
    grid_launch_dependents();

    // ================================ consumer warps
    const int gi = warp >> 2, wq = warp & 3;
    const int g = lane >> 2, c = lane & 3;
    float* scratch = reinterpret_cast<float*>(smem + LY::kScratch);
    float2* ml = reinterpret_cast<float2*>(smem + LY::kML);
    volatile uint32_t* q_sink = reinterpret_cast<volatile uint32_t*>(smem + LY::kSink);
    uint32_t seq = 0, mphase = 0;
    int qd = 0;
    // Failure-path test: a wait on a barrier that nothing completes runs out
    // after kTestWaitLimitNs, and the CTA leaves through its timeout path
    // (the producer then drains its copies in flight).
    if (p.test_wait_expiry && !wait_bounded(unset_bar, 0, abort_flag, kTestWaitLimitNs)) goto timeout;
    TaskAhead tw;
    tw.start(p, p.cta_off[blockIdx.x]);
    for (;;) {
        const int h = tw.t0.x, b = tw.t0.y, c0 = tw.t0.z, c1 = tw.t0.w, s = tw.s;
        if (h < 0) break;
        tw.next(p);
        if (!desc_ok(p, h, b, c0, c1, s)) continue;

        uint32_t qf[8][2];
        const int qs = qd & 1;
        if (!wait_bounded(&qfull[qs], (qd >> 1) & 1, abort_flag, kWaitLimitNs)) goto timeout;
        load_q_frags<FP8, QF8, QF8 ? kQPitchE4m3 : kQPitchBf16>(smem_u32(qbuf + qs * kQSlotBytes), lane, qf);
        float qsc[2] = {1.f, 1.f};
        if constexpr (QF8) {
            const float* qs_smem = reinterpret_cast<const float*>(qbuf + qs * kQSlotBytes + kQScaleOffE4m3);
            qsc[0] = qs_smem[2 * c];
            qsc[1] = qs_smem[2 * c + 1];
        }
        {
            // The slot may be refilled by TMA as soon as it is released, so the
            // release must wait until the fragment loads have returned: fold
            // every fragment word into a value that a store consumes first.
            uint32_t x = __float_as_uint(qsc[0]) ^ __float_as_uint(qsc[1]);
#pragma unroll
            for (int i = 0; i < 8; ++i) x ^= qf[i][0] ^ qf[i][1];
            __syncwarp();
            if (lane == 0) {
                q_sink[warp] = x;
                mbar_arrive(&qempty[qs]);
            }
        }
        ++qd;

        {
            float o[8][4];
#pragma unroll
            for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
            float m[2] = {kNegInf, kNegInf}, l[2] = {0.f, 0.f};

            for (int cc = c0; cc < c1; ++cc, ++seq) {
                if (NG > 1 && (int)(seq % NG) != gi) continue;
                const int st = (int)(seq % STAGES);
                if (!wait_bounded(&full[st], (seq / STAGES) & 1, abort_flag, kWaitLimitNs)) goto timeout;
                const int nv = meta[st] - 16 * wq;
                if (nv > 0)
                    chunk_compute<FP8, QF8>(smem + (size_t)st * Cfg::kStageBytes, wq, lane, nv < 16 ? nv : 16,
                                            qf, qsc, o, m, l, p.scale_log2, p.ks_off);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[st]);
            }

            // ---- merge the NCW warps' states of this descriptor (buffer mphase % 2;
            // every warp read buffer mphase % 2 of two descriptors back before it
            // arrived on the previous merge barrier, which this warp has passed)
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                l[0] += __shfl_xor_sync(0xffffffffu, l[0], off);
                l[1] += __shfl_xor_sync(0xffffffffu, l[1], off);
            }
            float* scr = scratch + (mphase & 1) * LY::kScratchFloats + warp * kGroup * kScratchStride;
            float2* mlw = ml + (mphase & 1) * (NCW * kGroup);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if constexpr (FP8) {
                    const int d = 16 * g + 2 * i;
                    *reinterpret_cast<float2*>(scr + (2 * c) * kScratchStride + d) = make_float2(o[i][0], o[i][2]);
                    *reinterpret_cast<float2*>(scr + (2 * c + 1) * kScratchStride + d) =
                        make_float2(o[i][1], o[i][3]);
                } else {
                    const int d = 16 * i + g;
                    scr[(2 * c) * kScratchStride + d] = o[i][0];
                    scr[(2 * c + 1) * kScratchStride + d] = o[i][1];
                    scr[(2 * c) * kScratchStride + d + 8] = o[i][2];
                    scr[(2 * c + 1) * kScratchStride + d + 8] = o[i][3];
                }
            }
            if (g == 0) {
                mlw[warp * kGroup + 2 * c] = make_float2(m[0], l[0]);
                mlw[warp * kGroup + 2 * c + 1] = make_float2(m[1], l[1]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(merge_bar);
        if (!wait_bounded(merge_bar, mphase & 1, abort_flag, kWaitLimitNs)) goto timeout;
        {
            const float* scr = scratch + (mphase & 1) * LY::kScratchFloats;
            const float2* mlr = ml + (mphase & 1) * (NCW * kGroup);
            const int ct = warp * 32 + lane;
            for (int idx = ct; idx < kGroup * 32; idx += NCW * 32) {
                const int qh = idx >> 5, d4 = idx & 31;
                float M = kNegInf;
#pragma unroll
                for (int w = 0; w < NCW; ++w) M = fmaxf(M, mlr[w * kGroup + qh].x);
                float lsum = 0.f;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                if (M != kNegInf) {
#pragma unroll
                    for (int w = 0; w < NCW; ++w) {
                        const float2 v = mlr[w * kGroup + qh];
                        const float f = fast_exp2(v.x - M);
                        lsum += v.y * f;
                        const float4 x = *reinterpret_cast<const float4*>(
                            scr + (w * kGroup + qh) * kScratchStride + 4 * d4);
                        acc.x += f * x.x;
                        acc.y += f * x.y;
                        acc.z += f * x.z;
                        acc.w += f * x.w;
                    }
                }
                const float inv = lsum > 0.f ? 1.f / (lsum * Cfg::kPScale) : 0.f;
                float4 r = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
                *reinterpret_cast<float4*>(p.split_o + ((long long)s * kGroup + qh) * kHeadDim + 4 * d4) = r;
                if (d4 == 0)
                    p.split_lse[(long long)s * kGroup + qh] = lsum > 0.f ? (M + __log2f(lsum)) * kLn2 : kNegInf;
            }
        }
        ++mphase;
    }
    return;
timeout:
    if (lane == 0) {
        *abort_flag = 1;
        atomicOr(p.err, (int)HPC_DEVERR_WAIT_TIMEOUT);
    }
}

// ------------------------------------------------------------------ host side

}  // namespace

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// 2-D map over a scale array [num_pages * Hkv rows][64 float32]; box = one
// 256-byte row (the 64 scales of one page and KV head).
bool make_scale_map(CUtensorMap* map, const float* base, int num_pages, int Hkv) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)kChunk, (cuuint64_t)num_pages * Hkv};
    cuuint64_t strides[1] = {kChunk * sizeof(float)};
    cuuint32_t box[2] = {(cuuint32_t)kChunk, 1u};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// One 3-D map over both scale arrays: [2 arrays at their distance][num_pages *
// Hkv rows][64 float32] from the lower array; box = one row of each (the lower
// array's first), so a page's two 256-byte scale rows land with one copy.
bool make_scale_maps(CUtensorMap* ks_map, CUtensorMap* vs_map, const float* k_scale, const float* v_scale,
                     int num_pages, int Hkv, int* pair, int* ks_off) {
    *pair = 0;
    *ks_off = 0;
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    const uintptr_t k = reinterpret_cast<uintptr_t>(k_scale), v = reinterpret_cast<uintptr_t>(v_scale);
    const bool k_low = k < v;
    const uintptr_t lo = k_low ? k : v, dist = k_low ? v - k : k - v;
    if (dist > 0 && dist % 16 == 0 && dist < (1ull << 40)) {
        cuuint64_t dims[3] = {(cuuint64_t)kChunk, (cuuint64_t)num_pages * Hkv, 2};
        cuuint64_t strides[2] = {kChunk * sizeof(float), (cuuint64_t)dist};
        cuuint32_t box[3] = {(cuuint32_t)kChunk, 1u, 2u};
        cuuint32_t estr[3] = {1, 1, 1};
        if (fn(ks_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, reinterpret_cast<void*>(lo), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS) {
            memset(vs_map, 0, sizeof(CUtensorMap));
            *pair = 1;
            *ks_off = k_low ? 0 : kChunk;
            return true;
        }
    }
    return make_scale_map(ks_map, k_scale, num_pages, Hkv) && make_scale_map(vs_map, v_scale, num_pages, Hkv);
}

// 3-D map over a paged cache [num_pages*64 tokens][Hkv][128]; box = 64 tokens
// x 1 head x (64 bf16 or 128 e4m3 = 128 bytes), 128-byte swizzle.
bool make_kv_map(CUtensorMap* map, const void* base, int fp8, int num_pages, int Hkv) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    const cuuint64_t esz = fp8 ? 1 : 2;
    cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)Hkv, (cuuint64_t)num_pages * kChunk};
    cuuint64_t strides[2] = {kHeadDim * esz, (cuuint64_t)Hkv * kHeadDim * esz};
    cuuint32_t box[3] = {fp8 ? 128u : 64u, 1u, (cuuint32_t)kChunk};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                    const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

namespace {

template <bool FP8, bool QF8, int STAGES, int NG>
struct Inst {
    using LY = Layout<FP8, STAGES, NG>;
    static const void* fn() { return reinterpret_cast<const void*>(&decode_attn_kernel<FP8, QF8, STAGES, NG>); }
    // The shared-memory opt-in is set once per device (the launch path then
    // makes no extra runtime calls, which keeps it cheap and capturable).
    static cudaError_t prepare() {
        static std::atomic<unsigned long long> done{0};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        const unsigned long long bit = 1ull << (dev & 63);
        if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
        e = cudaFuncSetAttribute(fn(), cudaFuncAttributeMaxDynamicSharedMemorySize, (int)LY::kAlloc);
        if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
        return e;
    }
    static cudaError_t launch(const CUtensorMap* maps, const Params& p, int grid, cudaStream_t s) {
        cudaError_t e = prepare();
        if (e != cudaSuccess) return e;
        return launch_pdl(decode_attn_kernel<FP8, QF8, STAGES, NG>, dim3(grid), dim3(LY::kThreads), LY::kAlloc, s,
                          maps[0], maps[1], maps[2], maps[3], p);
    }
    static int ctas_per_sm() {
        if (prepare() != cudaSuccess) return 0;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_attn_kernel<FP8, QF8, STAGES, NG>,
                                                          LY::kThreads, LY::kAlloc) != cudaSuccess)
            return 0;
        return n;
    }
};

// Persistent (load-balanced) instances, one CTA per SM. Two consumer groups
// work on alternate chunks; measured on GB300 (mixed-length batches) these
// ring depths were the best that fit in shared memory: bf16 4 x 32 KB
// stages, e4m3 8 x 17 KB stages.
using BalancedBf16 = Inst<false, false, 4, 2>;
using BalancedFp8 = Inst<true, false, 8, 2>;
using BalancedFp8Q = Inst<true, true, 8, 2>;
// Shallow instances: static split-KV maps (one descriptor per CTA, several
// CTAs per SM, as a non-persistent split-KV grid would) and balanced maps
// planned for more CTAs than the deep instance keeps resident.
using StaticBf16 = Inst<false, false, 2, 1>;
using StaticFp8 = Inst<true, false, 4, 1>;
using StaticFp8Q = Inst<true, true, 4, 1>;

}  // namespace

int attn_default_ctas(int fp8) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    const int per = fp8 ? BalancedFp8::ctas_per_sm() : BalancedBf16::ctas_per_sm();
    return sms * (per > 0 ? per : 1);
}

int attn_shallow_ctas(int fp8) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    const int per = fp8 ? StaticFp8::ctas_per_sm() : StaticBf16::ctas_per_sm();
    return sms * (per > 0 ? per : 1);
}

cudaError_t launch_attn(const AttnArgs& a, cudaStream_t s) {
    CUtensorMap maps[4];  // K, V, K scales, V scales (the last two unused for bf16)
    memset(maps, 0, sizeof maps);
    if (!make_kv_map(&maps[0], a.k_cache, a.fp8, a.num_pages, a.num_kv_heads) ||
        !make_kv_map(&maps[1], a.v_cache, a.fp8, a.num_pages, a.num_kv_heads))
        return cudaErrorInvalidValue;
    int pair = 0, ks_off = 0;
    if (a.fp8 &&
        !make_scale_maps(&maps[2], &maps[3], a.k_scale, a.v_scale, a.num_pages, a.num_kv_heads, &pair, &ks_off))
        return cudaErrorInvalidValue;
    const PlanLayout L = plan_layout(a.batch, a.num_kv_heads, a.num_ctas);
    Params p;
    memset(&p, 0, sizeof p);
    p.scale_pair = pair;
    p.ks_off = ks_off;
    p.q = reinterpret_cast<const __nv_bfloat16*>(a.q);
    p.q8 = reinterpret_cast<const uint8_t*>(a.q);
    p.q_scale = a.q_scale;
    p.k_scale = a.k_scale;
    p.v_scale = a.v_scale;
    p.page_table = a.page_table;
    p.pt_stride = a.pt_stride;
    p.seq_lens = a.seq_lens;
    p.batch = a.batch;
    p.num_q_heads = a.num_q_heads;
    p.num_kv_heads = a.num_kv_heads;
    p.num_pages = a.num_pages;
    p.q_len = 1;
    p.cta_off = a.plan + L.cta_off;
    p.tasks = a.plan + L.tasks;
    p.err = const_cast<int32_t*>(a.plan) + kHError;
    p.split_cap = a.split_cap;
    p.split_o = a.split_o;
    p.split_lse = a.split_lse;
    p.scale_log2 = 1.4426950408889634f / sqrtf((float)kHeadDim);
    p.early_kv = a.early_kv;
    p.max_tasks = (int)L.max_tasks;
    p.test_wait_expiry = a.test_wait_expiry;
    // A static map, or a balanced map planned for more CTAs than the deep
    // instance keeps resident (SMs x its CTAs per SM), runs the shallow
    // instance, which holds two CTAs per SM: a caller can plan a batch of many
    // short requests over 2 x SMs CTAs without a second wave of CTAs.
    static std::atomic<int> deep_cap[2] = {{0}, {0}};
    int cap = deep_cap[a.fp8 ? 1 : 0].load(std::memory_order_relaxed);
    if (cap == 0) {
        cap = attn_default_ctas(a.fp8);
        deep_cap[a.fp8 ? 1 : 0].store(cap, std::memory_order_relaxed);
    }
    const bool stat = a.mode == 1 || (cap > 0 && a.num_ctas > cap);
    if (a.fp8 && a.q_scale)
        return stat ? StaticFp8Q::launch(maps, p, a.num_ctas, s) : BalancedFp8Q::launch(maps, p, a.num_ctas, s);
    if (a.fp8)
        return stat ? StaticFp8::launch(maps, p, a.num_ctas, s) : BalancedFp8::launch(maps, p, a.num_ctas, s);
    return stat ? StaticBf16::launch(maps, p, a.num_ctas, s) : BalancedBf16::launch(maps, p, a.num_ctas, s);
}

}  // namespace hpc
