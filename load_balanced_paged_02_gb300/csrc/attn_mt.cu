// Persistent paged GQA decode attention for several new tokens per request:
// the rows that speculative decoding verifies in one step (SGLang Low-Latency
// Mode blog, "Where the Time Goes": one request verifies six token rows per
// step; vLLM x HPC-Ops blog, Hy3 section: an MTP layer for speculative
// decoding). The schedule is the load-balanced one of the one-token kernel
// (HPC-Ops/SGLang blog, "Scheduling around live KV work"): the same task map,
// one partial per descriptor, merged by the combine kernel.
//
// Causal reading: the q_len new tokens of request b are already in the cache
// (seq_lens counts them); new token i sees tokens [0, L_b - q_len + i].
//
// For descriptor (h, b, c0, c1, s) the CTA computes, for every new token i
// and query head 8h + j, attention over tokens [64*c0, min(64*c1, visible))
// and writes row (s * q_len + i) * 8 + j of the split buffers.
//
// Block = NG groups x (QS x TS) consumer warps + 1 producer warp (the
// producer is the one-token kernel's, staging q_len blocks of 8 query rows per
// descriptor).
//  * Group gi takes the chunks whose running index is gi mod NG. Inside a
//    group, warp (qw, ts) owns new tokens [qw*NTW, qw*NTW + NTW) and the
//    chunk's 16-token m-tiles [ts*4/TS, (ts+1)*4/TS). K and V fragments are
//    loaded from shared memory once per m-tile and reused for each of the
//    warp's NTW new tokens (n-tiles of the 8 query heads), so shared-memory
//    traffic per chunk is QS x (K + V) rather than q_len x (K + V).
//  * Each (group, token slice, new token) keeps its own online-softmax
//    state; at the end of a descriptor the NG x TS states of every new token
//    are merged in shared memory (the owners add their rescaled outputs one
//    after the other, so the sum order is fixed) and the normalised rows are
//    written out.
// mma.m16n8k16 with tokens as M and 8 query heads as N, as in the one-token
// kernel; e4m3 caches are widened exactly to f16 with the same permuted
// k / m indices. Every wait is bounded (2 s).
#include <atomic>
#include <cstring>

#include "attn_common.cuh"

namespace hpc {
namespace {

using namespace attn;

template <bool FP8, int NTW, int QS, int TS, int NG, int STAGES>
struct MtLayout {
    // Chunk k goes to group k % NG and stage k % STAGES: with STAGES a multiple
    // of NG a stage always belongs to the same group (no parity aliasing).
    static_assert(STAGES % NG == 0, "stage ring must be a multiple of the consumer groups");
    static_assert(TS == 1 || TS == 2 || TS == 4, "token slices split the 4 m-tiles of a chunk");
    static constexpr int kWPG = QS * TS;     // consumer warps per group
    static constexpr int kNCW = NG * kWPG;
    static constexpr int kOwners = NG * TS;  // partial states per (new token, head)
    static constexpr int kQCap = NTW * QS;   // new tokens per descriptor
    static constexpr int kQSlot = kQCap * kGroup * (int)kQPitchBf16;  // rows at the padded pitch
    static constexpr size_t kQ = (size_t)STAGES * KvCfg<FP8>::kStageBytes;
    static constexpr size_t kScratch = kQ + 2 * (size_t)kQSlot;
    // Merge scratch: one accumulator row set (owners add in turn), or, where
    // shared memory allows, one row set per owner (every owner writes at once
    // and all warps merge after one barrier).
    static constexpr size_t kScratchOne = (size_t)kQCap * kGroup * kScratchStride * 4;
    static constexpr size_t kMLBytes = (size_t)kOwners * kQCap * kGroup * 8;
    static constexpr size_t kTail = STAGES * 4 + (size_t)kNCW * 4 + 8 + (2 * STAGES + 5) * 8 + 16 + 1024;
    static constexpr bool kParMerge = kScratch + kOwners * kScratchOne + kMLBytes + kTail <= 232448;
    static constexpr size_t kML = kScratch + (kParMerge ? kOwners : 1) * kScratchOne;
    static constexpr size_t kMeta = kML + kMLBytes;
    static constexpr size_t kSink = kMeta + STAGES * 4;
    static constexpr size_t kBars = (kSink + kNCW * 4 + 7) / 8 * 8;
    static constexpr int kNumBars = 2 * STAGES + 5;
    static constexpr size_t kFlag = kBars + kNumBars * 8;
    static constexpr size_t kTotal = kFlag + 16;
    static constexpr size_t kAlloc = kTotal + 1024;  // base rounded up to 1 KB (128B swizzle)
    static constexpr int kThreads = (kNCW + 1) * 32;
    static_assert(kAlloc <= 232448, "over the 227 KB shared-memory limit of a CTA");
};

// One chunk for one consumer warp: the chunk's m-tiles [mt0, mt0 + MPW) (16
// tokens each) against the warp's ntl <= NTW new tokens. nv = valid tokens of
// the chunk; the warp's first new token sees lim0 tokens of the chunk (any
// integer; the t-th sees lim0 + t). Online-softmax state per new token in
// log2 domain.
template <bool FP8, int NTW, int MPW>
__device__ __forceinline__ void chunk_compute_mt(uint8_t* stage, int lane, int mt0, int nv, int lim0, int ntl,
                                                 const uint32_t (&qf)[NTW][8][2], float (&o)[NTW][8][4],
                                                 float (&m)[NTW][2], float (&l)[NTW][2], float scale_log2,
                                                 int ks_off) {
    const int g = lane >> 2, c = lane & 3, rr = lane & 7;
    const uint32_t sb = smem_u32(stage);
    const int last_lim = lim0 + ntl - 1;  // the warp's widest causal limit
    bool zeroed = false;
#pragma unroll 1
    for (int mt = mt0; mt < mt0 + MPW; ++mt) {
        const int nvm = nv - 16 * mt;
        if (nvm <= 0 || 16 * mt >= last_lim) break;  // the rest is invalid or masked for every token
        if (nvm < 16) {
            zero_v_tail<FP8>(stage, mt, nvm, lane);
            zeroed = true;
        }
        float acc[NTW][2][4];
#pragma unroll
        for (int t = 0; t < NTW; ++t)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[t][0][i] = acc[t][1][i] = 0.f;
        uint32_t pb[NTW][2];

        if constexpr (!FP8) {
            // ---- S^T = K Q^T, K fragments shared by the warp's new tokens
            const uint32_t krow = sb + (uint32_t)(16 * mt + ((lane >> 3) & 1) * 8 + rr) * 128u;
            const uint32_t kx = (uint32_t)((lane >> 4) ^ rr);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                uint32_t a[4];
                ldsm_x4(a, krow + (uint32_t)(ks >> 2) * 8192u + (((uint32_t)(2 * (ks & 3)) ^ kx) << 4));
#pragma unroll
                for (int t = 0; t < NTW; ++t)
                    if (t < ntl) mma_bf16(acc[t][ks & 1], a, qf[t][ks][0], qf[t][ks][1]);
            }
#pragma unroll
            for (int t = 0; t < NTW; ++t) {
                if (t >= ntl) continue;
                float s[4], p[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) s[i] = (acc[t][0][i] + acc[t][1][i]) * scale_log2;
                const int lim = min(nvm, lim0 + t - 16 * mt);
                if (g >= lim) s[0] = s[1] = kNegInf;
                if (g + 8 >= lim) s[2] = s[3] = kNegInf;
                softmax_step(s, m[t], l[t], o[t], p);
                pb[t][0] = movmatrix_t(pack_bf16x2(p[0], p[1]));
                pb[t][1] = movmatrix_t(pack_bf16x2(p[2], p[3]));
            }
            // ---- O^T += V^T P^T, V fragments shared by the warp's new tokens
            const uint32_t vrow = sb + 16384u + (uint32_t)(16 * mt + (lane >> 4) * 8 + rr) * 128u;
            const uint32_t vx = (uint32_t)(((lane >> 3) & 1) ^ rr);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                uint32_t a[4];
                ldsm_x4_t(a, vrow + (uint32_t)(i >> 2) * 8192u + (((uint32_t)(2 * (i & 3)) ^ vx) << 4));
#pragma unroll
                for (int t = 0; t < NTW; ++t)
                    if (t < ntl) mma_bf16(o[t][i], a, pb[t][0], pb[t][1]);
            }
        } else {
            const float* ksc = reinterpret_cast<const float*>(stage + 16384) + ks_off;
            const float* vsc = reinterpret_cast<const float*>(stage + 16384) + (kChunk - ks_off);
            const int r0 = 16 * mt + g;
            {
                // ---- S^T: thread reads dims [32c, 32c+32) of token rows r0, r0+8
                const uint4 k00 = lds128(sb + (uint32_t)r0 * 128u + ((uint32_t)((2 * c) ^ g) << 4));
                const uint4 k01 = lds128(sb + (uint32_t)r0 * 128u + ((uint32_t)((2 * c + 1) ^ g) << 4));
                const uint4 k10 = lds128(sb + (uint32_t)(r0 + 8) * 128u + ((uint32_t)((2 * c) ^ g) << 4));
                const uint4 k11 = lds128(sb + (uint32_t)(r0 + 8) * 128u + ((uint32_t)((2 * c + 1) ^ g) << 4));
                const uint32_t w0[8] = {k00.x, k00.y, k00.z, k00.w, k01.x, k01.y, k01.z, k01.w};
                const uint32_t w1[8] = {k10.x, k10.y, k10.z, k10.w, k11.x, k11.y, k11.z, k11.w};
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    uint32_t a[4];
                    e4m3x4_to_f16x2x2(w0[ks], a[0], a[2]);
                    e4m3x4_to_f16x2x2(w1[ks], a[1], a[3]);
#pragma unroll
                    for (int t = 0; t < NTW; ++t)
                        if (t < ntl) mma_f16(acc[t][ks & 1], a, qf[t][ks][0], qf[t][ks][1]);
                }
            }
            const float ks0 = ksc[r0] * scale_log2, ks1 = ksc[r0 + 8] * scale_log2;
            const bool v0 = g < nvm, v1 = g + 8 < nvm;
            const float vs0 = v0 ? vsc[r0] * KvCfg<true>::kPScale : 0.f;
            const float vs1 = v1 ? vsc[r0 + 8] * KvCfg<true>::kPScale : 0.f;
#pragma unroll
            for (int t = 0; t < NTW; ++t) {
                if (t >= ntl) continue;
                float s[4], p[4];
                s[0] = (acc[t][0][0] + acc[t][1][0]) * ks0;
                s[1] = (acc[t][0][1] + acc[t][1][1]) * ks0;
                s[2] = (acc[t][0][2] + acc[t][1][2]) * ks1;
                s[3] = (acc[t][0][3] + acc[t][1][3]) * ks1;
                const int lim = min(nvm, lim0 + t - 16 * mt);
                if (g >= lim) s[0] = s[1] = kNegInf;
                if (g + 8 >= lim) s[2] = s[3] = kNegInf;
                softmax_step(s, m[t], l[t], o[t], p);
                pb[t][0] = movmatrix_t(pack_f16x2(v0 ? p[0] * vs0 : 0.f, v0 ? p[1] * vs0 : 0.f));
                pb[t][1] = movmatrix_t(pack_f16x2(v1 ? p[2] * vs1 : 0.f, v1 ? p[3] * vs1 : 0.f));
            }
            // ---- O^T += V^T P^T: 16-byte column g of token rows 2c, 2c+1, 2c+8, 2c+9;
            // m-tile i row g is dim 16g+2i, row g+8 is dim 16g+2i+1
            const uint32_t vb = sb + 8192u;
            const int t0 = 16 * mt + 2 * c;
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
#pragma unroll
                for (int t = 0; t < NTW; ++t)
                    if (t < ntl) mma_f16(o[t][i], a, pb[t][0], pb[t][1]);
            }
        }
    }
    if (zeroed) fence_proxy_async_smem();  // generic zero-fill before the next TMA write
}

template <bool FP8, int NTW, int QS, int TS, int NG, int STAGES>
__global__ void __launch_bounds__(MtLayout<FP8, NTW, QS, TS, NG, STAGES>::kThreads, 1)
    decode_attn_mt_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                          const __grid_constant__ CUtensorMap tm_ks, const __grid_constant__ CUtensorMap tm_vs,
                          const Params p) {
    using LY = MtLayout<FP8, NTW, QS, TS, NG, STAGES>;
    using Cfg = KvCfg<FP8>;
    constexpr int NCW = LY::kNCW;
    constexpr int QCAP = LY::kQCap;
    constexpr int OWN = LY::kOwners;
    constexpr int MPW = 4 / TS;  // m-tiles per warp
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + LY::kBars);
    uint64_t* empty = full + STAGES;
    uint64_t* qfull = empty + STAGES;
    uint64_t* qempty = qfull + 2;
    uint64_t* merge_bar = qempty + 2;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + LY::kFlag);
    volatile int* meta = reinterpret_cast<volatile int*>(smem + LY::kMeta);
    uint8_t* qbuf = smem + LY::kQ;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], LY::kWPG);  // a stage is consumed by the warps of one group
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&qfull[i], 1);
            mbar_init(&qempty[i], NCW);
        }
        mbar_init(merge_bar, NCW);  // one arrival per consumer warp (lane 0, after __syncwarp)
        *abort_flag = 0;
        fence_mbar_init();
    }
    // every warp but the producer waits for the predecessor here (the producer
    // waits inside produce(), after its early loads when the caller allows
    // them); each thread releases the next kernel only after its own wait
    __syncthreads();
    const int Q = p.q_len;

    if (warp == NCW) {
        produce<FP8, STAGES, QStage::kBf16Rows>(p, &tm_k, &tm_v, &tm_ks, &tm_vs, lane, smem, qbuf,
                                                LY::kQSlot, full, empty, qfull, qempty, meta, abort_flag);
        return;
    }
    grid_dependency_wait();
    grid_launch_dependents();

    // ================================ consumer warps
    const int gi = warp / LY::kWPG, qw = (warp % LY::kWPG) / TS, ts = warp % TS;
    const int own = gi * TS + ts;               // this warp's partial-state owner index
    const int j0 = qw * NTW;                    // first new token of this warp
    const int ntl = max(0, min(NTW, Q - j0));   // new tokens this warp owns
    const int c = lane & 3, g = lane >> 2;
    float* scratch = reinterpret_cast<float*>(smem + LY::kScratch);
    float2* ml = reinterpret_cast<float2*>(smem + LY::kML);
    volatile uint32_t* q_sink = reinterpret_cast<volatile uint32_t*>(smem + LY::kSink);
    uint32_t seq = 0, mphase = 0;
    int qd = 0;
    TaskAhead tw;
    tw.start(p, p.cta_off[blockIdx.x]);
    for (;;) {
        const int h = tw.t0.x, b = tw.t0.y, c0 = tw.t0.z, c1 = tw.t0.w, s = tw.s;
        if (h < 0) break;
        tw.next(p);
        if (!desc_ok(p, h, b, c0, c1, s)) continue;
        const int L = __ldg(p.seq_lens + b);

        uint32_t qf[NTW][8][2];
        const int qs = qd & 1;
        if (!wait_bounded(&qfull[qs], (qd >> 1) & 1, abort_flag, kWaitLimitNs)) goto timeout;
#pragma unroll
        for (int t = 0; t < NTW; ++t) {
            if (t < ntl) {
                load_q_frags<FP8, false, kQPitchBf16>(
                    smem_u32(qbuf + qs * LY::kQSlot + (j0 + t) * kGroup * kQPitchBf16), lane, qf[t]);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) qf[t][i][0] = qf[t][i][1] = 0u;
            }
        }
        {
            // release the Q slot only after the fragment loads have returned
            uint32_t x = 0;
#pragma unroll
            for (int t = 0; t < NTW; ++t)
#pragma unroll
                for (int i = 0; i < 8; ++i) x ^= qf[t][i][0] ^ qf[t][i][1];
            __syncwarp();
            if (lane == 0) {
                q_sink[warp] = x;
                mbar_arrive(&qempty[qs]);
            }
        }
        ++qd;

        {
            float o[NTW][8][4];
            float m[NTW][2], l[NTW][2];
#pragma unroll
            for (int t = 0; t < NTW; ++t) {
#pragma unroll
                for (int i = 0; i < 8; ++i) o[t][i][0] = o[t][i][1] = o[t][i][2] = o[t][i][3] = 0.f;
                m[t][0] = m[t][1] = kNegInf;
                l[t][0] = l[t][1] = 0.f;
            }

            for (int cc = c0; cc < c1; ++cc, ++seq) {
                if (NG > 1 && (int)(seq % NG) != gi) continue;
                const int st = (int)(seq % STAGES);
                if (!wait_bounded(&full[st], (seq / STAGES) & 1, abort_flag, kWaitLimitNs)) goto timeout;
                const int nv = meta[st];
                // tokens of this chunk visible to new token j0: L - Q + j0 + 1 - 64 cc
                const int lim0 = L - kChunk * cc - (Q - 1 - j0);
                if (nv > 0 && ntl > 0)
                    chunk_compute_mt<FP8, NTW, MPW>(smem + (size_t)st * Cfg::kStageBytes, lane, ts * MPW, nv, lim0,
                                                    ntl, qf, o, m, l, p.scale_log2, p.ks_off);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[st]);
            }

            if constexpr (LY::kParMerge) {
                // ---- every owner writes its (m, l) and its unnormalised rows at once
#pragma unroll
                for (int t = 0; t < NTW; ++t) {
                    if (t >= ntl) continue;
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1) {
                        l[t][0] += __shfl_xor_sync(0xffffffffu, l[t][0], off);
                        l[t][1] += __shfl_xor_sync(0xffffffffu, l[t][1], off);
                    }
                    if (g == 0) {
                        float2* dst = ml + (own * QCAP + j0 + t) * kGroup + 2 * c;
                        dst[0] = make_float2(m[t][0], l[t][0]);
                        dst[1] = make_float2(m[t][1], l[t][1]);
                    }
                    float* r0 = scratch + ((own * QCAP + j0 + t) * kGroup + 2 * c) * kScratchStride;
                    float* r1 = r0 + kScratchStride;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        if constexpr (FP8) {
                            const int d = 16 * g + 2 * i;  // regs 0, 1: dim d; regs 2, 3: dim d + 1
                            *reinterpret_cast<float2*>(r0 + d) = make_float2(o[t][i][0], o[t][i][2]);
                            *reinterpret_cast<float2*>(r1 + d) = make_float2(o[t][i][1], o[t][i][3]);
                        } else {
                            const int d = 16 * i + g;  // regs 0, 1: dim d; regs 2, 3: dim d + 8
                            r0[d] = o[t][i][0];
                            r1[d] = o[t][i][1];
                            r0[d + 8] = o[t][i][2];
                            r1[d + 8] = o[t][i][3];
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(merge_bar);
                if (!wait_bounded(merge_bar, mphase & 1, abort_flag, kWaitLimitNs)) goto timeout;
                ++mphase;
            } else {
                // ---- phase 1: publish (m, l) of each (owner, new token, head)
#pragma unroll
                for (int t = 0; t < NTW; ++t) {
                    if (t >= ntl) continue;
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1) {
                        l[t][0] += __shfl_xor_sync(0xffffffffu, l[t][0], off);
                        l[t][1] += __shfl_xor_sync(0xffffffffu, l[t][1], off);
                    }
                    if (g == 0) {
                        float2* dst = ml + (own * QCAP + j0 + t) * kGroup + 2 * c;
                        dst[0] = make_float2(m[t][0], l[t][0]);
                        dst[1] = make_float2(m[t][1], l[t][1]);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(merge_bar);
                if (!wait_bounded(merge_bar, mphase & 1, abort_flag, kWaitLimitNs)) goto timeout;
                ++mphase;

                // ---- phase 2: owner k adds its rescaled outputs, k = 0 .. OWN-1
                for (int k = 0; k < OWN; ++k) {
                    if (own == k) {
#pragma unroll
                        for (int t = 0; t < NTW; ++t) {
                            if (t >= ntl) continue;
                            const int j = j0 + t;
                            float f[2];
#pragma unroll
                            for (int col = 0; col < 2; ++col) {
                                float M = kNegInf;
#pragma unroll
                                for (int gg = 0; gg < OWN; ++gg) M = fmaxf(M, ml[(gg * QCAP + j) * kGroup + 2 * c + col].x);
                                f[col] = m[t][col] == kNegInf ? 0.f : fast_exp2(m[t][col] - M);
                            }
                            float* r0 = scratch + (j * kGroup + 2 * c) * kScratchStride;
                            float* r1 = r0 + kScratchStride;
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                int d00, d01, d10, d11;  // dims of o[t][i][0..3]
                                if constexpr (FP8) {
                                    d00 = 16 * g + 2 * i;  // regs 0, 1: dim d; regs 2, 3: dim d + 1
                                    d01 = d00;
                                    d10 = d00 + 1;
                                    d11 = d00 + 1;
                                } else {
                                    d00 = 16 * i + g;  // regs 0, 1: dim d; regs 2, 3: dim d + 8
                                    d01 = d00;
                                    d10 = d00 + 8;
                                    d11 = d00 + 8;
                                }
                                const float a0 = o[t][i][0] * f[0], a1 = o[t][i][1] * f[1];
                                const float a2 = o[t][i][2] * f[0], a3 = o[t][i][3] * f[1];
                                if (k == 0) {
                                    r0[d00] = a0;
                                    r1[d01] = a1;
                                    r0[d10] = a2;
                                    r1[d11] = a3;
                                } else {
                                    r0[d00] += a0;
                                    r1[d01] += a1;
                                    r0[d10] += a2;
                                    r1[d11] += a3;
                                }
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(merge_bar);
                    if (!wait_bounded(merge_bar, mphase & 1, abort_flag, kWaitLimitNs)) goto timeout;
                    ++mphase;
                }
            }
        }
        if constexpr (LY::kParMerge) {
            // ---- all warps: rows (s * q_len + j) * 8 + head from every owner's state
            const int ct = warp * 32 + lane;
            for (int idx = ct; idx < Q * kGroup * 32; idx += NCW * 32) {
                const int row = idx >> 5, d4 = idx & 31;
                const int j = row >> 3, qh = row & 7;
                float M = kNegInf;
#pragma unroll
                for (int gg = 0; gg < OWN; ++gg) M = fmaxf(M, ml[(gg * QCAP + j) * kGroup + qh].x);
                float lsum = 0.f;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                if (M != kNegInf) {
#pragma unroll
                    for (int gg = 0; gg < OWN; ++gg) {
                        const float2 v = ml[(gg * QCAP + j) * kGroup + qh];
                        const float f = fast_exp2(v.x - M);
                        lsum += v.y * f;
                        const float4 x = *reinterpret_cast<const float4*>(
                            scratch + ((gg * QCAP + j) * kGroup + qh) * kScratchStride + 4 * d4);
                        acc.x += f * x.x;
                        acc.y += f * x.y;
                        acc.z += f * x.z;
                        acc.w += f * x.w;
                    }
                }
                const float inv = lsum > 0.f ? 1.f / (lsum * Cfg::kPScale) : 0.f;
                const long long orow = ((long long)s * Q + j) * kGroup + qh;
                *reinterpret_cast<float4*>(p.split_o + orow * kHeadDim + 4 * d4) =
                    make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
                if (d4 == 0) p.split_lse[orow] = lsum > 0.f ? (M + __log2f(lsum)) * kLn2 : kNegInf;
            }
        } else {
            // ---- phase 3: normalise and write rows (s * q_len + j) * 8 + head
            const int ct = warp * 32 + lane;
            for (int idx = ct; idx < Q * kGroup * 32; idx += NCW * 32) {
                const int row = idx >> 5, d4 = idx & 31;
                const int j = row >> 3, qh = row & 7;
                float M = kNegInf;
#pragma unroll
                for (int gg = 0; gg < OWN; ++gg) M = fmaxf(M, ml[(gg * QCAP + j) * kGroup + qh].x);
                float lsum = 0.f;
                if (M != kNegInf) {
#pragma unroll
                    for (int gg = 0; gg < OWN; ++gg) {
                        const float2 v = ml[(gg * QCAP + j) * kGroup + qh];
                        lsum += v.y * fast_exp2(v.x - M);
                    }
                }
                const float4 x = *reinterpret_cast<const float4*>(scratch + row * kScratchStride + 4 * d4);
                const float inv = lsum > 0.f ? 1.f / (lsum * Cfg::kPScale) : 0.f;
                const long long orow = ((long long)s * Q + j) * kGroup + qh;
                *reinterpret_cast<float4*>(p.split_o + orow * kHeadDim + 4 * d4) =
                    make_float4(x.x * inv, x.y * inv, x.z * inv, x.w * inv);
                if (d4 == 0) p.split_lse[orow] = lsum > 0.f ? (M + __log2f(lsum)) * kLn2 : kNegInf;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(merge_bar);
        if (!wait_bounded(merge_bar, mphase & 1, abort_flag, kWaitLimitNs)) goto timeout;
        ++mphase;
    }
    return;
timeout:
    if (lane == 0) {
        *abort_flag = 1;
        atomicOr(p.err, (int)HPC_DEVERR_WAIT_TIMEOUT);
    }
}

template <bool FP8, int NTW, int QS, int TS, int NG, int STAGES>
struct MtInst {
    using LY = MtLayout<FP8, NTW, QS, TS, NG, STAGES>;
    static constexpr int kMaxQ = LY::kQCap;
    static cudaError_t prepare() {
        static std::atomic<unsigned long long> done{0};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        const unsigned long long bit = 1ull << (dev & 63);
        if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
        e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&decode_attn_mt_kernel<FP8, NTW, QS, TS, NG, STAGES>),
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)LY::kAlloc);
        if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
        return e;
    }
    static cudaError_t launch(const CUtensorMap* maps, const Params& p, int grid, cudaStream_t s) {
        cudaError_t e = prepare();
        if (e != cudaSuccess) return e;
        return launch_pdl(decode_attn_mt_kernel<FP8, NTW, QS, TS, NG, STAGES>, dim3(grid), dim3(LY::kThreads),
                          LY::kAlloc, s, maps[0], maps[1], maps[2], maps[3], p);
    }
};

// Instances by q_len, chosen by a sweep of (NTW, QS, TS, NG) on GB300 over the
// mixed-length bf16 and e4m3 batches. A warp that owns NTW new tokens holds
// 32 x NTW output registers; with 9 warps a CTA may give each at most 168
// registers (the SM's register file is split over four sub-partitions), with
// 7 warps 255. bf16 favours many warps with one new token each (latency
// hiding); e4m3 favours sharing each widened K/V fragment over two new
// tokens (the f16 widening is paid once per fragment).
//                     NTW QS TS NG STAGES
//   bf16 q_len 2       1   2  4  1   4
//   bf16 q_len 3-4     1   4  1  2   4
//   bf16 q_len 5-6     2   3  1  2   4
//   bf16 q_len 7-8     3   3  1  2   4
//   e4m3 q_len 2       2   1  4  2   8
//   e4m3 q_len 3-4     2   2  2  2   8
//   e4m3 q_len 5-6     3   2  1  3   9
//   e4m3 q_len 7-8     3   3  1  2   8
template <bool FP8>
struct MtSet;
template <>
struct MtSet<false> {
    using Q2 = MtInst<false, 1, 2, 4, 1, 4>;
    using Q4 = MtInst<false, 1, 4, 1, 2, 4>;
    using Q6 = MtInst<false, 2, 3, 1, 2, 4>;
    using Q9 = MtInst<false, 3, 3, 1, 2, 4>;
};
template <>
struct MtSet<true> {
    using Q2 = MtInst<true, 2, 1, 4, 2, 8>;
    using Q4 = MtInst<true, 2, 2, 2, 2, 8>;
    using Q6 = MtInst<true, 3, 2, 1, 3, 9>;
    using Q9 = MtInst<true, 3, 3, 1, 2, 8>;
};

template <bool FP8>
cudaError_t launch_set(const CUtensorMap* maps, const Params& p, int grid, cudaStream_t s) {
    using S = MtSet<FP8>;
    if (p.q_len <= S::Q2::kMaxQ) return S::Q2::launch(maps, p, grid, s);
    if (p.q_len <= S::Q4::kMaxQ) return S::Q4::launch(maps, p, grid, s);
    if (p.q_len <= S::Q6::kMaxQ) return S::Q6::launch(maps, p, grid, s);
    if (p.q_len <= S::Q9::kMaxQ) return S::Q9::launch(maps, p, grid, s);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_attn_mt(const AttnArgs& a, int q_len, cudaStream_t s) {
    if (q_len < 2 || q_len > kMaxQLen || a.q_scale) return cudaErrorInvalidValue;
    CUtensorMap maps[4];
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
    p.k_scale = a.k_scale;
    p.v_scale = a.v_scale;
    p.page_table = a.page_table;
    p.pt_stride = a.pt_stride;
    p.seq_lens = a.seq_lens;
    p.batch = a.batch;
    p.num_q_heads = a.num_q_heads;
    p.num_kv_heads = a.num_kv_heads;
    p.num_pages = a.num_pages;
    p.q_len = q_len;
    p.cta_off = a.plan + L.cta_off;
    p.tasks = a.plan + L.tasks;
    p.err = const_cast<int32_t*>(a.plan) + kHError;
    p.split_cap = a.split_cap;
    p.split_o = a.split_o;
    p.split_lse = a.split_lse;
    p.scale_log2 = 1.4426950408889634f / sqrtf((float)kHeadDim);
    p.early_kv = a.early_kv;
    p.max_tasks = (int)L.max_tasks;
    return a.fp8 ? launch_set<true>(maps, p, a.num_ctas, s) : launch_set<false>(maps, p, a.num_ctas, s);
}

}  // namespace hpc
