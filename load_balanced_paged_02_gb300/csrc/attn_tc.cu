// Multi-token paged GQA decode attention on the fifth-generation tensor cores
// (tcgen05.mma with TMEM accumulators): the q_len new tokens of a request are
// the rows verified in one speculative-decoding step (SGLang Low-Latency Mode
// blog, "Where the Time Goes"; vLLM x HPC-Ops blog, Hy3's MTP layer). Same
// task map, causal reading and outputs as attn_mt.cu: new token i of request
// b sees tokens [0, L_b - q_len + i]; descriptor (h, b, c0, c1, s) writes rows
// (s * q_len + i) * 8 + j of the split buffers.
//
// One CTA per SM. bf16 caches, 11 warps:
//  * warp 8, producer: the shared producer (attn_common.cuh) streams K/V pages
//    into a ring of 128-byte-swizzled stages and the descriptor's query rows
//    into a 2-slot ring as one swizzled tile (two 3-D TMA loads).
//  * warp 9, S issuer: one thread issues, per chunk k of 64 tokens,
//      S_k = Q . K_k^T   (M = 64 query rows, N = 64 tokens, K = 128 dims)
//    into TMEM score buffer k % 2 (tcgen05.mma kind::f16, 16-bit operands in
//    shared memory, f32 accumulator; K and Q are K-major).
//  * warp 10, P.V issuer: one thread issues O_g += P_k . V_k (M = 64, N = 128
//    dims, K = 64 tokens; V is the MN-major operand) into TMEM output tile
//    g = k % 2 once softmax warpgroup g has written P_k. Separate issuers keep
//    the two MMA chains from waiting on each other; tcgen05.commit arrives on
//    the mbarriers that free score buffers, P buffers, stages and query slots.
//  * warps 0-3 and 4-7, two softmax warpgroups: warpgroup g takes the chunks
//    k with k % 2 == g. Thread (w, l < 16) of a warpgroup owns query row
//    r = 16 w + l (= new token r / 8, head r % 8), which the M = 64 layout puts
//    in TMEM lane 32 w + l. It loads its 64 scores, masks tokens past the
//    chunk's valid count and its causal limit, and keeps a reference max m and
//    sum l (log2 domain) for its warpgroup's chunks. P = exp2(s - m) goes to
//    shared memory as a 16-bit value; O_g is rescaled in TMEM only when a
//    chunk's max exceeds m by more than 8 (so P <= 256), which after the first
//    chunks is rare. At the descriptor's end warpgroup 1 publishes its (m, l)
//    and warpgroup 0 merges both states and both O tiles into the partial row
//    and its LSE.
// e4m3 caches (one float32 scale per token and KV head), 15 warps: the same
// roles on f16 operands, plus
//  * warps 11-14, converter: the producer fills a deeper ring of e4m3 stages
//    (K codes, V codes, their two 256-byte scale rows); the converter widens
//    each stage into an f16 operand slot laid out like a bf16 stage: K as its
//    exact codes (every e4m3 value is an f16 value), V dequantised (code x
//    scale, rounded to f16), rows past the live length zero. The K scales,
//    times log2(e)/sqrt(d), go beside the slot: the softmax multiplies score
//    column t by them in float32, so the scores carry no rounding of the
//    scales. The descriptor's bf16 query tile is converted to f16 in place
//    (exact for |q| in [2^-14, 65504]).
//    The dequantised V values must lie within the f16 range (|v| <= 65504).
// Every wait is bounded (2 s); on expiry the CTA records
// HPC_DEVERR_WAIT_TIMEOUT and, after a bounded drain, frees its TMEM and
// returns.
#include <atomic>
#include <cstring>

#include "attn_common.cuh"

namespace hpc {
namespace {

using namespace attn;

constexpr int kQTile = 16384;            // [2 dim halves][64 rows][128 B]
constexpr int kPTile = 8192;             // [64 rows][64 tokens x 2 B]
constexpr int kOpBytes = 32768;          // 16-bit K and V operand tiles of one chunk (a bf16 stage)
constexpr uint32_t kTmemCols = 512;      // S buffers 2 x 64 columns, O tiles 2 x 128 columns
constexpr uint32_t kOCol = 128;          // O tile g at column kOCol + 128 g
constexpr float kRescaleLog2 = 8.0f;     // lazy rescale threshold: P <= 2^8
constexpr int kSoftmaxThreads = 128;     // one warpgroup
constexpr int kConvWarp0 = 11;           // first converter warp (e4m3 instances)
constexpr int kConvThreads = 128;        // converter warpgroup
constexpr int kCMeta = 8;                // meta[kCMeta + slot]: valid tokens of a converted slot

template <bool FP8>
struct TcCfg {
    static constexpr int kStages = FP8 ? 6 : 4;                   // TMA ring depth
    static constexpr int kStageBytes = KvCfg<FP8>::kStageBytes;   // 17 KB e4m3, 32 KB bf16
    // operand slots the MMAs read: the TMA stages themselves for bf16, two
    // converted f16 slots for e4m3
    static constexpr int kOpSlots = FP8 ? 2 : kStages;
    static constexpr int kWarps = FP8 ? 15 : 11;
};

template <bool FP8>
struct TcLayout {
    using C = TcCfg<FP8>;
    static constexpr size_t kStages = 0;
    static constexpr size_t kOps = kStages + (size_t)C::kStages * C::kStageBytes;
    static constexpr size_t kQ = kOps + (FP8 ? (size_t)C::kOpSlots * kOpBytes : 0);
    static constexpr size_t kP = kQ + 2 * (size_t)kQTile;
    static constexpr size_t kKsl = kP + 2 * (size_t)kPTile;  // float [op slot][64]: K scale x log2(e)/sqrt(d)
    static constexpr size_t kML = kKsl + (FP8 ? (size_t)C::kOpSlots * 256 : 0);  // float2 [2 parities][64 rows]
    static constexpr size_t kMeta = kML + 2 * 64 * 8;  // int: stage valid counts, then slot counts at kCMeta
    static constexpr size_t kBars = kMeta + 128;
    // full, empty (stages); qfull, qempty, sfull, sfree, pfull, pvdone, published, consumed (2 each); ofree;
    // e4m3: cfull, cfree (op slots), qconv (2)
    static constexpr int kNumBars = 2 * C::kStages + 16 + 1 + (FP8 ? 2 * C::kOpSlots + 2 : 0);
    static constexpr size_t kTmemSlot = kBars + kNumBars * 8;
    static constexpr size_t kFlag = kTmemSlot + 8;
    static constexpr size_t kTotal = kFlag + 8;
    static constexpr size_t kAlloc = kTotal + 1024;
    static constexpr int kThreads = C::kWarps * 32;
    static_assert(kAlloc <= 232448, "over the 227 KB shared-memory limit of a CTA");
    static_assert(kOps % 1024 == 0 && kQ % 1024 == 0 && kP % 1024 == 0, "swizzled tiles need 1 KB alignment");
    static_assert(C::kStageBytes % 1024 == 0, "stages need 1 KB alignment");
    static_assert(C::kStages <= kCMeta && C::kOpSlots <= 8, "meta words");
};

// ------------------------------------------------------------------ tcgen05 wrappers

// Shared-memory matrix descriptor, 128-byte swizzle (rows of 128 B, 8-row
// atoms of 1024 B): start address, leading / stride byte offsets, the sm_100
// descriptor version (bit 46) and the swizzle mode (2 = 128B, bits 61-63).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16: f32 accumulator, A and B both f16
// (f16 = true) or both bf16, M x N, A K-major, B K-major (b_mn = 0) or
// MN-major (b_mn = 1).
__host__ __device__ constexpr uint32_t idesc_16bit(bool f16, int M, int N, int b_mn) {
    return (1u << 4) | ((f16 ? 0u : 1u) << 7) | ((f16 ? 0u : 1u) << 10) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
static_assert(idesc_16bit(false, 64, 64, 0) == ((1u << 4) | (1u << 7) | (1u << 10) | (8u << 17) | (4u << 24)),
              "bf16 descriptor");
static_assert(idesc_16bit(true, 64, 128, 1) == ((1u << 4) | (1u << 16) | (16u << 17) | (4u << 24)),
              "f16 descriptor");

// D (TMEM) (+)= A . B^T from shared-memory descriptors; the operand type
// comes from the instruction descriptor.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// Arrives on bar once every MMA this thread issued before it has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// bf16 pair -> f16 pair (exact for magnitudes in [2^-14, 65504]).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
    return pack_f16x2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// ------------------------------------------------------------------ kernel

// Register cap per thread. The register file is four sub-partitions of 16384
// registers and warp w runs on sub-partition w % 4: e4m3 (15 warps, four on
// some sub-partitions) gets 16384 / (4 x 32) = 128; bf16 (11 warps, at most
// three per sub-partition) could take 168, more than it needs.
template <bool FP8>
__global__ void __maxnreg__(FP8 ? 128 : 168)
    decode_attn_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                          const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_ks,
                          const __grid_constant__ CUtensorMap tm_vs, const Params p) {
    using LY = TcLayout<FP8>;
    using C = TcCfg<FP8>;
    constexpr int NS = C::kStages, NO = C::kOpSlots;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + LY::kBars);
    uint64_t* empty = full + NS;
    uint64_t* qfull = empty + NS;
    uint64_t* qempty = qfull + 2;
    uint64_t* sfull = qempty + 2;
    uint64_t* sfree = sfull + 2;
    uint64_t* pfull = sfree + 2;
    uint64_t* pvdone = pfull + 2;
    uint64_t* published = pvdone + 2;
    uint64_t* consumed = published + 2;
    uint64_t* ofree = consumed + 2;
    uint64_t* cfull = ofree + 1;      // e4m3: op slot converted
    uint64_t* cfree = cfull + NO;     // e4m3: op slot read by both MMAs
    uint64_t* qconv = cfree + NO;     // e4m3: query tile converted to f16
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + LY::kTmemSlot);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + LY::kFlag);
    volatile int* meta = reinterpret_cast<volatile int*>(smem + LY::kMeta);
    float2* mlx = reinterpret_cast<float2*>(smem + LY::kML);
    uint8_t* qbuf = smem + LY::kQ;
    uint8_t* pbuf = smem + LY::kP;
    // operand slot of the CTA's chunk number seq: where its 16-bit K and V
    // tiles are, the barrier that says they are ready, the one that frees them
    // and its valid-token count
    uint8_t* const opbase = FP8 ? smem + LY::kOps : smem;
    uint64_t* const op_ready = FP8 ? cfull : full;
    uint64_t* const op_free = FP8 ? cfree : empty;
    uint64_t* const q_ready = FP8 ? qconv : qfull;
    volatile int* const op_meta = FP8 ? meta + kCMeta : meta;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Q = p.q_len;
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1);
            // bf16: released by the P . V issuer's commit; e4m3: by the converter
            mbar_init(&empty[i], FP8 ? kConvThreads : 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&qfull[i], 1);
            mbar_init(&qempty[i], 1);
            mbar_init(&sfull[i], 1);
            mbar_init(&sfree[i], kSoftmaxThreads);
            mbar_init(&pfull[i], kSoftmaxThreads);
            mbar_init(&pvdone[i], 1);
            mbar_init(&published[i], kSoftmaxThreads);
            mbar_init(&consumed[i], kSoftmaxThreads);
        }
        mbar_init(ofree, kSoftmaxThreads);
        if constexpr (FP8) {
            for (int i = 0; i < NO; ++i) {
                mbar_init(&cfull[i], kConvThreads);
                mbar_init(&cfree[i], 1);
            }
            for (int i = 0; i < 2; ++i) mbar_init(&qconv[i], kConvThreads);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    // P rows of dead query rows (r >= 8 q_len) stay zero for the whole kernel
    for (int i = threadIdx.x; i < 2 * kPTile / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(pbuf)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(const_cast<uint32_t*>(tmem_slot))),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    grid_dependency_wait();
    grid_launch_dependents();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int list0 = p.cta_off[blockIdx.x];

    if (warp == 8) {
        produce<FP8, NS, QStage::kBf16Tile>(p, &tm_k, &tm_v, &tm_ks, &tm_vs, list0, lane, smem, qbuf, kQTile, full,
                                            empty, qfull, qempty, meta, abort_flag, &tm_q);
    } else if (warp == 9) {
        // ============================ S issuer (one thread): S_k = Q . K_k^T
        if (lane == 0) {
            constexpr uint32_t kIdS = idesc_16bit(FP8, 64, 64, 0);
            uint32_t seq = 0;  // chunks of this CTA
            int qd = 0;
            bool ok = true;
            for (int slot = list0; ok; ++slot) {
                const int4 t0 = __ldg(reinterpret_cast<const int4*>(p.tasks + (long long)slot * kTaskInts));
                const int4 t1 = __ldg(reinterpret_cast<const int4*>(p.tasks + (long long)slot * kTaskInts + 4));
                const int h = t0.x, b = t0.y, c0 = t0.z, c1 = t0.w;
                if (h < 0) break;
                if (!desc_ok(p, h, b, c0, c1, t1.x)) continue;
                const int qs = qd & 1;
                ok = wait_bounded(&q_ready[qs], (qd >> 1) & 1, abort_flag, kWaitLimitNs);
                if (!ok) break;
                tc_fence_after();
                const uint32_t qa = smem_u32(qbuf + qs * kQTile);
                for (int cc = c0; cc < c1 && ok; ++cc, ++seq) {
                    const uint32_t os = seq % NO;
                    const uint32_t sb = seq & 1;
                    ok = wait_bounded(&op_ready[os], (seq / NO) & 1, abort_flag, kWaitLimitNs);
                    if (ok && seq >= 2) ok = wait_bounded(&sfree[sb], ((seq - 2) >> 1) & 1, abort_flag, kWaitLimitNs);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t ka = smem_u32(opbase + (size_t)os * kOpBytes);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t off = (uint32_t)(kk >> 2) * 8192u + (uint32_t)(kk & 3) * 32u;
                        umma_f16(tmem + sb * 64, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(ka + off, 16, 1024),
                                 kIdS, kk > 0);
                    }
                    umma_commit(&sfull[sb]);
                    if (cc + 1 == c1) umma_commit(&qempty[qs]);  // the query slot is free once S is done
                }
                ++qd;
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(p.err, (int)HPC_DEVERR_WAIT_TIMEOUT);
            }
        }
        __syncwarp();
    } else if (warp == 10) {
        // ============================ P . V issuer (one thread): O_g += P_k . V_k
        if (lane == 0) {
            constexpr uint32_t kIdO = idesc_16bit(FP8, 64, 128, 1);
            uint32_t seq = 0;
            int nd = 0;
            bool ok = true;
            for (int slot = list0; ok; ++slot) {
                const int4 t0 = __ldg(reinterpret_cast<const int4*>(p.tasks + (long long)slot * kTaskInts));
                const int4 t1 = __ldg(reinterpret_cast<const int4*>(p.tasks + (long long)slot * kTaskInts + 4));
                const int h = t0.x, b = t0.y, c0 = t0.z, c1 = t0.w;
                if (h < 0) break;
                if (!desc_ok(p, h, b, c0, c1, t1.x)) continue;
                // the descriptor's first P . V overwrites the O tiles: the epilogue of
                // the previous descriptor must have read them
                if (nd > 0) {
                    ok = wait_bounded(ofree, (nd - 1) & 1, abort_flag, kWaitLimitNs);
                    if (!ok) break;
                }
                for (int cc = c0; cc < c1 && ok; ++cc, ++seq) {
                    const uint32_t os = seq % NO;
                    const uint32_t g = seq & 1;
                    ok = wait_bounded(&pfull[g], (seq >> 1) & 1, abort_flag, kWaitLimitNs);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t va = smem_u32(opbase + (size_t)os * kOpBytes + 16384);
                    const uint32_t pa = smem_u32(pbuf + g * kPTile);
                    const bool first = cc - c0 < 2;  // the first chunk of this parity overwrites
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_f16(tmem + kOCol + 128 * g, sdesc_sw128(pa + kk * 32, 16, 1024),
                                 sdesc_sw128(va + kk * 2048, 8192, 1024), kIdO, !first || kk > 0);
                    umma_commit(&pvdone[g]);
                    umma_commit(&op_free[os]);  // S_k finished before P_k was written
                }
                ++nd;
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(p.err, (int)HPC_DEVERR_WAIT_TIMEOUT);
            }
        }
        __syncwarp();
    } else if (warp >= kConvWarp0) {
        // ============================ converter (e4m3 instances only): e4m3 stage ->
        // f16 operand slot, bf16 query tile -> f16 in place
        if constexpr (FP8) {
            const int ct = threadIdx.x - kConvWarp0 * 32;
            float* ksl = reinterpret_cast<float*>(smem + LY::kKsl);
            uint32_t seq = 0;
            int qd = 0;
            bool ok = true;
            for (int slot = list0; ok; ++slot) {
                const int4 t0 = __ldg(reinterpret_cast<const int4*>(p.tasks + (long long)slot * kTaskInts));
                const int4 t1 = __ldg(reinterpret_cast<const int4*>(p.tasks + (long long)slot * kTaskInts + 4));
                const int h = t0.x, b = t0.y, c0 = t0.z, c1 = t0.w;
                if (h < 0) break;
                if (!desc_ok(p, h, b, c0, c1, t1.x)) continue;
                const int qs = qd & 1;
                ok = wait_bounded(&qfull[qs], (qd >> 1) & 1, abort_flag, kWaitLimitNs);
                if (!ok) break;
                {
                    // rows [0, 8 q_len) of both dim halves, 16-byte pieces (8 per row)
                    uint8_t* qt = qbuf + qs * kQTile;
                    const int npiece = kGroup * Q * 8;
                    for (int i = ct; i < 2 * npiece; i += kConvThreads) {
                        const int half = i >= npiece ? 1 : 0;
                        uint4* ptr = reinterpret_cast<uint4*>(qt + half * 8192 + (i - half * npiece) * 16);
                        uint4 v = *ptr;
                        v.x = bf16x2_to_f16x2(v.x);
                        v.y = bf16x2_to_f16x2(v.y);
                        v.z = bf16x2_to_f16x2(v.z);
                        v.w = bf16x2_to_f16x2(v.w);
                        *ptr = v;
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(&qconv[qs]);
                ++qd;
                for (int cc = c0; cc < c1 && ok; ++cc, ++seq) {
                    const uint32_t st = seq % NS, os = seq % NO;
                    ok = wait_bounded(&full[st], (seq / NS) & 1, abort_flag, kWaitLimitNs);
                    if (ok && seq >= (uint32_t)NO)
                        ok = wait_bounded(&cfree[os], ((seq / NO) - 1) & 1, abort_flag, kWaitLimitNs);
                    if (!ok) break;
                    const int nv = meta[st];  // 0: page id out of range (nothing loaded)
                    const uint8_t* sb = smem + (size_t)st * C::kStageBytes;
                    uint8_t* ob = opbase + (size_t)os * kOpBytes;
                    const float* ks = reinterpret_cast<const float*>(sb + 16384);
                    const float* vs = reinterpret_cast<const float*>(sb + 16640);
                    if (ct < kChunk) ksl[os * kChunk + ct] = ct < nv ? ks[ct] * p.scale_log2 : 0.f;
                    // 1024 source pieces of 16 codes: K then V, 8 per 128-byte row; a
                    // warp reads four whole rows per step
#pragma unroll 2
                    for (int i = ct; i < 1024; i += kConvThreads) {
                        const int mat = i >> 9, row = (i >> 3) & 63, c16 = i & 7;
                        uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
                        if (row < nv) {
                            const uint4 w = *reinterpret_cast<const uint4*>(sb + mat * 8192 + row * 128 +
                                                                           ((c16 ^ (row & 7)) << 4));
                            e4m3x4_to_f16x2x2(w.x, lo.x, lo.y);
                            e4m3x4_to_f16x2x2(w.y, lo.z, lo.w);
                            e4m3x4_to_f16x2x2(w.z, hi.x, hi.y);
                            e4m3x4_to_f16x2x2(w.w, hi.z, hi.w);
                            if (mat == 1) {
                                const float sv = vs[row];
                                const uint32_t s2 = pack_f16x2(sv, sv);
                                lo.x = hmul2_u32(lo.x, s2);
                                lo.y = hmul2_u32(lo.y, s2);
                                lo.z = hmul2_u32(lo.z, s2);
                                lo.w = hmul2_u32(lo.w, s2);
                                hi.x = hmul2_u32(hi.x, s2);
                                hi.y = hmul2_u32(hi.y, s2);
                                hi.z = hmul2_u32(hi.z, s2);
                                hi.w = hmul2_u32(hi.w, s2);
                            }
                        }
                        // dims [16 c16, 16 c16 + 16) = f16 pieces 2 (c16 & 3) and +1 of dim half
                        // c16 >> 2; the second half stores its pieces in the other order, so
                        // each store of a warp fills 8 distinct 16-byte bank groups per row
                        const int half = c16 >> 2, f0 = 2 * (c16 & 3);
                        uint8_t* rp = ob + mat * 16384 + half * 8192 + row * 128;
                        const int pa = half ? f0 + 1 : f0, pb = half ? f0 : f0 + 1;
                        *reinterpret_cast<uint4*>(rp + ((pa ^ (row & 7)) << 4)) = half ? hi : lo;
                        *reinterpret_cast<uint4*>(rp + ((pb ^ (row & 7)) << 4)) = half ? lo : hi;
                    }
                    if (ct == 0) op_meta[os] = nv;
                    fence_proxy_async_smem();
                    mbar_arrive(&empty[st]);
                    mbar_arrive(&cfull[os]);
                }
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(p.err, (int)HPC_DEVERR_WAIT_TIMEOUT);
            }
        }
    } else {
        // ============================ softmax warpgroups: g = warp / 4 takes the
        // computed chunks k with k % 2 == g, into S buffer g, P buffer g and O tile g
        const int g = warp >> 2, wq = warp & 3;
        const int tg = threadIdx.x & (kSoftmaxThreads - 1);
        const int r = 16 * wq + lane;            // query row (valid for lane < 16)
        const bool live = lane < 16 && r < kGroup * Q;
        const int qi = r >> 3;                   // new token of the row
        const uint32_t lane_addr = (uint32_t)(32 * wq) << 16;
        const uint32_t ocol = kOCol + 128 * g;
        // bf16: raw scores times log2(e)/sqrt(d) in the exponent; e4m3: the score
        // columns are already multiplied by their K scale times that factor
        const float sc = FP8 ? 1.f : p.scale_log2;
        uint32_t seq = 0;
        int nd = 0;
        for (int slot = list0;; ++slot) {
            const int4 t0 = __ldg(reinterpret_cast<const int4*>(p.tasks + (long long)slot * kTaskInts));
            const int4 t1 = __ldg(reinterpret_cast<const int4*>(p.tasks + (long long)slot * kTaskInts + 4));
            const int h = t0.x, b = t0.y, c0 = t0.z, c1 = t0.w, s = t1.x;
            if (h < 0) break;
            if (!desc_ok(p, h, b, c0, c1, s)) continue;
            const int L = __ldg(p.seq_lens + b);
            float m_ref = kNegInf, l_sum = 0.f;
            for (int cc = c0; cc < c1; ++cc, ++seq) {
                if ((int)(seq & 1) != g) continue;
                const uint32_t os = seq % NO;
                // the slot's valid-token word: the slot is not refilled before this
                // warpgroup releases P of this chunk, so waiting on its fill is exact
                if (!wait_bounded(&op_ready[os], (seq / NO) & 1, abort_flag, kWaitLimitNs)) goto timeout;
                if (!wait_bounded(&sfull[g], (seq >> 1) & 1, abort_flag, kWaitLimitNs)) goto timeout;
                tc_fence_after();
                uint32_t sr[2][32];
                tmem_ld32(tmem + lane_addr + g * 64, sr[0]);
                tmem_ld32(tmem + lane_addr + g * 64 + 32, sr[1]);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(&sfree[g]);
                const int nv = op_meta[os];  // 0: page id out of range (nothing loaded)
                if constexpr (FP8) {
                    const float4* kp = reinterpret_cast<const float4*>(smem + LY::kKsl + os * 256);
#pragma unroll
                    for (int t4 = 0; t4 < 16; ++t4) {
                        const float4 f = kp[t4];
                        const int t = 4 * t4;
                        sr[t >> 5][t & 31] = __float_as_uint(__uint_as_float(sr[t >> 5][t & 31]) * f.x);
                        sr[t >> 5][(t + 1) & 31] = __float_as_uint(__uint_as_float(sr[t >> 5][(t + 1) & 31]) * f.y);
                        sr[t >> 5][(t + 2) & 31] = __float_as_uint(__uint_as_float(sr[t >> 5][(t + 2) & 31]) * f.z);
                        sr[t >> 5][(t + 3) & 31] = __float_as_uint(__uint_as_float(sr[t >> 5][(t + 3) & 31]) * f.w);
                    }
                }
                // valid tokens of this chunk for this row: the chunk's and the causal limit
                const int lim = min(nv, L - kChunk * cc - (Q - 1 - qi));
                // tokens past the limit get -inf (after any scale, which is positive and
                // keeps the order); full chunks skip this
                if (!__all_sync(0xffffffffu, !live || lim >= kChunk)) {
#pragma unroll
                    for (int t = 0; t < 64; ++t)
                        if (t >= lim) sr[t >> 5][t & 31] = __float_as_uint(kNegInf);
                }
                // row max in eight independent chains, then a tree
                float m8[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    m8[j] = __uint_as_float(sr[0][j]);
#pragma unroll
                    for (int t = j + 8; t < 64; t += 8) m8[j] = fmaxf(m8[j], __uint_as_float(sr[t >> 5][t & 31]));
                }
                const float mraw = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                         fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
                float mx = mraw * sc;
                if (!live) mx = kNegInf;
                // P buffer g and O tile g were last used by this warpgroup's previous chunk
                if (seq >= 2 && !wait_bounded(&pvdone[g], ((seq - 2) >> 1) & 1, abort_flag, kWaitLimitNs))
                    goto timeout;
                tc_fence_after();
                // lazy rescale: move the reference max only when this chunk's max is far above it
                const bool move = mx != kNegInf && (m_ref == kNegInf || mx > m_ref + kRescaleLog2);
                const bool rescale_o = move && m_ref != kNegInf;
                if (__any_sync(0xffffffffu, rescale_o)) {
                    const float alpha = rescale_o ? fast_exp2(m_ref - mx) : 1.f;
#pragma unroll 1
                    for (int c4 = 0; c4 < 4; ++c4) {
                        uint32_t o[32];
                        tmem_ld32(tmem + lane_addr + ocol + 32 * c4, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                        tmem_st32(tmem + lane_addr + ocol + 32 * c4, o);
                    }
                    tmem_st_wait();
                }
                if (move) {
                    if (m_ref != kNegInf) l_sum *= fast_exp2(m_ref - mx);
                    m_ref = mx;
                }
                if (live) {
                    // P = exp2(s * scale - m), eight partial sums
                    const float nmu = m_ref == kNegInf ? 0.f : -m_ref;
                    uint8_t* prow = pbuf + g * kPTile + r * 128;
                    float l8[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) l8[j] = 0.f;
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) {
                        uint32_t w[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int t = 8 * c8 + 2 * u;
                            const float p0 = fast_exp2(fmaf(__uint_as_float(sr[t >> 5][t & 31]), sc, nmu));
                            const float p1 = fast_exp2(fmaf(__uint_as_float(sr[(t + 1) >> 5][(t + 1) & 31]), sc, nmu));
                            l8[2 * u] += p0;
                            l8[2 * u + 1] += p1;
                            w[u] = FP8 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
                        }
                        *reinterpret_cast<uint4*>(prow + ((c8 ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                    l_sum += ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
                }
                // rows of the last page past the live length may hold any bits: zero them
                // in V (the e4m3 converter already wrote zeros there)
                if (!FP8 && nv < kChunk) {
                    uint8_t* vst = opbase + (size_t)os * kOpBytes + 16384;
                    const int nz = (kChunk - nv) * 16;  // 16-byte pieces over both dim halves
                    for (int i = tg; i < nz; i += kSoftmaxThreads) {
                        const int row = nv + i / 16, part = i % 16;
                        *reinterpret_cast<uint4*>(vst + (part >> 3) * 8192 + row * 128 + (part & 7) * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&pfull[g]);
            }
            if (g == 1) {
                // ---- publish this warpgroup's (m, l) of the descriptor for warpgroup 0,
                // once warpgroup 0 has read what this slot held two descriptors ago
                if (nd >= 2 && !wait_bounded(&consumed[nd & 1], ((nd - 2) >> 1) & 1, abort_flag, kWaitLimitNs))
                    goto timeout;
                if (lane < 16) mlx[(nd & 1) * 64 + r] = make_float2(m_ref, l_sum);
                mbar_arrive(&published[nd & 1]);
            } else {
                // ---- epilogue: merge the two warpgroups' states and O tiles
                if (!wait_bounded(&published[nd & 1], (nd >> 1) & 1, abort_flag, kWaitLimitNs)) goto timeout;
                const uint32_t k_last = seq - 1;  // every P . V of the descriptor is done with it
                if (!wait_bounded(&pvdone[k_last & 1], (k_last >> 1) & 1, abort_flag, kWaitLimitNs)) goto timeout;
                tc_fence_after();
                // a warpgroup without a chunk in this descriptor published (-inf, 0) and
                // its O tile holds another descriptor's bits: weight 0, never multiplied
                const float2 other = mlx[(nd & 1) * 64 + (r & 63)];
                const float m1 = other.x, l1 = other.y;
                mbar_arrive(&consumed[nd & 1]);
                const float M = fmaxf(m_ref, m1);
                const float f0 = l_sum > 0.f ? fast_exp2(m_ref - M) : 0.f;
                const float f1 = l1 > 0.f ? fast_exp2(m1 - M) : 0.f;
                const float lt = f0 * l_sum + f1 * l1;
                const float inv = lt > 0.f ? 1.f / lt : 0.f;
                const float w0 = f0 * inv, w1 = f1 * inv;
                float* dst = p.split_o + (((long long)s * Q + qi) * kGroup + (r & 7)) * kHeadDim;
#pragma unroll 1
                for (int c4 = 0; c4 < 4; ++c4) {
                    uint32_t o0[32], o1[32];
                    tmem_ld32(tmem + lane_addr + kOCol + 32 * c4, o0);
                    tmem_ld32(tmem + lane_addr + kOCol + 128 + 32 * c4, o1);
                    tmem_ld_wait();
                    if (live) {
#pragma unroll
                        for (int j = 0; j < 32; j += 4) {
                            float4 v;
                            v.x = w0 * __uint_as_float(o0[j]) + (w1 != 0.f ? w1 * __uint_as_float(o1[j]) : 0.f);
                            v.y = w0 * __uint_as_float(o0[j + 1]) + (w1 != 0.f ? w1 * __uint_as_float(o1[j + 1]) : 0.f);
                            v.z = w0 * __uint_as_float(o0[j + 2]) + (w1 != 0.f ? w1 * __uint_as_float(o1[j + 2]) : 0.f);
                            v.w = w0 * __uint_as_float(o0[j + 3]) + (w1 != 0.f ? w1 * __uint_as_float(o1[j + 3]) : 0.f);
                            if (w0 == 0.f) {  // tile 0 holds nothing of this row: ignore its bits
                                v.x = w1 * __uint_as_float(o1[j]);
                                v.y = w1 * __uint_as_float(o1[j + 1]);
                                v.z = w1 * __uint_as_float(o1[j + 2]);
                                v.w = w1 * __uint_as_float(o1[j + 3]);
                                if (w1 == 0.f) v = make_float4(0.f, 0.f, 0.f, 0.f);
                            }
                            *reinterpret_cast<float4*>(dst + 32 * c4 + j) = v;
                        }
                    }
                }
                if (live)
                    p.split_lse[((long long)s * Q + qi) * kGroup + (r & 7)] = lt > 0.f ? (M + __log2f(lt)) * kLn2 : kNegInf;
                tc_fence_before();
                mbar_arrive(ofree);
            }
            ++nd;
        }
        goto done;
    timeout:
        if (lane == 0) {
            *abort_flag = 1;
            atomicOr(p.err, (int)HPC_DEVERR_WAIT_TIMEOUT);
        }
    done:;
    }
    // all roles done: in the normal path every MMA completed before warpgroup 0's
    // last wait; after a timeout give in-flight work a bounded drain
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) {
        if (*abort_flag) {
            const uint64_t t0 = global_timer_ns();
            while (global_timer_ns() - t0 < kDrainLimitNs) {
            }
        }
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// 3-D map over the query [B * q_len rows of (b, i)][Hq][128] bf16: box = 64
// dims x 8 heads x q_len new tokens, 128-byte swizzle (an MMA operand tile).
bool make_q_map(CUtensorMap* map, const void* q, int B, int Q, int Hq) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)Hq, (cuuint64_t)B * Q};
    cuuint64_t strides[2] = {kHeadDim * 2, (cuuint64_t)Hq * kHeadDim * 2};
    cuuint32_t box[3] = {64u, (cuuint32_t)kGroup, (cuuint32_t)Q};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <bool FP8>
cudaError_t tc_prepare() {
    static std::atomic<unsigned long long> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&decode_attn_tc_kernel<FP8>),
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TcLayout<FP8>::kAlloc);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

template <bool FP8>
cudaError_t launch_tc(const CUtensorMap (&maps)[5], const Params& p, int num_ctas, cudaStream_t s) {
    cudaError_t e = tc_prepare<FP8>();
    if (e != cudaSuccess) return e;
    return launch_pdl(decode_attn_tc_kernel<FP8>, dim3(num_ctas), dim3(TcLayout<FP8>::kThreads),
                      TcLayout<FP8>::kAlloc, s, maps[0], maps[1], maps[2], maps[3], maps[4], p);
}

}  // namespace

cudaError_t launch_attn_tc(const AttnArgs& a, int q_len, cudaStream_t s) {
    if (q_len < 1 || q_len > kMaxQLen || a.q_scale) return cudaErrorInvalidValue;
    CUtensorMap maps[5];  // K, V, Q, K scales, V scales (the last two e4m3 only)
    memset(maps, 0, sizeof maps);
    if (!make_kv_map(&maps[0], a.k_cache, a.fp8, a.num_pages, a.num_kv_heads) ||
        !make_kv_map(&maps[1], a.v_cache, a.fp8, a.num_pages, a.num_kv_heads) ||
        !make_q_map(&maps[2], a.q, a.batch, q_len, a.num_q_heads))
        return cudaErrorInvalidValue;
    if (a.fp8 && (!make_scale_map(&maps[3], a.k_scale, a.num_pages, a.num_kv_heads) ||
                  !make_scale_map(&maps[4], a.v_scale, a.num_pages, a.num_kv_heads)))
        return cudaErrorInvalidValue;
    const PlanLayout L = plan_layout(a.batch, a.num_kv_heads, a.num_ctas);
    Params p;
    memset(&p, 0, sizeof p);
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
    return a.fp8 ? launch_tc<true>(maps, p, a.num_ctas, s) : launch_tc<false>(maps, p, a.num_ctas, s);
}

}  // namespace hpc
