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
//    into TMEM score buffer k % 3 (tcgen05.mma kind::f16, 16-bit operands in
//    shared memory, f32 accumulator; K and Q are K-major).
//  * warp 10, P.V issuer: one thread issues O_g += P_k . V_k (M = 64, N = 128
//    dims, K = 64 tokens; V is the MN-major operand) into TMEM output tile
//    g = k % 2 once softmax warpgroup g has written P_k. Separate issuers keep
//    the two MMA chains from waiting on each other; tcgen05.commit arrives on
//    the mbarriers that free score buffers, P buffers, stages and query slots.
//  * warps 0-3 and 4-7, two softmax warpgroups: warpgroup g takes the chunks
//    k with k % 2 == g. The M = 64 layout puts query row r (= new token r / 8,
//    head r % 8) in TMEM lane 32 (r / 16) + r % 16; the 16x256b load shape
//    gives every thread of warp w half of rows 16 w + t / 4 and 16 w + t / 4 + 8
//    (all 32 lanes busy; a row's max and sum combine its four threads). The
//    warpgroup masks tokens past the chunk's valid count and each row's causal
//    limit, and keeps a reference max m and sum l (log2 domain) per row for its
//    chunks. P = exp2(s - m) goes to shared memory as 16-bit values, into one of
//    the warpgroup's two P buffers; O_g is rescaled in TMEM only when a chunk's
//    max exceeds m by more than 8 (so P <= 256), which after the first chunks
//    is rare. At the descriptor's end warpgroup 1 publishes its (m, l) and
//    warpgroup 0 merges both states and both O tiles into the partial rows and
//    their LSEs.
// e4m3 caches (one float32 scale per token and KV head), 12 warps, the same
// roles with these changes:
//  * warp 11, query splitter. Once per descriptor it splits each bf16 query
//    row in place into two e4m3 tiles, Q = (Q_hi + Q_lo) x 2^e_r with a
//    power-of-two row scale (exact to the bf16 input but for elements under
//    2^-11 of the row's maximum).
//  * S issuer: S = Q_hi . K^T + Q_lo . K^T as kind::f8f6f4 MMAs straight on
//    the K codes of the stage (4 steps of 32 dims, each hi then lo), so K is
//    never converted.
//  * softmax: score column t is multiplied by its K scale (read from the
//    stage) in float32 and the row by 2^e_r log2(e)/sqrt(d) in the exponent,
//    so the scores carry no rounding of the scales. The warpgroup that owns a
//    chunk also widens its V codes into the f16 V slot paired with its P
//    buffer (code x scale, rounded to f16; rows past the live length zero);
//    P is f16 and P . V runs kind::f16 on that slot. The dequantised V values
//    must lie within the f16 range (|v| <= 65504).
// Every wait is bounded (2 s); on expiry the CTA records
// HPC_DEVERR_WAIT_TIMEOUT and, after a bounded drain, frees its TMEM and
// returns.
#include <atomic>
#include <cstring>

#include <cuda_fp8.h>

#include "attn_common.cuh"

namespace hpc {
namespace {

using namespace attn;

constexpr int kQTile = 16384;            // [2 dim halves][64 rows][128 B]
constexpr int kPTile = 8192;             // [64 rows][64 tokens x 2 B]
constexpr int kPBufs = 4;                // two per softmax warpgroup
constexpr int kSBufs = 3;                // TMEM score buffers: S_k goes to buffer k % 3
constexpr uint32_t kTmemCols = 512;      // S buffers 3 x 64 columns, O tiles 2 x 128 columns
constexpr uint32_t kOCol = 64 * kSBufs;  // O tile g at column kOCol + 128 g
static_assert(kOCol + 256 <= kTmemCols, "TMEM columns");
constexpr float kRescaleLog2 = 8.0f;     // lazy rescale threshold: P <= 2^8
constexpr int kSoftmaxThreads = 128;     // one warpgroup
constexpr int kSplitWarp = 11;           // e4m3: the warp that splits each descriptor's query

template <bool FP8>
struct TcCfg {
    static constexpr int kStages = FP8 ? 5 : 4;                   // TMA ring depth
    static constexpr int kStageBytes = KvCfg<FP8>::kStageBytes;   // 17 KB e4m3, 32 KB bf16
    // operand slots the P . V product reads V from: the TMA stages themselves
    // for bf16; for e4m3 one f16 V slot per P buffer, filled by the softmax
    // warpgroup that writes that P
    static constexpr int kOpSlots = FP8 ? kPBufs : kStages;
    static constexpr int kOpBytes = FP8 ? 16384 : 32768;
    static constexpr int kVOff = FP8 ? 0 : 16384;                 // V tile inside an operand slot
    static constexpr int kWarps = FP8 ? 12 : 11;
};

template <bool FP8>
struct TcLayout {
    using C = TcCfg<FP8>;
    static constexpr size_t kStages = 0;
    static constexpr size_t kOps = kStages + (size_t)C::kStages * C::kStageBytes;
    static constexpr size_t kQ = kOps + (FP8 ? (size_t)C::kOpSlots * C::kOpBytes : 0);
    static constexpr size_t kP = kQ + 2 * (size_t)kQTile;
    static constexpr size_t kQsc = kP + kPBufs * (size_t)kPTile;  // float [2][64]: e4m3 Q row scales
    static constexpr size_t kML = kQsc + (FP8 ? 2 * 256 : 0);  // float2 [2 parities][64 rows]
    static constexpr size_t kMeta = kML + 2 * 64 * 8;  // int [stage]: valid tokens of the staged chunk
    static constexpr size_t kBars = kMeta + 128;
    // full, empty (stages); qfull, qempty, published, consumed (2 each); sfull, sfree (one per S buffer);
    // pfull, pvdone (one per P buffer, with its V slot for e4m3); ofree; e4m3: q8full, qdone (2 each)
    static constexpr int kNumBars = 2 * C::kStages + 8 + 2 * kSBufs + 2 * kPBufs + 1 + (FP8 ? 4 : 0);
    static constexpr size_t kTmemSlot = kBars + kNumBars * 8;
    static constexpr size_t kFlag = kTmemSlot + 8;
    static constexpr size_t kTotal = kFlag + 8;
    static constexpr size_t kAlloc = kTotal + 1024;
    static constexpr int kThreads = C::kWarps * 32;
    static_assert(kAlloc <= 232448, "over the 227 KB shared-memory limit of a CTA");
    static_assert(kOps % 1024 == 0 && kQ % 1024 == 0 && kP % 1024 == 0,
                  "swizzled tiles need 1 KB alignment");
    static_assert(C::kStageBytes % 1024 == 0 && C::kOpBytes % 1024 == 0, "stages and slots need 1 KB alignment");
    static_assert(C::kStages <= 32, "meta words");
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

// Instruction descriptor of kind::f8f6f4 with e4m3 A and B (format 0), f32
// accumulator, M x N, both operands K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D (TMEM) (+)= A . B^T, e4m3 operands from shared-memory descriptors (32
// elements of K per instruction).
__device__ __forceinline__ void umma_e4m3(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
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

// 16x256b shape, 16 lanes from the warp's base lane: register 4 m + k of
// thread t holds lane t / 4 (k < 2) or t / 4 + 8 (k >= 2), column
// 8 m + 2 (t % 4) + (k & 1), for m < 8 (x8: 64 columns) or m < 4 (x4: 32).
__device__ __forceinline__ void tmem_ld16_x8(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld16_x4(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_st16_x4(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Eight floats (exact multiples of the row scale's inverse, |x| <= 448) ->
// eight e4m3 "hi" codes (round to nearest even) and eight "lo" codes of the
// remainders x - hi. A bf16 value has eight significant bits; rounding it to
// e4m3's four leaves a remainder of at most four, so hi + lo is x exactly
// unless the remainder falls below e4m3's smallest subnormal (2^-9), i.e. for
// |x| < 2^-2 (elements under 2^-11 of the row maximum). Byte i of the
// outputs holds element i.
__device__ __forceinline__ void split_e4m3x8(const float (&x)[8], uint2& hi, uint2& lo) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const __nv_fp8x2_storage_t hc =
            __nv_cvt_float2_to_fp8x2(make_float2(x[2 * j], x[2 * j + 1]), __NV_SATFINITE, __NV_E4M3);
        const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(hc, __NV_E4M3);
        const float2 hv = __half22float2(*reinterpret_cast<const __half2*>(&hr));
        const __nv_fp8x2_storage_t lc = __nv_cvt_float2_to_fp8x2(
            make_float2(x[2 * j] - hv.x, x[2 * j + 1] - hv.y), __NV_SATFINITE, __NV_E4M3);
        h[j] = hc;
        l[j] = lc;
    }
    hi = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
    lo = make_uint2(l[0] | (l[1] << 16), l[2] | (l[3] << 16));
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// ------------------------------------------------------------------ kernel

// Register cap per thread. The register file is four sub-partitions of 16384
// registers and warp w runs on sub-partition w % 4: with at most three warps
// on a sub-partition (11 warps bf16, 12 e4m3) a thread may hold 168.
template <bool FP8>
__global__ void __maxnreg__(168)
    decode_attn_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                          const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_ks,
                          const __grid_constant__ CUtensorMap tm_vs, const Params p) {
    using LY = TcLayout<FP8>;
    using C = TcCfg<FP8>;
    constexpr int NS = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + LY::kBars);
    uint64_t* empty = full + NS;
    uint64_t* qfull = empty + NS;
    uint64_t* qempty = qfull + 2;
    uint64_t* sfull = qempty + 2;
    uint64_t* sfree = sfull + kSBufs;
    uint64_t* pfull = sfree + kSBufs;
    // pfull and pvdone: one per P buffer 2 g + j (chunks k with k % 2 = g and
    // (k / 2) % 2 = j); a warpgroup refills a buffer only after the P . V that
    // read it, so neither barrier can run two phases ahead of its waiter
    uint64_t* pvdone = pfull + kPBufs;
    uint64_t* published = pvdone + kPBufs;
    uint64_t* consumed = published + 2;
    uint64_t* ofree = consumed + 2;
    uint64_t* q8full = ofree + 1;     // e4m3: query rows split into hi / lo e4m3 tiles and scales
    // e4m3: both softmax warpgroups finished a descriptor, so its query slot
    // (split in place) is free for the producer
    uint64_t* qdone = q8full + 2;
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
    uint64_t* const q_ready = FP8 ? q8full : qfull;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Q = p.q_len;
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1);
            // bf16: released by the P . V issuer's commit; e4m3: by the S issuer's
            // commit (K codes read) and the chunk's softmax warpgroup (valid count,
            // scales and V codes read)
            mbar_init(&empty[i], FP8 ? 1 + kSoftmaxThreads : 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&qfull[i], 1);
            mbar_init(&qempty[i], 1);  // bf16 only (e4m3 frees query slots through qdone)
            mbar_init(&published[i], kSoftmaxThreads);
            mbar_init(&consumed[i], kSoftmaxThreads);
        }
        for (int i = 0; i < kSBufs; ++i) {
            mbar_init(&sfull[i], 1);
            mbar_init(&sfree[i], kSoftmaxThreads);
        }
        for (int i = 0; i < kPBufs; ++i) {
            mbar_init(&pfull[i], kSoftmaxThreads);
            mbar_init(&pvdone[i], 1);
        }
        mbar_init(ofree, kSoftmaxThreads);
        if constexpr (FP8) {
            for (int i = 0; i < 2; ++i) {
                mbar_init(&q8full[i], 32);
                mbar_init(&qdone[i], 2 * kSoftmaxThreads);
            }
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    // P rows of dead query rows (r >= 8 q_len) stay zero for the whole kernel
    for (int i = threadIdx.x; i < kPBufs * kPTile / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(pbuf)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(const_cast<uint32_t*>(tmem_slot))),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // every warp but the producer waits for the predecessor here (the producer
    // waits inside produce(), after its early loads when the caller allows
    // them); each thread releases the next kernel only after its own wait
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    int list0 = 0;
    if (warp != 8) {
        grid_dependency_wait();
        grid_launch_dependents();
        list0 = p.cta_off[blockIdx.x];
    }

    if (warp == 8) {
        produce<FP8, NS, QStage::kBf16Tile>(p, &tm_k, &tm_v, &tm_ks, &tm_vs, lane, smem, qbuf, kQTile, full,
                                            empty, qfull, FP8 ? qdone : qempty, meta, abort_flag, &tm_q);
    } else if (warp == 9) {
        // ============================ S issuer (one thread): S_k = Q . K_k^T
        if (lane == 0) {
            // bf16: Q . K^T in 8 steps of 16 dims; e4m3: (Q_hi + Q_lo) . K^T in 4
            // steps of 32 dims on the K codes of the TMA stage
            constexpr uint32_t kIdS = FP8 ? idesc_e4m3(64, 64) : idesc_16bit(false, 64, 64, 0);
            uint32_t seq = 0;  // chunks of this CTA
            int qd = 0;
            bool ok = true;
            TaskAhead tw;
            tw.start(p, list0);
            while (ok) {
                const int h = tw.t0.x, b = tw.t0.y, c0 = tw.t0.z, c1 = tw.t0.w, sx = tw.s;
                if (h < 0) break;
                tw.next(p);
                if (!desc_ok(p, h, b, c0, c1, sx)) continue;
                const int qs = qd & 1;
                ok = wait_bounded(&q_ready[qs], (qd >> 1) & 1, abort_flag, kWaitLimitNs);
                if (!ok) break;
                tc_fence_after();
                // e4m3: the slot holds the hi codes [64 rows][128 B], then the lo codes
                const uint32_t qa = smem_u32(qbuf + qs * kQTile);
                for (int cc = c0; cc < c1 && ok; ++cc, ++seq) {
                    const uint32_t sb = seq % kSBufs;
                    // bf16: the K tile of the chunk's stage; e4m3: its K codes
                    const uint32_t ks_ = seq % NS;
                    ok = wait_bounded(&full[ks_], (seq / NS) & 1, abort_flag, kWaitLimitNs);
                    if (ok && seq >= (uint32_t)kSBufs)
                        ok = wait_bounded(&sfree[sb], (seq / kSBufs - 1) & 1, abort_flag, kWaitLimitNs);
                    if (!ok) break;
                    tc_fence_after();
                    if constexpr (FP8) {
                        const uint32_t ka = smem_u32(smem + (size_t)ks_ * C::kStageBytes);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint32_t off = (uint32_t)kk * 32u;
                            umma_e4m3(tmem + sb * 64, sdesc_sw128(qa + off, 16, 1024),
                                      sdesc_sw128(ka + off, 16, 1024), kIdS, kk > 0);
                            umma_e4m3(tmem + sb * 64, sdesc_sw128(qa + 8192 + off, 16, 1024),
                                      sdesc_sw128(ka + off, 16, 1024), kIdS, 1);
                        }
                        umma_commit(&sfull[sb]);
                        umma_commit(&empty[ks_]);  // the K codes are read once S is done
                    } else {
                        const uint32_t ka = smem_u32(smem + (size_t)ks_ * C::kStageBytes);
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint32_t off = (uint32_t)(kk >> 2) * 8192u + (uint32_t)(kk & 3) * 32u;
                            umma_f16(tmem + sb * 64, sdesc_sw128(qa + off, 16, 1024),
                                     sdesc_sw128(ka + off, 16, 1024), kIdS, kk > 0);
                        }
                        umma_commit(&sfull[sb]);
                        if (cc + 1 == c1) umma_commit(&qempty[qs]);  // the query slot is free once S is done
                    }
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
            constexpr uint32_t kIdO = idesc_16bit(FP8, 64, 128, 1);  // f16 P and V for e4m3 caches
            uint32_t seq = 0;
            int nd = 0;
            bool ok = true;
            TaskAhead tw;
            tw.start(p, list0);
            while (ok) {
                const int h = tw.t0.x, b = tw.t0.y, c0 = tw.t0.z, c1 = tw.t0.w, sx = tw.s;
                if (h < 0) break;
                tw.next(p);
                if (!desc_ok(p, h, b, c0, c1, sx)) continue;
                // the descriptor's first P . V overwrites the O tiles: the epilogue of
                // the previous descriptor must have read them
                if (nd > 0) {
                    ok = wait_bounded(ofree, (nd - 1) & 1, abort_flag, kWaitLimitNs);
                    if (!ok) break;
                }
                for (int cc = c0; cc < c1 && ok; ++cc, ++seq) {
                    const uint32_t st = seq % NS;
                    const uint32_t g = seq & 1;
                    const uint32_t pb = 2 * g + ((seq >> 1) & 1);  // P buffer of the chunk
                    // P (and, e4m3, the widened V in slot pb) written by the softmax
                    ok = wait_bounded(&pfull[pb], (seq >> 2) & 1, abort_flag, kWaitLimitNs);
                    if (!ok) break;
                    tc_fence_after();
                    // bf16: V of the chunk's stage; e4m3: the f16 V slot paired with P buffer pb
                    const uint32_t va = smem_u32(FP8 ? opbase + (size_t)pb * C::kOpBytes : smem + (size_t)st * C::kStageBytes + C::kVOff);
                    const uint32_t pa = smem_u32(pbuf + pb * kPTile);
                    const bool first = cc - c0 < 2;  // the first chunk of this parity overwrites
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_f16(tmem + kOCol + 128 * g, sdesc_sw128(pa + kk * 32, 16, 1024),
                                 sdesc_sw128(va + kk * 2048, 8192, 1024), kIdO, !first || kk > 0);
                    umma_commit(&pvdone[pb]);  // P buffer pb and (e4m3) its V slot are free
                    // bf16: the stage (S_k finished before P_k was written)
                    if constexpr (!FP8) umma_commit(&empty[st]);
                }
                ++nd;
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(p.err, (int)HPC_DEVERR_WAIT_TIMEOUT);
            }
        }
        __syncwarp();
    } else if (warp == kSplitWarp) {
        // ============================ query splitter (e4m3 instances only): each
        // descriptor's bf16 query tile -> hi / lo e4m3 tiles in place, row scales
        if constexpr (FP8) {
            float* qsc = reinterpret_cast<float*>(smem + LY::kQsc);
            int qd = 0;
            bool ok = true;
            TaskAhead tw;
            tw.start(p, list0);
            while (ok) {
                const int h = tw.t0.x, b = tw.t0.y, c0 = tw.t0.z, c1 = tw.t0.w, sx = tw.s;
                if (h < 0) break;
                tw.next(p);
                if (!desc_ok(p, h, b, c0, c1, sx)) continue;
                const int qs = qd & 1;
                // (the producer refills slot qs only after both softmax warpgroups
                // finished the descriptor two back)
                ok = wait_bounded(&qfull[qs], (qd >> 1) & 1, abort_flag, kWaitLimitNs);
                if (!ok) break;
                uint8_t* qt = qbuf + qs * kQTile;
                // Lane pair (2 j, 2 j + 1) takes query row r = j + 16 u, u < 4; half hh
                // = lane & 1 reads bf16 dims [64 hh, 64 hh + 64), which sit where row r
                // of the hi tile (hh = 0) or of the lo tile (hh = 1) goes; each lane
                // writes the hi and lo codes of its dims once both lanes have read.
#pragma unroll 1
                for (int u = 0; u < 4; ++u) {
                    const int r = (lane >> 1) + 16 * u, hh = lane & 1;
                    const bool in = r < kGroup * Q;
                    uint4 raw[8];
                    float amax = 0.f;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        raw[c] = in ? *reinterpret_cast<const uint4*>(qt + hh * 8192 + r * 128 + ((c ^ (r & 7)) << 4))
                                    : make_uint4(0, 0, 0, 0);
                        const uint32_t w[4] = {raw[c].x, raw[c].y, raw[c].z, raw[c].w};
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[j] << 16)),
                                                     fabsf(__uint_as_float(w[j] & 0xffff0000u))));
                    }
                    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                    __syncwarp();  // the partner lane has read its half row
                    // the smallest power of two 2^ex with amax / 2^ex <= 448: q / 2^ex is exact
                    float qscale = 1.f, qinv = 1.f;
                    if (amax > 0.f && amax <= 3.0e38f) {
                        int e;
                        const float m = frexpf(amax * (1.f / 448.f), &e);
                        const int ex = m == 0.5f ? e - 1 : e;
                        qscale = ldexpf(1.f, ex);
                        qinv = ldexpf(1.f, -ex);
                    }
                    if (hh == 0) qsc[qs * 64 + r] = qscale;
#pragma unroll
                    for (int c2 = 0; c2 < 4; ++c2) {
                        // bf16 pieces c = 2 c2 + v (dims 64 hh + 8 c ...) -> bytes 8 v of the
                        // e4m3 row's 16-byte piece 4 hh + c2
                        uint2 hp[2], lp[2];
#pragma unroll
                        for (int v = 0; v < 2; ++v) {
                            const uint4 x4 = raw[2 * c2 + v];
                            const uint32_t w[4] = {x4.x, x4.y, x4.z, x4.w};
                            float x[8];
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                x[2 * j] = __uint_as_float(w[j] << 16) * qinv;
                                x[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u) * qinv;
                            }
                            split_e4m3x8(x, hp[v], lp[v]);
                        }
                        const int off = r * 128 + (((4 * hh + c2) ^ (r & 7)) << 4);
                        *reinterpret_cast<uint4*>(qt + off) = make_uint4(hp[0].x, hp[0].y, hp[1].x, hp[1].y);
                        *reinterpret_cast<uint4*>(qt + 8192 + off) = make_uint4(lp[0].x, lp[0].y, lp[1].x, lp[1].y);
                    }
                    __syncwarp();
                }
                fence_proxy_async_smem();
                mbar_arrive(&q8full[qs]);
                ++qd;
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(p.err, (int)HPC_DEVERR_WAIT_TIMEOUT);
            }
        }
    } else {
        // ============================ softmax warpgroups: g = warp / 4 takes the
        // computed chunks k with k % 2 == g, from S buffer k % 3, into P buffer
        // 2 g + (k / 2) % 2 and O tile g. The M = 64 accumulator holds query row i
        // in TMEM lane 32 (i / 16) + i % 16; the 16x256b load shape spreads warp
        // wq's 16 rows over all its threads: thread t holds half rows ra = 16 wq +
        // t / 4 and rb = ra + 8 (query head t / 4 of new tokens 2 wq and 2 wq + 1),
        // columns 8 m + 2 (t % 4) + {0, 1}, m < 8 (registers 4 m + {0, 1} of ra,
        // 4 m + {2, 3} of rb). A row's max and sum combine its four threads.
        const int g = warp >> 2, wq = warp & 3;
        const int tg = threadIdx.x & (kSoftmaxThreads - 1);
        const int hq = lane >> 2, cq = lane & 3;  // query head, column pair
        const int ra = 16 * wq + hq, rb = ra + 8;  // query rows
        const int qa = 2 * wq, qb = qa + 1;        // their new tokens
        const bool live_a = qa < Q, live_b = qb < Q;
        const uint32_t lane_addr = (uint32_t)(32 * wq) << 16;
        const uint32_t ocol = kOCol + 128 * g;
        // bf16: raw scores times log2(e)/sqrt(d) in the exponent; e4m3: the score
        // columns are multiplied by their K scales first, and the row's query
        // scale joins log2(e)/sqrt(d) in the exponent
        float sc_a = p.scale_log2, sc_b = p.scale_log2;
        uint32_t seq = 0;
        int nd = 0;
        TaskWalker<true, false> tw;
        tw.start(p, list0, lane);
        for (;;) {
            const int h = tw.t0.x, b = tw.t0.y, c0 = tw.t0.z, c1 = tw.t0.w, s = tw.t1.x;
            const int L = tw.len;
            if (h < 0) break;
            tw.next(p, lane);
            if (!desc_ok(p, h, b, c0, c1, s)) continue;
            // reference maxima (log2 domain) and this thread's part of the row sums
            float m_a = kNegInf, m_b = kNegInf, l_a = 0.f, l_b = 0.f;
            if constexpr (FP8) {
                // the rows' query scales, kept until both warpgroups arrive on qdone
                if (!wait_bounded(&q8full[nd & 1], (nd >> 1) & 1, abort_flag, kWaitLimitNs)) goto timeout;
                const float* qsc = reinterpret_cast<const float*>(smem + LY::kQsc) + (nd & 1) * 64;
                sc_a = qsc[ra] * p.scale_log2;
                sc_b = qsc[rb] * p.scale_log2;
            }
            for (int cc = c0; cc < c1; ++cc, ++seq) {
                if ((int)(seq & 1) != g) continue;
                // the staged chunk's valid-token word (and, e4m3, its K scales): the
                // stage is not refilled before this warpgroup releases it (e4m3) or
                // releases P of this chunk (bf16), so waiting on its fill is exact
                const uint32_t st = seq % NS;
                if (!wait_bounded(&full[st], (seq / NS) & 1, abort_flag, kWaitLimitNs)) goto timeout;
                const uint32_t sbuf = seq % kSBufs;
                if (!wait_bounded(&sfull[sbuf], (seq / kSBufs) & 1, abort_flag, kWaitLimitNs)) goto timeout;
                tc_fence_after();
                uint32_t sr[32];
                tmem_ld16_x8(tmem + lane_addr + sbuf * 64, sr);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(&sfree[sbuf]);
                const int nv = meta[st];  // 0: page id out of range (nothing loaded)
                if constexpr (FP8) {
                    // score column c times its K scale (tokens past nv are masked below)
                    const float* ks = reinterpret_cast<const float*>(smem + (size_t)st * C::kStageBytes + 16384) + p.ks_off;
#pragma unroll
                    for (int m = 0; m < 8; ++m) {
                        const float2 f = *reinterpret_cast<const float2*>(ks + 8 * m + 2 * cq);
                        sr[4 * m] = __float_as_uint(__uint_as_float(sr[4 * m]) * f.x);
                        sr[4 * m + 1] = __float_as_uint(__uint_as_float(sr[4 * m + 1]) * f.y);
                        sr[4 * m + 2] = __float_as_uint(__uint_as_float(sr[4 * m + 2]) * f.x);
                        sr[4 * m + 3] = __float_as_uint(__uint_as_float(sr[4 * m + 3]) * f.y);
                    }
                }
                // valid tokens of this chunk for each row: the chunk's and the causal limit;
                // tokens past it get -inf (after any scale, which is positive); full
                // chunks skip this
                const int lim_a = min(nv, L - kChunk * cc - (Q - 1 - qa));
                const int lim_b = min(nv, L - kChunk * cc - (Q - 1 - qb));
                if (!__all_sync(0xffffffffu, lim_a >= kChunk && lim_b >= kChunk)) {
#pragma unroll
                    for (int m = 0; m < 8; ++m) {
                        const int c = 8 * m + 2 * cq;
                        if (c >= lim_a) sr[4 * m] = __float_as_uint(kNegInf);
                        if (c + 1 >= lim_a) sr[4 * m + 1] = __float_as_uint(kNegInf);
                        if (c >= lim_b) sr[4 * m + 2] = __float_as_uint(kNegInf);
                        if (c + 1 >= lim_b) sr[4 * m + 3] = __float_as_uint(kNegInf);
                    }
                }
                // row maxima: two chains per row over the thread's 16 columns, then the
                // row's four threads
                float ma0 = __uint_as_float(sr[0]), ma1 = __uint_as_float(sr[1]);
                float mb0 = __uint_as_float(sr[2]), mb1 = __uint_as_float(sr[3]);
#pragma unroll
                for (int m = 1; m < 8; ++m) {
                    ma0 = fmaxf(ma0, __uint_as_float(sr[4 * m]));
                    ma1 = fmaxf(ma1, __uint_as_float(sr[4 * m + 1]));
                    mb0 = fmaxf(mb0, __uint_as_float(sr[4 * m + 2]));
                    mb1 = fmaxf(mb1, __uint_as_float(sr[4 * m + 3]));
                }
                float mra = fmaxf(ma0, ma1), mrb = fmaxf(mb0, mb1);
                mra = fmaxf(mra, __shfl_xor_sync(0xffffffffu, mra, 1));
                mrb = fmaxf(mrb, __shfl_xor_sync(0xffffffffu, mrb, 1));
                mra = fmaxf(mra, __shfl_xor_sync(0xffffffffu, mra, 2));
                mrb = fmaxf(mrb, __shfl_xor_sync(0xffffffffu, mrb, 2));
                const float mxa = live_a ? mra * sc_a : kNegInf;
                const float mxb = live_b ? mrb * sc_b : kNegInf;
                // this chunk's P buffer (2 g + pj) last served the chunk four back: its
                // P . V must be done; the one two back may still run
                const uint32_t pj = (seq >> 1) & 1;
                if (seq >= 4 && !wait_bounded(&pvdone[2 * g + pj], ((seq >> 2) - 1) & 1, abort_flag, kWaitLimitNs))
                    goto timeout;
                tc_fence_after();
                // lazy rescale: move a reference max only when the chunk's max is far above it
                const bool move_a = mxa != kNegInf && (m_a == kNegInf || mxa > m_a + kRescaleLog2);
                const bool move_b = mxb != kNegInf && (m_b == kNegInf || mxb > m_b + kRescaleLog2);
                const bool resc_a = move_a && m_a != kNegInf, resc_b = move_b && m_b != kNegInf;
                if (__any_sync(0xffffffffu, resc_a || resc_b)) {
                    // O tile g is final only once the P . V of the chunk two back is done
                    if (seq >= 2 &&
                        !wait_bounded(&pvdone[2 * g + (pj ^ 1)], ((seq - 2) >> 2) & 1, abort_flag, kWaitLimitNs))
                        goto timeout;
                    tc_fence_after();
                    const float al_a = resc_a ? fast_exp2(m_a - mxa) : 1.f;
                    const float al_b = resc_b ? fast_exp2(m_b - mxb) : 1.f;
#pragma unroll 1
                    for (int c32 = 0; c32 < 4; ++c32) {
                        uint32_t o[16];
                        tmem_ld16_x4(tmem + lane_addr + ocol + 32 * c32, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            o[j] = __float_as_uint(__uint_as_float(o[j]) * ((j & 2) ? al_b : al_a));
                        tmem_st16_x4(tmem + lane_addr + ocol + 32 * c32, o);
                    }
                    tmem_st_wait();
                }
                if (move_a) {
                    if (m_a != kNegInf) l_a *= fast_exp2(m_a - mxa);
                    m_a = mxa;
                }
                if (move_b) {
                    if (m_b != kNegInf) l_b *= fast_exp2(m_b - mxb);
                    m_b = mxb;
                }
                // P = exp2(s * scale - m) as 16-bit pairs; row r's columns 8 m .. 8 m + 7 are
                // the 16-byte piece m of its 128-byte P row (swizzled), pair cq at byte 4 cq
                {
                    const float na = m_a == kNegInf ? 0.f : -m_a, nb = m_b == kNegInf ? 0.f : -m_b;
                    uint8_t* pbase = pbuf + (2 * g + pj) * kPTile;
                    float sa0 = 0.f, sa1 = 0.f, sb0 = 0.f, sb1 = 0.f;
#pragma unroll
                    for (int m = 0; m < 8; ++m) {
                        const float pa0 = fast_exp2(fmaf(__uint_as_float(sr[4 * m]), sc_a, na));
                        const float pa1 = fast_exp2(fmaf(__uint_as_float(sr[4 * m + 1]), sc_a, na));
                        const float pb0 = fast_exp2(fmaf(__uint_as_float(sr[4 * m + 2]), sc_b, nb));
                        const float pb1 = fast_exp2(fmaf(__uint_as_float(sr[4 * m + 3]), sc_b, nb));
                        sa0 += pa0;
                        sa1 += pa1;
                        sb0 += pb0;
                        sb1 += pb1;
                        if (live_a)
                            *reinterpret_cast<uint32_t*>(pbase + ra * 128 + ((m ^ (ra & 7)) << 4) + 4 * cq) =
                                FP8 ? pack_f16x2(pa0, pa1) : pack_bf16x2(pa0, pa1);
                        if (live_b)
                            *reinterpret_cast<uint32_t*>(pbase + rb * 128 + ((m ^ (rb & 7)) << 4) + 4 * cq) =
                                FP8 ? pack_f16x2(pb0, pb1) : pack_bf16x2(pb0, pb1);
                    }
                    l_a += sa0 + sa1;
                    l_b += sb0 + sb1;
                }
                if constexpr (FP8) {
                    // V codes of the stage -> f16 V slot 2 g + pj (code x scale, rounded; rows
                    // past the live length zero). Thread tg takes the 16-code pieces
                    // c16 = (tg & 3) + 4 hf of rows 32 rr + tg / 4: a warp's loads cover 8
                    // rows x 4 pieces and its stores 8 rows x 4 f16 pieces, each in the
                    // minimum of four 16-byte bank-group passes. The slot was last read by
                    // the P . V of chunk k - 4, waited for above.
                    const uint8_t* sbv = smem + (size_t)st * C::kStageBytes + 8192;
                    const float* vs =
                        reinterpret_cast<const float*>(smem + (size_t)st * C::kStageBytes + 16384) + (kChunk - p.ks_off);
                    uint8_t* ob = opbase + (size_t)(2 * g + pj) * C::kOpBytes;
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr) {
                        const int row = 32 * rr + (tg >> 2);
                        const bool in = row < nv;
                        const float sv = in ? vs[row] : 0.f;
                        const uint32_t s2 = pack_f16x2(sv, sv);
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            const int c16 = (tg & 3) + 4 * hf;
                            uint4 vl = make_uint4(0, 0, 0, 0), vh = vl;
                            if (in) {
                                const uint4 vw = *reinterpret_cast<const uint4*>(sbv + row * 128 + ((c16 ^ (row & 7)) << 4));
                                e4m3x4_to_f16x2x2(vw.x, vl.x, vl.y);
                                e4m3x4_to_f16x2x2(vw.y, vl.z, vl.w);
                                e4m3x4_to_f16x2x2(vw.z, vh.x, vh.y);
                                e4m3x4_to_f16x2x2(vw.w, vh.z, vh.w);
                                vl.x = hmul2_u32(vl.x, s2);
                                vl.y = hmul2_u32(vl.y, s2);
                                vl.z = hmul2_u32(vl.z, s2);
                                vl.w = hmul2_u32(vl.w, s2);
                                vh.x = hmul2_u32(vh.x, s2);
                                vh.y = hmul2_u32(vh.y, s2);
                                vh.z = hmul2_u32(vh.z, s2);
                                vh.w = hmul2_u32(vh.w, s2);
                            }
                            // dims [16 c16, 16 c16 + 16) are f16 pieces f0 and f0 + 1 of dim
                            // half hf, f0 = 2 (c16 & 3)
                            const int f0 = 2 * (tg & 3);
                            *reinterpret_cast<uint4*>(ob + hf * 8192 + row * 128 + ((f0 ^ (row & 7)) << 4)) = vl;
                            *reinterpret_cast<uint4*>(ob + hf * 8192 + row * 128 + (((f0 + 1) ^ (row & 7)) << 4)) = vh;
                        }
                    }
                    mbar_arrive(&empty[st]);  // valid count, scales and V codes read
                }
                // rows of the last page past the live length may hold any bits: zero them
                // in V (the e4m3 path wrote zeros there above)
                if (!FP8 && nv < kChunk) {
                    uint8_t* vst = opbase + (size_t)st * C::kOpBytes + C::kVOff;  // bf16: the stage
                    const int nz = (kChunk - nv) * 16;  // 16-byte pieces over both dim halves
                    for (int i = tg; i < nz; i += kSoftmaxThreads) {
                        const int row = nv + i / 16, part = i % 16;
                        *reinterpret_cast<uint4*>(vst + (part >> 3) * 8192 + row * 128 + (part & 7) * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&pfull[2 * g + pj]);
            }
            // the rows' sums over their four threads
            l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
            l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
            l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
            l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
            if (g == 1) {
                // ---- publish this warpgroup's (m, l) of the descriptor for warpgroup 0,
                // once warpgroup 0 has read what this slot held two descriptors ago
                if (nd >= 2 && !wait_bounded(&consumed[nd & 1], ((nd - 2) >> 1) & 1, abort_flag, kWaitLimitNs))
                    goto timeout;
                if (cq == 0) {
                    mlx[(nd & 1) * 64 + ra] = make_float2(m_a, l_a);
                    mlx[(nd & 1) * 64 + rb] = make_float2(m_b, l_b);
                }
                mbar_arrive(&published[nd & 1]);
            } else {
                // ---- epilogue: merge the two warpgroups' states and O tiles
                if (!wait_bounded(&published[nd & 1], (nd >> 1) & 1, abort_flag, kWaitLimitNs)) goto timeout;
                const uint32_t k_last = seq - 1;  // every P . V of the descriptor is done with it
                if (!wait_bounded(&pvdone[2 * (k_last & 1) + ((k_last >> 1) & 1)], (k_last >> 2) & 1, abort_flag,
                                  kWaitLimitNs))
                    goto timeout;
                tc_fence_after();
                // a warpgroup without a chunk in this descriptor published (-inf, 0) and
                // its O tile holds another descriptor's bits: weight 0, never multiplied
                const float2 oa = mlx[(nd & 1) * 64 + ra], ob = mlx[(nd & 1) * 64 + rb];
                mbar_arrive(&consumed[nd & 1]);
                float w0a, w1a, w0b, w1b, lsa, lsb;
                {
                    const float M = fmaxf(m_a, oa.x);
                    const float f0 = l_a > 0.f ? fast_exp2(m_a - M) : 0.f;
                    const float f1 = oa.y > 0.f ? fast_exp2(oa.x - M) : 0.f;
                    const float lt = f0 * l_a + f1 * oa.y;
                    const float inv = lt > 0.f ? 1.f / lt : 0.f;
                    w0a = f0 * inv;
                    w1a = f1 * inv;
                    lsa = lt > 0.f ? (M + __log2f(lt)) * kLn2 : kNegInf;
                }
                {
                    const float M = fmaxf(m_b, ob.x);
                    const float f0 = l_b > 0.f ? fast_exp2(m_b - M) : 0.f;
                    const float f1 = ob.y > 0.f ? fast_exp2(ob.x - M) : 0.f;
                    const float lt = f0 * l_b + f1 * ob.y;
                    const float inv = lt > 0.f ? 1.f / lt : 0.f;
                    w0b = f0 * inv;
                    w1b = f1 * inv;
                    lsb = lt > 0.f ? (M + __log2f(lt)) * kLn2 : kNegInf;
                }
                float* dst_a = p.split_o + (((long long)s * Q + qa) * kGroup + hq) * kHeadDim;
                float* dst_b = p.split_o + (((long long)s * Q + qb) * kGroup + hq) * kHeadDim;
#pragma unroll 1
                for (int c32 = 0; c32 < 4; ++c32) {
                    uint32_t o0[16], o1[16];
                    tmem_ld16_x4(tmem + lane_addr + kOCol + 32 * c32, o0);
                    tmem_ld16_x4(tmem + lane_addr + kOCol + 128 + 32 * c32, o1);
                    tmem_ld_wait();
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const int col = 32 * c32 + 8 * m + 2 * cq;
                        // a tile whose weight is 0 may hold any bits: never multiplied
                        if (live_a) {
                            float2 v;
                            v.x = (w0a != 0.f ? w0a * __uint_as_float(o0[4 * m]) : 0.f) +
                                  (w1a != 0.f ? w1a * __uint_as_float(o1[4 * m]) : 0.f);
                            v.y = (w0a != 0.f ? w0a * __uint_as_float(o0[4 * m + 1]) : 0.f) +
                                  (w1a != 0.f ? w1a * __uint_as_float(o1[4 * m + 1]) : 0.f);
                            *reinterpret_cast<float2*>(dst_a + col) = v;
                        }
                        if (live_b) {
                            float2 v;
                            v.x = (w0b != 0.f ? w0b * __uint_as_float(o0[4 * m + 2]) : 0.f) +
                                  (w1b != 0.f ? w1b * __uint_as_float(o1[4 * m + 2]) : 0.f);
                            v.y = (w0b != 0.f ? w0b * __uint_as_float(o0[4 * m + 3]) : 0.f) +
                                  (w1b != 0.f ? w1b * __uint_as_float(o1[4 * m + 3]) : 0.f);
                            *reinterpret_cast<float2*>(dst_b + col) = v;
                        }
                    }
                }
                if (cq == 0) {
                    if (live_a) p.split_lse[((long long)s * Q + qa) * kGroup + hq] = lsa;
                    if (live_b) p.split_lse[((long long)s * Q + qb) * kGroup + hq] = lsb;
                }
                tc_fence_before();
                mbar_arrive(ofree);
            }
            if constexpr (FP8) mbar_arrive(&qdone[nd & 1]);  // this descriptor's query slot is free
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
    int pair = 0, ks_off = 0;
    if (a.fp8 &&
        !make_scale_maps(&maps[3], &maps[4], a.k_scale, a.v_scale, a.num_pages, a.num_kv_heads, &pair, &ks_off))
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
    return a.fp8 ? launch_tc<true>(maps, p, a.num_ctas, s) : launch_tc<false>(maps, p, a.num_ctas, s);
}

}  // namespace hpc
