// Pieces shared by the decode attention kernels (attn.cu: one new token per
// request; attn_mt.cu: several new tokens per request): launch parameters,
// bounded mbarrier waits, query fragment loads, the online-softmax step, the
// V tail fill and the producer warp that streams K/V pages with TMA.
#pragma once

#include <cudaTypedefs.h>

#include "hpc_internal.cuh"

namespace hpc {
namespace attn {

constexpr int kScratchStride = 132;  // floats per (query) merge row
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint64_t kDrainLimitNs = 200000000ull;
// limit of the failure-path test's wait (HPC_ATTN_TEST_WAIT_EXPIRY)
constexpr uint64_t kTestWaitLimitNs = 1000000ull;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kNegInf = -__builtin_huge_valf();

template <bool FP8>
struct KvCfg;
template <>
struct KvCfg<false> {
    static constexpr int kStageBytes = 32768;  // K dims 0-63 | K 64-127 | V 0-63 | V 64-127
    static constexpr uint32_t kTxBytes = 32768;
    static constexpr float kPScale = 1.0f;
};
template <>
struct KvCfg<true> {
    static constexpr int kStageBytes = 17408;  // K 8 KB | V 8 KB | K scales 256 B | V scales 256 B
    static constexpr uint32_t kTxBytes = 16384 + 512;
    static constexpr float kPScale = 256.0f;
};

struct Params {
    const __nv_bfloat16* q;
    const uint8_t* q8;      // e4m3 query codes (QF8 instances)
    const float* q_scale;   // one float32 scale per (request, query head) (QF8 instances)
    const float* k_scale;
    const float* v_scale;
    const int32_t* page_table;
    long long pt_stride;
    const int32_t* seq_lens;
    int batch, num_q_heads, num_kv_heads, num_pages;
    int q_len;              // new tokens per request (multi-token instances; 1 otherwise)
    const int32_t* cta_off;
    const int32_t* tasks;
    int* err;
    long long split_cap;
    float* split_o;
    float* split_lse;
    float scale_log2;
    // 1: the task map, page table, lengths and every cache slot but the last
    // q_len tokens of each request were final before the preceding kernel
    // released this one, so the producer may stream those chunks before it
    // waits for that kernel
    int early_kv;
    int max_tasks;  // descriptor slots in the task map (bounds the early walk)
    // 1: failure-path test (one-token kernel): the consumers first wait, with
    // kTestWaitLimitNs, on a barrier that nothing completes, so the CTA takes
    // its timeout path
    int test_wait_expiry;
    // e4m3: 1 when tm_ks is one 3-D map over both scale arrays (the lower
    // array's row, then the upper's, at their fixed distance), so a page's two
    // scale rows arrive in one copy; else two 2-D copies, K then V
    int scale_pair;
    // e4m3: where a stage's K scales sit among its two scale rows, in floats
    // from the first (0, or 64 when the V array lies below the K array and the
    // one copy lands V first); the V scales are in the other row
    int ks_off;
};

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity,
                                             volatile int* abort_flag, uint64_t limit_ns) {
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

__device__ __forceinline__ bool desc_ok(const Params& p, int h, int b, int c0, int c1, int s) {
    return h < p.num_kv_heads && b >= 0 && b < p.batch && c0 >= 0 && c1 > c0 && c1 <= p.pt_stride &&
           s >= 0 && s < p.split_cap;
}

// Walks a CTA's descriptor list one entry ahead. The entry after the current
// one is in flight while the current one is processed, and (LEN) the live
// length of its request and (PAGES) this lane's page id of its chunk c0 +
// lane are loaded as soon as it becomes current, so a list of short
// descriptors does not pay dependent global-memory round trips per
// descriptor. Call next() right after copying the current fields, before the
// descriptor's work. An entry past the current one is only read while the
// current one is not the terminator, so every read stays inside the list.
// len and pg are 0 for an entry outside the call's shapes (desc_ok false).
template <bool LEN, bool PAGES>
struct TaskWalker {
    int4 t0, t1;  // current entry
    int len;      // LEN: its request's live length
    int pg;       // PAGES: page id of chunk t0.z + lane, when below t0.w
    int4 n0, n1;  // the entry after it
    int slot;

    __device__ __forceinline__ static void fetch(const Params& p, int s, int4& a, int4& b) {
        a = __ldg(reinterpret_cast<const int4*>(p.tasks + (long long)s * kTaskInts));
        b = __ldg(reinterpret_cast<const int4*>(p.tasks + (long long)s * kTaskInts + 4));
    }
    __device__ __forceinline__ void side(const Params& p, int lane) {
        len = 0;
        pg = 0;
        if ((LEN || PAGES) && t0.x >= 0 && desc_ok(p, t0.x, t0.y, t0.z, t0.w, t1.x)) {
            if (LEN) len = __ldg(p.seq_lens + t0.y);
            if (PAGES && t0.z + lane < t0.w) pg = __ldg(p.page_table + (long long)t0.y * p.pt_stride + t0.z + lane);
        }
    }
    __device__ __forceinline__ void start(const Params& p, int list0, int lane) {
        slot = list0;
        fetch(p, slot, t0, t1);
        side(p, lane);
        n0 = make_int4(-1, -1, -1, -1);
        n1 = n0;
        if (t0.x >= 0) fetch(p, slot + 1, n0, n1);
    }
    __device__ __forceinline__ void next(const Params& p, int lane) {
        if (t0.x < 0) return;
        ++slot;
        t0 = n0;
        t1 = n1;
        side(p, lane);
        if (t0.x >= 0) fetch(p, slot + 1, n0, n1);
    }
};

// The lighter form for loops that need only the entry itself: the next entry
// (its kv head, request, chunk range and split index) is in flight while the
// current descriptor is processed. Call next() right after copying the
// current fields; the entry after the terminator is never read.
struct TaskAhead {
    int4 t0;  // current entry: kv head, request, first chunk, end chunk
    int s;    // its split index
    int slot;

    __device__ __forceinline__ void fetch(const Params& p) {
        t0 = __ldg(reinterpret_cast<const int4*>(p.tasks + (long long)slot * kTaskInts));
        s = __ldg(p.tasks + (long long)slot * kTaskInts + 4);
    }
    __device__ __forceinline__ void start(const Params& p, int list0) {
        slot = list0;
        fetch(p);
    }
    __device__ __forceinline__ void next(const Params& p) {
        if (t0.x < 0) return;
        ++slot;
        fetch(p);
    }
};

// ------------------------------------------------------------------ consumer math

// Query rows are staged PITCH bytes apart: 256 (bf16) or 128 (e4m3) packed,
// or padded by 16 bytes (kQPitchBf16 / kQPitchE4m3) so that the 8 rows read
// together fall into different shared-memory banks.
template <bool FP8, bool QF8, uint32_t PITCH = (QF8 ? 128u : 256u)>
__device__ __forceinline__ void load_q_frags(uint32_t qbase, int lane, uint32_t (&qf)[8][2]) {
    if constexpr (QF8) {
        // e4m3 Q codes, 128 bytes per row: thread (g, c) takes bytes [32c, 32c+32)
        // of query g and widens them exactly to f16, word ks (dims 32c+4ks ..
        // 32c+4ks+3) into the B-fragment pair of k-step ks, the order in which the
        // same thread widens the K words (see chunk_compute). On GB300 the f16
        // products measured faster than e4m3 x e4m3 mma.sync (m16n8k32) on the
        // codes (e4m3-query batch: 1261 against 1290 us).
        const int g = lane >> 2, c = lane & 3;
        const uint32_t base = qbase + (uint32_t)g * PITCH + (uint32_t)c * 32u;
        const uint4 v0 = lds128(base), v1 = lds128(base + 16u);
        const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) e4m3x4_to_f16x2x2(w[ks], qf[ks][0], qf[ks][1]);
    } else if constexpr (!FP8) {
        // Q^T B-fragments: rows are the 8 query heads, 16-byte columns are dims.
#pragma unroll
        for (int kp = 0; kp < 4; ++kp) {
            uint32_t r[4];
            ldsm_x4(r, qbase + (uint32_t)(lane & 7) * PITCH + (uint32_t)(4 * kp + (lane >> 3)) * 16u);
            qf[2 * kp][0] = r[0];
            qf[2 * kp][1] = r[1];
            qf[2 * kp + 1][0] = r[2];
            qf[2 * kp + 1][1] = r[3];
        }
    } else {
        // Thread (g, c) holds dims [32c, 32c+32) of query g; k-step ks uses
        // dims 32c+4ks+{0,1} (b0b1) and 32c+4ks+{2,3} (b2b3), widened to f16.
        const int g = lane >> 2, c = lane & 3;
        const uint32_t base = qbase + (uint32_t)g * PITCH + (uint32_t)c * 64u;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 v = lds128(base + 16u * i);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int word = 4 * i + j;  // dims 32c + 2*word, +1
                __nv_bfloat162 bv = *reinterpret_cast<const __nv_bfloat162*>(&w[j]);
                const float2 f = __bfloat1622float2(bv);
                qf[word >> 1][word & 1] = pack_f16x2(f.x, f.y);
            }
        }
    }
}

// Online-softmax update of one warp's state with a 16-token x 8-query score
// tile s (log2 domain, masked entries -inf). Returns P in p.
__device__ __forceinline__ void softmax_step(float (&s)[4], float (&m)[2], float (&l)[2],
                                             float (&o)[8][4], float (&p)[4]) {
    float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
    const float mu0 = (mn0 == kNegInf) ? 0.f : mn0;
    const float mu1 = (mn1 == kNegInf) ? 0.f : mn1;
    const float al0 = fast_exp2(m[0] - mu0), al1 = fast_exp2(m[1] - mu1);
    m[0] = mn0;
    m[1] = mn1;
    p[0] = fast_exp2(s[0] - mu0);
    p[1] = fast_exp2(s[1] - mu1);
    p[2] = fast_exp2(s[2] - mu0);
    p[3] = fast_exp2(s[3] - mu1);
    l[0] = l[0] * al0 + p[0] + p[2];
    l[1] = l[1] * al1 + p[1] + p[3];
    // Once a long sequence's running max settles, alpha is 1 for every lane;
    // skip the rescale of O then (warp-uniform branch).
    if (__any_sync(0xffffffffu, (al0 != 1.f) | (al1 != 1.f))) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            o[i][0] *= al0;
            o[i][1] *= al1;
            o[i][2] *= al0;
            o[i][3] *= al1;
        }
    }
}

// Zero V rows [16*wq + nv, 16*wq + 16) of a stage (tokens past the live length
// in the last page may hold any bits, and 0 * NaN would poison P V).
template <bool FP8>
__device__ __forceinline__ void zero_v_tail(uint8_t* stage, int wq, int nv, int lane) {
    constexpr int kVecPerRow = FP8 ? 8 : 16;
    const int n = (16 - nv) * kVecPerRow;
    for (int i = lane; i < n; i += 32) {
        const int r = 16 * wq + nv + i / kVecPerRow;
        const int part = i % kVecPerRow;
        uint8_t* dst;
        if constexpr (FP8)
            dst = stage + 8192 + r * 128 + part * 16;
        else
            dst = stage + 16384 + (part >> 3) * 8192 + r * 128 + (part & 7) * 16;
        *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
    }
    __syncwarp();
}



// How the producer stages the query rows of a descriptor.
enum class QStage {
    kBf16,      // one new token: 8 bf16 rows, kQPitchBf16 bytes apart
    kE4m3,      // one new token: 8 rows of e4m3 codes kQPitchE4m3 bytes apart, then their 8 float32 scales
    kBf16Rows,  // p.q_len new tokens: p.q_len blocks of 8 bf16 rows, kQPitchBf16 bytes apart
    kBf16Tile,  // p.q_len new tokens as one 128-byte-swizzled tile [2 dim halves][8 q_len rows][128 B]
                // by two 3-D TMA loads through tm_q (an MMA operand as it lands)
};

constexpr int kQRowsBytes = kGroup * kHeadDim * 2;  // 8 bf16 query rows
// padded row pitches of the one-token query slot (one 16-byte piece per row
// shifts the rows' banks: reads of all 8 rows at one column are conflict-free)
constexpr uint32_t kQPitchBf16 = 256 + 16;
constexpr uint32_t kQPitchE4m3 = 128 + 16;
constexpr uint32_t kQScaleOffE4m3 = kGroup * kQPitchE4m3;  // the 8 float32 scales after the codes

// Producer warp of a decode attention CTA. It waits for the preceding kernel
// itself (the kernel's other warps wait before they start): at once, or, with
// p.early_kv, after issuing the TMA loads of the CTA's leading chunks that
// hold no new token, up to a full ring, so the KV stream starts while the
// predecessor (the prologue writing Q and the new tokens' K/V) is still
// running. It walks the CTA's descriptor list;
// for each descriptor it stages the query rows into a 2-slot ring (qfull /
// qempty) and then streams every chunk (= page) of K and V, plus the page's
// two e4m3 scale rows, into the STAGES-deep ring (full / empty) with TMA. The
// lanes fetch 32 page ids at a time; lane 0 issues the copies. meta[stage]
// carries the chunk's valid token count (0: skip, page id out of range).
// Chunk k of the CTA goes to stage k % STAGES. Every wait is bounded; on
// expiry it raises the abort flag and records HPC_DEVERR_WAIT_TIMEOUT. On any
// exit it waits (bounded) for its own copies in flight before returning.
template <bool FP8, int STAGES>
__device__ __forceinline__ void issue_chunk(const Params& p, const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                            const CUtensorMap* tm_ks, const CUtensorMap* tm_vs, uint8_t* sbuf,
                                            uint64_t* full_st, int page, int h, uint64_t pol) {
    using Cfg = KvCfg<FP8>;
    mbar_arrive_expect_tx(full_st, Cfg::kTxBytes);
    const int tok = page * kChunk;
    if constexpr (FP8) {
        // The 256-byte scale rows go through tensor maps (on GB300 that
        // measured 6 % faster for the whole kernel than plain bulk copies of
        // the same rows), both rows in one copy when the arrays allow it.
        // Issued first, so they are not the last bytes of the stage to land.
        const int srow = page * p.num_kv_heads + h;
        if (p.scale_pair) {
            tma_load_3d(sbuf + 16384, tm_ks, full_st, 0, srow, 0, pol);  // both rows, lower array first
        } else {
            tma_load_2d(sbuf + 16384, tm_ks, full_st, 0, srow, pol);
            tma_load_2d(sbuf + 16640, tm_vs, full_st, 0, srow, pol);
        }
        tma_load_3d(sbuf, tm_k, full_st, 0, h, tok, pol);
        tma_load_3d(sbuf + 8192, tm_v, full_st, 0, h, tok, pol);
    } else {
        tma_load_3d(sbuf, tm_k, full_st, 0, h, tok, pol);
        tma_load_3d(sbuf + 8192, tm_k, full_st, 64, h, tok, pol);
        tma_load_3d(sbuf + 16384, tm_v, full_st, 0, h, tok, pol);
        tma_load_3d(sbuf + 24576, tm_v, full_st, 64, h, tok, pol);
    }
}

template <bool FP8, int STAGES, QStage QM>
__device__ __forceinline__ void produce(const Params& p, const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                        const CUtensorMap* tm_ks, const CUtensorMap* tm_vs, int lane,
                                        uint8_t* smem, uint8_t* qbuf, uint32_t q_slot_bytes, uint64_t* full,
                                        uint64_t* empty, uint64_t* qfull, uint64_t* qempty, volatile int* meta,
                                        volatile int* abort_flag, const CUtensorMap* tm_q = nullptr) {
    using Cfg = KvCfg<FP8>;
    const uint64_t pol = l2_evict_first_policy();
    // Early phase: the leading chunks of the CTA's list that hold no new token
    // (all 64 positions below seq_len - q_len), in list order, up to a full
    // ring, stopping at the first other chunk. Each is issued exactly as the
    // main loop would (stage npre of the first lap) and skipped there.
    uint32_t npre = 0;
    if (p.early_kv && lane == 0) {
        // the walk stays inside the task map even if the caller broke the
        // contract and the map is not yet written (wrong values, no fault)
        const int l0 = p.cta_off[blockIdx.x];
        for (int slot = max(l0, 0); slot < p.max_tasks && npre < (uint32_t)STAGES; ++slot) {
            const int4 t0 = __ldg(reinterpret_cast<const int4*>(p.tasks + (long long)slot * kTaskInts));
            const int4 t1 = __ldg(reinterpret_cast<const int4*>(p.tasks + (long long)slot * kTaskInts + 4));
            const int h = t0.x, b = t0.y, c0 = t0.z, c1 = t0.w;
            if (h < 0 || !desc_ok(p, h, b, c0, c1, t1.x)) break;
            const int L = __ldg(p.seq_lens + b);
            const int32_t* prow = p.page_table + (long long)b * p.pt_stride;
            bool stop = false;
            for (int cc = c0; cc < c1 && npre < (uint32_t)STAGES; ++cc) {
                const int page = __ldg(prow + cc);
                if (kChunk * (cc + 1) > L - p.q_len || (unsigned)page >= (unsigned)p.num_pages) {
                    stop = true;
                    break;
                }
                meta[npre] = kChunk;
                issue_chunk<FP8, STAGES>(p, tm_k, tm_v, tm_ks, tm_vs, smem + (size_t)npre * Cfg::kStageBytes,
                                         &full[npre], page, h, pol);
                ++npre;
            }
            if (stop) break;
        }
    }
    npre = __shfl_sync(0xffffffffu, npre, 0);
    grid_dependency_wait();
    grid_launch_dependents();
    TaskWalker<true, true> tw;
    tw.start(p, p.cta_off[blockIdx.x], lane);
    uint32_t seq = 0;
    int qd = 0;
    bool ok = true;
    while (ok) {
        const int4 t0 = tw.t0, t1 = tw.t1;
        const int L = tw.len, pg0 = tw.pg;
        const int h = t0.x, b = t0.y, c0 = t0.z, c1 = t0.w;
        if (h < 0) break;
        tw.next(p, lane);
        if (!desc_ok(p, h, b, c0, c1, t1.x)) {
            if (lane == 0) atomicOr(p.err, (int)HPC_DEVERR_BAD_DESCRIPTOR);
            continue;
        }
        const int qs = qd & 1;
        if (lane == 0) {
            ok = wait_bounded(&qempty[qs], ((qd >> 1) & 1) ^ 1, abort_flag, kWaitLimitNs);
            if (ok) {
                uint8_t* qdst = qbuf + qs * q_slot_bytes;
                if constexpr (QM == QStage::kBf16Tile) {
                    // rows (i, j) = new token i, query head 8h + j of request b; box
                    // 64 dims x 8 heads x q_len tokens per dim half
                    const uint32_t half = (uint32_t)p.q_len * kQRowsBytes / 2;
                    mbar_arrive_expect_tx(&qfull[qs], 2 * half);
                    tma_load_3d(qdst, tm_q, &qfull[qs], 0, h * kGroup, b * p.q_len, pol);
                    tma_load_3d(qdst + q_slot_bytes / 2, tm_q, &qfull[qs], 64, h * kGroup, b * p.q_len, pol);
                } else if constexpr (QM == QStage::kE4m3) {
                    // 8 rows of 128 e4m3 codes (padded pitch), then their 8 scales
                    const long long qrow = (long long)b * p.num_q_heads + (long long)h * kGroup;
                    mbar_arrive_expect_tx(&qfull[qs], kGroup * kHeadDim + kGroup * 4);
                    for (int r = 0; r < kGroup; ++r)
                        bulk_load_nohint(qdst + r * kQPitchE4m3, p.q8 + (qrow + r) * kHeadDim, kHeadDim, &qfull[qs]);
                    bulk_load_nohint(qdst + kQScaleOffE4m3, p.q_scale + qrow, kGroup * 4, &qfull[qs]);
                } else if constexpr (QM == QStage::kBf16) {
                    // 8 bf16 rows (padded pitch): query heads [8h, 8h + 8) of request b
                    const long long qrow = (long long)b * p.num_q_heads + (long long)h * kGroup;
                    mbar_arrive_expect_tx(&qfull[qs], kQRowsBytes);
                    for (int r = 0; r < kGroup; ++r)
                        bulk_load_nohint(qdst + r * kQPitchBf16, p.q + (qrow + r) * kHeadDim, kHeadDim * 2, &qfull[qs]);
                } else {
                    // q_len blocks of 8 bf16 rows: row (i, j) = new token i of request
                    // b, query head 8h + j, at the padded pitch; the warp's lanes issue
                    // the copies below, after this expectation is set
                    mbar_arrive_expect_tx(&qfull[qs], (uint32_t)p.q_len * kQRowsBytes);
                }
            }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if constexpr (QM == QStage::kBf16Rows) {
            uint8_t* qdst = qbuf + qs * q_slot_bytes;
            for (int r = lane; r < p.q_len * kGroup; r += 32) {
                const int i = r / kGroup, j = r % kGroup;
                const long long qrow = ((long long)b * p.q_len + i) * p.num_q_heads + (long long)h * kGroup + j;
                bulk_load_nohint(qdst + r * kQPitchBf16, p.q + qrow * kHeadDim, kHeadDim * 2, &qfull[qs]);
            }
        }
        ++qd;  // query copies issued
        const int32_t* prow = p.page_table + (long long)b * p.pt_stride;
        for (int cb = c0; cb < c1 && ok; cb += 32) {
            const int cl = cb + lane;
            const int pg = cb == c0 ? pg0 : (cl < c1 ? __ldg(prow + cl) : 0);
            const int n = min(32, c1 - cb);
            for (int j = 0; j < n; ++j, ++seq) {
                const int page = __shfl_sync(0xffffffffu, pg, j);
                const int cc = cb + j;
                const int nvalid = min(kChunk, L - kChunk * cc);
                const bool page_ok = (unsigned)page < (unsigned)p.num_pages;
                const int st = (int)(seq % STAGES);
                const uint32_t ph = (seq / STAGES) & 1;
                if (lane == 0 && seq >= npre) {  // (the first npre chunks were issued early)
                    ok = wait_bounded(&empty[st], ph ^ 1, abort_flag, kWaitLimitNs);
                    if (ok) {
                        if (!page_ok) atomicOr(p.err, (int)HPC_DEVERR_PAGE_OUT_OF_RANGE);
                        if (page_ok && nvalid > 0) {
                            meta[st] = nvalid;
                            issue_chunk<FP8, STAGES>(p, tm_k, tm_v, tm_ks, tm_vs,
                                                     smem + (size_t)st * Cfg::kStageBytes, &full[st], page, h, pol);
                        } else {
                            meta[st] = 0;
                            mbar_arrive(&full[st]);
                        }
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
            }
        }
    }
    if (!ok && lane == 0) {
        *abort_flag = 1;
        atomicOr(p.err, (int)HPC_DEVERR_WAIT_TIMEOUT);
    }
    // Every copy this warp issued lands before it returns, whichever way the
    // walk ended: after an abort the consumers may have left already, and a CTA
    // must not exit while copies into its shared memory are in flight. (On the
    // normal path they have landed or are about to: consumers wait for each.)
    // Chunk k < seq went to stage k % STAGES in lap k / STAGES, and every chunk
    // before the last STAGES was consumed before its stage was issued again;
    // query copy d < qd went to slot d % 2 in lap d / 2. Early copies the walk
    // did not reach (an abort, or a task map that changed under the caller's
    // contract) sit in stages [seq, npre) of the first lap.
    if (lane == 0) {
        const uint32_t first = seq > (uint32_t)STAGES ? seq - STAGES : 0u;
        for (uint32_t k = first; k < seq; ++k)
            wait_bounded(&full[k % STAGES], (k / STAGES) & 1, nullptr, kDrainLimitNs);
        for (int d = qd > 2 ? qd - 2 : 0; d < qd; ++d)
            wait_bounded(&qfull[d & 1], (d >> 1) & 1, nullptr, kDrainLimitNs);
        for (uint32_t k = seq; k < npre; ++k) wait_bounded(&full[k], 0, nullptr, kDrainLimitNs);
    }
}

}  // namespace attn

// Tensor maps (defined in attn.cu).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
bool make_kv_map(CUtensorMap* map, const void* base, int fp8, int num_pages, int Hkv);
bool make_scale_map(CUtensorMap* map, const float* base, int num_pages, int Hkv);
// The e4m3 scale maps of a launch: one 3-D map over both arrays, from the
// lower one (*pair = 1, vs_map unused; *ks_off = 0 when the K array is the
// lower, else 64), or one 2-D map each (*pair = 0, *ks_off = 0) when the
// arrays' distance is not a multiple of 16 bytes below 2^40 or the 3-D map
// cannot be encoded. False if a map cannot be encoded.
bool make_scale_maps(CUtensorMap* ks_map, CUtensorMap* vs_map, const float* k_scale, const float* v_scale,
                     int num_pages, int Hkv, int* pair, int* ks_off);

}  // namespace hpc
