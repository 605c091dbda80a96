// Internal definitions shared by the CUDA translation units of libhpcdecode:
// task-map layout arithmetic, launch entry points and sm_103a PTX wrappers
// (mbarrier, TMA bulk copies, warp-level mma / ldmatrix / movmatrix).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "hpc_decode.h"

namespace hpc {

constexpr int kChunk = 64;    // tokens per chunk == tokens per page
constexpr int kHeadDim = 128;
constexpr int kGroup = 8;     // query heads per KV head
constexpr int kHdrInts = 16;
constexpr int kTaskInts = 8;

enum HdrSlot {
    kHTotalChunks = 0,
    kHBucket = 1,
    kHUsedCtas = 2,
    kHTotalSplits = 3,
    kHNumCtas = 4,
    kHBatch = 5,
    kHNumKvHeads = 6,
    kHMinChunks = 7,
    kHMaxTasks = 8,
    kHMode = 9,
    kHChunksPerHead = 10,
    kHChunkTokens = 11,
    kHError = 12,
};

// Offsets (int32 units) of the sections of a task map.
struct PlanLayout {
    long long cta_off, tasks, pair_nsplit, pair_split0, total_ints, max_tasks;
};

__host__ __device__ inline PlanLayout plan_layout(long long B, long long Hkv, long long C) {
    PlanLayout L;
    L.max_tasks = Hkv * B + 2 * C;
    L.cta_off = kHdrInts;
    L.tasks = (kHdrInts + C + 1 + 7) / 8 * 8;
    L.pair_nsplit = L.tasks + L.max_tasks * kTaskInts;
    L.pair_split0 = L.pair_nsplit + Hkv * B;
    L.total_ints = L.pair_split0 + Hkv * B;
    return L;
}

// ----------------------------------------------------------------- launchers
// (defined in plan.cu / attn.cu / combine.cu; called by api.cu)

cudaError_t launch_plan(const int32_t* seq_lens, int B, int Hkv, int C, int m, int32_t* buf,
                        cudaStream_t s);
cudaError_t launch_plan_static(const int32_t* seq_lens, int B, int Hkv, int S, int32_t* buf,
                               cudaStream_t s);

struct AttnArgs {
    const void* q;          // bf16 [B][Hq][128], or e4m3 codes when q_scale is set
    const float* q_scale;   // e4m3 query only: float32 [B][Hq]
    const void* k_cache;
    const void* v_cache;
    const float* k_scale;
    const float* v_scale;
    int fp8;
    int num_pages;
    const int32_t* page_table;
    int pt_stride;
    const int32_t* seq_lens;
    int batch, num_q_heads, num_kv_heads;
    const int32_t* plan;
    int num_ctas, mode;
    long long split_cap;
    float* split_o;
    float* split_lse;
    int early_kv;  // see Params::early_kv (attn_common.cuh)
    int test_wait_expiry = 0;  // see Params::test_wait_expiry (one-token kernel only)
};
cudaError_t launch_attn(const AttnArgs& a, cudaStream_t s);
int attn_default_ctas(int fp8);
// CTAs of the shallow one-token instance resident in one wave (SMs x its CTAs per SM).
int attn_shallow_ctas(int fp8);

// Host-side checks of one decode step's arguments (api.cu): those that
// hpc_decode_plan, hpc_decode_attn and hpc_decode_combine make, minus the ones
// on a task map and split buffers, for entry points that provide those
// themselves. Enqueues nothing and makes no CUDA call.
hpc_status step_args_check(const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
                           const float* v_scale, int kv_dtype, int num_pages, const int32_t* page_table,
                           int page_table_stride, const int32_t* seq_lens, int batch, int num_q_heads,
                           int num_kv_heads, int head_dim, int page_size, int num_ctas, int min_chunks_per_cta,
                           const void* out);

// Several new tokens per request (attn_mt.cu): q is bf16 [B][q_len][Hq][128],
// split rows are [split][q_len][8]; 2 <= q_len <= kMaxQLen.
constexpr int kMaxQLen = HPC_MAX_Q_LEN;
cudaError_t launch_attn_mt(const AttnArgs& a, int q_len, cudaStream_t s);
// The same on tcgen05 tensor cores with TMEM accumulators (attn_tc.cu), bf16 KV.
cudaError_t launch_attn_tc(const AttnArgs& a, int q_len, cudaStream_t s);

struct RopeNormArgs {
    const void* qkv;
    const int32_t* positions;
    const float* cos_sin;
    int max_pos;
    const float* q_weight;
    const float* k_weight;
    float eps;
    const int32_t* slots;
    int num_tokens, num_q_heads, num_kv_heads;
    void* q_out;
    float* q_scale;
    void* k_cache;
    void* v_cache;
    float* k_scale;
    float* v_scale;
    int num_pages;
    int kv_fp8;
    int* err;
};
cudaError_t launch_rope_norm(const RopeNormArgs& a, cudaStream_t s);

// q_len new tokens per request (1 for plain decode): rows (b, i, qh) of out.
// One byte range for the zero-copy staging kernel (stage.cu).
struct StageCopy {
    const uint8_t* src;  // device-mapped host address
    uint8_t* dst;        // device address
    size_t bytes;
};
cudaError_t launch_stage_in(const StageCopy& a, const StageCopy& b, const StageCopy& c, cudaStream_t s);

cudaError_t launch_combine(const int32_t* plan, int C, const float* split_o,
                           const float* split_lse, __nv_bfloat16* out, float* out_lse, int B,
                           int Hq, int Hkv, int q_len, cudaStream_t s);

// ----------------------------------------------------------------- PTX helpers
#if defined(__CUDACC__)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// L2 policy for data that is read exactly once (the KV stream).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 3-D tiled TMA load into this CTA's shared memory, completion counted on bar.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)),
        "l"(policy)
        : "memory");
}

// 2-D tiled TMA load into this CTA's shared memory.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0,
                                            int c1, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Contiguous bulk copy global -> shared (16-byte aligned, size multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void bulk_load_nohint(void* dst, const void* src, uint32_t bytes,
                                                 uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// D(16x8, f32) += A(16x16) * B(16x8), bf16 operands.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D(16x8, f32) += A(16x16) * B(16x8), f16 operands.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Four e4m3 codes (bytes 0..3 of w) -> two f16x2, exact (every e4m3 value is
// an f16 value): lo = {b0, b1}, hi = {b2, b3}, lower byte to lower half.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t.reg .b16 a, b;\n\t"
        "mov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialization attribute may start before its predecessor finishes;
// it must wait here before it reads anything the predecessor wrote.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Lets the next kernel in the stream (if launched as a programmatic
// dependent) be scheduled now; it still waits for this grid to complete.
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

#endif  // __CUDACC__

// Launch `kernel` as a programmatic dependent of the previous kernel on the
// stream (its prologue overlaps the predecessor's tail); the kernel calls
// grid_dependency_wait() before reading predecessor outputs. Falls back to an
// ordinary launch if the attribute is refused.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    if (e == cudaErrorNotSupported || e == cudaErrorInvalidValue) {
        (void)cudaGetLastError();
        cfg.numAttrs = 0;
        e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    }
    // a refused launch is reported through the return value; leave no error
    // pending for the caller's next runtime call
    if (e != cudaSuccess) (void)cudaGetLastError();
    return e;
}

}  // namespace hpc
