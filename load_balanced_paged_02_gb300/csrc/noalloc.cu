// hpc_decode_noalloc: one decode step (plan -> attention -> combine) that
// allocates nothing. The task map and the split buffers, which the other
// entry points take from the caller, live here in one fixed device array.
//
// Who needs it: callers that cannot call cudaMalloc (or any allocator) at
// the point where they run the step, for instance a host engine whose memory
// pool takes all device memory at start-up and forbids allocations outside
// it, or plugin code that is handed only input and output pointers and has no
// allocator to reach. They still pass inputs and outputs; the intermediate
// storage comes from this file.
//
// The array is a file-scope __device__ symbol. In host code its name is only a
// host-side stand-in, not a device address, so the entry point looks the
// address up with cudaGetSymbolAddress, with the device current, on its first
// call on the device, and passes that address on. The address belongs to the
// device's current context: a device reset (or a primary context released and
// created again) loads the module again, maybe elsewhere. So the lookup is
// cached per device together with the context's unique ID, and a call that
// finds another context current looks the address up again.
#include <cudaTypedefs.h>

#include <mutex>

#include "hpc_internal.cuh"

namespace {

using hpc::kGroup;
using hpc::kHeadDim;

// 8 MiB: the task map plus split_o / split_lse rows. A split row takes
// kGroup * kHeadDim * 4 + kGroup * 4 = 4128 bytes, so about 2000 rows fit,
// e.g. 64 requests x 8 KV heads on 152 CTAs (663 rows, 2.8 MB).
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
struct ScratchAddr {
    unsigned long long ctx_id;  // the context the address was looked up in
    void* addr;
};
std::mutex g_scratch_mu;
ScratchAddr g_scratch[kMaxDevices] = {};

// cuCtxGetCurrent and cuCtxGetId through the runtime's driver entry points
// (the library does not link libcuda).
struct CtxFns {
    PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    PFN_cuCtxGetId_v12000 get_id = nullptr;
};

const CtxFns& ctx_fns() {
    static CtxFns f;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    return f;
}

// Unique ID of the calling thread's current context; 0 if none is current.
bool current_ctx_id(unsigned long long* id) {
    const CtxFns& f = ctx_fns();
    if (!f.get_current || !f.get_id) return false;
    CUcontext ctx = nullptr;
    if (f.get_current(&ctx) != CUDA_SUCCESS) return false;
    *id = 0;
    return !ctx || f.get_id(ctx, id) == CUDA_SUCCESS;
}

hpc_status scratch_base(void** base) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return HPC_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return HPC_ERR_UNSUPPORTED;
    unsigned long long id = 0;
    if (!current_ctx_id(&id)) return HPC_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchAddr& c = g_scratch[dev];
    if (!c.addr || id == 0 || c.ctx_id != id) {
        // set-up: the device address of the array in this device's current
        // context (the lookup also makes the primary context current when none
        // was, so the ID is read again afterwards)
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return HPC_ERR_CUDA;
        if (!current_ctx_id(&id) || id == 0) return HPC_ERR_CUDA;
        c.addr = p;
        c.ctx_id = id;
    }
    *base = c.addr;
    return HPC_OK;
}

inline size_t round256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

extern "C" hpc_status hpc_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                         const float* k_scale, const float* v_scale, int kv_dtype,
                                         int num_pages, const int32_t* page_table, int page_table_stride,
                                         const int32_t* seq_lens, int batch, int num_q_heads,
                                         int num_kv_heads, int head_dim, int page_size, int num_ctas,
                                         int min_chunks_per_cta, void* out, float* out_lse, void* stream) {
    const size_t plan_bytes = hpc_decode_plan_bytes(batch, num_kv_heads, num_ctas);
    const size_t cap = hpc_decode_split_capacity(batch, num_kv_heads, num_ctas);
    if (!plan_bytes || !cap) return HPC_ERR_INVALID_ARG;
    const size_t off_o = round256(plan_bytes);
    const size_t off_lse = off_o + round256(cap * kGroup * kHeadDim * sizeof(float));
    const size_t need = off_lse + round256(cap * kGroup * sizeof(float));
    if (need > kNoAllocScratchBytes) return HPC_ERR_WORKSPACE_TOO_SMALL;
    // every check the three calls below make, before any of them enqueues work
    // into the shared array
    hpc_status st = hpc::step_args_check(q, k_cache, v_cache, k_scale, v_scale, kv_dtype, num_pages, page_table,
                                         page_table_stride, seq_lens, batch, num_q_heads, num_kv_heads, head_dim,
                                         page_size, num_ctas, min_chunks_per_cta, out);
    if (st != HPC_OK) return st;

    void* base = nullptr;
    if ((st = scratch_base(&base)) != HPC_OK) return st;
    unsigned char* s = static_cast<unsigned char*>(base);
    float* split_o = reinterpret_cast<float*>(s + off_o);
    float* split_lse = reinterpret_cast<float*>(s + off_lse);

    // Nothing in the array has to start at zero: the planner rewrites the whole
    // task map, and the attention kernel writes every split row the combine reads.
    hpc_plan plan{};
    plan.buf = reinterpret_cast<int32_t*>(s);
    plan.bytes = plan_bytes;
    if ((st = hpc_decode_plan(seq_lens, batch, num_kv_heads, num_ctas, min_chunks_per_cta, &plan, stream)) !=
        HPC_OK)
        return st;
    if ((st = hpc_decode_attn(q, k_cache, v_cache, k_scale, v_scale, kv_dtype, num_pages, page_table,
                              page_table_stride, seq_lens, batch, num_q_heads, num_kv_heads, head_dim, page_size,
                              &plan, split_o, split_lse, stream)) != HPC_OK)
        return st;
    return hpc_decode_combine(&plan, split_o, split_lse, out, out_lse, batch, num_q_heads, num_kv_heads, head_dim,
                              stream);
}
