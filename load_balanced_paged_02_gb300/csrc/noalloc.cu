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
// address up with cudaGetSymbolAddress, once per device, with that device
// current, on its first call on the device, and passes that address on.
#include <mutex>

#include "hpc_internal.cuh"

namespace {

// 8 MiB: the task map plus split_o / split_lse rows. A split row takes
// 8 * 128 * 4 + 8 * 4 = 4128 bytes, so about 2000 rows fit, e.g.
// 64 requests x 8 KV heads on 152 CTAs (663 rows, 2.8 MB).
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

hpc_status scratch_base(void** base) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return HPC_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return HPC_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return HPC_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *base = g_scratch_addr[dev];
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
    const size_t off_lse = off_o + round256(cap * 8 * 128 * sizeof(float));
    const size_t need = off_lse + round256(cap * 8 * sizeof(float));
    if (need > kNoAllocScratchBytes) return HPC_ERR_WORKSPACE_TOO_SMALL;

    void* base = nullptr;
    hpc_status st = scratch_base(&base);
    if (st != HPC_OK) return st;
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
