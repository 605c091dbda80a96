// extern "C" entry points of libhpcdecode (declared in include/hpc_decode.h):
// host-side argument checks, then the launches in plan.cu, attn.cu and
// combine.cu. Nothing here allocates device memory or synchronises, except
// hpc_decode_read_error.
#include <algorithm>
#include <new>
#include <vector>

#include "hpc_internal.cuh"

using namespace hpc;

namespace {

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// hpc_decode_suggest_num_ctas: two CTAs per SM when some CTA of the one-per-SM
// plan holds at least kFewDescriptors descriptors and at least
// kDescriptorsPerChunkPct descriptors per hundred chunks of its budget, i.e.
// when fixed per-descriptor costs are a sizable share of that CTA's work. On
// GB300 every batch measured followed the rule (step time planned for 152 and
// for 304 CTAs): 1024 x 128 tokens (54 descriptors in 108 chunks), the
// decode-latency table's 32 x 128 + 32 x 4096 mix at 8/1 (7 in 14) and 64/8
// heads (34 in 112) and its 64 x 512 mix at 64/8 (5 in 27) ran faster on 304;
// the mixed-length (12 in 491), e4m3 (13 in 3195) and skewed (10 in 134)
// batches and the table's other mixes ran faster, or the same, on 152.
constexpr int kFewDescriptors = 4;
constexpr int kDescriptorsPerChunkPct = 15;

bool sizes_ok(int batch, int num_kv_heads, long long num_ctas) {
    return batch >= 1 && batch <= HPC_MAX_BATCH && num_kv_heads >= 1 &&
           num_kv_heads <= HPC_MAX_KV_HEADS && num_ctas >= 1 && num_ctas <= HPC_MAX_CTAS;
}

size_t plan_bytes_ll(int batch, int num_kv_heads, long long num_ctas) {
    if (!sizes_ok(batch, num_kv_heads, num_ctas)) return 0;
    return (size_t)plan_layout(batch, num_kv_heads, num_ctas).total_ints * sizeof(int32_t);
}

hpc_status shape_check(int num_q_heads, int num_kv_heads, int head_dim, int page_size) {
    if (num_q_heads < 1 || num_kv_heads < 1) return HPC_ERR_INVALID_ARG;
    if (head_dim != kHeadDim || page_size != kChunk || num_q_heads != kGroup * num_kv_heads)
        return HPC_ERR_UNSUPPORTED;
    return HPC_OK;
}

hpc_status plan_check(const hpc_plan* plan, int batch, int num_kv_heads) {
    if (!plan || !plan->buf) return HPC_ERR_INVALID_ARG;
    if (plan->batch != batch || plan->num_kv_heads != num_kv_heads) return HPC_ERR_INVALID_ARG;
    if (plan->num_ctas < 1 || plan->bytes < plan_bytes_ll(batch, num_kv_heads, plan->num_ctas))
        return HPC_ERR_INVALID_ARG;
    return HPC_OK;
}

// The device address of page-locked, device-mapped host memory; nullptr for
// anything else (pageable or device memory, or a failed query).
void* mapped_host(const void* h) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, h) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

struct StepWorkspace {
    size_t q, seq_lens, page_table, plan, split_o, split_lse, out, out_lse, total;
};

StepWorkspace step_workspace(int batch, int num_q_heads, int num_kv_heads, int pt_stride, int num_ctas) {
    StepWorkspace w{};
    const size_t cap = hpc_decode_split_capacity(batch, num_kv_heads, num_ctas);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t at = off;
        off = align_up(off + bytes, 256);
        return at;
    };
    w.q = take((size_t)batch * num_q_heads * kHeadDim * 2);
    w.seq_lens = take((size_t)batch * 4);
    w.page_table = take((size_t)batch * pt_stride * 4);
    w.plan = take(hpc_decode_plan_bytes(batch, num_kv_heads, num_ctas));
    w.split_o = take(cap * kGroup * kHeadDim * 4);
    w.split_lse = take(cap * kGroup * 4);
    w.out = take((size_t)batch * num_q_heads * kHeadDim * 2);
    w.out_lse = take((size_t)batch * num_q_heads * 4);
    w.total = off;
    return w;
}

}  // namespace

extern "C" {

size_t hpc_decode_plan_bytes(int batch, int num_kv_heads, int num_ctas) {
    return plan_bytes_ll(batch, num_kv_heads, num_ctas);
}

size_t hpc_decode_split_capacity(int batch, int num_kv_heads, int num_ctas) {
    if (!sizes_ok(batch, num_kv_heads, num_ctas)) return 0;
    long long cap = (long long)num_kv_heads * batch + num_ctas - 1;
    return (size_t)(cap < 1 ? 1 : cap);
}

int hpc_decode_default_num_ctas(int kv_dtype) {
    if (kv_dtype != HPC_KV_BF16 && kv_dtype != HPC_KV_FP8_E4M3) return 0;
    return attn_default_ctas(kv_dtype == HPC_KV_FP8_E4M3);
}

int hpc_decode_suggest_num_ctas(const int32_t* h_seq_lens, int batch, int num_kv_heads, int min_chunks_per_cta,
                                int kv_dtype, int q_len) {
    if (!h_seq_lens || !sizes_ok(batch, num_kv_heads, 1) || min_chunks_per_cta < 0) return 0;
    if (kv_dtype != HPC_KV_BF16 && kv_dtype != HPC_KV_FP8_E4M3) return 0;
    if (q_len < 1 || q_len > HPC_MAX_Q_LEN) return 0;
    const bool fp8 = kv_dtype == HPC_KV_FP8_E4M3;
    const int deep = attn_default_ctas(fp8);
    if (deep <= 0 || q_len > 1) return deep;  // the multi-token kernels keep one CTA per SM
    // chunk counts per request and the total over the head-major walk
    long long per_head = 0;
    for (int b = 0; b < batch; ++b) per_head += h_seq_lens[b] > 0 ? (h_seq_lens[b] + kChunk - 1) / kChunk : 0;
    const long long T = per_head * num_kv_heads;
    if (T == 0) return deep;
    const long long bucket = std::max<long long>({(T + deep - 1) / deep, (long long)min_chunks_per_cta, 1LL});
    // descriptors per CTA of the deep plan: pair (h, b) with chunks [g0, g0 + n) of
    // the walk has one descriptor in every CTA its range touches; every head
    // walks the same requests, so the walk is a head's run repeated
    std::vector<int> desc((size_t)deep + 1, 0);
    long long g0 = 0;
    int most = 0;
    for (int h = 0; h < num_kv_heads; ++h) {
        for (int b = 0; b < batch; ++b) {
            const int L = h_seq_lens[b];
            const long long n = L > 0 ? (L + kChunk - 1) / kChunk : 0;
            if (n == 0) continue;
            const long long c0 = g0 / bucket, c1 = (g0 + n - 1) / bucket;
            for (long long c = c0; c <= c1 && c <= deep; ++c) most = std::max(most, ++desc[(size_t)c]);
            g0 += n;
        }
    }
    // Each descriptor costs its CTA a fixed amount (query staging, the merge of
    // its warps' states, the partial's write) on top of its chunks; where that
    // is a sizable share of the busiest CTA's work, two CTAs per SM halve the
    // lists and overlap one CTA's merges with the other's loads. Otherwise one
    // CTA per SM: more CTAs only add partials to combine.
    if (most < kFewDescriptors || 100LL * most < (long long)kDescriptorsPerChunkPct * bucket) return deep;
    const int shallow = attn_shallow_ctas(fp8);
    return shallow > deep ? shallow : deep;
}

hpc_status hpc_decode_plan(const int32_t* d_seq_lens, int batch, int num_kv_heads, int num_ctas,
                           int min_chunks_per_cta, hpc_plan* plan, void* stream) {
    if (!d_seq_lens || !plan || !plan->buf || min_chunks_per_cta < 0) return HPC_ERR_INVALID_ARG;
    if (!sizes_ok(batch, num_kv_heads, num_ctas)) return HPC_ERR_INVALID_ARG;
    if ((long long)num_kv_heads * batch > HPC_MAX_CTAS || !aligned(plan->buf, 16)) return HPC_ERR_INVALID_ARG;
    if (plan->bytes < plan_bytes_ll(batch, num_kv_heads, num_ctas)) return HPC_ERR_WORKSPACE_TOO_SMALL;
    plan->batch = batch;
    plan->num_kv_heads = num_kv_heads;
    plan->num_ctas = num_ctas;
    plan->min_chunks = min_chunks_per_cta;
    plan->mode = 0;
    plan->max_tasks = (int)plan_layout(batch, num_kv_heads, num_ctas).max_tasks;
    cudaError_t e = launch_plan(d_seq_lens, batch, num_kv_heads, num_ctas, min_chunks_per_cta, plan->buf,
                                static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? HPC_OK : HPC_ERR_CUDA;
}

hpc_status hpc_decode_plan_static(const int32_t* d_seq_lens, int batch, int num_kv_heads, int num_splits,
                                  hpc_plan* plan, void* stream) {
    if (!d_seq_lens || !plan || !plan->buf || num_splits < 1) return HPC_ERR_INVALID_ARG;
    const long long C = (long long)num_kv_heads * batch * num_splits;
    if (!sizes_ok(batch, num_kv_heads, C) || !aligned(plan->buf, 16)) return HPC_ERR_INVALID_ARG;
    if (plan->bytes < plan_bytes_ll(batch, num_kv_heads, C)) return HPC_ERR_WORKSPACE_TOO_SMALL;
    plan->batch = batch;
    plan->num_kv_heads = num_kv_heads;
    plan->num_ctas = (int)C;
    plan->min_chunks = num_splits;
    plan->mode = 1;
    plan->max_tasks = (int)plan_layout(batch, num_kv_heads, C).max_tasks;
    cudaError_t e = launch_plan_static(d_seq_lens, batch, num_kv_heads, num_splits, plan->buf,
                                       static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? HPC_OK : HPC_ERR_CUDA;
}

}  // extern "C"

namespace {

// Engine used by HPC_ENGINE_AUTO, as measured on GB300 (median attention
// launch on the full batches). bf16 (mixed-length batch): the warp-level
// kernels are fastest for one and two new tokens (367 / 389 us against
// 389 / 391 us), the tcgen05 kernel from three on (about 395 us for any q_len,
// against 440 us at three and 831 us at six). e4m3 (the long-context batch):
// the warp-level kernels for one and two new tokens (1309 / 1777 us), the
// tcgen05 kernel from three (about 2165 us for any q_len, against 3252 us at
// three, 4660 at six and 6954 at eight).
int multi_engine_for(bool fp8, int q_len) {
    if (fp8) return q_len >= 3 ? HPC_ENGINE_TCGEN05 : HPC_ENGINE_MMA_SYNC;
    return q_len >= 3 ? HPC_ENGINE_TCGEN05 : HPC_ENGINE_MMA_SYNC;
}

// The checks of an attention call on everything but the task map and the
// split buffers.
hpc_status attn_inputs_check(const void* q, const float* q_scale, const void* k_cache, const void* v_cache,
                             const float* k_scale, const float* v_scale, int kv_dtype, int num_pages,
                             const int32_t* page_table, int page_table_stride, const int32_t* seq_lens,
                             int num_q_heads, int num_kv_heads, int head_dim, int page_size) {
    hpc_status st = shape_check(num_q_heads, num_kv_heads, head_dim, page_size);
    if (st != HPC_OK) return st;
    if (kv_dtype != HPC_KV_BF16 && kv_dtype != HPC_KV_FP8_E4M3) return HPC_ERR_UNSUPPORTED;
    const bool fp8 = kv_dtype == HPC_KV_FP8_E4M3;
    if (!q || !k_cache || !v_cache || !page_table || !seq_lens) return HPC_ERR_INVALID_ARG;
    if (fp8 && (!k_scale || !v_scale)) return HPC_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16)) return HPC_ERR_INVALID_ARG;
    if (fp8 && (!aligned(k_scale, 16) || !aligned(v_scale, 16))) return HPC_ERR_INVALID_ARG;
    if (num_pages < 1 || (long long)num_pages * kChunk > 2147483647LL || page_table_stride < 1)
        return HPC_ERR_INVALID_ARG;
    if (fp8 && (long long)num_pages * num_kv_heads > 2147483647LL) return HPC_ERR_INVALID_ARG;
    if (q_scale && (!fp8 || !aligned(q_scale, 16))) return fp8 ? HPC_ERR_INVALID_ARG : HPC_ERR_UNSUPPORTED;
    return HPC_OK;
}

// Shared by hpc_decode_attn (bf16 Q), hpc_decode_attn_q8 (e4m3 Q + scales)
// and hpc_decode_attn_multi (q_len bf16 query rows per request).
hpc_status attn_common(const void* q, const float* q_scale, const void* k_cache, const void* v_cache,
                       const float* k_scale, const float* v_scale, int kv_dtype, int num_pages,
                       const int32_t* page_table, int page_table_stride, const int32_t* seq_lens, int batch,
                       int num_q_heads, int num_kv_heads, int head_dim, int page_size, const hpc_plan* plan,
                       float* split_o, float* split_lse, void* stream, int q_len = 1,
                       int engine = HPC_ENGINE_AUTO, int flags = 0) {
    hpc_status st = attn_inputs_check(q, q_scale, k_cache, v_cache, k_scale, v_scale, kv_dtype, num_pages,
                                      page_table, page_table_stride, seq_lens, num_q_heads, num_kv_heads,
                                      head_dim, page_size);
    if (st != HPC_OK) return st;
    const bool fp8 = kv_dtype == HPC_KV_FP8_E4M3;
    if (!split_o || !split_lse || !aligned(split_o, 16)) return HPC_ERR_INVALID_ARG;
    if ((st = plan_check(plan, batch, num_kv_heads)) != HPC_OK) return st;
    if (q_len < 1 || q_len > HPC_MAX_Q_LEN || (q_len > 1 && q_scale)) return HPC_ERR_INVALID_ARG;
    if (engine < HPC_ENGINE_AUTO || engine > HPC_ENGINE_TCGEN05) return HPC_ERR_INVALID_ARG;
    if (flags & ~(HPC_ATTN_EARLY_KV | HPC_ATTN_TEST_WAIT_EXPIRY)) return HPC_ERR_INVALID_ARG;
    AttnArgs a;
    a.q = q;
    a.q_scale = q_scale;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.k_scale = fp8 ? k_scale : nullptr;
    a.v_scale = fp8 ? v_scale : nullptr;
    a.fp8 = fp8;
    a.num_pages = num_pages;
    a.page_table = page_table;
    a.pt_stride = page_table_stride;
    a.seq_lens = seq_lens;
    a.batch = batch;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.plan = plan->buf;
    a.num_ctas = plan->num_ctas;
    a.mode = plan->mode;
    a.split_cap = (long long)hpc_decode_split_capacity(batch, num_kv_heads, plan->num_ctas);
    a.split_o = split_o;
    a.split_lse = split_lse;
    a.early_kv = (flags & HPC_ATTN_EARLY_KV) ? 1 : 0;
    a.test_wait_expiry = (flags & HPC_ATTN_TEST_WAIT_EXPIRY) ? 1 : 0;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (engine == HPC_ENGINE_AUTO) engine = multi_engine_for(fp8, q_len);
    // the failure-path test exists in the one-token kernel only
    if (a.test_wait_expiry && (q_len != 1 || engine == HPC_ENGINE_TCGEN05)) return HPC_ERR_UNSUPPORTED;
    cudaError_t e;
    if (engine == HPC_ENGINE_TCGEN05)
        e = launch_attn_tc(a, q_len, cs);
    else
        e = q_len == 1 ? launch_attn(a, cs) : launch_attn_mt(a, q_len, cs);
    if (e == cudaErrorInvalidValue) return HPC_ERR_INVALID_ARG;
    return e == cudaSuccess ? HPC_OK : HPC_ERR_CUDA;
}

}  // namespace

// Every host-side check that hpc_decode_plan, hpc_decode_attn and
// hpc_decode_combine make for one step with one new token per request, except
// those on the task map and split buffers the caller does not provide.
hpc_status hpc::step_args_check(const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
                                const float* v_scale, int kv_dtype, int num_pages, const int32_t* page_table,
                                int page_table_stride, const int32_t* seq_lens, int batch, int num_q_heads,
                                int num_kv_heads, int head_dim, int page_size, int num_ctas,
                                int min_chunks_per_cta, const void* out) {
    if (min_chunks_per_cta < 0 || !sizes_ok(batch, num_kv_heads, num_ctas)) return HPC_ERR_INVALID_ARG;
    if ((long long)num_kv_heads * batch > HPC_MAX_CTAS) return HPC_ERR_INVALID_ARG;
    hpc_status st = attn_inputs_check(q, nullptr, k_cache, v_cache, k_scale, v_scale, kv_dtype, num_pages,
                                      page_table, page_table_stride, seq_lens, num_q_heads, num_kv_heads,
                                      head_dim, page_size);
    if (st != HPC_OK) return st;
    if (!out || !aligned(out, 8)) return HPC_ERR_INVALID_ARG;
    return HPC_OK;
}

extern "C" {

hpc_status hpc_decode_attn(const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
                           const float* v_scale, int kv_dtype, int num_pages, const int32_t* page_table,
                           int page_table_stride, const int32_t* seq_lens, int batch, int num_q_heads,
                           int num_kv_heads, int head_dim, int page_size, const hpc_plan* plan,
                           float* split_o, float* split_lse, void* stream) {
    return attn_common(q, nullptr, k_cache, v_cache, k_scale, v_scale, kv_dtype, num_pages, page_table,
                       page_table_stride, seq_lens, batch, num_q_heads, num_kv_heads, head_dim, page_size, plan,
                       split_o, split_lse, stream);
}

hpc_status hpc_decode_attn_q8(const void* q8, const float* q_scale, const void* k_cache, const void* v_cache,
                              const float* k_scale, const float* v_scale, int num_pages,
                              const int32_t* page_table, int page_table_stride, const int32_t* seq_lens,
                              int batch, int num_q_heads, int num_kv_heads, int head_dim, int page_size,
                              const hpc_plan* plan, float* split_o, float* split_lse, void* stream) {
    if (!q_scale) return HPC_ERR_INVALID_ARG;
    return attn_common(q8, q_scale, k_cache, v_cache, k_scale, v_scale, HPC_KV_FP8_E4M3, num_pages, page_table,
                       page_table_stride, seq_lens, batch, num_q_heads, num_kv_heads, head_dim, page_size, plan,
                       split_o, split_lse, stream);
}

hpc_status hpc_decode_attn_multi(const void* q, int q_len, const void* k_cache, const void* v_cache,
                                 const float* k_scale, const float* v_scale, int kv_dtype, int num_pages,
                                 const int32_t* page_table, int page_table_stride, const int32_t* seq_lens,
                                 int batch, int num_q_heads, int num_kv_heads, int head_dim, int page_size,
                                 const hpc_plan* plan, float* split_o, float* split_lse, void* stream) {
    if (q_len < 1 || q_len > HPC_MAX_Q_LEN) return HPC_ERR_INVALID_ARG;
    return attn_common(q, nullptr, k_cache, v_cache, k_scale, v_scale, kv_dtype, num_pages, page_table,
                       page_table_stride, seq_lens, batch, num_q_heads, num_kv_heads, head_dim, page_size, plan,
                       split_o, split_lse, stream, q_len);
}

int hpc_decode_attn_multi_auto_engine(int kv_dtype, int q_len) {
    if (kv_dtype != HPC_KV_BF16 && kv_dtype != HPC_KV_FP8_E4M3) return 0;
    if (q_len < 1 || q_len > HPC_MAX_Q_LEN) return 0;
    return multi_engine_for(kv_dtype == HPC_KV_FP8_E4M3, q_len);
}

hpc_status hpc_decode_attn_multi_engine(const void* q, int q_len, const void* k_cache, const void* v_cache,
                                        const float* k_scale, const float* v_scale, int kv_dtype, int num_pages,
                                        const int32_t* page_table, int page_table_stride, const int32_t* seq_lens,
                                        int batch, int num_q_heads, int num_kv_heads, int head_dim, int page_size,
                                        const hpc_plan* plan, float* split_o, float* split_lse, int engine,
                                        void* stream) {
    if (q_len < 1 || q_len > HPC_MAX_Q_LEN) return HPC_ERR_INVALID_ARG;
    return attn_common(q, nullptr, k_cache, v_cache, k_scale, v_scale, kv_dtype, num_pages, page_table,
                       page_table_stride, seq_lens, batch, num_q_heads, num_kv_heads, head_dim, page_size, plan,
                       split_o, split_lse, stream, q_len, engine);
}

hpc_status hpc_decode_attn_ex(const void* q, const float* q_scale, int q_len, const void* k_cache,
                              const void* v_cache, const float* k_scale, const float* v_scale, int kv_dtype,
                              int num_pages, const int32_t* page_table, int page_table_stride,
                              const int32_t* seq_lens, int batch, int num_q_heads, int num_kv_heads, int head_dim,
                              int page_size, const hpc_plan* plan, float* split_o, float* split_lse, int engine,
                              int flags, void* stream) {
    if (q_len < 1 || q_len > HPC_MAX_Q_LEN) return HPC_ERR_INVALID_ARG;
    return attn_common(q, q_scale, k_cache, v_cache, k_scale, v_scale, kv_dtype, num_pages, page_table,
                       page_table_stride, seq_lens, batch, num_q_heads, num_kv_heads, head_dim, page_size, plan,
                       split_o, split_lse, stream, q_len, engine, flags);
}

hpc_status hpc_decode_combine_multi(const hpc_plan* plan, int q_len, const float* split_o, const float* split_lse,
                                    void* out, float* out_lse, int batch, int num_q_heads, int num_kv_heads,
                                    int head_dim, void* stream) {
    hpc_status st = shape_check(num_q_heads, num_kv_heads, head_dim, kChunk);
    if (st != HPC_OK) return st;
    if (q_len < 1 || q_len > HPC_MAX_Q_LEN) return HPC_ERR_INVALID_ARG;
    if (!split_o || !split_lse || !out || !aligned(split_o, 16) || !aligned(out, 8)) return HPC_ERR_INVALID_ARG;
    if ((st = plan_check(plan, batch, num_kv_heads)) != HPC_OK) return st;
    cudaError_t e = launch_combine(plan->buf, plan->num_ctas, split_o, split_lse,
                                   static_cast<__nv_bfloat16*>(out), out_lse, batch, num_q_heads, num_kv_heads,
                                   q_len, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? HPC_OK : HPC_ERR_CUDA;
}

hpc_status hpc_decode_combine(const hpc_plan* plan, const float* split_o, const float* split_lse, void* out,
                              float* out_lse, int batch, int num_q_heads, int num_kv_heads, int head_dim,
                              void* stream) {
    return hpc_decode_combine_multi(plan, 1, split_o, split_lse, out, out_lse, batch, num_q_heads, num_kv_heads,
                                    head_dim, stream);
}

hpc_status hpc_rope_norm(const void* qkv, const int32_t* positions, const float* cos_sin, int max_pos,
                         const float* q_weight, const float* k_weight, float eps, const int32_t* slot_mapping,
                         int num_tokens, int num_q_heads, int num_kv_heads, int head_dim, int page_size,
                         void* q_out, float* q_scale_out, void* k_cache, void* v_cache, float* k_scale,
                         float* v_scale, int kv_dtype, int num_pages, int* d_error_word, void* stream) {
    if (head_dim != kHeadDim || page_size != kChunk) return HPC_ERR_UNSUPPORTED;
    if (kv_dtype != HPC_KV_BF16 && kv_dtype != HPC_KV_FP8_E4M3) return HPC_ERR_UNSUPPORTED;
    if (num_tokens < 0 || num_q_heads < 1 || num_kv_heads < 1 || num_kv_heads > HPC_MAX_KV_HEADS ||
        num_q_heads > 4096 || max_pos < 1 || num_pages < 1 || !(eps >= 0.f))
        return HPC_ERR_INVALID_ARG;
    const bool fp8 = kv_dtype == HPC_KV_FP8_E4M3;
    if (!qkv || !positions || !cos_sin || !q_weight || !k_weight || !slot_mapping || !q_out || !k_cache ||
        !v_cache)
        return HPC_ERR_INVALID_ARG;
    if (fp8 && (!k_scale || !v_scale)) return HPC_ERR_INVALID_ARG;
    if (!aligned(qkv, 16) || !aligned(cos_sin, 16) || !aligned(q_weight, 16) || !aligned(k_weight, 16) ||
        !aligned(q_out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
        return HPC_ERR_INVALID_ARG;
    if ((long long)num_pages * kChunk * num_kv_heads > (1LL << 40)) return HPC_ERR_INVALID_ARG;
    if (num_tokens == 0) return HPC_OK;
    RopeNormArgs a;
    a.qkv = qkv;
    a.positions = positions;
    a.cos_sin = cos_sin;
    a.max_pos = max_pos;
    a.q_weight = q_weight;
    a.k_weight = k_weight;
    a.eps = eps;
    a.slots = slot_mapping;
    a.num_tokens = num_tokens;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.q_out = q_out;
    a.q_scale = q_scale_out;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.k_scale = fp8 ? k_scale : nullptr;
    a.v_scale = fp8 ? v_scale : nullptr;
    a.num_pages = num_pages;
    a.kv_fp8 = fp8;
    a.err = d_error_word;
    return launch_rope_norm(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? HPC_OK : HPC_ERR_CUDA;
}

size_t hpc_decode_step_workspace_bytes(int batch, int num_q_heads, int num_kv_heads, int page_table_stride,
                                       int num_ctas) {
    if (!sizes_ok(batch, num_kv_heads, num_ctas) || page_table_stride < 1 || num_q_heads < 1) return 0;
    return step_workspace(batch, num_q_heads, num_kv_heads, page_table_stride, num_ctas).total;
}

hpc_status hpc_decode_step_host(const void* h_q, const int32_t* h_seq_lens, const int32_t* h_page_table,
                                int page_table_stride, const void* d_k_cache, const void* d_v_cache,
                                const float* d_k_scale, const float* d_v_scale, int kv_dtype, int num_pages,
                                int batch, int num_q_heads, int num_kv_heads, int head_dim, int page_size,
                                int num_ctas, int min_chunks_per_cta, void* d_workspace,
                                size_t workspace_bytes, void* h_out, float* h_out_lse, void* stream) {
    hpc_status st = shape_check(num_q_heads, num_kv_heads, head_dim, page_size);
    if (st != HPC_OK) return st;
    if (!h_q || !h_seq_lens || !h_page_table || !d_workspace || !h_out) return HPC_ERR_INVALID_ARG;
    if (!sizes_ok(batch, num_kv_heads, num_ctas) || page_table_stride < 1 || !aligned(d_workspace, 256))
        return HPC_ERR_INVALID_ARG;
    const StepWorkspace w = step_workspace(batch, num_q_heads, num_kv_heads, page_table_stride, num_ctas);
    if (workspace_bytes < w.total) return HPC_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(d_workspace);
    const size_t q_bytes = (size_t)batch * num_q_heads * kHeadDim * 2;
    const size_t pt_bytes = (size_t)batch * page_table_stride * 4;
    // Page-locked, device-mapped host buffers are read and written by the
    // kernels themselves (one staging kernel in, the combine out); any other
    // host memory goes through the copy engine.
    void* m_q = mapped_host(h_q);
    void* m_sl = mapped_host(h_seq_lens);
    void* m_pt = mapped_host(h_page_table);
    void* m_out = mapped_host(h_out);
    void* m_lse = h_out_lse ? mapped_host(h_out_lse) : nullptr;
    const bool zero_copy = m_q && m_sl && m_pt && m_out && (!h_out_lse || m_lse) && aligned(m_out, 8);
    if (zero_copy) {
        const StageCopy cq{static_cast<const uint8_t*>(m_q), ws + w.q, q_bytes};
        const StageCopy csl{static_cast<const uint8_t*>(m_sl), ws + w.seq_lens, (size_t)batch * 4};
        const StageCopy cpt{static_cast<const uint8_t*>(m_pt), ws + w.page_table, pt_bytes};
        if (launch_stage_in(cq, csl, cpt, s) != cudaSuccess) return HPC_ERR_CUDA;
    } else if (cudaMemcpyAsync(ws + w.q, h_q, q_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess ||
               cudaMemcpyAsync(ws + w.seq_lens, h_seq_lens, (size_t)batch * 4, cudaMemcpyHostToDevice, s) !=
                   cudaSuccess ||
               cudaMemcpyAsync(ws + w.page_table, h_page_table, pt_bytes, cudaMemcpyHostToDevice, s) !=
                   cudaSuccess) {
        return HPC_ERR_CUDA;
    }
    hpc_plan plan{};
    plan.buf = reinterpret_cast<int32_t*>(ws + w.plan);
    plan.bytes = hpc_decode_plan_bytes(batch, num_kv_heads, num_ctas);
    const int32_t* d_sl = reinterpret_cast<const int32_t*>(ws + w.seq_lens);
    if ((st = hpc_decode_plan(d_sl, batch, num_kv_heads, num_ctas, min_chunks_per_cta, &plan, stream)) != HPC_OK)
        return st;
    float* so = reinterpret_cast<float*>(ws + w.split_o);
    float* sl = reinterpret_cast<float*>(ws + w.split_lse);
    if ((st = hpc_decode_attn(ws + w.q, d_k_cache, d_v_cache, d_k_scale, d_v_scale, kv_dtype, num_pages,
                              reinterpret_cast<const int32_t*>(ws + w.page_table), page_table_stride, d_sl,
                              batch, num_q_heads, num_kv_heads, head_dim, page_size, &plan, so, sl, stream)) !=
        HPC_OK)
        return st;
    float* d_lse = reinterpret_cast<float*>(ws + w.out_lse);
    if (zero_copy) {
        return hpc_decode_combine(&plan, so, sl, m_out, static_cast<float*>(m_lse), batch, num_q_heads,
                                  num_kv_heads, head_dim, stream);
    }
    if ((st = hpc_decode_combine(&plan, so, sl, ws + w.out, d_lse, batch, num_q_heads, num_kv_heads, head_dim,
                                 stream)) != HPC_OK)
        return st;
    if (cudaMemcpyAsync(h_out, ws + w.out, q_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess) return HPC_ERR_CUDA;
    if (h_out_lse &&
        cudaMemcpyAsync(h_out_lse, d_lse, (size_t)batch * num_q_heads * 4, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return HPC_ERR_CUDA;
    return HPC_OK;
}

}  // extern "C"

struct hpc_step_graph {
    cudaGraphExec_t exec;
};

extern "C" {

hpc_status hpc_decode_step_graph_create(const void* h_q, const int32_t* h_seq_lens, const int32_t* h_page_table,
                                        int page_table_stride, const void* d_k_cache, const void* d_v_cache,
                                        const float* d_k_scale, const float* d_v_scale, int kv_dtype,
                                        int num_pages, int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                        int page_size, int num_ctas, int min_chunks_per_cta, void* d_workspace,
                                        size_t workspace_bytes, void* h_out, float* h_out_lse,
                                        hpc_step_graph** graph) {
    if (!graph) return HPC_ERR_INVALID_ARG;
    *graph = nullptr;
    // the checks of hpc_decode_step_host, before any CUDA call
    hpc_status st = shape_check(num_q_heads, num_kv_heads, head_dim, page_size);
    if (st != HPC_OK) return st;
    if (kv_dtype != HPC_KV_BF16 && kv_dtype != HPC_KV_FP8_E4M3) return HPC_ERR_UNSUPPORTED;
    if (!h_q || !h_seq_lens || !h_page_table || !d_workspace || !h_out) return HPC_ERR_INVALID_ARG;
    if (!sizes_ok(batch, num_kv_heads, num_ctas) || page_table_stride < 1 || !aligned(d_workspace, 256))
        return HPC_ERR_INVALID_ARG;
    if (workspace_bytes < step_workspace(batch, num_q_heads, num_kv_heads, page_table_stride, num_ctas).total)
        return HPC_ERR_WORKSPACE_TOO_SMALL;
    // one-time launcher setup (kernel attributes) outside the capture
    if (attn_default_ctas(kv_dtype == HPC_KV_FP8_E4M3) <= 0) return HPC_ERR_CUDA;
    cudaStream_t cs = nullptr;
    if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) return HPC_ERR_CUDA;
    cudaGraph_t g = nullptr;
    if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
        cudaStreamDestroy(cs);
        return HPC_ERR_CUDA;
    }
    st = hpc_decode_step_host(h_q, h_seq_lens, h_page_table, page_table_stride, d_k_cache, d_v_cache, d_k_scale,
                              d_v_scale, kv_dtype, num_pages, batch, num_q_heads, num_kv_heads, head_dim,
                              page_size, num_ctas, min_chunks_per_cta, d_workspace, workspace_bytes, h_out,
                              h_out_lse, cs);
    const cudaError_t ce = cudaStreamEndCapture(cs, &g);
    cudaStreamDestroy(cs);
    if (st != HPC_OK || ce != cudaSuccess) {
        if (g) cudaGraphDestroy(g);
        (void)cudaGetLastError();
        return st != HPC_OK ? st : HPC_ERR_CUDA;
    }
    cudaGraphExec_t exec = nullptr;
    const cudaError_t ie = cudaGraphInstantiate(&exec, g, 0);
    cudaGraphDestroy(g);
    if (ie != cudaSuccess) {
        (void)cudaGetLastError();
        return HPC_ERR_CUDA;
    }
    hpc_step_graph* out = new (std::nothrow) hpc_step_graph{exec};
    if (!out) {
        cudaGraphExecDestroy(exec);
        return HPC_ERR_CUDA;
    }
    *graph = out;
    return HPC_OK;
}

hpc_status hpc_decode_step_graph_launch(hpc_step_graph* graph, void* stream) {
    if (!graph || !graph->exec) return HPC_ERR_INVALID_ARG;
    return cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream)) == cudaSuccess ? HPC_OK : HPC_ERR_CUDA;
}

hpc_status hpc_decode_step_graph_destroy(hpc_step_graph* graph) {
    if (!graph) return HPC_OK;
    const cudaError_t e = graph->exec ? cudaGraphExecDestroy(graph->exec) : cudaSuccess;
    delete graph;
    return e == cudaSuccess ? HPC_OK : HPC_ERR_CUDA;
}

hpc_status hpc_decode_read_error(const hpc_plan* plan, int* device_error_word) {
    if (!plan || !plan->buf || !device_error_word) return HPC_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return HPC_ERR_CUDA;
    int w = 0;
    if (cudaMemcpy(&w, plan->buf + kHError, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return HPC_ERR_CUDA;
    *device_error_word = w;
    return w ? HPC_ERR_DEVICE_CHECK : HPC_OK;
}

const char* hpc_status_string(hpc_status status) {
    switch (status) {
        case HPC_OK: return "ok";
        case HPC_ERR_INVALID_ARG: return "invalid argument";
        case HPC_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case HPC_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case HPC_ERR_CUDA: return "CUDA launch or copy failed";
        case HPC_ERR_DEVICE_CHECK: return "device-side check failed (see the error word)";
    }
    return "unknown status";
}

}  // extern "C"
