/*
 * hpc_decode.h - C ABI of the load-balanced paged GQA decode attention
 * library for NVIDIA GB300 (sm_103a).
 *
 * The method (two blog posts on the HPC-Ops attention backend):
 *   [SGL]  "HPC-Ops, integrated into SGLang", sections "Attention: load
 *          balancing for mixed-length decode" and "Scheduling around live KV
 *          work".
 *   [VLLM] "vLLM x HPC-Ops: High-Performance Attention and MoE Backends from
 *          Tencent Hunyuan", sub-section "解决方案：按步负载均衡的 decode
 *          调度器" (assign -> compute and combine), and "关于 Hy3 系列模型的
 *          简要说明" (GQA shape: 64 query heads, 8 KV heads, head dim 128).
 *   [LL]   "SGLang Low-Latency Mode: Kernels and Runtime", section "Where the
 *          Time Goes" (several verified token rows per request and step).
 *
 * One decode step is three calls on one stream:
 *   hpc_decode_plan     once per step: live lengths -> task map (reused by
 *                       every layer of the step)
 *   hpc_decode_attn     per layer: persistent grid drains the task map and
 *                       writes one partial output + LSE per descriptor
 *   hpc_decode_combine  per layer: LSE-weighted merge into the BF16 output
 *
 * Conventions for every call:
 *   - Pointers named d_* or documented as "device" are device pointers; h_*
 *     are host pointers. The caller owns all memory. The library never
 *     allocates, frees or synchronises inside these calls (except
 *     hpc_decode_read_error, which synchronises by design, and
 *     hpc_decode_step_graph_create / _destroy, which allocate and free a
 *     captured step).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Work is enqueued asynchronously on it.
 *   - Supported shapes: head_dim == 128, page_size == 64 (one chunk is one
 *     page), num_q_heads == 8 * num_kv_heads. Anything else returns
 *     HPC_ERR_UNSUPPORTED before any work is enqueued.
 *   - Host-side argument checks return HPC_ERR_INVALID_ARG and enqueue
 *     nothing. Launch failures return HPC_ERR_CUDA. No call traps or aborts.
 *   - Device-side checks (negative length, page id out of range, a
 *     descriptor outside the shapes, a bounded wait that ran out) set bits in
 *     the error word stored in the task map (HPC_DEVERR_*) and skip the
 *     offending work; read it with hpc_decode_read_error.
 *
 * Data layouts (row-major, contiguous):
 *   q          bf16 [batch][num_q_heads][128]; query head qh belongs to KV
 *              head qh / 8 (contiguous GQA groups).
 *   k_cache,   [num_pages][64][num_kv_heads][128], bf16 or e4m3 (OCP
 *   v_cache    e4m3fn). Token t of request b lives in page
 *              page_table[b * page_table_stride + t / 64], slot t % 64.
 *   k_scale,   e4m3 caches only: float32 [num_pages][num_kv_heads][64], one
 *   v_scale    scale per (token, KV head); the value is code * scale.
 *   page_table int32 [batch][page_table_stride]; only entries
 *              [0, ceil(seq_lens[b] / 64)) of row b are read.
 *   seq_lens   int32 [batch], live KV length of each request (>= 0).
 *   split_o    float32 [split_capacity][8][128]: normalised partial output of
 *              each descriptor for the 8 query heads of its KV head.
 *   split_lse  float32 [split_capacity][8]: natural-log LSE of each partial
 *              (scores scaled by 1/sqrt(128)).
 *   out        bf16 [batch][num_q_heads][128] (round to nearest even).
 *   out_lse    float32 [batch][num_q_heads] (nullable). A request of length 0
 *              gets out = 0 and out_lse = -inf.
 */
#ifndef HPC_DECODE_H
#define HPC_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum hpc_status {
    HPC_OK = 0,
    HPC_ERR_INVALID_ARG = 1,
    HPC_ERR_UNSUPPORTED = 2,
    HPC_ERR_WORKSPACE_TOO_SMALL = 3,
    HPC_ERR_CUDA = 4,
    HPC_ERR_DEVICE_CHECK = 5
} hpc_status;

typedef enum hpc_kv_dtype { HPC_KV_BF16 = 0, HPC_KV_FP8_E4M3 = 1 } hpc_kv_dtype;

/* Bits of the device error word (hpc_decode_read_error). */
#define HPC_DEVERR_NEGATIVE_LENGTH 1u    /* planner saw seq_lens[b] < 0 (counted as 0) */
#define HPC_DEVERR_CHUNK_OVERFLOW 2u     /* chunk total over all heads exceeds INT32_MAX */
#define HPC_DEVERR_PAGE_OUT_OF_RANGE 4u  /* a page id outside [0, num_pages): chunk skipped */
#define HPC_DEVERR_WAIT_TIMEOUT 8u       /* a bounded wait inside the kernel ran out */
#define HPC_DEVERR_BAD_DESCRIPTOR 16u    /* a task descriptor outside the call's shapes */
#define HPC_DEVERR_BAD_POSITION 32u      /* prologue: a position outside [0, max_pos): not rotated */

/* Limits checked on the host. */
#define HPC_MAX_BATCH 16384
#define HPC_MAX_KV_HEADS 256
#define HPC_MAX_CTAS (1 << 22)
#define HPC_MAX_Q_LEN 8          /* new tokens per request in hpc_decode_attn_multi */

/*
 * Task map ([SGL] "Scheduling around live KV work": a global task map built
 * once per decode step from device-side lengths and reused across layers).
 * The caller fills `buf` (device memory of at least hpc_decode_plan_bytes)
 * and `bytes`; hpc_decode_plan / hpc_decode_plan_static fill the rest.
 *
 * Byte layout of buf (int32):
 *   [0, 16)            header {total_chunks, bucket, used_ctas, total_splits,
 *                      num_ctas, batch, num_kv_heads, min_chunks (or the
 *                      static split count), max_tasks, mode, chunks_per_head,
 *                      chunk_tokens (64), error word, 0, 0, 0}
 *   [16, 16 + C + 1)   first task row of each CTA's list; entry C = end
 *   tasks              32-byte aligned, max_tasks rows of 8 int32
 *                      {kv_head, request, chunk_begin, chunk_end, split,
 *                       rank_in_pair, splits_in_pair, 0}; each CTA's list is
 *                      closed by a row of -1 (terminator); unused rows are -1
 *   pair_nsplit        [num_kv_heads * batch], pair p = kv_head * batch + b
 *   pair_split0        [num_kv_heads * batch], first split of pair p
 *   max_tasks = num_kv_heads * batch + 2 * num_ctas.
 * The buffer is deterministic: the same lengths give the same bytes.
 */
typedef struct hpc_plan {
    int32_t* buf;      /* device, caller-owned */
    size_t bytes;      /* size of buf in bytes */
    int batch;         /* filled by the planner from here on */
    int num_kv_heads;
    int num_ctas;      /* grid size hpc_decode_attn launches */
    int min_chunks;    /* floor m (dynamic) or split count S (static) */
    int mode;          /* 0 load-balanced, 1 static split count */
    int max_tasks;
} hpc_plan;

/* Bytes of the task map for (batch, num_kv_heads, num_ctas); independent of
 * the lengths, so one buffer serves every step. 0 on invalid sizes. */
size_t hpc_decode_plan_bytes(int batch, int num_kv_heads, int num_ctas);

/* Rows needed in split_o / split_lse: num_kv_heads * batch + num_ctas - 1
 * (at least 1). A descriptor is a maximal run of one (kv head, request) inside
 * one bucket, so each used CTA adds at most one split beyond one per pair.
 * For a static plan pass num_ctas = num_kv_heads * batch * num_splits. */
size_t hpc_decode_split_capacity(int batch, int num_kv_heads, int num_ctas);

/* Persistent CTA count for the attention kernel on the current device:
 * SM count x resident CTAs per SM of the kernel instance for `kv_dtype`.
 * Returns 0 if the device cannot be queried. A plan for more CTAs than this
 * runs a shallower instance that keeps two CTAs per SM resident (up to twice
 * this count in one wave): finer buckets for batches of many short requests,
 * at the price of more partials for long ones. */
int hpc_decode_default_num_ctas(int kv_dtype);

/*
 * A CTA count to plan a batch for, from its lengths on the host (int32
 * [batch], host memory; nothing is enqueued). The pages leave the CTA count to
 * the caller ([SGL] "Scheduling around live KV work": the planner divides the
 * work by the number of CTAs). The rule: plan the batch for
 * hpc_decode_default_num_ctas(kv_dtype) CTAs (one per SM); if the CTA of that
 * plan with the most descriptors holds at least 4 of them and at least 0.15
 * per chunk of its budget (each descriptor costs a fixed amount beyond its
 * chunks, a sizable share there), return the count of the shallow instance
 * (two CTAs per SM), which halves such lists; otherwise the default count. With several new tokens per request (q_len >
 * 1) the default count. Any count gives the same outputs up to rounding; the
 * task map for each count is exact. Returns 0 for bad arguments or when the
 * device cannot be queried.
 */
int hpc_decode_suggest_num_ctas(const int32_t* h_seq_lens, int batch, int num_kv_heads,
                                int min_chunks_per_cta, int kv_dtype, int q_len);

/*
 * Load-balanced planner ([SGL] "Scheduling around live KV work"; [VLLM]
 * "解决方案：按步负载均衡的 decode 调度器", assign stage). For each request
 * n_b = ceil(seq_lens[b] / 64); T = num_kv_heads * sum(n_b);
 * bucket = max(ceil(T / num_ctas), min_chunks_per_cta, 1). Chunks are walked
 * kv head by kv head, request by request, chunk by chunk; global chunk g goes
 * to CTA g / bucket, and each maximal run of one (kv head, request) inside one
 * CTA is one descriptor. One block, integer only, reads d_seq_lens on the
 * device (no host synchronisation).
 *   d_seq_lens  device int32 [batch]
 *   plan        caller fills buf/bytes; other fields are written here
 * Errors: HPC_ERR_INVALID_ARG (null pointers, sizes outside the limits,
 * min_chunks_per_cta < 0), HPC_ERR_WORKSPACE_TOO_SMALL, HPC_ERR_CUDA.
 */
hpc_status hpc_decode_plan(const int32_t* d_seq_lens, int batch, int num_kv_heads, int num_ctas,
                           int min_chunks_per_cta, hpc_plan* plan, void* stream);

/*
 * Static split-KV comparison schedule ([SGL] "Attention: load balancing for
 * mixed-length decode", policy (1): a fixed split count). One virtual CTA per
 * (kv head, request, split s), num_ctas = num_kv_heads * batch * num_splits;
 * split s of a pair with n chunks covers [s*q, min((s+1)*q, n)) with
 * q = ceil(n / num_splits) and is empty when s*q >= n. Same layout and same
 * attention kernel as the load-balanced map.
 */
hpc_status hpc_decode_plan_static(const int32_t* d_seq_lens, int batch, int num_kv_heads,
                                  int num_splits, hpc_plan* plan, void* stream);

/*
 * Persistent decode attention ([SGL] "Scheduling around live KV work", the
 * paragraph on execution; [VLLM] compute stage). Launches plan->num_ctas CTAs;
 * CTA j walks its descriptor list until the terminator. For descriptor
 * (h, b, c0, c1, s) and each j < 8 it writes
 *   split_o[s][j][:]  = sum_t softmax_t(q[b][8h+j] . k_t / sqrt(128)) v_t
 *   split_lse[s][j]   = ln sum_t exp(q[b][8h+j] . k_t / sqrt(128))
 * over tokens t in [64*c0, min(64*c1, seq_lens[b])) of KV head h.
 *   q, k_cache, v_cache   device, 16-byte aligned (TMA sources)
 *   k_scale, v_scale      device float32, 16-byte aligned, e4m3 only (NULL
 *                         for bf16)
 *   num_pages             physical pages in each cache (page ids outside
 *                         [0, num_pages) set HPC_DEVERR_PAGE_OUT_OF_RANGE)
 *   seq_lens              device int32 [batch], the lengths the plan saw
 *   split_o, split_lse    device float32, hpc_decode_split_capacity rows
 * Errors: HPC_ERR_INVALID_ARG, HPC_ERR_UNSUPPORTED, HPC_ERR_CUDA.
 */
hpc_status hpc_decode_attn(const void* q, const void* k_cache, const void* v_cache,
                           const float* k_scale, const float* v_scale, int kv_dtype, int num_pages,
                           const int32_t* page_table, int page_table_stride,
                           const int32_t* seq_lens, int batch, int num_q_heads, int num_kv_heads,
                           int head_dim, int page_size, const hpc_plan* plan, float* split_o,
                           float* split_lse, void* stream);

/*
 * Persistent decode attention with an e4m3 query ([SGL] "A fused attention
 * prologue": the prologue emits Q in FP8 with one scale per token and head
 * and passes both to the attention kernel, which does not requantise). Same
 * task map, cache, outputs and errors as hpc_decode_attn with
 * kv_dtype = HPC_KV_FP8_E4M3; the query is q8[b][qh][d] * q_scale[b][qh].
 *   q8        device e4m3 codes [batch][num_q_heads][128], 16-byte aligned
 *   q_scale   device float32 [batch][num_q_heads], 16-byte aligned, not NULL
 * QK^T multiplies the K and Q codes, both widened exactly to f16, with float32
 * accumulation (exact products: the same values as e4m3 x e4m3 products); the
 * scores are then multiplied by the K and Q scales.
 */
hpc_status hpc_decode_attn_q8(const void* q8, const float* q_scale, const void* k_cache,
                              const void* v_cache, const float* k_scale, const float* v_scale,
                              int num_pages, const int32_t* page_table, int page_table_stride,
                              const int32_t* seq_lens, int batch, int num_q_heads,
                              int num_kv_heads, int head_dim, int page_size, const hpc_plan* plan,
                              float* split_o, float* split_lse, void* stream);

/*
 * Persistent decode attention for q_len new tokens per request, the rows that
 * speculative decoding verifies in one step ([LL] "SGLang Low-Latency Mode:
 * Kernels and Runtime", section "Where the Time Goes": six token rows per
 * step; [VLLM] Hy3: an MTP layer for speculative decoding). Same task map,
 * caches and errors as hpc_decode_attn; the plan does not depend on q_len.
 * The pages give no mask; the causal reading is taken: the q_len new tokens
 * are already in the cache and counted by seq_lens, and new token i of
 * request b attends to tokens [0, seq_lens[b] - q_len + i]. For descriptor
 * (h, b, c0, c1, s), new token i and j < 8 it writes row (s * q_len + i) * 8 + j:
 *   split_o[.][:]  = normalised attention of q[b][i][8h+j] over tokens
 *                    [64*c0, min(64*c1, seq_lens[b] - q_len + i + 1))
 *   split_lse[.]   = its natural-log LSE (-inf and 0 outputs when empty)
 *   q          device bf16 [batch][q_len][num_q_heads][128], 16-byte aligned
 *   q_len      1 <= q_len <= HPC_MAX_Q_LEN (1 runs hpc_decode_attn's kernel)
 *   split_o    device float32 [split_capacity][q_len][8][128]
 *   split_lse  device float32 [split_capacity][q_len][8]
 * Errors: HPC_ERR_INVALID_ARG (also q_len out of range), HPC_ERR_UNSUPPORTED,
 * HPC_ERR_CUDA.
 */
hpc_status hpc_decode_attn_multi(const void* q, int q_len, const void* k_cache, const void* v_cache,
                                 const float* k_scale, const float* v_scale, int kv_dtype, int num_pages,
                                 const int32_t* page_table, int page_table_stride,
                                 const int32_t* seq_lens, int batch, int num_q_heads,
                                 int num_kv_heads, int head_dim, int page_size, const hpc_plan* plan,
                                 float* split_o, float* split_lse, void* stream);

/* Kernels behind hpc_decode_attn_multi_engine. */
#define HPC_ENGINE_AUTO 0       /* the faster one for the cache dtype and q_len (below) */
#define HPC_ENGINE_MMA_SYNC 1   /* warp-level mma.sync kernels (every dtype and q_len) */
#define HPC_ENGINE_TCGEN05 2    /* tcgen05.mma with TMEM accumulators (every dtype and q_len) */

/*
 * hpc_decode_attn_multi with a choice of kernel, for callers that pin one and
 * for tests. HPC_ENGINE_AUTO (what hpc_decode_attn_multi uses) takes the
 * faster kernel measured for the cache dtype and q_len (see multi_engine_for
 * in api.cu). Both compute the same rows with 16-bit probabilities and float32
 * accumulation; they differ in summation order and in where the softmax
 * reference maximum moves. On an e4m3 cache the tcgen05 kernel multiplies the
 * exact K codes by Q in f16 and applies the K scales to the float32 scores (as
 * the warp-level kernel does); V enters the P . V product dequantised and
 * rounded to f16, so its values must lie within the f16 range (|v| <= 65504),
 * and Q must fit f16 as well (as for the warp-level e4m3 kernel).
 * Errors: as hpc_decode_attn_multi, plus HPC_ERR_INVALID_ARG for an unknown
 * engine.
 */
hpc_status hpc_decode_attn_multi_engine(const void* q, int q_len, const void* k_cache, const void* v_cache,
                                        const float* k_scale, const float* v_scale, int kv_dtype,
                                        int num_pages, const int32_t* page_table, int page_table_stride,
                                        const int32_t* seq_lens, int batch, int num_q_heads,
                                        int num_kv_heads, int head_dim, int page_size,
                                        const hpc_plan* plan, float* split_o, float* split_lse,
                                        int engine, void* stream);

/* The kernel HPC_ENGINE_AUTO runs for a cache dtype and q_len new tokens per
 * request: HPC_ENGINE_MMA_SYNC or HPC_ENGINE_TCGEN05 (the measured faster one;
 * q_len = 1 runs hpc_decode_attn's kernel, reported as HPC_ENGINE_MMA_SYNC).
 * Returns 0 for an unknown kv_dtype or q_len outside [1, HPC_MAX_Q_LEN]. Host
 * only, no device call. */
int hpc_decode_attn_multi_auto_engine(int kv_dtype, int q_len);

/* Flags of hpc_decode_attn_ex. */
#define HPC_ATTN_EARLY_KV 1  /* gather KV before waiting for the predecessor kernel */
#define HPC_ATTN_TEST_WAIT_EXPIRY 2  /* failure-path test: make a bounded wait run out */

/*
 * Every attention form in one call: q_scale NULL takes a bf16 query
 * [batch][q_len][num_q_heads][128] (hpc_decode_attn_multi_engine; q_len = 1
 * is hpc_decode_attn), non-NULL an e4m3 query with per-(token, head) scales
 * (hpc_decode_attn_q8: kv_dtype HPC_KV_FP8_E4M3, q_len 1, HPC_ENGINE_AUTO or
 * HPC_ENGINE_MMA_SYNC). Outputs and errors as those calls, plus
 * HPC_ERR_INVALID_ARG for an unknown flag bit.
 *
 * HPC_ATTN_EARLY_KV ([LL] "SGLang Low-Latency Mode: Kernels and Runtime",
 * section "Low-Latency-Specific Optimizations", item 1: with programmatic
 * dependent launch, attention starts gathering KV before it waits for the
 * query). The kernel always waits for the kernel before it in the stream
 * before it reads the query; with this flag each CTA's producer first issues
 * the copies of the leading chunks of its task list that hold no new token
 * (all 64 positions below seq_lens[b] - q_len), up to its ring depth, and
 * only then waits. Results are bit-identical to the call without the flag.
 * Contract, the caller's: the plan, seq_lens, page_table and every cache
 * slot outside the last q_len tokens of each request are final before the
 * kernel preceding this call in the stream triggers its dependents (the
 * library's kernels trigger only after their own wait for their
 * predecessor; a kernel launched without programmatic serialisation counts
 * as triggering when it ends). That kernel may write the query and the new
 * tokens' K and V (hpc_rope_norm does). Breaking the contract yields wrong
 * outputs, never an out-of-bounds access: early copies are bounds-checked
 * like the others and every copy lands before the CTA exits.
 *
 * HPC_ATTN_TEST_WAIT_EXPIRY exists to test the failure path without a fault
 * (the pages have no counterpart). Every wait inside the attention kernels is
 * bounded (2 s); when one runs out, the CTA sets HPC_DEVERR_WAIT_TIMEOUT in
 * the task map's error word, waits (bounded) for its own copies in flight
 * and returns, leaving the device usable. With this flag the consumer warps
 * of every CTA first wait, with a 1 ms limit, on a barrier that nothing
 * completes, so every CTA takes that path: the call computes no partial
 * (split_o / split_lse keep their contents) and hpc_decode_read_error then
 * reports HPC_DEVERR_WAIT_TIMEOUT. Plan again before the next use of the
 * task map (the planner clears the error word). One new token per request on
 * the warp-level kernel only (q_len 1, engine AUTO or MMA_SYNC); other forms
 * return HPC_ERR_UNSUPPORTED.
 */
hpc_status hpc_decode_attn_ex(const void* q, const float* q_scale, int q_len, const void* k_cache,
                              const void* v_cache, const float* k_scale, const float* v_scale,
                              int kv_dtype, int num_pages, const int32_t* page_table,
                              int page_table_stride, const int32_t* seq_lens, int batch,
                              int num_q_heads, int num_kv_heads, int head_dim, int page_size,
                              const hpc_plan* plan, float* split_o, float* split_lse, int engine,
                              int flags, void* stream);

/*
 * Combine ([SGL] the paragraph on execution; [VLLM] combine stage). For every
 * (request b, query head qh) with h = qh / 8, j = qh % 8 and the pair's
 * n = pair_nsplit[h*batch+b] partials starting at s0 = pair_split0[...]:
 * M = max_i lse_i, w_i = exp(lse_i - M), out = sum w_i o_i / sum w_i (to
 * bf16, round to nearest even), out_lse = M + ln sum w_i. n == 0 gives 0 and
 * -inf. One warp per output row.
 *   out       device bf16 [batch][num_q_heads][128], 8-byte aligned
 *   out_lse   device float32 [batch][num_q_heads] or NULL
 */
hpc_status hpc_decode_combine(const hpc_plan* plan, const float* split_o, const float* split_lse,
                              void* out, float* out_lse, int batch, int num_q_heads,
                              int num_kv_heads, int head_dim, void* stream);

/*
 * Combine for q_len new tokens per request (the partials of
 * hpc_decode_attn_multi): the same merge for every (b, i, qh), reading the
 * partial rows (s * q_len + i) * 8 + qh % 8 of the pair's splits.
 *   out       device bf16 [batch][q_len][num_q_heads][128], 8-byte aligned
 *   out_lse   device float32 [batch][q_len][num_q_heads] or NULL
 * q_len == 1 is hpc_decode_combine.
 */
hpc_status hpc_decode_combine_multi(const hpc_plan* plan, int q_len, const float* split_o,
                                    const float* split_lse, void* out, float* out_lse, int batch,
                                    int num_q_heads, int num_kv_heads, int head_dim, void* stream);

/*
 * Fused attention prologue, HpcRopeNorm ([SGL] "A fused attention prologue";
 * [VLLM] "融合的注意力前奏"). For every token t and head of the fused QKV
 * projection output:
 *   query and key heads: RMS QK-norm, y = x / sqrt(mean(x^2) + eps) * w
 *     (w = q_weight or k_weight, shared by all heads), then rotary embedding
 *     on pairs (i, i+64): y_i' = y_i c_i - y_{i+64} s_i,
 *     y_{i+64}' = y_{i+64} c_i + y_i s_i, with (c, s) = row positions[t] of
 *     cos_sin;
 *   value heads: unchanged.
 * Queries go to q_out: bf16, or (q_scale_out != NULL) e4m3 codes with one
 * float32 scale per (token, query head), the input of hpc_decode_attn_q8.
 * Keys and values go straight into the cache at slot_mapping[t] =
 * page * 64 + offset (negative: not written): bf16, or e4m3 with one scale
 * per (token, KV head) in k_scale / v_scale ([num_pages][num_kv_heads][64]).
 * e4m3 scales are amax / 448 over the head's 128 values (1 if all are 0);
 * codes are round-to-nearest-even of x / scale, saturated.
 *   qkv          device bf16 [num_tokens][num_q_heads + 2*num_kv_heads][128],
 *                heads in the order Q, K, V; 16-byte aligned
 *   positions    device int32 [num_tokens]
 *   cos_sin      device float32 [max_pos][128]: 64 cosines then 64 sines
 *   q_weight,    device float32 [128], 16-byte aligned
 *   k_weight
 *   q_out        device bf16 or e4m3 [num_tokens][num_q_heads][128]
 *   d_error_word device int32 or NULL: HPC_DEVERR_BAD_POSITION (row left
 *                unrotated), HPC_DEVERR_PAGE_OUT_OF_RANGE (slot skipped)
 * Errors: HPC_ERR_INVALID_ARG, HPC_ERR_UNSUPPORTED (head_dim != 128,
 * page_size != 64), HPC_ERR_CUDA. num_tokens == 0 enqueues nothing.
 */
hpc_status hpc_rope_norm(const void* qkv, const int32_t* positions, const float* cos_sin, int max_pos,
                         const float* q_weight, const float* k_weight, float eps,
                         const int32_t* slot_mapping, int num_tokens, int num_q_heads,
                         int num_kv_heads, int head_dim, int page_size, void* q_out,
                         float* q_scale_out, void* k_cache, void* v_cache, float* k_scale,
                         float* v_scale, int kv_dtype, int num_pages, int* d_error_word,
                         void* stream);

/*
 * Workspace bytes for hpc_decode_step_host: device copies of q, seq_lens and
 * the page table, the task map, the split buffers and the outputs, each
 * 256-byte aligned. 0 on invalid sizes.
 */
size_t hpc_decode_step_workspace_bytes(int batch, int num_q_heads, int num_kv_heads,
                                       int page_table_stride, int num_ctas);

/*
 * One decode step from host buffers: brings h_q, h_seq_lens and h_page_table
 * into d_workspace, plans with num_ctas and min_chunks_per_cta, runs attention
 * over the device-resident caches, combines, and delivers out (and out_lse,
 * if h_out_lse is non-NULL) to the host. Everything is enqueued on `stream`;
 * the caller synchronises the stream before reading h_out.
 * When all the host buffers are page-locked and mapped into the device's
 * address space (cudaHostAlloc, or cudaHostRegister with
 * cudaHostRegisterMapped; cudaPointerGetAttributes reports them as host
 * memory with a device pointer), one staging kernel reads the inputs over the
 * host link and the combine writes the outputs straight into h_out and
 * h_out_lse (h_out 8-byte aligned). Otherwise the inputs and outputs go
 * through cudaMemcpyAsync (synchronous for pageable memory). Same errors as
 * the calls it chains.
 */
hpc_status hpc_decode_step_host(const void* h_q, const int32_t* h_seq_lens,
                                const int32_t* h_page_table, int page_table_stride,
                                const void* d_k_cache, const void* d_v_cache,
                                const float* d_k_scale, const float* d_v_scale, int kv_dtype,
                                int num_pages, int batch, int num_q_heads, int num_kv_heads,
                                int head_dim, int page_size, int num_ctas, int min_chunks_per_cta,
                                void* d_workspace, size_t workspace_bytes, void* h_out,
                                float* h_out_lse, void* stream);

/* One hpc_decode_step_host call captured as a CUDA graph (opaque). */
typedef struct hpc_step_graph hpc_step_graph;

/*
 * Captures the work of hpc_decode_step_host (the three host -> device copies,
 * plan, attention, combine and the copies back into h_out and h_out_lse) as a
 * CUDA graph, so that each step is one graph launch instead of eight
 * enqueues. Every pointer and size is fixed at capture: the caller refills
 * the host input buffers in place and reads the output buffers after each
 * launch. Host buffers must be pinned (capture of a copy from pageable memory
 * fails). Capture runs on a stream of its own, so this call performs no step;
 * it sets the kernels' one-time attributes first and allocates the graph and
 * its handle (host and driver memory) until hpc_decode_step_graph_destroy.
 * Errors: as hpc_decode_step_host; HPC_ERR_INVALID_ARG for graph == NULL;
 * HPC_ERR_CUDA if capture or instantiation fails (*graph is then NULL).
 */
hpc_status hpc_decode_step_graph_create(const void* h_q, const int32_t* h_seq_lens,
                                        const int32_t* h_page_table, int page_table_stride,
                                        const void* d_k_cache, const void* d_v_cache,
                                        const float* d_k_scale, const float* d_v_scale,
                                        int kv_dtype, int num_pages, int batch, int num_q_heads,
                                        int num_kv_heads, int head_dim, int page_size, int num_ctas,
                                        int min_chunks_per_cta, void* d_workspace,
                                        size_t workspace_bytes, void* h_out, float* h_out_lse,
                                        hpc_step_graph** graph);

/* Enqueues one captured step on `stream`; synchronise the stream before
 * reading the outputs. Launches on one graph are ordered by the stream; two
 * launches of the same graph must not overlap (they share the workspace and
 * the host buffers). Errors: HPC_ERR_INVALID_ARG, HPC_ERR_CUDA. */
hpc_status hpc_decode_step_graph_launch(hpc_step_graph* graph, void* stream);

/* Frees a captured step (NULL is a no-op). Its launches must have completed. */
hpc_status hpc_decode_step_graph_destroy(hpc_step_graph* graph);

/*
 * One decode step (plan -> attention -> combine) that allocates nothing. The
 * pages describe no counterpart: this entry point exists for callers that
 * cannot call cudaMalloc where they run the step, for example an engine
 * whose memory pool takes all device memory at start-up and forbids
 * allocations outside it, or plugin code that is handed only input and output
 * pointers and has no allocator to reach. The caller passes the inputs (as
 * for hpc_decode_attn) and the outputs (as for hpc_decode_combine); the task
 * map and the split buffers live in one fixed 8 MiB device array inside the
 * library, which every GPU that loads the library holds until the process
 * exits.
 *   - Limit: the task map for (batch, num_kv_heads, num_ctas) plus
 *     hpc_decode_split_capacity rows of 4128 bytes (each part rounded up to
 *     256 bytes) must fit in 8 MiB, about 2000 split rows; larger sizes return
 *     HPC_ERR_WORKSPACE_TOO_SMALL before any work is enqueued.
 *   - Every argument check of hpc_decode_plan, hpc_decode_attn and
 *     hpc_decode_combine runs before the first launch: a refused call
 *     enqueues nothing and leaves the array as it was.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress with that device current); make that first call
 *     before any stream capture. The address is kept with the ID of the
 *     context it was found in: after a device reset (or the primary context
 *     released and created again) the next call looks it up again, so make
 *     that call outside stream capture too.
 *   - Every call on a device shares the array: calls whose work overlaps on
 *     the GPU (other streams, no ordering between them) race on it. Nothing in
 *     the array needs to start at zero; each call rewrites what it reads.
 *   - The device error word lives in that array and is not reported.
 * Errors: as hpc_decode_plan, hpc_decode_attn and hpc_decode_combine.
 */
hpc_status hpc_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                              const float* k_scale, const float* v_scale, int kv_dtype,
                              int num_pages, const int32_t* page_table, int page_table_stride,
                              const int32_t* seq_lens, int batch, int num_q_heads,
                              int num_kv_heads, int head_dim, int page_size, int num_ctas,
                              int min_chunks_per_cta, void* out, float* out_lse, void* stream);

/* Synchronises the device, then reads the task map's error word into
 * *device_error_word. Returns HPC_ERR_DEVICE_CHECK when it is non-zero.
 * For tests and diagnostics, not for the hot loop. */
hpc_status hpc_decode_read_error(const hpc_plan* plan, int* device_error_word);

/* Static string for a status code. */
const char* hpc_status_string(hpc_status status);

#ifdef __cplusplus
}
#endif

#endif /* HPC_DECODE_H */
