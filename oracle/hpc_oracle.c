/*
 * Float64 CPU oracle for load-balanced paged GQA decode attention.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg may load or run this library. It shares no
 * code, header, table or constant generator with the CUDA library that it
 * checks, and it never reads anything the CUDA library produced except to
 * compare against it in a test.
 *
 * Sources (two blog posts on the HPC-Ops attention backend):
 *   [SGL]  "HPC-Ops, integrated into SGLang" (English text), section
 *          "Scheduling around live KV work" and the paragraph after it.
 *   [VLLM] "vLLM x HPC-Ops: High-Performance Attention and MoE Backends from
 *          Tencent Hunyuan", section "Attention 后端：动态负载均衡调度"
 *          (attention backend: dynamic load-balanced scheduling), sub-section
 *          "解决方案：按步负载均衡的 decode 调度器" (per-step load-balanced
 *          decode scheduler: assign, compute and combine), and the section
 *          "关于 Hy3 系列模型的简要说明" (Hy3: GQA with 64 query heads, 8 KV
 *          heads, head dim 128).
 *
 * What the method computes, restated:
 *   assign   Each (KV head, request) KV sequence is cut into 64-token chunks.
 *            The per-CTA budget (bucket) is the chunk total over all heads and
 *            requests divided by the number of persistent CTAs, and never
 *            below a minimum-work floor. Chunks are walked head-major, then
 *            request by request, and poured into CTA buckets in order; a full
 *            bucket spills into the next CTA. Each CTA's bucket is a list of
 *            task descriptors closed by a terminator; a descriptor is one
 *            (KV head, request, contiguous chunk range).
 *   compute  Each descriptor yields, for each query head of its GQA group, a
 *            partial attention output over its token range plus the
 *            log-sum-exp of that range.
 *   combine  Per (request, query head) the partials are merged with weights
 *            exp(lse_i - max lse) into the output under the global softmax.
 *
 * Readings where the pages are silent (each one is listed with its reason in
 * the design notes of the repository):
 *   - bucket = max(ceil(T / C), m, 1) where T is the chunk total, C the CTA
 *     count and m the floor; CTAs past ceil(T / bucket) get an empty list.
 *   - one partial per descriptor (a maximal run of one pair inside one bucket).
 *   - softmax scale 1/sqrt(head_dim); LSE is the natural log of the sum of
 *     exp of scaled scores; partial outputs are normalised by their own sum.
 *   - query head qh reads KV head qh / G with G = Hq / Hkv (contiguous groups).
 *   - KV cache layout [num_pages][64][Hkv][128]; FP8 scale layout
 *     [num_pages][Hkv][64] (per token, per head); FP8 is OCP e4m3fn.
 *   - a request of length 0 has no chunks; its output is 0 and its LSE -inf.
 *
 * Several new tokens per request (q_len > 1), as in speculative verification:
 *   [LL] "SGLang Low-Latency Mode: Kernels and Runtime", section "Where the
 *   Time Goes" (one request verifies six token rows per step), and the Hy3
 *   section of [VLLM] (an MTP layer for speculative decoding). The pages give
 *   no masking rule; the reading taken here is the usual causal one:
 *   - the q_len new tokens are already in the cache and seq_lens counts them;
 *     new token qi (0-based) sees tokens [0, L - q_len + qi];
 *   - the task map is the same as for one token (it walks the chunks of L);
 *     each descriptor computes q_len * G rows, and a new token whose visible
 *     range misses the descriptor's chunks gets O = 0, LSE = -inf there;
 *   - q is [B][q_len][Hq][128] and the split buffers [split][q_len][G][128].
 *
 * Task-map byte layout (all int32; the CUDA planner must reproduce it
 * bit for bit):
 *   [0, 16)                 header, see the OR_H_* slots below
 *   [16, 16 + C + 1)        cta_off: first task slot of each CTA's list, and
 *                           the end of the last list at index C
 *   tasks (32-byte aligned) max_tasks rows of 8 ints:
 *                           {kv_head, request, chunk_begin, chunk_end,
 *                            split_index, rank_in_pair, splits_in_pair, 0}
 *                           a terminator row and every unused row are all -1
 *   pair_nsplit[Hkv * B]    descriptor count of pair p = h * B + b
 *   pair_split0[Hkv * B]    split index of the pair's first descriptor
 *                           (exclusive running count in walk order)
 *   max_tasks = Hkv * B + 2 * C.
 *
 * A descriptor's split index is its position in the global walk order; the
 * split buffers are [split][q_len][G][head_dim] (outputs) and [split][q_len][G]
 * (LSE).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_CHUNK_TOKENS 64
#define OR_HEAD_DIM 128
#define OR_HDR_INTS 16
#define OR_TASK_INTS 8

enum {
    OR_H_TOTAL_CHUNKS = 0,
    OR_H_BUCKET = 1,
    OR_H_USED_CTAS = 2,
    OR_H_TOTAL_SPLITS = 3,
    OR_H_NUM_CTAS = 4,
    OR_H_BATCH = 5,
    OR_H_NUM_KV_HEADS = 6,
    OR_H_MIN_CHUNKS = 7, /* the floor m; the split count S for a static plan */
    OR_H_MAX_TASKS = 8,
    OR_H_MODE = 9, /* 0 load-balanced, 1 static split count */
    OR_H_CHUNKS_PER_HEAD = 10,
    OR_H_CHUNK_TOKENS = 11,
    OR_H_ERROR = 12 /* bit 0: a negative length was seen; bit 1: chunk total overflowed int32 */
};

typedef struct {
    long long cta_off, tasks, nsplit, split0, total;
    long long max_tasks;
} or_layout;

static or_layout or_layout_of(long long B, long long Hkv, long long C) {
    or_layout L;
    L.max_tasks = Hkv * B + 2 * C;
    L.cta_off = OR_HDR_INTS;
    long long t = OR_HDR_INTS + C + 1;
    L.tasks = (t + 7) / 8 * 8;
    L.nsplit = L.tasks + L.max_tasks * OR_TASK_INTS;
    L.split0 = L.nsplit + Hkv * B;
    L.total = L.split0 + Hkv * B;
    return L;
}

long long oracle_plan_ints(int B, int Hkv, int C) {
    if (B < 1 || Hkv < 1 || C < 1) return -1;
    return or_layout_of(B, Hkv, C).total;
}

/* ---------------------------------------------------------------- numbers */

/* OCP 8-bit E4M3 ("fn": no infinities). 1 sign bit, 4 exponent bits with bias
 * 7, 3 mantissa bits. Exponent field 0 is subnormal: mant/8 * 2^-6. The code
 * with all exponent and mantissa bits set is NaN; the largest finite value is
 * 448 = 1.75 * 2^8. */
double oracle_e4m3_to_f64(uint8_t x) {
    int sign = (x >> 7) & 1;
    int e = (x >> 3) & 15;
    int mant = x & 7;
    double v;
    if (e == 15 && mant == 7) return NAN;
    if (e == 0)
        v = ldexp((double)mant / 8.0, -6);
    else
        v = ldexp(1.0 + (double)mant / 8.0, e - 7);
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32. */
double oracle_bf16_to_f64(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ---------------------------------------------------------------- planner */

typedef struct {
    int h, b, c0, c1;
    long long cta;
} or_desc;

/* Writes the descriptor list d[0..nd) (already in walk order, CTA index
 * non-decreasing) into the canonical buffer. */
static void or_emit(const or_desc* d, long long nd, int B, int Hkv, long long C, long long T,
                    long long bucket, long long m_or_s, int mode, long long N, int err, int32_t* out) {
    or_layout L = or_layout_of(B, Hkv, C);
    for (long long i = 0; i < L.total; ++i) out[i] = 0;
    for (long long i = 0; i < L.max_tasks * OR_TASK_INTS; ++i) out[L.tasks + i] = -1;

    /* pair tables: descriptors of one pair are consecutive in walk order */
    long long P = (long long)Hkv * B;
    int32_t* nsplit = out + L.nsplit;
    int32_t* split0 = out + L.split0;
    for (long long p = 0; p < P; ++p) nsplit[p] = 0;
    for (long long i = 0; i < nd; ++i) nsplit[(long long)d[i].h * B + d[i].b] += 1;
    long long run = 0;
    for (long long p = 0; p < P; ++p) {
        split0[p] = (int32_t)run;
        run += nsplit[p];
    }

    /* per-CTA lists, each closed by a terminator */
    long long pos = 0, i = 0;
    for (long long j = 0; j < C; ++j) {
        out[L.cta_off + j] = (int32_t)pos;
        while (i < nd && d[i].cta == j) {
            int32_t* t = out + L.tasks + pos * OR_TASK_INTS;
            long long p = (long long)d[i].h * B + d[i].b;
            t[0] = d[i].h;
            t[1] = d[i].b;
            t[2] = d[i].c0;
            t[3] = d[i].c1;
            t[4] = (int32_t)i;
            t[5] = (int32_t)(i - split0[p]);
            t[6] = nsplit[p];
            t[7] = 0;
            ++pos;
            ++i;
        }
        ++pos; /* terminator row stays -1 */
    }
    out[L.cta_off + C] = (int32_t)pos;

    long long used = 0;
    for (long long k = 0; k < nd; ++k)
        if (k == 0 || d[k].cta != d[k - 1].cta) ++used;

    int32_t* hdr = out;
    hdr[OR_H_TOTAL_CHUNKS] = (int32_t)T;
    hdr[OR_H_BUCKET] = (int32_t)bucket;
    hdr[OR_H_USED_CTAS] = (int32_t)used;
    hdr[OR_H_TOTAL_SPLITS] = (int32_t)nd;
    hdr[OR_H_NUM_CTAS] = (int32_t)C;
    hdr[OR_H_BATCH] = B;
    hdr[OR_H_NUM_KV_HEADS] = Hkv;
    hdr[OR_H_MIN_CHUNKS] = (int32_t)m_or_s;
    hdr[OR_H_MAX_TASKS] = (int32_t)L.max_tasks;
    hdr[OR_H_MODE] = mode;
    hdr[OR_H_CHUNKS_PER_HEAD] = (int32_t)N;
    hdr[OR_H_CHUNK_TOKENS] = OR_CHUNK_TOKENS;
    hdr[OR_H_ERROR] = err;
}

/* Chunk counts n_b = ceil(L_b / 64); negative lengths count as 0 and set bit 0
 * of the error word. Returns N = sum of n_b, or -1 when the chunk total over
 * all heads would not fit in int32 (then every n_b is zeroed, bit 1 set). */
static long long or_chunks(const int32_t* seq_lens, int B, int Hkv, long long* n, int* err) {
    long long N = 0;
    for (int b = 0; b < B; ++b) {
        long long len = seq_lens[b];
        if (len < 0) {
            *err |= 1;
            len = 0;
        }
        n[b] = (len + OR_CHUNK_TOKENS - 1) / OR_CHUNK_TOKENS;
        N += n[b];
    }
    if (N * (long long)Hkv > 2147483647LL) {
        *err |= 2;
        for (int b = 0; b < B; ++b) n[b] = 0;
        return 0;
    }
    return N;
}

/* Load-balanced task map: the walk of [SGL] / [VLLM] written as a triple
 * loop over (kv head, request, chunk) with a running global chunk counter g;
 * chunk g goes to CTA g / bucket, and a new descriptor starts whenever the
 * pair or the CTA changes. */
int oracle_plan(const int32_t* seq_lens, int B, int Hkv, int C, int m, int32_t* out,
                long long out_ints) {
    if (B < 1 || Hkv < 1 || C < 1 || m < 0) return -1;
    or_layout L = or_layout_of(B, Hkv, C);
    if (out_ints < L.total) return -2;
    long long* n = (long long*)malloc(sizeof(long long) * (size_t)B);
    or_desc* d = (or_desc*)malloc(sizeof(or_desc) * (size_t)L.max_tasks);
    if (!n || !d) {
        free(n);
        free(d);
        return -3;
    }
    int err = 0;
    long long N = or_chunks(seq_lens, B, Hkv, n, &err);
    long long T = N * Hkv;
    long long bucket = (T + C - 1) / C;
    if (bucket < m) bucket = m;
    if (bucket < 1) bucket = 1;

    long long nd = 0, g = 0;
    for (int h = 0; h < Hkv; ++h)
        for (int b = 0; b < B; ++b)
            for (long long c = 0; c < n[b]; ++c, ++g) {
                long long cta = g / bucket;
                if (c > 0 && d[nd - 1].cta == cta) {
                    d[nd - 1].c1 = (int)(c + 1);
                } else {
                    d[nd].h = h;
                    d[nd].b = b;
                    d[nd].c0 = (int)c;
                    d[nd].c1 = (int)(c + 1);
                    d[nd].cta = cta;
                    ++nd;
                }
            }
    or_emit(d, nd, B, Hkv, C, T, bucket, m, 0, N, err, out);
    free(n);
    free(d);
    return 0;
}

/* Static split-KV comparison schedule ([SGL], "Attention: load balancing for
 * mixed-length decode", policy (1): a fixed split count). One virtual CTA per
 * (kv head, request, split s) in that order; split s of a pair with n chunks
 * covers chunks [s*q, min((s+1)*q, n)) with q = ceil(n / S), and is empty when
 * s*q >= n. */
int oracle_plan_static(const int32_t* seq_lens, int B, int Hkv, int S, int32_t* out,
                       long long out_ints) {
    if (B < 1 || Hkv < 1 || S < 1) return -1;
    long long C = (long long)Hkv * B * S;
    if (C > 2147483647LL / 4) return -1;
    or_layout L = or_layout_of(B, Hkv, C);
    if (out_ints < L.total) return -2;
    long long* n = (long long*)malloc(sizeof(long long) * (size_t)B);
    or_desc* d = (or_desc*)malloc(sizeof(or_desc) * (size_t)L.max_tasks);
    if (!n || !d) {
        free(n);
        free(d);
        return -3;
    }
    int err = 0;
    long long N = or_chunks(seq_lens, B, Hkv, n, &err);
    long long nd = 0;
    for (int h = 0; h < Hkv; ++h)
        for (int b = 0; b < B; ++b) {
            long long q = (n[b] + S - 1) / S;
            for (int s = 0; s < S; ++s) {
                if (q == 0 || (long long)s * q >= n[b]) continue;
                long long e = ((long long)s + 1) * q;
                d[nd].h = h;
                d[nd].b = b;
                d[nd].c0 = (int)((long long)s * q);
                d[nd].c1 = (int)(e < n[b] ? e : n[b]);
                d[nd].cta = ((long long)h * B + b) * S + s;
                ++nd;
            }
        }
    or_emit(d, nd, B, Hkv, C, N * Hkv, 0, S, 1, N, err, out);
    free(n);
    free(d);
    return 0;
}

/* ---------------------------------------------------------------- attention */

typedef struct {
    const void* q;     /* bf16 bits, or e4m3 codes when q_scale is set: [B][Hq][128] */
    const float* q_scale; /* e4m3 query only: [B][Hq] */
    const void* kc;    /* [P][64][Hkv][128] bf16 bits or e4m3 bytes */
    const void* vc;
    const float* ks; /* e4m3 only: [P][Hkv][64] */
    const float* vs;
    int fp8;
    int num_pages;
    const int32_t* pt;
    int pt_stride;
    const int32_t* seq_lens;
    int B, Hq, Hkv;
    int q_len; /* new tokens per request (1 for plain decode); q is [B][q_len][Hq][128] */
} or_kv;

static double or_elem(const or_kv* kv, const void* cache, const float* scale, long long page,
                      int slot, int h, int dim) {
    long long idx = ((page * OR_CHUNK_TOKENS + slot) * kv->Hkv + h) * OR_HEAD_DIM + dim;
    if (kv->fp8) {
        double s = scale[(page * kv->Hkv + h) * OR_CHUNK_TOKENS + slot];
        return oracle_e4m3_to_f64(((const uint8_t*)cache)[idx]) * s;
    }
    return oracle_bf16_to_f64(((const uint16_t*)cache)[idx]);
}

/* Softmax attention of query row (b, qh) over tokens [t0, t1) of request b,
 * two passes in float64: scores, max, sum of exp, weighted sum of values.
 * Returns -1 if a page id is outside [0, num_pages). */
static int or_attend(const or_kv* kv, int b, int qi, int qh, long long t0, long long t1, double* o,
                     double* lse) {
    int G = kv->Hq / kv->Hkv;
    int h = qh / G;
    for (int dd = 0; dd < OR_HEAD_DIM; ++dd) o[dd] = 0.0;
    if (t1 <= t0) {
        *lse = -INFINITY;
        return 0;
    }
    double qv[OR_HEAD_DIM];
    const long long row = ((long long)b * kv->q_len + qi) * kv->Hq + qh;
    const long long qoff = row * OR_HEAD_DIM;
    if (kv->q_scale) {
        /* e4m3 query with one scale per (request, query head), the form the fused
         * attention prologue hands to the attention kernel */
        const uint8_t* qrow = (const uint8_t*)kv->q + qoff;
        const double qs = kv->q_scale[row];
        for (int dd = 0; dd < OR_HEAD_DIM; ++dd) qv[dd] = oracle_e4m3_to_f64(qrow[dd]) * qs;
    } else {
        const uint16_t* qrow = (const uint16_t*)kv->q + qoff;
        for (int dd = 0; dd < OR_HEAD_DIM; ++dd) qv[dd] = oracle_bf16_to_f64(qrow[dd]);
    }
    long long n = t1 - t0;
    double* s = (double*)malloc(sizeof(double) * (size_t)n);
    if (!s) return -3;
    const double scale = 1.0 / sqrt((double)OR_HEAD_DIM);
    for (long long t = t0; t < t1; ++t) {
        long long page = kv->pt[(long long)b * kv->pt_stride + t / OR_CHUNK_TOKENS];
        if (page < 0 || page >= kv->num_pages) {
            free(s);
            return -1;
        }
        int slot = (int)(t % OR_CHUNK_TOKENS);
        double acc = 0.0;
        for (int dd = 0; dd < OR_HEAD_DIM; ++dd)
            acc += qv[dd] * or_elem(kv, kv->kc, kv->ks, page, slot, h, dd);
        s[t - t0] = acc * scale;
    }
    double mx = -INFINITY;
    for (long long i = 0; i < n; ++i)
        if (s[i] > mx) mx = s[i];
    double sum = 0.0;
    for (long long i = 0; i < n; ++i) {
        s[i] = exp(s[i] - mx);
        sum += s[i];
    }
    for (long long t = t0; t < t1; ++t) {
        long long page = kv->pt[(long long)b * kv->pt_stride + t / OR_CHUNK_TOKENS];
        int slot = (int)(t % OR_CHUNK_TOKENS);
        double w = s[t - t0];
        for (int dd = 0; dd < OR_HEAD_DIM; ++dd)
            o[dd] += w * or_elem(kv, kv->vc, kv->vs, page, slot, h, dd);
    }
    for (int dd = 0; dd < OR_HEAD_DIM; ++dd) o[dd] /= sum;
    *lse = mx + log(sum);
    free(s);
    return 0;
}

/* Causal length of new token qi of request b: it sees tokens [0, L - q_len + qi]
 * (the cache already holds all q_len new tokens; seq_lens counts them). */
static long long or_visible(const or_kv* kv, int b, int qi) {
    long long len = kv->seq_lens[b] > 0 ? kv->seq_lens[b] : 0;
    long long v = len - kv->q_len + qi + 1;
    return v < 0 ? 0 : (v > len ? len : v);
}

static int or_check_kv(const or_kv* kv) {
    if (kv->q_len < 1) return -1;
    if (kv->B < 1 || kv->Hkv < 1 || kv->Hq < kv->Hkv || kv->Hq % kv->Hkv) return -1;
    if (kv->num_pages < 1 || kv->pt_stride < 1) return -1;
    if (kv->fp8 && (!kv->ks || !kv->vs)) return -1;
    return 0;
}

/* Full-sequence attention for selected rows. rows holds nrows (b, r) pairs with
 * r = qi * Hq + qh (new token qi, query head qh); rows == NULL means every row
 * in (b, qi, qh) order (nrows must be B * q_len * Hq). New token qi attends
 * causally: to tokens [0, L_b - q_len + qi].
 * q is bf16 bits, or e4m3 codes scaled by q_scale[b][qi][qh] when q_scale != NULL.
 * Outputs: out_o [nrows][128], out_lse [nrows]. */
int oracle_attn_rows(const void* q, const float* q_scale, const void* kc, const void* vc,
                     const float* ks, const float* vs, int kv_fp8, int num_pages, const int32_t* pt,
                     int pt_stride, const int32_t* seq_lens, int B, int Hq, int Hkv, int q_len,
                     int nrows, const int32_t* rows, double* out_o, double* out_lse) {
    or_kv kv = {q, q_scale, kc, vc, ks, vs, kv_fp8, num_pages, pt, pt_stride, seq_lens, B, Hq, Hkv,
                q_len};
    if (or_check_kv(&kv)) return -1;
    const int R = q_len * Hq; /* query rows per request: (new token, head) */
    if (!rows && nrows != B * R) return -1;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int r = 0; r < nrows; ++r) {
        int b = rows ? rows[2 * r] : r / R;
        int rr = rows ? rows[2 * r + 1] : r % R;
        if (b < 0 || b >= B || rr < 0 || rr >= R) {
            bad |= 1;
            continue;
        }
        int qi = rr / Hq, qh = rr % Hq;
        if (or_attend(&kv, b, qi, qh, 0, or_visible(&kv, b, qi), out_o + (long long)r * OR_HEAD_DIM,
                      out_lse + r))
            bad |= 2;
    }
    return bad ? -4 : 0;
}

/* Partial outputs of every descriptor of a task map written by oracle_plan /
 * oracle_plan_static: for descriptor s = (h, b, c0, c1), each new token qi and
 * each j < G the attention of row (b, qi, h*G + j) over tokens
 * [64*c0, min(64*c1, visible length of qi)).
 * Outputs: split_o [total_splits][q_len][G][128], split_lse [total_splits][q_len][G]. */
int oracle_attn_splits(const int32_t* plan, const void* q, const float* q_scale, const void* kc,
                       const void* vc, const float* ks, const float* vs, int kv_fp8, int num_pages,
                       const int32_t* pt, int pt_stride, const int32_t* seq_lens, int B, int Hq,
                       int Hkv, int q_len, double* split_o, double* split_lse) {
    or_kv kv = {q, q_scale, kc, vc, ks, vs, kv_fp8, num_pages, pt, pt_stride, seq_lens, B, Hq, Hkv,
                q_len};
    if (or_check_kv(&kv)) return -1;
    if (plan[OR_H_BATCH] != B || plan[OR_H_NUM_KV_HEADS] != Hkv) return -1;
    int G = Hq / Hkv;
    or_layout L = or_layout_of(B, Hkv, plan[OR_H_NUM_CTAS]);
    const int32_t* tasks = plan + L.tasks;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (long long i = 0; i < L.max_tasks; ++i) {
        const int32_t* t = tasks + i * OR_TASK_INTS;
        if (t[0] < 0) continue;
        int h = t[0], b = t[1], s = t[4];
        long long t0 = (long long)t[2] * OR_CHUNK_TOKENS;
        for (int qi = 0; qi < q_len; ++qi) {
            long long t1 = (long long)t[3] * OR_CHUNK_TOKENS;
            long long len = or_visible(&kv, b, qi);
            if (t1 > len) t1 = len;
            for (int j = 0; j < G; ++j) {
                long long row = ((long long)s * q_len + qi) * G + j;
                if (or_attend(&kv, b, qi, h * G + j, t0, t1, split_o + row * OR_HEAD_DIM,
                              split_lse + row))
                    bad |= 1;
            }
        }
    }
    return bad ? -4 : 0;
}

/* Merge of the partials of each (request, new token, query head) under the
 * global softmax: M = max lse_i, w_i = exp(lse_i - M), O = sum w_i o_i / sum w_i,
 * LSE = M + log(sum w_i). Pairs without partials give O = 0, LSE = -inf.
 * Outputs: out_o [B][q_len][Hq][128], out_lse [B][q_len][Hq]. */
int oracle_combine(const int32_t* plan, const double* split_o, const double* split_lse, int B,
                   int Hq, int Hkv, int q_len, double* out_o, double* out_lse) {
    if (plan[OR_H_BATCH] != B || plan[OR_H_NUM_KV_HEADS] != Hkv || Hq % Hkv || q_len < 1) return -1;
    int G = Hq / Hkv;
    or_layout L = or_layout_of(B, Hkv, plan[OR_H_NUM_CTAS]);
    const int32_t* nsplit = plan + L.nsplit;
    const int32_t* split0 = plan + L.split0;
    for (int b = 0; b < B; ++b)
        for (int qi = 0; qi < q_len; ++qi)
        for (int qh = 0; qh < Hq; ++qh) {
            int h = qh / G, j = qh % G;
            long long p = (long long)h * B + b;
            long long orow = ((long long)b * q_len + qi) * Hq + qh;
            double* o = out_o + orow * OR_HEAD_DIM;
            double* lse = out_lse + orow;
            for (int dd = 0; dd < OR_HEAD_DIM; ++dd) o[dd] = 0.0;
            int ns = nsplit[p];
            long long s0 = split0[p];
            double M = -INFINITY;
            for (int i = 0; i < ns; ++i) {
                double v = split_lse[((s0 + i) * q_len + qi) * G + j];
                if (v > M) M = v;
            }
            if (ns == 0 || M == -INFINITY) {
                *lse = -INFINITY;
                continue;
            }
            double wsum = 0.0;
            for (int i = 0; i < ns; ++i) {
                long long srow = ((s0 + i) * q_len + qi) * G + j;
                double w = exp(split_lse[srow] - M);
                wsum += w;
                const double* oi = split_o + srow * OR_HEAD_DIM;
                for (int dd = 0; dd < OR_HEAD_DIM; ++dd) o[dd] += w * oi[dd];
            }
            for (int dd = 0; dd < OR_HEAD_DIM; ++dd) o[dd] /= wsum;
            *lse = M + log(wsum);
        }
    return 0;
}

/* ---------------------------------------------------------------- prologue */

/* Fused attention prologue ([SGL] "A fused attention prologue"; [VLLM]
 * "融合的注意力前奏", HpcRopeNorm): from the fused QKV projection output,
 * RMS QK-norm, then rotary position embedding, for every query and key head;
 * value heads pass through. Returns the float64 values before any output
 * rounding or quantisation (the tests check the CUDA outputs against them).
 *   qkv      bf16 bits [T][Hq + 2*Hkv][128], heads in the order Q, K, V
 *   pos      int32 [T], position of each token (row of cos_sin)
 *   cos_sin  float32 [max_pos][128]: cos(theta_i) for i < 64, then sin(theta_i)
 *   qw, kw   float32 [128] RMSNorm weights shared by all query / key heads
 *   q_out    [T][Hq][128], k_out / v_out [T][Hkv][128]
 * RMSNorm: y_d = x_d / sqrt(mean_d x_d^2 + eps) * w_d.
 * Rotation (pairs (i, i+64), i < 64): y_i = x_i c_i - x_{i+64} s_i,
 * y_{i+64} = x_{i+64} c_i + x_i s_i. */
int oracle_rope_norm(const uint16_t* qkv, const int32_t* pos, const float* cos_sin, int max_pos,
                     const float* qw, const float* kw, double eps, int T, int Hq, int Hkv,
                     double* q_out, double* k_out, double* v_out) {
    if (T < 0 || Hq < 1 || Hkv < 1 || max_pos < 1) return -1;
    const int H3 = Hq + 2 * Hkv;
    const int half = OR_HEAD_DIM / 2;
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (long long r = 0; r < (long long)T * H3; ++r) {
        const int t = (int)(r / H3), j = (int)(r % H3);
        const uint16_t* src = qkv + r * OR_HEAD_DIM;
        double x[OR_HEAD_DIM];
        for (int d = 0; d < OR_HEAD_DIM; ++d) x[d] = oracle_bf16_to_f64(src[d]);
        double* dst;
        if (j >= Hq + Hkv) {
            dst = v_out + ((long long)t * Hkv + (j - Hq - Hkv)) * OR_HEAD_DIM;
            for (int d = 0; d < OR_HEAD_DIM; ++d) dst[d] = x[d];
            continue;
        }
        const float* w = j < Hq ? qw : kw;
        dst = j < Hq ? q_out + ((long long)t * Hq + j) * OR_HEAD_DIM
                     : k_out + ((long long)t * Hkv + (j - Hq)) * OR_HEAD_DIM;
        double ss = 0.0;
        for (int d = 0; d < OR_HEAD_DIM; ++d) ss += x[d] * x[d];
        const double inv = 1.0 / sqrt(ss / OR_HEAD_DIM + eps);
        for (int d = 0; d < OR_HEAD_DIM; ++d) x[d] = x[d] * inv * (double)w[d];
        const int p = pos[t];
        if (p < 0 || p >= max_pos) {
            bad |= 1;
            continue;
        }
        const float* cs = cos_sin + (long long)p * OR_HEAD_DIM;
        for (int i = 0; i < half; ++i) {
            const double c = cs[i], sn = cs[half + i];
            dst[i] = x[i] * c - x[i + half] * sn;
            dst[i + half] = x[i + half] * c + x[i] * sn;
        }
    }
    return bad ? -4 : 0;
}
