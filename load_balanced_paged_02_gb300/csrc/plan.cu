// Task-map planners (integer only). The balanced map's planner runs over
// several blocks when the batch has many (kv head, request) pairs; the static
// map's planner is one block.
//
// Load-balanced map: HPC-Ops/SGLang blog, "Scheduling around live KV work";
// vLLM x HPC-Ops blog, "解决方案：按步负载均衡的 decode 调度器" (assign stage).
// Static map: HPC-Ops/SGLang blog, "Attention: load balancing for mixed-length
// decode", policy (1), a fixed split count.
//
// The planner never walks chunks one by one. For pair p = (h, b) with n_b
// chunks starting at global chunk g0 = h*N + prefix_b, the CTAs it touches are
// g0/bucket .. (g0+n_b-1)/bucket; descriptor k of the pair lives in CTA
// g0/bucket + k and covers [max(g0, cta*bucket), min(g0+n_b, (cta+1)*bucket)).
// Its split index s is the running descriptor count, and its task row is
// s + cta (every earlier CTA contributed one terminator row).
#include "hpc_internal.cuh"

namespace hpc {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kPlanWarps = kPlanThreads / 32;
// Blocks of the balanced planner: one per 1024 pairs, at most this many (each
// block then takes several 1024-pair tiles).
constexpr int kPlanMaxBlocks = 64;

// Exclusive scan of one value per thread across the block. All threads must
// call it. Returns the exclusive prefix; *total receives the block sum.
template <typename V>
__device__ V block_exclusive_scan(V v, V* total, V* warp_sums) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    V x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        V y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[wid] = x;
    __syncthreads();
    if (wid == 0) {
        V w = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            V y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        warp_sums[lane] = w;
    }
    __syncthreads();
    V prefix = (wid > 0 ? warp_sums[wid - 1] : 0) + x - v;
    *total = warp_sums[kPlanWarps - 1];
    __syncthreads();
    return prefix;
}

// Division of 32-bit unsigned integers by a divisor fixed for the launch, as a
// multiply and shifts (T. Granlund and P. L. Montgomery, "Division by invariant
// integers using multiplication", PLDI 1994, section 4): with l = ceil(log2 d)
// and m = floor(2^32 (2^l - d) / d) + 1, the quotient is
// (t + ((n - t) >> min(l, 1))) >> max(l - 1, 0), t = high half of m * n, for
// 1 <= d < 2^32 and every 32-bit n. A planner block is bound by instruction
// issue and latency; hardware-sequence divisions by the bucket and the batch
// for every pair cost about a tenth of its time.
struct FastDiv {
    uint32_t m;
    int s1, s2;
    __device__ __forceinline__ explicit FastDiv(uint32_t d) {
        const int l = 32 - __clz((int)(d - 1u));  // ceil(log2 d); 0 for d = 1
        m = (uint32_t)(((((uint64_t)1 << l) - d) << 32) / d + 1);
        s1 = l < 1 ? l : 1;
        s2 = l > 0 ? l - 1 : 0;
    }
    __device__ __forceinline__ uint32_t div(uint32_t n) const {
        const uint32_t t = __umulhi(m, n);
        return (t + ((n - t) >> s1)) >> s2;
    }
};

__device__ __forceinline__ void write_row(int32_t* row, int a, int b, int c, int d, int e, int f,
                                          int g) {
    reinterpret_cast<int4*>(row)[0] = make_int4(a, b, c, d);
    reinterpret_cast<int4*>(row)[1] = make_int4(e, f, g, 0);
}

__device__ __forceinline__ void write_term(int32_t* row) {
    reinterpret_cast<int4*>(row)[0] = make_int4(-1, -1, -1, -1);
    reinterpret_cast<int4*>(row)[1] = make_int4(-1, -1, -1, -1);
}

// Chunk prefix sums pre[0..B] (pre[B] = N) of n_b = ceil(max(L_b, 0) / 64).
// Returns N, or 0 with every prefix zeroed when Hkv * N overflows int32.
__device__ long long chunk_prefix(const int32_t* __restrict__ seq_lens, int B, int Hkv, int32_t* pre,
                                  long long* warp_sums, int* s_err) {
    const int tid = threadIdx.x;
    long long running = 0;
    for (int base = 0; base < B; base += kPlanThreads) {
        const int b = base + tid;
        long long n = 0;
        if (b < B) {
            long long L = seq_lens[b];
            if (L < 0) {
                atomicOr(s_err, (int)HPC_DEVERR_NEGATIVE_LENGTH);
                L = 0;
            }
            n = (L + kChunk - 1) / kChunk;
        }
        long long tot;
        long long ex = block_exclusive_scan<long long>(n, &tot, warp_sums);
        if (b < B) pre[b] = (int32_t)(running + ex);
        running += tot;
    }
    const bool overflow = running * (long long)Hkv > 2147483647LL;
    __syncthreads();
    if (overflow) {
        for (int b = tid; b <= B; b += kPlanThreads) pre[b] = 0;
        if (tid == 0) atomicOr(s_err, (int)HPC_DEVERR_CHUNK_OVERFLOW);
        running = 0;
    } else if (tid == 0) {
        pre[B] = (int32_t)running;
    }
    __syncthreads();
    return running;
}

__device__ void write_header(int32_t* buf, long long T, long long bucket, long long used,
                             long long splits, int C, int B, int Hkv, int m, long long max_tasks,
                             int mode, long long N, int err) {
    buf[kHTotalChunks] = (int32_t)T;
    buf[kHBucket] = (int32_t)bucket;
    buf[kHUsedCtas] = (int32_t)used;
    buf[kHTotalSplits] = (int32_t)splits;
    buf[kHNumCtas] = C;
    buf[kHBatch] = B;
    buf[kHNumKvHeads] = Hkv;
    buf[kHMinChunks] = m;
    buf[kHMaxTasks] = (int32_t)max_tasks;
    buf[kHMode] = mode;
    buf[kHChunksPerHead] = (int32_t)N;
    buf[kHChunkTokens] = kChunk;
    buf[kHError] = err;
    buf[13] = buf[14] = buf[15] = 0;
}

__global__ void __launch_bounds__(kPlanThreads, 1)
    plan_balanced_kernel(const int32_t* __restrict__ seq_lens, int B, int Hkv, int C, int m,
                         int32_t* __restrict__ buf) {
    extern __shared__ int32_t pre[];  // [B + 1]
    __shared__ long long warp_sums[32];
    __shared__ unsigned warp_sums32[32];
    __shared__ int s_err;
    const int tid = threadIdx.x;
    if (tid == 0) s_err = 0;
    grid_dependency_wait();   // seq_lens may come from the previous kernel
    grid_launch_dependents();
    __syncthreads();

    const PlanLayout L = plan_layout(B, Hkv, C);
    int32_t* cta_off = buf + L.cta_off;
    int32_t* tasks = buf + L.tasks;
    int32_t* nsplit = buf + L.pair_nsplit;
    int32_t* split0 = buf + L.pair_split0;

    const long long N = chunk_prefix(seq_lens, B, Hkv, pre, warp_sums, &s_err);
    const long long T = N * Hkv;
    long long bucket = (T + C - 1) / C;
    if (bucket < m) bucket = m;
    if (bucket < 1) bucket = 1;
    const long long used = T ? (T + bucket - 1) / bucket : 0;
    const long long P = (long long)Hkv * B;

    // Chunk indices stay below T <= INT32_MAX (checked in chunk_prefix), and so do
    // split and task-row indices (P + 2C rows), so the per-pair work runs in 32-bit
    // unsigned arithmetic (each block is bound by instruction issue and latency).
    // A CTA range ends below T + bucket < 2^32.
    const unsigned ubucket = (unsigned)bucket, uB = (unsigned)B, uN = (unsigned)N, uT = (unsigned)T;
    const FastDiv by_bucket(ubucket), by_batch(uB);
    const int Pi = (int)P;  // P <= HPC_MAX_CTAS

    // Block k takes pairs [p_lo, p_hi), a whole number of 1024-pair tiles; every
    // block computes the same chunk prefixes, bucket and error bits itself, and
    // starts its split indices at the number of descriptors of all earlier pairs,
    // which it sums in closed form (no block waits for another).
    const int per_block = (int)(((P + kPlanThreads - 1) / kPlanThreads + gridDim.x - 1) / gridDim.x) * kPlanThreads;
    const int p_lo = min(Pi, (int)blockIdx.x * per_block), p_hi = min(Pi, p_lo + per_block);
    auto pair_splits = [&](int p) -> unsigned {
        const unsigned h = by_batch.div((unsigned)p), b = (unsigned)p - h * uB;
        const unsigned nb = (unsigned)(pre[b + 1] - pre[b]);
        const unsigned g0 = h * uN + (unsigned)pre[b];
        return nb ? by_bucket.div(g0 + nb - 1) - by_bucket.div(g0) + 1 : 0u;
    };
    unsigned running = 0;
    {
        unsigned acc = 0;
        for (int p = tid; p < p_lo; p += kPlanThreads) acc += pair_splits(p);
        unsigned tot;
        (void)block_exclusive_scan<unsigned>(acc, &tot, warp_sums32);
        running = tot;
    }

    // split count of each of the block's pairs, then its first split index
    for (int base = p_lo; base < p_hi; base += kPlanThreads) {
        const int p = base + tid;
        const unsigned ns = p < p_hi ? pair_splits(p) : 0u;
        unsigned tot;
        const unsigned ex = block_exclusive_scan<unsigned>(ns, &tot, warp_sums32);
        if (p < p_hi) {
            nsplit[p] = (int32_t)ns;
            split0[p] = (int32_t)(running + ex);
        }
        running += tot;
    }

    // Descriptors, by the thread that scanned the pair (its split0 write is its own).
    // Descriptor k of a pair lies in CTA first + k; the one that reaches the end of
    // its CTA's range [cta*bucket, min((cta+1)*bucket, T)) is the CTA's last, and the
    // CTA's terminator row follows it.
    for (int p = p_lo + tid; p < p_hi; p += kPlanThreads) {
        const unsigned h = by_batch.div((unsigned)p), b = (unsigned)p - h * uB;
        const unsigned nb = (unsigned)(pre[b + 1] - pre[b]);
        if (!nb) continue;
        const unsigned g0 = h * uN + (unsigned)pre[b], end = g0 + nb;
        const unsigned first = by_bucket.div(g0);
        const unsigned ns = by_bucket.div(end - 1) - first + 1;
        const unsigned s0 = (unsigned)split0[p];
        for (unsigned k = 0; k < ns; ++k) {
            const unsigned cta = first + k;
            const unsigned lo = cta * ubucket, hi = lo + ubucket;
            const unsigned cs = g0 > lo ? g0 : lo;
            const unsigned ce = end < hi ? end : hi;
            const unsigned s = s0 + k, slot = s + cta;
            int32_t* row = tasks + (size_t)slot * kTaskInts;
            write_row(row, (int)h, (int)b, (int)(cs - g0), (int)(ce - g0), (int)s, (int)k, (int)ns);
            if (cs == lo) cta_off[cta] = (int32_t)slot;
            if (ce == hi || ce == uT) write_term(row + kTaskInts);
        }
    }
    // the last block, whose running count is now every pair's, fills the rest
    if (blockIdx.x != gridDim.x - 1) return;
    const long long total = running;

    // unused CTAs: an empty task list each, then terminators up to the row capacity
    for (long long j = used + tid; j <= C; j += kPlanThreads) cta_off[j] = (int32_t)(total + j);
    for (long long i = L.cta_off + C + 1 + tid; i < L.tasks; i += kPlanThreads) buf[i] = 0;
    for (long long r = total + used + tid; r < L.max_tasks; r += kPlanThreads) write_term(tasks + r * kTaskInts);
    if (tid == 0)
        write_header(buf, T, bucket, used, total, C, B, Hkv, m, L.max_tasks, 0, N, s_err);
}

__global__ void __launch_bounds__(kPlanThreads, 1)
    plan_static_kernel(const int32_t* __restrict__ seq_lens, int B, int Hkv, int S,
                       int32_t* __restrict__ buf) {
    extern __shared__ int32_t pre[];  // [B + 1]
    __shared__ long long warp_sums[32];
    __shared__ int s_err;
    const int tid = threadIdx.x;
    if (tid == 0) s_err = 0;
    grid_dependency_wait();   // seq_lens may come from the previous kernel
    grid_launch_dependents();
    __syncthreads();

    const long long C = (long long)Hkv * B * S;
    const PlanLayout L = plan_layout(B, Hkv, C);
    int32_t* cta_off = buf + L.cta_off;
    int32_t* tasks = buf + L.tasks;
    int32_t* nsplit = buf + L.pair_nsplit;
    int32_t* split0 = buf + L.pair_split0;

    const long long N = chunk_prefix(seq_lens, B, Hkv, pre, warp_sums, &s_err);
    const long long P = (long long)Hkv * B;
    const FastDiv by_batch((unsigned)B);

    // non-empty splits of a pair: s*q < n_b  <=>  s < ceil(n_b / q), q = ceil(n_b / S)
    long long running = 0;
    for (long long base = 0; base < P; base += kPlanThreads) {
        const long long p = base + tid;
        long long ns = 0;
        if (p < P) {
            const unsigned b = (unsigned)p - by_batch.div((unsigned)p) * (unsigned)B;
            const unsigned nb = (unsigned)(pre[b + 1] - pre[b]);
            const unsigned q = (nb + (unsigned)S - 1) / (unsigned)S;
            ns = q ? (long long)((nb + q - 1) / q) : 0;
        }
        long long tot;
        long long ex = block_exclusive_scan(ns, &tot, warp_sums);
        if (p < P) {
            nsplit[p] = (int32_t)ns;
            split0[p] = (int32_t)(running + ex);
        }
        running += tot;
    }
    const long long total = running;
    __syncthreads();

    const unsigned uS = (unsigned)S, uB = (unsigned)B;
    const FastDiv by_splits(uS);
    for (long long j = tid; j < C; j += kPlanThreads) {
        const unsigned uj = (unsigned)j;  // C <= HPC_MAX_CTAS < 2^31
        const unsigned up = by_splits.div(uj);
        const int s = (int)(uj - up * uS);
        const int h = (int)by_batch.div(up), b = (int)(up - (unsigned)h * uB);
        const long long p = up;
        const long long nb = pre[b + 1] - pre[b];
        const long long q = ((unsigned)nb + uS - 1) / uS;
        const int ns = nsplit[p];
        const long long s0 = split0[p];
        const long long off = s0 + (s < ns ? s : ns) + j;
        cta_off[j] = (int32_t)off;
        if (s < ns) {
            const long long c0 = (long long)s * q;
            const long long c1 = (c0 + q) < nb ? (c0 + q) : nb;
            write_row(tasks + off * kTaskInts, h, b, (int)c0, (int)c1, (int)(s0 + s), s, ns);
            write_term(tasks + (off + 1) * kTaskInts);
        } else {
            write_term(tasks + off * kTaskInts);
        }
    }
    if (tid == 0) cta_off[C] = (int32_t)(total + C);
    for (long long i = L.cta_off + C + 1 + tid; i < L.tasks; i += kPlanThreads) buf[i] = 0;
    for (long long r = total + C + tid; r < L.max_tasks; r += kPlanThreads) write_term(tasks + r * kTaskInts);
    if (tid == 0)
        write_header(buf, N * Hkv, 0, total, total, (int)C, B, Hkv, S, L.max_tasks, 1, N, s_err);
}

cudaError_t set_smem(const void* fn, size_t bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

cudaError_t launch_plan(const int32_t* seq_lens, int B, int Hkv, int C, int m, int32_t* buf,
                        cudaStream_t s) {
    const size_t smem = sizeof(int32_t) * ((size_t)B + 1);
    cudaError_t e = set_smem((const void*)plan_balanced_kernel, smem);
    if (e != cudaSuccess) return e;
    const long long tiles = ((long long)Hkv * B + kPlanThreads - 1) / kPlanThreads;
    const int blocks = (int)(tiles < kPlanMaxBlocks ? tiles : kPlanMaxBlocks);
    return launch_pdl(plan_balanced_kernel, dim3(blocks), dim3(kPlanThreads), smem, s, seq_lens, B, Hkv, C, m, buf);
}

cudaError_t launch_plan_static(const int32_t* seq_lens, int B, int Hkv, int S, int32_t* buf,
                               cudaStream_t s) {
    const size_t smem = sizeof(int32_t) * ((size_t)B + 1);
    cudaError_t e = set_smem((const void*)plan_static_kernel, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(plan_static_kernel, dim3(1), dim3(kPlanThreads), smem, s, seq_lens, B, Hkv, S, buf);
}

}  // namespace hpc
