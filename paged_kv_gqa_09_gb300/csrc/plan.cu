// plan.cu -- row-local bounds and the compact workqueue, built on the device.
//
// "PersistentKV: Page-Aware Decode Scheduling for Long-Context LLM Serving on
// Commodity GPUs", technical summary, Methodology 1, "Row-local bounds" and
// "Compact workqueue": split counts come from each row's real length N*_i and
// the scheduler emits a 1D list holding only the non-empty (row, kv-head,
// split) intervals.
//
// One CTA of 1024 threads:
//   n_i = ceil(N*_i / C); offsets = exclusive scan of n (block scan in chunks
//   of 1024 rows); T = Hkv * sum n; task k of row i (Hkv*offsets[i] <= k <
//   Hkv*offsets[i+1]) is {i, g, j, (offsets[i] + j)*Hq + g*G} with
//   g = (k - Hkv*offsets[i]) / n_i, j = ... % n_i -- the lexicographic
//   (row, kv-head, split) order.  The host never reads T back.
// A second copy of the same records, in balance order (every full-length
// split first, by row, split and kv head, then the shorter last splits,
// longest length class first, by row and kv head), is what the decode
// kernel's CTAs claim from: the launch ends on its shortest tasks, and the kv
// heads of one split, claimed together, read the same pages at about the
// same time.
#include "pkv_device.cuh"
#include "pkv_kernels.h"
#include "plan_map.cuh"

namespace pkv {
namespace {

constexpr int kPlanThreads = 1024;

// Block-wide exclusive scan of one int per thread; returns the exclusive prefix
// and sets *total to the block sum.
__device__ __forceinline__ int block_exclusive_scan(int x, int *warp_tot, int *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += y;
    }
    if (lane == 31)
        warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int t = warp_tot[lane];
        int sc = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, sc, o);
            if (lane >= o)
                sc += y;
        }
        warp_tot[lane] = sc - t;
        if (lane == 31)
            warp_tot[32] = sc;
    }
    __syncthreads();
    const int ex = warp_tot[warp] + incl - x;
    *total = warp_tot[32];
    __syncthreads();
    return ex;
}

// A row's counts for the plan: its splits n_i, and its shorter split (if
// any) as a one-hot 16-bit counter of its length class -- classes 0..3 in
// `lo`, 4..7 in `hi` (each counter stays below 2^16 within one block of
// rows), so that the sum of the eight counters is r_i.
struct RowCounts {
    int n;
    unsigned long long lo, hi;
};

__device__ __forceinline__ RowCounts operator+(const RowCounts &x, const RowCounts &y)
{
    return RowCounts{x.n + y.n, x.lo + y.lo, x.hi + y.hi};
}

__device__ __forceinline__ RowCounts operator-(const RowCounts &x, const RowCounts &y)
{
    return RowCounts{x.n - y.n, x.lo - y.lo, x.hi - y.hi};
}

__device__ __forceinline__ RowCounts shfl_up_counts(const RowCounts &x, int o)
{
    return RowCounts{__shfl_up_sync(0xffffffffu, x.n, o), __shfl_up_sync(0xffffffffu, x.lo, o),
                     __shfl_up_sync(0xffffffffu, x.hi, o)};
}

// Block-wide exclusive scan of every count of a row at once (one pass, one
// set of barriers); sets *total to the block sums.
__device__ __forceinline__ RowCounts block_exclusive_scan_counts(const RowCounts &x, RowCounts *warp_tot,
                                                                 RowCounts *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    RowCounts incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const RowCounts y = shfl_up_counts(incl, o);
        if (lane >= o)
            incl = incl + y;
    }
    if (lane == 31)
        warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const RowCounts t = warp_tot[lane];
        RowCounts sc = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const RowCounts y = shfl_up_counts(sc, o);
            if (lane >= o)
                sc = sc + y;
        }
        warp_tot[lane] = sc - t;
        if (lane == 31)
            warp_tot[32] = sc;
    }
    __syncthreads();
    const RowCounts ex = warp_tot[warp] + incl - x;
    *total = warp_tot[32];
    __syncthreads();
    return ex;
}

// Counter c (0..7) of a row's packed class counters, and the sum of all
// eight (the shorter splits).
__device__ __forceinline__ int class_count(const RowCounts &x, int c)
{
    return (int)(((c < 4 ? x.lo : x.hi) >> (16 * (c & 3))) & 0xffffull);
}

__device__ __forceinline__ int short_count(const RowCounts &x)
{
    int r = 0;
#pragma unroll
    for (int c = 0; c < kShortClasses; ++c)
        r += class_count(x, c);
    return r;
}

// The fused append: for every row i with length N, write k_new[i], v_new[i]
// into page block_table[i][N / P], slot N % P, and set the length to N + 1.
// With a free list, a row whose new token starts a page (N % P == 0) takes
// free_pages[count - 1 - rank], rank = the row's place among such rows (a
// block scan, so the assignment is deterministic), and the table names it.
// A row that cannot append (no room in its table, no free page, a bad page
// id) keeps its length and the error is recorded.  Rows are processed in
// chunks of one block: each thread settles its row's destination, then the
// whole block copies the chunk's tokens 16 bytes at a time.
__device__ void append_tokens(const PlanParams &p, int *warp_tot, long long *s_dst)
{
    const int tid = threadIdx.x;
    const int P = 1 << p.log2P;
    const int chunks = p.Hkv * p.d / 8;  // 16-byte chunks of one token's K (or V)
    const int avail = p.free_pages ? *p.free_count : 0;
    int taken = 0;
    for (int base = 0; base < p.B; base += kPlanThreads) {
        const int i = base + tid;
        int N = 0, need = 0;
        if (i < p.B) {
            N = p.seq_lens_rw[i];
            need = (p.free_pages && N >= 0 && (N & (P - 1)) == 0 && N < p.len_cap) ? 1 : 0;
        }
        int tot;
        const int rank = block_exclusive_scan(need, warp_tot, &tot);
        int page = -1;
        bool ok = i < p.B && N >= 0 && N < p.len_cap;
        if (i < p.B && !ok)
            report_error(p.ws, N < 0 ? kErrNegLen : kErrTooLong, i, N, p.len_cap);
        if (ok && need) {
            const int slot = avail - 1 - (taken + rank);
            if (slot < 0) {
                report_error(p.ws, kErrNoPage, i, N, avail);
                ok = false;
            } else {
                page = p.free_pages[slot];
                p.bt[(int64_t)i * p.bt_stride + (N >> p.log2P)] = page;
            }
        } else if (ok) {
            page = p.bt[(int64_t)i * p.bt_stride + (N >> p.log2P)];
        }
        if (ok && (page < 0 || page >= p.num_pages)) {
            report_error(p.ws, kErrBadPage, i, N >> p.log2P, page);
            ok = false;
        }
        s_dst[tid] = ok ? (long long)(((size_t)page * P + (N & (P - 1))) * (size_t)chunks) : -1ll;
        if (ok)
            p.seq_lens_rw[i] = N + 1;
        __syncthreads();
        const int rows = min(kPlanThreads, p.B - base);
        const int total = rows * chunks;
        constexpr int U = 4;
        for (int e0 = tid; e0 < total; e0 += kPlanThreads * U) {
            int4 a[U], b[U];
            long long dst[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int e = e0 + u * kPlanThreads;
                dst[u] = -1;
                if (e < total) {
                    const int r = e / chunks, c = e - r * chunks;
                    if (s_dst[r] >= 0) {
                        dst[u] = s_dst[r] + c;
                        const size_t src = (size_t)(base + r) * chunks + c;
                        a[u] = reinterpret_cast<const int4 *>(p.k_new)[src];
                        b[u] = reinterpret_cast<const int4 *>(p.v_new)[src];
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (dst[u] >= 0) {
                    reinterpret_cast<int4 *>(p.k_cache)[dst[u]] = a[u];
                    reinterpret_cast<int4 *>(p.v_cache)[dst[u]] = b[u];
                }
            }
        }
        taken += tot;
        __syncthreads();
    }
    if (tid == 0 && p.free_pages)
        *p.free_count = avail - (taken < avail ? taken : avail);
    __syncthreads();
}

// n_i = ceil(N_i / C) of row i, r_i = 1 when it ends in a shorter split and
// that split's length class (-1 without one), the length clamped to
// [0, len_cap] (reported when it was outside).
__device__ __forceinline__ void row_splits(const PlanParams &p, int i, bool report, int &n, int &r, int &cls)
{
    int N = p.k_new ? p.seq_lens_rw[i] : p.seq_lens[i];  // the same thread appended to it
    if (report && (N < 0 || N > p.len_cap))
        report_error(p.ws, N < 0 ? kErrNegLen : kErrTooLong, i, N, p.len_cap);
    N = N < 0 ? 0 : (N > p.len_cap ? p.len_cap : N);
    n = (N + p.C - 1) / p.C;
    r = (N % p.C) != 0 ? 1 : 0;
    cls = r ? plan_short_class(N % p.C, p.C) : -1;
}

// A row's counts from its splits and its shorter split's class (-1: none).
__device__ __forceinline__ RowCounts row_counts(int n, int cls)
{
    RowCounts x{n, 0ull, 0ull};
    if (cls >= 0 && cls < 4)
        x.lo = 1ull << (16 * cls);
    else if (cls >= 4)
        x.hi = 1ull << (16 * (cls - 4));
    return x;
}
static_assert(kShortClasses == 8, "two packed words of four classes");

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const PlanParams p)
{
    __shared__ int warp_tot[33];
    __shared__ RowCounts warp_counts[33];
    __shared__ long long s_dst[kPlanThreads];
    // offsets and short-split prefix of the current chunk's rows (+ the row
    // after), and each row's place among the shorter splits in balance order
    __shared__ int s_off[kPlanThreads + 1];
    __shared__ int s_sb[kPlanThreads + 1];
    __shared__ int s_srank[kPlanThreads];
    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x;

    if (p.k_new)
        append_tokens(p, warp_tot, s_dst);
    // the balance order puts every full-length split before the shorter last
    // splits, and those by length class, so the totals are needed before the
    // first task is written: one extra pass over the lengths when the rows
    // span several chunks
    int total = 0, total_r = 0;
    int in_class[kShortClasses] = {};
    const bool chunks = p.B > kPlanThreads;
    if (chunks) {
        for (int base = 0; base < p.B; base += kPlanThreads) {
            int n = 0, r = 0, cls = -1;
            if (base + tid < p.B)
                row_splits(p, base + tid, false, n, r, cls);
            RowCounts tot;
            block_exclusive_scan_counts(row_counts(n, cls), warp_counts, &tot);
            total += tot.n;
            total_r += short_count(tot);
#pragma unroll
            for (int c = 0; c < kShortClasses; ++c)
                in_class[c] += class_count(tot, c);
        }
    }
    int carry = 0, carry_r = 0;
    int class_next[kShortClasses];  // next place among the shorter splits, per class
    bool overflow = false;
    int64_t n_full = 0;
    for (int base = 0; base < p.B || base == 0; base += kPlanThreads) {
        const int i = base + tid;
        int n = 0, r = 0, cls = -1;
        if (i < p.B)
            row_splits(p, i, true, n, r, cls);
        RowCounts tot;
        const RowCounts ex = block_exclusive_scan_counts(row_counts(n, cls), warp_counts, &tot);
        const int ex_r = short_count(ex), tot_r = short_count(tot);
        const int rows = min(kPlanThreads, p.B - base);
        if (base == 0) {
            if (!chunks) {
                total = tot.n;
                total_r = tot_r;
#pragma unroll
                for (int c = 0; c < kShortClasses; ++c)
                    in_class[c] = class_count(tot, c);
            }
            int acc = 0;
#pragma unroll
            for (int c = kShortClasses - 1; c >= 0; --c) {
                class_next[c] = acc;
                acc += in_class[c];
            }
            const int64_t T = (int64_t)total * p.Hkv;
            overflow = T > p.max_tasks;
            n_full = T - (int64_t)total_r * p.Hkv;
            if (tid == 0) {
                p.offsets[p.B] = total;
                p.ws->task_count = overflow ? 0 : (int32_t)T;
                p.ws->state_rows = total;
                p.ws->overflow = overflow ? 1 : 0;
                if (overflow)
                    report_error(p.ws, kErrCapacity, (int32_t)(T > 0x7fffffff ? 0x7fffffff : T),
                                 (int32_t)p.max_tasks, 0);
            }
        }
        if (i < p.B) {
            p.offsets[i] = carry + ex.n;
            p.short_before[i] = carry_r + ex_r;
            s_off[tid] = carry + ex.n;
            s_sb[tid] = carry_r + ex_r;
            if (cls >= 0)
                s_srank[tid] = class_next[cls] + class_count(ex, cls);
        }
        if (tid == 0) {
            s_off[rows] = carry + tot.n;
            s_sb[rows] = carry_r + tot_r;
        }
        __syncthreads();
        if (!overflow) {
            // this chunk's tasks: k in [Hkv * carry, Hkv * (carry + tot.n)), lexicographic
            const int64_t k1 = (int64_t)(carry + tot.n) * p.Hkv;
            for (int64_t k = (int64_t)carry * p.Hkv + tid; k < k1; k += kPlanThreads) {
                // last chunk row lo with Hkv * offsets <= k (rows without splits share
                // the next row's offset, so the search lands on the row holding k)
                int lo = 0, hi = rows - 1;
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if ((int64_t)s_off[mid] * p.Hkv <= k)
                        lo = mid;
                    else
                        hi = mid - 1;
                }
                const int oi = s_off[lo];
                const int ni = s_off[lo + 1] - oi;
                const int kk = (int)(k - (int64_t)oi * p.Hkv);
                const int g = kk / ni, j = kk - g * ni;
                const int4 rec = make_int4(base + lo, g, j, (oi + j) * p.Hq + g * p.G);
                p.tasks[k] = rec;
                // balance order: a shorter split goes after every full one, at
                // its row's place among them, then by kv head; a full split j
                // of row i sits at Hkv * (full splits before row i + j) + g
                const int sb = s_sb[lo];
                const int has_short = s_sb[lo + 1] - sb;
                const bool is_short = has_short && j == ni - 1;
                const int64_t pos = is_short ? n_full + (int64_t)s_srank[lo] * p.Hkv + g
                                             : ((int64_t)(oi - sb) + j) * p.Hkv + g;
                p.tasks_ordered[pos] = rec;
            }
        }
        carry += tot.n;
        carry_r += tot_r;
#pragma unroll
        for (int c = 0; c < kShortClasses; ++c)
            class_next[c] += class_count(tot, c);
        __syncthreads();  // the chunk's shared offsets are rewritten next
        if (base + kPlanThreads >= p.B)
            break;
    }
}

}  // namespace

cudaError_t launch_plan(const PlanParams &p, cudaStream_t s, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kPlanThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, plan_kernel, p);
}

}  // namespace pkv
