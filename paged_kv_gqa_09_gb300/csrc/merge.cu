// merge.cu -- the exact log-sum-exp merge of split states, and the per-step
// KV append.
//
// Merge: "PersistentKV: Page-Aware Decode Scheduling for Long-Context LLM
// Serving on Commodity GPUs", technical summary, Methodology 1, "Sequence
// splitting": a separate kernel combines the partial online-softmax states
// exactly.  Each (row i, query head h) reads only the row's
// n_i = ceil(N*_i / C) states (row-local bounds):
//   M = max_j m_j; L = sum_j l_j e^{m_j - M}; o = sum_j acc_j e^{m_j - M} / L;
//   lse = M + ln L; a row with N*_i = 0 gets o = 0, lse = -inf.
// The states are few and were just written (L2-resident), so the kernel is
// latency-bound.  A 4-warp CTA per (row, head): warp w takes states
// j = w, w+4, ... with all of its loads in flight at once, and the four
// partial sums meet in shared memory; or, on batches of many (row, head)
// pairs, one warp per pair and four heads of a row per CTA.
#include "pkv_device.cuh"
#include "pkv_kernels.h"

namespace pkv {
namespace {

constexpr int kMergeWarps = 4;
// Batches up to this many rows: the workqueue's merge finds its row's first
// state itself, from the lengths of the rows before it.
constexpr int kEarlyBaseRows = 512;
constexpr float kLog2e = 1.4426950408889634f;

// kRowCta = false: one CTA per (row, head), its four warps folding states
// j = w, w + 4, ... and meeting in shared memory (rows of many splits, few
// (row, head) pairs).  kRowCta = true: one warp per (row, head), a CTA serving
// four heads of one row, each warp folding all of its row's states (batches of
// many (row, head) pairs with few splits each: a quarter of the CTAs, all
// resident at once, and no exchange).
template <int D, bool kRowCta>
__global__ void __launch_bounds__(32 * kMergeWarps) merge_kernel(const MergeParams p)
{
    constexpr int VPL = D / 32;  // values per lane: 4 (d=128) or 2 (d=64)
    __shared__ float s_max[kMergeWarps];
    __shared__ float s_l[kMergeWarps];
    __shared__ __align__(16) float s_acc[kRowCta ? 1 : kMergeWarps][D];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int cpr = kRowCta ? (p.Hq + kMergeWarps - 1) / kMergeWarps : p.Hq;  // CTAs per row
    const int lr = blockIdx.x / cpr;
    const int h = kRowCta ? (blockIdx.x - lr * cpr) * kMergeWarps + warp : blockIdx.x - lr * cpr;
    // The merge reads the row list and the lengths while the decode it follows
    // is still running: both are inputs that no kernel writes between a step's
    // decode and its merge (an append that advances the lengths finished before
    // the decode started, and the next one waits for this merge), so after the
    // wait only the state loads remain.  The workqueue's offsets come from the
    // plan, which its own decode may write: on batches of up to kEarlyBaseRows
    // rows the CTA instead sums ceil(N / C) over the rows before its own (the
    // plan's definition of offsets[i]); larger ones read offsets after the wait.
    const bool rect = p.mode != kModeQueue;
    const bool early = rect || p.B <= kEarlyBaseRows;
    int i = -1, N = 0;
    int64_t base = 0;
    if (early && lr < p.n_rows) {
        i = p.rows ? p.rows[lr] : lr;
        if (i >= 0 && i < p.B)
            N = p.seq_lens[i];
    }
    if (!rect && early && lr < p.n_rows) {  // the same branch for the whole CTA
        __shared__ long long s_part[kMergeWarps];
        long long sum = 0;
        for (int r = threadIdx.x; r < i; r += 32 * kMergeWarps) {
            int Nr = p.seq_lens[r];
            Nr = Nr < 0 ? 0 : (Nr > p.len_cap ? p.len_cap : Nr);
            sum += (Nr + p.C - 1) / p.C;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane == 0)
            s_part[warp] = sum;
        __syncthreads();
        for (int w = 0; w < kMergeWarps; ++w)
            base += s_part[w];
    }
    // otherwise every libpkv kernel waits for its predecessor before touching
    // global memory, so the next one may be scheduled as soon as this one runs
    pdl_wait();
    pdl_trigger();
    if (lr >= p.n_rows || h >= p.Hq)
        return;
    if (!early) {
        i = p.rows ? p.rows[lr] : lr;  // row of the batch
        if (i >= 0 && i < p.B)
            N = p.seq_lens[i];
    }
    if (i < 0 || i >= p.B)
        return;  // reported by the decode kernel
    const int64_t wg = (int64_t)i * p.Hq + h;  // (row, head) of o and lse
    N = N < 0 ? 0 : (N > p.len_cap ? p.len_cap : N);
    int n = (N + p.C - 1) / p.C;
    bool bad = false;
    if (p.mode == kModeQueue) {
        if (!early)
            base = p.offsets[i];
        bad = p.ws->overflow != 0 || base + n > p.state_rows_cap;
    } else {
        base = (int64_t)lr * p.S_b;
        n = min(n, p.S_b);
    }
    if (bad || n == 0) {
        if (kRowCta || warp == 0) {
            __half *out = p.o + (size_t)wg * D + lane * VPL;
            const __half fill = bad ? __float2half(NAN) : __float2half(0.f);
#pragma unroll
            for (int v = 0; v < VPL; ++v)
                out[v] = fill;
            if (p.lse && lane == 0)
                p.lse[wg] = bad ? NAN : -INFINITY;
        }
        return;
    }
    // warp w folds states j = w, w+4, ... with its own running maximum, all
    // of its loads in flight together; the four warp results are then
    // rescaled to the common maximum (exact: every term keeps its e^{m_j - M})
    float Mw = -INFINITY, L = 0.f, acc[VPL];
#pragma unroll
    for (int v = 0; v < VPL; ++v)
        acc[v] = 0.f;
    // states j = first, first + js, ... in batches of kBatch: a batch's loads
    // are all issued before its first fold, so a warp waits one L2 round
    // trip per batch rather than one per state
    constexpr int kBatch = 8;
    const int js = kRowCta ? 1 : kMergeWarps;
    for (int j0 = kRowCta ? 0 : warp; j0 < n; j0 += kBatch * js) {
        float mj[kBatch], lj[kBatch], x[kBatch][VPL];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int j = j0 + u * js;
            mj[u] = -INFINITY;
            lj[u] = 0.f;
#pragma unroll
            for (int v = 0; v < VPL; ++v)
                x[u][v] = 0.f;
            if (j < n) {
                const int64_t slot = (base + j) * p.Hq + h;
                mj[u] = p.part_m[slot];
                lj[u] = p.part_l[slot];
                const float *a = p.part_acc + slot * D + lane * VPL;
                if constexpr (VPL == 4) {
                    const float4 t = *reinterpret_cast<const float4 *>(a);
                    x[u][0] = t.x;
                    x[u][1] = t.y;
                    x[u][2] = t.z;
                    x[u][3] = t.w;
                } else {
                    const float2 t = *reinterpret_cast<const float2 *>(a);
                    x[u][0] = t.x;
                    x[u][1] = t.y;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            if (j0 + u * js >= n)
                break;
            const float mn = fmaxf(Mw, mj[u]);
            const float so = ex2((Mw - mn) * kLog2e), sj = ex2((mj[u] - mn) * kLog2e);
            L = L * so + lj[u] * sj;
#pragma unroll
            for (int v = 0; v < VPL; ++v)
                acc[v] = acc[v] * so + x[u][v] * sj;
            Mw = mn;
        }
    }
    __half *out = p.o + (size_t)wg * D + lane * VPL;
    if constexpr (kRowCta) {
        // the warp holds the whole (row, head): normalise and write
        const float inv = 1.f / L;
        float o[VPL];
#pragma unroll
        for (int v = 0; v < VPL; ++v)
            o[v] = acc[v] * inv;
        if constexpr (VPL == 4) {
            *reinterpret_cast<uint2 *>(out) = make_uint2(pack_half2(o[0], o[1]), pack_half2(o[2], o[3]));
        } else {
            *reinterpret_cast<uint32_t *>(out) = pack_half2(o[0], o[1]);
        }
        if (p.lse && lane == 0)
            p.lse[wg] = Mw + logf(L);
        return;
    }
    if (lane == 0) {
        s_max[warp] = Mw;
        s_l[warp] = L;
    }
#pragma unroll
    for (int v = 0; v < VPL; ++v)
        s_acc[warp][lane * VPL + v] = acc[v];
    __syncthreads();
    if (warp != 0)
        return;
    float M = -INFINITY;
#pragma unroll
    for (int w2 = 0; w2 < kMergeWarps; ++w2)
        M = fmaxf(M, s_max[w2]);
    float sc[kMergeWarps], Lt = 0.f;
#pragma unroll
    for (int w2 = 0; w2 < kMergeWarps; ++w2) {
        sc[w2] = ex2((s_max[w2] - M) * kLog2e);  // 0 for a warp that saw no state
        Lt += s_l[w2] * sc[w2];
    }
    const float inv = 1.f / Lt;
    float o[VPL];
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
        float t = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < kMergeWarps; ++w2)
            t += s_acc[w2][lane * VPL + v] * sc[w2];
        o[v] = t * inv;
    }
    if constexpr (VPL == 4) {
        *reinterpret_cast<uint2 *>(out) = make_uint2(pack_half2(o[0], o[1]), pack_half2(o[2], o[3]));
    } else {
        *reinterpret_cast<uint32_t *>(out) = pack_half2(o[0], o[1]);
    }
    if (p.lse && lane == 0)
        p.lse[wg] = M + logf(Lt);
}

// Append: one CTA per row, its threads copying the row's new K and V 16 bytes
// at a time into page block_table[i][N / P], slot N % P, then N -> N + 1.
constexpr int kAppendThreads = 128;

// A row's new token starts a page that the free list must supply.
__device__ __forceinline__ bool append_needs_page(const AppendParams &p, int N, int64_t cap)
{
    return N >= 0 && (int64_t)N < cap && (N & ((1 << p.log2P) - 1)) == 0;
}

// Where row i's token goes: its page, or -1 when the row cannot append (no
// room in its table, no free page left, a bad page id).  With `commit` (the
// row's own CTA) an allocated page is entered in the block table and a
// failure is reported; without, nothing is written.
__device__ int append_page(const AppendParams &p, int i, int N, int avail, int rank, bool commit)
{
    const int64_t cap = (int64_t)p.bt_stride << p.log2P;
    if (N < 0 || (int64_t)N >= cap) {
        if (commit)
            report_error(p.ws, N < 0 ? kErrNegLen : kErrTooLong, i, N, (int32_t)cap);
        return -1;
    }
    int page;
    const int64_t entry = (int64_t)i * p.bt_stride + (N >> p.log2P);
    if (p.free_pages && append_needs_page(p, N, cap)) {
        const int slot = avail - 1 - rank;
        if (slot < 0) {
            if (commit)
                report_error(p.ws, kErrNoPage, i, N, avail);
            return -1;
        }
        page = p.free_pages[slot];
        if (commit)
            p.bt[entry] = page;
    } else {
        page = p.bt[entry];
    }
    if (page < 0 || page >= p.num_pages) {
        if (commit)
            report_error(p.ws, kErrBadPage, i, N >> p.log2P, page);
        return -1;
    }
    return page;
}

// Sum of one int per thread over the CTA (every thread gets it).
__device__ __forceinline__ int append_block_sum(int x, int *s_warp)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        x += __shfl_xor_sync(0xffffffffu, x, o);
    __syncthreads();
    if ((threadIdx.x & 31) == 0)
        s_warp[threadIdx.x >> 5] = x;
    __syncthreads();
    int t = 0;
#pragma unroll
    for (int w = 0; w < kAppendThreads / 32; ++w)
        t += s_warp[w];
    return t;
}

// Without a free list every row's CTA advances its own length.  With one, a
// row whose token starts a page takes free_pages[avail - 1 - rank], rank = the
// rows before it that need one (the order the fused append-and-plan launch
// serves them in); each CTA counts those rows from the lengths itself, so no
// length may change before every CTA has read them: the last CTA to finish
// (a counter in the workspace header, which it zeroes again) advances the
// lengths of every row that appended and lowers the free count.
__global__ void __launch_bounds__(kAppendThreads) append_kernel(const AppendParams p)
{
    __shared__ int s_warp[kAppendThreads / 32];
    __shared__ int s_last;
    pdl_wait();
    pdl_trigger();
    const int i = blockIdx.x;
    if (i >= p.B)
        return;
    const int64_t cap = (int64_t)p.bt_stride << p.log2P;
    const int N = p.seq_lens[i];
    int avail = 0, rank = 0;
    if (p.free_pages) {
        avail = *p.free_count;
        int before = 0;
        for (int r = threadIdx.x; r < i; r += kAppendThreads)
            before += append_needs_page(p, p.seq_lens[r], cap) ? 1 : 0;
        rank = append_block_sum(before, s_warp);
    }
    __shared__ int s_page;
    if (threadIdx.x == 0)
        s_page = append_page(p, i, N, avail, rank, true);
    __syncthreads();
    const int page = s_page;
    if (page >= 0) {
        const int chunks = p.Hkv * p.d / 8;  // 16-byte chunks per token
        const size_t dst = ((size_t)page << p.log2P | (size_t)(N & ((1 << p.log2P) - 1))) * chunks;
        const size_t src = (size_t)i * chunks;
        for (int c = threadIdx.x; c < chunks; c += kAppendThreads) {
            reinterpret_cast<int4 *>(p.k_cache)[dst + c] = reinterpret_cast<const int4 *>(p.k_new)[src + c];
            reinterpret_cast<int4 *>(p.v_cache)[dst + c] = reinterpret_cast<const int4 *>(p.v_new)[src + c];
        }
    }
    if (!p.free_pages) {
        __syncthreads();  // every thread has read N before it changes
        if (page >= 0 && threadIdx.x == 0)
            p.seq_lens[i] = N + 1;
        return;
    }
    __syncthreads();  // this CTA's reads of the lengths are done
    if (threadIdx.x == 0) {
        __threadfence();
        s_last = atomicAdd(&p.ws->append_done, 1) == (int)gridDim.x - 1;
    }
    __syncthreads();
    if (!s_last)
        return;
    __threadfence();
    // every other CTA has read what it needed: settle each row as its CTA did
    // (same inputs, none of them written by this launch) and advance it
    int carry = 0;
    for (int base = 0; base < p.B; base += kAppendThreads) {
        const int r = base + threadIdx.x;
        const int Nr = r < p.B ? p.seq_lens[r] : -1;
        const int need = r < p.B && append_needs_page(p, Nr, cap) ? 1 : 0;
        // exclusive prefix of `need` over this chunk's rows
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        int incl = need;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += y;
        }
        __syncthreads();
        if (lane == 31)
            s_warp[warp] = incl;
        __syncthreads();
        int before_warp = 0, chunk_total = 0;
#pragma unroll
        for (int w = 0; w < kAppendThreads / 32; ++w) {
            before_warp += w < warp ? s_warp[w] : 0;
            chunk_total += s_warp[w];
        }
        const int rank_r = carry + before_warp + incl - need;
        if (r < p.B && append_page(p, r, Nr, avail, rank_r, false) >= 0)
            p.seq_lens[r] = Nr + 1;
        carry += chunk_total;
    }
    if (threadIdx.x == 0) {
        *p.free_count = avail - (carry < avail ? carry : avail);
        p.ws->append_done = 0;
    }
}

cudaLaunchConfig_t make_cfg(dim3 grid, dim3 block, cudaStream_t s, cudaLaunchAttribute *attr, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

}  // namespace

cudaError_t launch_merge(int d, const MergeParams &p, cudaStream_t s, bool pdl)
{
    const int per_row = p.row_cta ? (p.Hq + kMergeWarps - 1) / kMergeWarps : p.Hq;
    const int blocks = p.n_rows * per_row > 0 ? p.n_rows * per_row : 1;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = make_cfg(dim3(blocks), dim3(32 * kMergeWarps), s, attr, pdl);
    if (p.row_cta)
        return d == 128 ? cudaLaunchKernelEx(&cfg, merge_kernel<128, true>, p)
                        : cudaLaunchKernelEx(&cfg, merge_kernel<64, true>, p);
    return d == 128 ? cudaLaunchKernelEx(&cfg, merge_kernel<128, false>, p)
                    : cudaLaunchKernelEx(&cfg, merge_kernel<64, false>, p);
}

cudaError_t launch_append(const AppendParams &p, cudaStream_t s, bool pdl)
{
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = make_cfg(dim3(p.B > 0 ? p.B : 1), dim3(kAppendThreads), s, attr, pdl);
    return cudaLaunchKernelEx(&cfg, append_kernel, p);
}

}  // namespace pkv
