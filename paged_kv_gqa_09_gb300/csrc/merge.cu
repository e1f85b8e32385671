// merge.cu -- the exact log-sum-exp merge of split states, and the per-step
// KV append.
//
// Merge: "PersistentKV: Page-Aware Decode Scheduling for Long-Context LLM
// Serving on Commodity GPUs", technical summary, Methodology 1, "Sequence
// splitting": a separate kernel combines the partial online-softmax states
// exactly.  One 4-warp CTA per (row i, query head h) reads only the row's
// n_i = ceil(N*_i / C) states (row-local bounds):
//   M = max_j m_j; L = sum_j l_j e^{m_j - M}; o = sum_j acc_j e^{m_j - M} / L;
//   lse = M + ln L; a row with N*_i = 0 gets o = 0, lse = -inf.
// The states are few and were just written (L2-resident), so the kernel is
// latency-bound: warp w takes states j = w, w+4, ... with all of its loads
// in flight at once, and the four partial sums meet in shared memory.
#include "pkv_device.cuh"
#include "pkv_kernels.h"

namespace pkv {
namespace {

constexpr int kMergeWarps = 4;
// Batches up to this many rows: the workqueue's merge finds its row's first
// state itself, from the lengths of the rows before it.
constexpr int kEarlyBaseRows = 512;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
__global__ void __launch_bounds__(32 * kMergeWarps) merge_kernel(const MergeParams p)
{
    constexpr int VPL = D / 32;  // values per lane: 4 (d=128) or 2 (d=64)
    __shared__ float s_max[kMergeWarps];
    __shared__ float s_l[kMergeWarps];
    __shared__ __align__(16) float s_acc[kMergeWarps][D];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int lr = blockIdx.x / p.Hq, h = blockIdx.x - lr * p.Hq;
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
    if (lr >= p.n_rows)
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
        if (warp == 0) {
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
#pragma unroll 8
    for (int j = warp; j < n; j += kMergeWarps) {
        const int64_t slot = (base + j) * p.Hq + h;
        const float mj = p.part_m[slot];
        const float lj = p.part_l[slot];
        const float *a = p.part_acc + slot * D + lane * VPL;
        float x[VPL];
        if constexpr (VPL == 4) {
            const float4 t = *reinterpret_cast<const float4 *>(a);
            x[0] = t.x;
            x[1] = t.y;
            x[2] = t.z;
            x[3] = t.w;
        } else {
            const float2 t = *reinterpret_cast<const float2 *>(a);
            x[0] = t.x;
            x[1] = t.y;
        }
        const float mn = fmaxf(Mw, mj);
        const float so = ex2((Mw - mn) * kLog2e), sj = ex2((mj - mn) * kLog2e);
        L = L * so + lj * sj;
#pragma unroll
        for (int v = 0; v < VPL; ++v)
            acc[v] = acc[v] * so + x[v] * sj;
        Mw = mn;
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
    __half *out = p.o + (size_t)wg * D + lane * VPL;
    if constexpr (VPL == 4) {
        *reinterpret_cast<uint2 *>(out) = make_uint2(pack_half2(o[0], o[1]), pack_half2(o[2], o[3]));
    } else {
        *reinterpret_cast<uint32_t *>(out) = pack_half2(o[0], o[1]);
    }
    if (p.lse && lane == 0)
        p.lse[wg] = M + logf(Lt);
}

// Append: one CTA per row, one thread per 16 bytes of the row's new K and V.
__global__ void __launch_bounds__(256) append_kernel(const AppendParams p)
{
    pdl_wait();
    pdl_trigger();
    const int i = blockIdx.x;
    if (i >= p.B)
        return;
    const int N = p.seq_lens[i];
    const int P = 1 << p.log2P;
    const int chunks = p.Hkv * p.d / 8;  // 16-byte chunks per token
    bool ok = N >= 0 && (int64_t)N < (int64_t)p.bt_stride * P;
    int page = 0;
    if (ok) {
        page = p.bt[(int64_t)i * p.bt_stride + (N >> p.log2P)];
        if (page < 0 || page >= p.num_pages) {
            if (threadIdx.x == 0)
                report_error(p.ws, kErrBadPage, i, N >> p.log2P, page);
            ok = false;
        }
    } else if (threadIdx.x == 0) {
        report_error(p.ws, N < 0 ? kErrNegLen : kErrTooLong, i, N, p.bt_stride * P);
    }
    if (ok) {
        const size_t dst = ((size_t)page * P + (N & (P - 1))) * (size_t)chunks;
        const size_t src = (size_t)i * chunks;
        for (int c = threadIdx.x; c < chunks; c += blockDim.x) {
            reinterpret_cast<int4 *>(p.k_cache)[dst + c] = reinterpret_cast<const int4 *>(p.k_new)[src + c];
            reinterpret_cast<int4 *>(p.v_cache)[dst + c] = reinterpret_cast<const int4 *>(p.v_new)[src + c];
        }
    }
    __syncthreads();  // every thread has read N before it changes
    if (ok && threadIdx.x == 0)
        p.seq_lens[i] = N + 1;
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
    const int blocks = p.n_rows * p.Hq > 0 ? p.n_rows * p.Hq : 1;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = make_cfg(dim3(blocks), dim3(32 * kMergeWarps), s, attr, pdl);
    if (d == 128)
        return cudaLaunchKernelEx(&cfg, merge_kernel<128>, p);
    return cudaLaunchKernelEx(&cfg, merge_kernel<64>, p);
}

cudaError_t launch_append(const AppendParams &p, cudaStream_t s, bool pdl)
{
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = make_cfg(dim3(p.B > 0 ? p.B : 1), dim3(128), s, attr, pdl);
    return cudaLaunchKernelEx(&cfg, append_kernel, p);
}

}  // namespace pkv
