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
#include "pkv_device.cuh"
#include "pkv_kernels.h"

namespace pkv {
namespace {

constexpr int kPlanThreads = 1024;

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const PlanParams p)
{
    __shared__ int warp_tot[32];
    __shared__ int chunk_tot;
    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    int carry = 0;
    for (int base = 0; base < p.B; base += kPlanThreads) {
        const int i = base + tid;
        int n = 0;
        if (i < p.B) {
            int N = p.seq_lens[i];
            N = N < 0 ? 0 : (N > p.len_cap ? p.len_cap : N);
            n = (N + p.C - 1) / p.C;
        }
        int x = n;  // inclusive warp scan
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o)
                x += y;
        }
        if (lane == 31)
            warp_tot[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int t = warp_tot[lane];
            int s = t;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, s, o);
                if (lane >= o)
                    s += y;
            }
            warp_tot[lane] = s - t;  // exclusive prefix of warp totals
            if (lane == 31)
                chunk_tot = s;
        }
        __syncthreads();
        if (i < p.B)
            p.offsets[i] = carry + warp_tot[warp] + x - n;
        carry += chunk_tot;
        __syncthreads();
    }
    const int64_t T = (int64_t)carry * p.Hkv;
    const bool overflow = T > p.max_tasks;
    if (tid == 0) {
        p.offsets[p.B] = carry;
        p.ws->task_count = overflow ? 0 : (int32_t)T;
        p.ws->state_rows = carry;
        p.ws->overflow = overflow ? 1 : 0;
        if (overflow)
            report_error(p.ws, kErrCapacity, (int32_t)(T > 0x7fffffff ? 0x7fffffff : T),
                         (int32_t)p.max_tasks, 0);
    }
    __syncthreads();
    if (overflow)
        return;
    for (int64_t k = tid; k < T; k += kPlanThreads) {
        // last row i in [0, B-1] with Hkv * offsets[i] <= k
        int lo = 0, hi = p.B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if ((int64_t)__ldcg(p.offsets + mid) * p.Hkv <= k)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int oi = __ldcg(p.offsets + lo);
        const int ni = __ldcg(p.offsets + lo + 1) - oi;
        const int kk = (int)(k - (int64_t)oi * p.Hkv);
        const int g = kk / ni, j = kk - g * ni;
        p.tasks[k] = make_int4(lo, g, j, (oi + j) * p.Hq + g * p.G);
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
