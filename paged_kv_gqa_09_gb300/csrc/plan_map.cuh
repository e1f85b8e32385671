// plan_map.cuh -- one position of the workqueue's balance order -> its task.
//
// "PersistentKV: Page-Aware Decode Scheduling for Long-Context LLM Serving on
// Commodity GPUs", technical summary, Methodology 1, "Row-local bounds" and
// "Compact workqueue".  Row i of length N_i has f_i = floor(N_i / C) full
// splits and r_i = 1 more, shorter, split when C does not divide N_i; its
// n_i = f_i + r_i states start at offsets_i = F_i + R_i, where F and R are the
// exclusive prefix sums of f and r over the rows.  The task list in
// lexicographic (row, kv head, split) order is the contract; the decode's CTAs
// consume the same records in balance order:
//   positions [0, Hkv*F_B)         every full split by (row, split, kv head):
//                                  row i owns Hkv*f_i of them, and the Hkv
//                                  heads of one split sit side by side, so
//                                  CTAs that claim them together read the
//                                  same pages at about the same time;
//   positions [Hkv*F_B, Hkv*(F_B+R_B))  each shorter last split, longest
//                                  class first, then by row, then kv head.
//                                  The class of a shorter split of
//                                  N_i mod C tokens is
//                                  floor(kShortClasses * (N_i mod C) / C):
//                                  the launch ends on its shortest tasks, so
//                                  the CTAs finish closer together.
// Both lists are the plan kernel's output; the self-planning decode rebuilds
// the mapping from F, R and the class-ordered list of rows with a shorter
// split (S), held in shared memory.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv {

// Rows that the self-planning decode keeps in shared memory.
constexpr int kSelfPlanMaxB = 512;

// Length classes of the shorter last splits (the balance order takes them
// from the longest class down).
constexpr int kShortClasses = 8;

// Class of a shorter split of r tokens, 0 < r < C.
__host__ __device__ inline int plan_short_class(int r, int C)
{
    return (int)(((int64_t)r * kShortClasses) / C);
}

// Largest i in [0, B) with key * pre[i] <= x (pre non-decreasing, pre[0] = 0 <= x).
__host__ __device__ inline int plan_last_row_at_or_below(const int *pre, int B, int key, int x)
{
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)key * pre[mid] <= x)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// The task at balance position t (0 <= t < Hkv*(F[B]+R[B])) as the record
// {row, kv head, split, first state slot}, and its lexicographic index.
// F and R hold B + 1 entries each; S holds the R[B] rows that end in a
// shorter split, in balance order.
__host__ __device__ inline int4 plan_task_at(int t, const int *F, const int *R, const int16_t *S, int B,
                                             int Hkv, int Hq, int G, int64_t *lex)
{
    const int n_full = Hkv * F[B];
    int i, g, j;
    if (t < n_full) {
        i = plan_last_row_at_or_below(F, B, Hkv, t);
        const int kk = t - Hkv * F[i];
        j = kk / Hkv;
        g = kk - j * Hkv;
    } else {
        const int u = t - n_full;
        const int q = u / Hkv;
        g = u - q * Hkv;
        i = S[q];
        j = F[i + 1] - F[i];  // the shorter split comes after the row's full ones
    }
    const int off = F[i] + R[i];
    const int n = (F[i + 1] - F[i]) + (R[i + 1] - R[i]);
    if (lex)
        *lex = (int64_t)Hkv * off + (int64_t)g * n + j;
    return make_int4(i, g, j, (off + j) * Hq + g * G);
}

}  // namespace pkv
