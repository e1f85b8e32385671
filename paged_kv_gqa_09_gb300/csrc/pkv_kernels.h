// pkv_kernels.h -- kernel parameter blocks and launchers shared between the
// kernels (*.cu) and the C-ABI layer (api.cu).  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv {

struct WsHeader;

enum Mode : int { kModeRect = 0, kModeQueue = 1, kModeSingle = 2 };

// Byte offsets inside the plan workspace.
constexpr size_t kWsHeaderBytes = 64;
inline size_t ws_offsets_off() { return kWsHeaderBytes; }
inline size_t ws_tasks_off(int B)
{
    size_t o = kWsHeaderBytes + sizeof(int32_t) * (size_t)(B + 1);
    return (o + 15) & ~(size_t)15;
}
// Workqueue-only regions after the canonical task list (max_tasks records):
// the balance-ordered copy, then short_before[B].
inline size_t ws_ordered_off(int B, int64_t max_tasks) { return ws_tasks_off(B) + 16 * (size_t)max_tasks; }
inline size_t ws_short_off(int B, int64_t max_tasks) { return ws_ordered_off(B, max_tasks) + 16 * (size_t)max_tasks; }

struct PlanParams {
    const int32_t *seq_lens;
    WsHeader *ws;
    int32_t *offsets;       // [B+1]
    int32_t *short_before;  // [B]: rows before i whose last split is shorter than C
    int4 *tasks;            // [max_tasks], canonical order
    int4 *tasks_ordered;    // [max_tasks], balance order
    int B, Hq, Hkv, G, C;
    int len_cap;       // bt_stride * page_size: lengths are clamped to it
    int64_t max_tasks;
    // fused append (k_new != nullptr): before planning, write one new token per
    // row and advance its length; with free_pages, a token that starts a page
    // takes one from the free list
    const __half *k_new, *v_new;
    __half *k_cache, *v_cache;
    int32_t *bt;                // written when a page is allocated
    int32_t *seq_lens_rw;       // the lengths, advanced in place
    const int32_t *free_pages;  // free page ids, top of the stack at the end
    int32_t *free_count;        // entries of free_pages in use
    int d, log2P, num_pages, bt_stride;
};

struct DecodeParams {
    const __half *q;
    const int32_t *bt;
    const int32_t *seq_lens;
    const int4 *tasks;  // workqueue mode
    const int32_t *rows;  // rect mode: the launch covers rows[0..n_rows) (nullptr: rows 0..B)
    WsHeader *ws;
    float *part_acc, *part_m, *part_l;  // split modes
    __half *o;                           // single-pass and fused-merge modes
    float *lse;                          // single-pass and fused-merge modes (nullable)
    // fused merge (split modes): after a grid-wide barrier the CTAs merge the
    // rows' states into o / lse
    int fuse;
    const int32_t *offsets;  // workqueue: first state row of each batch row
    int n_rows;              // rows of the launch (rect: rows[] entries, else B)
    // self-planning workqueue (self_plan != 0, B <= kSelfPlanMaxB, no fused
    // merge): every CTA derives the tasks from the lengths in shared memory,
    // and the launch writes the plan -- header, offsets, short_before and both
    // task lists -- exactly as the plan kernel would
    int self_plan;
    int32_t *plan_offsets, *plan_short_before;
    int4 *plan_tasks, *plan_ordered;
    int B, Hq, Hkv, G, num_pages, bt_stride;
    int log2P;         // page size = 1 << log2P
    int box_log2;      // tokens per TMA box = 1 << box_log2 (min(P, 64))
    int C;             // split tokens (split modes)
    int S_b;           // rectangular grid splits per row
    int n_tasks;       // rect/single: tasks in the grid; queue: capacity
    int len_cap;       // bt_stride * page_size
    float scale_log2;  // scale * log2(e)
    int starve_first_stage;  // test hook: CTA 0 never fills its first stage
};

struct MergeParams {
    const int32_t *rows;  // rect mode: merge rows[0..n_rows) (nullptr: rows 0..B)
    int n_rows;
    const int32_t *seq_lens;
    const int32_t *offsets;  // workqueue mode
    const WsHeader *ws;
    const float *part_acc, *part_m, *part_l;
    __half *o;
    float *lse;  // nullable
    int B, Hq, C, S_b, mode;
    int len_cap;
    int64_t state_rows_cap;  // partial-state rows the buffer holds
    int row_cta;             // one warp per (row, head), four heads of a row per CTA
};

struct AppendParams {
    const __half *k_new, *v_new;
    int32_t *bt;  // written only when a page is allocated
    int32_t *seq_lens;
    __half *k_cache, *v_cache;
    WsHeader *ws;
    // with free_pages, a token that starts a page takes one from the free list
    const int32_t *free_pages;  // free page ids, top of the stack at the end
    int32_t *free_count;        // entries of free_pages in use
    int B, Hkv, d, log2P, num_pages, bt_stride;
};

cudaError_t launch_plan(const PlanParams &p, cudaStream_t s, bool pdl);
cudaError_t launch_decode(int d, int mode, const CUtensorMap &tk, const CUtensorMap &tv,
                          const DecodeParams &p, int grid, cudaStream_t s, bool pdl);
cudaError_t launch_merge(int d, const MergeParams &p, cudaStream_t s, bool pdl);
cudaError_t launch_append(const AppendParams &p, cudaStream_t s, bool pdl);

// Dynamic shared memory a decode CTA uses for head dim d, and how many such
// CTAs an SM holds.
int decode_smem_bytes(int d);
cudaError_t decode_ctas_per_sm(int d, int *out);

// Set the calling thread's pkv_last_error_string() and return `code`.
int record_error(int code, const char *msg);

}  // namespace pkv
