// decode.cu -- the split-decode kernel of "PersistentKV: Page-Aware Decode
// Scheduling for Long-Context LLM Serving on Commodity GPUs" (technical
// summary, Methodology 1: native block-table decode engine), written for
// sm_103a.
//
// One persistent kernel serves the three task sources:
//   rect   -- the length-bucketed rectangular grid B x Hkv x S_b
//             ("Row-local bounds": an empty split writes the neutral state and
//             reads no KV);
//   queue  -- the compact 1D workqueue of non-empty (row, kv-head, split)
//             tasks ("Compact workqueue"), read from the plan kernel's list or,
//             for batches of up to kSelfPlanMaxB rows, derived by the CTA's
//             producer warp from the row lengths (the launch then writes the
//             plan itself);
//   single -- one task per (row, kv-head) over the whole row, writing o/lse
//             directly (the policy's no-split route).
//
// CTA layout (160 threads, two CTAs per SM, ~104 KB shared memory each):
//   warp 4      producer: walks this CTA's tasks (claimed one at a time in
//               the workqueue's balance order, or a static stride over the
//               task index), reads block-table entries, and streams each 64-token
//               tile of K and V straight from the pages into a ring of
//               shared-memory stages with TMA (cp.async.bulk.tensor, 128-byte
//               swizzle, evict-first L2 policy).  No page is repacked.
//   warps 0..3  consumers: warp w owns tokens [16w, 16w+16) of every tile and
//               keeps its own online-softmax state for the G query heads of
//               the task.  Scores S^T = K q^T (16 tokens x 8 heads) and the
//               update O^T += V^T P^T (d x 8 heads) run on tensor cores
//               (mma.sync m16n8k16, fp16 in, fp32 accumulate); P^T is formed
//               from the score fragment with movmatrix.  At a task's last tile
//               warps 1..3 park their states in their own, already consumed,
//               K rows of that stage; warp 0 merges the four states exactly,
//               writes the task's partial state (m, l, acc) -- or, in single
//               mode, o and lse -- and releases the stage for all four warps.
//               While the producer waits for the previous kernel, warp 0
//               prefetches the CTA's first tiles into L2.
// Two CTAs per SM keep every task of a 256-task launch in flight at once, so
// the DRAM bandwidth is shared per task rather than per wave of tasks.
// Every barrier wait is bounded (1 s); a timeout records an error in the
// workspace header and the CTA drains its own copies and exits.
#include "pkv_device.cuh"
#include "pkv_kernels.h"
#include "plan_map.cuh"

namespace pkv {
namespace {

constexpr int kCW = 4;                   // consumer warps
constexpr int kTile = 16 * kCW;          // tokens per pipeline stage
constexpr int kThreads = 32 * (kCW + 1); // + producer warp
constexpr int kMaxG = 8;                 // query heads per KV head handled by one n8 tile
constexpr int kSegRegs = 4;              // block-table entries per producer lane per segment
constexpr int kSeg = 32 * kSegRegs;      // pages per segment
constexpr uint64_t kWaitNs = 1000000000ull;  // bound on any barrier wait
constexpr uint64_t kDrainNs = 20000000ull;   // bound when draining after a timeout
constexpr float kLn2 = 0.6931471805599453f;

// tiles of the first task prefetched into L2 early: the workqueue's first
// tasks are full splits of at least a few tiles; deeper prefetch on the
// rectangular grid's one-row launches only competed with the real loads
constexpr int kPrefetchTiles = 4;
constexpr int kQueuePrefetchTiles = 8;

constexpr int kFirst = 1 << 16;  // stage flags (low 16 bits: valid tokens)
constexpr int kLast = 1 << 17;
constexpr int kEnd = 1 << 18;

template <int D>
struct Layout {
    static constexpr int kDch = D / 64;                 // 128-byte column blocks per row
    static constexpr int kTileBytes = kTile * D * 2;    // one K (or V) tile
    static constexpr int kQBytes = kMaxG * D * 2;
    static constexpr int kStageBytes = 2 * kTileBytes + kQBytes;
    static constexpr int kStages = (D == 128) ? 3 : 6;
    static constexpr int kMetaOff = kStages * kStageBytes;           // int4 per stage
    static constexpr int kRedOff = kMetaOff + kStages * 16;          // [stage][warp 1..3][m 8, l 8]
    static constexpr int kBarOff = kRedOff + kStages * (kCW - 1) * 2 * kMaxG * 4;
    // barriers: full[S], empty[S], merge[S]
    static constexpr int kBytes = kBarOff + 3 * kStages * 8;
    static constexpr int kAlloc = kBytes + 1024;                     // slack for alignment
    static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");
    static_assert(2 * (kAlloc + 1024) <= 228 * 1024, "two CTAs per SM");
};

struct TaskInfo {
    int i, g, sbase, t0, t1;  // row, kv head, first state slot, token range [t0, t1)
};

__device__ __forceinline__ TaskInfo shfl_task(const TaskInfo &a, int src)
{
    TaskInfo r;
    r.i = __shfl_sync(0xffffffffu, a.i, src);
    r.g = __shfl_sync(0xffffffffu, a.g, src);
    r.sbase = __shfl_sync(0xffffffffu, a.sbase, src);
    r.t0 = __shfl_sync(0xffffffffu, a.t0, src);
    r.t1 = __shfl_sync(0xffffffffu, a.t1, src);
    return r;
}

// Prefix sums of a self-planning workqueue launch in shared memory: F[i] full
// splits and R[i] shorter last splits in the rows before i (B + 1 entries
// each), and S the rows that end in a shorter split, in balance order;
// F == nullptr when the plan kernel wrote the task list.
struct SelfPlan {
    const int *F, *R;
    const int16_t *S;
};

// Workqueue task k (balance order) as {row, kv head, split, first state slot}.
__device__ __forceinline__ int4 queue_record(const DecodeParams &p, const SelfPlan &sp, int k)
{
    if (sp.F)
        return plan_task_at(k, sp.F, sp.R, sp.S, p.B, p.Hkv, p.Hq, p.G, nullptr);
    return p.tasks[k];
}

// Task k of this launch, with its row-local token range.
template <int MODE>
__device__ __forceinline__ TaskInfo load_task(const DecodeParams &p, const SelfPlan &sp, int k, int ntasks)
{
    TaskInfo ti{0, 0, 0, 0, 0};
    if (k >= ntasks)
        return ti;
    int j = 0;
    if (MODE == kModeQueue) {
        const int4 r = queue_record(p, sp, k);
        ti.i = r.x;
        ti.g = r.y;
        j = r.z;
        ti.sbase = r.w;
    } else if (MODE == kModeRect) {
        const int per_row = p.Hkv * p.S_b;
        const int lr = k / per_row;  // row of the launch (index into rows[] when given)
        const int r = k - lr * per_row;
        ti.g = r / p.S_b;
        j = r - ti.g * p.S_b;
        ti.sbase = (lr * p.S_b + j) * p.Hq + ti.g * p.G;
        ti.i = p.rows ? p.rows[lr] : lr;
        if (ti.i < 0 || ti.i >= p.B) {
            report_error(p.ws, kErrBadRow, lr, ti.i, p.B);
            ti.i = 0;
            ti.t0 = ti.t1 = 0;  // an empty task: neutral state, no KV read
            return ti;
        }
    } else {
        ti.i = k / p.Hkv;
        ti.g = k - ti.i * p.Hkv;
        ti.sbase = ti.i * p.Hq + ti.g * p.G;
    }
    int N = p.seq_lens[ti.i];
    if (N < 0) {
        report_error(p.ws, kErrNegLen, ti.i, N, 0);
        N = 0;
    }
    if (N > p.len_cap) {
        report_error(p.ws, kErrTooLong, ti.i, N, p.len_cap);
        N = p.len_cap;
    }
    if (MODE == kModeSingle) {
        ti.t0 = 0;
        ti.t1 = N;
    } else {
        if (MODE == kModeRect && N > p.S_b * p.C)
            report_error(p.ws, kErrTooLong, ti.i, N, p.S_b * p.C);
        ti.t0 = j * p.C;
        ti.t1 = min(ti.t0 + p.C, N);
    }
    return ti;
}

// Byte offset of (tile token t, 16-byte column chunk c) inside a K/V tile that
// TMA filled with 128-byte-swizzled boxes of (1 << btl) tokens x D columns,
// laid out [box][column block][token][128 bytes].
template <int D>
__device__ __forceinline__ uint32_t row_base(int t, int btl)
{
    const int b = t >> btl, s = t & ((1 << btl) - 1);
    return (uint32_t)(((b << btl) * Layout<D>::kDch + s) * 128);
}

// ---------------------------------------------------------------- fused merge
//
// With p.fuse the exact log-sum-exp merge ("Sequence splitting": the split
// states are combined exactly) runs on the decode's tail instead of in a
// second kernel: every split writes its state, the CTAs meet at a grid-wide
// barrier, then share the (row, query head) merges out (grid_merge).  A row
// with one split writes o / lse from registers at its task's end, and rows
// without tokens are filled by the producer warps after their tasks.

constexpr float kLog2e = 1.4426950408889634f;

// Splits of batch row i that hold tokens: ceil(N*_i / C), the length clamped
// as load_task clamps it (a rectangular grid holds at most S_b of them).
template <int MODE>
__device__ __forceinline__ int split_count(const DecodeParams &p, int i)
{
    int N = p.seq_lens[i];
    N = N < 0 ? 0 : (N > p.len_cap ? p.len_cap : N);
    const int n = (N + p.C - 1) / p.C;
    return MODE == kModeRect ? min(n, p.S_b) : n;
}

// The fused merge: once every CTA has finished its tasks
// (a grid-wide barrier; the grid never exceeds the CTAs the GPU holds at once,
// and dependents launch only after all of them have started, so all of them
// become resident), each CTA merges (row, query head) units u = blockIdx.x,
// blockIdx.x + gridDim.x, ... the way the merge kernel does: consumer warp w
// folds states j = w, w + 4, ... with its own running maximum, all loads in
// flight, and the four warp results meet in shared memory.  The barrier's wait
// is bounded; a CTA that gives up records a timeout and merges nothing.

template <int D, int MODE>
__device__ void grid_merge(const DecodeParams &p, uint8_t *basep, volatile int *ctl)
{
    constexpr int VPL = D / 32;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    __syncthreads();  // this CTA's states are written and all of its waits have ended
    if (tid == 0) {
        // every CTA arrives, also after a timeout, so that no other waits on it
        int ok = 1;
        const int gen = ld_acquire_gpu(&p.ws->bar_gen);
        __threadfence();  // the CTA's state stores, ordered by the barrier above, go first
        if (atomicAdd(&p.ws->bar_count, 1) == (int)gridDim.x - 1) {
            p.ws->bar_count = 0;  // ready for the next launch
            st_release_gpu(&p.ws->bar_gen, gen + 1);
        } else {
            const uint64_t t0 = globaltimer_ns();
            while (ld_acquire_gpu(&p.ws->bar_gen) == gen) {
                if (globaltimer_ns() - t0 > kWaitNs) {
                    report_error(p.ws, kErrTimeout, (int)blockIdx.x, 0, 5);
                    ok = 0;
                    break;
                }
                __nanosleep(64);
            }
        }
        ctl[1] = ok;
    }
    __syncthreads();
    if (!ctl[1] || ctl[0])
        return;
    if (MODE == kModeQueue && p.ws->overflow)
        return;  // no task ran: the producers' fill pass wrote NaN, as the merge kernel does
    float *s_m = reinterpret_cast<float *>(basep);  // [kCW] maxima, [kCW] sums, [kCW][D] acc
    float *s_l = s_m + kCW;
    float *s_acc = s_m + 4 * kCW;
    const int U = p.n_rows * p.Hq;
    for (int u = blockIdx.x; u < U; u += gridDim.x) {
        const int lr = u / p.Hq, h = u - lr * p.Hq;
        int i = lr;
        if (MODE == kModeRect && p.rows) {
            i = p.rows[lr];
            if (i < 0 || i >= p.B)
                continue;
        }
        const int n = split_count<MODE>(p, i);
        if (n <= 1)
            continue;  // written at its task's end, or by the producers' fill pass
        const int base = MODE == kModeQueue ? p.offsets[i] : lr * p.S_b;
        if (warp < kCW) {
            float Mw = -INFINITY, Lw = 0.f, acc[VPL];
#pragma unroll
            for (int v = 0; v < VPL; ++v)
                acc[v] = 0.f;
            // states j = warp, warp + kCW, ... in batches of kBatch, each
            // batch's loads issued before its first fold (one L2 round trip
            // per batch); read past L1, since this launch wrote them
            constexpr int kBatch = 8;
            for (int j0 = warp; j0 < n; j0 += kBatch * kCW) {
                float mj[kBatch], lj[kBatch], x[kBatch][VPL];
#pragma unroll
                for (int q = 0; q < kBatch; ++q) {
                    const int j = j0 + q * kCW;
                    mj[q] = -INFINITY;
                    lj[q] = 0.f;
#pragma unroll
                    for (int v = 0; v < VPL; ++v)
                        x[q][v] = 0.f;
                    if (j < n) {
                        const int64_t slot = (int64_t)(base + j) * p.Hq + h;
                        mj[q] = __ldcg(p.part_m + slot);
                        lj[q] = __ldcg(p.part_l + slot);
                        if constexpr (VPL == 4) {
                            const float4 t = __ldcg(reinterpret_cast<const float4 *>(p.part_acc + slot * D) + lane);
                            x[q][0] = t.x;
                            x[q][1] = t.y;
                            x[q][2] = t.z;
                            x[q][3] = t.w;
                        } else {
                            const float2 t = __ldcg(reinterpret_cast<const float2 *>(p.part_acc + slot * D) + lane);
                            x[q][0] = t.x;
                            x[q][1] = t.y;
                        }
                    }
                }
#pragma unroll
                for (int q = 0; q < kBatch; ++q) {
                    if (j0 + q * kCW >= n)
                        break;
                    const float mn = fmaxf(Mw, mj[q]);
                    const float so = ex2((Mw - mn) * kLog2e), sj = ex2((mj[q] - mn) * kLog2e);
                    Lw = Lw * so + lj[q] * sj;
#pragma unroll
                    for (int v = 0; v < VPL; ++v)
                        acc[v] = acc[v] * so + x[q][v] * sj;
                    Mw = mn;
                }
            }
            if (lane == 0) {
                s_m[warp] = Mw;
                s_l[warp] = Lw;
            }
#pragma unroll
            for (int v = 0; v < VPL; ++v)
                s_acc[warp * D + lane * VPL + v] = acc[v];
        }
        __syncthreads();
        if (warp == 0) {
            float M = -INFINITY;
#pragma unroll
            for (int w2 = 0; w2 < kCW; ++w2)
                M = fmaxf(M, s_m[w2]);
            float sc[kCW], L = 0.f;
#pragma unroll
            for (int w2 = 0; w2 < kCW; ++w2) {
                sc[w2] = ex2((s_m[w2] - M) * kLog2e);  // 0 for a warp that saw no state
                L += s_l[w2] * sc[w2];
            }
            const float inv = 1.f / L;
            float o[VPL];
#pragma unroll
            for (int v = 0; v < VPL; ++v) {
                float t = 0.f;
#pragma unroll
                for (int w2 = 0; w2 < kCW; ++w2)
                    t += s_acc[w2 * D + lane * VPL + v] * sc[w2];
                o[v] = t * inv;
            }
            const int64_t oh = (int64_t)i * p.Hq + h;
            __half *out = p.o + oh * D + lane * VPL;
            if constexpr (VPL == 4)
                *reinterpret_cast<uint2 *>(out) = make_uint2(pack_half2(o[0], o[1]), pack_half2(o[2], o[3]));
            else
                *reinterpret_cast<uint32_t *>(out) = pack_half2(o[0], o[1]);
            if (p.lse && lane == 0)
                p.lse[oh] = M + logf(L);
        }
        __syncthreads();  // the shared scratch is reused by the next unit
    }
}

// Rows of the launch that no task covers: o = 0 and lse = -inf for a row
// without tokens; after a workqueue overflow (no tasks ran) every row gets
// NaN, as the merge kernel writes.  CTAs stride over the rows.
template <int D, int MODE>
__device__ void fill_uncovered_rows(const DecodeParams &p, int lane)
{
    const bool bad = MODE == kModeQueue && p.ws->overflow != 0;
    const uint32_t w2 = bad ? 0x7e007e00u : 0u;  // two fp16 NaNs, or zeros
    const int4 fill = make_int4((int)w2, (int)w2, (int)w2, (int)w2);
    for (int lr = blockIdx.x; lr < p.n_rows; lr += gridDim.x) {
        int i = lr;
        if (MODE == kModeRect && p.rows) {
            i = p.rows[lr];
            if (i < 0 || i >= p.B)
                continue;  // reported by load_task
        }
        if (!bad && split_count<MODE>(p, i) > 0)
            continue;
        int4 *out = reinterpret_cast<int4 *>(p.o + (size_t)i * p.Hq * D);
        for (int x = lane; x < p.Hq * D / 8; x += 32)
            out[x] = fill;
        if (p.lse)
            for (int h = lane; h < p.Hq; h += 32)
                p.lse[(size_t)i * p.Hq + h] = bad ? NAN : -INFINITY;
    }
}

// ---------------------------------------------------------------- producer

// Block-table entries of pages [s0, s0 + kSeg) of row i, clipped to pg_end:
// lane l holds pages s0 + l + 32 r in pid[r].  An entry outside
// [0, num_pages) is reported and replaced by num_pages, an out-of-range page
// coordinate that TMA fills with zeros.
__device__ __forceinline__ void fetch_pages(const DecodeParams &p, int i, int s0, int pg_end, int lane,
                                            int (&pid)[kSegRegs])
{
    const int64_t row_off = (int64_t)i * p.bt_stride;
#pragma unroll
    for (int r = 0; r < kSegRegs; ++r) {
        const int pp = s0 + lane + 32 * r;
        pid[r] = pp < pg_end ? p.bt[row_off + pp] : 0;
    }
}

__device__ __forceinline__ void check_pages(const DecodeParams &p, int i, int s0, int pg_end, int lane,
                                            int (&pid)[kSegRegs])
{
#pragma unroll
    for (int r = 0; r < kSegRegs; ++r) {
        const int pp = s0 + lane + 32 * r;
        if (pp < pg_end && (pid[r] < 0 || pid[r] >= p.num_pages)) {
            report_error(p.ws, kErrBadPage, i, pp, pid[r]);
            pid[r] = p.num_pages;
        }
    }
}

__device__ __forceinline__ void load_pages(const DecodeParams &p, int i, int s0, int pg_end, int lane,
                                           int (&pid)[kSegRegs])
{
    fetch_pages(p, i, s0, pg_end, lane, pid);
    check_pages(p, i, s0, pg_end, lane, pid);
}

template <int D, int MODE, bool FUSE>
__device__ __forceinline__ void run_producer(const CUtensorMap *tmK, const CUtensorMap *tmV,
                                             const DecodeParams &p, int ntasks, uint32_t sbase,
                                             uint8_t *basep, int4 *meta, uint32_t bar_full0,
                                             uint32_t bar_empty0, volatile int *fail, const SelfPlan sp)
{
    using L = Layout<D>;
    const int lane = threadIdx.x & 31;
    const int btl = p.box_log2;
    const int log2P = p.log2P;
    const uint32_t box_bytes = (uint32_t)((128 << btl) * L::kDch);
    const uint64_t pol = l2_evict_first_policy();
    const int nloc = ntasks > (int)blockIdx.x ? (ntasks - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int G = p.G;

    // task infos of this CTA's local tasks t, lane-held in windows of 32
    auto task_of = [&](int t) {
        return t < nloc ? load_task<MODE>(p, sp, (int)blockIdx.x + t * (int)gridDim.x, ntasks)
                        : TaskInfo{0, 0, 0, 0, 0};
    };
    auto seg_end = [&](const TaskInfo &ti) { return ((ti.t1 - 1) >> log2P) + 1; };
    int pid[kSegRegs], pnx[kSegRegs];
    // The first task's block-table entries are fetched before its length is
    // known (the widest range the task can cover, clipped to the row), so
    // the two loads overlap; only entries below the row end are checked.
    if (nloc > 0) {
        int i0, j0;
        if (MODE == kModeQueue) {
            const int4 r = queue_record(p, sp, (int)blockIdx.x);
            i0 = r.x;
            j0 = r.z;
        } else if (MODE == kModeRect) {
            i0 = (int)blockIdx.x / (p.Hkv * p.S_b);
            j0 = (int)blockIdx.x % p.S_b;
            if (p.rows)
                i0 = p.rows[i0];
            i0 = min(max(i0, 0), p.B - 1);  // a bad row id is reported by load_task
        } else {
            i0 = (int)blockIdx.x / p.Hkv;
            j0 = 0;
        }
        const int s00 = MODE == kModeSingle ? 0 : (j0 * p.C) >> log2P;
        const int span = MODE == kModeSingle ? kSeg : min(kSeg, p.C >> log2P);
        fetch_pages(p, i0, s00, min(p.bt_stride, s00 + span), lane, pid);
    }
    TaskInfo wa = task_of(lane), wb = task_of(32 + lane);
    TaskInfo cur = shfl_task(wa, 0);
    if (nloc > 0 && cur.t0 < cur.t1)
        check_pages(p, cur.i, cur.t0 >> log2P, min(seg_end(cur), (cur.t0 >> log2P) + kSeg), lane, pid);

    int stage = 0;
    uint32_t ph = 0;                  // lap parity of the ring
    uint32_t pend = 0, pend_par = 0;  // stages with copies in flight, and their parity
    bool ok = true;

    // The workqueue's CTAs (without the fused merge, whose end phase re-walks a
    // CTA's strided tasks) claim tasks dynamically: the first round is static,
    // then each CTA takes the next balance-order task from a counter once it
    // has issued the copies of its current one, so the longest tasks go first
    // and the short ones fill in wherever a CTA runs free.  The claim, the task
    // record and its block-table entries arrive while the consumers drain the
    // stages in flight.  Other modes stride statically over their tasks.
    constexpr bool kDyn = MODE == kModeQueue;
    int k_cur = (int)blockIdx.x;  // kDyn: balance-order index of cur
    for (int t = 0; (kDyn ? k_cur < ntasks : t < nloc) && ok; ++t) {
        TaskInfo nxt{0, 0, 0, 0, 0};
        bool nxt_live = false;
        if (!kDyn) {
            if (t > 0 && (t & 31) == 0) {
                wa = wb;
                wb = task_of(t + 32 + lane);
            }
            // the next task's first block-table entries load while this one streams
            const int tn = t + 1;
            nxt = shfl_task(((tn & 31) != 0) ? wa : wb, tn & 31);
            nxt_live = tn < nloc && nxt.t0 < nxt.t1;
            if (nxt_live)
                load_pages(p, nxt.i, nxt.t0 >> log2P, min(seg_end(nxt), (nxt.t0 >> log2P) + kSeg), lane,
                           pnx);
        }

        if (cur.t0 >= cur.t1) {
            // empty task: neutral state (split modes) or o = 0, lse = -inf (single)
            if (MODE == kModeSingle) {
                for (int x = lane; x < G * D / 8; x += 32)
                    reinterpret_cast<int4 *>(p.o + (size_t)cur.sbase * D)[x] = make_int4(0, 0, 0, 0);
                if (p.lse && lane < G)
                    p.lse[cur.sbase + lane] = -INFINITY;
            } else if (!FUSE) {  // the fused merge reads only the splits that hold tokens
                for (int x = lane; x < G * D / 4; x += 32)
                    reinterpret_cast<float4 *>(p.part_acc + (size_t)cur.sbase * D)[x] =
                        make_float4(0.f, 0.f, 0.f, 0.f);
                if (lane < G) {
                    p.part_m[cur.sbase + lane] = -INFINITY;
                    p.part_l[cur.sbase + lane] = 0.f;
                }
            }
        } else {
            const int pg_end = seg_end(cur);
            for (int s0 = cur.t0 >> log2P; s0 < pg_end && ok; s0 += kSeg) {
                if (s0 != (cur.t0 >> log2P))  // later segments of long single-pass rows
                    load_pages(p, cur.i, s0, min(pg_end, s0 + kSeg), lane, pid);
                const int ts = max(cur.t0, s0 << log2P);
                const int te = min(cur.t1, (s0 + kSeg) << log2P);
                for (int tt = ts; tt < te; tt += kTile) {
                    const int nv = min(kTile, te - tt);
                    const int flags = nv | (tt == cur.t0 ? kFirst : 0) | (tt + nv >= cur.t1 ? kLast : 0);
                    const uint32_t full = bar_full0 + stage * 8, empty = bar_empty0 + stage * 8;
                    if (!__all_sync(0xffffffffu, mbar_wait(empty, ph ^ 1, kWaitNs))) {
                        report_error(p.ws, kErrTimeout, (int)blockIdx.x, stage, 0);
                        *fail = 1;
                        ok = false;
                        break;
                    }
                    pend &= ~(1u << stage);
                    if (p.starve_first_stage && blockIdx.x == 0 && stage == 0 && ph == 0) {
                        // test hook: leave the consumers' first full barrier
                        // without arrival or copies, so their bounded wait runs out
                        if (lane == 0)
                            meta[stage] = make_int4(cur.i, cur.g, cur.sbase, flags);
                        if (++stage == L::kStages) {
                            stage = 0;
                            ph ^= 1;
                        }
                        continue;
                    }
                    const int nb = (nv + (1 << btl) - 1) >> btl;
                    const uint32_t kdst = sbase + stage * L::kStageBytes;
                    const uint32_t vdst = kdst + L::kTileBytes;
                    if (lane == 0) {
                        meta[stage] = make_int4(cur.i, cur.g, cur.sbase, flags);
                        // a task's first tile also carries its q rows, stored below:
                        // its arrival then comes after them
                        if (flags & kFirst)
                            mbar_expect_tx(full, 2u * nb * box_bytes);
                        else
                            mbar_arrive_expect_tx(full, 2u * nb * box_bytes);
                    }
                    __syncwarp();
                    // box b of the tile is page rel0 + b of the segment; the lane
                    // holding that page's entry issues its K and V copies
                    const int rel0 = (tt >> log2P) - s0;
                    const int b = (lane - rel0) & 31;
                    if (b < nb) {
                        int pg = pid[0];
#pragma unroll
                        for (int r = 1; r < kSegRegs; ++r)
                            if ((rel0 >> 5) == r)
                                pg = pid[r];
                        const int slot = (tt + (b << btl)) & ((1 << log2P) - 1);
                        tma_load_5d(kdst + b * box_bytes, tmK, full, 0, slot, 0, cur.g, pg, pol);
                        tma_load_5d(vdst + b * box_bytes, tmV, full, 0, slot, 0, cur.g, pg, pol);
                    }
                    if (flags & kFirst) {
                        // the G query rows of the task, copied with plain 16-byte loads
                        // (q may live in page-locked host memory, which kernels can
                        // address) while the K/V copies are in flight; lane 0's
                        // arrival then publishes them to the consumers
                        const int4 *qsrc = reinterpret_cast<const int4 *>(
                            p.q + ((size_t)cur.i * p.Hq + (size_t)cur.g * G) * D);
                        int4 *qdst = reinterpret_cast<int4 *>(basep + (kdst - sbase) + 2 * L::kTileBytes);
                        if constexpr (MODE == kModeQueue) {
                            for (int x = lane; x < G * D / 8; x += 32)
                                qdst[x] = qsrc[x];
                        } else {
                            // all of a lane's loads first, then its stores: one round
                            // trip (a step's first and only task per CTA on one-row
                            // launches; the workqueue measured ~0.2% slower with it)
                            constexpr int kQPerLane = kMaxG * D / 8 / 32;
                            int4 qv[kQPerLane];
#pragma unroll
                            for (int u = 0; u < kQPerLane; ++u)
                                if (lane + 32 * u < G * D / 8)
                                    qv[u] = qsrc[lane + 32 * u];
#pragma unroll
                            for (int u = 0; u < kQPerLane; ++u)
                                if (lane + 32 * u < G * D / 8)
                                    qdst[lane + 32 * u] = qv[u];
                        }
                        __syncwarp();
                        if (lane == 0)
                            mbar_arrive(full);
                    }
                    pend |= 1u << stage;
                    pend_par = (pend_par & ~(1u << stage)) | (ph << stage);
                    if (++stage == L::kStages) {
                        stage = 0;
                        ph ^= 1;
                    }
                }
            }
        }
        if (kDyn && ok) {
            int kn = 0;
            if (lane == 0)
                kn = (int)gridDim.x + atomicAdd(&p.ws->next_task, 1);
            kn = __shfl_sync(0xffffffffu, kn, 0);
            if (kn < ntasks) {
                nxt = load_task<MODE>(p, sp, kn, ntasks);
                nxt_live = nxt.t0 < nxt.t1;
                if (nxt_live)
                    load_pages(p, nxt.i, nxt.t0 >> log2P, min(seg_end(nxt), (nxt.t0 >> log2P) + kSeg),
                               lane, pnx);
            }
            k_cur = kn;
        }
        cur = nxt;
#pragma unroll
        for (int r = 0; r < kSegRegs; ++r)
            pid[r] = pnx[r];
    }
    if (kDyn && lane == 0) {
        // this CTA claims no more; the last one to get here resets the counters
        // for the next launch on this workspace (every claim precedes the fence)
        __threadfence();
        if (atomicAdd(&p.ws->done_ctas, 1) == (int)gridDim.x - 1) {
            p.ws->next_task = 0;
            p.ws->done_ctas = 0;
        }
    }
    if (ok) {
        // end-of-work sentinel
        if (__all_sync(0xffffffffu, mbar_wait(bar_empty0 + stage * 8, ph ^ 1, kWaitNs))) {
            pend &= ~(1u << stage);
            if (lane == 0) {
                meta[stage] = make_int4(0, 0, 0, kEnd);
                mbar_arrive(bar_full0 + stage * 8);
            }
            if (FUSE)
                fill_uncovered_rows<D, MODE>(p, lane);
        } else {
            report_error(p.ws, kErrTimeout, (int)blockIdx.x, stage, 1);
            *fail = 1;
            ok = false;
        }
    }
    if (!ok && lane == 0) {
        // let every copy this CTA issued land before the CTA's shared memory goes away
        for (int s = 0; s < L::kStages; ++s)
            if (pend & (1u << s))
                mbar_wait(bar_full0 + s * 8, (pend_par >> s) & 1u, kDrainNs);
    }
}

// L2 prefetch of the first `span` tokens from token t0 of row i0, kv head g0:
// lane l takes page s0 + l of the range (tiles hold whole pages when
// P <= 64); block-table entries are read past L1 and only valid page ids
// drive a prefetch.
__device__ __forceinline__ void prefetch_task_tiles(const CUtensorMap *tmK, const CUtensorMap *tmV,
                                                    const DecodeParams &p, int i0, int g0, int t0, int span)
{
    const int lane = threadIdx.x & 31;
    const int log2P = p.log2P, btl = p.box_log2;
    const int n_pages = ((span - 1) >> log2P) + 1;
    const int64_t row = (int64_t)i0 * p.bt_stride;
    const int s0 = t0 >> log2P;
    if (lane < n_pages && s0 + lane < p.bt_stride) {
        const int pg = __ldcg(p.bt + row + s0 + lane);
        if (pg >= 0 && pg < p.num_pages) {
            // one box per page when P <= 64, else the page's boxes inside the span
            for (int b = 0; (b << btl) < (1 << log2P) && (b << btl) < span; ++b) {
                tma_prefetch_5d(tmK, 0, b << btl, 0, g0, pg);
                tma_prefetch_5d(tmV, 0, b << btl, 0, g0, pg);
            }
        }
    }
}

// Before the kernel may read its inputs (griddepcontrol.wait), warm L2 with
// the first tiles of this CTA's first task: block-table entries are read
// L2-only (they may still be changing, so they must not land in L1) and only
// drive TMA prefetches, which cannot change any result.  The real loads after
// the wait re-read everything.  Rectangular and single modes: the workqueue's
// task list is being written by the plan kernel right before, and a
// self-planning workqueue finds its first task itself
// (prefetch_first_queue_tiles).
template <int D, int MODE>
__device__ __forceinline__ void prefetch_first_tiles(const CUtensorMap *tmK, const CUtensorMap *tmV,
                                                     const DecodeParams &p)
{
    if (MODE == kModeQueue || (int)blockIdx.x >= p.n_tasks)
        return;
    int i0, g0, j0;
    if (MODE == kModeRect) {
        const int per_row = p.Hkv * p.S_b;
        const int lr = (int)blockIdx.x / per_row, r = (int)blockIdx.x - lr * per_row;
        g0 = r / p.S_b;
        j0 = r - g0 * p.S_b;
        i0 = p.rows ? __ldcg(p.rows + lr) : lr;
    } else {
        i0 = (int)blockIdx.x / p.Hkv;
        g0 = (int)blockIdx.x - i0 * p.Hkv;
        j0 = 0;
    }
    if (i0 < 0 || i0 >= p.B)
        return;
    prefetch_task_tiles(tmK, tmV, p, i0, g0, MODE == kModeSingle ? 0 : j0 * p.C,
                        MODE == kModeSingle ? kPrefetchTiles * kTile : min(p.C, kPrefetchTiles * kTile));
}

// The self-planning workqueue's version, run by consumer warp 0 while the
// producer waits for the previous kernel and then plans: the CTA's first task
// is balance position blockIdx.x, and when that is a full split (the whole
// first round on a batch of long rows) its row, kv head and split follow from
// a scan of f_i = floor(N_i / C) over the lengths as they are now (read past
// L1, since they may still be changing).  Shorter first tasks are not
// prefetched.  Nothing is written; the producer's own plan decides.
__device__ __forceinline__ void prefetch_first_queue_tiles(const CUtensorMap *tmK, const CUtensorMap *tmV,
                                                           const DecodeParams &p)
{
    constexpr int kRounds = kSelfPlanMaxB / 32;
    if (p.B > kSelfPlanMaxB)
        return;
    const int lane = threadIdx.x & 31;
    const long long b = blockIdx.x;
    int len[kRounds];
#pragma unroll
    for (int u = 0; u < kRounds; ++u) {
        const int i = u * 32 + lane;
        len[u] = u * 32 < p.B && i < p.B ? __ldcg(p.seq_lens + i) : 0;
    }
    long long carry = 0;  // full splits of the rows before this round
#pragma unroll
    for (int u = 0; u < kRounds; ++u) {
        if (u * 32 >= p.B)
            break;
        const int N = min(max(len[u], 0), p.len_cap);
        const int f = N / p.C;
        long long x = f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o)
                x += y;
        }
        const long long lo = (carry + x - f) * p.Hkv;
        const unsigned m = __ballot_sync(0xffffffffu, b >= lo && b < (carry + x) * p.Hkv);
        if (m) {
            const int src = __ffs(m) - 1;
            const int kk = (int)(b - __shfl_sync(0xffffffffu, lo, src));
            const int j0 = kk / p.Hkv;
            prefetch_task_tiles(tmK, tmV, p, u * 32 + src, kk - j0 * p.Hkv, j0 * p.C,
                                min(p.C, kQueuePrefetchTiles * kTile));
            return;
        }
        carry += __shfl_sync(0xffffffffu, x, 31);
    }
}

// ---------------------------------------------------------------- consumer

// Shared-memory address where lane `lane` of consumer warp w parks 16-byte
// chunk x of its state at a task's end: inside the warp's own 16 K rows of
// the stage (16 rows x D*2 bytes == 32 lanes x D/16 chunks), chunks XOR-spread
// over the row's 16-byte slots.
template <int D>
__device__ __forceinline__ uint32_t park_addr(uint32_t ktile, int w, int lane, int x, int btl)
{
    constexpr int CPR = D / 8;  // 16-byte chunks per row
    const int e = lane * (D / 16) + x;
    const int r = e / CPR, c = e % CPR;
    return ktile + row_base<D>(16 * w + r, btl) + (uint32_t)((c >> 3) * (128 << btl)) +
           (uint32_t)(((c & 7) ^ (r & 7)) << 4);
}

template <int D, int MODE, bool FUSE>
__device__ __forceinline__ void run_consumer(const DecodeParams &p, uint32_t sbase, uint8_t *basep,
                                             const int4 *meta, uint32_t bar_full0,
                                             uint32_t bar_empty0, uint32_t bar_merge0,
                                             volatile int *fail)
{
    using L = Layout<D>;
    constexpr int KS = D / 16;  // k-steps of the QK product == m-blocks of the PV product
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int btl = p.box_log2;
    const uint32_t blk_bytes = 128u << btl;  // one 128-byte column block of a box
    const int mi = lane >> 3, r8 = lane & 7;
    // per-lane ldmatrix row addresses (see row_base): K tiles are read as
    // A = K (tokens x d), V tiles transposed as A = V^T (d x tokens)
    const uint32_t rowK = row_base<D>(16 * w + (mi & 1) * 8 + r8, btl);
    const uint32_t rowV = row_base<D>(16 * w + (mi >> 1) * 8 + r8, btl);
    const int r0 = lane >> 2;       // score fragment: tokens r0 and r0 + 8
    const int hq = lane >> 2;       // B-fragment column: query head
    const int h0 = 2 * (lane & 3);  // this lane's two heads in C fragments
    const float sl2 = p.scale_log2;
    const int G = p.G;
    float *red = reinterpret_cast<float *>(basep + L::kRedOff);

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float O[KS][4];
#pragma unroll
    for (int x = 0; x < KS; ++x)
        O[x][0] = O[x][1] = O[x][2] = O[x][3] = 0.f;
    uint32_t qf[KS][2];
#pragma unroll
    for (int x = 0; x < KS; ++x)
        qf[x][0] = qf[x][1] = 0u;

    int stage = 0;
    uint32_t ph = 0, mpar = 0;  // ring lap parity; per-stage merge-barrier parities
    for (;;) {
        const uint32_t full = bar_full0 + stage * 8;
        const bool got = __all_sync(0xffffffffu, mbar_wait(full, ph, kWaitNs));
        if (!got) {
            report_error(p.ws, kErrTimeout, (int)blockIdx.x, stage, 2);
            *fail = 1;
            return;
        }
        const int4 mt = meta[stage];
        const int fl = mt.w;
        if (fl & kEnd)
            return;
        const uint32_t kt = sbase + stage * L::kStageBytes;
        const uint32_t vt = kt + L::kTileBytes;
        if (fl & kFirst) {
            const uint8_t *qs = basep + (kt - sbase) + 2 * L::kTileBytes;
#pragma unroll
            for (int x = 0; x < KS; ++x) {
                uint32_t b0 = 0, b1 = 0;
                if (hq < G) {
                    const uint32_t *row = reinterpret_cast<const uint32_t *>(qs + hq * D * 2);
                    b0 = row[(16 * x + 2 * (lane & 3)) / 2];
                    b1 = row[(16 * x + 8 + 2 * (lane & 3)) / 2];
                }
                qf[x][0] = b0;
                qf[x][1] = b1;
            }
        }
        const int nv = fl & 0xffff;
        const int nvw = min(max(nv - 16 * w, 0), 16);
        if (nvw > 0) {
            if (nvw < 16) {
                // rows past the row end hold other tokens' (or stale) data: zero
                // them in V so that p = 0 cannot meet a NaN in the PV product
                uint8_t *vtp = basep + (vt - sbase);
                for (int x = lane; x < (16 - nvw) * (D / 8); x += 32) {
                    const int rr = nvw + x / (D / 8), c = x % (D / 8);
                    const int tok = 16 * w + rr;
                    const uint32_t off = row_base<D>(tok, btl) + (c >> 3) * blk_bytes +
                                         (uint32_t)((((c & 7) ^ (tok & 7))) << 4);
                    *reinterpret_cast<int4 *>(vtp + off) = make_int4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            // S^T = K q^T : 16 tokens x 8 heads, two accumulation chains
            float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int x = 0; x < KS; ++x) {
                const uint32_t cc = (uint32_t)((((2 * x) & 7) + (mi >> 1)) ^ r8) << 4;
                uint32_t a0, a1, a2, a3;
                ldsm_x4(kt + rowK + (x >> 2) * blk_bytes + cc, a0, a1, a2, a3);
                if (x & 1)
                    mma_16816(sb, a0, a1, a2, a3, qf[x][0], qf[x][1]);
                else
                    mma_16816(sa, a0, a1, a2, a3, qf[x][0], qf[x][1]);
            }
            const bool v0 = r0 < nvw, v1 = r0 + 8 < nvw;
            const float x0 = v0 ? (sa[0] + sb[0]) * sl2 : -INFINITY;
            const float x1 = v0 ? (sa[1] + sb[1]) * sl2 : -INFINITY;
            const float x2 = v1 ? (sa[2] + sb[2]) * sl2 : -INFINITY;
            const float x3 = v1 ? (sa[3] + sb[3]) * sl2 : -INFINITY;
            float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
            }
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float al0 = ex2(m0 - mn0), al1 = ex2(m1 - mn1);
            const float p0 = ex2(x0 - mn0), p1 = ex2(x1 - mn1);
            const float p2 = ex2(x2 - mn0), p3 = ex2(x3 - mn1);
            l0 = l0 * al0 + (p0 + p2);
            l1 = l1 * al1 + (p1 + p3);
            m0 = mn0;
            m1 = mn1;
            const uint32_t P0 = movmatrix_t(pack_half2(p0, p1));
            const uint32_t P1 = movmatrix_t(pack_half2(p2, p3));
            // O^T += V^T P^T : D x 8 heads
#pragma unroll
            for (int x = 0; x < KS; ++x) {
                O[x][0] *= al0;
                O[x][1] *= al1;
                O[x][2] *= al0;
                O[x][3] *= al1;
                const uint32_t cc = (uint32_t)((((2 * x) & 7) + (mi & 1)) ^ r8) << 4;
                uint32_t a0, a1, a2, a3;
                ldsm_x4_t(vt + rowV + (x >> 2) * blk_bytes + cc, a0, a1, a2, a3);
                mma_16816(O[x], a0, a1, a2, a3, P0, P1);
            }
        }
        __syncwarp();
        if (!(fl & kLast)) {
            if (lane == 0)
                mbar_arrive(bar_empty0 + stage * 8);
        } else {
            // ---- exact merge of the four warp states of this task
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                l0 += __shfl_xor_sync(0xffffffffu, l0, o);
                l1 += __shfl_xor_sync(0xffffffffu, l1, o);
            }
            float *rs = red + stage * (kCW - 1) * 2 * kMaxG;  // [warp 1..3][m 8 | l 8]
            // fused merge: a row of one split writes o / lse directly
            const bool direct = FUSE && split_count<MODE>(p, mt.x) == 1;
            const uint32_t mbar = bar_merge0 + stage * 8;
            const uint32_t mp = (mpar >> stage) & 1u;
            mpar ^= 1u << stage;
            if (w > 0) {
                // park: this warp has finished reading its K rows of the stage
#pragma unroll
                for (int x = 0; x < KS; ++x)
                    *reinterpret_cast<float4 *>(basep + (park_addr<D>(kt, w, lane, x, btl) - sbase)) =
                        make_float4(O[x][0], O[x][1], O[x][2], O[x][3]);
                if (lane < 4) {
                    rs[(w - 1) * 16 + h0] = m0;
                    rs[(w - 1) * 16 + h0 + 1] = m1;
                    rs[(w - 1) * 16 + 8 + h0] = l0;
                    rs[(w - 1) * 16 + 8 + h0 + 1] = l1;
                }
                fence_proxy_async_smem();  // these K rows are refilled by TMA later
                mbar_arrive(mbar);
                // warp 0 releases the stage once it has read the parked states
            } else {
                if (!__all_sync(0xffffffffu, mbar_wait(mbar, mp, kWaitNs))) {
                    report_error(p.ws, kErrTimeout, (int)blockIdx.x, stage, 3);
                    *fail = 1;
                    return;
                }
                float M0 = m0, M1 = m1;
#pragma unroll
                for (int w2 = 0; w2 < kCW - 1; ++w2) {
                    M0 = fmaxf(M0, rs[w2 * 16 + h0]);
                    M1 = fmaxf(M1, rs[w2 * 16 + h0 + 1]);
                }
                float s0 = ex2(m0 - M0), s1 = ex2(m1 - M1);
                float L0 = l0 * s0, L1 = l1 * s1;
#pragma unroll
                for (int x = 0; x < KS; ++x) {
                    O[x][0] *= s0;
                    O[x][1] *= s1;
                    O[x][2] *= s0;
                    O[x][3] *= s1;
                }
#pragma unroll
                for (int w2 = 1; w2 < kCW; ++w2) {
                    const float t0 = ex2(rs[(w2 - 1) * 16 + h0] - M0);
                    const float t1 = ex2(rs[(w2 - 1) * 16 + h0 + 1] - M1);
                    L0 += rs[(w2 - 1) * 16 + 8 + h0] * t0;
                    L1 += rs[(w2 - 1) * 16 + 8 + h0 + 1] * t1;
#pragma unroll
                    for (int x = 0; x < KS; ++x) {
                        const float4 v = *reinterpret_cast<const float4 *>(
                            basep + (park_addr<D>(kt, w2, lane, x, btl) - sbase));
                        O[x][0] += v.x * t0;
                        O[x][1] += v.y * t1;
                        O[x][2] += v.z * t0;
                        O[x][3] += v.w * t1;
                    }
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive_n(bar_empty0 + stage * 8, kCW);  // release for all four warps
                const int sb0 = mt.z;
                const bool ok0 = h0 < G, ok1 = h0 + 1 < G;
                if (MODE == kModeSingle || direct) {
                    // o / lse from registers: the whole row (single pass), or a
                    // row of one split (fused merge)
                    const int ob = MODE == kModeSingle ? sb0 : mt.x * p.Hq + mt.y * G;
                    const float i0 = 1.f / L0, i1 = 1.f / L1;
#pragma unroll
                    for (int x = 0; x < KS; ++x) {
                        const int d0 = 16 * x + r0;
                        if (ok0) {
                            p.o[(size_t)(ob + h0) * D + d0] = __float2half_rn(O[x][0] * i0);
                            p.o[(size_t)(ob + h0) * D + d0 + 8] = __float2half_rn(O[x][2] * i0);
                        }
                        if (ok1) {
                            p.o[(size_t)(ob + h0 + 1) * D + d0] = __float2half_rn(O[x][1] * i1);
                            p.o[(size_t)(ob + h0 + 1) * D + d0 + 8] = __float2half_rn(O[x][3] * i1);
                        }
                    }
                    if (lane < 4 && p.lse) {
                        if (ok0)
                            p.lse[ob + h0] = (M0 + log2f(L0)) * kLn2;
                        if (ok1)
                            p.lse[ob + h0 + 1] = (M1 + log2f(L1)) * kLn2;
                    }
                } else {
                    // the merge reads these states back soon: they are written to
                    // stay in L2 ahead of the KV stream, whose write-back into
                    // DRAM would interrupt the stream's reads
                    const uint64_t keep = l2_evict_last_policy();
#pragma unroll
                    for (int x = 0; x < KS; ++x) {
                        const int d0 = 16 * x + r0;
                        if (ok0) {
                            st_global_hint(p.part_acc + (size_t)(sb0 + h0) * D + d0, O[x][0], keep);
                            st_global_hint(p.part_acc + (size_t)(sb0 + h0) * D + d0 + 8, O[x][2], keep);
                        }
                        if (ok1) {
                            st_global_hint(p.part_acc + (size_t)(sb0 + h0 + 1) * D + d0, O[x][1], keep);
                            st_global_hint(p.part_acc + (size_t)(sb0 + h0 + 1) * D + d0 + 8, O[x][3], keep);
                        }
                    }
                    if (lane < 4) {
                        if (ok0) {
                            st_global_hint(p.part_m + sb0 + h0, M0 * kLn2, keep);
                            st_global_hint(p.part_l + sb0 + h0, L0, keep);
                        }
                        if (ok1) {
                            st_global_hint(p.part_m + sb0 + h0 + 1, M1 * kLn2, keep);
                            st_global_hint(p.part_l + sb0 + h0 + 1, L1, keep);
                        }
                    }
                }
            }
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.f;
#pragma unroll
            for (int x = 0; x < KS; ++x)
                O[x][0] = O[x][1] = O[x][2] = O[x][3] = 0.f;
        }
        if (++stage == L::kStages) {
            stage = 0;
            ph ^= 1;
        }
    }
}

// ---------------------------------------------------------- self-planning workqueue

// The plan of a workqueue launch, built by the producer warp of every CTA
// from the row lengths ("Row-local bounds": n_i = ceil(N*_i / C), row i's
// states start at the exclusive prefix of n).  Rows go 32 at a time, one per
// lane (all lengths loaded at once); a warp scan per round plus a carry gives
// the prefixes F (full splits) and R (shorter last splits) of every row,
// B + 1 entries each, in shared memory, and a ballot per length class counts
// the shorter splits of each class; a second pass over the lengths then
// places each row with a shorter split in S, longest class first and by row
// within a class.  CTA 0 also writes what the merge and the workspace's
// readers expect of the plan kernel: offsets, short_before, the header's task
// count, state rows and overflow flag, and any bad length.  Returns the task
// count (0 after an overflow of the launch's capacity).
__device__ __forceinline__ int self_plan_warp(const DecodeParams &p, int *F, int *R, int16_t *S)
{
    constexpr int kRounds = kSelfPlanMaxB / 32;
    const int lane = threadIdx.x & 31;
    const bool cta0 = blockIdx.x == 0;
    if (p.B > kSelfPlanMaxB) {  // the host never launches this; decode nothing, merge NaN
        if (cta0 && lane == 0) {
            p.ws->task_count = 0;
            p.ws->overflow = 1;
            report_error(p.ws, kErrCapacity, p.B, kSelfPlanMaxB, 1);
        }
        return 0;
    }
    int len[kRounds];
#pragma unroll
    for (int u = 0; u < kRounds; ++u) {
        const int i = u * 32 + lane;
        len[u] = i < p.B ? p.seq_lens[i] : 0;
    }
    long long cf = 0, cr = 0;  // splits of the rows before this round
    int in_class[kShortClasses];  // shorter splits per length class
#pragma unroll
    for (int c = 0; c < kShortClasses; ++c)
        in_class[c] = 0;
#pragma unroll
    for (int u = 0; u < kRounds; ++u) {
        if (u * 32 >= p.B)
            break;
        const int i = u * 32 + lane;
        int N = len[u];
        if (N < 0 || N > p.len_cap) {
            if (cta0)
                report_error(p.ws, N < 0 ? kErrNegLen : kErrTooLong, i, N, p.len_cap);
            N = N < 0 ? 0 : p.len_cap;
        }
        len[u] = N;
        const int f = N / p.C, r = (N % p.C) != 0 ? 1 : 0;
        const int cls = r ? plan_short_class(N % p.C, p.C) : -1;
#pragma unroll
        for (int c = 0; c < kShortClasses; ++c)
            in_class[c] += __popc(__ballot_sync(0xffffffffu, cls == c));
        long long xf = f, xr = r;  // inclusive warp scans
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long yf = __shfl_up_sync(0xffffffffu, xf, o);
            const long long yr = __shfl_up_sync(0xffffffffu, xr, o);
            if (lane >= o) {
                xf += yf;
                xr += yr;
            }
        }
        const long long ef = cf + xf - f, er = cr + xr - r;
        if (i < p.B) {  // after an overflow F and R go unused
            F[i] = (int)ef;
            R[i] = (int)er;
            if (cta0) {
                p.plan_offsets[i] = (int)(ef + er);
                p.plan_short_before[i] = (int)er;
            }
        }
        cf += __shfl_sync(0xffffffffu, xf, 31);
        cr += __shfl_sync(0xffffffffu, xr, 31);
    }
    // S: the longest class first; within a class, rows in order
    int next[kShortClasses];
    int acc = 0;
#pragma unroll
    for (int c = kShortClasses - 1; c >= 0; --c) {
        next[c] = acc;
        acc += in_class[c];
    }
    const unsigned below = (1u << lane) - 1u;
#pragma unroll
    for (int u = 0; u < kRounds; ++u) {
        if (u * 32 >= p.B)
            break;
        const int N = len[u];  // clamped above; 0 past the last row
        const int cls = (N % p.C) != 0 ? plan_short_class(N % p.C, p.C) : -1;
#pragma unroll
        for (int c = 0; c < kShortClasses; ++c) {
            const unsigned m = __ballot_sync(0xffffffffu, cls == c);
            if (cls == c)
                S[next[c] + __popc(m & below)] = (int16_t)(u * 32 + lane);
            next[c] += __popc(m);
        }
    }
    const long long T = (cf + cr) * p.Hkv;
    const bool over = T > p.n_tasks;  // the capacity, at most INT32_MAX: F and R fit in int
    if (lane == 0) {
        F[p.B] = (int)cf;
        R[p.B] = (int)cr;
        if (cta0) {
            p.plan_offsets[p.B] = (int)(cf + cr);
            p.ws->task_count = over ? 0 : (int)T;
            p.ws->state_rows = (int)(cf + cr);
            p.ws->overflow = over ? 1 : 0;
            if (over)
                report_error(p.ws, kErrCapacity, (int)(T > 0x7fffffffLL ? 0x7fffffffLL : T), p.n_tasks, 0);
        }
    }
    __syncwarp();
    return over ? 0 : (int)T;
}

// Named barrier between the planning producer warp (arrives) and the
// consumer warps (wait), so that only the consumers wait for the plan.
constexpr int kPlanBarrier = 1;

__device__ __forceinline__ void plan_barrier_arrive()
{
    asm volatile("bar.arrive %0, %1;" ::"n"(kPlanBarrier), "n"(kThreads) : "memory");
}

__device__ __forceinline__ void plan_barrier_sync()
{
    asm volatile("bar.sync %0, %1;" ::"n"(kPlanBarrier), "n"(kThreads) : "memory");
}

// Both task lists of the plan, written by the consumer warps of all CTAs
// (task t of the balance order goes to position t of the balanced list and
// to its lexicographic index in the canonical one) while the first tiles
// are in flight; nothing in this launch reads them back.
__device__ __forceinline__ void self_plan_write_tasks(const DecodeParams &p, const SelfPlan &sp, int ntasks)
{
    constexpr int kWriters = 32 * kCW;
    for (int64_t t = (int64_t)blockIdx.x * kWriters + threadIdx.x; t < ntasks; t += (int64_t)gridDim.x * kWriters) {
        int64_t lex;
        const int4 rec = plan_task_at((int)t, sp.F, sp.R, sp.S, p.B, p.Hkv, p.Hq, p.G, &lex);
        p.plan_ordered[t] = rec;
        p.plan_tasks[lex] = rec;
    }
}

template <int D, int MODE, bool FUSE>
__global__ void __launch_bounds__(kThreads, 2)
    decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const DecodeParams p)
{
    using L = Layout<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *basep = smem_raw + (sbase - raw);
    int4 *meta = reinterpret_cast<int4 *>(basep + L::kMetaOff);
    const uint32_t bar_full0 = sbase + L::kBarOff;
    const uint32_t bar_empty0 = bar_full0 + L::kStages * 8;
    const uint32_t bar_merge0 = bar_empty0 + L::kStages * 8;
    const int warp = threadIdx.x >> 5;
    __shared__ int s_ctl[2];  // [0]: a wait timed out in this CTA; [1]: fused merge may proceed
    // the self-planning workqueue's prefix sums F, R (the other instances keep one word)
    constexpr bool kSelf = MODE == kModeQueue && !FUSE;
    __shared__ int s_plan[kSelf ? 2 * (kSelfPlanMaxB + 1) + 1 : 1];  // + the task count
    __shared__ int16_t s_short_rows[kSelf ? kSelfPlanMaxB : 1];           // and S

    if (threadIdx.x == 0) {
        s_ctl[0] = s_ctl[1] = 0;
        for (int s = 0; s < L::kStages; ++s) {
            mbar_init(bar_full0 + s * 8, 1);
            mbar_init(bar_empty0 + s * 8, kCW);
            mbar_init(bar_merge0 + s * 8, (kCW - 1) * 32);
        }
        fence_mbar_init();
    }
    if (warp == kCW && (threadIdx.x & 31) == 0) {
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
    }
    __syncthreads();
    // consumer warp 0 warms L2 with the CTA's first tiles while the producer
    // waits for the previous kernel (and plans)
    if (warp == 0) {
        if constexpr (kSelf) {
            if (p.self_plan)
                prefetch_first_queue_tiles(&tmK, &tmV, p);
        } else {
            prefetch_first_tiles<D, MODE>(&tmK, &tmV, p);
        }
    }
    // everything above overlaps the previous kernel; nothing below runs before
    // it has finished and its writes are visible
    pdl_wait();
    pdl_trigger();
    SelfPlan sp{nullptr, nullptr, nullptr};
    int ntasks = p.n_tasks;
    if constexpr (kSelf) {
        if (p.self_plan) {
            sp = SelfPlan{s_plan, s_plan + kSelfPlanMaxB + 1, s_short_rows};
            int *s_count = s_plan + 2 * (kSelfPlanMaxB + 1);
            if (warp == kCW) {
                ntasks = self_plan_warp(p, s_plan, s_plan + kSelfPlanMaxB + 1, s_short_rows);
                if ((threadIdx.x & 31) == 0)
                    *s_count = ntasks;
                plan_barrier_arrive();
            } else {
                plan_barrier_sync();
                ntasks = *s_count;
            }
        } else {
            ntasks = min(p.ws->task_count, p.n_tasks);
        }
    } else if (MODE == kModeQueue) {
        ntasks = min(p.ws->task_count, p.n_tasks);
    }
    if (warp == kCW) {
        run_producer<D, MODE, FUSE>(&tmK, &tmV, p, ntasks, sbase, basep, meta, bar_full0, bar_empty0,
                                    s_ctl, sp);
    } else {
        if constexpr (kSelf)
            if (sp.F)
                self_plan_write_tasks(p, sp, ntasks);
        run_consumer<D, MODE, FUSE>(p, sbase, basep, meta, bar_full0, bar_empty0, bar_merge0, s_ctl);
    }
    if constexpr (FUSE)
        grid_merge<D, MODE>(p, basep, s_ctl);
}

template <int D, int MODE, bool FUSE>
cudaError_t launch_one(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p, int grid,
                       cudaStream_t s, bool pdl)
{
    static_assert(!FUSE || MODE != kModeSingle, "the single pass has no merge");
    auto kern = decode_kernel<D, MODE, FUSE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Layout<D>::kAlloc);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Layout<D>::kAlloc;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tk, tv, p);
}

template <int D>
cudaError_t occupancy(int *out)
{
    auto kern = decode_kernel<D, kModeQueue, true>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Layout<D>::kAlloc);
    if (e != cudaSuccess)
        return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, kern, kThreads, Layout<D>::kAlloc);
}

}  // namespace

int decode_smem_bytes(int d) { return d == 64 ? Layout<64>::kAlloc : Layout<128>::kAlloc; }

cudaError_t decode_ctas_per_sm(int d, int *out)
{
    return d == 64 ? occupancy<64>(out) : occupancy<128>(out);
}

template <int D>
cudaError_t launch_d(int mode, const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p,
                     int grid, cudaStream_t s, bool pdl)
{
    // the fused merge is a separate instance, so the split kernels without it
    // carry none of its code or registers
    if (mode == kModeRect)
        return p.fuse ? launch_one<D, kModeRect, true>(tk, tv, p, grid, s, pdl)
                      : launch_one<D, kModeRect, false>(tk, tv, p, grid, s, pdl);
    if (mode == kModeQueue)
        return p.fuse ? launch_one<D, kModeQueue, true>(tk, tv, p, grid, s, pdl)
                      : launch_one<D, kModeQueue, false>(tk, tv, p, grid, s, pdl);
    return launch_one<D, kModeSingle, false>(tk, tv, p, grid, s, pdl);
}

cudaError_t launch_decode(int d, int mode, const CUtensorMap &tk, const CUtensorMap &tv,
                          const DecodeParams &p, int grid, cudaStream_t s, bool pdl)
{
    return d == 128 ? launch_d<128>(mode, tk, tv, p, grid, s, pdl)
                    : launch_d<64>(mode, tk, tv, p, grid, s, pdl);
}

}  // namespace pkv
