// api.cu -- the C ABI of libpkv (declared in include/pkv.h): argument
// validation, TMA descriptor encoding, kernel launches on the caller's stream,
// launch counters, the calibrated path policy and error reporting.
#include "pkv.h"
#include "pkv_device.cuh"
#include "pkv_kernels.h"
#include "plan_map.cuh"

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <cudaTypedefs.h>
#include <mutex>
#include <string>

using namespace pkv;

namespace {

thread_local std::string g_err;

int fail(int code, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char *what)
{
    return fail(PKV_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

struct Counters {
    std::atomic<int64_t> plan{0}, decode{0}, merge{0}, single{0}, append{0};
} g_cnt;

std::atomic<int32_t> g_starve{0};  // decode launches left to run with the test hook

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
int ilog2(int x)
{
    int l = 0;
    while ((1 << l) < x)
        ++l;
    return l;
}
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(const pkv_shape_t *s)
{
    if (!s)
        return fail(PKV_EINVAL, "shape is NULL");
    if (s->B < 0 || s->Hq <= 0 || s->Hkv <= 0 || s->d <= 0 || s->page_size <= 0 ||
        s->num_pages <= 0 || s->bt_stride <= 0)
        return fail(PKV_EINVAL, "shape has a non-positive field (B=%d Hq=%d Hkv=%d d=%d P=%d "
                                "num_pages=%d bt_stride=%d)",
                    s->B, s->Hq, s->Hkv, s->d, s->page_size, s->num_pages, s->bt_stride);
    if (s->Hq % s->Hkv)
        return fail(PKV_EINVAL, "Hq=%d is not a multiple of Hkv=%d", s->Hq, s->Hkv);
    if (!std::isfinite(s->scale))
        return fail(PKV_EINVAL, "scale is not finite");
    if (s->d != 64 && s->d != 128)
        return fail(PKV_EUNSUPPORTED, "head dim d=%d (supported: 64, 128)", s->d);
    if (s->Hq / s->Hkv > 8)
        return fail(PKV_EUNSUPPORTED, "G=Hq/Hkv=%d (supported: 1..8)", s->Hq / s->Hkv);
    if (!is_pow2(s->page_size) || s->page_size < 8 || s->page_size > 256)
        return fail(PKV_EUNSUPPORTED, "page_size=%d (supported: powers of two in [8, 256])",
                    s->page_size);
    if ((int64_t)s->bt_stride * s->page_size > 0x7fffffffLL)
        return fail(PKV_EINVAL, "bt_stride*page_size overflows int32");
    return PKV_OK;
}

int check_cfg(const pkv_shape_t *s, const pkv_plan_cfg_t *c)
{
    if (!c)
        return fail(PKV_EINVAL, "plan cfg is NULL");
    if (c->path != PKV_PATH_BUCKETED_SPLIT && c->path != PKV_PATH_WORKQUEUE &&
        c->path != PKV_PATH_SINGLE_PASS)
        return fail(PKV_EINVAL, "unknown path %d", (int)c->path);
    if (c->path == PKV_PATH_SINGLE_PASS)
        return PKV_OK;
    if (c->split_tokens <= 0 || c->split_tokens % s->page_size)
        return fail(PKV_EINVAL, "split_tokens=%d must be a positive multiple of page_size=%d",
                    c->split_tokens, s->page_size);
    if (c->bucket_len < 0 || c->max_tasks < 0)
        return fail(PKV_EINVAL, "negative bucket_len or max_tasks");
    if (c->merge != PKV_MERGE_SEPARATE && c->merge != PKV_MERGE_FUSED)
        return fail(PKV_EINVAL, "unknown merge mode %d", (int)c->merge);
    if (c->plan != PKV_PLAN_SEPARATE && c->plan != PKV_PLAN_IN_DECODE)
        return fail(PKV_EINVAL, "unknown plan mode %d", (int)c->plan);
    return PKV_OK;
}

static_assert(pkv::kSelfPlanMaxB == PKV_SELF_PLAN_MAX_B, "one row limit for the self-planning decode");

// The workqueue decode of this shape and cfg builds its own plan.
bool self_plans(const pkv_shape_t *s, const pkv_plan_cfg_t *c)
{
    return c->path == PKV_PATH_WORKQUEUE && c->plan == PKV_PLAN_IN_DECODE && s->B <= kSelfPlanMaxB;
}

WsHeader *ws_hdr(void *ws) { return reinterpret_cast<WsHeader *>(ws); }

// pkv_append_plan leaves the plan to the decode that follows it: that decode
// plans for itself (the fused merge's decode reads a plan built before it).
bool append_defers_plan(const pkv_shape_t *s, const pkv_plan_cfg_t *c)
{
    return self_plans(s, c) && c->merge == PKV_MERGE_SEPARATE;
}

AppendParams append_params(const pkv_shape_t *s, void *d_ws, const void *k_new, const void *v_new,
                           int32_t *bt, int32_t *sl, void *k_cache, void *v_cache)
{
    AppendParams p = {};
    p.k_new = static_cast<const __half *>(k_new);
    p.v_new = static_cast<const __half *>(v_new);
    p.bt = bt;
    p.seq_lens = sl;
    p.k_cache = static_cast<__half *>(k_cache);
    p.v_cache = static_cast<__half *>(v_cache);
    p.ws = ws_hdr(d_ws);
    p.B = s->B;
    p.Hkv = s->Hkv;
    p.d = s->d;
    p.log2P = ilog2(s->page_size);
    p.num_pages = s->num_pages;
    p.bt_stride = s->bt_stride;
    return p;
}

int len_cap(const pkv_shape_t *s) { return s->bt_stride * s->page_size; }

int s_b(const pkv_shape_t *s, const pkv_plan_cfg_t *c)
{
    const int64_t bl = c->bucket_len > 0 ? c->bucket_len : len_cap(s);
    return (int)((bl + c->split_tokens - 1) / c->split_tokens);
}

int64_t max_tasks(const pkv_shape_t *s, const pkv_plan_cfg_t *c)
{
    if (c->max_tasks > 0)
        return c->max_tasks;
    const int64_t per_row = ((int64_t)len_cap(s) + c->split_tokens - 1) / c->split_tokens;
    return (int64_t)s->Hkv * s->B * per_row;
}

int64_t partial_slots(const pkv_shape_t *s, const pkv_plan_cfg_t *c, int64_t rows = -1)
{
    if (c->path == PKV_PATH_BUCKETED_SPLIT)
        return (rows >= 0 ? rows : (int64_t)s->B) * s_b(s, c) * s->Hq;
    if (c->path == PKV_PATH_WORKQUEUE)
        return max_tasks(s, c) * (s->Hq / s->Hkv);
    return 0;
}

int check_ptr(const void *p, const char *name, bool nullable = false)
{
    if (!p)
        return nullable ? PKV_OK : fail(PKV_EINVAL, "%s is NULL", name);
    if (!aligned16(p))
        return fail(PKV_EINVAL, "%s is not 16-byte aligned", name);
    return PKV_OK;
}

#define PKV_TRY(x)               \
    do {                         \
        int rc_ = (x);           \
        if (rc_ != PKV_OK)       \
            return rc_;          \
    } while (0)

// ---------------------------------------------------------------- devices

struct DevInfo {
    int sms = 0;
    int ctas_per_sm[2] = {0, 0};  // decode CTAs an SM holds, d = 64 / 128
};
std::mutex g_dev_mu;
DevInfo g_dev[64];

// Resident decode CTAs the current device holds at once (SMs x occupancy).
int device_slots(int d, int *out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64)
        return fail(PKV_EUNSUPPORTED, "device ordinal %d", dev);
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DevInfo &di = g_dev[dev];
    if (!di.sms) {
        e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
    }
    int &occ = di.ctas_per_sm[d == 128 ? 1 : 0];
    if (!occ) {
        e = decode_ctas_per_sm(d, &occ);
        if (e != cudaSuccess)
            return cuda_fail(e, "occupancy query");
        if (occ < 1)
            return fail(PKV_ECUDA, "decode kernel does not fit on an SM");
    }
    *out = di.sms * occ;
    return PKV_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

int encode_kv_map(CUtensorMap *m, const void *base, const pkv_shape_t *s, int box_tok)
{
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!g_encode)
        return fail(PKV_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");
    // Pages viewed as a 5-D tensor (innermost first):
    //   d low (64 halves, 128 B) | slot (P) | d high (d/64) | kv head | page
    // so one box {64, box_tok, d/64, 1, 1} is box_tok tokens x all d columns of
    // one KV head of one page, landing as [d high][token][128 B] rows that the
    // 128-byte swizzle spreads over all shared-memory banks.
    const cuuint64_t es = 2;
    cuuint64_t dims[5] = {64, (cuuint64_t)s->page_size, (cuuint64_t)(s->d / 64), (cuuint64_t)s->Hkv,
                          (cuuint64_t)s->num_pages};
    cuuint64_t strides[4] = {(cuuint64_t)s->Hkv * s->d * es, 128, (cuuint64_t)s->d * es,
                             (cuuint64_t)s->page_size * s->Hkv * s->d * es};
    cuuint32_t box[5] = {64, (cuuint32_t)box_tok, (cuuint32_t)(s->d / 64), 1, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 5, const_cast<void *>(base), dims, strides,
                          box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PKV_ECUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return PKV_OK;
}

// State slots are int32 in the task records and the kernels: a split path
// whose partial-state buffer would hold more is refused before any launch.
int check_slots(const pkv_shape_t *s, const pkv_plan_cfg_t *c, int64_t rows = -1)
{
    const int64_t slots = partial_slots(s, c, rows);
    if (slots > 0x7fffffffLL)
        return fail(PKV_EUNSUPPORTED, "%lld partial-state slots exceed int32 (lower max_tasks, "
                    "bucket_len or B)", (long long)slots);
    return PKV_OK;
}

int run_decode(const pkv_shape_t *s, int mode, const pkv_plan_cfg_t *c, void *d_ws, const void *q,
               const void *k, const void *v, const int32_t *bt, const int32_t *sl, float *part,
               void *o, float *lse, cudaStream_t st, const int32_t *rows = nullptr,
               int n_rows = -1, bool fuse = false)
{
    if (mode != kModeSingle)
        PKV_TRY(check_slots(s, c, rows ? n_rows : -1));
    int slots = 0;
    PKV_TRY(device_slots(s->d, &slots));
    const int box_tok = s->page_size < 64 ? s->page_size : 64;
    alignas(64) CUtensorMap tk, tv;
    PKV_TRY(encode_kv_map(&tk, k, s, box_tok));
    PKV_TRY(encode_kv_map(&tv, v, s, box_tok));
    DecodeParams p = {};
    p.q = static_cast<const __half *>(q);
    p.bt = bt;
    p.seq_lens = sl;
    p.ws = ws_hdr(d_ws);
    p.B = s->B;
    p.Hq = s->Hq;
    p.Hkv = s->Hkv;
    p.G = s->Hq / s->Hkv;
    p.num_pages = s->num_pages;
    p.bt_stride = s->bt_stride;
    p.log2P = ilog2(s->page_size);
    p.box_log2 = ilog2(box_tok);
    p.len_cap = len_cap(s);
    p.scale_log2 = s->scale * 1.4426950408889634f;
    for (int32_t n = g_starve.load(); n > 0;)
        if (g_starve.compare_exchange_weak(n, n - 1)) {
            p.starve_first_stage = 1;
            break;
        }
    int64_t ntasks = 0;
    if (mode == kModeSingle) {
        p.o = static_cast<__half *>(o);
        p.lse = lse;
        ntasks = (int64_t)s->B * s->Hkv;
    } else {
        const int64_t slots = partial_slots(s, c, rows ? n_rows : -1);
        p.part_acc = part;
        p.part_m = part + slots * s->d;
        p.part_l = p.part_m + slots;
        p.C = c->split_tokens;
        p.S_b = s_b(s, c);
        if (mode == kModeRect) {
            p.rows = rows;
            ntasks = (int64_t)(rows ? n_rows : s->B) * s->Hkv * p.S_b;
        } else {
            ntasks = max_tasks(s, c);
            char *w = static_cast<char *>(d_ws);
            p.tasks = reinterpret_cast<const int4 *>(w + ws_ordered_off(s->B, ntasks));
            if (!fuse && self_plans(s, c)) {
                p.self_plan = 1;
                p.plan_offsets = reinterpret_cast<int32_t *>(w + ws_offsets_off());
                p.plan_short_before = reinterpret_cast<int32_t *>(w + ws_short_off(s->B, ntasks));
                p.plan_tasks = reinterpret_cast<int4 *>(w + ws_tasks_off(s->B));
                p.plan_ordered = reinterpret_cast<int4 *>(w + ws_ordered_off(s->B, ntasks));
            }
        }
        if (fuse) {
            p.fuse = 1;
            p.o = static_cast<__half *>(o);
            p.lse = lse;
            p.offsets = reinterpret_cast<const int32_t *>(static_cast<char *>(d_ws) + ws_offsets_off());
            p.n_rows = rows ? n_rows : s->B;
        }
    }
    if (ntasks > 0x7fffffffLL)
        return fail(PKV_EUNSUPPORTED, "%lld tasks exceed int32", (long long)ntasks);
    p.n_tasks = (int)ntasks;
    const int grid = (int)(ntasks < slots ? (ntasks > 0 ? ntasks : 1) : slots);
    cudaError_t e = launch_decode(s->d, mode, tk, tv, p, grid, st, true);
    if (e != cudaSuccess)
        return cuda_fail(e, "decode launch");
    (mode == kModeSingle ? g_cnt.single : g_cnt.decode)++;
    return PKV_OK;
}

}  // namespace

int pkv::record_error(int code, const char *msg) { return fail(code, "%s", msg); }

extern "C" {

size_t pkv_plan_workspace_size(const pkv_shape_t *s, const pkv_plan_cfg_t *c)
{
    if (check_shape(s) || check_cfg(s, c))
        return 0;
    if (c->path != PKV_PATH_WORKQUEUE)
        return ws_tasks_off(s->B);
    return ws_short_off(s->B, max_tasks(s, c)) + sizeof(int32_t) * (size_t)s->B;
}

size_t pkv_partials_size(const pkv_shape_t *s, const pkv_plan_cfg_t *c)
{
    if (check_shape(s) || check_cfg(s, c))
        return 0;
    return (size_t)partial_slots(s, c) * (size_t)(s->d + 2) * sizeof(float);
}

}  // extern "C"

namespace {

PlanParams plan_params(const pkv_shape_t *s, const pkv_plan_cfg_t *c, const int32_t *d_seq_lens,
                       void *d_ws)
{
    PlanParams p = {};
    p.seq_lens = d_seq_lens;
    p.ws = ws_hdr(d_ws);
    p.offsets = reinterpret_cast<int32_t *>(static_cast<char *>(d_ws) + ws_offsets_off());
    const int64_t cap = max_tasks(s, c);
    p.tasks = reinterpret_cast<int4 *>(static_cast<char *>(d_ws) + ws_tasks_off(s->B));
    p.tasks_ordered = reinterpret_cast<int4 *>(static_cast<char *>(d_ws) + ws_ordered_off(s->B, cap));
    p.short_before = reinterpret_cast<int32_t *>(static_cast<char *>(d_ws) + ws_short_off(s->B, cap));
    p.B = s->B;
    p.Hq = s->Hq;
    p.Hkv = s->Hkv;
    p.G = s->Hq / s->Hkv;
    p.C = c->split_tokens;
    p.len_cap = len_cap(s);
    p.max_tasks = cap;
    return p;
}

}  // namespace

extern "C" {

int pkv_plan(const pkv_shape_t *s, const pkv_plan_cfg_t *c, const int32_t *d_seq_lens, void *d_ws,
             void *stream)
{
    PKV_TRY(check_shape(s));
    PKV_TRY(check_cfg(s, c));
    if (s->B == 0)
        return PKV_OK;  // an empty batch: nothing to do
    if (c->path != PKV_PATH_WORKQUEUE)
        return PKV_OK;
    PKV_TRY(check_slots(s, c));
    PKV_TRY(check_ptr(d_seq_lens, "seq_lens"));
    PKV_TRY(check_ptr(d_ws, "workspace"));
    const PlanParams p = plan_params(s, c, d_seq_lens, d_ws);
    cudaError_t e = launch_plan(p, static_cast<cudaStream_t>(stream), true);
    if (e != cudaSuccess)
        return cuda_fail(e, "plan launch");
    g_cnt.plan++;
    return PKV_OK;
}

int pkv_append_plan(const pkv_shape_t *s, const pkv_plan_cfg_t *c, void *d_ws, const void *k_new,
                    const void *v_new, int32_t *bt, int32_t *sl, const int32_t *free_pages,
                    int32_t *free_count, void *k_cache, void *v_cache, void *stream)
{
    PKV_TRY(check_shape(s));
    PKV_TRY(check_cfg(s, c));
    if (s->B == 0)
        return PKV_OK;  // an empty batch: nothing to do
    if (c->path != PKV_PATH_WORKQUEUE)
        return fail(PKV_EINVAL, "pkv_append_plan builds the WORKQUEUE plan");
    PKV_TRY(check_slots(s, c));
    PKV_TRY(check_ptr(d_ws, "workspace"));
    PKV_TRY(check_ptr(k_new, "k_new"));
    PKV_TRY(check_ptr(v_new, "v_new"));
    PKV_TRY(check_ptr(bt, "block_table"));
    PKV_TRY(check_ptr(sl, "seq_lens"));
    PKV_TRY(check_ptr(k_cache, "k_cache"));
    PKV_TRY(check_ptr(v_cache, "v_cache"));
    if ((free_pages == nullptr) != (free_count == nullptr))
        return fail(PKV_EINVAL, "free_pages and free_count go together");
    if (free_pages) {
        PKV_TRY(check_ptr(free_pages, "free_pages"));
        if (reinterpret_cast<uintptr_t>(free_count) & 3u)
            return fail(PKV_EINVAL, "free_count is not 4-byte aligned");
    }
    if (append_defers_plan(s, c)) {
        // append (and allocate) only: the decode that follows builds the plan
        AppendParams a = append_params(s, d_ws, k_new, v_new, bt, sl, k_cache, v_cache);
        a.free_pages = free_pages;
        a.free_count = free_count;
        cudaError_t e = launch_append(a, static_cast<cudaStream_t>(stream), true);
        if (e != cudaSuccess)
            return cuda_fail(e, "append launch");
        g_cnt.append++;
        return PKV_OK;
    }
    PlanParams p = plan_params(s, c, sl, d_ws);
    p.k_new = static_cast<const __half *>(k_new);
    p.v_new = static_cast<const __half *>(v_new);
    p.k_cache = static_cast<__half *>(k_cache);
    p.v_cache = static_cast<__half *>(v_cache);
    p.bt = bt;
    p.seq_lens_rw = sl;
    p.free_pages = free_pages;
    p.free_count = free_count;
    p.d = s->d;
    p.log2P = ilog2(s->page_size);
    p.num_pages = s->num_pages;
    p.bt_stride = s->bt_stride;
    cudaError_t e = launch_plan(p, static_cast<cudaStream_t>(stream), true);
    if (e != cudaSuccess)
        return cuda_fail(e, "plan launch");
    g_cnt.plan++;
    return PKV_OK;
}

int pkv_decode(const pkv_shape_t *s, const pkv_plan_cfg_t *c, void *d_ws, const void *q, const void *k,
               const void *v, const int32_t *bt, const int32_t *sl, float *part, void *stream)
{
    PKV_TRY(check_shape(s));
    PKV_TRY(check_cfg(s, c));
    if (s->B == 0)
        return PKV_OK;  // an empty batch: nothing to do
    if (c->path == PKV_PATH_SINGLE_PASS)
        return fail(PKV_EINVAL, "pkv_decode takes a split path; use pkv_single_pass");
    PKV_TRY(check_ptr(d_ws, "workspace"));
    PKV_TRY(check_ptr(q, "q"));
    PKV_TRY(check_ptr(k, "k_cache"));
    PKV_TRY(check_ptr(v, "v_cache"));
    PKV_TRY(check_ptr(bt, "block_table"));
    PKV_TRY(check_ptr(sl, "seq_lens"));
    PKV_TRY(check_ptr(part, "partials"));
    const int mode = c->path == PKV_PATH_WORKQUEUE ? kModeQueue : kModeRect;
    return run_decode(s, mode, c, d_ws, q, k, v, bt, sl, part, nullptr, nullptr,
                      static_cast<cudaStream_t>(stream));
}

int pkv_decode_merge(const pkv_shape_t *s, const pkv_plan_cfg_t *c, void *d_ws, const void *q,
                     const void *k, const void *v, const int32_t *bt, const int32_t *sl, float *part,
                     void *o, float *lse, void *stream)
{
    PKV_TRY(check_shape(s));
    PKV_TRY(check_cfg(s, c));
    if (s->B == 0)
        return PKV_OK;  // an empty batch: nothing to do
    if (c->path == PKV_PATH_SINGLE_PASS)
        return fail(PKV_EINVAL, "pkv_decode_merge takes a split path; use pkv_single_pass");
    PKV_TRY(check_ptr(d_ws, "workspace"));
    PKV_TRY(check_ptr(q, "q"));
    PKV_TRY(check_ptr(k, "k_cache"));
    PKV_TRY(check_ptr(v, "v_cache"));
    PKV_TRY(check_ptr(bt, "block_table"));
    PKV_TRY(check_ptr(sl, "seq_lens"));
    PKV_TRY(check_ptr(part, "partials"));
    PKV_TRY(check_ptr(o, "o"));
    PKV_TRY(check_ptr(lse, "lse", true));
    const int mode = c->path == PKV_PATH_WORKQUEUE ? kModeQueue : kModeRect;
    return run_decode(s, mode, c, d_ws, q, k, v, bt, sl, part, o, lse,
                      static_cast<cudaStream_t>(stream), nullptr, -1, true);
}

}  // extern "C"

namespace {

// (row, head) pairs from which the merge gives each pair one warp instead of
// a four-warp CTA.
constexpr int64_t kMergeRowCtaPairs = 2048;

int run_merge(const pkv_shape_t *s, const pkv_plan_cfg_t *c, void *d_ws, const int32_t *sl,
              const float *part, void *o, float *lse, void *stream, const int32_t *rows,
              int n_rows)
{
    PKV_TRY(check_slots(s, c, rows ? n_rows : -1));
    const int64_t slots = partial_slots(s, c, rows ? n_rows : -1);
    MergeParams p = {};
    p.rows = rows;
    p.n_rows = rows ? n_rows : s->B;
    p.seq_lens = sl;
    p.ws = ws_hdr(d_ws);
    p.offsets = reinterpret_cast<const int32_t *>(static_cast<char *>(d_ws) + ws_offsets_off());
    p.part_acc = part;
    p.part_m = part + slots * s->d;
    p.part_l = p.part_m + slots;
    p.o = static_cast<__half *>(o);
    p.lse = lse;
    p.B = s->B;
    p.Hq = s->Hq;
    p.C = c->split_tokens;
    p.S_b = s_b(s, c);
    p.mode = c->path == PKV_PATH_WORKQUEUE ? kModeQueue : kModeRect;
    p.len_cap = len_cap(s);
    p.state_rows_cap = slots / s->Hq;
    // many (row, head) pairs: one warp each, all resident in one wave
    p.row_cta = (int64_t)p.n_rows * s->Hq >= kMergeRowCtaPairs ? 1 : 0;
    cudaError_t e = launch_merge(s->d, p, static_cast<cudaStream_t>(stream), true);
    if (e != cudaSuccess)
        return cuda_fail(e, "merge launch");
    g_cnt.merge++;
    return PKV_OK;
}

}  // namespace

extern "C" {

int pkv_merge(const pkv_shape_t *s, const pkv_plan_cfg_t *c, void *d_ws, const int32_t *sl,
              const float *part, void *o, float *lse, void *stream)
{
    PKV_TRY(check_shape(s));
    PKV_TRY(check_cfg(s, c));
    if (s->B == 0)
        return PKV_OK;  // an empty batch: nothing to do
    if (c->path == PKV_PATH_SINGLE_PASS)
        return fail(PKV_EINVAL, "pkv_merge takes a split path");
    PKV_TRY(check_ptr(d_ws, "workspace"));
    PKV_TRY(check_ptr(sl, "seq_lens"));
    PKV_TRY(check_ptr(part, "partials"));
    PKV_TRY(check_ptr(o, "o"));
    PKV_TRY(check_ptr(lse, "lse", true));
    return run_merge(s, c, d_ws, sl, part, o, lse, stream, nullptr, -1);
}

int pkv_decode_step_rows(const pkv_shape_t *s, const pkv_plan_cfg_t *c, void *d_ws,
                         const int32_t *d_rows, int32_t n_rows, const void *q, const void *k,
                         const void *v, const int32_t *bt, const int32_t *sl, float *part, void *o,
                         float *lse, void *stream)
{
    PKV_TRY(check_shape(s));
    PKV_TRY(check_cfg(s, c));
    if (s->B == 0)
        return PKV_OK;  // an empty batch: nothing to do
    if (c->path != PKV_PATH_BUCKETED_SPLIT)
        return fail(PKV_EINVAL, "pkv_decode_step_rows runs the BUCKETED_SPLIT path");
    if (n_rows < 1 || n_rows > s->B)
        return fail(PKV_EINVAL, "n_rows=%d must be in [1, B=%d]", n_rows, s->B);
    PKV_TRY(check_ptr(d_rows, "rows"));
    PKV_TRY(check_ptr(d_ws, "workspace"));
    PKV_TRY(check_ptr(q, "q"));
    PKV_TRY(check_ptr(k, "k_cache"));
    PKV_TRY(check_ptr(v, "v_cache"));
    PKV_TRY(check_ptr(bt, "block_table"));
    PKV_TRY(check_ptr(sl, "seq_lens"));
    PKV_TRY(check_ptr(part, "partials"));
    PKV_TRY(check_ptr(o, "o"));
    PKV_TRY(check_ptr(lse, "lse", true));
    if (c->merge == PKV_MERGE_FUSED)
        return run_decode(s, kModeRect, c, d_ws, q, k, v, bt, sl, part, o, lse,
                          static_cast<cudaStream_t>(stream), d_rows, n_rows, true);
    PKV_TRY(run_decode(s, kModeRect, c, d_ws, q, k, v, bt, sl, part, nullptr, nullptr,
                       static_cast<cudaStream_t>(stream), d_rows, n_rows));
    return run_merge(s, c, d_ws, sl, part, o, lse, stream, d_rows, n_rows);
}

int pkv_single_pass(const pkv_shape_t *s, void *d_ws, const void *q, const void *k, const void *v,
                    const int32_t *bt, const int32_t *sl, void *o, float *lse, void *stream)
{
    PKV_TRY(check_shape(s));
    if (s->B == 0)
        return PKV_OK;  // an empty batch: nothing to do
    PKV_TRY(check_ptr(d_ws, "workspace"));
    PKV_TRY(check_ptr(q, "q"));
    PKV_TRY(check_ptr(k, "k_cache"));
    PKV_TRY(check_ptr(v, "v_cache"));
    PKV_TRY(check_ptr(bt, "block_table"));
    PKV_TRY(check_ptr(sl, "seq_lens"));
    PKV_TRY(check_ptr(o, "o"));
    PKV_TRY(check_ptr(lse, "lse", true));
    return run_decode(s, kModeSingle, nullptr, d_ws, q, k, v, bt, sl, nullptr, o, lse,
                      static_cast<cudaStream_t>(stream));
}

int pkv_decode_step(const pkv_shape_t *s, const pkv_plan_cfg_t *c, void *d_ws, const void *q,
                    const void *k, const void *v, const int32_t *bt, const int32_t *sl, float *part,
                    void *o, float *lse, void *stream)
{
    PKV_TRY(check_shape(s));
    PKV_TRY(check_cfg(s, c));
    if (s->B == 0)
        return PKV_OK;  // an empty batch: nothing to do
    if (c->path == PKV_PATH_SINGLE_PASS)
        return pkv_single_pass(s, d_ws, q, k, v, bt, sl, o, lse, stream);
    PKV_TRY(check_ptr(o, "o"));
    PKV_TRY(check_ptr(lse, "lse", true));
    if (c->merge == PKV_MERGE_FUSED) {
        PKV_TRY(pkv_plan(s, c, sl, d_ws, stream));
        return pkv_decode_merge(s, c, d_ws, q, k, v, bt, sl, part, o, lse, stream);
    }
    if (!self_plans(s, c))
        PKV_TRY(pkv_plan(s, c, sl, d_ws, stream));
    PKV_TRY(pkv_decode(s, c, d_ws, q, k, v, bt, sl, part, stream));
    return pkv_merge(s, c, d_ws, sl, part, o, lse, stream);
}

namespace {

// The current device's address of a page-locked host buffer that kernels may
// read or write in place over the host link, or nullptr when `h` is pageable,
// not 16-byte aligned or not mapped for the device.
void *mapped_host(const void *h)
{
    if (!h || !aligned16(h))
        return nullptr;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, h) != cudaSuccess) {
        cudaGetLastError();  // an unknown pointer: not an error of this call
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

}  // namespace

int pkv_decode_step_host(const pkv_shape_t *s, const pkv_plan_cfg_t *c, void *d_ws, float *part,
                         const void *h_q, void *d_q, const int32_t *h_bt, int32_t *d_bt,
                         const int32_t *h_sl, int32_t *d_sl, const void *k, const void *v, void *d_o,
                         void *h_o, float *d_lse, float *h_lse, void *stream)
{
    PKV_TRY(check_shape(s));
    PKV_TRY(check_cfg(s, c));
    if (s->B == 0)
        return PKV_OK;  // an empty batch: nothing to do
    PKV_TRY(check_ptr(d_ws, "workspace"));
    PKV_TRY(check_ptr(d_q, "q"));
    PKV_TRY(check_ptr(k, "k_cache"));
    PKV_TRY(check_ptr(v, "v_cache"));
    PKV_TRY(check_ptr(d_bt, "block_table"));
    PKV_TRY(check_ptr(d_sl, "seq_lens"));
    PKV_TRY(check_ptr(d_o, "o"));
    PKV_TRY(check_ptr(d_lse, "lse", true));
    if (c->path != PKV_PATH_SINGLE_PASS)
        PKV_TRY(check_ptr(part, "partials"));
    if (!h_q || !h_o)
        return fail(PKV_EINVAL, "host q and o are required");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t qbytes = (size_t)s->B * s->Hq * s->d * 2;
    // page-locked inputs are read in place by the step's kernels, pageable ones
    // are copied into the device buffers first
    const void *q_in = mapped_host(h_q);
    const int32_t *bt_in = static_cast<const int32_t *>(h_bt ? mapped_host(h_bt) : nullptr);
    const int32_t *sl_in = static_cast<const int32_t *>(h_sl ? mapped_host(h_sl) : nullptr);
    cudaError_t e = cudaSuccess;
    if (!q_in) {
        e = cudaMemcpyAsync(d_q, h_q, qbytes, cudaMemcpyHostToDevice, st);
        q_in = d_q;
    }
    if (e == cudaSuccess && h_bt && !bt_in)
        e = cudaMemcpyAsync(d_bt, h_bt, (size_t)s->B * s->bt_stride * 4, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess && h_sl && !sl_in)
        e = cudaMemcpyAsync(d_sl, h_sl, (size_t)s->B * 4, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess)
        return cuda_fail(e, "host-to-device copy");
    if (!bt_in)
        bt_in = d_bt;
    if (!sl_in)
        sl_in = d_sl;
    // o / lse are written once: page-locked host buffers take them in place
    void *o_out = mapped_host(h_o);
    float *lse_out = static_cast<float *>(h_lse ? mapped_host(h_lse) : nullptr);
    const bool copy_o = o_out == nullptr, copy_lse = h_lse && d_lse && lse_out == nullptr;
    if (copy_o)
        o_out = d_o;
    if (!lse_out)
        lse_out = d_lse;
    PKV_TRY(pkv_decode_step(s, c, d_ws, q_in, k, v, bt_in, sl_in, part, o_out, lse_out, stream));
    e = cudaSuccess;
    if (copy_o)
        e = cudaMemcpyAsync(h_o, d_o, qbytes, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess && copy_lse)
        e = cudaMemcpyAsync(h_lse, d_lse, (size_t)s->B * s->Hq * 4, cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess)
        return cuda_fail(e, "device-to-host copy");
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaStreamSynchronize");
    return PKV_OK;
}

int pkv_append_decode_step_host(const pkv_shape_t *s, const pkv_plan_cfg_t *c, void *d_ws,
                                float *part, const void *h_q, void *d_q, const void *h_k_new,
                                const void *h_v_new, void *d_k_new, void *d_v_new, int32_t *d_bt,
                                int32_t *d_sl, const int32_t *free_pages, int32_t *free_count,
                                void *k, void *v, void *d_o, void *h_o, float *d_lse,
                                float *h_lse, void *stream)
{
    // every argument is checked here, so that a call that fails enqueues nothing
    PKV_TRY(check_shape(s));
    PKV_TRY(check_cfg(s, c));
    if (s->B == 0)
        return PKV_OK;  // an empty batch: nothing to do
    if (c->path != PKV_PATH_SINGLE_PASS)
        PKV_TRY(check_slots(s, c));
    PKV_TRY(check_ptr(d_ws, "workspace"));
    PKV_TRY(check_ptr(d_q, "q"));
    PKV_TRY(check_ptr(d_k_new, "k_new"));
    PKV_TRY(check_ptr(d_v_new, "v_new"));
    PKV_TRY(check_ptr(k, "k_cache"));
    PKV_TRY(check_ptr(v, "v_cache"));
    PKV_TRY(check_ptr(d_bt, "block_table"));
    PKV_TRY(check_ptr(d_sl, "seq_lens"));
    PKV_TRY(check_ptr(d_o, "o"));
    PKV_TRY(check_ptr(d_lse, "lse", true));
    if (c->path != PKV_PATH_SINGLE_PASS)
        PKV_TRY(check_ptr(part, "partials"));
    if ((free_pages == nullptr) != (free_count == nullptr))
        return fail(PKV_EINVAL, "free_pages and free_count go together");
    if (free_pages) {
        if (c->path != PKV_PATH_WORKQUEUE)
            return fail(PKV_EINVAL, "device page allocation comes with the WORKQUEUE path");
        PKV_TRY(check_ptr(free_pages, "free_pages"));
        if (reinterpret_cast<uintptr_t>(free_count) & 3u)
            return fail(PKV_EINVAL, "free_count is not 4-byte aligned");
    }
    if (!h_q || !h_k_new || !h_v_new || !h_o)
        return fail(PKV_EINVAL, "host q, k_new, v_new and o are required");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t qbytes = (size_t)s->B * s->Hq * s->d * 2;
    const size_t nbytes = (size_t)s->B * s->Hkv * s->d * 2;
    // page-locked host buffers are used in place by the step's kernels (q,
    // which every split of every kv head re-reads, mostly from L2), pageable
    // ones go through the device buffers
    const void *q_in = mapped_host(h_q);
    const void *kn = mapped_host(h_k_new), *vn = mapped_host(h_v_new);
    if (!kn || !vn)
        kn = vn = nullptr;
    void *o_out = mapped_host(h_o);
    float *lse_out = static_cast<float *>(h_lse ? mapped_host(h_lse) : nullptr);
    const bool copy_o = o_out == nullptr, copy_lse = h_lse && d_lse && lse_out == nullptr;
    if (copy_o)
        o_out = d_o;
    if (!lse_out)
        lse_out = d_lse;
    cudaError_t e = cudaSuccess;
    if (!q_in) {
        e = cudaMemcpyAsync(d_q, h_q, qbytes, cudaMemcpyHostToDevice, st);
        q_in = d_q;
    }
    if (e == cudaSuccess && !kn)
        e = cudaMemcpyAsync(d_k_new, h_k_new, nbytes, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess && !vn)
        e = cudaMemcpyAsync(d_v_new, h_v_new, nbytes, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess)
        return cuda_fail(e, "host-to-device copy");
    if (!kn) {
        kn = d_k_new;
        vn = d_v_new;
    }
    if (c->path == PKV_PATH_WORKQUEUE) {
        // the append launch allocates pages and, unless the decode plans, plans
        PKV_TRY(pkv_append_plan(s, c, d_ws, kn, vn, d_bt, d_sl, free_pages, free_count, k, v,
                                stream));
        // the decode then plans for itself, or reads the plan the append built
        if (c->merge == PKV_MERGE_FUSED) {
            PKV_TRY(pkv_decode_merge(s, c, d_ws, q_in, k, v, d_bt, d_sl, part, o_out, lse_out,
                                     stream));
        } else {
            PKV_TRY(pkv_decode(s, c, d_ws, q_in, k, v, d_bt, d_sl, part, stream));
            PKV_TRY(pkv_merge(s, c, d_ws, d_sl, part, o_out, lse_out, stream));
        }
    } else {
        PKV_TRY(pkv_append(s, d_ws, kn, vn, d_bt, d_sl, k, v, stream));
        PKV_TRY(pkv_decode_step(s, c, d_ws, q_in, k, v, d_bt, d_sl, part, o_out, lse_out, stream));
    }
    e = cudaSuccess;
    if (copy_o)
        e = cudaMemcpyAsync(h_o, d_o, qbytes, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess && copy_lse)
        e = cudaMemcpyAsync(h_lse, d_lse, (size_t)s->B * s->Hq * 4, cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess)
        return cuda_fail(e, "device-to-host copy");
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaStreamSynchronize");
    return PKV_OK;
}

int pkv_append(const pkv_shape_t *s, void *d_ws, const void *k_new, const void *v_new,
               const int32_t *bt, int32_t *sl, void *k_cache, void *v_cache, void *stream)
{
    PKV_TRY(check_shape(s));
    if (s->B == 0)
        return PKV_OK;  // an empty batch: nothing to do
    PKV_TRY(check_ptr(d_ws, "workspace"));
    PKV_TRY(check_ptr(k_new, "k_new"));
    PKV_TRY(check_ptr(v_new, "v_new"));
    PKV_TRY(check_ptr(bt, "block_table"));
    PKV_TRY(check_ptr(sl, "seq_lens"));
    PKV_TRY(check_ptr(k_cache, "k_cache"));
    PKV_TRY(check_ptr(v_cache, "v_cache"));
    // no free list: the kernel writes no block-table entry
    AppendParams p = append_params(s, d_ws, k_new, v_new, const_cast<int32_t *>(bt), sl, k_cache,
                                   v_cache);
    cudaError_t e = launch_append(p, static_cast<cudaStream_t>(stream), true);
    if (e != cudaSuccess)
        return cuda_fail(e, "append launch");
    g_cnt.append++;
    return PKV_OK;
}

// ------------------------------------------------------ exact-length groups

int pkv_exact_length_groups(const int32_t *seq_lens, int32_t B, int32_t *rows,
                            int32_t *group_start, int32_t *group_len, int32_t *n_groups)
{
    if (B < 0 || !n_groups)
        return fail(PKV_EINVAL, "pkv_exact_length_groups: negative B or NULL n_groups");
    if (B > 0 && (!seq_lens || !rows || !group_start || !group_len))
        return fail(PKV_EINVAL, "pkv_exact_length_groups: NULL array");
    // rows by (length, index): a counting pass would need the length range, so
    // sort the row indices (B is a batch: small) by a stable insertion order
    int32_t n = 0;
    for (int32_t i = 0; i < B; ++i) {
        if (seq_lens[i] < 0)
            return fail(PKV_EINVAL, "pkv_exact_length_groups: row %d has a negative length", i);
        if (seq_lens[i] == 0)
            continue;
        int32_t k = n++;
        while (k > 0 && seq_lens[rows[k - 1]] > seq_lens[i]) {
            rows[k] = rows[k - 1];
            --k;
        }
        rows[k] = i;
    }
    int32_t g = 0;
    for (int32_t k = 0; k < n; ++k) {
        if (k == 0 || seq_lens[rows[k]] != seq_lens[rows[k - 1]]) {
            group_start[g] = k;
            group_len[g] = seq_lens[rows[k]];
            ++g;
        }
    }
    group_start[g] = n;
    for (int32_t i = 0, k = n; i < B; ++i)  // the rows without tokens, after the groups
        if (seq_lens[i] == 0)
            rows[k++] = i;
    *n_groups = g;
    return PKV_OK;
}

// ------------------------------------------------------------------ policy

// Thresholds calibrated on a GB300 (152 SMs) by paged_kv_gqa_09_gb300/calibrate.py:
// 252 traces (bucketed, bimodal, uniform, Zipf; B 1..64; N_max 256..65536;
// Hq=32, Hkv=8, d=128, P=16) drawn with the calibration seed 20260622, timed as
// synchronized wall-clock per step (the workqueue with its plan built inside the
// decode); held-out seed 20260623 mean regret 1.028 (worst 1.22x).
void pkv_policy_default(pkv_policy_cfg_t *c)
{
    if (!c)
        return;
    c->bucketed_min_tokens = 1024;
    c->bucketed_max_batch = 4;
    c->workqueue_min_tokens = 2048;
    c->workqueue_min_batch = 1;
    c->split_tokens = 256;
    c->bucketed_split_tokens = 512;
    c->workqueue_max_split_tokens = 1024;
    c->workqueue_target_splits = 32;
    c->workqueue_min_long_splits = 8;
}

int pkv_policy(int32_t B, int32_t n_max, const pkv_policy_cfg_t *cfg, pkv_path_t *out_path,
               int32_t *out_split)
{
    if (!out_path || !out_split)
        return fail(PKV_EINVAL, "policy outputs are NULL");
    if (B < 0 || n_max < 0)
        return fail(PKV_EINVAL, "negative B or n_max");
    pkv_policy_cfg_t d;
    pkv_policy_default(&d);
    const pkv_policy_cfg_t *c = cfg ? cfg : &d;
    if (c->split_tokens <= 0 || c->bucketed_split_tokens <= 0 || c->workqueue_target_splits < 0 ||
        c->workqueue_min_long_splits < 0)
        return fail(PKV_EINVAL, "policy split sizes must be positive");
    pkv_path_t path = PKV_PATH_SINGLE_PASS;
    int32_t C = c->split_tokens;
    if (B >= 1 && B <= c->bucketed_max_batch && n_max >= c->bucketed_min_tokens) {
        path = PKV_PATH_BUCKETED_SPLIT;
        C = c->bucketed_split_tokens;
    } else if (B >= c->workqueue_min_batch && n_max >= c->workqueue_min_tokens) {
        path = PKV_PATH_WORKQUEUE;
        // fewer, longer splits for larger batches: every split writes a state
        while (c->workqueue_target_splits > 0 && C < c->workqueue_max_split_tokens &&
               (int64_t)B * ((n_max + (int64_t)C - 1) / C) > c->workqueue_target_splits &&
               (n_max + 2 * (int64_t)C - 1) / (2 * (int64_t)C) >= c->workqueue_min_long_splits)
            C *= 2;
    }
    *out_path = path;
    *out_split = C;
    return PKV_OK;
}

// ------------------------------------------------------------ learned model

// Routes and weights fitted by paged_kv_gqa_09_gb300/calibrate.py (least
// squares of log step time, calibration seed 20260622, 252 GB300 traces, the
// workqueue with its plan built inside the decode and its full splits claimed
// kv heads side by side); held-out seed 20260623 mean regret 1.028 (worst 1.27x).
static const pkv_cost_route_t kGb300Routes[] = {
    {0, 128, {6.32596585f, 0.161054287f, 0.0567319871f, -0.817394585f, -0.000291889516f, 0.00947691535f, 0.00720108639f, 0.278543951f, -0.0380039254f, 0.0323045397f}},
    {0, 256, {6.76135326f, 0.123543866f, 0.0806977112f, -0.874130438f, 0.00196533382f, 0.00523261849f, 0.00287883712f, 0.237565484f, -0.0550019129f, 0.0360926702f}},
    {0, 512, {6.92285841f, 0.0309477548f, 0.0682869668f, -0.84860889f, 0.00766998863f, 0.0044188007f, 0.00124586854f, 0.18332268f, -0.0487189545f, 0.0359124603f}},
    {0, 1024, {6.54865388f, -0.10686691f, 0.105374087f, -0.776884156f, 0.0154875338f, 0.00774054743f, -0.00151910083f, 0.116170665f, -0.0313161385f, 0.0333337912f}},
    {0, 2048, {5.55392319f, -0.180748252f, 0.278615937f, -0.747356823f, 0.0184875087f, 0.011382734f, -0.00797789108f, 0.054136097f, -0.00713310756f, 0.0314061685f}},
    {1, 256, {7.80428606f, 0.100382416f, 0.00343302636f, -0.906483809f, -0.00775595531f, 0.00188807613f, 0.00241907309f, -0.0205244659f, -0.00163554316f, 0.0405911339f}},
    {1, 512, {7.81364181f, 0.119356165f, 0.102866709f, -0.977378568f, -0.00810699919f, -0.000969304075f, -0.00273632032f, -0.00624230515f, -0.0159528335f, 0.0432357342f}},
    {1, 1024, {7.10032599f, 0.144580042f, 0.320125701f, -1.04372929f, -0.00945893095f, -0.00183146496f, -0.0113625829f, 0.00372923372f, -0.0141489341f, 0.0448997306f}},
    {1, 2048, {5.59301125f, 0.194205683f, 0.655522869f, -1.10398165f, -0.0133785116f, -0.000962689672f, -0.0234915754f, 0.0112598486f, -0.00844457495f, 0.0458395646f}},
    {1, 4096, {3.79049579f, 0.210621293f, 0.959115882f, -1.09954352f, -0.017013829f, 0.00504941651f, -0.0323231097f, -0.0105836929f, 0.0205952306f, 0.0434405961f}},
    {2, 1024, {5.19843729f, -0.169887795f, -0.194825525f, -0.369044046f, -0.00811396268f, 0.0392129519f, 0.0286692397f, -0.410672607f, 0.169898182f, 0.0128228085f}},
};

void pkv_cost_model_default(pkv_cost_model_t *m)
{
    if (!m)
        return;
    std::memset(m, 0, sizeof *m);
    m->n_routes = (int32_t)(sizeof kGb300Routes / sizeof kGb300Routes[0]);
    for (int r = 0; r < m->n_routes; ++r)
        m->route[r] = kGb300Routes[r];
}

int pkv_policy_learned(int32_t B, int32_t n_max, int64_t n_sum, const pkv_cost_model_t *model,
                       pkv_path_t *out_path, int32_t *out_split)
{
    if (!out_path || !out_split)
        return fail(PKV_EINVAL, "policy outputs are NULL");
    if (B < 0 || n_max < 0 || n_sum < 0)
        return fail(PKV_EINVAL, "negative B, n_max or n_sum");
    pkv_cost_model_t d;
    if (!model) {
        pkv_cost_model_default(&d);
        model = &d;
    }
    if (model->n_routes < 1 || model->n_routes > PKV_COST_MAX_ROUTES)
        return fail(PKV_EINVAL, "cost model has %d routes", model->n_routes);
    *out_path = PKV_PATH_SINGLE_PASS;
    *out_split = 1024;
    if (B == 0 || n_max == 0)
        return PKV_OK;
    const double lb = std::log2((double)B), ln = std::log2((double)n_max);
    const double ls = std::log2((double)(n_sum > 1 ? n_sum : 1));
    const double fill = (double)n_sum / ((double)B * (double)n_max);
    const double f[PKV_COST_FEATURES] = {1.0, lb, ln, ls, lb * ln, lb * lb, ln * ln, fill, fill * lb,
                                          ls * ls};
    double best = INFINITY;
    for (int r = 0; r < model->n_routes; ++r) {
        const pkv_cost_route_t &rt = model->route[r];
        if (rt.path < 0 || rt.path > 2 || (rt.path != 2 && rt.split_tokens <= 0))
            return fail(PKV_EINVAL, "cost model route %d is invalid", r);
        double t = 0.0;
        for (int k = 0; k < PKV_COST_FEATURES; ++k)
            t += (double)rt.w[k] * f[k];
        if (t < best) {
            best = t;
            *out_path = (pkv_path_t)rt.path;
            *out_split = rt.split_tokens;
        }
    }
    return PKV_OK;
}

// ---------------------------------------------------------------- counters

int pkv_get_counters(pkv_counters_t *out)
{
    if (!out)
        return fail(PKV_EINVAL, "counters output is NULL");
    out->plan_launches = g_cnt.plan.load();
    out->decode_launches = g_cnt.decode.load();
    out->merge_launches = g_cnt.merge.load();
    out->single_pass_launches = g_cnt.single.load();
    out->append_launches = g_cnt.append.load();
    return PKV_OK;
}

int pkv_reset_counters(void)
{
    g_cnt.plan = 0;
    g_cnt.decode = 0;
    g_cnt.merge = 0;
    g_cnt.single = 0;
    g_cnt.append = 0;
    return PKV_OK;
}

int pkv_step_model(int32_t path, const pkv_shape_t *s, int32_t C, int32_t bucket_len,
                   const int32_t *seq_lens, pkv_step_model_t *out)
{
    if (!s || !out || (s->B > 0 && !seq_lens))
        return fail(PKV_EINVAL, "NULL argument");
    if (s->B < 0 || s->Hq <= 0 || s->Hkv <= 0 || s->Hq % s->Hkv || s->d <= 0)
        return fail(PKV_EINVAL, "bad shape");
    if (path != 2 && C <= 0)
        return fail(PKV_EINVAL, "split_tokens must be positive");
    std::memset(out, 0, sizeof *out);
    int64_t rows = 0, toks = 0, n_max = 0;
    for (int i = 0; i < s->B; ++i) {
        const int64_t N = seq_lens[i] < 0 ? 0 : seq_lens[i];
        toks += N;
        if (path != 2)
            rows += (N + C - 1) / C;
        n_max = N > n_max ? N : n_max;
    }
    const int64_t state = (int64_t)(s->d + 2) * 4;
    out->kv_bytes = toks * s->Hkv * s->d * 4;
    if (path == PKV_PATH_BUCKETED_SPLIT) {
        const int64_t bl = bucket_len > 0 ? bucket_len : n_max;
        const int64_t sb = (bl + C - 1) / C;
        out->attn_launches = 2;
        out->tasks = rows * s->Hkv;
        out->grid_tasks = (int64_t)s->B * s->Hkv * sb;
        out->states_written = (int64_t)s->B * sb * s->Hq;
        out->states_read = rows * s->Hq;
    } else if (path == PKV_PATH_WORKQUEUE) {
        out->attn_launches = 2;
        out->plan_launches = 1;
        out->tasks = out->grid_tasks = rows * s->Hkv;
        out->states_written = out->states_read = rows * s->Hq;
    } else if (path == PKV_PATH_SINGLE_PASS) {
        out->attn_launches = 1;
        out->tasks = out->grid_tasks = (int64_t)s->B * s->Hkv;
    } else if (path == 3) {
        // exact-length buckets: one (split, merge) launch pair per distinct length
        int64_t groups = 0;
        for (int i = 0; i < s->B; ++i) {
            if (seq_lens[i] <= 0)
                continue;
            bool seen = false;
            for (int k = 0; k < i && !seen; ++k)
                seen = seq_lens[k] == seq_lens[i];
            groups += seen ? 0 : 1;
        }
        out->attn_launches = 2 * groups;
        out->tasks = out->grid_tasks = rows * s->Hkv;
        out->states_written = out->states_read = rows * s->Hq;
    } else {
        return fail(PKV_EINVAL, "unknown path %d", path);
    }
    out->merge_state_bytes = (out->states_written + out->states_read) * state;
    return PKV_OK;
}

// ------------------------------------------------------------------ errors

int pkv_get_error(void *d_ws, void *stream)
{
    PKV_TRY(check_ptr(d_ws, "workspace"));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaStreamSynchronize");
    WsHeader hd;
    e = cudaMemcpy(&hd, d_ws, sizeof hd, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMemcpy (error word)");
    const int32_t h[4] = {hd.err, hd.err_a, hd.err_b, hd.err_c};
    if (h[0] == kErrNone)
        return PKV_OK;
    e = cudaMemset(d_ws, 0, sizeof h);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMemset (error word)");
    switch (h[0]) {
    case kErrBadPage:
        return fail(PKV_EDEVICE, "block-table entry out of range: row %d, logical page %d, value %d",
                    h[1], h[2], h[3]);
    case kErrTooLong:
        return fail(PKV_EDEVICE, "row %d has length %d beyond its limit %d", h[1], h[2], h[3]);
    case kErrNegLen:
        return fail(PKV_EDEVICE, "row %d has negative length %d", h[1], h[2]);
    case kErrNoPage:
        return fail(PKV_EDEVICE, "no free page for row %d at length %d (%d pages were free)", h[1],
                    h[2], h[3]);
    case kErrBadRow:
        return fail(PKV_EDEVICE, "row list entry %d is %d, outside [0, %d)", h[1], h[2], h[3]);
    case kErrTimeout:
        return fail(PKV_ETIMEOUT, "a barrier wait timed out (CTA %d, stage %d, site %d)", h[1], h[2],
                    h[3]);
    case kErrCapacity:
        return fail(PKV_ECAPACITY, "workqueue needs %d tasks, capacity %d", h[1], h[2]);
    default:
        return fail(PKV_EDEVICE, "device error code %d", h[0]);
    }
}

int pkv_test_starve_next_decodes(int32_t n)
{
    // off unless the process opted in: a production caller cannot make its
    // decodes time out by accident
    const char *opt_in = std::getenv("PKV_TEST_HOOKS");
    if (!opt_in || std::strcmp(opt_in, "1") != 0)
        return fail(PKV_EUNSUPPORTED, "test hooks are off (set PKV_TEST_HOOKS=1 in the environment)");
    if (n < 0)
        return fail(PKV_EINVAL, "negative count");
    g_starve = n;
    return PKV_OK;
}

const char *pkv_last_error_string(void) { return g_err.c_str(); }

int pkv_version(void) { return PKV_VERSION; }

}  // extern "C"
