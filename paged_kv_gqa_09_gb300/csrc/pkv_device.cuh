// pkv_device.cuh -- device-side building blocks shared by the libpkv kernels:
// the workspace header, bounded mbarrier waits, TMA / bulk copies, warp-level
// tensor-core fragments (ldmatrix, movmatrix, mma.sync m16n8k16) and
// programmatic dependent launch.  Everything is inline PTX for sm_103a.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace pkv {

// ----------------------------------------------------------- workspace

// Device error codes recorded in WsHeader::err (first one wins).
enum DevErr : int32_t {
    kErrNone = 0,
    kErrBadPage = 1,   // block-table entry outside [0, num_pages): page read as zeros
    kErrTooLong = 2,   // N*_i beyond the block table or the bucket: tail dropped
    kErrTimeout = 3,   // a bounded barrier wait gave up
    kErrCapacity = 4,  // workqueue larger than max_tasks: nothing decoded
    kErrNegLen = 5,    // negative length: row treated as empty
    kErrBadRow = 6,    // a row list entry outside [0, B): that row skipped
    kErrNoPage = 7,    // the free list ran out: that row's token not appended
};

// First 64 bytes of the plan workspace.
struct WsHeader {
    int32_t err;          // DevErr of the first failure
    int32_t err_a, err_b, err_c;  // detail (row, value, limit)
    int32_t task_count;   // tasks written by the plan (0 after an overflow)
    int32_t state_rows;   // sum_i n_i
    int32_t overflow;     // 1 when the plan exceeded max_tasks
    // dynamic task claims of the workqueue decode: next balance-order index to
    // hand out (beyond the first round) and CTAs finished; the last CTA to
    // finish zeroes both for the next launch
    int32_t next_task;
    int32_t done_ctas;
    // grid-wide barrier of the fused merge: CTAs arrived, and a generation the
    // last arrival advances (the count is back at zero after every launch)
    int32_t bar_count;
    int32_t bar_gen;
    // CTAs of an allocating append that have read the lengths; the last one
    // zeroes it after advancing them
    int32_t append_done;
    int32_t pad[4];
};
static_assert(sizeof(WsHeader) == 64, "workspace header is 64 bytes");

__device__ __forceinline__ void report_error(WsHeader *ws, int32_t code, int32_t a, int32_t b,
                                             int32_t c)
{
    if (atomicCAS(&ws->err, 0, code) == 0) {
        ws->err_a = a;
        ws->err_b = b;
        ws->err_c = c;
    }
}

// ------------------------------------------------------------- misc PTX

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// 2^x (hardware approximation, relative error about 2^-22; 2^-inf = +0).
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// GPU-scope acquire load / release store of one int (grid-wide barrier words).
__device__ __forceinline__ int ld_acquire_gpu(const int *p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_gpu(int *p, int v)
{
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Programmatic dependent launch: wait for the preceding grid (and its memory),
// and allow the next grid in the stream to be scheduled early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Arrive `count` times at once (on behalf of several threads or warps).
__device__ __forceinline__ void mbar_arrive_n(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Raise the barrier's expected transaction bytes without arriving (the
// arrival follows separately, e.g. after the thread's own shared stores).
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete, giving up after
// limit_ns nanoseconds (returns false).  Every barrier wait in libpkv goes
// through here, so no kernel can spin forever.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > limit_ns)
            return false;
    }
    return true;
}

// ------------------------------------------------------------------ TMA

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *m)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// L2 policy for data read exactly once (the KV stream).
__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// L2 policy for data written now and read back soon (the split states the
// merge reads): kept ahead of the evict-first KV stream.
__device__ __forceinline__ uint64_t l2_evict_last_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Global store of one float with an L2 cache-eviction policy.
__device__ __forceinline__ void st_global_hint(float *p, float v, uint64_t policy)
{
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(policy) : "memory");
}

// 5-D tiled TMA load into shared memory, completing on `bar` (tx bytes).
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap *m, uint32_t bar,
                                            int c0, int c1, int c2, int c3, int c4,
                                            uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4, %5, %6, %7}], [%2], %8;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
        "r"(c4), "l"(policy)
        : "memory");
}

// Prefetch the same 5-D box into L2 (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_5d(const CUtensorMap *m, int c0, int c1, int c2, int c3,
                                                int c4)
{
    asm volatile("cp.async.bulk.prefetch.tensor.5d.L2.global.tile [%0, {%1, %2, %3, %4, %5}];" ::"l"(
                     reinterpret_cast<uint64_t>(m)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
                 : "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) writes to the same addresses.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------- warp tensor-core ops

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

// Transpose an 8x8 b16 matrix held one fragment per lane.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t a)
{
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

// D += A (16x16, row) * B (16x8, col); fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi)
{
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

}  // namespace pkv
