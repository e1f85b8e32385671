// noalloc.cu -- pkv_decode_step_noalloc: a whole decode step for callers that
// cannot allocate device memory.
//
// Who needs this: code that runs where cudaMalloc is off limits -- inside a
// custom allocator's own callbacks, in plugins of runtimes that own every
// device allocation and forbid others, or on paths that must not stall on the
// allocator's implicit synchronisation.  Such callers can still pass their
// inputs and outputs, but not the plan workspace and partial-state buffers the
// split paths need.
//
// The scratch lives in one file-scope device array of PKV_NOALLOC_SCRATCH_BYTES
// that every GPU loading this library holds until the process exits.  Host code
// must not pass the array's name to a kernel: on the host that name is only a
// stand-in, not a device address.  Its address is looked up once per device,
// with that device current, by cudaGetSymbolAddress on the first call made on
// that device.  With lazy module loading (CUDA's default) that lookup, and the
// first launch of each kernel, load code and the array onto the device: that
// first call is set-up, to be made where allocating is still allowed.
#include "pkv.h"
#include "pkv_kernels.h"

#include <cstdio>
#include <mutex>

#include <cuda_runtime.h>

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_addr[kMaxDevices];  // device address of g_noalloc_scratch per device

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Device address of the scratch array on the current device (set up once).
int scratch_address(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return pkv::record_error(PKV_ECUDA, "pkv_decode_step_noalloc: cudaGetDevice failed");
    if (dev < 0 || dev >= kMaxDevices)
        return pkv::record_error(PKV_EUNSUPPORTED, "pkv_decode_step_noalloc: device ordinal too large");
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return pkv::record_error(PKV_ECUDA,
                                     "pkv_decode_step_noalloc: cudaGetSymbolAddress failed");
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return PKV_OK;
}

}  // namespace

extern "C" int pkv_decode_step_noalloc(const pkv_shape_t *shape, const pkv_plan_cfg_t *cfg,
                                       const void *d_q, const void *d_k_cache,
                                       const void *d_v_cache, const int32_t *d_block_table,
                                       const int32_t *d_seq_lens, void *d_o, float *d_lse,
                                       void *stream)
{
    // sizes of this step's scratch; 0 means the shape or cfg is invalid, and
    // pkv_decode_step rejects it (with its reason) before touching any pointer
    const size_t ws = pkv_plan_workspace_size(shape, cfg);
    if (ws == 0)
        return pkv_decode_step(shape, cfg, nullptr, d_q, d_k_cache, d_v_cache, d_block_table,
                               d_seq_lens, nullptr, d_o, d_lse, stream);
    if (shape->B == 0)
        return PKV_OK;  // an empty batch: nothing to do
    const size_t part = pkv_partials_size(shape, cfg);
    const size_t ws_slot = round_up(ws, 256);
    if (ws_slot + part > (size_t)PKV_NOALLOC_SCRATCH_BYTES) {
        char buf[200];
        snprintf(buf, sizeof buf,
                 "pkv_decode_step_noalloc: this step needs %zu bytes of scratch, the static "
                 "scratch holds %d",
                 ws_slot + part, (int)PKV_NOALLOC_SCRATCH_BYTES);
        return pkv::record_error(PKV_ECAPACITY, buf);
    }
    void *base = nullptr;
    const int rc = scratch_address(&base);
    if (rc != PKV_OK)
        return rc;
    // the array keeps the previous call's contents: clear the workspace header
    // (error word, task count, the decode's task-claim and barrier counters),
    // which must start at zero; the rest is written before it is read
    if (cudaMemsetAsync(base, 0, 64, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return pkv::record_error(PKV_ECUDA, "pkv_decode_step_noalloc: cudaMemsetAsync failed");
    float *partials = part ? reinterpret_cast<float *>(static_cast<unsigned char *>(base) + ws_slot)
                           : nullptr;
    return pkv_decode_step(shape, cfg, base, d_q, d_k_cache, d_v_cache, d_block_table, d_seq_lens,
                           partials, d_o, d_lse, stream);
}
