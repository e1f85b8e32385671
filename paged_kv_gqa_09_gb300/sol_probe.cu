// sol_probe.cu -- the streaming speed of light of the decode's launch shape.
//
// A measurement tool, not part of libpkv.  It moves a paged K/V pool from HBM
// into shared memory with the decode kernel's machinery -- 5-D TMA boxes with
// 128-byte swizzle and an evict-first L2 policy, a 3-stage ring filled by one
// producer warp and released by four consumer warps, bounded mbarrier waits --
// but does no math, walks no block table (pages come from one random
// permutation, as a block table would give) and merges nothing.  So the time
// it takes for a given volume and grid is what any kernel of that shape pays to
// stream the bytes; comparing the decode kernel with it separates the cost of
// the method's work from the fixed cost of launching and draining a grid.
//
// Pool: K and V each [pages][16 slots][8 kv heads][128] fp16 (32 KB a page).
// Patterns (one box per page per stage row):
//   head  per-head boxes {64, 16, 2, 1, 1} = 4 KB; a stage = 4 pages of one kv
//         head, K+V = 32 KB; 2 CTAs per SM; tasks (head, 64 pages)  <- the decode
//   quad  4-head boxes {64, 16, 2, 4, 1} = 16 KB; a stage = 1 page of 4 heads,
//         K+V = 32 KB; 2 CTAs per SM; tasks (head group, 64 pages)
//   page  whole-page boxes {64, 16, 2, 8, 1} = 32 KB; a stage = 1 page, K+V =
//         64 KB; 1 CTA per SM; tasks (64 pages)
// Tasks stride statically over the CTAs; grid = min(tasks, SMs x CTAs per SM).
// Each run streams a fresh window of the pool (never what the last run left in
// L2).  Output: one line per (pages, pattern) with the mean and the best of
// 9 runs.
//
// Usage: sol_probe [pages ...]   (default: 2048 4096, and SMs x 128)
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <random>
#include <vector>

#include "pkv_device.cuh"

using namespace pkv;

#define CK(x)                                                                        \
    do {                                                                             \
        cudaError_t e_ = (x);                                                        \
        if (e_ != cudaSuccess) {                                                     \
            std::printf("CUDA error %s at line %d\n", cudaGetErrorString(e_), __LINE__); \
            std::exit(1);                                                            \
        }                                                                            \
    } while (0)

namespace {

constexpr int kConsumers = 4;
constexpr int kThreadsPerCta = 32 * (kConsumers + 1);
constexpr int kStages = 3;
constexpr int kPagesPerTask = 64;
constexpr uint64_t kWaitNs = 1000000000ull;
constexpr int kPageBytes = 32768;

struct Params {
    const int *perm;  // logical page -> physical page
    int npages, ntasks, off;
    int heads_per_box, pages_per_stage;
    int stage_bytes;
    int *err;
};

__global__ void __launch_bounds__(kThreadsPerCta, 1)
    stream_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv, Params p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sb = (raw + 1023) & ~1023u;
    const uint32_t full0 = sb + kStages * p.stage_bytes, empty0 = full0 + kStages * 8;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kConsumers);
        }
        fence_mbar_init();
    }
    __syncthreads();
    const int groups = 8 / p.heads_per_box;
    const int box_bytes = p.stage_bytes / 2 / p.pages_per_stage;
    const int steps = kPagesPerTask / p.pages_per_stage;
    if (warp == kConsumers) {
        const uint64_t pol = l2_evict_first_policy();
        int st = 0;
        uint32_t ph = 0;
        for (int t = blockIdx.x; t < p.ntasks; t += gridDim.x) {
            const int grp = t % groups, first = (t / groups) * kPagesPerTask;
            for (int s = 0; s < steps; ++s) {
                if (!__all_sync(0xffffffffu, mbar_wait(empty0 + 8 * st, ph ^ 1, kWaitNs))) {
                    atomicExch(p.err, 1);
                    return;  // the consumers' own bounded waits end them too
                }
                const uint32_t dst = sb + st * p.stage_bytes, bar = full0 + 8 * st;
                if (lane == 0)
                    mbar_arrive_expect_tx(bar, p.stage_bytes);
                __syncwarp();
                if (lane < p.pages_per_stage) {
                    const int lp = first + s * p.pages_per_stage + lane;
                    const int pg = p.perm[(lp + p.off) % p.npages];
                    tma_load_5d(dst + lane * box_bytes, &tk, bar, 0, 0, 0, grp * p.heads_per_box, pg, pol);
                    tma_load_5d(dst + p.stage_bytes / 2 + lane * box_bytes, &tv, bar, 0, 0, 0,
                                grp * p.heads_per_box, pg, pol);
                }
                __syncwarp();
                if (++st == kStages) {
                    st = 0;
                    ph ^= 1;
                }
            }
        }
        return;  // every copy lands before the consumers exit: they wait for each stage
    }
    int st = 0;
    uint32_t ph = 0;
    float touch = 0.f;
    for (int t = blockIdx.x; t < p.ntasks; t += gridDim.x) {
        for (int s = 0; s < steps; ++s) {
            if (!__all_sync(0xffffffffu, mbar_wait(full0 + 8 * st, ph, kWaitNs))) {
                atomicExch(p.err, 2);
                return;
            }
            touch += reinterpret_cast<const float *>(smem_raw + (sb - raw) + st * p.stage_bytes)[threadIdx.x];
            __syncwarp();
            if (lane == 0)
                mbar_arrive(empty0 + 8 * st);
            if (++st == kStages) {
                st = 0;
                ph ^= 1;
            }
        }
    }
    if (touch == 123456.f)
        atomicAdd(p.err, 0);  // keeps the reads
}

struct Pattern {
    const char *name;
    int heads_per_box, pages_per_stage, ctas_per_sm;
};

}  // namespace

int main(int argc, char **argv)
{
    int sms = 0;
    CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
    std::vector<int> sizes;
    for (int a = 1; a < argc; ++a)
        sizes.push_back(std::atoi(argv[a]));
    if (sizes.empty())
        sizes = {2048, 4096, sms * 128};
    int pool = 0;
    for (int n : sizes) {
        if (n <= 0 || n % kPagesPerTask) {
            std::printf("page counts must be positive multiples of %d\n", kPagesPerTask);
            return 1;
        }
        pool = std::max(pool, n);
    }
    pool = std::max(pool, sms * 128);  // room for fresh windows
    const size_t bytes = (size_t)pool * kPageBytes;
    char *k = nullptr, *v = nullptr;
    CK(cudaMalloc(&k, bytes));
    CK(cudaMalloc(&v, bytes));
    CK(cudaMemset(k, 1, bytes));
    CK(cudaMemset(v, 2, bytes));
    std::vector<int> perm(pool);
    for (int i = 0; i < pool; ++i)
        perm[i] = i;
    std::mt19937 rng(20260623);
    std::shuffle(perm.begin(), perm.end(), rng);
    int *dperm = nullptr, *derr = nullptr;
    CK(cudaMalloc(&dperm, pool * sizeof(int)));
    CK(cudaMemcpy(dperm, perm.data(), pool * sizeof(int), cudaMemcpyHostToDevice));
    CK(cudaMalloc(&derr, sizeof(int)));
    CK(cudaMemset(derr, 0, sizeof(int)));

    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    CK(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q));
    auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    auto make_map = [&](CUtensorMap *m, void *base, int heads) {
        cuuint64_t dims[5] = {64, 16, 2, 8, (cuuint64_t)pool};
        cuuint64_t strides[4] = {2048, 128, 256, (cuuint64_t)kPageBytes};
        cuuint32_t box[5] = {64, 16, 2, (cuuint32_t)heads, 1}, es[5] = {1, 1, 1, 1, 1};
        if (encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 5, base, dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE)) {
            std::printf("cuTensorMapEncodeTiled failed\n");
            std::exit(1);
        }
    };
    CK(cudaFuncSetAttribute(stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024));
    cudaEvent_t e0, e1;
    CK(cudaEventCreate(&e0));
    CK(cudaEventCreate(&e1));
    const Pattern patterns[] = {{"head", 1, 4, 2}, {"quad", 4, 1, 2}, {"page", 8, 1, 1}};
    std::printf("sms %d pool_pages %d\n", sms, pool);
    for (int pages : sizes) {
        for (const Pattern &pt : patterns) {
            CUtensorMap mk, mv;
            make_map(&mk, k, pt.heads_per_box);
            make_map(&mv, v, pt.heads_per_box);
            const int box = kPageBytes / 8 * pt.heads_per_box;
            const int stage = 2 * box * pt.pages_per_stage;
            const int smem = kStages * stage + 2 * kStages * 8 + 1024;
            int occ = 0;
            CK(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, stream_kernel, kThreadsPerCta, smem));
            Params p{dperm, pool, (8 / pt.heads_per_box) * (pages / kPagesPerTask), 0,
                     pt.heads_per_box, pt.pages_per_stage, stage, derr};
            const int grid = std::min(sms * std::min(occ, pt.ctas_per_sm), p.ntasks);
            float best = 1e30f, sum = 0.f;
            constexpr int kRuns = 9;
            for (int r = 0; r < kRuns; ++r) {
                p.off = (r % 5) * pages;  // a fresh window of the pool each run
                CK(cudaEventRecord(e0));
                stream_kernel<<<grid, kThreadsPerCta, smem>>>(mk, mv, p);
                CK(cudaEventRecord(e1));
                CK(cudaEventSynchronize(e1));
                float ms = 0.f;
                CK(cudaEventElapsedTime(&ms, e0, e1));
                best = std::min(best, ms);
                sum += ms;
            }
            int err = 0;
            CK(cudaMemcpy(&err, derr, sizeof(int), cudaMemcpyDeviceToHost));
            const double moved = 2.0 * pages * (double)kPageBytes;
            const float mean = sum / kRuns;
            std::printf("pages %d pattern %s grid %d tasks %d us %.2f best %.2f gbs %.0f err %d\n", pages,
                        pt.name, grid, p.ntasks, mean * 1e3, best * 1e3, moved / (mean * 1e-3) / 1e9, err);
        }
    }
    return 0;
}
