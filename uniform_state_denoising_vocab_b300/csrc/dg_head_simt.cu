// dg_head_simt.cu -- fp32 vocabulary head on the CUDA cores, with the same online-softmax
// epilogue as the tensor-core head. Used for fp32 operands, which the tensor cores would round
// (tf32); it serves small heads (hidden size 64, vocabulary 4096 in the fp32 workload).
//
// One CTA of 256 threads per (row block, vocabulary group) unit: threads t and t + 128 own slot
// row mb*128 + t, each keeping 32 hidden values of the row in registers and accumulating its half
// (32 logits) of every 64-column vocabulary tile against a 64 x 32 slice of W staged in shared
// memory (broadcast reads); each half folds its columns into its own running state and writes
// its own partial (two per row and unit).
#include <cuda_runtime.h>

#include "dg_common.cuh"
#include "dg_internal.h"

namespace dg {
namespace {

constexpr int BM = kSimtBM;  // 128 rows per CTA
constexpr int BN = kSimtBN;  // 64 vocabulary columns per tile
constexpr int KC = 32;       // hidden values per staging step
constexpr int THREADS = 2 * BM;
constexpr int HC = BN / 2;   // columns of a tile per thread
static_assert(HC == 32, "one 32-column fold per thread and tile");

__global__ void __launch_bounds__(THREADS)
    head_simt_kernel(const float* __restrict__ h, const float* __restrict__ w, const HeadArgs args) {
    __shared__ __align__(16) float ws[BN][KC];
    const int t = threadIdx.x & (BM - 1);
    const int half = threadIdx.x / BM;
    grid_dependency_wait();
    const int units = (args.stop != nullptr && *args.stop != 0) ? 0 : args.MB * args.n_groups;
    const int tl_pass = args.timeline != nullptr ? *args.pass_ptr : 0;
    const float crow_base = pass_crow_base(args);
    if (units > 0) timeline_begin(args.timeline, tl_pass, DG_TL_HEAD);
    unsigned long long* const clk_slot = units > 0 ? head_clock_slot(args) : nullptr;
    head_clock_stamp(clk_slot, 0);
    grid_launch_dependents();
    for (int unit = blockIdx.x; unit < units; unit += gridDim.x) {
        const int mb = unit % args.MB, grp = unit / args.MB;
        const int row = mb * BM + t;
        const bool row_ok = row < args.R;
        const float crow = crow_base;
        RowState st = row_state_init();
        for (int nb = grp; nb < args.NT; nb += args.n_groups) {
            float acc[HC];
#pragma unroll
            for (int j = 0; j < HC; ++j) acc[j] = 0.f;
            for (int k0 = 0; k0 < args.d; k0 += KC) {
                float hr[KC];
#pragma unroll
                for (int j = 0; j < KC; ++j) {
                    const int k = k0 + j;
                    hr[j] = (row_ok && k < args.d) ? h[static_cast<size_t>(row) * args.d + k] : 0.f;
                }
                __syncthreads();
                for (int i = threadIdx.x; i < BN * KC; i += THREADS) {
                    const int n = nb * BN + i / KC, k = k0 + i % KC;
                    ws[i / KC][i % KC] =
                        (n < args.V && k < args.d) ? w[static_cast<size_t>(n) * args.d + k] : 0.f;
                }
                __syncthreads();
#pragma unroll
                for (int n = 0; n < HC; ++n) {
                    const float4* wr = reinterpret_cast<const float4*>(ws[half * HC + n]);
                    float a = acc[n];
#pragma unroll
                    for (int q = 0; q < KC / 4; ++q) {
                        const float4 v = wr[q];
                        a = fmaf(hr[4 * q + 0], v.x, a);
                        a = fmaf(hr[4 * q + 1], v.y, a);
                        a = fmaf(hr[4 * q + 2], v.z, a);
                        a = fmaf(hr[4 * q + 3], v.w, a);
                    }
                    acc[n] = a;
                }
            }
            const int n0 = nb * BN + half * HC;
            const int valid = args.V - n0;
            if (valid >= HC)
                row_state_update<false>(st, acc, crow, n0, HC);
            else if (valid > 0)
                row_state_update<true>(st, acc, crow, n0, valid);
        }
        if (row_ok)
            args.partials[static_cast<size_t>(row) * (2 * args.n_groups) + 2 * grp + half] =
                pack(row_state_partial(st));
    }
    if (units > 0) timeline_end(args.timeline, tl_pass, DG_TL_HEAD);
    head_clock_stamp(clk_slot, 1);
}

}  // namespace

cudaError_t launch_head_simt(const float* h, const float* w, const HeadArgs& args, int grid,
                             cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(THREADS);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    set_pdl_attr(&attr[0]);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, head_simt_kernel, h, w, args);
}

}  // namespace dg
