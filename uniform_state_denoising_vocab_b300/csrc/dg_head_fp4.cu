// dg_head_fp4.cu -- vocabulary head with NVFP4 operands on the 5th-generation tensor cores:
// block-scaled E2M1 x E2M1 MMAs (tcgen05 kind::mxf4nvf4, UE4M3 scale factors per 16 elements
// along K) with the same fused online-softmax epilogue as the bf16 / E4M3 heads. For every slot
// row r and vocabulary id n,
//   l[r, n] = inv_temp * g_h[r] * g_w[n] * sum_k (q_h[r,k] sb_h[r,k/16]) (q_w[n,k] sb_w[n,k/16])
// with E2M1 codes q, E4M3 block scales sb and fp32 row scales g; logits are never stored. The
// 4-bit variant follows the NVFP4-quantised model the pages mention ("DiffusionGemma: When Text
// Generation Stops Being Sequential" (laura-martel.com), introduction; "DiffusionGemma 26B: How
// Google's Text Diffusion Model Generates Tokens in Parallel" (dev.to), memory table).
//
// Operand layouts (device, prepared by dg_quantize_nvfp4 / dg_nvfp4_pack_scales):
//   codes: [rows][d/2] bytes, element 2j in the low nibble of byte j;
//   block scales: one 512-byte atom per (128-row group, 64-element K step): byte
//     (m % 32) * 16 + (m / 32) * 4 + kb holds the scale of row 128 g + m, K block 4 j + kb, which
//     a 32x128b tensor-memory copy places at lane m % 32, column m / 32 (replicated over the four
//     lane quadrants): the scale-factor layout the block-scaled MMA reads.
//
// Structure (one CTA of 192 threads per SM; 128 x 256 tiles; K slices of 256 elements):
//   warp 0     TMA loads of the A / B code slices (128-byte swizzle) and bulk loads of their
//              scale atoms into a 4-stage ring;
//   warp 1     owns 512 TMEM columns: the accumulator and one set of scale-factor columns per
//              stage; one thread copies each stage's scale atoms into tensor memory (tcgen05.cp,
//              12 copies of 512 bytes) and issues 4 block-scaled MMAs (M=128, N=256, K=64);
//   warps 2-5  epilogue as in the other heads (one slot row per thread).
// The scale factors of every stage in flight share the 512 TMEM columns with the accumulator, so
// a 256-column tile has a single accumulator and its epilogue does not overlap the next tile's
// MMAs. Measured on the 256 x 262144 x 2816 head: 156 us per launch, of which removing the scale
// copies saves ~55 us (each copy costs ~30 ns in the tensor pipe's issue order) and removing the
// epilogue ~40 us; both are the known limits of this kernel.
#include <cuda.h>
#include <cuda_runtime.h>

#include "dg_common.cuh"
#include "dg_head_epi.cuh"
#include "dg_internal.h"
#include "dg_ptx.cuh"

namespace dg {
namespace {

constexpr int BM = 128, BN = kFp4BN, NACC = kFp4Acc, STAGES = kFp4Stages;
constexpr int KSLICE = 256;                      // FP4 elements per 128-byte K slice
constexpr int KSTEP = 64;                        // elements per MMA
constexpr int A_BYTES = BM * 128;
constexpr int B_BYTES = BN * 128;
constexpr int SF_ATOM = 512;
constexpr int BGROUPS = BN / 128;                // 128-row scale groups per B tile
constexpr int SFA_BYTES = 4 * SF_ATOM;           // 4 K steps x one 128-row group
constexpr int SFB_BYTES = BGROUPS * 4 * SF_ATOM; // groups x 4 K steps
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
constexpr int TMEM_COLS = 512;
constexpr uint32_t SF_COL0 = NACC * BN;          // scale-factor columns after the accumulators
constexpr uint32_t SFB_COLS = BN / 32;           // scale columns of B per MMA
constexpr uint32_t SF_COLS_PER_STAGE = 4 * 4 + 4 * SFB_COLS;
static_assert(SF_COL0 + STAGES * SF_COLS_PER_STAGE <= TMEM_COLS, "TMEM budget");
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + 4 * BN * 4 + 256;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

struct SmemCtl {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[NACC], tempty[NACC], drain;
    uint32_t tmem_base;
    int abort;
};

__device__ __forceinline__ void set_abort(SmemCtl* c, uint32_t* status) {
    *reinterpret_cast<volatile int*>(&c->abort) = 1;
    flag_status(status, DG_ST_TIMEOUT);
}

__global__ void __launch_bounds__(kTcThreads, 1)
    head_fp4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const HeadArgs args, const uint8_t* __restrict__ sfa_g,
                    const uint8_t* __restrict__ sfb_g) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;
    uint8_t* sB = sA + STAGES * A_BYTES;
    uint8_t* sSFA = sB + STAGES * B_BYTES;
    uint8_t* sSFB = sSFA + STAGES * SFA_BYTES;
    float* s_csc = reinterpret_cast<float*>(sSFB + STAGES * SFB_BYTES);
    SmemCtl* ctl = reinterpret_cast<SmemCtl*>(s_csc + 4 * BN);
    const volatile int* abort_flag = &ctl->abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nks = args.num_kb * (KSLICE / KSTEP);  // 64-element K steps per row

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&ctl->full[i], 1);
            mbar_init(&ctl->empty[i], 1);
        }
        for (int i = 0; i < NACC; ++i) {
            mbar_init(&ctl->tfull[i], 1);
            mbar_init(&ctl->tempty[i], 4);
        }
        mbar_init(&ctl->drain, 1);
        ctl->abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(&ctl->tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    grid_dependency_wait();  // the prologue above overlaps the previous kernel of the stream
    const int units = (args.stop != nullptr && *args.stop != 0) ? 0 : args.MB * args.n_groups;
    const int tl_pass = args.timeline != nullptr ? *args.pass_ptr : 0;
    const float crow_base = pass_crow_base(args);
    if (units > 0) timeline_begin(args.timeline, tl_pass, DG_TL_HEAD);
    grid_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ loads
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_h = policy_evict_last();
            uint32_t stage = 0, phase = 0, issued = 0, parity_bits = 0;
            bool ok = true;
            for (int unit = blockIdx.x; unit < units && ok; unit += gridDim.x) {
                const int mb = unit % args.MB, grp = unit / args.MB;
                for (int nb = grp; nb < args.NT && ok; nb += args.n_groups) {
                    for (int kb = 0; kb < args.num_kb; ++kb) {
                        if (!mbar_wait(&ctl->empty[stage], phase ^ 1u, abort_flag)) {
                            set_abort(ctl, args.status);
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&ctl->full[stage], STAGE_BYTES);
                        tma_load_2d(sA + stage * A_BYTES, &tmA, kb * 128, mb * BM,
                                    &ctl->full[stage], pol_h);
                        tma_load_2d(sB + stage * B_BYTES, &tmB, kb * 128, nb * BN,
                                    &ctl->full[stage], pol_w);
                        // scale atoms of the slice: K steps 4 kb .. 4 kb + 3 are contiguous
                        bulk_load(sSFA + stage * SFA_BYTES,
                                  sfa_g + (static_cast<size_t>(mb) * nks + 4 * kb) * SF_ATOM,
                                  SFA_BYTES, &ctl->full[stage]);
                        for (int g = 0; g < BGROUPS; ++g)
                            bulk_load(sSFB + stage * SFB_BYTES + g * 4 * SF_ATOM,
                                      sfb_g + (static_cast<size_t>(BGROUPS * nb + g) * nks + 4 * kb) *
                                                  SF_ATOM,
                                      4 * SF_ATOM, &ctl->full[stage]);
                        parity_bits = (parity_bits & ~(1u << stage)) | (phase << stage);
                        ++issued;
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
            const uint32_t n = issued < STAGES ? issued : STAGES;
            for (uint32_t i = 0; i < n; ++i) {
                const uint32_t s = (stage + STAGES - 1 - i) % STAGES;
                if (!mbar_wait(&ctl->full[s], (parity_bits >> s) & 1u))
                    flag_status(args.status, DG_ST_TIMEOUT);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------------ scale copies + MMAs
            constexpr uint32_t idesc = idesc_nvfp4(BM, BN);
            uint32_t stage = 0, phase = 0, tcount = 0;
            bool ok = true;
            for (int unit = blockIdx.x; unit < units && ok; unit += gridDim.x) {
                const int grp = unit / args.MB;
                for (int nb = grp; nb < args.NT && ok; nb += args.n_groups, ++tcount) {
                    const uint32_t buf = tcount % NACC, tph = (tcount / NACC) & 1u;
                    if (!mbar_wait(&ctl->tempty[buf], tph ^ 1u, abort_flag)) {
                        set_abort(ctl, args.status);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + buf * BN;
                    for (int kb = 0; kb < args.num_kb; ++kb) {
                        if (!mbar_wait(&ctl->full[stage], phase, abort_flag)) {
                            set_abort(ctl, args.status);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sf_col = tmem_base + SF_COL0 + stage * SF_COLS_PER_STAGE;
                        const uint32_t sa = smem_u32(sSFA + stage * SFA_BYTES);
                        const uint32_t sb = smem_u32(sSFB + stage * SFB_BYTES);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            tmem_cp_32x128b_x4(sf_col + 4 * j, sdesc_rows16_noswizzle(sa + j * SF_ATOM));
#pragma unroll
                            for (int g = 0; g < BGROUPS; ++g)
                                tmem_cp_32x128b_x4(
                                    sf_col + 16 + SFB_COLS * j + 4 * g,
                                    sdesc_rows16_noswizzle(sb + (g * 4 + j) * SF_ATOM));
                        }
                        const uint64_t ad = sdesc_kmajor_sw128(smem_u32(sA + stage * A_BYTES));
                        const uint64_t bd = sdesc_kmajor_sw128(smem_u32(sB + stage * B_BYTES));
#pragma unroll
                        for (int j = 0; j < 4; ++j)  // 4 x 32 bytes (64 FP4) per 128-byte slice
                            mma_nvfp4(d_tmem, ad + 2 * j, bd + 2 * j, idesc, sf_col + 4 * j,
                                      sf_col + 16 + SFB_COLS * j, (kb | j) != 0 ? 1u : 0u);
                        mma_commit(&ctl->empty[stage]);
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (ok) mma_commit(&ctl->tfull[buf]);
                }
            }
            mma_commit(&ctl->drain);
            if (!mbar_wait(&ctl->drain, 0)) flag_status(args.status, DG_ST_TIMEOUT);
        }
    } else {
        // ---------------------------------------------------------------- epilogue
        const int quad = warp & 3;
        const int row_in_block = quad * 32 + lane;
        float* csc = s_csc + (warp - 2) * BN;
        uint32_t tcount = 0;
        bool ok = true;
        for (int unit = blockIdx.x; unit < units && ok; unit += gridDim.x) {
            const int mb = unit % args.MB, grp = unit / args.MB;
            const int row = mb * BM + row_in_block;
            float crow = crow_base;
            if (args.h_scale != nullptr && row < args.R) crow *= args.h_scale[row];
            RowState st = row_state_init();
            for (int nb = grp; nb < args.NT && ok; nb += args.n_groups, ++tcount) {
                const uint32_t buf = tcount % NACC, tph = (tcount / NACC) & 1u;
                const int n_base = nb * BN;
                stage_column_scales<BN>(csc, args.w_scale, n_base, args.V, lane);
                if (!mbar_wait(&ctl->tfull[buf], tph, abort_flag)) {
                    set_abort(ctl, args.status);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr0 =
                    tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + buf * BN;
                drain_tile<1, BN>(st, taddr0, csc, crow, n_base, args.V - n_base);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->tempty[buf]);
            }
            if (ok && row < args.R)
                args.partials[static_cast<size_t>(row) * args.n_groups + grp] =
                    pack(row_state_partial(st));
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
    if (units > 0) timeline_end(args.timeline, tl_pass, DG_TL_HEAD);
}

}  // namespace

bool make_map_u8(CUtensorMap* m, const void* base, int rows, int cols_bytes, int box_rows);

cudaError_t launch_head_fp4(const void* qh, const uint8_t* sfa, const void* qw, const uint8_t* sfb,
                            const HeadArgs& args, int grid, cudaStream_t stream) {
    CUtensorMap ma, mb;
    if (!make_map_u8(&ma, qh, args.R, args.d / 2, BM) ||
        !make_map_u8(&mb, qw, args.V, args.d / 2, BN))
        return cudaErrorInvalidValue;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(head_fp4_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    set_pdl_attr(&attr[0]);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, head_fp4_kernel, ma, mb, args, sfa, sfb);
}

}  // namespace dg
