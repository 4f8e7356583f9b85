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
//   block scales of w: packed, one 4096-byte chunk per (256-row group, 256-element K slice);
//   block scales of h: the row-block layout, two 4096-byte tiles per (128-row block, K slice)
//     (both layouts in dg_nvfp4.cu). The block-scaled MMA reads the scale of tile row m (lane
//     quadrant q = m / 32) for a 64-element step from TMEM lane m, column (scale address + q);
//     the scales of the 256 w rows of a step occupy 8 columns of every lane quadrant.
//
// Structure (one CTA of 320 threads per SM; 128 x 256 tiles; K slices of 256 elements):
//   warp 0     TMA loads of the A / B code slices (128-byte swizzle) and bulk loads of the scales
//              into a 3-stage ring: the h row block's two tiles, the w chunk four times (one copy
//              per lane quadrant, so that a single 128x256b copy fills all four);
//   warp 1     owns 512 TMEM columns: the accumulator and one set of scale-factor columns per
//              stage; one thread copies each stage's scales into tensor memory (two 128x256b
//              copies of h scales, one per pair of 64-element steps; one 128x256b copy of w
//              scales per step) and issues 4 block-scaled MMAs (M=128, N=256, K=64);
//   warps 2-9  epilogue: two warps per lane quadrant (one slot row per thread), each folding one
//              half of the tile's 256 columns into its own running state, so a unit writes two
//              partials per row.
// The scale factors of every stage in flight share the 512 TMEM columns with the accumulator, so
// a 256-column tile has a single accumulator; each epilogue thread loads its 128 columns into
// registers in one TMEM load and releases the accumulator before folding them, so the softmax
// arithmetic of a tile overlaps the MMAs of the next. Scale copies are issued in order with the
// MMAs and cost time per instruction (the quadrant-replicating 32x128b.warpx4 form about twice a
// 128x256b copy), so every scale tile is laid out for 128x256b copies: 6 per K slice instead of
// 12 replicated ones.
#include <cuda.h>
#include <cuda_runtime.h>

#include "dg_common.cuh"
#include "dg_head_epi.cuh"
#include "dg_internal.h"
#include "dg_ptx.cuh"

namespace dg {
namespace {

constexpr int BM = 128, BN = kFp4BN, NACC = kFp4Acc, STAGES = kFp4Stages;
constexpr int A_BYTES = BM * 128;
constexpr int B_BYTES = BN * 128;
constexpr int SF_CHUNK = 4096;                   // packed scales of 256 rows x one K slice
constexpr int SFA_BYTES = 2 * 4096;             // row-block layout: two 128x256b copy sources
constexpr int SFB_BYTES = 4 * SF_CHUNK;          // the w chunk once per TMEM lane quadrant
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
constexpr int EPI_WARPS = kFp4Threads / 32 - 2;  // two per lane quadrant
constexpr int HALF = BN / 2;                     // columns per epilogue warp
static_assert(BN == 256, "a w scale chunk covers 256 vocabulary rows");
static_assert(EPI_WARPS == 8, "two epilogue warps per lane quadrant");
static_assert(HALF == 128, "one 32x32b.x128 TMEM load per epilogue warp and tile");
constexpr int TMEM_COLS = 512;
constexpr uint32_t SF_COL0 = NACC * BN;          // scale-factor columns after the accumulators
constexpr uint32_t SFB_COLS = BN / 32;           // scale columns of B per MMA
constexpr uint32_t SF_COLS_PER_STAGE = 4 * 4 + 4 * SFB_COLS;
static_assert(SF_COL0 + STAGES * SF_COLS_PER_STAGE <= TMEM_COLS, "TMEM budget");
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_WARPS * HALF * 4 + 256;
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

__global__ void __launch_bounds__(kFp4Threads, 1)
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
    SmemCtl* ctl = reinterpret_cast<SmemCtl*>(s_csc + EPI_WARPS * HALF);
    const volatile int* abort_flag = &ctl->abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nsl = args.num_kb;  // 256-element K slices per row (one scale chunk each)

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&ctl->full[i], 1);
            mbar_init(&ctl->empty[i], 1);
        }
        for (int i = 0; i < NACC; ++i) {
            mbar_init(&ctl->tfull[i], 1);
            mbar_init(&ctl->tempty[i], EPI_WARPS);
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
    unsigned long long* const clk_slot = units > 0 ? head_clock_slot(args) : nullptr;
    head_clock_stamp(clk_slot, 0);
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
                        // scales of the slice: the h row block's tiles, the w chunk per quadrant
                        bulk_load(sSFA + stage * SFA_BYTES,
                                  sfa_g + (static_cast<size_t>(mb) * nsl + kb) * SFA_BYTES,
                                  SFA_BYTES, &ctl->full[stage]);
                        const uint8_t* wchunk =
                            sfb_g + (static_cast<size_t>(nb) * nsl + kb) * SF_CHUNK;
                        for (int q = 0; q < 4; ++q)
                            bulk_load(sSFB + stage * SFB_BYTES + q * SF_CHUNK, wchunk, SF_CHUNK,
                                      &ctl->full[stage]);
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
                        // h scales: steps 2p, 2p + 1 from tile p of the row-block layout into
                        // columns 8p .. 8p + 7 (step j's scale address: column 4j); w scales of
                        // step j from byte j * 256 of the four chunk copies (quadrant q's rows
                        // 4096 q on; 8-row groups 1024 bytes apart) into 8 columns
#pragma unroll
                        for (int p = 0; p < 2; ++p)
                            tmem_cp_128x256b(sf_col + 8 * p, sdesc_noswizzle(sa + p * 4096, 128, 256));
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            tmem_cp_128x256b(sf_col + 16 + SFB_COLS * j,
                                             sdesc_noswizzle(sb + j * 256, 128, 1024));
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
        const int ew = warp - 2;
        const int quad = warp & 3;       // TMEM lane quadrant this warp may access
        const int half = ew >> 2;        // columns [half * HALF, half * HALF + HALF) of each tile
        const int row_in_block = quad * 32 + lane;
        const int parts_per_row = 2 * args.n_groups;
        float* csc = s_csc + ew * HALF;
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
                const int n_base = nb * BN + half * HALF;
                stage_column_scales<HALF>(csc, args.w_scale, n_base, args.V, lane);
                if (!mbar_wait(&ctl->tfull[buf], tph, abort_flag)) {
                    set_abort(ctl, args.status);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr0 =
                    tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + buf * BN + half * HALF;
                // take the 128 columns into registers and hand the accumulator back at once: the
                // arithmetic below overlaps the next tile's MMAs
                float v[HALF];
                tmem_ld128(taddr0, v);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->tempty[buf]);
                fold_columns<1, HALF>(st, v, csc, crow, n_base, args.V - n_base);
            }
            if (ok && row < args.R)
                args.partials[static_cast<size_t>(row) * parts_per_row + 2 * grp + half] =
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
    head_clock_stamp(clk_slot, 1);
}

}  // namespace

bool make_map_u8(CUtensorMap* m, const void* base, int rows, int cols_bytes, int box_rows);

cudaError_t launch_head_fp4(const void* qh, const uint8_t* sfa, const void* qw, const uint8_t* sfb,
                            const HeadArgs& args, int grid, cudaStream_t stream) {
    CUtensorMap ma, mb;
    if (!make_map_u8(&ma, qh, args.R, args.d / 2, BM) ||
        !make_map_u8(&mb, qw, args.V, args.d / 2, BN))
        return cudaErrorInvalidValue;
    if (cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(head_fp4_kernel), SMEM_BYTES);
        e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kFp4Threads);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    set_pdl_attr(&attr[0]);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, head_fp4_kernel, ma, mb, args, sfa, sfb);
}

}  // namespace dg
