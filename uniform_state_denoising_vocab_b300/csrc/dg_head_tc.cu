// dg_head_tc.cu -- vocabulary-head contraction on the 5th-generation tensor cores with a fused
// online-softmax epilogue. Computes, for every slot row r and every vocabulary id n,
//   l[r, n] = inv_temp * sum_k h[r, k] * W[n, k]   (times h_scale[r] * w_scale[n] for E4M3)
// in fp32 TMEM accumulators and folds each 128 x 256 tile straight into per-row softmax
// partials (running max, argmax, sum of exponentials, sum of exponential-weighted logits);
// logits are never written to memory. Each pass predicts every slot of the canvas through the
// head ("When to use a diffusion LLM" (devengoratela.com), "How block diffusion works"; the
// vocabulary is 262K per "DiffusionGemma 26B: How Google's Text Diffusion Model Generates Tokens
// in Parallel" (dev.to), "Architecture Details").
//
// Structure (one persistent CTA per SM, 192 threads):
//   warp 0     one elected thread issues TMA loads of A = h (128 x 128 B) and B = W (256 x 128 B)
//              K-slices into a 4-stage shared-memory ring (128-byte swizzle);
//   warp 1     allocates 512 TMEM columns (two 128 x 256 fp32 accumulators) and one elected
//              thread issues tcgen05.mma (M=128, N=256, K=16 bf16 / K=32 e4m3) per slice;
//   warps 2-5  epilogue: each thread owns one TMEM lane (= one slot row), drains its 256
//              columns in 32-column tcgen05.ld chunks and updates its running softmax state,
//              while the MMA warp fills the other accumulator.
// Each CTA walks (row block, vocabulary group) units; the state of a row stays in registers for
// all tiles of a unit and is written once as a 16-byte partial at the end.
#include <cuda.h>
#include <cuda_runtime.h>

#include "dg_common.cuh"
#include "dg_internal.h"
#include "dg_head_epi.cuh"
#include "dg_ptx.cuh"

namespace dg {
namespace {

constexpr int BM = kTcBM, BN = kTcBN, STAGES = kTcStages;
constexpr int A_BYTES = BM * 128;
constexpr int B_BYTES = BN * 128;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 2 * BN;
constexpr int SMEM_BYTES = 1024 /*align slack*/ + STAGES * STAGE_BYTES +
                           4 * BN * 4 /*per-warp column scales*/ + 256 /*barriers and flags*/;

struct SmemCtl {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(SmemCtl) <= 256, "control block too large");

__device__ __forceinline__ void set_abort(SmemCtl* c, uint32_t* status) {
    *reinterpret_cast<volatile int*>(&c->abort) = 1;
    flag_status(status, DG_ST_TIMEOUT);
}

template <int KIND>
__global__ void __launch_bounds__(kTcThreads, 1)
    head_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const HeadArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * A_BYTES;
    float* s_csc = reinterpret_cast<float*>(sB + STAGES * B_BYTES);  // [4 epilogue warps][BN]
    SmemCtl* ctl = reinterpret_cast<SmemCtl*>(s_csc + 4 * BN);
    const volatile int* abort_flag = &ctl->abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr int KB_ELEMS = (KIND == 0) ? 64 : 128;  // elements per 128-byte K slice

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&ctl->full[i], 1);
            mbar_init(&ctl->empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
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
    // a pass after the loop has ended (second pass of a graph iteration) does no work
    const int units = (args.stop != nullptr && *args.stop != 0) ? 0 : args.MB * args.n_groups;
    const int tl_pass = args.timeline != nullptr ? *args.pass_ptr : 0;
    const float crow_base = pass_crow_base(args);
    if (units > 0) timeline_begin(args.timeline, tl_pass, DG_TL_HEAD);
    unsigned long long* const clk_slot = units > 0 ? head_clock_slot(args) : nullptr;
    head_clock_stamp(clk_slot, 0);
    grid_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ TMA producer
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_h = policy_evict_last();
            uint32_t stage = 0, phase = 0, issued = 0;
            uint32_t parity_bits = 0;  // bit s: parity of the last phase issued on stage s
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
                        tma_load_2d(sA + stage * A_BYTES, &tmA, kb * KB_ELEMS, mb * BM,
                                    &ctl->full[stage], pol_h);
                        tma_load_2d(sB + stage * B_BYTES, &tmB, kb * KB_ELEMS, nb * BN,
                                    &ctl->full[stage], pol_w);
                        parity_bits = (parity_bits & ~(1u << stage)) | (phase << stage);
                        ++issued;
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
            // Drain: every load this thread issued must have landed before the CTA exits.
            const uint32_t n = issued < STAGES ? issued : STAGES;
            for (uint32_t i = 0; i < n; ++i) {
                const uint32_t s = (stage + STAGES - 1 - i) % STAGES;
                if (!mbar_wait(&ctl->full[s], (parity_bits >> s) & 1u)) flag_status(args.status, DG_ST_TIMEOUT);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------------ MMA issuer
            constexpr uint32_t idesc = idesc_f32acc(KIND == 0 ? 1u : 0u, BM, BN);
            uint32_t stage = 0, phase = 0, tcount = 0;
            bool ok = true;
            for (int unit = blockIdx.x; unit < units && ok; unit += gridDim.x) {
                const int grp = unit / args.MB;
                for (int nb = grp; nb < args.NT && ok; nb += args.n_groups, ++tcount) {
                    const uint32_t buf = tcount & 1u, tph = (tcount >> 1) & 1u;
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
                        const uint64_t ad = sdesc_kmajor_sw128(smem_u32(sA + stage * A_BYTES));
                        const uint64_t bd = sdesc_kmajor_sw128(smem_u32(sB + stage * B_BYTES));
#pragma unroll
                        for (int k = 0; k < 4; ++k)  // 4 x 32 bytes along K per 128-byte slice
                            mma_ss<KIND>(d_tmem, ad + 2 * k, bd + 2 * k, idesc,
                                         (kb | k) != 0 ? 1u : 0u);
                        mma_commit(&ctl->empty[stage]);
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (ok) mma_commit(&ctl->tfull[buf]);
                }
            }
            // Drain: all MMAs issued by this thread complete before TMEM is released.
            mma_commit(&ctl->drain);
            if (!mbar_wait(&ctl->drain, 0)) flag_status(args.status, DG_ST_TIMEOUT);
        }
    } else {
        // ---------------------------------------------------------------- epilogue
        const int quad = warp & 3;                 // TMEM lane quadrant this warp may access
        const int row_in_block = quad * 32 + lane;
        float* csc = s_csc + (warp - 2) * BN;     // this warp's copy of the column scales
        uint32_t tcount = 0;
        bool ok = true;
        for (int unit = blockIdx.x; unit < units && ok; unit += gridDim.x) {
            const int mb = unit % args.MB, grp = unit / args.MB;
            const int row = mb * BM + row_in_block;
            float crow = crow_base;
            if (KIND == 1 && args.h_scale != nullptr && row < args.R) crow *= args.h_scale[row];
            RowState st = row_state_init();
            for (int nb = grp; nb < args.NT && ok; nb += args.n_groups, ++tcount) {
                const uint32_t buf = tcount & 1u, tph = (tcount >> 1) & 1u;
                const int n_base = nb * BN;
                if (KIND == 1) stage_column_scales<BN>(csc, args.w_scale, n_base, args.V, lane);
                if (!mbar_wait(&ctl->tfull[buf], tph, abort_flag)) {
                    set_abort(ctl, args.status);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr0 = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                        buf * BN;
                drain_tile<KIND, BN>(st, taddr0, csc, crow, n_base, args.V - n_base);
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
    head_clock_stamp(clk_slot, 1);
}

// cuTensorMapEncodeTiled from the driver, resolved once through the runtime.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// Row-major [rows, cols] matrix of 1- or 2-byte elements; box = 128 bytes x box_rows, 128B swizzle.
bool make_map(CUtensorMap* m, const void* base, int elem_bytes, int rows, int cols, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * elem_bytes};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / elem_bytes),
                               static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt =
        elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Row-major [rows, cols_bytes] byte matrix, box 128 bytes x box_rows, 128-byte swizzle.
bool make_map_u8(CUtensorMap* m, const void* base, int rows, int cols_bytes, int box_rows) {
    return make_map(m, base, 1, rows, cols_bytes, box_rows);
}

cudaError_t launch_head_tc(int kind, const void* h, const void* w, const HeadArgs& args,
                           const HeadPlan& plan, cudaStream_t stream) {
    const int eb = kind == 0 ? 2 : 1;
    CUtensorMap ma, mb;
    if (!make_map(&ma, h, eb, args.R, args.d, BM) ||
        !make_map(&mb, w, eb, args.V, args.d, plan.pair ? BN / 2 : BN))
        return cudaErrorInvalidValue;
    if (plan.pair) return launch_head_tc2(kind, ma, mb, args, plan.grid, stream);
    const void* fn = kind == 0 ? reinterpret_cast<const void*>(head_tc_kernel<0>)
                               : reinterpret_cast<const void*>(head_tc_kernel<1>);
    if (cudaError_t ea = ensure_smem_attr(fn, SMEM_BYTES); ea != cudaSuccess) return ea;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    set_pdl_attr(&attr[0]);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = kind == 0 ? cudaLaunchKernelEx(&cfg, head_tc_kernel<0>, ma, mb, args)
                              : cudaLaunchKernelEx(&cfg, head_tc_kernel<1>, ma, mb, args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace dg
