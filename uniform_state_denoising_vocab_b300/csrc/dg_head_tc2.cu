// dg_head_tc2.cu -- vocabulary-head contraction on a CTA pair (tcgen05 cta_group::2) with the
// fused online-softmax epilogue. Same result as dg_head_tc.cu: for every slot row r and
// vocabulary id n,
//   l[r, n] = inv_temp * sum_k h[r, k] * W[n, k]   (times h_scale[r] * w_scale[n] for E4M3)
// accumulated in fp32 TMEM and folded tile by tile into per-row softmax partials; logits are
// never written to memory. Each pass scores every slot of the canvas against the whole
// vocabulary ("When to use a diffusion LLM" (devengoratela.com), "How block diffusion works";
// 262K vocabulary per "DiffusionGemma 26B: How Google's Text Diffusion Model Generates Tokens in
// Parallel" (dev.to), "Architecture Details").
//
// Why a pair: one tcgen05.mma.cta_group::2 computes a 256 x 256 tile over two SMs. Each CTA
// stages 128 slot rows of h and 128 of the tile's 256 vocabulary rows of W, so every W byte
// crosses L2 -> SM once per pair (twice with two independent 128-row CTAs), and each SM's
// tensor core reads half as many B bytes from shared memory per FLOP. Stages are 32 KB per CTA:
// seven fit in shared memory for bf16 (six for E4M3, which also stages the tile's column scales),
// and the loads in flight cover DRAM latency under load.
//
// Roles (192 threads per CTA; cluster of 2, CTA rank 0 = "leader"):
//   warp 0     producer: one thread waits for a free stage (its own `empty` barrier, signalled
//              by the leader's MMA commits in both CTAs) and loads its A and B halves by TMA;
//              the loads of both CTAs complete on the leader's `full` barrier, on which the
//              leader's producer alone registers the byte count of both halves;
//   warp 1     allocates 512 TMEM columns in both CTAs (pair allocation); in the leader one
//              thread issues the pair MMAs (M=256, N=256) and commits to both CTAs' barriers;
//   warps 2-5  epilogue, in both CTAs: each thread owns one TMEM lane (one slot row) and folds
//              the tile's 256 columns into its running state; the four warps of each CTA arrive
//              on the leader's `tempty` barrier (8 arrivals) when an accumulator is drained.
// A pair walks (row block of 256, vocabulary group) units; a row's state stays in registers for
// the whole unit and is written once as a 16-byte partial.
#include <cuda.h>
#include <cuda_runtime.h>

#include "dg_common.cuh"
#include "dg_head_epi.cuh"
#include "dg_internal.h"
#include "dg_ptx.cuh"

namespace dg {
namespace {

constexpr int BM = 128;               // slot rows per CTA (256 per pair)
constexpr int BN = kTcBN;             // vocabulary ids per tile (256; 128 staged per CTA)
// Ring depth: the bf16 head stages no column scales, which leaves room for one more stage.
template <int KIND>
constexpr int stages_of() { return KIND == 0 ? kTc2Stages + 1 : kTc2Stages; }
constexpr int kMaxStages = kTc2Stages + 1;
constexpr int A_BYTES = BM * 128;     // one 128-byte K slice of 128 rows
constexpr int B_BYTES = (BN / 2) * 128;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 2 * BN;
template <int KIND>
constexpr int smem_of() { return 1024 + stages_of<KIND>() * STAGE_BYTES + (KIND == 1 ? 4 * BN * 4 : 0) + 256; }
static_assert(smem_of<0>() <= 227 * 1024 && smem_of<1>() <= 227 * 1024, "shared memory budget");

struct SmemCtl {
    uint64_t full[kMaxStages];   // leader: both CTAs' A/B halves of a stage have landed
    uint64_t empty[kMaxStages];  // each CTA: the stage's MMAs are done (commit multicast)
    uint64_t tfull[2];       // each CTA: accumulator complete (commit multicast)
    uint64_t tempty[2];      // leader: accumulator drained by both CTAs (8 warp arrivals)
    uint64_t drain;          // leader: every MMA issued has completed
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
    head_tc2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const HeadArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;
    constexpr int STAGES = stages_of<KIND>();
    uint8_t* sB = smem + STAGES * A_BYTES;
    float* s_csc = reinterpret_cast<float*>(sB + STAGES * B_BYTES);  // [4 epilogue warps][BN]
    SmemCtl* ctl = reinterpret_cast<SmemCtl*>(s_csc + (KIND == 1 ? 4 * BN : 0));
    const volatile int* abort_flag = &ctl->abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1;
    const int n_pairs = gridDim.x >> 1;
    constexpr int KB_ELEMS = (KIND == 0) ? 64 : 128;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&ctl->full[i], 1);
            mbar_init(&ctl->empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ctl->tfull[i], 1);
            mbar_init(&ctl->tempty[i], 8);
        }
        mbar_init(&ctl->drain, 1);
        ctl->abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc_pair(&ctl->tmem_base, TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();  // barriers of both CTAs initialised and TMEM allocated before any use
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
            for (int unit = pair; unit < units && ok; unit += n_pairs) {
                const int mb = unit % args.MB, grp = unit / args.MB;
                const int arow = mb * (2 * BM) + static_cast<int>(rank) * BM;
                for (int nb = grp; nb < args.NT && ok; nb += args.n_groups) {
                    const int brow = nb * BN + static_cast<int>(rank) * (BN / 2);
                    for (int kb = 0; kb < args.num_kb; ++kb) {
                        if (!mbar_wait(&ctl->empty[stage], phase ^ 1u, abort_flag)) {
                            set_abort(ctl, args.status);
                            ok = false;
                            break;
                        }
                        if (leader) mbar_arrive_expect_tx(&ctl->full[stage], 2 * STAGE_BYTES);
                        const uint32_t fbar = mapa_shared(smem_u32(&ctl->full[stage]), 0);
                        tma_load_2d_pair(sA + stage * A_BYTES, &tmA, kb * KB_ELEMS, arow, fbar,
                                         pol_h);
                        tma_load_2d_pair(sB + stage * B_BYTES, &tmB, kb * KB_ELEMS, brow, fbar,
                                         pol_w);
                        parity_bits = (parity_bits & ~(1u << stage)) | (phase << stage);
                        ++issued;
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
            // Drain (leader): every stage phase either CTA loaded must have landed before exit.
            if (leader) {
                const uint32_t n = issued < STAGES ? issued : STAGES;
                for (uint32_t i = 0; i < n; ++i) {
                    const uint32_t s = (stage + STAGES - 1 - i) % STAGES;
                    if (!mbar_wait(&ctl->full[s], (parity_bits >> s) & 1u))
                        flag_status(args.status, DG_ST_TIMEOUT);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ------------------------------------------------------------ MMA issuer
            constexpr uint32_t idesc = idesc_f32acc(KIND == 0 ? 1u : 0u, 2 * BM, BN);
            uint32_t stage = 0, phase = 0, tcount = 0;
            bool ok = true;
            for (int unit = pair; unit < units && ok; unit += n_pairs) {
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
                            mma_ss_pair<KIND>(d_tmem, ad + 2 * k, bd + 2 * k, idesc,
                                              (kb | k) != 0 ? 1u : 0u);
                        mma_commit_pair(&ctl->empty[stage], 0x3);
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (ok) mma_commit_pair(&ctl->tfull[buf], 0x3);
                }
            }
            // Drain: every MMA this thread issued completes before TMEM is released.
            mma_commit_pair(&ctl->drain, 0x1);
            if (!mbar_wait(&ctl->drain, 0)) flag_status(args.status, DG_ST_TIMEOUT);
        }
    } else {
        // ---------------------------------------------------------------- epilogue
        const int quad = warp & 3;  // TMEM lane quadrant this warp may access
        const int row_in_cta = quad * 32 + lane;
        float* csc = s_csc + (warp - 2) * BN;
        uint32_t tcount = 0;
        bool ok = true;
        for (int unit = pair; unit < units && ok; unit += n_pairs) {
            const int mb = unit % args.MB, grp = unit / args.MB;
            const int row = mb * (2 * BM) + static_cast<int>(rank) * BM + row_in_cta;
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
                if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&ctl->tempty[buf]), 0));
            }
            if (ok && row < args.R)
                args.partials[static_cast<size_t>(row) * args.n_groups + grp] =
                    pack(row_state_partial(st));
        }
    }

    // Neither CTA leaves while the other may still signal its barriers or use the pair's TMEM.
    __syncwarp();
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
    if (units > 0) timeline_end(args.timeline, tl_pass, DG_TL_HEAD);
    head_clock_stamp(clk_slot, 1);
}

}  // namespace

cudaError_t launch_head_tc2(int kind, const CUtensorMap& ma, const CUtensorMap& mb,
                            const HeadArgs& args, int n_pairs, cudaStream_t stream) {
    const void* fn = kind == 0 ? reinterpret_cast<const void*>(head_tc2_kernel<0>)
                               : reinterpret_cast<const void*>(head_tc2_kernel<1>);
    const int smem = kind == 0 ? smem_of<0>() : smem_of<1>();
    cudaError_t e = ensure_smem_attr(fn, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * n_pairs);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    set_pdl_attr(&attr[1]);
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (kind == 0) return cudaLaunchKernelEx(&cfg, head_tc2_kernel<0>, ma, mb, args);
    return cudaLaunchKernelEx(&cfg, head_tc2_kernel<1>, ma, mb, args);
}

int head_tc2_max_pairs() {
    // Clusters of two CTAs of this kernel that can be resident at once (a GPC with an odd number
    // of free SMs leaves one SM out), so that a persistent grid never waits for a second wave.
    constexpr int kMaxDevices = 64;
    static int cached[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    if (cached[dev] > 0) return cached[dev];
    if (ensure_smem_attr(reinterpret_cast<const void*>(head_tc2_kernel<0>), smem_of<0>()) !=
        cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem_of<0>();
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(head_tc2_kernel<0>), &cfg) !=
        cudaSuccess)
        return 0;
    cached[dev] = n;
    return n;
}

}  // namespace dg
