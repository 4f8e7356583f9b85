// dg_internal.h -- what the C ABI (dg_abi.cu) and the kernel files share: tile geometry, the head
// work plan, the argument blocks of each launch, the launch functions, and the small device helpers
// every kernel of a pass uses (programmatic dependent launch, the per-pass timeline, the pass's
// temperature).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/dgcanvas.h"

namespace dg {

// Tile geometry of the tensor-core head: 128 slot rows x 256 vocabulary columns per tile, one
// 128-byte K slice (64 bf16 or 128 e4m3 elements) per pipeline stage.
constexpr int kTcBM = 128;
constexpr int kTcBN = 256;
constexpr int kTcStages = 4;
constexpr int kTc2Stages = 6;    // pair kernel: 32 KB stages (128 h rows + 128 W rows); bf16 +1
constexpr int kTcThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
// NVFP4 head: vocabulary rows per tile, accumulator buffers, pipeline stages and threads. TMEM
// holds kFp4Acc accumulators of kFp4BN columns plus the scale factors of every stage in flight; of
// the configurations that fit, 256-row tiles with one accumulator measured fastest (128-row tiles
// with two accumulators re-read h twice as often and issue more scale copies per column). Each
// stage carries four copies of the w scale chunk (one per TMEM lane quadrant), which leaves shared
// memory for 3 stages. 8 epilogue warps: two per lane quadrant, one per half of the tile's columns.
constexpr int kFp4BN = 256;
constexpr int kFp4Acc = 1;
constexpr int kFp4Stages = 3;
constexpr int kFp4Threads = 320;
// Geometry of the fp32 CUDA-core head.
constexpr int kSimtBM = 128;
constexpr int kSimtBN = 64;

// Work decomposition of a head pass: MB row blocks x NT vocabulary tiles, each row block split
// into n_groups vocabulary groups (group g takes tiles g, g + n_groups, ...). A (row block,
// group) unit writes `parts` Partials per row (one per column subset of its tiles) into
// partials[row * n_groups * parts + g * parts + part].
// For the CTA-pair kernel (pair = 1) a row block is 256 rows and `grid` counts pairs.
struct HeadPlan {
    int R, V, d;
    int BM, BN;
    int MB, NT, n_groups, units, grid;
    int pair;
    int parts;
};

HeadPlan plan_head(int R, int V, int d, int BM, int BN, int num_sms);
// Pair plan: groups chosen so that units = lcm(MB, pairs) spread evenly over the pairs.
HeadPlan plan_head_pair(int R, int V, int d, int max_pairs);

struct HeadArgs {
    int R, V, d;
    int MB, NT, n_groups, num_kb;
    float crow_base;          // inv_temp * log2(e)
    const float* h_scale;     // [R] or null
    const float* w_scale;     // [V] or null
    float4* partials;         // [R][n_groups * parts]: the partials of one row are contiguous
    uint32_t* status;         // sticky status word or null
    unsigned long long* timeline;  // loop timeline (dg_loop_params.trace_timeline) or null
    const int32_t* pass_ptr;       // loop mode: the pass index (device), else null
    const int32_t* stop;           // loop mode: non-zero = the loop has ended, do nothing
    float temp_start, temp_end;    // loop temperature schedule (temp_passes > 0)
    int temp_passes;               // max_passes of the schedule, 0 = none
    unsigned long long* clk;       // SM clock sample [n][4] or null (head_clock_slot)
    int clk_per_pass;              // 1: row *pass_ptr of clk (loop trace), 0: row 0
};

// The logit scale of a pass, in base-2 units: crow_base (= inv_temp * log2 e), divided by the
// pass's temperature T_p = t0 + (t1 - t0) * p / (P - 1) when a schedule is set (fp32).
__device__ __forceinline__ float pass_crow_base(const HeadArgs& a) {
    if (a.temp_passes <= 0 || a.pass_ptr == nullptr) return a.crow_base;
    const int p = *a.pass_ptr;
    const float T = a.temp_passes > 1
                        ? a.temp_start + __fdiv_rn((a.temp_end - a.temp_start) * static_cast<float>(p),
                                                   static_cast<float>(a.temp_passes - 1))
                        : a.temp_start;
    return __fdiv_rn(a.crow_base, T);
}

// Programmatic dependent launch. Every kernel of a pass is launched with the programmatic
// stream-serialization attribute, so it may be scheduled while its predecessor in the stream is
// still running; it calls grid_dependency_wait() before its first global-memory access, which
// returns once the predecessor grid has completed and its writes are visible (a no-op for a
// normal launch). grid_launch_dependents() lets the successor be scheduled early.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Per-pass kernel timeline: the first CTA past its dependency wait sets `begin`, the last CTA to
// finish sets `end` (atomic min / max of the device global timer, in ns). Thread 0 of each CTA.
__device__ __forceinline__ unsigned long long globaltimer_now() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void timeline_begin(unsigned long long* tl, int pass, int kernel) {
    if (tl != nullptr && threadIdx.x == 0)
        atomicMin(tl + 2 * (static_cast<size_t>(pass) * DG_TL_KERNELS + kernel), globaltimer_now());
}
__device__ __forceinline__ void timeline_end(unsigned long long* tl, int pass, int kernel) {
    if (tl != nullptr && threadIdx.x == 0)
        atomicMax(tl + 2 * (static_cast<size_t>(pass) * DG_TL_KERNELS + kernel) + 1, globaltimer_now());
}

// SM clock sample of a head launch: CTA 0 / thread 0 stores its clock64 and the global timer
// (ns) when it gets past its dependency wait (slot[0], slot[1]) and when it leaves (slot[2],
// slot[3]); cycles over nanoseconds is the SM clock the kernel actually ran at, and the cycle
// count is the kernel's duration independent of that clock.
__device__ __forceinline__ unsigned long long* head_clock_slot(const HeadArgs& a) {
    if (a.clk == nullptr || blockIdx.x != 0 || threadIdx.x != 0) return nullptr;
    return a.clk + 4 * static_cast<size_t>(a.clk_per_pass && a.pass_ptr ? *a.pass_ptr : 0);
}
__device__ __forceinline__ void head_clock_stamp(unsigned long long* slot, int i) {
    if (slot != nullptr) {
        slot[2 * i] = static_cast<unsigned long long>(clock64());
        slot[2 * i + 1] = globaltimer_now();
    }
}

inline void set_pdl_attr(cudaLaunchAttribute* a) {
    a->id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a->val.programmaticStreamSerializationAllowed = 1;
}

// Opts kernel `fn` in to `bytes` of dynamic shared memory on the current device, once per
// (device, kernel, size). The attribute belongs to the device's context, so a process that
// drives several GPUs sets it on each; thread-safe.
cudaError_t ensure_smem_attr(const void* fn, int bytes);

// Tensor-core head (bf16: kind = 0, e4m3: kind = 1). h and w are device row-major matrices.
// Runs the CTA-pair kernel when plan.pair, else the single-CTA kernel.
cudaError_t launch_head_tc(int kind, const void* h, const void* w, const HeadArgs& args,
                           const HeadPlan& plan, cudaStream_t stream);
cudaError_t launch_head_tc2(int kind, const CUtensorMap& ma, const CUtensorMap& mb,
                            const HeadArgs& args, int n_pairs, cudaStream_t stream);
// Resident clusters of the pair kernel on the current device (0 if it cannot run).
int head_tc2_max_pairs();
// NVFP4 head (single-CTA, block-scaled MMAs): codes of h and w, h block scales in the row-block
// layout, w block scales packed.
cudaError_t launch_head_fp4(const void* qh, const uint8_t* sfa, const void* qw, const uint8_t* sfb,
                            const HeadArgs& args, int grid, cudaStream_t stream);
// NVFP4 preparation (dg_nvfp4.cu). Packed block-scale arrays cover nvfp4_rows_pad(rows) rows;
// the row-block layout of the head's A operand takes nvfp4_rowblock_bytes(rows, d) bytes.
// layout: 0 = packed (dg_nvfp4_pack_scales), 1 = row-block.
int nvfp4_rows_pad(int rows);
size_t nvfp4_rowblock_bytes(int rows, int d);
cudaError_t launch_quant_rows_nvfp4(const uint16_t* h, int R, int d, uint8_t* q, uint8_t* sf,
                                    float* scale, uint32_t* status, cudaStream_t stream,
                                    int layout = 0);
cudaError_t launch_repack_rowblock(const uint8_t* packed, int R, int d, uint8_t* out,
                                   cudaStream_t stream);
cudaError_t launch_pack_scales(const uint8_t* plain, int rows, int d, uint8_t* packed,
                               cudaStream_t stream);
// fp32 CUDA-core head.
cudaError_t launch_head_simt(const float* h, const float* w, const HeadArgs& args, int grid,
                             cudaStream_t stream);

// Loop control block in the workspace (device).
struct LoopCtl {
    int32_t pass;       // index of the pass about to run
    uint32_t ticket;    // canvases of the merge kernel finished in this pass
    int32_t max_passes;
    int32_t stop;       // set once the loop has ended: later passes of a graph iteration are no-ops
    uint64_t row_offset;  // added to the row index of every re-draw key
};

struct SelectArgs {
    const float4* partials;           // [R][n_groups]
    int n_groups, R, S, B, V;
    int32_t* argmax;                  // per-row statistics: caller's arrays or workspace scratch
    float* conf;
    float* entropy;
    float* mean_entropy;              // optional [B]
    uint8_t* kept;
    const int32_t* canvas_in;         // null: statistics only
    int32_t* canvas_out;
    double inv_v;                     // RN(1 / V) for the exact draw modulo
    int keep_rule;                    // DG_KEEP_CONFIDENCE / DG_KEEP_ENTROPY
    int redraw_mode;                  // DG_REDRAW_UNIFORM / DG_REDRAW_MASK
    int mask_id;
    int keep_k;                       // fixed K when keep_k0 < 0
    int keep_k0;                      // >= 0: K_t = min(keep_k0 * (p + 1), S)
    const int32_t* keep_sched;        // optional [max_passes]
    uint64_t seed;
    uint32_t pass;                    // host pass index when ctl == null
    dg_canvas_state* state;           // optional [B]
    dg_stop_rule rule;
    int has_rule;
    LoopCtl* ctl;                     // loop mode: pass from ctl, advance it, set condition
    cudaGraphConditionalHandle cond;
    int set_cond;
    float* trace_mean_entropy;        // optional [max_passes * B]
    int32_t* trace_canvas;            // optional [max_passes * R]
    int32_t* trace_argmax;            // optional [max_passes * R] (loop mode)
    float* trace_conf;
    float* trace_entropy;
    unsigned long long* timeline;     // optional loop timeline
    uint32_t* status;
};

cudaError_t launch_select(const SelectArgs& a, cudaStream_t stream);

// Per-row absmax E4M3 quantisation of bf16 rows.
cudaError_t launch_quant_rows(const uint16_t* h, int R, int d, uint8_t* q, float* scale,
                              uint32_t* status, cudaStream_t stream);

// Loop set-up: optional random initial canvas, state reset, control block reset.
// init_random: 1 = uniform draws key(seed, 0xFFFFFFFF, row_offset + r) mod V, 2 = mask_id.
cudaError_t launch_loop_init(int32_t* canvas, int R, int S, int B, int V, uint64_t seed,
                             int init_random, int mask_id, uint64_t row_offset,
                             dg_canvas_state* state, int keep_stable, LoopCtl* ctl,
                             int start_pass, int max_passes, uint32_t* status,
                             unsigned long long* timeline, cudaStream_t stream);

// Copy rows of one pass into a trace buffer at offset pass * bytes (pass read on device).
cudaError_t launch_trace_copy(const void* src, void* dst, size_t bytes, const LoopCtl* ctl,
                              cudaStream_t stream);

// Built-in synthetic denoiser (stop: optional loop stop flag, non-zero = do nothing). With
// q_out/scale_out non-null it also quantises each bf16 row it writes to E4M3 with the per-row
// absmax rule of launch_quant_rows (one kernel instead of two).
cudaError_t launch_synth_denoise(const dg_head_desc* desc, const int32_t* y, int n_content,
                                 float s_content, float s_pad, const int32_t* canvas,
                                 const int32_t* pass, uint16_t* h_out, uint32_t* status,
                                 cudaStream_t stream, uint8_t* q_out = nullptr,
                                 float* scale_out = nullptr,
                                 unsigned long long* timeline = nullptr,
                                 const int32_t* stop = nullptr);

}  // namespace dg
