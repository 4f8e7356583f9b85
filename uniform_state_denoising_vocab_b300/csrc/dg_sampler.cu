// dg_sampler.cu -- the per-canvas part of a pass and the loop plumbing:
//   merge_select    merge the vocabulary-group partials of every slot into argmax, confidence
//                   and entropy (one warp per slot); then, in the last CTA of each canvas to
//                   finish: mean entropy (fixed-order tree), rank slots by
//                   (confidence desc, slot asc), keep the top K at their argmax, re-draw the
//                   rest uniformly with the SplitMix64 counter key, and apply the stop rules.
//                   "Each pass, the model predicts every slot at once, keeps the ones it's most
//                   confident about, and re-randomizes the rest" ("When to use a diffusion LLM"
//                   (devengoratela.com), "How block diffusion works"); stop on mean entropy
//                   below a threshold or tokens stable across two consecutive steps, at most 48
//                   steps ("DiffusionGemma 26B: How Google's Text Diffusion Model Generates Tokens
//                   in Parallel" (dev.to), "How Diffusion Changes the Equation").
//   quant_rows      per-row absmax E4M3 quantisation of bf16 hidden states (FP8 head).
//   loop_init       random initial canvas (uniform-state start, same devengoratela.com section),
//                   state and control-block reset.
//   trace_copy      per-pass trace of the hidden states for checking.
//   synth_denoise   built-in synthetic denoiser (test workload, not part of the method).
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "dg_common.cuh"
#include "dg_internal.h"
#include "dg_ptx.cuh"

namespace dg {
namespace {

// The same monoid over several partials at once, maximum first: M = max mx, then every non-empty
// term rescaled to M with its own 2^(mx - M) (independent special-function operations instead of
// a chain of pairwise merges), S = sum 2^(mx - M) s, U = sum 2^(mx - M) (u + s (mx - M)), argmax
// the lowest index among the terms attaining M. Empty partials (s = 0) contribute nothing; a
// non-finite s or u propagates into the result, where the merge's finiteness check sees it.
__device__ __forceinline__ Partial fold_max_first(const Partial (&p)[4]) {
    float M = p[0].mx;
#pragma unroll
    for (int i = 1; i < 4; ++i) M = fmaxf(M, p[i].mx);
    Partial r;
    r.mx = M;
    r.s = 0.f;
    r.u = 0.f;
    r.idx = 0x7FFFFFFF;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (p[i].s == 0.f) continue;
        const float d = p[i].mx - M;
        const float e = ex2_fast(d);
        r.s = fmaf(e, p[i].s, r.s);
        r.u = fmaf(e, fmaf(p[i].s, d, p[i].u), r.u);
        if (p[i].mx == M) r.idx = min(r.idx, p[i].idx);
    }
    return r;
}

// Across the 32 lanes of a warp (each holding one partial): maximum by xor butterfly, each lane
// rescales its own terms, then sums and the lowest attaining index by xor butterflies; every
// lane ends with the same result (each butterfly step adds the same two values on both lanes).
__device__ __forceinline__ Partial warp_fold_max_first(const Partial& a) {
    float M = a.mx;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const bool live = a.s != 0.f;
    const float d = a.mx - M;
    const float e = live ? ex2_fast(d) : 0.f;
    float S = live ? e * a.s : 0.f;
    float U = live ? e * fmaf(a.s, d, a.u) : 0.f;
    int idx = (live && a.mx == M) ? a.idx : 0x7FFFFFFF;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        S += __shfl_xor_sync(0xffffffffu, S, off);
        U += __shfl_xor_sync(0xffffffffu, U, off);
        idx = min(idx, __shfl_xor_sync(0xffffffffu, idx, off));
    }
    return Partial{M, S, U, idx};
}

// ---------------------------------------------------------------------------------------------
// The per-canvas step, on one thread-block cluster per canvas (kMergeCluster CTAs).
// ---------------------------------------------------------------------------------------------
constexpr int kMergeCluster = 8;              // CTAs per canvas (one cluster)
constexpr int kMergeThreads = 1024;           // 32 warps per CTA: one slot row per warp at S = 256
constexpr int kMergeWarps = kMergeThreads / 32;
constexpr int kMaxRowsPerCta = 1024 / kMergeCluster;

__device__ __forceinline__ float ld_cluster_f32(uint32_t cluster_addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr) : "memory");
    return v;
}
__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

struct MergeSmem {
    float key[kMaxRowsPerCta];       // this CTA's rows: keep key (larger = kept first),
    float conf[kMaxRowsPerCta];      // confidence, entropy, argmax
    float ent[kMaxRowsPerCta];
    int32_t arg[kMaxRowsPerCta];
    int32_t old[kMaxRowsPerCta];     // this CTA's slots' tokens before the pass
    int32_t draw[kMaxRowsPerCta];    // this CTA's slots' re-randomised tokens for the pass
    float all_key[1024];             // every slot's keep key (gathered over the cluster)
    float warp_ent[32];              // CTA 0: per-warp sums of the entropy tree
    uint32_t changed[kMergeCluster]; // CTA 0: per-CTA "some slot changed" flags (pushed)
};

// Cluster b (kMergeCluster CTAs of kMergeThreads) handles canvas b. CTA c owns slots
// [c * rpc, (c + 1) * rpc) with rpc = ceil(S / kMergeCluster); warp w merges the vocabulary-group
// partials of its slots w, w + 32, ...: lane l takes groups l, l + 32, ..., four at a time
// (maximum first), then the lanes combine maximum first with fixed xor butterflies, so every run
// merges in the same order and all lanes end with the same result. After a cluster barrier every CTA reads
// the whole canvas's confidences from the cluster's shared memory and ranks its own slots by
// (key desc, slot asc), the key being the confidence or the negated entropy: kept <=> rank < K;
// kept slots take their argmax, the others the counter-hash draw (or the mask token). CTA 0 forms the mean entropy (fixed-order pairwise tree over the slots) and,
// after a second barrier, applies the stop rules; in loop mode the last canvas of the pass
// advances the pass and sets the graph condition.
__global__ void __cluster_dims__(kMergeCluster, 1, 1) __maxnreg__(40)
    merge_select_kernel(const SelectArgs a) {
    __shared__ MergeSmem sm;
    grid_dependency_wait();
    // the next pass's first kernel may be scheduled now and run its prologue beside this grid;
    // it waits for this grid's completion before touching the canvas or the statistics
    grid_launch_dependents();
    if (a.ctl != nullptr && *reinterpret_cast<const volatile int32_t*>(&a.ctl->stop) != 0)
        return;  // the loop ended in an earlier pass of this graph iteration (uniform)
    const int b = blockIdx.x / kMergeCluster;
    const uint32_t c = cluster_ctarank();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = a.S;
    const int rpc = (S + kMergeCluster - 1) / kMergeCluster;
    const int j0 = static_cast<int>(c) * rpc;
    const int nrows = max(0, min(rpc, S - j0));
    const int base = b * S;
    const int p = a.ctl ? a.ctl->pass : static_cast<int>(a.pass);
    timeline_begin(a.timeline, p, DG_TL_MERGE);
    // Loads that do not depend on whether the canvas is frozen go out first: its state word,
    // the old tokens of this CTA's slots and the partials of each warp's rows.
    const int done = a.state != nullptr ? __ldcg(&a.state[b].done) : 0;  // same in every CTA of b
    const uint64_t row_off = a.ctl != nullptr ? __ldcg(&a.ctl->row_offset) : 0ull;
    int old_tok = 0;
    if (a.canvas_out && tid < nrows) old_tok = __ldcg(a.canvas_in + base + j0 + tid);
    // CTA 0 applies the stop rule: its inputs are fetched now
    dg_canvas_state st0 = {};
    int max_passes = 0;
    if (c == 0 && tid == 0) {
        if (a.state != nullptr) st0 = a.state[b];
        if (a.ctl != nullptr) max_passes = a.ctl->max_passes;
    }
    const bool frozen = done != 0;
    int my_done = frozen ? 1 : 0;  // CTA 0 thread 0: this canvas is stopped after the pass

    // The rows are merged whether or not the canvas is frozen (the partials are this pass's), so
    // that no load waits for the state word; a frozen canvas's outputs are left untouched.
    for (int jj = warp; jj < nrows; jj += kMergeWarps) {
        const int r = base + j0 + jj;
        const float4* q = a.partials + static_cast<size_t>(r) * a.n_groups;
        Partial acc = partial_empty();
        // all of this lane's partials (groups lane, lane + 32, ...) in flight at once,
        // then merged in increasing group order
        for (int g0 = 0; g0 < a.n_groups; g0 += 4 * 32) {
            float4 v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int g = g0 + lane + 32 * i;
                v[i] = g < a.n_groups ? __ldcg(q + g) : pack(partial_empty());
            }
            if (g0 == 0 && lane == 0 && a.canvas_out)  // integer work while the loads fly
                sm.draw[jj] = a.redraw_mode == DG_REDRAW_MASK
                                  ? a.mask_id
                                  : static_cast<int32_t>(mod_u64_by_u32(
                                        draw_key(a.seed, static_cast<uint32_t>(p),
                                                 row_off + static_cast<uint64_t>(r)),
                                        static_cast<uint32_t>(a.V), a.inv_v));
            Partial pc[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) pc[i] = unpack(v[i]);
            acc = partial_merge(acc, fold_max_first(pc));
        }
        acc = warp_fold_max_first(acc);
        if (lane == 0 && !frozen) {
            const float s = acc.s;
            sm.conf[jj] = 1.0f / s;
            sm.ent[jj] = fmaxf(kLn2 * (log2f(s) - acc.u / s), 0.0f);
            sm.key[jj] = a.keep_rule == DG_KEEP_ENTROPY ? -sm.ent[jj] : sm.conf[jj];
            sm.arg[jj] = acc.idx;
            if (!(isfinite(s) && isfinite(acc.u) && isfinite(acc.mx) && s >= 1.0f - 1e-3f))
                flag_status(a.status, DG_ST_NONFINITE);
        }
    }

    if (!frozen) {
        if (tid < nrows) sm.old[tid] = old_tok;
        cluster_sync();  // every CTA's statistics are in its shared memory

        // this CTA's rows' statistics to the caller's arrays (and traces): after the barrier, so
        // that its release does not wait for these stores
        for (int jj = tid; jj < nrows; jj += kMergeThreads) {
            const int r = base + j0 + jj;
            a.argmax[r] = sm.arg[jj];
            a.conf[r] = sm.conf[jj];
            a.entropy[r] = sm.ent[jj];
            if (a.ctl) {
                const size_t tr = static_cast<size_t>(p) * a.R + r;
                if (a.trace_argmax) a.trace_argmax[tr] = sm.arg[jj];
                if (a.trace_conf) a.trace_conf[tr] = sm.conf[jj];
                if (a.trace_entropy) a.trace_entropy[tr] = sm.ent[jj];
            }
        }

        // gather the canvas's keep keys from the cluster; CTA 0 also sums the entropies with a
        // fixed-order tree: pairwise within each warp of 32 consecutive slots (xor butterfly),
        // then the per-warp sums in increasing order
        float ent_i = 0.0f;
        for (int i = tid; i < S; i += kMergeThreads) {
            const uint32_t owner = static_cast<uint32_t>(i / rpc);
            const int off = i - static_cast<int>(owner) * rpc;
            sm.all_key[i] = ld_cluster_f32(mapa_shared(smem_u32(&sm.key[off]), owner));
            if (c == 0) ent_i = ld_cluster_f32(mapa_shared(smem_u32(&sm.ent[off]), owner));
        }
        if (c == 0) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ent_i += __shfl_xor_sync(0xffffffffu, ent_i, off);
            if (lane == 0) sm.warp_ent[warp] = ent_i;
        }
        __syncthreads();

        uint32_t changed = 0;
        if (a.canvas_out) {
            long long K;
            if (a.keep_sched)
                K = a.keep_sched[p];
            else if (a.keep_k0 >= 0)
                K = static_cast<long long>(a.keep_k0) * (p + 1);
            else
                K = a.keep_k;
            K = K < 0 ? 0 : (K > S ? S : K);
            // tpr threads per slot (a power of two dividing 32) split the rank count
            const int rpow2 = max(1, 1 << (32 - __clz(max(nrows, 1) - 1)));
            int tpr = kMergeThreads / rpow2;
            tpr = tpr > 32 ? 32 : tpr;
            const int jj = tid / tpr, sub = tid % tpr;
            int rank = 0;
            const bool act = jj < nrows;
            const int j = j0 + jj;
            if (act) {
                const float cj = sm.all_key[j];
                for (int i = sub; i < S; i += tpr) {
                    const float ci = sm.all_key[i];
                    rank += (ci > cj) || (ci == cj && i < j);
                }
            }
            for (int off = 1; off < tpr; off <<= 1) rank += __shfl_xor_sync(0xffffffffu, rank, off);
            if (act && sub == 0) {
                const int r = base + j;
                const bool kp = rank < K;
                const int oldt = sm.old[jj];
                const int nw = kp ? sm.arg[jj] : sm.draw[jj];
                if (oldt < 0 || oldt >= a.V) flag_status(a.status, DG_ST_BAD_TOKEN);
                if (a.trace_canvas && a.ctl) a.trace_canvas[static_cast<size_t>(p) * a.R + r] = oldt;
                a.canvas_out[r] = nw;
                if (a.kept) a.kept[r] = kp ? 1 : 0;
                changed = (nw != oldt);
            }
        }
        changed = __syncthreads_or(changed);
        if (tid == 0) st_cluster_u32(mapa_shared(smem_u32(&sm.changed[c]), 0), changed);

        float meanH = 0.0f;
        if (c == 0) {
            const int nw = (S + 31) / 32;
            float sum = 0.0f;
            for (int i = 0; i < nw; ++i) sum += sm.warp_ent[i];
            meanH = sum / static_cast<float>(S);
        }
        cluster_sync();  // changed flags delivered; no CTA reads another's shared memory after this
        if (c != 0) {
            timeline_end(a.timeline, p, DG_TL_MERGE);
            return;
        }
        if (tid == 0) {
            if (a.mean_entropy) a.mean_entropy[b] = meanH;
            if (a.trace_mean_entropy && a.ctl) a.trace_mean_entropy[p * a.B + b] = meanH;
            if (a.canvas_out && a.state && a.has_rule) {
                uint32_t any = 0;
                for (int i = 0; i < kMergeCluster; ++i) any |= sm.changed[i];
                dg_canvas_state st = st0;
                st.stable = any ? 0 : st.stable + 1;
                const bool ent = meanH < a.rule.entropy_threshold;
                const bool stb = st.stable >= a.rule.stable_passes;
                const bool cap = p + 1 >= a.rule.max_passes;
                const bool stop =
                    (a.rule.stop_mode == DG_STOP_AND ? (ent && stb) : (ent || stb)) || cap;
                st.mean_entropy = meanH;
                st.last_pass = p;
                if (stop) {
                    st.done = 1;
                    st.passes = p + 1;
                    st.reason = (ent ? DG_REASON_ENTROPY : 0) | (stb ? DG_REASON_STABLE : 0) |
                                (cap ? DG_REASON_CAP : 0);
                }
                a.state[b] = st;
                my_done = st.done;
            }
        }
    }

    if (frozen && a.canvas_out && tid < nrows) {
        const int r = base + j0 + tid;
        if (a.canvas_out != a.canvas_in) a.canvas_out[r] = old_tok;
        // a stopped canvas enters every later pass unchanged: its canvas trace says so
        if (a.trace_canvas && a.ctl) a.trace_canvas[static_cast<size_t>(p) * a.R + r] = old_tok;
    }

    // loop mode: the last canvas of the pass advances the pass and sets the graph condition
    if (a.ctl && c == 0 && tid == 0) {
        unsigned t = 0;
        if (a.B > 1) {
            __threadfence();
            t = atomicAdd(&a.ctl->ticket, 1u);
        }
        if (t == static_cast<unsigned>(a.B) - 1u) {
            if (a.B > 1) __threadfence();
            int all_done = a.state != nullptr ? my_done : 0;
            if (a.state != nullptr && a.B > 1)
                for (int bb = 0; bb < a.B; ++bb)
                    all_done &= (*reinterpret_cast<volatile int*>(&a.state[bb].done) != 0);
            a.ctl->ticket = 0;
            const int np = p + 1;
            a.ctl->pass = np;
            // the condition is 1 at every graph launch; it is only ever set to stop the loop
            if (all_done || np >= max_passes) {
                a.ctl->stop = 1;
                if (a.set_cond) cudaGraphSetConditional(a.cond, 0u);
            }
        }
    }
    timeline_end(a.timeline, p, DG_TL_MERGE);
}

// Block-wide max of a non-negative value (blockDim.x a multiple of 32, at most 1024).
__device__ __forceinline__ float block_max(float v, float* red) {
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    __syncthreads();  // `red` may still be in use by a previous reduction
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x < 32) {
        float m = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (threadIdx.x == 0) red[0] = m;
    }
    __syncthreads();
    return red[0];
}

// E4M3 codes of one bf16 row given its absmax: amax = 0 gives scale 1 and all-zero codes,
// otherwise inv = fp32(448 / amax), q_k = e4m3_rn_satfinite(fp32(h_k * inv)), scale = amax / 448.
__device__ __forceinline__ void quant_row(const __nv_bfloat16* hr, int d, float amax, uint8_t* qr,
                                          float* scale) {
    if (amax == 0.f) {
        for (int k = threadIdx.x; k < d; k += blockDim.x) qr[k] = 0;
        if (threadIdx.x == 0) *scale = 1.0f;
        return;
    }
    const float inv = __fdiv_rn(448.0f, amax);
    for (int k = threadIdx.x; k < d; k += blockDim.x) {
        const float x = __fmul_rn(__bfloat162float(hr[k]), inv);
        qr[k] = static_cast<uint8_t>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3));
    }
    if (threadIdx.x == 0) *scale = __fdiv_rn(amax, 448.0f);
}

__global__ void quant_rows_kernel(const __nv_bfloat16* __restrict__ h, int d, uint8_t* __restrict__ q,
                                  float* __restrict__ scale, uint32_t* status) {
    __shared__ float red[32];
    grid_dependency_wait();
    grid_launch_dependents();
    const int r = blockIdx.x;
    const __nv_bfloat16* hr = h + static_cast<size_t>(r) * d;
    float amax = 0.f;
    bool bad = false;
    for (int k = threadIdx.x; k < d; k += blockDim.x) {
        const float v = __bfloat162float(hr[k]);
        bad |= !isfinite(v);
        amax = fmaxf(amax, fabsf(v));
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) flag_status(status, DG_ST_NONFINITE);
    amax = block_max(amax, red);
    quant_row(hr, d, amax, q + static_cast<size_t>(r) * d, scale + r);
}

__global__ void loop_init_kernel(int32_t* canvas, int S, int V, uint64_t seed, int init_random,
                                 int mask_id, uint64_t row_offset, dg_canvas_state* state,
                                 int keep_stable, LoopCtl* ctl, int start_pass, int max_passes,
                                 uint32_t* status, unsigned long long* timeline) {
    const int b = blockIdx.x;
    if (timeline)
        for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < max_passes * DG_TL_KERNELS;
             i += gridDim.x * blockDim.x) {
            timeline[2 * i] = ~0ull;
            timeline[2 * i + 1] = 0ull;
        }
    for (int j = threadIdx.x; j < S; j += blockDim.x) {
        const int r = b * S + j;
        if (init_random == 2) {
            canvas[r] = mask_id;
        } else if (init_random) {
            canvas[r] = static_cast<int32_t>(
                draw_key(seed, kInitPass, row_offset + static_cast<uint64_t>(r)) %
                static_cast<uint64_t>(V));
        } else {
            const int c = canvas[r];
            if (c < 0 || c >= V) flag_status(status, DG_ST_BAD_TOKEN);
        }
    }
    if (threadIdx.x == 0) {
        dg_canvas_state st;
        st.passes = 0;
        st.reason = 0;
        st.stable = keep_stable ? state[b].stable : 0;
        st.done = 0;
        st.mean_entropy = __int_as_float(0x7fc00000);
        st.last_pass = -1;
        st.reserved[0] = st.reserved[1] = 0;
        state[b] = st;
        if (b == 0) {
            ctl->pass = start_pass;
            ctl->ticket = 0;
            ctl->max_passes = max_passes;
            ctl->stop = 0;
            ctl->row_offset = row_offset;
        }
    }
}

__global__ void trace_copy_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                  size_t bytes, const LoopCtl* ctl) {
    if (ctl->stop != 0) return;
    uint8_t* out = dst + static_cast<size_t>(ctl->pass) * bytes;
    const size_t n16 = bytes / 16;
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(out);
    for (size_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += gridDim.x * blockDim.x)
        d4[i] = s4[i];
    for (size_t i = n16 * 16 + blockIdx.x * blockDim.x + threadIdx.x; i < bytes;
         i += gridDim.x * blockDim.x)
        out[i] = src[i];
}

__device__ __forceinline__ float head_value(int dtype, const void* w, const float* ws, int64_t row,
                                            int64_t d, int64_t k) {
    if (dtype == DG_BF16)
        return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(w)[row * d + k]);
    if (dtype == DG_E4M3) {
        __nv_fp8_e4m3 q;
        q.__x = reinterpret_cast<const uint8_t*>(w)[row * d + k];
        return static_cast<float>(q) * ws[row];
    }
    return reinterpret_cast<const float*>(w)[row * d + k];
}

__global__ void synth_denoise_kernel(int dtype, const void* __restrict__ w, const float* ws, int S,
                                     int d, int V, const int32_t* __restrict__ y, int n_content,
                                     float s_content, float s_pad, const int32_t* __restrict__ canvas,
                                     const int32_t* __restrict__ pass, __nv_bfloat16* __restrict__ h,
                                     uint32_t* status, uint8_t* __restrict__ q,
                                     float* __restrict__ qscale, unsigned long long* timeline,
                                     const int32_t* stop) {
    __shared__ float red[32];
    grid_dependency_wait();
    grid_launch_dependents();
    if (stop != nullptr && *stop != 0) return;
    const int r = blockIdx.x;
    const int t = pass[0] + 1;
    timeline_begin(timeline, t - 1, DG_TL_DENOISE);
    const float at = fminf(1.0f, __fdiv_rn(static_cast<float>(2 + t), 10.0f));
    const float bt = 1.0f - at;
    const int yy = y[r], cc = canvas[r];
    __nv_bfloat16* hr = h + static_cast<size_t>(r) * d;
    if (yy < 0 || yy >= V || cc < 0 || cc >= V) {
        if (threadIdx.x == 0) flag_status(status, DG_ST_BAD_TOKEN);
        for (int k = threadIdx.x; k < d; k += blockDim.x) hr[k] = __float2bfloat16_rn(0.f);
        if (q) {
            for (int k = threadIdx.x; k < d; k += blockDim.x) q[static_cast<size_t>(r) * d + k] = 0;
            if (threadIdx.x == 0) qscale[r] = 1.0f;
        }
        timeline_end(timeline, t - 1, DG_TL_DENOISE);
        return;
    }
    float n2 = 0.f;
    for (int k = threadIdx.x; k < d; k += blockDim.x) {
        const float x = at * head_value(dtype, w, ws, yy, d, k) + bt * head_value(dtype, w, ws, cc, d, k);
        n2 = fmaf(x, x, n2);
    }
    for (int o = 16; o > 0; o >>= 1) n2 += __shfl_xor_sync(0xffffffffu, n2, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = n2;
    __syncthreads();
    if (threadIdx.x < 32) {
        float m = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
        for (int o = 16; o > 0; o >>= 1) m += __shfl_xor_sync(0xffffffffu, m, o);
        if (threadIdx.x == 0) red[0] = m;
    }
    __syncthreads();
    n2 = red[0];
    const float s = (r % S) < n_content ? s_content : s_pad;
    const float inv = n2 > 0.f ? s / sqrtf(n2) : 0.f;
    float amax = 0.f;
    bool bad = false;
    for (int k = threadIdx.x; k < d; k += blockDim.x) {
        const float x = at * head_value(dtype, w, ws, yy, d, k) + bt * head_value(dtype, w, ws, cc, d, k);
        const __nv_bfloat16 hb = __float2bfloat16_rn(x * inv);
        hr[k] = hb;
        const float v = __bfloat162float(hb);
        bad |= !isfinite(v);
        amax = fmaxf(amax, fabsf(v));
    }
    if (q) {
        if (__syncthreads_or(bad) && threadIdx.x == 0) flag_status(status, DG_ST_NONFINITE);
        // the row's own bf16 values, written above by this CTA, are visible after the barrier
        // inside block_max
        amax = block_max(amax, red);
        quant_row(hr, d, amax, q + static_cast<size_t>(r) * d, qscale + r);
    }
    timeline_end(timeline, t - 1, DG_TL_DENOISE);
}

// Vectorised synthetic denoiser (same arithmetic as synth_denoise_kernel): one CTA of
// kDenThreads per row; thread t holds 16-byte chunks t, t + kDenThreads, ... of both head rows
// (ES-byte elements: 2 = bf16, 1 = E4M3 codes), so the mixed row x stays in registers between the
// norm, the bf16 write and the optional E4M3 quantisation.
constexpr int kDenThreads = 128;

template <int ES>
__device__ __forceinline__ void unpack16(const uint4& v, float scale, float (&out)[16 / ES]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    if constexpr (ES == 2) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            out[2 * i] = __uint_as_float(w[i] << 16);
            out[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(
                static_cast<__nv_fp8x2_storage_t>(w[i] & 0xFFFFu), __NV_E4M3);
            const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(
                static_cast<__nv_fp8x2_storage_t>(w[i] >> 16), __NV_E4M3);
            const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
            const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
            out[4 * i] = a.x * scale;
            out[4 * i + 1] = a.y * scale;
            out[4 * i + 2] = b.x * scale;
            out[4 * i + 3] = b.y * scale;
        }
    }
}

__device__ __forceinline__ float block_sum128(float v, float* red) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    return (red[0] + red[1]) + (red[2] + red[3]);
}

__device__ __forceinline__ float block_max128(float v, float* red) {
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if ((threadIdx.x & 31) == 0) red[4 + (threadIdx.x >> 5)] = v;
    __syncthreads();
    return fmaxf(fmaxf(red[4], red[5]), fmaxf(red[6], red[7]));
}

template <int ES, int MAXC>
__global__ void __launch_bounds__(kDenThreads)
    synth_denoise_vec_kernel(const uint8_t* __restrict__ w, const float* __restrict__ ws, int S,
                             int d, int V, const int32_t* __restrict__ y, int n_content,
                             float s_content, float s_pad, const int32_t* __restrict__ canvas,
                             const int32_t* __restrict__ pass, __nv_bfloat16* __restrict__ h,
                             uint32_t* status, uint8_t* __restrict__ q, float* __restrict__ qscale,
                             unsigned long long* timeline, const int32_t* stop) {
    constexpr int EPC = 16 / ES;  // elements per 16-byte chunk
    __shared__ float red[8];
    grid_dependency_wait();
    grid_launch_dependents();
    if (stop != nullptr && *stop != 0) return;
    const int r = blockIdx.x;
    const int tid = threadIdx.x;
    const int t = pass[0] + 1;
    timeline_begin(timeline, t - 1, DG_TL_DENOISE);
    const int yy = y[r], cc = canvas[r];
    const float at = fminf(1.0f, __fdiv_rn(static_cast<float>(2 + t), 10.0f));
    const float bt = 1.0f - at;
    __nv_bfloat16* hr = h + static_cast<size_t>(r) * d;
    const int nch = d / EPC;
    if (yy < 0 || yy >= V || cc < 0 || cc >= V) {
        if (tid == 0) flag_status(status, DG_ST_BAD_TOKEN);
        for (int k = tid; k < d; k += kDenThreads) hr[k] = __float2bfloat16_rn(0.f);
        if (q) {
            for (int k = tid; k < d; k += kDenThreads) q[static_cast<size_t>(r) * d + k] = 0;
            if (tid == 0) qscale[r] = 1.0f;
        }
        timeline_end(timeline, t - 1, DG_TL_DENOISE);
        return;
    }
    const uint4* wy = reinterpret_cast<const uint4*>(w + static_cast<size_t>(yy) * d * ES);
    const uint4* wc = reinterpret_cast<const uint4*>(w + static_cast<size_t>(cc) * d * ES);
    uint4 vy[MAXC], vc[MAXC];
#pragma unroll
    for (int i = 0; i < MAXC; ++i) {
        const int ch = tid + i * kDenThreads;
        if (ch < nch) {
            vy[i] = __ldg(wy + ch);
            vc[i] = __ldg(wc + ch);
        }
    }
    const float sy = ES == 1 ? ws[yy] : 1.0f, sc = ES == 1 ? ws[cc] : 1.0f;
    float x[MAXC][EPC];
    float n2 = 0.f;
#pragma unroll
    for (int i = 0; i < MAXC; ++i) {
        const int ch = tid + i * kDenThreads;
        if (ch < nch) {
            float a[EPC], b[EPC];
            unpack16<ES>(vy[i], sy, a);
            unpack16<ES>(vc[i], sc, b);
#pragma unroll
            for (int e = 0; e < EPC; ++e) {
                x[i][e] = at * a[e] + bt * b[e];
                n2 = fmaf(x[i][e], x[i][e], n2);
            }
        }
    }
    n2 = block_sum128(n2, red);
    const float s = (r % S) < n_content ? s_content : s_pad;
    const float inv = n2 > 0.f ? s / sqrtf(n2) : 0.f;
    float amax = 0.f;
    bool bad = false;
#pragma unroll
    for (int i = 0; i < MAXC; ++i) {
        const int ch = tid + i * kDenThreads;
        if (ch < nch) {
            uint32_t packed[EPC / 2];
#pragma unroll
            for (int e = 0; e < EPC; e += 2) {
                const __nv_bfloat16 h0 = __float2bfloat16_rn(x[i][e] * inv);
                const __nv_bfloat16 h1 = __float2bfloat16_rn(x[i][e + 1] * inv);
                x[i][e] = __bfloat162float(h0);  // keep the rounded value for the quantiser
                x[i][e + 1] = __bfloat162float(h1);
                bad |= !isfinite(x[i][e]) || !isfinite(x[i][e + 1]);
                amax = fmaxf(amax, fmaxf(fabsf(x[i][e]), fabsf(x[i][e + 1])));
                packed[e / 2] = static_cast<uint32_t>(__bfloat16_as_ushort(h0)) |
                                (static_cast<uint32_t>(__bfloat16_as_ushort(h1)) << 16);
            }
            uint4* dst = reinterpret_cast<uint4*>(hr + static_cast<size_t>(ch) * EPC);
#pragma unroll
            for (int v = 0; v < EPC / 8; ++v)
                dst[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
        }
    }
    if (!q) {
        timeline_end(timeline, t - 1, DG_TL_DENOISE);
        return;
    }
    if (__syncthreads_or(bad) && tid == 0) flag_status(status, DG_ST_NONFINITE);
    amax = block_max128(amax, red);
    uint8_t* qr = q + static_cast<size_t>(r) * d;
    const float qinv = amax == 0.f ? 0.f : __fdiv_rn(448.0f, amax);
#pragma unroll
    for (int i = 0; i < MAXC; ++i) {
        const int ch = tid + i * kDenThreads;
        if (ch < nch) {
            uint32_t codes[EPC / 4];
#pragma unroll
            for (int e = 0; e < EPC; e += 4) {
                uint32_t c4 = 0;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t cu = amax == 0.f ? 0u
                        : static_cast<uint32_t>(__nv_cvt_float_to_fp8(__fmul_rn(x[i][e + u], qinv),
                                                                      __NV_SATFINITE, __NV_E4M3));
                    c4 |= cu << (8 * u);
                }
                codes[e / 4] = c4;
            }
            if constexpr (EPC == 16) {
                reinterpret_cast<uint4*>(qr)[ch] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
            } else {
                reinterpret_cast<uint2*>(qr)[ch] = make_uint2(codes[0], codes[1]);
            }
        }
    }
    if (tid == 0) qscale[r] = amax == 0.f ? 1.0f : __fdiv_rn(amax, 448.0f);
    timeline_end(timeline, t - 1, DG_TL_DENOISE);
}

}  // namespace

cudaError_t launch_select(const SelectArgs& a, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.B) * kMergeCluster);
    cfg.blockDim = dim3(kMergeThreads);
    cfg.stream = stream;
    // Programmatic dependent launch: the merge grid may be scheduled while the head kernel
    // drains; griddepcontrol.wait at its top orders every read after the head's writes.
    cudaLaunchAttribute attr[1];
    set_pdl_attr(&attr[0]);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, merge_select_kernel, a);
}

cudaError_t launch_quant_rows(const uint16_t* h, int R, int d, uint8_t* q, float* scale,
                              uint32_t* status, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(R);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    set_pdl_attr(&attr[0]);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, quant_rows_kernel, reinterpret_cast<const __nv_bfloat16*>(h), d,
                              q, scale, status);
}

// Self-test of the bounded waits: one thread waits on an mbarrier that nothing ever arrives on,
// with the same wait the head kernels use. It gives up after the wall-time bound (kWaitNs), sets
// DG_ST_TIMEOUT and returns, as a head kernel does when a wait of one of its roles runs out.
__global__ void wait_selftest_kernel(uint32_t* status) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    if (!mbar_wait(&bar, 0)) flag_status(status, DG_ST_TIMEOUT);
}

cudaError_t launch_wait_selftest(uint32_t* status, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(status);
    return cudaGetLastError();
}

cudaError_t launch_loop_init(int32_t* canvas, int R, int S, int B, int V, uint64_t seed,
                             int init_random, int mask_id, uint64_t row_offset,
                             dg_canvas_state* state, int keep_stable, LoopCtl* ctl,
                             int start_pass, int max_passes, uint32_t* status,
                             unsigned long long* timeline, cudaStream_t stream) {
    (void)R;
    loop_init_kernel<<<B, 256, 0, stream>>>(canvas, S, V, seed, init_random, mask_id, row_offset,
                                            state, keep_stable, ctl, start_pass, max_passes,
                                            status, timeline);
    return cudaGetLastError();
}

cudaError_t launch_trace_copy(const void* src, void* dst, size_t bytes, const LoopCtl* ctl,
                              cudaStream_t stream) {
    trace_copy_kernel<<<148, 256, 0, stream>>>(reinterpret_cast<const uint8_t*>(src),
                                               reinterpret_cast<uint8_t*>(dst), bytes, ctl);
    return cudaGetLastError();
}

cudaError_t launch_synth_denoise(const dg_head_desc* desc, const int32_t* y, int n_content,
                                 float s_content, float s_pad, const int32_t* canvas,
                                 const int32_t* pass, uint16_t* h_out, uint32_t* status,
                                 cudaStream_t stream, uint8_t* q_out, float* scale_out,
                                 unsigned long long* timeline, const int32_t* stop) {
    const int R = desc->B * desc->S;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(R);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    set_pdl_attr(&attr[0]);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    constexpr int MAXC = 4;
    const int es = desc->w_dtype == DG_BF16 ? 2 : 1;
    const long long chunks = static_cast<long long>(desc->d) * es / 16;  // d * es % 16 == 0
    auto hb = reinterpret_cast<__nv_bfloat16*>(h_out);
    auto wb = static_cast<const uint8_t*>(desc->w);
    if ((desc->w_dtype == DG_BF16 || desc->w_dtype == DG_E4M3) &&
        chunks <= static_cast<long long>(MAXC) * kDenThreads) {
        cfg.blockDim = dim3(kDenThreads);
        if (es == 2)
            return cudaLaunchKernelEx(&cfg, synth_denoise_vec_kernel<2, MAXC>, wb, desc->w_scale,
                                      static_cast<int>(desc->S), static_cast<int>(desc->d),
                                      static_cast<int>(desc->V), y, n_content, s_content, s_pad,
                                      canvas, pass, hb, status, q_out, scale_out, timeline, stop);
        return cudaLaunchKernelEx(&cfg, synth_denoise_vec_kernel<1, MAXC>, wb, desc->w_scale,
                                  static_cast<int>(desc->S), static_cast<int>(desc->d),
                                  static_cast<int>(desc->V), y, n_content, s_content, s_pad, canvas,
                                  pass, hb, status, q_out, scale_out, timeline, stop);
    }
    cfg.blockDim = dim3(256);
    return cudaLaunchKernelEx(&cfg, synth_denoise_kernel, static_cast<int>(desc->w_dtype),
                              desc->w, desc->w_scale, static_cast<int>(desc->S),
                              static_cast<int>(desc->d), static_cast<int>(desc->V), y, n_content,
                              s_content, s_pad, canvas, pass, hb, status, q_out, scale_out, timeline, stop);
}

}  // namespace dg
