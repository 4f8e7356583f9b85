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

namespace dg {
namespace {

__device__ __forceinline__ Partial shfl_xor_partial(const Partial& p, int off) {
    Partial q;
    q.mx = __shfl_xor_sync(0xffffffffu, p.mx, off);
    q.s = __shfl_xor_sync(0xffffffffu, p.s, off);
    q.u = __shfl_xor_sync(0xffffffffu, p.u, off);
    q.idx = __shfl_xor_sync(0xffffffffu, p.idx, off);
    return q;
}

// Wait until the grid this launch depends on (the head kernel, when launched as a programmatic
// dependent) has completed and its memory is visible. A no-op for a normal launch.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

constexpr int kMergeWarps = 16;            // slot rows merged per CTA (one warp per row)
constexpr int kMergeThreads = kMergeWarps * 32;

// Per-canvas part of a pass, run by the last CTA of the canvas to finish its rows:
// mean entropy (fixed-order pairwise tree over the slots), rank by (confidence desc, slot asc),
// keep the top K at their argmax, re-draw the rest with the counter key, stop rules.
__device__ void canvas_tail(const SelectArgs& a, int b, int p, bool frozen, float* sh_red,
                            float* sh_conf, int rows_pow2) {
    const int tid = threadIdx.x;
    const int base = b * a.S;
    if (frozen) {
        if (a.canvas_out && a.canvas_out != a.canvas_in)
            for (int j = tid; j < a.S; j += blockDim.x) a.canvas_out[base + j] = a.canvas_in[base + j];
        return;
    }
    // statistics of the canvas's rows, written by every CTA of the canvas (L2, not L1)
    for (int j = tid; j < rows_pow2; j += blockDim.x) {
        sh_red[j] = j < a.S ? __ldcg(a.entropy + base + j) : 0.0f;
        sh_conf[j] = j < a.S ? __ldcg(a.conf + base + j) : 0.0f;
    }
    __syncthreads();
    for (int off = rows_pow2 >> 1; off > 0; off >>= 1) {
        for (int j = tid; j < off; j += blockDim.x) sh_red[j] += sh_red[j + off];
        __syncthreads();
    }
    const float meanH = sh_red[0] / static_cast<float>(a.S);
    if (tid == 0 && a.mean_entropy) a.mean_entropy[b] = meanH;
    if (tid == 0 && a.trace_mean_entropy && a.ctl) a.trace_mean_entropy[p * a.B + b] = meanH;
    if (!a.canvas_out) return;

    long long K;
    if (a.keep_sched)
        K = a.keep_sched[p];
    else if (a.keep_k0 >= 0)
        K = static_cast<long long>(a.keep_k0) * (p + 1);
    else
        K = a.keep_k;
    K = K < 0 ? 0 : (K > a.S ? a.S : K);

    // tpr threads per slot (a power of two dividing 32) split the rank count
    int tpr = static_cast<int>(blockDim.x) / rows_pow2;
    tpr = tpr < 1 ? 1 : (tpr > 8 ? 8 : tpr);
    const int sub = tid % tpr;
    const int slots_per_round = static_cast<int>(blockDim.x) / tpr;
    int changed = 0;
    for (int j0 = 0; j0 < rows_pow2; j0 += slots_per_round) {
        const int j = j0 + tid / tpr;
        const bool act = j < a.S;
        const float cj = act ? sh_conf[j] : 0.0f;
        int rank = 0;
        if (act)
            for (int i = sub; i < a.S; i += tpr) {
                const float ci = sh_conf[i];
                rank += (ci > cj) || (ci == cj && i < j);
            }
        for (int off = 1; off < tpr; off <<= 1) rank += __shfl_xor_sync(0xffffffffu, rank, off);
        if (act && sub == 0) {
            const int r = base + j;
            const bool kp = rank < K;
            const int old = a.canvas_in[r];
            const int nw = kp ? __ldcg(a.argmax + r)
                              : static_cast<int>(draw_key(a.seed, static_cast<uint32_t>(p),
                                                          static_cast<uint64_t>(r)) %
                                                 static_cast<uint64_t>(a.V));
            if (old < 0 || old >= a.V) flag_status(a.status, DG_ST_BAD_TOKEN);
            if (a.trace_canvas && a.ctl) a.trace_canvas[static_cast<size_t>(p) * a.R + r] = old;
            a.canvas_out[r] = nw;
            if (a.kept) a.kept[r] = kp ? 1 : 0;
            changed |= (nw != old);
        }
    }
    changed = __syncthreads_or(changed);
    if (tid == 0 && a.state && a.has_rule) {
        dg_canvas_state st = a.state[b];
        st.stable = changed ? 0 : st.stable + 1;
        const bool ent = meanH < a.rule.entropy_threshold;
        const bool stb = st.stable >= a.rule.stable_passes;
        const bool cap = p + 1 >= a.rule.max_passes;
        const bool stop = (a.rule.stop_mode == DG_STOP_AND ? (ent && stb) : (ent || stb)) || cap;
        st.mean_entropy = meanH;
        st.last_pass = p;
        if (stop) {
            st.done = 1;
            st.passes = p + 1;
            st.reason = (ent ? DG_REASON_ENTROPY : 0) | (stb ? DG_REASON_STABLE : 0) |
                        (cap ? DG_REASON_CAP : 0);
        }
        a.state[b] = st;
    }
}

// Grid: B x ceil(S / kMergeWarps) CTAs of kMergeThreads. Warp w of CTA (b, x) merges the
// vocabulary-group partials of slot x * kMergeWarps + w of canvas b: lane l takes groups
// l, l + 32, ... in increasing order, then the lanes combine with a fixed xor butterfly (lower
// lane first), so every run merges in the same order and all lanes end with the same result.
// The last CTA of a canvas to arrive (arrival counter in a.tickets) runs the canvas tail; in
// loop mode the last canvas tail of the pass advances the pass and sets the graph condition.
__global__ void __launch_bounds__(kMergeThreads) merge_select_kernel(const SelectArgs a,
                                                                      int ctas_per_canvas) {
    extern __shared__ float sh[];  // [2 * rows_pow2]: entropy tree, confidences
    __shared__ int sh_last;
    grid_dependency_wait();
    const int rows_pow2 = max(32, 1 << (32 - __clz(a.S - 1)));
    const int b = blockIdx.x / ctas_per_canvas;
    const int x = blockIdx.x % ctas_per_canvas;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j = x * kMergeWarps + warp;
    const int p = a.ctl ? a.ctl->pass : static_cast<int>(a.pass);
    const bool frozen = a.state != nullptr && a.state[b].done != 0;

    if (!frozen && j < a.S) {
        const int r = b * a.S + j;
        const float4* q = a.partials + static_cast<size_t>(r) * a.n_groups;
        Partial acc = partial_empty();
        int g = lane;
        for (; g + 96 < a.n_groups; g += 128) {
            const float4 v0 = __ldcg(q + g), v1 = __ldcg(q + g + 32), v2 = __ldcg(q + g + 64),
                         v3 = __ldcg(q + g + 96);
            acc = partial_merge(acc, unpack(v0));
            acc = partial_merge(acc, unpack(v1));
            acc = partial_merge(acc, unpack(v2));
            acc = partial_merge(acc, unpack(v3));
        }
        for (; g < a.n_groups; g += 32) acc = partial_merge(acc, unpack(__ldcg(q + g)));
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const Partial o = shfl_xor_partial(acc, off);
            acc = (lane & off) ? partial_merge(o, acc) : partial_merge(acc, o);
        }
        if (lane == 0) {
            const float s = acc.s;
            const float conf = 1.0f / s;
            const float H = fmaxf(kLn2 * (log2f(s) - acc.u / s), 0.0f);
            if (!(isfinite(s) && isfinite(acc.u) && isfinite(acc.mx) && s >= 1.0f - 1e-3f))
                flag_status(a.status, DG_ST_NONFINITE);
            a.argmax[r] = acc.idx;
            a.conf[r] = conf;
            a.entropy[r] = H;
            if (a.ctl) {
                const size_t tr = static_cast<size_t>(p) * a.R + r;
                if (a.trace_argmax) a.trace_argmax[tr] = acc.idx;
                if (a.trace_conf) a.trace_conf[tr] = conf;
                if (a.trace_entropy) a.trace_entropy[tr] = H;
            }
        }
    }

    // arrival: the last CTA of canvas b (in arrival order) sees every row's statistics
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned t = atomicAdd(&a.tickets[b], 1u);
        sh_last = (t == static_cast<unsigned>(ctas_per_canvas) - 1u);
        if (sh_last) {
            a.tickets[b] = 0;  // ready for the next pass
            __threadfence();
        }
    }
    __syncthreads();
    if (!sh_last) return;
    canvas_tail(a, b, p, frozen, sh, sh + rows_pow2, rows_pow2);

    // loop mode: the last canvas tail of the pass advances the pass and sets the graph condition
    if (a.ctl) {
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            const unsigned t = atomicAdd(&a.ctl->ticket, 1u);
            if (t == static_cast<unsigned>(a.B) - 1u) {
                __threadfence();
                int all_done = 1;
                if (a.state)
                    for (int bb = 0; bb < a.B; ++bb)
                        all_done &= (*reinterpret_cast<volatile int*>(&a.state[bb].done) != 0);
                else
                    all_done = 0;
                a.ctl->ticket = 0;
                const int np = p + 1;
                a.ctl->pass = np;
                if (a.set_cond)
                    cudaGraphSetConditional(a.cond, (!all_done && np < a.ctl->max_passes) ? 1u : 0u);
            }
        }
    }
}

__global__ void quant_rows_kernel(const __nv_bfloat16* __restrict__ h, int d, uint8_t* __restrict__ q,
                                  float* __restrict__ scale, uint32_t* status) {
    __shared__ float red[32];
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
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    if (threadIdx.x < 32) {
        float m = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (threadIdx.x == 0) red[0] = m;
    }
    __syncthreads();
    amax = red[0];
    uint8_t* qr = q + static_cast<size_t>(r) * d;
    if (amax == 0.f) {
        for (int k = threadIdx.x; k < d; k += blockDim.x) qr[k] = 0;
        if (threadIdx.x == 0) scale[r] = 1.0f;
        return;
    }
    const float inv = __fdiv_rn(448.0f, amax);
    for (int k = threadIdx.x; k < d; k += blockDim.x) {
        const float x = __fmul_rn(__bfloat162float(hr[k]), inv);
        qr[k] = static_cast<uint8_t>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3));
    }
    if (threadIdx.x == 0) scale[r] = __fdiv_rn(amax, 448.0f);
}

__global__ void loop_init_kernel(int32_t* canvas, int S, int V, uint64_t seed, int init_random,
                                 dg_canvas_state* state, int keep_stable, LoopCtl* ctl,
                                 int start_pass, int max_passes, uint32_t* status) {
    const int b = blockIdx.x;
    for (int j = threadIdx.x; j < S; j += blockDim.x) {
        const int r = b * S + j;
        if (init_random) {
            canvas[r] = static_cast<int32_t>(draw_key(seed, kInitPass, static_cast<uint64_t>(r)) %
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
        }
    }
}

__global__ void trace_copy_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                  size_t bytes, const LoopCtl* ctl) {
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
                                     uint32_t* status) {
    __shared__ float red[32];
    const int r = blockIdx.x;
    const int t = pass[0] + 1;
    const float at = fminf(1.0f, __fdiv_rn(static_cast<float>(2 + t), 10.0f));
    const float bt = 1.0f - at;
    const int yy = y[r], cc = canvas[r];
    __nv_bfloat16* hr = h + static_cast<size_t>(r) * d;
    if (yy < 0 || yy >= V || cc < 0 || cc >= V) {
        if (threadIdx.x == 0) flag_status(status, DG_ST_BAD_TOKEN);
        for (int k = threadIdx.x; k < d; k += blockDim.x) hr[k] = __float2bfloat16_rn(0.f);
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
    for (int k = threadIdx.x; k < d; k += blockDim.x) {
        const float x = at * head_value(dtype, w, ws, yy, d, k) + bt * head_value(dtype, w, ws, cc, d, k);
        hr[k] = __float2bfloat16_rn(x * inv);
    }
}

int pow2_at_least(int x) {
    int p = 32;
    while (p < x) p <<= 1;
    return p;
}

}  // namespace

cudaError_t launch_select(const SelectArgs& a, cudaStream_t stream) {
    const int rows = pow2_at_least(a.S);  // 32 .. 1024
    const int cpc = (a.S + kMergeWarps - 1) / kMergeWarps;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(static_cast<long long>(a.B) * cpc));
    cfg.blockDim = dim3(kMergeThreads);
    cfg.dynamicSmemBytes = 2 * rows * sizeof(float);
    cfg.stream = stream;
    // Programmatic dependent launch: the merge grid may be scheduled while the head kernel
    // drains; griddepcontrol.wait at its top orders every read after the head's writes.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, merge_select_kernel, a, cpc);
}

cudaError_t launch_quant_rows(const uint16_t* h, int R, int d, uint8_t* q, float* scale,
                              uint32_t* status, cudaStream_t stream) {
    quant_rows_kernel<<<R, 256, 0, stream>>>(reinterpret_cast<const __nv_bfloat16*>(h), d, q, scale,
                                             status);
    return cudaGetLastError();
}

cudaError_t launch_loop_init(int32_t* canvas, int R, int S, int B, int V, uint64_t seed,
                             int init_random, dg_canvas_state* state, int keep_stable, LoopCtl* ctl,
                             int start_pass, int max_passes, uint32_t* status, cudaStream_t stream) {
    (void)R;
    loop_init_kernel<<<B, 256, 0, stream>>>(canvas, S, V, seed, init_random, state, keep_stable, ctl,
                                            start_pass, max_passes, status);
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
                                 cudaStream_t stream) {
    const int R = desc->B * desc->S;
    synth_denoise_kernel<<<R, 256, 0, stream>>>(desc->w_dtype, desc->w, desc->w_scale, desc->S,
                                                desc->d, desc->V, y, n_content, s_content, s_pad,
                                                canvas, pass,
                                                reinterpret_cast<__nv_bfloat16*>(h_out), status);
    return cudaGetLastError();
}

}  // namespace dg
