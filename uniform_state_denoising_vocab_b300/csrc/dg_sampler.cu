// dg_sampler.cu -- the per-canvas part of a pass and the loop plumbing:
//   select_kernel   merge the vocabulary-group partials of every slot into argmax, confidence
//                   and entropy; per canvas: mean entropy (fixed-order tree), rank slots by
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

// One CTA per canvas, `tpr` (1..8, a power of two) consecutive threads per slot row:
// the threads of a row merge disjoint, strided subsets of the vocabulary-group partials with
// their loads batched, then combine them with a fixed xor butterfly (lower sub-lane first), so
// every run merges in the same order.
__global__ void __launch_bounds__(1024) select_kernel(const SelectArgs a, int tpr) {
    extern __shared__ float sh[];  // [2 * rows_pow2]: reduction scratch, confidences
    const int rows_pow2 = blockDim.x / tpr;
    float* sh_red = sh;
    float* sh_conf = sh + rows_pow2;
    const int b = blockIdx.x;
    const int j = threadIdx.x / tpr;       // slot
    const int sub = threadIdx.x % tpr;
    const bool act = j < a.S;
    const int r = b * a.S + j;
    const int p = a.ctl ? a.ctl->pass : static_cast<int>(a.pass);

    const bool frozen = a.state != nullptr && a.state[b].done != 0;
    if (frozen) {
        if (act && sub == 0 && a.canvas_out && a.canvas_out != a.canvas_in)
            a.canvas_out[r] = a.canvas_in[r];
    } else {
        // ---- merge the partials of this row ----
        Partial acc = partial_empty();
        if (act) {
            const size_t stride = static_cast<size_t>(a.R) * tpr;
            int g = sub;
            const float4* q = a.partials + r + static_cast<size_t>(g) * a.R;
            for (; g + 3 * tpr < a.n_groups; g += 4 * tpr, q += 4 * stride) {
                const float4 v0 = __ldg(q), v1 = __ldg(q + stride), v2 = __ldg(q + 2 * stride),
                             v3 = __ldg(q + 3 * stride);
                acc = partial_merge(acc, unpack(v0));
                acc = partial_merge(acc, unpack(v1));
                acc = partial_merge(acc, unpack(v2));
                acc = partial_merge(acc, unpack(v3));
            }
            for (; g < a.n_groups; g += tpr, q += stride) acc = partial_merge(acc, unpack(__ldg(q)));
        }
        for (int off = 1; off < tpr; off <<= 1) {
            const Partial o = shfl_xor_partial(acc, off);
            acc = (sub & off) ? partial_merge(o, acc) : partial_merge(acc, o);
        }
        const float s = acc.s;
        const float conf = 1.0f / s;
        float H = kLn2 * (log2f(s) - acc.u / s);
        H = fmaxf(H, 0.0f);
        if (act && sub == 0) {
            if (!(isfinite(s) && isfinite(acc.u) && isfinite(acc.mx) && s >= 1.0f - 1e-3f))
                flag_status(a.status, DG_ST_NONFINITE);
            if (a.argmax) a.argmax[r] = acc.idx;
            if (a.conf) a.conf[r] = conf;
            if (a.entropy) a.entropy[r] = H;
            if (a.ctl) {
                const size_t tr = static_cast<size_t>(p) * a.R + r;
                if (a.trace_argmax) a.trace_argmax[tr] = acc.idx;
                if (a.trace_conf) a.trace_conf[tr] = conf;
                if (a.trace_entropy) a.trace_entropy[tr] = H;
            }
        }
        // ---- mean entropy of the canvas: fixed-order pairwise tree over the slots ----
        if (sub == 0) {
            sh_red[j] = act ? H : 0.0f;
            sh_conf[j] = act ? conf : 0.0f;
        }
        __syncthreads();
        for (int off = rows_pow2 >> 1; off > 0; off >>= 1) {
            if (threadIdx.x < off) sh_red[threadIdx.x] += sh_red[threadIdx.x + off];
            __syncthreads();
        }
        const float meanH = sh_red[0] / static_cast<float>(a.S);
        if (threadIdx.x == 0 && a.mean_entropy) a.mean_entropy[b] = meanH;
        if (threadIdx.x == 0 && a.trace_mean_entropy && a.ctl) a.trace_mean_entropy[p * a.B + b] = meanH;

        if (a.canvas_out) {
            // ---- keep the K most confident slots, re-draw the rest ----
            long long K;
            if (a.keep_sched)
                K = a.keep_sched[p];
            else if (a.keep_k0 >= 0)
                K = static_cast<long long>(a.keep_k0) * (p + 1);
            else
                K = a.keep_k;
            K = K < 0 ? 0 : (K > a.S ? a.S : K);
            int rank = 0;
            for (int i = sub; i < a.S; i += tpr) {
                const float ci = sh_conf[i];
                rank += (ci > conf) || (ci == conf && i < j);
            }
            for (int off = 1; off < tpr; off <<= 1) rank += __shfl_xor_sync(0xffffffffu, rank, off);
            const bool kp = act && rank < K;
            int old = 0, nw = 0;
            if (act) {
                old = a.canvas_in[r];
                nw = kp ? acc.idx
                        : static_cast<int>(draw_key(a.seed, static_cast<uint32_t>(p),
                                                    static_cast<uint64_t>(r)) %
                                           static_cast<uint64_t>(a.V));
            }
            __syncthreads();  // every slot read its old token before any slot writes (in place)
            if (act && sub == 0) {
                if (old < 0 || old >= a.V) flag_status(a.status, DG_ST_BAD_TOKEN);
                if (a.trace_canvas && a.ctl) a.trace_canvas[static_cast<size_t>(p) * a.R + r] = old;
                a.canvas_out[r] = nw;
                if (a.kept) a.kept[r] = kp ? 1 : 0;
            }
            const int changed = __syncthreads_or(act && nw != old);
            if (threadIdx.x == 0 && a.state && a.has_rule) {
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
    }

    // ---- loop mode: the last CTA of the pass advances the pass and sets the graph condition ----
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
    const int rows = pow2_at_least(a.S);      // 32 .. 1024
    int tpr = 1024 / rows;
    if (tpr > 8) tpr = 8;
    select_kernel<<<a.B, rows * tpr, 2 * rows * sizeof(float), stream>>>(a, tpr);
    return cudaGetLastError();
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
