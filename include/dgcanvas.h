/*
 * dgcanvas.h -- C ABI of libdgcanvas.so: the per-pass canvas update of a uniform-state block
 * text-diffusion sampler, on one B300 (sm_103a).
 *
 * The method (as the pages describe it):
 *   - A canvas is a fixed block of 256 token slots ("DiffusionGemma 26B: How Google's Text
 *     Diffusion Model Generates Tokens in Parallel" (dev.to), "Architecture Details": canvas
 *     length 256, vocabulary 262K).
 *   - Uniform-state diffusion: the canvas starts from random vocabulary tokens and any slot can
 *     be revised later. Each pass predicts every slot at once, keeps the slots it is most
 *     confident about and re-randomises the rest ("When to use a diffusion LLM"
 *     (devengoratela.com), "How block diffusion works").
 *   - The loop stops when the average canvas entropy drops below a threshold or the tokens are
 *     stable across two consecutive steps, after at most 48 steps (dev.to page, "How Diffusion
 *     Changes the Equation"); the average runs over all 256 slots including padding
 *     (devengoratela.com page, "How block diffusion works").
 *
 * Readings fixed by this library where the pages are silent:
 *   - confidence of a slot = max_n p_n of its softmax over the vocabulary; entropy in nats;
 *   - keep the K most confident slots of each canvas, ties to the lower slot index; argmax ties
 *     to the lower vocabulary index;
 *   - re-randomised token of row r = b*S + slot at pass p: key(seed, p, r) mod V with
 *     key(seed, p, r) = sm64(sm64(sm64(seed) ^ p) ^ r) and sm64 one SplitMix64 output
 *     (Steele, Lea & Flood, OOPSLA 2014); the initial random canvas uses p = 0xFFFFFFFF;
 *   - the stop rules are OR-combined by default (DG_STOP_AND requires entropy AND stability),
 *     "stable" = the update left the whole canvas unchanged for `stable_passes` consecutive
 *     passes, the entropy test is strict (mean H < threshold).
 *
 * Conventions for every entry point:
 *   - All data pointers are DEVICE pointers owned by the caller (for example PyTorch tensors),
 *     16-byte aligned; dg_canvas_step_host's hidden states and canvases are the one exception
 *     (host memory). The library allocates no device memory on the step path: the caller
 *     passes a workspace of at least dg_workspace_bytes() bytes, 256-byte aligned.
 *   - `stream` is the caller's cudaStream_t (NULL = legacy default stream). Calls only enqueue
 *     work and never synchronise; results are valid once the stream reaches them.
 *   - Return value: DG_OK or a negative DG_ERR_* code; on error nothing was enqueued (except
 *     DG_ERR_CUDA, which reports a failed launch). Data problems found on the device (token ids
 *     outside [0, V), non-finite logits, a bounded wait that ran out) do not trap: they set
 *     sticky DG_ST_* bits in the caller's device `status` word (which the caller zeroes), and
 *     the affected outputs are unspecified.
 */
#ifndef DGCANVAS_H
#define DGCANVAS_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DG_API __attribute__((visibility("default")))
#else
#define DG_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dg_stream_t; /* identical to cudaStream_t */

typedef enum { DG_F32 = 0, DG_BF16 = 1, DG_E4M3 = 2, DG_NVFP4 = 3 } dg_dtype;

enum {
    DG_OK = 0,
    DG_ERR_INVALID_ARG = -1,  /* null/negative/inconsistent argument */
    DG_ERR_ALIGNMENT = -2,    /* pointer not 16-byte aligned, or d*elem_size % 16 != 0 */
    DG_ERR_UNSUPPORTED = -3,  /* not sm_103, dtype pair not supported, S > 1024, V >= 2^31 */
    DG_ERR_WORKSPACE = -4,    /* workspace NULL, misaligned or smaller than required */
    DG_ERR_CUDA = -5          /* a CUDA runtime call or kernel launch failed */
};

/* Sticky device status bits. */
enum {
    DG_ST_BAD_TOKEN = 1u,  /* an input canvas or target id was outside [0, V) */
    DG_ST_NONFINITE = 2u,  /* a non-finite logit or hidden value reached the statistics */
    DG_ST_TIMEOUT = 4u     /* a bounded on-device wait ran out; that kernel returned early */
};

/* Stop reasons (bitmask of every rule true at the stopping pass). */
enum { DG_REASON_ENTROPY = 1, DG_REASON_STABLE = 2, DG_REASON_CAP = 4 };
enum { DG_STOP_OR = 0, DG_STOP_AND = 1 };
/* Which slots a pass keeps: the K most confident (max-prob), or the K lowest-entropy ones
   ("lowest-entropy tokens locked first", dev.to page, "Architecture Details"); ties to the lower
   slot either way. */
enum { DG_KEEP_CONFIDENCE = 0, DG_KEEP_ENTROPY = 1 };
/* What the other slots become: a uniform re-draw key(seed, pass, row) mod V (uniform-state
   diffusion), or a fixed mask token (the masked-diffusion variant: "DiffusionGemma: When Text
   Generation Stops Being Sequential" (laura-martel.com), introduction). */
enum { DG_REDRAW_UNIFORM = 0, DG_REDRAW_MASK = 1 };

/*
 * The vocabulary head and the hidden states of one batch of canvases.
 *   h       [B*S, d] row-major, row r = b*S + slot. dtype h_dtype.
 *   h_scale [B*S] fp32 per-row scales when h_dtype == DG_E4M3, else NULL.
 *   w       [V, d] row-major vocabulary head. dtype w_dtype.
 *   w_scale [V] fp32 per-row scales when w_dtype == DG_E4M3, else NULL.
 * logits l[r, n] = inv_temp * sum_k h[r,k] * w[n,k] (times h_scale[r] * w_scale[n] for E4M3),
 * accumulated in fp32 and never stored.
 * Supported (h_dtype, w_dtype): (F32, F32) on CUDA cores; (BF16, BF16) and (E4M3, E4M3) on the
 * tensor cores; (BF16, E4M3) quantises h per row to E4M3 first (absmax scaling:
 * scale = amax/448, q = e4m3_rn_satfinite(h * (448/amax)), all in fp32; amax = 0 gives scale 1).
 * NVFP4 (4-bit; the NVFP4-quantised variant of the laura-martel.com page, introduction):
 * (NVFP4, NVFP4) and (BF16, NVFP4), the latter quantising h on the device with dg_quantize_nvfp4's
 * rule. An NVFP4 operand is three arrays: E2M1 codes [rows, d/2] bytes (element 2j in the low
 * nibble of byte j), the fp32 row scale (h_scale / w_scale) and E4M3 block scales, one per 16
 * elements along d, in the packed layout of dg_nvfp4_pack_scales (h_block_scale /
 * w_block_scale); element value = e2m1(code) * e4m3(block scale) * row scale.
 * Limits: 1 <= S <= 1024, B >= 1, 1 <= V < 2^31, d >= 1 with d*elem_size(dtype) % 16 == 0
 * (elem_size 4 / 2 / 1 / 0.5); NVFP4 also needs d % 256 == 0.
 */
typedef struct {
    int32_t B, S, d, V;
    int32_t h_dtype, w_dtype; /* dg_dtype */
    const void* h;
    const float* h_scale;
    const void* w;
    const float* w_scale;
    float inv_temp;           /* 1.0f = untempered statistics */
    const uint8_t* h_block_scale;  /* NVFP4 h: packed E4M3 block scales, else NULL */
    const uint8_t* w_block_scale;  /* NVFP4 w: packed E4M3 block scales, else NULL */
} dg_head_desc;

/* Per-canvas loop state in device memory (32 bytes per canvas). */
typedef struct {
    int32_t passes;       /* passes completed when the canvas stopped, else 0 */
    int32_t reason;       /* DG_REASON_* bitmask at the stopping pass, else 0 */
    int32_t stable;       /* consecutive passes that left the canvas unchanged */
    int32_t done;         /* 1 once stopped: later passes leave the canvas frozen */
    float mean_entropy;   /* mean slot entropy (nats) of the last pass that ran */
    int32_t last_pass;    /* index of the last pass that updated this canvas, -1 before */
    int32_t reserved[2];
} dg_canvas_state;

/* The rules of a pass: its stop test (used by dg_canvas_step with a state, and by
   dg_canvas_loop) and its keep / re-draw variant (used by every pass given a rule; a NULL rule
   means DG_KEEP_CONFIDENCE and DG_REDRAW_UNIFORM). A zero-initialised tail selects the defaults. */
typedef struct {
    int32_t max_passes;        /* pass cap (48 in the pages) */
    float entropy_threshold;   /* stop when mean H < threshold (nats) */
    int32_t stable_passes;     /* stop when unchanged for this many consecutive passes (2) */
    int32_t stop_mode;         /* DG_STOP_OR or DG_STOP_AND */
    int32_t keep_rule;         /* DG_KEEP_CONFIDENCE (default) or DG_KEEP_ENTROPY */
    int32_t redraw_mode;       /* DG_REDRAW_UNIFORM (default) or DG_REDRAW_MASK */
    int32_t mask_id;           /* the mask token, in [0, V), with DG_REDRAW_MASK */
} dg_stop_rule;

/* Bytes of workspace a call with this descriptor needs (same for stats/step/loop). */
DG_API int dg_workspace_bytes(const dg_head_desc* desc, size_t* bytes);

/*
 * Softmax statistics of every slot, without storing logits:
 *   argmax[r] (int32), conf[r] = max_n p_n (fp32), entropy[r] = -sum_n p_n ln p_n (fp32, nats),
 *   mean_entropy[b] = mean over the S slots of canvas b (fp32, fixed summation order).
 * Any output pointer may be NULL. status: device uint32 (sticky DG_ST_* bits), may be NULL.
 */
DG_API int dg_canvas_stats(const dg_head_desc* desc, int32_t* argmax, float* conf, float* entropy,
                    float* mean_entropy, void* workspace, size_t workspace_bytes,
                    uint32_t* status, dg_stream_t stream);

/*
 * One canvas pass: statistics, keep the K = min(keep_k, S) most confident slots of each canvas
 * at their argmax, re-draw the others as key(seed, pass, r) mod V, write canvas_out [B*S].
 * canvas_in == canvas_out is allowed. kept [B*S] (uint8 0/1) and the statistics outputs may be
 * NULL. If `state` (device, [B]) and `rule` (host) are given, the pass also applies the stop
 * test: it updates stable/done/passes/reason, and canvases already done are left unchanged
 * (copied to canvas_out). rule may only be NULL when state is NULL; without a state only its
 * keep / re-draw variant is used.
 */
DG_API int dg_canvas_step(const dg_head_desc* desc, const int32_t* canvas_in, int32_t* canvas_out,
                   int32_t keep_k, uint64_t seed, uint32_t pass, int32_t* argmax, float* conf,
                   float* entropy, uint8_t* kept, float* mean_entropy, dg_canvas_state* state,
                   const dg_stop_rule* rule, void* workspace, size_t workspace_bytes,
                   uint32_t* status, dg_stream_t stream);

/*
 * Denoiser hook of the loop: enqueue, on `stream`, work that reads the canvas (device int32
 * [B*S]) and the pass index (device int32 scalar) and writes the hidden states h_out (device,
 * [B*S, d] in the descriptor's h_dtype; BF16 when the head is E4M3 and h is quantised by the
 * library). It must be stream-ordered and capturable into a CUDA graph (no host sync, no
 * allocation): the library calls it while it captures the loop's graph, not once per pass, and
 * the pass index is only known on the device. Return 0 on success.
 * The captured graph is cached and replayed by later dg_canvas_loop calls whose arguments are
 * all the same (the same hook function and `user` pointer included), without calling the hook
 * again. So the work a hook enqueues for one (hook, user) must not change between such calls:
 * the memory it reads may change in content, not in address. Pass a different `user` (or
 * function) to have the loop captured afresh.
 */
typedef int (*dg_denoise_fn)(void* user, const int32_t* canvas, const int32_t* pass,
                             void* h_out, dg_stream_t stream);

/*
 * Built-in synthetic denoiser (test workload, not part of the method): with t = pass + 1 and
 * a_t = min(1, fp32((2 + t)/10)), x = a_t * w[y_r] + (1 - a_t) * w[c_r] in fp32 (E4M3 rows
 * dequantised as code * w_scale), h_r = s_r * x / ||x||_2 (0 when x = 0), s_r = s_content
 * for the first n_content slots of each canvas and s_pad for the rest, rounded to bf16.
 * Pass dg_synth_denoise as the hook and a dg_synth_params* (host memory, read at call time)
 * as `user`.
 */
typedef struct {
    const dg_head_desc* desc; /* head whose rows are mixed (the head is tied) */
    const int32_t* y;         /* device [B*S] target ids */
    int32_t n_content;
    float s_content, s_pad;
    uint32_t* status;         /* optional device status word (DG_ST_BAD_TOKEN on bad ids) */
} dg_synth_params;

DG_API int dg_synth_denoise(void* user, const int32_t* canvas, const int32_t* pass, void* h_out,
                     dg_stream_t stream);

/*
 * The whole denoising loop, stream-ordered with no host synchronisation: a CUDA graph whose
 * conditional WHILE node runs [denoise -> (quantise) -> statistics -> keep/re-randomise/stop]
 * until every canvas has stopped or max_passes is reached.
 *   canvas [B*S]: the canvas (in/out). If init_random, it is first overwritten with
 *     key(seed, 0xFFFFFFFF, row_offset + r) mod V (with DG_REDRAW_MASK: the mask token).
 *   h_buffer: device [B*S, d] buffer the denoiser writes (desc->h must equal it).
 *   K_t = keep_sched ? keep_sched[p] : min(keep_k0 * (p + 1), S) for 0-based pass p.
 *   Re-draws of pass p use key(seed, p, row_offset + r) (a block's offset in a
 *   block-autoregressive run; 0 otherwise).
 *   With temp_start > 0 the statistics of pass p are those of softmax(l / T_p), l the logits of
 *   the descriptor (inv_temp included), T_p = temp_start + (temp_end - temp_start) * p /
 *   (max_passes - 1) in fp32 (temp_start alone when max_passes = 1): the 0.8 -> 0.4 anneal of
 *   the dev.to page, "Architecture Details", and the devengoratela.com page, "Appendix:
 *   Methodology / Decoding". The argmax is unaffected; confidence, entropy, the keep order and
 *   the entropy stop test are.
 *   state [B] (device): on entry `stable` is the resume count when start_pass > 0 (and is
 *     reset to 0 otherwise); on exit it holds passes/reason/mean_entropy per canvas.
 *   argmax/conf/entropy: optional device outputs of the last pass that ran.
 *   trace_mean_entropy [max_passes * B], trace_canvas [max_passes * B*S] (row p holds the
 *   canvas entering pass p; the canvas left by the last pass is the `canvas` argument itself),
 *   trace_h [max_passes * B*S*d] (bytes of h_dtype), trace_argmax/conf/entropy
 *   [max_passes * B*S]: optional device traces of every pass, for checking. Rows of passes
 *   that did not run are left as they were; so are a stopped canvas's statistics and mean
 *   entropy in later passes, while its canvas trace keeps showing its frozen canvas.
 */
typedef struct {
    dg_stop_rule rule;
    int32_t keep_k0;
    const int32_t* keep_sched;  /* optional device [max_passes] */
    uint64_t seed;
    uint32_t start_pass;
    uint32_t init_random;
    float* trace_mean_entropy;
    int32_t* trace_canvas;
    void* trace_h;
    int32_t* trace_argmax;      /* optional device [max_passes * B*S] per-pass statistics */
    float* trace_conf;
    float* trace_entropy;
    /* optional device [max_passes * DG_TL_KERNELS * 2] uint64: per pass p and kernel k the
       device global timer (ns) when the first CTA of k got past its wait on the previous kernel
       (index (p * DG_TL_KERNELS + k) * 2) and when the last CTA of k finished (+1). Entries of
       passes that did not run, and of the built-in denoiser when the caller supplies its own,
       stay at (UINT64_MAX, 0). Costs one branch per CTA when NULL. */
    unsigned long long* trace_timeline;
    float temp_start, temp_end;  /* temperature schedule; temp_start = 0: none */
    uint64_t row_offset;         /* added to the row index of every re-draw key */
    /* optional device [max_passes * 4] uint64: per pass p, the SM clock sample of its head
       kernel (see dg_profile_next_head_clock) at index p * 4; rows of passes that did not run
       stay as they were. */
    unsigned long long* trace_sm_clock;
} dg_loop_params;

/* Kernels recorded in dg_loop_params.trace_timeline. */
enum { DG_TL_DENOISE = 0, DG_TL_HEAD = 1, DG_TL_MERGE = 2, DG_TL_KERNELS = 3 };

DG_API int dg_canvas_loop(const dg_head_desc* desc, int32_t* canvas, void* h_buffer,
                   const dg_loop_params* params, dg_denoise_fn denoise, void* user,
                   dg_canvas_state* state, int32_t* argmax, float* conf, float* entropy,
                   void* workspace, size_t workspace_bytes, uint32_t* status,
                   dg_stream_t stream);

/*
 * Block-autoregressive generation with the built-in synthetic denoiser: block i (0-based) runs
 * the whole loop (dg_canvas_loop with init_random, start_pass 0 and row_offset =
 * params->row_offset + i*B*S) on a fresh canvas with targets y_blocks[i*B*S ...], then commits its
 * final canvas to tokens_out[i*B*S ...] and its per-canvas state to states_out[i*B ...]; block
 * i+1 starts after it, on the same stream, with no host synchronisation. The model would condition
 * each block on the committed ones through its KV cache; the synthetic denoiser does not.
 *   y_work [B*S], canvas [B*S], state [B]: device work buffers (written); desc->h == h_buffer.
 *   One captured loop graph serves every block (only y_work's contents and the row offset change).
 */
DG_API int dg_block_generate(const dg_head_desc* desc, int32_t n_blocks, const int32_t* y_blocks,
                             int32_t* y_work, int32_t* canvas, dg_canvas_state* state,
                             void* h_buffer, const dg_loop_params* params, int32_t n_content,
                             float s_content, float s_pad, int32_t* tokens_out,
                             dg_canvas_state* states_out, void* workspace, size_t workspace_bytes,
                             uint32_t* status, dg_stream_t stream);

/*
 * Per-row E4M3 quantisation of bf16 rows [rows, d] on the device (step a0 of an FP8 pass, the
 * rule a (BF16, E4M3) descriptor applies inside a pass), in IEEE binary32: amax = max_k |h_k|;
 * amax == 0 gives row scale 1 and zero codes; else inv = 448 / amax,
 * codes q_k = e4m3_rn_satfinite(h_k * inv) and row scale amax / 448 (each operation rounded to
 * nearest). Writes codes [rows, d] (E4M3 bytes) and row_scale [rows]; sets DG_ST_NONFINITE in
 * *status (may be NULL) on non-finite input. Device pointers; h_bf16 16-byte aligned.
 */
DG_API int dg_quantize_e4m3(const void* h_bf16, int32_t rows, int32_t d, uint8_t* codes,
                            float* row_scale, uint32_t* status, dg_stream_t stream);

/*
 * NVFP4 operand preparation (4-bit heads).
 *   dg_nvfp4_scale_bytes: size of the packed block-scale array of `rows` rows of width d:
 *     ceil(rows / 256) * 256 * d / 16 bytes.
 *   dg_nvfp4_pack_scales: block scales [rows, d/16] (row-major, E4M3) -> the packed layout the
 *     block-scaled MMA consumes: one 4096-byte chunk per (256-row group G, 256-element K slice s)
 *     at offset (G * d/256 + s) * 4096; the scale of row 256 G + m (l = m % 32, c = m / 32),
 *     block 16 s + 4 j + kb sits at byte
 *       (l / 8) * 1024 + j * 256 + (c / 4) * 128 + (l % 8) * 16 + (c % 4) * 4 + kb
 *     of its chunk; rows past `rows` are zero. Device pointers, d % 256 == 0.
 *   dg_quantize_nvfp4: two-level NVFP4 quantisation of bf16 rows [rows, d] on the device, in
 *     IEEE binary32: amax = max |h|; amax == 0 gives row scale 1 and zero codes / block scales;
 *     else g = amax / 2688, per block of 16: sb = e4m3_rn_satfinite(bmax / (6 g)), codes
 *     q = e2m1_rn_satfinite(h / (value(sb) g)) (0 where sb = 0). Writes codes [rows, d/2], packed
 *     block scales (dg_nvfp4_scale_bytes) and row scales [rows]. Sets DG_ST_NONFINITE on
 *     non-finite input. d % 256 == 0.
 */
DG_API int dg_nvfp4_scale_bytes(int32_t rows, int32_t d, size_t* bytes);
DG_API int dg_nvfp4_pack_scales(const uint8_t* block_scales, int32_t rows, int32_t d,
                                uint8_t* packed, dg_stream_t stream);
DG_API int dg_quantize_nvfp4(const void* h_bf16, int32_t rows, int32_t d, uint8_t* codes,
                             uint8_t* block_scale_packed, float* row_scale, uint32_t* status,
                             dg_stream_t stream);

/*
 * dg_canvas_step without a caller-supplied workspace, for callers that cannot allocate device
 * memory: plugins hosted by a framework that owns all device allocations, and latency-critical
 * code that must not risk the implicit synchronisation of cudaMalloc/cudaFree or that runs under
 * a device-memory budget fixed in advance. (The pages describe no such entry point; it has no
 * counterpart in the method.)
 * Same arguments and results as dg_canvas_step minus the workspace. Its scratch is one array of
 * DG_NOALLOC_SCRATCH_BYTES compiled into the library (held by every GPU that loads it until the
 * process exits); descriptors needing more scratch than that (dg_workspace_bytes) are rejected
 * with DG_ERR_WORKSPACE. The function allocates nothing. Its first call on a device looks up the
 * array's device address (cudaGetSymbolAddress), so make that first call before any stream
 * capture. All calls share the array: calls that overlap on the GPU (unordered streams or
 * threads) race and corrupt each other's results, so order them on one stream. Nothing in the
 * array needs clearing between calls: each pass rewrites every scratch byte it reads.
 */
#define DG_NOALLOC_SCRATCH_BYTES (4u << 20)
DG_API int dg_canvas_step_noalloc(const dg_head_desc* desc, const int32_t* canvas_in,
                                  int32_t* canvas_out, int32_t keep_k, uint64_t seed,
                                  uint32_t pass, int32_t* argmax, float* conf, float* entropy,
                                  uint8_t* kept, float* mean_entropy, dg_canvas_state* state,
                                  const dg_stop_rule* rule, uint32_t* status, dg_stream_t stream);

/*
 * One canvas pass on HOST buffers: the hidden states (desc->h, and desc->h_scale /
 * desc->h_block_scale when h is E4M3 / NVFP4) and canvas_in [B*S] are read from host memory, the
 * new canvas is written to canvas_out [B*S] and, if non-NULL, the per-canvas mean entropy to
 * mean_entropy [B], both host memory. w, w_scale, w_block_scale, state and status stay device
 * pointers; keep_k, seed, pass and rule are those of dg_canvas_step, whose pass this runs. (The
 * pages describe no such entry point; it serves callers whose data lives on the host.)
 * Everything is enqueued and the call returns: the uploads run on a copy stream owned by the
 * library and are ordered before the pass on `stream` by events; the read-backs run on `stream`
 * after the pass. Host results are valid once `stream` has synchronised; host inputs must stay
 * valid and unchanged until then. Use page-locked host memory for the copies to be asynchronous.
 * The device copies live in the workspace, in two staging sets used by successive calls in turn,
 * so the uploads of one call overlap the previous call's kernels; a set is not rewritten before
 * the pass that last used it has finished. Calls sharing a workspace must share `stream`. Not for
 * use under stream capture (DG_ERR_UNSUPPORTED): capture dg_canvas_step instead. The library
 * keeps one copy stream and four events per (workspace address, device) it has seen, for the
 * life of the process.
 * dg_workspace_bytes_host: workspace bytes for this entry point (dg_workspace_bytes plus the two
 * staging sets).
 */
DG_API int dg_workspace_bytes_host(const dg_head_desc* desc, size_t* bytes);
DG_API int dg_canvas_step_host(const dg_head_desc* desc, const int32_t* canvas_in,
                               int32_t* canvas_out, float* mean_entropy, int32_t keep_k,
                               uint64_t seed, uint32_t pass, dg_canvas_state* state,
                               const dg_stop_rule* rule, void* workspace, size_t workspace_bytes,
                               uint32_t* status, dg_stream_t stream);

/*
 * Instrumentation: make the next dg_canvas_stats / dg_canvas_step call issued by this host
 * thread record `start_event` on its stream just before its vocabulary-head kernel and
 * `stop_event` just after it (cudaEvent_t handles created by the caller). One-shot; calls that
 * are being captured into a graph do not consume it. Passing NULLs clears a pending request.
 */
DG_API int dg_profile_next_head(void* start_event, void* stop_event);

/*
 * Instrumentation: make the next dg_canvas_stats / dg_canvas_step call issued by this host
 * thread (not being captured) have its vocabulary-head kernel write an SM clock sample to
 * clock_sample (device, 4 x uint64, 8-byte aligned): CTA 0's clock64 counter and the global
 * timer (ns) when it got past its wait on the previous kernel, then the same two when it
 * finished. (cycles / ns) is the SM clock the kernel ran at, and the cycle count its duration
 * independent of that clock. One-shot; NULL clears a pending request. Independent of
 * dg_profile_next_head; both may be pending for the same call.
 */
DG_API int dg_profile_next_head_clock(unsigned long long* clock_sample);

/*
 * Self-test of the failure detection every kernel relies on: launches one kernel on `stream`
 * whose single mbarrier wait can never complete (nothing arrives on it). The wait gives up after
 * its wall-time bound (about 2 s, the bound of every on-device wait in this library), the kernel
 * sets DG_ST_TIMEOUT in *status (device, caller-owned, sticky bits OR-ed in) and returns, and the
 * CUDA context stays usable: no trap, no fault. Returns DG_ERR_INVALID_ARG for a NULL status,
 * DG_ERR_UNSUPPORTED off sm_103, DG_ERR_CUDA if the launch fails.
 */
DG_API int dg_selftest_wait_timeout(uint32_t* status, dg_stream_t stream);

/* Human-readable name of a DG_ERR_* code or DG_ST_* bit set. */
DG_API const char* dg_status_string(int code);

/* Library version, e.g. 100 for 0.1.0. */
DG_API int dg_version(void);

#ifdef __cplusplus
}
#endif
#endif /* DGCANVAS_H */
