// dg_host.cu -- dg_canvas_step_host: one canvas pass on host buffers. Uploads the pass's hidden
// states and canvas into one of two device staging sets in the workspace (on a copy stream the
// library owns), runs dg_canvas_step on the caller's stream, and reads the new canvas and mean
// entropy back. Successive calls alternate between the staging sets, so a call's uploads overlap
// the previous call's kernels; events keep a set from being rewritten before the pass that last
// used it has finished.
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <utility>

#include "../../include/dgcanvas.h"
#include "dg_nvtx.h"

namespace {

constexpr int kSets = 2;

size_t up256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Byte sizes of one staging set for a descriptor: hidden states, their scales, canvas in / out,
// mean entropy; offsets relative to the start of the set.
struct Staging {
    size_t h, h_scale, h_bscale, cin, cout, mean, bytes;
    size_t n_h, n_h_scale, n_h_bscale, n_canvas, n_mean;
};

int staging_for(const dg_head_desc* d, Staging* s) {
    const size_t R = static_cast<size_t>(d->B) * d->S;
    size_t row;
    switch (d->h_dtype) {
    case DG_F32: row = static_cast<size_t>(d->d) * 4; break;
    case DG_BF16: row = static_cast<size_t>(d->d) * 2; break;
    case DG_E4M3: row = static_cast<size_t>(d->d); break;
    case DG_NVFP4: row = static_cast<size_t>(d->d) / 2; break;
    default: return DG_ERR_UNSUPPORTED;
    }
    s->n_h = R * row;
    s->n_h_scale = d->h_scale ? R * 4 : 0;
    s->n_h_bscale = 0;
    if (d->h_block_scale) {
        const int rc = dg_nvfp4_scale_bytes(static_cast<int32_t>(R), d->d, &s->n_h_bscale);
        if (rc != DG_OK) return rc;
    }
    s->n_canvas = R * 4;
    s->n_mean = static_cast<size_t>(d->B) * 4;
    size_t off = 0;
    s->h = off;
    off = up256(off + s->n_h);
    s->h_scale = off;
    off = up256(off + s->n_h_scale);
    s->h_bscale = off;
    off = up256(off + s->n_h_bscale);
    s->cin = off;
    off = up256(off + s->n_canvas);
    s->cout = off;
    off = up256(off + s->n_canvas);
    s->mean = off;
    off = up256(off + s->n_mean);
    s->bytes = off;
    return DG_OK;
}

// Per (workspace, device) copy stream and events, created on the first call that uses them.
struct Session {
    cudaStream_t copy = nullptr;
    cudaEvent_t ready[kSets] = {};
    cudaEvent_t freed[kSets] = {};
    bool used[kSets] = {};
    int next = 0;
};

using SessionKey = std::pair<const void*, int>;
std::mutex g_mu;
std::map<SessionKey, Session>& sessions() {
    static std::map<SessionKey, Session> m;
    return m;
}

int session_for(const void* ws, Session** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DG_ERR_CUDA;
    auto& m = sessions();
    const SessionKey key(ws, dev);
    auto it = m.find(key);
    if (it != m.end()) {
        *out = &it->second;
        return DG_OK;
    }
    Session s;
    if (cudaStreamCreateWithFlags(&s.copy, cudaStreamNonBlocking) != cudaSuccess) return DG_ERR_CUDA;
    for (int i = 0; i < kSets; ++i)
        if (cudaEventCreateWithFlags(&s.ready[i], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&s.freed[i], cudaEventDisableTiming) != cudaSuccess)
            return DG_ERR_CUDA;
    *out = &(m[key] = s);
    return DG_OK;
}

}  // namespace

extern "C" {

int dg_workspace_bytes_host(const dg_head_desc* desc, size_t* bytes) {
    if (!desc || !bytes) return DG_ERR_INVALID_ARG;
    size_t base = 0;
    int rc = dg_workspace_bytes(desc, &base);
    if (rc != DG_OK) return rc;
    Staging s;
    rc = staging_for(desc, &s);
    if (rc != DG_OK) return rc;
    *bytes = up256(base) + kSets * s.bytes;
    return DG_OK;
}

int dg_canvas_step_host(const dg_head_desc* desc, const int32_t* canvas_in, int32_t* canvas_out,
                        float* mean_entropy, int32_t keep_k, uint64_t seed, uint32_t pass,
                        dg_canvas_state* state, const dg_stop_rule* rule, void* workspace,
                        size_t workspace_bytes, uint32_t* status, dg_stream_t stream) {
    dg::NvtxRange nvtx_range("dg_canvas_step_host");
    if (!desc || !desc->h || !canvas_in || !canvas_out || !workspace) return DG_ERR_INVALID_ARG;
    size_t base = 0;
    int rc = dg_workspace_bytes(desc, &base);
    if (rc != DG_OK) return rc;
    Staging sz;
    rc = staging_for(desc, &sz);
    if (rc != DG_OK) return rc;
    base = up256(base);
    if (workspace_bytes < base + kSets * sz.bytes ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return DG_ERR_WORKSPACE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) return DG_ERR_CUDA;
    if (cap != cudaStreamCaptureStatusNone) return DG_ERR_UNSUPPORTED;

    std::lock_guard<std::mutex> lock(g_mu);
    Session* s = nullptr;
    rc = session_for(workspace, &s);
    if (rc != DG_OK) return rc;
    const int b = s->next;
    uint8_t* set = static_cast<uint8_t*>(workspace) + base + b * sz.bytes;

    // uploads, once the pass that last used this set has finished
    if (s->used[b] && cudaStreamWaitEvent(s->copy, s->freed[b], 0) != cudaSuccess) return DG_ERR_CUDA;
    if (cudaMemcpyAsync(set + sz.h, desc->h, sz.n_h, cudaMemcpyHostToDevice, s->copy) != cudaSuccess ||
        (sz.n_h_scale && cudaMemcpyAsync(set + sz.h_scale, desc->h_scale, sz.n_h_scale,
                                         cudaMemcpyHostToDevice, s->copy) != cudaSuccess) ||
        (sz.n_h_bscale && cudaMemcpyAsync(set + sz.h_bscale, desc->h_block_scale, sz.n_h_bscale,
                                          cudaMemcpyHostToDevice, s->copy) != cudaSuccess) ||
        cudaMemcpyAsync(set + sz.cin, canvas_in, sz.n_canvas, cudaMemcpyHostToDevice, s->copy) !=
            cudaSuccess ||
        cudaEventRecord(s->ready[b], s->copy) != cudaSuccess ||
        cudaStreamWaitEvent(st, s->ready[b], 0) != cudaSuccess)
        return DG_ERR_CUDA;

    // the pass, on the staged copies
    dg_head_desc dd = *desc;
    dd.h = set + sz.h;
    dd.h_scale = sz.n_h_scale ? reinterpret_cast<const float*>(set + sz.h_scale) : nullptr;
    dd.h_block_scale = sz.n_h_bscale ? set + sz.h_bscale : nullptr;
    int32_t* cout = reinterpret_cast<int32_t*>(set + sz.cout);
    float* mean = reinterpret_cast<float*>(set + sz.mean);
    rc = dg_canvas_step(&dd, reinterpret_cast<const int32_t*>(set + sz.cin), cout, keep_k, seed,
                        pass, nullptr, nullptr, nullptr, nullptr, mean, state, rule, workspace,
                        base, status, stream);
    if (rc != DG_OK) return rc;

    // read-backs, then mark the set free for the call after next
    if (cudaMemcpyAsync(canvas_out, cout, sz.n_canvas, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        (mean_entropy && cudaMemcpyAsync(mean_entropy, mean, sz.n_mean, cudaMemcpyDeviceToHost,
                                         st) != cudaSuccess) ||
        cudaEventRecord(s->freed[b], st) != cudaSuccess)
        return DG_ERR_CUDA;
    s->used[b] = true;
    s->next = (b + 1) % kSets;
    return DG_OK;
}

}  // extern "C"
