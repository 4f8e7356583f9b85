// dg_noalloc.cu -- dg_canvas_step_noalloc: one canvas pass whose scratch memory is a fixed
// array compiled into the library, for callers that cannot allocate device memory.
//
// Who cannot allocate: plugins and custom operators hosted by a framework that owns every
// device allocation and forbids its extensions from calling the CUDA allocator, and
// latency-critical callers that must never risk the implicit device synchronisation that
// cudaMalloc/cudaFree can cause, or that run under a fixed device-memory budget set before they
// start. They pass only inputs and outputs; the softmax partials (and, for an E4M3 head fed
// bf16 hidden states, the quantised copy of h) live in `g_scratch` below.
//
// Set-up: the first call on each device looks up the array's device address with
// cudaGetSymbolAddress (with that device current) and caches it; make that first call before
// any stream capture.
//
// Sharing rules: every call in the process on the same device uses the same array, and the
// array keeps the previous call's contents. Each pass fully rewrites every scratch byte it
// later reads (the head kernel writes one partial per (vocabulary group, row) before the merge
// reads it, and the quantised rows are rewritten before the head reads them), so nothing needs
// clearing between calls. Calls whose work overlaps on the GPU (issued on different streams,
// or from different threads, without ordering between them) race on the array and corrupt each
// other's results: order them on one stream.
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "../../include/dgcanvas.h"
#include "dg_nvtx.h"

namespace {

// Every GPU that loads the library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_scratch[DG_NOALLOC_SCRATCH_BYTES];

// Device address of g_scratch per device. In host code `g_scratch` names a host-side stand-in,
// not device memory, so the address must come from cudaGetSymbolAddress with the device current.
int scratch_address(void** out) {
    static std::mutex mu;
    static std::vector<void*> addr;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DG_ERR_CUDA;
    std::lock_guard<std::mutex> lk(mu);
    if (static_cast<int>(addr.size()) <= dev) addr.resize(dev + 1, nullptr);
    if (!addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return DG_ERR_CUDA;
        addr[dev] = p;
    }
    *out = addr[dev];
    return DG_OK;
}

}  // namespace

extern "C" int dg_canvas_step_noalloc(const dg_head_desc* desc, const int32_t* canvas_in,
                                      int32_t* canvas_out, int32_t keep_k, uint64_t seed,
                                      uint32_t pass, int32_t* argmax, float* conf, float* entropy,
                                      uint8_t* kept, float* mean_entropy, dg_canvas_state* state,
                                      const dg_stop_rule* rule, uint32_t* status,
                                      dg_stream_t stream) {
    dg::NvtxRange nvtx_range("dg_canvas_step_noalloc");
    size_t need = 0;
    int rc = dg_workspace_bytes(desc, &need);
    if (rc != DG_OK) return rc;
    if (need > DG_NOALLOC_SCRATCH_BYTES) return DG_ERR_WORKSPACE;
    void* scratch = nullptr;
    rc = scratch_address(&scratch);
    if (rc != DG_OK) return rc;
    return dg_canvas_step(desc, canvas_in, canvas_out, keep_k, seed, pass, argmax, conf, entropy,
                          kept, mean_entropy, state, rule, scratch, DG_NOALLOC_SCRATCH_BYTES,
                          status, stream);
}
