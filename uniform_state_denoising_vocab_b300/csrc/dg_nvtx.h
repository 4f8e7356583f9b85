// dg_nvtx.h -- NVTX ranges around the C ABI's entry points. A tool that records NVTX (Nsight
// Systems, ncu's --nvtx range filters) sees each call as a range named after the entry point;
// it spans the host-side enqueue of the call's work, which then runs asynchronously on the
// stream. Without such a tool the push and pop cost a few loads (header-only NVTX 3).
#pragma once
#include <nvtx3/nvToolsExt.h>

namespace dg {

struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

}  // namespace dg
