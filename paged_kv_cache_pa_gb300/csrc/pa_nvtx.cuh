// pa_nvtx.cuh -- optional NVTX ranges around the C-ABI calls.  Built with
// -DPA_NVTX (header-only NVTX v3: nothing extra to link), every compute call
// pushes a range named after itself for the host thread that made it, so a
// timeline tool shows where each call's launches were enqueued; otherwise
// PA_NVTX_RANGE expands to nothing.
#pragma once

#ifdef PA_NVTX
#include <nvtx3/nvToolsExt.h>

namespace pa {
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};
}  // namespace pa
#define PA_NVTX_RANGE(name) ::pa::NvtxRange pa_nvtx_range_(name)
#else
#define PA_NVTX_RANGE(name) ((void)0)
#endif
