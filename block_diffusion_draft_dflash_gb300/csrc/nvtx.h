// One NVTX range per C-ABI call, so a profiler's timeline groups each call's kernels under
// the call's name.  NVTX 3 is header-only: with no tool attached a range costs a branch.
#pragma once
#include <nvtx3/nvToolsExt.h>

namespace df {
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
}  // namespace df

#define DF_NVTX(name) ::df::NvtxRange df_nvtx_range_(name)
