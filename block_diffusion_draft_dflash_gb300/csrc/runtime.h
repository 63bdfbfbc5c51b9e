// Per-device host state of the library: SM counts and kernel attributes.
//
// Kernel attributes (the dynamic shared-memory opt-in) and device properties belong to a
// device, not to the process, so every cached value here is keyed by the current device:
// a process may call the library on several GPUs in turn.
#pragma once
#include <cuda_runtime.h>

namespace df {

// SM count of the current device (cached per device).
int num_sms();

// Makes sure `func` may be launched with `bytes` of dynamic shared memory (beside its
// static shared memory) on the current device: cudaFuncSetAttribute on the first launch
// per device and kernel, again when a larger size is asked for.  Returns cudaSuccess or
// the error of the attribute call.
cudaError_t ensure_dynamic_smem(const void* func, size_t bytes);

template <typename F>
cudaError_t ensure_dynamic_smem(F* func, size_t bytes) {
  return ensure_dynamic_smem(reinterpret_cast<const void*>(func), bytes);
}

}  // namespace df
