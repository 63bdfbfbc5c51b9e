// Index checks of the checked build (compiled with -DDFLASH_CHECKED, the library built by
// build.py when DFLASH_CHECKED=1): a failed check records DF_ERR_BOUNDS with the check's id
// in the status word and the guarded access is skipped; nothing traps.  In the default
// build a check is the constant true.
#pragma once
#include "common.cuh"

namespace df {
#ifdef DFLASH_CHECKED
DF_DEV bool checked_ok(bool ok, int* status, int where) {
  if (!ok) set_status(status, DF_ERR_BOUNDS, where);
  return ok;
}
#define DF_IN_BOUNDS(cond, status, where) (::df::checked_ok((cond), (status), (where)))
#else
#define DF_IN_BOUNDS(cond, status, where) (true)
#endif
}  // namespace df
