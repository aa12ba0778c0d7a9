// m2rnn_check.cuh -- index checks of the checked build.
//
// Built with -DM2RNN_CHECK=1 (libm2rnn_check.so), every global-memory access
// whose index the kernels compute is tested against the extent that the
// launch's shape gives the array.  A violation records M2RNN_ERR_BOUNDS and
// the site's code in the device status word (the first recorded error
// wins) and the access is skipped: nothing traps, and the host reads the
// status with m2rnn_device_status.  In the normal build the checks compile
// to nothing.
#pragma once
#include <cstddef>

#include "m2rnn_internal.h"

#ifndef M2RNN_CHECK
#define M2RNN_CHECK 0
#endif

namespace m2rnn {

// True when elements [off, off + n) lie inside an array of `extent`
// elements.  Checked build: records the violation at `site` and returns false.
__device__ __forceinline__ bool in_range(int* status, size_t off, size_t n, size_t extent, int site) {
#if M2RNN_CHECK
  if (off <= extent && n <= extent - off) return true;
  if (status != nullptr && atomicCAS(&status[0], 0, kStatusBounds) == 0) atomicExch(&status[1], site);
  return false;
#else
  (void)status;
  (void)off;
  (void)n;
  (void)extent;
  (void)site;
  return true;
#endif
}

}  // namespace m2rnn
