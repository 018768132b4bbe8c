// State of the bounded grid-wide barrier used by cooperative kernels (see
// grid_barrier() in common.cuh).  Plain data, shared by host and device code.
#pragma once

namespace moe {

// Lives in global memory; zeroed (by the host, or by a kernel earlier on the
// same stream) before each cooperative launch that uses it.
struct GridBarrier {
  unsigned count;         // arrivals so far, over every barrier of the launch
  int abort;              // raised by the first CTA whose wait ran out
};

}  // namespace moe
