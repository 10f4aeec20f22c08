// forward_bf16.cu -- the forward scan (every mode) for bf16 inputs (one translation unit per input
// dtype, so that the library's units compile in parallel).
#include "forward_launch.cuh"

namespace csscan_host {
int forward_bf16(const Args& a, const csscan_options_t& o, cudaStream_t st, const FixedScratch* fixed) {
  return forward_dispatch<uint16_t>(a, o, st, fixed);
}
}  // namespace csscan_host
