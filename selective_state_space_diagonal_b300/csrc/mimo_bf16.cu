// mimo_bf16.cu -- csscan_forward_mimo and csscan_backward_mimo for bfloat16 inputs (mimo_launch.cuh).
#include "mimo_launch.cuh"

namespace csscan_host {
int mimo_bf16(const MimoArgs& a, cudaStream_t st) { return mimo_detail::mimo_dispatch<uint16_t>(a, st); }
int mimo_backward_bf16(const MimoBwdArgs& a, cudaStream_t st) {
  return mimo_detail::mimo_backward_dispatch<uint16_t>(a, st);
}
}  // namespace csscan_host
