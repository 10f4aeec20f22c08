// mimo_f32.cu -- csscan_forward_mimo and csscan_backward_mimo for float32 inputs (mimo_launch.cuh).
#include "mimo_launch.cuh"

namespace csscan_host {
int mimo_f32(const MimoArgs& a, cudaStream_t st) { return mimo_detail::mimo_dispatch<float>(a, st); }
int mimo_backward_f32(const MimoBwdArgs& a, cudaStream_t st) {
  return mimo_detail::mimo_backward_dispatch<float>(a, st);
}
}  // namespace csscan_host
