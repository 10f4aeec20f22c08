// backward_f32.cu -- csscan_backward for float32 inputs (one translation unit per input dtype, so
// that the library's units compile in parallel).
#include "backward_launch.cuh"

namespace csscan_host {
int backward_f32(const BwdArgs& a, cudaStream_t st) { return backward_dispatch<float>(a, st); }
}  // namespace csscan_host
