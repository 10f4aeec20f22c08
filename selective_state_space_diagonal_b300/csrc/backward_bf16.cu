// backward_bf16.cu -- csscan_backward for bf16 inputs (one translation unit per input dtype, so
// that the library's units compile in parallel).
#include "backward_launch.cuh"

namespace csscan_host {
int backward_bf16(const BwdArgs& a, cudaStream_t st) { return backward_dispatch<uint16_t>(a, st); }
}  // namespace csscan_host
