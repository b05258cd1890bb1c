// q8_gemv_r16.cu -- instantiations of the GEMV kernel for 16-row tiles.
#include "q8_gemv_impl.cuh"

namespace q8 {
Q8_INSTANTIATE_R(16)
}  // namespace q8
