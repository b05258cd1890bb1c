// q8_gemv_r32.cu -- instantiations of the GEMV kernel for 32-row tiles.
#include "q8_gemv_impl.cuh"

namespace q8 {
Q8_INSTANTIATE_R(32)
}  // namespace q8
