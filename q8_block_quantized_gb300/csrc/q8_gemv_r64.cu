// q8_gemv_r64.cu -- instantiations of the GEMV kernel for 64-row tiles.
#include "q8_gemv_impl.cuh"

namespace q8 {
Q8_INSTANTIATE_R(64)
}  // namespace q8
