// q8_gemv_r128.cu -- instantiations of the GEMV kernel for 128-row tiles.
#include "q8_gemv_impl.cuh"

namespace q8 {
Q8_INSTANTIATE_R(128)
}  // namespace q8
