// q8_gemv_vt_m32.cu -- instantiations of the virtual-tile GEMV for passes of
// up to 32 activation rows.
#include "q8_gemv_vt.cuh"

namespace q8 {
namespace vt {
Q8_VT_INSTANTIATE(32)
}  // namespace vt
}  // namespace q8
