// q8_gemv_vt_m4.cu -- instantiations of the virtual-tile GEMV for passes of
// up to 4 activation rows.
#include "q8_gemv_vt.cuh"

namespace q8 {
namespace vt {
Q8_VT_INSTANTIATE(4)
}  // namespace vt
}  // namespace q8
