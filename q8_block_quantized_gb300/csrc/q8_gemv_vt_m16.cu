// q8_gemv_vt_m16.cu -- instantiations of the virtual-tile GEMV for passes of
// up to 16 activation rows.
#include "q8_gemv_vt.cuh"

namespace q8 {
namespace vt {
Q8_VT_INSTANTIATE(16)
}  // namespace vt
}  // namespace q8
