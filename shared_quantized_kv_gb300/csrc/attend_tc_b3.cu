// Tensor-core attention instances for layers with 3-bit V codes (one
// translation unit per bit width keeps the build parallel).
#include "attend_tc_impl.cuh"

namespace kvp {
template cudaError_t launch_attend_tc_bits<3>(const Shape&, const LayerBufs&, const AttendArgs&, int*,
                                               cudaStream_t);
}  // namespace kvp
