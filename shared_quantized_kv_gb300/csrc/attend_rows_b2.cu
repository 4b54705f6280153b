// Row-per-thread tensor-core attention instances for layers with 2-bit V
// codes (one translation unit per bit width keeps the build parallel).
#include "attend_rows.cuh"

namespace kvp {
template cudaError_t launch_attend_rows_bits<2, false>(const Shape&, const LayerBufs&, const AttendArgs&, int*,
                                                         cudaStream_t);
}  // namespace kvp
