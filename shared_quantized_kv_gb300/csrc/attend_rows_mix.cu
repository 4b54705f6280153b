// Row-per-thread tensor-core attention instances for block-scaled layers whose
// 32-token groups have their own V widths (at most 3 or 4 bits).
#include "attend_rows.cuh"

namespace kvp {
template cudaError_t launch_attend_rows_bits<3, true>(const Shape&, const LayerBufs&, const AttendArgs&, int*,
                                                      cudaStream_t);
template cudaError_t launch_attend_rows_bits<4, true>(const Shape&, const LayerBufs&, const AttendArgs&, int*,
                                                      cudaStream_t);
}  // namespace kvp
