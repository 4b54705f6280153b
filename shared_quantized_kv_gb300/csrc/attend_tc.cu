// Dispatch of the tensor-core attention by V bit width (the kernel and its
// launcher are in attend_rows.cuh; one instance file per width).
#include "kvpool_internal.cuh"

namespace kvp {

template <int BITS>
cudaError_t launch_attend_rows_bits(const Shape& s, const LayerBufs& L, const AttendArgs& a, int* status,
                                    cudaStream_t st);
extern template cudaError_t launch_attend_rows_bits<2>(const Shape&, const LayerBufs&, const AttendArgs&,
                                                        int*, cudaStream_t);
extern template cudaError_t launch_attend_rows_bits<3>(const Shape&, const LayerBufs&, const AttendArgs&,
                                                        int*, cudaStream_t);
extern template cudaError_t launch_attend_rows_bits<4>(const Shape&, const LayerBufs&, const AttendArgs&,
                                                        int*, cudaStream_t);

cudaError_t launch_attend_tc(const Shape& s, const LayerBufs& L, const AttendArgs& a, int* status,
                             int sm_count, cudaStream_t st) {
    (void)sm_count;
    if (L.bits == 2) return launch_attend_rows_bits<2>(s, L, a, status, st);
    if (L.bits == 3) return launch_attend_rows_bits<3>(s, L, a, status, st);
    return launch_attend_rows_bits<4>(s, L, a, status, st);
}

}  // namespace kvp
