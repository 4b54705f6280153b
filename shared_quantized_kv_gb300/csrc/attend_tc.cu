// Dispatch of the tensor-core attention by V bit width (the kernel and its
// launcher are in attend_rows.cuh; one instance file per width, and one for
// layers of per-group widths).
#include "kvpool_internal.cuh"

namespace kvp {

template <int BITS, bool MIX>
cudaError_t launch_attend_rows_bits(const Shape& s, const LayerBufs& L, const AttendArgs& a, int* status,
                                    cudaStream_t st);
extern template cudaError_t launch_attend_rows_bits<2, false>(const Shape&, const LayerBufs&, const AttendArgs&,
                                                               int*, cudaStream_t);
extern template cudaError_t launch_attend_rows_bits<3, false>(const Shape&, const LayerBufs&, const AttendArgs&,
                                                               int*, cudaStream_t);
extern template cudaError_t launch_attend_rows_bits<4, false>(const Shape&, const LayerBufs&, const AttendArgs&,
                                                               int*, cudaStream_t);
extern template cudaError_t launch_attend_rows_bits<3, true>(const Shape&, const LayerBufs&, const AttendArgs&,
                                                              int*, cudaStream_t);
extern template cudaError_t launch_attend_rows_bits<4, true>(const Shape&, const LayerBufs&, const AttendArgs&,
                                                              int*, cudaStream_t);

cudaError_t launch_attend_tc(const Shape& s, const LayerBufs& L, const AttendArgs& a, int* status,
                             int sm_count, cudaStream_t st) {
    (void)sm_count;
    if (L.mixed) {  // per-group widths: at most the layer's width, which is then 3 or 4
        if (L.bits == 3) return launch_attend_rows_bits<3, true>(s, L, a, status, st);
        if (L.bits == 4) return launch_attend_rows_bits<4, true>(s, L, a, status, st);
        return cudaErrorInvalidValue;
    }
    if (L.bits == 2) return launch_attend_rows_bits<2, false>(s, L, a, status, st);
    if (L.bits == 3) return launch_attend_rows_bits<3, false>(s, L, a, status, st);
    return launch_attend_rows_bits<4, false>(s, L, a, status, st);
}

}  // namespace kvp
