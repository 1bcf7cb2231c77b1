// warp_rows.cuh -- sums of several per-lane values over a warp at once.
#pragma once

namespace ssd {

// Sums each of the R values over the warp's 32 lanes at once (R a power of two
// <= 32): each butterfly stage exchanges half of the values still held, so R
// rows take R - 1 + log2(32 / R) shuffles instead of 5 R.  Afterwards vals[0]
// of lane l is the total of row summed_row<R>(l).
template <int R>
__device__ __forceinline__ void warp_sum_rows_all(float (&vals)[R], int lane)
{
    int cnt = R;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        if (cnt > 1) {
            const int half = cnt >> 1;
            const bool upper = (lane & o) != 0;
#pragma unroll
            for (int j = 0; j < R / 2; ++j) {
                if (j < half) {
                    const float send = upper ? vals[j] : vals[j + half];
                    const float keep = upper ? vals[j + half] : vals[j];
                    vals[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
            cnt = half;
        } else {
            vals[0] += __shfl_xor_sync(0xffffffffu, vals[0], o);
        }
    }
}

// the row whose total lane l holds after warp_sum_rows_all<R>
template <int R>
__device__ __forceinline__ int summed_row(int lane)
{
    int row = 0, half = R >> 1;
#pragma unroll
    for (int o = 16; o >= 1 && half >= 1; o >>= 1, half >>= 1)
        if (lane & o)
            row += half;
    return row;
}

}  // namespace ssd
