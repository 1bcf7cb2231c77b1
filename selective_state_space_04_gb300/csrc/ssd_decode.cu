// ssd_decode.cu -- one step of the SSD recurrence (L = 1): the decode step.
//
// With a single time step the scan is the recurrence applied once to the
// carried state (the direct form of the SSD module's ssd_chunk_forward on the
// @seanhogg/builderforce-memory-engine 2026.6.18 page: decay the state, add
// the input term, read out from the updated state, add the skip):
//   h[p,n] = dA * h[p,n] + dt * B[n] * x[p]        dt = softplus(dt_raw + dt_bias)
//   y[p]   = sum_n C[n] * h[p,n] + D * x[p]        dA = exp(dt * A), A = -exp(A_log)
// per (batch row b, head h), state stored [P, N] (n fastest).
//
// The work is streaming the state in and out (P*N*4 bytes each way per (b, h)
// against P + 2N values of x, B, C), so the layout is chosen for the memory
// system: one CTA of 4 warps per (b, h); a warp owns whole state rows p, lane l
// holding n = 4l .. 4l+3 (+128 per further float4), so every state load and
// store of a warp is one coalesced 512-byte row.  The readout is a warp
// shuffle reduction.  A warp issues the loads of all its rows before it uses
// the first, so several rows per warp are in flight.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ssd_internal.h"

namespace ssd {
namespace {

// 4 warps of 8 rows in flight measured best on the 2.7B layer's decode step
// (100.7 us against 112.7 for 8 warps of 8 rows, 104.1 for 4 of 4, 239.5 for 8 of 16)
constexpr int kWarps = 4;
constexpr int kRowsPerWarp = 8;   // rows of one warp in flight together

struct DecodeParams {
    const void *x;
    const float *dt_raw, *dt_bias, *A_log, *D;
    const void *B, *C;
    const float *init_state;   // may be null (zero state)
    void *y;
    float *final_state;        // may be null
    int H, P, N, G;
};

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v)
{
    return __float2bfloat16_rn(v);
}

__device__ __forceinline__ float softplus_f32(float z)
{
    return fmaxf(z, 0.f) + log1pf(expf(-fabsf(z)));
}

// NV: float4 chunks of a state row per lane (N <= 128 * NV)
template <typename T, int NV>
__global__ void __launch_bounds__(kWarps * 32) ssd_decode_kernel(DecodeParams p)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = p.H, P = p.P, N = p.N;
    const long long bh = blockIdx.x;   // b * H + h
    const long long b = bh / H;
    const int h = (int)(bh - b * H);
    const int g = h / (H / p.G);

    const float dt = softplus_f32(p.dt_raw[bh] + p.dt_bias[h]);
    const float dA = expf(dt * -expf(p.A_log[h]));
    const float Dh = p.D[h];

    // B and C of this group: lane l holds n = 4l + 128 k + {0..3}
    const T *Bg = static_cast<const T *>(p.B) + (b * p.G + g) * (long long)N;
    const T *Cg = static_cast<const T *>(p.C) + (b * p.G + g) * (long long)N;
    float bv[NV][4], cv[NV][4];
#pragma unroll
    for (int k = 0; k < NV; ++k)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int n = 4 * lane + 128 * k + e;
            bv[k][e] = n < N ? to_f32<T>(Bg[n]) : 0.f;
            cv[k][e] = n < N ? to_f32<T>(Cg[n]) : 0.f;
        }
    const T *xg = static_cast<const T *>(p.x) + bh * P;
    T *yg = static_cast<T *>(p.y) + bh * P;
    const size_t sbase = (size_t)bh * P * N;

    // rows p = warp * kRowsPerWarp + i, then the next block of kWarps * kRowsPerWarp rows
    for (int p0 = warp * kRowsPerWarp; p0 < P; p0 += kWarps * kRowsPerWarp) {
        float4 hv[kRowsPerWarp][NV];
        float xv[kRowsPerWarp];
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
            const int pr = p0 + i;
            xv[i] = pr < P ? to_f32<T>(xg[pr]) : 0.f;
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const int n = 4 * lane + 128 * k;
                hv[i][k] = (p.init_state && pr < P && n < N)
                               ? __ldcs(reinterpret_cast<const float4 *>(p.init_state + sbase + (size_t)pr * N + n))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
            const int pr = p0 + i;
            const float dtx = dt * xv[i];
            float acc = 0.f;
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                float4 &v = hv[i][k];
                v.x = fmaf(dA, v.x, dtx * bv[k][0]);
                v.y = fmaf(dA, v.y, dtx * bv[k][1]);
                v.z = fmaf(dA, v.z, dtx * bv[k][2]);
                v.w = fmaf(dA, v.w, dtx * bv[k][3]);
                acc = fmaf(cv[k][0], v.x, acc);
                acc = fmaf(cv[k][1], v.y, acc);
                acc = fmaf(cv[k][2], v.z, acc);
                acc = fmaf(cv[k][3], v.w, acc);
                const int n = 4 * lane + 128 * k;
                if (p.final_state && pr < P && n < N)
                    __stcs(reinterpret_cast<float4 *>(p.final_state + sbase + (size_t)pr * N + n), v);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0 && pr < P)
                yg[pr] = from_f32<T>(fmaf(Dh, xv[i], acc));
        }
    }
}

template <typename T, int NV>
cudaError_t launch_nv(const DecodeParams &dp, long long grid, cudaStream_t st)
{
    ssd_decode_kernel<T, NV><<<(unsigned)grid, kWarps * 32, 0, st>>>(dp);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(int nv, const DecodeParams &dp, long long grid, cudaStream_t st)
{
    switch (nv) {
    case 1: return launch_nv<T, 1>(dp, grid, st);
    case 2: return launch_nv<T, 2>(dp, grid, st);
    case 4: return launch_nv<T, 4>(dp, grid, st);
    default: return cudaErrorInvalidValue;
    }
}

int decode_nv(int N)
{
    return N <= 128 ? 1 : (N <= 256 ? 2 : 4);
}

}  // namespace

bool decode_supported(const ScanArgs &a)
{
    // whole float4 chunks of a state row (16-byte aligned rows), at most 512 states
    return a.seqlen == 1 && a.dstate % 4 == 0 && a.dstate <= 512 && a.headdim >= 1 &&
           a.batch * (long long)a.nheads <= 0x7FFFFFFFLL;
}

cudaError_t decode_launch(const ScanArgs &a, cudaStream_t stream)
{
    SSD_NVTX_RANGE("decode_launch");
    if (!decode_supported(a))
        return cudaErrorInvalidValue;
    DecodeParams dp;
    dp.x = a.x;
    dp.dt_raw = a.dt_raw;
    dp.dt_bias = a.dt_bias;
    dp.A_log = a.A_log;
    dp.D = a.D;
    dp.B = a.B;
    dp.C = a.C;
    dp.init_state = a.init_state;
    dp.y = a.y;
    dp.final_state = a.final_state;
    dp.H = a.nheads;
    dp.P = a.headdim;
    dp.N = a.dstate;
    dp.G = a.ngroups;
    const long long grid = a.batch * (long long)a.nheads;
    const int nv = decode_nv(a.dstate);
    cudaError_t e = a.dtype == SSD_DTYPE_BF16 ? launch_t<__nv_bfloat16>(nv, dp, grid, stream)
                                              : launch_t<float>(nv, dp, grid, stream);
    if (e == cudaSuccess)
        note_launches(1);
    return e;
}

}  // namespace ssd
