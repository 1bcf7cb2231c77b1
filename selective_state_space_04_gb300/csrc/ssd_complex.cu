// ssd_complex.cu -- the complex-valued scan with exponential-trapezoidal (ET)
// discretisation (the Mamba-3 complex SSD module of the pages, as its header
// defines it), sequential in time.
//
// Per batch row b and head h, with A = exp(log|A| + i arg A) (polar pair per
// head) and dt_t = softplus(dt_raw_t + dt_bias):
//   A_bar_t = exp(dt_t A),   B_bar_t = (A_bar_t - 1) A^-1 B_t   (the exact hold)
//   h_t = A_bar_t h_{t-1} + B_bar_t x_t^T,   y_t = Re(C_t^T h_t) + D x_t
// B, C and the state hold N/2 complex numbers as (re, im) pairs along N.
//
// Layout as the trapezoidal scan: one CTA per (b, h), one warp per block of
// state rows p, lane l holding n = 4l .. 4l+3 (two complex components, +128
// per further float4) of each of its rows, so the state is read and written as
// coalesced 512-byte rows and stays in registers for the whole sequence.  Time
// is walked in blocks: A_bar per step, B_bar = (A_bar - 1) A^-1 B (the complex
// scalar times the complex B, formed once per step and component while
// staging), C and x are staged in shared memory; y_t[p] is a warp reduction.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "f32x2.cuh"
#include "ssd_internal.h"
#include "warp_rows.cuh"

namespace ssd {
namespace {

struct CplxParams {
    const void *x, *B, *C;            // x [B,L,H,P]; B, C [B,L,G,N] (interleaved re, im)
    const float *dt_raw, *dt_bias, *A_polar, *D;
    const float *h0;                  // [B,H,P,N] or null
    void *y;
    float *h_final;                   // [B,H,P,N] or null
    long long L;
    int H, P, N, G, tblk;
    int Pp;                           // staged x row stride: the CTA's rows (warps x rows per warp)
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

__device__ __forceinline__ float softplus_f32(float z) { return fmaxf(z, 0.f) + log1pf(expf(-fabsf(z))); }

constexpr int kStateFloat4PerLane = 8;   // RPW * NV float4 of state per lane
constexpr int kMaxWarps = 16;

template <typename T, int NV>
__global__ void __launch_bounds__(kMaxWarps * 32) ssd_complex_seq_kernel(CplxParams p)
{
    constexpr int RPW = kStateFloat4PerLane / NV;
    extern __shared__ float sm[];
    const int P = p.P, N = p.N, H = p.H, TB = p.tblk;
    const long long L = p.L;
    // B_bar and C staged per 4-float group of two components k, k+1 as
    // (re_k, re_k+1, im_k, im_k+1), C's imaginary parts negated: the packed
    // arithmetic below then takes pairs straight from the 16-byte loads
    float *bb = sm;                  // [TB][N]: B_bar
    float *cs = bb + TB * N;         // [TB][N]: C (re, re, -im, -im)
    float *xs = cs + TB * N;         // [TB][Pp], zero past P
    float *ab = xs + TB * p.Pp;      // [TB][4]: A_bar (re, im), (A_bar - 1) A^-1 (re, im)
    const int Pp = p.Pp;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nthr = blockDim.x;
    const long long bh = blockIdx.x;
    const long long b = bh / H;
    const int h = (int)(bh - b * H);
    const int g = h / (H / p.G);
    const int p0 = warp * RPW;
    const T *xg = static_cast<const T *>(p.x), *Bg = static_cast<const T *>(p.B), *Cg = static_cast<const T *>(p.C);
    T *yg = static_cast<T *>(p.y);
    const size_t sbase = (size_t)bh * P * N;

    // A = |A| (cos arg, sin arg); A^-1 = (cos arg, -sin arg) / |A|
    const float lm = p.A_polar[2 * h], ph = p.A_polar[2 * h + 1];
    float sph, cph;
    sincosf(ph, &sph, &cph);
    const float mag = expf(lm), imag_ = expf(-lm);
    const float Ar = mag * cph, Ai = mag * sph, Ir = imag_ * cph, Ii = -imag_ * sph;
    const float Dh = p.D[h];

    // (re, re) and (im, im) of components n/2, n/2 + 1 (the state is stored (re, im, re, im))
    f32x2 hre[RPW][NV], him[RPW][NV];
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        const int pr = p0 + r;
#pragma unroll
        for (int c = 0; c < NV; ++c) {
            const int n = 4 * lane + 128 * c;
            const float4 v = (p.h0 && pr < P && n < N)
                                 ? __ldcs(reinterpret_cast<const float4 *>(p.h0 + sbase + (size_t)pr * N + n))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
            hre[r][c] = pk2(v.x, v.z);
            him[r][c] = pk2(v.y, v.w);
        }
    }

    for (long long t0 = 0; t0 < L; t0 += TB) {
        const int nt = (int)min((long long)TB, L - t0);
        __syncthreads();   // the previous block is consumed
        for (int i = threadIdx.x; i < nt; i += nthr) {
            const float dt = softplus_f32(p.dt_raw[(size_t)(b * L + t0 + i) * H + h] + p.dt_bias[h]);
            float s, c;
            sincosf(dt * Ai, &s, &c);
            const float e = expf(dt * Ar);
            const float abr = e * c, abi = e * s;
            ab[4 * i + 0] = abr;
            ab[4 * i + 1] = abi;
            ab[4 * i + 2] = (abr - 1.f) * Ir - abi * Ii;   // (A_bar - 1) A^-1
            ab[4 * i + 3] = (abr - 1.f) * Ii + abi * Ir;
        }
        for (int i = threadIdx.x; i < nt * Pp; i += nthr) {
            const int tt = i / Pp, pp = i - tt * Pp;
            xs[i] = pp < P ? to_f32<T>(xg[((size_t)(b * L + t0 + tt) * H + h) * P + pp]) : 0.f;
        }
        __syncthreads();
        const int K = N / 2;
        for (int i = threadIdx.x; i < nt * K; i += nthr) {
            const int tt = i / K, k = i - tt * K;
            const size_t gi = ((size_t)(b * L + t0 + tt) * p.G + g) * N + 2 * k;
            const float br = to_f32<T>(Bg[gi]), bi = to_f32<T>(Bg[gi + 1]);
            const float fr = ab[4 * tt + 2], fi = ab[4 * tt + 3];
            const int o = tt * N + 4 * (k >> 1) + (k & 1);   // re at o, im at o + 2
            bb[o] = fr * br - fi * bi;
            bb[o + 2] = fr * bi + fi * br;
            cs[o] = to_f32<T>(Cg[gi]);
            cs[o + 2] = -to_f32<T>(Cg[gi + 1]);
        }
        __syncthreads();
        // unrolled: the readout reductions of a step (shuffle chains, not on the
        // recurrence) overlap the next steps' state updates
#pragma unroll 4
        for (int i = 0; i < nt; ++i) {
            const float abr = ab[4 * i], abi = ab[4 * i + 1];
            const f32x2 abr2 = pk2(abr, abr), abi2 = pk2(abi, abi), nabi2 = pk2(-abi, -abi);
            float4 bt[NV], ct[NV];
#pragma unroll
            for (int c = 0; c < NV; ++c) {
                const int n = 4 * lane + 128 * c;
                const bool in = n < N;   // N % 4 == 0: whole float4 chunks
                bt[c] = in ? *reinterpret_cast<const float4 *>(bb + i * N + n) : make_float4(0.f, 0.f, 0.f, 0.f);
                ct[c] = in ? *reinterpret_cast<const float4 *>(cs + i * N + n) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            float acc[RPW], xr[RPW];   // this warp's RPW rows of x_t: 16- or 8-byte loads
            if constexpr (RPW >= 4) {
#pragma unroll
                for (int v = 0; v < RPW / 4; ++v) {
                    const float4 x4 = *reinterpret_cast<const float4 *>(xs + i * Pp + p0 + 4 * v);
                    xr[4 * v] = x4.x;
                    xr[4 * v + 1] = x4.y;
                    xr[4 * v + 2] = x4.z;
                    xr[4 * v + 3] = x4.w;
                }
            } else {
                const float2 x2 = *reinterpret_cast<const float2 *>(xs + i * Pp + p0);
                xr[0] = x2.x;
                xr[1] = x2.y;
            }
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
                const f32x2 x2 = pk2(xr[r], xr[r]);
                f32x2 s = pk2(0.f, 0.f);
#pragma unroll
                for (int c = 0; c < NV; ++c) {
                    // h <- A_bar h + B_bar x, per component in the order
                    // re = abr re + (-abi im + Br x), im = abr im + (abi re + Bi x)
                    const f32x2 re = hre[r][c], im = him[r][c];
                    const f32x2 nre = fma2(abr2, re, fma2(nabi2, im, mul2(pk2(bt[c].x, bt[c].y), x2)));
                    const f32x2 nim = fma2(abr2, im, fma2(abi2, re, mul2(pk2(bt[c].z, bt[c].w), x2)));
                    hre[r][c] = nre;
                    him[r][c] = nim;
                    s = fma2(pk2(ct[c].x, ct[c].y), nre, s);   // Re(C h) = Cr hr - Ci hi
                    s = fma2(pk2(ct[c].z, ct[c].w), nim, s);
                }
                acc[r] = lo2(s) + hi2(s);
            }
            warp_sum_rows_all<RPW>(acc, lane);
            const int pr = p0 + summed_row<RPW>(lane);
            if ((lane & (32 / RPW - 1)) == 0 && pr < P)
                yg[((size_t)(b * L + t0 + i) * H + h) * P + pr] = from_f32<T>(fmaf(Dh, xs[i * Pp + pr], acc[0]));
        }
    }

    if (p.h_final) {
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            const int pr = p0 + r;
#pragma unroll
            for (int c = 0; c < NV; ++c) {
                const int n = 4 * lane + 128 * c;
                if (pr < P && n < N)
                    __stcs(reinterpret_cast<float4 *>(p.h_final + sbase + (size_t)pr * N + n),
                           make_float4(lo2(hre[r][c]), lo2(him[r][c]), hi2(hre[r][c]), hi2(him[r][c])));
            }
        }
    }
}

// One step (seqlen 1): a stream of the state.  One CTA of 4 warps per (b, h),
// no shared memory and no barrier; each warp takes blocks of 8 rows, loads all
// of a block's state before using it, writes the updated rows straight back
// and reduces each row's readout with shuffles.
constexpr int kDecWarps = 4, kDecRows = 8;

template <typename T, int NV>
__global__ void __launch_bounds__(kDecWarps * 32, NV == 1 ? 5 : 1) ssd_complex_decode_kernel(CplxParams p)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = p.H, P = p.P, N = p.N;
    const long long bh = blockIdx.x;   // b * H + h (seqlen 1: also the token index)
    const long long b = bh / H;
    const int h = (int)(bh - b * H), g = h / (H / p.G);
    const float lm = p.A_polar[2 * h], ph = p.A_polar[2 * h + 1];
    float sph, cph;
    sincosf(ph, &sph, &cph);
    const float mag = expf(lm), imag_ = expf(-lm);
    const float Ar = mag * cph, Ai = mag * sph, Ir = imag_ * cph, Ii = -imag_ * sph;
    const float dt = softplus_f32(p.dt_raw[bh] + p.dt_bias[h]);
    float s, c;
    sincosf(dt * Ai, &s, &c);
    const float e = expf(dt * Ar);
    const float abr = e * c, abi = e * s;
    const float fr = (abr - 1.f) * Ir - abi * Ii, fi = (abr - 1.f) * Ii + abi * Ir;   // (A_bar - 1) A^-1
    const float Dh = p.D[h];
    const T *Bg = static_cast<const T *>(p.B) + (b * p.G + g) * (long long)N;
    const T *Cg = static_cast<const T *>(p.C) + (b * p.G + g) * (long long)N;
    float bb[NV][4], cv[NV][4];   // this lane's B_bar and C: two complex components per float4
#pragma unroll
    for (int q = 0; q < NV; ++q) {
        const int n = 4 * lane + 128 * q;
        float bv[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            bv[k] = n < N ? to_f32<T>(Bg[n + k]) : 0.f;
            cv[q][k] = n < N ? to_f32<T>(Cg[n + k]) : 0.f;
        }
        bb[q][0] = fr * bv[0] - fi * bv[1];
        bb[q][1] = fr * bv[1] + fi * bv[0];
        bb[q][2] = fr * bv[2] - fi * bv[3];
        bb[q][3] = fr * bv[3] + fi * bv[2];
    }
    const T *xg = static_cast<const T *>(p.x) + bh * P;
    T *yg = static_cast<T *>(p.y) + bh * P;
    const size_t sbase = (size_t)bh * P * N;
    for (int p0 = warp * kDecRows; p0 < P; p0 += kDecWarps * kDecRows) {
        float4 hv[kDecRows][NV];
        float xv[kDecRows];
#pragma unroll
        for (int i = 0; i < kDecRows; ++i) {
            const int pr = p0 + i;
            xv[i] = pr < P ? to_f32<T>(xg[pr]) : 0.f;
#pragma unroll
            for (int q = 0; q < NV; ++q) {
                const int n = 4 * lane + 128 * q;
                hv[i][q] = (p.h0 && pr < P && n < N)
                               ? __ldcs(reinterpret_cast<const float4 *>(p.h0 + sbase + (size_t)pr * N + n))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int i = 0; i < kDecRows; ++i) {
            const int pr = p0 + i;
            float acc = 0.f;
#pragma unroll
            for (int q = 0; q < NV; ++q) {
                const float4 z = hv[i][q];
                const float r0 = fmaf(abr, z.x, fmaf(-abi, z.y, bb[q][0] * xv[i]));
                const float i0 = fmaf(abr, z.y, fmaf(abi, z.x, bb[q][1] * xv[i]));
                const float r1 = fmaf(abr, z.z, fmaf(-abi, z.w, bb[q][2] * xv[i]));
                const float i1 = fmaf(abr, z.w, fmaf(abi, z.z, bb[q][3] * xv[i]));
                acc = fmaf(cv[q][0], r0, acc);   // Re(C h)
                acc = fmaf(-cv[q][1], i0, acc);
                acc = fmaf(cv[q][2], r1, acc);
                acc = fmaf(-cv[q][3], i1, acc);
                const int n = 4 * lane + 128 * q;
                if (p.h_final && pr < P && n < N)
                    __stcs(reinterpret_cast<float4 *>(p.h_final + sbase + (size_t)pr * N + n),
                           make_float4(r0, i0, r1, i1));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0 && pr < P)
                yg[pr] = from_f32<T>(fmaf(Dh, xv[i], acc));
        }
    }
}

int complex_nv(int N) { return N <= 128 ? 1 : N <= 256 ? 2 : 4; }

}  // namespace

bool complex_supported(const ComplexArgs &a)
{
    if (a.dstate % 4 != 0 || a.dstate < 4 || a.dstate > 512 || a.headdim < 1)
        return false;
    const int rows = kStateFloat4PerLane / complex_nv(a.dstate);
    return a.headdim <= kMaxWarps * rows && a.batch * (long long)a.nheads <= 0x7FFFFFFFLL &&
           a.seqlen < (1LL << 31);
}

cudaError_t complex_launch(const ComplexArgs &a, cudaStream_t st)
{
    SSD_NVTX_RANGE("complex_launch");
    if (!complex_supported(a))
        return cudaErrorInvalidValue;
    CplxParams p;
    p.x = a.x;
    p.B = a.B;
    p.C = a.C;
    p.dt_raw = a.dt_raw;
    p.dt_bias = a.dt_bias;
    p.A_polar = a.A_polar;
    p.D = a.D;
    p.h0 = a.init_state;
    p.y = a.y;
    p.h_final = a.final_state;
    p.L = a.seqlen;
    p.H = a.nheads;
    p.P = a.headdim;
    p.N = a.dstate;
    p.G = a.ngroups;
    const int nv = complex_nv(a.dstate), rows = kStateFloat4PerLane / nv;
    const int warps = (a.headdim + rows - 1) / rows;
    p.Pp = warps * rows;
    // steps per staged block: up to 64, within about 200 KB of shared memory
    const long long per_step = (long long)(2 * a.dstate + p.Pp + 4) * (long long)sizeof(float);
    p.tblk = (int)std::max<long long>(1, std::min<long long>({64LL, a.seqlen, (200LL << 10) / per_step}));
    const size_t smem = (size_t)(p.tblk * (2 * a.dstate + p.Pp + 4)) * sizeof(float);
    const dim3 grid((unsigned)(a.batch * a.nheads));
    const bool bf = a.dtype == SSD_DTYPE_BF16;
    if (a.seqlen == 1) {   // the decode step: the specialised stream of the state
        if (nv == 1)
            bf ? ssd_complex_decode_kernel<__nv_bfloat16, 1><<<grid, kDecWarps * 32, 0, st>>>(p)
               : ssd_complex_decode_kernel<float, 1><<<grid, kDecWarps * 32, 0, st>>>(p);
        else if (nv == 2)
            bf ? ssd_complex_decode_kernel<__nv_bfloat16, 2><<<grid, kDecWarps * 32, 0, st>>>(p)
               : ssd_complex_decode_kernel<float, 2><<<grid, kDecWarps * 32, 0, st>>>(p);
        else
            bf ? ssd_complex_decode_kernel<__nv_bfloat16, 4><<<grid, kDecWarps * 32, 0, st>>>(p)
               : ssd_complex_decode_kernel<float, 4><<<grid, kDecWarps * 32, 0, st>>>(p);
        const cudaError_t e = cudaGetLastError();
        if (e == cudaSuccess)
            note_launches(1);
        return e;
    }
#define SSD_CPLX_LAUNCH(NVV)                                                                                    \
    do {                                                                                                         \
        if (bf)                                                                                                  \
            ssd_complex_seq_kernel<__nv_bfloat16, NVV><<<grid, 32 * warps, smem, st>>>(p);                       \
        else                                                                                                     \
            ssd_complex_seq_kernel<float, NVV><<<grid, 32 * warps, smem, st>>>(p);                               \
    } while (0)
    if (smem > 48 * 1024) {
        const cudaError_t e =
            nv == 1 ? (bf ? cudaFuncSetAttribute(ssd_complex_seq_kernel<__nv_bfloat16, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)
                          : cudaFuncSetAttribute(ssd_complex_seq_kernel<float, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem))
            : nv == 2 ? (bf ? cudaFuncSetAttribute(ssd_complex_seq_kernel<__nv_bfloat16, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)
                            : cudaFuncSetAttribute(ssd_complex_seq_kernel<float, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem))
                      : (bf ? cudaFuncSetAttribute(ssd_complex_seq_kernel<__nv_bfloat16, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)
                            : cudaFuncSetAttribute(ssd_complex_seq_kernel<float, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        if (e != cudaSuccess)
            return e;
    }
    if (nv == 1)
        SSD_CPLX_LAUNCH(1);
    else if (nv == 2)
        SSD_CPLX_LAUNCH(2);
    else
        SSD_CPLX_LAUNCH(4);
#undef SSD_CPLX_LAUNCH
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess)
        note_launches(1);
    return e;
}

}  // namespace ssd
