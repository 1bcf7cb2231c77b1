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

// staged x elements per thread and block for CTAs of one or two warps:
// 64 steps x (2 warps x RPW rows) / 64 threads
constexpr int kXPerThread = 64 * kStateFloat4PerLane / 32;
constexpr int kSmallWarps = 8;   // CTAs of up to 8 warps: 3 (N <= 128) or 2 per SM

// asynchronous 16- and 8-byte copies of B or C rows into the staging area
// (completed by cp.async.wait_all)
template <typename T>
__device__ __forceinline__ void cp_async16(T *dst, const T *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((unsigned)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
template <typename T>
__device__ __forceinline__ void cp_async8(T *dst, const T *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"((unsigned)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
// 4 staged values (two components as re, im, re, im) as floats
__device__ __forceinline__ float4 load4f(const float *src) { return *reinterpret_cast<const float4 *>(src); }
__device__ __forceinline__ float4 load4f(const __nv_bfloat16 *src)
{
    const uint2 v = *reinterpret_cast<const uint2 *>(src);
    return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u), __uint_as_float(v.y << 16),
                       __uint_as_float(v.y & 0xffff0000u));
}

// One CTA per (b, h), one warp per block of RPW state rows p, lane l holding
// the components n/2, n/2 + 1 of n = 4l (+128 per further float4) of each row,
// kept in registers as (re, re) and (im, im) pairs.  Per time block (up to 64
// steps) the CTA stages B_t and C_t as stored (bf16 stays bf16) by cp.async
// copies, x_t as fp32 and the step's coefficients A_bar_t and (A_bar_t - 1) A^-1;
// each lane forms B_bar = ((A_bar - 1) A^-1) B for its two components at use,
// once per step for all of its rows.
template <typename T, int NV, int MAXT, int MINB>
__global__ void __launch_bounds__(MAXT, MINB) ssd_complex_seq_kernel(CplxParams p)
{
    constexpr int RPW = kStateFloat4PerLane / NV;
    extern __shared__ float sm[];
    const int P = p.P, N = p.N, H = p.H, TB = p.tblk;
    const long long L = p.L;
    const int Pp = p.Pp;
    float *xs = sm;                  // [TB][Pp], zero past P
    float *ab = xs + TB * Pp;        // [TB][4]: A_bar (re, im), (A_bar - 1) A^-1 (re, im)
    T *bs = reinterpret_cast<T *>(sm + ((TB * (Pp + 4) + 3) & ~3));   // [TB][N]: B_t as stored (16-byte aligned)
    T *cs = bs + (size_t)TB * N;     // [TB][N]: C_t as stored

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nthr = blockDim.x, nwarps = nthr >> 5;
    const long long bh = blockIdx.x;
    const long long b = bh / H;
    const int h = (int)(bh - b * H);
    const int g = h / (H / p.G);
    const int p0 = warp * RPW;
    const T *xg = static_cast<const T *>(p.x), *Bg = static_cast<const T *>(p.B), *Cg = static_cast<const T *>(p.C);
    T *yg = static_cast<T *>(p.y);
    const size_t sbase = (size_t)bh * P * N;
    const bool wide16 = (N * (int)sizeof(T)) % 16 == 0;   // staged rows in 16-byte copies

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
        // B_t and C_t by asynchronous copies (all in flight at once)
        if (wide16) {   // 16-byte copies: 8 bf16 or 4 fp32 elements
            constexpr int E = 16 / (int)sizeof(T);
            for (int i = threadIdx.x; i < nt * (N / E); i += nthr) {
                const int tt = i / (N / E), q = E * (i - tt * (N / E));
                const size_t row = ((size_t)(b * L + t0 + tt) * p.G + g) * N;
                cp_async16(bs + (size_t)tt * N + q, Bg + row + q);
                cp_async16(cs + (size_t)tt * N + q, Cg + row + q);
            }
        } else {        // bf16 rows of N % 8 == 4 elements: 8-byte copies
            for (int i = threadIdx.x; i < nt * (N / 4); i += nthr) {
                const int tt = i / (N / 4), q = 4 * (i - tt * (N / 4));
                const size_t row = ((size_t)(b * L + t0 + tt) * p.G + g) * N;
                cp_async8(bs + (size_t)tt * N + q, Bg + row + q);
                cp_async8(cs + (size_t)tt * N + q, Cg + row + q);
            }
        }
        if (nwarps <= 2) {
            // few warps (small P): each thread's x loads all issued before its first store
            float xv[kXPerThread];
#pragma unroll
            for (int k = 0; k < kXPerThread; ++k) {
                const int i = threadIdx.x + k * nthr;
                xv[k] = 0.f;
                if (i < nt * Pp) {
                    const int tt = i / Pp, pp = i - tt * Pp;
                    if (pp < P)
                        xv[k] = to_f32<T>(xg[((size_t)(b * L + t0 + tt) * H + h) * P + pp]);
                }
            }
#pragma unroll
            for (int k = 0; k < kXPerThread; ++k) {
                const int i = threadIdx.x + k * nthr;
                if (i < nt * Pp)
                    xs[i] = xv[k];
            }
        } else {
            for (int tt = warp; tt < nt; tt += nwarps) {
                const size_t row = (size_t)(b * L + t0 + tt);
                for (int pp = lane; pp < Pp; pp += 32)
                    xs[tt * Pp + pp] = pp < P ? to_f32<T>(xg[(row * H + h) * P + pp]) : 0.f;
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        __syncthreads();
        // unrolled: the readout reductions of a step (shuffle chains, not on the
        // recurrence) overlap the next steps' state updates
#pragma unroll 4
        for (int i = 0; i < nt; ++i) {
            const float abr = ab[4 * i], abi = ab[4 * i + 1], fr = ab[4 * i + 2], fi = ab[4 * i + 3];
            const f32x2 abr2 = pk2(abr, abr), abi2 = pk2(abi, abi), nabi2 = pk2(-abi, -abi);
            f32x2 bre[NV], bim[NV], cre[NV], ncim[NV];   // B_bar (re, re), (im, im); C (re, re), (-im, -im)
#pragma unroll
            for (int c = 0; c < NV; ++c) {
                const int n = 4 * lane + 128 * c;
                if (n < N) {   // N % 4 == 0: whole float4 chunks
                    const float4 bv = load4f(bs + (size_t)i * N + n), cv = load4f(cs + (size_t)i * N + n);
                    bre[c] = pk2(fr * bv.x - fi * bv.y, fr * bv.z - fi * bv.w);
                    bim[c] = pk2(fr * bv.y + fi * bv.x, fr * bv.w + fi * bv.z);
                    cre[c] = pk2(cv.x, cv.z);
                    ncim[c] = pk2(-cv.y, -cv.w);
                } else {
                    bre[c] = bim[c] = cre[c] = ncim[c] = pk2(0.f, 0.f);
                }
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
                    const f32x2 nre = fma2(abr2, re, fma2(nabi2, im, mul2(bre[c], x2)));
                    const f32x2 nim = fma2(abr2, im, fma2(abi2, re, mul2(bim[c], x2)));
                    hre[r][c] = nre;
                    him[r][c] = nim;
                    s = fma2(cre[c], nre, s);    // Re(C h) = Cr hr - Ci hi
                    s = fma2(ncim[c], nim, s);
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

template <typename T, int NV, int MAXT, int MINB>
cudaError_t seq_launch_t(const CplxParams &p, dim3 grid, int warps, size_t smem, cudaStream_t st)
{
    auto kern = ssd_complex_seq_kernel<T, NV, MAXT, MINB>;
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
    }
    kern<<<grid, 32 * warps, smem, st>>>(p);
    return cudaSuccess;
}

template <typename T, int MAXT, int MINB>
cudaError_t seq_launch_nv(int nv, const CplxParams &p, dim3 grid, int warps, size_t smem, cudaStream_t st)
{
    switch (nv) {
    case 1: return seq_launch_t<T, 1, MAXT, MINB>(p, grid, warps, smem, st);
    case 2: return seq_launch_t<T, 2, MAXT, MINB>(p, grid, warps, smem, st);
    default: return seq_launch_t<T, 4, MAXT, MINB>(p, grid, warps, smem, st);
    }
}


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
    const bool bf = a.dtype == SSD_DTYPE_BF16;
    const dim3 grid((unsigned)(a.batch * a.nheads));
    // steps per staged block: up to 64, within a third of the SM's shared memory for
    // CTAs of up to 8 warps (3 per SM) and about 200 KB otherwise (x and the step's
    // coefficients as fp32, B and C as stored)
    const bool small = warps <= kSmallWarps;
    const long long per_step = (long long)(p.Pp + 4) * (long long)sizeof(float) +
                               2LL * a.dstate * (long long)(bf ? sizeof(__nv_bfloat16) : sizeof(float));
    const long long budget = small ? (72LL << 10) : (200LL << 10);
    p.tblk = (int)std::max<long long>(1, std::min<long long>({64LL, a.seqlen, (budget - 16) / per_step}));
    const size_t smem = (size_t)p.tblk * (size_t)per_step + 16;   // (+ the B_t area's alignment)
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
    // (3 CTAs per SM where one float4 of each state row per lane leaves the
    // registers for it; 2 for the wider states)
    const cudaError_t le =
        bf ? (small ? (nv == 1 ? seq_launch_t<__nv_bfloat16, 1, kSmallWarps * 32, 3>(p, grid, warps, smem, st)
                               : seq_launch_nv<__nv_bfloat16, kSmallWarps * 32, 2>(nv, p, grid, warps, smem, st))
                    : seq_launch_nv<__nv_bfloat16, kMaxWarps * 32, 1>(nv, p, grid, warps, smem, st))
           : (small ? (nv == 1 ? seq_launch_t<float, 1, kSmallWarps * 32, 3>(p, grid, warps, smem, st)
                               : seq_launch_nv<float, kSmallWarps * 32, 2>(nv, p, grid, warps, smem, st))
                    : seq_launch_nv<float, kMaxWarps * 32, 1>(nv, p, grid, warps, smem, st));
    if (le != cudaSuccess)
        return le;
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess)
        note_launches(1);
    return e;
}

}  // namespace ssd
