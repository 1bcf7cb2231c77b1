// ssd_trap.cu -- the trapezoidal (Mamba-3 SISO) scan, sequential in time.
//
// Per batch row b and head h, with v = x, k = B, q = C of the head's group
// (the Mamba-3 SISO GPU forward page: its step F5b replaces the exponential
// update by a trapezoidal one with three coefficients, and the layer keeps
// the previous step's k and v as persistent state):
//   alpha_t = exp(a_t dt_t),  beta_t = alpha_t dt_t (1 - trap_t),  gamma_t = trap_t dt_t
//   h_t = alpha_t h_{t-1} + beta_t k_{t-1} v_{t-1}^T + gamma_t k_t v_t^T
//   y_t = q_t^T h_t + D v_t
// k_{-1}, v_{-1} are the carried k/v states; the state is stored [P, N].
//
// One CTA per (b, h), one warp per block of state rows p: lane l holds
// n = 4l .. 4l+3 (+128 per further float4) of each of the warp's rows, so the
// state in and out are coalesced 512-byte rows (at seqlen 1 the kernel is a
// stream of the state, like the decode step), and the state stays in
// registers for the whole sequence.  Time is walked in blocks whose k, q, v and
// coefficients are staged in shared memory by the whole CTA; the readout
// y_t[p] is a warp shuffle reduction.  The coefficient step (F5b) is fused:
// alpha, beta, gamma are computed from dt, a, trap as they are staged.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "ssd_internal.h"
#include "warp_rows.cuh"

namespace ssd {
namespace {

struct TrapParams {
    const void *v, *k, *q;
    const float *dt, *a, *trap, *D;
    const float *h0;
    const void *k0, *v0;
    void *y;
    float *h_final;
    void *k_final, *v_final;
    long long L;
    int H, P, N, G, tblk;
    int Pp;   // staged v row stride: the CTA's rows (warps x rows per warp)
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

// rows of one warp: RPW * NV = 8 float4 of state per lane stay in registers,
// and a CTA has at most 16 warps (so at most 128 registers per thread)
constexpr int kStateFloat4PerLane = 8;
constexpr int kMaxWarps = 16;

// NV: float4 chunks of a state row per lane (N <= 128 NV); RPW: rows per warp
template <typename T, int NV>
__global__ void __launch_bounds__(kMaxWarps * 32) ssd_trap_seq_kernel(TrapParams p)
{
    constexpr int RPW = kStateFloat4PerLane / NV;
    extern __shared__ float sm[];
    const int P = p.P, N = p.N, H = p.H, TB = p.tblk;
    const long long L = p.L;
    float *ks = sm;                  // [TB][N]
    float *qs = ks + TB * N;         // [TB][N]
    float *vs = qs + TB * N;         // [TB][Pp], zero past P
    float *cf = vs + TB * p.Pp;      // [TB][3]: alpha, beta, gamma
    const int Pp = p.Pp;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nthr = blockDim.x;
    const long long bh = blockIdx.x;
    const long long b = bh / H;
    const int h = (int)(bh - b * H);
    const int g = h / (H / p.G);
    const int p0 = warp * RPW;

    const T *vg = static_cast<const T *>(p.v);
    const T *kg = static_cast<const T *>(p.k);
    const T *qg = static_cast<const T *>(p.q);
    T *yg = static_cast<T *>(p.y);
    const size_t sbase = (size_t)bh * P * N;

    // state rows of this warp, and the previous step's k (lane's n) and v (rows)
    float4 hs[RPW][NV];
    float kp[NV][4], vp[RPW];
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        const int pr = p0 + r;
#pragma unroll
        for (int c = 0; c < NV; ++c) {
            const int n = 4 * lane + 128 * c;
            hs[r][c] = (p.h0 && pr < P && n < N)
                           ? __ldcs(reinterpret_cast<const float4 *>(p.h0 + sbase + (size_t)pr * N + n))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        vp[r] = (p.v0 && pr < P) ? to_f32<T>(static_cast<const T *>(p.v0)[bh * P + pr]) : 0.f;
    }
#pragma unroll
    for (int c = 0; c < NV; ++c)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int n = 4 * lane + 128 * c + e;
            kp[c][e] = (p.k0 && n < N) ? to_f32<T>(static_cast<const T *>(p.k0)[bh * N + n]) : 0.f;
        }

    for (long long t0 = 0; t0 < L; t0 += TB) {
        const int nt = (int)min((long long)TB, L - t0);
        __syncthreads();   // the previous block is consumed
        for (int i = threadIdx.x; i < nt * N; i += nthr) {
            const int tt = i / N, n = i - tt * N;
            const size_t gi = ((size_t)(b * L + t0 + tt) * p.G + g) * N + n;
            ks[i] = to_f32<T>(kg[gi]);
            qs[i] = to_f32<T>(qg[gi]);
        }
        for (int i = threadIdx.x; i < nt * Pp; i += nthr) {
            const int tt = i / Pp, pp = i - tt * Pp;
            vs[i] = pp < P ? to_f32<T>(vg[((size_t)(b * L + t0 + tt) * H + h) * P + pp]) : 0.f;
        }
        for (int i = threadIdx.x; i < nt; i += nthr) {
            const size_t ci = (size_t)(b * L + t0 + i) * H + h;
            const float dt = p.dt[ci];
            const float alpha = expf(p.a[ci] * dt);
            cf[3 * i + 0] = alpha;
            cf[3 * i + 1] = alpha * dt * (1.f - p.trap[ci]);
            cf[3 * i + 2] = p.trap[ci] * dt;
        }
        __syncthreads();
        for (int i = 0; i < nt; ++i) {
            const float alpha = cf[3 * i], beta = cf[3 * i + 1], gamma = cf[3 * i + 2];
            float kt[NV][4], qt[NV][4];
#pragma unroll
            for (int c = 0; c < NV; ++c) {
                const int n = 4 * lane + 128 * c;
                const bool in = n < N;   // N % 4 == 0: whole float4 chunks
                const float4 k4 = in ? *reinterpret_cast<const float4 *>(ks + i * N + n) : make_float4(0.f, 0.f, 0.f, 0.f);
                const float4 q4 = in ? *reinterpret_cast<const float4 *>(qs + i * N + n) : make_float4(0.f, 0.f, 0.f, 0.f);
                kt[c][0] = k4.x; kt[c][1] = k4.y; kt[c][2] = k4.z; kt[c][3] = k4.w;
                qt[c][0] = q4.x; qt[c][1] = q4.y; qt[c][2] = q4.z; qt[c][3] = q4.w;
            }
            float acc[RPW], vr[RPW];   // this warp's RPW rows of v_t: 16- or 8-byte loads
            if constexpr (RPW >= 4) {
#pragma unroll
                for (int u = 0; u < RPW / 4; ++u) {
                    const float4 v4 = *reinterpret_cast<const float4 *>(vs + i * Pp + p0 + 4 * u);
                    vr[4 * u] = v4.x;
                    vr[4 * u + 1] = v4.y;
                    vr[4 * u + 2] = v4.z;
                    vr[4 * u + 3] = v4.w;
                }
            } else {
                const float2 v2 = *reinterpret_cast<const float2 *>(vs + i * Pp + p0);
                vr[0] = v2.x;
                vr[1] = v2.y;
            }
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
                const float vt = vr[r];
                const float bv = beta * vp[r], gv = gamma * vt;
                float s = 0.f;
#pragma unroll
                for (int c = 0; c < NV; ++c) {
                    float4 &x = hs[r][c];
                    x.x = fmaf(alpha, x.x, fmaf(bv, kp[c][0], gv * kt[c][0]));
                    x.y = fmaf(alpha, x.y, fmaf(bv, kp[c][1], gv * kt[c][1]));
                    x.z = fmaf(alpha, x.z, fmaf(bv, kp[c][2], gv * kt[c][2]));
                    x.w = fmaf(alpha, x.w, fmaf(bv, kp[c][3], gv * kt[c][3]));
                    s = fmaf(qt[c][0], x.x, s);
                    s = fmaf(qt[c][1], x.y, s);
                    s = fmaf(qt[c][2], x.z, s);
                    s = fmaf(qt[c][3], x.w, s);
                }
                acc[r] = s;
                vp[r] = vt;
            }
#pragma unroll
            for (int c = 0; c < NV; ++c)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    kp[c][e] = kt[c][e];
            warp_sum_rows_all<RPW>(acc, lane);
            const int pr = p0 + summed_row<RPW>(lane);
            if ((lane & (32 / RPW - 1)) == 0 && pr < P)
                yg[((size_t)(b * L + t0 + i) * H + h) * P + pr] =
                    from_f32<T>(fmaf(p.D[h], vs[i * Pp + pr], acc[0]));
        }
    }

    // updated state, and the last step's k and v for the next call
    if (p.h_final) {
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            const int pr = p0 + r;
#pragma unroll
            for (int c = 0; c < NV; ++c) {
                const int n = 4 * lane + 128 * c;
                if (pr < P && n < N)
                    __stcs(reinterpret_cast<float4 *>(p.h_final + sbase + (size_t)pr * N + n), hs[r][c]);
            }
        }
    }
    if (p.v_final && lane == 0) {
#pragma unroll
        for (int r = 0; r < RPW; ++r)
            if (p0 + r < P)
                static_cast<T *>(p.v_final)[bh * P + p0 + r] = from_f32<T>(vp[r]);
    }
    if (p.k_final && warp == 0) {
        __syncwarp();
#pragma unroll
        for (int c = 0; c < NV; ++c)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int n = 4 * lane + 128 * c + e;
                if (n < N)
                    static_cast<T *>(p.k_final)[bh * N + n] = from_f32<T>(kp[c][e]);
            }
    }
}

// The carried k and v states after a scan run by the chunked kernel: the last
// step's k of the head's group and v of the head.  One CTA per (b, h).
template <typename T>
__global__ void __launch_bounds__(128) ssd_trap_carry_kernel(const T *v, const T *k, T *k_final, T *v_final,
                                                             long long L, int H, int P, int N, int G)
{
    const long long bh = blockIdx.x;
    const long long b = bh / H;
    const int h = (int)(bh - b * H), g = h / (H / G);
    for (int i = threadIdx.x; i < N && k_final; i += blockDim.x)
        k_final[bh * N + i] = k[((b * L + L - 1) * G + g) * N + i];
    for (int i = threadIdx.x; i < P && v_final; i += blockDim.x)
        v_final[bh * P + i] = v[((b * L + L - 1) * H + h) * P + i];
}

// One step (seqlen 1): the state is only streamed in and out, so the layout of
// the SSD decode step is used: one CTA of 4 warps per (b, h), 8 rows of a warp
// in flight, each state row one coalesced 512-byte load and store, no staging.
constexpr int kDecWarps = 4, kDecRows = 8;

template <typename T, int NV>
__global__ void __launch_bounds__(kDecWarps * 32, NV == 1 ? 5 : 1) ssd_trap_decode_kernel(TrapParams p)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = p.H, P = p.P, N = p.N;
    const long long bh = blockIdx.x;   // b * H + h (seqlen 1: also the token index)
    const long long b = bh / H;
    const int h = (int)(bh - b * H), g = h / (H / p.G);
    const float dt = p.dt[bh], trap = p.trap[bh];
    const float alpha = expf(p.a[bh] * dt), beta = alpha * dt * (1.f - trap), gamma = trap * dt;
    const float Dh = p.D[h];
    const T *kg = static_cast<const T *>(p.k) + (b * p.G + g) * (long long)N;
    const T *qg = static_cast<const T *>(p.q) + (b * p.G + g) * (long long)N;
    const T *k0 = p.k0 ? static_cast<const T *>(p.k0) + bh * N : nullptr;
    float kv[NV][4], qv[NV][4], kp[NV][4];
#pragma unroll
    for (int c = 0; c < NV; ++c)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int n = 4 * lane + 128 * c + e;
            kv[c][e] = n < N ? to_f32<T>(kg[n]) : 0.f;
            qv[c][e] = n < N ? to_f32<T>(qg[n]) : 0.f;
            kp[c][e] = (k0 && n < N) ? to_f32<T>(k0[n]) : 0.f;
        }
    const T *vg = static_cast<const T *>(p.v) + bh * P;
    const T *v0 = p.v0 ? static_cast<const T *>(p.v0) + bh * P : nullptr;
    T *yg = static_cast<T *>(p.y) + bh * P;
    const size_t sbase = (size_t)bh * P * N;
    for (int p0 = warp * kDecRows; p0 < P; p0 += kDecWarps * kDecRows) {
        float4 hv[kDecRows][NV];
        float vt[kDecRows], vp[kDecRows];
#pragma unroll
        for (int i = 0; i < kDecRows; ++i) {
            const int pr = p0 + i;
            vt[i] = pr < P ? to_f32<T>(vg[pr]) : 0.f;
            vp[i] = (v0 && pr < P) ? to_f32<T>(v0[pr]) : 0.f;
#pragma unroll
            for (int c = 0; c < NV; ++c) {
                const int n = 4 * lane + 128 * c;
                hv[i][c] = (p.h0 && pr < P && n < N)
                               ? __ldcs(reinterpret_cast<const float4 *>(p.h0 + sbase + (size_t)pr * N + n))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int i = 0; i < kDecRows; ++i) {
            const int pr = p0 + i;
            const float bv = beta * vp[i], gv = gamma * vt[i];
            float acc = 0.f;
#pragma unroll
            for (int c = 0; c < NV; ++c) {
                float4 &x = hv[i][c];
                x.x = fmaf(alpha, x.x, fmaf(bv, kp[c][0], gv * kv[c][0]));
                x.y = fmaf(alpha, x.y, fmaf(bv, kp[c][1], gv * kv[c][1]));
                x.z = fmaf(alpha, x.z, fmaf(bv, kp[c][2], gv * kv[c][2]));
                x.w = fmaf(alpha, x.w, fmaf(bv, kp[c][3], gv * kv[c][3]));
                acc = fmaf(qv[c][0], x.x, acc);
                acc = fmaf(qv[c][1], x.y, acc);
                acc = fmaf(qv[c][2], x.z, acc);
                acc = fmaf(qv[c][3], x.w, acc);
                const int n = 4 * lane + 128 * c;
                if (p.h_final && pr < P && n < N)
                    __stcs(reinterpret_cast<float4 *>(p.h_final + sbase + (size_t)pr * N + n), x);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0 && pr < P) {
                yg[pr] = from_f32<T>(fmaf(Dh, vt[i], acc));
                if (p.v_final)   // v_t from the register (exact: it was read as T)
                    static_cast<T *>(p.v_final)[bh * P + pr] = from_f32<T>(vt[i]);
            }
        }
    }
    if (p.k_final) {   // uniform over the CTA
        __syncthreads();   // every warp has read k0, which k_final may be
        if (warp == 0) {
#pragma unroll
            for (int c = 0; c < NV; ++c)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int n = 4 * lane + 128 * c + e;
                    if (n < N)
                        static_cast<T *>(p.k_final)[bh * N + n] = from_f32<T>(kv[c][e]);
                }
        }
    }
}

int trap_nv(int N) { return N <= 128 ? 1 : (N <= 256 ? 2 : 4); }

// warps per CTA: each holds kStateFloat4PerLane / NV rows
int trap_warps(int P, int N)
{
    const int rpw = kStateFloat4PerLane / trap_nv(N);
    return (P + rpw - 1) / rpw;
}

// the staged v row stride: the rows of all of the CTA's warps
int trap_pp(int P, int N) { return trap_warps(P, N) * (kStateFloat4PerLane / trap_nv(N)); }

// time steps per staged block: k, q (2N), v (Pp) and three coefficients per step
int trap_tblk(int P, int N)
{
    const size_t per_step = (size_t)(2 * N + trap_pp(P, N) + 3) * sizeof(float);
    return (int)std::max<size_t>(1, std::min<size_t>(64, (48u * 1024u) / per_step));
}

size_t trap_smem(int P, int N, int tb) { return (size_t)tb * (2 * N + trap_pp(P, N) + 3) * sizeof(float); }

template <typename T, int NV>
cudaError_t trap_launch_nv(const TrapParams &tp, long long grid, int threads, size_t smem, cudaStream_t st)
{
    if (tp.L == 1)
        ssd_trap_decode_kernel<T, NV><<<(unsigned)grid, kDecWarps * 32, 0, st>>>(tp);
    else
        ssd_trap_seq_kernel<T, NV><<<(unsigned)grid, threads, smem, st>>>(tp);
    return cudaGetLastError();
}

template <typename T>
cudaError_t trap_launch_t(int nv, const TrapParams &tp, long long grid, int threads, size_t smem, cudaStream_t st)
{
    switch (nv) {
    case 1: return trap_launch_nv<T, 1>(tp, grid, threads, smem, st);
    case 2: return trap_launch_nv<T, 2>(tp, grid, threads, smem, st);
    case 4: return trap_launch_nv<T, 4>(tp, grid, threads, smem, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool trap_supported(const TrapArgs &a)
{
    // whole float4 chunks of a state row, at most 512 states, at most kMaxWarps warps
    // (P <= 128 for N <= 128, P <= 64 for N <= 256, P <= 32 for N <= 512)
    return a.dstate % 4 == 0 && a.dstate <= 512 && a.headdim >= 1 && trap_warps(a.headdim, a.dstate) <= kMaxWarps &&
           a.batch * (long long)a.nheads <= 0x7FFFFFFFLL;
}

cudaError_t trap_carry_launch(const TrapArgs &a, cudaStream_t stream)
{
    SSD_NVTX_RANGE("trap_carry_launch");
    if (!a.k_final && !a.v_final)
        return cudaSuccess;
    const long long grid = a.batch * (long long)a.nheads;
    if (a.dtype == SSD_DTYPE_BF16)
        ssd_trap_carry_kernel<__nv_bfloat16><<<(unsigned)grid, 128, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(a.v), static_cast<const __nv_bfloat16 *>(a.k),
            static_cast<__nv_bfloat16 *>(a.k_final), static_cast<__nv_bfloat16 *>(a.v_final), a.seqlen, a.nheads,
            a.headdim, a.dstate, a.ngroups);
    else
        ssd_trap_carry_kernel<float><<<(unsigned)grid, 128, 0, stream>>>(
            static_cast<const float *>(a.v), static_cast<const float *>(a.k), static_cast<float *>(a.k_final),
            static_cast<float *>(a.v_final), a.seqlen, a.nheads, a.headdim, a.dstate, a.ngroups);
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess)
        note_launches(1);
    return e;
}

cudaError_t trap_launch(const TrapArgs &a, cudaStream_t stream)
{
    SSD_NVTX_RANGE("trap_launch");
    if (!trap_supported(a))
        return cudaErrorInvalidValue;
    TrapParams tp;
    tp.v = a.v;
    tp.k = a.k;
    tp.q = a.q;
    tp.dt = a.dt;
    tp.a = a.a;
    tp.trap = a.trap;
    tp.D = a.D;
    tp.h0 = a.h0;
    tp.k0 = a.k0;
    tp.v0 = a.v0;
    tp.y = a.y;
    tp.h_final = a.h_final;
    tp.k_final = a.k_final;
    tp.v_final = a.v_final;
    tp.L = a.seqlen;
    tp.H = a.nheads;
    tp.P = a.headdim;
    tp.N = a.dstate;
    tp.G = a.ngroups;
    tp.tblk = trap_tblk(a.headdim, a.dstate);
    tp.Pp = trap_pp(a.headdim, a.dstate);
    const size_t smem = trap_smem(a.headdim, a.dstate, tp.tblk);
    const int threads = 32 * trap_warps(a.headdim, a.dstate);
    const long long grid = a.batch * (long long)a.nheads;
    const int nv = trap_nv(a.dstate);
    cudaError_t e = a.dtype == SSD_DTYPE_BF16 ? trap_launch_t<__nv_bfloat16>(nv, tp, grid, threads, smem, stream)
                                              : trap_launch_t<float>(nv, tp, grid, threads, smem, stream);
    if (e == cudaSuccess)
        note_launches(1);
    return e;
}

}  // namespace ssd
