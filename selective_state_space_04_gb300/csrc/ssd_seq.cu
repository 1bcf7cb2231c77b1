// ssd_seq.cu -- sequential SSD scan (direct recurrence), fp32 FFMA.
//
// One CTA per (batch row b, head h).  The N x P state of that head lives in
// registers: thread (slice, p) owns the NPT state entries
// n = slice*NPT .. slice*NPT+NPT-1 of channel p, so no thread holds more than
// NPT (<= 64) floats -- the register limit that a one-thread-per-channel scan
// runs into for large N is avoided by splitting N over `slices` threads.
// Time is processed in blocks of `tblk` steps: B_t, C_t, x_t, dt_t and dA_t
// of the block are staged in shared memory (B and C are read once per CTA
// and broadcast to every thread of a warp, since a warp holds one slice),
// the per-slice partial readouts are collected in shared memory and summed
// once per block, and y is written with coalesced row stores.
//
// Recurrence (per step, the order of the SSD module's WGSL ssd_chunk_forward
// on the @seanhogg/builderforce-memory-engine 2026.6.18 page: decay the
// state, add the input term, read out from the updated state, add the skip):
//   h[n,p] = dA_t * h[n,p] + dt_t * B_t[n] * x_t[p]
//   y_t[p] = sum_n C_t[n] * h[n,p] + D * x_t[p]
// with dt_t = softplus(dt_raw + dt_bias), dA_t = exp(dt_t * A), A = -exp(A_log).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "f32x2.cuh"
#include "ssd_internal.h"
#include "warp_rows.cuh"

namespace ssd {
namespace {

struct SeqParams {
    const void *x;
    const float *dt_raw, *dt_bias, *A_log, *D;
    const void *B, *C;
    const float *init_state;
    void *y;
    float *final_state;
    long long L;
    int H, P, N, G, slices, tblk;
};

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v)
{
    return __bfloat162float(v);
}
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

template <int NPT, typename T>
__global__ void __launch_bounds__(512) ssd_seq_kernel(SeqParams p)
{
    extern __shared__ float sm[];
    const int P = p.P, N = p.N, S = p.slices, TB = p.tblk, H = p.H, G = p.G;
    const long long L = p.L;
    float *Bs = sm;                  // [TB][N]
    float *Cs = Bs + TB * N;         // [TB][N]
    float *xs = Cs + TB * N;         // [TB][P]
    float *dts = xs + TB * P;        // [TB]
    float *dAs = dts + TB;           // [TB]
    float *yp = dAs + TB;            // [S][TB][P]

    const int tid = threadIdx.x;
    const int nthr = S * P;
    const int slice = tid / P, pc = tid - slice * P;
    const long long b = blockIdx.x / H;
    const int h = blockIdx.x % H;
    const int g = h / (H / G);
    const int n0 = slice * NPT;
    const int nvalid = min(NPT, N - n0);  // may be <= 0 for padding slices

    const T *xg = static_cast<const T *>(p.x);
    const T *Bg = static_cast<const T *>(p.B);
    const T *Cg = static_cast<const T *>(p.C);
    T *yg = static_cast<T *>(p.y);

    float hs[NPT];
    const size_t sbase = ((size_t)(b * H + h) * P + pc) * N + n0;
#pragma unroll
    for (int j = 0; j < NPT; ++j)
        hs[j] = (p.init_state && j < nvalid) ? p.init_state[sbase + j] : 0.f;

    const float A = -expf(p.A_log[h]);
    const float bias = p.dt_bias[h];
    const float Dh = p.D[h];

    for (long long t0 = 0; t0 < L; t0 += TB) {
        const int nt = (int)min((long long)TB, L - t0);
        __syncthreads();  // previous block fully consumed
        for (int i = tid; i < nt * N; i += nthr) {
            const int tt = i / N, n = i - tt * N;
            const size_t gi = ((size_t)(b * L + t0 + tt) * G + g) * N + n;
            Bs[i] = to_f32<T>(Bg[gi]);
            Cs[i] = to_f32<T>(Cg[gi]);
        }
        for (int i = tid; i < nt * P; i += nthr) {
            const int tt = i / P, pp = i - tt * P;
            xs[i] = to_f32<T>(xg[((size_t)(b * L + t0 + tt) * H + h) * P + pp]);
        }
        for (int i = tid; i < nt; i += nthr) {
            const float dt = softplus_f32(p.dt_raw[(size_t)(b * L + t0 + i) * H + h] + bias);
            dts[i] = dt;
            dAs[i] = expf(dt * A);
        }
        __syncthreads();
        for (int i = 0; i < nt; ++i) {
            const float dA = dAs[i];
            const float dtx = dts[i] * xs[i * P + pc];
            const float *Bt = Bs + i * N + n0;
            const float *Ct = Cs + i * N + n0;
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < NPT; ++j) {
                if (j < nvalid) {
                    hs[j] = fmaf(dA, hs[j], dtx * Bt[j]);
                    acc = fmaf(Ct[j], hs[j], acc);
                }
            }
            yp[(slice * TB + i) * P + pc] = acc;
        }
        __syncthreads();
        for (int i = tid; i < nt * P; i += nthr) {
            const int tt = i / P, pp = i - tt * P;
            float acc = 0.f;
            for (int s = 0; s < S; ++s)
                acc += yp[(s * TB + tt) * P + pp];
            acc = fmaf(Dh, xs[i], acc);
            yg[((size_t)(b * L + t0 + tt) * H + h) * P + pp] = from_f32<T>(acc);
        }
    }
    if (p.final_state) {
#pragma unroll
        for (int j = 0; j < NPT; ++j)
            if (j < nvalid)
                p.final_state[sbase + j] = hs[j];
    }
}


// ---- the row layout (N % 4 == 0, N <= 512): one CTA per (b, h), one warp per
// block of RPW = 8 / NV state rows p, lane l holding n = 4l .. 4l+3 (+128 per
// further float4) of each row, so the state is read and written as coalesced
// 512-byte rows and stays in registers.  Per time block (up to 64 steps) the
// CTA stages B_t and C_t as stored (bf16 stays bf16: half the shared memory, so
// more CTAs overlap their loads with the others' steps), x_t as fp32 and dt_t,
// dA_t, with vector copies and no index division.  Each element takes
// dA h + (dt x) B, the decode step's operations in its order (one decode step
// equals one step of this scan bit for bit), two elements per instruction with
// the packed fp32 multiply and FMA; y_t[p] is a warp butterfly over the
// per-lane readouts (each an fp32 pair, summed at the end).  The step loop is
// unrolled so that a step's readout reduction overlaps the next steps'
// updates, and each warp reads its rows of x_t as 16-byte (8-byte) words from a
// stride padded to the CTA's rows.
constexpr int kRowF4PerLane = 8;   // RPW * NV float4 of state per lane
constexpr int kRowMaxWarps = 16;
constexpr int kRowSmallWarps = 8;  // CTAs of up to 8 warps: 2 or 3 per SM
// x elements a thread stages per block: steps x rows / threads <= 64 * (8 warps' RPW rows) / 32
constexpr int kXPerThread = 64 * kRowF4PerLane / 32;

struct RowParams {
    SeqParams s;
    int Pp;                         // staged x row stride (the CTA's rows)
};

// 4 staged values of B or C as two fp32 pairs
__device__ __forceinline__ void load4(const float *src, f32x2 (&o)[2])
{
    const float4 v = *reinterpret_cast<const float4 *>(src);
    o[0] = pk2(v.x, v.y);
    o[1] = pk2(v.z, v.w);
}
__device__ __forceinline__ void load4(const __nv_bfloat16 *src, f32x2 (&o)[2])
{
    const uint2 v = *reinterpret_cast<const uint2 *>(src);
    o[0] = pk2(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u));
    o[1] = pk2(__uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
}
// asynchronous 16- and 8-byte copies of B or C into the staging area (the
// 16-byte ones bypass L1); completed by cp.async.wait_all
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

template <typename T, int NV, int MAXT, int MINB>
__global__ void __launch_bounds__(MAXT, MINB) ssd_seq_rows_kernel(RowParams rp)
{
    constexpr int RPW = kRowF4PerLane / NV;
    const SeqParams &p = rp.s;
    extern __shared__ float sm[];
    const int P = p.P, N = p.N, H = p.H, TB = p.tblk, Pp = rp.Pp;
    const long long L = p.L;
    float *xs = sm;                  // [TB][Pp], zero past P
    float *da = xs + TB * Pp;        // [TB]: dA_t
    float *ds = da + TB;             // [TB]: dt_t
    T *bs = reinterpret_cast<T *>(sm + ((TB * (Pp + 2) + 3) & ~3));   // [TB][N]: B_t as stored (16-byte aligned)
    T *cs = bs + (size_t)TB * N;     // [TB][N]: C_t
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nthr = blockDim.x, nwarps = nthr >> 5;
    const long long bh = blockIdx.x;
    const long long b = bh / H;
    const int h = (int)(bh - b * H);
    const int g = h / (H / p.G);
    const int p0 = warp * RPW;
    const T *xg = static_cast<const T *>(p.x), *Bg = static_cast<const T *>(p.B), *Cg = static_cast<const T *>(p.C);
    T *yg = static_cast<T *>(p.y);
    const size_t sbase = (size_t)bh * P * N;
    const float A = -expf(p.A_log[h]), bias = p.dt_bias[h], Dh = p.D[h];
    const bool wide16 = (N * (int)sizeof(T)) % 16 == 0;   // staged rows in 16-byte copies

    f32x2 hs[RPW][NV][2];
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        const int pr = p0 + r;
#pragma unroll
        for (int c = 0; c < NV; ++c) {
            const int n = 4 * lane + 128 * c;
            const float4 v = (p.init_state && pr < P && n < N)
                                 ? __ldcs(reinterpret_cast<const float4 *>(p.init_state + sbase + (size_t)pr * N + n))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
            hs[r][c][0] = pk2(v.x, v.y);
            hs[r][c][1] = pk2(v.z, v.w);
        }
    }

    for (long long t0 = 0; t0 < L; t0 += TB) {
        const int nt = (int)min((long long)TB, L - t0);
        __syncthreads();   // the previous block is consumed
        for (int i = threadIdx.x; i < nt; i += nthr) {
            const float dt = softplus_f32(p.dt_raw[(size_t)(b * L + t0 + i) * H + h] + bias);
            da[i] = expf(dt * A);
            ds[i] = dt;
        }
        // B_t and C_t by asynchronous copies (all in flight at once), x_t converted to
        // fp32 on the way, so that a block costs few memory round trips
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
            // a warp per step row (measured faster than the batch above with 8 warps)
            for (int tt = warp; tt < nt; tt += nwarps) {
                const size_t row = (size_t)(b * L + t0 + tt);
                for (int pp = lane; pp < Pp; pp += 32)
                    xs[tt * Pp + pp] = pp < P ? to_f32<T>(xg[(row * H + h) * P + pp]) : 0.f;
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        __syncthreads();
#pragma unroll 4
        for (int i = 0; i < nt; ++i) {
            const float dt = ds[i];
            const f32x2 dA2 = pk2(da[i], da[i]);
            f32x2 bt[NV][2], ct[NV][2];
#pragma unroll
            for (int c = 0; c < NV; ++c) {
                const int n = 4 * lane + 128 * c;
                if (n < N) {   // N % 4 == 0: whole 4-element chunks
                    load4(bs + (size_t)i * N + n, bt[c]);
                    load4(cs + (size_t)i * N + n, ct[c]);
                } else {
                    bt[c][0] = bt[c][1] = ct[c][0] = ct[c][1] = 0ull;
                }
            }
            float acc[RPW], xr[RPW];
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
                const float dtx = dt * xr[r];
                const f32x2 dtx2 = pk2(dtx, dtx);
                f32x2 s = 0ull;
#pragma unroll
                for (int c = 0; c < NV; ++c) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        f32x2 &z = hs[r][c][e];
                        z = fma2(dA2, z, mul2(dtx2, bt[c][e]));
                        s = fma2(ct[c][e], z, s);
                    }
                }
                acc[r] = lo2(s) + hi2(s);
            }
            warp_sum_rows_all<RPW>(acc, lane);
            const int pr = p0 + summed_row<RPW>(lane);
            if ((lane & (32 / RPW - 1)) == 0 && pr < P)
                yg[((size_t)(b * L + t0 + i) * H + h) * P + pr] = from_f32<T>(fmaf(Dh, xs[i * Pp + pr], acc[0]));
        }
    }

    if (p.final_state) {
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            const int pr = p0 + r;
#pragma unroll
            for (int c = 0; c < NV; ++c) {
                const int n = 4 * lane + 128 * c;
                if (pr < P && n < N)
                    __stcs(reinterpret_cast<float4 *>(p.final_state + sbase + (size_t)pr * N + n),
                           make_float4(lo2(hs[r][c][0]), hi2(hs[r][c][0]), lo2(hs[r][c][1]), hi2(hs[r][c][1])));
            }
        }
    }
}

int rows_nv(int N) { return N <= 128 ? 1 : N <= 256 ? 2 : 4; }

bool rows_supported(int P, int N)
{
    if (N % 4 != 0 || N < 4 || N > 512 || P < 1)
        return false;
    return P <= kRowMaxWarps * (kRowF4PerLane / rows_nv(N));
}

template <typename T, int NV, int MAXT, int MINB>
cudaError_t rows_launch_t(const RowParams &rp, int grid, int threads, size_t smem, cudaStream_t st)
{
    auto kern = ssd_seq_rows_kernel<T, NV, MAXT, MINB>;
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
    }
    kern<<<grid, threads, smem, st>>>(rp);
    return cudaGetLastError();
}

template <typename T, int MAXT, int MINB>
cudaError_t rows_launch_nv(int nv, const RowParams &rp, int grid, int threads, size_t smem, cudaStream_t st)
{
    switch (nv) {
    case 1: return rows_launch_t<T, 1, MAXT, MINB>(rp, grid, threads, smem, st);
    case 2: return rows_launch_t<T, 2, MAXT, MINB>(rp, grid, threads, smem, st);
    default: return rows_launch_t<T, 4, MAXT, MINB>(rp, grid, threads, smem, st);
    }
}

template <typename T>
cudaError_t rows_launch(const SeqParams &sp, int grid, cudaStream_t st)
{
    const int nv = rows_nv(sp.N), rpw = kRowF4PerLane / nv;
    const int warps = (sp.P + rpw - 1) / rpw;
    const bool small = warps <= kRowSmallWarps;   // 3 CTAs per SM
    RowParams rp;
    rp.s = sp;
    rp.Pp = warps * rpw;
    // steps per staged block: up to 64, within a third of the SM's shared memory for
    // the small CTAs (3 per SM) and about 200 KB otherwise (x as fp32, B and C as
    // stored, dA and dt per step)
    const long long per_step =
        (long long)(rp.Pp + 2) * (long long)sizeof(float) + 2LL * sp.N * (long long)sizeof(T);
    const long long budget = small ? (72LL << 10) : (200LL << 10);
    rp.s.tblk = (int)std::max<long long>(1, std::min<long long>({64LL, sp.L, (budget - 16) / per_step}));
    const size_t smem = (size_t)rp.s.tblk * (size_t)per_step + 16;   // (+ the B_t area's alignment)
    // (3 CTAs per SM where one float4 of each state row per lane leaves the registers
    // for it; 2 for the wider states, which would spill at 3)
    if (small && nv == 1)
        return rows_launch_t<T, 1, kRowSmallWarps * 32, 3>(rp, grid, 32 * warps, smem, st);
    return small ? rows_launch_nv<T, kRowSmallWarps * 32, 2>(nv, rp, grid, 32 * warps, smem, st)
                 : rows_launch_nv<T, kRowMaxWarps * 32, 1>(nv, rp, grid, 32 * warps, smem, st);
}

struct SeqShape {
    int slices, npt, tblk;
    size_t smem;
};

int pow2ceil(int v)
{
    int r = 1;
    while (r < v)
        r <<= 1;
    return r;
}

bool seq_shape(int P, int N, SeqShape *out)
{
    if (P < 1 || P > 512 || N < 1)
        return false;
    int S = std::min(32, pow2ceil((N + 31) / 32));
    while (S > 1 && S * P > 512)
        S >>= 1;
    if (S * P > 512)
        return false;
    const int npt = pow2ceil((N + S - 1) / S);
    if (npt > 64)
        return false;
    // per time step: B, C rows (2N), x row (P), dt and dA (2), partial readouts (S*P)
    const size_t per_step = (size_t)(2 * N + P + 2 + S * P) * sizeof(float);
    const size_t budget = 160 * 1024;
    int tb = (int)std::min<size_t>(64, budget / per_step);
    if (tb < 1)
        return false;
    out->slices = S;
    out->npt = npt;
    out->tblk = tb;
    out->smem = per_step * tb;
    return true;
}

template <int NPT, typename T>
cudaError_t launch_t(const SeqParams &sp, int grid, int threads, size_t smem, cudaStream_t st)
{
    auto kern = ssd_seq_kernel<NPT, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    kern<<<grid, threads, smem, st>>>(sp);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_npt(int npt, const SeqParams &sp, int grid, int threads, size_t smem,
                       cudaStream_t st)
{
    switch (npt) {
    case 1: return launch_t<1, T>(sp, grid, threads, smem, st);
    case 2: return launch_t<2, T>(sp, grid, threads, smem, st);
    case 4: return launch_t<4, T>(sp, grid, threads, smem, st);
    case 8: return launch_t<8, T>(sp, grid, threads, smem, st);
    case 16: return launch_t<16, T>(sp, grid, threads, smem, st);
    case 32: return launch_t<32, T>(sp, grid, threads, smem, st);
    case 64: return launch_t<64, T>(sp, grid, threads, smem, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool seq_supported(int headdim, int dstate)
{
    SeqShape s;
    return seq_shape(headdim, dstate, &s);
}

cudaError_t seq_launch(const ScanArgs &a, cudaStream_t stream)
{
    SSD_NVTX_RANGE("seq_launch");
    SeqShape s;
    if (!seq_shape(a.headdim, a.dstate, &s))
        return cudaErrorInvalidValue;
    SeqParams sp;
    sp.x = a.x;
    sp.dt_raw = a.dt_raw;
    sp.dt_bias = a.dt_bias;
    sp.A_log = a.A_log;
    sp.D = a.D;
    sp.B = a.B;
    sp.C = a.C;
    sp.init_state = a.init_state;
    sp.y = a.y;
    sp.final_state = a.final_state;
    sp.L = a.seqlen;
    sp.H = a.nheads;
    sp.P = a.headdim;
    sp.N = a.dstate;
    sp.G = a.ngroups;
    sp.slices = s.slices;
    sp.tblk = s.tblk;
    const long long grid = a.batch * (long long)a.nheads;
    if (grid > 0x7FFFFFFFLL)
        return cudaErrorInvalidValue;
    if (rows_supported(a.headdim, a.dstate)) {   // the row layout where it applies
        const cudaError_t e = a.dtype == SSD_DTYPE_BF16 ? rows_launch<__nv_bfloat16>(sp, (int)grid, stream)
                                                        : rows_launch<float>(sp, (int)grid, stream);
        if (e == cudaSuccess)
            note_launches(1);
        return e;
    }
    const int threads = s.slices * a.headdim;
    cudaError_t e;
    if (a.dtype == SSD_DTYPE_BF16)
        e = launch_npt<__nv_bfloat16>(s.npt, sp, (int)grid, threads, s.smem, stream);
    else
        e = launch_npt<float>(s.npt, sp, (int)grid, threads, s.smem, stream);
    if (e == cudaSuccess)
        note_launches(1);
    return e;
}

}  // namespace ssd
