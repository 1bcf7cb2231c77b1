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

#include "ssd_internal.h"

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
