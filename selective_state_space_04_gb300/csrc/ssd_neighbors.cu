// ssd_neighbors.cu -- the steps on either side of the scan in the Mamba blocks
// of the pages.
//
// * Causal depthwise conv1d + SiLU over the fused x | B | C channels (the
//   builderforce Mamba2Block convolves the fused x, B and C projection
//   channels; the conv1d kernel page: y[b,t,d] = sum_k weight[d,k] x[b,t-k,d]
//   + bias[d], zero before the sequence; the mamba-rs 0.4.0 S6 forward applies
//   SiLU in the conv's kernel and carries the conv state between calls),
//   written straight into the scan's x [B,L,H,P], B and C [B,L,G,N].
// * Gated RMSNorm of the scan's output (Mamba-3 forward, step F7:
//   RMSNorm(y) * weight * SiLU(z)) over the H*P channels of each token.
//
// Both are streams of HBM; the layouts follow from that (16-byte vectors along
// the channels, each input read once).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "ssd_internal.h"

namespace ssd {
namespace {

// 8 channels of one 16-byte (bf16) or two 16-byte (fp32) vectors
template <typename T> struct Vec8;
template <> struct Vec8<__nv_bfloat16> {
    uint4 u;
    __device__ __forceinline__ void load(const __nv_bfloat16 *p) { u = *reinterpret_cast<const uint4 *>(p); }
    __device__ __forceinline__ void store(__nv_bfloat16 *p) const { *reinterpret_cast<uint4 *>(p) = u; }
    __device__ __forceinline__ void load_cs(const __nv_bfloat16 *p) { u = __ldcs(reinterpret_cast<const uint4 *>(p)); }
    __device__ __forceinline__ void store_cs(__nv_bfloat16 *p) const { __stcs(reinterpret_cast<uint4 *>(p), u); }
    __device__ __forceinline__ void get(float (&f)[8]) const
    {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ __forceinline__ void set(const float (&f)[8])
    {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t *>(&h);
        }
        u = make_uint4(w[0], w[1], w[2], w[3]);
    }
};
template <> struct Vec8<float> {
    float4 a, b;
    __device__ __forceinline__ void load(const float *p)
    {
        a = reinterpret_cast<const float4 *>(p)[0];
        b = reinterpret_cast<const float4 *>(p)[1];
    }
    __device__ __forceinline__ void store(float *p) const
    {
        reinterpret_cast<float4 *>(p)[0] = a;
        reinterpret_cast<float4 *>(p)[1] = b;
    }
    __device__ __forceinline__ void load_cs(const float *p)
    {
        a = __ldcs(reinterpret_cast<const float4 *>(p));
        b = __ldcs(reinterpret_cast<const float4 *>(p) + 1);
    }
    __device__ __forceinline__ void store_cs(float *p) const
    {
        __stcs(reinterpret_cast<float4 *>(p), a);
        __stcs(reinterpret_cast<float4 *>(p) + 1, b);
    }
    __device__ __forceinline__ void get(float (&f)[8]) const
    {
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
        f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    }
    __device__ __forceinline__ void set(const float (&f)[8])
    {
        a = make_float4(f[0], f[1], f[2], f[3]);
        b = make_float4(f[4], f[5], f[6], f[7]);
    }
};

// 4 channels of one 8-byte (bf16) or 16-byte (fp32) vector
template <typename T> struct Vec4;
template <> struct Vec4<__nv_bfloat16> {
    uint2 u;
    __device__ __forceinline__ void load(const __nv_bfloat16 *p) { u = *reinterpret_cast<const uint2 *>(p); }
    __device__ __forceinline__ void load_cs(const __nv_bfloat16 *p) { u = __ldcs(reinterpret_cast<const uint2 *>(p)); }
    __device__ __forceinline__ void store(__nv_bfloat16 *p) const { *reinterpret_cast<uint2 *>(p) = u; }
    __device__ __forceinline__ void get(float (&f)[4]) const
    {
        f[0] = __uint_as_float(u.x << 16);
        f[1] = __uint_as_float(u.x & 0xffff0000u);
        f[2] = __uint_as_float(u.y << 16);
        f[3] = __uint_as_float(u.y & 0xffff0000u);
    }
    __device__ __forceinline__ void set(const float (&f)[4])
    {
        const __nv_bfloat162 a = __floats2bfloat162_rn(f[0], f[1]), b = __floats2bfloat162_rn(f[2], f[3]);
        u = make_uint2(*reinterpret_cast<const uint32_t *>(&a), *reinterpret_cast<const uint32_t *>(&b));
    }
};
template <> struct Vec4<float> {
    float4 a;
    __device__ __forceinline__ void load(const float *p) { a = *reinterpret_cast<const float4 *>(p); }
    __device__ __forceinline__ void load_cs(const float *p) { a = __ldcs(reinterpret_cast<const float4 *>(p)); }
    __device__ __forceinline__ void store(float *p) const { *reinterpret_cast<float4 *>(p) = a; }
    __device__ __forceinline__ void get(float (&f)[4]) const
    {
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    }
    __device__ __forceinline__ void set(const float (&f)[4]) { a = make_float4(f[0], f[1], f[2], f[3]); }
};

// SiLU with the fast exp and divide intrinsics (a few ulp; the IEEE forms cost
// about 40 instructions per element, which made the conv arithmetic-bound).
// For v below about -88 the divisor overflows and the result is 0, as SiLU's is.
__device__ __forceinline__ float silu_f32(float v) { return __fdividef(v, 1.f + __expf(-v)); }

__device__ __forceinline__ float tanh_approx(float x)
{
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// For outputs rounded to bf16 (8 significant bits): SiLU(v) = h + h tanh(h),
// h = v / 2, with the hardware tanh approximation (relative error about 2^-11):
// one special-function operation per element instead of two, which bounds the
// conv's throughput.  fp32 outputs keep silu_f32.
template <typename T> __device__ __forceinline__ float silu_out(float v);
template <> __device__ __forceinline__ float silu_out<float>(float v) { return silu_f32(v); }
template <> __device__ __forceinline__ float silu_out<__nv_bfloat16>(float v)
{
    const float h = 0.5f * v;
    return fmaf(h, tanh_approx(h), h);
}

constexpr int kConvTile = 64;     // time steps per thread
constexpr int kConvThreads = 128;

struct ConvParams {
    const void *xbc;            // [B,L,C]
    const float *w, *bias;      // [C,K], [C] or null
    const void *state_in;       // [B,K-1,C] or null
    void *x, *B, *C;            // [B,L,H*P], [B,L,G*N] x2
    void *state_out;            // [B,K-1,C] or null
    long long L;
    int Cc, HP, GN, nvec;       // nvec = C / channels per thread
    int vbase = 0;              // first vector handled (the launch covers vbase .. nvec-1)
};

// Asynchronous 16-byte copies from global into shared memory (cp.async, L1
// bypassed): the bytes in flight wait in shared memory, not in registers.
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem)
{
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

constexpr int kConvStages = 16;   // steps of each thread in flight (its own ring of 16-byte slots)
static_assert((kConvStages & (kConvStages - 1)) == 0, "a power of two (slot = step & (stages - 1))");

template <typename T, int V> struct VecSel;
template <typename T> struct VecSel<T, 4> { using type = Vec4<T>; };
template <typename T> struct VecSel<T, 8> { using type = Vec8<T>; };

// a 16-byte vector from its raw bits
__device__ __forceinline__ void from_raw(Vec8<__nv_bfloat16> &v, const uint4 &r) { v.u = r; }
__device__ __forceinline__ void from_raw(Vec4<float> &v, const uint4 &r)
{
    v.a = make_float4(__uint_as_float(r.x), __uint_as_float(r.y), __uint_as_float(r.z), __uint_as_float(r.w));
}

// thread: V consecutive channels (one 16-byte vector v) over kConvTile steps
// of one batch row; the K-1 inputs before the current step stay in registers.
// Each thread streams its inputs through its own ring of kConvStages 16-byte
// slots in shared memory (cp.async), so kConvStages steps are in flight per
// thread; no slot is shared, so no barrier is needed.
template <typename T, int K, int V>
__global__ void __launch_bounds__(kConvThreads, 4) ssd_conv1d_silu_kernel(ConvParams p)
{
    using Vec = typename VecSel<T, V>::type;
    static_assert(V * sizeof(T) == 16, "one 16-byte vector per step");
    __shared__ uint4 ring[kConvStages * kConvThreads];
    const int v = p.vbase + blockIdx.x * blockDim.x + threadIdx.x;
    if (v >= p.nvec)
        return;   // (no barrier in this kernel)
    const long long b = blockIdx.z, L = p.L;
    const long long t0 = (long long)blockIdx.y * kConvTile;
    const int c0 = V * v, Cc = p.Cc;
    const T *in = static_cast<const T *>(p.xbc) + (size_t)b * L * Cc + c0;
    float wv[K][V], bv[V];
#pragma unroll
    for (int e = 0; e < V; ++e) {
#pragma unroll
        for (int k = 0; k < K; ++k)
            wv[k][e] = p.w[(size_t)(c0 + e) * K + k];
        bv[e] = p.bias ? p.bias[c0 + e] : 0.f;
    }
    // win[j]: the input at step t - (K-1) + j, j < K-1
    float win[K - 1][V];
#pragma unroll
    for (int j = 0; j < K - 1; ++j) {
        const long long tt = t0 - (K - 1) + j;
        Vec u;
        if (tt >= 0) {
            u.load(in + (size_t)tt * Cc);
            u.get(win[j]);
        } else if (p.state_in) {
            u.load(static_cast<const T *>(p.state_in) + ((size_t)b * (K - 1) + (K - 1) + tt) * Cc + c0);
            u.get(win[j]);
        } else {
#pragma unroll
            for (int e = 0; e < V; ++e)
                win[j][e] = 0.f;
        }
    }
    // this vector's output tensor (the vector lies inside one of x, B, C)
    T *out;
    int stride, off;
    if (c0 < p.HP) {
        out = static_cast<T *>(p.x);
        stride = p.HP;
        off = c0;
    } else if (c0 < p.HP + p.GN) {
        out = static_cast<T *>(p.B);
        stride = p.GN;
        off = c0 - p.HP;
    } else {
        out = static_cast<T *>(p.C);
        stride = p.GN;
        off = c0 - p.HP - p.GN;
    }
    const int nt = (int)min((long long)kConvTile, L - t0);
    const T *src = in + (size_t)t0 * Cc;
    T *dst = out + ((size_t)b * L + t0) * stride + off;
    // one step: the output from the window and the current input, then the window moves on
    auto step = [&](const Vec &u, T *d) {
        float cur[V], acc[V];
        u.get(cur);
#pragma unroll
        for (int e = 0; e < V; ++e) {
            float s = fmaf(wv[0][e], cur[e], bv[e]);
#pragma unroll
            for (int k = 1; k < K; ++k)
                s = fmaf(wv[k][e], win[K - 1 - k][e], s);   // the input k steps back
            acc[e] = silu_out<T>(s);
        }
        Vec o;
        o.set(acc);
        o.store(d);
#pragma unroll
        for (int j = 0; j + 1 < K - 1; ++j)
#pragma unroll
            for (int e = 0; e < V; ++e)
                win[j][e] = win[j + 1][e];
#pragma unroll
        for (int e = 0; e < V; ++e)
            win[K - 2][e] = cur[e];
    };
    // the ring: slot s holds step i with i % kConvStages == s; one commit
    // group per step (empty past the tile's end), so after the wait below at
    // most kConvStages - 1 groups, the steps after i, are still in flight
    uint4 *mine = ring + threadIdx.x;
#pragma unroll
    for (int s = 0; s < kConvStages; ++s) {
        if (s < nt)
            cp_async16(mine + s * kConvThreads, src + (size_t)s * Cc);
        cp_async_commit();
    }
    const T *next = src + (size_t)kConvStages * Cc;   // the step kConvStages ahead
#pragma unroll 4
    for (int i = 0; i < nt; ++i) {
        cp_async_wait<kConvStages - 1>();
        uint4 *slot = mine + (i & (kConvStages - 1)) * kConvThreads;
        const uint4 raw = *slot;
        if (i + kConvStages < nt)
            cp_async16(slot, next);   // after the read of this slot, in program order
        cp_async_commit();
        next += Cc;
        Vec u;
        from_raw(u, raw);
        step(u, dst);
        dst += stride;
    }
    cp_async_wait<0>();
    if (p.state_out && t0 + nt == L) {   // the last tile: the last K-1 inputs
#pragma unroll
        for (int j = 0; j < K - 1; ++j) {
            Vec o;
            o.set(win[j]);
            o.store(static_cast<T *>(p.state_out) + ((size_t)b * (K - 1) + j) * Cc + c0);
        }
    }
}

// bf16: 8 channels (one 16-byte vector) per thread; fp32: 4 (one 16-byte vector)
template <typename T> constexpr int conv_vec() { return sizeof(T) == 2 ? 8 : 4; }

template <typename T>
cudaError_t conv_launch_t(int K, const ConvParams &cp, dim3 grid, cudaStream_t st)
{
    constexpr int V = conv_vec<T>();
    switch (K) {
    case 2: ssd_conv1d_silu_kernel<T, 2, V><<<grid, kConvThreads, 0, st>>>(cp); break;
    case 3: ssd_conv1d_silu_kernel<T, 3, V><<<grid, kConvThreads, 0, st>>>(cp); break;
    case 4: ssd_conv1d_silu_kernel<T, 4, V><<<grid, kConvThreads, 0, st>>>(cp); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

constexpr int kNormVPT = 4;   // 8-channel vectors of y and of z per thread, held in registers
constexpr int kNormMaxThreads = 512;

struct NormParams {
    const void *y, *z;
    const float *w;
    void *out;
    int D;          // channels per token (H*P), a multiple of 8, at most kNormMaxThreads * kNormVPT * 8
    float eps;
};

// One CTA per token; thread i holds vectors i, i + blockDim, ... (kNormVPT of
// them) of y and z, all loaded before the sum of squares is reduced, so a
// token's row is read once: out = y / sqrt(mean(y^2) + eps) * w * SiLU(z).
template <typename T>
__global__ void __launch_bounds__(kNormMaxThreads) ssd_gated_rmsnorm_kernel(NormParams p)
{
    __shared__ float part[kNormMaxThreads / 32];
    const size_t row = blockIdx.x;
    const int nv = p.D / 8;
    const T *y = static_cast<const T *>(p.y) + row * p.D;
    const T *z = static_cast<const T *>(p.z) + row * p.D;
    T *out = static_cast<T *>(p.out) + row * p.D;
    Vec8<T> uy[kNormVPT], uz[kNormVPT];
#pragma unroll
    for (int a = 0; a < kNormVPT; ++a) {
        const int v = threadIdx.x + a * blockDim.x;
        if (v < nv) {
            uy[a].load_cs(y + 8 * v);
            uz[a].load_cs(z + 8 * v);
        }
    }
    float ss = 0.f;
#pragma unroll
    for (int a = 0; a < kNormVPT; ++a) {
        if (threadIdx.x + a * blockDim.x < nv) {
            float f[8];
            uy[a].get(f);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                ss = fmaf(f[e], f[e], ss);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0)
        part[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i)
        tot += part[i];
    const float inv = rsqrtf(tot / (float)p.D + p.eps);
#pragma unroll
    for (int a = 0; a < kNormVPT; ++a) {
        const int v = threadIdx.x + a * blockDim.x;
        if (v >= nv)
            break;
        float fy[8], fz[8], o[8];
        uy[a].get(fy);
        uz[a].get(fz);
        const float4 w0 = reinterpret_cast<const float4 *>(p.w)[2 * v];
        const float4 w1 = reinterpret_cast<const float4 *>(p.w)[2 * v + 1];
        const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e)
            o[e] = fy[e] * inv * wv[e] * silu_out<T>(fz[e]);
        Vec8<T> uo;
        uo.set(o);
        uo.store(out + 8 * v);
    }
}

}  // namespace

bool conv_supported(const NeighborArgs &a)
{
    const long long HP = (long long)a.nheads * a.headdim, GN = (long long)a.ngroups * a.dstate;
    return HP % 8 == 0 && GN % 8 == 0 && a.kernel_size >= 2 && a.kernel_size <= 4 && a.seqlen < (1LL << 31) &&
           a.batch <= 65535;
}

cudaError_t conv_launch(const NeighborArgs &a, cudaStream_t st)
{
    SSD_NVTX_RANGE("conv_launch");
    if (!conv_supported(a))
        return cudaErrorInvalidValue;
    ConvParams cp;
    cp.xbc = a.xbc;
    cp.w = a.w;
    cp.bias = a.bias;
    cp.state_in = a.state_in;
    cp.x = a.x;
    cp.B = a.B;
    cp.C = a.C;
    cp.state_out = a.state_out;
    cp.L = a.seqlen;
    cp.HP = a.nheads * a.headdim;
    cp.GN = a.ngroups * a.dstate;
    cp.Cc = cp.HP + 2 * cp.GN;
    cp.nvec = cp.Cc / (a.dtype == SSD_DTYPE_BF16 ? conv_vec<__nv_bfloat16>() : conv_vec<float>());
    const dim3 grid((unsigned)((cp.nvec + kConvThreads - 1) / kConvThreads),
                    (unsigned)((a.seqlen + kConvTile - 1) / kConvTile), (unsigned)a.batch);
    const cudaError_t e = a.dtype == SSD_DTYPE_BF16 ? conv_launch_t<__nv_bfloat16>(a.kernel_size, cp, grid, st)
                                                    : conv_launch_t<float>(a.kernel_size, cp, grid, st);
    if (e == cudaSuccess)
        note_launches(1);
    return e;
}

// The x channels' part of the conv state after the sequence: the last K-1
// inputs (from the carried state when the sequence is shorter than K-1 steps,
// zero where neither has them).  Thread: one 8-channel bf16 vector of one batch row.
__global__ void __launch_bounds__(256) ssd_conv_state_tail_kernel(const __nv_bfloat16 *xbc, const __nv_bfloat16 *state_in,
                                                                  __nv_bfloat16 *state_out, long long L, int Cc,
                                                                  int nvec, int K)
{
    const int v = blockIdx.x * blockDim.x + threadIdx.x;
    if (v >= nvec)
        return;
    const long long b = blockIdx.y;
    for (int j = 0; j < K - 1; ++j) {
        const long long tt = L - (K - 1) + j;
        uint4 u = make_uint4(0u, 0u, 0u, 0u);
        if (tt >= 0)
            u = *reinterpret_cast<const uint4 *>(xbc + ((size_t)b * L + tt) * Cc + 8 * v);
        else if (state_in)
            u = *reinterpret_cast<const uint4 *>(state_in + ((size_t)b * (K - 1) + (K - 1) + tt) * Cc + 8 * v);
        *reinterpret_cast<uint4 *>(state_out + ((size_t)b * (K - 1) + j) * Cc + 8 * v) = u;
    }
}

cudaError_t conv_bc_launch(const NeighborArgs &a, cudaStream_t st)
{
    SSD_NVTX_RANGE("conv_bc_launch");
    if (!conv_supported(a) || a.dtype != SSD_DTYPE_BF16)
        return cudaErrorInvalidValue;
    ConvParams cp;
    cp.xbc = a.xbc;
    cp.w = a.w;
    cp.bias = a.bias;
    cp.state_in = a.state_in;
    cp.x = nullptr;   // (no x channel is handled)
    cp.B = a.B;
    cp.C = a.C;
    cp.state_out = a.state_out;
    cp.L = a.seqlen;
    cp.HP = a.nheads * a.headdim;
    cp.GN = a.ngroups * a.dstate;
    cp.Cc = cp.HP + 2 * cp.GN;
    constexpr int V = conv_vec<__nv_bfloat16>();
    cp.vbase = cp.HP / V;
    cp.nvec = cp.Cc / V;
    const dim3 grid((unsigned)((cp.nvec - cp.vbase + kConvThreads - 1) / kConvThreads),
                    (unsigned)((a.seqlen + kConvTile - 1) / kConvTile), (unsigned)a.batch);
    cudaError_t e = conv_launch_t<__nv_bfloat16>(a.kernel_size, cp, grid, st);
    if (e != cudaSuccess)
        return e;
    note_launches(1);
    if (a.state_out) {
        const int nv = cp.HP / V;
        ssd_conv_state_tail_kernel<<<dim3((unsigned)((nv + 255) / 256), (unsigned)a.batch), 256, 0, st>>>(
            static_cast<const __nv_bfloat16 *>(a.xbc), static_cast<const __nv_bfloat16 *>(a.state_in),
            static_cast<__nv_bfloat16 *>(a.state_out), a.seqlen, cp.Cc, nv, a.kernel_size);
        e = cudaGetLastError();
        if (e == cudaSuccess)
            note_launches(1);
    }
    return e;
}

bool gnorm_supported(const NeighborArgs &a)
{
    const long long D = (long long)a.nheads * a.headdim;
    return D % 8 == 0 && D <= (long long)kNormMaxThreads * kNormVPT * 8 && a.batch * a.seqlen <= 0x7FFFFFFFLL;
}

cudaError_t gnorm_launch(const NeighborArgs &a, cudaStream_t st)
{
    SSD_NVTX_RANGE("gnorm_launch");
    if (!gnorm_supported(a))
        return cudaErrorInvalidValue;
    NormParams np;
    np.y = a.y;
    np.z = a.z;
    np.w = a.w;
    np.out = a.out;
    np.D = a.nheads * a.headdim;
    np.eps = a.eps;
    const unsigned grid = (unsigned)(a.batch * a.seqlen);
    const int nv = np.D / 8;
    const int threads = ((nv + kNormVPT - 1) / kNormVPT + 31) / 32 * 32;   // whole warps
    if (a.dtype == SSD_DTYPE_BF16)
        ssd_gated_rmsnorm_kernel<__nv_bfloat16><<<grid, threads, 0, st>>>(np);
    else
        ssd_gated_rmsnorm_kernel<float><<<grid, threads, 0, st>>>(np);
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess)
        note_launches(1);
    return e;
}

}  // namespace ssd
