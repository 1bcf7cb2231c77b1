// ssd_bwd.cu -- the backward of the SSD scan, sequential in time.
//
// Forward (per batch row b, head h; dt_t = softplus(r_t + bias), a = -exp(A_log),
// dA_t = exp(dt_t a)):  h_t = dA_t h_{t-1} + dt_t B_t x_t^T,  y_t = C_t^T h_t + D x_t.
// Backward: the gradient of the state runs in reverse,
//   G_{L-1} = d_final + C_{L-1} dy_{L-1}^T,   G_t = dA_{t+1} G_{t+1} + C_t dy_t^T,
// and per step dx_t = D dy_t + dt_t G_t^T B_t, dB_t = dt_t G_t x_t, dC_t = h_t dy_t,
// ddt_t = sum G_t o (a dA_t h_{t-1} + B_t x_t^T), da += sum G_t o (dt_t dA_t h_{t-1}),
// dD += dy_t . x_t, d init = dA_0 G_0 (the derivatives of the recurrence the SSD
// module's forward defines).
//
// One CTA per (b, h); warp w owns state rows p = 4w .. 4w+3, lane l the states
// n = 4l .. 4l+3 (N <= 128), so G and the forward state sit in registers.  The
// reverse pass needs h_{t-1} and h_t at every step: the forward pass stores the
// state entering every segment of kSeg steps (checkpoints), and the reverse pass
// recomputes each segment's states into a per-(b, h) buffer (each thread writes
// and reads back only its own elements) before walking it backwards.  Sums over
// the rows (dB, dC, ddt) go through shared memory each step; sums over heads of
// a group and over batch rows are left to ssd_bwd_reduce_kernel, in a fixed
// order (no atomics: the gradients are deterministic).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ssd_internal.h"
#include "warp_rows.cuh"

namespace ssd {
namespace {

constexpr int kSeg = 64;      // steps per recomputed segment
constexpr int kRows = 4;      // state rows per warp
constexpr int kMaxWarps = 32; // P <= 128

struct BwdParams {
    const void *x, *B, *C, *dy;          // x, dy [B,L,H,P]; B, C [B,L,G,N] (dtype T)
    const float *dt_raw, *dt_bias, *A_log, *D;
    const float *init_state, *d_final;   // [B,H,P,N] or null
    float *dx, *ddt_raw;                 // [B,L,H,P], [B,L,H]
    float *d_init;                       // [B,H,P,N] or null
    float *ckpt, *seg;                   // [B,H,nseg,P,N], [B,H,kSeg,P,N]
    float *dB_head, *dC_head;            // [B,L,H,N]
    float *part;                         // [3][B,H]: da * a, d bias, dD per batch row
    long long L;
    int H, P, N, G, nseg;
};

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

__device__ __forceinline__ float softplus_f32(float z) { return fmaxf(z, 0.f) + log1pf(expf(-fabsf(z))); }

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// lane's 4 values of a row of N (n = 4 lane + e), zero past N
template <typename T>
__device__ __forceinline__ void load4(const T *row, int lane, int N, float (&v)[4])
{
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int n = 4 * lane + e;
        v[e] = n < N ? to_f32<T>(row[n]) : 0.f;
    }
}

template <typename T>
__global__ void __launch_bounds__(kMaxWarps * 32) ssd_bwd_kernel(BwdParams p)
{
    __shared__ float red_b[kMaxWarps][128];   // per-warp partial sums over its rows, per state n
    __shared__ float red_c[kMaxWarps][128];
    __shared__ float red_s[kMaxWarps][3];     // G.h_{t-1}, G.(B x^T), dy.x
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, W = blockDim.x >> 5;
    const int H = p.H, P = p.P, N = p.N, Gg = p.G;
    const long long L = p.L, bh = blockIdx.x, b = bh / H;
    const int h = (int)(bh - b * H), g = h / (H / Gg);
    const int p0 = warp * kRows;
    const bool ln = 4 * lane < N;             // this lane holds states
    const float a = -expf(p.A_log[h]), bias = p.dt_bias[h], Dh = p.D[h];
    const T *xg = static_cast<const T *>(p.x), *dyg = static_cast<const T *>(p.dy);
    const T *Bg = static_cast<const T *>(p.B), *Cg = static_cast<const T *>(p.C);
    const size_t PN = (size_t)P * N;
    auto ok = [&](int r) { return p0 + r < P && ln; };
    auto at = [&](int r) { return (size_t)(p0 + r) * N + 4 * lane; };   // offset in a [P,N] state

    float4 hs[kRows];
    // h <- dA_t h + dt_t B_t x_t^T for this thread's elements
    auto fwd_step = [&](long long t) {
        const size_t ti = (size_t)(b * L + t);
        const float dt = softplus_f32(p.dt_raw[ti * H + h] + bias), dA = expf(dt * a);
        float bv[4];
        load4(Bg + (ti * Gg + g) * N, lane, N, bv);
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const float dtx = dt * (p0 + r < P ? to_f32<T>(xg[(ti * H + h) * P + p0 + r]) : 0.f);
            hs[r].x = fmaf(dA, hs[r].x, dtx * bv[0]);
            hs[r].y = fmaf(dA, hs[r].y, dtx * bv[1]);
            hs[r].z = fmaf(dA, hs[r].z, dtx * bv[2]);
            hs[r].w = fmaf(dA, hs[r].w, dtx * bv[3]);
        }
    };

    // ---- phase 1: forward, storing the state entering each segment
#pragma unroll
    for (int r = 0; r < kRows; ++r)
        hs[r] = (p.init_state && ok(r)) ? *reinterpret_cast<const float4 *>(p.init_state + bh * PN + at(r))
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
    for (long long t = 0; t < L; ++t) {
        if (t % kSeg == 0) {
#pragma unroll
            for (int r = 0; r < kRows; ++r)
                if (ok(r))
                    *reinterpret_cast<float4 *>(p.ckpt + ((size_t)bh * p.nseg + t / kSeg) * PN + at(r)) = hs[r];
        }
        fwd_step(t);
    }

    // ---- phase 2: reverse, segment by segment
    float4 Gs[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r)
        Gs[r] = (p.d_final && ok(r)) ? *reinterpret_cast<const float4 *>(p.d_final + bh * PN + at(r))
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
    float acc_da = 0.f, acc_db = 0.f, acc_dd = 0.f;   // thread 0 / lane 0 of each warp
    float *segb = p.seg + (size_t)bh * kSeg * PN;
    for (int j = p.nseg - 1; j >= 0; --j) {
        const long long tb = (long long)j * kSeg, te = min(L, tb + kSeg);
        const float *ck = p.ckpt + ((size_t)bh * p.nseg + j) * PN;
#pragma unroll
        for (int r = 0; r < kRows; ++r)
            hs[r] = ok(r) ? *reinterpret_cast<const float4 *>(ck + at(r)) : make_float4(0.f, 0.f, 0.f, 0.f);
        for (long long t = tb; t < te; ++t) {   // recompute h_t, t in the segment
            fwd_step(t);
#pragma unroll
            for (int r = 0; r < kRows; ++r)
                if (ok(r))
                    *reinterpret_cast<float4 *>(segb + (size_t)(t - tb) * PN + at(r)) = hs[r];
        }
        for (long long t = te - 1; t >= tb; --t) {
            const size_t ti = (size_t)(b * L + t);
            const float z = p.dt_raw[ti * H + h] + bias;
            const float dt = softplus_f32(z), dA = expf(dt * a);
            if (t + 1 < L) {   // G_t = dA_{t+1} G_{t+1} + C_t dy_t^T
                const float dAn = expf(softplus_f32(p.dt_raw[(ti + 1) * H + h] + bias) * a);
#pragma unroll
                for (int r = 0; r < kRows; ++r) {
                    Gs[r].x *= dAn;
                    Gs[r].y *= dAn;
                    Gs[r].z *= dAn;
                    Gs[r].w *= dAn;
                }
            }
            float cv[4], bv[4], dyr[kRows], xr[kRows];
            load4(Cg + (ti * Gg + g) * N, lane, N, cv);
            load4(Bg + (ti * Gg + g) * N, lane, N, bv);
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                const bool in = p0 + r < P;
                dyr[r] = in ? to_f32<T>(dyg[(ti * H + h) * P + p0 + r]) : 0.f;
                xr[r] = in ? to_f32<T>(xg[(ti * H + h) * P + p0 + r]) : 0.f;
                Gs[r].x = fmaf(cv[0], dyr[r], Gs[r].x);
                Gs[r].y = fmaf(cv[1], dyr[r], Gs[r].y);
                Gs[r].z = fmaf(cv[2], dyr[r], Gs[r].z);
                Gs[r].w = fmaf(cv[3], dyr[r], Gs[r].w);
            }
            // dx_t rows: D dy + dt G^T B
            float sx[kRows];
#pragma unroll
            for (int r = 0; r < kRows; ++r)
                sx[r] = Gs[r].x * bv[0] + Gs[r].y * bv[1] + Gs[r].z * bv[2] + Gs[r].w * bv[3];
            warp_sum_rows_all<kRows>(sx, lane);
            {
                const int rr = summed_row<kRows>(lane);
                float dv = 0.f;
#pragma unroll
                for (int r = 0; r < kRows; ++r)
                    dv = r == rr ? dyr[r] : dv;
                if ((lane & (32 / kRows - 1)) == 0 && p0 + rr < P)
                    p.dx[(ti * H + h) * P + p0 + rr] = fmaf(Dh, dv, dt * sx[0]);
            }
            // per-lane partial sums over this warp's rows
            float pb[4] = {0.f, 0.f, 0.f, 0.f}, pc[4] = {0.f, 0.f, 0.f, 0.f}, gh = 0.f, gbx = 0.f, xd = 0.f;
            const bool has_prev = t > tb;
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                float4 ht = make_float4(0.f, 0.f, 0.f, 0.f), hp = ht;
                if (ok(r)) {
                    ht = *reinterpret_cast<const float4 *>(segb + (size_t)(t - tb) * PN + at(r));
                    hp = *reinterpret_cast<const float4 *>((has_prev ? segb + (size_t)(t - 1 - tb) * PN : ck) + at(r));
                }
                const float gv[4] = {Gs[r].x, Gs[r].y, Gs[r].z, Gs[r].w};
                const float hv[4] = {ht.x, ht.y, ht.z, ht.w}, pv[4] = {hp.x, hp.y, hp.z, hp.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    pb[e] = fmaf(gv[e], xr[r], pb[e]);
                    pc[e] = fmaf(hv[e], dyr[r], pc[e]);
                    gh = fmaf(gv[e], pv[e], gh);
                    gbx = fmaf(gv[e] * bv[e], xr[r], gbx);
                }
                xd = fmaf(dyr[r], xr[r], xd);
            }
            if (ln) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    red_b[warp][4 * lane + e] = pb[e];
                    red_c[warp][4 * lane + e] = pc[e];
                }
            }
            gh = warp_sum(gh);
            gbx = warp_sum(gbx);
            if (lane == 0) {
                red_s[warp][0] = gh;
                red_s[warp][1] = gbx;
                acc_dd += xd;
            }
            __syncthreads();
            for (int n = threadIdx.x; n < N; n += blockDim.x) {
                float sb = 0.f, sc = 0.f;
                for (int w = 0; w < W; ++w) {
                    sb += red_b[w][n];
                    sc += red_c[w][n];
                }
                p.dB_head[(ti * H + h) * N + n] = dt * sb;
                p.dC_head[(ti * H + h) * N + n] = sc;
            }
            if (threadIdx.x == 0) {
                float ghT = 0.f, gbT = 0.f;
                for (int w = 0; w < W; ++w) {
                    ghT += red_s[w][0];
                    gbT += red_s[w][1];
                }
                const float dr = fmaf(a * dA, ghT, gbT) / (1.f + expf(-z));   // ddt times sigmoid(z)
                p.ddt_raw[ti * H + h] = dr;
                acc_da = fmaf(dt * dA, ghT, acc_da);
                acc_db += dr;
            }
            __syncthreads();
        }
    }

    // ---- d init = dA_0 G_0; per-(b, h) partials of the per-head gradients
    if (p.d_init) {
        const float dA0 = expf(softplus_f32(p.dt_raw[(size_t)b * L * H + h] + bias) * a);
#pragma unroll
        for (int r = 0; r < kRows; ++r)
            if (ok(r))
                *reinterpret_cast<float4 *>(p.d_init + bh * PN + at(r)) =
                    make_float4(dA0 * Gs[r].x, dA0 * Gs[r].y, dA0 * Gs[r].z, dA0 * Gs[r].w);
    }
    if (lane == 0)
        red_s[warp][2] = acc_dd;
    __syncthreads();
    if (threadIdx.x == 0) {
        float dd = 0.f;
        for (int w = 0; w < W; ++w)
            dd += red_s[w][2];
        const long long BH = gridDim.x;
        p.part[bh] = acc_da * a;
        p.part[BH + bh] = acc_db;
        p.part[2 * BH + bh] = dd;
    }
}

// dB, dC [B,L,G,N]: the per-head gradients summed over the heads of each group,
// in head order.  One thread per (token, group, n).
__global__ void __launch_bounds__(256) ssd_bwd_reduce_kernel(const float *dB_head, const float *dC_head, float *dB,
                                                              float *dC, long long total, int H, int G, int N)
{
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;   // (row, g, n)
    if (i >= total)
        return;
    const int n = (int)(i % N);
    const long long rg = i / N;
    const int g = (int)(rg % G);
    const long long row = rg / G;
    const int hpg = H / G;
    float sb = 0.f, sc = 0.f;
    for (int k = 0; k < hpg; ++k) {
        const size_t o = ((size_t)row * H + g * hpg + k) * N + n;
        sb += dB_head[o];
        sc += dC_head[o];
    }
    dB[i] = sb;
    dC[i] = sc;
}

// dA_log, d dt_bias, dD [H]: the partials of (b, h) (nper of them, one per
// chunk or one per sequence) summed over batch rows and partials in order (b,
// then c).  They are loaded kBatch at a time so that those loads are in flight
// together; the sums and their order are those of the plain loop.
__device__ __forceinline__ void heads_sum(const float *part, float *dA_log, float *ddt_bias, float *dD, int Bt, int H,
                                          int nper, int h)
{
    const size_t BHC = (size_t)Bt * H * nper;
    float s0 = 0.f, s1 = 0.f, s2 = 0.f;
    constexpr int kBatch = 16;
    const long long n = (long long)Bt * nper;
    for (long long j0 = 0; j0 < n; j0 += kBatch) {
        float v0[kBatch], v1[kBatch], v2[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k)
            if (j0 + k < n) {
                const long long j = j0 + k, b = j / nper, c = j - b * nper;
                const size_t i = ((size_t)b * H + h) * nper + c;
                v0[k] = part[i];
                v1[k] = part[BHC + i];
                v2[k] = part[2 * BHC + i];
            }
#pragma unroll
        for (int k = 0; k < kBatch; ++k)
            if (j0 + k < n) {
                s0 += v0[k];
                s1 += v1[k];
                s2 += v2[k];
            }
    }
    dA_log[h] = s0;
    ddt_bias[h] = s1;
    dD[h] = s2;
}

__global__ void ssd_bwd_heads_kernel(const float *part, float *dA_log, float *ddt_bias, float *dD, int Bt, int H,
                                     int nper)
{
    const int h = blockIdx.x * blockDim.x + threadIdx.x;
    if (h < H)
        heads_sum(part, dA_log, ddt_bias, dD, Bt, H, nper, h);
}

// Both reductions in one launch.  The first hblocks CTAs sum the per-head
// partials (one thread per head).  The others take dB and dC with four
// consecutive n per thread (16-byte loads; N % 4 == 0 and 16-byte aligned
// tensors) and the loads of 8 heads in flight at once; each element is still
// summed over the heads in order, so the results are those of the scalar form
// bit for bit.  The two parts read what the launch before wrote and share
// nothing.
__global__ void __launch_bounds__(256) ssd_bwd_finish4_kernel(const float4 *dB_head, const float4 *dC_head,
                                                               float4 *dB, float4 *dC, long long total4, int H, int G,
                                                               int N4, const float *part, float *dA_log,
                                                               float *ddt_bias, float *dD, int Bt, int nper,
                                                               int hblocks)
{
    if ((int)blockIdx.x < hblocks) {
        const int h = blockIdx.x * blockDim.x + threadIdx.x;
        if (h < H)
            heads_sum(part, dA_log, ddt_bias, dD, Bt, H, nper, h);
        return;
    }
    const long long i = (long long)(blockIdx.x - hblocks) * blockDim.x + threadIdx.x;   // (row, g, n / 4)
    if (i >= total4)
        return;
    const int n4 = (int)(i % N4);
    const long long rg = i / N4;
    const int g = (int)(rg % G);
    const long long row = rg / G;
    const int hpg = H / G;
    const float4 *pb = dB_head + ((size_t)row * H + (size_t)g * hpg) * N4 + n4;
    const float4 *pc = dC_head + ((size_t)row * H + (size_t)g * hpg) * N4 + n4;
    float4 sb = make_float4(0.f, 0.f, 0.f, 0.f), sc = sb;
    constexpr int kBatch = 8;
    for (int k0 = 0; k0 < hpg; k0 += kBatch) {
        float4 vb[kBatch], vc[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k)
            if (k0 + k < hpg) {
                vb[k] = __ldcs(pb + (size_t)(k0 + k) * N4);
                vc[k] = __ldcs(pc + (size_t)(k0 + k) * N4);
            }
#pragma unroll
        for (int k = 0; k < kBatch; ++k)
            if (k0 + k < hpg) {
                sb.x += vb[k].x; sb.y += vb[k].y; sb.z += vb[k].z; sb.w += vb[k].w;
                sc.x += vc[k].x; sc.y += vc[k].y; sc.z += vc[k].z; sc.w += vc[k].w;
            }
    }
    dB[i] = sb;
    dC[i] = sc;
}

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

}  // namespace

bool bwd_seq_supported(const BwdArgs &a)
{
    return a.dstate % 4 == 0 && a.dstate <= 128 && a.headdim >= 1 && a.headdim <= kMaxWarps * kRows &&
           a.batch * (long long)a.nheads <= 0x7FFFFFFFLL && a.seqlen < (1LL << 31);
}

bool bwd_supported(const BwdArgs &a)
{
    return a.path == SSD_PATH_CHUNKED ? bwd_chunk_supported(a) : bwd_seq_supported(a);
}

size_t bwd_workspace_bytes(const BwdArgs &a)
{
    if (a.path == SSD_PATH_CHUNKED)
        return bwd_chunk_workspace_bytes(a);
    const size_t BH = (size_t)a.batch * a.nheads, PN = (size_t)a.headdim * a.dstate;
    const size_t nseg = (size_t)((a.seqlen + kSeg - 1) / kSeg);
    const size_t BLHN = (size_t)a.batch * a.seqlen * a.nheads * a.dstate;
    return align256(BH * nseg * PN * 4) + align256(BH * kSeg * PN * 4) + 2 * align256(BLHN * 4) +
           align256(3 * BH * 4);
}

cudaError_t bwd_finish_launch(const BwdArgs &a, const float *dB_head, const float *dC_head, const float *part,
                              int nper, cudaStream_t st)
{
    SSD_NVTX_RANGE("bwd_finish_launch");
    const long long total = (long long)a.batch * a.seqlen * a.ngroups * a.dstate;
    auto aligned16 = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
    if (a.dstate % 4 == 0 && aligned16(dB_head) && aligned16(dC_head) && aligned16(a.dB) && aligned16(a.dC)) {
        const int hblocks = (a.nheads + 255) / 256;
        ssd_bwd_finish4_kernel<<<(unsigned)(hblocks + (total / 4 + 255) / 256), 256, 0, st>>>(
            reinterpret_cast<const float4 *>(dB_head), reinterpret_cast<const float4 *>(dC_head),
            reinterpret_cast<float4 *>(a.dB), reinterpret_cast<float4 *>(a.dC), total / 4, a.nheads, a.ngroups,
            a.dstate / 4, part, a.dA_log, a.ddt_bias, a.dD, (int)a.batch, nper, hblocks);
        const cudaError_t e = cudaGetLastError();
        if (e == cudaSuccess)
            note_launches(1);
        return e;
    }
    ssd_bwd_reduce_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(dB_head, dC_head, a.dB, a.dC, total,
                                                                          a.nheads, a.ngroups, a.dstate);
    ssd_bwd_heads_kernel<<<(a.nheads + 127) / 128, 128, 0, st>>>(part, a.dA_log, a.ddt_bias, a.dD, (int)a.batch,
                                                                 a.nheads, nper);
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess)
        note_launches(2);
    return e;
}

cudaError_t bwd_launch(const BwdArgs &a, void *ws, cudaStream_t st)
{
    SSD_NVTX_RANGE("bwd_launch");
    if (!bwd_supported(a))
        return cudaErrorInvalidValue;
    if (a.path == SSD_PATH_CHUNKED)
        return bwd_chunk_launch(a, ws, st);
    const size_t BH = (size_t)a.batch * a.nheads, PN = (size_t)a.headdim * a.dstate;
    const int nseg = (int)((a.seqlen + kSeg - 1) / kSeg);
    const size_t BLHN = (size_t)a.batch * a.seqlen * a.nheads * a.dstate;
    char *w = static_cast<char *>(ws);
    BwdParams p;
    p.x = a.x;
    p.B = a.B;
    p.C = a.C;
    p.dy = a.dy;
    p.dt_raw = a.dt_raw;
    p.dt_bias = a.dt_bias;
    p.A_log = a.A_log;
    p.D = a.D;
    p.init_state = a.init_state;
    p.d_final = a.d_final;
    p.dx = a.dx;
    p.ddt_raw = a.ddt_raw;
    p.d_init = a.d_init;
    p.ckpt = reinterpret_cast<float *>(w);
    w += align256(BH * nseg * PN * 4);
    p.seg = reinterpret_cast<float *>(w);
    w += align256(BH * kSeg * PN * 4);
    p.dB_head = reinterpret_cast<float *>(w);
    w += align256(BLHN * 4);
    p.dC_head = reinterpret_cast<float *>(w);
    w += align256(BLHN * 4);
    p.part = reinterpret_cast<float *>(w);
    p.L = a.seqlen;
    p.H = a.nheads;
    p.P = a.headdim;
    p.N = a.dstate;
    p.G = a.ngroups;
    p.nseg = nseg;
    const int threads = 32 * ((a.headdim + kRows - 1) / kRows);
    if (a.dtype == SSD_DTYPE_BF16)
        ssd_bwd_kernel<__nv_bfloat16><<<(unsigned)BH, threads, 0, st>>>(p);
    else
        ssd_bwd_kernel<float><<<(unsigned)BH, threads, 0, st>>>(p);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    note_launches(1);
    return bwd_finish_launch(a, p.dB_head, p.dC_head, p.part, 1, st);
}

}  // namespace ssd
