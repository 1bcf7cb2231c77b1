// ssd_bwd_chunk.cu -- the backward of the SSD scan in chunk form (chunks of
// kQ = 64 steps processed in parallel), the chunk structure of the Mamba-2 SSD
// algorithm run in reverse.
//
// Per batch row b and head h, within one chunk (local steps i = 0 .. Q-1,
// cs_i = sum_{k <= i} dt_k a the inclusive cumsum of the log decays, h_in the
// state entering the chunk, G_out = dL/dh at the chunk's last step through
// the later steps only):
//   h_i  = e^{cs_i} h_in + sum_{j <= i} e^{cs_i - cs_j} dt_j B_j x_j^T
//   G_i  = sum_{s >= i} e^{cs_s - cs_i} C_s dy_s^T + e^{cs_last - cs_i} G_out
// and the chunks are linked by
//   h_in(c+1)  = e^{cs_last(c)} h_in(c) + S(c),   S(c) = sum_j e^{cs_last - cs_j} dt_j B_j x_j^T
//   G_out(c-1) = e^{cs_last(c)} G_out(c) + R(c),  R(c) = sum_s e^{cs_s} C_s dy_s^T
// (G_out(-1) = dA_0 G_0 is d init).  Three launches:
//   1. ssd_bwd_local_kernel: S(c), R(c) and e^{cs_last(c)} for every chunk;
//   2. ssd_bwd_pass_kernel: the two chains above, element-wise over the state,
//      overwriting S(c) by h_in(c) (and the slot past the last by the final
//      state) and R(c) by G_out(c);
//   3. ssd_bwd_grad_kernel: every gradient of one chunk from h_in, G_out and
//      the chunk's inputs, as dense contractions (CB = C B^T, DX = dy x^T,
//      E = causal e^{cs_s - cs_j}):
//        dx_j = D dy_j + dt_j (sum_s E CB [s,j] dy_s + e^{cs_last-cs_j} G_out^T B_j)
//        dB_j = dt_j (sum_s E DX [s,j] C_s + e^{cs_last-cs_j} G_out x_j)
//        dC_s = sum_j E DX [s,j] dt_j B_j + e^{cs_s} h_in dy_s
//      and d log dA_j = sum_{k >= j} dL/dcs_k, with dL/dcs_k the row-minus-
//      column sum of W = E CB DX dt_j, plus e^{cs_k} dy_k . (h_in^T C_k), minus
//      e^{cs_last-cs_k} dt_k x_k . (G_out^T B_k), plus <G_out, h_last> at the
//      chunk's last step; ddt = x . (G^T B) + a d log dA, dA_log = a sum dt d log dA.
// The contractions are shared-memory tiled fp32 FFMA: every operand sits in
// shared memory (the states also transposed) with rows of 4 mod 32 words,
// each thread owns a 4 x 4, 4 x 8 or 8 x 4 output tile, and every operand
// read is a conflict-free 16-byte load (see contract()).  Sums over chunks,
// batch rows and a group's heads are left to the fixed-order reduction
// kernels (deterministic gradients).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "f32x2.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kQ = 64;        // steps per chunk
constexpr int kPM = 64;       // largest headdim of this path
constexpr int kNM = 128;      // largest dstate of this path
constexpr int kLP = kPM + 4;  // shared-memory row strides: 16-byte rows, = 4 mod 32 words
constexpr int kLN = kNM + 4;
constexpr int kLQ = kQ + 4;
constexpr int kThreads = 256; // 16 x 16 threads, output tiles strided by 16

struct ChunkBwdParams {
    const void *x, *B, *C, *dy;          // x, dy [B,L,H,P]; B, C [B,L,G,N]
    const float *dt_raw, *dt_bias, *A_log, *D;
    const float *init_state, *d_final;   // [B,H,P,N] or null
    float *dx, *ddt_raw, *d_init;        // [B,L,H,P], [B,L,H], [B,H,P,N] or null
    float *S;                            // [B*H][nc+1][N][P]: S(c), then h_in(c); slot nc the final state
    float *R;                            // [B*H][nc][N][P]: R(c), then G_out(c)
    float *dec;                          // [B*H][nc]: e^{cs_last(c)}
    float *dB_head, *dC_head;            // [B,L,H,N]
    float *part;                         // [3][B*H*nc]: a * sum dt dlogdA, sum ddt_raw, sum dy.x per chunk
    long long L;
    int H, P, N, G, nc;
};

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

__device__ __forceinline__ float softplus_f32(float z) { return fmaxf(z, 0.f) + log1pf(expf(-fabsf(z))); }

// Thread (ty, tx) = (tid / 16, tid % 16) owns a TM x TN output tile.  Its
// rows are TM ty + i (contiguous, RC) or ty + 16 i; its columns 4 tx + j % 4
// + 64 (j / 4) (contiguous groups of four) when B is k-major, else tx + 16 j.
template <int TM, bool RC>
__device__ __forceinline__ int tile_row(int i) { return RC ? TM * (threadIdx.x >> 4) + i : (threadIdx.x >> 4) + 16 * i; }
template <bool BK>
__device__ __forceinline__ int tile_col(int j) { return BK ? 4 * (threadIdx.x & 15) + (j & 3) + 64 * (j >> 2) : (threadIdx.x & 15) + 16 * j; }

// acc[i][j] += sum_{k_lo <= k < k_hi} A(row_i, k) B(k, col_j) (times kscale[k]
// if given; k_hi = -1 means K), operands in shared memory, rows 16-byte
// aligned, K, k_lo and k_hi multiples of 4.  The bounds let a contraction with
// a causal factor skip the blocks of k where that factor is zero for all of
// the thread's rows (adding those exact zeros would not change the sums).  A is k-major
// (A[k * lda + m]; needs RC) when AK, else m-major (A[m * lda + k]); B is
// k-major (B[k * ldb + n]) when BK, else n-major (B[n * ldb + k]; ldb = 4 mod
// 32).  Every read is a 16-byte load: along m or n for a k-major operand,
// along k otherwise.  Within a warp A reads hit two addresses (broadcast) and
// B reads 16 distinct 16-byte words in distinct banks: no conflicts.
template <int TM, int TN, int K, bool AK, bool RC, bool BK>
__device__ __forceinline__ void contract(float (&acc)[TM][TN], const float *A, int lda, const float *B, int ldb,
                                         const float *kscale = nullptr, int k_lo = 0, int k_hi = -1)
{
    static_assert(!AK || RC, "a k-major A needs contiguous rows");
    static_assert(TM % 4 == 0 && TN % 4 == 0 && K % 4 == 0, "whole 16-byte words");
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int kend = k_hi < 0 ? K : k_hi;
    // packed accumulators (f32x2): along j for a k-major B (starting from acc), else
    // along k (starting from zero, added to acc at the end)
    f32x2 accj[TM][BK ? TN / 2 : 1], acck[TM][BK ? 1 : TN];
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        if constexpr (BK) {
#pragma unroll
            for (int j = 0; j < TN / 2; ++j)
                accj[i][j] = pk2(acc[i][2 * j], acc[i][2 * j + 1]);
        } else {
#pragma unroll
            for (int j = 0; j < TN; ++j)
                acck[i][j] = pk2(0.f, 0.f);
        }
    }
#pragma unroll 2
    for (int k = k_lo; k < kend; k += 4) {
        float av[TM][4], bv[4][TN];
        if constexpr (AK) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                for (int iv = 0; iv < TM / 4; ++iv) {
                    const float4 t = *reinterpret_cast<const float4 *>(A + (k + kk) * lda + TM * ty + 4 * iv);
                    av[4 * iv][kk] = t.x;
                    av[4 * iv + 1][kk] = t.y;
                    av[4 * iv + 2][kk] = t.z;
                    av[4 * iv + 3][kk] = t.w;
                }
        } else {
#pragma unroll
            for (int i = 0; i < TM; ++i) {
                const float4 t = *reinterpret_cast<const float4 *>(A + tile_row<TM, RC>(i) * lda + k);
                av[i][0] = t.x;
                av[i][1] = t.y;
                av[i][2] = t.z;
                av[i][3] = t.w;
            }
        }
        if (kscale) {
            const float4 s = *reinterpret_cast<const float4 *>(kscale + k);
#pragma unroll
            for (int i = 0; i < TM; ++i) {
                av[i][0] *= s.x;
                av[i][1] *= s.y;
                av[i][2] *= s.z;
                av[i][3] *= s.w;
            }
        }
        if constexpr (BK) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                for (int jv = 0; jv < TN / 4; ++jv) {
                    const float4 t = *reinterpret_cast<const float4 *>(B + (k + kk) * ldb + 4 * tx + 64 * jv);
                    bv[kk][4 * jv] = t.x;
                    bv[kk][4 * jv + 1] = t.y;
                    bv[kk][4 * jv + 2] = t.z;
                    bv[kk][4 * jv + 3] = t.w;
                }
        } else {
#pragma unroll
            for (int j = 0; j < TN; ++j) {
                const float4 t = *reinterpret_cast<const float4 *>(B + (tx + 16 * j) * ldb + k);
                bv[0][j] = t.x;
                bv[1][j] = t.y;
                bv[2][j] = t.z;
                bv[3][j] = t.w;
            }
        }
        if constexpr (BK) {
            // B's 16-byte words hold neighbouring columns: pairs along j, the
            // operations of acc[i][j] += A B unchanged
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                for (int i = 0; i < TM; ++i) {
                    const f32x2 a2 = pk2(av[i][kk], av[i][kk]);
#pragma unroll
                    for (int j = 0; j < TN / 2; ++j)
                        accj[i][j] = fma2(a2, pk2(bv[kk][2 * j], bv[kk][2 * j + 1]), accj[i][j]);
                }
        } else {
            // both operands' words run along k: pairs along k, two partial sums
#pragma unroll
            for (int kk = 0; kk < 4; kk += 2)
#pragma unroll
                for (int i = 0; i < TM; ++i) {
                    const f32x2 a2 = pk2(av[i][kk], av[i][kk + 1]);
#pragma unroll
                    for (int j = 0; j < TN; ++j)
                        acck[i][j] = fma2(a2, pk2(bv[kk][j], bv[kk + 1][j]), acck[i][j]);
                }
        }
    }
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        if constexpr (BK) {
#pragma unroll
            for (int j = 0; j < TN / 2; ++j) {
                acc[i][2 * j] = lo2(accj[i][j]);
                acc[i][2 * j + 1] = hi2(accj[i][j]);
            }
        } else {
#pragma unroll
            for (int j = 0; j < TN; ++j)
                acc[i][j] += lo2(acck[i][j]) + hi2(acck[i][j]);
        }
    }
}

template <int TM, int TN>
__device__ __forceinline__ void zero(float (&acc)[TM][TN])
{
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j)
            acc[i][j] = 0.f;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// v[0..3] to row[c0 .. c0 + 3], the columns below cols only (one 16-byte
// store where the row and cols allow it)
__device__ __forceinline__ void store4(float *row, int c0, int cols, const float (&v)[4])
{
    if (cols % 4 == 0 && (reinterpret_cast<uintptr_t>(row) & 15) == 0) {
        if (c0 < cols)
            *reinterpret_cast<float4 *>(row + c0) = make_float4(v[0], v[1], v[2], v[3]);
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (c0 + e < cols)
                row[c0 + e] = v[e];
    }
}

// sum over the 16 threads of a half warp (the threads sharing a tile row)
__device__ __forceinline__ float half_warp_sum(float v)
{
#pragma unroll
    for (int o = 8; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// the chunk's dt, z = dt_raw + bias and inclusive cumsum of dt a, in shared
// memory (zero dt past the sequence's end, so cs stays flat there)
__device__ __forceinline__ void chunk_decays(const ChunkBwdParams &p, long long b, int h, long long t0, int nq,
                                             float a, float *dt_s, float *z_s, float *cs_s)
{
    const int tid = threadIdx.x;
    if (tid < kQ) {
        float dt = 0.f, z = 0.f;
        if (tid < nq) {
            z = p.dt_raw[(size_t)(b * p.L + t0 + tid) * p.H + h] + p.dt_bias[h];
            dt = softplus_f32(z);
        }
        dt_s[tid] = dt;
        z_s[tid] = z;
        float v = dt * a;   // inclusive scan within each of the two warps
        const int lane = tid & 31;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float u = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o)
                v += u;
        }
        cs_s[tid] = v;
    }
    __syncthreads();
    if (tid >= 32 && tid < kQ)
        cs_s[tid] += cs_s[31];
    __syncthreads();
}

// the V = 16 / sizeof(T) values of a 16-byte vector as fp32
__device__ __forceinline__ void unpack(const uint4 &u, float (&v)[4]) {
    v[0] = __uint_as_float(u.x);
    v[1] = __uint_as_float(u.y);
    v[2] = __uint_as_float(u.z);
    v[3] = __uint_as_float(u.w);
}
__device__ __forceinline__ void unpack(const uint4 &u, float (&v)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {   // little-endian: the lower half is the earlier element
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// Rows r < nrows (of ROWS) and columns c < cols (of CMAX) of a row-major
// tensor (row stride row_stride elements) into shared memory as fp32, row
// stride ld, each row times scale[r] when scale is given; zero elsewhere.
// load() issues this thread's 16-byte loads and store() writes them, so a
// kernel can have the loads of several tiles in flight at once.  Where rows
// are not 16-byte aligned, store() falls back to scalar loads.
template <typename T, int ROWS, int CMAX>
struct RowTile {
    static constexpr int V = 16 / sizeof(T), VPR = CMAX / V, IT = ROWS * VPR / kThreads;
    static_assert(ROWS * VPR % kThreads == 0, "whole vectors per thread");
    uint4 buf[IT];
    const T *src;
    size_t row_stride;
    int nrows, cols;
    bool vec;
    __device__ __forceinline__ void load(const T *src_, size_t row_stride_, int nrows_, int cols_)
    {
        src = src_;
        row_stride = row_stride_;
        nrows = nrows_;
        cols = cols_;
        vec = cols % V == 0 && row_stride % V == 0 && (reinterpret_cast<uintptr_t>(src) & 15) == 0;
        if (!vec)
            return;
#pragma unroll
        for (int it = 0; it < IT; ++it) {
            const int idx = it * kThreads + threadIdx.x, r = idx / VPR, cv = idx % VPR;
            buf[it] = (r < nrows && cv * V < cols)
                          ? *reinterpret_cast<const uint4 *>(src + (size_t)r * row_stride + cv * V)
                          : make_uint4(0u, 0u, 0u, 0u);
        }
    }
    __device__ __forceinline__ void store(float *dst, int ld, const float *scale = nullptr) const
    {
        if (vec) {
#pragma unroll
            for (int it = 0; it < IT; ++it) {
                const int idx = it * kThreads + threadIdx.x, r = idx / VPR, cv = idx % VPR;
                float v[V];
                unpack(buf[it], v);
                const float s = scale ? scale[r] : 1.f;
#pragma unroll
                for (int e = 0; e < V; ++e)
                    dst[r * ld + cv * V + e] = s * v[e];
            }
        } else {
            for (int i = threadIdx.x; i < ROWS * CMAX; i += kThreads) {
                const int r = i / CMAX, c = i % CMAX;
                dst[r * ld + c] = (r < nrows && c < cols)
                                      ? (scale ? scale[r] : 1.f) * to_f32<T>(src[(size_t)r * row_stride + c])
                                      : 0.f;
            }
        }
    }
};

template <typename T, int ROWS, int CMAX>
__device__ __forceinline__ void stage(float *dst, int ld, const T *src, size_t row_stride, int nrows, int cols)
{
    RowTile<T, ROWS, CMAX> t;
    t.load(src, row_stride, nrows, cols);
    t.store(dst, ld);
}

// 1. S(c) = sum_j e^{cs_last - cs_j} dt_j B_j x_j^T and R(c) = sum_s e^{cs_s} C_s dy_s^T
//    ([N,P] each) and e^{cs_last(c)}.  Grid (nc, B*H).  Thread tile: 8 rows n
//    (ty + 16 i) x 4 columns p (tx + 16 j).
template <typename T>
__global__ void __launch_bounds__(kThreads) ssd_bwd_local_kernel(ChunkBwdParams p)
{
    extern __shared__ __align__(16) float smem[];
    float *Bs = smem, *Cs = Bs + kQ * kLN, *xw = Cs + kQ * kLN, *dyw = xw + kQ * kLP;
    float *dt_s = dyw + kQ * kLP, *z_s = dt_s + kQ, *cs_s = z_s + kQ, *w_s = cs_s + kQ, *e_s = w_s + kQ;
    const int H = p.H, P = p.P, N = p.N, Gg = p.G, nc = p.nc;
    const long long bh = blockIdx.y, b = bh / H;
    const int h = (int)(bh - b * H), g = h / (H / Gg), c = blockIdx.x;
    const long long t0 = (long long)c * kQ;
    const int nq = (int)min((long long)kQ, p.L - t0);
    const float a = -expf(p.A_log[h]);
    const T *xg = static_cast<const T *>(p.x) + ((size_t)(b * p.L + t0) * H + h) * P;
    const T *dyg = static_cast<const T *>(p.dy) + ((size_t)(b * p.L + t0) * H + h) * P;
    const T *Bg = static_cast<const T *>(p.B) + ((size_t)(b * p.L + t0) * Gg + g) * N;
    const T *Cg = static_cast<const T *>(p.C) + ((size_t)(b * p.L + t0) * Gg + g) * N;
    RowTile<T, kQ, kNM> tB, tC;
    RowTile<T, kQ, kPM> tx, tdy;
    tB.load(Bg, (size_t)Gg * N, nq, N);   // every load in flight before the first store
    tC.load(Cg, (size_t)Gg * N, nq, N);
    tx.load(xg, (size_t)H * P, nq, P);
    tdy.load(dyg, (size_t)H * P, nq, P);
    chunk_decays(p, b, h, t0, nq, a, dt_s, z_s, cs_s);
    if (threadIdx.x < kQ) {
        const int j = threadIdx.x;
        w_s[j] = expf(cs_s[kQ - 1] - cs_s[j]) * dt_s[j];
        e_s[j] = expf(cs_s[j]);
    }
    __syncthreads();
    tB.store(Bs, kLN);
    tC.store(Cs, kLN);
    tx.store(xw, kLP, w_s);
    tdy.store(dyw, kLP, e_s);
    __syncthreads();
    const size_t NP = (size_t)N * P;
    const int p0 = tile_col<true>(0);   // this thread's four columns p0 .. p0 + 3
    float acc[8][4];
    zero(acc);
    contract<8, 4, kQ, true, true, true>(acc, Bs, kLN, xw, kLP);
    float *Sd = p.S + ((size_t)bh * (nc + 1) + c) * NP;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int n = tile_row<8, true>(i);
        if (n < N)
            store4(Sd + (size_t)n * P, p0, P, acc[i]);
    }
    zero(acc);
    contract<8, 4, kQ, true, true, true>(acc, Cs, kLN, dyw, kLP);
    float *Rd = p.R + ((size_t)bh * nc + c) * NP;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int n = tile_row<8, true>(i);
        if (n < N)
            store4(Rd + (size_t)n * P, p0, P, acc[i]);
    }
    if (threadIdx.x == 0)
        p.dec[bh * nc + c] = expf(cs_s[kQ - 1]);
}

// 2. The chains over chunks.  blockIdx.z = 0: S(c) <- h_in(c) (slot nc <- the
//    final state); blockIdx.z = 1: R(c) <- G_out(c), d init <- G_out(-1).  Each
//    thread runs one chain over kVec consecutive state elements (n, p) of one
//    (b, h), loading kBatch chunks ahead so that the loads of a batch are all
//    in flight together (the stores of a batch go to other addresses).  Two
//    blocks per SM (128 registers): one block per SM at 142 registers left the
//    loads of only 8 warps per SM in flight (the whole backward on 2 x 1024
//    steps, 80 heads: 0.370 ms, against 0.344 ms capped); batches of 8 at three
//    blocks per SM measured 0.375 ms.
constexpr int kVec = 4, kBatch = 16;
template <int V>
__device__ __forceinline__ void chain(float *buf, size_t stride, const float *dec, int nc, bool reverse,
                                      float (&v)[V])
{
    for (int c0 = 0; c0 < nc; c0 += kBatch) {
        float x[kBatch][V], d[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const int c = reverse ? nc - 1 - (c0 + k) : c0 + k;
            if (c0 + k < nc) {
                d[k] = dec[c];
                if constexpr (V == 4) {
                    const float4 t = *reinterpret_cast<const float4 *>(buf + c * stride);
                    x[k][0] = t.x; x[k][1] = t.y; x[k][2] = t.z; x[k][3] = t.w;
                } else {
                    x[k][0] = buf[c * stride];
                }
            }
        }
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const int c = reverse ? nc - 1 - (c0 + k) : c0 + k;
            if (c0 + k < nc) {
                if constexpr (V == 4)
                    *reinterpret_cast<float4 *>(buf + c * stride) = make_float4(v[0], v[1], v[2], v[3]);
                else
                    buf[c * stride] = v[0];
#pragma unroll
                for (int e = 0; e < V; ++e)
                    v[e] = fmaf(d[k], v[e], x[k][e]);
            }
        }
    }
}

// kTr (P = 64, N % 16 == 0, V = 4, 16-byte aligned [B,H,P,N] tensors): a block's
// 1024 elements are 16 whole rows n, and the [P][N] tensors (the initial state
// or d final in, d init out) pass through a shared-memory transpose, so their
// loads and stores are 64-byte segments rather than 4-byte pieces 4 N bytes
// apart.
constexpr int kTrLd = 17;   // transpose row stride (floats)
template <int V, bool kTr>
__global__ void __launch_bounds__(kThreads, 2) ssd_bwd_pass_kernel(ChunkBwdParams p)
{
    const int P = p.P, N = p.N, nc = p.nc;
    const long long bh = blockIdx.y;
    const int NP = N * P, e0 = (blockIdx.x * kThreads + threadIdx.x) * V;
    __shared__ float tr[kTr ? kPM * kTrLd : 1];
    if (!kTr && e0 >= NP)
        return;
    const float *dec = p.dec + bh * nc;
    const bool fwd = blockIdx.z == 0;
    const float *in = fwd ? p.init_state : p.d_final;   // [B,H,P,N] or null
    const int nb = (int)blockIdx.x * (kThreads * V / kPM);   // kTr: the block's first row n
    float v[V];
    if constexpr (kTr) {
        const int t = threadIdx.x, pr = t >> 2, n4 = 4 * (t & 3);
        const float4 f = in ? *reinterpret_cast<const float4 *>(in + (size_t)bh * NP + (size_t)pr * N + nb + n4)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
        tr[pr * kTrLd + n4] = f.x;
        tr[pr * kTrLd + n4 + 1] = f.y;
        tr[pr * kTrLd + n4 + 2] = f.z;
        tr[pr * kTrLd + n4 + 3] = f.w;
        __syncthreads();
        const int nn = e0 / P - nb, col = e0 % P;
#pragma unroll
        for (int e = 0; e < V; ++e)
            v[e] = tr[(col + e) * kTrLd + nn];
    } else {
#pragma unroll
        for (int e = 0; e < V; ++e) {
            const int n = (e0 + e) / P, col = (e0 + e) - n * P;
            v[e] = in ? in[(size_t)bh * NP + (size_t)col * N + n] : 0.f;
        }
    }
    if (fwd) {
        float *S = p.S + (size_t)bh * (nc + 1) * NP + e0;
        chain<V>(S, (size_t)NP, dec, nc, false, v);
        if constexpr (V == 4)
            *reinterpret_cast<float4 *>(S + (size_t)nc * NP) = make_float4(v[0], v[1], v[2], v[3]);
        else
            S[(size_t)nc * NP] = v[0];
    } else {
        chain<V>(p.R + (size_t)bh * nc * NP + e0, (size_t)NP, dec, nc, true, v);
        if (p.d_init) {
            if constexpr (kTr) {
                const int nn = e0 / P - nb, col = e0 % P;
                __syncthreads();   // every thread has read its initial values
#pragma unroll
                for (int e = 0; e < V; ++e)
                    tr[(col + e) * kTrLd + nn] = v[e];
                __syncthreads();
                const int t = threadIdx.x, pr = t >> 2, n4 = 4 * (t & 3);
                *reinterpret_cast<float4 *>(p.d_init + (size_t)bh * NP + (size_t)pr * N + nb + n4) =
                    make_float4(tr[pr * kTrLd + n4], tr[pr * kTrLd + n4 + 1], tr[pr * kTrLd + n4 + 2],
                                tr[pr * kTrLd + n4 + 3]);
            } else {
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    const int n = (e0 + e) / P, col = (e0 + e) - n * P;
                    p.d_init[(size_t)bh * NP + (size_t)col * N + n] = v[e];
                }
            }
        }
    }
}

// A [N,P] fp32 state (N <= kNM, P <= kPM) in two steps: load() issues this
// thread's 16-byte loads (consecutive threads take consecutive rows n), the
// stores then put it into shared memory straight (row stride kLP) and / or
// transposed (dst[p * kLN + n]); zero past N, P.  Both store patterns are
// free of bank conflicts.  Needs P % 4 == 0 (else the scalar fallbacks).
struct StateTile {
    static constexpr int IT = kNM * (kPM / 4) / kThreads;
    float4 v[IT];
    __device__ __forceinline__ static int row(int it) { return (it * kThreads + (int)threadIdx.x) % kNM; }
    __device__ __forceinline__ static int cv(int it) { return (it * kThreads + (int)threadIdx.x) / kNM; }
    __device__ __forceinline__ void load(const float *src, int N, int P)
    {
#pragma unroll
        for (int it = 0; it < IT; ++it)
            v[it] = (row(it) < N && 4 * cv(it) < P)
                        ? *reinterpret_cast<const float4 *>(src + (size_t)row(it) * P + 4 * cv(it))
                        : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __device__ __forceinline__ void store(float *dst) const
    {
#pragma unroll
        for (int it = 0; it < IT; ++it)
            *reinterpret_cast<float4 *>(dst + row(it) * kLP + 4 * cv(it)) = v[it];
    }
    __device__ __forceinline__ void store_t(float *dst) const
    {
#pragma unroll
        for (int it = 0; it < IT; ++it) {
            float *d = dst + (4 * cv(it)) * kLN + row(it);
            d[0] = v[it].x;
            d[kLN] = v[it].y;
            d[2 * kLN] = v[it].z;
            d[3 * kLN] = v[it].w;
        }
    }
    // sum of this thread's elements times the same elements of another state
    __device__ __forceinline__ float dot(const float *other, int N, int P) const
    {
        float s = 0.f;
        float4 o[IT];
#pragma unroll
        for (int it = 0; it < IT; ++it)
            o[it] = (row(it) < N && 4 * cv(it) < P)
                        ? *reinterpret_cast<const float4 *>(other + (size_t)row(it) * P + 4 * cv(it))
                        : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int it = 0; it < IT; ++it)
            s = fmaf(v[it].x, o[it].x, fmaf(v[it].y, o[it].y, fmaf(v[it].z, o[it].z, fmaf(v[it].w, o[it].w, s))));
        return s;
    }
};

// scalar fallbacks (P % 4 != 0): straight and transposed
__device__ __forceinline__ void stage_state(float *dst, const float *src, int N, int P)
{
    stage<float, kNM, kPM>(dst, kLP, src, (size_t)P, N, P);
}

// the same state transposed: dst[p * kLN + n], zero past N, P.  Consecutive
// threads take consecutive n, so the shared-memory stores do not conflict.
__device__ __forceinline__ void stage_state_t(float *dst, const float *src, int N, int P)
{
    for (int i = threadIdx.x; i < kNM * kPM; i += kThreads) {
        const int n = i % kNM, col = i / kNM;
        dst[col * kLN + n] = (n < N && col < P) ? src[(size_t)n * P + col] : 0.f;
    }
}

// 3. Every gradient of one chunk.  Grid (nc, B*H).
template <typename T>
__global__ void __launch_bounds__(kThreads) ssd_bwd_grad_kernel(ChunkBwdParams p)
{
    extern __shared__ __align__(16) float smem[];
    float *xs = smem, *dys = xs + kQ * kLP, *Bs = dys + kQ * kLP, *Cs = Bs + kQ * kLN;
    float *Mt = Cs + kQ * kLN, *A2 = Mt + kQ * kLQ, *St = A2 + kQ * kLQ, *StT = St + kNM * kLP;
    float *rowp = StT + kPM * kLN, *colp = rowp + 16 * kQ;
    float *dt_s = colp + 16 * kQ, *z_s = dt_s + kQ, *cs_s = z_s + kQ;
    float *ddir = cs_s + kQ, *vv = ddir + kQ, *uu = vv + kQ, *dcs = uu + kQ;
    float *red = dcs + kQ;   // [32]: per-warp sums (fixed order: deterministic)
    const int H = p.H, P = p.P, N = p.N, Gg = p.G, nc = p.nc;
    const long long bh = blockIdx.y, b = bh / H;
    const int h = (int)(bh - b * H), g = h / (H / Gg), c = blockIdx.x;
    const long long t0 = (long long)c * kQ;
    const int nq = (int)min((long long)kQ, p.L - t0);
    const float a = -expf(p.A_log[h]), Dh = p.D[h];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4, lane = tid & 31, warp = tid >> 5;
    const size_t NP = (size_t)N * P;
    const float *Gout = p.R + ((size_t)bh * nc + c) * NP;
    const float *hin = p.S + ((size_t)bh * (nc + 1) + c) * NP, *hlast = hin + NP;

    // every global load of the chunk in flight together, then the stores
    const size_t rowx = (size_t)(b * p.L + t0) * H + h, rowb = (size_t)(b * p.L + t0) * Gg + g;
    const bool pv = P % 4 == 0;   // 16-byte rows of the states
    RowTile<T, kQ, kPM> tX, tdy;
    RowTile<T, kQ, kNM> tB, tC;
    StateTile sg, sh;
    tX.load(static_cast<const T *>(p.x) + rowx * P, (size_t)H * P, nq, P);
    tdy.load(static_cast<const T *>(p.dy) + rowx * P, (size_t)H * P, nq, P);
    tB.load(static_cast<const T *>(p.B) + rowb * N, (size_t)Gg * N, nq, N);
    tC.load(static_cast<const T *>(p.C) + rowb * N, (size_t)Gg * N, nq, N);
    if (pv) {
        sg.load(Gout, N, P);
        sh.load(hlast, N, P);
    }
    chunk_decays(p, b, h, t0, nq, a, dt_s, z_s, cs_s);
    tX.store(xs, kLP);
    tdy.store(dys, kLP);
    tB.store(Bs, kLN);
    tC.store(Cs, kLN);
    float gh = 0.f;   // <G_out, h_last>, this thread's share
    if (pv) {
        sg.store(St);
        sg.store_t(StT);
#pragma unroll
        for (int it = 0; it < StateTile::IT; ++it)
            gh = fmaf(sg.v[it].x, sh.v[it].x,
                      fmaf(sg.v[it].y, sh.v[it].y, fmaf(sg.v[it].z, sh.v[it].z, fmaf(sg.v[it].w, sh.v[it].w, gh))));
    } else {
        stage_state(St, Gout, N, P);
        stage_state_t(StT, Gout, N, P);
        for (size_t e = tid; e < NP; e += kThreads)
            gh = fmaf(Gout[e], hlast[e], gh);
    }
    gh = warp_sum(gh);
    if (lane == 0)
        red[warp] = gh;
    __syncthreads();
    const float cs_last = cs_s[kQ - 1];
    float dd = 0.f;   // sum dy . x, this thread's share
    for (int i = tid; i < kQ * kPM; i += kThreads)
        dd = fmaf(dys[(i / kPM) * kLP + i % kPM], xs[(i / kPM) * kLP + i % kPM], dd);
    dd = warp_sum(dd);
    if (lane == 0)
        red[8 + warp] = dd;

    // CB = C B^T, DX = dy x^T; Mt = E CB, A2 = E DX; row / column sums of W = Mt DX dt_j.
    // Rows s = ty + 16 i, columns j = tx + 16 jj.
    {
        float cb[4][4], dx[4][4];
        zero(cb);
        zero(dx);
        contract<4, 4, kNM, false, false, false>(cb, Cs, kLN, Bs, kLN);
        contract<4, 4, kPM, false, false, false>(dx, dys, kLP, xs, kLP);
        float rp[4] = {0.f, 0.f, 0.f, 0.f}, cp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int s = ty + 16 * i, jj = tx + 16 * j;
                const float E = (jj <= s && s < nq) ? expf(cs_s[s] - cs_s[jj]) : 0.f;
                const float mt = E * cb[i][j], a2 = E * dx[i][j];
                Mt[s * kLQ + jj] = mt;
                A2[s * kLQ + jj] = a2;
                const float w = mt * dt_s[jj] * dx[i][j];
                rp[i] += w;
                cp[j] += w;
            }
#pragma unroll
        for (int i = 0; i < 4; ++i)
            rowp[tx * kQ + ty + 16 * i] = rp[i];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            colp[ty * kQ + tx + 16 * j] = cp[j];
    }
    __syncthreads();

    // dx_j = D dy_j + dt_j (Mt^T dy + e^{cs_last - cs_j} B G_out)_j; x . (G^T B) and v.
    // Rows j = 4 ty + i, columns p = 4 tx + q.
    const int c4 = 4 * tx;
    {
        float in[4][4], out[4][4];
        zero(in);
        zero(out);
        contract<4, 4, kQ, true, true, true>(in, Mt, kLQ, dys, kLP, nullptr, 4 * ty);   // Mt[s][j] = 0 for s < j
        contract<4, 4, kNM, false, true, true>(out, Bs, kLN, St, kLP);
        float *dxg = p.dx + rowx * P;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int j = tile_row<4, true>(i);
            const float eo = expf(cs_last - cs_s[j]), dtj = dt_s[j];
            const float4 x4 = *reinterpret_cast<const float4 *>(xs + j * kLP + c4);
            const float4 y4 = *reinterpret_cast<const float4 *>(dys + j * kLP + c4);
            const float xv[4] = {x4.x, x4.y, x4.z, x4.w}, yv[4] = {y4.x, y4.y, y4.z, y4.w};
            float dsum = 0.f, vsum = 0.f, o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float gx = fmaf(eo, out[i][q], in[i][q]);
                dsum = fmaf(xv[q], gx, dsum);
                vsum = fmaf(xv[q], out[i][q], vsum);
                o[q] = fmaf(Dh, yv[q], dtj * gx);
            }
            if (j < nq)
                store4(dxg + (size_t)j * H * P, c4, P, o);
            dsum = half_warp_sum(dsum);
            vsum = half_warp_sum(vsum);
            if (tx == 0) {
                ddir[j] = dsum;
                vv[j] = dtj * eo * vsum;
            }
        }
    }

    // dB_j = dt_j (A2^T C + e^{cs_last - cs_j} x G_out^T)_j.  Rows j = 4 ty + i,
    // columns n = 4 tx + q and 64 + 4 tx + q.  The loads of h_in are in flight meanwhile.
    if (pv)
        sh.load(hin, N, P);
    {
        float in[4][8], out[4][8];
        zero(in);
        zero(out);
        contract<4, 8, kQ, true, true, true>(in, A2, kLQ, Cs, kLN, nullptr, 4 * ty);   // A2[s][j] = 0 for s < j
        contract<4, 8, kPM, false, true, true>(out, xs, kLP, StT, kLN);
        float *dbg = p.dB_head + rowx * N;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int j = tile_row<4, true>(i);
            const float eo = expf(cs_last - cs_s[j]), dtj = dt_s[j];
            float o0[4], o1[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                o0[q] = dtj * fmaf(eo, out[i][q], in[i][q]);
                o1[q] = dtj * fmaf(eo, out[i][q + 4], in[i][q + 4]);
            }
            if (j < nq) {
                store4(dbg + (size_t)j * H * N, c4, N, o0);
                store4(dbg + (size_t)j * H * N, 64 + c4, N, o1);
            }
        }
    }
    __syncthreads();
    if (pv)
        sh.store_t(StT);
    else
        stage_state_t(StT, hin, N, P);
    __syncthreads();

    // dC_s = (A2 dt) B + e^{cs_s} dy h_in^T; u_s = C_s . (e^{cs_s} h_in dy_s).
    // Rows s = 4 ty + i, columns n = 4 tx + q and 64 + 4 tx + q.
    {
        float in[4][8], out[4][8];
        zero(in);
        zero(out);
        contract<4, 8, kQ, false, true, true>(in, A2, kLQ, Bs, kLN, dt_s, 0, 4 * ty + 4);   // A2[s][j] = 0 for j > s
        contract<4, 8, kPM, false, true, true>(out, dys, kLP, StT, kLN);
        float *dcg = p.dC_head + rowx * N;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int s = tile_row<4, true>(i);
            const float es = expf(cs_s[s]);
            const float4 ca = *reinterpret_cast<const float4 *>(Cs + s * kLN + c4);
            const float4 cb = *reinterpret_cast<const float4 *>(Cs + s * kLN + 64 + c4);
            const float cv[8] = {ca.x, ca.y, ca.z, ca.w, cb.x, cb.y, cb.z, cb.w};
            float usum = 0.f, o0[4], o1[4];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float inter = es * out[i][q];
                usum = fmaf(cv[q], inter, usum);
                if (q < 4)
                    o0[q] = in[i][q] + inter;
                else
                    o1[q - 4] = in[i][q] + inter;
            }
            if (s < nq) {
                store4(dcg + (size_t)s * H * N, c4, N, o0);
                store4(dcg + (size_t)s * H * N, 64 + c4, N, o1);
            }
            usum = half_warp_sum(usum);
            if (tx == 0)
                uu[s] = usum;
        }
    }
    __syncthreads();

    // dL/dcs_k, its suffix sums d log dA_j, ddt_raw and the chunk's per-head partials
    if (tid < kQ) {
        float r = 0.f, cl = 0.f;
        for (int q = 0; q < 16; ++q) {
            r += rowp[q * kQ + tid];
            cl += colp[q * kQ + tid];
        }
        dcs[tid] = r - cl + uu[tid] - vv[tid];
    }
    __syncthreads();
    if (warp == 0) {   // suffix sums over the 64 steps, two per lane; <G_out, h_last> enters at the last
        float ghs = 0.f;
        for (int q = 0; q < 8; ++q)
            ghs += red[q];
        const float v0 = dcs[2 * lane], v1 = dcs[2 * lane + 1];
        float s = v0 + v1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float t = __shfl_down_sync(0xffffffffu, s, o);
            if (lane + o < 32)
                s += t;
        }
        float after = __shfl_down_sync(0xffffffffu, s, 1);   // sum over the lanes past this one
        if (lane == 31)
            after = 0.f;
        const float s1 = ghs + after + v1;
        dcs[2 * lane + 1] = s1;
        dcs[2 * lane] = s1 + v0;
    }
    __syncthreads();
    if (warp < 2) {
        float cda = 0.f, cdb = 0.f;
        if (tid < nq) {
            const float ddt = fmaf(a, dcs[tid], ddir[tid]);
            cdb = ddt / (1.f + expf(-z_s[tid]));
            p.ddt_raw[(size_t)(b * p.L + t0 + tid) * H + h] = cdb;
            cda = dt_s[tid] * dcs[tid];
        }
        cda = warp_sum(cda);
        cdb = warp_sum(cdb);
        if (lane == 0) {
            red[16 + warp] = cda;
            red[18 + warp] = cdb;
        }
    }
    __syncthreads();
    if (tid == 0) {
        const float sa = red[16] + red[17], sb = red[18] + red[19];
        float sd = 0.f;
        for (int q = 0; q < 8; ++q)
            sd += red[8 + q];
        const size_t BHC = (size_t)gridDim.y * nc, i = (size_t)bh * nc + c;
        p.part[i] = a * sa;
        p.part[BHC + i] = sb;
        p.part[2 * BHC + i] = sd;
    }
}

constexpr size_t kLocalSmem = (size_t)(2 * kQ * kLN + 2 * kQ * kLP + 5 * kQ) * sizeof(float);
constexpr size_t kGradSmem =
    (size_t)(2 * kQ * kLP + 2 * kQ * kLN + 2 * kQ * kLQ + kNM * kLP + kPM * kLN + 32 * kQ + 7 * kQ + 32) * sizeof(float);
static_assert(kGradSmem <= 227 * 1024, "grad kernel shared memory");

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

}  // namespace

bool bwd_chunk_supported(const BwdArgs &a)
{
    return a.headdim >= 1 && a.headdim <= kPM && a.dstate >= 1 && a.dstate <= kNM &&
           a.batch * (long long)a.nheads <= 65535 && a.seqlen < (1LL << 31) &&
           (a.seqlen + kQ - 1) / kQ <= 0x7FFFFFFFLL;
}

size_t bwd_chunk_workspace_bytes(const BwdArgs &a)
{
    const size_t BH = (size_t)a.batch * a.nheads, NP = (size_t)a.headdim * a.dstate;
    const size_t nc = (size_t)((a.seqlen + kQ - 1) / kQ);
    const size_t BLHN = (size_t)a.batch * a.seqlen * a.nheads * a.dstate;
    return align256(BH * (nc + 1) * NP * 4) + align256(BH * nc * NP * 4) + align256(BH * nc * 4) +
           2 * align256(BLHN * 4) + align256(3 * BH * nc * 4);
}

cudaError_t bwd_chunk_launch(const BwdArgs &a, void *ws, cudaStream_t st)
{
    SSD_NVTX_RANGE("bwd_chunk_launch");
    if (!bwd_chunk_supported(a))
        return cudaErrorInvalidValue;
    const size_t BH = (size_t)a.batch * a.nheads, NP = (size_t)a.headdim * a.dstate;
    const int nc = (int)((a.seqlen + kQ - 1) / kQ);
    const size_t BLHN = (size_t)a.batch * a.seqlen * a.nheads * a.dstate;
    char *w = static_cast<char *>(ws);
    ChunkBwdParams p;
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
    p.S = reinterpret_cast<float *>(w);
    w += align256(BH * (nc + 1) * NP * 4);
    p.R = reinterpret_cast<float *>(w);
    w += align256(BH * nc * NP * 4);
    p.dec = reinterpret_cast<float *>(w);
    w += align256(BH * nc * 4);
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
    p.nc = nc;
    const dim3 grid((unsigned)nc, (unsigned)BH);
    const bool bf = a.dtype == SSD_DTYPE_BF16;
    // the tensor-core form (ssd_bwd_tc.cu) of the chunk states and of the gradient pass
    // (its tensor maps need 16-byte aligned bases)
    auto aligned16 = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
    const bool tc = bf && !a.fp32_form && bwd_tc_supported(a.dtype, a.headdim, a.dstate) && aligned16(a.x) &&
                    aligned16(a.B) && aligned16(a.C) && aligned16(a.dy) && aligned16(a.dx);
    cudaError_t e;
    if (bf) {
        e = cudaFuncSetAttribute(ssd_bwd_local_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kLocalSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(ssd_bwd_grad_kernel<__nv_bfloat16>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGradSmem);
    } else {
        e = cudaFuncSetAttribute(ssd_bwd_local_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kLocalSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(ssd_bwd_grad_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kGradSmem);
    }
    if (e != cudaSuccess)
        return e;
    // the tensor-core form's chunk states: one launch walking each (b, h) through its
    // chunks (the state in TMEM) when 2 B H CTAs fill the SMs or the walk is short,
    // else every chunk at once and then the chains
    int sms = 0;
    if (tc) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return cudaErrorInvalidValue;
    }
    const bool walk = tc && !a.split_states && (2 * (long long)BH >= sms || nc <= 8);
    if (walk) {
        BwdTcChainArgs t;
        t.x = a.x;
        t.B = a.B;
        t.C = a.C;
        t.dy = a.dy;
        t.dt_raw = a.dt_raw;
        t.dt_bias = a.dt_bias;
        t.A_log = a.A_log;
        t.init_state = a.init_state;
        t.d_final = a.d_final;
        t.S = p.S;
        t.R = p.R;
        t.d_init = a.d_init;
        t.batch = a.batch;
        t.seqlen = a.seqlen;
        t.nheads = a.nheads;
        t.ngroups = a.ngroups;
        t.nc = nc;
        e = bwd_tc_chain_launch(t, st);
        if (e != cudaSuccess)
            return e;
    } else if (tc) {
        BwdTcLocalArgs t;
        t.x = a.x;
        t.B = a.B;
        t.C = a.C;
        t.dy = a.dy;
        t.dt_raw = a.dt_raw;
        t.dt_bias = a.dt_bias;
        t.A_log = a.A_log;
        t.S = p.S;
        t.R = p.R;
        t.dec = p.dec;
        t.batch = a.batch;
        t.seqlen = a.seqlen;
        t.nheads = a.nheads;
        t.ngroups = a.ngroups;
        t.nc = nc;
        e = bwd_tc_local_launch(t, st);
        if (e != cudaSuccess)
            return e;
    } else if (bf) {
        ssd_bwd_local_kernel<__nv_bfloat16><<<grid, kThreads, kLocalSmem, st>>>(p);
    } else {
        ssd_bwd_local_kernel<float><<<grid, kThreads, kLocalSmem, st>>>(p);
    }
    const bool tr = a.headdim == kPM && a.dstate % 16 == 0 && aligned16(a.init_state) && aligned16(a.d_final) &&
                    aligned16(a.d_init);
    if (walk)
        ;   // the walk has linked the chunks
    else if (tr)
        ssd_bwd_pass_kernel<kVec, true><<<dim3((unsigned)(NP / kVec / kThreads), (unsigned)BH, 2), kThreads, 0, st>>>(p);
    else if (NP % kVec == 0)
        ssd_bwd_pass_kernel<kVec, false><<<dim3((unsigned)((NP / kVec + kThreads - 1) / kThreads), (unsigned)BH, 2),
                                           kThreads, 0, st>>>(p);
    else
        ssd_bwd_pass_kernel<1, false><<<dim3((unsigned)((NP + kThreads - 1) / kThreads), (unsigned)BH, 2), kThreads, 0,
                                        st>>>(p);
    if (tc) {
        // the gradient pass on the tensor cores
        BwdTcArgs t;
        t.x = a.x;
        t.B = a.B;
        t.C = a.C;
        t.dy = a.dy;
        t.dt_raw = a.dt_raw;
        t.dt_bias = a.dt_bias;
        t.A_log = a.A_log;
        t.D = a.D;
        t.S = p.S;
        t.R = p.R;
        t.dx = a.dx;
        t.ddt_raw = a.ddt_raw;
        t.dB_head = p.dB_head;
        t.dC_head = p.dC_head;
        t.part = p.part;
        t.batch = a.batch;
        t.seqlen = a.seqlen;
        t.nheads = a.nheads;
        t.ngroups = a.ngroups;
        t.nc = nc;
        e = bwd_tc_grad_launch(t, st);
    } else if (bf) {
        ssd_bwd_grad_kernel<__nv_bfloat16><<<grid, kThreads, kGradSmem, st>>>(p);
    } else {
        ssd_bwd_grad_kernel<float><<<grid, kThreads, kGradSmem, st>>>(p);
    }
    if (e == cudaSuccess)
        e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    note_launches(walk ? 2 : 3);
    return bwd_finish_launch(a, p.dB_head, p.dC_head, p.part, nc, st);
}

}  // namespace ssd
