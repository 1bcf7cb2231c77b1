// ssd_chunk.cu -- chunked SSD forward scan on the sm_103a tensor cores.
//
// One persistent kernel evaluates the whole scan.  Work unit = (chunk c,
// batch row b, pair of heads h0, h0+1 of one group).  Units are ordered
// chunk-major, so the CTAs running at any moment work on the same chunk of
// many head pairs (the group's B/C tiles are shared through L2), and the unit
// that needs the state left by chunk c-1 of its chain was scheduled about one
// round of the grid earlier.
//
// Inside a unit the chunk is walked in sub-chunks of T = 128 steps.  For a
// sub-chunk with carried-in state P (N x P per head) and the sub-chunk-local
// inclusive cumulative sum cs_t = sum_{k<=t} dt_k A:
//
//   S      = C B^T                                   (T x T, shared by both heads)
//   M[t,s] = S[t,s] exp(cs_t - cs_s) dt_s  (s <= t),  M[t,t] += D
//   y_t    = (M x)_t + exp(cs_t) (C P)_t
//   P     <- exp(cs_{T-1}) P + B^T (w o x),   w_s = exp(cs_{T-1} - cs_s) dt_s
//
// This is the quadratic ("dual") form inside the sub-chunk and the linear
// recurrence between sub-chunks; chunk boundaries are where the state is
// handed from one unit to the next through global memory.  Source: the SSD
// module of @seanhogg/builderforce-memory-engine 2026.6.18 (chunked evaluation
// with a carried state) and the chunked-scan pipeline of mamba-rs 0.2.1
// mamba3_siso/gpu/mamba3_gpu.rs (decay cumsum, chunk state, state passing,
// chunk scan), applied to the Mamba-2 recurrence.
//
// Roles (10 warps):
//   warps 0-7  "math": cumulative sums and decay factors, the masked decay
//              matrix M (written to tensor memory as a bf16 MMA operand), the
//              w-scaling of x, the state rescale, the output epilogue and the
//              state handoff.
//   warp 8     TMA producer: B/C tiles (2 stages) and x tiles (2 stages).
//   warp 9     tcgen05 MMA issuer (one lane) and TMEM owner.
// Tensor memory (512 columns x 128 lanes, fp32):
//   [  0,128)  Y_diag = M x            lanes t, columns (head, p)
//   [128,256)  S = C B^T, then Y_off = C P   (lanes t)
//   [256,384)  M for both heads (bf16 pairs, MMA A operand)
//   [384,512)  P, the carried state, fp32    lanes n, columns (head, p)
// Every wait is bounded (about 2 s); on expiry the kernel records
// SSD_ERR_TIMEOUT, stops issuing work, drains its own copies and MMAs, frees
// tensor memory and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <chrono>

#include "ptx.cuh"
#include "ssd_internal.h"
#include "tmap.h"

namespace ssd {

__device__ unsigned int g_chunk_error;

namespace {

using namespace ssd::ptx;

constexpr int kT = 128;          // sub-chunk length (MMA M)
constexpr int kP = 64;           // head dimension
constexpr int kN = 128;          // state size
constexpr int kMathWarps = 8;
constexpr int kMathThreads = kMathWarps * 32;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 320;

constexpr uint32_t kTileBytes = 16384;              // 128 rows x 128 bytes
constexpr uint32_t kBCStageBytes = 4 * kTileBytes;  // C lo/hi, B lo/hi
constexpr uint32_t kXStageBytes = 2 * kTileBytes;   // x of two heads

// dynamic shared memory layout (offsets from a 1024-aligned base)
constexpr uint32_t kOffBC = 0;
constexpr uint32_t kOffX = kOffBC + 2 * kBCStageBytes;
constexpr uint32_t kOffSmall = kOffX + 2 * kXStageBytes;
constexpr uint32_t kSmallFloats = 2 /*parity*/ * 2 /*head*/ * kT * 3 /*cs2, dt, colf*/;
constexpr uint32_t kOffWsum = kOffSmall + kSmallFloats * 4;
constexpr uint32_t kOffBars = kOffWsum + 64;
constexpr int kNumBars = 20;
constexpr uint32_t kOffTmemHolder = kOffBars + kNumBars * 8;
constexpr uint32_t kSmemBytes = kOffTmemHolder + 16 + 1024;  // + alignment slack

// tensor memory columns
constexpr uint32_t kColYd = 0, kColSY = 128, kColM = 256, kColP = 384;

// barrier indices
enum {
    BAR_BC_FULL = 0,   // 2
    BAR_BC_EMPTY = 2,  // 2
    BAR_X_FULL = 4,    // 2
    BAR_X_EMPTY = 6,   // 2
    BAR_S_DONE = 8,
    BAR_M_READY,
    BAR_YD_DONE,
    BAR_XS_READY,
    BAR_YOFF_DONE,
    BAR_STATE_DONE,
    BAR_PB_READY,
    BAR_EPI_DONE,
    BAR_DRAIN,
    BAR_MSYNC,   // math-warp group barrier (bounded, unlike bar.sync)
};

struct ChunkParams {
    const float *dt_raw;
    const float *dt_bias;
    const float *A_log;
    const float *D;
    const float *init_state;          // may be null
    __nv_bfloat16 *y;
    float *slot;                      // [B, H, P, N] fp32: handoff states, final state
    unsigned long long *flags;        // [nunits]
    unsigned long long *abort_word;
    unsigned long long epoch;
    unsigned long long timeout_ns;
    long long L;
    long long nunits;
    int H, Q, nchunks, nhp, nchains, hpg;
};

struct Maps {
    CUtensorMap x, B, C;
};

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_u64(unsigned long long *p, unsigned long long v)
{
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void st_global_cs_v4(void *ptr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.global.cs.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(ptr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

__device__ void raise_timeout(const ChunkParams &p)
{
    atomicCAS(&g_chunk_error, 0u, (unsigned)SSD_ERR_TIMEOUT);
    atomicExch(p.abort_word, p.epoch);
}

__device__ __forceinline__ bool aborted(const ChunkParams &p)
{
    return *reinterpret_cast<volatile unsigned long long *>(p.abort_word) == p.epoch;
}

// Bounded wait for the phase of `bar` with the given parity.
__device__ bool wait_bar(uint64_t *bar, uint32_t parity, const ChunkParams &p)
{
    if (mbar_test(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_test(bar, parity))
            return true;
        if ((it & 255u) == 0) {
            if (aborted(p))
                return false;
            if (globaltimer_ns() - t0 > p.timeout_ns) {
                raise_timeout(p);
                return false;
            }
        }
    }
}

// Group barrier of the math warps on an mbarrier, so that it is bounded too.
__device__ __forceinline__ bool math_sync(uint64_t *bar, uint32_t &phase, const ChunkParams &p)
{
    mbar_arrive(bar);
    const bool ok = wait_bar(bar, phase, p);
    phase ^= 1u;
    return ok;
}

// Bounded wait until flag == epoch (the predecessor unit published its state).
__device__ bool wait_flag(const unsigned long long *flag, const ChunkParams &p)
{
    if (ld_acquire_u64(flag) == p.epoch)
        return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        __nanosleep(64);
        if (ld_acquire_u64(flag) == p.epoch)
            return true;
        if ((it & 63u) == 0) {
            if (aborted(p))
                return false;
            if (globaltimer_ns() - t0 > p.timeout_ns) {
                raise_timeout(p);
                return false;
            }
        }
    }
}

struct Unit {
    int c, b, h0, g, nsub, clen;
    long long cstart;
};

__device__ __forceinline__ Unit decode_unit(long long u, const ChunkParams &p)
{
    Unit w;
    w.c = (int)(u / p.nchains);
    const int chain = (int)(u - (long long)w.c * p.nchains);
    w.b = chain / p.nhp;
    const int hp = chain - w.b * p.nhp;
    w.h0 = 2 * hp;
    w.g = w.h0 / p.hpg;
    w.cstart = (long long)w.c * p.Q;
    w.clen = (int)min((long long)p.Q, p.L - w.cstart);
    w.nsub = (w.clen + kT - 1) / kT;
    return w;
}

__device__ __forceinline__ float softplus_f32(float z)
{
    return fmaxf(z, 0.f) + log1pf(expf(-fabsf(z)));
}

// byte offset of 16-byte chunk `c` of row `r` in a 128-byte-swizzled tile
__device__ __forceinline__ uint32_t sw128(uint32_t r, uint32_t c)
{
    return r * 128u + ((c ^ (r & 7u)) << 4);
}

__global__ void __launch_bounds__(kThreads, 1)
    ssd_chunk_fused_kernel(const __grid_constant__ Maps maps, const ChunkParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBars);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + kOffTmemHolder);
    float *small = reinterpret_cast<float *>(smem + kOffSmall);
    float *wsum = reinterpret_cast<float *>(smem + kOffWsum);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[BAR_BC_FULL + i], 1);
            mbar_init(&bars[BAR_BC_EMPTY + i], 1);
            mbar_init(&bars[BAR_X_FULL + i], 1);
            mbar_init(&bars[BAR_X_EMPTY + i], 1);
        }
        mbar_init(&bars[BAR_S_DONE], 1);
        mbar_init(&bars[BAR_M_READY], kMathThreads);
        mbar_init(&bars[BAR_YD_DONE], 1);
        mbar_init(&bars[BAR_XS_READY], kMathThreads);
        mbar_init(&bars[BAR_YOFF_DONE], 1);
        mbar_init(&bars[BAR_STATE_DONE], 1);
        mbar_init(&bars[BAR_PB_READY], kMathThreads);
        mbar_init(&bars[BAR_EPI_DONE], kMathThreads);
        mbar_init(&bars[BAR_DRAIN], 1);
        mbar_init(&bars[BAR_MSYNC], kMathThreads);
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_holder, 512);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        prefetch_tmap(&maps.x);
        prefetch_tmap(&maps.B);
        prefetch_tmap(&maps.C);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ TMA
        if (lane == 0) {
            const uint64_t pol_stream = policy_evict_first();
            const uint64_t pol_keep = policy_evict_last();
            uint32_t j = 0;
            bool ok = true;
            int last_bc[2] = {-1, -1}, last_x[2] = {-1, -1};  // last sub-chunk loaded per stage
            for (long long u = blockIdx.x; ok && u < p.nunits; u += gridDim.x) {
                const Unit w = decode_unit(u, p);
                for (int k = 0; k < w.nsub; ++k, ++j) {
                    const int s = j & 1;
                    const int t0 = (int)(w.cstart + (long long)k * kT);
                    if (j >= 2 && !(ok = wait_bar(&bars[BAR_BC_EMPTY + s], ((j >> 1) + 1) & 1, p)))
                        break;
                    uint8_t *bc = smem + kOffBC + s * kBCStageBytes;
                    mbar_arrive_expect_tx(&bars[BAR_BC_FULL + s], kBCStageBytes);
                    tma_load_3d(bc, &maps.C, &bars[BAR_BC_FULL + s], w.g * kN, t0, w.b, pol_keep);
                    tma_load_3d(bc + kTileBytes, &maps.C, &bars[BAR_BC_FULL + s], w.g * kN + 64, t0, w.b, pol_keep);
                    tma_load_3d(bc + 2 * kTileBytes, &maps.B, &bars[BAR_BC_FULL + s], w.g * kN, t0, w.b, pol_keep);
                    tma_load_3d(bc + 3 * kTileBytes, &maps.B, &bars[BAR_BC_FULL + s], w.g * kN + 64, t0, w.b, pol_keep);
                    last_bc[s] = (int)j;
                    if (j >= 1 && !(ok = wait_bar(&bars[BAR_X_EMPTY + s], ((j - 1) >> 1) & 1, p)))
                        break;
                    uint8_t *xs = smem + kOffX + s * kXStageBytes;
                    mbar_arrive_expect_tx(&bars[BAR_X_FULL + s], kXStageBytes);
                    tma_load_3d(xs, &maps.x, &bars[BAR_X_FULL + s], w.h0 * kP, t0, w.b, pol_stream);
                    tma_load_3d(xs + kTileBytes, &maps.x, &bars[BAR_X_FULL + s], (w.h0 + 1) * kP, t0, w.b, pol_stream);
                    last_x[s] = (int)j;
                }
            }
            if (!ok) {
                // every load issued by this thread must land before the CTA exits
                const uint64_t t0 = globaltimer_ns();
                for (int st = 0; st < 2; ++st) {
                    if (last_bc[st] >= 0)
                        while (!mbar_test(&bars[BAR_BC_FULL + st], (last_bc[st] >> 1) & 1) &&
                               globaltimer_ns() - t0 < p.timeout_ns) {
                        }
                    if (last_x[st] >= 0)
                        while (!mbar_test(&bars[BAR_X_FULL + st], (last_x[st] >> 1) & 1) &&
                               globaltimer_ns() - t0 < p.timeout_ns) {
                        }
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            const uint32_t id_S = idesc_bf16_f32(128, 128, 0, 0);      // C (K-major) x B (K-major)
            const uint32_t id_Yd = idesc_bf16_f32(128, 64, 0, 1);      // M (TMEM) x x (MN-major)
            const uint32_t id_Yoff = idesc_bf16_f32(128, 128, 0, 1);   // C (K-major) x P (MN-major)
            const uint32_t id_St = idesc_bf16_f32(128, 128, 1, 1);     // B^T (MN-major) x wx (MN-major)
            uint32_t j = 0;
            bool ok = true;
            for (long long u = blockIdx.x; ok && u < p.nunits; u += gridDim.x) {
                const Unit w = decode_unit(u, p);
                for (int k = 0; k < w.nsub; ++k, ++j) {
                    const int s = j & 1;
                    const uint32_t par = j & 1;
                    const uint32_t bc = smem_u32(smem + kOffBC + s * kBCStageBytes);
                    const uint32_t cA = bc, bB = bc + 2 * kTileBytes;
                    const uint32_t xs = smem_u32(smem + kOffX + s * kXStageBytes);
                    const uint32_t pb = smem_u32(smem + kOffX + (s ^ 1) * kXStageBytes);
                    // 1. S = C B^T
                    if (!(ok = wait_bar(&bars[BAR_BC_FULL + s], (j >> 1) & 1, p)))
                        break;
                    if (j >= 1 && !(ok = wait_bar(&bars[BAR_EPI_DONE], (j - 1) & 1, p)))
                        break;
                    tc_fence_after();
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t ko = (kk >> 2) * kTileBytes + (kk & 3) * 32;
                        mma_ss(tmem + kColSY, sdesc_sw128(cA + ko, 16, 1024), sdesc_sw128(bB + ko, 16, 1024),
                               id_S, kk > 0);
                    }
                    mma_commit(&bars[BAR_S_DONE]);
                    // 2. Y_diag[h] = M[h] x[h]
                    if (!(ok = wait_bar(&bars[BAR_X_FULL + s], (j >> 1) & 1, p)))
                        break;
                    if (!(ok = wait_bar(&bars[BAR_M_READY], par, p)))
                        break;
                    tc_fence_after();
                    for (int h = 0; h < 2; ++h)
                        for (int kk = 0; kk < 8; ++kk)
                            mma_ts(tmem + kColYd + 64 * h, tmem + kColM + 64 * h + 8 * kk,
                                   sdesc_sw128(xs + h * kTileBytes + kk * 2048, kTileBytes, 1024), id_Yd, kk > 0);
                    mma_commit(&bars[BAR_YD_DONE]);
                    // 3. Y_off = C P   (P as bf16 in the other x stage)
                    if (!(ok = wait_bar(&bars[BAR_PB_READY], par, p)))
                        break;
                    tc_fence_after();
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t ko = (kk >> 2) * kTileBytes + (kk & 3) * 32;
                        mma_ss(tmem + kColSY, sdesc_sw128(cA + ko, 16, 1024),
                               sdesc_sw128(pb + kk * 2048, kTileBytes, 1024), id_Yoff, kk > 0);
                    }
                    mma_commit(&bars[BAR_YOFF_DONE]);
                    mma_commit(&bars[BAR_X_EMPTY + (s ^ 1)]);
                    // 4. P += B^T (w o x)   (P already rescaled by the math warps)
                    if (!(ok = wait_bar(&bars[BAR_XS_READY], par, p)))
                        break;
                    tc_fence_after();
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ss(tmem + kColP, sdesc_sw128(bB + kk * 2048, kTileBytes, 1024),
                               sdesc_sw128(xs + kk * 2048, kTileBytes, 1024), id_St, 1);
                    mma_commit(&bars[BAR_STATE_DONE]);
                    mma_commit(&bars[BAR_BC_EMPTY + s]);
                }
            }
            // make sure no MMA is in flight before tensor memory is released
            mma_commit(&bars[BAR_DRAIN]);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_test(&bars[BAR_DRAIN], 0) && globaltimer_ns() - t0 < p.timeout_ns) {
            }
        }
    } else {
        // ------------------------------------------------------------ math
        const int q = warp & 3;        // TMEM lane quarter
        const int hf = warp >> 2;      // head of this thread for per-head work; column half for M
        const int r = q * 32 + lane;   // row: token t / state row n
        const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
        const float LOG2E = 1.4426950408889634f;
        uint32_t j = 0, msync = 0;
        bool ok = true;
        for (long long u = blockIdx.x; ok && u < p.nunits; u += gridDim.x) {
            const Unit w = decode_unit(u, p);
            const int hh = w.h0 + hf;  // this thread's head
            const float A2 = -expf(p.A_log[hh]) * LOG2E;
            const float bias = p.dt_bias[hh];
            const float Dh0 = p.D[w.h0], Dh1 = p.D[w.h0 + 1];
            // state slot of (b, hh): [P][N], this thread's row n = r
            const size_t slot_base = ((size_t)w.b * p.H + hh) * (size_t)(kP * kN) + r;
            for (int k = 0; k < w.nsub; ++k, ++j) {
                const int s = j & 1;
                const uint32_t par = j & 1;
                const long long t0 = w.cstart + (long long)k * kT;
                const int valid = min(kT, w.clen - k * kT);
                float *cs2 = small + ((s * 2) * kT) * 3;          // [2 heads][T]
                float *dtv = cs2 + 2 * kT;
                float *colf = dtv + 2 * kT;
                // ---- 0a. unit start: carried-in state into TMEM (fp32) and bf16 operand
                if (k == 0) {
                    if (w.c > 0) {
                        if (threadIdx.x == 0 && !(ok = wait_flag(p.flags + (u - p.nchains), p)))
                            break;
                        if (!(ok = math_sync(&bars[BAR_MSYNC], msync, p)))
                            break;
                    }
                    uint32_t v[32];
                    uint8_t *pb = smem + kOffX + (s ^ 1) * kXStageBytes + hf * kTileBytes;
                    for (int half = 0; half < 2; ++half) {
                        for (int i = 0; i < 32; ++i) {
                            const size_t off = slot_base + (size_t)(half * 32 + i) * kN;
                            float val = 0.f;
                            if (w.c > 0)
                                val = __ldcg(p.slot + off);
                            else if (p.init_state)
                                val = __ldg(p.init_state + off);
                            v[i] = __float_as_uint(val);
                        }
                        tmem_st32(tmem + lane_addr + kColP + hf * 64 + half * 32, v);
                        for (int c8 = 0; c8 < 4; ++c8) {
                            uint4 o;
                            o.x = pack_bf16x2(__uint_as_float(v[c8 * 8 + 0]), __uint_as_float(v[c8 * 8 + 1]));
                            o.y = pack_bf16x2(__uint_as_float(v[c8 * 8 + 2]), __uint_as_float(v[c8 * 8 + 3]));
                            o.z = pack_bf16x2(__uint_as_float(v[c8 * 8 + 4]), __uint_as_float(v[c8 * 8 + 5]));
                            o.w = pack_bf16x2(__uint_as_float(v[c8 * 8 + 6]), __uint_as_float(v[c8 * 8 + 7]));
                            *reinterpret_cast<uint4 *>(pb + sw128(r, half * 4 + c8)) = o;
                        }
                    }
                    tmem_wait_st();
                    fence_proxy_async_smem();
                    tc_fence_before();
                    mbar_arrive(&bars[BAR_PB_READY]);
                }
                // ---- 0b. dt, sub-chunk-local cumulative sum of dt*A (base 2), decay factors
                float dt = 0.f;
                if (r < valid)
                    dt = softplus_f32(p.dt_raw[((size_t)w.b * p.L + t0 + r) * p.H + hh] + bias);
                float l = dt * A2;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float nb = __shfl_up_sync(0xffffffffu, l, o);
                    if (lane >= o)
                        l += nb;
                }
                if (lane == 31)
                    wsum[hf * 4 + q] = l;
                if (!(ok = math_sync(&bars[BAR_MSYNC], msync, p)))
                    break;
                for (int qq = 0; qq < q; ++qq)
                    l += wsum[hf * 4 + qq];
                cs2[hf * kT + r] = l;
                dtv[hf * kT + r] = dt;
                if (!(ok = math_sync(&bars[BAR_MSYNC], msync, p)))
                    break;
                colf[hf * kT + r] = ex2_approx(cs2[hf * kT + (r | 31)] - l) * dt;
                const float cs_last = cs2[hf * kT + kT - 1];
                const float ecs = ex2_approx(l);                  // exp(cs_t), for C P
                const float wsc = ex2_approx(cs_last - l) * dt;   // state input weight
                const float dtot = ex2_approx(cs_last);           // state decay over the sub-chunk
                if (!(ok = math_sync(&bars[BAR_MSYNC], msync, p)))
                    break;
                // ---- 1. masked decay matrix M (both heads) from S
                if (!(ok = wait_bar(&bars[BAR_S_DONE], par, p)))
                    break;
                tc_fence_after();
                {
                    uint32_t m0[32], m1[32];
                    const int rb = r >> 5;
                    for (int jb = 0; jb < 2; ++jb) {
                        const int J = hf * 2 + jb;   // 32-column block of s
                        uint32_t sv[32];
                        tmem_ld32(tmem + lane_addr + kColSY + J * 32, sv);
                        tmem_wait_ld();
                        for (int hh2 = 0; hh2 < 2; ++hh2) {
                            uint32_t *mo = (hh2 == 0 ? m0 : m1) + jb * 16;
                            const float *cs = cs2 + hh2 * kT;
                            const float *dd = dtv + hh2 * kT;
                            const float *cf = colf + hh2 * kT;
                            const float Dh = hh2 == 0 ? Dh0 : Dh1;
                            if (J > rb) {
#pragma unroll
                                for (int i = 0; i < 16; ++i)
                                    mo[i] = 0u;
                            } else if (J == rb) {
                                const float csr = cs[r];
#pragma unroll
                                for (int i = 0; i < 16; ++i) {
                                    const int s0 = J * 32 + 2 * i, s1 = s0 + 1;
                                    float a = 0.f, b2 = 0.f;
                                    if (s0 <= r)
                                        a = __uint_as_float(sv[2 * i]) * ex2_approx(csr - cs[s0]) * dd[s0];
                                    if (s1 <= r)
                                        b2 = __uint_as_float(sv[2 * i + 1]) * ex2_approx(csr - cs[s1]) * dd[s1];
                                    if (s0 == r)
                                        a += Dh;
                                    if (s1 == r)
                                        b2 += Dh;
                                    mo[i] = pack_bf16x2(a, b2);
                                }
                            } else {
                                const float rf = ex2_approx(cs[r] - cs[J * 32 + 31]);
#pragma unroll
                                for (int i = 0; i < 16; ++i) {
                                    const int s0 = J * 32 + 2 * i;
                                    mo[i] = pack_bf16x2(__uint_as_float(sv[2 * i]) * rf * cf[s0],
                                                        __uint_as_float(sv[2 * i + 1]) * rf * cf[s0 + 1]);
                                }
                            }
                        }
                    }
                    tmem_st32(tmem + lane_addr + kColM + 0 * 64 + hf * 32, m0);
                    tmem_st32(tmem + lane_addr + kColM + 1 * 64 + hf * 32, m1);
                    tmem_wait_st();
                }
                tc_fence_before();
                mbar_arrive(&bars[BAR_M_READY]);
                // ---- 2. x <- w o x in place (row r of head hf), P <- dtot P
                if (!(ok = wait_bar(&bars[BAR_YD_DONE], par, p)))
                    break;
                tc_fence_after();
                {
                    uint8_t *xrow = smem + kOffX + s * kXStageBytes + hf * kTileBytes + r * 128;
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) {
                        uint4 v4 = *reinterpret_cast<uint4 *>(xrow + c8 * 16);
                        v4.x = pack_bf16x2(bf16lo_to_f32(v4.x) * wsc, bf16hi_to_f32(v4.x) * wsc);
                        v4.y = pack_bf16x2(bf16lo_to_f32(v4.y) * wsc, bf16hi_to_f32(v4.y) * wsc);
                        v4.z = pack_bf16x2(bf16lo_to_f32(v4.z) * wsc, bf16hi_to_f32(v4.z) * wsc);
                        v4.w = pack_bf16x2(bf16lo_to_f32(v4.w) * wsc, bf16hi_to_f32(v4.w) * wsc);
                        *reinterpret_cast<uint4 *>(xrow + c8 * 16) = v4;
                    }
                    for (int half = 0; half < 2; ++half) {
                        uint32_t v[32];
                        const uint32_t ta = tmem + lane_addr + kColP + hf * 64 + half * 32;
                        tmem_ld32(ta, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            v[i] = __float_as_uint(__uint_as_float(v[i]) * dtot);
                        tmem_st32(ta, v);
                    }
                    tmem_wait_st();
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&bars[BAR_XS_READY]);
                // ---- 3. y = Y_diag + exp(cs_t) Y_off   (row t = r, head hf)
                if (!(ok = wait_bar(&bars[BAR_YOFF_DONE], par, p)))
                    break;
                tc_fence_after();
                {
                    __nv_bfloat16 *yrow = p.y + (((size_t)w.b * p.L + t0 + r) * p.H + hh) * kP;
                    for (int half = 0; half < 2; ++half) {
                        uint32_t yd[32], yo[32];
                        tmem_ld32(tmem + lane_addr + kColYd + hf * 64 + half * 32, yd);
                        tmem_ld32(tmem + lane_addr + kColSY + hf * 64 + half * 32, yo);
                        tmem_wait_ld();
                        if (r < valid) {
#pragma unroll
                            for (int c8 = 0; c8 < 4; ++c8) {
                                uint32_t o[4];
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const int i = c8 * 8 + 2 * e;
                                    o[e] = pack_bf16x2(fmaf(ecs, __uint_as_float(yo[i]), __uint_as_float(yd[i])),
                                                       fmaf(ecs, __uint_as_float(yo[i + 1]), __uint_as_float(yd[i + 1])));
                                }
                                st_global_cs_v4(yrow + half * 32 + c8 * 8, o[0], o[1], o[2], o[3]);
                            }
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(&bars[BAR_EPI_DONE]);
                // ---- 4. carried state: hand off (end of unit) or bf16 operand for the next sub-chunk
                if (!(ok = wait_bar(&bars[BAR_STATE_DONE], par, p)))
                    break;
                tc_fence_after();
                const bool last = (k == w.nsub - 1);
                if (last) {
                    for (int half = 0; half < 2; ++half) {
                        uint32_t v[32];
                        tmem_ld32(tmem + lane_addr + kColP + hf * 64 + half * 32, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            p.slot[slot_base + (size_t)(half * 32 + i) * kN] = __uint_as_float(v[i]);
                    }
                    tc_fence_before();
                    if (!(ok = math_sync(&bars[BAR_MSYNC], msync, p)))
                        break;
                    if (threadIdx.x == 0 && w.c < p.nchunks - 1) {
                        __threadfence();
                        st_release_u64(p.flags + u, p.epoch);
                    }
                } else {
                    uint8_t *pb = smem + kOffX + s * kXStageBytes + hf * kTileBytes;
                    for (int half = 0; half < 2; ++half) {
                        uint32_t v[32];
                        tmem_ld32(tmem + lane_addr + kColP + hf * 64 + half * 32, v);
                        tmem_wait_ld();
                        for (int c8 = 0; c8 < 4; ++c8) {
                            uint4 o;
                            o.x = pack_bf16x2(__uint_as_float(v[c8 * 8 + 0]), __uint_as_float(v[c8 * 8 + 1]));
                            o.y = pack_bf16x2(__uint_as_float(v[c8 * 8 + 2]), __uint_as_float(v[c8 * 8 + 3]));
                            o.z = pack_bf16x2(__uint_as_float(v[c8 * 8 + 4]), __uint_as_float(v[c8 * 8 + 5]));
                            o.w = pack_bf16x2(__uint_as_float(v[c8 * 8 + 6]), __uint_as_float(v[c8 * 8 + 7]));
                            *reinterpret_cast<uint4 *>(pb + sw128(r, half * 4 + c8)) = o;
                        }
                    }
                    fence_proxy_async_smem();
                    tc_fence_before();
                    mbar_arrive(&bars[BAR_PB_READY]);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp)
        tmem_dealloc(tmem, 512);
}

std::atomic<unsigned long long> g_epoch{0};

unsigned long long next_epoch()
{
    unsigned long long e = g_epoch.fetch_add(1, std::memory_order_relaxed);
    if (e == 0) {
        // first use: start from a value that stale memory is unlikely to hold
        const unsigned long long seed =
            (unsigned long long)std::chrono::steady_clock::now().time_since_epoch().count() *
                0x9E3779B97F4A7C15ull ^
            (unsigned long long)(uintptr_t)&g_epoch;
        unsigned long long expect = 1;
        g_epoch.compare_exchange_strong(expect, seed | 1ull);
        e = g_epoch.fetch_add(1, std::memory_order_relaxed);
    }
    return e == 0 ? next_epoch() : e;
}

struct Geometry {
    long long nchunks, nchains, nunits;
    size_t flags_off, slot_off, total;
};

Geometry geometry(const ScanArgs &a)
{
    Geometry g;
    g.nchunks = (a.seqlen + a.chunk - 1) / a.chunk;
    g.nchains = a.batch * (a.nheads / 2);
    g.nunits = g.nchunks * g.nchains;
    g.flags_off = 256;
    g.slot_off = (g.flags_off + (size_t)g.nunits * 8 + 255) & ~(size_t)255;
    const size_t slot_bytes = a.final_state ? 0 : (size_t)a.batch * a.nheads * kP * kN * 4;
    g.total = g.slot_off + slot_bytes;
    return g;
}

}  // namespace

bool chunk_supported(const ScanArgs &a)
{
    if (a.dtype != SSD_DTYPE_BF16 || a.headdim != kP || a.dstate != kN)
        return false;
    if (a.chunk % 64 != 0 || a.chunk <= 0)
        return false;
    if ((a.nheads / a.ngroups) % 2 != 0)
        return false;
    if (a.batch >= (1LL << 31) || a.seqlen >= (1LL << 31))
        return false;
    return true;
}

size_t chunk_workspace_bytes(const ScanArgs &a) { return geometry(a).total; }

ssd_status_t chunk_launch(const ScanArgs &a, void *workspace, cudaStream_t stream)
{
    const Geometry geo = geometry(a);
    Maps maps;
    const uint64_t HP = (uint64_t)a.nheads * kP, GN = (uint64_t)a.ngroups * kN, L = (uint64_t)a.seqlen;
    if (!make_tmap_bf16_3d(&maps.x, a.x, HP, L, (uint64_t)a.batch, HP * 2, HP * 2 * L, 64, 128) ||
        !make_tmap_bf16_3d(&maps.B, a.B, GN, L, (uint64_t)a.batch, GN * 2, GN * 2 * L, 64, 128) ||
        !make_tmap_bf16_3d(&maps.C, a.C, GN, L, (uint64_t)a.batch, GN * 2, GN * 2 * L, 64, 128))
        return SSD_ERR_CUDA;
    ChunkParams p;
    p.dt_raw = a.dt_raw;
    p.dt_bias = a.dt_bias;
    p.A_log = a.A_log;
    p.D = a.D;
    p.init_state = a.init_state;
    p.y = static_cast<__nv_bfloat16 *>(a.y);
    char *ws = static_cast<char *>(workspace);
    p.abort_word = reinterpret_cast<unsigned long long *>(ws);
    p.flags = reinterpret_cast<unsigned long long *>(ws + geo.flags_off);
    p.slot = a.final_state ? a.final_state : reinterpret_cast<float *>(ws + geo.slot_off);
    p.epoch = next_epoch();
    p.timeout_ns = 2000000000ull;
    p.L = a.seqlen;
    p.nunits = geo.nunits;
    p.H = a.nheads;
    p.Q = a.chunk;
    p.nchunks = (int)geo.nchunks;
    p.nhp = a.nheads / 2;
    p.nchains = (int)geo.nchains;
    p.hpg = a.nheads / a.ngroups;

    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return SSD_ERR_CUDA;
    if (cudaFuncSetAttribute(ssd_chunk_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes) != cudaSuccess)
        return SSD_ERR_CUDA;
    const long long grid = std::min<long long>(sms, geo.nunits);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs co-resident: chunk handoff waits are safe
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, ssd_chunk_fused_kernel, maps, p) != cudaSuccess)
        return SSD_ERR_CUDA;
    note_launches(1);
    return SSD_OK;
}

ssd_status_t chunk_read_device_error(cudaStream_t stream, uint32_t *code)
{
    unsigned int v = 0, zero = 0;
    if (cudaStreamSynchronize(stream) != cudaSuccess)
        return SSD_ERR_CUDA;
    if (cudaMemcpyFromSymbol(&v, g_chunk_error, sizeof(v)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_chunk_error, &zero, sizeof(zero)) != cudaSuccess)
        return SSD_ERR_CUDA;
    *code = v;
    return SSD_OK;
}

}  // namespace ssd
