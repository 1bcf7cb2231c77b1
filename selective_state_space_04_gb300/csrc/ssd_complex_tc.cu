// ssd_complex_tc.cu -- the complex-valued scan with ET discretisation in chunk
// form on the tensor cores, for bf16 inputs with P = 64 and N = 128 (64 complex
// state components, stored as (re, im) pairs along N).
//
// Per batch row b and head h, with A = exp(log|A| + i arg A) = a_r + i a_i and
// dt_t = softplus(dt_raw_t + dt_bias), the recurrence h_t = A_bar_t h_{t-1} +
// B_bar_t x_t^T (A_bar_t = e^{A dt_t}, B_bar_t = f_t B_t, f_t = (A_bar_t - 1) / A)
// unrolled over a chunk of 64 steps with tau_t = sum_{j <= t} dt_j (steps of the
// chunk), H the state entering it and C_t . B_s = sum_k C_t[k] B_s[k]:
//   y_t = Re( sum_{s <= t} e^{A (tau_t - tau_s)} f_s (C_t . B_s) x_s
//             + Lambda_t (C_t . H) ) + D x_t,          Lambda_t = e^{A tau_t}
//   H'  = Lambda_63 H + sum_s g_s B_s x_s^T,            g_s = e^{A (tau_63 - tau_s)} f_s
// (products of A_bar over the steps between, as the recurrence composes them).
// In real products over the interleaved (re, im) index n:
//   S_re = C^ B^T and S_im = C~ B^T, with C^ = (C_r, -C_i) and C~ = (C_i, C_r);
//   M[t][s] = Re(E_ts) S_re - Im(E_ts) S_im, E_ts = e^{A (tau_t - tau_s)} f_s (s <= t);
//   Y = M x + C_L H_bf16, C_L[t] = (Re(Lambda_t C_t[k]), -Im(Lambda_t C_t[k]));
//   H' = rot(Lambda_63) H + B~^T x, B~[s] = (Re(g_s B_s[k]), Im(g_s B_s[k])),
// rot(z) multiplying each complex component of H (the lane pair 2k, 2k+1) by z.
//
// A work item is two batch rows of one head, stacked as the 128 rows of every
// tcgen05 MMA (kind::f16, bf16 operands in shared memory with the 128-byte
// swizzle, fp32 accumulators in TMEM; lane = row), whose chunks are walked
// together with both states in TMEM.  One persistent CTA per SM takes items in
// turn; each step's C and B load once the previous step's S products have read
// theirs, its x once the previous epilogue has, and an item's entering states
// are prefetched into L2 an item ahead.  E is zero across the two rows, so M is
// block diagonal; the products with a row's state are issued once per state
// over all 128 rows, and each row keeps its own one.  M is factored per 16-step
// block (ending at step e) as e^{A (tau_t - tau_e)} . e^{A (tau_e - tau_s)} f_s:
// below a row's diagonal block both factors have modulus at most 1 for decaying
// modes; on it the row factor is at most e^{|a_r| span}, so the factored form
// (masked to s <= t) is taken while that stays far inside fp32, and
// e^{A (tau_t - tau_s)} f_s per element otherwise.  M, C_L, B~ and H enter as
// single bf16 operands, as the real chunked scan rounds its M, its state copy
// and its scaled inputs.  Eight row warps: the two warps of a TMEM lane quarter
// split the tile columns, M's blocks, the two states and the y columns.
//
// Phases per chunk, one mbarrier hand-off each (all waits bounded):
//   TMA: C, B, x of both rows.    rows: dt, tau and the complex factors; C^, C~,
//   C_L, B~ from C and B; each state's bf16 copy, then the state rotated by
//   Lambda_63 in TMEM.    MMA: S_re, S_im; then H_r += B~^T x (its rows) and
//   C_L H_0.    rows: M in place of S_re.    MMA: Y = M x; C_L H_1 in place of S_im.
//   rows: y = Y + C_L H_r + D x by tensor stores.  After the last chunk the
//   states go out.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "ptx.cuh"
#include "ssd_internal.h"
#include "tmap.h"

namespace ssd {

__device__ unsigned int g_complex_tc_error;

namespace {

using namespace ssd::ptx;

constexpr int kR = 128;                    // rows: two batch rows' chunks of 64 steps
constexpr int kQ = 64;                     // steps per chunk
constexpr int kP = 64, kN = 128;
constexpr int kRowWarps = 8;               // warps 0-7: warp w reads TMEM lane quarter w & 3 (one row
                                           // per thread) and takes half w >> 2 of that quarter's work
constexpr int kIssueWarp = 8;              // TMA and MMA issue, TMEM owner
constexpr int kThreads = 9 * 32;
constexpr uint32_t kT16 = 16384;           // one [128 rows][64 bf16] tile, 128-byte swizzle

// shared memory (from a 1024-aligned base)
constexpr uint32_t kOffC = 0;                      // C [t][n], two tiles (n 0-63, 64-127); then C^
constexpr uint32_t kOffCT = kOffC + 2 * kT16;      // C~; after S, y staging (2 KB per warp)
constexpr uint32_t kOffCL = kOffCT + 2 * kT16;     // C_L
constexpr uint32_t kOffB = kOffCL + 2 * kT16;      // B [s][n]
constexpr uint32_t kOffBT = kOffB + 2 * kT16;      // B~
constexpr uint32_t kOffX = kOffBT + 2 * kT16;      // x [s][p]
constexpr uint32_t kOffHB = kOffX + kT16;          // the states entering the chunk, bf16 [n][p], one tile each
constexpr uint32_t kOffArr = kOffHB + 2 * kT16;
// per row: tau, f, the column factor of M's blocks, Lambda, g
enum { A_TAU = 0, A_FR, A_FI, A_CR, A_CI, A_LR, A_LI, A_GR, A_GI, A_NUM };
constexpr uint32_t kOffRed = kOffArr + A_NUM * kR * 4;   // 8 floats: warp totals of dt
constexpr uint32_t kOffBars = kOffRed + 8 * 4;
enum { BAR_FULL = 0, BAR_ROWS_A, BAR_MMA_S, BAR_ROWS_M, BAR_MMA_Y, BAR_EPI, BAR_RSYNC, BAR_DRAIN, kNumBars };
constexpr uint32_t kOffHolder = kOffBars + kNumBars * 8;
constexpr uint32_t kSmemBytes = kOffHolder + 16 + 1024;

// TMEM columns
constexpr uint32_t kColS = 0;       // S_re; M (bf16 pairs) in the first 8 columns of each 16
constexpr uint32_t kColSI = 128;    // S_im; then C_L H_1
constexpr uint32_t kColY = 256;     // M x
constexpr uint32_t kColH = 320;     // the states: row r at +64 r
constexpr uint32_t kColYO0 = 448;   // C_L H_0 (issued with S, before M is built)

constexpr uint64_t kTimeoutNs = 2000000000ull;

struct CtcParams {
    const float *dt_raw, *dt_bias, *A_polar, *D;
    const float *h0;      // [B,H,P,N] or null
    float *h_final;       // [B,H,P,N] or null
    long long L;
    int Bt, H, G;
};

struct CtcMaps {
    CUtensorMap x, B, C;  // bf16 loads, boxes of 64 x 64
    CUtensorMap y;        // bf16 stores, boxes of 32 x 32, no swizzle
};

__device__ __forceinline__ uint32_t sw128(uint32_t r, uint32_t c) { return r * 128u + ((c ^ (r & 7u)) << 4); }

__device__ void raise_error() { atomicCAS(&g_complex_tc_error, 0u, (unsigned)SSD_ERR_TIMEOUT); }

// bounded wait (each probe suspends up to 1 ms); false after kTimeoutNs
__device__ bool wait_bar(uint64_t *bar, uint32_t parity)
{
    if (mbar_wait_for(bar, parity, 1000000u))
        return true;
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < kTimeoutNs)
        if (mbar_wait_for(bar, parity, 1000000u))
            return true;
    raise_error();
    return false;
}

__device__ __forceinline__ void warp_arrive(uint64_t *bar)
{
    __syncwarp();
    if ((threadIdx.x & 31) == 0)
        mbar_arrive(bar);
}

// bounded barrier of the row warps on an mbarrier (phase: this thread's copy)
__device__ __forceinline__ bool rsync(uint64_t *bar, uint32_t &phase)
{
    warp_arrive(bar);
    const bool ok = wait_bar(bar, phase);
    phase ^= 1u;
    return ok;
}

__device__ __forceinline__ float softplus_f32(float z) { return fmaxf(z, 0.f) + log1pf(expf(-fabsf(z))); }

// e^{A u} for real u: (e^{a_r u} cos(a_i u), e^{a_r u} sin(a_i u))
__device__ __forceinline__ float2 cexp_a(float ar, float ai, float u)
{
    float s, c;
    sincosf(ai * u, &s, &c);
    const float m = expf(ar * u);
    return make_float2(m * c, m * s);
}

__device__ __forceinline__ float2 cmul(float2 a, float2 b) { return make_float2(a.x * b.x - a.y * b.y, a.x * b.y + a.y * b.x); }

// 8 bf16 of a swizzled tile row as floats, and back (rounded to nearest)
__device__ __forceinline__ void ld8(const uint8_t *tile, int r, int c, float (&v)[8])
{
    const uint4 u = *reinterpret_cast<const uint4 *>(tile + sw128(r, c));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ void st8(uint8_t *tile, int r, int c, const float (&v)[8])
{
    *reinterpret_cast<uint4 *>(tile + sw128(r, c)) = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                                                pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
}

__global__ void __launch_bounds__(kThreads, 1) ssd_complex_tc_kernel(const __grid_constant__ CtcMaps maps,
                                                                     const CtcParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBars);
    uint32_t *holder = reinterpret_cast<uint32_t *>(smem + kOffHolder);
    float *arr = reinterpret_cast<float *>(smem + kOffArr);
    float *tau_s = arr + A_TAU * kR, *fr_s = arr + A_FR * kR, *fi_s = arr + A_FI * kR;
    float *cr_s = arr + A_CR * kR, *ci_s = arr + A_CI * kR;
    float *red = reinterpret_cast<float *>(smem + kOffRed);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = p.H;
    const int nch = (int)((p.L + kQ - 1) / kQ);
    const size_t NP = (size_t)kN * kP;
    // work items: (pair of batch rows, head), pair-major so that the CTAs running
    // at once share a group's B and C; CTA i takes items i, i + grid, ...
    const long long nitems = (long long)((p.Bt + 1) / 2) * H;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNumBars; ++i)
            mbar_init(&bars[i], (i == BAR_ROWS_A || i == BAR_ROWS_M || i == BAR_EPI || i == BAR_RSYNC) ? kRowWarps : 1);
        fence_mbar_init();
    }
    if (warp == kIssueWarp) {
        tmem_alloc(holder, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *holder;
    bool ok = true;
    uint32_t armed = 0;   // steps whose loads were issued (issue lane)

    if (warp == kIssueWarp) {
        if (lane == 0) {
            const uint64_t once = policy_evict_first(), shared = policy_evict_last();
            const uint32_t sC = smem_u32(smem + kOffC), sCT = smem_u32(smem + kOffCT), sCL = smem_u32(smem + kOffCL);
            const uint32_t sB = smem_u32(smem + kOffB), sBT = smem_u32(smem + kOffBT), sX = smem_u32(smem + kOffX);
            const uint32_t sHB = smem_u32(smem + kOffHB);
            // K-major operand over two 64-column tiles (K = 128): 8 k-steps of 16
            auto kmaj = [](uint32_t base, int kk) { return sdesc_sw128(base + (kk >> 2) * kT16 + (kk & 3) * 32, 16, 1024); };
            // MN-major operand: k-step kk = rows 16 kk .. +15; the 64-element MN blocks kT16 apart
            auto mnmaj = [](uint32_t base, int kk) { return sdesc_sw128(base + kk * 2048, kT16, 1024); };
            const uint32_t i128kk = idesc_bf16_f32(128, 128, 0, 0), i64kn = idesc_bf16_f32(128, 64, 0, 1);
            const uint32_t i64nn = idesc_bf16_f32(128, 64, 1, 1);
            // the loads of one step (item u, chunk c): C and B once the previous step's S
            // products have read theirs, x once the previous step's epilogue has read
            // its x; the barrier is armed for all of them with the first
            auto load_cb = [&](long long u, int c) {
                const int bp = (int)(u / H), hh = (int)(u - (long long)bp * H), gg = hh / (H / p.G);
                mbar_arrive_expect_tx(&bars[BAR_FULL], 5 * kT16);
                for (int r = 0; r < 2; ++r) {
                    const uint32_t ro = r * (kT16 / 2);   // rows 64 r ..
                    const int t0 = c * kQ, br = 2 * bp + r;
                    tma_load_3d(smem + kOffC + ro, &maps.C, &bars[BAR_FULL], gg * kN, t0, br, shared);
                    tma_load_3d(smem + kOffC + kT16 + ro, &maps.C, &bars[BAR_FULL], gg * kN + 64, t0, br, shared);
                    tma_load_3d(smem + kOffB + ro, &maps.B, &bars[BAR_FULL], gg * kN, t0, br, shared);
                    tma_load_3d(smem + kOffB + kT16 + ro, &maps.B, &bars[BAR_FULL], gg * kN + 64, t0, br, shared);
                }
                ++armed;
            };
            auto load_x = [&](long long u, int c) {
                const int bp = (int)(u / H), hh = (int)(u - (long long)bp * H);
                for (int r = 0; r < 2; ++r)
                    tma_load_3d(smem + kOffX + r * (kT16 / 2), &maps.x, &bars[BAR_FULL], hh * kP, c * kQ, 2 * bp + r,
                                once);
            };
            // an item's entering states into L2 one item ahead (the row warps load them)
            auto prefetch_states = [&](long long u) {
                if (!p.h0 || u >= nitems)
                    return;
                const int bp = (int)(u / H), hh = (int)(u - (long long)bp * H);
                for (int r = 0; r < 2; ++r)
                    if (2 * bp + r < p.Bt)
                        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                                         p.h0 + ((size_t)(2 * bp + r) * H + hh) * NP),
                                     "r"((uint32_t)(NP * 4))
                                     : "memory");
            };
            uint32_t k = 0;   // steps so far (the barriers' phases)
            if ((long long)blockIdx.x < nitems) {
                load_cb(blockIdx.x, 0);
                load_x(blockIdx.x, 0);
            }
            for (long long u = blockIdx.x; u < nitems && ok; u += gridDim.x) {
                prefetch_states(u + gridDim.x);
                for (int c = 0; c < nch && ok; ++c, ++k) {
                    const uint32_t par = k & 1;
                    const long long un = c + 1 < nch ? u : u + gridDim.x;   // the next step
                    const int cn = c + 1 < nch ? c + 1 : 0;
                    const bool has_next = un < nitems;
                    // ---- S_re = C^ B^T, S_im = C~ B^T
                    if (!(ok = wait_bar(&bars[BAR_ROWS_A], par)))
                        break;
                    tc_fence_after();
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ss(tmem + kColS, kmaj(sC, kk), kmaj(sB, kk), i128kk, kk > 0);
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ss(tmem + kColSI, kmaj(sCT, kk), kmaj(sB, kk), i128kk, kk > 0);
                    mma_commit(&bars[BAR_MMA_S]);
                    // H_r += B~^T x over row r's steps, and C_L H_0: their operands are ready,
                    // so they run while M is built
                    for (int r = 0; r < 2; ++r)
                        for (int kk = 4 * r; kk < 4 * r + 4; ++kk)
                            mma_ss(tmem + kColH + 64 * r, mnmaj(sBT, kk), mnmaj(sX, kk), i64nn, 1);
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ss(tmem + kColYO0, kmaj(sCL, kk), mnmaj(sHB, kk), i64kn, kk > 0);
                    // the next step's C and B, once S has read this step's
                    if (has_next) {
                        if (!(ok = wait_bar(&bars[BAR_MMA_S], par)))
                            break;
                        load_cb(un, cn);
                    }
                    // ---- Y = M x; C_L H_1 (in S_im's columns, once M has been built from them)
                    if (!(ok = wait_bar(&bars[BAR_ROWS_M], par)))
                        break;
                    tc_fence_after();
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ts(tmem + kColY, tmem + kColS + 16 * kk, mnmaj(sX, kk), i64kn, kk > 0);
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ss(tmem + kColSI, kmaj(sCL, kk), mnmaj(sHB + kT16, kk), i64kn, kk > 0);
                    mma_commit(&bars[BAR_MMA_Y]);
                    // the next step's x, once this step's epilogue has read its x
                    if (has_next) {
                        if (!(ok = wait_bar(&bars[BAR_EPI], par)))
                            break;
                        load_x(un, cn);
                    }
                }
            }
            // no MMA may be in flight when tensor memory is released, nor a TMA load
            // when the CTA exits
            const uint64_t tw = globaltimer_ns();
            if (armed > 0)
                while (!mbar_wait_for(&bars[BAR_FULL], (armed - 1) & 1, 1000000u) &&
                       globaltimer_ns() - tw < kTimeoutNs) {
                }
            mma_commit(&bars[BAR_DRAIN]);   // (arrives once every MMA issued so far has completed)
        }
    } else {
        // ------------------------------------------------------------ rows
        const int q = warp & 3;                  // TMEM lane quarter
        const int hf = warp >> 2;                // half: tile columns 64 hf.., M's blocks of parity hf,
                                                 // state hf, y columns 32 hf..
        const int t = 32 * q + lane;             // this thread's step row (and state row n = t)
        const int rr = q >> 1, i = t & (kQ - 1); // the step row's batch row (0, 1) and step in the chunk
        const uint32_t trow = tmem + (static_cast<uint32_t>(32 * q) << 16);
        uint8_t *tC = smem + kOffC, *tCT = smem + kOffCT, *tCL = smem + kOffCL, *tB = smem + kOffB;
        uint8_t *tBT = smem + kOffBT, *tX = smem + kOffX, *tHB = smem + kOffHB;
        float *lr_s = arr + A_LR * kR, *li_s = arr + A_LI * kR, *gr_s = arr + A_GR * kR, *gi_s = arr + A_GI * kR;
        uint32_t rphase = 0, k = 0;   // (k: steps so far, the barriers' phases)
        // (every wait's result is made warp-uniform: the TMEM loads and stores that
        // follow are collective)
        for (long long u = blockIdx.x; u < nitems && ok; u += gridDim.x) {
            const int bp = (int)(u / H), h = (int)(u - (long long)bp * H);
            const int b0 = 2 * bp, b = b0 + rr;      // batch rows b0, b0 + 1; this step row's
            const float la = p.A_polar[2 * h], th = p.A_polar[2 * h + 1];
            const float ar = expf(la) * cosf(th), ai = expf(la) * sinf(th);
            const float inv = 1.f / (ar * ar + ai * ai);            // 1 / |A|^2
            const float Dh = p.D[h];
            auto dt_raw_of = [&](int c) {
                const long long l = (long long)c * kQ + i;
                return (b < p.Bt && l < p.L) ? p.dt_raw[((size_t)b * p.L + l) * H + h] : 0.f;
            };
            float zr = (nch > 0 && hf == 0) ? dt_raw_of(0) : 0.f;
            // state hf entering the item's first chunk (row n = t), loaded now: the loads
            // overlap the chunk's tiles and factors
            uint32_t hv[2][32];
            {
                const float *src = (p.h0 && b0 + hf < p.Bt) ? p.h0 + ((size_t)(b0 + hf) * H + h) * NP + t : nullptr;
#pragma unroll
                for (int kk = 0; kk < 64; ++kk)
                    hv[kk >> 5][kk & 31] = __float_as_uint(src ? __ldg(src + (size_t)kk * kN) : 0.f);
            }
            for (int c = 0; c < nch && ok; ++c, ++k) {
                const uint32_t par = k & 1;
                const long long l = (long long)c * kQ + i;
                const bool valid = b < p.Bt && l < p.L;
                // ---- dt, tau within the row's chunk (its two warps of half 0), the complex factors
                float dt = 0.f, tau = 0.f;
                if (hf == 0) {
                    dt = valid ? softplus_f32(zr + p.dt_bias[h]) : 0.f;
                    if (c + 1 < nch)
                        zr = dt_raw_of(c + 1);   // in flight through this chunk
                    tau = dt;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const float u = __shfl_up_sync(0xffffffffu, tau, o);
                        if (lane >= o)
                            tau += u;
                    }
                    if (lane == 31)
                        red[q] = tau;
                }
                if (!(ok = __all_sync(0xffffffffu, rsync(&bars[BAR_RSYNC], rphase))))
                    break;
                if (hf == 0) {
                    tau += (q & 1) ? red[q - 1] : 0.f;
                    const float tau_end = red[2 * rr] + red[2 * rr + 1];
                    // f = (e^{A dt} - 1) / A, with e^{A dt} - 1 = expm1(a_r dt) cos(a_i dt) - 2 sin^2(a_i dt / 2)
                    //     + i e^{a_r dt} sin(a_i dt)
                    float sd, cd;
                    sincosf(ai * dt, &sd, &cd);
                    const float sh = sinf(0.5f * ai * dt);
                    const float nr = expm1f(ar * dt) * cd - 2.f * sh * sh, ni = expf(ar * dt) * sd;
                    const float2 f = make_float2((nr * ar + ni * ai) * inv, (ni * ar - nr * ai) * inv);
                    const float2 lam = cexp_a(ar, ai, tau);                      // Lambda_t
                    const float2 gw = cmul(cexp_a(ar, ai, tau_end - tau), f);    // g_t
                    const float tau_e = __shfl_sync(0xffffffffu, tau, lane | 15);   // the end of this 16-step block
                    const float2 cf = cmul(cexp_a(ar, ai, tau_e - tau), f);      // column factor of M's blocks
                    tau_s[t] = tau;
                    fr_s[t] = f.x;
                    fi_s[t] = f.y;
                    cr_s[t] = cf.x;
                    ci_s[t] = cf.y;
                    lr_s[t] = lam.x;
                    li_s[t] = lam.y;
                    gr_s[t] = gw.x;
                    gi_s[t] = gw.y;
                }
                // (every row's entries are read by the other half and by the M build)
                if (!(ok = __all_sync(0xffffffffu, rsync(&bars[BAR_RSYNC], rphase))) ||
                    !(ok = __all_sync(0xffffffffu, wait_bar(&bars[BAR_FULL], par))))
                    break;
                // ---- C^ (in place), C~, C_L from row t of C; B~ from row t of B (tile hf)
                {
                    const float2 lam = make_float2(lr_s[t], li_s[t]), gw = make_float2(gr_s[t], gi_s[t]);
                    uint8_t *c0 = tC + hf * kT16, *b1 = tB + hf * kT16;
#pragma unroll 1
                    for (int ch = 0; ch < 8; ++ch) {
                        float v[8], w1[8], w2[8], w3[8];
                        ld8(c0, t, ch, v);
#pragma unroll
                        for (int j = 0; j < 8; j += 2) {
                            const float re = v[j], im = v[j + 1];
                            w1[j] = im;                              // C~ = (C_i, C_r)
                            w1[j + 1] = re;
                            w2[j] = lam.x * re - lam.y * im;         // C_L = (Re(Lambda C), -Im(Lambda C))
                            w2[j + 1] = -(lam.x * im + lam.y * re);
                            w3[j] = re;                              // C^ = (C_r, -C_i)
                            w3[j + 1] = -im;
                        }
                        st8(tCT + hf * kT16, t, ch, w1);
                        st8(tCL + hf * kT16, t, ch, w2);
                        st8(c0, t, ch, w3);
                        ld8(b1, t, ch, v);
#pragma unroll
                        for (int j = 0; j < 8; j += 2) {
                            const float re = v[j], im = v[j + 1];
                            w1[j] = gw.x * re - gw.y * im;           // B~ = g B
                            w1[j + 1] = gw.x * im + gw.y * re;
                        }
                        st8(tBT + hf * kT16, t, ch, w1);
                    }
                }
                // ---- state hf (row n = t): its bf16 copy for C_L H, then rotated by Lambda_63
                //      of its batch row (lanes 2k, 2k+1 hold a component's re, im)
                {
                    if (c > 0) {
                        tmem_ld32(trow + kColH + 64 * hf, hv[0]);
                        tmem_ld32(trow + kColH + 64 * hf + 32, hv[1]);
                        tmem_wait_ld();
                    }
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) {
                        float w[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            w[e] = __uint_as_float(hv[cc >> 2][8 * (cc & 3) + e]);
                        st8(tHB + hf * kT16, t, cc, w);
                    }
                    const float te = red[2 * hf] + red[2 * hf + 1];   // tau at the end of row hf's chunk
                    const float2 z = cexp_a(ar, ai, te);
                    const bool odd = lane & 1;
#pragma unroll
                    for (int j = 0; j < 64; ++j) {
                        const float mine = __uint_as_float(hv[j >> 5][j & 31]);
                        const float other = __shfl_xor_sync(0xffffffffu, mine, 1);
                        // even lane: re' = z_r re - z_i im; odd lane: im' = z_r im + z_i re
                        const float out = odd ? fmaf(z.x, mine, z.y * other) : fmaf(z.x, mine, -z.y * other);
                        hv[j >> 5][j & 31] = __float_as_uint(out);
                    }
                    tmem_st32(trow + kColH + 64 * hf, hv[0]);
                    tmem_st32(trow + kColH + 64 * hf + 32, hv[1]);
                }
                tmem_wait_st();
                fence_proxy_async_smem();
                tc_fence_before();
                warp_arrive(&bars[BAR_ROWS_A]);
                // ---- M from S_re, S_im in place (row t; the blocks of 16 steps of parity hf)
                if (!(ok = __all_sync(0xffffffffu, wait_bar(&bars[BAR_MMA_S], par))))
                    break;
                tc_fence_after();
                {
                    const int gdiag = t >> 4;   // the block holding step t (2q or 2q + 1 within the warp)
                    const float tau_t = tau_s[t];   // (computed by half 0)
#pragma unroll 1
                    for (int G = hf; G < 8; G += 2) {
                        uint32_t m[8];
                        // warp-uniform: some row of this warp reaches block G (the TMEM loads are
                        // collective); each lane then takes its own case
                        if ((G >> 2) != rr || G > 2 * q + 1) {
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                m[e] = 0u;
                        } else {
                            uint32_t sr[16], si[16];
                            tmem_ld16(trow + kColS + 16 * G, sr);
                            tmem_ld16(trow + kColSI + 16 * G, si);
                            const int s0 = 16 * G, se = s0 + 15;
                            // e^{A (tau_t - tau_e)}: at most 1 in modulus below the diagonal block and
                            // at most e^{|a_r| span} on it; the factored form there while that stays
                            // far inside fp32 (the span test is the same for the whole block)
                            const bool factored = G < gdiag || fabsf(ar) * (tau_s[se] - tau_s[s0]) < 60.f;
                            const float2 rf = cexp_a(ar, ai, tau_t - tau_s[se]);
                            tmem_wait_ld();
                            float mv[16];
                            if (G > gdiag) {    // above this row's diagonal
#pragma unroll
                                for (int e = 0; e < 16; ++e)
                                    mv[e] = 0.f;
                            } else if (factored) {
#pragma unroll
                                for (int e = 0; e < 16; ++e) {
                                    const int s = s0 + e;
                                    const float2 E = cmul(rf, make_float2(cr_s[s], ci_s[s]));
                                    const float v = E.x * __uint_as_float(sr[e]) - E.y * __uint_as_float(si[e]);
                                    mv[e] = s <= t ? v : 0.f;
                                }
                            } else {            // the diagonal block, directly: e^{A (tau_t - tau_s)} f_s, s <= t
#pragma unroll
                                for (int e = 0; e < 16; ++e) {
                                    const int s = s0 + e;
                                    float val = 0.f;
                                    if (s <= t) {
                                        const float2 E = cmul(cexp_a(ar, ai, tau_t - tau_s[s]), make_float2(fr_s[s], fi_s[s]));
                                        val = E.x * __uint_as_float(sr[e]) - E.y * __uint_as_float(si[e]);
                                    }
                                    mv[e] = val;
                                }
                            }
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                m[e] = pack_bf16x2(mv[2 * e], mv[2 * e + 1]);
                        }
                        tmem_st8(trow + kColS + 16 * G, m);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                warp_arrive(&bars[BAR_ROWS_M]);
                // ---- y = M x + C_L H_r + D x (row t, columns 32 hf ..), by a tensor store per warp
                if (!(ok = __all_sync(0xffffffffu, wait_bar(&bars[BAR_MMA_Y], par))))
                    break;
                tc_fence_after();
                {
                    uint8_t *stg = tCT + warp * 2048;   // this warp's box: 32 rows x 32 bf16, plain (C~ is dead)
#pragma unroll 1
                    for (int g16 = 2 * hf; g16 < 2 * hf + 2; ++g16) {
                        uint32_t ym[16], yo[16];
                        tmem_ld16(trow + kColY + 16 * g16, ym);
                        tmem_ld16(trow + (rr ? kColSI : kColYO0) + 16 * g16, yo);
                        tmem_wait_ld();
                        float xv[8], o[8];
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            ld8(tX, t, 2 * g16 + hh, xv);
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                o[e] = fmaf(Dh, xv[e], __uint_as_float(ym[8 * hh + e]) + __uint_as_float(yo[8 * hh + e]));
                            *reinterpret_cast<uint4 *>(stg + lane * 64 + 16 * (2 * (g16 & 1) + hh)) =
                                make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]), pack_bf16x2(o[4], o[5]),
                                           pack_bf16x2(o[6], o[7]));
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        const long long r0 = (long long)c * kQ + 32 * (q & 1);
                        if (b < p.Bt && r0 < p.L)
                            tma_store_3d(&maps.y, stg, h * kP + 32 * hf, (int)r0, b);
                        bulk_commit_group();
                        bulk_wait_read_all();   // the box is rewritten next chunk
                    }
                }
                warp_arrive(&bars[BAR_EPI]);
            }
            // ---- the item's final state hf (row n = t), [P][N]
            if (ok && p.h_final && b0 + hf < p.Bt) {
                tmem_ld32(trow + kColH + 64 * hf, hv[0]);
                tmem_ld32(trow + kColH + 64 * hf + 32, hv[1]);
                tmem_wait_ld();
                float *dst = p.h_final + ((size_t)(b0 + hf) * H + h) * NP + t;
#pragma unroll
                for (int kk = 0; kk < 64; ++kk)
                    dst[(size_t)kk * kN] = __uint_as_float(hv[kk >> 5][kk & 31]);
            }
        }
        if (lane == 0)
            bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kIssueWarp) {
        // no MMA in flight when tensor memory is released (the drain commit arrives
        // once every MMA issued before it has completed)
        if (lane == 0) {
            const uint64_t tw = globaltimer_ns();
            while (!mbar_wait_for(&bars[BAR_DRAIN], 0, 1000000u) && globaltimer_ns() - tw < kTimeoutNs) {
            }
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

bool complex_tc_supported(const ComplexArgs &a)
{
    auto al = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
    return a.dtype == SSD_DTYPE_BF16 && a.headdim == kP && a.dstate == kN && a.seqlen >= 2 &&
           a.batch >= 1 && a.batch < (1LL << 30) && a.seqlen < (1LL << 31) &&
           (long long)((a.batch + 1) / 2) * a.nheads < (1LL << 40) && al(a.x) && al(a.B) && al(a.C) && al(a.y);
}

cudaError_t complex_tc_launch(const ComplexArgs &a, cudaStream_t st)
{
    SSD_NVTX_RANGE("complex_tc_launch");
    if (!complex_tc_supported(a))
        return cudaErrorInvalidValue;
    CtcMaps maps;
    const uint64_t HP = (uint64_t)a.nheads * kP, GN = (uint64_t)a.ngroups * kN, L = (uint64_t)a.seqlen;
    const uint64_t Bt = (uint64_t)a.batch;
    if (!make_tmap_bf16_3d(&maps.x, a.x, HP, L, Bt, HP * 2, HP * 2 * L, 64, kQ) ||
        !make_tmap_bf16_3d(&maps.B, a.B, GN, L, Bt, GN * 2, GN * 2 * L, 64, kQ) ||
        !make_tmap_bf16_3d(&maps.C, a.C, GN, L, Bt, GN * 2, GN * 2 * L, 64, kQ) ||
        !make_tmap_bf16_3d(&maps.y, a.y, HP, L, Bt, HP * 2, HP * 2 * L, 32, 32, false))
        return cudaErrorInvalidValue;
    CtcParams p;
    p.dt_raw = a.dt_raw;
    p.dt_bias = a.dt_bias;
    p.A_polar = a.A_polar;
    p.D = a.D;
    p.h0 = a.init_state;
    p.h_final = a.final_state;
    p.L = a.seqlen;
    p.Bt = (int)a.batch;
    p.H = a.nheads;
    p.G = a.ngroups;
    const cudaError_t e =
        cudaFuncSetAttribute(ssd_complex_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess)
        return e;
    // persistent: one CTA per SM (its shared memory), each walking items
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaErrorInvalidValue;
    const long long nitems = (long long)((a.batch + 1) / 2) * a.nheads;
    const dim3 grid((unsigned)std::min<long long>(nitems, sms));
    ssd_complex_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(maps, p);
    return cudaGetLastError();
}

ssd_status_t complex_tc_read_device_error(uint32_t *code)
{
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_complex_tc_error, sizeof(v)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_complex_tc_error, &zero, sizeof(zero)) != cudaSuccess)
        return SSD_ERR_CUDA;
    *code = v;
    return SSD_OK;
}

}  // namespace ssd
