// ssd_chunk.cu -- chunked SSD forward scan on the sm_103a tensor cores.
//
// One persistent cooperative kernel evaluates the whole scan.  A work unit is
// a range of R consecutive chunks (R*Q steps) of one chain, a chain being a
// batch row b and a pair of heads h0, h0+1 of one group.  Units are ordered
// range-major (all chains' first ranges, then all second ranges, ...): the
// CTAs running at any moment share the group's B/C tiles through L2, and the
// unit that needs the state left by the previous range of its chain was
// scheduled about one grid round earlier.  R is chosen on the host to balance
// the grid against the cost of handing a state from unit to unit.
//
// Inside a unit the steps are walked in sub-chunks of T = 128.  For a
// sub-chunk with carried-in state P (N x P per head) and the sub-chunk-local
// inclusive cumulative sum cs_t = sum_{k<=t} dt_k A:
//
//   S      = C B^T                                   (T x T, shared by both heads)
//   M[t,s] = S[t,s] exp(cs_t - cs_s) dt_s  (s <= t)
//   y_t    = (M x)_t + D x_t + exp(cs_t) (C P)_t      (D x added in fp32 to M x)
//   P     <- exp(cs_{T-1}) P + B^T (w o x),   w_s = exp(cs_{T-1} - cs_s) dt_s
//
// This is the quadratic ("dual") form inside a sub-chunk and the linear
// recurrence between sub-chunks and chunks.  Source: the SSD module of
// @seanhogg/builderforce-memory-engine 2026.6.18 (chunked evaluation with a
// carried state) and the chunked-scan pipeline of mamba-rs 0.2.1
// mamba3_siso/gpu/mamba3_gpu.rs (decay cumsum, chunk state, state passing,
// chunk scan), applied to the Mamba-2 recurrence.
//
// Roles (18 warps):
//   warps 0-7   decay group: dt, cumulative sums and decay factors; the masked
//               decay matrix M, built in tensor memory as a bf16 MMA operand
//   warps 8-15  state group: w-scaling of x, state rescale, output epilogue,
//               state handoff between units
//   warp 16     TMA producer: B/C tiles (2 stages), x tiles (2 stages)
//               (the state warps issue the TMA stores of y themselves)
//   warp 17     tcgen05 MMA issuer (one lane) and TMEM owner
// The decay group prepares sub-chunk j+1 while the state group finishes j.
// Tensor memory (512 columns x 128 lanes, fp32):
//   [  0,128)  Y_diag = M x            lanes t, columns head*64 + p
//   [128,256)  Y_off  = C P            lanes t, columns head*64 + p
//   [256,384)  S = C B^T, then in place M of both heads (bf16 pairs)
//   [384,512)  P, the carried state    lanes n, columns head*64 + p
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
constexpr int kGroupWarps = 8;   // warps per math group
constexpr int kStateWarp0 = 8;   // first warp of the state group
constexpr int kProducerWarp = 16;
constexpr int kMmaWarp = 17;
constexpr int kThreads = 18 * 32;

constexpr uint32_t kTileBytes = 16384;              // 128 rows x 128 bytes
constexpr uint32_t kBCStageBytes = 4 * kTileBytes;  // C lo/hi, B lo/hi
constexpr uint32_t kXStageBytes = 2 * kTileBytes;   // x of two heads

// dynamic shared memory layout (offsets from a 1024-aligned base)
constexpr uint32_t kOffBC = 0;
constexpr uint32_t kOffX = kOffBC + 2 * kBCStageBytes;
// decay arrays, 3 buffers (sub-chunk j uses buffer j % 3), each:
//   cs2 [2][T], dt [2][T], colf [2][T], ecs [2][T], wsc [2][T], dtot [2] (+pad),
//   dcr [2][T] (trapezoidal mode: diagonal weight minus input weight)
constexpr int kDecayFloats = 6 * 2 * kT + 4;
constexpr uint32_t kOffDecay = kOffX + 2 * kXStageBytes;
constexpr uint32_t kOffWsum = kOffDecay + 3 * kDecayFloats * 4;
constexpr int kMaxHeads = 512;                       // per-head parameters staged in shared memory
constexpr uint32_t kOffHead = kOffWsum + 64;          // A*log2(e), dt_bias, D  (3 x kMaxHeads floats)
// conv mode: the conv1d weights of the head pair's 128 x channels, per head and
// 8-channel chunk c: taps 0..3 (tap k multiplies the input k steps back; zero
// past the kernel size) then the bias, 8 channels each (40 floats); and the 3
// raw input rows before the sub-chunk, per head (the halo carried between the
// sub-chunks of a unit)
constexpr uint32_t kOffConvW = kOffHead + 3 * kMaxHeads * 4;
constexpr int kConvWFloats = 2 * 8 * 40;
constexpr uint32_t kOffHalo = kOffConvW + kConvWFloats * 4;   // [2 heads][3 rows][128 bytes]
constexpr uint32_t kOffBars = kOffHalo + 2 * 3 * 128;
constexpr int kNumBars = 24;
constexpr uint32_t kOffTmemHolder = kOffBars + kNumBars * 8;
constexpr uint32_t kSmemBytes = kOffTmemHolder + 16 + 1024;  // + alignment slack

// tensor memory columns (128 lanes each)
//   SM: S = C B^T (fp32, column s), then, in place, M of both heads as bf16
//       pairs: for each 16-step group s0, columns s0 + 8*head + c hold
//       s = s0 + 2c, s0 + 2c + 1 (so M is built group by group in place)
constexpr uint32_t kColYd = 0, kColYo = 128, kColSM = 256, kColP = 384;

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
    BAR_MSYNC,   // decay-group barrier (bounded, unlike bar.sync)
    BAR_CSYNC,   // conv mode: decay-group barrier around the conv (bounded)
};

struct ChunkParams {
    const float *dt_raw;
    const float *dt_bias;
    const float *A_log;
    const float *D;
    const float *init_state;          // [B,H,P,N] or null
    __nv_bfloat16 *y;
    float *final_state;               // [B,H,P,N] or null
    float *slots;                     // handoff states, [chains][2][16][N][4] (chained) or [units][2][16][N][4]
                                      // (split); null when no unit hands a state on
    float *unit_decay;                // split pass 1: exp(sum dt A) over each unit, [units][2]
    unsigned long long *flags;        // [nunits][state-group warps]: warp w of a unit publishes its rows
    unsigned long long *abort_word;
    unsigned long long epoch;
    unsigned long long timeout_ns;
    long long L;
    long long nunits;                 // range schedule: units
    long long total_subs;             // piece schedule: sub-chunks of all chains
    int H, span, nranges, nhp, nchains, hpg;   // span = steps per unit (R*Q)
    int nsub_chain;                   // sub-chunks per chain
    int diag_stall;                   // first units wait for a handoff nobody publishes
    // trapezoidal mode: per-token dt, a, trap [B,L,H]; carried k0 [B,H,N], v0 [B,H,P] (bf16, or null)
    const float *tdt, *ta, *ttrap;
    const __nv_bfloat16 *k0, *v0;
    int mode;                         // kChained, kSplitLocal or kSplitEntering
    // conv mode: raw xbc [B,L,conv_cc] (the x tensor map reads its x channels), the conv
    // weights [conv_cc, conv_k] and bias [conv_cc] (or null), the carried conv state
    // [B, conv_k - 1, conv_cc] (or null)
    const __nv_bfloat16 *xbc;
    const float *conv_w, *conv_b;
    const __nv_bfloat16 *conv_state;
    int conv_k, conv_cc;
};

// How the units of a chain get their entering state:
//   kChained        from the preceding unit of the chain, through a slot per chain
//                   and a release/acquire flag (one launch)
//   kSplitLocal     split pass 1: every unit starts from zero and stores its end
//                   state and its total decay in a slot of its own (no y)
//   kSplitEntering  split pass 3: every unit reads its entering state, combined
//                   between the passes, from its own slot
enum { kChained = 0, kSplitLocal = 1, kSplitEntering = 2 };

struct Maps {
    CUtensorMap x, B, C;
    CUtensorMap y;         // store boxes of 32 steps x 64 channels
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

__device__ void raise_timeout(const ChunkParams &p)
{
    atomicCAS(&g_chunk_error, 0u, (unsigned)SSD_ERR_TIMEOUT);
    atomicExch(p.abort_word, p.epoch);
}

__device__ __forceinline__ bool aborted(const ChunkParams &p)
{
    return *reinterpret_cast<volatile unsigned long long *>(p.abort_word) == p.epoch;
}

// Bounded wait for the phase of `bar` with the given parity.  Each probe
// suspends the thread for up to 1 ms (it resumes as soon as the phase
// completes), so waiting warps do not take issue slots from working ones.
__device__ bool wait_bar(uint64_t *bar, uint32_t parity, const ChunkParams &p)
{
    if (mbar_wait_for(bar, parity, 1000000u))
        return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_wait_for(bar, parity, 1000000u))
            return true;
        if (aborted(p))
            return false;
        if (globaltimer_ns() - t0 > p.timeout_ns) {
            raise_timeout(p);
            return false;
        }
    }
}

// One arrival per warp (lane 0, after the warp's own writes are ordered).
__device__ __forceinline__ void warp_arrive(uint64_t *bar)
{
    __syncwarp();
    if ((threadIdx.x & 31) == 0)
        mbar_arrive(bar);
}

// Group barrier of the decay warps on an mbarrier, so that it is bounded too.
__device__ __forceinline__ bool group_sync(uint64_t *bar, uint32_t &phase, const ChunkParams &p)
{
    warp_arrive(bar);
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
        __nanosleep(128);
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

// A run of consecutive sub-chunks of one chain (one batch row, one head pair).
// Kept small: every warp role holds two of them (this sub-chunk's, the next).
struct Unit {
    int b, h0, nsub, len, start;   // start: first step (sequences are shorter than 2^31)
    int flags;                     // kFirst: begins its chain; kLast: ends it
};
constexpr int kFirst = 1, kLast = 2;

// Range schedule: unit u is step range u / nchains of chain u % nchains (units
// number fewer than 2^31: 32-bit index arithmetic).
__device__ __forceinline__ Unit decode_unit(int u, const ChunkParams &p)
{
    Unit w;
    const int rg = u / p.nchains;
    const int chain = u - rg * p.nchains;
    w.b = chain / p.nhp;
    w.h0 = 2 * (chain - w.b * p.nhp);
    w.start = rg * p.span;
    w.len = min(p.span, (int)(p.L - w.start));
    w.nsub = (w.len + kT - 1) / kT;
    w.flags = (rg == 0 ? kFirst : 0) | (rg == p.nranges - 1 ? kLast : 0);
    return w;
}

// Piece schedule: the chains' sub-chunks, chain after chain, are cut into
// gridDim.x runs of equal length (to one sub-chunk), CTA i taking run i.  A
// run is at least one chain long, so it holds at most: the head of a chain
// that the next CTA finishes, whole chains, and the tail of a chain that the
// previous CTA began.  It takes them in that order, so a head is handed on
// first and a tail is taken up last.  The state crossing the boundary between
// CTAs i and i+1 goes through slot i.  Unit e of this CTA's run (nsub == 0
// past its end).
__device__ __forceinline__ Unit decode_piece(int e, const ChunkParams &p)
{
    Unit w;
    const long long T = p.total_subs, G = gridDim.x, i = blockIdx.x, ns = p.nsub_chain;
    const long long lo = i * T / G, hi = (i + 1) * T / G;
    const int head = hi % ns != 0 ? 1 : 0;
    const int tail = lo % ns != 0 ? 1 : 0;
    const long long f0 = (lo + ns - 1) / ns;
    const int nfull = (int)(hi / ns - f0);
    long long chain, kb, ke;
    if (e < head) {
        chain = hi / ns;
        kb = 0;
        ke = hi - chain * ns;
        w.flags = kFirst;
    } else if (e < head + nfull) {
        chain = f0 + (e - head);
        kb = 0;
        ke = ns;
        w.flags = kFirst | kLast;
    } else if (e < head + nfull + tail) {
        chain = lo / ns;
        kb = lo - chain * ns;
        ke = ns;
        w.flags = kLast;
    } else {
        w.nsub = 0;
        return w;
    }
    w.b = (int)(chain / p.nhp);
    w.h0 = 2 * (int)(chain - (long long)w.b * p.nhp);
    w.start = (int)(kb * kT);
    w.len = (int)(min(ke * kT, p.L) - w.start);
    w.nsub = (int)(ke - kb);
    return w;
}

// Position in this CTA's sequence of sub-chunks: units blockIdx.x,
// blockIdx.x + gridDim.x, ... (range schedule) or units 0, 1, ... of the
// CTA's run (piece schedule), each walked in sub-chunks of kT steps.
struct Cursor {
    int u;
    int k;
    Unit w;
    __device__ __forceinline__ int valid() const { return min(kT, w.len - k * kT); }
    __device__ __forceinline__ long long t0() const { return (long long)w.start + k * kT; }
    __device__ __forceinline__ bool first() const { return (w.flags & kFirst) != 0; }
    __device__ __forceinline__ bool last() const { return (w.flags & kLast) != 0; }
};

template <bool kPieces>
__device__ __forceinline__ bool cursor_load(Cursor &c, const ChunkParams &p)
{
    c.k = 0;
    if constexpr (kPieces) {
        c.w = decode_piece(c.u, p);
        return c.w.nsub > 0;
    }
    if (c.u >= p.nunits)
        return false;
    c.w = decode_unit(c.u, p);
    return true;
}

template <bool kPieces>
__device__ __forceinline__ bool cursor_first(Cursor &c, const ChunkParams &p)
{
    c.u = kPieces ? 0 : (int)blockIdx.x;
    return cursor_load<kPieces>(c, p);
}

template <bool kPieces>
__device__ __forceinline__ bool cursor_next(Cursor &c, const ChunkParams &p)
{
    if (c.k + 1 < c.w.nsub) {
        ++c.k;
        return true;
    }
    c.u += kPieces ? 1 : (int)gridDim.x;
    return cursor_load<kPieces>(c, p);
}

// Handoff slot of the unit's entering and/or end state: chained range schedule,
// one per chain; piece schedule, one per boundary between CTAs (a head hands on
// through this CTA's, a tail takes up through the previous CTA's); split, one
// per unit.
template <bool kPieces>
__device__ __forceinline__ int unit_slot(const Cursor &c, const ChunkParams &p)
{
    if (kPieces)
        return c.first() ? (int)blockIdx.x : (int)blockIdx.x - 1;
    return p.mode == kChained ? c.w.b * p.nhp + (c.w.h0 >> 1) : c.u;
}

// Flag rows (chained only): the one the predecessor publishes, and this unit's.
template <bool kPieces>
__device__ __forceinline__ int wait_row(const Cursor &c, const ChunkParams &p)
{
    return kPieces ? (int)blockIdx.x - 1 : c.u - p.nchains;
}
template <bool kPieces>
__device__ __forceinline__ int post_row_of(const Cursor &c, const ChunkParams &p)
{
    return kPieces ? (int)blockIdx.x : c.u;
}

// SiLU for outputs rounded to bf16: SiLU(v) = h + h tanh(h), h = v / 2, with the
// hardware tanh approximation (the form and the operation order of the library's
// conv kernel, so that the conv mode's x matches its output bit for bit)
__device__ __forceinline__ float silu_bf16_out(float v)
{
    const float h = 0.5f * v;
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(h));
    return fmaf(h, t, h);
}

// conv mode: 4 channels (8 bytes) of the raw input at step t of batch row b,
// channels ch .. ch+3 of xbc: from xbc for t >= 0, else from the carried conv
// state (its row K-1+t), zero where neither has it
__device__ __forceinline__ uint2 conv_input_row4(const ChunkParams &p, int b, long long t, int ch)
{
    if (t >= 0)
        return __ldg(reinterpret_cast<const uint2 *>(p.xbc + ((size_t)b * p.L + t) * p.conv_cc + ch));
    const long long rs = p.conv_k - 1 + t;
    if (p.conv_state && rs >= 0)
        return __ldg(reinterpret_cast<const uint2 *>(p.conv_state + ((size_t)b * (p.conv_k - 1) + rs) * p.conv_cc + ch));
    return make_uint2(0u, 0u);
}

__device__ __forceinline__ void bf16x4_to_f32(const uint2 &u, float (&f)[4])
{
    f[0] = __uint_as_float(u.x << 16);
    f[1] = __uint_as_float(u.x & 0xffff0000u);
    f[2] = __uint_as_float(u.y << 16);
    f[3] = __uint_as_float(u.y & 0xffff0000u);
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

__device__ __forceinline__ uint4 pack8(const uint32_t *v)
{
    uint4 o;
    o.x = pack_bf16x2(__uint_as_float(v[0]), __uint_as_float(v[1]));
    o.y = pack_bf16x2(__uint_as_float(v[2]), __uint_as_float(v[3]));
    o.z = pack_bf16x2(__uint_as_float(v[4]), __uint_as_float(v[5]));
    o.w = pack_bf16x2(__uint_as_float(v[6]), __uint_as_float(v[7]));
    return o;
}

__device__ __forceinline__ uint32_t pack_pair(uint64_t v)
{
    float lo, hi;
    f32x2_split(v, lo, hi);
    return pack_bf16x2(lo, hi);
}

// Largest decay span (log2 units) of one 16-step group for which the factored
// form below is used inside the group; beyond it the direct form is.
constexpr float kSpanMax = 64.f;

// One 16-column group of M for both heads: columns s0 .. s0+15 of row t, from
// the S values sv[0..15], as 8 packed bf16 pairs per head.
//   M[t,s] = S[t,s] exp(cs_t - cs_s) dt_s  (s <= t, else 0),   M[t,t] += D
// (the kernel passes D = 0: it adds D x to the fp32 Y_diag accumulator instead)
// is evaluated as S[t,s] rf colf[s] with the row factor rf = exp(cs_t - cs_e)
// and the column factor colf[s] = exp(cs_e - cs_s) dt_s, e = s0 + 15 the
// group's last step (the caller passes rf and colf + s0).  For rows below the
// group both factors are <= 1.  For a row inside the group rf >= 1 is at most
// exp(span of the group) and colf >= exp(-span) dt, so the product is exact to
// rounding while the span stays below kSpanMax (checked by the caller).
// kMask: some rows are inside or above the group (k = t - s0 < 15): entries
// with s > t are zeroed and D lands on s == t.
// kTrap (the trapezoidal mode): the diagonal entry also gets S[t,t] dc, where
// dc (dc0, dc1 per head) is the diagonal weight of row t minus its input weight.
template <bool kMask, bool kTrap = false>
__device__ __forceinline__ void build_group(const uint32_t (&sv)[16], uint32_t (&m0)[8], uint32_t (&m1)[8], int k,
                                            float rf0, float rf1, const float *colf, float D0, float D1,
                                            float dc0 = 0.f, float dc1 = 0.f)
{
    const uint64_t r0 = f32x2(rf0, rf0), r1 = f32x2(rf1, rf1);
    const uint64_t dd0 = f32x2(D0, D0), dd1 = f32x2(D1, D1);
    const uint64_t cc0 = f32x2(dc0, dc0), cc1 = f32x2(dc1, dc1);
#pragma unroll
    for (int i4 = 0; i4 < 4; ++i4) {
        const float4 c0 = *reinterpret_cast<const float4 *>(colf + 4 * i4);
        const float4 c1 = *reinterpret_cast<const float4 *>(colf + kT + 4 * i4);
        const uint64_t rc0[2] = {mul_f32x2(r0, f32x2(c0.x, c0.y)), mul_f32x2(r0, f32x2(c0.z, c0.w))};
        const uint64_t rc1[2] = {mul_f32x2(r1, f32x2(c1.x, c1.y)), mul_f32x2(r1, f32x2(c1.z, c1.w))};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int i = 4 * i4 + 2 * e;   // columns s0+i, s0+i+1
            float a = __uint_as_float(sv[i]), b = __uint_as_float(sv[i + 1]);
            if (kMask) {
                a = i <= k ? a : 0.f;
                b = i + 1 <= k ? b : 0.f;
            }
            const uint64_t ab = f32x2(a, b);
            uint64_t v0 = mul_f32x2(ab, rc0[e]);
            uint64_t v1 = mul_f32x2(ab, rc1[e]);
            if (kMask) {
                const uint64_t ind = f32x2(i == k ? 1.f : 0.f, i + 1 == k ? 1.f : 0.f);
                if (kTrap) {
                    v0 = fma_f32x2(ind, fma_f32x2(ab, cc0, dd0), v0);
                    v1 = fma_f32x2(ind, fma_f32x2(ab, cc1, dd1), v1);
                } else {
                    v0 = fma_f32x2(ind, dd0, v0);
                    v1 = fma_f32x2(ind, dd1, v1);
                }
            }
            m0[2 * i4 + e] = pack_pair(v0);
            m1[2 * i4 + e] = pack_pair(v1);
        }
    }
}

// The same group in the direct form exp(cs_t - cs_s) dt_s per entry, for a
// group whose decay span is too large for the factored form (rare: kept out
// of line; it reads S from and writes M to tensor memory at `ta` itself).
// dc0, dc1: diagonal correction as in build_group (0 outside the trapezoidal mode).
__device__ __noinline__ void build_group_direct(uint32_t ta, int s0, int t, const float *cs2, const float *dtv,
                                                float D0, float D1, float dc0, float dc1)
{
    uint32_t sv[16], m0[8], m1[8];
    tmem_ld16(ta, sv);
    tmem_wait_ld();
    const float cr0 = cs2[t], cr1 = cs2[kT + t];
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
        float e0[2], e1[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int s = s0 + i + u;
            const float v = __uint_as_float(sv[i + u]);
            const bool keep = s <= t;
            e0[u] = keep ? v * ex2_approx(cr0 - cs2[s]) * dtv[s] : 0.f;
            e1[u] = keep ? v * ex2_approx(cr1 - cs2[kT + s]) * dtv[kT + s] : 0.f;
            if (s == t) {
                e0[u] += fmaf(v, dc0, D0);
                e1[u] += fmaf(v, dc1, D1);
            }
        }
        m0[i >> 1] = pack_bf16x2(e0[0], e0[1]);
        m1[i >> 1] = pack_bf16x2(e1[0], e1[1]);
    }
    tmem_st8(ta, m0);
    tmem_st8(ta + 8, m1);
}

// Trapezoidal mode, per-token values of thread row r of sub-chunk c: dt_t, a_t,
// trap_t, and dt, trap of the next step (0 and 1 past the end of the sequence,
// so that the last step's input weight is its own gamma only).
__device__ __forceinline__ void load_trap_tok(const Cursor &c, int r, int hd, const ChunkParams &p, float (&o)[5])
{
    const long long t = c.t0() + r;
    const size_t idx = ((size_t)c.w.b * p.L + t) * p.H + c.w.h0 + hd;
    o[0] = __ldg(p.tdt + idx);
    o[1] = __ldg(p.ta + idx);
    o[2] = __ldg(p.ttrap + idx);
    const bool more = t + 1 < p.L;
    o[3] = more ? __ldg(p.tdt + idx + p.H) : 0.f;
    o[4] = more ? __ldg(p.ttrap + idx + p.H) : 1.f;
}

// conv mode: the causal conv1d + SiLU over the x tile of sub-chunk jj (cursor
// cur), in place: raw xbc x channels in, the scan's x out.  Run by the 8 warps of
// the decay group (g: the warp's index in it; csync: the phase of its barrier).
// Warp g takes head g >> 2 and rows 32 (g & 3) .. +31; lane l takes 4 channels,
// half (l >> 3) & 1 of the 16-byte chunk l & 7, of the 16 rows from 16 (l >> 4)
// on.  The 16 lanes on one row then cover its 128 bytes once (8-byte accesses
// without bank conflicts), and a lane's 4 taps and bias stay in registers for all
// its rows.  The 3 rows before a lane's first row are read before anyone writes;
// the raw rows 125 .. 127 become the next sub-chunk's halo.  At a unit start the
// weights of the unit's head pair are staged first.  False on abort or timeout.
__device__ __forceinline__ bool conv_x_tile(uint8_t *smem, uint64_t *bars, const ChunkParams &p, const Cursor &cur,
                                            uint32_t jj, int g, int lane, uint32_t &csync)
{
    const int s = jj & 1;
    const int hc = g >> 2, c = lane & 7, h4 = (lane >> 3) & 1;
    const int r0 = 32 * (g & 3) + 16 * (lane >> 4);
    float *cw = reinterpret_cast<float *>(smem + kOffConvW);
    uint8_t *halo = smem + kOffHalo + hc * (3 * 128) + 16 * c + 8 * h4;
    if (cur.k == 0) {   // unit start: this head pair's weights
        for (int i = g * 32 + lane; i < kConvWFloats; i += kGroupWarps * 32) {
            const int hh2 = i / 320, rem = i % 320, cq = rem / 40, k = (rem % 40) / 8, e = rem % 8;
            const int ch = (cur.w.h0 + hh2) * kP + 8 * cq + e;
            float v;
            if (rem % 40 < 32)
                v = k < p.conv_k ? p.conv_w[(size_t)ch * p.conv_k + k] : 0.f;
            else
                v = p.conv_b ? p.conv_b[ch] : 0.f;
            cw[i] = v;
        }
    }
    if (!wait_bar(&bars[BAR_X_FULL + s], (jj >> 1) & 1, p))
        return false;
    uint8_t *xt = smem + kOffX + s * kXStageBytes + hc * kTileBytes + 8 * h4;
    uint2 hal[3];
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        const int rr = r0 - 3 + i;
        if (rr >= 0)
            hal[i] = *reinterpret_cast<const uint2 *>(xt + sw128(rr, c));
        else if (cur.k > 0)
            hal[i] = *reinterpret_cast<const uint2 *>(halo + (rr + 3) * 128);
        else
            hal[i] = conv_input_row4(p, cur.w.b, cur.t0() + rr, (cur.w.h0 + hc) * kP + 8 * c + 4 * h4);
    }
    if (!group_sync(&bars[BAR_CSYNC], csync, p))
        return false;
    {
        // (the group barrier's arrive releases and its wait acquires the weights)
        const float *wc = cw + (hc * 8 + c) * 40 + 4 * h4;
        const float4 w0 = *reinterpret_cast<const float4 *>(wc);
        const float4 w1 = *reinterpret_cast<const float4 *>(wc + 8);
        const float4 w2 = *reinterpret_cast<const float4 *>(wc + 16);
        const float4 w3 = *reinterpret_cast<const float4 *>(wc + 24);
        const float4 bq = *reinterpret_cast<const float4 *>(wc + 32);
        const float W0[4] = {w0.x, w0.y, w0.z, w0.w}, W1[4] = {w1.x, w1.y, w1.z, w1.w};
        const float W2[4] = {w2.x, w2.y, w2.z, w2.w}, W3[4] = {w3.x, w3.y, w3.z, w3.w};
        const float Bq[4] = {bq.x, bq.y, bq.z, bq.w};
        float win[3][4];   // win[i]: the input 3 - i steps back
#pragma unroll
        for (int i = 0; i < 3; ++i)
            bf16x4_to_f32(hal[i], win[i]);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int rr = r0 + i;
            uint2 *cell = reinterpret_cast<uint2 *>(xt + sw128(rr, c));
            const uint2 raw = *cell;
            if (rr >= 125)   // raw rows 125 .. 127: the next sub-chunk's halo
                *reinterpret_cast<uint2 *>(halo + (rr - 125) * 128) = raw;
            float cur4[4], out[4];
            bf16x4_to_f32(raw, cur4);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                float v = fmaf(W0[u], cur4[u], Bq[u]);
                v = fmaf(W1[u], win[2][u], v);
                v = fmaf(W2[u], win[1][u], v);
                v = fmaf(W3[u], win[0][u], v);
                out[u] = silu_bf16_out(v);
            }
            *cell = make_uint2(pack_bf16x2(out[0], out[1]), pack_bf16x2(out[2], out[3]));
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                win[0][u] = win[1][u];
                win[1][u] = win[2][u];
                win[2][u] = cur4[u];
            }
        }
    }
    fence_proxy_async_smem();   // (the MMAs read the tile through the async proxy)
    // the halo rows and every read of this tile's rows are done before the next tile
    return group_sync(&bars[BAR_CSYNC], csync, p);
}

// kPieces: the piece schedule (else the range schedule, or a split pass).
// kLocal: split pass 1, which computes every unit's end state from zero and
//   nothing else (no C loads, no M, no Y MMAs, no y); only the state MMA runs.
// kTrap: the trapezoidal (Mamba-3 SISO) recurrence
//   h_t = alpha_t h_{t-1} + beta_t k_{t-1} v_{t-1}^T + gamma_t k_t v_t^T
// (alpha = exp(a dt), beta = alpha dt (1 - trap), gamma = trap dt) evaluated as
// this kernel's SSD recurrence on h~_t = h_t + (beta_{t+1}/alpha_{t+1}) k_t v_t^T:
// decay alpha_t, input weight w_t = gamma_t + dt_{t+1} (1 - trap_{t+1}) (gamma
// alone at the last step), y_t = q_t h~_t + (D - dt_{t+1} (1 - trap_{t+1}) q_t.k_t) v_t
// (a correction on the diagonal of M), entering state h0 + dt_0 (1 - trap_0) k0 v0^T.
// kFold: split pass 3 with the combine folded in, for few ranges: a unit's
//   entering state is formed at its start from the initial state and the end
//   states and decays its predecessors left in pass 1, by the combine's
//   arithmetic (E_0 = h0 or 0, E_{j+1} = Lambda_j E_j + S_j, in range order).
template <bool kPieces, bool kTrap, bool kLocal, bool kConv = false, bool kFold = false>
__global__ void __launch_bounds__(kThreads, 1)
    ssd_chunk_fused_kernel(const __grid_constant__ Maps maps, const ChunkParams p)
{
    static_assert(!kFold || (!kPieces && !kTrap && !kLocal && !kConv), "the folded combine is split pass 3 only");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBars);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + kOffTmemHolder);
    float *decay_base = reinterpret_cast<float *>(smem + kOffDecay);
    float *wsum = reinterpret_cast<float *>(smem + kOffWsum);
    float *hA2 = reinterpret_cast<float *>(smem + kOffHead);   // -exp(A_log) * log2(e)
    float *hBias = hA2 + kMaxHeads;
    float *hD = hBias + kMaxHeads;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    for (int h = threadIdx.x; h < p.H; h += blockDim.x) {
        if constexpr (!kTrap) {   // the trapezoidal mode has per-token a and dt instead
            hA2[h] = -expf(p.A_log[h]) * 1.4426950408889634f;
            hBias[h] = p.dt_bias[h];
        }
        hD[h] = p.D[h];
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[BAR_BC_FULL + i], 1);
            // the state MMA's commit (B read) and the state warps (their y stores have read the C area)
            mbar_init(&bars[BAR_BC_EMPTY + i], 1 + kGroupWarps);
            mbar_init(&bars[BAR_X_FULL + i], 1);
            mbar_init(&bars[BAR_X_EMPTY + i], 1);
        }
        mbar_init(&bars[BAR_S_DONE], 1);
        mbar_init(&bars[BAR_M_READY], kGroupWarps);
        mbar_init(&bars[BAR_YD_DONE], 1);
        mbar_init(&bars[BAR_XS_READY], kGroupWarps);
        mbar_init(&bars[BAR_YOFF_DONE], 1);
        mbar_init(&bars[BAR_STATE_DONE], 1);
        mbar_init(&bars[BAR_PB_READY], kGroupWarps);
        mbar_init(&bars[BAR_EPI_DONE], kGroupWarps);
        mbar_init(&bars[BAR_DRAIN], 1);
        mbar_init(&bars[BAR_MSYNC], kGroupWarps);
        mbar_init(&bars[BAR_CSYNC], kGroupWarps);
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
        prefetch_tmap(&maps.y);
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
            Cursor cur;
            for (bool has = cursor_first<kPieces>(cur, p); has; has = cursor_next<kPieces>(cur, p), ++j) {
                const int s = j & 1;
                const int t0 = (int)cur.t0();
                if (j >= 2 && !(ok = wait_bar(&bars[BAR_BC_EMPTY + s], ((j >> 1) + 1) & 1, p)))
                    break;
                uint8_t *bc = smem + kOffBC + s * kBCStageBytes;
                const int gc = (cur.w.h0 / p.hpg) * kN;
                // split pass 1 computes end states only: it needs B and x, not C
                constexpr bool with_c = !kLocal;
                mbar_arrive_expect_tx(&bars[BAR_BC_FULL + s], with_c ? kBCStageBytes : 2 * kTileBytes);
                if (with_c) {
                    tma_load_3d(bc, &maps.C, &bars[BAR_BC_FULL + s], gc, t0, cur.w.b, pol_keep);
                    tma_load_3d(bc + kTileBytes, &maps.C, &bars[BAR_BC_FULL + s], gc + 64, t0, cur.w.b, pol_keep);
                }
                tma_load_3d(bc + 2 * kTileBytes, &maps.B, &bars[BAR_BC_FULL + s], gc, t0, cur.w.b, pol_keep);
                tma_load_3d(bc + 3 * kTileBytes, &maps.B, &bars[BAR_BC_FULL + s], gc + 64, t0, cur.w.b, pol_keep);
                last_bc[s] = (int)j;
                // the x stage is free once Y_off(j-1) has read the bf16 P staged in it; in
                // split pass 1 (no P there) once the state MMA of sub-chunk j-2 has read it
                if constexpr (kLocal) {
                    if (j >= 2 && !(ok = wait_bar(&bars[BAR_X_EMPTY + s], ((j >> 1) + 1) & 1, p)))
                        break;
                } else {
                    if (j >= 1 && !(ok = wait_bar(&bars[BAR_X_EMPTY + s], ((j - 1) >> 1) & 1, p)))
                        break;
                }
                uint8_t *xs = smem + kOffX + s * kXStageBytes;
                mbar_arrive_expect_tx(&bars[BAR_X_FULL + s], kXStageBytes);
                tma_load_3d(xs, &maps.x, &bars[BAR_X_FULL + s], cur.w.h0 * kP, t0, cur.w.b, pol_stream);
                tma_load_3d(xs + kTileBytes, &maps.x, &bars[BAR_X_FULL + s], (cur.w.h0 + 1) * kP, t0, cur.w.b,
                            pol_stream);
                last_x[s] = (int)j;
            }
            if (!ok) {
                // every load issued by this thread must land before the CTA exits
                const uint64_t t0 = globaltimer_ns();
                for (int st = 0; st < 2; ++st) {
                    if (last_bc[st] >= 0)
                        while (!mbar_wait_for(&bars[BAR_BC_FULL + st], (last_bc[st] >> 1) & 1, 1000000u) &&
                               globaltimer_ns() - t0 < p.timeout_ns) {
                        }
                    if (last_x[st] >= 0)
                        while (!mbar_wait_for(&bars[BAR_X_FULL + st], (last_x[st] >> 1) & 1, 1000000u) &&
                               globaltimer_ns() - t0 < p.timeout_ns) {
                        }
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA
        // order per sub-chunk j:  Y_diag(j), Y_off(j), S(j+1), state(j).  Split pass 1
        // issues the state MMA alone; the other commits still arrive, so every role
        // keeps its hand-offs
        if (lane == 0) {
            constexpr bool with_y = !kLocal;
            const uint32_t id_S = idesc_bf16_f32(128, 128, 0, 0);      // C (K-major) x B (K-major)
            const uint32_t id_Yd = idesc_bf16_f32(128, 64, 0, 1);      // M (TMEM) x x (MN-major)
            const uint32_t id_Yoff = idesc_bf16_f32(128, 128, 0, 1);   // C (K-major) x P (MN-major)
            const uint32_t id_St = idesc_bf16_f32(128, 128, 1, 1);     // B^T (MN-major) x wx (MN-major)
            auto issue_S = [&](int stage) {
                const uint32_t bc = smem_u32(smem + kOffBC + stage * kBCStageBytes);
                for (int kk = 0; with_y && kk < 8; ++kk) {
                    const uint32_t ko = (kk >> 2) * kTileBytes + (kk & 3) * 32;
                    mma_ss(tmem + kColSM, sdesc_sw128(bc + ko, 16, 1024),
                           sdesc_sw128(bc + 2 * kTileBytes + ko, 16, 1024), id_S, kk > 0);
                }
                mma_commit(&bars[BAR_S_DONE]);
            };
            uint32_t j = 0;
            bool ok = true;
            Cursor cur;
            bool has = cursor_first<kPieces>(cur, p);
            if (has) {
                if ((ok = wait_bar(&bars[BAR_BC_FULL + 0], 0, p))) {
                    tc_fence_after();
                    issue_S(0);
                }
            }
            while (ok && has) {
                Cursor nxt = cur;
                const bool has_next = cursor_next<kPieces>(nxt, p);
                const int s = j & 1;
                const uint32_t par = j & 1;
                const uint32_t bc = smem_u32(smem + kOffBC + s * kBCStageBytes);
                const uint32_t cA = bc, bB = bc + 2 * kTileBytes;
                const uint32_t xs = smem_u32(smem + kOffX + s * kXStageBytes);
                const uint32_t pb = smem_u32(smem + kOffX + (s ^ 1) * kXStageBytes);
                auto issue_Yoff = [&]() {
                    tc_fence_after();
                    for (int kk = 0; with_y && kk < 8; ++kk) {
                        const uint32_t ko = (kk >> 2) * kTileBytes + (kk & 3) * 32;
                        mma_ss(tmem + kColYo, sdesc_sw128(cA + ko, 16, 1024), sdesc_sw128(pb + kk * 2048, kTileBytes, 1024),
                               id_Yoff, kk > 0);
                    }
                    mma_commit(&bars[BAR_YOFF_DONE]);
                    if constexpr (!kLocal)
                        mma_commit(&bars[BAR_X_EMPTY + (s ^ 1)]);
                };
                // Bounded poll loop: calls step(progressed) until it returns true, sleeping
                // after the calls that issued nothing; false on abort or timeout
                auto poll = [&](auto &&step) -> bool {
                    const uint64_t tw = globaltimer_ns();
                    uint32_t spins = 0;
                    for (;;) {
                        bool progressed = false;
                        if (step(progressed))
                            return true;
                        if (progressed)
                            continue;
                        __nanosleep(32);
                        if ((++spins & 255u) == 0) {
                            if (aborted(p))
                                return false;
                            if (globaltimer_ns() - tw > p.timeout_ns) {
                                raise_timeout(p);
                                return false;
                            }
                        }
                    }
                };
                bool yo_done = false;
                // Y_diag[h] = M[h] x[h]
                if (j >= 1 && !(ok = wait_bar(&bars[BAR_EPI_DONE], (j - 1) & 1, p)))
                    break;
                if constexpr (kConv) {
                    // conv mode: Y_off(j) goes ahead of Y_diag(j) when its operand is ready
                    // first.  The x stage it frees then takes the next raw tile, which the
                    // decay group convolves once it has published M(j).
                    // (M_READY(j) also says that the decay group has convolved x(j))
                    if (!(ok = poll([&](bool &progressed) {
                              if (!yo_done && mbar_poll(&bars[BAR_PB_READY], par)) {
                                  issue_Yoff();
                                  yo_done = progressed = true;
                              }
                              return mbar_poll(&bars[BAR_M_READY], par);
                          })))
                        break;
                } else if (!(ok = wait_bar(&bars[BAR_X_FULL + s], (j >> 1) & 1, p)) ||
                           !(ok = wait_bar(&bars[BAR_M_READY], par, p))) {
                    break;
                }
                tc_fence_after();
                for (int h = 0; with_y && h < 2; ++h)
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ts(tmem + kColYd + 64 * h, tmem + kColSM + 16 * kk + 8 * h,
                               sdesc_sw128(xs + h * kTileBytes + kk * 2048, kTileBytes, 1024), id_Yd, kk > 0);
                mma_commit(&bars[BAR_YD_DONE]);
                // Y_off(j) = C P (P as bf16 in the other x stage) and S(j+1), in place of
                // M once Y_diag has read it: whichever is ready first goes first, S first
                // when both are (the next M build waits on it)
                {
                    bool s_done = !has_next;
                    if (!(ok = poll([&](bool &progressed) {
                              // (split pass 1 has no S, so no wait for the next B/C tile here: the
                              // state MMA waits for its own tile instead, and two loads stay in flight)
                              if (!s_done &&
                                  (!with_y || mbar_poll(&bars[BAR_BC_FULL + (s ^ 1)], ((j + 1) >> 1) & 1)) &&
                                  mbar_poll(&bars[BAR_YD_DONE], par)) {
                                  tc_fence_after();
                                  issue_S(s ^ 1);
                                  s_done = progressed = true;
                              }
                              if (!yo_done && mbar_poll(&bars[BAR_PB_READY], par)) {
                                  issue_Yoff();
                                  yo_done = progressed = true;
                              }
                              return yo_done && s_done;
                          })))
                        break;
                }
                // P += B^T (w o x)   (P already rescaled by the state group)
                if (!(ok = wait_bar(&bars[BAR_XS_READY], par, p)) ||
                    (!with_y && !(ok = wait_bar(&bars[BAR_BC_FULL + s], (j >> 1) & 1, p))))
                    break;
                tc_fence_after();
                for (int kk = 0; kk < 8; ++kk)
                    mma_ss(tmem + kColP, sdesc_sw128(bB + kk * 2048, kTileBytes, 1024),
                           sdesc_sw128(xs + kk * 2048, kTileBytes, 1024), id_St, 1);
                mma_commit(&bars[BAR_STATE_DONE]);
                mma_commit(&bars[BAR_BC_EMPTY + s]);
                if constexpr (kLocal)
                    mma_commit(&bars[BAR_X_EMPTY + s]);   // (split pass 1: see the producer)
                cur = nxt;
                has = has_next;
                ++j;
            }
            // make sure no MMA is in flight before tensor memory is released
            mma_commit(&bars[BAR_DRAIN]);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_wait_for(&bars[BAR_DRAIN], 0, 1000000u) && globaltimer_ns() - t0 < p.timeout_ns) {
            }
        }
    } else if (warp < kStateWarp0) {
        // ------------------------------------------------------------ decay group
        // per sub-chunk j: dt and the local cumulative sum of dt*A (thread: step r,
        // head hd), decay factors for both groups, then M from S (thread: row r,
        // both heads).  Conv mode: once M(j) is published the group computes the
        // decay factors of sub-chunk j+1 and applies the conv to x(j+1), so that
        // M_READY(j+1) also says that x(j+1) holds the scan's input.
        const int q = warp & 3;        // TMEM lane quarter
        const int hd = warp >> 2;      // head (decay) / column-group parity (M)
        const int r = q * 32 + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
        uint32_t msync = 0, csync = 0;
        Cursor cur;
        bool has = cursor_first<kPieces>(cur, p);
        float dt_raw = 0.f;
        float tq[5] = {0.f, 0.f, 0.f, 0.f, 0.f};   // trapezoidal mode: see load_trap_tok
        if (has && r < cur.valid()) {
            if constexpr (kTrap)
                load_trap_tok(cur, r, hd, p, tq);
            else
                dt_raw = __ldg(p.dt_raw + ((size_t)cur.w.b * p.L + cur.t0() + r) * p.H + cur.w.h0 + hd);
        }
        // decay factors of sub-chunk jj (cursor c; dt_raw dr, trapezoidal tokens tv) into
        // buffer jj % 3; false on abort or timeout
        auto prep = [&](const Cursor &c, uint32_t jj, float dr, const float (&tv)[5]) -> bool {
            const int hh = c.w.h0 + hd;
            float *dk = decay_base + (jj % 3) * kDecayFloats;
            float *cs2 = dk, *dtv = dk + 2 * kT, *colf = dk + 4 * kT, *ecs = dk + 6 * kT, *wsc = dk + 8 * kT,
                  *dtot = dk + 10 * kT;
            // log2 decay l and input weight wgt of this step; dcv: diagonal weight minus wgt
            float l, wgt, dcv = 0.f;
            if constexpr (kTrap) {
                const float carried = tv[3] * (1.f - tv[4]);   // dt_{t+1} (1 - trap_{t+1})
                l = tv[1] * tv[0] * 1.4426950408889634f;
                wgt = fmaf(tv[2], tv[0], carried);
                dcv = -carried;
            } else {
                float dt = 0.f;
                if (r < c.valid())
                    dt = softplus_f32(dr + hBias[hh]);
                l = dt * hA2[hh];
                wgt = dt;
            }
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float nb = __shfl_up_sync(0xffffffffu, l, o);
                if (lane >= o)
                    l += nb;
            }
            if (lane == 31)
                wsum[hd * 4 + q] = l;
            if (!group_sync(&bars[BAR_MSYNC], msync, p))
                return false;
            float pre = 0.f, tot = 0.f;
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
                const float v = wsum[hd * 4 + qq];
                pre += qq < q ? v : 0.f;
                tot += v;
            }
            l += pre;
            const float l_end = __shfl_sync(0xffffffffu, l, lane | 15);   // cs at the end of this 16-step group
            cs2[hd * kT + r] = l;
            dtv[hd * kT + r] = wgt;
            colf[hd * kT + r] = ex2_approx(l_end - l) * wgt;
            ecs[hd * kT + r] = ex2_approx(l);                 // exp(cs_t), scales C P
            wsc[hd * kT + r] = ex2_approx(tot - l) * wgt;     // state input weight
            if constexpr (kTrap)
                dk[10 * kT + 4 + hd * kT + r] = dcv;
            if (r == 0)
                dtot[hd] = ex2_approx(tot);                   // state decay over the sub-chunk
            return group_sync(&bars[BAR_MSYNC], msync, p);
        };
        if constexpr (kConv) {
            if (has && !(prep(cur, 0, dt_raw, tq) && conv_x_tile(smem, bars, p, cur, 0, warp, lane, csync)))
                has = false;
        }
        for (uint32_t j = 0; has; ++j) {
            Cursor nxt = cur;
            const bool has_next = cursor_next<kPieces>(nxt, p);
            float dt_next = 0.f;   // issued one sub-chunk ahead
            float tn[5] = {0.f, 0.f, 0.f, 0.f, 0.f};
            if (has_next && r < nxt.valid()) {
                if constexpr (kTrap)
                    load_trap_tok(nxt, r, hd, p, tn);
                else
                    dt_next = __ldg(p.dt_raw + ((size_t)nxt.w.b * p.L + nxt.t0() + r) * p.H + nxt.w.h0 + hd);
            }
            if constexpr (!kConv) {
                if (!prep(cur, j, dt_raw, tq))
                    break;
            }
            float *dk = decay_base + (j % 3) * kDecayFloats;
            const float *cs2 = dk, *dtv = dk + 2 * kT, *colf = dk + 4 * kT;
            // ---- M from S, in place, 16 columns at a time (row r, both heads).  The
            //      rows 32q .. 32q+31 of this lane quarter lie below every column
            //      group G < 2q, hold the diagonal in G = 2q, 2q+1 and lie above
            //      G > 2q+1 (M = 0 there); the quarter's two warps take alternate groups.
            if (!wait_bar(&bars[BAR_S_DONE], j & 1, p))
                break;
            tc_fence_after();
            if constexpr (!kLocal) {   // split pass 1 has no y, so no M
                // (D x is added in fp32 to Y_diag by the state group, not through M)
                const float D0 = 0.f, D1 = 0.f;
                const float ct0 = cs2[r], ct1 = cs2[kT + r];
                const float dc0 = kTrap ? dk[10 * kT + 4 + r] : 0.f, dc1 = kTrap ? dk[11 * kT + 4 + r] : 0.f;
#pragma unroll 1
                for (int G = hd; G < 8; G += 2) {
                    const uint32_t ta = tmem + lane_addr + kColSM + 16 * G;
                    uint32_t m0[8], m1[8];
                    const int s0 = 16 * G;
                    if (G <= 2 * q + 1 && G >= 2 * q &&
                        !(cs2[s0] - cs2[s0 + 15] <= kSpanMax && cs2[kT + s0] - cs2[kT + s0 + 15] <= kSpanMax)) {
                        build_group_direct(ta, s0, r, cs2, dtv, D0, D1, dc0, dc1);
                        continue;
                    }
                    if (G > 2 * q + 1) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            m0[i] = 0u;
                            m1[i] = 0u;
                        }
                    } else {
                        uint32_t sv[16];
                        tmem_ld16(ta, sv);
                        const float e0 = cs2[s0 + 15], e1 = cs2[kT + s0 + 15];
                        const float rf0 = ex2_approx(fminf(ct0 - e0, kSpanMax));
                        const float rf1 = ex2_approx(fminf(ct1 - e1, kSpanMax));
                        tmem_wait_ld();
                        if (G < 2 * q)
                            build_group<false>(sv, m0, m1, 0, rf0, rf1, colf + s0, 0.f, 0.f);
                        else
                            build_group<true, kTrap>(sv, m0, m1, r - s0, rf0, rf1, colf + s0, D0, D1, dc0, dc1);
                    }
                    tmem_st8(ta, m0);
                    tmem_st8(ta + 8, m1);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            // M(j) is published only after the state group has passed its wait on
            // M(j-1) (it signals XS_READY(j-1) after that wait), so M_READY never
            // runs two phases ahead of that group's parity wait
            if (j >= 1 && !wait_bar(&bars[BAR_XS_READY], (j - 1) & 1, p))
                break;
            warp_arrive(&bars[BAR_M_READY]);
            if constexpr (kConv) {
                if (has_next && !(prep(nxt, j + 1, dt_next, tn) &&
                                  conv_x_tile(smem, bars, p, nxt, j + 1, warp, lane, csync)))
                    break;
            }
            cur = nxt;
            has = has_next;
            dt_raw = dt_next;
#pragma unroll
            for (int i = 0; i < 5; ++i)
                tq[i] = tn[i];
        }
    } else if (warp < kProducerWarp) {
        // ------------------------------------------------------------ state group
        // per sub-chunk j (thread: row r, head hf):
        //   [carried-in state](j) at a unit start, [x <- w o x, P <- dtot P](j),
        //   [y](j), [state handoff or bf16 P](j)
        const int sw = warp - kStateWarp0;   // 0..7
        const int q = warp & 3;              // TMEM lane quarter
        const int hf = sw >> 2;              // this thread's head
        const int r = q * 32 + lane;         // row: token t, or state row n
        const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
        const uint32_t ta = tmem + lane_addr + kColP + hf * 64;
        float unit_decay = 1.f;
        bool ok = true;
        Cursor cur;
        bool has = cursor_first<kPieces>(cur, p);
        for (uint32_t j = 0; ok && has; ++j) {
            Cursor nxt = cur;
            const bool has_next = cursor_next<kPieces>(nxt, p);
            const int s = j & 1;
            const uint32_t par = j & 1;
            const int hh = cur.w.h0 + hf;
            if (cur.k == 0) {
                if (p.mode == kChained && p.diag_stall && cur.first()) {
                    // diagnostic: a handoff that never comes (the word stays 0, never the epoch)
                    bool okf = true;
                    if (lane == 0)
                        okf = wait_flag(p.abort_word + 8, p);
                    if (!(ok = __shfl_sync(0xffffffffu, okf ? 1 : 0, 0) != 0))
                        break;
                }
                // ---- carried-in state at a unit start: TMEM (fp32) and the bf16 operand of
                //      C P in x stage (j-1)&1
                if (p.mode == kChained && !cur.first()) {
                    // rows n of this warp were written by the same warp of the predecessor unit
                    bool okf = true;
                    if (lane == 0)
                        okf = wait_flag(p.flags + (size_t)wait_row<kPieces>(cur, p) * kGroupWarps + sw, p);
                    if (!(ok = __shfl_sync(0xffffffffu, okf ? 1 : 0, 0) != 0))
                        break;
                }
                uint8_t *pb = smem + kOffX + (s ^ 1) * kXStageBytes + hf * kTileBytes;
                // chained: the slot the predecessor filled; split pass 3: this unit's own
                // slot; split pass 1 starts every unit from zero (the combine adds the
                // initial state), except in the trapezoidal mode, where it starts each
                // chain's first unit from the chain's entering state (the initial state
                // and the carried k0 v0^T term) and the combine starts from zero
                // all 64 loads of the row are issued before the first use (one round trip)
                const size_t slot_of = (size_t)unit_slot<kPieces>(cur, p);
                const bool chain_entry = cur.first() && (kTrap || p.mode != kSplitLocal);
                if constexpr (!kPieces) {
                    // The initial state of this CTA's next unit, when that unit starts its
                    // chain, into L2 ahead of its loads (64 KB, contiguous for the head
                    // pair).  Handoff slots are not prefetched: a chained predecessor may
                    // still be running, and split pass 3 measured no gain.
                    if (sw == 0 && lane == 0 && p.init_state && p.mode != kSplitLocal &&
                        cur.u + (long long)gridDim.x < p.nunits) {
                        const Unit w2 = decode_unit(cur.u + (int)gridDim.x, p);
                        if (w2.flags & kFirst) {
                            const float *nxt_state = p.init_state + ((size_t)w2.b * p.H + w2.h0) * (size_t)(kP * kN);
                            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(nxt_state),
                                         "r"((uint32_t)(2 * kP * kN * sizeof(float)))
                                         : "memory");
                        }
                    }
                }
                uint32_t v[2][32];
                // split pass 3 is launched as a programmatic dependent of the combine
                // (of pass 1 with the combine folded in): its other roles start on the
                // inputs, and this group waits for the launch before it here (a no-op
                // once passed)
                if (p.mode == kSplitEntering)
                    asm volatile("griddepcontrol.wait;" ::: "memory");
                if (kFold && !cur.first()) {
                    // E_0: the initial state (or 0), then each predecessor's end state S_j and
                    // decay Lambda_j from pass 1, half a row (8 float4) of S_j at a time
                    if (p.init_state) {
                        const float *src = p.init_state + ((size_t)cur.w.b * p.H + hh) * (size_t)(kP * kN) + r;
#pragma unroll
                        for (int i = 0; i < 64; ++i)
                            v[i >> 5][i & 31] = __float_as_uint(__ldg(src + (size_t)i * kN));
                    } else {
#pragma unroll
                        for (int i = 0; i < 64; ++i)
                            v[i >> 5][i & 31] = 0u;
                    }
                    const int rg = cur.u / p.nchains, chain = cur.u - rg * p.nchains;
                    for (int jj = 0; jj < rg; ++jj) {
                        const size_t uj = (size_t)jj * p.nchains + chain;
                        const float lam = __ldcg(p.unit_decay + uj * 2 + hf);
                        const float4 *src = reinterpret_cast<const float4 *>(p.slots) + (uj * 2 + hf) * 16 * kN + r;
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            float4 sv[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                sv[i] = __ldcg(src + (size_t)(8 * half + i) * kN);
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                uint32_t *e = &v[half][4 * i];
                                e[0] = __float_as_uint(fmaf(lam, __uint_as_float(e[0]), sv[i].x));
                                e[1] = __float_as_uint(fmaf(lam, __uint_as_float(e[1]), sv[i].y));
                                e[2] = __float_as_uint(fmaf(lam, __uint_as_float(e[2]), sv[i].z));
                                e[3] = __float_as_uint(fmaf(lam, __uint_as_float(e[3]), sv[i].w));
                            }
                        }
                    }
                } else if (!cur.first() && p.mode != kSplitLocal) {
                    const float4 *src = reinterpret_cast<const float4 *>(p.slots) + (slot_of * 2 + hf) * 16 * kN + r;
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float4 f = __ldcg(src + (size_t)i * kN);
                        v[i >> 3][4 * (i & 7) + 0] = __float_as_uint(f.x);
                        v[i >> 3][4 * (i & 7) + 1] = __float_as_uint(f.y);
                        v[i >> 3][4 * (i & 7) + 2] = __float_as_uint(f.z);
                        v[i >> 3][4 * (i & 7) + 3] = __float_as_uint(f.w);
                    }
                } else if (p.init_state && chain_entry) {
                    const float *src = p.init_state + ((size_t)cur.w.b * p.H + hh) * (size_t)(kP * kN) + r;
#pragma unroll
                    for (int i = 0; i < 64; ++i)
                        v[i >> 5][i & 31] = __float_as_uint(__ldg(src + (size_t)i * kN));
                } else {
#pragma unroll
                    for (int i = 0; i < 64; ++i)
                        v[i >> 5][i & 31] = 0u;
                }
                if constexpr (kTrap) {
                    // the chain's first step also takes the carried k0 v0^T, weighted
                    // dt_0 (1 - trap_0) before the decay (see the kernel's comment)
                    if (chain_entry && p.k0 && p.v0) {
                        const size_t i0 = (size_t)cur.w.b * p.L * p.H + hh;   // step 0
                        const float c = __ldg(p.tdt + i0) * (1.f - __ldg(p.ttrap + i0));
                        const float ck = c * __bfloat162float(p.k0[((size_t)cur.w.b * p.H + hh) * kN + r]);
                        const __nv_bfloat16 *v0 = p.v0 + ((size_t)cur.w.b * p.H + hh) * kP;
#pragma unroll
                        for (int i = 0; i < 64; ++i)
                            v[i >> 5][i & 31] = __float_as_uint(
                                fmaf(ck, __bfloat162float(v0[i]), __uint_as_float(v[i >> 5][i & 31])));
                    }
                }
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    tmem_st32(ta + 32 * half, v[half]);
                    if constexpr (!kLocal) {   // (split pass 1 has no C P; x(j+1) may be landing there)
#pragma unroll
                        for (int c8 = 0; c8 < 4; ++c8)
                            *reinterpret_cast<uint4 *>(pb + sw128(r, 4 * half + c8)) = pack8(v[half] + 8 * c8);
                    }
                }
                tmem_wait_st();
                fence_proxy_async_smem();
                tc_fence_before();
                warp_arrive(&bars[BAR_PB_READY]);
            }
            // ---- x <- w o x in place (row r, head hf); P <- dtot P
            if (!(ok = wait_bar(&bars[BAR_M_READY], par, p)) || !(ok = wait_bar(&bars[BAR_YD_DONE], par, p)))
                break;
            // split pass 1 issues no Y_diag MMA to read x first: wait for its load here
            if (kLocal && !(ok = wait_bar(&bars[BAR_X_FULL + s], (j >> 1) & 1, p)))
                break;
            tc_fence_after();
            const float *dk = decay_base + (j % 3) * kDecayFloats;
            const float ecs = dk[6 * kT + hf * kT + r];
            const float wsc = dk[8 * kT + hf * kT + r];
            const float dtot = dk[10 * kT + hf];
            unit_decay = (cur.k == 0 ? 1.f : unit_decay) * dtot;   // decay of the state over the unit so far
            {
                uint8_t *xrow = smem + kOffX + s * kXStageBytes + hf * kTileBytes + r * 128;
                const uint32_t w2 = pack_bf16x2(wsc, wsc);
                const float Dh = hD[hh];
                // The skip term D x goes into the fp32 Y_diag accumulator from the row of x
                // as loaded (before it is scaled), half a row (32 channels, one TMEM round
                // trip) at a time; then the row is scaled in place for the state MMA.  Chunks
                // are visited in swizzled order: 8 consecutive rows hit 8 distinct banks.
#pragma unroll 1
                for (int hx = 0; hx < 2; ++hx) {
                    uint4 v4[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        v4[i] = *reinterpret_cast<const uint4 *>(xrow + ((4 * hx + i) ^ (r & 7)) * 16);
                    if constexpr (!kLocal) {
                        const uint32_t tcol = tmem + lane_addr + kColYd + hf * 64 + 32 * hx;
                        uint32_t yd[32];
                        tmem_ld32(tcol, yd);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint32_t xw[4] = {v4[i].x, v4[i].y, v4[i].z, v4[i].w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float lo = __uint_as_float(xw[e] << 16), hi = __uint_as_float(xw[e] & 0xffff0000u);
                                yd[8 * i + 2 * e] = __float_as_uint(fmaf(Dh, lo, __uint_as_float(yd[8 * i + 2 * e])));
                                yd[8 * i + 2 * e + 1] =
                                    __float_as_uint(fmaf(Dh, hi, __uint_as_float(yd[8 * i + 2 * e + 1])));
                            }
                        }
                        tmem_st32(tcol, yd);
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint4 o = v4[i];
                        o.x = mul_bf16x2(o.x, w2);
                        o.y = mul_bf16x2(o.y, w2);
                        o.z = mul_bf16x2(o.z, w2);
                        o.w = mul_bf16x2(o.w, w2);
                        *reinterpret_cast<uint4 *>(xrow + ((4 * hx + i) ^ (r & 7)) * 16) = o;
                    }
                }
                for (int half = 0; half < 2; ++half) {
                    uint32_t v[32];
                    tmem_ld32(ta + 32 * half, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        v[i] = __float_as_uint(__uint_as_float(v[i]) * dtot);
                    tmem_st32(ta + 32 * half, v);
                }
                tmem_wait_st();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            warp_arrive(&bars[BAR_XS_READY]);
            // ---- y = Y_diag + exp(cs_t) Y_off   (TMEM lane r = step r, head hf).  Each warp
            //      stages its 32 rows in its own 4 KB of the C area of this sub-chunk's B/C
            //      stage (C is dead after Y_off) and stores them with one TMA store; the
            //      warp releases the C area once that store has read it
            if (!(ok = wait_bar(&bars[BAR_YOFF_DONE], par, p)))
                break;
            tc_fence_after();
            if constexpr (!kLocal) {
                uint8_t *stg = smem + kOffBC + s * kBCStageBytes + sw * 4096;   // this warp's 32 rows
                for (int half = 0; half < 2; ++half) {
                    uint32_t yd[32], yo[32];
                    tmem_ld32(tmem + lane_addr + kColYd + hf * 64 + 32 * half, yd);
                    tmem_ld32(tmem + lane_addr + kColYo + hf * 64 + 32 * half, yo);
                    tmem_wait_ld();
                    if (half == 1) {
                        tc_fence_before();
                        warp_arrive(&bars[BAR_EPI_DONE]);
                    }
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8) {
                        uint4 o;
                        uint32_t *ov = reinterpret_cast<uint32_t *>(&o);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int i = c8 * 8 + 2 * e;
                            ov[e] = pack_bf16x2(fmaf(ecs, __uint_as_float(yo[i]), __uint_as_float(yd[i])),
                                                fmaf(ecs, __uint_as_float(yo[i + 1]), __uint_as_float(yd[i + 1])));
                        }
                        *reinterpret_cast<uint4 *>(stg + sw128(lane, 4 * half + c8)) = o;
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && 32 * q < cur.valid()) {
                    tma_store_3d(&maps.y, stg, hh * kP, (int)cur.t0() + 32 * q, cur.w.b);
                    bulk_commit_group();
                }
            } else {
                // split pass 1 has no y: only the hand-off of the TMEM columns
                tc_fence_before();
                warp_arrive(&bars[BAR_EPI_DONE]);
            }
            // ---- carried state after sub-chunk j
            if (!(ok = wait_bar(&bars[BAR_STATE_DONE], par, p)))
                break;
            tc_fence_after();
            if (cur.k == cur.w.nsub - 1) {
                // end of the unit: hand the state to the next unit of this chain, or
                // write the final state; split pass 1 stores every unit's end state and
                // total decay in its own slot
                const bool to_slot = p.mode == kSplitLocal || (p.mode == kChained && !cur.last());
                if (to_slot) {
                    // slot layout [slot][head][16-byte chunk c][row n]: a warp writes 512
                    // contiguous bytes per chunk
                    const size_t slot_of = (size_t)unit_slot<kPieces>(cur, p);
                    float4 *dst = reinterpret_cast<float4 *>(p.slots) + (slot_of * 2 + hf) * 16 * kN + r;
                    for (int half = 0; half < 2; ++half) {
                        uint32_t v[32];
                        tmem_ld32(ta + 32 * half, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            __stcg(dst + (size_t)(8 * half + i) * kN,
                                   make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                               __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3])));
                    }
                    if (p.mode == kSplitLocal) {
                        if (q == 0 && lane == 0)
                            p.unit_decay[(size_t)cur.u * 2 + hf] = unit_decay;
                    } else {
                        __syncwarp();
                        if (lane == 0) {
                            __threadfence();
                            st_release_u64(p.flags + (size_t)post_row_of<kPieces>(cur, p) * kGroupWarps + sw, p.epoch);
                        }
                    }
                } else if (p.final_state && cur.last()) {
                    float *dst = p.final_state + ((size_t)cur.w.b * p.H + hh) * (size_t)(kP * kN) + r;
                    for (int half = 0; half < 2; ++half) {
                        uint32_t v[32];
                        tmem_ld32(ta + 32 * half, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            dst[(size_t)(32 * half + i) * kN] = __uint_as_float(v[i]);
                    }
                }
                tc_fence_before();
            } else {
                // bf16 copy of P for the next sub-chunk's C P, in this sub-chunk's x stage
                uint8_t *pb = smem + kOffX + s * kXStageBytes + hf * kTileBytes;
                for (int half = 0; half < 2 && !kLocal; ++half) {   // pass 1: no C P
                    uint32_t v[32];
                    tmem_ld32(ta + 32 * half, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8)
                        *reinterpret_cast<uint4 *>(pb + sw128(r, 4 * half + c8)) = pack8(v + 8 * c8);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                warp_arrive(&bars[BAR_PB_READY]);
            }
            if (lane == 0)
                bulk_wait_read_all();
            warp_arrive(&bars[BAR_BC_EMPTY + s]);
            cur = nxt;
            has = has_next;
        }
        if (lane == 0)
            bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp)
        tmem_dealloc(tmem, 512);
}

// Entering states of the split evaluation, between its two passes.  For each
// chain, range by range: E_0 = the initial state (or 0) and
// E_{k+1} = Lambda_k E_k + S_k, where S_k is the end state of the chain's unit k
// started from zero and Lambda_k = exp(sum of dt A over that unit) (the linear
// recurrence between chunks, applied to whole unit ranges).  E_k replaces S_k in
// unit k's slot for k >= 1.  One thread per (chain, head, 4 channels, state row).
__global__ void __launch_bounds__(256) ssd_split_combine_kernel(float *slots, const float *unit_decay,
                                                                const float *init_state, int nchains,
                                                                int nranges, int nhp, int H)
{
    constexpr int kPerChain = 2 * 16 * kN;   // float4 per slot
    // launched as a programmatic dependent of pass 1: its slots and decays are
    // complete and visible after this wait.  (No early trigger for pass 3: its
    // CTAs, resident beside this grid's, measured slower on the 64k sequences.)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (tid >= (long long)nchains * kPerChain)
        return;
    const int chain = (int)(tid / kPerChain);
    const int e = (int)(tid % kPerChain);   // (hf * 16 + c) * N + n
    const int hf = e / (16 * kN), c = (e / kN) % 16, n = e % kN;
    const int b = chain / nhp, h = 2 * (chain % nhp) + hf;
    float4 E = make_float4(0.f, 0.f, 0.f, 0.f);
    if (init_state) {
        const float *src = init_state + ((size_t)b * H + h) * (size_t)(kP * kN) + (size_t)(4 * c) * kN + n;
        E = make_float4(src[0], src[kN], src[2 * kN], src[3 * kN]);
    }
    float4 *sl = reinterpret_cast<float4 *>(slots);
    float4 S = __ldcg(sl + (size_t)chain * kPerChain + e);   // unit (range 0, chain)
    // The end states and decays of the next kBatch units are all loaded before the
    // first of them is replaced, so the chain of ranges costs one memory round trip
    // per batch rather than one per range.
    constexpr int kBatch = 8;
    for (int k0 = 0; k0 + 1 < nranges; k0 += kBatch) {
        float4 nx[kBatch];
        float lam[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int k = k0 + i;
            if (k + 1 < nranges) {
                const size_t u = (size_t)k * nchains + chain;
                lam[i] = __ldcg(unit_decay + u * 2 + hf);
                nx[i] = __ldcg(sl + (u + nchains) * kPerChain + e);   // the next unit's own end state
            }
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int k = k0 + i;
            if (k + 1 < nranges) {
                const float l = lam[i];
                E = make_float4(fmaf(l, E.x, S.x), fmaf(l, E.y, S.y), fmaf(l, E.z, S.z), fmaf(l, E.w, S.w));
                __stcg(sl + ((size_t)(k + 1) * nchains + chain) * kPerChain + e, E);
                S = nx[i];
            }
        }
    }
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

int sm_count()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return sms;
}

struct Geometry {
    long long nchunks, nchains, chunks_per_unit, nranges, nunits, grid;
    long long seqlen, span;   // steps per unit: chunks_per_unit chunks, or (split) whole sub-chunks
    bool split;    // two passes with a combine in between, instead of chained units
    bool pieces;   // chained, one run of equal length per CTA (see decode_piece)
    long long nsub_chain, total_subs;
    size_t flags_off, slot_off, decay_off, total;
};

// Candidate chunks-per-unit values: 1, 2, 3, 4, 8, 16, ... and all chunks.
int unit_candidates(long long nchunks, long long *cand)
{
    int nc = 0;
    for (long long R = 1; R < nchunks && nc < 62; R = (R < 4 ? R + 1 : R * 2))
        cand[nc++] = R;
    cand[nc++] = nchunks;
    return nc;
}

// Estimated time (in 128-step sub-chunk times) of the chained schedule with R
// chunks per unit: ceil(units / grid) rounds of units of R chunks, each unit
// boundary costing about one sub-chunk of handoff latency, and never less than
// one chain's ranges run one after another.
double chained_estimate(long long R, long long nchunks, long long nchains, int Q, long long grid)
{
    const double subs_per_chunk = (double)Q / kT;
    const long long ranges = (nchunks + R - 1) / R;
    const long long rounds = (ranges * nchains + grid - 1) / grid;
    const double unit_time = R * subs_per_chunk + 1.0;
    return std::max(rounds * unit_time, ranges * unit_time);
}

// Estimated time of the split schedule with units of `len` blocks of
// `subs_per_block` sub-chunks each (nblocks blocks per chain): two passes over
// independent units (no handoff wait, about half a sub-chunk to refill the
// pipeline per unit), of which pass 1 (end states only: B and x loads and the
// state MMA) measured about half as long as pass 3; then the combine, whose
// batched loads stream every unit's state (64 KB) in and out at about 2 ns per
// unit (in sub-chunk times of about 3 us), and about one sub-chunk for the two
// extra launches.
double split_estimate(long long len, long long nblocks, long long nchains, double subs_per_block, long long grid)
{
    const long long ranges = (nblocks + len - 1) / len;
    const long long units = ranges * nchains;
    const long long rounds = (units + grid - 1) / grid;
    const double pass = rounds * (len * subs_per_block + 0.5);
    const double combine = units * 0.002 + 1.0;
    return 1.5 * pass + combine;
}

void layout(Geometry &g, long long grid_p, int sms);

Geometry geometry(const ScanArgs &a)
{
    Geometry g;
    g.seqlen = a.seqlen;
    g.nchunks = (a.seqlen + a.chunk - 1) / a.chunk;
    g.nchains = a.batch * (a.nheads / 2);
    g.nsub_chain = (a.seqlen + kT - 1) / kT;
    g.total_subs = g.nsub_chain * g.nchains;
    const int sms = std::max(1, sm_count());
    long long cand[64];
    const int nc = unit_candidates(g.nchunks, cand);
    double best = 1e300;
    g.chunks_per_unit = 1;
    for (int i = 0; i < nc; ++i) {
        const double est = chained_estimate(cand[i], g.nchunks, g.nchains, a.chunk, sms);
        if (est < best * 0.999) {
            best = est;
            g.chunks_per_unit = cand[i];
        }
    }
    // piece schedule: every run must hold at least one whole chain, so at most
    // nchains runs.  Only on request, or to bound the scratch: with all CTAs in
    // step (the range schedule) neighbouring head pairs read and write the same
    // rows of x and y at the same time, which measured faster on the 2.7B layer
    // than the better balance of the pieces.
    g.pieces = false;
    const long long grid_p = std::min<long long>(sms, g.nchains);
    const bool pieces_ok = g.nsub_chain > 0 && grid_p > 0 && g.total_subs / grid_p >= g.nsub_chain &&
                           g.total_subs < (1LL << 40);
    if (pieces_ok && a.sched_req == SSD_SCHEDULE_PIECES)
        g.pieces = true;
    g.split = false;
    const bool split_allowed = a.sched_req == SSD_SCHEDULE_SPLIT || (a.sched_req == 0 && a.scratch_cap == 0);
    g.span = g.chunks_per_unit * a.chunk;
    if (split_allowed && g.nchunks > 1) {
        double best_split = 1e300;
        long long span_split = a.chunk;
        for (int i = 0; i + 1 < nc; ++i) {   // at least two ranges
            const double est = split_estimate(cand[i], g.nchunks, g.nchains, (double)a.chunk / kT, sms);
            if (est < best_split * 0.999) {
                best_split = est;
                span_split = cand[i] * a.chunk;
            }
        }
        if (best_split < 0.8 * best || a.sched_req == SSD_SCHEDULE_SPLIT) {
            g.split = true;
            g.pieces = false;
            // Once split, where a chunk is a whole number of the kernel's 128-step
            // sub-chunks, a unit may be any whole number of sub-chunks (the sub-chunk
            // grid of every chain stays where it is): the lengths that make the units
            // fill whole rounds of the grid.  Units stay fewer than 2^31.
            if (a.chunk % kT == 0) {
                const long long smax = std::min<long long>(g.nsub_chain - 1, 4096);
                for (long long S = 1; S <= smax; ++S) {
                    if ((g.nsub_chain + S - 1) / S > ((1LL << 31) - 1) / std::max<long long>(1, g.nchains))
                        continue;
                    const double est = split_estimate(S, g.nsub_chain, g.nchains, 1.0, sms);
                    if (est < best_split * 0.99) {
                        best_split = est;
                        span_split = S * kT;
                    }
                }
            }
            g.span = span_split;
        }
    }
    layout(g, grid_p, sms);
    if (a.sched_req == 0 && a.scratch_cap != 0 && g.total > a.scratch_cap && pieces_ok && !g.pieces) {
        g.pieces = true;   // at most one state slot per CTA
        layout(g, grid_p, sms);
    }
    return g;
}

// Split evaluations of at most this many ranges per chain fold the combine into
// pass 3 (ssd_chunk_fused_kernel's kFold): each unit then reads at most three
// predecessors' end states at its start, in place of one combine launch.
constexpr long long kFoldMaxRanges = 4;

bool split_folds(const ScanArgs &a, const Geometry &g)
{
    return g.split && !a.conv && !a.trap && g.nranges <= kFoldMaxRanges;
}

// Grid and scratch layout of the chosen schedule.
void layout(Geometry &g, long long grid_p, int sms)
{
    const size_t slot_state = (size_t)kN * 2 * kP * 4;   // one head pair, fp32
    size_t flag_rows, slot_bytes;
    if (g.pieces) {
        g.chunks_per_unit = g.nchunks;
        g.span = g.seqlen;
        g.nranges = 1;
        g.grid = grid_p;
        g.nunits = 0;
        flag_rows = (size_t)g.grid;   // one per boundary between CTAs
        slot_bytes = g.grid > 1 ? (size_t)g.grid * slot_state : 0;
    } else {
        g.nranges = (g.seqlen + g.span - 1) / g.span;
        g.nunits = g.nranges * g.nchains;
        g.grid = std::min<long long>(sms, g.nunits);
        flag_rows = (size_t)g.nunits;
        slot_bytes = g.split ? (size_t)g.nunits * slot_state
                             : (g.nranges > 1 ? (size_t)g.nchains * slot_state : 0);
    }
    g.flags_off = 256;
    g.slot_off = (g.flags_off + flag_rows * kGroupWarps * 8 + 255) & ~(size_t)255;
    g.decay_off = g.slot_off + slot_bytes;
    g.total = g.decay_off + (g.split ? (((size_t)g.nunits * 2 * 4 + 255) & ~(size_t)255) : 0);
}

}  // namespace

bool chunk_supported(const ScanArgs &a)
{
    if (a.nheads > kMaxHeads)
        return false;
    if (a.dtype != SSD_DTYPE_BF16 || a.headdim != kP || a.dstate != kN)
        return false;
    if (a.chunk % 64 != 0 || a.chunk <= 0)
        return false;
    if ((a.nheads / a.ngroups) % 2 != 0)
        return false;
    if (a.batch >= (1LL << 31) || a.seqlen >= (1LL << 31))
        return false;
    // work units (at most chunks x chains) are indexed with 32-bit arithmetic
    const long long nchunks = (a.seqlen + a.chunk - 1) / a.chunk, nchains = a.batch * (a.nheads / 2);
    if (nchains > 0 && nchunks > ((1LL << 31) - 1) / nchains)
        return false;
    return true;
}

size_t chunk_workspace_bytes(const ScanArgs &a) { return geometry(a).total; }

ssd_status_t chunk_launch(const ScanArgs &a, void *workspace, cudaStream_t stream)
{
    SSD_NVTX_RANGE("chunk_launch");
    const Geometry geo = geometry(a);
    Maps maps;
    const uint64_t HP = (uint64_t)a.nheads * kP, GN = (uint64_t)a.ngroups * kN, L = (uint64_t)a.seqlen;
    // conv mode: x tiles come from the x channels (the first H*P) of the raw xbc rows
    const uint64_t xrow = a.conv ? (uint64_t)a.conv_cc * 2 : HP * 2;
    if (!make_tmap_bf16_3d(&maps.x, a.conv ? a.xbc : a.x, HP, L, (uint64_t)a.batch, xrow, xrow * L, 64, 128) ||
        !make_tmap_bf16_3d(&maps.B, a.B, GN, L, (uint64_t)a.batch, GN * 2, GN * 2 * L, 64, 128) ||
        !make_tmap_bf16_3d(&maps.C, a.C, GN, L, (uint64_t)a.batch, GN * 2, GN * 2 * L, 64, 128) ||
        !make_tmap_bf16_3d(&maps.y, a.y, HP, L, (uint64_t)a.batch, HP * 2, HP * 2 * L, 64, 32))
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
    p.final_state = a.final_state;
    p.slots = (geo.split || geo.nranges > 1 || (geo.pieces && geo.grid > 1)) ? reinterpret_cast<float *>(ws + geo.slot_off)
                                                                            : nullptr;
    p.unit_decay = geo.split ? reinterpret_cast<float *>(ws + geo.decay_off) : nullptr;
    p.mode = kChained;
    p.epoch = next_epoch();
    p.timeout_ns = a.diag_stall ? 20000000ull : 2000000000ull;
    p.diag_stall = a.diag_stall ? 1 : 0;
    p.tdt = a.tdt;
    p.ta = a.ta;
    p.ttrap = a.ttrap;
    p.k0 = static_cast<const __nv_bfloat16 *>(a.k0);
    p.v0 = static_cast<const __nv_bfloat16 *>(a.v0);
    if (a.diag_stall && cudaMemsetAsync(ws + 64, 0, 8, stream) != cudaSuccess)
        return SSD_ERR_CUDA;
    p.L = a.seqlen;
    p.nunits = geo.nunits;
    p.H = a.nheads;
    p.span = (int)geo.span;
    p.nranges = (int)geo.nranges;
    p.nsub_chain = (int)geo.nsub_chain;
    p.total_subs = geo.total_subs;
    p.nhp = a.nheads / 2;
    p.nchains = (int)geo.nchains;
    p.hpg = a.nheads / a.ngroups;

    p.xbc = static_cast<const __nv_bfloat16 *>(a.xbc);
    p.conv_w = a.conv_w;
    p.conv_b = a.conv_b;
    p.conv_state = static_cast<const __nv_bfloat16 *>(a.conv_state);
    p.conv_k = a.conv_k;
    p.conv_cc = a.conv_cc;
    auto kernel = a.conv ? (geo.pieces ? ssd_chunk_fused_kernel<true, false, false, true>
                                       : ssd_chunk_fused_kernel<false, false, false, true>)
                : a.trap ? (geo.pieces ? ssd_chunk_fused_kernel<true, true, false>
                                       : ssd_chunk_fused_kernel<false, true, false>)
                         : (geo.pieces ? ssd_chunk_fused_kernel<true, false, false>
                                       : ssd_chunk_fused_kernel<false, false, false>);
    auto kernel_local = a.conv   ? ssd_chunk_fused_kernel<false, false, true, true>
                        : a.trap ? ssd_chunk_fused_kernel<false, true, true>
                                 : ssd_chunk_fused_kernel<false, false, true>;   // split pass 1
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes) != cudaSuccess)
        return SSD_ERR_CUDA;
    if (geo.split && cudaFuncSetAttribute(kernel_local, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)kSmemBytes) != cudaSuccess)
        return SSD_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)geo.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs co-resident: chunk handoff waits are safe
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (!geo.split) {
        if (cudaLaunchKernelEx(&cfg, kernel, maps, p) != cudaSuccess)
            return SSD_ERR_CUDA;
        note_launches(1);
        return SSD_OK;
    }
    // split: pass 1 (end state of every unit from zero), combine (entering state of
    // every unit), pass 3 (the scan itself, all units independent); with few ranges
    // the combine is folded into pass 3
    const bool fold = split_folds(a, geo);
    auto kernel_fold = ssd_chunk_fused_kernel<false, false, false, false, true>;
    if (fold && cudaFuncSetAttribute(kernel_fold, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
                    cudaSuccess)
        return SSD_ERR_CUDA;
    p.mode = kSplitLocal;
    if (cudaLaunchKernelEx(&cfg, kernel_local, maps, p) != cudaSuccess)
        return SSD_ERR_CUDA;
    note_launches(1);
    // The combine and pass 3 are programmatic dependents of the launch before them
    // (each waits with griddepcontrol.wait before it reads what that launch wrote),
    // so their launch and setup overlap the previous kernel's tail.
    cudaLaunchAttribute pdl[2];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    if (!fold) {
        const long long threads = geo.nchains * 2 * 16 * kN;
        cudaLaunchConfig_t ccfg = {};
        ccfg.gridDim = dim3((unsigned)((threads + 255) / 256));
        ccfg.blockDim = dim3(256);
        ccfg.stream = stream;
        ccfg.attrs = pdl;
        ccfg.numAttrs = 1;
        // (the trapezoidal pass 1 has put each chain's entering state into its first unit)
        if (cudaLaunchKernelEx(&ccfg, ssd_split_combine_kernel, p.slots, (const float *)p.unit_decay,
                               a.trap ? nullptr : a.init_state, (int)geo.nchains, (int)geo.nranges, a.nheads / 2,
                               a.nheads) != cudaSuccess)
            return SSD_ERR_CUDA;
        note_launches(1);
    }
    p.mode = kSplitEntering;
    p.epoch = next_epoch();
    pdl[1] = attr[0];   // cooperative
    cfg.attrs = pdl;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, fold ? kernel_fold : kernel, maps, p) != cudaSuccess)
        return SSD_ERR_CUDA;
    note_launches(1);
    return SSD_OK;
}

int chunk_launches(const ScanArgs &a)
{
    const Geometry g = geometry(a);
    return g.split ? (split_folds(a, g) ? 2 : 3) : 1;
}

int chunk_schedule(const ScanArgs &a)
{
    const Geometry g = geometry(a);
    return g.split ? SSD_SCHEDULE_SPLIT : (g.pieces ? SSD_SCHEDULE_PIECES : SSD_SCHEDULE_RANGES);
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
