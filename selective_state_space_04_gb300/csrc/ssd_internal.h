// ssd_internal.h -- shared declarations between the host layer (ssd_api.cu)
// and the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "ssd.h"

// NVTX ranges, compiled in with -DSSD_NVTX (the build's SSD_NVTX=1): one range per
// call of a public entry point and one per launch function inside it, named after
// them, so that a timeline tool shows which call and which kernel family each
// kernel came from.  Without the flag the macro is empty.
#ifdef SSD_NVTX
#include <nvtx3/nvToolsExt.h>
namespace ssd {
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};
}  // namespace ssd
#define SSD_NVTX_RANGE(name) const ::ssd::NvtxRange ssd_nvtx_range_(name)
#else
#define SSD_NVTX_RANGE(name) ((void)0)
#endif

namespace ssd {

// Everything one scan needs, after validation.  Device pointers.
struct ScanArgs {
    const void *x;
    const float *dt_raw;
    const float *dt_bias;
    const float *A_log;
    const void *B;
    const void *C;
    const float *D;
    const float *init_state;   // may be null
    void *y;
    float *final_state;        // may be null
    int64_t batch, seqlen;
    int nheads, headdim, dstate, ngroups, chunk;
    int dtype;                 // ssd_dtype_t
    bool diag_stall;           // SSD_DIAG_STALL_HANDOFF
    int sched_req;             // requested SSD_SCHEDULE_*, or 0: the library chooses
    // trapezoidal (Mamba-3 SISO) mode of the chunked path: x = v, B = k, C = q,
    // init_state = h0, final_state = h_final; per-token dt, a, trap replace
    // dt_raw, dt_bias, A_log; k0, v0 ([B,H,N], [B,H,P], bf16) may be null
    bool trap = false;
    const float *tdt = nullptr, *ta = nullptr, *ttrap = nullptr;
    const void *k0 = nullptr, *v0 = nullptr;
    size_t scratch_cap = 0;   // nonzero: the chunked path takes no split schedule and, when it
                              // chooses, the piece schedule (at most one state slot per SM)
                              // if the one it would choose needs more scratch than this
    // conv mode of the chunked path: x is not an input; the kernel reads the x
    // channels of the fused xbc [B,L,conv_cc] (bf16) and applies the causal conv1d
    // + SiLU to them itself (weights [conv_cc, conv_k] and bias, fp32; the carried
    // conv state [B, conv_k - 1, conv_cc] or null).  B and C are the conv's outputs.
    bool conv = false;
    const void *xbc = nullptr;
    const float *conv_w = nullptr, *conv_b = nullptr;
    const void *conv_state = nullptr;
    int conv_k = 0, conv_cc = 0;
};

// The trapezoidal (Mamba-3 SISO) scan, after validation.  Device pointers.
struct TrapArgs {
    const void *v, *k, *q;               // x [B,L,H,P]; B, C [B,L,G,N] (storage dtype)
    const float *dt, *a, *trap, *D;       // [B,L,H] x3, [H]
    const float *h0;                      // [B,H,P,N] or null
    const void *k0, *v0;                  // [B,H,N], [B,H,P] (storage dtype) or null
    void *y;                              // [B,L,H,P]
    float *h_final;                       // or null
    void *k_final, *v_final;              // or null
    int64_t batch, seqlen;
    int nheads, headdim, dstate, ngroups;
    int dtype;
};

// ---- trapezoidal scan: ssd_trap.cu
bool trap_supported(const TrapArgs &a);
cudaError_t trap_launch(const TrapArgs &a, cudaStream_t stream);
// k_final, v_final (the last step's k and v) after a chunked-path run
cudaError_t trap_carry_launch(const TrapArgs &a, cudaStream_t stream);

// The steps on either side of the scan (ssd_neighbors.cu), after validation.
struct NeighborArgs {
    // causal conv1d + SiLU over the fused x | B | C channels
    const void *xbc = nullptr;                        // [B,L,H*P + 2*G*N]
    const float *w = nullptr, *bias = nullptr;        // [C,K] (also the norm weight [H*P]), [C] or null
    const void *state_in = nullptr;                   // [B,K-1,C] or null
    void *x = nullptr, *B = nullptr, *C = nullptr;    // [B,L,H,P], [B,L,G,N] x2
    void *state_out = nullptr;                        // [B,K-1,C] or null
    int kernel_size = 0;
    // gated RMSNorm
    const void *y = nullptr, *z = nullptr;            // [B,L,H,P]
    void *out = nullptr;                              // [B,L,H,P]
    float eps = 0.f;
    int64_t batch = 0, seqlen = 0;
    int nheads = 0, headdim = 0, dstate = 0, ngroups = 0;
    int dtype = 0;
};
bool conv_supported(const NeighborArgs &a);
cudaError_t conv_launch(const NeighborArgs &a, cudaStream_t stream);
// The conv over the B and C channels only (writing B, C and their part of
// state_out), and the x channels' part of state_out (the last K-1 inputs):
// the part of the conv that the chunked path's conv mode does not do itself.
cudaError_t conv_bc_launch(const NeighborArgs &a, cudaStream_t stream);
bool gnorm_supported(const NeighborArgs &a);
cudaError_t gnorm_launch(const NeighborArgs &a, cudaStream_t stream);

// The backward of the SSD scan (ssd_bwd.cu), after validation.
struct BwdArgs {
    const void *x, *B, *C, *dy;                 // [B,L,H,P], [B,L,G,N] x2, [B,L,H,P] (dtype)
    const float *dt_raw, *dt_bias, *A_log, *D;
    const float *init_state, *d_final;          // [B,H,P,N] or null
    float *dx, *ddt_raw, *ddt_bias, *dA_log;    // [B,L,H,P], [B,L,H], [H], [H]
    float *dB, *dC, *dD;                        // [B,L,G,N] x2, [H]
    float *d_init;                              // [B,H,P,N] or null
    int64_t batch, seqlen;
    int nheads, headdim, dstate, ngroups;
    int dtype;
    uint32_t path;                              // SSD_PATH_SEQUENTIAL or SSD_PATH_CHUNKED (resolved)
    bool fp32_form = false;                     // the chunk form's fp32 contractions even where the
                                                // tensor-core gradient pass applies (SSD_BWD_FP32_FORM)
    bool split_states = false;                  // the tensor-core form's chunk states and chains as two
                                                // launches (SSD_BWD_SPLIT_STATES)
};
// ssd_bwd.cu: dispatch, the sequential kernel and the fixed-order reductions
bool bwd_seq_supported(const BwdArgs &a);
bool bwd_supported(const BwdArgs &a);
size_t bwd_workspace_bytes(const BwdArgs &a);
cudaError_t bwd_launch(const BwdArgs &a, void *workspace, cudaStream_t stream);
// dB, dC from the per-head buffers; dA_log, ddt_bias, dD from nper partials per (b, h)
cudaError_t bwd_finish_launch(const BwdArgs &a, const float *dB_head, const float *dC_head, const float *part,
                              int nper, cudaStream_t stream);
// ssd_bwd_tc.cu: the chunk form's gradient pass on the tensor cores (bf16, P = 64,
// N = 128), from the chunk states and state gradients the first two launches left
struct BwdTcArgs {
    const void *x, *B, *C, *dy;                 // bf16
    const float *dt_raw, *dt_bias, *A_log, *D;
    const float *S, *R;                         // [B*H][nc+1][N][P] entering states; [B*H][nc][N][P] G_out
    float *dx, *ddt_raw, *dB_head, *dC_head, *part;
    int64_t batch, seqlen;
    int nheads, ngroups, nc;
};
struct BwdTcLocalArgs {
    const void *x, *B, *C, *dy;                 // bf16
    const float *dt_raw, *dt_bias, *A_log;
    float *S, *R, *dec;                         // [B*H][nc+1][N][P] (slots 0 .. nc-1 written), [B*H][nc][N][P], [B*H][nc]
    int64_t batch, seqlen;
    int nheads, ngroups, nc;
};
bool bwd_tc_supported(int dtype, int headdim, int dstate);
cudaError_t bwd_tc_local_launch(const BwdTcLocalArgs &a, cudaStream_t stream);
struct BwdTcChainArgs {
    const void *x, *B, *C, *dy;                 // bf16
    const float *dt_raw, *dt_bias, *A_log;
    const float *init_state, *d_final;          // [B,H,P,N] or null
    float *S, *R, *d_init;                      // [B*H][nc+1][N][P] (all slots), [B*H][nc][N][P], [B,H,P,N] or null
    int64_t batch, seqlen;
    int nheads, ngroups, nc;
};
cudaError_t bwd_tc_chain_launch(const BwdTcChainArgs &a, cudaStream_t stream);
cudaError_t bwd_tc_grad_launch(const BwdTcArgs &a, cudaStream_t stream);
ssd_status_t bwd_tc_read_device_error(uint32_t *code);
// ssd_bwd_chunk.cu: the chunk-parallel backward (P <= 64, N <= 128)
bool bwd_chunk_supported(const BwdArgs &a);
size_t bwd_chunk_workspace_bytes(const BwdArgs &a);
cudaError_t bwd_chunk_launch(const BwdArgs &a, void *workspace, cudaStream_t stream);

// ---- complex-valued scan with ET discretisation: ssd_complex.cu
struct ComplexArgs {
    const void *x, *B, *C;                      // [B,L,H,P], [B,L,G,N] x2 (dtype; N/2 complex as re, im)
    const float *dt_raw, *dt_bias, *A_polar, *D; // [B,L,H], [H], [H,2] (log|A|, arg A), [H]
    const float *init_state;                    // [B,H,P,N] or null
    void *y;                                    // [B,L,H,P]
    float *final_state;                         // [B,H,P,N] or null
    int64_t batch, seqlen;
    int nheads, headdim, dstate, ngroups;
    int dtype;
};
bool complex_supported(const ComplexArgs &a);
cudaError_t complex_launch(const ComplexArgs &a, cudaStream_t stream);
// ssd_complex_tc.cu: the chunk form on the tensor cores (bf16, P = 64, N = 128, seqlen >= 2)
bool complex_tc_supported(const ComplexArgs &a);
cudaError_t complex_tc_launch(const ComplexArgs &a, cudaStream_t stream);
ssd_status_t complex_tc_read_device_error(uint32_t *code);

// ---- sequential (direct recurrence) path: ssd_seq.cu
bool seq_supported(int headdim, int dstate);
cudaError_t seq_launch(const ScanArgs &a, cudaStream_t stream);

// ---- decode step (seqlen 1): ssd_decode.cu
bool decode_supported(const ScanArgs &a);
cudaError_t decode_launch(const ScanArgs &a, cudaStream_t stream);

// ---- chunked tcgen05 path: ssd_chunk.cu
bool chunk_supported(const ScanArgs &a);
// Bytes of scratch the chunked path needs for these sizes (flags and, when
// final_state is null, the chunk-handoff states).
size_t chunk_workspace_bytes(const ScanArgs &a);
// `workspace` must hold chunk_workspace_bytes(a) bytes, 16-byte aligned;
// its contents on entry do not matter.
ssd_status_t chunk_launch(const ScanArgs &a, void *workspace, cudaStream_t stream);
// kernel launches chunk_launch makes for these sizes (1, or 3 for the split schedule)
int chunk_launches(const ScanArgs &a);
// SSD_SCHEDULE_RANGES, _PIECES or _SPLIT for these sizes
int chunk_schedule(const ScanArgs &a);
ssd_status_t chunk_read_device_error(cudaStream_t stream, uint32_t *code);

// launch accounting
void note_launches(int n);

}  // namespace ssd
