"""ctypes binding for libssd (argument marshalling only).

Every step of the scan runs in libssd's CUDA kernels.  If the shared library
has not been built, importing this module raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB_PATH

PATH_AUTO = 0
DIAG_STALL_HANDOFF = 0x100
BWD_FP32_FORM = 0x200   # ssd_scan_bwd: the chunk form's fp32 contractions even where the tensor-core pass applies
BWD_SPLIT_STATES = 0x400   # ssd_scan_bwd: the tensor-core form's chunk states and chains as two launches
PATH_SEQUENTIAL = 1
PATH_CHUNKED = 2
PATH_DECODE = 3
_PATHS = {"auto": PATH_AUTO, "sequential": PATH_SEQUENTIAL, "seq": PATH_SEQUENTIAL,
          "chunked": PATH_CHUNKED, "decode": PATH_DECODE}

DTYPE_F32 = 0
DTYPE_BF16 = 1

STATUS = {0: "SSD_OK", 1: "SSD_ERR_INVALID_DIMS", 2: "SSD_ERR_NULL_PTR", 3: "SSD_ERR_MISALIGNED",
          4: "SSD_ERR_UNSUPPORTED", 5: "SSD_ERR_CUDA", 6: "SSD_ERR_TIMEOUT", 7: "SSD_ERR_ALIASING",
          8: "SSD_ERR_SCRATCH_LIMIT", 9: "SSD_ERR_UNSUPPORTED_DTYPE"}


class SsdError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{STATUS.get(status, status)}: {what}")


class SsdDims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64),
                ("nheads", ctypes.c_int32), ("headdim", ctypes.c_int32),
                ("dstate", ctypes.c_int32), ("ngroups", ctypes.c_int32),
                ("chunk", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("flags", ctypes.c_uint32), ("reserved", ctypes.c_uint32)]


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"libssd is not built ({path} missing); run "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    vp, fp = ctypes.c_void_p, ctypes.c_void_p
    sig = [vp, fp, fp, fp, vp, vp, fp, fp, vp, fp, ctypes.POINTER(SsdDims), vp]
    for name in ("ssd_scan_fwd", "ssd_scan_fwd_host", "ssd_scan_fwd_noalloc"):
        f = getattr(lib, name)
        f.restype = ctypes.c_int
        f.argtypes = sig
    lib.ssd_scan_fwd_ws.restype = ctypes.c_int
    lib.ssd_scan_fwd_ws.argtypes = sig[:10] + [vp, ctypes.c_uint64, ctypes.POINTER(SsdDims), vp]
    lib.ssd_scan_fwd_workspace_size.restype = ctypes.c_int
    lib.ssd_scan_fwd_workspace_size.argtypes = [ctypes.POINTER(SsdDims), ctypes.POINTER(ctypes.c_uint64)]
    lib.ssd_select_path.restype = ctypes.c_int32
    lib.ssd_select_path.argtypes = [ctypes.POINTER(SsdDims)]
    lib.ssd_launches_per_call.restype = ctypes.c_int32
    lib.ssd_launches_per_call.argtypes = [ctypes.POINTER(SsdDims)]
    lib.ssd_chunk_schedule.restype = ctypes.c_int32
    lib.ssd_chunk_schedule.argtypes = [ctypes.POINTER(SsdDims)]
    lib.ssd_launch_count.restype = ctypes.c_uint64
    lib.ssd_launch_count.argtypes = []
    lib.ssd_get_device_error.restype = ctypes.c_int
    lib.ssd_get_device_error.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.ssd_status_string.restype = ctypes.c_char_p
    lib.ssd_status_string.argtypes = [ctypes.c_int32]
    lib.ssd_abi_version.restype = ctypes.c_int32
    lib.ssd_abi_version.argtypes = []
    lib.ssd_trap_scan_fwd.restype = ctypes.c_int
    lib.ssd_trap_scan_fwd.argtypes = [vp] * 14 + [ctypes.POINTER(SsdDims), vp]
    lib.ssd_conv1d_silu_fwd.restype = ctypes.c_int
    lib.ssd_conv1d_silu_fwd.argtypes = [vp] * 8 + [ctypes.c_int32, ctypes.POINTER(SsdDims), vp]
    lib.ssd_conv_scan_fwd.restype = ctypes.c_int
    lib.ssd_conv_scan_fwd.argtypes = [vp] * 4 + [ctypes.c_int32] + [vp] * 8 + [ctypes.POINTER(SsdDims), vp]
    lib.ssd_gated_rmsnorm_fwd.restype = ctypes.c_int
    lib.ssd_gated_rmsnorm_fwd.argtypes = [vp, vp, vp, ctypes.c_float, vp, ctypes.POINTER(SsdDims), vp]
    lib.ssd_scan_bwd.restype = ctypes.c_int
    lib.ssd_scan_bwd.argtypes = [vp] * 18 + [ctypes.POINTER(SsdDims), vp]
    lib.ssd_complex_scan_fwd.restype = ctypes.c_int
    lib.ssd_complex_scan_fwd.argtypes = [vp] * 10 + [ctypes.POINTER(SsdDims), vp]
    return lib


_lib = load_library()


def lib() -> ctypes.CDLL:
    return _lib


SCHEDULE_SHIFT = 4
_SCHEDULE_REQUESTS = {"auto": 0, "ranges": 1, "pieces": 2, "split": 3}


def make_dims(batch, seqlen, nheads, headdim, dstate, ngroups, chunk, dtype, path="auto",
              schedule="auto") -> SsdDims:
    d = SsdDims()
    d.batch, d.seqlen, d.nheads, d.headdim = batch, seqlen, nheads, headdim
    d.dstate, d.ngroups, d.chunk = dstate, ngroups, chunk
    if isinstance(dtype, int):     # an ssd_dtype_t value, passed through as given
        d.dtype = dtype
    else:
        d.dtype = DTYPE_BF16 if dtype in ("bf16", torch.bfloat16) else DTYPE_F32
    d.flags = (_PATHS[path] if isinstance(path, str) else int(path)) | \
        (_SCHEDULE_REQUESTS[schedule] << SCHEDULE_SHIFT)
    d.reserved = 0
    return d


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(status: int, what: str):
    if status != 0:
        raise SsdError(status, what)


def _dims_from(x, B, chunk, path, schedule="auto"):
    Bt, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    return make_dims(Bt, L, H, P, N, G, chunk, x.dtype, path, schedule)


def select_path(x_shape, ngroups, dstate, chunk, dtype="bf16", path="auto", schedule="auto") -> int:
    Bt, L, H, P = x_shape
    d = make_dims(Bt, L, H, P, dstate, ngroups, chunk, dtype, path, schedule)
    return _lib.ssd_select_path(ctypes.byref(d))


def launches_per_call(x_shape, ngroups, dstate, chunk, dtype="bf16", path="auto", schedule="auto") -> int:
    Bt, L, H, P = x_shape
    d = make_dims(Bt, L, H, P, dstate, ngroups, chunk, dtype, path, schedule)
    return _lib.ssd_launches_per_call(ctypes.byref(d))


SCHEDULES = {0: "none", 1: "ranges", 2: "pieces", 3: "split"}


def chunk_schedule(x_shape, ngroups, dstate, chunk, dtype="bf16", path="auto", schedule="auto") -> str:
    """How ``ssd_scan_fwd`` orders the chunked path's work for these sizes on the current device."""
    Bt, L, H, P = x_shape
    d = make_dims(Bt, L, H, P, dstate, ngroups, chunk, dtype, path, schedule)
    v = _lib.ssd_chunk_schedule(ctypes.byref(d))
    if v < 0:
        _check(-v, "ssd_chunk_schedule")
    return SCHEDULES[v]


def workspace_size(x_shape, ngroups, dstate, chunk, dtype="bf16", path="auto", schedule="auto") -> int:
    """Bytes of scratch ``ssd_scan_fwd_ws`` needs for these sizes on the current device."""
    Bt, L, H, P = x_shape
    d = make_dims(Bt, L, H, P, dstate, ngroups, chunk, dtype, path, schedule)
    n = ctypes.c_uint64(0)
    _check(_lib.ssd_scan_fwd_workspace_size(ctypes.byref(d), ctypes.byref(n)), "ssd_scan_fwd_workspace_size")
    return int(n.value)


def launch_count() -> int:
    return int(_lib.ssd_launch_count())


def device_error(stream=None) -> int:
    st = torch.cuda.current_stream() if stream is None else stream
    code = ctypes.c_uint32(0)
    _check(_lib.ssd_get_device_error(ctypes.c_void_p(st.cuda_stream), ctypes.byref(code)),
           "ssd_get_device_error")
    return int(code.value)


def ssd_scan_fwd(x, dt_raw, dt_bias, A_log, B, C, D, init_state=None, *, chunk=256,
                 path="auto", return_final_state=True, y=None, final_state=None, stream=None,
                 diag_stall_handoff=False, schedule="auto"):
    """Forward SSD scan on CUDA tensors.  Returns ``(y, final_state)``.

    ``x [B,L,H,P]`` and ``B, C [B,L,G,N]`` share one dtype (bf16 or fp32);
    ``dt_raw [B,L,H]``, ``dt_bias, A_log, D [H]`` and the states
    ``[B,H,P,N]`` are fp32.  Work is enqueued on ``stream`` (default: the
    current torch stream); the call does not synchronise.  ``schedule``
    requests the chunked path's schedule ("ranges", "pieces", "split"), or
    lets the library choose ("auto").
    """
    if y is None:
        y = torch.empty_like(x)
    if final_state is None and return_final_state:
        Bt, L, H, P = x.shape
        final_state = torch.empty((Bt, H, P, B.shape[3]), dtype=torch.float32, device=x.device)
    for name, t in (("x", x), ("dt_raw", dt_raw), ("dt_bias", dt_bias), ("A_log", A_log),
                    ("B", B), ("C", C), ("D", D), ("init_state", init_state), ("y", y),
                    ("final_state", final_state)):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    d = _dims_from(x, B, chunk, path, schedule)
    if diag_stall_handoff:
        d.flags |= DIAG_STALL_HANDOFF
    st = torch.cuda.current_stream(x.device) if stream is None else stream
    _check(_lib.ssd_scan_fwd(_ptr(x), _ptr(dt_raw), _ptr(dt_bias), _ptr(A_log), _ptr(B), _ptr(C),
                             _ptr(D), _ptr(init_state), _ptr(y), _ptr(final_state),
                             ctypes.byref(d), ctypes.c_void_p(st.cuda_stream)),
           "ssd_scan_fwd")
    return y, final_state


def ssd_scan_fwd_host(x, dt_raw, dt_bias, A_log, B, C, D, init_state=None, *, chunk=256,
                      path="auto", return_final_state=True, y=None, final_state=None,
                      stream=None, device=None, schedule="auto"):
    """Same scan on CPU tensors (pinned for asynchronous copies).  The library
    copies in, runs, copies out and synchronises before returning."""
    if y is None:
        y = torch.empty_like(x)
    if final_state is None and return_final_state:
        Bt, L, H, P = x.shape
        final_state = torch.empty((Bt, H, P, B.shape[3]), dtype=torch.float32)
    for name, t in (("x", x), ("dt_raw", dt_raw), ("dt_bias", dt_bias), ("A_log", A_log),
                    ("B", B), ("C", C), ("D", D), ("init_state", init_state), ("y", y),
                    ("final_state", final_state)):
        if t is not None and (t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CPU tensor")
    d = _dims_from(x, B, chunk, path, schedule)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(dev):
        st = torch.cuda.current_stream(dev) if stream is None else stream
        _check(_lib.ssd_scan_fwd_host(_ptr(x), _ptr(dt_raw), _ptr(dt_bias), _ptr(A_log), _ptr(B),
                                      _ptr(C), _ptr(D), _ptr(init_state), _ptr(y),
                                      _ptr(final_state), ctypes.byref(d),
                                      ctypes.c_void_p(st.cuda_stream)),
               "ssd_scan_fwd_host")
    return y, final_state


def ssd_scan_fwd_noalloc(x, dt_raw, dt_bias, A_log, B, C, D, init_state=None, *, chunk=256,
                         path="auto", y=None, final_state=None, return_final_state=True,
                         stream=None, schedule="auto"):
    """``ssd_scan_fwd`` on the chunked path with the library's fixed scratch
    array instead of a pool allocation (the library allocates nothing; outputs
    not passed in are created here by torch).  Calls that may overlap on one
    device share that array and race; calls ordered on one stream are safe."""
    if y is None:
        y = torch.empty_like(x)
    if final_state is None and return_final_state:
        Bt, L, H, P = x.shape
        final_state = torch.empty((Bt, H, P, B.shape[3]), dtype=torch.float32, device=x.device)
    for name, t in (("x", x), ("dt_raw", dt_raw), ("dt_bias", dt_bias), ("A_log", A_log),
                    ("B", B), ("C", C), ("D", D), ("init_state", init_state), ("y", y),
                    ("final_state", final_state)):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    d = _dims_from(x, B, chunk, path, schedule)
    st = torch.cuda.current_stream(x.device) if stream is None else stream
    _check(_lib.ssd_scan_fwd_noalloc(_ptr(x), _ptr(dt_raw), _ptr(dt_bias), _ptr(A_log), _ptr(B),
                                     _ptr(C), _ptr(D), _ptr(init_state), _ptr(y),
                                     _ptr(final_state), ctypes.byref(d),
                                     ctypes.c_void_p(st.cuda_stream)),
           "ssd_scan_fwd_noalloc")
    return y, final_state


def ssd_scan_fwd_ws(x, dt_raw, dt_bias, A_log, B, C, D, init_state=None, *, workspace,
                    chunk=256, path="auto", y=None, final_state=None, return_final_state=True,
                    stream=None, schedule="auto"):
    """``ssd_scan_fwd`` with caller-provided scratch: ``workspace`` is a CUDA
    tensor of at least ``workspace_size(...)`` bytes (or None when that is 0).
    The library allocates nothing; calls that may overlap must not share a
    workspace."""
    if y is None:
        y = torch.empty_like(x)
    if final_state is None and return_final_state:
        Bt, L, H, P = x.shape
        final_state = torch.empty((Bt, H, P, B.shape[3]), dtype=torch.float32, device=x.device)
    for name, t in (("x", x), ("dt_raw", dt_raw), ("dt_bias", dt_bias), ("A_log", A_log),
                    ("B", B), ("C", C), ("D", D), ("init_state", init_state), ("y", y),
                    ("final_state", final_state), ("workspace", workspace)):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    d = _dims_from(x, B, chunk, path, schedule)
    st = torch.cuda.current_stream(x.device) if stream is None else stream
    _check(_lib.ssd_scan_fwd_ws(_ptr(x), _ptr(dt_raw), _ptr(dt_bias), _ptr(A_log), _ptr(B), _ptr(C),
                                _ptr(D), _ptr(init_state), _ptr(y), _ptr(final_state),
                                _ptr(workspace), ctypes.c_uint64(nbytes), ctypes.byref(d),
                                ctypes.c_void_p(st.cuda_stream)),
           "ssd_scan_fwd_ws")
    return y, final_state


def ssd_trap_scan_fwd(v, k, q, dt, a, trap, D, h0=None, k0=None, v0=None, *, chunk=256, path="auto", y=None,
                      h_final=None, k_final=None, v_final=None, return_states=True, stream=None, schedule="auto"):
    """Trapezoidal (Mamba-3 SISO) scan on CUDA tensors.  Returns
    ``(y, h_final, k_final, v_final)`` (the states None when not returned).
    ``schedule`` requests a schedule of the chunked kernel, as for ``ssd_scan_fwd``.

    ``v [B,L,H,P]``, ``k, q [B,L,G,N]``, ``k0/k_final [B,H,N]`` and
    ``v0/v_final [B,H,P]`` share one dtype (bf16 or fp32); ``dt, a, trap
    [B,L,H]``, ``D [H]`` and ``h0/h_final [B,H,P,N]`` are fp32.
    """
    Bt, L, H, P = v.shape
    G, N = k.shape[2], k.shape[3]
    if y is None:
        y = torch.empty_like(v)
    if return_states:
        if h_final is None:
            h_final = torch.empty((Bt, H, P, N), dtype=torch.float32, device=v.device)
        if k_final is None:
            k_final = torch.empty((Bt, H, N), dtype=v.dtype, device=v.device)
        if v_final is None:
            v_final = torch.empty((Bt, H, P), dtype=v.dtype, device=v.device)
    named = (("v", v), ("k", k), ("q", q), ("dt", dt), ("a", a), ("trap", trap), ("D", D), ("h0", h0),
             ("k0", k0), ("v0", v0), ("y", y), ("h_final", h_final), ("k_final", k_final), ("v_final", v_final))
    for name, t in named:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    d = make_dims(Bt, L, H, P, N, G, chunk, v.dtype, path, schedule)
    st = torch.cuda.current_stream(v.device) if stream is None else stream
    _check(_lib.ssd_trap_scan_fwd(*(_ptr(t) for _, t in named), ctypes.byref(d),
                                  ctypes.c_void_p(st.cuda_stream)), "ssd_trap_scan_fwd")
    return y, h_final, k_final, v_final


def complex_scan_fwd(x, dt_raw, dt_bias, A_polar, B, C, D, init_state=None, *, path="auto", y=None,
                     final_state=None, return_state=True, stream=None):
    """Complex-valued scan with ET discretisation on CUDA tensors.  Returns
    ``(y, final_state)`` (the state None when not returned).

    ``x [B,L,H,P]`` and ``B, C [B,L,G,N]`` share one dtype (bf16 or fp32); B
    and C hold N/2 complex numbers as (re, im) pairs along N.  ``A_polar
    [H,2]`` = (log|A|, arg A), ``dt_raw [B,L,H]``, ``dt_bias, D [H]`` and the
    states ``[B,H,P,N]`` (complex as (re, im) pairs) are fp32.
    """
    Bt, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    if y is None:
        y = torch.empty_like(x)
    if final_state is None and return_state:
        final_state = torch.empty((Bt, H, P, N), dtype=torch.float32, device=x.device)
    named = (("x", x), ("dt_raw", dt_raw), ("dt_bias", dt_bias), ("A_polar", A_polar), ("B", B), ("C", C),
             ("D", D), ("init_state", init_state), ("y", y), ("final_state", final_state))
    _require_cuda(named)
    d = make_dims(Bt, L, H, P, N, G, 1, x.dtype, path)
    st = torch.cuda.current_stream(x.device) if stream is None else stream
    _check(_lib.ssd_complex_scan_fwd(*(_ptr(t) for _, t in named), ctypes.byref(d),
                                     ctypes.c_void_p(st.cuda_stream)), "ssd_complex_scan_fwd")
    return y, final_state


def _require_cuda(named):
    for name, t in named:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CUDA tensor")


def conv1d_silu_fwd(xbc, weight, bias=None, conv_state=None, *, nheads, headdim, ngroups, dstate,
                    x=None, B=None, C=None, conv_state_out=None, return_state=True, stream=None):
    """Causal depthwise conv1d + SiLU over the fused x | B | C channels of
    ``xbc [B,L,C]`` (``weight [C,K]``, ``bias [C]``, ``conv_state [B,K-1,C]``).
    Returns ``(x [B,L,H,P], B [B,L,G,N], C [B,L,G,N], conv_state_out)``."""
    Bt, L, Cc = xbc.shape
    K = weight.shape[1]
    if x is None:
        x = torch.empty((Bt, L, nheads, headdim), dtype=xbc.dtype, device=xbc.device)
    if B is None:
        B = torch.empty((Bt, L, ngroups, dstate), dtype=xbc.dtype, device=xbc.device)
    if C is None:
        C = torch.empty((Bt, L, ngroups, dstate), dtype=xbc.dtype, device=xbc.device)
    if conv_state_out is None and return_state:
        conv_state_out = torch.empty((Bt, K - 1, Cc), dtype=xbc.dtype, device=xbc.device)
    named = (("xbc", xbc), ("weight", weight), ("bias", bias), ("conv_state", conv_state), ("x", x),
             ("B", B), ("C", C), ("conv_state_out", conv_state_out))
    _require_cuda(named)
    d = make_dims(Bt, L, nheads, headdim, dstate, ngroups, 1, xbc.dtype)
    st = torch.cuda.current_stream(xbc.device) if stream is None else stream
    _check(_lib.ssd_conv1d_silu_fwd(*(_ptr(t) for _, t in named), ctypes.c_int32(K), ctypes.byref(d),
                                    ctypes.c_void_p(st.cuda_stream)), "ssd_conv1d_silu_fwd")
    return x, B, C, conv_state_out


def conv_scan_fwd(xbc, weight, bias, conv_state, dt_raw, dt_bias, A_log, D, init_state=None, *, nheads, headdim,
                  ngroups, dstate, chunk=256, y=None, final_state=None, conv_state_out=None, return_final_state=True,
                  return_conv_state=True, stream=None, path="auto", schedule="auto"):
    """``ssd_conv_scan_fwd``: the causal conv1d + SiLU over ``xbc [B,L,C]`` and the
    forward scan of its output, with the conv of the x channels inside the chunked
    scan kernel.  Returns ``(y [B,L,H,P], final_state, conv_state_out)``."""
    Bt, L, Cc = xbc.shape
    K = weight.shape[1]
    if y is None:
        y = torch.empty((Bt, L, nheads, headdim), dtype=xbc.dtype, device=xbc.device)
    if final_state is None and return_final_state:
        final_state = torch.empty((Bt, nheads, headdim, dstate), dtype=torch.float32, device=xbc.device)
    if conv_state_out is None and return_conv_state:
        conv_state_out = torch.empty((Bt, K - 1, Cc), dtype=xbc.dtype, device=xbc.device)
    named = (("xbc", xbc), ("weight", weight), ("bias", bias), ("conv_state", conv_state))
    rest = (("dt_raw", dt_raw), ("dt_bias", dt_bias), ("A_log", A_log), ("D", D), ("init_state", init_state),
            ("y", y), ("final_state", final_state), ("conv_state_out", conv_state_out))
    _require_cuda(named + rest)
    d = make_dims(Bt, L, nheads, headdim, dstate, ngroups, chunk, xbc.dtype, path, schedule)
    st = torch.cuda.current_stream(xbc.device) if stream is None else stream
    _check(_lib.ssd_conv_scan_fwd(*(_ptr(t) for _, t in named), ctypes.c_int32(K), *(_ptr(t) for _, t in rest),
                                  ctypes.byref(d), ctypes.c_void_p(st.cuda_stream)), "ssd_conv_scan_fwd")
    return y, final_state, conv_state_out


def gated_rmsnorm_fwd(y, z, weight, eps=1e-6, *, out=None, stream=None):
    """RMSNorm(y) * weight * SiLU(z) per token over the H*P channels of
    ``y, z [B,L,H,P]`` (``weight [H*P]`` fp32)."""
    Bt, L, H, P = y.shape
    if out is None:
        out = torch.empty_like(y)
    named = (("y", y), ("z", z), ("weight", weight), ("out", out))
    _require_cuda(named)
    d = make_dims(Bt, L, H, P, 1, 1, 1, y.dtype)
    st = torch.cuda.current_stream(y.device) if stream is None else stream
    _check(_lib.ssd_gated_rmsnorm_fwd(_ptr(y), _ptr(z), _ptr(weight), ctypes.c_float(eps), _ptr(out),
                                      ctypes.byref(d), ctypes.c_void_p(st.cuda_stream)), "ssd_gated_rmsnorm_fwd")
    return out


def ssd_scan_bwd(x, dt_raw, dt_bias, A_log, B, C, D, init_state, dy, d_final=None, *, path="auto",
                 stream=None, fp32_form=False, split_states=False):
    """Gradients of ``ssd_scan_fwd`` given ``dy`` (and ``d_final``).  Returns a
    dict of fp32 CUDA tensors: dx, ddt_raw, ddt_bias, dA_log, dB, dC, dD, d_init.
    ``fp32_form`` keeps the chunk form's fp32 contractions where its tensor-core
    form would apply (bf16, P = 64, N = 128); ``split_states`` computes that
    form's chunk states and chains in two launches instead of one walk."""
    Bt, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    f32 = dict(dtype=torch.float32, device=x.device)
    out = dict(dx=torch.empty((Bt, L, H, P), **f32), ddt_raw=torch.empty((Bt, L, H), **f32),
               ddt_bias=torch.empty((H,), **f32), dA_log=torch.empty((H,), **f32),
               dB=torch.empty((Bt, L, G, N), **f32), dC=torch.empty((Bt, L, G, N), **f32),
               dD=torch.empty((H,), **f32), d_init=torch.empty((Bt, H, P, N), **f32))
    named = (("x", x), ("dt_raw", dt_raw), ("dt_bias", dt_bias), ("A_log", A_log), ("B", B), ("C", C), ("D", D),
             ("init_state", init_state), ("dy", dy), ("d_final", d_final)) + tuple(out.items())
    _require_cuda(named)
    d = make_dims(Bt, L, H, P, N, G, 1, x.dtype, path)
    if fp32_form:
        d.flags |= BWD_FP32_FORM
    if split_states:
        d.flags |= BWD_SPLIT_STATES
    st = torch.cuda.current_stream(x.device) if stream is None else stream
    _check(_lib.ssd_scan_bwd(*(_ptr(t) for _, t in named), ctypes.byref(d), ctypes.c_void_p(st.cuda_stream)),
           "ssd_scan_bwd")
    return out
