"""fp64 CPU oracle for the forward Mamba-2 SSD scan -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
leg of ``bench.py`` may import this package.  The product library (``libssd``)
and its Python binding never import it, and nothing here imports them.

Two independent statements of what the scan computes:

* :func:`ssd_fwd` -- the sequential recurrence (``ssd_oracle.c``), the plain
  definition, one time step after another in double precision.
* :func:`ssd_quadratic` (``quadratic.py``) -- the materialised quadratic
  ("dual") form ``y = (L o C B^T)(dt o X) + D x + decay * C h0``, written with
  numpy.  It is used to pin the recurrence on tiny inputs by brute force.

Parity status of every function is stated in ``pins`` of the test suite
(``tests/test_oracle.py``); both functions are pinned there.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .quadratic import ssd_quadratic  # noqa: F401  (re-export)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libssd_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``ssd_oracle.c`` into ``oracle/_build/libssd_oracle.so``.

    Plain ``gcc -O2 -fopenmp``; portable C, so the same source builds on the
    x86 development host and on the aarch64 GPU host.
    """
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            d = ctypes.POINTER(ctypes.c_double)
            lib.ssd_oracle_fwd.restype = ctypes.c_int
            lib.ssd_oracle_fwd.argtypes = [d] * 10 + [ctypes.c_long] * 6 + [ctypes.c_int]
            lib.ssd_oracle_softplus.restype = ctypes.c_double
            lib.ssd_oracle_softplus.argtypes = [ctypes.c_double]
            lib.ssd_oracle_max_threads.restype = ctypes.c_int
            lib.ssd_oracle_max_threads.argtypes = []
            _lib = lib
    return _lib


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor -> exact float64 copy
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def softplus(z: float) -> float:
    """The oracle's softplus, ``log(1 + e^z)`` in overflow-free form."""
    return _load().ssd_oracle_softplus(float(z))


def max_threads() -> int:
    """OpenMP threads the oracle uses when ``nthreads`` is 0."""
    return _load().ssd_oracle_max_threads()


def ssd_fwd(x, dt_raw, dt_bias, A_log, B, C, D, init_state=None,
            want_final: bool = True, nthreads: int = 0):
    """Sequential fp64 recurrence.  Returns ``(y, final_state)`` as float64.

    Shapes: ``x [Bt,L,H,P]``, ``dt_raw [Bt,L,H]``, ``dt_bias/A_log/D [H]``,
    ``B/C [Bt,L,G,N]``, ``init_state [Bt,H,P,N]`` or None (zero state).
    Inputs may be numpy arrays or CPU/GPU torch tensors of any float dtype;
    they are converted exactly to float64 (bf16 and fp32 embed in fp64).
    """
    x, dt_raw, dt_bias, A_log, B, C, D = (_f64(v) for v in (x, dt_raw, dt_bias, A_log, B, C, D))
    init_state = _f64(init_state)
    Bt, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    assert dt_raw.shape == (Bt, L, H) and B.shape == (Bt, L, G, N) and C.shape == B.shape
    assert dt_bias.shape == (H,) and A_log.shape == (H,) and D.shape == (H,)
    if init_state is not None:
        assert init_state.shape == (Bt, H, P, N)
    y = np.empty_like(x)
    final = np.empty((Bt, H, P, N), dtype=np.float64) if want_final else None
    rc = _load().ssd_oracle_fwd(_ptr(x), _ptr(dt_raw), _ptr(dt_bias), _ptr(A_log), _ptr(B),
                                _ptr(C), _ptr(D), _ptr(init_state), _ptr(y), _ptr(final),
                                Bt, L, H, P, N, G, int(nthreads))
    if rc != 0:
        raise ValueError(f"ssd_oracle_fwd failed with status {rc}")
    return y, final
