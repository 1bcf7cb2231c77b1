"""libssd: GB300-native forward Mamba-2 SSD (structured state-space duality) scan.

The compute path is the C-ABI shared library ``libssd.so`` (hand-written
sm_103a CUDA kernels); :mod:`.ssd` is a thin ctypes binding over it.  The
binding is imported lazily so that :mod:`.inputs` can be used without the
compiled library.
"""
__all__ = ["ssd_scan_fwd", "ssd_scan_fwd_host", "SsdError", "inputs"]


def __getattr__(name):
    if name in ("ssd_scan_fwd", "ssd_scan_fwd_host", "SsdError", "PATH_AUTO",
                "PATH_SEQUENTIAL", "PATH_CHUNKED", "load_library"):
        from . import ssd
        return getattr(ssd, name)
    raise AttributeError(name)
