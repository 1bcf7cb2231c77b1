"""CPU checks of the C ABI: the library builds, loads, exports every symbol
that include/ssd.h declares, and rejects bad arguments before touching a GPU.

No call here launches a kernel (validation runs before any CUDA call)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def libssd():
    from selective_state_space_04_gb300 import build
    path = build.build()
    from selective_state_space_04_gb300 import ssd
    return ssd


def declared_functions():
    src = open(os.path.join(ROOT, "include", "ssd.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(ssd_[a-z_0-9]+)\s*\(", src)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("ssd_scan_fwd", "ssd_scan_fwd_host", "ssd_status_string",
                     "ssd_get_device_error", "ssd_select_path"):
        assert required in names


def test_every_declared_symbol_is_exported(libssd):
    lib = libssd.lib()
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in ssd.h but not exported"


def test_abi_version_and_status_strings(libssd):
    lib = libssd.lib()
    assert lib.ssd_abi_version() == 2
    for code in range(10):
        s = lib.ssd_status_string(code)
        assert s and s != b"unknown status"
    assert lib.ssd_status_string(99) == b"unknown status"


def call(libssd, dims, ptrs=None):
    lib = libssd.lib()
    p = ptrs or {}
    fake = ctypes.c_void_p(0x10000)   # aligned, never dereferenced on these paths
    args = [p.get(k, fake) for k in ("x", "dt_raw", "dt_bias", "A_log", "B", "C", "D")]
    args += [p.get("init_state", None), p.get("y", ctypes.c_void_p(0x90000000)),
             p.get("final_state", None)]
    return lib.ssd_scan_fwd(*args, ctypes.byref(dims) if dims is not None else None, None)


def dims(libssd, **kw):
    base = dict(batch=1, seqlen=8, nheads=2, headdim=8, dstate=16, ngroups=1, chunk=16,
                dtype="bf16", path="auto")
    base.update(kw)
    return libssd.make_dims(**base)


@pytest.mark.parametrize("kw", [dict(nheads=3, ngroups=2), dict(nheads=0), dict(headdim=0),
                                dict(dstate=0), dict(ngroups=0), dict(chunk=0), dict(batch=-1),
                                dict(seqlen=-5), dict(path=7)])
def test_invalid_dims_rejected(libssd, kw):
    assert call(libssd, dims(libssd, **kw)) == 1


def test_reserved_must_be_zero(libssd):
    d = dims(libssd)
    d.reserved = 1
    assert call(libssd, d) == 1


def test_null_dims_and_pointers(libssd):
    assert call(libssd, None) == 2
    assert call(libssd, dims(libssd), {"x": None}) == 2
    assert call(libssd, dims(libssd), {"y": None}) == 2


def test_misaligned_pointer(libssd):
    assert call(libssd, dims(libssd), {"x": ctypes.c_void_p(0x10002)}) == 3


def test_output_aliasing_input(libssd):
    d = dims(libssd)
    assert call(libssd, d, {"x": ctypes.c_void_p(0x90000000), "y": ctypes.c_void_p(0x90000000)}) == 7
    # final_state overlapping B
    assert call(libssd, d, {"B": ctypes.c_void_p(0xA0000000),
                            "final_state": ctypes.c_void_p(0xA0000000)}) == 7


def test_chunked_path_needs_bf16_64_128(libssd):
    lib = libssd.lib()
    d = dims(libssd, dtype="f32", path="chunked", headdim=64, dstate=128, chunk=256)
    assert lib.ssd_select_path(ctypes.byref(d)) == -9      # SSD_ERR_UNSUPPORTED_DTYPE
    d = dims(libssd, path="chunked", headdim=32, dstate=128, chunk=256)
    assert lib.ssd_select_path(ctypes.byref(d)) == -4
    d = dims(libssd, path="chunked", headdim=64, dstate=128, chunk=100)
    assert lib.ssd_select_path(ctypes.byref(d)) == -4
    d = dims(libssd, path="chunked", nheads=3, ngroups=1, headdim=64, dstate=128, chunk=256)
    assert lib.ssd_select_path(ctypes.byref(d)) == -4


def test_unknown_dtype_rejected(libssd):
    # a dtype value outside ssd_dtype_t: SSD_ERR_UNSUPPORTED_DTYPE from every entry
    # point, before any device access
    lib = libssd.lib()
    d = dims(libssd)
    d.dtype = 7
    assert call(libssd, d) == 9
    assert lib.ssd_select_path(ctypes.byref(d)) == -9
    assert lib.ssd_launches_per_call(ctypes.byref(d)) == -9
    assert _trap_call(libssd, d) == 9
    assert _bwd_call(libssd, d) == 9
    assert _complex_call(libssd, d) == 9
    with pytest.raises(libssd.SsdError) as e:
        libssd.workspace_size((1, 64, 2, 64), 1, 128, 256, dtype=7)
    assert e.value.status == 9


def test_noalloc_refuses_other_paths_before_cuda(libssd):
    # the allocation-free entry point has only the chunked path: an explicit
    # sequential or decode request, or a split schedule, is refused before any
    # CUDA call; so is a dtype the chunked path does not take
    lib = libssd.lib()
    fake = ctypes.c_void_p(0x10000)
    args = [fake] * 7 + [None, ctypes.c_void_p(0x90000000), None]
    for path in ("sequential", "decode"):
        d = libssd.make_dims(1, 64, 2, 64, 128, 1, 64, "bf16", path=path)
        assert lib.ssd_scan_fwd_noalloc(*args, ctypes.byref(d), None) == 4
    d = libssd.make_dims(1, 64, 2, 64, 128, 1, 64, "bf16", schedule="split")
    assert lib.ssd_scan_fwd_noalloc(*args, ctypes.byref(d), None) == 4
    d = libssd.make_dims(1, 64, 2, 64, 128, 1, 64, "f32")
    assert lib.ssd_scan_fwd_noalloc(*args, ctypes.byref(d), None) == 9


def test_sequential_path_limits(libssd):
    lib = libssd.lib()
    assert lib.ssd_select_path(ctypes.byref(dims(libssd, path="sequential"))) == 1
    assert lib.ssd_select_path(ctypes.byref(dims(libssd, path="sequential", headdim=1024))) == -4


def test_empty_work_launches_nothing(libssd):
    lib = libssd.lib()
    assert lib.ssd_launches_per_call(ctypes.byref(dims(libssd, batch=0))) == 0
    assert lib.ssd_launches_per_call(ctypes.byref(dims(libssd, seqlen=0))) == 0
    # batch == 0 is a no-op that returns OK without any device access
    assert call(libssd, dims(libssd, batch=0)) == 0


def test_workspace_size_of_empty_and_sequential_work(libssd):
    assert libssd.workspace_size((2, 0, 4, 64), 1, 128, 256) == 0
    assert libssd.workspace_size((0, 64, 4, 64), 1, 128, 256) == 0
    # fp32 always takes the sequential path, which needs no scratch
    assert libssd.workspace_size((1, 64, 2, 8), 1, 16, 16, dtype="f32") == 0


def test_workspace_size_rejects_bad_dims(libssd):
    with pytest.raises(libssd.SsdError) as e:
        libssd.workspace_size((1, 64, 3, 64), 2, 128, 256)    # H % G != 0
    assert e.value.status == 1


def _ws_call(libssd, ws, ws_bytes):
    lib = libssd.lib()
    d = libssd.make_dims(1, 64, 2, 64, 128, 1, 64, "bf16")
    fake = ctypes.c_void_p(0x10000)
    args = [fake] * 7 + [None, ctypes.c_void_p(0x90000000), None]
    return lib.ssd_scan_fwd_ws(*args, ws, ctypes.c_uint64(ws_bytes), ctypes.byref(d), None)


def test_workspace_misaligned_or_overlapping_rejected_before_cuda(libssd):
    assert _ws_call(libssd, ctypes.c_void_p(0x20008), 4096) == 3   # SSD_ERR_MISALIGNED
    # overlaps y at 0x90000000
    assert _ws_call(libssd, ctypes.c_void_p(0x90000000 - 256), 4096) == 7   # SSD_ERR_ALIASING


def test_diagnostic_flag_accepted_other_flags_rejected(libssd):
    lib = libssd.lib()
    d = libssd.make_dims(1, 64, 2, 8, 16, 1, 16, "f32")
    d.flags = libssd.DIAG_STALL_HANDOFF
    assert lib.ssd_select_path(ctypes.byref(d)) == libssd.PATH_SEQUENTIAL
    d.flags = 0x200
    assert lib.ssd_select_path(ctypes.byref(d)) == -1


def test_chunk_schedule_query(libssd):
    # no chunked work: empty, or fp32 (sequential path)
    assert libssd.chunk_schedule((0, 64, 4, 64), 1, 128, 256) == "none"
    assert libssd.chunk_schedule((1, 64, 2, 8), 1, 16, 16, dtype="f32") == "none"
    # "none" without a GB300-class device (the auto path is then sequential)
    assert libssd.chunk_schedule((2, 640, 4, 64), 1, 128, 256) in ("none", "ranges", "pieces", "split")
    with pytest.raises(libssd.SsdError) as e:
        libssd.chunk_schedule((1, 64, 3, 64), 2, 128, 256)    # H % G != 0
    assert e.value.status == 1


def test_schedule_request_bits(libssd):
    lib = libssd.lib()
    for sched in ("auto", "ranges", "pieces", "split"):
        d = libssd.make_dims(1, 64, 2, 8, 16, 1, 16, "f32", schedule=sched)
        assert lib.ssd_select_path(ctypes.byref(d)) == libssd.PATH_SEQUENTIAL
    d = libssd.make_dims(1, 64, 2, 8, 16, 1, 16, "f32")
    d.flags = 0x40     # beyond the schedule request field
    assert lib.ssd_select_path(ctypes.byref(d)) == -1


def test_decode_path_selection(libssd):
    lib = libssd.lib()
    # one step: the decode path, with no scratch and one launch
    for dtype in ("bf16", "f32"):
        d = libssd.make_dims(4, 1, 8, 64, 128, 2, 256, dtype)
        assert lib.ssd_select_path(ctypes.byref(d)) == libssd.PATH_DECODE
        assert lib.ssd_launches_per_call(ctypes.byref(d)) == 1
    assert libssd.workspace_size((4, 1, 8, 64), 2, 128, 256) == 0
    assert libssd.chunk_schedule((4, 1, 8, 64), 2, 128, 256) == "none"
    # N not a multiple of 4: the auto path falls back; an explicit request is refused
    d = libssd.make_dims(4, 1, 8, 64, 126, 1, 256, "f32")
    assert lib.ssd_select_path(ctypes.byref(d)) == libssd.PATH_SEQUENTIAL
    d = libssd.make_dims(4, 1, 8, 64, 126, 1, 256, "f32", path="decode")
    assert lib.ssd_select_path(ctypes.byref(d)) == -4
    # more than one step: never the decode path
    d = libssd.make_dims(4, 2, 8, 64, 128, 1, 256, "f32", path="decode")
    assert lib.ssd_select_path(ctypes.byref(d)) == -4
    d = libssd.make_dims(4, 2, 8, 64, 128, 1, 256, "f32")
    assert lib.ssd_select_path(ctypes.byref(d)) == libssd.PATH_SEQUENTIAL


def _trap_call(libssd, dims_, **override):
    lib = libssd.lib()
    base = 0x10000000
    # 14 distinct, 16-byte aligned, widely spaced fake addresses (validation only)
    names = ["v", "k", "q", "dt", "a", "trap", "D", "h0", "k0", "v0", "y", "h_final", "k_final", "v_final"]
    ptrs = {n: ctypes.c_void_p(base + i * 0x1000000) for i, n in enumerate(names)}
    ptrs.update(override)
    return lib.ssd_trap_scan_fwd(*(ptrs[n] for n in names), ctypes.byref(dims_), None)


def test_trap_entry_validation_before_cuda(libssd):
    d = libssd.make_dims(2, 8, 4, 16, 32, 2, 1, "f32")
    assert _trap_call(libssd, d, v=None) == 2                                  # SSD_ERR_NULL_PTR
    assert _trap_call(libssd, d, dt=ctypes.c_void_p(0x30000008)) == 3          # SSD_ERR_MISALIGNED
    assert _trap_call(libssd, d, y=ctypes.c_void_p(0x10000000 + 0x100)) == 7   # y inside v: SSD_ERR_ALIASING
    # h_final overlapping h0 without being it
    assert _trap_call(libssd, d, h_final=ctypes.c_void_p(0x10000000 + 7 * 0x1000000 + 0x10)) == 7
    d2 = libssd.make_dims(2, 8, 4, 16, 32, 2, 1, "f32", path="chunked")
    assert _trap_call(libssd, d2) == 9                                         # SSD_ERR_UNSUPPORTED_DTYPE
    d3 = libssd.make_dims(2, 8, 4, 16, 32, 2, 1, "f32")
    d3.flags = 0x40                                                            # beyond the schedule field
    assert _trap_call(libssd, d3) == 1                                         # SSD_ERR_INVALID_DIMS
    # a schedule request passes the flag check (then fp32 on the chunked kernel is refused)
    d5 = libssd.make_dims(2, 8, 4, 16, 32, 2, 1, "f32", path="chunked", schedule="split")
    assert _trap_call(libssd, d5) == 9
    d4 = libssd.make_dims(2, 8, 4, 16, 30, 2, 1, "f32")                        # N % 4 != 0
    assert _trap_call(libssd, d4) == 4
    # empty batch: nothing to do, no device access
    assert _trap_call(libssd, libssd.make_dims(0, 8, 4, 16, 32, 2, 1, "f32")) == 0


def _bwd_call(libssd, dims_, **override):
    lib = libssd.lib()
    base = 0x10000000
    # 18 distinct, 16-byte aligned, widely spaced fake addresses (validation only)
    names = ["x", "dt_raw", "dt_bias", "A_log", "B", "C", "D", "init_state", "dy", "d_final",
             "dx", "ddt_raw", "ddt_bias", "dA_log", "dB", "dC", "dD", "d_init"]
    ptrs = {n: ctypes.c_void_p(base + i * 0x1000000) for i, n in enumerate(names)}
    ptrs.update(override)
    return lib.ssd_scan_bwd(*(ptrs[n] for n in names), ctypes.byref(dims_), None)


def test_bwd_entry_validation_before_cuda(libssd):
    d = libssd.make_dims(2, 8, 4, 16, 32, 2, 1, "f32")
    assert _bwd_call(libssd, d, dy=None) == 2                                   # SSD_ERR_NULL_PTR
    assert _bwd_call(libssd, d, dB=ctypes.c_void_p(0x30000008)) == 3            # SSD_ERR_MISALIGNED
    assert _bwd_call(libssd, d, dx=ctypes.c_void_p(0x10000000 + 0x100)) == 7    # dx inside x: SSD_ERR_ALIASING
    assert _bwd_call(libssd, libssd.make_dims(2, 8, 4, 16, 32, 2, 1, "f32", path="decode")) == 4
    assert _bwd_call(libssd, libssd.make_dims(2, 8, 4, 16, 32, 2, 1, "f32", schedule="pieces")) == 1
    # the chunk-parallel kernels take P <= 64, N <= 128; the sequential kernel P <= 128, N % 4 == 0
    assert _bwd_call(libssd, libssd.make_dims(1, 8, 2, 96, 32, 1, 1, "f32", path="chunked")) == 4
    assert _bwd_call(libssd, libssd.make_dims(1, 8, 2, 16, 30, 1, 1, "f32", path="sequential")) == 4
    assert _bwd_call(libssd, libssd.make_dims(1, 8, 2, 16, 160, 1, 1, "f32")) == 4
    assert _bwd_call(libssd, libssd.make_dims(0, 8, 4, 16, 32, 2, 1, "f32")) == 0   # empty: no device access


def _complex_call(libssd, dims_, **override):
    lib = libssd.lib()
    base = 0x10000000
    # 10 distinct, 16-byte aligned, widely spaced fake addresses (validation only)
    names = ["x", "dt_raw", "dt_bias", "A_polar", "B", "C", "D", "init_state", "y", "final_state"]
    ptrs = {n: ctypes.c_void_p(base + i * 0x1000000) for i, n in enumerate(names)}
    ptrs.update(override)
    return lib.ssd_complex_scan_fwd(*(ptrs[n] for n in names), ctypes.byref(dims_), None)


def test_complex_entry_validation_before_cuda(libssd):
    d = libssd.make_dims(2, 8, 4, 16, 32, 2, 1, "f32")
    assert _complex_call(libssd, d, A_polar=None) == 2                             # SSD_ERR_NULL_PTR
    assert _complex_call(libssd, d, B=ctypes.c_void_p(0x30000008)) == 3            # SSD_ERR_MISALIGNED
    assert _complex_call(libssd, d, y=ctypes.c_void_p(0x10000000 + 0x100)) == 7    # y inside x: SSD_ERR_ALIASING
    assert _complex_call(libssd, libssd.make_dims(2, 8, 4, 16, 32, 2, 1, "f32", path="chunked")) == 4
    assert _complex_call(libssd, libssd.make_dims(2, 8, 4, 16, 30, 2, 1, "f32")) == 4   # N % 4 != 0
    assert _complex_call(libssd, libssd.make_dims(2, 8, 4, 16, 1024, 2, 1, "f32")) == 4  # N > 512
    assert _complex_call(libssd, libssd.make_dims(0, 8, 4, 16, 32, 2, 1, "f32")) == 0    # empty: no device access


def _conv_scan_call(libssd, dims_, K=4, **override):
    lib = libssd.lib()
    base = 0x10000000
    names = ["xbc", "w", "bias", "state", "dt_raw", "dt_bias", "A_log", "D", "init", "y", "final", "state_out"]
    ptrs = {n: ctypes.c_void_p(base + i * 0x4000000) for i, n in enumerate(names)}
    ptrs.update(override)
    args = [ptrs[n] for n in names[:4]] + [ctypes.c_int32(K)] + [ptrs[n] for n in names[4:]]
    return lib.ssd_conv_scan_fwd(*args, ctypes.byref(dims_), None)


def test_conv_scan_entry_validation_before_cuda(libssd):
    d = libssd.make_dims(2, 64, 4, 64, 128, 1, 64, "bf16")
    assert _conv_scan_call(libssd, d, xbc=None) == 2                                   # SSD_ERR_NULL_PTR
    assert _conv_scan_call(libssd, d, w=ctypes.c_void_p(0x30000008)) == 3             # SSD_ERR_MISALIGNED
    assert _conv_scan_call(libssd, d, y=ctypes.c_void_p(0x10000000 + 0x100)) == 7     # y inside xbc
    assert _conv_scan_call(libssd, d, state_out=ctypes.c_void_p(0x10000000 + 3 * 0x4000000)) == 7   # = conv_state
    assert _conv_scan_call(libssd, d, K=5) == 1                                       # kernel size 2..4
    assert _conv_scan_call(libssd, d, K=1) == 1
    assert _conv_scan_call(libssd, libssd.make_dims(2, 64, 4, 64, 128, 1, 64, "f32")) == 9
    assert _conv_scan_call(libssd, libssd.make_dims(2, 64, 4, 64, 128, 1, 64, "bf16", path="sequential")) == 4
    d = libssd.make_dims(2, 64, 4, 64, 128, 1, 64, "bf16")
    d.flags = libssd.DIAG_STALL_HANDOFF
    assert _conv_scan_call(libssd, d) == 1
    assert _conv_scan_call(libssd, libssd.make_dims(0, 64, 4, 64, 128, 1, 64, "bf16")) == 0   # empty: no device access


def test_backward_takes_its_own_flags_only(libssd):
    # ssd_scan_bwd accepts SSD_BWD_FP32_FORM (0x200) and SSD_BWD_SPLIT_STATES (0x400)
    # beside a path and nothing else; an empty batch returns before any device access
    lib = libssd.lib()
    names = ["x", "dt_raw", "dt_bias", "A_log", "B", "C", "D", "init_state", "dy", "d_final",
             "dx", "ddt_raw", "ddt_bias", "dA_log", "dB", "dC", "dD", "d_init"]
    ptrs = [ctypes.c_void_p(0x10000000 + i * 0x1000000) for i in range(len(names))]
    d = libssd.make_dims(0, 64, 2, 64, 128, 1, 16, "bf16")
    d.flags = libssd.BWD_FP32_FORM
    assert lib.ssd_scan_bwd(*ptrs, ctypes.byref(d), None) == 0
    d.flags = libssd.BWD_SPLIT_STATES | libssd.BWD_FP32_FORM
    assert lib.ssd_scan_bwd(*ptrs, ctypes.byref(d), None) == 0
    d.flags = 0x800
    assert lib.ssd_scan_bwd(*ptrs, ctypes.byref(d), None) == 1                 # SSD_ERR_INVALID_DIMS
    # the forward entry points do not take it
    d.flags = libssd.BWD_FP32_FORM
    assert lib.ssd_select_path(ctypes.byref(d)) == -1
