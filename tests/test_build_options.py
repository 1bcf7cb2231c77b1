"""Build options (CPU only): the SSD_NVTX=1 option compiles NVTX ranges into the
host layer and nothing else, and changing the option makes the library stale."""
import os
import shutil
import subprocess

import pytest

from selective_state_space_04_gb300 import build as b


def _compile_api(tmp_path, flags):
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("no nvcc")
    obj = tmp_path / "ssd_api.o"
    subprocess.run([b.nvcc(), *b.ARCH, "-O1", "-std=c++17", "-I", b.INCLUDE, "-I", b.CSRC, *flags, "-c",
                    os.path.join(b.CSRC, "ssd_api.cu"), "-o", str(obj)], check=True)
    nm = subprocess.run(["nm", str(obj)], check=True, capture_output=True, text=True).stdout
    return nm


def test_nvtx_ranges_only_with_the_option(tmp_path):
    assert "nvtx" not in _compile_api(tmp_path, []).lower()
    assert "nvtx" in _compile_api(tmp_path, ["-DSSD_NVTX"]).lower()


def test_option_flags_follow_the_environment(monkeypatch):
    monkeypatch.delenv("SSD_NVTX", raising=False)
    assert b.option_flags() == []
    monkeypatch.setenv("SSD_NVTX", "1")
    assert b.option_flags() == ["-DSSD_NVTX"]


def test_changed_options_make_the_library_stale(tmp_path, monkeypatch):
    lib = tmp_path / "libssd.so"
    stamp = tmp_path / "flags"
    lib.write_bytes(b"")
    monkeypatch.setattr(b, "LIB_PATH", str(lib))
    monkeypatch.setattr(b, "FLAGS_STAMP", str(stamp))
    monkeypatch.setattr(b, "_inputs", lambda: [])
    stamp.write_text("")
    assert not b.is_stale([])
    assert b.is_stale(["-DSSD_NVTX"])
    stamp.write_text("-DSSD_NVTX")
    assert not b.is_stale(["-DSSD_NVTX"])
    stamp.unlink()
    assert b.is_stale([])
