"""The boundary used from plain C: ``include/sp_boundary.h`` compiles as strict
ISO C, and ``tests/c_abi/sp_roundtrip.c`` (a C11 program that uses only the
CUDA runtime API and the header: no C++, no Python, no PyTorch) links against
the library's exports and, on a GPU, gives the same bits as the ctypes
binding for the same inputs."""
import glob
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

from sp_boundary_norm_gb300 import _build
from sp_boundary_norm_gb300 import workloads as wl

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "c_abi", "sp_roundtrip.c")

CC = shutil.which("gcc") or shutil.which("cc")
needs_cc = pytest.mark.skipif(CC is None, reason="no C compiler")


def _cuda_dirs():
    home = os.environ.get("CUDA_HOME") or "/usr/local/cuda"
    inc = os.path.join(home, "include")
    libs = [d for d in [os.path.join(home, "lib64")] + glob.glob(os.path.join(home, "targets",
                                                                              "*", "lib"))
            if glob.glob(os.path.join(d, "libcudart.so*"))]
    if not os.path.exists(os.path.join(inc, "cuda_runtime_api.h")) or not libs:
        pytest.skip("CUDA runtime headers or library not found")
    return inc, libs[0]


def _compile(out_dir):
    inc, libdir = _cuda_dirs()
    exe = os.path.join(str(out_dir), "sp_roundtrip")
    cmd = [CC, "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror", "-pedantic", SRC,
           "-I", _build.INCLUDE, "-I", inc, "-L", _build.OUT_DIR, "-lspboundary",
           "-L", libdir, "-lcudart", f"-Wl,-rpath,{_build.OUT_DIR}:{libdir}", "-o", exe]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    return exe


@needs_cc
@pytest.mark.parametrize("std", ["c89", "c99", "c11"])
def test_header_compiles_as_strict_iso_c(tmp_path, std):
    src = tmp_path / "use.c"
    src.write_text('#include "sp_boundary.h"\n'
                   "int main(void) { return sp_abi_version() > 0 ? 0 : 1; }\n")
    res = subprocess.run([CC, f"-std={std}", "-pedantic", "-Wall", "-Wextra", "-Werror",
                          "-fsyntax-only", "-I", _build.INCLUDE, str(src)],
                         capture_output=True, text=True)
    assert res.returncode == 0, res.stderr


@needs_cc
def test_c_consumer_compiles_and_links(lib, tmp_path):
    exe = _compile(tmp_path)
    assert os.access(exe, os.X_OK)
    # without its arguments it prints its usage and fails: no device work
    res = subprocess.run([exe], capture_output=True, text=True)
    assert res.returncode == 1 and "usage" in res.stderr


def _bits(x):
    x = x.contiguous().cpu()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().tobytes()
    return x.numpy().tobytes()


@needs_cc
@pytest.mark.gpu
@pytest.mark.parametrize("variant,bits", [
    (dict(), False),
    (dict(t=3, b=2, s=48, h=520, norm="rmsnorm", eps=1e-6, p=0.3, seed=2**40 + 9, offset=77),
     False),
    (dict(t=4, b=1, s=64, h=544, p=0.2, seed=5, offset=3), True),   # the bit-packed mask
])
def test_c_consumer_gives_the_bits_of_the_binding(lib, tmp_path, variant, bits):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    C = pytest.importorskip("_cases")
    w = wl.WORKLOADS["tiny"].with_(**variant)
    dev = C.DEV
    inp = wl.forward_inputs(w, dev)
    dy = wl.backward_inputs(w, dev)["dy"]
    ln = w.norm == "layernorm"
    with open(tmp_path / "in.bin", "wb") as f:
        for x in inp["partials"] + inp["residual"]:
            f.write(_bits(x))
        beta = inp["beta"] if ln else torch.zeros(w.h, dtype=torch.bfloat16)   # unused for RMS
        for x in (inp["bias"], inp["gamma"], beta):
            f.write(_bits(x))
        for x in dy:
            f.write(_bits(x))
    exe = _compile(tmp_path)
    res = subprocess.run([exe, str(tmp_path / "in.bin"), str(tmp_path / "out.bin"), str(w.t),
                          str(w.b), str(w.s), str(w.h), w.norm, repr(w.p), str(w.seed),
                          str(w.offset), repr(w.eps)] + (["bits"] if bits else []),
                         capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, res.stdout + res.stderr

    if bits:
        fwd, bwd = C.run_bitmask_pair(w, inp, dy, None, 1, 1)
        fwd["mask"] = fwd["mask_bits"]
    else:
        fwd = C.run_fwd(w, inp, n_gather=1)
        bwd = C.run_bwd(w, fwd, inp["gamma"], dy, None, n_gather=1)
    torch.cuda.synchronize()
    C.sp.check_device_status(dev)
    want = b"".join(
        [_bits(x) for x in fwd["z"]] + [_bits(x) for x in fwd["mask"]]
        + ([_bits(x) for x in fwd["mean"]] if ln else []) + [_bits(x) for x in fwd["rstd"]]
        + [_bits(fwd["gathered"][0])] + [_bits(x) for x in bwd["dres"]] + [_bits(bwd["dgat"][0])]
        + [_bits(bwd["dgamma"])] + ([_bits(bwd["dbeta"])] if ln else []) + [_bits(bwd["dbias"])]
        + [np.zeros(1, np.int32).tobytes()])
    got = (tmp_path / "out.bin").read_bytes()
    assert len(got) == len(want)
    assert got == want
