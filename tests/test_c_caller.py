"""The C ABI from a plain C program (tests/c/host_only_caller.c): compiled
with gcc against include/nts.h and linked to libnts.so, no CUDA header and
no torch.  On the CPU it runs the argument checks; on the GPU it runs the
host-buffer MXNorm entry point on rows written by Python and must produce
the codes and scales of the device path bit for bit."""
import os
import shutil
import subprocess

import numpy as np
import pytest

from conftest import ROOT

nts = pytest.importorskip("normalization_token_split_gb300")
from normalization_token_split_gb300 import _lib  # noqa: E402


@pytest.fixture(scope="module")
def caller(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = _lib.LIB_PATH
    if not os.path.exists(lib):
        pytest.skip("libnts.so not built")
    exe = tmp_path_factory.mktemp("c") / "host_only_caller"
    subprocess.run([cc, "-O2", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c", "host_only_caller.c"), "-o", str(exe),
                    lib, "-Wl,-rpath," + os.path.dirname(lib)], check=True)
    return str(exe)


def test_argument_checks_from_c(caller):
    r = subprocess.run([caller, "--checks"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr


@pytest.mark.gpu
def test_host_only_c_caller_matches_device_path(caller, tmp_path):
    import torch
    import workloads
    T, D = 300, 2048
    X, _ = workloads.mx_inputs(T, D, seed=1234, t_frac=0.05)
    bits = workloads.bf16_bits(X)
    inp, out = tmp_path / "x.bin", tmp_path / "y.bin"
    bits.tofile(inp)
    r = subprocess.run([caller, str(inp), str(out), str(T), str(D)], capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    got = np.fromfile(out, dtype=np.uint8)
    ref = nts.mxnorm_cast(X.to("cuda:0"), None, B=32, fmt="e4m3", p=2)
    nts.check_status()
    assert np.array_equal(got[:T * D].reshape(T, D), ref.codes.cpu().numpy())
    assert np.array_equal(got[T * D:].reshape(T, D // 32), ref.scales.cpu().numpy())
    assert torch.cuda.is_available()
