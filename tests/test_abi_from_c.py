"""The C ABI used from a plain C program (tests/csrc/abi_from_c.c): no Python or C++ between the
caller and the library.  On the CPU the program compiles as strict C99 against
include/flint_moe.h and runs the host-side checks; on the GPU it also runs the layer on weights
and inputs it reads from raw files, and its outputs are checked against the fp64 oracle with
the parity rule."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import synth
import sparse_moe_layer_15_b300 as fm
from tests import parity

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "csrc", "abi_from_c.c")
LIBDIR = os.path.join(ROOT, "sparse_moe_layer_15_b300")
CUDA = "/usr/local/cuda"


def build(out, with_cuda):
    fm.load_library()  # the library is built
    cmd = ["gcc", "-std=c11" if with_cuda else "-std=c99", "-Wall", "-Wextra", "-Werror",
           "-I" + os.path.join(ROOT, "include"), SRC, "-L" + LIBDIR, "-lflint_moe", "-Wl,-rpath," + LIBDIR, "-o", out]
    if with_cuda:
        cmd[4:4] = ["-DWITH_CUDA", "-I" + os.path.join(CUDA, "include")]
        cmd += ["-L" + os.path.join(CUDA, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.join(CUDA, "lib64")]
    else:
        cmd.insert(2, "-pedantic")
    subprocess.run(cmd, check=True, capture_output=True, text=True)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_c_program_compiles_as_c99_and_passes_host_checks(tmp_path):
    exe = str(tmp_path / "abi_from_c")
    build(exe, with_cuda=False)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "host checks ok"


@pytest.mark.gpu
def test_c_program_forward_matches_oracle(tmp_path):
    exe = str(tmp_path / "abi_from_c")
    build(exe, with_cuda=True)
    w = synth.flint_weights(seed=0, device="cuda:0")
    for name in ("w_router", "w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down"):
        parity.to_np_bf16(w[name]).tofile(str(tmp_path / f"{name}.bin"))
    sizes = (4, 300)  # the decode-size kernel and the tensor-core path
    xs = {}
    for T in sizes:
        xs[T] = synth.torch_normal_bf16((T, fm.HIDDEN), 5000 + T, synth.TAG_X, 1.0, device="cuda:0")
        parity.to_np_bf16(xs[T]).tofile(str(tmp_path / f"x_{T}.bin"))
    r = subprocess.run([exe, str(tmp_path)] + [str(T) for T in sizes], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "host checks and forwards ok"
    for T in sizes:
        y = np.fromfile(str(tmp_path / f"y_{T}.bin"), dtype=np.uint16).reshape(T, fm.HIDDEN)
        yh = np.fromfile(str(tmp_path / f"yh_{T}.bin"), dtype=np.uint16).reshape(T, fm.HIDDEN)
        idx = np.fromfile(str(tmp_path / f"idx_{T}.bin"), dtype=np.int32).reshape(T, fm.TOP_K)
        gw = np.fromfile(str(tmp_path / f"gw_{T}.bin"), dtype=np.float32).reshape(T, fm.TOP_K)
        assert np.array_equal(y, yh)  # the host-buffer call is the device call plus the copies
        yt = torch.from_numpy(y.view(np.int16)).view(torch.bfloat16)
        ref = parity.oracle_reference(w, xs[T], range(T))
        rep = parity.compare(ref, yt, torch.from_numpy(idx), torch.from_numpy(gw))
        assert rep["ok"], (T, rep)
