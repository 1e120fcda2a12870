"""The chunked-backward kernel bodies (csrc/kda_backward_chunk.cuh), compiled for the
host and stepped there with one thread per CUDA thread (tests/host_step), against
the oracle: the kernels' arithmetic and indexing checked without a GPU, and every
shared- and global-memory access bounds-checked under AddressSanitizer."""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

import kda_inputs as ki
import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "host_step", "kda_bwd_host_step.cpp")
CSRC = os.path.join(os.path.dirname(HERE), "gated_delta_rule_gb300", "csrc")
TOL = 1e-4  # fp32 arithmetic on fp32 inputs; relative Frobenius per gradient


def _cuda_include():
    for root in (os.environ.get("CUDA_HOME"), os.environ.get("CUDA_PATH"), "/usr/local/cuda"):
        if root and os.path.exists(os.path.join(root, "include", "cuda_runtime.h")):
            return os.path.join(root, "include")
    return None


def _compile(out, extra):
    gxx = shutil.which("g++")
    inc = _cuda_include()
    if not gxx or not inc:
        pytest.skip("needs g++ and the CUDA headers")
    cmd = [gxx, "-std=c++20", "-I", CSRC, "-I", inc, *extra, "-o", out, SRC, "-lpthread"]
    return subprocess.run(cmd, capture_output=True, text=True)


@pytest.fixture(scope="module")
def step(tmp_path_factory):
    so = str(tmp_path_factory.mktemp("host_step") / "kda_bwd_host_step.so")
    r = _compile(so, ["-O2", "-fPIC", "-shared"])
    assert r.returncode == 0, r.stderr[-2000:]
    lib = ctypes.CDLL(so)
    lib.host_step_backward.restype = ctypes.c_int
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(x):
    return None if x is None else np.ascontiguousarray(x.numpy() if hasattr(x, "numpy") else x, dtype=np.float32)


def _run(step, B, T, H, dk, dv, lens=None, s0=True, dst=True, strong=False, seed=0):
    d = ki.prefill_inputs(B, T, H, dk, dv, "f32", seed=seed, s0=s0, n_states=None if lens is None else len(lens))
    q, k, v, g, beta, S0 = (_f32(d[n]) for n in ("q", "k", "v", "g", "beta", "initial_state"))
    if strong:
        g[..., : dk // 2] = -5.0
    rng = np.random.default_rng(seed)
    cu = None if lens is None else ki.cu_seqlens_from_lengths(lens).astype(np.int32)
    N = B if lens is None else len(lens)
    do = rng.standard_normal((B, T, H, dv)).astype(np.float32)
    dST = rng.standard_normal((N, H, dk, dv)).astype(np.float32) if dst else None
    out = dict(dq=np.zeros((B, T, H, dk), np.float32), dk=np.zeros((B, T, H, dk), np.float32),
               dv=np.zeros((B, T, H, dv), np.float32), dg=np.zeros((B, T, H, dk), np.float32),
               dbeta=np.zeros((B, T, H), np.float32), d_initial_state=np.zeros((N, H, dk, dv), np.float32))
    rc = step.host_step_backward(B, T, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S0),
                                 ctypes.c_float(d["scale"]), _ptr(cu), N, _ptr(do), _ptr(dST),
                                 *(_ptr(out[n]) for n in ("dq", "dk", "dv", "dg", "dbeta", "d_initial_state")))
    assert rc == 0
    ref = oracle.backward(q, k, v, g, beta, S0, d["scale"], do, dST, cu_seqlens=cu)
    for name, x in out.items():
        assert np.isfinite(x).all(), name
        err = np.linalg.norm(x - ref[name]) / max(np.linalg.norm(ref[name]), 1e-30)
        assert err <= TOL, f"{name}: {err:.3g}"


@pytest.mark.parametrize("case", [
    dict(B=1, T=1, H=1, dk=64, dv=64),
    dict(B=2, T=64, H=2, dk=64, dv=64, s0=False, dst=False),
    dict(B=1, T=65, H=1, dk=128, dv=128),
    dict(B=1, T=150, H=2, dk=64, dv=128, strong=True),
    dict(B=1, T=130, H=1, dk=128, dv=64, strong=True),
    dict(B=1, T=181, H=2, dk=64, dv=64, lens=[0, 40, 1, 70, 0, 70]),
], ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
def test_host_stepped_kernels_match_oracle(step, case):
    _run(step, **case)


def test_host_stepped_kernels_stay_in_bounds(tmp_path):
    exe = str(tmp_path / "kda_bwd_host_step_asan")
    r = _compile(exe, ["-O0", "-fsanitize=address,undefined", "-fno-omit-frame-pointer", "-DKB_HOST_STEP_MAIN"])
    if r.returncode != 0:
        pytest.skip("sanitizer build unavailable: " + r.stderr.strip().splitlines()[-1][:200])
    p = subprocess.run([exe], capture_output=True, text=True, timeout=600,
                       env={**os.environ, "ASAN_OPTIONS": "detect_leaks=0:abort_on_error=0"})
    assert p.returncode == 0, (p.stdout[-2000:], p.stderr[-4000:])
    assert "ERROR: AddressSanitizer" not in p.stderr and "runtime error" not in p.stderr, p.stderr[-4000:]
