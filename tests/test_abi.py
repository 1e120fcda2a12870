"""The C-ABI library builds, loads and exports every entry point include/kda.h
declares, and rejects invalid arguments on the host before touching the GPU
(these calls never reach CUDA, so they run without a GPU)."""
import ctypes
import os
import re

import pytest

import gated_delta_rule_gb300 as kda
from gated_delta_rule_gb300 import KdaTensor

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 1 << 40  # a 16-byte aligned address that is never dereferenced


@pytest.fixture(scope="module")
def lib():
    kda.build()
    return kda.load_library()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "kda.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(kda_\w+)\s*\(", src, flags=re.M)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"kda_chunk_fwd", "kda_recurrent_step", "kda_get_device_error"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    assert set(kda.EXPORTED) >= set(names)


def test_status_strings(lib):
    for code, name in kda.STATUS.items():
        assert lib.kda_status_string(code).decode() == name
    assert lib.kda_status_string(99).decode() == "KDA_ERR_UNKNOWN"


def T(shape, dtype=1, addr=FAKE, stride=None):
    d = KdaTensor()
    d.data = addr
    d.dtype = dtype
    d.ndim = len(shape)
    if stride is None:
        stride, acc = [], 1
        for s in reversed(shape):
            stride.insert(0, acc)
            acc *= s
    for i, (s, st) in enumerate(zip(shape, stride)):
        d.shape[i] = s
        d.stride[i] = st
    return d


def prefill_args(B=1, Tn=64, H=2, dk=128, dv=128, dt=1):
    base = FAKE
    step = 1 << 30
    return dict(q=T([B, Tn, H, dk], dt, base), k=T([B, Tn, H, dk], dt, base + step),
                v=T([B, Tn, H, dv], dt, base + 2 * step), g=T([B, Tn, H, dk], 0, base + 3 * step),
                beta=T([B, Tn, H], 0, base + 4 * step), s0=None, cu=None,
                out=T([B, Tn, H, dv], dt, base + 5 * step), sT=None)


def call_prefill(lib, a, scale=0.1):
    r = lambda x: None if x is None else ctypes.byref(x)
    st = lib.kda_chunk_fwd(r(a["q"]), r(a["k"]), r(a["v"]), r(a["g"]), r(a["beta"]), r(a["s0"]),
                           scale, r(a["cu"]), r(a["out"]), r(a["sT"]), None)
    return st, lib.kda_last_error_message().decode()


@pytest.mark.parametrize("mutate,needle", [
    (lambda a: a.update(q=None), "q: descriptor is NULL"),
    (lambda a: a.update(k=T([1, 64, 2, 128], 0, FAKE + (1 << 30))), "k: dtype"),
    (lambda a: a.update(v=T([1, 64, 2, 96], 1, FAKE + (2 << 30))), "head dims"),
    (lambda a: a.update(g=T([1, 64, 2, 128], 1, FAKE + (3 << 30))), "g: dtype"),
    (lambda a: a.update(beta=T([1, 64, 3], 0, FAKE + (4 << 30))), "beta: size"),
    (lambda a: a.update(out=T([1, 64, 2, 128], 1, FAKE + 8)), "out: data pointer"),
    (lambda a: a.update(out=T([1, 64, 2, 128], 1, FAKE + 16)), "out overlaps q"),
    (lambda a: a.update(q=T([1, 64, 2, 128], 1, FAKE, stride=[64 * 256, 256, 129, 1])), "stride of dim 2"),
    (lambda a: a.update(q=T([1, 64, 2, 128], 1, FAKE, stride=[64 * 256, 256, 128, 2])), "innermost"),
    (lambda a: a.update(s0=T([1, 2, 128, 64], 0, FAKE + (6 << 30))), "initial_state: size"),
    (lambda a: a.update(s0=T([1, 2, 128, 128], 0, FAKE + (6 << 30)),
                        sT=T([1, 2, 128, 128], 0, FAKE + (6 << 30) + 4096)), "partly overlaps"),
    (lambda a: a.update(prefill_args(B=2), cu=T([3], 2, FAKE + (7 << 30))), "requires B == 1"),
    (lambda a: a.update(cu=T([3], 0, FAKE + (7 << 30))), "cu_seqlens: dtype"),
])
def test_prefill_rejects_invalid_arguments(lib, mutate, needle):
    a = prefill_args()
    mutate(a)
    st, msg = call_prefill(lib, a)
    assert st in (1, 2), (st, msg)
    assert needle in msg, msg


def test_prefill_rejects_nonfinite_scale(lib):
    st, msg = call_prefill(lib, prefill_args(), scale=float("inf"))
    assert st == 1 and "scale" in msg


def test_prefill_empty_problem_is_a_no_op(lib):
    a = prefill_args(B=0)
    st, msg = call_prefill(lib, a)
    assert st == 0, msg


def test_decode_rejects_invalid_arguments(lib):
    r = ctypes.byref
    N, H = 4, 2
    state = T([N, H, 128, 128], 0, FAKE)
    q = T([N, H, 128], 1, FAKE + (1 << 30))
    k = T([N, H, 128], 1, FAKE + (2 << 30))
    v = T([N, H, 128], 1, FAKE + (3 << 30))
    g = T([N, H, 128], 0, FAKE + (4 << 30))
    beta = T([N, H], 0, FAKE + (5 << 30))
    out = T([N, H, 128], 1, FAKE + 64)  # inside the state
    st = lib.kda_recurrent_step(r(state), r(q), r(k), r(v), r(g), r(beta), 1.0, r(out), None)
    assert st == 1 and "out overlaps state" in lib.kda_last_error_message().decode()
    out = T([N, H, 128], 0, FAKE + (6 << 30))
    st = lib.kda_recurrent_step(r(state), r(q), r(k), r(v), r(g), r(beta), 1.0, r(out), None)
    assert st == 1 and "out: dtype" in lib.kda_last_error_message().decode()


def test_fused_decode_requires_channel_pair_aligned_caches(lib):
    """The fused decode moves conv-cache channels in pairs: a cache that starts one
    bf16 element off a 4-byte boundary is refused before any launch."""
    r = ctypes.byref
    N, H, d = 2, 2, 128
    G = 1 << 30
    state = T([N, H, d, d], 0, FAKE)
    cq, ck, cv = (T([N, 3, H, d], 1, FAKE + i * G) for i in (1, 2, 3))
    q, k, v = (T([N, H, d], 1, FAKE + i * G) for i in (4, 5, 6))
    wq, wk, wv = (T([H, d, 4], 0, FAKE + i * G) for i in (7, 8, 9))
    g = T([N, H, d], 0, FAKE + 10 * G)
    beta = T([N, H], 0, FAKE + 11 * G)
    gate = T([N, H, d], 1, FAKE + 12 * G)
    out = T([N, H, d], 1, FAKE + 13 * G)

    def call(conv_q):
        return lib.kda_decode_step_fused(r(state), r(conv_q), r(ck), r(cv), r(q), r(k), r(v), r(wq), r(wk), r(wv),
                                         r(g), r(beta), r(gate), None, ctypes.c_float(1.0), ctypes.c_float(1e-6), r(out),
                                         None)

    st = call(T([N, 3, H, d], 1, FAKE + G + 2))
    assert st == 1 and "conv_q" in lib.kda_last_error_message().decode()
    st = call(T([N, 3, H, d], 1, FAKE + G, stride=[3 * H * d + 1, H * d, d, 1]))
    assert st == 1 and "conv_q" in lib.kda_last_error_message().decode()


def test_binding_fails_loudly_without_library(tmp_path):
    import importlib
    m = importlib.import_module("gated_delta_rule_gb300")
    saved = m._lib
    m._lib = None
    try:
        with pytest.raises(ImportError):
            m.load_library(str(tmp_path / "missing.so"))
    finally:
        m._lib = saved


def test_noalloc_rejects_requests_beyond_its_workspace(lib):
    """kda_chunk_fwd_noalloc refuses, before touching the GPU, a call whose chunk
    records would not fit its fixed workspace (1024 (chunk, head) pairs here)."""
    r = lambda x: None if x is None else ctypes.byref(x)
    a = prefill_args(B=1, Tn=4096, H=16)
    st = lib.kda_chunk_fwd_noalloc(r(a["q"]), r(a["k"]), r(a["v"]), r(a["g"]), r(a["beta"]), None,
                                   0.1, None, r(a["out"]), None, None)
    msg = lib.kda_last_error_message().decode()
    assert st == 2 and "fixed workspace" in msg, msg


def test_launch_events_argument_checks(lib):
    assert lib.kda_set_launch_events(None, -1) == 1
    assert lib.kda_set_launch_events(None, 3) == 1
    assert lib.kda_set_launch_events(None, 0) == 0  # disarm


def test_failed_call_reports_no_launches(lib):
    """A call rejected on the host enqueues nothing, and says so."""
    assert lib.kda_recurrent_step(None, None, None, None, None, None, ctypes.c_float(1.0), None,
                                  None) == 1
    assert lib.kda_last_launch_count() == 0


def test_multi_step_requires_q_and_out_together(lib):
    import torch
    r = lambda x: ctypes.byref(x)
    N, n, H, dk = 2, 3, 1, 64
    k = KdaTensor(); k.data = FAKE; k.dtype = 1; k.ndim = 4
    for i, (sh, st) in enumerate(zip((N, n, H, dk), (n * H * dk, H * dk, dk, 1))):
        k.shape[i] = sh
        k.stride[i] = st
    v, g, q = KdaTensor.from_buffer_copy(k), KdaTensor.from_buffer_copy(k), KdaTensor.from_buffer_copy(k)
    g.dtype = 0
    beta = KdaTensor(); beta.data = FAKE; beta.dtype = 0; beta.ndim = 3
    for i, (sh, st) in enumerate(zip((N, n, H), (n * H, H, 1))):
        beta.shape[i] = sh
        beta.stride[i] = st
    S = KdaTensor(); S.data = FAKE; S.dtype = 0; S.ndim = 4
    for i, (sh, st) in enumerate(zip((N, H, dk, dk), (H * dk * dk, dk * dk, dk, 1))):
        S.shape[i] = sh
        S.stride[i] = st
    st = lib.kda_recurrent_multi_step(r(S), r(q), r(k), r(v), r(g), r(beta), ctypes.c_float(1.0), None,
                                      None, None)
    assert st == 1 and b"both" in lib.kda_last_error_message()


def test_chunk_bwd_rejects_more_chunks_than_an_int_indexes(lib):
    """65536 sequences of 2^22 tokens are 2^32 chunks of 64: refused on the host
    (KDA_ERR_UNSUPPORTED) before any launch."""
    r = ctypes.byref
    B, Tn, H, d = 1 << 16, 1 << 22, 1, 64
    base = lambda i: (i + 1) << 46  # extents of up to 2^45 bytes never overlap
    q, k, v, do = (T([B, Tn, H, d], 1, base(i)) for i in range(4))
    g, dq, dk, dv, dg = (T([B, Tn, H, d], 0, base(4 + i)) for i in range(5))
    beta, dbeta = T([B, Tn, H], 0, base(9)), T([B, Tn, H], 0, base(10))
    st = lib.kda_chunk_bwd(r(q), r(k), r(v), r(g), r(beta), None, ctypes.c_float(0.125), None, r(do), None,
                           r(dq), r(dk), r(dv), r(dg), r(dbeta), None, None)
    assert st == 2, (st, lib.kda_last_error_message().decode())
    assert "64-token chunks" in lib.kda_last_error_message().decode()
