"""Parity of kda_backward (gradients of the KDA core) with the CPU oracle, which
differentiates a plain fp64 token loop with torch autograd (itself pinned to finite
differences)."""
import numpy as np
import pytest
import torch

import kda_inputs as ki
import oracle
from tests.parity import rel_fro, to_dev

pytestmark = pytest.mark.gpu

TOL = 1e-3  # fp32 arithmetic on exact bf16 / fp32 inputs; relative Frobenius per gradient


@pytest.fixture(scope="module")
def kda():
    import gated_delta_rule_gb300 as m
    m.build()
    m.load_library()
    return m


def _grads(kda, d, do, dST, need_s0=True):
    t = to_dev(d)
    return kda.kda_backward(t["q"], t["k"], t["v"], t["g"], t["beta"], t["initial_state"], t["scale"],
                            do.cuda(), None if dST is None else dST.cuda(), cu_seqlens=t.get("cu_seqlens"),
                            need_initial_state_grad=need_s0)


def _check(kda, d, do, dST, label, need_s0=True):
    got = _grads(kda, d, do, dST, need_s0)
    ref = oracle.backward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"], d["scale"], do,
                          dST, cu_seqlens=d.get("cu_seqlens"))
    for name in ("dq", "dk", "dv", "dg", "dbeta") + (("d_initial_state",) if need_s0 else ()):
        err = rel_fro(got[name], ref[name])
        assert err <= TOL, f"{label} {name}: {err:.3g}"
        assert torch.isfinite(got[name]).all(), (label, name)


def _do(B, T, H, dv, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(B, T, H, dv, generator=g).to(ki.torch_dtype(dtype))


@pytest.mark.parametrize("T", [1, 31, 32, 33, 100])
def test_backward_lengths(kda, T):
    d = ki.prefill_inputs(2, T, 2, 64, 64, "f32", seed=100 + T, s0=True)
    g = torch.Generator().manual_seed(T)
    dST = torch.randn(2, 2, 64, 64, generator=g)
    _check(kda, d, _do(2, T, 2, 64, "f32", T), dST, f"T={T}")


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128), (128, 64), (64, 64)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_backward_head_dims(kda, dk, dv, dtype):
    d = ki.prefill_inputs(1, 70, 2, dk, dv, dtype, seed=110, s0=True)
    _check(kda, d, _do(1, 70, 2, dv, dtype, 5), None, f"{dk}x{dv} {dtype}")


def test_backward_without_state_gradients(kda):
    d = ki.prefill_inputs(1, 45, 1, 128, 128, "bf16", seed=111, s0=False)
    _check(kda, d, _do(1, 45, 1, 128, "bf16", 6), None, "no s0", need_s0=False)


def test_backward_varlen(kda):
    lens = [0, 40, 1, 70]
    cu = ki.cu_seqlens_from_lengths(lens)
    d = ki.prefill_inputs(1, int(cu[-1]), 2, 64, 128, "bf16", seed=112, s0=True, n_states=len(lens))
    d["cu_seqlens"] = torch.from_numpy(cu)
    g = torch.Generator().manual_seed(7)
    dST = torch.randn(len(lens), 2, 64, 128, generator=g)
    _check(kda, d, _do(1, int(cu[-1]), 2, 128, "bf16", 8), dST, "varlen")


def test_backward_long_sequence(kda):
    d = ki.prefill_inputs(1, 512, 2, 128, 128, "bf16", seed=113, s0=True)
    _check(kda, d, _do(1, 512, 2, 128, "bf16", 9), None, "T=512")


@pytest.mark.parametrize("dv", [64, 128])
@pytest.mark.parametrize("H", [4, 48, 96])
def test_backward_value_slices(kda, dv, H):
    """d_v split into four or two 32-column slices, two 64-column slices, or none,
    by how many (sequence, head) pairs there are: every split matches the oracle,
    and two runs give the same bits (the partial row sums meet in a fixed order)."""
    d = ki.prefill_inputs(1, 40, H, 128, dv, "bf16", seed=120 + H + dv, s0=True)
    do = _do(1, 40, H, dv, "bf16", 11)
    _check(kda, d, do, None, f"H={H} dv={dv}")
    g1 = _grads(kda, d, do, None)
    g2 = _grads(kda, d, do, None)
    for name in ("dq", "dk", "dv", "dg", "dbeta", "d_initial_state"):
        assert torch.equal(g1[name], g2[name]), name
