"""Parity of kda_chunk_bwd (gradients of the KDA core by the chunked form) with the
CPU oracles: torch autograd of the fp64 token loop on small cases (itself pinned to
finite differences), and the fp64 chunk-level backward of the numpy oracle (pinned
to that autograd) on sampled heads of the full prefill workload."""
import numpy as np
import pytest
import torch

import kda_inputs as ki
import oracle
from oracle import kda_numpy as kn
from tests.parity import rel_fro, to_dev

pytestmark = pytest.mark.gpu

TOL = 1e-3  # fp32 arithmetic on exact bf16 / fp32 inputs; relative Frobenius per gradient
NAMES = ("dq", "dk", "dv", "dg", "dbeta")


@pytest.fixture(scope="module")
def kda():
    import gated_delta_rule_gb300 as m
    m.build()
    m.load_library()
    return m


def _do(B, T, H, dv, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(B, T, H, dv, generator=g).to(ki.torch_dtype(dtype))


def _grads(kda, d, do, dST, need_s0=True):
    t = to_dev(d)
    return kda.kda_chunk_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["initial_state"], t["scale"],
                             do.cuda(), None if dST is None else dST.cuda(), cu_seqlens=t.get("cu_seqlens"),
                             need_initial_state_grad=need_s0)


def _check(kda, d, do, dST, label, need_s0=True):
    got = _grads(kda, d, do, dST, need_s0)
    torch.cuda.synchronize()
    ref = oracle.backward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"], d["scale"], do,
                          dST, cu_seqlens=d.get("cu_seqlens"))
    for name in NAMES + (("d_initial_state",) if need_s0 else ()):
        assert torch.isfinite(got[name]).all(), (label, name)
        err = rel_fro(got[name], ref[name])
        assert err <= TOL, f"{label} {name}: {err:.3g}"
    return got


@pytest.mark.parametrize("T", [1, 15, 16, 17, 63, 64, 65, 130, 200])
def test_chunk_bwd_lengths(kda, T):
    d = ki.prefill_inputs(2, T, 2, 64, 64, "f32", seed=200 + T, s0=True)
    g = torch.Generator().manual_seed(T)
    dST = torch.randn(2, 2, 64, 64, generator=g)
    _check(kda, d, _do(2, T, 2, 64, "f32", T), dST, f"T={T}")


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128), (128, 64), (64, 64)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_chunk_bwd_head_dims(kda, dk, dv, dtype):
    d = ki.prefill_inputs(1, 140, 2, dk, dv, dtype, seed=210, s0=True)
    g = torch.Generator().manual_seed(3)
    dST = torch.randn(1, 2, dk, dv, generator=g)
    _check(kda, d, _do(1, 140, 2, dv, dtype, 5), dST, f"{dk}x{dv} {dtype}")


@pytest.mark.parametrize("T", [1, 17, 64, 65, 200])
def test_chunk_bwd_tensor_core_lengths(kda, T):
    """d_k = d_v = 128 with bf16 inputs (the tensor-core gradient kernel) at ragged
    lengths: partial last chunks, a single token, exact multiples of the chunk."""
    d = ki.prefill_inputs(2, T, 2, 128, 128, "bf16", seed=220 + T, s0=True)
    g = torch.Generator().manual_seed(T + 1)
    dST = torch.randn(2, 2, 128, 128, generator=g)
    _check(kda, d, _do(2, T, 2, 128, "bf16", T + 2), dST, f"tc T={T}")


def test_chunk_bwd_tensor_core_varlen_and_strongest_decay(kda):
    lens = [0, 40, 1, 70, 0, 129, 64]
    cu = ki.cu_seqlens_from_lengths(lens)
    T = int(cu[-1])
    d = ki.prefill_inputs(1, T, 2, 128, 128, "bf16", seed=226, s0=True, n_states=len(lens))
    d["cu_seqlens"] = torch.from_numpy(cu)
    d["g"][..., 64:] = -5.0
    g = torch.Generator().manual_seed(17)
    dST = torch.randn(len(lens), 2, 128, 128, generator=g)
    _check(kda, d, _do(1, T, 2, 128, "bf16", 18), dST, "tc varlen, g=-5")


def test_chunk_bwd_tensor_core_strided_views(kda):
    """q, k, v as head slices of a fused projection and d_out inside a wider buffer
    (non-contiguous head and token strides), on the tensor-core kernels."""
    B, T, H, D = 1, 150, 3, 128
    d = ki.prefill_inputs(B, T, H, D, D, "bf16", seed=230, s0=True)
    fused = torch.empty(B, T, H, 3 * D, dtype=torch.bfloat16, device="cuda")
    fused[..., :D] = d["q"].cuda()
    fused[..., D:2 * D] = d["k"].cuda()
    fused[..., 2 * D:] = d["v"].cuda()
    q, k, v = fused[..., :D], fused[..., D:2 * D], fused[..., 2 * D:]
    do = _do(B, T, H, D, "bf16", 231)
    wide = torch.zeros(B, T, H, D + 64, dtype=torch.bfloat16, device="cuda")
    wide[..., :D] = do.cuda()
    dST = torch.randn(B, H, D, D, generator=torch.Generator().manual_seed(232))
    got = kda.kda_chunk_bwd(q, k, v, d["g"].cuda(), d["beta"].cuda(), d["initial_state"].cuda(), d["scale"],
                            wide[..., :D], dST.cuda())
    ref = oracle.backward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"], d["scale"], do, dST)
    for name in NAMES + ("d_initial_state",):
        err = rel_fro(got[name], ref[name])
        assert err <= TOL, f"{name}: {err:.3g}"


@pytest.mark.parametrize("beta_value", [0.0, 1.0])
def test_chunk_bwd_tensor_core_extreme_beta(kda, beta_value):
    """beta = 0 (no writes: T = I, the state only decays) and beta = 1 (full
    delta-rule overwrite) on the tensor-core kernels."""
    d = ki.prefill_inputs(1, 130, 2, 128, 128, "bf16", seed=233, s0=True)
    d["beta"] = torch.full_like(d["beta"], beta_value)
    dST = torch.randn(1, 2, 128, 128, generator=torch.Generator().manual_seed(234))
    _check(kda, d, _do(1, 130, 2, 128, "bf16", 235), dST, f"beta={beta_value}")


def test_chunk_bwd_without_states(kda):
    d = ki.prefill_inputs(1, 100, 1, 128, 128, "bf16", seed=211, s0=False)
    _check(kda, d, _do(1, 100, 1, 128, "bf16", 6), None, "no s0", need_s0=False)


def test_chunk_bwd_strongest_decay(kda):
    """Half the channels at g = -5 in every token: 16-token cumulative decays reach
    -80, the edge of the exponent range the chunked form relies on."""
    d = ki.prefill_inputs(1, 150, 2, 128, 128, "f32", seed=212, s0=True)
    d["g"][..., :64] = -5.0
    g = torch.Generator().manual_seed(9)
    dST = torch.randn(1, 2, 128, 128, generator=g)
    _check(kda, d, _do(1, 150, 2, 128, "f32", 9), dST, "g=-5")


def test_chunk_bwd_varlen(kda):
    lens = [0, 40, 1, 70, 0, 129, 64]
    cu = ki.cu_seqlens_from_lengths(lens)
    T = int(cu[-1])
    d = ki.prefill_inputs(1, T, 2, 64, 128, "bf16", seed=213, s0=True, n_states=len(lens))
    d["cu_seqlens"] = torch.from_numpy(cu)
    g = torch.Generator().manual_seed(7)
    dST = torch.randn(len(lens), 2, 64, 128, generator=g)
    _check(kda, d, _do(1, T, 2, 128, "bf16", 8), dST, "varlen")


def test_chunk_bwd_matches_token_loop_kernel_and_is_deterministic(kda):
    d = ki.prefill_inputs(1, 300, 2, 128, 128, "bf16", seed=214, s0=True)
    t = to_dev(d)
    do = _do(1, 300, 2, 128, "bf16", 10).cuda()
    a = kda.kda_chunk_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["initial_state"], t["scale"], do)
    b = kda.kda_chunk_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["initial_state"], t["scale"], do)
    r = kda.kda_backward(t["q"], t["k"], t["v"], t["g"], t["beta"], t["initial_state"], t["scale"], do)
    for name in NAMES + ("d_initial_state",):
        assert torch.equal(a[name], b[name]), name
        err = rel_fro(a[name], r[name].double().cpu().numpy())
        assert err <= TOL, f"{name}: {err:.3g}"


@pytest.mark.parametrize("problem", [(0, 3), (1, 12)])
def test_chunk_bwd_full_prefill_workload_sampled_heads(kda, problem):
    """B=2, H=16, T=4096, d=128, bf16 (the prefill workload), launched whole; one
    (sequence, head) is compared with the fp64 chunk-level oracle."""
    B, T, H, D = 2, 4096, 16, 128
    d = ki.prefill_inputs(B, T, H, D, D, "bf16", seed=215, s0=True)
    g = torch.Generator().manual_seed(11)
    dST = torch.randn(B, H, D, D, generator=g)
    do = _do(B, T, H, D, "bf16", 12)
    got = _grads(kda, d, do, dST)
    b, h = problem
    ref = kn.backward_chunked(d["q"][b, :, h], d["k"][b, :, h], d["v"][b, :, h], d["g"][b, :, h],
                              d["beta"][b, :, h], d["initial_state"][b, h], d["scale"], do[b, :, h],
                              dST[b, h], 64)
    for name in NAMES:
        x = got[name][b, :, h]
        assert torch.isfinite(x).all(), name
        err = rel_fro(x, ref[name])
        assert err <= TOL, f"{name}: {err:.3g}"
    err = rel_fro(got["d_initial_state"][b, h], ref["d_initial_state"])
    assert err <= TOL, f"d_initial_state: {err:.3g}"


def test_chunk_bwd_empty_sequence_passes_state_gradient(kda):
    """T = 0: no token gradients, and the initial-state gradient equals the final one."""
    d = ki.prefill_inputs(1, 0, 2, 64, 64, "bf16", seed=216, s0=True)
    g = torch.Generator().manual_seed(13)
    dST = torch.randn(1, 2, 64, 64, generator=g)
    got = _grads(kda, d, _do(1, 0, 2, 64, "bf16", 13), dST)
    assert torch.equal(got["d_initial_state"].cpu(), dST)
    assert got["dq"].numel() == 0 and got["dbeta"].numel() == 0
