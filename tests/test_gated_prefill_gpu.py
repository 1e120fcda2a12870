"""Parity of kda_chunk_fwd_gated (log-decay formed in the kernel from decay logits,
g = -5 sigmoid(A_h z)) with the CPU oracle, which forms g itself in fp64."""
import pytest
import torch

import kda_inputs as ki
import oracle
from tests.parity import TOL, max_abs, rel_fro, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    import gated_delta_rule_gb300 as m
    m.build()
    m.load_library()
    return m


def _check(kda, d, tol=None, label=""):
    t = to_dev(d)
    out, sT = kda.kda_chunk_fwd_gated(t["q"], t["k"], t["v"], t["z"], t["gate_scale"], t["beta"],
                                      t["initial_state"], t["scale"], cu_seqlens=t.get("cu_seqlens"))
    g = oracle.gate_log_decay(d["z"], d["gate_scale"])
    o_ref, s_ref = oracle.prefill(d["q"], d["k"], d["v"], g, d["beta"], d["initial_state"], d["scale"],
                                  cu_seqlens=d.get("cu_seqlens"))
    to, ts = tol or TOL["bf16" if d["q"].dtype == torch.bfloat16 else "f32"]
    eo, es = max_abs(out, o_ref), rel_fro(sT, s_ref)
    assert eo <= to and es <= ts, f"{label}: {eo:.3g} {es:.3g}"
    return out, sT


@pytest.mark.parametrize("T", [1, 63, 64, 200])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128), (128, 64), (64, 64)])
def test_gated_bf16(kda, T, dk, dv):
    d = ki.gate_logits(ki.prefill_inputs(2, T, 3, dk, dv, "bf16", seed=70 + T, s0=True), seed=70 + T)
    _check(kda, d, label=f"gated T={T} {dk}x{dv}")


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128)])
def test_gated_f32(kda, dk, dv):
    d = ki.gate_logits(ki.prefill_inputs(1, 130, 2, dk, dv, "f32", seed=71, s0=True), seed=71)
    _check(kda, d, label="gated f32")


def test_gated_extreme_logits(kda):
    """Logits far out on both sides: g saturates at -5 and 0 without NaN."""
    d = ki.gate_logits(ki.prefill_inputs(1, 100, 2, 128, 128, "bf16", seed=72, s0=True), seed=72)
    z = d["z"].float()
    z[:, :30] *= 1e4
    z[:, 30:60] *= -1e4
    d["z"] = z.to(torch.bfloat16)
    out, sT = _check(kda, d, label="gated extremes")
    assert torch.isfinite(out).all() and torch.isfinite(sT).all()


def test_gated_equals_ungated_on_same_log_decay(kda):
    """With A_h = 1 the gated call and kda_chunk_fwd on g = -5 sigmoid(z) (formed
    in fp32 here from the same bf16 logits) agree to fp32 rounding of g."""
    d = ki.gate_logits(ki.prefill_inputs(2, 150, 2, 128, 128, "bf16", seed=73, s0=True), seed=73)
    d["gate_scale"] = torch.ones_like(d["gate_scale"])
    t = to_dev(d)
    o1, s1 = kda.kda_chunk_fwd_gated(t["q"], t["k"], t["v"], t["z"], t["gate_scale"], t["beta"],
                                     t["initial_state"], t["scale"])
    g = torch.from_numpy(oracle.gate_log_decay(d["z"], d["gate_scale"])).float().cuda()
    o2, s2 = kda.kda_chunk_fwd(t["q"], t["k"], t["v"], g, t["beta"], t["initial_state"], t["scale"])
    assert max_abs(o1, o2.float().cpu().numpy()) <= 2e-3
    assert rel_fro(s1, s2.double().cpu().numpy()) <= 1e-3


def test_gated_varlen(kda):
    lens = [0, 70, 1, 129]
    cu = ki.cu_seqlens_from_lengths(lens)
    d = ki.gate_logits(ki.prefill_inputs(1, int(cu[-1]), 2, 128, 128, "bf16", seed=74, s0=True,
                                         n_states=len(lens)), seed=74)
    d["cu_seqlens"] = torch.from_numpy(cu)
    _check(kda, d, label="gated varlen")
