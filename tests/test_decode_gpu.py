"""Parity of kda_recurrent_step (in-place decode) with the CPU oracle."""
import numpy as np
import pytest
import torch

import kda_inputs as ki
import oracle
from tests.parity import TOL, max_abs, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    import gated_delta_rule_gb300 as m
    m.build()
    m.load_library()
    return m


def _step(kda, S_dev, d):
    dev = S_dev.device
    return kda.kda_recurrent_step(S_dev, d["q"].to(dev), d["k"].to(dev), d["v"].to(dev),
                                  d["g"].to(dev), d["beta"].to(dev), scale=d["scale"])


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64), (128, 128)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_steps_small(kda, dk, dv, dtype):
    N, H, steps = 5, 3, 8
    S = ki.decode_state(N, H, dk, dv, seed=3)
    Sd = S.cuda()
    S_ref = S.double().numpy()
    to, ts = TOL[dtype]
    for s in range(steps):
        d = ki.decode_inputs(N, H, dk, dv, dtype, seed=3, step=s)
        o = _step(kda, Sd, d)
        o_ref, S_ref = oracle.decode_step(S_ref, d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"])
        assert max_abs(o, o_ref) <= to, s
    assert rel_fro(Sd, S_ref) <= ts


def test_decode_unit_key_row_exact(kda):
    """beta = 1 and k = e_i: the new state row i is v, bit for bit."""
    N, H, dk, dv = 4, 2, 128, 128
    S = ki.decode_state(N, H, dk, dv, seed=8).cuda()
    d = ki.decode_inputs(N, H, dk, dv, "bf16", seed=8, step=0)
    idx = torch.randint(0, dk, (N, H), generator=torch.Generator().manual_seed(1))
    d["k"] = torch.nn.functional.one_hot(idx, dk).to(torch.bfloat16)
    d["beta"] = torch.ones(N, H)
    _step(kda, S, d)
    rows = S.cpu()[torch.arange(N)[:, None], torch.arange(H)[None, :], idx]
    assert torch.equal(rows, d["v"].float())


def test_decode_strided_views(kda):
    """Non-contiguous head/request strides (views into larger buffers) are honoured."""
    N, H, dk, dv = 3, 4, 128, 64
    S = ki.decode_state(N, H, dk, dv, seed=4)
    d = ki.decode_inputs(N, H, dk, dv, "bf16", seed=4, step=0)
    big = torch.zeros(N, H, 2 * dk, dtype=torch.bfloat16, device="cuda")
    big[:, :, :dk] = d["q"].cuda()
    q = big[:, :, :dk]
    Sbig = torch.zeros(N, 2 * H, dk, dv, device="cuda")
    Sbig[:, ::2] = S.cuda()
    Sv = Sbig[:, ::2]
    o = kda.kda_recurrent_step(Sv, q, d["k"].cuda(), d["v"].cuda(), d["g"].cuda(),
                               d["beta"].cuda(), scale=d["scale"])
    o_ref, S_ref = oracle.decode_step(S, d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"])
    assert max_abs(o, o_ref) <= 2e-2 and rel_fro(Sv, S_ref) <= 1e-2
    assert torch.count_nonzero(Sbig[:, 1::2]) == 0


def test_decode_workload_sampled(kda):
    """Decode workload (256 requests x 96 heads x 128 x 128, 64 steps) at full size on
    the GPU; the oracle replays a sample of heads for all 64 steps."""
    w = ki.WORKLOADS[3]
    N, H, dk, dv, steps = w["N"], w["H"], w["dk"], w["dv"], w["steps"]
    seed = ki.SEED_BASE + 3
    heads = [0, 37, 95]
    Sd = ki.decode_state(N, H, dk, dv, seed=seed).cuda()
    S_ref = ki.decode_state(N, H, dk, dv, seed=seed, heads=heads).double().numpy()
    worst_o = 0.0
    for s in range(steps):
        d = ki.decode_inputs(N, H, dk, dv, "bf16", seed=seed, step=s)
        o = _step(kda, Sd, d)
        sub = {x: d[x][:, heads] for x in ("q", "k", "v", "g", "beta")}
        o_ref, S_ref = oracle.decode_step(S_ref, sub["q"], sub["k"], sub["v"], sub["g"],
                                          sub["beta"], d["scale"])
        worst_o = max(worst_o, max_abs(o[:, heads], o_ref))
    assert worst_o <= 2e-2
    assert rel_fro(Sd[:, heads], S_ref) <= 1e-2
    assert torch.isfinite(Sd).all()
