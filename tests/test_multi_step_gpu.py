"""Parity of kda_recurrent_multi_step (n decode tokens per request, state kept after
an accepted count, read once and written once) with the CPU oracle, and its
agreement with n calls of kda_recurrent_step."""
import numpy as np
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


def _inputs(N, n, H, dk, dv, dtype, seed):
    S = ki.decode_state(N, H, dk, dv, seed=seed)
    d = ki.prefill_inputs(N, n, H, dk, dv, dtype, seed=seed)
    return S, d


@pytest.mark.parametrize("n", [1, 3, 8])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128), (128, 64), (64, 64)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_multi_step_matches_oracle(kda, n, dk, dv, dtype):
    N, H = 6, 3
    S, d = _inputs(N, n, H, dk, dv, dtype, seed=50 + n)
    acc = torch.tensor([0, 1, n, n + 3, -1, max(n - 1, 0)], dtype=torch.int32)
    Sd, t = S.cuda(), to_dev(d)
    out = kda.kda_recurrent_multi_step(Sd, t["q"], t["k"], t["v"], t["g"], t["beta"], d["scale"],
                                       num_accepted=acc.cuda())
    o_ref, s_ref = oracle.multi_step(S, d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], acc)
    to, ts = TOL[dtype]
    assert max_abs(out, o_ref) <= to
    assert rel_fro(Sd, s_ref) <= ts
    assert torch.equal(Sd.cpu()[0], S[0]) and torch.equal(Sd.cpu()[4], S[4])  # nothing accepted


def test_all_accepted_equals_single_steps(kda):
    """With every token accepted, one call equals n calls of kda_recurrent_step up to
    fp32 rounding (the multi-token kernel takes four tokens per pass over the state,
    the single step one): states within 1e-5 of their scale, outputs within one bf16
    rounding step of theirs."""
    N, n, H, dk, dv = 4, 5, 2, 128, 128
    S, d = _inputs(N, n, H, dk, dv, "bf16", seed=60)
    t = to_dev(d)
    S1 = S.cuda()
    out1 = kda.kda_recurrent_multi_step(S1, t["q"], t["k"], t["v"], t["g"], t["beta"], d["scale"])
    S2 = S.cuda()
    outs = [kda.kda_recurrent_step(S2, t["q"][:, j].contiguous(), t["k"][:, j].contiguous(),
                                   t["v"][:, j].contiguous(), t["g"][:, j].contiguous(),
                                   t["beta"][:, j].contiguous(), scale=d["scale"]) for j in range(n)]
    assert (S1 - S2).abs().max().item() <= 1e-5 * S2.abs().max().item()
    o2 = torch.stack(outs, dim=1).float()
    assert ((out1.float() - o2).abs() <= 2 ** -7 * o2.abs() + 1e-5).all()


def test_verify_then_commit(kda):
    """Speculative decoding: verify the drafts with nothing accepted (state untouched),
    then commit the accepted prefix with no outputs."""
    N, n, H, dk, dv = 8, 4, 2, 128, 128
    S, d = _inputs(N, n, H, dk, dv, "bf16", seed=61)
    t = to_dev(d)
    Sd = S.cuda()
    zero = torch.zeros(N, dtype=torch.int32, device="cuda")
    out = kda.kda_recurrent_multi_step(Sd, t["q"], t["k"], t["v"], t["g"], t["beta"], d["scale"],
                                       num_accepted=zero)
    assert torch.equal(Sd.cpu(), S)
    acc = torch.tensor([4, 0, 2, 1, 3, 4, 2, 0], dtype=torch.int32)
    res = kda.kda_recurrent_multi_step(Sd, None, t["k"], t["v"], t["g"], t["beta"], d["scale"],
                                       num_accepted=acc.cuda())
    assert res is None
    o_ref, s_ref = oracle.multi_step(S, d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], acc)
    assert max_abs(out, o_ref) <= 2e-2
    assert rel_fro(Sd, s_ref) <= 1e-2


def test_replay_then_draft_in_one_call(kda):
    """The fused form: previous step's accepted tokens followed by new drafts in one
    call, num_accepted = the replayed count; the kept state and the draft outputs
    match the oracle."""
    N, H, dk, dv = 3, 2, 128, 128
    n = 6  # 2 replayed + 4 drafts
    S, d = _inputs(N, n, H, dk, dv, "bf16", seed=62)
    t = to_dev(d)
    Sd = S.cuda()
    acc = torch.full((N,), 2, dtype=torch.int32)
    out = kda.kda_recurrent_multi_step(Sd, t["q"], t["k"], t["v"], t["g"], t["beta"], d["scale"],
                                       num_accepted=acc.cuda())
    o_ref, s_ref = oracle.multi_step(S, d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], acc)
    assert max_abs(out, o_ref) <= 2e-2 and rel_fro(Sd, s_ref) <= 1e-2


def test_multi_step_workload_sampled(kda):
    """Decode-sized batch (256 requests x 96 heads x 128 x 128) with 4 tokens per
    request; the oracle replays a sample of heads."""
    N, n, H, dk, dv = 256, 4, 96, 128, 128
    seed = ki.SEED_BASE + 3
    heads = [0, 41, 95]
    Sd = ki.decode_state(N, H, dk, dv, seed=seed).cuda()
    S_ref0 = ki.decode_state(N, H, dk, dv, seed=seed, heads=heads)
    d = ki.prefill_inputs(N, n, H, dk, dv, "bf16", seed=seed + 100)
    acc = torch.randint(0, n + 1, (N,), generator=torch.Generator().manual_seed(3), dtype=torch.int32)
    t = to_dev(d)
    out = kda.kda_recurrent_multi_step(Sd, t["q"], t["k"], t["v"], t["g"], t["beta"], d["scale"],
                                       num_accepted=acc.cuda())
    sub = {x: d[x][:, :, heads] for x in ("q", "k", "v", "g", "beta")}
    o_ref, s_ref = oracle.multi_step(S_ref0, sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"],
                                     d["scale"], acc)
    assert max_abs(out[:, :, heads], o_ref) <= 2e-2
    assert rel_fro(Sd[:, heads], s_ref) <= 1e-2
