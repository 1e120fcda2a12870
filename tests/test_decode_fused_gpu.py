"""Parity of kda_decode_step_fused (short convolutions, SiLU, L2 norm, the decode
step, RMSNorm and the sigmoid output gate in one kernel) with the CPU oracle."""
import numpy as np
import pytest
import torch

import kda_inputs as ki
import oracle
from tests.parity import max_abs, rel_fro, to_dev

pytestmark = pytest.mark.gpu

EPS = 1e-6


@pytest.fixture(scope="module")
def kda():
    import gated_delta_rule_gb300 as m
    m.build()
    m.load_library()
    return m


def _step(kda, S, C, d, x, norm=True):
    t, xt = to_dev(d), to_dev(x)
    return kda.kda_decode_step_fused(S, C["q"], C["k"], C["v"], t["q"], t["k"], t["v"], xt["w_q"], xt["w_k"],
                                     xt["w_v"], t["g"], t["beta"], xt["out_gate"],
                                     xt["norm_weight"] if norm else None, scale=d["scale"], eps=EPS)


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128), (128, 64), (64, 64)])
@pytest.mark.parametrize("dtype,tol_o,tol_s", [("bf16", 2e-2, 1e-2), ("f32", 1e-4, 1e-4)])
def test_fused_steps_match_oracle(kda, dk, dv, dtype, tol_o, tol_s):
    N, H, steps = 5, 3, 6
    seed = 90 + dk + dv
    S = ki.decode_state(N, H, dk, dv, seed=seed)
    x0 = ki.fused_decode_extras(N, H, dk, dv, dtype, seed=seed)
    Sd = S.cuda()
    C = {k: x0[f"conv_{k}"].cuda() for k in "qkv"}
    S_ref = S.double().numpy()
    c_ref = {k: x0[f"conv_{k}"] for k in "qkv"}
    for st in range(steps):
        d = ki.decode_inputs(N, H, dk, dv, dtype, seed=seed, step=st)
        x = ki.fused_decode_extras(N, H, dk, dv, dtype, seed=seed, step=st)
        y = _step(kda, Sd, C, d, x, norm=(st % 2 == 0))
        y_ref, S_ref, cq, ck, cv = oracle.decode_fused(
            S_ref, c_ref["q"], c_ref["k"], c_ref["v"], d["q"], d["k"], d["v"], x["w_q"], x["w_k"], x["w_v"],
            d["g"], d["beta"], x["out_gate"], x["norm_weight"] if st % 2 == 0 else None, d["scale"], EPS)
        c_ref = {"q": cq, "k": ck, "v": cv}
        assert max_abs(y, y_ref) <= tol_o, st
        for k in "qkv":  # the caches hold raw inputs: exact
            assert np.array_equal(C[k].double().cpu().numpy(), c_ref[k]), (st, k)
    assert rel_fro(Sd, S_ref) <= tol_s


def test_fused_identity_front_end_equals_plain_step(kda):
    """Conv weights (0, 0, 0, 1) and inputs whose SiLU and norm are applied by hand:
    the state update equals kda_recurrent_step on the processed inputs."""
    N, H, dk, dv = 4, 2, 128, 128
    S = ki.decode_state(N, H, dk, dv, seed=95)
    d = ki.decode_inputs(N, H, dk, dv, "f32", seed=95, step=0)
    x = ki.fused_decode_extras(N, H, dk, dv, "f32", seed=95)
    for w in ("w_q", "w_k", "w_v"):
        x[w].zero_()
        x[w][..., 3] = 1.0
    S1 = S.cuda()
    C = {k: x[f"conv_{k}"].cuda() for k in "qkv"}
    _step(kda, S1, C, d, x)
    silu = torch.nn.functional.silu
    qa = torch.nn.functional.normalize(silu(d["q"]), dim=-1, eps=1e-6)
    ka = torch.nn.functional.normalize(silu(d["k"]), dim=-1, eps=1e-6)
    S2 = S.cuda()
    kda.kda_recurrent_step(S2, qa.cuda(), ka.cuda(), silu(d["v"]).cuda(), d["g"].cuda(), d["beta"].cuda(),
                           scale=d["scale"])
    assert rel_fro(S1, S2.double().cpu().numpy()) <= 1e-5


def test_fused_decode_sized_batch(kda):
    """256 requests x 96 heads x 128 x 128, two steps; the oracle replays sampled heads."""
    N, H, dk, dv = 256, 96, 128, 128
    seed = ki.SEED_BASE + 3
    heads = [0, 50, 95]
    Sd = ki.decode_state(N, H, dk, dv, seed=seed).cuda()
    S_ref = ki.decode_state(N, H, dk, dv, seed=seed, heads=heads).double().numpy()
    x0 = ki.fused_decode_extras(N, H, dk, dv, "bf16", seed=seed)
    C = {k: x0[f"conv_{k}"].cuda() for k in "qkv"}
    c_ref = {k: x0[f"conv_{k}"][:, :, heads] for k in "qkv"}
    for st in range(2):
        d = ki.decode_inputs(N, H, dk, dv, "bf16", seed=seed, step=st)
        x = ki.fused_decode_extras(N, H, dk, dv, "bf16", seed=seed, step=st)
        y = _step(kda, Sd, C, d, x)
        sub = lambda a: a[:, heads]
        y_ref, S_ref, cq, ck, cv = oracle.decode_fused(
            S_ref, c_ref["q"], c_ref["k"], c_ref["v"], sub(d["q"]), sub(d["k"]), sub(d["v"]),
            x["w_q"][heads], x["w_k"][heads], x["w_v"][heads], sub(d["g"]), sub(d["beta"]),
            sub(x["out_gate"]), x["norm_weight"], d["scale"], EPS)
        c_ref = {"q": cq, "k": ck, "v": cv}
        assert max_abs(y[:, heads], y_ref) <= 2e-2
    assert rel_fro(Sd[:, heads], S_ref) <= 1e-2
