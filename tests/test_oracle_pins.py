"""Pins of the CPU oracle to facts the KDA pages and the mathematics fix.

No page prints a numeric worked example, so the oracle is pinned by an
independent formulation (explicit transition matrix), an independent algorithm
(the chunked form at several chunk sizes), closed forms of special cases,
exact invariants, a hand-worked two-token example and brute force on tiny
inputs.  ``test_planted_mistakes_are_caught`` plants typical mistakes into a
copy of the token loop and checks that the pins reject every one of them.
"""
import math
import os

import numpy as np
import pytest

import oracle
from oracle import kda_numpy as kn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# implementations under test: one problem -> (o [T, dv], S_T [dk, dv])

def cpp_oracle(q, k, v, g, beta, S0, scale):
    f = lambda a: np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    q, k, v, g, beta = map(f, (q, k, v, g, beta))
    S0 = None if S0 is None else f(S0)[None]
    o, S, _ = oracle.run_problems([0], [q.shape[0]], q, k, v, g, beta, S0, scale)
    return o, S[0]


def problem(T, dk, dv, seed, s0=True, gscale=5.0, unit_keys=True):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, dk))
    k = rng.standard_normal((T, dk))
    if unit_keys:
        q /= np.linalg.norm(q, axis=1, keepdims=True)
        k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((T, dv))
    g = -gscale / (1 + np.exp(-rng.standard_normal((T, dk))))
    beta = 1 / (1 + np.exp(-rng.standard_normal(T)))
    S0 = 0.1 * rng.standard_normal((dk, dv)) if s0 else None
    return q, k, v, g, beta, S0


def rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


# ---------------------------------------------------------------------------
# the pins, written as predicates over an implementation so that the planted
# mistake test can run them against broken copies

def pin_full_matrix(impl):
    """Explicit d_k x d_k transition (I - b k k^T) Diag(alpha) (naive DPLR form)."""
    for (T, dk, dv, seed) in [(1, 3, 2, 1), (7, 4, 3, 2), (32, 8, 5, 3), (20, 5, 8, 4)]:
        p = problem(T, dk, dv, seed)
        o, S = impl(*p, 0.7)
        o2, S2 = kn.recurrence_full_matrix(*p, 0.7)
        if not (np.allclose(o, o2, rtol=0, atol=1e-12) and np.allclose(S, S2, rtol=0, atol=1e-12)):
            return False
    return True


def pin_beta_zero(impl):
    """beta = 0: pure channel-wise decay, S_t = Diag(exp(sum_{r<=t} g_r)) S0."""
    q, k, v, g, beta, S0 = problem(19, 6, 4, 11)
    beta = np.zeros_like(beta)
    o, S = impl(q, k, v, g, beta, S0, 0.5)
    cum = np.cumsum(g, axis=0)
    o_ref = 0.5 * np.stack([(np.exp(cum[t])[:, None] * S0).T @ q[t] for t in range(19)])
    S_ref = np.exp(cum[-1])[:, None] * S0
    return rel(S, S_ref) < 1e-13 and np.abs(o - o_ref).max() < 1e-13


def pin_unit_key_exact(impl):
    """k_t a unit basis vector e_i, beta = 1: row i of S_t equals v_t exactly, so
    with q_t = e_i and scale 1 the output is v_t bit for bit."""
    rng = np.random.default_rng(5)
    T, dk, dv = 40, 6, 5
    idx = rng.integers(0, dk, T)
    k = np.eye(dk)[idx]
    q = k.copy()
    v = rng.standard_normal((T, dv))
    g = -5 / (1 + np.exp(-rng.standard_normal((T, dk))))
    beta = np.ones(T)
    S0 = rng.standard_normal((dk, dv))
    o, S = impl(q, k, v, g, beta, S0, 1.0)
    return np.array_equal(o, v) and np.array_equal(S[idx[-1]], v[-1])


def pin_linear_attention(impl):
    """Orthonormal keys, g = 0, beta = 1, S0 = 0 (T <= d_k): the delta rule never
    erases, so o_t = scale * sum_{j<=t} (q_t . k_j) v_j (causal linear attention,
    including j = t)."""
    rng = np.random.default_rng(7)
    T, dk, dv = 8, 8, 3
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    k = Qm.T[:T]
    q = rng.standard_normal((T, dk))
    v = rng.standard_normal((T, dv))
    g = np.zeros((T, dk))
    beta = np.ones(T)
    o, S = impl(q, k, v, g, beta, None, 0.3)
    o_ref = 0.3 * np.stack([sum((q[t] @ k[j]) * v[j] for j in range(t + 1)) for t in range(T)])
    S_ref = k.T @ v
    return np.abs(o - o_ref).max() < 1e-13 and np.abs(S - S_ref).max() < 1e-13


def pin_repeated_key(impl):
    """One key repeated, beta = 1, g = 0: after every step S_t^T k = v_t."""
    rng = np.random.default_rng(9)
    T, dk, dv = 12, 5, 4
    kk = rng.standard_normal(dk)
    kk /= np.linalg.norm(kk)
    k = np.tile(kk, (T, 1))
    v = rng.standard_normal((T, dv))
    o, S = impl(k.copy(), k, v, np.zeros((T, dk)), np.ones(T), rng.standard_normal((dk, dv)), 1.0)
    return np.abs(o - v).max() < 1e-13


def pin_chunkwise(impl):
    """An independent chunked implementation agrees at every chunk size, partial tails included."""
    for (T, dk, dv, seed) in [(37, 8, 6, 21), (64, 16, 16, 22), (130, 8, 4, 23)]:
        p = problem(T, dk, dv, seed)
        o, S = impl(*p, 0.25)
        for C in (1, 2, 4, 16, 32, 64):
            oc, Sc = kn.chunkwise(*p, 0.25, C)
            if rel(o, oc) > 1e-10 or rel(S, Sc) > 1e-10:
                return False
    return True


def pin_segment_composition(impl):
    """A segment acts as S_out = M S_in + S~ with M and S~ independent of S_in."""
    q, k, v, g, beta, S0 = problem(25, 6, 4, 31)
    M, St = kn.segment_transition(k, g, beta, v)
    _, S = impl(q, k, v, g, beta, S0, 1.0)
    return rel(S, M @ S0 + St) < 1e-12


def pin_hand_example(impl):
    vals = {}
    with open(os.path.join(GOLDEN, "kda_two_steps_by_hand.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            name, rest = line.split(":", 1)
            vals[name.strip()] = np.array([float(x) for x in rest.split()])
    o, S = impl(vals["q"].reshape(2, 2), vals["k"].reshape(2, 2), vals["v"].reshape(2, 2),
                vals["g"].reshape(2, 2), vals["beta"], vals["S0"].reshape(2, 2), 1.0)
    return (np.abs(o - vals["o"].reshape(2, 2)).max() < 1e-14 and
            np.abs(S - vals["S_T"].reshape(2, 2)).max() < 1e-14)


PINS = [pin_full_matrix, pin_beta_zero, pin_unit_key_exact, pin_linear_attention,
        pin_repeated_key, pin_chunkwise, pin_segment_composition, pin_hand_example]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_cpp_oracle_pins(pin):
    assert pin(cpp_oracle)


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_numpy_loop_pins(pin):
    assert pin(kn.recurrence_three_step)


def test_contraction_bound():
    """With ||k|| = 1 and beta in [0, 1] every transition has spectral norm <= 1, so
    ||S_t||_2 <= ||S_{t-1}||_2 + beta_t ||v_t||."""
    q, k, v, g, beta, S0 = problem(50, 8, 8, 41)
    prev = np.linalg.norm(S0, 2)
    for t in range(1, 51):
        _, S = cpp_oracle(q[:t], k[:t], v[:t], g[:t], beta[:t], S0, 1.0)
        cur = np.linalg.norm(S, 2)
        assert cur <= prev + beta[t - 1] * np.linalg.norm(v[t - 1]) + 1e-12
        prev = cur


def test_resume_equals_straight_run():
    """Prefill of T tokens equals prefill of T1 tokens then T - T1 more from S_{T1}."""
    p = problem(45, 8, 6, 51)
    o, S = cpp_oracle(*p, 0.5)
    q, k, v, g, beta, S0 = p
    o1, S1 = cpp_oracle(q[:17], k[:17], v[:17], g[:17], beta[:17], S0, 0.5)
    o2, S2 = cpp_oracle(q[17:], k[17:], v[17:], g[17:], beta[17:], S1, 0.5)
    assert np.array_equal(np.concatenate([o1, o2]), o) and np.array_equal(S2, S)


def test_cpp_matches_numpy_loop_bitwise_shape_mix():
    for (T, dk, dv, seed) in [(0, 4, 4, 1), (1, 64, 64, 2), (33, 128, 64, 3), (9, 64, 128, 4)]:
        p = problem(T, dk, dv, seed)
        o, S = cpp_oracle(*p, 0.125)
        o2, S2 = kn.recurrence_three_step(*p, 0.125)
        assert o.shape == (T, dv) and S.shape == (dk, dv)
        assert np.abs(o - o2).max(initial=0) < 1e-13 and np.abs(S - S2).max() < 1e-13


def test_empty_sequence_keeps_initial_state():
    p = problem(0, 4, 3, 3)
    o, S = cpp_oracle(*p, 1.0)
    assert o.shape == (0, 3) and np.array_equal(S, p[5])


def test_varlen_packing_matches_separate_runs():
    import torch
    import kda_inputs as ki
    lens = [5, 0, 17, 64, 1]
    cu = ki.cu_seqlens_from_lengths(lens)
    d = ki.prefill_inputs(1, int(cu[-1]), 3, 16, 8, "bf16", seed=77, s0=True, n_states=len(lens))
    out, ST = oracle.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"],
                             d["scale"], cu_seqlens=torch.from_numpy(cu))
    for n in range(len(lens)):
        a, b = int(cu[n]), int(cu[n + 1])
        sl = lambda t: t[:, a:b]
        o1, S1 = oracle.prefill(sl(d["q"]), sl(d["k"]), sl(d["v"]), sl(d["g"]), sl(d["beta"]),
                                d["initial_state"][n:n + 1], d["scale"])
        assert np.array_equal(out[:, a:b], o1) and np.array_equal(ST[n:n + 1], S1)


def test_decode_step_is_one_token_prefill():
    import kda_inputs as ki
    S = ki.decode_state(3, 2, 16, 8, seed=5)
    d = ki.decode_inputs(3, 2, 16, 8, "bf16", seed=5, step=0)
    o, S1 = oracle.decode_step(S, d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"])
    o2, S2 = oracle.prefill(d["q"][:, None], d["k"][:, None], d["v"][:, None], d["g"][:, None],
                            d["beta"][:, None], S, d["scale"])
    assert np.array_equal(o, o2[:, 0]) and np.array_equal(S1, S2)


def test_gate_closed_forms():
    """g = -5 sigmoid(A z): -2.5 at z = 0, -5 and 0 in the limits, g(-z) = -5 - g(z),
    strictly inside (-5, 0) for finite A z, and A scales the logit, not the output."""
    z = np.array([[[[0.0, 1e6, -1e6, 1.3, -1.3, 0.2]]]])
    A = np.array([1.0])
    g = oracle.gate_log_decay(z, A)[0, 0, 0]
    assert g[0] == -2.5 and g[1] == -5.0 and g[2] == 0.0
    assert math.isclose(g[3] + g[4], -5.0, abs_tol=1e-15)
    assert -5.0 < g[5] < 0.0
    assert math.isclose(g[3], -5.0 / (1.0 + math.exp(-1.3)), rel_tol=1e-15)
    g2 = oracle.gate_log_decay(z, np.array([2.0]))[0, 0, 0]
    assert math.isclose(g2[5], oracle.gate_log_decay(2 * z, A)[0, 0, 0][5], rel_tol=1e-15)
    zz = np.zeros((1, 1, 2, 3))
    assert np.all(oracle.gate_log_decay(zz, np.array([0.5, 3.0])) == -2.5)


def test_checkpoints_match_numpy_token_loop():
    """Checkpoint j is the numpy loop's state after (j + 1) * ck tokens; rows past a
    sequence's end are NaN."""
    import kda_inputs as ki
    d = ki.prefill_inputs(2, 17, 2, 8, 4, "bf16", seed=8, s0=True)
    ck, C = 5, 4
    res = oracle.prefill_checkpoints(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"],
                                     d["scale"], ck, C)
    f = lambda x: np.asarray(x.double(), dtype=np.float64)
    q, k, v, g, beta, S0 = map(f, (d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"]))
    for b in range(2):
        for h in range(2):
            for j in range(3):
                n_tok = (j + 1) * ck
                _, s_ref = kn.recurrence_three_step(q[b, :n_tok, h], k[b, :n_tok, h], v[b, :n_tok, h],
                                                    g[b, :n_tok, h], beta[b, :n_tok, h], S0[b, h], d["scale"])
                assert np.allclose(res[b * C + j, h], s_ref, rtol=0, atol=1e-12)
            assert np.isnan(res[b * C + 3]).all()  # 17 tokens hold three checkpoints of 5


def test_decode_fused_special_cases():
    """Fused decode front/back ends: an identity convolution (weight only on the
    current input) with inputs whose SiLU is known; q, k come out unit-length; the
    cache shifts by one; a zero gate logit halves, and the RMS norm makes the output
    of a constant vector equal to the norm weight."""
    rng = np.random.default_rng(3)
    N, H, dk, dv = 2, 2, 4, 3
    S = rng.standard_normal((N, H, dk, dv))
    cq, ck = rng.standard_normal((N, 3, H, dk)), rng.standard_normal((N, 3, H, dk))
    cv = rng.standard_normal((N, 3, H, dv))
    q, k, v = rng.standard_normal((N, H, dk)), rng.standard_normal((N, H, dk)), rng.standard_normal((N, H, dv))
    w_id_k = np.zeros((H, dk, 4)); w_id_k[..., 3] = 1.0
    w_id_v = np.zeros((H, dv, 4)); w_id_v[..., 3] = 1.0
    g = -rng.uniform(0, 5, (N, H, dk)); beta = rng.uniform(0, 1, (N, H))
    gate = np.zeros((N, H, dv)); wn = rng.uniform(0.5, 2, dv)
    y, S1, nq, nk, nv = oracle.decode_fused(S, cq, ck, cv, q, k, v, w_id_k, w_id_k, w_id_v, g, beta,
                                            gate, wn, 0.5, 0.0)
    silu = lambda x: x / (1 + np.exp(-x))
    qa, ka = silu(q), silu(k)
    qa /= np.linalg.norm(qa, axis=-1, keepdims=True)
    ka /= np.linalg.norm(ka, axis=-1, keepdims=True)
    for n in range(N):
        for h in range(H):
            o, s_ref = kn.recurrence_three_step(qa[n, h][None], ka[n, h][None], silu(v[n, h])[None],
                                                g[n, h][None], beta[n, h][None], S[n, h], 0.5)
            assert np.allclose(S1[n, h], s_ref, rtol=0, atol=1e-12)
            o = o[0]
            assert np.allclose(y[n, h], o / np.sqrt(np.mean(o * o)) * wn * 0.5, rtol=1e-12, atol=0)
    assert np.array_equal(nq[:, :2], cq[:, 1:]) and np.array_equal(nq[:, 2], q)
    assert np.array_equal(nv[:, 2], v)
    # a convolution that only sees the oldest cached input
    w_old = np.zeros((H, dk, 4)); w_old[..., 0] = 2.0
    y2, S2, *_ = oracle.decode_fused(S, cq, ck, cv, q, k, v, w_old, w_old, np.concatenate(
        [np.zeros((H, dv, 3)), np.ones((H, dv, 1))], -1), g, beta, gate, None, 0.5, 0.0)
    qa2 = silu(2.0 * cq[:, 0]); qa2 /= np.linalg.norm(qa2, axis=-1, keepdims=True)
    ka2 = silu(2.0 * ck[:, 0]); ka2 /= np.linalg.norm(ka2, axis=-1, keepdims=True)
    _, s2 = kn.recurrence_three_step(qa2[0, 0][None], ka2[0, 0][None], silu(v[0, 0])[None], g[0, 0][None],
                                     beta[0, 0][None], S[0, 0], 0.5)
    assert np.allclose(S2[0, 0], s2, rtol=0, atol=1e-12)


def test_backward_matches_finite_differences():
    """The backward oracle's gradients equal central finite differences of the C++
    forward oracle's loss <o, d_out> + <S_T, d_final_state>, for every input."""
    rng = np.random.default_rng(11)
    B, T, H, dk, dv = 1, 5, 1, 3, 2
    q = rng.standard_normal((B, T, H, dk)); k = rng.standard_normal((B, T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, dv)); g = -rng.uniform(0.05, 2.0, (B, T, H, dk))
    beta = rng.uniform(0.1, 0.9, (B, T, H)); S0 = rng.standard_normal((B, H, dk, dv))
    do = rng.standard_normal((B, T, H, dv)); dST = rng.standard_normal((B, H, dk, dv))
    scale = 0.7
    gr = oracle.backward(q, k, v, g, beta, S0, scale, do, dST)

    def loss(q, k, v, g, beta, S0):
        o, ST = oracle.prefill(q, k, v, g, beta, S0, scale)
        return float(np.sum(o * do) + np.sum(ST * dST))

    args = dict(q=q, k=k, v=v, g=g, beta=beta, S0=S0)
    names = dict(q="dq", k="dk", v="dv", g="dg", beta="dbeta", S0="d_initial_state")
    eps = 1e-6
    for a, arr in args.items():
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            p, m = {x: y.copy() for x, y in args.items()}, {x: y.copy() for x, y in args.items()}
            p[a][idx] += eps
            m[a][idx] -= eps
            num[idx] = (loss(**p) - loss(**m)) / (2 * eps)
        assert np.allclose(gr[names[a]], num, rtol=1e-6, atol=1e-7), a


def test_multi_step_matches_numpy_token_loop():
    """Multi-token decode: every request's outputs are those of the numpy three-step
    loop over its n tokens, and the kept state is that loop stopped after the
    accepted count (clamped to [0, n])."""
    import kda_inputs as ki
    N, n, H, dk, dv = 5, 4, 2, 16, 8
    S = ki.decode_state(N, H, dk, dv, seed=6).double().numpy()
    d = ki.prefill_inputs(N, n, H, dk, dv, "bf16", seed=6)
    acc = np.array([0, 1, 4, 7, -2])
    out, Sk = oracle.multi_step(S, d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], acc)
    f = lambda x: np.asarray(x.double() if hasattr(x, "double") else x, dtype=np.float64)
    q, k, v, g, beta = map(f, (d["q"], d["k"], d["v"], d["g"], d["beta"]))
    for i in range(N):
        a = min(max(int(acc[i]), 0), n)
        for h in range(H):
            o_ref, _ = kn.recurrence_three_step(q[i, :, h], k[i, :, h], v[i, :, h], g[i, :, h],
                                                beta[i, :, h], S[i, h], d["scale"])
            _, s_ref = kn.recurrence_three_step(q[i, :a, h], k[i, :a, h], v[i, :a, h], g[i, :a, h],
                                                beta[i, :a, h], S[i, h], d["scale"])
            assert np.allclose(out[i, :, h], o_ref, rtol=0, atol=1e-12)
            assert np.allclose(Sk[i, h], s_ref, rtol=0, atol=1e-12)
    assert np.array_equal(Sk[0], S[0])  # nothing accepted: the state is untouched


def test_multi_step_outputs_do_not_depend_on_acceptance():
    import kda_inputs as ki
    S = ki.decode_state(2, 1, 8, 8, seed=7).double().numpy()
    d = ki.prefill_inputs(2, 3, 1, 8, 8, "f32", seed=7)
    o1, _ = oracle.multi_step(S, d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, np.array([0, 0]))
    o2, S2 = oracle.multi_step(S, d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, None)
    assert np.array_equal(o1, o2)
    _, S3 = oracle.multi_step(S, None, d["k"], d["v"], d["g"], d["beta"], 1.0, np.array([3, 3]))
    assert np.array_equal(S2, S3)


# ---------------------------------------------------------------------------
# planted mistakes: each broken copy of the loop must fail at least one pin

def _loop(variant):
    def impl(q, k, v, g, beta, S0, scale):
        q, k, v, g, beta = (np.asarray(a, dtype=np.float64) for a in (q, k, v, g, beta))
        dk, dv = k.shape[1], v.shape[1]
        S = np.zeros((dk, dv)) if S0 is None else np.array(S0, dtype=np.float64)
        o = np.zeros((q.shape[0], dv))
        for t in range(q.shape[0]):
            a = np.exp(-g[t]) if variant == "decay_sign" else np.exp(g[t])
            if variant == "read_before_update":
                o[t] = scale * (S.T @ q[t])
            if variant != "decay_after_write":
                S = S * a[:, None]
            base = S
            sgn = 1.0 if variant == "correction_sign" else -1.0
            S = S + sgn * beta[t] * np.outer(k[t], k[t] @ base)
            wb = 1.0 if variant == "write_without_beta" else beta[t]
            S = S + wb * np.outer(k[t], v[t])
            if variant == "decay_after_write":
                S = S * a[:, None]
            if variant == "decay_on_columns" and dk == dv:
                S = S * (a[None, :] / a[:, None])
            if variant == "readout_transposed" and dk == dv:
                o[t] = scale * (S @ q[t])
            elif variant == "drop_scale":
                o[t] = S.T @ q[t]
            elif variant != "read_before_update":
                o[t] = scale * (S.T @ q[t])
        return o, S
    return impl


@pytest.mark.parametrize("variant", ["read_before_update", "decay_after_write", "decay_sign",
                                     "correction_sign", "write_without_beta", "decay_on_columns",
                                     "readout_transposed", "drop_scale"])
def test_planted_mistakes_are_caught(variant):
    assert all(pin(_loop("none")) for pin in PINS)
    assert not all(pin(_loop(variant)) for pin in PINS), variant


@pytest.mark.parametrize("T,C,with_state", [(11, 1, True), (11, 4, True), (70, 16, False), (70, 64, True),
                                            (64, 64, True), (1, 64, False)])
def test_chunked_backward_matches_token_autograd(T, C, with_state):
    """The chunk-by-chunk hand derivative of the chunked form gives the same gradients
    as reverse-mode differentiation of the token recurrence (itself pinned to finite
    differences), for full, partial and single-token chunks, with and without an
    initial state and a final-state gradient."""
    rng = np.random.default_rng(T * 100 + C)
    B, H, dk, dv = 1, 1, 8, 5
    q = rng.standard_normal((B, T, H, dk)); k = rng.standard_normal((B, T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, dv)); g = -rng.uniform(0.01, 0.5, (B, T, H, dk))
    beta = rng.uniform(0.1, 0.9, (B, T, H)); do = rng.standard_normal((B, T, H, dv))
    S0 = rng.standard_normal((B, H, dk, dv)) if with_state else None
    dST = rng.standard_normal((B, H, dk, dv)) if with_state else None
    ref = oracle.backward(q, k, v, g, beta, S0, 0.6, do, dST)
    got = kn.backward_chunked(q[0, :, 0], k[0, :, 0], v[0, :, 0], g[0, :, 0], beta[0, :, 0],
                              None if S0 is None else S0[0, 0], 0.6, do[0, :, 0],
                              None if dST is None else dST[0, 0], C)
    for name in ("dq", "dk", "dv", "dg", "dbeta"):
        assert np.allclose(got[name], ref[name][0, :, 0], rtol=1e-9, atol=1e-10), name
    assert np.allclose(got["d_initial_state"], ref["d_initial_state"][0, 0], rtol=1e-9, atol=1e-10)


def test_numpy_oracle_keeps_fp64_torch_inputs_exact():
    """fp64 torch tensors reach the numpy oracle unrounded: the result equals the one
    from the same numbers as numpy arrays bit for bit, and differs from the result on
    the fp32-rounded numbers (so a silent fp32 round trip would be caught)."""
    import torch
    p = problem(9, 6, 5, 11)
    o_np, S_np = kn.recurrence_three_step(*p, 0.5)
    tp = [None if a is None else torch.from_numpy(np.array(a)) for a in p]
    o_t, S_t = kn.recurrence_three_step(*tp, 0.5)
    assert np.array_equal(o_t, o_np) and np.array_equal(S_t, S_np)
    rounded = [None if a is None else np.asarray(a, dtype=np.float32).astype(np.float64) for a in p]
    o_r, _ = kn.recurrence_three_step(*rounded, 0.5)
    assert not np.array_equal(o_r, o_np)
