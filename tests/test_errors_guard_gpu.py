"""Device-side error paths and output bounds of the prefill and decode entry points.

* Timeout path: with the testing hook kda_test_stall_next_prefill, the serial
  kernel of the next prefill call issues no chunk-record copies and its bounded
  waits give up after about 0.1 ms.  Nothing is left in flight (the kernel stops
  issuing, drains what it issued and frees its tensor memory), so the device
  error word reports KDA_ERR_TIMEOUT and the very next call, on the same context,
  matches the oracle.  No GPU fault, trap or endless wait is involved.
* KDA_VALIDATE: the optional domain check reports KDA_ERR_DOMAIN for a g outside
  [-5, 0], a beta outside [0, 1] or a non-finite input, and changes no result.
* Guard bands: out and final_state are views inside larger buffers filled with a
  sentinel (bands before and after, and padding between rows, heads and
  sequences); every sentinel byte survives the call, at ragged lengths and with
  varlen packing.
"""
import numpy as np
import pytest
import torch

import kda_inputs as ki
import oracle
from tests.parity import TOL, check_prefill, max_abs, rel_fro, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    import gated_delta_rule_gb300 as m
    m.build()
    m.load_library()
    return m


def _call(kda, t, **kw):
    return kda.kda_chunk_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["initial_state"], t["scale"],
                             cu_seqlens=t.get("cu_seqlens"), **kw)


@pytest.mark.parametrize("case", ["fixed", "varlen"])
def test_stalled_serial_kernel_times_out_and_the_next_call_is_exact(kda, case):
    if case == "fixed":
        d = ki.prefill_inputs(2, 300, 4, 128, 128, "bf16", seed=501, s0=True)
    else:
        lens = [130, 0, 64, 257]
        d = ki.prefill_inputs(1, sum(lens), 3, 128, 128, "bf16", seed=502, s0=True, n_states=len(lens))
        d["cu_seqlens"] = torch.from_numpy(ki.cu_seqlens_from_lengths(lens))
    t = to_dev(d)
    kda.kda_get_device_error()  # start from a clear word
    kda.kda_test_stall_next_prefill(True)
    _call(kda, t)
    with pytest.raises(kda.KdaError) as e:
        kda.kda_get_device_error()
    assert e.value.status == 5, e.value
    kda.kda_get_device_error()  # the word was cleared by the read
    check_prefill(kda.kda_chunk_fwd, d, label=f"after the timeout ({case})")
    kda.kda_get_device_error()


def test_stall_hook_is_consumed_by_one_call(kda):
    d = ki.prefill_inputs(1, 100, 2, 128, 128, "bf16", seed=503, s0=True)
    kda.kda_test_stall_next_prefill(True)
    kda.kda_test_stall_next_prefill(False)  # disarmed: the call runs normally
    check_prefill(kda.kda_chunk_fwd, d, label="disarmed")
    kda.kda_get_device_error()


@pytest.fixture
def validate(monkeypatch):
    monkeypatch.setenv("KDA_VALIDATE", "1")
    yield
    monkeypatch.delenv("KDA_VALIDATE", raising=False)


def _domain_error(kda):
    with pytest.raises(kda.KdaError) as e:
        kda.kda_get_device_error()
    return e.value.status


@pytest.mark.parametrize("entry", ["kda_chunk_fwd", "kda_fused_recurrent_fwd", "kda_chunk_bwd"])
def test_validate_flags_out_of_domain_inputs(kda, validate, entry):
    d = ki.prefill_inputs(1, 90, 2, 128, 128, "bf16", seed=504, s0=True)
    fn = getattr(kda, entry)

    def run(x):
        t = to_dev(x)
        if entry == "kda_chunk_bwd":
            do = torch.ones(t["v"].shape, dtype=t["v"].dtype, device="cuda")
            fn(t["q"], t["k"], t["v"], t["g"], t["beta"], t["initial_state"], t["scale"], do, None)
        else:
            fn(t["q"], t["k"], t["v"], t["g"], t["beta"], t["initial_state"], t["scale"])

    run(d)
    kda.kda_get_device_error()  # in the domain: no error
    for name, idx, val in (("g", (0, 17, 1, 5), -5.5), ("g", (0, 3, 0, 0), 0.25), ("beta", (0, 40, 1), 1.5),
                           ("beta", (0, 2, 0), -0.1), ("v", (0, 89, 1, 127), float("nan")),
                           ("q", (0, 0, 0, 3), float("inf")), ("g", (0, 60, 0, 64), float("nan"))):
        x = {k: (v.clone() if torch.is_tensor(v) else v) for k, v in d.items()}
        x[name][idx] = val
        run(x)
        assert _domain_error(kda) == 6, (name, idx, val)
    # the edges of the domain are accepted
    x = {k: (v.clone() if torch.is_tensor(v) else v) for k, v in d.items()}
    x["g"][0, 5, 0, :] = -5.0
    x["g"][0, 6, 1, :] = 0.0
    x["beta"][0, 7, :] = 0.0
    x["beta"][0, 8, :] = 1.0
    run(x)
    kda.kda_get_device_error()


def test_validate_changes_no_result(kda, monkeypatch):
    d = to_dev(ki.prefill_inputs(2, 150, 3, 128, 128, "bf16", seed=505, s0=True))
    o1, s1 = _call(kda, d)
    monkeypatch.setenv("KDA_VALIDATE", "1")
    o2, s2 = _call(kda, d)
    n_checked = kda.kda_last_launch_count()
    monkeypatch.delenv("KDA_VALIDATE")
    _call(kda, d)
    assert n_checked == kda.kda_last_launch_count() + 1  # exactly one extra (checking) kernel
    kda.kda_get_device_error()
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


def test_validate_decode_and_gate(kda, validate):
    N, H = 4, 3
    S = ki.decode_state(N, H, 128, 128, seed=506).cuda()
    x = to_dev(ki.decode_inputs(N, H, 128, 128, "bf16", seed=506, step=0))
    kda.kda_recurrent_step(S, x["q"], x["k"], x["v"], x["g"], x["beta"], scale=x["scale"])
    kda.kda_get_device_error()
    x["g"][2, 1, 7] = 1.0
    kda.kda_recurrent_step(S, x["q"], x["k"], x["v"], x["g"], x["beta"], scale=x["scale"])
    assert _domain_error(kda) == 6
    # fused gate: the logits may take any finite value, an infinite one is flagged
    d = ki.gate_logits(ki.prefill_inputs(1, 70, 2, 128, 128, "bf16", seed=507), seed=507)
    t = to_dev(d)
    t["z"][0, 3, 1, 9] = 40.0
    kda.kda_chunk_fwd_gated(t["q"], t["k"], t["v"], t["z"], t["gate_scale"], t["beta"], None, t["scale"])
    kda.kda_get_device_error()
    t["z"][0, 3, 1, 9] = float("inf")
    kda.kda_chunk_fwd_gated(t["q"], t["k"], t["v"], t["z"], t["gate_scale"], t["beta"], None, t["scale"])
    assert _domain_error(kda) == 6


# ---- guard bands ----

SENT_BF16 = -12345.0   # exactly representable in bf16
SENT_F32 = 7.0e30
BAND = 4096            # elements of sentinel before and after each view


def _guarded(shape, dtype, sentinel, pad_last=0, pad_outer=0):
    """A view of `shape` inside a sentinel-filled buffer: BAND elements before and
    after it, `pad_last` extra elements after each innermost row (a multiple of 8 so
    rows stay 16-byte aligned) and `pad_outer` extra rows per outermost index."""
    shp = list(shape)
    inner = shp[-1] + pad_last
    rows_per_outer = int(np.prod(shp[1:-1])) + pad_outer
    n = shp[0] * rows_per_outer * inner
    buf = torch.full((2 * BAND + n,), sentinel, dtype=dtype, device="cuda")
    body = buf[BAND:BAND + n].view(shp[0], rows_per_outer, inner)
    mid = body[:, : int(np.prod(shp[1:-1])), : shp[-1]]
    view = mid.reshape(shp) if len(shp) == 3 else mid.unflatten(1, tuple(shp[1:-1]))
    mask = torch.ones_like(buf, dtype=torch.bool)
    marker = torch.zeros_like(buf)
    marker[BAND:BAND + n].view(shp[0], rows_per_outer, inner)[:, : int(np.prod(shp[1:-1])), : shp[-1]] = 1
    mask &= marker == 0
    return buf, view, mask


def _untouched(buf, mask, sentinel):
    return bool((buf[mask] == sentinel).all())


@pytest.mark.parametrize("case", ["ragged", "varlen", "segments"])
def test_outputs_stay_inside_their_views(kda, case):
    if case == "ragged":
        d = ki.prefill_inputs(2, 201, 3, 128, 128, "bf16", seed=510, s0=True)
    elif case == "varlen":
        lens = [0, 1, 63, 65, 0, 130, 17]
        d = ki.prefill_inputs(1, sum(lens), 2, 128, 64, "bf16", seed=511, s0=True, n_states=len(lens))
        d["cu_seqlens"] = torch.from_numpy(ki.cu_seqlens_from_lengths(lens))
    else:  # a sequence long enough for the segment split, next to a short one
        lens = [(1152 + 128) * 64 + 333, 90]  # a first segment and two tail segments
        d = ki.prefill_inputs(1, sum(lens), 2, 128, 128, "bf16", seed=512, s0=True, n_states=len(lens))
        d["cu_seqlens"] = torch.from_numpy(ki.cu_seqlens_from_lengths(lens))
    t = to_dev(d)
    B, T, H, dk = t["q"].shape
    dv = t["v"].shape[-1]
    N = B if t.get("cu_seqlens") is None else t["cu_seqlens"].shape[0] - 1
    ob, out, om = _guarded((B, T, H, dv), torch.bfloat16, SENT_BF16, pad_last=8)
    sb, sT, sm = _guarded((N, H, dk, dv), torch.float32, SENT_F32, pad_outer=dk // 2)
    assert out.stride(-1) == 1 and out.stride(2) == dv + 8 and sT.stride(0) == (H * dk + dk // 2) * dv
    _call(kda, t, out=out, final_state=sT)
    torch.cuda.synchronize()
    kda.kda_get_device_error()
    assert _untouched(ob, om, SENT_BF16), "out wrote outside its view"
    assert _untouched(sb, sm, SENT_F32), "final_state wrote outside its view"
    o_ref, s_ref = oracle.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"], d["scale"],
                                  cu_seqlens=d.get("cu_seqlens"))
    to, ts = TOL["bf16"]
    assert max_abs(out, o_ref) <= to and rel_fro(sT, s_ref) <= ts


def test_decode_outputs_stay_inside_their_views(kda):
    N, H, dk, dv = 5, 3, 128, 128
    S0 = ki.decode_state(N, H, dk, dv, seed=513)
    x = ki.decode_inputs(N, H, dk, dv, "bf16", seed=513, step=0)
    t = to_dev(x)
    ob, out, om = _guarded((N, H, dv), torch.bfloat16, SENT_BF16, pad_last=8)
    sb, S, sm = _guarded((N, H, dk, dv), torch.float32, SENT_F32, pad_outer=8)
    S.copy_(S0.cuda())
    kda.kda_recurrent_step(S, t["q"], t["k"], t["v"], t["g"], t["beta"], scale=t["scale"], out=out)
    torch.cuda.synchronize()
    assert _untouched(ob, om, SENT_BF16) and _untouched(sb, sm, SENT_F32)
    o_ref, s_ref = oracle.decode_step(S0, x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"])
    assert max_abs(out, o_ref) <= 2e-2 and rel_fro(S, s_ref) <= 1e-2
