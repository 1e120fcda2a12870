"""Launch accounting (kda_set_launch_events / kda_last_launch_count): the number of
kernels each path enqueues, and per-kernel event times that add up to the call."""
import pytest
import torch

import kda_inputs as ki
from tests.parity import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    import gated_delta_rule_gb300 as m
    m.build()
    m.load_library()
    return m


def _events(n, stream):
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in ev:
        e.record(stream)  # creates the handle
    stream.synchronize()
    return ev


def _prefill(kda, entry, d, stream):
    t = to_dev(d)
    getattr(kda, entry)(t["q"], t["k"], t["v"], t["g"], t["beta"], t["initial_state"],
                        t["scale"], cu_seqlens=t.get("cu_seqlens"), stream=stream)


@pytest.mark.parametrize("entry,dtype,varlen,want", [
    ("kda_chunk_fwd", "bf16", False, 2),         # chunk prep, serial chunk loop
    ("kda_chunk_fwd", "bf16", True, 4),          # + cu_seqlens check, chunk offsets
    ("kda_chunk_fwd_noalloc", "bf16", False, 2),
    ("kda_chunk_fwd", "f32", False, 1),          # fp32 inputs: the recurrent kernel
    ("kda_fused_recurrent_fwd", "bf16", True, 2),
])
def test_prefill_launch_counts_and_times(kda, entry, dtype, varlen, want):
    stream = torch.cuda.Stream()
    if varlen:
        lens = [70, 0, 130]
        cu = ki.cu_seqlens_from_lengths(lens)
        d = ki.prefill_inputs(1, int(cu[-1]), 2, 128, 128, dtype, seed=30, s0=True,
                              n_states=len(lens))
        d["cu_seqlens"] = torch.from_numpy(cu)
    else:
        d = ki.prefill_inputs(2, 300, 2, 128, 128, dtype, seed=30, s0=True)
    ev = _events(6, stream)
    outer = _events(2, stream)
    kda.kda_set_launch_events(ev)
    with torch.cuda.stream(stream):
        outer[0].record(stream)
        _prefill(kda, entry, d, stream)
        outer[1].record(stream)
    stream.synchronize()
    kda.kda_get_device_error(stream)
    assert kda.kda_last_launch_count() == want
    parts = [ev[i].elapsed_time(ev[i + 1]) for i in range(want)]
    assert all(p > 0 for p in parts)
    assert sum(parts) <= outer[0].elapsed_time(outer[1]) * 1.001 + 1e-3
    # the arm lasts for one call: the next call leaves the events where they were
    stamp = ev[0].elapsed_time(ev[want])
    _prefill(kda, entry, d, stream)
    stream.synchronize()
    assert kda.kda_last_launch_count() == want
    assert ev[0].elapsed_time(ev[want]) == stamp


def test_decode_launch_count(kda):
    stream = torch.cuda.Stream()
    S = ki.decode_state(4, 3, 128, 128, seed=31).cuda()
    x = to_dev(ki.decode_inputs(4, 3, 128, 128, "bf16", seed=31, step=0))
    ev = _events(3, stream)
    kda.kda_set_launch_events(ev)
    kda.kda_recurrent_step(S, x["q"], x["k"], x["v"], x["g"], x["beta"], scale=x["scale"],
                           stream=stream)
    stream.synchronize()
    assert kda.kda_last_launch_count() == 1
    assert ev[0].elapsed_time(ev[1]) > 0


def test_fewer_events_than_kernels(kda):
    """Only as many events as given are recorded; the count still covers every kernel."""
    stream = torch.cuda.Stream()
    d = ki.prefill_inputs(1, 200, 2, 128, 128, "bf16", seed=32, s0=True)
    ev = _events(2, stream)
    kda.kda_set_launch_events(ev)
    _prefill(kda, "kda_chunk_fwd", d, stream)
    stream.synchronize()
    assert kda.kda_last_launch_count() == 2
    assert ev[0].elapsed_time(ev[1]) > 0
