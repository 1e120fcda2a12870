"""kda_chunk_fwd_noalloc: the prefill entry point for callers that cannot allocate
device memory during a call (their device memory is pre-sized and owned by the
host application's own allocator, or they run where cudaMalloc is not allowed).

It keeps its chunk records in a fixed device array built into the library, so
every call shares that array.  These checks call it through the C ABI twice in a
row, with different shapes (so a second call cannot lean on what the first left
behind), and compare each result with kda_chunk_fwd on the same inputs, within
the tolerances the other GPU tests use; and, in a fresh process, check that a call
leaves the device's free memory exactly where it was.  This file is collected
last on purpose.
"""
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest
import torch

import kda_inputs as ki
from tests.parity import TOL, max_abs, rel_fro, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    import gated_delta_rule_gb300 as m
    m.build()
    m.load_library()
    return m


def _run(fn, t, cu=None):
    out = torch.full(t["v"].shape, float("nan"), dtype=t["q"].dtype, device="cuda")
    N = t["q"].shape[0] if cu is None else cu.shape[0] - 1
    H, dk, dv = t["q"].shape[2], t["q"].shape[3], t["v"].shape[3]
    sT = torch.full((N, H, dk, dv), float("nan"), dtype=torch.float32, device="cuda")
    fn(t["q"], t["k"], t["v"], t["g"], t["beta"], t["initial_state"], t["scale"], cu_seqlens=cu,
       out=out, final_state=sT)
    torch.cuda.synchronize()
    return out, sT


def test_noalloc_matches_chunk_fwd_on_two_calls_in_a_row(kda):
    to, ts = TOL["bf16"]
    # call 1: fixed length, ragged tail
    d1 = to_dev(ki.prefill_inputs(2, 300, 4, 128, 128, "bf16", seed=901, s0=True))
    o_ref, s_ref = _run(kda.kda_chunk_fwd, d1)
    o1, s1 = _run(kda.kda_chunk_fwd_noalloc, d1)
    # call 2: varlen with an empty sequence, other head dims
    lens = [100, 0, 37, 200]
    cu = torch.from_numpy(ki.cu_seqlens_from_lengths(lens)).cuda()
    d2 = to_dev(ki.prefill_inputs(1, sum(lens), 3, 64, 128, "bf16", seed=902, s0=True,
                                  n_states=len(lens)))
    o2_ref, s2_ref = _run(kda.kda_chunk_fwd, d2, cu)
    o2, s2 = _run(kda.kda_chunk_fwd_noalloc, d2, cu)
    kda.kda_get_device_error()
    for o, s, orf, srf in ((o1, s1, o_ref, s_ref), (o2, s2, o2_ref, s2_ref)):
        assert torch.isfinite(o).all() and torch.isfinite(s).all()
        assert max_abs(o, orf.float().cpu().numpy()) <= to
        assert rel_fro(s, srf.cpu().numpy().astype(np.float64)) <= ts


def test_noalloc_rejects_oversized_request(kda):
    d = {k: (v.cuda() if torch.is_tensor(v) else v)
         for k, v in ki.prefill_inputs(1, 4096, 16, 128, 128, "bf16", seed=903).items()}
    with pytest.raises(kda.KdaError) as e:
        kda.kda_chunk_fwd_noalloc(d["q"], d["k"], d["v"], d["g"], d["beta"], None, d["scale"])
    assert e.value.status == 2 and "fixed workspace" in e.value.message


_FRESH = textwrap.dedent("""
    import torch, kda_inputs as ki, gated_delta_rule_gb300 as kda
    kda.load_library()
    def dev(d):
        return {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in d.items()}
    small = dev(ki.prefill_inputs(1, 640, 4, 128, 128, "bf16", seed=904, s0=True))       # 40 chunk-heads
    large = dev(ki.prefill_inputs(1, 64 * 225, 4, 128, 128, "bf16", seed=905, s0=True))  # 900 chunk-heads
    outs = [(torch.empty_like(x["v"]), torch.empty_like(x["initial_state"])) for x in (small, large)]
    def call(x, o):
        kda.kda_chunk_fwd_noalloc(x["q"], x["k"], x["v"], x["g"], x["beta"], x["initial_state"], x["scale"],
                                  out=o[0], final_state=o[1])
    call(small, outs[0])            # warm: kernels loaded, the fixed array's address looked up
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    call(large, outs[1])            # 60 MB of chunk records: a pool would have to grow for them
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    kda.kda_get_device_error()
    assert torch.isfinite(outs[1][0]).all()
    print("FREE", free0, free1)
""")


def test_noalloc_call_leaves_device_memory_untouched():
    """In a fresh process that never calls kda_chunk_fwd: after one warm call, a call
    whose records need 60 MB (15 times the warm call's) changes the device's free
    memory by nothing, so no pool or allocation sits behind the entry point."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FRESH], cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    free0, free1 = (int(x) for x in r.stdout.split("FREE")[-1].split())
    assert free0 == free1, (free0, free1)
