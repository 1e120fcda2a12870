"""Prefix-cache checkpoints of kda_chunk_fwd_checkpointed: the state after every
checkpoint_tokens tokens of each sequence, against the oracle, and a prefill resumed
from a checkpoint continues the original run bit for bit."""
import numpy as np
import pytest
import torch

import kda_inputs as ki
import oracle
from tests.parity import max_abs, rel_fro, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    import gated_delta_rule_gb300 as m
    m.build()
    m.load_library()
    return m


def _run(kda, d, ck, C):
    t = to_dev(d)
    return kda.kda_chunk_fwd_checkpointed(t["q"], t["k"], t["v"], t["g"], t["beta"], t["initial_state"],
                                          t["scale"], cu_seqlens=t.get("cu_seqlens"), checkpoint_tokens=ck,
                                          num_checkpoints=C)


def _compare(ck_gpu, ref, tol):
    got = ck_gpu.double().cpu().numpy()
    for r in range(ref.shape[0]):
        if np.isnan(ref[r]).all():
            assert not got[r].any(), r  # untouched rows stay zero
        else:
            assert rel_fro(got[r], ref[r]) <= tol, r


@pytest.mark.parametrize("dtype,tol", [("bf16", 1e-2), ("f32", 1e-4)])
def test_checkpoints_fixed_length(kda, dtype, tol):
    d = ki.prefill_inputs(2, 1000, 3, 128, 128, dtype, seed=80, s0=True)
    ck, C = 128, 7
    out, sT, cks = _run(kda, d, ck, C)
    ref = oracle.prefill_checkpoints(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"],
                                     d["scale"], ck, C)
    _compare(cks, ref, tol)


def test_checkpoints_varlen_and_short_buffer(kda):
    lens = [300, 0, 1024, 77, 512]
    cu = ki.cu_seqlens_from_lengths(lens)
    d = ki.prefill_inputs(1, int(cu[-1]), 2, 128, 64, "bf16", seed=81, s0=True, n_states=len(lens))
    d["cu_seqlens"] = torch.from_numpy(cu)
    ck, C = 256, 3  # the 1024-token sequence has a fourth checkpoint that does not fit
    out, sT, cks = _run(kda, d, ck, C)
    ref = oracle.prefill_checkpoints(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"],
                                     d["scale"], ck, C, cu_seqlens=d["cu_seqlens"])
    _compare(cks, ref, 1e-2)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_resume_from_checkpoint_is_bit_exact(kda, dtype):
    """A prefill resumed from checkpoint j on the rest of the sequence gives the
    original outputs and final state bit for bit (bf16: the chunked kernels; fp32:
    the token-recurrent kernel, whose four-token blocks start at the sequence start
    and so at every checkpoint)."""
    B, T, H, ck = 2, 640 + 3, 2, 256
    d = ki.prefill_inputs(B, T, H, 128, 128, dtype, seed=82, s0=True)
    out, sT, cks = _run(kda, d, ck, 2)
    t = to_dev(d)
    j = 1
    start = (j + 1) * ck
    S_resume = cks.view(B, 2, H, 128, 128)[:, j].contiguous()
    sl = lambda x: x[:, start:].contiguous()
    o2, s2 = kda.kda_chunk_fwd(sl(t["q"]), sl(t["k"]), sl(t["v"]), sl(t["g"]), sl(t["beta"]), S_resume,
                               t["scale"])
    assert torch.equal(o2, out[:, start:]) and torch.equal(s2, sT)


def test_checkpoint_on_segment_boundary(kda):
    """Checkpoints every 8192 tokens, two of them where the segment split cuts the
    sequence (after the 1152-chunk first segment and after the first 128-chunk
    tail segment)."""
    T = (1152 + 128) * 64 + 200
    d = ki.prefill_inputs(1, T, 1, 128, 128, "bf16", seed=83, s0=True)
    ck, C = 8192, 10
    out, sT, cks = _run(kda, d, ck, C)
    ref = oracle.prefill_checkpoints(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"],
                                     d["scale"], ck, C)
    _compare(cks, ref, 1e-2)


def test_checkpoint_at_sequence_end(kda):
    d = ki.prefill_inputs(1, 512, 2, 64, 64, "bf16", seed=84, s0=True)
    out, sT, cks = _run(kda, d, 256, 2)
    assert torch.equal(cks[1], sT[0])  # the last checkpoint is the final state


def test_checkpoints_with_full_width_slices(kda):
    """96 heads at d_v = 128: the serial kernel runs one 128-column CTA per head
    (eight TMEM warps, each holding half of a state row), while one head alone runs
    as four 32-column CTAs.  Checkpoints, outputs and final states of the two
    agree bit for bit (columns never mix), and a head matches the oracle."""
    d = ki.prefill_inputs(1, 640 + 37, 96, 128, 128, "bf16", seed=85, s0=True)
    ck, C = 128, 5
    out, sT, cks = _run(kda, d, ck, C)
    for h in (0, 47, 95):
        one = {k: (v[:, :, h:h + 1].contiguous() if k in ("q", "k", "v", "g") else v) for k, v in d.items()}
        one["beta"] = d["beta"][:, :, h:h + 1].contiguous()
        one["initial_state"] = d["initial_state"][:, h:h + 1].contiguous()
        o1, s1, c1 = _run(kda, one, ck, C)
        assert torch.equal(o1, out[:, :, h:h + 1]) and torch.equal(s1, sT[:, h:h + 1]), h
        assert torch.equal(c1, cks[:, h:h + 1]), h
    h = 47
    ref = oracle.prefill_checkpoints(d["q"][:, :, h:h + 1], d["k"][:, :, h:h + 1], d["v"][:, :, h:h + 1],
                                     d["g"][:, :, h:h + 1], d["beta"][:, :, h:h + 1],
                                     d["initial_state"][:, h:h + 1], d["scale"], ck, C)
    _compare(cks[:, h:h + 1], ref, 1e-2)
