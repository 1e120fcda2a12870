"""Parity of the prefill entry points (kda_chunk_fwd, kda_fused_recurrent_fwd) with the
CPU oracle: ragged lengths around the 64-token chunk, every head-dim pair, both
dtypes, initial states, in-place states, strided views, varlen packing with
empty sequences and bit-exact sequence boundaries, and the full-size workloads
(sampled heads / sequences)."""
import numpy as np
import pytest
import torch

import kda_inputs as ki
import oracle
from tests.parity import TOL, check_prefill, max_abs, rel_fro, to_dev

pytestmark = pytest.mark.gpu

ENTRIES = ["kda_chunk_fwd", "kda_fused_recurrent_fwd"]


@pytest.fixture(scope="module")
def kda():
    import gated_delta_rule_gb300 as m
    m.build()
    m.load_library()
    return m


@pytest.mark.parametrize("entry", ENTRIES)
@pytest.mark.parametrize("T", [1, 15, 16, 17, 63, 64, 65, 200])
def test_ragged_lengths(kda, entry, T):
    d = ki.prefill_inputs(2, T, 3, 128, 128, "bf16", seed=100 + T, s0=True)
    check_prefill(getattr(kda, entry), d, label=f"{entry} T={T}")


@pytest.mark.parametrize("entry", ENTRIES)
@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64), (128, 128)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_head_dims_and_dtypes(kda, entry, dk, dv, dtype):
    d = ki.prefill_inputs(1, 130, 2, dk, dv, dtype, seed=7, s0=True)
    check_prefill(getattr(kda, entry), d, label=f"{entry} {dk}x{dv} {dtype}")


@pytest.mark.parametrize("entry", ENTRIES)
def test_zero_initial_state_and_no_final_state(kda, entry):
    d = ki.prefill_inputs(1, 70, 2, 128, 128, "bf16", seed=9, s0=False)
    t = to_dev(d)
    out, sT = getattr(kda, entry)(t["q"], t["k"], t["v"], t["g"], t["beta"], None, t["scale"],
                                  output_final_state=False)
    assert sT is None
    o_ref, _ = oracle.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], None, d["scale"])
    assert max_abs(out, o_ref) <= 2e-2


@pytest.mark.parametrize("entry", ENTRIES)
def test_in_place_state(kda, entry):
    d = ki.prefill_inputs(2, 90, 2, 128, 128, "bf16", seed=10, s0=True)
    t = to_dev(d)
    S = t["initial_state"].clone()
    out, sT = getattr(kda, entry)(t["q"], t["k"], t["v"], t["g"], t["beta"], S, t["scale"],
                                  final_state=S)
    assert sT is S
    o_ref, s_ref = oracle.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"],
                                  d["scale"])
    assert max_abs(out, o_ref) <= 2e-2 and rel_fro(S, s_ref) <= 1e-2


@pytest.mark.parametrize("entry", ENTRIES)
def test_strided_views(kda, entry):
    """q/k/v/g as head-slices of fused projections (non-contiguous head stride)."""
    B, T, H, dk, dv = 1, 100, 2, 128, 128
    d = ki.prefill_inputs(B, T, H, dk, dv, "bf16", seed=11, s0=True)
    fused = torch.empty(B, T, H, 3 * dk, dtype=torch.bfloat16, device="cuda")
    fused[..., :dk] = d["q"].cuda()
    fused[..., dk:2 * dk] = d["k"].cuda()
    fused[..., 2 * dk:] = d["v"].cuda()
    q, k, v = fused[..., :dk], fused[..., dk:2 * dk], fused[..., 2 * dk:]
    out, sT = getattr(kda, entry)(q, k, v, d["g"].cuda(), d["beta"].cuda(),
                                  d["initial_state"].cuda(), d["scale"])
    o_ref, s_ref = oracle.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"],
                                  d["scale"])
    assert max_abs(out, o_ref) <= 2e-2 and rel_fro(sT, s_ref) <= 1e-2


@pytest.mark.parametrize("entry", ENTRIES)
def test_varlen_with_empty_sequences(kda, entry):
    lens = [0, 1, 64, 65, 0, 200, 17, 128]
    cu = ki.cu_seqlens_from_lengths(lens)
    d = ki.prefill_inputs(1, int(cu[-1]), 3, 128, 128, "bf16", seed=12, s0=True,
                          n_states=len(lens))
    d["cu_seqlens"] = torch.from_numpy(cu)
    check_prefill(getattr(kda, entry), d, label=f"{entry} varlen")


@pytest.mark.parametrize("entry", ENTRIES)
def test_varlen_boundaries_bit_exact(kda, entry):
    """Each packed sequence's out and final state are bit-identical to the same
    sequence run alone, and to a packing whose other sequences hold different data."""
    fn = getattr(kda, entry)
    lens = [37, 150, 64, 1, 99]
    cu = ki.cu_seqlens_from_lengths(lens)
    Tt = int(cu[-1])
    d = to_dev(ki.prefill_inputs(1, Tt, 2, 128, 128, "bf16", seed=13, s0=True, n_states=len(lens)))
    cu_d = torch.from_numpy(cu).cuda()
    out, sT = fn(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"], d["scale"],
                 cu_seqlens=cu_d)
    other = to_dev(ki.prefill_inputs(1, Tt, 2, 128, 128, "bf16", seed=14, s0=True,
                                     n_states=len(lens)))
    for n in range(len(lens)):
        a, b = int(cu[n]), int(cu[n + 1])
        sl = lambda x: x[:, a:b].contiguous()
        o1, s1 = fn(sl(d["q"]), sl(d["k"]), sl(d["v"]), sl(d["g"]), sl(d["beta"]),
                    d["initial_state"][n:n + 1].contiguous(), d["scale"])
        assert torch.equal(out[:, a:b], o1) and torch.equal(sT[n:n + 1], s1), n
        mixed = {x: other[x].clone() for x in ("q", "k", "v", "g", "beta")}
        for x in mixed:
            mixed[x][:, a:b] = d[x][:, a:b]
        S0m = other["initial_state"].clone()
        S0m[n] = d["initial_state"][n]
        o2, s2 = fn(mixed["q"], mixed["k"], mixed["v"], mixed["g"], mixed["beta"], S0m,
                    d["scale"], cu_seqlens=cu_d)
        assert torch.equal(o2[:, a:b], out[:, a:b]) and torch.equal(s2[n], sT[n]), n


@pytest.mark.parametrize("T", [1500, 1600])
def test_fixed_length_equals_varlen_packing(kda, T):
    """A fixed-length batch (chunk indices n * chunks + c) and the same sequences
    packed with cu_seqlens (chunk offsets built on the device) give bit-identical
    outputs, final states and per-chunk checkpoints, in place as well, and match
    the oracle.  24 and 25 chunks (the last one partial at T = 1500)."""
    B, H = 2, 4
    d = ki.prefill_inputs(B, T, H, 128, 128, "bf16", seed=31, s0=True)
    check_prefill(kda.kda_chunk_fwd, d, label=f"fixed length T={T}")
    t = to_dev(d)
    C = T // 64
    out, sT, ck = kda.kda_chunk_fwd_checkpointed(t["q"], t["k"], t["v"], t["g"], t["beta"],
                                                 t["initial_state"], t["scale"], checkpoint_tokens=64,
                                                 num_checkpoints=C)
    pk = lambda x: x.reshape(1, B * T, *x.shape[2:]).contiguous()
    cu = torch.tensor([0, T, 2 * T], dtype=torch.int32, device="cuda")
    out2, sT2, ck2 = kda.kda_chunk_fwd_checkpointed(pk(t["q"]), pk(t["k"]), pk(t["v"]), pk(t["g"]),
                                                    pk(t["beta"]), t["initial_state"], t["scale"],
                                                    cu_seqlens=cu, checkpoint_tokens=64, num_checkpoints=C)
    assert torch.equal(out, out2.reshape(out.shape))
    assert torch.equal(sT, sT2) and torch.equal(ck, ck2)
    S = t["initial_state"].clone()
    out3, _ = kda.kda_chunk_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], S, t["scale"], final_state=S)
    assert torch.equal(out3, out) and torch.equal(S, sT)


@pytest.mark.parametrize("dv", [64, 128])
@pytest.mark.parametrize("H", [4, 48, 96])
def test_value_column_slices(kda, dv, H):
    """The serial kernel splits d_v into 32- or 64-column CTAs when the SMs hold
    that many (4 heads: 32 columns; 48 heads: 64, or 32 at d_v = 64; 96 heads at
    d_v = 128: unsplit).  Every split matches the oracle, and the slices together
    equal the unsplit result bit for bit (columns never mix)."""
    d = ki.prefill_inputs(1, 200, H, 128, dv, "bf16", seed=40 + H + dv, s0=True)
    check_prefill(kda.kda_chunk_fwd, d, label=f"H={H} dv={dv}")
    if H != 96:
        return
    # heads of the unsplit run, one at a time (4-slice split), bitwise
    t = to_dev(d)
    out, sT = kda.kda_chunk_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["initial_state"], t["scale"])
    for h in (0, 37, 95):
        sl = lambda x: x[:, :, h:h + 1].contiguous()
        o1, s1 = kda.kda_chunk_fwd(sl(t["q"]), sl(t["k"]), sl(t["v"]), sl(t["g"]), sl(t["beta"]),
                                   t["initial_state"][:, h:h + 1].contiguous(), t["scale"])
        assert torch.equal(o1, out[:, :, h:h + 1]) and torch.equal(s1, sT[:, h:h + 1]), h


def test_bad_cu_seqlens_sets_device_error(kda):
    d = to_dev(ki.prefill_inputs(1, 50, 1, 64, 64, "bf16", seed=15, n_states=2))
    for bad in ([0, 30, 20], [1, 20, 50], [0, 20, 49]):
        cu = torch.tensor(bad, dtype=torch.int32, device="cuda")
        kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], None, d["scale"],
                          cu_seqlens=cu)
        with pytest.raises(kda.KdaError) as e:
            kda.kda_get_device_error()
        assert e.value.status == 4
    kda.kda_get_device_error()  # cleared


def test_workload0_fp32(kda):
    d = ki.workload_inputs(0)
    eo, es = check_prefill(kda.kda_chunk_fwd, d, tol=(1e-4, 1e-4), label="fp32 workload")


def test_workload1_full(kda):
    d = ki.workload_inputs(1)
    check_prefill(kda.kda_chunk_fwd, d, label="B2 H16 T4096")


def test_workload2_sampled_heads(kda):
    """96 heads x 32768 tokens on the GPU; the oracle recomputes 3 heads."""
    d = ki.workload_inputs(2)
    t = to_dev(d)
    out, sT = kda.kda_chunk_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], None, t["scale"])
    heads = [0, 50, 95]
    o_ref, s_ref = oracle.prefill(d["q"][:, :, heads], d["k"][:, :, heads], d["v"][:, :, heads],
                                  d["g"][:, :, heads], d["beta"][:, :, heads], None, d["scale"])
    assert max_abs(out[:, :, heads], o_ref) <= 2e-2
    assert rel_fro(sT[:, heads], s_ref) <= 1e-2
    assert torch.isfinite(out).all() and torch.isfinite(sT).all()


def test_workload4_sampled_sequences(kda):
    """1M-token varlen packing (16 sequences x 8 heads) on the GPU; the oracle
    recomputes the shortest, a mid-length and the longest sequence on two heads.
    The longest (194893 tokens, 3046 chunks) runs the segment split: a first
    segment of 1152 chunks from its initial state, then fifteen tail segments of
    128 chunks from the chained (M, S~) transitions, each rerun with outputs."""
    d = ki.workload_inputs(4)
    t = to_dev(d)
    out, sT = kda.kda_chunk_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["initial_state"],
                                t["scale"], cu_seqlens=t["cu_seqlens"])
    kda.kda_get_device_error()
    cu = d["cu_seqlens"].numpy()
    lens = np.diff(cu)
    order = np.argsort(lens)
    assert -(-int(lens[order[-1]]) // 64) > 1152 + 14 * 128  # the longest spans sixteen segments
    heads = [1, 6]
    for n in (int(order[0]), int(order[len(order) // 2]), int(order[-1])):
        a, b = int(cu[n]), int(cu[n + 1])
        sub = {x: d[x][:, a:b][:, :, heads] for x in ("q", "k", "v", "g", "beta")}
        o_ref, s_ref = oracle.prefill(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"],
                                      d["initial_state"][n:n + 1, heads], d["scale"])
        assert max_abs(out[:, a:b][:, :, heads], o_ref) <= 2e-2, n
        assert rel_fro(sT[n:n + 1, heads], s_ref) <= 1e-2, n
    assert torch.isfinite(sT).all()


# ---- segment split: sequences longer than 1152 chunks (73728 tokens) ----

SEG = 1152 * 64   # tokens of a sequence's first segment
TAIL = 128 * 64   # tokens of each later segment


@pytest.mark.parametrize("B,T,H", [(1, SEG + 100, 2),             # two segments, the second of 2 chunks
                                   (2, SEG + 2 * TAIL + 200, 1)])  # four segments per sequence
def test_segment_split_matches_oracle(kda, B, T, H):
    d = ki.prefill_inputs(B, T, H, 128, 128, "bf16", seed=40 + B, s0=True)
    check_prefill(kda.kda_chunk_fwd, d, label=f"segments B{B} T{T}")


@pytest.mark.parametrize("dk,dv", [(64, 128), (128, 64), (64, 64)])
def test_segment_split_head_dims(kda, dk, dv):
    d = ki.prefill_inputs(1, SEG + TAIL + 64 * 7 + 5, 1, dk, dv, "bf16", seed=43, s0=True)
    check_prefill(kda.kda_chunk_fwd, d, label=f"segments {dk}x{dv}")


def test_segment_split_varlen_bit_exact(kda):
    """Packed long and short sequences: each matches the oracle, and equals the same
    sequence run alone bit for bit (segments are cut from each sequence start)."""
    lens = [100, SEG + 6000, 0, SEG + 3 * TAIL + 4000, SEG + 200]
    cu = ki.cu_seqlens_from_lengths(lens)
    d = ki.prefill_inputs(1, int(cu[-1]), 1, 128, 128, "bf16", seed=44, s0=True, n_states=len(lens))
    d["cu_seqlens"] = torch.from_numpy(cu)
    check_prefill(kda.kda_chunk_fwd, d, label="segments varlen")
    t = to_dev(d)
    out, sT = kda.kda_chunk_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["initial_state"], t["scale"],
                                cu_seqlens=t["cu_seqlens"])
    for n in (1, 3, 4):
        a, b = int(cu[n]), int(cu[n + 1])
        sl = lambda x: x[:, a:b].contiguous()
        o1, s1 = kda.kda_chunk_fwd(sl(t["q"]), sl(t["k"]), sl(t["v"]), sl(t["g"]), sl(t["beta"]),
                                   t["initial_state"][n:n + 1].contiguous(), t["scale"])
        assert torch.equal(out[:, a:b], o1) and torch.equal(sT[n:n + 1], s1), n


def test_segment_split_64_column_units(kda):
    """20 heads of one 73828-token sequence: with its tail segment the first pass
    holds 60 units, so the serial kernel runs 64-column slices (120 CTAs).  Two
    heads match the oracle, and a head run alone (32-column slices) equals its
    slice of the batch bit for bit."""
    d = ki.prefill_inputs(1, SEG + 100, 20, 128, 128, "bf16", seed=46, s0=True)
    t = to_dev(d)
    out, sT = kda.kda_chunk_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["initial_state"], t["scale"])
    kda.kda_get_device_error()
    for h in (3, 17):
        sub = {x: d[x][:, :, h:h + 1] for x in ("q", "k", "v", "g", "beta")}
        o_ref, s_ref = oracle.prefill(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"],
                                      d["initial_state"][:, h:h + 1], d["scale"])
        assert max_abs(out[:, :, h:h + 1], o_ref) <= 2e-2, h
        assert rel_fro(sT[:, h:h + 1], s_ref) <= 1e-2, h
    h = 17
    sl = lambda x: x[:, :, h:h + 1].contiguous()
    o1, s1 = kda.kda_chunk_fwd(sl(t["q"]), sl(t["k"]), sl(t["v"]), sl(t["g"]), sl(t["beta"]),
                               t["initial_state"][:, h:h + 1].contiguous(), t["scale"])
    assert torch.equal(o1, out[:, :, h:h + 1]) and torch.equal(s1, sT[:, h:h + 1])


def test_segment_split_full_width_units(kda):
    """80 sequence-heads at d = 128: one 128-column CTA per serial unit, and the
    tail segment's S~ and M halves as two CTAs.  The long sequence matches the
    oracle and equals the same sequence run alone (one head pair, 32-column CTAs)
    bit for bit; so do two short ones."""
    lens = [SEG + 3000] + [300 + 7 * i for i in range(39)]
    cu = ki.cu_seqlens_from_lengths(lens)
    d = ki.prefill_inputs(1, int(cu[-1]), 2, 128, 128, "bf16", seed=45, s0=True, n_states=len(lens))
    d["cu_seqlens"] = torch.from_numpy(cu)
    t = to_dev(d)
    out, sT = kda.kda_chunk_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["initial_state"], t["scale"],
                                cu_seqlens=t["cu_seqlens"])
    kda.kda_get_device_error()
    a, b = int(cu[0]), int(cu[1])
    sub = {x: d[x][:, a:b] for x in ("q", "k", "v", "g", "beta")}
    o_ref, s_ref = oracle.prefill(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"],
                                  d["initial_state"][0:1], d["scale"])
    assert max_abs(out[:, a:b], o_ref) <= 2e-2
    assert rel_fro(sT[0:1], s_ref) <= 1e-2
    for n in (0, 5, 39):
        a, b = int(cu[n]), int(cu[n + 1])
        sl = lambda x: x[:, a:b].contiguous()
        o1, s1 = kda.kda_chunk_fwd(sl(t["q"]), sl(t["k"]), sl(t["v"]), sl(t["g"]), sl(t["beta"]),
                                   t["initial_state"][n:n + 1].contiguous(), t["scale"])
        assert torch.equal(out[:, a:b], o1) and torch.equal(sT[n:n + 1], s1), n
