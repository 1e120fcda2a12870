"""Seeded synthetic inputs for the KDA core.

This module is shared by the tests, ``bench.py`` and the oracle harness.  It holds
none of the method's arithmetic: it draws Gaussian numbers, L2-normalises q and k
(the KDA layer does this before the core, "把注意力换成一块「会遗忘的内存」",
section on the layer implementation; "Kimi K3 四个核心模块的公式与真实张量流" §1.2),
maps logits into the input domain (log-decay g = -5*sigmoid(z), "Kimi K3 技术报告解读"
§3.3 and §3.5; write strength beta = sigmoid(z)) and rounds to the storage dtype.

Recipe (fixed, so every consumer sees the same numbers):
  * every (tensor, head) pair has its own numpy PCG64 stream seeded by
    SeedSequence([seed, tensor_code, head]) (decode steps add the step index),
    so any subset of heads can be regenerated on its own;
  * a head's rows are drawn in (batch, time) order as one [B*T, d] block;
  * q, k ~ N(0, 1), then divided by their L2 norm over d_k in fp32;
  * v ~ N(0, 1); g = -5*sigmoid(z), z ~ N(0, 1); beta = sigmoid(z), z ~ N(0, 1);
  * "slow" configs shift the logit of channels c < d_k/2 to z - 3 (slower decay);
    ``slow="literal"`` applies z + 3 instead (faster decay), as the text is printed;
  * initial states S0 ~ N(0, 0.1^2) (0.1 is the standard deviation);
  * q, k, v are then rounded to the config dtype (bf16 round-to-nearest-even via
    torch); g, beta and S0 stay fp32.

The seed of workload i is ``SEED_BASE + i``.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

SEED_BASE = 20260

Q, K, V, GATE, BETA, S0, LENGTHS = 1, 2, 3, 4, 5, 6, 7
GATE_SCALE = 8
CONV_W, CONV_CACHE, OUT_GATE, NORM_W = 9, 10, 11, 12

# The five workloads: sizes and distributions as the KDA pages describe them
# (96 heads x 128 head dim from "Kimi K3 四个核心模块的公式与真实张量流" §0-§1,
# up to 1M tokens of context).
WORKLOADS = {
    0: dict(name="kda_prefill_fp32_B1_H2_T256_d64", kind="prefill", B=1, H=2, T=256,
            dk=64, dv=64, dtype="f32", s0=False, slow=False),
    1: dict(name="kda_prefill_B2_H16_T4096_d128", kind="prefill", B=2, H=16, T=4096,
            dk=128, dv=128, dtype="bf16", s0=True, slow=False),
    2: dict(name="kda_prefill_B1_H96_T32768_d128", kind="prefill", B=1, H=96, T=32768,
            dk=128, dv=128, dtype="bf16", s0=False, slow=True),
    3: dict(name="kda_decode_N256_H96_d128_64steps", kind="decode", N=256, H=96,
            dk=128, dv=128, dtype="bf16", s0=True, steps=64),
    4: dict(name="kda_varlen_H8_T1048576_16seqs_d128", kind="varlen", H=8, T=1 << 20,
            nseq=16, lo=1024, hi=262144, dk=128, dv=128, dtype="bf16", s0=True, slow=False),
}

_TORCH_DTYPES = {"bf16": torch.bfloat16, "f32": torch.float32}


def torch_dtype(name: str) -> torch.dtype:
    return _TORCH_DTYPES[name]


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(x) for x in key])))


def _normal(key, shape) -> np.ndarray:
    return _rng(*key).standard_normal(shape, dtype=np.float32)


def _l2norm_rows(x: np.ndarray) -> np.ndarray:
    n = np.sqrt(np.einsum("...d,...d->...", x, x, dtype=np.float32))
    return x / np.maximum(n, np.float32(1e-6))[..., None]


def _sigmoid(z: np.ndarray) -> np.ndarray:
    return (np.float32(1.0) / (np.float32(1.0) + np.exp(-z))).astype(np.float32)


def _gate_from_logits(z: np.ndarray, slow) -> np.ndarray:
    dk = z.shape[-1]
    if slow:
        shift = np.float32(-3.0 if slow is True or slow == "slow" else 3.0)
        z = z.copy()
        z[..., : dk // 2] += shift
    return (np.float32(-5.0) * _sigmoid(z)).astype(np.float32)


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def varlen_lengths(seed: int, nseq: int, total: int, lo: int, hi: int) -> np.ndarray:
    """Sequence lengths: log-uniform in [lo, hi], rescaled to sum to ``total``.

    L_i = exp(U(ln lo, ln hi)), multiplied by total / sum(L), floored; the
    remainder is handed out one token at a time to the longest sequences.
    """
    u = _rng(seed, LENGTHS).uniform(math.log(lo), math.log(hi), size=nseq)
    raw = np.exp(u)
    scaled = raw * (total / raw.sum())
    lens = np.floor(scaled).astype(np.int64)
    rem = int(total - lens.sum())
    order = np.argsort(-scaled, kind="stable")
    for i in range(rem):
        lens[order[i % nseq]] += 1
    assert lens.sum() == total and (lens >= 0).all()
    return lens


def cu_seqlens_from_lengths(lens) -> np.ndarray:
    lens = np.asarray(lens, dtype=np.int64)
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)


def prefill_inputs(B: int, T: int, H: int, dk: int, dv: int, dtype: str = "bf16", *,
                   seed: int, s0: bool = False, slow=False, n_states: int | None = None,
                   heads=None, scale: float | None = None) -> dict:
    """Inputs of one ``kda_chunk_fwd`` call as CPU torch tensors.

    q, k: [B, T, H', dk] (dtype); v: [B, T, H', dv] (dtype); g: [B, T, H', dk] fp32;
    beta: [B, T, H'] fp32; initial_state: [n_states, H', dk, dv] fp32 or None, with
    n_states = B unless given (varlen calls pass the number of sequences).  H' is
    ``len(heads)`` when a subset of heads is requested (each head's numbers do not
    depend on which other heads are generated).
    """
    heads = list(range(H)) if heads is None else [int(h) for h in heads]
    Hs = len(heads)
    tdt = torch_dtype(dtype)
    rows = B * T
    q = torch.empty((rows, Hs, dk), dtype=tdt)
    k = torch.empty((rows, Hs, dk), dtype=tdt)
    v = torch.empty((rows, Hs, dv), dtype=tdt)
    g = torch.empty((rows, Hs, dk), dtype=torch.float32)
    beta = torch.empty((rows, Hs), dtype=torch.float32)
    N = B if n_states is None else int(n_states)
    S = torch.empty((N, Hs, dk, dv), dtype=torch.float32) if s0 else None

    def one(j_h):
        j, h = j_h
        q[:, j] = torch.from_numpy(_l2norm_rows(_normal((seed, Q, h), (rows, dk)))).to(tdt)
        k[:, j] = torch.from_numpy(_l2norm_rows(_normal((seed, K, h), (rows, dk)))).to(tdt)
        v[:, j] = torch.from_numpy(_normal((seed, V, h), (rows, dv))).to(tdt)
        g[:, j] = torch.from_numpy(_gate_from_logits(_normal((seed, GATE, h), (rows, dk)), slow))
        beta[:, j] = torch.from_numpy(_sigmoid(_normal((seed, BETA, h), (rows,))))
        if S is not None:
            S[:, j] = torch.from_numpy(np.float32(0.1) * _normal((seed, S0, h), (N, dk, dv)))

    with ThreadPoolExecutor(min(_threads(), max(1, Hs))) as ex:
        list(ex.map(one, enumerate(heads)))
    return dict(q=q.view(B, T, Hs, dk), k=k.view(B, T, Hs, dk), v=v.view(B, T, Hs, dv),
                g=g.view(B, T, Hs, dk), beta=beta.view(B, T, Hs), initial_state=S,
                scale=float(scale if scale is not None else 1.0 / math.sqrt(dk)))


def gate_logits(d: dict, *, seed: int, heads=None) -> dict:
    """Decay logits for the fused-gate prefill, added to the inputs ``d`` of
    :func:`prefill_inputs`: ``z`` [B, T, H', dk] ~ N(0, 1) in q's dtype (the same
    draws that ``d["g"]`` was formed from) and ``gate_scale`` [H'] fp32, one
    draw per head from U(0.5, 2).  Random numbers only."""
    B, T, Hs, dk = d["q"].shape
    H_all = heads if heads is not None else list(range(Hs))
    rows = B * T
    z = torch.empty((rows, Hs, dk), dtype=d["q"].dtype)
    A = torch.empty((Hs,), dtype=torch.float32)
    for j, h in enumerate(H_all):
        z[:, j] = torch.from_numpy(_normal((seed, GATE, h), (rows, dk))).to(d["q"].dtype)
        A[j] = float(_rng(seed, GATE_SCALE, h).uniform(0.5, 2.0))
    out = dict(d)
    out["z"] = z.view(B, T, Hs, dk)
    out["gate_scale"] = A
    return out


def fused_decode_extras(N: int, H: int, dk: int, dv: int, dtype: str = "bf16", *, seed: int,
                        step: int = 0) -> dict:
    """Synthetic tensors of the fused decode step: convolution weights w_q, w_k
    [H, dk, 4], w_v [H, dv, 4] ~ N(0, 0.5^2) fp32; conv caches conv_q, conv_k [N, 3,
    H, dk], conv_v [N, 3, H, dv] ~ N(0, 1) in ``dtype``; output-gate logits out_gate
    [N, H, dv] ~ N(0, 1) in ``dtype`` (fresh per step); norm_weight [dv] ~ U(0.5,
    1.5).  Random numbers only."""
    tdt = torch_dtype(dtype)
    f = lambda key, shape: torch.from_numpy(_normal((seed,) + key, shape))
    return dict(
        w_q=0.5 * f((CONV_W, 0), (H, dk, 4)), w_k=0.5 * f((CONV_W, 1), (H, dk, 4)),
        w_v=0.5 * f((CONV_W, 2), (H, dv, 4)),
        conv_q=f((CONV_CACHE, 0), (N, 3, H, dk)).to(tdt), conv_k=f((CONV_CACHE, 1), (N, 3, H, dk)).to(tdt),
        conv_v=f((CONV_CACHE, 2), (N, 3, H, dv)).to(tdt),
        out_gate=f((OUT_GATE, step), (N, H, dv)).to(tdt),
        norm_weight=torch.from_numpy(_rng(seed, NORM_W).uniform(0.5, 1.5, dv).astype(np.float32)))


def decode_state(N: int, H: int, dk: int, dv: int, *, seed: int, heads=None) -> torch.Tensor:
    heads = list(range(H)) if heads is None else [int(h) for h in heads]
    S = torch.empty((N, len(heads), dk, dv), dtype=torch.float32)

    def one(j_h):
        j, h = j_h
        S[:, j] = torch.from_numpy(np.float32(0.1) * _normal((seed, S0, h), (N, dk, dv)))

    with ThreadPoolExecutor(min(_threads(), len(heads))) as ex:
        list(ex.map(one, enumerate(heads)))
    return S


def decode_inputs(N: int, H: int, dk: int, dv: int, dtype: str = "bf16", *, seed: int,
                  step: int, heads=None, scale: float | None = None) -> dict:
    """Inputs of one ``kda_recurrent_step`` call: q, k [N, H', dk]; v [N, H', dv]
    (dtype); g [N, H', dk] fp32; beta [N, H'] fp32."""
    heads = list(range(H)) if heads is None else [int(h) for h in heads]
    Hs = len(heads)
    tdt = torch_dtype(dtype)
    q = torch.empty((N, Hs, dk), dtype=tdt)
    k = torch.empty((N, Hs, dk), dtype=tdt)
    v = torch.empty((N, Hs, dv), dtype=tdt)
    g = torch.empty((N, Hs, dk), dtype=torch.float32)
    beta = torch.empty((N, Hs), dtype=torch.float32)
    st = 1000 + int(step)

    def one(j_h):
        j, h = j_h
        q[:, j] = torch.from_numpy(_l2norm_rows(_normal((seed, Q, h, st), (N, dk)))).to(tdt)
        k[:, j] = torch.from_numpy(_l2norm_rows(_normal((seed, K, h, st), (N, dk)))).to(tdt)
        v[:, j] = torch.from_numpy(_normal((seed, V, h, st), (N, dv))).to(tdt)
        g[:, j] = torch.from_numpy(_gate_from_logits(_normal((seed, GATE, h, st), (N, dk)), False))
        beta[:, j] = torch.from_numpy(_sigmoid(_normal((seed, BETA, h, st), (N,))))

    with ThreadPoolExecutor(min(_threads(), max(1, Hs))) as ex:
        list(ex.map(one, enumerate(heads)))
    return dict(q=q, k=k, v=v, g=g, beta=beta,
                scale=float(scale if scale is not None else 1.0 / math.sqrt(dk)))


def workload_inputs(idx: int, heads=None) -> dict:
    """Inputs of prefill workload ``idx`` (0, 1, 2 or 4), optionally for a head subset."""
    w = WORKLOADS[idx]
    seed = SEED_BASE + idx
    if w["kind"] == "prefill":
        d = prefill_inputs(w["B"], w["T"], w["H"], w["dk"], w["dv"], w["dtype"], seed=seed,
                           s0=w["s0"], slow=w["slow"], heads=heads)
        d["cu_seqlens"] = None
        return d
    if w["kind"] == "varlen":
        lens = varlen_lengths(seed, w["nseq"], w["T"], w["lo"], w["hi"])
        d = prefill_inputs(1, w["T"], w["H"], w["dk"], w["dv"], w["dtype"], seed=seed,
                           s0=w["s0"], slow=w["slow"], n_states=w["nseq"], heads=heads)
        d["cu_seqlens"] = torch.from_numpy(cu_seqlens_from_lengths(lens))
        return d
    raise ValueError(f"workload {idx} is not a prefill workload")
