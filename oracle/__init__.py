"""CPU fp64 oracle for the KDA core.

TEST INFRASTRUCTURE ONLY.  The product path (the ``gated_delta_rule_gb300``
package and its CUDA library) never imports, links or runs anything here; only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg do.
The oracle shares no code with the CUDA path; both only read the seeded inputs of
``kda_inputs``.

Contents:
  * ``kda_oracle.cpp`` - the main oracle: the token-by-token recurrence in fp64,
    OpenMP across independent (sequence, head) problems (built to
    ``_kda_oracle.so`` by :func:`build`);
  * ``kda_numpy``      - numpy restatements (three-step loop, explicit transition
    matrix, chunked form, segment transition) used to pin the C++ oracle.

Every function here takes the exact values of the tensors the GPU sees (bf16 or
fp32, widened to fp64) and returns fp64 numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from . import kda_numpy  # noqa: F401  (re-exported)

_DIR = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_DIR, "kda_oracle.cpp")
_LIB = os.path.join(_DIR, "_kda_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C++ oracle (g++ -O2 -fopenmp).  Returns the library path."""
    with _lock:
        fresh = os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)
        if force or not fresh:
            tmp = _LIB + f".{os.getpid()}.tmp"
            subprocess.run(["g++", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c++17", _SRC,
                            "-o", tmp], check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.kda_oracle_run.restype = ctypes.c_int
        lib.kda_oracle_run.argtypes = [ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_int, ctypes.c_int] + [ctypes.c_void_p] * 6 + [
            ctypes.c_double, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        lib.kda_oracle_threads.restype = ctypes.c_int
        lib.kda_oracle_threads.argtypes = [ctypes.c_int]
        _lib = lib
    return _lib


def threads(nthreads: int = 0) -> int:
    return int(_load().kda_oracle_threads(int(nthreads)))


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu()
        if not x.dtype.is_floating_point:
            return np.ascontiguousarray(x.numpy().astype(np.float64))
        x = x.double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def run_problems(row_start, row_count, q, k, v, g, beta, S0, scale, nthreads=0):
    """Low-level entry: problem p runs rows [row_start[p], +row_count[p]) of the
    row-major fp64 arrays q, k, g [rows, dk], v [rows, dv], beta [rows].
    Returns (out [rows, dv], S_T [P, dk, dv], threads used)."""
    lib = _load()
    rs = np.ascontiguousarray(row_start, dtype=np.int64)
    rc = np.ascontiguousarray(row_count, dtype=np.int64)
    P = rs.shape[0]
    dk, dv = q.shape[1], v.shape[1]
    out = np.zeros((q.shape[0], dv))
    ST = np.zeros((P, dk, dv))
    S0c = None if S0 is None else np.ascontiguousarray(S0, dtype=np.float64).reshape(P, dk, dv)
    nt = lib.kda_oracle_run(P, _ptr(rs), _ptr(rc), dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                            _ptr(beta), _ptr(S0c), float(scale), _ptr(out), _ptr(ST),
                            int(nthreads))
    if nt < 0:
        raise ValueError(f"kda_oracle_run rejected its arguments ({nt})")
    return out, ST, nt


def prefill(q, k, v, g, beta, initial_state, scale, cu_seqlens=None, nthreads=0):
    """Oracle of ``kda_chunk_fwd``.

    q, k, g: [B, T, H, dk]; v: [B, T, H, dv]; beta: [B, T, H]; initial_state:
    [N, H, dk, dv] or None; cu_seqlens: [N+1] offsets (then B == 1) or None (then
    N == B and every batch row is one sequence).  Returns (out [B, T, H, dv],
    final_state [N, H, dk, dv]) in fp64.
    """
    q, k, v, g, beta = (_f64(a) for a in (q, k, v, g, beta))
    B, T, H, dk = q.shape
    dv = v.shape[3]
    # head-major packing: [B, H, T, d] rows, so one problem's rows are contiguous
    qp, kp, gp = (np.ascontiguousarray(a.transpose(0, 2, 1, 3)).reshape(B * H * T, dk)
                  for a in (q, k, g))
    vp = np.ascontiguousarray(v.transpose(0, 2, 1, 3)).reshape(B * H * T, dv)
    bp = np.ascontiguousarray(beta.transpose(0, 2, 1)).reshape(B * H * T)
    if cu_seqlens is None:
        N = B
        starts = [(b * H + h) * T for b in range(B) for h in range(H)]
        counts = [T] * (B * H)
    else:
        cu = _f64(cu_seqlens).astype(np.int64)
        if B != 1:
            raise ValueError("varlen inputs must have B == 1")
        N = cu.shape[0] - 1
        starts = [h * T + int(cu[n]) for n in range(N) for h in range(H)]
        counts = [int(cu[n + 1] - cu[n]) for n in range(N) for h in range(H)]
    S0 = None if initial_state is None else _f64(initial_state).reshape(N * H, dk, dv)
    out, ST, _ = run_problems(starts, counts, qp, kp, vp, gp, bp, S0, scale, nthreads)
    out = out.reshape(B, H, T, dv).transpose(0, 2, 1, 3)
    return np.ascontiguousarray(out), ST.reshape(N, H, dk, dv)


def decode_step(state, q, k, v, g, beta, scale, nthreads=0):
    """Oracle of ``kda_recurrent_step``: state [N, H, dk, dv]; q, k, g [N, H, dk];
    v [N, H, dv]; beta [N, H].  Returns (out [N, H, dv], new_state) in fp64."""
    q, k, v, g, beta, S = (_f64(a) for a in (q, k, v, g, beta, state))
    N, H, dk = q.shape
    dv = v.shape[2]
    P = N * H
    out, ST, _ = run_problems(np.arange(P), np.ones(P), q.reshape(P, dk), k.reshape(P, dk),
                              v.reshape(P, dv), g.reshape(P, dk), beta.reshape(P),
                              S.reshape(P, dk, dv), scale, nthreads)
    return out.reshape(N, H, dv), ST.reshape(N, H, dk, dv)


def multi_step(state, q, k, v, g, beta, scale, num_accepted=None, nthreads=0):
    """Oracle of ``kda_recurrent_multi_step``: state [N, H, dk, dv]; q (or None), k, g
    [N, n, H, dk]; v [N, n, H, dv]; beta [N, n, H]; num_accepted [N] or None (= n).

    The n tokens of a request run the recurrence in order, token j's output read
    from the state after tokens 0..j ("Kimi K3 核心算子拆解" (devpress.csdn.net)
    §2.3, one step per token); the state kept is the one after the first
    clamp(num_accepted, 0, n) tokens, the replay of accepted draft tokens of
    "Kimi K3 技术报告解读" (marsggbo.github.io) §9.  Returns (out [N, n, H, dv] or
    None when q is None, kept state [N, H, dk, dv]) in fp64.
    """
    k, v, g, beta, S = (_f64(a) for a in (k, v, g, beta, state))
    N, n, H, dk = k.shape
    dv = v.shape[3]
    if num_accepted is None:
        acc = np.full(N, n, dtype=np.int64)
    else:
        acc = np.clip(_f64(num_accepted).astype(np.int64).reshape(N), 0, n)
    out = None
    if q is not None:
        out, _ = prefill(q, k, v, g, beta, S, scale, nthreads=nthreads)
    kp, gp = (np.ascontiguousarray(a.transpose(0, 2, 1, 3)).reshape(N * H * n, dk) for a in (k, g))
    vp = np.ascontiguousarray(v.transpose(0, 2, 1, 3)).reshape(N * H * n, dv)
    bp = np.ascontiguousarray(beta.transpose(0, 2, 1)).reshape(N * H * n)
    starts = [(i * H + h) * n for i in range(N) for h in range(H)]
    counts = [int(acc[i]) for i in range(N) for h in range(H)]
    # the kept state only: the read-outs of this run (q = k here) are discarded
    _, ST, _ = run_problems(starts, counts, kp, kp, vp, gp, bp, S.reshape(N * H, dk, dv), scale,
                            nthreads)
    return out, ST.reshape(N, H, dk, dv)


def gate_log_decay(z, gate_scale):
    """Log-decay of the fused-gate prefill: g = -5 sigmoid(A_h z) in fp64, z
    [..., H, dk], A [H] ("Kimi K3 技术报告解读" (marsggbo.github.io) §3.5: a scaled
    sigmoid of the decay logit with a learnable per-head scale, keeping every
    per-step decay factor above e^-5; the formula's reading is that bound's)."""
    z = _f64(z)
    A = _f64(gate_scale).reshape(-1)
    x = z * A[:, None]
    with np.errstate(over="ignore"):  # exp(-x) = inf for very negative x gives g = -0
        return -5.0 / (1.0 + np.exp(-x))


def prefill_checkpoints(q, k, v, g, beta, initial_state, scale, checkpoint_tokens, num_checkpoints,
                        cu_seqlens=None, nthreads=0):
    """Oracle of the checkpoints of ``kda_chunk_fwd_checkpointed``: [N * C, H, dk, dv]
    fp64 with row n * C + j = the state after the first (j + 1) * checkpoint_tokens
    tokens of sequence n (the prefix-cache checkpoints of "Kimi K3 技术报告解读"
    (marsggbo.github.io) §9), NaN where the sequence is shorter.  The recurrence
    runs from checkpoint to checkpoint, carrying the state."""
    q, k, v, g, beta = (_f64(a) for a in (q, k, v, g, beta))
    B, T, H, dk = q.shape
    dv = v.shape[3]
    C, ck = int(num_checkpoints), int(checkpoint_tokens)
    if cu_seqlens is None:
        N = B
        spans = [(b, 0, T) for b in range(B)]
    else:
        cu = _f64(cu_seqlens).astype(np.int64)
        N = cu.shape[0] - 1
        spans = [(0, int(cu[n]), int(cu[n + 1])) for n in range(N)]
    S0 = None if initial_state is None else _f64(initial_state).reshape(N, H, dk, dv)
    res = np.full((N * C, H, dk, dv), np.nan)
    for n, (b, t0, t1) in enumerate(spans):
        S = np.zeros((H, dk, dv)) if S0 is None else S0[n].copy()
        for j in range(min(C, (t1 - t0) // ck)):
            a, e = t0 + j * ck, t0 + (j + 1) * ck
            _, S = prefill(q[b:b + 1, a:e], k[b:b + 1, a:e], v[b:b + 1, a:e], g[b:b + 1, a:e],
                           beta[b:b + 1, a:e], S[None], scale, nthreads=nthreads)
            S = S[0]
            res[n * C + j] = S
    return res


def decode_fused(state, conv_q, conv_k, conv_v, q, k, v, w_q, w_k, w_v, g, beta, out_gate,
                 norm_weight, scale, eps, l2_eps=1e-6, nthreads=0):
    """Oracle of ``kda_decode_step_fused``: one decode token with the layer's front
    and back ends, in fp64.

    Front ("Kimi K3 四个核心模块的公式与真实张量流" (gentlecold.top) §1.2; "Kimi K3
    核心算子拆解" (devpress.csdn.net) §2.6): each of q, k, v goes through a causal
    depthwise convolution of width 4 over its last three raw inputs (conv_* [N, 3, H,
    d], oldest first) and itself, weights w_* [H, d, 4] (w[..., 3] on the current
    input), then SiLU; q and k are L2-normalised (x / max(||x||, l2_eps)).  Core: the
    decode step.  Back ("把注意力换成一块「会遗忘的内存」" (jokeuncle.github.io), the
    output gate; devpress §2.5): y = o / sqrt(mean(o^2) + eps) * norm_weight *
    sigmoid(out_gate).  Returns (y [N, H, dv], new state, new conv_q, conv_k, conv_v).
    """
    S = _f64(state)
    cq, ck, cv = (_f64(a) for a in (conv_q, conv_k, conv_v))
    xq, xk, xv = (_f64(a) for a in (q, k, v))
    wq, wk, wv = (_f64(a) for a in (w_q, w_k, w_v))

    def conv_silu(cache, x, w):
        y = (w[None, :, :, 0] * cache[:, 0] + w[None, :, :, 1] * cache[:, 1] +
             w[None, :, :, 2] * cache[:, 2] + w[None, :, :, 3] * x)
        return y / (1.0 + np.exp(-y))

    def l2n(x):
        n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
        return x / np.maximum(n, l2_eps)

    qa = l2n(conv_silu(cq, xq, wq))
    ka = l2n(conv_silu(ck, xk, wk))
    va = conv_silu(cv, xv, wv)
    o, S1 = decode_step(S, qa, ka, va, g, beta, scale, nthreads)
    gate = _f64(out_gate)
    wn = np.ones(o.shape[-1]) if norm_weight is None else _f64(norm_weight)
    y = o / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps) * wn / (1.0 + np.exp(-gate))
    shift = lambda c, x: np.concatenate([c[:, 1:], x[:, None]], axis=1)
    return y, S1, shift(cq, xq), shift(ck, xk), shift(cv, xv)


def backward(q, k, v, g, beta, initial_state, scale, d_out, d_final_state=None, cu_seqlens=None):
    """Oracle of ``kda_backward``: gradients of the KDA core with respect to q, k, v,
    g, beta and the initial state, given the gradients of the outputs (d_out [B, T,
    H, dv]) and of the final state (d_final_state [N, H, dk, dv] or None).

    The forward is the token recurrence in the three-step order of "Kimi K3
    核心算子拆解" (devpress.csdn.net) §2.3 (decay, correct, write; read-out after the
    update), written with plain torch fp64 operations on the CPU; the gradients come
    from torch's reverse-mode differentiation of that loop ("尝试对Kimi
    KDA的数学推导&算子实现分析" (hjcheng0602.cn/blog/kdd) gives only the forward;
    the backward is its exact derivative).  Returns a dict of fp64 numpy arrays
    dq, dk, dv, dg, dbeta and d_initial_state (zeros when initial_state is None).
    """
    import torch
    t = lambda x: None if x is None else torch.as_tensor(_f64(x), dtype=torch.float64)
    q, k, v, g, beta, do = (t(a).clone().requires_grad_(True) if i < 5 else t(a)
                            for i, a in enumerate((q, k, v, g, beta, d_out)))
    B, T, H, dk = q.shape
    dv = v.shape[3]
    if cu_seqlens is None:
        N = B
        spans = [(b, 0, T) for b in range(B)]
    else:
        cu = _f64(cu_seqlens).astype(np.int64)
        N = cu.shape[0] - 1
        spans = [(0, int(cu[n]), int(cu[n + 1])) for n in range(N)]
    S0 = torch.zeros(N, H, dk, dv, dtype=torch.float64) if initial_state is None else t(initial_state)
    S0 = S0.clone().requires_grad_(True)
    loss = torch.zeros((), dtype=torch.float64)
    dS_T = None if d_final_state is None else t(d_final_state)
    for n, (b, t0, t1) in enumerate(spans):
        for h in range(H):
            S = S0[n, h]
            for s in range(t0, t1):
                S = S * torch.exp(g[b, s, h])[:, None]
                kS = k[b, s, h] @ S
                S = S + beta[b, s, h] * torch.outer(k[b, s, h], v[b, s, h] - kS)
                o = scale * (S.T @ q[b, s, h])
                loss = loss + o @ do[b, s, h]
            if dS_T is not None:
                loss = loss + torch.sum(S * dS_T[n, h])
    loss.backward()
    grads = dict(dq=q.grad, dk=k.grad, dv=v.grad, dg=g.grad, dbeta=beta.grad, d_initial_state=S0.grad)
    return {name: gr.detach().numpy() for name, gr in grads.items()}
