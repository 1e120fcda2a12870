"""Helpers shared by the GPU parity tests: run the CUDA path and the oracle on the
same seeded inputs and compare element by element.

Tolerances (stated for the KDA core: bf16 inputs with fp32 accumulation, and an
fp32-input mode):
  * bf16 inputs: max |o - o_ref| <= 2e-2 and ||S_T - S_ref||_F / ||S_ref||_F <= 1e-2;
  * fp32 inputs: both <= 1e-4.
"""
import numpy as np
import torch

import oracle

TOL = {"bf16": (2e-2, 1e-2), "f32": (1e-4, 1e-4)}


def dtype_name(t):
    return "bf16" if t.dtype == torch.bfloat16 else "f32"


def to_dev(d, dev="cuda"):
    return {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in d.items()}


def max_abs(a, b):
    a = a.float().cpu().numpy() if torch.is_tensor(a) else a
    return float(np.abs(a - b).max()) if np.size(b) else 0.0


def rel_fro(a, b):
    a = a.float().cpu().numpy().astype(np.float64) if torch.is_tensor(a) else a
    nb = np.linalg.norm(b)
    if nb == 0:
        return float(np.linalg.norm(a))
    return float(np.linalg.norm(a - b) / nb)


def check_prefill(fn, d, tol=None, label=""):
    """Run ``fn`` (a binding entry point) on device copies of ``d`` and compare with the
    oracle.  Returns (err_o, err_S)."""
    t = to_dev(d)
    out, sT = fn(t["q"], t["k"], t["v"], t["g"], t["beta"], t["initial_state"], t["scale"],
                 cu_seqlens=t.get("cu_seqlens"))
    torch.cuda.synchronize()
    o_ref, s_ref = oracle.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"],
                                  d["scale"], cu_seqlens=d.get("cu_seqlens"))
    eo, es = max_abs(out, o_ref), rel_fro(sT, s_ref)
    to, ts = tol or TOL[dtype_name(d["q"])]
    assert eo <= to and es <= ts, f"{label}: max|o-o_ref|={eo:.3g} (tol {to}), rel_F(S)={es:.3g} (tol {ts})"
    assert np.isfinite(out.float().cpu().numpy()).all()
    return eo, es
