"""Test-side glue: oracle expectations for seeded torch inputs, and the error measure.

Error measure (relative Frobenius with an underflow floor):
    err = ||X_gpu - X_ref||_F / max(||X_ref||_F, tau),  tau = 1e-30,
taken per unit (one head's T_C, S or output block) and maximised over units.
The floor matters for long gated-delta segments, whose T_C decays below the
fp32 range (the kernel then returns zeros).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

TAU = 1e-30
TOL_F32 = 1e-5   # fp32 inputs and state
TOL_BF16 = 2e-3  # bf16 inputs, fp32 state and accumulation


def np64(t):
    return None if t is None else t.detach().to("cpu").to(torch.float64).numpy()


def relerr(x, ref, tau=TAU):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), tau))


def gates(family, tok, h, b, e):
    """Oracle gate arrays of head h over tokens [b, e)."""
    alpha, beta = tok["alpha"], tok["beta"]
    if family == "scalar_const":
        a = np64(alpha[h:h + 1])
    elif family == "delta":
        a = None
    else:
        a = np64(alpha[b:e, h])
    bb = np64(beta[b:e, h]) if family in ("delta", "gated_delta", "kda") else None
    return a, bb


def ref_pair(family, tok, h, b, e):
    a, bb = gates(family, tok, h, b, e)
    return oracle.segment_pair(family, np64(tok["k"][b:e, h]), np64(tok["v"][b:e, h]), a, bb)


def ref_run(family, tok, h, b, e, S0=None, want_o=False):
    a, bb = gates(family, tok, h, b, e)
    q = np64(tok["q"][b:e, h]) if want_o else None
    return oracle.run(family, np64(tok["k"][b:e, h]), np64(tok["v"][b:e, h]), a, bb, q=q, S0=S0)


def t_as_dense(family, T, d):
    T = np.asarray(T, dtype=np.float64)
    if family in ("scalar_const", "scalar"):
        return float(T.reshape(-1)[0]) * np.eye(d)
    if family == "diag":
        return np.diag(T.reshape(-1))
    return T.reshape(d, d)


def host_tokens(tok, heads):
    """Copy the listed heads' token tensors to the host (oracle side)."""
    out = {}
    for key, t in tok.items():
        if t is None:
            out[key] = None
        elif key == "alpha" and t.dim() == 1:
            out[key] = t[heads].cpu()
        else:
            out[key] = t[:, heads].cpu()
    return out
