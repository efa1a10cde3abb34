"""Float64 oracle for the boundary patches of the reuse path.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: the product library never imports,
links or runs anything here.  Plain numpy with explicit loops; no code is shared with the
CUDA path.

What it computes (HYPIC reading notes, Method part 6, "causal convolution and RoPE must be
handled together"; paper Sec. 4.2-4.3, Eqs. (7) and (8)):

* Causal convolution at a segment boundary.  A depthwise causal convolution of width k on
  the q/k/v path makes the first k - 1 outputs of a segment depend on the previous segment's
  last k - 1 inputs.  The cache keeps those inputs (the segment's conv tail) and the seam
  window recomputes the first tokens from them.  Reading: weights [C, k] in the
  cross-correlation order of a depthwise conv1d with left padding k - 1, i.e.
      y_t[c] = act(bias[c] + sum_{j=0}^{k-1} W[c, j] x_{t-k+1+j}[c]),
  act = identity or SiLU (the pages name no activation; SiLU is offered because the
  short convolutions of gated-delta layers commonly use it); a segment shorter than k - 1
  tokens pads its tail with zeros at the front (a segment prefilled alone starts from a zero
  conv state).
* RoPE key re-rotation, Eq. (8): K_b = R(b - a) K_a.  Reading: rotate-half pairing (dims i and
  i + r/2 form a pair, i < r/2), r = rotary dims (r <= d, even; dims >= r are not rotated),
  frequencies theta_i = base^(-2i/r); R(D) turns pair i by the angle D * theta_i.
* Linear-layer state re-rotation for the scalar families, Eq. (7): S_{C|b} = R(b - a) S_{C|a},
  R acting on the key index (rows) of S.  It holds because gamma I commutes with R; the pages
  do not extend it to transitions that do not commute with rotations (diagonal, delta), and
  neither does the library.
"""
from __future__ import annotations

import math

import numpy as np


def _f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def rope_angles(delta, r, base):
    """Angle of pair i (i < r/2) for a shift of delta positions: delta * base^(-2i/r)."""
    assert r % 2 == 0 and r > 0
    return np.array([float(delta) * base ** (-2.0 * i / r) for i in range(r // 2)], dtype=np.float64)


def rope_shift(K, delta, r, base=10000.0):
    """R(delta) applied to the last axis of K (Eq. (8)); dims >= r pass through."""
    K = _f64(K)
    d = K.shape[-1]
    assert r <= d
    out = K.copy()
    h = r // 2
    ang = rope_angles(delta, r, base)
    flat_in = K.reshape(-1, d)
    flat_out = out.reshape(-1, d)
    for row in range(flat_in.shape[0]):
        for i in range(h):
            c, s = math.cos(ang[i]), math.sin(ang[i])
            x, y = flat_in[row, i], flat_in[row, i + h]
            flat_out[row, i] = c * x - s * y
            flat_out[row, i + h] = s * x + c * y
    return out


def state_rerotate(S, delta, r, base=10000.0):
    """S_{C|b} = R(delta) S_{C|a} for the scalar families (Eq. (7)): rows of S [d_k, d_v]."""
    S = _f64(S)
    # R acts on the key index, which is the row index: rotate the columns of S^T as vectors.
    return np.ascontiguousarray(rope_shift(S.T, delta, r, base).T)


def conv_tail(x, beg, end, k):
    """Last k - 1 inputs of the segment body x[beg:end] ([k-1, C]), zero-padded at the front."""
    x = _f64(x)
    C = x.shape[1]
    tail = np.zeros((max(k - 1, 0), C))
    for m in range(k - 1):
        t = end - (k - 1) + m
        if t >= beg:
            tail[m] = x[t]
    return tail


def _silu(z):
    return z / (1.0 + math.exp(-z))


def conv_seam(x_seam, tail, W, bias=None, act="identity"):
    """Outputs of the first tokens of a segment: x_seam [w, C], the previous tail [k-1, C]."""
    x_seam, tail, W = _f64(x_seam), _f64(tail), _f64(W)
    w, C = x_seam.shape
    k = W.shape[1]
    y = np.zeros((w, C))
    for t in range(w):
        for c in range(C):
            acc = 0.0 if bias is None else float(bias[c])
            for j in range(k):
                src = t - k + 1 + j  # position relative to the segment start
                xv = x_seam[src, c] if src >= 0 else tail[k - 1 + src, c]
                acc += W[c, j] * xv
            y[t, c] = _silu(acc) if act == "silu" else acc
    return y
