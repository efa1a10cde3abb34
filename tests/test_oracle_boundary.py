"""Pins for the boundary-patch oracle (``oracle/boundary.py``).

Each pin states the same quantity independently of the oracle's loops:

* RoPE shift (HYPIC notes, Method 6, paper Eq. (8)): the pairs as complex numbers multiplied
  by exp(i D theta_j); the group law R(a) R(b) = R(a + b); R(0) = I; pair norms kept; the
  relative-position property that makes the cache reusable (a key prefilled at its
  segment-local position and shifted by b equals the key prefilled at its global position,
  and attention scores depend only on position differences).
* State re-rotation for the scalar families (Eq. (7)): a segment built by the float64 C
  oracle from keys rotated by R(D) has S = R(D) S_{C|0} of the unrotated keys and the same
  T_C; for the diagonal family the identity fails (why the library refuses it).
* Causal convolution: seam outputs equal the full-sequence depthwise conv1d (torch on the
  CPU) over [previous segment | this segment] at the boundary; a short segment's tail
  equals that of the segment prefilled alone from a zero state.

``test_pins_catch_planted_mistakes`` plants plausible mistakes in a copy of the oracle and
checks that some pin catches each.
"""
from __future__ import annotations

import importlib.util
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import boundary as B


def rel(a, b):
    return float(np.linalg.norm(np.asarray(a) - np.asarray(b)) / max(np.linalg.norm(b), 1e-300))


# ---- RoPE ------------------------------------------------------------------------------------

def pin_rope_complex(mod):
    rng = np.random.default_rng(1)
    for d, r, base, delta in [(8, 8, 10000.0, 3), (16, 8, 500.0, 1000), (128, 128, 1e6, 131071), (6, 2, 10.0, -7)]:
        K = rng.standard_normal((5, d))
        out = mod.rope_shift(K, delta, r, base)
        h = r // 2
        z = K[:, :h] + 1j * K[:, h:r]
        theta = base ** (-2.0 * np.arange(h) / r)
        zr = z * np.exp(1j * delta * theta)
        ref = K.copy()
        ref[:, :h], ref[:, h:r] = zr.real, zr.imag
        assert rel(out, ref) < 1e-12


def pin_rope_group_law(mod):
    rng = np.random.default_rng(2)
    K = rng.standard_normal((4, 32))
    a, b = 17, 345
    two = mod.rope_shift(mod.rope_shift(K, a, 24, 1e4), b, 24, 1e4)
    one = mod.rope_shift(K, a + b, 24, 1e4)
    assert rel(two, one) < 1e-12
    assert rel(mod.rope_shift(K, 0, 24, 1e4), K) == 0.0
    back = mod.rope_shift(one, -(a + b), 24, 1e4)
    assert rel(back, K) < 1e-12
    out = mod.rope_shift(K, 99, 24, 1e4)
    assert np.array_equal(out[:, 24:], K[:, 24:])  # partial rotary: the rest passes through
    n_in = K[:, :12] ** 2 + K[:, 12:24] ** 2
    n_out = out[:, :12] ** 2 + out[:, 12:24] ** 2
    assert np.allclose(n_in, n_out, rtol=1e-12)


def pin_rope_relative_positions(mod):
    """Why Eq. (8) makes segment caches position-independent."""
    rng = np.random.default_rng(3)
    d, r, base = 16, 16, 1e4
    raw = rng.standard_normal((6, d))  # un-rotated keys of a 6-token segment
    b = 1234                            # the segment's start in the request
    cached = np.stack([mod.rope_shift(raw[p], p, r, base) for p in range(6)])  # local positions
    global_ = np.stack([mod.rope_shift(raw[p], b + p, r, base) for p in range(6)])
    assert rel(mod.rope_shift(cached, b, r, base), global_) < 1e-12
    q = rng.standard_normal(d)
    m = 2000
    qm = mod.rope_shift(q, m, r, base)
    for p in range(6):
        score = float(qm @ global_[p])
        assert abs(score - float(q @ mod.rope_shift(raw[p], b + p - m, r, base))) < 1e-9 * (1 + abs(score))


# ---- state re-rotation -----------------------------------------------------------------------

def pin_state_rerotate(mod):
    rng = np.random.default_rng(4)
    dk, dv, L, r, base, D = 8, 5, 11, 8, 100.0, 37
    k = rng.standard_normal((L, dk))
    v = rng.standard_normal((L, dv))
    for fam, alpha in (("scalar_const", np.array([0.93])), ("scalar", 0.5 + 0.5 * rng.random(L))):
        T0, S0 = oracle.segment_pair(fam, k, v, alpha)
        kr = mod.rope_shift(k, D, r, base)
        T1, S1 = oracle.segment_pair(fam, kr, v, alpha)
        assert rel(mod.state_rerotate(S0, D, r, base), S1) < 1e-12
        assert abs(float(np.asarray(T0).reshape(-1)[0]) - float(np.asarray(T1).reshape(-1)[0])) < 1e-15
    # diagonal transitions do not commute with rotations: the identity fails there
    alpha = 0.3 + 0.7 * rng.random((L, dk))
    _, S0 = oracle.segment_pair("diag", k, v, alpha)
    _, S1 = oracle.segment_pair("diag", mod.rope_shift(k, D, r, base), v, alpha)
    assert rel(mod.state_rerotate(S0, D, r, base), S1) > 1e-3


# ---- causal convolution ----------------------------------------------------------------------

def torch_causal_conv(x, W, bias, act):
    """Depthwise causal conv1d over a whole sequence x [L, C] (library routine, CPU, float64)."""
    C, k = W.shape
    xt = torch.tensor(x.T[None], dtype=torch.float64)
    wt = torch.tensor(W[:, None, :], dtype=torch.float64)
    bt = None if bias is None else torch.tensor(bias, dtype=torch.float64)
    y = torch.nn.functional.conv1d(torch.nn.functional.pad(xt, (k - 1, 0)), wt, bt, groups=C)[0].T
    if act == "silu":
        y = torch.nn.functional.silu(y)
    return y.numpy()


def pin_conv_boundary(mod):
    rng = np.random.default_rng(5)
    for k, w, act, use_bias in [(4, 8, "identity", True), (4, 3, "silu", False), (1, 5, "identity", True),
                                (2, 1, "silu", True), (4, 0, "identity", False)]:
        C, L1, L2 = 6, 13, max(w, 1) + 4
        x = rng.standard_normal((L1 + L2, C))
        W = rng.standard_normal((C, k))
        bias = rng.standard_normal(C) if use_bias else None
        full = torch_causal_conv(x, W, bias, act)
        tail = mod.conv_tail(x, 0, L1, k)
        y = mod.conv_seam(x[L1:L1 + w], tail, W, bias, act)
        assert y.shape == (w, C)
        if w:
            assert rel(y, full[L1:L1 + w]) < 1e-12


def pin_conv_short_segment(mod):
    rng = np.random.default_rng(6)
    C, k = 3, 5
    seg = rng.standard_normal((2, C))  # shorter than k - 1
    x = np.concatenate([rng.standard_normal((7, C)), seg])
    tail = mod.conv_tail(x, 7, 9, k)
    alone = np.concatenate([np.zeros((k - 1, C)), seg])  # prefilled alone from a zero state
    assert np.array_equal(tail, alone[-(k - 1):])
    assert mod.conv_tail(x, 0, 9, 1).shape == (0, C)


PINS = [pin_rope_complex, pin_rope_group_law, pin_rope_relative_positions, pin_state_rerotate,
        pin_conv_boundary, pin_conv_short_segment]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_boundary_pin(pin):
    pin(B)


MUTANTS = {
    "rotation_sign_flipped": ("flat_out[row, i] = c * x - s * y", "flat_out[row, i] = c * x + s * y"),
    "interleaved_pairs": ("x, y = flat_in[row, i], flat_in[row, i + h]", "x, y = flat_in[row, 2 * i], flat_in[row, 2 * i + 1]"),
    "frequency_exponent": ("base ** (-2.0 * i / r)", "base ** (-1.0 * i / r)"),
    "state_rotates_columns": ("return np.ascontiguousarray(rope_shift(S.T, delta, r, base).T)",
                              "return np.ascontiguousarray(rope_shift(S, delta, r, base))"),
    "conv_tap_reversed": ("acc += W[c, j] * xv", "acc += W[c, k - 1 - j] * xv"),
    "conv_tail_off_by_one": ("t = end - (k - 1) + m", "t = end - k + m"),
    "conv_drops_bias": ("acc = 0.0 if bias is None else float(bias[c])", "acc = 0.0"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(name, tmp_path):
    src = open(os.path.join(os.path.dirname(B.__file__), "boundary.py")).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    path = tmp_path / "boundary_mutant.py"
    path.write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location("boundary_mutant", str(path))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    caught = []
    for pin in PINS:
        try:
            pin(mod)
        except (AssertionError, IndexError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name}"
