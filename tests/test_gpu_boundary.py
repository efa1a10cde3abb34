"""GPU parity of the boundary patches against the float64 oracle (``oracle/boundary.py``).

RoPE key shift (Eq. (8)), scalar-family state re-rotation (Eq. (7)), the causal-conv tail
of segment bodies and the conv over the seam window (HYPIC notes, Method 6), in fp32 and
bf16, with ragged sizes (rows and channel counts that are not multiples of a warp), partial
rotary dims, large and negative shifts, short and empty segments, and the degenerate
widths k = 1 and w = 0.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import linear_attention_state_gb300 as hy
import workloads as W
from oracle import boundary as B
from refs import TOL_BF16, TOL_F32, np64, relerr

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from linear_attention_state_gb300 import build
    build.build_library()
    hy.load()
    assert hy.stream_status() == 0


def randn(shape, key, dtype=torch.float32):
    return torch.randn(shape, device=DEV, generator=W.generator(DEV, 8800, key)).to(dtype)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("d,rot,base,delta", [(128, 128, 1e4, 5), (128, 32, 1e6, -3), (96, 64, 500.0, 131071),
                                              (128, 128, 1e7, 0)])
def test_rope_shift(dtype, d, rot, base, delta):
    K = randn((37, 3, d), key=d + rot, dtype=dtype)
    out = hy.rope_shift(K, delta, rot_dim=rot, base=base)
    assert hy.stream_status() == 0
    ref = B.rope_shift(np64(K).reshape(-1, d), delta, rot, base).reshape(37, 3, d)
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    assert relerr(np64(out), ref) <= tol
    assert torch.equal(out[..., rot:], K[..., rot:])  # pass-through dims are copied bit for bit
    # in place
    K2 = K.clone()
    hy.rope_shift(K2, delta, rot_dim=rot, base=base, out=K2)
    assert torch.equal(K2, out)


@pytest.mark.parametrize("dtype,rot", [(torch.float32, 96), (torch.bfloat16, 96), (torch.bfloat16, 100)])
def test_rope_shift_many_rows(dtype, rot):
    """Enough rows for several grid-stride passes of every CTA, with a ragged last pass (and, at
    rot = 100 in bf16, rows that are not whole 16-byte groups): sampled rows against the oracle,
    the pass-through dims bit for bit."""
    d, delta, base = 128, 70_001, 1e6
    K = randn((10007, 4, d), key=77 + rot, dtype=dtype)
    out = hy.rope_shift(K, delta, rot_dim=rot, base=base)
    assert hy.stream_status() == 0
    fin, fout = K.reshape(-1, d), out.reshape(-1, d)
    n = fin.shape[0]
    rows = sorted({0, 1, n - 2, n - 1, *np.random.default_rng(5).integers(0, n, 200).tolist()})
    ref = B.rope_shift(np64(fin[rows]), delta, rot, base)
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    assert relerr(np64(fout[rows]), ref) <= tol
    assert torch.equal(out[..., rot:], K[..., rot:])
    # in place over the same rows: every block is read before any of its rows is written
    K2 = K.clone()
    hy.rope_shift(K2, delta, rot_dim=rot, base=base, out=K2)
    assert hy.stream_status() == 0
    assert torch.equal(K2, out)


def test_state_rerotate_many_matrices():
    """In place over 40 x 32 matrices (several grid-stride passes): sampled matrices against the
    oracle."""
    S = randn((40, 32, 128, 128), key=91)
    S0 = S.clone()
    hy.state_rerotate(S, 70_001, rot_dim=128, base=1e6, family="scalar")
    assert hy.stream_status() == 0
    for n, h in [(0, 0), (17, 5), (39, 31), (39, 30)]:
        assert relerr(np64(S[n, h]), B.state_rerotate(np64(S0[n, h]), 70_001, 128, 1e6)) <= TOL_F32


def test_rope_shift_makes_cached_keys_global():
    """Keys rotated at segment-local positions, shifted by the segment start, equal keys rotated
    at their global positions (computed by the oracle)."""
    d, start, L = 128, 70_001, 16
    raw = np64(randn((L, d), key=3))
    cached = np.stack([B.rope_shift(raw[p], p, d, 1e4) for p in range(L)]).astype(np.float32)
    moved = hy.rope_shift(torch.tensor(cached, device=DEV), start, base=1e4)
    glob = np.stack([B.rope_shift(raw[p], start + p, d, 1e4) for p in range(L)])
    assert relerr(np64(moved), glob) <= TOL_F32


@pytest.mark.parametrize("rot", [128, 64])
def test_state_rerotate(rot):
    S = randn((3, 2, 128, 128), key=rot)
    S0 = S.clone()
    hy.state_rerotate(S, 4097, rot_dim=rot, base=1e4, family="scalar")
    assert hy.stream_status() == 0
    for n in range(3):
        for h in range(2):
            assert relerr(np64(S[n, h]), B.state_rerotate(np64(S0[n, h]), 4097, rot, 1e4)) <= TOL_F32
    with pytest.raises(hy.HypicError):
        hy.state_rerotate(S, 5, family="diag")


def test_state_rerotate_equals_build_from_rotated_keys():
    """For a scalar-gate segment, building from keys rotated by R(D) gives R(D) S_{C|0} (Eq. (7))."""
    L, H, d, D = 300, 2, 128, 513
    g = W.generator(DEV, 8801, 0)
    tok = W.draw_tokens(g, L, H, d, "scalar", "f32", DEV, need_q=False)
    T0, S0 = hy.segment_build(tok["k"], tok["v"], tok["alpha"], family="scalar")
    T1, S1 = hy.segment_build(hy.rope_shift(tok["k"], D), tok["v"], tok["alpha"], family="scalar")
    hy.state_rerotate(S0[None], D, family="scalar")
    assert hy.stream_status() == 0
    assert relerr(np64(S0), np64(S1)) <= TOL_F32
    assert relerr(np64(T0), np64(T1)) <= TOL_F32


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("k", [1, 2, 4])
def test_conv_tail(dtype, k):
    C = 200
    lens = [0, 1, 2, 3, 17, 64]
    gap = 2
    n = sum(lens) + gap * (len(lens) + 1)
    x = randn((n, C), key=10 + k, dtype=dtype)
    bounds, off = [], gap
    for L_ in lens:
        bounds.append((off, off + L_))
        off += L_ + gap
    tail = hy.conv_tail(x, torch.tensor(bounds, device=DEV), k)
    assert hy.stream_status() == 0
    assert tail.shape == (len(lens), k - 1, C)
    xh = np64(x)
    for s, (b, e) in enumerate(bounds):
        ref = torch.tensor(B.conv_tail(xh, b, e, k)).to(dtype)
        assert torch.equal(tail[s].cpu(), ref)  # a copy: bit for bit


def test_conv_tail_bad_bounds_are_reported():
    from linear_attention_state_gb300 import _lib as L
    x = randn((10, 8), key=20)
    tail = hy.conv_tail(x, torch.tensor([[2, 5], [4, 11]], device=DEV), 4)
    assert hy.stream_status() == L.HYPIC_EDEVICE
    assert hy.stream_status() == 0
    assert float(tail[1].abs().max()) == 0.0


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("k,w,act,use_bias", [(4, 8, "identity", True), (4, 3, "silu", False), (1, 5, "silu", True),
                                              (2, 1, "identity", False), (4, 0, "identity", True)])
def test_conv_seam(dtype, k, w, act, use_bias):
    Bn, C = 3, 200
    xs = randn((Bn, w, C), key=30 + k + w, dtype=dtype)
    tail = randn((Bn, k - 1, C), key=40 + k, dtype=dtype) if k > 1 else None
    Wt = randn((C, k), key=50 + k)
    bias = randn((C,), key=60) if use_bias else None
    y = hy.conv_seam(xs, tail, Wt, bias, act=act)
    assert hy.stream_status() == 0
    assert y.shape == (Bn, w, C)
    for b in range(Bn):
        ref = B.conv_seam(np64(xs[b]), np64(tail[b]) if k > 1 else np.zeros((0, C)), np64(Wt),
                          None if bias is None else np64(bias), act)
        if w:
            assert relerr(np64(y[b]), ref) <= TOL_F32


def test_conv_seam_continues_the_previous_segment():
    """Tails from conv_tail feed conv_seam: the seam outputs equal the conv over the whole token
    axis at each boundary (oracle over the concatenated sequence)."""
    C, k, w = 64, 4, 8
    lens = [40, 33, 21]
    x = randn((sum(lens), C), key=70)
    Wt, bias = randn((C, k), key=71), randn((C,), key=72)
    bounds, off = [], 0
    for L_ in lens:
        bounds.append((off, off + L_))
        off += L_
    tails = hy.conv_tail(x, torch.tensor(bounds, device=DEV), k)
    seams = torch.stack([x[bounds[j][0]:bounds[j][0] + w] for j in (1, 2)])
    y = hy.conv_seam(seams, tails[:2].contiguous(), Wt, bias, act="silu")
    assert hy.stream_status() == 0
    xh = np64(x)
    for i, j in enumerate((1, 2)):
        b0 = bounds[j][0]
        # the conv at positions b0 .. b0 + w - 1 of the whole sequence, by the oracle
        ref = B.conv_seam(xh[b0:b0 + w], xh[b0 - (k - 1):b0], np64(Wt), np64(bias), "silu")
        assert relerr(np64(y[i]), ref) <= TOL_F32
