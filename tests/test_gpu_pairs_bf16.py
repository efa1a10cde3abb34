"""GPU parity of 16-bit pair storage: rounding to bf16, and composition over bf16 pools.

The paper sizes its cache with 16-bit T_C and S (HYPIC notes, Method 3, Table 3).
hypic_pairs_to_bf16 must round exactly as IEEE round-to-nearest-even does (checked bit
for bit against the CPU conversion, including ties, subnormals and a ragged tail).
Composition over bf16 pools takes the stored values exactly, so it is checked against
the float64 oracle composing the same stored values, at the fp32 tolerance.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import linear_attention_state_gb300 as hy
import oracle
import workloads as W
from refs import TOL_BF16, TOL_F32, np64, relerr

pytestmark = pytest.mark.gpu
FAMS = ["scalar_const", "scalar", "diag", "delta", "gated_delta", "kda"]
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from linear_attention_state_gb300 import build
    build.build_library()
    hy.load()
    assert hy.stream_status() == 0


def random_pool(family, P, H, d, key):
    T, S = W.random_pairs(P, H, d, DEV, key=key)
    if family in ("scalar_const", "scalar"):
        T = 0.5 + 0.5 * torch.rand((P, H), device=DEV, generator=W.generator(DEV, 41, key))
    elif family == "diag":
        T = 0.5 + 0.5 * torch.rand((P, H, d), device=DEV, generator=W.generator(DEV, 42, key))
    return T.contiguous(), S


def bits(t):
    return t.cpu().view(torch.int16).numpy()


@pytest.mark.parametrize("family", ["gated_delta", "diag", "scalar"])
def test_rounding_is_nearest_even_bit_for_bit(family):
    P, H, d = 3, 5, 16 if family != "gated_delta" else 128
    T, S = random_pool(family, P, H, d, key=1)
    # values that probe the rounding: exact ties (1 + 2^-8 rounds down to even, 1 + 3 * 2^-8 up),
    # just above a tie, fp32 subnormals, signed zeros, large magnitudes
    probe = torch.tensor([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -8 + 2.0 ** -20, -(1.0 + 2.0 ** -8),
                          1e-40, -3e-39, 0.0, -0.0, 3.0e38, -2.5e38, 65504.0, 2.0 ** -126], dtype=torch.float32)
    flat = S.view(-1)
    flat[:probe.numel()] = probe.to(DEV)
    T_lp, S_lp = hy.pairs_to_bf16(T, S, family=family)
    assert hy.stream_status() == 0
    assert T_lp.dtype == torch.bfloat16 and T_lp.shape == T.shape
    assert np.array_equal(bits(T_lp), bits(T.cpu().to(torch.bfloat16)))
    assert np.array_equal(bits(S_lp), bits(S.cpu().to(torch.bfloat16)))
    # T of the scalar families has P * H = 15 elements: not a multiple of the 8-wide groups
    if family == "scalar":
        assert T.numel() % 8 != 0


@pytest.mark.parametrize("family", FAMS)
@pytest.mark.parametrize("d", [16, 128])
def test_compose_over_bf16_pool(family, d):
    if d != 128 and family in ("delta", "gated_delta", "kda"):
        pytest.skip("bf16 pools of the delta families run on the d = 128 tensor-core chain only")
    P, H, B, n = 11, 3, 4, 7
    T, S = random_pool(family, P, H, d, key=10 + d + FAMS.index(family))
    T_lp, S_lp = T.to(torch.bfloat16), S.to(torch.bfloat16)  # stored values, rounded outside the library
    g = W.generator("cpu", 43, d)
    idx = torch.stack([torch.randperm(P, generator=g)[:n] for _ in range(B)]).to(torch.int32)
    S_init = torch.randn((B, H, d, d), device=DEV, generator=W.generator(DEV, 44, d))
    Th, Sh = np64(T_lp), np64(S_lp)
    for init in (None, S_init):
        out = hy.compose(T_lp, S_lp, idx.to(DEV), S_init=init, family=family)
        assert hy.stream_status() == 0
        worst = 0.0
        for b in range(B):
            for h in range(H):
                ids = idx[b].tolist()
                ref = oracle.compose(family, Th[ids, h].reshape(n, -1), Sh[ids, h],
                                     S_init=None if init is None else np64(init[b, h]))
                worst = max(worst, relerr(np64(out[b, h]), ref))
        assert worst <= TOL_F32, worst


def test_long_chains_over_bf16_pool():
    """Chains of 1, 2, 3 and 41 steps over a bf16 pool, so every load buffer and signal of the
    pipelined composition is reused many times and the short chains end before the pipeline
    fills, against the oracle composing the same stored values."""
    P, H, d = 13, 2, 128
    T, S = random_pool("delta", P, H, d, key=123)
    T_lp, S_lp = hy.pairs_to_bf16(T, S, family="delta")
    Th, Sh = np64(T_lp), np64(S_lp)
    g = np.random.default_rng(7)
    for n in (1, 2, 3, 41):
        idx = torch.tensor(g.integers(0, P, size=(3, n)), dtype=torch.int32)
        S_init = torch.randn((3, H, d, d), device=DEV, generator=W.generator(DEV, 46, n))
        out = hy.compose(T_lp, S_lp, idx.to(DEV), S_init=S_init, family="delta")
        assert hy.stream_status() == 0
        worst = 0.0
        for b in range(3):
            for h in range(H):
                ids = idx[b].tolist()
                ref = oracle.compose("delta", Th[ids, h].reshape(n, -1), Sh[ids, h], S_init=np64(S_init[b, h]))
                worst = max(worst, relerr(np64(out[b, h]), ref))
        assert worst <= TOL_F32, (n, worst)


def test_bf16_pool_differs_from_fp32_pool_by_the_storage_rounding():
    """Composing the rounded pool differs from composing the fp32 pool by the storage rounding
    (about 2^-9 relative per stored value), not by anything larger."""
    P, H, d, n = 8, 2, 128, 8
    T, S = random_pool("gated_delta", P, H, d, key=77)
    idx = torch.arange(n, dtype=torch.int32, device=DEV)[None]
    full = hy.compose(T, S, idx, family="gated_delta")
    T_lp, S_lp = hy.pairs_to_bf16(T, S, family="gated_delta")
    low = hy.compose(T_lp, S_lp, idx, family="gated_delta")
    assert hy.stream_status() == 0
    for h in range(H):
        e = relerr(np64(low[0, h]), np64(full[0, h]))
        assert 0.0 < e < 1e-2, e


@pytest.mark.parametrize("family", ["gated_delta", "diag", "kda"])
@pytest.mark.parametrize("d,storage", [(128, "bf16"), (128, "f32"), (16, "f32")])
def test_assemble_with_seams(family, d, storage):
    """Seams then composition per segment; the seam update of each family (KDA's per-channel gate
    included) on the tensor-core chain (d = 128) and the SIMT chains (d = 16)."""
    P, H, B, n, w = 6, 2, 2, 4, 8
    T, S = random_pool(family, P, H, d, key=90 + d + FAMS.index(family))
    if storage == "bf16":
        T, S = hy.pairs_to_bf16(T, S, family=family)
    idx = torch.tensor([[0, 3, 1, 5], [2, 4, 0, 1]], dtype=torch.int32, device=DEV)
    g = W.generator(DEV, 45, FAMS.index(family) + d)
    in_dtype = "bf16" if d == 128 else "f32"
    tok = W.draw_tokens(g, B * (n - 1) * w, H, d, family, in_dtype, DEV,
                        gate_div=16.0 if family in ("diag", "kda") else None)
    shp = (B, n - 1, w, H, d)
    sk, sv, sq = tok["k"].view(shp), tok["v"].view(shp), tok["q"].view(shp)
    sa = tok["alpha"].view((B, n - 1, w) + tok["alpha"].shape[1:])
    sb = tok["beta"].view(B, n - 1, w, H)
    S_out, o = hy.assemble(T, S, idx, sk, sv, seam_alpha=sa, seam_beta=sb, seam_q=sq, family=family)
    assert hy.stream_status() == 0
    Th, Sh = np64(T), np64(S)
    worst_s = worst_o = 0.0
    for b in range(B):
        for h in range(H):
            Sr = None
            for j in range(n):
                if j >= 1:
                    bb = np64(sb[b, j - 1, :, h]) if family in ("delta", "gated_delta", "kda") else None
                    Sr, orf = oracle.run(family, np64(sk[b, j - 1, :, h]), np64(sv[b, j - 1, :, h]),
                                         np64(sa[b, j - 1, :, h]), bb, q=np64(sq[b, j - 1, :, h]), S0=Sr)
                    worst_o = max(worst_o, relerr(np64(o[b, j - 1, :, h]), orf))
                p = int(idx[b, j])
                Sr = oracle.compose(family, Th[p:p + 1, h].reshape(1, -1), Sh[p:p + 1, h], S_init=Sr)
            worst_s = max(worst_s, relerr(np64(S_out[b, h]), Sr))
    tol = TOL_BF16 if in_dtype == "bf16" else TOL_F32
    assert worst_s <= tol and worst_o <= tol, (worst_s, worst_o)


def test_n_zero_and_in_place_over_bf16_pool():
    d, H, P = 128, 2, 5
    T, S = random_pool("gated_delta", P, H, d, key=9)
    T_lp, S_lp = hy.pairs_to_bf16(T, S)
    S_cur = torch.randn((1, H, d, d), device=DEV)
    S_keep = S_cur.clone()
    idx0 = torch.zeros((1, 0), dtype=torch.int32, device=DEV)
    assert torch.equal(hy.compose(T_lp, S_lp, idx0, S_init=S_cur), S_keep)
    idx = torch.tensor([[3, 1, 4]], dtype=torch.int32, device=DEV)
    ref = hy.compose(T_lp, S_lp, idx, S_init=S_keep)
    hy.compose(T_lp, S_lp, idx, S_init=S_cur, out=S_cur)
    assert hy.stream_status() == 0
    assert torch.equal(S_cur, ref)
