"""GPU parity: libhypic through its C ABI against the float64 oracle on the same seeded inputs.

Small and medium cases that span several token tiles, ragged tails, every
family, both input precisions and the degenerate cases (empty segments, n = 0,
bad indices and bounds reported through the status word).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import linear_attention_state_gb300 as hy
import oracle
import workloads as W
from refs import TOL_BF16, TOL_F32, host_tokens, np64, ref_pair, ref_run, relerr, t_as_dense

pytestmark = pytest.mark.gpu
FAMS = ["scalar_const", "scalar", "diag", "delta", "gated_delta", "kda"]
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from linear_attention_state_gb300 import build
    build.build_library()
    hy.load()
    torch.cuda.init()
    assert hy.stream_status() == 0


def tol(in_dtype):
    return TOL_F32 if in_dtype == "f32" else TOL_BF16


def draw(n, H, d, family, in_dtype, key):
    g = W.generator(DEV, 5000, key)
    return W.draw_tokens(g, n, H, d, family, in_dtype, DEV, gate_div=16.0 if family == "diag" else None)


# ---- workload 0: tiny fp32 gated delta, 2 heads, d = 16, 4 x 64 tokens, w = 4 -------------

def test_tiny_build_pairs_and_outputs():
    w = W.TINY
    tok = w.draw_request(DEV)
    bounds = torch.tensor(w.body_bounds(), dtype=torch.int64, device=DEV)
    T, S, o = hy.segment_build_batched(tok["k"], tok["v"], bounds, tok["alpha"], tok["beta"], q=tok["q"],
                                       family=w.family, want_o=True)
    assert hy.stream_status() == 0
    host = host_tokens(tok, list(range(w.H)))
    errs = []
    for s, (b, e) in enumerate(w.body_bounds()):
        for h in range(w.H):
            Tr, Sr = ref_pair(w.family, host, h, b, e)
            errs.append(relerr(np64(T[s, h]), Tr))
            errs.append(relerr(np64(S[s, h]), Sr))
            _, orf = ref_run(w.family, host, h, b, e, want_o=True)
            errs.append(relerr(np64(o[b:e, h]), orf))
    assert max(errs) <= TOL_F32, max(errs)


def test_tiny_assemble_matches_full_recurrence():
    w = W.TINY
    tok = w.draw_request(DEV)
    bounds = w.body_bounds()
    T, S = hy.segment_build_batched(tok["k"], tok["v"], torch.tensor(bounds, device=DEV), tok["alpha"],
                                    tok["beta"], family=w.family)
    seam_pos = torch.tensor(w.seam_positions(), device=DEV)
    sk = tok["k"][seam_pos].reshape(1, w.n_seg - 1, w.w, w.H, w.d).contiguous()
    sv = tok["v"][seam_pos].reshape(1, w.n_seg - 1, w.w, w.H, w.d).contiguous()
    sq = tok["q"][seam_pos].reshape(1, w.n_seg - 1, w.w, w.H, w.d).contiguous()
    sa = tok["alpha"][seam_pos].reshape(1, w.n_seg - 1, w.w, w.H).contiguous()
    sb = tok["beta"][seam_pos].reshape(1, w.n_seg - 1, w.w, w.H).contiguous()
    idx = torch.arange(w.n_seg, dtype=torch.int32, device=DEV)[None]
    S_out, o = hy.assemble(T, S, idx, sk, sv, sa, sb, seam_q=sq, family=w.family)
    assert hy.stream_status() == 0
    host = host_tokens(tok, list(range(w.H)))
    n_tok = w.n_seg * w.seg_len
    pos = w.seam_positions()
    for h in range(w.H):
        S_ref, o_ref = ref_run(w.family, host, h, 0, n_tok, want_o=True)
        assert relerr(np64(S_out[0, h]), S_ref) <= TOL_F32
        got = np64(o[0, :, :, h]).reshape(len(pos), w.d)
        assert relerr(got, o_ref[pos]) <= TOL_F32


# ---- build: every family, both precisions, ragged and empty bodies -----------------------

@pytest.mark.parametrize("family", FAMS)
@pytest.mark.parametrize("d,in_dtype", [(16, "f32"), (32, "f32"), (64, "bf16"), (128, "bf16"), (128, "f32")])
def test_build_families(family, d, in_dtype):
    H = 3
    lens = [0, 1, 37, 200, 64]
    n = sum(lens) + 5
    tok = draw(n, H, d, family, in_dtype, key=d * 10 + FAMS.index(family))
    bounds, off = [], 3
    for L_ in lens:
        bounds.append((off, off + L_))
        off += L_
    T, S, o = hy.segment_build_batched(tok["k"], tok["v"], torch.tensor(bounds, device=DEV), tok["alpha"],
                                       tok["beta"], q=tok["q"], family=family, want_o=True)
    assert hy.stream_status() == 0
    host = host_tokens(tok, list(range(H)))
    worst = 0.0
    for s, (b, e) in enumerate(bounds):
        for h in range(H):
            Tr, Sr = ref_pair(family, host, h, b, e)
            worst = max(worst, relerr(t_as_dense(family, np64(T[s, h]), d), t_as_dense(family, Tr, d)))
            if e > b:
                worst = max(worst, relerr(np64(S[s, h]), Sr))
                _, orf = ref_run(family, host, h, b, e, want_o=True)
                worst = max(worst, relerr(np64(o[b:e, h]), orf))
            else:
                assert float(S[s, h].abs().max()) == 0.0
    assert worst <= tol(in_dtype), worst


def test_single_segment_build_and_empty():
    d, H = 128, 2
    tok = draw(300, H, d, "gated_delta", "bf16", key=77)
    T, S = hy.segment_build(tok["k"], tok["v"], tok["alpha"], tok["beta"], family="gated_delta")
    host = host_tokens(tok, list(range(H)))
    for h in range(H):
        Tr, Sr = ref_pair("gated_delta", host, h, 0, 300)
        assert relerr(np64(T[h]), Tr) <= TOL_BF16
        assert relerr(np64(S[h]), Sr) <= TOL_BF16
    e = tok["k"][:0]
    T0, S0 = hy.segment_build(e, tok["v"][:0], tok["alpha"][:0], tok["beta"][:0], family="gated_delta")
    assert torch.equal(T0, torch.eye(d, device=DEV).expand(H, d, d))
    assert float(S0.abs().max()) == 0.0


# ---- compose / scan / seam advance on generator-drawn pairs --------------------------------

def random_pool(family, P, H, d, key):
    T, S = W.random_pairs(P, H, d, DEV, key=key)
    if family in ("scalar_const", "scalar"):
        T = 0.5 + 0.5 * torch.rand((P, H), device=DEV, generator=W.generator(DEV, 31, key))
    elif family == "diag":
        T = 0.5 + 0.5 * torch.rand((P, H, d), device=DEV, generator=W.generator(DEV, 32, key))
    return T.contiguous(), S


@pytest.mark.parametrize("family", FAMS)
@pytest.mark.parametrize("d", [16, 64, 128])
def test_compose_random_pairs(family, d):
    P, H, B, n = 11, 3, 4, 7
    pool_T, pool_S = random_pool(family, P, H, d, key=d + FAMS.index(family))
    g = W.generator("cpu", 33, d)
    idx = torch.stack([torch.randperm(P, generator=g)[:n] for _ in range(B)]).to(torch.int32)
    S_init = torch.randn((B, H, d, d), device=DEV, generator=W.generator(DEV, 34, d))
    for init in (None, S_init):
        out = hy.compose(pool_T, pool_S, idx.to(DEV), S_init=init, family=family)
        assert hy.stream_status() == 0
        Th, Sh = np64(pool_T), np64(pool_S)
        for b in range(B):
            for h in range(H):
                ids = idx[b].tolist()
                ref = oracle.compose(family, Th[ids, h].reshape(n, -1), Sh[ids, h],
                                     S_init=None if init is None else np64(init[b, h]))
                assert relerr(np64(out[b, h]), ref) <= TOL_F32


def test_compose_in_place_and_n_zero():
    d, H, P = 128, 2, 5
    pool_T, pool_S = random_pool("gated_delta", P, H, d, key=9)
    S = torch.randn((1, H, d, d), device=DEV)
    S0 = S.clone()
    idx0 = torch.zeros((1, 0), dtype=torch.int32, device=DEV)
    out = hy.compose(pool_T, pool_S, idx0, S_init=S, family="gated_delta")
    assert torch.equal(out, S0)
    out = hy.compose(pool_T, pool_S, idx0, family="gated_delta")
    assert float(out.abs().max()) == 0.0
    idx = torch.tensor([[3, 1, 4]], dtype=torch.int32, device=DEV)
    ref = hy.compose(pool_T, pool_S, idx, S_init=S0, family="gated_delta")
    hy.compose(pool_T, pool_S, idx, S_init=S, family="gated_delta", out=S)
    assert torch.equal(S, ref)


@pytest.mark.parametrize("family", FAMS)
@pytest.mark.parametrize("d", [16, 128])
def test_affine_scan(family, d):
    n, H = 9, 2
    T, S = random_pool(family, n, H, d, key=200 + d + FAMS.index(family))
    Tp, Sp = hy.affine_scan(T, S, family=family)
    assert hy.stream_status() == 0
    Th, Sh = np64(T), np64(S)
    for h in range(H):
        Tr, Sr = oracle.affine_scan(family, Th[:, h].reshape(n, -1), Sh[:, h])
        for i in range(n):
            assert relerr(t_as_dense(family, np64(Tp[i, h]), d), t_as_dense(family, Tr[i], d)) <= TOL_F32
            assert relerr(np64(Sp[i, h]), Sr[i]) <= TOL_F32


def test_long_chains_and_scan_fp32_pairs():
    """Compose chains and scans of 1, 2, 3 and 41 steps over fp32 DeltaNet pairs, so every
    split buffer and signal of the pipelined chain is reused many times and the short chains end
    before it fills, against the oracle."""
    d, H, P = 128, 2, 13
    pool_T, pool_S = random_pool("delta", P, H, d, key=515)
    Th, Sh = np64(pool_T), np64(pool_S)
    g = np.random.default_rng(8)
    for n in (1, 2, 3, 41):
        idx = torch.tensor(g.integers(0, P, size=(3, n)), dtype=torch.int32)
        S_init = torch.randn((3, H, d, d), device=DEV, generator=W.generator(DEV, 36, n))
        out = hy.compose(pool_T, pool_S, idx.to(DEV), S_init=S_init, family="delta")
        assert hy.stream_status() == 0
        for b in range(3):
            for h in range(H):
                ids = idx[b].tolist()
                ref = oracle.compose("delta", Th[ids, h].reshape(n, -1), Sh[ids, h], S_init=np64(S_init[b, h]))
                assert relerr(np64(out[b, h]), ref) <= TOL_F32, (n, b, h)
    for n in (1, 2, 3, 41):
        T, S = random_pool("delta", n, H, d, key=516 + n)
        Tp, Sp = hy.affine_scan(T, S, family="delta")
        assert hy.stream_status() == 0
        for h in range(H):
            Tr, Sr = oracle.affine_scan("delta", np64(T[:, h]).reshape(n, -1), np64(S[:, h]))
            for i in sorted({0, 1, 2, 20, n - 1} & set(range(n))):
                assert relerr(np64(Tp[i, h]), Tr[i].reshape(d, d)) <= TOL_F32, (n, h, i)
                assert relerr(np64(Sp[i, h]), Sr[i]) <= TOL_F32, (n, h, i)


@pytest.mark.parametrize("H,n", [(2, 64), (1, 48), (3, 40), (2, 200)])
def test_two_level_scan(H, n):
    """With few heads the scan runs in two levels (chunk totals, a scan of the totals, every chunk
    again from its carry).  Transitions are orthogonal matrices, so the prefixes keep norm 1 and
    the relative error stays meaningful over long chains; every prefix is checked against the
    oracle, for the two-level scan and for the plain one (no workspace).  Chains up to 64 pairs
    (the workloads' lengths) are held to the fp32 tolerance.  Beyond that each fp32 composition step
    adds its own rounding (about sqrt(128) units of 2^-24 for a 128-term product), so a chain of n
    steps is held to n * 6.7e-7 and both scans must stay within it."""
    d = 128
    g = torch.Generator().manual_seed(1000 * H + n)
    Q, _ = torch.linalg.qr(torch.randn((n, H, d, d), generator=g, dtype=torch.float64))
    T = Q.to(torch.float32).contiguous().to(DEV)
    S = torch.randn((n, H, d, d), generator=g).to(DEV)
    outs = {"two-level": hy.affine_scan(T, S, family="delta"),
            "plain": hy.affine_scan(T, S, family="delta", two_level=False)}
    assert hy.stream_status() == 0
    tol = TOL_F32 if n <= 64 else n * 6.7e-7
    worst = {name: 0.0 for name in outs}
    for h in range(H):
        Tr, Sr = oracle.affine_scan("delta", np64(T[:, h]).reshape(n, -1), np64(S[:, h]))
        for name, (Tp, Sp) in outs.items():
            for i in range(n):
                worst[name] = max(worst[name], relerr(np64(Tp[i, h]), Tr[i].reshape(d, d)),
                                  relerr(np64(Sp[i, h]), Sr[i]))
    print(f"two-level scan H={H} n={n}: {worst}")
    assert max(worst.values()) <= tol, worst


@pytest.mark.parametrize("family", FAMS)
@pytest.mark.parametrize("d,in_dtype", [(16, "f32"), (128, "bf16")])
def test_seam_advance(family, d, in_dtype):
    B, w, H = 3, 8, 2
    tok = draw(B * w, H, d, family, in_dtype, key=300 + d + FAMS.index(family))
    S = torch.randn((B, H, d, d), device=DEV, generator=W.generator(DEV, 35, d))
    S_before = S.clone()

    def bw(t):
        return None if t is None else t.reshape(B, w, *t.shape[1:]).contiguous()

    alpha = tok["alpha"] if family == "scalar_const" else bw(tok["alpha"])
    o = hy.seam_advance(S, bw(tok["k"]), bw(tok["v"]), alpha, bw(tok["beta"]) if tok["beta"] is not None else None,
                        q=bw(tok["q"]), family=family)
    assert hy.stream_status() == 0
    host = host_tokens(tok, list(range(H)))
    for b in range(B):
        for h in range(H):
            Sr, orf = ref_run(family, host, h, b * w, (b + 1) * w, S0=np64(S_before[b, h]), want_o=True)
            assert relerr(np64(S[b, h]), Sr) <= tol(in_dtype)
            assert relerr(np64(o[b, :, h]), orf) <= tol(in_dtype)


# ---- device-side checks report through the status word, never fault -----------------------

def test_bad_pool_index_is_reported():
    d, H, P = 16, 2, 4
    pool_T, pool_S = random_pool("gated_delta", P, H, d, key=5)
    idx = torch.tensor([[0, 7]], dtype=torch.int32, device=DEV)
    hy.compose(pool_T, pool_S, idx, family="gated_delta")
    assert hy.stream_status() == hy._lib.HYPIC_EDEVICE
    assert hy.stream_status() == 0  # cleared


def test_bad_bounds_are_reported():
    tok = draw(32, 2, 16, "gated_delta", "f32", key=6)
    bounds = torch.tensor([[0, 16], [20, 40]], dtype=torch.int64, device=DEV)  # 40 > 32 tokens
    hy.segment_build_batched(tok["k"], tok["v"], bounds, tok["alpha"], tok["beta"], family="gated_delta",
                             max_len=20)
    assert hy.stream_status() == hy._lib.HYPIC_EDEVICE
    bounds = torch.tensor([[0, 16], [10, 5]], dtype=torch.int64, device=DEV)
    hy.segment_build_batched(tok["k"], tok["v"], bounds, tok["alpha"], tok["beta"], family="gated_delta",
                             max_len=16)
    assert hy.stream_status() == hy._lib.HYPIC_EDEVICE
    assert hy.stream_status() == 0
