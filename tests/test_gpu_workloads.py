"""GPU parity on the full-size workloads, in the launch configuration the bench times.

Each test runs the whole workload on the GPU and checks a seeded sample of heads
(or request chains) against the float64 oracle computed from the same seeded
inputs.  The oracle never consumes anything the CUDA path produced: build and
assembly are checked end to end against the plain recurrence over the request.
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
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from linear_attention_state_gb300 import build
    build.build_library()
    hy.load()
    assert hy.stream_status() == 0
    yield
    torch.cuda.empty_cache()


def seams_of(w, tok, dev=DEV):
    pos = torch.tensor(w.seam_positions(), device=dev)
    shp = (1, w.n_seg - 1, w.w, w.H)
    return (tok["k"][pos].reshape(*shp, w.d).contiguous(), tok["v"][pos].reshape(*shp, w.d).contiguous(),
            tok["alpha"][pos].reshape(shp).contiguous(), tok["beta"][pos].reshape(shp).contiguous(),
            tok["q"][pos].reshape(*shp, w.d).contiguous())


def test_build_32k_full_size_sampled_heads():
    """8 segments x 4096 tokens, 32 heads, bf16: pairs, seam outputs and composed state."""
    w = W.BUILD_32K
    tok = w.draw_request(DEV)
    bounds = w.body_bounds()
    T, S = hy.segment_build_batched(tok["k"], tok["v"], torch.tensor(bounds, device=DEV), tok["alpha"],
                                    tok["beta"], family=w.family, max_len=max(e - b for b, e in bounds))
    sk, sv, sa, sb, sq = seams_of(w, tok)
    S_out, o = hy.assemble(T, S, torch.arange(w.n_seg, dtype=torch.int32, device=DEV)[None], sk, sv, sa, sb,
                           seam_q=sq, family=w.family)
    assert hy.stream_status() == 0
    heads = [0, 13, 31]
    host = host_tokens(tok, heads)
    n_tok = w.n_seg * w.seg_len
    pos = w.seam_positions()

    def ref(i):
        pairs = [ref_pair(w.family, host, i, b, e) for b, e in bounds]
        S_full, o_full = ref_run(w.family, host, i, 0, n_tok, want_o=True)
        return pairs, S_full, o_full[pos]

    res = oracle.parallel_map(ref, range(len(heads)))
    worst = {"T": 0.0, "S": 0.0, "S_out": 0.0, "o": 0.0}
    for i, h in enumerate(heads):
        pairs, S_full, o_ref = res[i]
        for s, (Tr, Sr) in enumerate(pairs):
            worst["T"] = max(worst["T"], relerr(np64(T[s, h]), Tr))
            worst["S"] = max(worst["S"], relerr(np64(S[s, h]), Sr))
        worst["S_out"] = max(worst["S_out"], relerr(np64(S_out[0, h]), S_full))
        worst["o"] = max(worst["o"], relerr(np64(o[0, :, :, h]).reshape(len(pos), w.d), o_ref))
    print("build 32k:", {k: f"{v:.2e}" for k, v in worst.items()})
    assert max(worst.values()) <= TOL_BF16, worst


@pytest.mark.parametrize("variant", ["scalar_const", "diag", "gated_delta"])
def test_decay_families_full_size_sampled_heads(variant):
    """64 segments x 512 tokens, 32 heads, bf16, w = 0: every pair, then compose all 64 from zero."""
    w = W.DECAY_FAMILIES[variant]
    tok = w.draw_request(DEV, need_q=False)
    bounds = w.body_bounds()
    T, S = hy.segment_build_batched(tok["k"], tok["v"], torch.tensor(bounds, device=DEV), tok["alpha"],
                                    tok["beta"], family=w.family, max_len=w.seg_len)
    S_out = hy.compose(T.reshape(w.n_seg, w.H, -1).contiguous() if variant != "gated_delta" else T, S,
                       torch.arange(w.n_seg, dtype=torch.int32, device=DEV)[None], family=w.family)
    assert hy.stream_status() == 0
    heads = [0, 17, 31]
    host = host_tokens(tok, heads)

    def ref(i):
        pairs = [ref_pair(w.family, host, i, b, e) for b, e in bounds]
        S_full, _ = ref_run(w.family, host, i, 0, w.n_seg * w.seg_len)
        return pairs, S_full

    res = oracle.parallel_map(ref, range(len(heads)))
    wT = wS = wC = 0.0
    for i, h in enumerate(heads):
        pairs, S_full = res[i]
        for s, (Tr, Sr) in enumerate(pairs):
            wT = max(wT, relerr(t_as_dense(w.family, np64(T[s, h]), w.d), t_as_dense(w.family, Tr, w.d)))
            wS = max(wS, relerr(np64(S[s, h]), Sr))
        wC = max(wC, relerr(np64(S_out[0, h]), S_full))
        if variant == "scalar_const":  # closed form of the constant-decay transition
            g = float(tok["alpha"][h])
            assert abs(float(T[0, h]) / (np.float64(g) ** w.seg_len) - 1.0) < 1e-4
    print(f"decay {variant}: T {wT:.2e} S {wS:.2e} composed {wC:.2e}")
    assert max(wT, wS, wC) <= TOL_BF16


def _oracle_pool(P, heads_flat, gate_div, key):
    """Pool pairs built by the oracle (float64, then rounded to fp32) from seeded 1024-token segments."""
    pw = W.COMPOSE_POOL
    Hs = len(heads_flat)
    toks = []
    for p in range(P):
        if gate_div is None:
            t = pw.pair_inputs(p, DEV, heads=heads_flat)
        else:
            t = W.draw_tokens(W.generator(DEV, 8000 + key, p), pw.pair_tokens, Hs, pw.d, "gated_delta", "bf16", DEV,
                              gate_div=gate_div, need_q=False)
        toks.append(host_tokens(t, list(range(Hs))))

    def one(job):
        p, i = job
        return ref_pair("gated_delta", toks[p], i, 0, pw.pair_tokens)

    jobs = [(p, i) for p in range(P) for i in range(Hs)]
    out = oracle.parallel_map(one, jobs)
    T = np.zeros((P, Hs, pw.d, pw.d), np.float32)
    S = np.zeros((P, Hs, pw.d, pw.d), np.float32)
    for (p, i), (Tr, Sr) in zip(jobs, out):
        T[p, i] = Tr
        S[p, i] = Sr
    return T, S


@pytest.mark.parametrize("gate_div", [None, 1024.0], ids=["config_gates", "slow_decay"])
def test_compose_oracle_built_pool(gate_div):
    """Composition on pairs the oracle built (fp32 path, 1e-5): 16 of a pool of 20, 6 requests."""
    heads_flat = [0, 3 * 32 + 5, 17 * 32 + 9, 29 * 32 + 31]
    P, B, n = 20, 6, 16
    T, S = _oracle_pool(P, heads_flat, gate_div, key=1)
    g = W.generator("cpu", 8100, int(gate_div or 0))
    idx = torch.stack([torch.randperm(P, generator=g)[:n] for _ in range(B)]).to(torch.int32)
    out = hy.compose(torch.from_numpy(T).to(DEV), torch.from_numpy(S).to(DEV), idx.to(DEV), family="gated_delta")
    assert hy.stream_status() == 0
    T64, S64 = T.astype(np.float64), S.astype(np.float64)
    worst = 0.0
    for b in range(B):
        ids = idx[b].tolist()
        for i in range(len(heads_flat)):
            ref = oracle.compose("gated_delta", T64[ids, i].reshape(n, -1), S64[ids, i])
            worst = max(worst, relerr(np64(out[b, i]), ref))
    if gate_div is not None:
        assert float(np.linalg.norm(T64[0, 0])) > 1e-2  # the T path really matters here
    print(f"compose on oracle-built pool ({gate_div}): {worst:.2e}")
    assert worst <= TOL_F32


def test_compose_full_size_random_pairs():
    """30 x 32 heads, pool of 256 fp32 pairs, 64 requests x 16: the bench's launch, sampled chains."""
    pw = W.COMPOSE_POOL
    pool_T, pool_S = W.random_pairs(pw.pool, pw.H, pw.d, DEV, key=17)
    idx = pw.request_indices(DEV)
    out = hy.compose(pool_T, pool_S, idx, family="gated_delta")
    assert hy.stream_status() == 0
    g = np.random.default_rng(5)
    worst = 0.0
    idx_h = idx.cpu()
    for _ in range(12):
        b, h = int(g.integers(pw.B)), int(g.integers(pw.H))
        ids = idx_h[b].tolist()
        Tn = np64(pool_T[ids, h]).reshape(pw.n, -1)
        Sn = np64(pool_S[ids, h])
        ref = oracle.compose("gated_delta", Tn, Sn)
        worst = max(worst, relerr(np64(out[b, h]), ref))
    print(f"compose full size random pairs: {worst:.2e}")
    del pool_T, pool_S
    assert worst <= TOL_F32


def test_compose_full_size_bf16_pool():
    """The bench's bf16-pool launch: 30 x 32 heads, pool of 256 pairs stored in bf16, 64 requests x
    16; sampled chains against the oracle composing the same stored values."""
    pw = W.COMPOSE_POOL
    pool_T, pool_S = W.random_pairs(pw.pool, pw.H, pw.d, DEV, key=17)
    T_lp, S_lp = hy.pairs_to_bf16(pool_T, pool_S, family="gated_delta")
    del pool_T, pool_S
    idx = pw.request_indices(DEV)
    out = hy.compose(T_lp, S_lp, idx, family="gated_delta")
    assert hy.stream_status() == 0
    g = np.random.default_rng(6)
    worst = 0.0
    idx_h = idx.cpu()
    for _ in range(12):
        b, h = int(g.integers(pw.B)), int(g.integers(pw.H))
        ids = idx_h[b].tolist()
        ref = oracle.compose("gated_delta", np64(T_lp[ids, h]).reshape(pw.n, -1), np64(S_lp[ids, h]))
        worst = max(worst, relerr(np64(out[b, h]), ref))
    print(f"compose full size bf16 pool: {worst:.2e}")
    del T_lp, S_lp
    assert worst <= TOL_F32


def test_affine_scan_full_size_sampled_heads():
    """The bench's scan launch: 64 fp32 pairs x 960 heads; every prefix of sampled heads against the
    oracle."""
    n, H, d = 64, 960, 128
    T, S = W.random_pairs(n, H, d, DEV, key=11)
    Tp, Sp = hy.affine_scan(T, S, family="gated_delta")
    assert hy.stream_status() == 0
    worst = 0.0
    for h in (0, 1, 479, 959):
        Tr, Sr = oracle.affine_scan("gated_delta", np64(T[:, h]).reshape(n, -1), np64(S[:, h]))
        for i in range(n):
            worst = max(worst, relerr(np64(Tp[i, h]), Tr[i].reshape(d, d)), relerr(np64(Sp[i, h]), Sr[i]))
    print(f"affine scan full size: {worst:.2e}")
    del T, S, Tp, Sp
    assert worst <= TOL_F32


def test_long_mixed_full_size_sampled_heads():
    """30 x 32 heads, 128 segments x 1024 tokens, 96 cached + 32 cold, w = 8 on every inner segment."""
    w = W.LONG_MIXED
    H, d, n, Ls, ww = w.H, w.d, w.n_seg, w.seg_len, w.w
    cold = set(W.long_mixed_cold(w))
    pool_T = torch.empty((n, H, d, d), device=DEV)
    pool_S = torch.empty((n, H, d, d), device=DEV)
    sk = torch.empty((1, n - 1, ww, H, d), dtype=torch.bfloat16, device=DEV)
    sv = torch.empty_like(sk)
    sq = torch.empty_like(sk)
    sa = torch.empty((1, n - 1, ww, H), device=DEV)
    sb = torch.empty_like(sa)
    ws = torch.empty(hy.build_workspace_bytes(H, d, 1, Ls), dtype=torch.uint8, device=DEV)
    cold_list = sorted(cold)
    ck = torch.empty((len(cold_list) * Ls, H, d), dtype=torch.bfloat16, device=DEV)
    cv = torch.empty_like(ck)
    ca = torch.empty((len(cold_list) * Ls, H), device=DEV)
    cb = torch.empty_like(ca)
    cbounds = []
    for j in range(n):
        tok = w.draw_segment(j, DEV)
        lo = 0 if j == 0 else ww
        if j >= 1:
            sk[0, j - 1], sv[0, j - 1], sq[0, j - 1] = tok["k"][:ww], tok["v"][:ww], tok["q"][:ww]
            sa[0, j - 1], sb[0, j - 1] = tok["alpha"][:ww], tok["beta"][:ww]
        if j in cold:
            c = cold_list.index(j)
            ck[c * Ls:(c + 1) * Ls], cv[c * Ls:(c + 1) * Ls] = tok["k"], tok["v"]
            ca[c * Ls:(c + 1) * Ls], cb[c * Ls:(c + 1) * Ls] = tok["alpha"], tok["beta"]
            cbounds.append((c * Ls + lo, (c + 1) * Ls))
        else:
            body = {key: tok[key][lo:].contiguous() for key in ("k", "v", "alpha", "beta")}
            T, S = hy.segment_build_batched(body["k"], body["v"], torch.tensor([[0, Ls - lo]], device=DEV),
                                            body["alpha"], body["beta"], family=w.family, max_len=Ls, ws=ws)
            pool_T[j].copy_(T[0])
            pool_S[j].copy_(S[0])
        del tok
    # the cold segments, built in one batched call
    ws_c = torch.empty(hy.build_workspace_bytes(H, d, len(cold_list), Ls), dtype=torch.uint8, device=DEV)
    Tc, Sc = hy.segment_build_batched(ck, cv, torch.tensor(cbounds, device=DEV), ca, cb, family=w.family,
                                      max_len=Ls, ws=ws_c)
    for c, j in enumerate(cold_list):
        pool_T[j].copy_(Tc[c])
        pool_S[j].copy_(Sc[c])
    del ck, cv, ca, cb, Tc, Sc, ws_c
    S_out, o = hy.assemble(pool_T, pool_S, torch.arange(n, dtype=torch.int32, device=DEV)[None], sk, sv, sa, sb,
                           seam_q=sq, family=w.family)
    assert hy.stream_status() == 0

    heads = [0, 17 * 32 + 9, 29 * 32 + 31]
    parts = [host_tokens(w.draw_segment(j, DEV, heads=heads), list(range(len(heads)))) for j in range(n)]
    host = {key: torch.cat([p[key] for p in parts], dim=0) for key in ("k", "q", "v", "alpha", "beta")}
    pos = w.seam_positions()

    def ref(i):
        S_full, o_full = ref_run(w.family, host, i, 0, n * Ls, want_o=True)
        return S_full, o_full[pos]

    res = oracle.parallel_map(ref, range(len(heads)))
    wS = wo = 0.0
    for i, h in enumerate(heads):
        S_full, o_ref = res[i]
        wS = max(wS, relerr(np64(S_out[0, h]), S_full))
        wo = max(wo, relerr(np64(o[0, :, :, h]).reshape(len(pos), d), o_ref))
    print(f"long mixed: S {wS:.2e} seams {wo:.2e}")
    del pool_T, pool_S
    assert max(wS, wo) <= TOL_BF16


def test_build_32k_with_outputs_sampled_heads():
    """The 32k-token build emitting every body token's output (the cold-segment forward fused
    with pair construction): outputs of two sampled heads against the oracle run per body."""
    w = W.BUILD_32K
    tok = w.draw_request(DEV)
    bounds = w.body_bounds()
    T, S, o = hy.segment_build_batched(tok["k"], tok["v"], torch.tensor(bounds, device=DEV), tok["alpha"],
                                       tok["beta"], q=tok["q"], family=w.family, max_len=w.seg_len, want_o=True)
    assert hy.stream_status() == 0
    heads = [0, w.H - 1]
    host = host_tokens(tok, heads)
    worst = 0.0
    for i, h in enumerate(heads):
        for (b, e) in bounds[:3]:
            _, orf = ref_run(w.family, host, i, b, e, want_o=True)
            worst = max(worst, relerr(np64(o[b:e, h]), orf))
    print(f"build 32k outputs: {worst:.2e}")
    assert worst <= TOL_BF16
