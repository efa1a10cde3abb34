"""The allocation-free batched build.

hypic_segment_build_batched_noalloc serves callers that cannot allocate device
memory (code inside a framework that owns all device memory through its own
pool, or a process that must not allocate after start-up).  It must give the
same pairs (and, with q and o_out, the same per-token outputs) as
hypic_segment_build_batched with a caller-provided workspace, call after call,
while using only the library's own fixed scratch array, and those results must
match the oracle.

This file is named so that pytest collects it last.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

from linear_attention_state_gb300 import _lib as L
from refs import TOL_BF16, host_tokens, np64, ref_pair, ref_run, relerr

SCRATCH = 64 << 20
RECORD = 49664      # bytes per (64-token chunk, head), pairs only
RECORD_O = 66560    # with per-token outputs


@pytest.fixture(scope="module")
def lib():
    from linear_attention_state_gb300 import build
    build.build_library()
    return L.load()


def _call(lib, sh, n_seg, bounds, max_len, n_tokens, k, v, q, alpha, beta, T, S, o, stream):
    vp = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return lib.hypic_segment_build_batched_noalloc(ctypes.byref(sh), n_seg, vp(bounds), max_len, n_tokens, vp(k),
                                                   vp(v), vp(q), vp(alpha), vp(beta), vp(T), vp(S), vp(o), stream)


def test_sizes_beyond_the_scratch_are_rejected_on_the_host(lib):
    sh = L.shape(2, 128, "gated_delta", "bf16")
    p = ctypes.c_void_p(0x10000)
    chunks = SCRATCH // RECORD + 1  # one head's records no longer fit
    r = lib.hypic_segment_build_batched_noalloc(ctypes.byref(sh), 1, p, chunks * 64, chunks * 64, p, p, None, p, p,
                                                p, p, None, None)
    assert r == L.HYPIC_ENOSPACE
    r = lib.hypic_segment_build_batched_noalloc(None, 1, p, 64, 64, p, p, None, p, p, p, p, None, None)
    assert r == L.HYPIC_EINVAL


def test_outputs_limit_uses_the_larger_record(lib):
    """With q and o_out the build keeps 66,560-byte records, so fewer chunk-segments fit: a size
    between the two limits is rejected on the host, before anything is enqueued."""
    assert SCRATCH // RECORD_O == 1008 and SCRATCH // RECORD == 1351
    sh = L.shape(2, 128, "gated_delta", "bf16")
    p = ctypes.c_void_p(0x10000)
    for chunks in (1009, 1200, 1351):
        r = lib.hypic_segment_build_batched_noalloc(ctypes.byref(sh), 1, p, chunks * 64, chunks * 64, p, p, p, p, p,
                                                    p, p, p, None)
        assert r == L.HYPIC_ENOSPACE, chunks


def _tokens(dev, key, H, lens, gap, need_q, family="gated_delta"):
    import workloads as W
    n = sum(lens) + gap * (len(lens) + 1)
    g = W.generator(dev, 7100, key)
    tok = W.draw_tokens(g, n, H, 128, family, "bf16", dev, need_q=need_q,
                        gate_div=16.0 if family == "kda" else None)
    bounds, off = [], gap
    for L_ in lens:
        bounds.append((off, off + L_))
        off += L_ + gap
    return tok, bounds, n


@pytest.mark.gpu
def test_noalloc_build_matches_the_workspace_build_twice(lib):
    """40 heads of four bodies: the scratch holds the records of fewer heads, so the build runs in
    head blocks; two calls in a row against the workspace build, and one head against the oracle."""
    import linear_attention_state_gb300 as hy

    dev = "cuda"
    H, d = 40, 128
    lens = [1000, 937, 1024, 64]
    tok, bounds, n = _tokens(dev, 1, H, lens, 5, need_q=False)
    b_dev = torch.tensor(bounds, dtype=torch.int64, device=dev)
    max_len = max(lens)
    # per head: 4 bodies x 16 chunks x 49,664 B = 3.2 MB, so 40 heads take two blocks of the scratch
    assert len(lens) * ((max_len + 63) // 64) * RECORD * H > SCRATCH

    T_ref, S_ref = hy.segment_build_batched(tok["k"], tok["v"], b_dev, tok["alpha"], tok["beta"],
                                            family="gated_delta", max_len=max_len)
    assert hy.stream_status() == 0
    sh = L.shape(H, d, "gated_delta", "bf16")
    T = torch.empty((len(lens), H, d, d), device=dev)
    S = torch.empty((len(lens), H, d, d), device=dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        T.fill_(float("nan"))
        S.fill_(float("nan"))
        r = _call(lib, sh, len(lens), b_dev, max_len, n, tok["k"], tok["v"], None, tok["alpha"], tok["beta"], T, S,
                  None, stream)
        assert r == L.HYPIC_OK, (call, r)
        assert hy.stream_status() == 0
        worst = 0.0
        for s in range(len(lens)):
            for h in range(H):
                worst = max(worst, relerr(np64(T[s, h]), np64(T_ref[s, h])),
                            relerr(np64(S[s, h]), np64(S_ref[s, h])))
        assert worst <= TOL_BF16, (call, worst)
    # one head of the second call against the oracle
    h = H - 1
    host = host_tokens(tok, [h])
    for s, (b, e) in enumerate(bounds):
        Tr, Sr = ref_pair("gated_delta", host, 0, b, e)
        assert relerr(np64(T[s, h]), Tr) <= TOL_BF16 and relerr(np64(S[s, h]), Sr) <= TOL_BF16, s


@pytest.mark.gpu
def test_noalloc_split_schedule_on_the_reused_scratch_against_the_oracle(lib):
    """Few long bodies: the records leave room in the scratch for the split chain schedule (pair
    slots, publish flags, per-CTA schedule), which then runs on the never-cleared static array.  Two
    calls in a row, each against the oracle."""
    import linear_attention_state_gb300 as hy

    dev = "cuda"
    H, d = 2, 128
    lens = [2048, 1984]  # 4 units of 32 and 31 chunk steps: each unit cut into several pieces
    tok, bounds, n = _tokens(dev, 2, H, lens, 3, need_q=False)
    b_dev = torch.tensor(bounds, dtype=torch.int64, device=dev)
    max_len = max(lens)
    sh = L.shape(H, d, "gated_delta", "bf16")
    T = torch.empty((len(lens), H, d, d), device=dev)
    S = torch.empty((len(lens), H, d, d), device=dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    host = host_tokens(tok, list(range(H)))
    refs = {(s, h): ref_pair("gated_delta", host, h, b, e) for s, (b, e) in enumerate(bounds) for h in range(H)}
    for call in range(2):
        T.fill_(float("nan"))
        S.fill_(float("nan"))
        r = _call(lib, sh, len(lens), b_dev, max_len, n, tok["k"], tok["v"], None, tok["alpha"], tok["beta"], T, S,
                  None, stream)
        assert r == L.HYPIC_OK, (call, r)
        assert hy.stream_status() == 0
        worst = 0.0
        for (s, h), (Tr, Sr) in refs.items():
            worst = max(worst, relerr(np64(T[s, h]), Tr), relerr(np64(S[s, h]), Sr))
        assert np.isfinite(worst) and worst <= TOL_BF16, (call, worst)


@pytest.mark.gpu
def test_noalloc_build_with_outputs_matches_the_workspace_build_twice(lib):
    """q and o_out through the allocation-free entry: pairs and per-token outputs equal the workspace
    build's, two calls in a row, and one head's outputs match the oracle."""
    import linear_attention_state_gb300 as hy

    dev = "cuda"
    H, d = 3, 128
    lens = [700, 512, 1]
    tok, bounds, n = _tokens(dev, 3, H, lens, 9, need_q=True)
    b_dev = torch.tensor(bounds, dtype=torch.int64, device=dev)
    max_len = max(lens)
    T_ref, S_ref, o_ref = hy.segment_build_batched(tok["k"], tok["v"], b_dev, tok["alpha"], tok["beta"], q=tok["q"],
                                                   family="gated_delta", max_len=max_len, want_o=True)
    assert hy.stream_status() == 0
    sh = L.shape(H, d, "gated_delta", "bf16")
    T = torch.empty((len(lens), H, d, d), device=dev)
    S = torch.empty((len(lens), H, d, d), device=dev)
    o = torch.zeros((n, H, d), device=dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        T.fill_(float("nan"))
        S.fill_(float("nan"))
        for b, e in bounds:
            o[b:e].fill_(float("nan"))
        r = _call(lib, sh, len(lens), b_dev, max_len, n, tok["k"], tok["v"], tok["q"], tok["alpha"], tok["beta"], T,
                  S, o, stream)
        assert r == L.HYPIC_OK, (call, r)
        assert hy.stream_status() == 0
        worst = 0.0
        for s, (b, e) in enumerate(bounds):
            for h in range(H):
                worst = max(worst, relerr(np64(T[s, h]), np64(T_ref[s, h])),
                            relerr(np64(S[s, h]), np64(S_ref[s, h])),
                            relerr(np64(o[b:e, h]), np64(o_ref[b:e, h])))
        assert worst <= TOL_BF16, (call, worst)
    host = host_tokens(tok, [1])
    for b, e in bounds:
        _, o_or = ref_run("gated_delta", host, 0, b, e, want_o=True)
        assert relerr(np64(o[b:e, 1]), o_or) <= TOL_BF16


@pytest.mark.gpu
def test_noalloc_kda_build_in_head_blocks_against_the_oracle(lib):
    """The KDA family keeps its larger records (82,432 bytes per chunk and head): 16 heads of four
    bodies take two head blocks of the scratch.  Two calls in a row against the workspace build,
    and one head against the oracle."""
    import linear_attention_state_gb300 as hy

    dev = "cuda"
    H, d = 16, 128
    lens = [1000, 937, 1024, 64]
    tok, bounds, n = _tokens(dev, 4, H, lens, 5, need_q=False, family="kda")
    b_dev = torch.tensor(bounds, dtype=torch.int64, device=dev)
    max_len = max(lens)
    assert len(lens) * ((max_len + 63) // 64) * 82432 * H > SCRATCH
    T_ref, S_ref = hy.segment_build_batched(tok["k"], tok["v"], b_dev, tok["alpha"], tok["beta"], family="kda",
                                            max_len=max_len)
    assert hy.stream_status() == 0
    sh = L.shape(H, d, "kda", "bf16")
    T = torch.empty((len(lens), H, d, d), device=dev)
    S = torch.empty((len(lens), H, d, d), device=dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        T.fill_(float("nan"))
        S.fill_(float("nan"))
        r = _call(lib, sh, len(lens), b_dev, max_len, n, tok["k"], tok["v"], None, tok["alpha"], tok["beta"], T, S,
                  None, stream)
        assert r == L.HYPIC_OK, (call, r)
        assert hy.stream_status() == 0
        worst = 0.0
        for s_ in range(len(lens)):
            for h in range(H):
                worst = max(worst, relerr(np64(T[s_, h]), np64(T_ref[s_, h])),
                            relerr(np64(S[s_, h]), np64(S_ref[s_, h])))
        assert worst <= 1e-6, (call, worst)
    h = H - 1
    host = host_tokens(tok, [h])
    for s_, (b, e) in enumerate(bounds):
        Tr, Sr = ref_pair("kda", host, 0, b, e)
        assert relerr(np64(T[s_, h]), Tr) <= TOL_BF16 and relerr(np64(S[s_, h]), Sr) <= TOL_BF16, s_
