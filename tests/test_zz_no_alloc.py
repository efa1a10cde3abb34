"""The allocation-free batched build.

hypic_segment_build_batched_noalloc serves callers that cannot allocate device
memory (code inside a framework that owns all device memory through its own
pool, or a process that must not allocate after start-up).  It must give the
same pairs as hypic_segment_build_batched with a caller-provided workspace,
call after call, while using only the library's own fixed scratch array.

This file is named so that pytest collects it last.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

from linear_attention_state_gb300 import _lib as L
from refs import TOL_BF16, np64, relerr

SCRATCH = 64 << 20
RECORD = 49664


@pytest.fixture(scope="module")
def lib():
    from linear_attention_state_gb300 import build
    build.build_library()
    return L.load()


def test_sizes_beyond_the_scratch_are_rejected_on_the_host(lib):
    sh = L.shape(2, 128, "gated_delta", "bf16")
    p = ctypes.c_void_p(0x10000)
    chunks = SCRATCH // RECORD + 1  # one head's records no longer fit
    r = lib.hypic_segment_build_batched_noalloc(ctypes.byref(sh), 1, p, chunks * 64, chunks * 64, p, p, None, p, p,
                                                p, p, None, None)
    assert r == L.HYPIC_ENOSPACE
    r = lib.hypic_segment_build_batched_noalloc(None, 1, p, 64, 64, p, p, None, p, p, p, p, None, None)
    assert r == L.HYPIC_EINVAL


@pytest.mark.gpu
def test_noalloc_build_matches_the_workspace_build_twice(lib):
    import linear_attention_state_gb300 as hy
    import workloads as W

    dev = "cuda"
    H, d = 40, 128
    lens = [1000, 937, 1024, 64]
    gap = 5
    n = sum(lens) + gap * (len(lens) + 1)
    g = W.generator(dev, 7100, 1)
    tok = W.draw_tokens(g, n, H, d, "gated_delta", "bf16", dev, need_q=False)
    bounds, off = [], gap
    for L_ in lens:
        bounds.append((off, off + L_))
        off += L_ + gap
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
        r = lib.hypic_segment_build_batched_noalloc(
            ctypes.byref(sh), len(lens), ctypes.c_void_p(b_dev.data_ptr()), max_len, n,
            ctypes.c_void_p(tok["k"].data_ptr()), ctypes.c_void_p(tok["v"].data_ptr()), None,
            ctypes.c_void_p(tok["alpha"].data_ptr()), ctypes.c_void_p(tok["beta"].data_ptr()),
            ctypes.c_void_p(T.data_ptr()), ctypes.c_void_p(S.data_ptr()), None, stream)
        assert r == L.HYPIC_OK, (call, r)
        assert hy.stream_status() == 0
        worst = 0.0
        for s in range(len(lens)):
            for h in range(H):
                worst = max(worst, relerr(np64(T[s, h]), np64(T_ref[s, h])),
                            relerr(np64(S[s, h]), np64(S_ref[s, h])))
        assert worst <= TOL_BF16, (call, worst)
