"""GPU parity of the tensor-core build for the scalar and diagonal decay families.

At d = 128 with bf16 inputs and no per-token outputs, these families build each
(segment, head) pair as one accumulating GEMM over suffix-decayed keys.  Bodies
of ragged lengths on one token axis (empty, shorter than a chunk, exact multiples,
long, and a body whose last chunk runs past the end of the token axis) are checked
against the float64 oracle at the bf16-path tolerance; slow gates keep T_C far from
underflow so the T half is really tested; and the path must agree with the
token-by-token build.
"""
from __future__ import annotations

import os

import pytest
import torch

import linear_attention_state_gb300 as hy
import workloads as W
from refs import TOL_BF16, host_tokens, np64, ref_pair, relerr, t_as_dense

pytestmark = pytest.mark.gpu
DEV = "cuda"
FAMS = ["scalar_const", "scalar", "diag"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from linear_attention_state_gb300 import build
    build.build_library()
    hy.load()
    assert hy.stream_status() == 0


def run_case(family, lens, H, key, gate_div=None, gap=7, tail_gap=True):
    n = sum(lens) + gap * (len(lens) + (1 if tail_gap else 0))
    g = W.generator(DEV, 6100, key)
    tok = W.draw_tokens(g, n, H, 128, family, "bf16", DEV, gate_div=gate_div, need_q=False)
    bounds, off = [], gap
    for L_ in lens:
        bounds.append((off, off + L_))
        off += L_ + gap
    if not tail_gap:
        assert bounds[-1][1] == n
    T, S = hy.segment_build_batched(tok["k"], tok["v"], torch.tensor(bounds, device=DEV), tok["alpha"],
                                    tok["beta"], family=family)
    assert hy.stream_status() == 0
    return tok, bounds, T, S


def check(family, tok, bounds, T, S, H):
    host = host_tokens(tok, list(range(H)))
    eT, eS = [], []
    for s, (b, e) in enumerate(bounds):
        for h in range(H):
            Tr, Sr = ref_pair(family, host, h, b, e)
            eT.append(relerr(t_as_dense(family, np64(T[s, h]), 128), t_as_dense(family, Tr, 128)))
            if e > b:
                eS.append(relerr(np64(S[s, h]), Sr))
            else:
                assert float(S[s, h].abs().max()) == 0.0
                assert torch.all(T[s, h] == 1.0)
    return max(eT), max(eS) if eS else 0.0


@pytest.mark.parametrize("family", FAMS)
def test_ragged_bodies(family):
    lens = [0, 1, 37, 63, 64, 65, 128, 200, 1000, 2053]
    H = 3
    tok, bounds, T, S = run_case(family, lens, H, key=FAMS.index(family))
    eT, eS = check(family, tok, bounds, T, S, H)
    print(f"{family}: max rel err T {eT:.2e} S {eS:.2e}")
    assert eT <= TOL_BF16 and eS <= TOL_BF16


@pytest.mark.parametrize("family", FAMS)
def test_several_units_per_cta_with_empty_and_ragged_bodies(family):
    """More units than SMs, so every CTA walks several (segment, head) units and reads each next
    unit's bounds and gates ahead of time, across empty, one-token and ragged bodies."""
    lens = [0, 1, 37, 64, 65, 130, 300]
    H = 48  # 336 units over at most 152 CTAs
    tok, bounds, T, S = run_case(family, lens, H, key=40 + FAMS.index(family))
    eT, eS = check(family, tok, bounds, T, S, H)
    print(f"{family} several units per CTA: max rel err T {eT:.2e} S {eS:.2e}")
    assert eT <= TOL_BF16 and eS <= TOL_BF16


@pytest.mark.parametrize("family", FAMS)
def test_last_chunk_runs_past_the_token_axis(family):
    # the final body ends at the last token and its length is not a multiple of 64, so the
    # tensor-map loads of its last chunk read past the axis (zero fill)
    lens = [100, 29]
    H = 2
    tok, bounds, T, S = run_case(family, lens, H, key=10 + FAMS.index(family), gap=3, tail_gap=False)
    eT, eS = check(family, tok, bounds, T, S, H)
    assert eT <= TOL_BF16 and eS <= TOL_BF16


@pytest.mark.parametrize("family", ["scalar", "diag"])
def test_slow_decay_keeps_T_large(family):
    lens = [256, 1000, 3000]
    H = 2
    tok, bounds, T, S = run_case(family, lens, H, key=20 + FAMS.index(family), gate_div=1024.0)
    eT, eS = check(family, tok, bounds, T, S, H)
    print(f"slow {family}: T {eT:.2e} S {eS:.2e}, min T {float(T.min()):.3e}")
    assert float(T.min()) > 1e-3
    assert eT <= TOL_BF16 and eS <= TOL_BF16


@pytest.mark.parametrize("family", FAMS)
def test_tensor_core_path_agrees_with_recurrent_path(family, monkeypatch):
    lens = [300, 64, 5, 0]
    H = 2
    tok, bounds, T, S = run_case(family, lens, H, key=30 + FAMS.index(family))
    monkeypatch.setenv("HYPIC_BUILD_PATH", "recurrent")
    T2, S2 = hy.segment_build_batched(tok["k"], tok["v"], torch.tensor(bounds, device=DEV), tok["alpha"],
                                      tok["beta"], family=family)
    monkeypatch.delenv("HYPIC_BUILD_PATH")
    assert hy.stream_status() == 0
    for s in range(len(lens)):
        for h in range(H):
            assert relerr(np64(S[s, h]), np64(S2[s, h])) <= TOL_BF16
            assert relerr(np64(T[s, h]), np64(T2[s, h])) <= TOL_BF16
    assert os.environ.get("HYPIC_BUILD_PATH") is None


@pytest.mark.parametrize("family", FAMS)
def test_single_segment_entry_point(family):
    H = 4
    g = W.generator(DEV, 6200, FAMS.index(family))
    tok = W.draw_tokens(g, 333, H, 128, family, "bf16", DEV, need_q=False)
    T, S = hy.segment_build(tok["k"], tok["v"], tok["alpha"], tok["beta"], family=family)
    assert hy.stream_status() == 0
    host = host_tokens(tok, list(range(H)))
    for h in range(H):
        Tr, Sr = ref_pair(family, host, h, 0, 333)
        assert relerr(t_as_dense(family, np64(T[h]), 128), t_as_dense(family, Tr, 128)) <= TOL_BF16
        assert relerr(np64(S[h]), Sr) <= TOL_BF16
