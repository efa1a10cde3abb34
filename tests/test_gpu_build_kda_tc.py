"""The chunked tensor-core KDA build (d = 128, bf16 inputs, pairs only) against the oracle.

KDA (HYPIC reading notes, Method 3, Table 1): T_i = (I - b_i k_i k_i^T) diag(g_i), u_i = b_i k_i v_i^T
with a per-channel gate g_i.  The build runs the per-channel decay inside a factored Gram, the
W_k product and the update's key operand; chunks whose decay spans more than 2^100 in some channel
form L term by term instead.  Every case is checked against the float64 oracle.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import linear_attention_state_gb300 as hy
import workloads as W
from refs import TOL_BF16, host_tokens, np64, ref_pair, relerr

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_case(lens, H, key, gate_div=16.0, gap=5, ws=None):
    n = sum(lens) + gap * (len(lens) + 1)
    g = W.generator(DEV, 8200, key)
    tok = W.draw_tokens(g, n, H, 128, "kda", "bf16", DEV, gate_div=gate_div, need_q=False)
    bounds, off = [], gap
    for L_ in lens:
        bounds.append((off, off + L_))
        off += L_ + gap
    T, S = hy.segment_build_batched(tok["k"], tok["v"], torch.tensor(bounds, device=DEV), tok["alpha"],
                                    tok["beta"], family="kda", ws=ws)
    assert hy.stream_status() == 0
    return tok, bounds, T, S


def check(tok, bounds, T, S, H, heads=None):
    host = host_tokens(tok, list(range(H)))
    eT, eS = 0.0, 0.0
    for s, (b, e) in enumerate(bounds):
        for h in (heads if heads is not None else range(H)):
            Tr, Sr = ref_pair("kda", host, h, b, e)
            eT = max(eT, relerr(np64(T[s, h]).reshape(128, 128), Tr))
            if e > b:
                eS = max(eS, relerr(np64(S[s, h]), Sr))
            else:
                assert float(S[s, h].abs().max()) == 0.0
                assert torch.equal(T[s, h].reshape(128, 128).cpu(), torch.eye(128))
    return eT, eS


def test_ragged_bodies():
    lens = [0, 1, 37, 63, 64, 65, 128, 200, 1000]
    H = 3
    tok, bounds, T, S = run_case(lens, H, key=1)
    eT, eS = check(tok, bounds, T, S, H)
    print(f"kda ragged: T {eT:.2e} S {eS:.2e}")
    assert eT <= TOL_BF16 and eS <= TOL_BF16


def test_slow_decay_keeps_T_large():
    """Channel gates close to one: T_C stays far above the fp32 range over thousands of tokens
    (only the erase terms shrink it), so the T half of the chain is checked where it matters."""
    lens = [512, 3000]
    H = 2
    tok, bounds, T, S = run_case(lens, H, key=2, gate_div=1024.0)
    eT, eS = check(tok, bounds, T, S, H)
    host = host_tokens(tok, [0])
    Tr, _ = ref_pair("kda", host, 0, *bounds[1])
    assert float(np.linalg.norm(Tr)) > 1e-6
    print(f"kda slow decay: T {eT:.2e} S {eS:.2e}")
    assert eT <= TOL_BF16 and eS <= TOL_BF16


@pytest.mark.parametrize("gate_div", [2.0, 0.1])
def test_strong_decay_forms_L_term_by_term(gate_div):
    """Gates strong enough that a chunk's decay spans more than 2^100 in some channel (some chunks
    at gate_div 2, all at 0.1): those chunks take the direct form of L."""
    lens = [300, 64, 129]
    H = 2
    tok, bounds, T, S = run_case(lens, H, key=3 + int(gate_div * 10), gate_div=gate_div)
    eT, eS = check(tok, bounds, T, S, H)
    print(f"kda strong decay ({gate_div}): T {eT:.2e} S {eS:.2e}")
    assert eT <= TOL_BF16 and eS <= TOL_BF16


def test_tensor_core_path_agrees_with_recurrent_path(monkeypatch):
    lens = [300, 64, 5, 0]
    H = 2
    tok, bounds, T, S = run_case(lens, H, key=6)
    monkeypatch.setenv("HYPIC_BUILD_PATH", "recurrent")
    T2, S2 = hy.segment_build_batched(tok["k"], tok["v"], torch.tensor(bounds, device=DEV), tok["alpha"],
                                      tok["beta"], family="kda")
    assert hy.stream_status() == 0
    worst = max(relerr(np64(T[s, h]), np64(T2[s, h])) + relerr(np64(S[s, h]), np64(S2[s, h]))
                for s in range(len(lens)) for h in range(H) if bounds[s][1] > bounds[s][0])
    assert worst <= 2 * TOL_BF16, worst


def test_head_blocks_in_a_one_head_workspace():
    """A workspace that holds one head's records makes the build run head by head."""
    lens = [200, 70]
    H = 3
    ws_bytes = hy.build_workspace_bytes(1, 128, len(lens), max(lens), family="kda", in_dtype="bf16")
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV)
    tok, bounds, T, S = run_case(lens, H, key=7, ws=ws)
    eT, eS = check(tok, bounds, T, S, H)
    assert eT <= TOL_BF16 and eS <= TOL_BF16


def test_decay_family_workload_full_size_sampled_heads():
    """The KDA build of the decay-family workload (32 heads, 64 segments x 512 tokens): the bench's
    launch, sampled (segment, head) units against the oracle."""
    w = W.KDA_BUILD
    tok = w.draw_request(DEV, need_q=False)
    bounds = w.body_bounds()
    T, S = hy.segment_build_batched(tok["k"], tok["v"], torch.tensor(bounds, device=DEV), tok["alpha"],
                                    tok["beta"], family="kda", max_len=w.seg_len)
    assert hy.stream_status() == 0
    heads = [0, 13, 31]
    host = host_tokens(tok, heads)
    worst = 0.0
    for s in (0, 21, 63):
        b, e = bounds[s]
        for i, h in enumerate(heads):
            Tr, Sr = ref_pair("kda", host, i, b, e)
            worst = max(worst, relerr(np64(T[s, h]).reshape(128, 128), Tr), relerr(np64(S[s, h]), Sr))
    print(f"kda full size: {worst:.2e}")
    assert worst <= TOL_BF16
