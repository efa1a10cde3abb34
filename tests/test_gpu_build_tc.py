"""GPU parity of the chunked tensor-core build (d = 128, bf16 inputs, delta families).

Bodies of ragged lengths (empty, shorter than a chunk, exact multiples, long) on
one token axis, against the float64 oracle at the bf16-path tolerance.  Extra
cases keep T_C far from underflow so the T half is really tested: DeltaNet
(a = 1) and gated delta with slow decay a = exp(-softplus(z) / 1024).
"""
from __future__ import annotations

import os

import pytest
import torch

import linear_attention_state_gb300 as hy
import workloads as W
from refs import TOL_BF16, host_tokens, np64, ref_pair, ref_run, relerr

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from linear_attention_state_gb300 import build
    build.build_library()
    hy.load()
    assert hy.stream_status() == 0


def run_case(family, lens, H, key, gate_div=None, gap=7):
    n = sum(lens) + gap * (len(lens) + 1)
    g = W.generator(DEV, 6000, key)
    tok = W.draw_tokens(g, n, H, 128, family, "bf16", DEV, gate_div=gate_div, need_q=False)
    bounds, off = [], gap
    for L_ in lens:
        bounds.append((off, off + L_))
        off += L_ + gap
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
            eT.append(relerr(np64(T[s, h]), Tr))
            if e > b:
                eS.append(relerr(np64(S[s, h]), Sr))
    return max(eT), max(eS) if eS else 0.0


@pytest.mark.parametrize("family", ["delta", "gated_delta"])
def test_ragged_bodies(family):
    lens = [0, 1, 37, 63, 64, 65, 128, 200, 1000]
    H = 3
    tok, bounds, T, S = run_case(family, lens, H, key=1 if family == "delta" else 2)
    eT, eS = check(family, tok, bounds, T, S, H)
    print(f"{family}: max rel err T {eT:.2e} S {eS:.2e}")
    assert eT <= TOL_BF16 and eS <= TOL_BF16
    for s, (b, e) in enumerate(bounds):
        if e == b:
            assert torch.equal(T[s], torch.eye(128, device=DEV).expand(H, 128, 128))
            assert float(S[s].abs().max()) == 0.0


def test_slow_decay_keeps_T_large():
    lens = [256, 512, 1024]
    H = 2
    tok, bounds, T, S = run_case("gated_delta", lens, H, key=3, gate_div=1024.0)
    eT, eS = check("gated_delta", tok, bounds, T, S, H)
    print(f"slow-decay GDN: T {eT:.2e} S {eS:.2e}, |T| {float(T.norm(dim=(-2, -1)).min()):.3e}")
    assert float(T.norm(dim=(-2, -1)).min()) > 1e-3
    assert eT <= TOL_BF16 and eS <= TOL_BF16


def test_strong_decay_takes_per_entry_exponentials():
    """Gates near 0.2 make a chunk's total decay exceed 2^-100, so the prep kernel forms every decay
    factor of L as its own exponential instead of the separable product; T_C underflows to 0
    (the tolerance floor covers it) and S must still match."""
    lens = [64, 200, 1000, 37]
    H = 2
    tok, bounds, T, S = run_case("gated_delta", lens, H, key=41, gate_div=0.5)
    a = tok["alpha"][bounds[2][0]:bounds[2][0] + 64]
    assert float(torch.log2(a).sum(0).max()) < -100.0  # the chunk really is non-separable
    eT, eS = check("gated_delta", tok, bounds, T, S, H)
    print(f"strong decay: T {eT:.2e} S {eS:.2e}")
    assert eT <= TOL_BF16 and eS <= TOL_BF16


def test_deltanet_four_segments_of_256():
    lens = [256, 256, 256, 256]
    H = 4
    tok, bounds, T, S = run_case("delta", lens, H, key=4, gap=0)
    eT, eS = check("delta", tok, bounds, T, S, H)
    print(f"DeltaNet 4 x 256: T {eT:.2e} S {eS:.2e}")
    assert eT <= TOL_BF16 and eS <= TOL_BF16


@pytest.mark.parametrize("family,gate_div", [("delta", None), ("gated_delta", 1024.0)])
def test_more_units_than_resident_ctas(family, gate_div):
    """More (segment, head) units than chain CTAs fit on the GPU at once: the chain then runs one CTA
    per SM over equal shares of all chunk steps and rejoins each segment it cuts by composing the two
    pairs.  Ragged lengths put the cuts everywhere (inside a body, on its last chunk, past its end,
    on empty bodies); a = 1 or slow decay keeps T_C large so the composed T half is really checked.
    The same build with a workspace that holds only the records runs one CTA per unit."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    H = 4
    n_seg = sms // H + 10
    special = [0, 1, 63, 64, 65, 127, 128, 129, 255, 256, 257, 511, 512]
    gen = torch.Generator().manual_seed(77)
    lens = [special[i % len(special)] if i % 3 == 0 else int(torch.randint(0, 513, (1,), generator=gen))
            for i in range(n_seg)]
    tok, bounds, T, S = run_case(family, lens, H, key=11, gate_div=gate_div)
    records = n_seg * ((max(lens) + 63) // 64) * 49664 * H
    ws = torch.empty(records, dtype=torch.uint8, device=DEV)
    T1, S1 = hy.segment_build_batched(tok["k"], tok["v"], torch.tensor(bounds, device=DEV), tok["alpha"],
                                      tok["beta"], family=family, ws=ws)
    assert hy.stream_status() == 0
    host = host_tokens(tok, list(range(H)))
    err = {"split": [0.0, 0.0], "per unit": [0.0, 0.0]}
    for s, (b, e) in enumerate(bounds):
        for h in range(H):
            Tr, Sr = ref_pair(family, host, h, b, e)
            for key, (Tg, Sg) in (("split", (T, S)), ("per unit", (T1, S1))):
                err[key][0] = max(err[key][0], relerr(np64(Tg[s, h]), Tr))
                if e > b:
                    err[key][1] = max(err[key][1], relerr(np64(Sg[s, h]), Sr))
    print(f"{family}: {n_seg} x {H} units, max rel err T/S {err}")
    for key in err:
        assert err[key][0] <= TOL_BF16 and err[key][1] <= TOL_BF16, key
    for s, (b, e) in enumerate(bounds):
        if e == b:
            assert torch.equal(T[s], torch.eye(128, device=DEV).expand(H, 128, 128))
            assert float(S[s].abs().max()) == 0.0


@pytest.mark.parametrize("family,gate_div", [("delta", None), ("gated_delta", 1024.0)])
def test_fewer_units_than_sms_cut_several_times(family, gate_div):
    """Fewer (segment, head) units than SMs: the chain spreads each unit over several CTAs in pieces
    of at least 8 chunks, and the CTA holding a unit's head composes the later pieces' published
    pairs onto it in order.  Long ragged bodies give heads with up to seven pairs to compose;
    a = 1 or slow decay keeps T_C large, so the composed T half is really checked."""
    lens = [4096, 3001, 577, 0]
    H = 2
    tok, bounds, T, S = run_case(family, lens, H, key=31, gate_div=gate_div)
    records = len(lens) * 64 * 49664 * H
    ws = torch.empty(records, dtype=torch.uint8, device=DEV)
    T1, S1 = hy.segment_build_batched(tok["k"], tok["v"], torch.tensor(bounds, device=DEV), tok["alpha"],
                                      tok["beta"], family=family, ws=ws)
    assert hy.stream_status() == 0
    host = host_tokens(tok, list(range(H)))
    eT = eS = 0.0
    for s, (b, e) in enumerate(bounds):
        for h in range(H):
            Tr, Sr = ref_pair(family, host, h, b, e)
            eT = max(eT, relerr(np64(T[s, h]), Tr))
            if e > b:
                eS = max(eS, relerr(np64(S[s, h]), Sr))
                assert relerr(np64(S[s, h]), np64(S1[s, h])) <= 1e-4
    print(f"{family} cut into pieces: max rel err T {eT:.2e} S {eS:.2e}")
    assert eT <= TOL_BF16 and eS <= TOL_BF16
    assert torch.equal(T[3], torch.eye(128, device=DEV).expand(H, 128, 128))


@pytest.mark.parametrize("family,gate_div,with_split", [("delta", None, False), ("gated_delta", 1024.0, True)])
def test_head_blocks_in_a_one_head_workspace(family, gate_div, with_split):
    """A workspace that holds one head's records (and, with_split, the split schedule's slots for
    one head's units) makes the build run over the heads one block at a time; every head is checked
    against the oracle, and the result against the build with the full preferred workspace."""
    lens = [640, 0, 64, 129, 1000]
    H = 3
    tok, bounds, T, S = run_case(family, lens, H, key=43, gate_div=gate_div)
    one_head = hy.build_workspace_bytes(1, 128, len(lens), max(lens), family=family)
    records = len(lens) * ((max(lens) + 63) // 64) * 49664
    ws_bytes = one_head if with_split else records
    assert ws_bytes >= records and ws_bytes < 2 * records
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV)
    T1, S1 = hy.segment_build_batched(tok["k"], tok["v"], torch.tensor(bounds, device=DEV), tok["alpha"],
                                      tok["beta"], family=family, ws=ws)
    assert hy.stream_status() == 0
    eT, eS = check(family, tok, bounds, T1, S1, H)
    print(f"{family} head by head: max rel err T {eT:.2e} S {eS:.2e}")
    assert eT <= TOL_BF16 and eS <= TOL_BF16
    for s, (b, e) in enumerate(bounds):
        if e > b:
            assert relerr(np64(S1[s]), np64(S[s])) <= 1e-4
        else:
            assert torch.equal(T1[s], torch.eye(128, device=DEV).expand(H, 128, 128))
            assert float(S1[s].abs().max()) == 0.0


@pytest.mark.parametrize("family,gate_div", [("delta", None), ("gated_delta", 1024.0)])
def test_one_long_body_cut_into_many_pieces(family, gate_div):
    """Two units of 32,768 tokens (512 chunks each): the split schedule cuts each into about 64
    pieces of eight chunks, and the CTA holding a unit's head composes some 63 published pairs onto
    it in order.  Over the whole body T_C decays far below one even with a = 1 or slow decay, so the
    check rests on S_{C|0}: every composed piece's T_B (512 tokens, far from underflow) multiplies
    the S of the pieces before it."""
    lens = [32768]
    H = 2
    tok, bounds, T, S = run_case(family, lens, H, key=47, gate_div=gate_div, gap=3)
    eT, eS = check(family, tok, bounds, T, S, H)
    print(f"{family} one 32k body in pieces: max rel err T {eT:.2e} S {eS:.2e}")
    assert eT <= TOL_BF16 and eS <= TOL_BF16


def test_tensor_core_path_agrees_with_recurrent_path(monkeypatch):
    lens = [300, 64, 5]
    H = 2
    tok, bounds, T, S = run_case("gated_delta", lens, H, key=5)
    monkeypatch.setenv("HYPIC_BUILD_PATH", "recurrent")
    T2, S2 = hy.segment_build_batched(tok["k"], tok["v"], torch.tensor(bounds, device=DEV), tok["alpha"],
                                      tok["beta"], family="gated_delta")
    monkeypatch.delenv("HYPIC_BUILD_PATH")
    assert hy.stream_status() == 0
    for s in range(len(lens)):
        for h in range(H):
            assert relerr(np64(S[s, h]), np64(S2[s, h])) <= TOL_BF16
            assert relerr(np64(T[s, h]), np64(T2[s, h]), tau=1e-30) <= TOL_BF16
    assert os.environ.get("HYPIC_BUILD_PATH") is None


# ---- builds that also emit per-token outputs (o_t = q_t^T S_t from the zero state) ----------

@pytest.mark.parametrize("family", ["delta", "gated_delta"])
def test_ragged_bodies_with_outputs(family):
    lens = [0, 1, 37, 63, 64, 65, 128, 200, 1000]
    H, gap = 3, 7
    n = sum(lens) + gap * (len(lens) + 1)
    g = W.generator(DEV, 6300, 1 if family == "delta" else 2)
    tok = W.draw_tokens(g, n, H, 128, family, "bf16", DEV)
    bounds, off = [], gap
    for L_ in lens:
        bounds.append((off, off + L_))
        off += L_ + gap
    T, S, o = hy.segment_build_batched(tok["k"], tok["v"], torch.tensor(bounds, device=DEV), tok["alpha"],
                                       tok["beta"], q=tok["q"], family=family, want_o=True)
    assert hy.stream_status() == 0
    host = host_tokens(tok, list(range(H)))
    eT = eS = eO = 0.0
    for s, (b, e) in enumerate(bounds):
        for h in range(H):
            Tr, Sr = ref_pair(family, host, h, b, e)
            eT = max(eT, relerr(np64(T[s, h]), Tr))
            if e > b:
                eS = max(eS, relerr(np64(S[s, h]), Sr))
                _, orf = ref_run(family, host, h, b, e, want_o=True)
                eO = max(eO, relerr(np64(o[b:e, h]), orf))
    print(f"{family} with outputs: T {eT:.2e} S {eS:.2e} o {eO:.2e}")
    assert eT <= TOL_BF16 and eS <= TOL_BF16 and eO <= TOL_BF16
    # tokens outside every body keep the zeros the binding put there
    assert float(o[:gap].abs().max()) == 0.0


def test_outputs_agree_with_recurrent_path(monkeypatch):
    lens = [300, 64, 5]
    H = 2
    n = sum(lens) + 8
    g = W.generator(DEV, 6301, 0)
    tok = W.draw_tokens(g, n, H, 128, "gated_delta", "bf16", DEV)
    bounds = torch.tensor([(0, 300), (300, 364), (364, 369)], device=DEV)
    _, _, o1 = hy.segment_build_batched(tok["k"], tok["v"], bounds, tok["alpha"], tok["beta"], q=tok["q"],
                                        family="gated_delta", want_o=True)
    monkeypatch.setenv("HYPIC_BUILD_PATH", "recurrent")
    _, _, o2 = hy.segment_build_batched(tok["k"], tok["v"], bounds, tok["alpha"], tok["beta"], q=tok["q"],
                                        family="gated_delta", want_o=True)
    monkeypatch.delenv("HYPIC_BUILD_PATH")
    assert hy.stream_status() == 0
    for h in range(H):
        assert relerr(np64(o1[:369, h]), np64(o2[:369, h])) <= TOL_BF16


def test_build_from_host_inputs_matches_device_inputs():
    """hypic_segment_build_batched_host: the bodies' rows are copied in segment groups on a second
    stream while earlier groups build; the pairs equal those of the device-input build bit for bit
    (same kernels, one CTA per unit in both) and the oracle's within the bf16-path tolerance."""
    lens = [0, 1, 63, 64, 300, 700, 129, 2, 1000, 65]
    H = 4
    tok, bounds, T, S = run_case("gated_delta", lens, H, key=21)
    host = {n: tok[n].cpu().pin_memory() for n in ("k", "v", "alpha", "beta")}
    b_host = torch.tensor(bounds, dtype=torch.int64)
    dev = tuple(torch.full_like(tok[n], float("nan")) for n in ("k", "v", "alpha", "beta")) + \
        (torch.zeros(len(lens), 2, dtype=torch.int64, device=DEV),)
    copy_stream = torch.cuda.Stream()
    for _ in range(2):  # a second call reuses the device buffers and the library's events
        T2, S2 = hy.segment_build_batched_host(host["k"], host["v"], b_host, host["alpha"], host["beta"],
                                               family="gated_delta", dev=dev, copy_stream=copy_stream)
        assert hy.stream_status() == 0
        assert torch.equal(T2, T) and torch.equal(S2, S)
    assert torch.equal(dev[4].cpu(), b_host)
    hk = host_tokens(tok, list(range(H)))
    for s in (4, 5, 8):
        for h in range(H):
            Tr, Sr = ref_pair("gated_delta", hk, h, *bounds[s])
            assert relerr(np64(T2[s, h]), Tr) <= TOL_BF16 and relerr(np64(S2[s, h]), Sr) <= TOL_BF16


@pytest.mark.parametrize("n_seg,H,seg_len", [(50, 4, 130), (2, 2, 2000)])
def test_bad_bounds_in_the_split_chain_are_reported_without_waiting(n_seg, H, seg_len):
    """One body running past the token axis, in a build whose chain cuts units between CTAs (more
    units than SMs: cut once; fewer: cut several times).  The CTAs holding that unit stop at once
    and raise their publish flags with a failure mark, so no neighbour's bounded wait has to run
    out: the call reports HYPIC_EDEVICE quickly, and the next, valid build is clean and correct."""
    import time
    n = n_seg * seg_len
    g = W.generator(DEV, 6400, n_seg)
    tok = W.draw_tokens(g, n, H, 128, "gated_delta", "bf16", DEV, need_q=False)
    good = [(i * seg_len, (i + 1) * seg_len) for i in range(n_seg)]
    bad = list(good)
    bad[n_seg // 2] = (bad[n_seg // 2][0], n + 64)  # past the token axis
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    hy.segment_build_batched(tok["k"], tok["v"], torch.tensor(bad, device=DEV), tok["alpha"], tok["beta"],
                             family="gated_delta", max_len=seg_len + 64)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert hy.stream_status() == hy._lib.HYPIC_EDEVICE
    assert dt < 0.5, f"a bounded wait seems to have run out ({dt:.2f} s)"
    T, S = hy.segment_build_batched(tok["k"], tok["v"], torch.tensor(good, device=DEV), tok["alpha"],
                                    tok["beta"], family="gated_delta")
    assert hy.stream_status() == 0
    host = host_tokens(tok, list(range(H)))
    for s_ in (0, n_seg // 2, n_seg - 1):
        Tr, Sr = ref_pair("gated_delta", host, H - 1, *good[s_])
        assert relerr(np64(S[s_, H - 1]), Sr) <= TOL_BF16
        assert relerr(np64(T[s_, H - 1]), Tr) <= TOL_BF16


def test_host_input_builds_in_a_serving_loop_with_ready_events():
    """Four different requests through hypic_segment_build_batched_host, alternating between two sets
    of device buffers: each request's copies wait only for the event recorded after the build that
    last read its set, so they overlap the previous request's build.  Every request's pairs equal
    those of the device-input build of the same tokens bit for bit."""
    lens = [300, 64, 1000, 5, 700]
    H = 4
    reqs = [run_case("gated_delta", lens, H, key=50 + r) for r in range(4)]
    n_tok = reqs[0][0]["k"].shape[0]
    sets = [tuple(torch.empty_like(reqs[0][0][n]) for n in ("k", "v", "alpha", "beta")) +
            (torch.empty(len(lens), 2, dtype=torch.int64, device=DEV),) for _ in range(2)]
    free = [torch.cuda.Event(), torch.cuda.Event()]
    copy_stream = torch.cuda.Stream()
    out = []
    for r, (tok, bounds, _, _) in enumerate(reqs):
        host = {n: tok[n].cpu().pin_memory() for n in ("k", "v", "alpha", "beta")}
        assert tok["k"].shape[0] == n_tok
        T, S = hy.segment_build_batched_host(host["k"], host["v"], torch.tensor(bounds, dtype=torch.int64),
                                             host["alpha"], host["beta"], family="gated_delta", dev=sets[r % 2],
                                             copy_stream=copy_stream, ready_event=free[r % 2] if r >= 2 else None)
        free[r % 2].record()
        out.append((T, S, host))  # keep the pinned inputs alive until the copies have run
    torch.cuda.synchronize()
    assert hy.stream_status() == 0
    for (tok, bounds, T0, S0), (T, S, _) in zip(reqs, out):
        assert torch.equal(T, T0) and torch.equal(S, S0)
