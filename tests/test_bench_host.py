"""Host logic of bench.py that needs no GPU: the parity check of the bench line."""
from __future__ import annotations

import types

import numpy as np
import pytest
import torch

import bench


def _fake_request(n_seg=3, H=2, d=4, w=2, seed=0):
    """A request's output buffers (as the timed loop leaves them) and matching oracle results."""
    g = np.random.default_rng(seed)
    T = g.standard_normal((n_seg, H, d, d))
    S = g.standard_normal((n_seg, H, d, d))
    So = g.standard_normal((1, H, d, d))
    o = g.standard_normal((1, n_seg - 1, w, H, d))
    req = types.SimpleNamespace(T=torch.tensor(T, dtype=torch.float32), S=torch.tensor(S, dtype=torch.float32),
                                S_out=torch.tensor(So, dtype=torch.float32), o=torch.tensor(o, dtype=torch.float32))
    wl = types.SimpleNamespace(n_seg=n_seg)
    # the references are the float32 buffers' own values, so the errors are exactly zero
    ref = {h: ([req.T[j, h].double().numpy().reshape(-1) for j in range(n_seg)],
               [req.S[j, h].double().numpy() for j in range(n_seg)],
               [req.o[0, j, :, h].double().numpy() for j in range(n_seg - 1)],
               req.S_out[0, h].double().numpy()) for h in range(H)}
    return req, wl, ref


def test_parity_of_identical_buffers_is_zero():
    req, wl, ref = _fake_request()
    p = bench.request_parity(req, wl, ref, 2e-3)
    assert p["ok"] and p["heads"] == 2
    assert all(e == 0.0 for e in p["max_rel_err"].values())


@pytest.mark.parametrize("which", ["T", "S", "o", "S_out"])
def test_parity_catches_a_planted_error_in_each_quantity(which):
    req, wl, ref = _fake_request()
    buf = getattr(req, which)
    flat = buf.view(-1)
    flat[flat.numel() // 2] += 10.0  # one entry of one unit far off
    p = bench.request_parity(req, wl, ref, 2e-3)
    assert not p["ok"]
    key = {"T": "T_C", "S": "S", "o": "seam_o", "S_out": "composed_S"}[which]
    assert p["max_rel_err"][key] > 2e-3
    assert all(v == 0.0 for k, v in p["max_rel_err"].items() if k != key)


def test_parity_floor_keeps_underflowed_transitions_quiet():
    """A T_C that underflowed to zero on the GPU against a float64 value far below the 1e-30 floor
    counts as agreement (the measure's floor), not as a relative error of one."""
    req, wl, ref = _fake_request()
    req.T.zero_()
    tiny = {h: ([np.full(16, 1e-154) for _ in range(3)], Ss, os_, Sf) for h, (_, Ss, os_, Sf) in ref.items()}
    p = bench.request_parity(req, wl, tiny, 2e-3)
    assert p["max_rel_err"]["T_C"] < 1e-100 and p["ok"]


def test_traffic_is_reported_only_for_the_sources_it_was_captured_on(monkeypatch):
    """A captured DRAM figure carries the digest of its kernel sources; once they change, the line
    reports null instead of a stale number."""
    entry = {"bytes": 123, "src": ("build_tc.cu",), "digest": bench.src_digest(("build_tc.cu",)), "commit": "x"}
    monkeypatch.setitem(bench.TRAFFIC, "build_tc", entry)
    assert bench.traffic("build_tc") == 123
    monkeypatch.setitem(bench.TRAFFIC, "build_tc", dict(entry, digest="000000000000"))
    assert bench.traffic("build_tc") is None
    monkeypatch.setitem(bench.TRAFFIC, "build_tc", dict(entry, bytes=None))
    assert bench.traffic("build_tc") is None


def test_traffic_digest_covers_code_not_comments():
    """Comment and layout edits leave a source's code, and so its captured traffic, in force; a change
    to the code (a string literal included) does not."""
    base = 'asm volatile("tcgen05.commit; // not a comment");\nint x = a + b;  // sum\n'
    same = '/* the sum */ asm volatile("tcgen05.commit; // not a comment");\n\n  int x  =  a + b;\n'
    assert bench.code_text(base) == bench.code_text(same)
    assert bench.code_text(base) != bench.code_text(base.replace("a + b", "a - b"))
    assert bench.code_text(base) != bench.code_text(base.replace("// not a comment", "// changed"))


def test_summary_is_compact_and_tolerates_missing_legs():
    import json
    line = {"value": 45977012.07, "e2e": {"value": 11924399.0}, "build": {"ms": 0.70312},
            "roofline": {"frac": 0.13812345}, "assemble": {"ms": 0.105},
            "compose_pool": {"compositions_per_s": 3.6e7, "roofline": {"frac": 0.718, "dram_frac": 0.25},
                             "bf16_pool": {"compositions_per_s": 6.3e7, "roofline": {"frac": 0.65, "dram_frac": None}}},
            "decay_builds": {"scalar_const": {"roofline": {"frac": 0.703}}}, "affine_scan": None,
            "build_with_outputs": None, "long_mixed": None, "parity": {"ok": True}, "parity_t_path": None}
    s = bench.summary(line)
    assert s["build_tensor_frac"] == 0.138 and s["compose_f32"]["dram_frac"] == 0.25
    assert s["scan_hbm_frac"] is None and s["long_mixed"]["tok_per_s"] is None
    assert s["parity_ok"] == {"request": True, "t_path": None, "long_mixed": None}
    assert len(json.dumps(s)) < 900


def test_both_arms_print_the_same_config():
    import workloads as W
    assert bench.bench_config(W.BUILD_32K, 1) == bench.bench_config(W.BUILD_32K, 1)
    src = open(bench.__file__).read()
    assert src.count('"config": bench_config(w, world)') == 2
