"""C-ABI checks that need no GPU: the library loads, exports what the header declares,
and rejects bad arguments on the host before anything reaches CUDA.

Only calls that fail host validation, empty no-op batches and pure-host queries
are made here; none of them touches the CUDA runtime's device API.
"""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from linear_attention_state_gb300 import _lib as L
from linear_attention_state_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hypic.h")


@pytest.fixture(scope="module")
def lib():
    B.build_library()
    return L.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(hypic_[a-z_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("hypic_segment_build", "hypic_segment_build_batched", "hypic_compose", "hypic_affine_scan",
                     "hypic_seam_advance", "hypic_assemble", "hypic_stream_status", "hypic_strerror"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/hypic.h but not exported"
        assert name in L.SIGNATURES, f"{name} has no ctypes signature in the binding"


def test_exports_are_plain_c(lib):
    out = os.popen(f"nm -D --defined-only {L.LIB_PATH}").read()
    exported = set(re.findall(r" T (hypic_\w+)", out))
    assert set(declared_functions()) <= exported


def test_host_queries(lib):
    assert lib.hypic_abi_version() == 1
    for fam, want in (("scalar_const", 1), ("scalar", 1), ("diag", 128), ("delta", 128 * 128),
                      ("gated_delta", 128 * 128)):
        sh = L.shape(4, 128, fam, "bf16")
        assert lib.hypic_t_size(ctypes.byref(sh)) == want
    bad = L.Shape(4, 128, 64, 4, 1)
    assert lib.hypic_t_size(ctypes.byref(bad)) == 0
    for st in (0, -1, -2, -3, -4, -5, -6):
        assert lib.hypic_strerror(st)
    assert lib.hypic_strerror(-99) == b"unknown status"


def _fake(addr=0x10000):
    return ctypes.c_void_p(addr)


def test_shape_validation(lib):
    S = _fake()
    cases = [
        (L.Shape(-1, 128, 128, 4, 1), L.HYPIC_EINVAL),
        (L.Shape(4, 0, 0, 4, 1), L.HYPIC_EINVAL),
        (L.Shape(4, 128, 128, 9, 1), L.HYPIC_EINVAL),
        (L.Shape(4, 128, 128, 4, 7), L.HYPIC_EINVAL),
        (L.Shape(4, 128, 64, 4, 1), L.HYPIC_EUNSUPPORTED),
        (L.Shape(4, 96, 96, 4, 1), L.HYPIC_EUNSUPPORTED),
    ]
    for sh, want in cases:
        r = lib.hypic_compose(ctypes.byref(sh), 1, 1, S, 1, S, S, None, S, None)
        assert r == want, (sh.H, sh.d_k, sh.d_v, sh.family, sh.in_dtype, r)
    assert lib.hypic_compose(None, 1, 1, S, 1, S, S, None, S, None) == L.HYPIC_EINVAL


def test_pointer_validation(lib):
    sh = L.shape(4, 128, "gated_delta", "bf16")
    p = _fake()
    mis = _fake(0x10004)  # not 16-byte aligned
    # build: missing k, misaligned v, missing beta for a delta family, o without q
    assert lib.hypic_segment_build(ctypes.byref(sh), None, p, None, p, p, 8, p, p, None, None, 0, None) == L.HYPIC_EINVAL
    assert lib.hypic_segment_build(ctypes.byref(sh), p, mis, None, p, p, 8, p, p, None, None, 0, None) == L.HYPIC_EINVAL
    assert lib.hypic_segment_build(ctypes.byref(sh), p, p, None, p, None, 8, p, p, None, None, 0, None) == L.HYPIC_EINVAL
    assert lib.hypic_segment_build(ctypes.byref(sh), p, p, None, p, p, 8, p, p, p, None, 0, None) == L.HYPIC_EINVAL
    assert lib.hypic_segment_build(ctypes.byref(sh), p, p, None, p, p, -1, p, p, None, None, 0, None) == L.HYPIC_EINVAL
    # batched: negative counts, missing bounds
    assert lib.hypic_segment_build_batched(ctypes.byref(sh), -1, p, 8, 8, p, p, None, p, p, p, p, None, None, 0,
                                           None) == L.HYPIC_EINVAL
    assert lib.hypic_segment_build_batched(ctypes.byref(sh), 2, None, 8, 8, p, p, None, p, p, p, p, None, None, 0,
                                           None) == L.HYPIC_EINVAL
    # compose: missing idx with n > 0, empty pool
    assert lib.hypic_compose(ctypes.byref(sh), 1, 2, None, 4, p, p, None, p, None) == L.HYPIC_EINVAL
    assert lib.hypic_compose(ctypes.byref(sh), 1, 2, p, 0, p, p, None, p, None) == L.HYPIC_EINVAL
    assert lib.hypic_compose(ctypes.byref(sh), 1, 2, p, 4, p, p, mis, p, None) == L.HYPIC_EINVAL
    # assemble: seams without seam tokens
    assert lib.hypic_assemble(ctypes.byref(sh), 1, 3, 8, p, 4, p, p, None, None, None, None, None, None, p, None,
                              None) == L.HYPIC_EINVAL
    # seam advance: missing v
    assert lib.hypic_seam_advance(ctypes.byref(sh), 1, p, None, p, None, p, p, 8, None, None) == L.HYPIC_EINVAL
    # scan: missing S
    assert lib.hypic_affine_scan(ctypes.byref(sh), 3, p, None, p, p, None, 0, None) == L.HYPIC_EINVAL


def test_gate_requirements_by_family(lib):
    p = _fake()
    # delta needs no alpha; scalar families need no beta
    sh = L.shape(2, 16, "delta", "f32")
    assert lib.hypic_segment_build(ctypes.byref(sh), p, p, None, None, None, 8, p, p, None, None, 0,
                                   None) == L.HYPIC_EINVAL  # beta still required
    sh = L.shape(2, 16, "scalar", "f32")
    assert lib.hypic_segment_build(ctypes.byref(sh), p, p, None, None, None, 8, p, p, None, None, 0,
                                   None) == L.HYPIC_EINVAL  # alpha required


def test_empty_batches_are_noops(lib):
    sh = L.shape(4, 128, "gated_delta", "bf16")
    sh0 = L.shape(0, 128, "gated_delta", "bf16")
    assert lib.hypic_compose(ctypes.byref(sh), 0, 4, None, 0, None, None, None, None, None) == L.HYPIC_OK
    assert lib.hypic_compose(ctypes.byref(sh0), 3, 4, None, 0, None, None, None, None, None) == L.HYPIC_OK
    assert lib.hypic_segment_build_batched(ctypes.byref(sh), 0, None, 0, 0, None, None, None, None, None, None, None,
                                           None, None, 0, None) == L.HYPIC_OK
    assert lib.hypic_seam_advance(ctypes.byref(sh), 0, None, None, None, None, None, None, 8, None,
                                  None) == L.HYPIC_OK
    assert lib.hypic_affine_scan(ctypes.byref(sh), 0, None, None, None, None, None, 0, None) == L.HYPIC_OK
    assert lib.hypic_assemble(ctypes.byref(sh), 0, 4, 8, None, 0, None, None, None, None, None, None, None, None,
                              None, None, None) == L.HYPIC_OK


def test_workspace_queries_are_host_only(lib):
    sh = L.shape(32, 128, "gated_delta", "bf16")
    a = lib.hypic_build_workspace_bytes(ctypes.byref(sh), 8, 4096)
    b = lib.hypic_build_workspace_bytes(ctypes.byref(sh), 16, 4096)
    assert b >= a >= 0
    assert lib.hypic_scan_workspace_bytes(ctypes.byref(sh), 16) >= 0


def test_binding_refuses_cpu_tensors():
    import torch

    import linear_attention_state_gb300 as hy
    k = torch.zeros(4, 2, 16)
    with pytest.raises(ValueError, match="CUDA"):
        hy.segment_build(k, k, torch.zeros(4, 2), torch.zeros(4, 2))


def test_build_workspace_contract(lib):
    sh = L.shape(32, 128, "gated_delta", "bf16")
    per_head = 8 * 64 * 49664
    # the records of all heads, then pair slots for the chain (up to 256 CTAs), flags and schedule
    split = min(8 * 32, 256) * 2 * 128 * 128 * 4 + 3 * 256 * 4
    assert lib.hypic_build_workspace_bytes(ctypes.byref(sh), 8, 4096) == 32 * per_head + split
    # shapes that run without a workspace
    for fam, dt in (("scalar", "bf16"), ("gated_delta", "f32")):
        s2 = L.shape(32, 128, fam, dt)
        assert lib.hypic_build_workspace_bytes(ctypes.byref(s2), 8, 4096) == 0
    # less than one head's records: rejected on the host before any launch
    p = _fake()
    r = lib.hypic_segment_build(ctypes.byref(sh), p, p, None, p, p, 4096, p, p, None, p, per_head // 8 - 16,
                                None)
    assert r == L.HYPIC_ENOSPACE
    r = lib.hypic_segment_build(ctypes.byref(sh), p, p, None, p, p, 4096, p, p, None, None, 0, None)
    assert r == L.HYPIC_ENOSPACE


def test_host_input_build_checks_bounds_on_the_host(lib):
    sh = L.shape(4, 128, "gated_delta", "bf16")
    p = _fake()
    bounds = (ctypes.c_int64 * 4)(0, 10, 10, 30)
    args = [p] * 4 + [p] * 5 + [p, p, p, 1 << 20, None, None, None]
    # a body past the token axis, and one longer than max_len: rejected before anything runs
    assert lib.hypic_segment_build_batched_host(ctypes.byref(sh), 2, bounds, 64, 20, *args) == L.HYPIC_EINVAL
    assert lib.hypic_segment_build_batched_host(ctypes.byref(sh), 2, bounds, 16, 30, *args) == L.HYPIC_EINVAL
    assert lib.hypic_segment_build_batched_host(ctypes.byref(sh), 2, None, 64, 30, *args) == L.HYPIC_EINVAL
    assert lib.hypic_segment_build_batched_host(ctypes.byref(sh), 0, None, 0, 0, *args) == L.HYPIC_OK


def test_bf16_pair_storage_validation(lib):
    p = _fake()
    mis = _fake(0x10004)
    # the delta families take bf16 pools on the d = 128 tensor-core chain only: rejected on the host
    sh64 = L.shape(2, 64, "gated_delta", "f32")
    assert lib.hypic_compose_bf16(ctypes.byref(sh64), 1, 2, p, 4, p, p, None, p, None) == L.HYPIC_EUNSUPPORTED
    assert lib.hypic_assemble_bf16(ctypes.byref(sh64), 1, 2, 0, p, 4, p, p, None, None, None, None, None, None, p,
                                   None, None) == L.HYPIC_EUNSUPPORTED
    sh = L.shape(2, 128, "gated_delta", "f32")
    assert lib.hypic_compose_bf16(ctypes.byref(sh), 1, 2, None, 4, p, p, None, p, None) == L.HYPIC_EINVAL
    assert lib.hypic_compose_bf16(ctypes.byref(sh), 0, 2, None, 0, None, None, None, None, None) == L.HYPIC_OK
    # conversion: negative count, misaligned or missing pointers; zero pairs is a no-op
    assert lib.hypic_pairs_to_bf16(ctypes.byref(sh), -1, p, p, p, p, None) == L.HYPIC_EINVAL
    assert lib.hypic_pairs_to_bf16(ctypes.byref(sh), 3, p, mis, p, p, None) == L.HYPIC_EINVAL
    assert lib.hypic_pairs_to_bf16(ctypes.byref(sh), 3, p, p, None, p, None) == L.HYPIC_EINVAL
    assert lib.hypic_pairs_to_bf16(ctypes.byref(sh), 0, None, None, None, None, None) == L.HYPIC_OK
