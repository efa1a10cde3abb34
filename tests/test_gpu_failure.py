"""Failure detection without a GPU fault.

Every wait in the tensor-core kernels is bounded by a cycle limit; when a wait runs
out, the kernel records HYPIC_ETIMEOUT in the per-device status word and returns.
Here a wait that nothing can satisfy (an mbarrier no one arrives at) runs out on
purpose, the host reads the status, and the device keeps working afterwards.
Device-side index and bound checks report the same way (HYPIC_EDEVICE).
"""
from __future__ import annotations

import ctypes

import pytest
import torch

import linear_attention_state_gb300 as hy
from linear_attention_state_gb300 import _lib as L

DEV = "cuda"


@pytest.fixture(scope="module")
def lib():
    from linear_attention_state_gb300 import build
    build.build_library()
    return L.load()


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def test_selftest_rejects_bad_limits_on_the_host(lib):
    assert lib.hypic_selftest_bounded_wait(-1, None) == L.HYPIC_EINVAL
    assert lib.hypic_selftest_bounded_wait(5_000_000_000, None) == L.HYPIC_EINVAL


@pytest.mark.gpu
def test_unsatisfiable_wait_times_out_and_is_reported(lib):
    assert hy.stream_status() == 0
    assert lib.hypic_selftest_bounded_wait(1_000_000, _stream()) == L.HYPIC_OK
    assert hy.stream_status() == L.HYPIC_ETIMEOUT
    assert hy.stream_status() == 0  # read and cleared
    # the context is still usable: a normal composition right after runs and is correct
    d, H = 16, 2
    T = torch.eye(d, device=DEV).expand(3, H, d, d).contiguous()
    S = torch.ones((3, H, d, d), device=DEV)
    out = hy.compose(T, S, torch.tensor([[0, 1, 2]], dtype=torch.int32, device=DEV), family="gated_delta")
    assert hy.stream_status() == 0
    assert torch.allclose(out, torch.full_like(out, 3.0))


@pytest.mark.gpu
def test_first_error_wins_until_read(lib):
    d, H = 128, 2
    T = torch.zeros((2, H, d, d), device=DEV)
    S = torch.zeros((2, H, d, d), device=DEV)
    hy.compose(T, S, torch.tensor([[0, 5]], dtype=torch.int32, device=DEV), family="gated_delta")  # bad index
    lib.hypic_selftest_bounded_wait(100_000, _stream())
    assert hy.stream_status() == L.HYPIC_EDEVICE  # the first recorded error is kept
    assert hy.stream_status() == 0
