"""GB300-native linear-attention segment transition cache (HYPIC's linear-layer hot path).

The compute runs in ``libhypic.so`` (hand-written sm_103a CUDA behind the C ABI
in ``include/hypic.h``); this package is its thin ctypes binding.  There is no
CPU or PyTorch fallback: calls raise if the library is not built.
"""
from ._lib import HypicError, load  # noqa: F401
from .api import (affine_scan, assemble, build_workspace_bytes, compose, conv_seam, conv_tail,  # noqa: F401
                  pairs_to_bf16, rope_shift, seam_advance, segment_build, segment_build_batched,
                  segment_build_batched_host, state_rerotate,
                  stream_status, t_size)

__all__ = ["segment_build", "segment_build_batched", "segment_build_batched_host", "build_workspace_bytes", "compose", "affine_scan", "seam_advance",
           "assemble", "pairs_to_bf16", "rope_shift", "state_rerotate", "conv_tail", "conv_seam", "stream_status",
           "t_size", "load", "HypicError"]
