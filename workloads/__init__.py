"""Seeded synthetic inputs for the segment transition cache: shared by tests, bench and smoke.

This module holds no arithmetic of the method: it only draws random numbers
with the distributions the workloads state and rounds them to the input
precision.  Both the CUDA path and the float64 oracle consume exactly the
tensors it returns (the oracle upcasts the rounded values to float64).

Input recipe (one unit = one (config, layer, segment) draw; every unit has its
own torch.Generator so any unit can be regenerated alone):

* k, q ~ N(0, 1) per element, then each token's vector is L2-normalised in
  fp32 and rounded to the input dtype (fp32 or bf16, round-to-nearest-even);
* v ~ N(0, 1), rounded to the input dtype;
* beta = sigmoid(N(0, 1)) in fp32;
* alpha = exp(-softplus(N(0, 1)) / 8) in fp32 per token and head (scalar and
  gated-delta families), or exp(-softplus(N(0, 1)) / 16) per channel (diagonal
  family), or gamma_h = 1 - 2^(-5 - h/4) per head (constant scalar decay).

Layouts: k, q, v [tokens, H, d]; alpha [tokens, H] ([tokens, H, d] for diag,
[H] for constant decay); beta [tokens, H].  Multi-layer workloads fold the
layer axis into the head axis (head index = layer * heads + head), since
layers are independent given their inputs.

Draw order inside a unit: k, q, v, beta logits, alpha logits.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

SEED = 0


def unit_seed(*key: int) -> int:
    """Stable 63-bit seed for a unit key like (config_id, layer, segment)."""
    s = SEED
    for x in key:
        s = (s * 1000003 + int(x) + 1) % (1 << 63)
    return s


def generator(device, *key: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(unit_seed(*key))
    return g


def _dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def draw_tokens(gen: torch.Generator, n: int, H: int, d: int, family: str, in_dtype: str,
                device, gate_div: float | None = None, need_q: bool = True) -> dict:
    """Draw n tokens for H heads.  Returns k, q, v (in_dtype) and alpha, beta (fp32)."""
    dt = _dtype(in_dtype)
    f32 = torch.float32

    def unit_rows():
        x = torch.randn((n, H, d), generator=gen, device=device, dtype=f32)
        return (x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)).to(dt)

    k = unit_rows()
    q = unit_rows() if need_q else None
    v = torch.randn((n, H, d), generator=gen, device=device, dtype=f32).to(dt)
    beta = torch.sigmoid(torch.randn((n, H), generator=gen, device=device, dtype=f32))
    if family in ("diag", "kda"):
        z = torch.randn((n, H, d), generator=gen, device=device, dtype=f32)
        alpha = torch.exp(-torch.nn.functional.softplus(z) / (gate_div or 16.0))
    elif family == "scalar_const":
        alpha = const_gamma(H, device)
    else:
        z = torch.randn((n, H), generator=gen, device=device, dtype=f32)
        alpha = torch.exp(-torch.nn.functional.softplus(z) / (gate_div or 8.0))
    return {"k": k, "q": q, "v": v, "alpha": alpha.contiguous(), "beta": beta.contiguous()}


def const_gamma(H: int, device) -> torch.Tensor:
    """gamma_h = 1 - 2^(-5 - h/4), one per head, rounded to fp32."""
    h = torch.arange(H, dtype=torch.float64)
    return (1.0 - torch.pow(2.0, -5.0 - h / 4.0)).to(torch.float32).to(device)


@dataclass
class Workload:
    """A synthetic request: `layers` x `heads` heads, segments of `seg_len` tokens."""
    name: str
    cfg_id: int
    layers: int
    heads: int
    d: int
    in_dtype: str
    family: str
    n_seg: int
    seg_len: int
    w: int
    gate_div: float | None = None
    extra: dict = field(default_factory=dict)

    @property
    def H(self) -> int:
        """Flattened head count (layer-major)."""
        return self.layers * self.heads

    def body_bounds(self) -> list[tuple[int, int]]:
        """[begin, end) of each segment body on the request's token axis.

        Segment 0 (the system prompt) has no seam; every inner segment's first
        w tokens are its seam window and the cached pair covers the rest.
        """
        out = []
        for j in range(self.n_seg):
            b = j * self.seg_len
            e = b + self.seg_len
            out.append((b if j == 0 else min(b + self.w, e), e))
        return out

    def seam_positions(self) -> list[int]:
        """Global token positions of all seam tokens, segment by segment."""
        pos = []
        for j in range(1, self.n_seg):
            pos.extend(range(j * self.seg_len, j * self.seg_len + min(self.w, self.seg_len)))
        return pos

    def draw_segment(self, seg: int, device, heads: list[int] | None = None, need_q: bool = True) -> dict:
        """All tokens of one segment for all layers (or the listed flat heads)."""
        parts = []
        layers = range(self.layers) if heads is None else sorted({h // self.heads for h in heads})
        for layer in layers:
            g = generator(device, self.cfg_id, layer, seg)
            parts.append(draw_tokens(g, self.seg_len, self.heads, self.d, self.family, self.in_dtype,
                                     device, self.gate_div, need_q=need_q))
        out = {}
        for key in ("k", "q", "v", "alpha", "beta"):
            if parts[0][key] is None:
                out[key] = None
                continue
            if key == "alpha" and self.family == "scalar_const":
                out[key] = torch.cat([p[key] for p in parts], dim=0)
            else:
                out[key] = torch.cat([p[key] for p in parts], dim=1)
        if heads is not None:
            pos = {layer: i for i, layer in enumerate(layers)}
            sel = [pos[h // self.heads] * self.heads + h % self.heads for h in heads]
            for key in out:
                if out[key] is None:
                    continue
                if key == "alpha" and self.family == "scalar_const":
                    out[key] = out[key][sel]
                else:
                    out[key] = out[key][:, sel]
        return out

    def draw_request(self, device, need_q: bool = True) -> dict:
        """The whole request's tokens, segments concatenated on the token axis."""
        segs = [self.draw_segment(j, device, need_q=need_q) for j in range(self.n_seg)]
        out = {}
        for key in ("k", "q", "v", "beta"):
            out[key] = None if segs[0][key] is None else torch.cat([s[key] for s in segs], dim=0)
        if self.family == "scalar_const":
            out["alpha"] = segs[0]["alpha"]
        else:
            out["alpha"] = torch.cat([s["alpha"] for s in segs], dim=0)
        return out


# The five workloads.  Sizes follow the pages' workloads: segments of 256-4096
# tokens, 8-segment 32k requests, 30 linear layers of 32 heads at d = 128.
TINY = Workload("tiny_f32_2h_d16_4x64", 0, 1, 2, 16, "f32", "gated_delta", 4, 64, 4)
BUILD_32K = Workload("build_32h_d128_8x4096", 1, 1, 32, 128, "bf16", "gated_delta", 8, 4096, 8)
DECAY_FAMILIES = {
    "scalar_const": Workload("decay_scalar_32h_d128_64x512", 3, 1, 32, 128, "bf16", "scalar_const", 64, 512, 0),
    "diag": Workload("decay_diag_32h_d128_64x512", 3, 1, 32, 128, "bf16", "diag", 64, 512, 0, gate_div=16.0),
    "gated_delta": Workload("decay_gdn_32h_d128_64x512", 3, 1, 32, 128, "bf16", "gated_delta", 64, 512, 0),
}
# KDA (per-channel gate before the erase) on the decay-family shape, channel gates as the diagonal family's.
KDA_BUILD = Workload("decay_kda_32h_d128_64x512", 3, 1, 32, 128, "bf16", "kda", 64, 512, 0, gate_div=16.0)
LONG_MIXED = Workload("long_30x32_d128_128x1024", 4, 30, 32, 128, "bf16", "gated_delta", 128, 1024, 8,
                      extra={"n_cold": 32})


@dataclass
class PoolWorkload:
    """Warm-cache composition: B requests, each composes n distinct pool entries."""
    name: str
    cfg_id: int
    layers: int
    heads: int
    d: int
    pool: int
    B: int
    n: int
    pair_tokens: int

    @property
    def H(self) -> int:
        return self.layers * self.heads

    def request_indices(self, device="cpu") -> torch.Tensor:
        """[B, n] int32: each request draws n distinct pool ids in random order."""
        g = generator("cpu", self.cfg_id, 99991)
        rows = [torch.randperm(self.pool, generator=g)[: self.n] for _ in range(self.B)]
        return torch.stack(rows).to(torch.int32).to(device)

    def pair_inputs(self, p: int, device, heads: list[int] | None = None) -> dict:
        """The 1024 gated-delta tokens (config-0 distributions, bf16) pool entry p is built from."""
        w = Workload(self.name, self.cfg_id, self.layers, self.heads, self.d, "bf16", "gated_delta",
                     self.pool, self.pair_tokens, 0)
        return w.draw_segment(p, device, heads=heads, need_q=False)


COMPOSE_POOL = PoolWorkload("compose_30x32_d128_pool256_B64x16", 2, 30, 32, 128, 256, 64, 16, 1024)


def long_mixed_cold(w: Workload = LONG_MIXED) -> list[int]:
    """The seeded choice of cold segments (built in the step); the rest arrive cached."""
    g = generator("cpu", w.cfg_id, 77777)
    return sorted(torch.randperm(w.n_seg, generator=g)[: w.extra.get("n_cold", 32)].tolist())


def random_pairs(P: int, H: int, d: int, device, key: int = 0, t_scale: float = 0.5) -> tuple:
    """Random fp32 affine pairs: T entries N(0, (t_scale^2)/d), S entries N(0, 1).

    Used where a test needs compose inputs that do not come from a build.
    """
    g = generator(device, 424242, key)
    T = torch.randn((P, H, d, d), generator=g, device=device) * (t_scale / d ** 0.5)
    S = torch.randn((P, H, d, d), generator=g, device=device)
    return T.contiguous(), S.contiguous()
