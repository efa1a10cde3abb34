"""Benchmark of the segment transition cache hot path on GB300.

One step = the whole hot path over one synthetic request: build the
(T_C, S_{C|0}) pair of every segment body, then the fused request assembly
(seam advance through the first w tokens of each inner segment, emitting their
outputs, and composition S <- T_C S + S_{C|0} in prompt order).

Default workload: 1 layer x 32 heads, d_k = d_v = 128, bf16 q/k/v, fp32 gates
and state, 8 segments x 4096 tokens (32k), w = 8, composed from a zero state.
A second measurement times warm-cache composition alone: 30 layers x 32 heads,
a pool of 256 fp32 pairs per head, 64 requests x 16 segments.

Prints ONE JSON line (rank 0).  Under torchrun each rank runs its own
independent request (weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import functools
import json
import os
import re
import statistics
import subprocess
import sys
import time
import types

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "segment tokens/s (build) and compositions/s, % tensor/HBM roofline, 1 GB300"

# Algorithmic work per unit: the FLOP and bytes a direct implementation of each step needs.
D = 128
FLOP_PER_CHUNK_WY = 3 * 2 * 64 * 64 * D + 2 * 2 * 64 * D * (2 * D)  # G, U, W; W.X and K^T.R per 64-token chunk
FLOP_PER_HEAD_TOKEN_WY = FLOP_PER_CHUNK_WY // 64                    # 180,224
# with per-token outputs: + Q S_p (2 C d^2), Q K^T and M Wm (2 C^2 d each) per chunk
FLOP_PER_HEAD_TOKEN_WY_O = (FLOP_PER_CHUNK_WY + 2 * 64 * D * D + 4 * 64 * 64 * D) // 64  # 245,760
FLOP_PER_HEAD_TOKEN_RECURRENT = 4 * D * (2 * D)                      # k.x and rank-1 update on [T|S]
FLOP_PER_HEAD_TOKEN_KDA_RECURRENT = FLOP_PER_HEAD_TOKEN_RECURRENT + D * (2 * D)  # + the channel gate
BYTES_PER_COMPOSITION = 2 * D * D * 4                                # T_C and S_{C|0}, fp32

# Captured DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch, from the ncu
# captures summarised under profiles/.  Each entry carries the digest of the kernel code it was
# captured on (sha1 of the listed csrc files without comments and with whitespace runs made one
# space, first 12 hex digits) and the commit of the capture; the bench reports a figure only while
# that code is unchanged, and null once it differs.
TRAFFIC = {
    # wy_prep_kernel + chain_tc_kernel, one build of the 8 x 4096-token, 32-head request (--build-only)
    "build_tc": {"bytes": 2_428_619_264, "src": ("build_tc.cu", "tc_ptx.cuh"), "digest": "f58ecee7ded7",
                 "commit": "3dd9139"},
    # wy_prep_kernel<1> + T-half chain_tc_kernel + chain_so_kernel, same request with outputs
    "build_outputs_tc": {"bytes": 5_338_161_835, "src": ("build_tc.cu", "tc_ptx.cuh"), "digest": "f58ecee7ded7",
                         "commit": "3dd9139"},
    # build_decay_tc_kernel, 64 x 512-token, 32-head decay workloads (--decay-only)
    "decay_scalar_const": {"bytes": 645_570_645, "src": ("build_decay_tc.cu", "tc_ptx.cuh"),
                           "digest": "75f0a1f85a8e", "commit": "1b1b1f2"},
    "decay_diag": {"bytes": 1_193_678_251, "src": ("build_decay_tc.cu", "tc_ptx.cuh"), "digest": "75f0a1f85a8e",
                   "commit": "1b1b1f2"},
    # wy_prep_kernel + chain_tc_kernel on the decay-family shape (--decay-only, plain gated delta)
    "decay_gated_delta": {"bytes": 2_676_390_229, "src": ("build_tc.cu", "tc_ptx.cuh"), "digest": "f58ecee7ded7",
                          "commit": "3dd9139"},
    # kda_prep_kernel + chain_kda_kernel on the decay-family shape (--decay-only)
    "decay_kda": {"bytes": 3_970_410_325, "src": ("build_kda_tc.cu", "tc_ptx.cuh"), "digest": "1ede637113ef",
                  "commit": "6d2df0b"},
    # compose_pipe32_kernel / compose_pipe_kernel (the kernels composition without seam windows runs)
    # on the warm-cache workload (fp32 and bf16 pools):
    # captured at 4 layers (128 heads, --compose-layers 4) and scaled by 7.5 to 960 heads (each
    # head's pool entries and requests are independent, the grid head-major)
    "compose_f32": {"bytes": 46_755_327_360, "src": ("compose_pipe.cu", "tc_ptx.cuh"),
                    "digest": "b2832f896031", "commit": "ae10944"},
    "compose_bf16": {"bytes": 19_951_943_680, "src": ("compose_pipe.cu", "tc_ptx.cuh"),
                     "digest": "b2832f896031", "commit": "ae10944"},
    # compose_pipe32_kernel in scan mode, 64 pairs: captured at 128 heads (--scan-heads 128) and
    # scaled by 7.5 to 960 heads
    "scan": {"bytes": 15_826_974_720, "src": ("compose_pipe.cu", "tc_ptx.cuh"), "digest": "b2832f896031",
             "commit": "ae10944"},
    # staged RoPE shift and state re-rotation
    "rope_shift_32768x8x128_bf16": {"bytes": 82_962_944, "src": ("boundary.cu",), "digest": "12e85b19d684",
                                    "commit": "ae9cc2f"},
    "state_rerotate_64x32_128x128_fp32": {"bytes": 206_485_504, "src": ("boundary.cu",), "digest": "12e85b19d684",
                                          "commit": "ae9cc2f"},
}


_CODE_TOKENS = re.compile(r'//[^\n]*|/\*.*?\*/|"(?:\\.|[^"\\\n])*"|\'(?:\\.|[^\'\\\n])*\'', re.S)


def code_text(src: str) -> str:
    """A source's code alone: comments dropped (string and character literals kept as they are) and
    every run of whitespace made one space, so that comment or layout edits keep the digest."""
    out = _CODE_TOKENS.sub(lambda m: " " if m.group(0)[0] == "/" else m.group(0), src)
    return " ".join(out.split())


def src_digest(names) -> str:
    """sha1 (first 12 hex digits) of the listed csrc files' code (see code_text)."""
    import hashlib
    h = hashlib.sha1()
    for n in names:
        with open(os.path.join(ROOT, "linear_attention_state_gb300", "csrc", n), encoding="utf-8") as f:
            h.update(code_text(f.read()).encode())
    return h.hexdigest()[:12]


def traffic(key):
    """Captured DRAM bytes of one launch, or None when not captured on the current sources."""
    t = TRAFFIC[key]
    if t["bytes"] is None or t["digest"] != src_digest(t["src"]):
        return None
    return t["bytes"]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"],
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained"), "sm_max_mhz": j.get("sm_max_mhz", 2070.0),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0,
                "source": "fallback"}


def fp32_simt_peak_tflops(sm_mhz):
    # 152 SMs x 128 FP32 lanes x 2 FLOP per FMA at the given clock.
    return 152 * 128 * 2 * sm_mhz * 1e6 / 1e12


# ---------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.t0 = time.time()
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            sel = str(device_index)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", sel], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------------------
class RequestStep:
    """Device-resident inputs and outputs of one request; step() runs the hot path once."""

    def __init__(self, w, dev, seed_offset=0):
        import torch

        import linear_attention_state_gb300 as hy
        self.hy = hy
        self.w = w
        tok = w.draw_request(dev)
        self.k, self.v = tok["k"], tok["v"]
        self.alpha, self.beta = tok["alpha"], tok["beta"]
        pos = torch.tensor(w.seam_positions(), device=dev)
        shp = (1, w.n_seg - 1, w.w, w.H)
        self.seam_q = tok["q"][pos].reshape(*shp, w.d).contiguous()
        self.seam_k = tok["k"][pos].reshape(*shp, w.d).contiguous()
        self.seam_v = tok["v"][pos].reshape(*shp, w.d).contiguous()
        self.seam_a = tok["alpha"][pos].reshape(shp).contiguous()
        self.seam_b = tok["beta"][pos].reshape(shp).contiguous()
        self.q_full = tok["q"]  # kept for the parity check of the bench line
        del tok
        self.bounds_list = w.body_bounds()
        self.bounds = torch.tensor(self.bounds_list, dtype=torch.int64, device=dev)
        self.max_len = max(e - b for b, e in self.bounds_list)
        self.T = torch.empty((w.n_seg, w.H, w.d, w.d), device=dev)
        self.S = torch.empty((w.n_seg, w.H, w.d, w.d), device=dev)
        # Requests run as a serving loop would: request i's assembly (one CTA per head) runs on its
        # own stream while request i + 1 builds, so the pairs alternate between two buffers and a
        # build waits for the assembly that last read its buffer.
        self.pairs = [(self.T, self.S), (torch.empty_like(self.T), torch.empty_like(self.S))]
        self.asm_stream = torch.cuda.Stream(device=dev)
        self.asm_done = [torch.cuda.Event(), torch.cuda.Event()]
        self.turn = 0
        self.idx = torch.arange(w.n_seg, dtype=torch.int32, device=dev)[None]
        self.S_out = torch.empty((1, w.H, w.d, w.d), device=dev)
        self.o = torch.empty((1, w.n_seg - 1, w.w, w.H, w.d), device=dev)
        ws_bytes = hy.build_workspace_bytes(w.H, w.d, w.n_seg, self.max_len, family=w.family, in_dtype=w.in_dtype)
        self.ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev) if ws_bytes else None
        # kernels per step: build (prep + chain per head block, or one recurrent launch) + assemble
        per_block = ws_bytes // max(1, w.H) if ws_bytes else 0
        blocks = -(-w.H // max(1, ws_bytes // per_block)) if ws_bytes else 0
        self.launches_per_step = (2 * blocks if ws_bytes and os.environ.get("HYPIC_BUILD_PATH") != "recurrent"
                                  else 1) + 1
        self.body_head_tokens = sum(e - b for b, e in self.bounds_list) * w.H
        self.tokens = w.n_seg * w.seg_len * w.layers
        self.compositions = w.n_seg * w.H
        self.seam_head_tokens = (w.n_seg - 1) * w.w * w.H

    def step(self, ev=None):
        import torch
        hy = self.hy
        i = self.turn % 2
        T, S = self.pairs[i]
        cur = torch.cuda.current_stream()
        if self.turn >= 2:
            cur.wait_event(self.asm_done[i])
        if ev is not None:
            ev[0].record()
        hy.segment_build_batched(self.k, self.v, self.bounds, self.alpha, self.beta, family=self.w.family,
                                 max_len=self.max_len, out=(T, S), ws=self.ws)
        built = torch.cuda.Event()
        built.record()
        if ev is not None:
            ev[1].record()
        self.asm_stream.wait_event(built)
        with torch.cuda.stream(self.asm_stream):
            hy.assemble(T, S, self.idx, self.seam_k, self.seam_v, self.seam_a, self.seam_b,
                        seam_q=self.seam_q, family=self.w.family, out=self.S_out, o_out=self.o)
            if ev is not None:
                ev[2].record()
            self.asm_done[i].record()
        self.turn += 1

    def join(self):
        """Makes the current stream wait for the last assembly."""
        import torch
        torch.cuda.current_stream().wait_stream(self.asm_stream)

    def host_copies(self):
        """Pinned host copies of the step's inputs (for the end-to-end measurement)."""
        names = ["k", "v", "alpha", "beta", "seam_q", "seam_k", "seam_v", "seam_a", "seam_b"]
        return {n: getattr(self, n).cpu().pin_memory() for n in names}


def run_timed(fn, steps, warmup, sync_all, kernel_events=True, finish=None):
    """Times `steps` calls of fn after `warmup` untimed ones, with CUDA events on the current stream.

    With kernel_events, fn records three events per step (before, between and after
    its two launches) and the per-launch durations are returned too.
    """
    import torch
    for _ in range(warmup):
        fn(None)
    if finish is not None:
        finish()
    sync_all()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    start.record()
    for i in range(steps):
        fn(evs[i] if kernel_events else None)
    if finish is not None:
        finish()
    end.record()
    sync_all()
    total_ms = start.elapsed_time(end)
    if not kernel_events:
        return total_ms, [], []
    k1 = [e[0].elapsed_time(e[1]) for e in evs]
    k2 = [e[1].elapsed_time(e[2]) for e in evs]
    return total_ms, k1, k2


def cpu_baseline(w, n_heads, threads, tok=None):
    """The oracle, as it stands, on a sample of heads of the same request: pairs, seams, compose.

    tok: the request's inputs on the host (the device request copied back), so that the results
    can be checked against the buffers the timed loop wrote; drawn on the host if None.  Returns
    (tokens/s, seconds, {head: (T_C per segment, S per segment, seam outputs, composed S)})."""
    import numpy as np

    import oracle
    if tok is None:
        tok = w.draw_request("cpu")
    heads = list(range(n_heads))
    bounds = w.body_bounds()

    def one_head(h):
        f = lambda t: t[:, h].double().numpy()  # noqa: E731
        k, v, q, a, b = f(tok["k"]), f(tok["v"]), f(tok["q"]), f(tok["alpha"]), f(tok["beta"])
        Ts, Ss, os_ = [], [], []
        for (b0, e0) in bounds:
            T, S = oracle.segment_pair(w.family, k[b0:e0], v[b0:e0], a[b0:e0], b[b0:e0])
            Ts.append(T.reshape(-1))
            Ss.append(S)
        S = np.zeros((w.d, w.d))
        for j in range(w.n_seg):
            if j >= 1 and w.w > 0:
                s0 = j * w.seg_len
                S, o = oracle.run(w.family, k[s0:s0 + w.w], v[s0:s0 + w.w], a[s0:s0 + w.w], b[s0:s0 + w.w],
                                  q=q[s0:s0 + w.w], S0=S)
                os_.append(o)
            S = oracle.compose(w.family, Ts[j][None], Ss[j][None], S_init=S)
        return Ts, Ss, os_, S

    t0 = time.perf_counter()
    res = oracle.parallel_map(one_head, heads, threads=threads)
    dt = time.perf_counter() - t0
    tokens_equiv = w.n_seg * w.seg_len * w.layers * n_heads / w.H
    return tokens_equiv / dt, dt, dict(zip(heads, res))


def request_parity(req, w, ref, tol):
    """The timed loop's last request against the oracle on the sampled heads: relative Frobenius
    error max(||gpu - ref|| / max(||ref||, 1e-30)) over heads and segments, for T_C, S_{C|0}, the
    seam outputs and the composed state."""
    import numpy as np

    def rel(x, r):
        return float(np.linalg.norm(x - r) / max(np.linalg.norm(r), 1e-30))

    T = req.T.double().cpu().numpy()
    S = req.S.double().cpu().numpy()
    So = req.S_out.double().cpu().numpy()
    o = req.o.double().cpu().numpy()
    err = {"T_C": 0.0, "S": 0.0, "seam_o": 0.0, "composed_S": 0.0}
    for h, (Ts, Ss, os_, Sf) in ref.items():
        for j in range(w.n_seg):
            err["T_C"] = max(err["T_C"], rel(T[j, h].reshape(-1), Ts[j]))
            err["S"] = max(err["S"], rel(S[j, h], Ss[j]))
        for j, oj in enumerate(os_):
            err["seam_o"] = max(err["seam_o"], rel(o[0, j, :, h], oj))
        err["composed_S"] = max(err["composed_S"], rel(So[0, h], Sf))
    return {"heads": len(ref), "max_rel_err": err, "tol": tol, "ok": all(e <= tol for e in err.values())}


def decay_build_measure(steps, warmup, dev, peaks):
    """Decay-family builds (64 segments x 512 tokens, 32 heads, bf16) and the 64-step compose of each.

    Roofline of the scalar and diagonal builds: HBM, algorithmic bytes per head-token = k and v
    (bf16, 2 x 256 B) + the gates (none for a constant gate, 4 B scalar, 512 B diagonal), plus
    the pairs written.  The gated-delta
    build is reported against the bf16 tensor peak with the chunked count.
    """
    import torch

    import linear_attention_state_gb300 as hy
    import workloads as W
    out = {}
    for fam, w in list(W.DECAY_FAMILIES.items()) + [("kda", W.KDA_BUILD)]:
        tok = w.draw_request(dev, need_q=False)
        bounds = torch.tensor(w.body_bounds(), device=dev)
        ws_bytes = hy.build_workspace_bytes(w.H, w.d, w.n_seg, w.seg_len, family=fam, in_dtype=w.in_dtype)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev) if ws_bytes else None
        T = torch.empty((w.n_seg, w.H, hy.t_size(fam, w.d)), device=dev)
        S = torch.empty((w.n_seg, w.H, w.d, w.d), device=dev)
        idx = torch.arange(w.n_seg, dtype=torch.int32, device=dev)[None]
        S_out = torch.empty((1, w.H, w.d, w.d), device=dev)

        def fn(ev):
            if ev is not None:
                ev[0].record()
            hy.segment_build_batched(tok["k"], tok["v"], bounds, tok["alpha"], tok["beta"], family=fam,
                                     max_len=w.seg_len, out=(T, S), ws=ws)
            if ev is not None:
                ev[1].record()
            hy.compose(T, S, idx, family=fam, out=S_out)
            if ev is not None:
                ev[2].record()

        _, kb, kc = run_timed(fn, steps, warmup, torch.cuda.synchronize)
        tb, tc = sum(kb) / len(kb) / 1e3, sum(kc) / len(kc) / 1e3
        ht = w.n_seg * w.seg_len * w.H
        entry = {"build_head_tokens_per_s": ht / tb, "build_ms": tb * 1e3,
                 "compose_ms": tc * 1e3, "compositions_per_s": w.n_seg * w.H / tc}
        recurrent = os.environ.get("HYPIC_BUILD_PATH") == "recurrent"
        if fam == "gated_delta" or (fam == "kda" and not recurrent):
            # chunked WY count (the per-channel decay of KDA leaves the products' shapes unchanged)
            fl = FLOP_PER_HEAD_TOKEN_WY * ht
            entry["roofline"] = {"bound": "tensor", "achieved": fl / tb / 1e12, "peak": peaks["bf16_tflops"],
                                 "unit": "TFLOP/s", "frac": fl / tb / 1e12 / peaks["bf16_tflops"],
                                 "flop_per_unit": FLOP_PER_HEAD_TOKEN_WY,
                                 "traffic": traffic("decay_kda" if fam == "kda" else "decay_gated_delta"),
                                 "kernel": ("kda_prep_kernel + chain_kda_kernel" if fam == "kda" else
                                            "wy_prep_kernel + chain_tc_kernel")}
        elif fam == "kda":
            # token-by-token fp32 kernel (no chunked KDA build): fp32 FMA roofline
            fl = FLOP_PER_HEAD_TOKEN_KDA_RECURRENT * ht
            alu = fp32_simt_peak_tflops(peaks["sm_max_mhz"])
            entry["roofline"] = {"bound": "alu", "achieved": fl / tb / 1e12, "peak": alu, "unit": "TFLOP/s",
                                 "frac": fl / tb / 1e12 / alu, "kernel": "recurrent_kernel (fp32 SIMT)",
                                 "flop_per_unit": FLOP_PER_HEAD_TOKEN_KDA_RECURRENT,
                                 "peak_source": "fp32 FMA: 152 SMs x 128 lanes x 2 FLOP x max SM clock"}
        else:
            per = 2 * w.d * 2 + {"scalar_const": 0, "scalar": 4, "diag": 4 * w.d}[fam]
            by = per * ht + w.n_seg * w.H * w.d * w.d * 4
            entry["roofline"] = {"bound": "hbm", "achieved": by / tb / 1e9, "peak": peaks["hbm_gbs"],
                                 "unit": "GB/s", "frac": by / tb / 1e9 / peaks["hbm_gbs"],
                                 "bytes_per_head_token": per, "traffic": traffic("decay_" + fam),
                                 "kernel": "build_decay_tc_kernel"}
        entry["status"] = hy.stream_status()
        out[fam] = entry
        del tok, T, S, ws
    torch.cuda.empty_cache()
    return out


def scan_measure(steps, warmup, dev, peaks, heads=None):
    """Affine scan of 64 pairs per head over 960 heads (d = 128, fp32): prefix pairs/s.  `heads`
    runs a reduced case (fewer heads, same per-head work) for counter captures."""
    import torch

    import linear_attention_state_gb300 as hy
    import workloads as W
    n, H, d = 64, heads or 960, 128
    T, S = W.random_pairs(n, H, d, dev, key=11)

    def fn(ev):
        if ev is not None:
            ev[0].record()
        hy.affine_scan(T, S, family="gated_delta")
        if ev is not None:
            ev[1].record()
            ev[2].record()

    total, k1, _ = run_timed(fn, steps, warmup, torch.cuda.synchronize)
    t = sum(k1) / len(k1) / 1e3
    by = n * H * (2 * d * d * 4) * 2  # read T and S, write both prefixes
    res = {"workload": f"scan_{n}x{H}heads_d{d}_fp32", "prefix_pairs_per_s": n * H / t, "ms": t * 1e3,
           "roofline": {"bound": "hbm", "achieved": by / t / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": by / t / 1e9 / peaks["hbm_gbs"], "traffic": traffic("scan")},
           "status": hy.stream_status()}
    del T, S
    # Few heads, a long chain: the two-level scan against one sequential chain per head.
    n2, H2 = 1024, 4
    T, S = W.random_pairs(n2, H2, d, dev, key=12)
    small = {"workload": f"scan_{n2}x{H2}heads_d{d}_fp32"}
    for name, two in (("two_level", True), ("plain", False)):
        def fn2(ev):
            if ev is not None:
                ev[0].record()
            hy.affine_scan(T, S, family="gated_delta", two_level=two)
            if ev is not None:
                ev[1].record()
                ev[2].record()
        _, k2, _ = run_timed(fn2, steps, warmup, torch.cuda.synchronize)
        small[f"ms_{name}"] = sum(k2) / len(k2)
    small["status"] = hy.stream_status()
    res["few_heads"] = small
    del T, S
    torch.cuda.empty_cache()
    return res


def build_outputs_measure(steps, warmup, dev, peaks):
    """The 32k-token build with every body token's output (q read, o written): the cold-segment
    forward fused with pair construction.  Reported beside the pair-only build of the headline."""
    import torch

    import linear_attention_state_gb300 as hy
    import workloads as W
    w = W.BUILD_32K
    tok = w.draw_request(dev)
    bounds = torch.tensor(w.body_bounds(), device=dev)
    ws_bytes = hy.build_workspace_bytes(w.H, w.d, w.n_seg, w.seg_len, family=w.family, in_dtype=w.in_dtype,
                                        want_o=True)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    T = torch.empty((w.n_seg, w.H, w.d * w.d), device=dev)
    S = torch.empty((w.n_seg, w.H, w.d, w.d), device=dev)
    o = torch.zeros((tok["k"].shape[0], w.H, w.d), device=dev)

    def fn(ev):
        if ev is not None:
            ev[0].record()
        hy.segment_build_batched(tok["k"], tok["v"], bounds, tok["alpha"], tok["beta"], q=tok["q"], family=w.family,
                                 max_len=w.seg_len, want_o=True, out=(T, S), ws=ws, o_out=o)
        if ev is not None:
            ev[1].record()
            ev[2].record()

    _, k1, _ = run_timed(fn, steps, warmup, torch.cuda.synchronize)
    tb = sum(k1) / len(k1) / 1e3
    ht = sum(e - b for b, e in w.body_bounds()) * w.H
    fl = FLOP_PER_HEAD_TOKEN_WY_O * ht
    res = {"workload": w.name + "_with_outputs", "build_ms": tb * 1e3, "body_head_tokens_per_s": ht / tb,
           "roofline": {"bound": "tensor", "achieved": fl / tb / 1e12, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                        "frac": fl / tb / 1e12 / peaks["bf16_tflops"], "flop_per_unit": FLOP_PER_HEAD_TOKEN_WY_O,
                        "traffic": traffic("build_outputs_tc") if os.environ.get("HYPIC_BUILD_PATH") != "recurrent" else None},
           "status": hy.stream_status()}
    del tok, ws, T, S, o
    torch.cuda.empty_cache()
    return res


def boundary_measure(steps, warmup, dev, peaks):
    """Boundary patches, HBM-bound: RoPE shift of one 32k-token segment's keys (8 heads x 128
    dims, bf16, out of place) and re-rotation of 2,048 scalar-family states (64 segments x 32
    heads, 128 x 128 fp32, in place).  Bytes are one read and one write of each tensor."""
    import torch

    import linear_attention_state_gb300 as hy
    g = torch.Generator(device=dev)
    g.manual_seed(881)
    K = torch.randn((32768, 8, 128), device=dev, generator=g).to(torch.bfloat16)
    K_out = torch.empty_like(K)
    S = torch.randn((64, 32, 128, 128), device=dev, generator=g)
    out = {}
    for name, fn_call, nbytes in (
            ("rope_shift_32768x8x128_bf16", lambda: hy.rope_shift(K, 70_001, base=1e6, out=K_out), 2 * K.numel() * 2),
            ("state_rerotate_64x32_128x128_fp32", lambda: hy.state_rerotate(S, 70_001, base=1e6, family="scalar"),
             2 * S.numel() * 4)):
        def fn(ev, f=fn_call):
            if ev is not None:
                ev[0].record()
            f()
            if ev is not None:
                ev[1].record()
                ev[2].record()

        _, k1, _ = run_timed(fn, steps, warmup, torch.cuda.synchronize)
        avg = sum(k1) / len(k1) / 1e3
        out[name] = {"ms": avg * 1e3, "roofline": {"bound": "hbm", "achieved": nbytes / avg / 1e9,
                                                    "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                                    "frac": nbytes / avg / 1e9 / peaks["hbm_gbs"],
                                                    "traffic": traffic(name)}}
    out["status"] = hy.stream_status()
    del K, K_out, S
    torch.cuda.empty_cache()
    return out


def compose_pool_measure(steps, warmup, dev, peaks, pool=None, n=None, random_pairs=False, storage="both",
                         layers=None):
    """Warm-cache composition: 30 layers x 32 heads, pool of 256 pairs, 64 requests x 16 segments.

    storage "f32": fp32 pairs (128 KiB per composition); "bf16": the same pairs rounded to bf16
    (64 KiB per composition, 16-bit cache storage); "both": fp32 first, then bf16 as "bf16_pool".
    """
    import dataclasses

    import torch

    import linear_attention_state_gb300 as hy
    import workloads as W
    pw = W.COMPOSE_POOL
    if pool is not None or n is not None or layers is not None:
        pw = dataclasses.replace(pw, pool=pool or pw.pool, n=n or pw.n, layers=layers or pw.layers,
                                 name=f"compose_{layers or pw.layers}x32_d128_pool{pool or pw.pool}_B{pw.B}x{n or pw.n}")
    H, d, P = pw.H, pw.d, pw.pool
    if random_pairs:
        pool_T, pool_S = W.random_pairs(P, H, d, dev, key=3)
    else:
        pool_T = torch.empty((P, H, d, d), device=dev)
        pool_S = torch.empty((P, H, d, d), device=dev)
        # Pool pairs: built (untimed) from 1024 seeded gated-delta tokens each.
        for p in range(P):
            tok = pw.pair_inputs(p, dev)
            T, S = hy.segment_build(tok["k"], tok["v"], tok["alpha"], tok["beta"], family="gated_delta")
            pool_T[p].copy_(T)
            pool_S[p].copy_(S)
            del tok, T, S
    idx = pw.request_indices(dev)
    out = torch.empty((pw.B, H, d, d), device=dev)
    comps = pw.B * pw.n * H

    def timed(pT, pS, bytes_per_comp, name, traffic_bytes):
        torch.cuda.synchronize()

        def fn(ev):
            if ev is not None:
                ev[0].record()
            hy.compose(pT, pS, idx, family="gated_delta", out=out)
            if ev is not None:
                ev[1].record()
                ev[2].record()

        total_ms, k1, _ = run_timed(fn, steps, warmup, torch.cuda.synchronize)
        avg = sum(k1) / len(k1) / 1e3
        bytes_ = comps * bytes_per_comp
        return {"workload": name, "compositions_per_s": comps / (total_ms / 1e3 / steps),
                "ms_per_step": total_ms / steps,
                "roofline": {"bound": "hbm", "achieved": bytes_ / avg / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                             "frac": bytes_ / avg / 1e9 / peaks["hbm_gbs"],
                             "traffic": traffic_bytes if (pool is None and n is None and layers is None) else None,
                             "dram_frac": (traffic_bytes / avg / 1e9 / peaks["hbm_gbs"]
                                           if traffic_bytes is not None and pool is None and n is None
                                           and layers is None else None),
                             "bytes_per_composition": bytes_per_comp, "peak_source": peaks["source"]},
                "status": hy.stream_status()}

    # Algorithmic bytes per composition: the pair read (T_C and S_{C|0}) plus the request's final
    # state, written once per chain of n compositions.
    out_per_comp = D * D * 4 / pw.n
    res = None
    if storage in ("f32", "both"):
        res = timed(pool_T, pool_S, BYTES_PER_COMPOSITION + out_per_comp, pw.name, traffic("compose_f32"))
    if storage in ("bf16", "both"):
        T_lp, S_lp = hy.pairs_to_bf16(pool_T, pool_S, family="gated_delta")
        del pool_T, pool_S
        torch.cuda.empty_cache()
        lp = timed(T_lp, S_lp, BYTES_PER_COMPOSITION // 2 + out_per_comp, pw.name + "_bf16pairs",
                   traffic("compose_bf16"))
        del T_lp, S_lp
        if res is None:
            res = lp
        else:
            res["bf16_pool"] = lp
    else:
        del pool_T, pool_S
    torch.cuda.empty_cache()
    return res


def t_path_parity(dev, threads):
    """The build on DeltaNet bodies (a = 1, 32 heads, 2 x 4096 tokens), whose T_C stays far above the
    fp32 range where the headline workload's T_C underflows: T_C and S_{C|0} of sampled heads against
    the oracle, so the line also checks the T half of the build."""
    import numpy as np
    import torch

    import linear_attention_state_gb300 as hy
    import oracle
    import workloads as W
    H, d, L_, nseg = 32, 128, 4096, 2
    g = W.generator(dev, 5151, 0)
    tok = W.draw_tokens(g, nseg * L_, H, d, "delta", "bf16", dev, need_q=False)
    bounds = [(j * L_, (j + 1) * L_) for j in range(nseg)]
    T, S = hy.segment_build_batched(tok["k"], tok["v"], torch.tensor(bounds, device=dev), None, tok["beta"],
                                    family="delta", max_len=L_)
    status = hy.stream_status()
    heads = [0, 13, 31]
    hk, hv, hb = (tok[x][:, heads].double().cpu().numpy() for x in ("k", "v", "beta"))
    Tg = T[:, heads].double().cpu().numpy()
    Sg = S[:, heads].double().cpu().numpy()
    units = [(i, j) for i in range(len(heads)) for j in range(nseg)]

    def ref(u):
        i, j = u
        b, e = bounds[j]
        return oracle.segment_pair("delta", hk[b:e, i], hv[b:e, i], None, hb[b:e, i])

    res = oracle.parallel_map(ref, units, threads=threads)
    eT = eS = 0.0
    tmin = float("inf")
    for (i, j), (Tr, Sr) in zip(units, res):
        eT = max(eT, float(np.linalg.norm(Tg[j, i].reshape(d, d) - Tr) / max(np.linalg.norm(Tr), 1e-30)))
        eS = max(eS, float(np.linalg.norm(Sg[j, i] - Sr) / max(np.linalg.norm(Sr), 1e-30)))
        tmin = min(tmin, float(np.linalg.norm(Tr)))
    del tok, T, S
    return {"workload": f"delta_{H}h_d{d}_{nseg}x{L_}", "heads": heads, "max_rel_err": {"T_C": eT, "S": eS},
            "min_ref_T_C_norm": tmin, "tol": 2e-3, "ok": max(eT, eS) <= 2e-3, "status": status}


def long_mixed_measure(steps, warmup, dev, peaks, threads, cpu=True):
    """Long mixed request: 30 layers x 32 heads (960 layer-heads), d = 128, bf16 inputs, 128 segments x
    1024 tokens (131,072 tokens); 32 cold segments built in the step, 96 arriving as cached fp32 pairs
    (built beforehand, untimed); seam window w = 8 on every inner segment, with outputs.

    One step = the cold builds (one batched launch over all layers) + the assembly (seams and 128
    compositions per layer-head, one launch).  A secondary schedule runs the same work layer by layer
    as a real stack would, a build and an assembly per layer (60 launches).  The oracle runs the step's
    work for three sampled layer-heads on the host cores (cpu_baseline; its cached pairs oracle-built
    beforehand, untimed) and the step's outputs are checked against it."""
    import numpy as np
    import torch

    import linear_attention_state_gb300 as hy
    import oracle
    import workloads as W
    w = W.LONG_MIXED
    H, d, n, Ls, ww, hpl = w.H, w.d, w.n_seg, w.seg_len, w.w, w.heads
    cold = W.long_mixed_cold(w)
    cold_set = set(cold)
    cached = [j for j in range(n) if j not in cold_set]
    slot = {j: i for i, j in enumerate(cached + cold)}  # cached pairs first, the cold builds last
    nc, nh = len(cached), len(cold)
    bf = torch.bfloat16
    pool_T = torch.empty((n, H, d, d), device=dev)
    pool_S = torch.empty((n, H, d, d), device=dev)
    ck = torch.empty((nh * Ls, H, d), dtype=bf, device=dev)
    cv = torch.empty_like(ck)
    ca = torch.empty((nh * Ls, H), device=dev)
    cb = torch.empty_like(ca)
    sk = torch.empty((1, n - 1, ww, H, d), dtype=bf, device=dev)
    sv, sq = torch.empty_like(sk), torch.empty_like(sk)
    sa = torch.empty((1, n - 1, ww, H), device=dev)
    sb = torch.empty_like(sa)
    ws1 = torch.empty(hy.build_workspace_bytes(H, d, 1, Ls), dtype=torch.uint8, device=dev)
    cbounds = []
    for j in range(n):
        tok = w.draw_segment(j, dev)
        lo = 0 if j == 0 else ww
        if j >= 1:
            sk[0, j - 1], sv[0, j - 1], sq[0, j - 1] = tok["k"][:ww], tok["v"][:ww], tok["q"][:ww]
            sa[0, j - 1], sb[0, j - 1] = tok["alpha"][:ww], tok["beta"][:ww]
        if j in cold_set:
            c = cold.index(j)
            ck[c * Ls:(c + 1) * Ls], cv[c * Ls:(c + 1) * Ls] = tok["k"], tok["v"]
            ca[c * Ls:(c + 1) * Ls], cb[c * Ls:(c + 1) * Ls] = tok["alpha"], tok["beta"]
            cbounds.append((c * Ls + lo, (c + 1) * Ls))
        else:
            i = slot[j]
            hy.segment_build_batched(tok["k"][lo:], tok["v"][lo:], torch.tensor([[0, Ls - lo]], device=dev),
                                     tok["alpha"][lo:], tok["beta"][lo:], family=w.family, max_len=Ls,
                                     out=(pool_T[i:i + 1], pool_S[i:i + 1]), ws=ws1)
        del tok
    del ws1
    cb_dev = torch.tensor(cbounds, dtype=torch.int64, device=dev)
    ws_c = torch.empty(hy.build_workspace_bytes(H, d, nh, Ls), dtype=torch.uint8, device=dev)
    idx = torch.tensor([[slot[j] for j in range(n)]], dtype=torch.int32, device=dev)
    S_out = torch.empty((1, H, d, d), device=dev)
    o = torch.empty((1, n - 1, ww, H, d), device=dev)
    Tc, Sc = pool_T[nc:], pool_S[nc:]

    def step(ev):
        if ev is not None:
            ev[0].record()
        hy.segment_build_batched(ck, cv, cb_dev, ca, cb, family=w.family, max_len=Ls, out=(Tc, Sc), ws=ws_c)
        if ev is not None:
            ev[1].record()
        hy.assemble(pool_T, pool_S, idx, sk, sv, sa, sb, seam_q=sq, family=w.family, out=S_out, o_out=o)
        if ev is not None:
            ev[2].record()

    total_ms, kb, ka = run_timed(step, steps, warmup, torch.cuda.synchronize)
    status = hy.stream_status()
    step_s = total_ms / 1e3 / steps
    tb, ta = sum(kb) / len(kb) / 1e3, sum(ka) / len(ka) / 1e3
    build_ht = sum(e - b for b, e in cbounds) * H
    comps = n * H
    seam_ht = (n - 1) * ww * H
    fl = FLOP_PER_HEAD_TOKEN_WY * build_ht
    # assembly bytes: the pairs read, the seam tokens (q, k, v bf16 and two fp32 gates) read, their
    # outputs written (fp32), the final state written
    asm_bytes = comps * BYTES_PER_COMPOSITION + seam_ht * (3 * d * 2 + 8 + d * 4) + H * d * d * 4
    res = {"workload": w.name, "cold_segments": nh, "cached_segments": nc,
           "request_tokens_per_s": n * Ls / step_s, "ms_per_step": step_s * 1e3,
           "build": {"ms": tb * 1e3, "body_head_tokens_per_s": build_ht / tb,
                     "roofline": {"bound": "tensor", "achieved": fl / tb / 1e12, "peak": peaks["bf16_tflops"],
                                  "unit": "TFLOP/s", "frac": fl / tb / 1e12 / peaks["bf16_tflops"],
                                  "flop_per_unit": FLOP_PER_HEAD_TOKEN_WY, "units_per_launch": build_ht}},
           "assemble": {"ms": ta * 1e3, "compositions_per_s": comps / ta, "seam_head_tokens_per_s": seam_ht / ta,
                        "roofline": {"bound": "hbm", "achieved": asm_bytes / ta / 1e9, "peak": peaks["hbm_gbs"],
                                     "unit": "GB/s", "frac": asm_bytes / ta / 1e9 / peaks["hbm_gbs"],
                                     "bytes_per_step": asm_bytes}},
           "status": status}
    sample_heads = [0, 17 * hpl + 9, 29 * hpl + 31]
    S_g = S_out[0, sample_heads].double().cpu().numpy()
    o_g = o[0, :, :, sample_heads].double().cpu().numpy()           # [n-1, w, 3, d]
    Tc_g = Tc[:, sample_heads].double().cpu().numpy()
    Sc_g = Sc[:, sample_heads].double().cpu().numpy()

    # Secondary schedule: layer by layer, a build of that layer's cold segments and its assembly.
    del ws_c
    per_layer = []
    for layer in range(w.layers):
        hs = slice(layer * hpl, (layer + 1) * hpl)
        lp_T, lp_S = pool_T[:, hs].contiguous(), pool_S[:, hs].contiguous()
        per_layer.append({"k": ck[:, hs].contiguous(), "v": cv[:, hs].contiguous(), "a": ca[:, hs].contiguous(),
                          "b": cb[:, hs].contiguous(), "T": lp_T, "S": lp_S,
                          "sk": sk[:, :, :, hs].contiguous(), "sv": sv[:, :, :, hs].contiguous(),
                          "sq": sq[:, :, :, hs].contiguous(), "sa": sa[:, :, :, hs].contiguous(),
                          "sb": sb[:, :, :, hs].contiguous(), "S_out": torch.empty((1, hpl, d, d), device=dev),
                          "o": torch.empty((1, n - 1, ww, hpl, d), device=dev)})
    del pool_T, pool_S, ck, cv, ca, cb, Tc, Sc
    torch.cuda.empty_cache()
    ws_l = torch.empty(hy.build_workspace_bytes(hpl, d, nh, Ls), dtype=torch.uint8, device=dev)

    def serial(ev):
        if ev is not None:
            ev[0].record()
        for L_ in per_layer:
            hy.segment_build_batched(L_["k"], L_["v"], cb_dev, L_["a"], L_["b"], family=w.family, max_len=Ls,
                                     out=(L_["T"][nc:], L_["S"][nc:]), ws=ws_l)
            hy.assemble(L_["T"], L_["S"], idx, L_["sk"], L_["sv"], L_["sa"], L_["sb"], seam_q=L_["sq"],
                        family=w.family, out=L_["S_out"], o_out=L_["o"])
        if ev is not None:
            ev[1].record()
            ev[2].record()

    s_ms, _, _ = run_timed(serial, steps, min(warmup, 3), torch.cuda.synchronize)
    s_step = s_ms / 1e3 / steps
    res["per_layer_serial"] = {"launches": 2 * w.layers, "ms_per_step": s_step * 1e3,
                               "request_tokens_per_s": n * Ls / s_step, "status": hy.stream_status()}
    # the serial schedule computes the same request state as the batched one (the build's chain
    # schedule differs with the head count, so the two agree to rounding, not bit for bit)
    dev_err = 0.0
    for i, h in enumerate(sample_heads):
        x = per_layer[h // hpl]["S_out"][0, h % hpl].double().cpu().numpy()
        dev_err = max(dev_err, float(np.linalg.norm(x - S_g[i]) / max(np.linalg.norm(S_g[i]), 1e-30)))
    res["per_layer_serial"]["max_rel_diff_vs_batched"] = dev_err
    del per_layer, ws_l
    torch.cuda.empty_cache()
    if not cpu:
        return res

    # Oracle on the host: the step's work for the sampled layer-heads (cold builds + assembly), and the
    # step's outputs against it.  Inputs are the device draws of those heads, copied to the host.
    host = {key: [] for key in ("k", "q", "v", "alpha", "beta")}
    for j in range(n):
        t = w.draw_segment(j, dev, heads=sample_heads)
        for key in host:
            host[key].append(t[key].double().cpu().numpy())
        del t
    fam = w.family

    def body(i, j):
        lo = 0 if j == 0 else ww
        return tuple(host[x][j][lo:, i] for x in ("k", "v", "alpha", "beta"))

    cached_units = [(i, j) for i in range(len(sample_heads)) for j in cached]
    pairs = dict(zip(cached_units, oracle.parallel_map(lambda u: oracle.segment_pair(fam, *body(*u)), cached_units,
                                                       threads=threads)))
    cold_units = [(i, j) for i in range(len(sample_heads)) for j in cold]
    t0 = time.perf_counter()
    pairs.update(zip(cold_units, oracle.parallel_map(lambda u: oracle.segment_pair(fam, *body(*u)), cold_units,
                                                     threads=threads)))

    def assemble_ref(i):
        S = np.zeros((d, d))
        outs = []
        for j in range(n):
            if j >= 1:
                S, oj = oracle.run(fam, host["k"][j][:ww, i], host["v"][j][:ww, i], host["alpha"][j][:ww, i],
                                   host["beta"][j][:ww, i], q=host["q"][j][:ww, i], S0=S)
                outs.append(oj)
            T, S0 = pairs[(i, j)]
            S = oracle.compose(fam, T[None], S0[None], S_init=S)
        return S, outs

    ref = oracle.parallel_map(assemble_ref, list(range(len(sample_heads))), threads=threads)
    dt = time.perf_counter() - t0

    def rel(x, r):
        return float(np.linalg.norm(x - r) / max(np.linalg.norm(r), 1e-30))

    err = {"cold_T_C": 0.0, "cold_S": 0.0, "seam_o": 0.0, "composed_S": 0.0}
    for i in range(len(sample_heads)):
        for c, j in enumerate(cold):
            Tr, Sr = pairs[(i, j)]
            err["cold_T_C"] = max(err["cold_T_C"], rel(Tc_g[c, i], Tr))
            err["cold_S"] = max(err["cold_S"], rel(Sc_g[c, i], Sr))
        Sf, outs = ref[i]
        err["composed_S"] = max(err["composed_S"], rel(S_g[i], Sf))
        for jj, oj in enumerate(outs):
            err["seam_o"] = max(err["seam_o"], rel(o_g[jj, :, i], oj))
    res["parity"] = {"layer_heads": sample_heads, "max_rel_err": err, "tol": 2e-3,
                     "ok": all(v <= 2e-3 for v in err.values())}
    frac = len(sample_heads) / H
    res["cpu_baseline"] = {"value": n * Ls * frac / dt, "unit": "request tokens/s", "cores": threads, "kind": "oracle",
                           "sample": f"{len(sample_heads)} of {H} layer-heads: {nh} cold builds + the assembly "
                                     f"({n - 1} seam windows, {n} compositions), float64, {dt:.1f} s wall"}
    return res


# ---------------------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-compose", action="store_true", help="skip the warm-cache composition measurement")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--compose-only", action="store_true",
                    help="time only the warm-cache composition (profiling aid; prints its own line)")
    ap.add_argument("--compose-pool", type=int, default=None, help="pool entries per head (default 256)")
    ap.add_argument("--compose-n", type=int, default=None, help="segments per request (default 16)")
    ap.add_argument("--compose-random", action="store_true", help="generator-drawn pairs instead of built ones")
    ap.add_argument("--compose-layers", type=int, default=None,
                    help="layers of 32 heads in the composition measurement (default 30; fewer for profiling)")
    ap.add_argument("--build-only", action="store_true",
                    help="time only the headline request's build and assembly loop (profiling aid)")
    ap.add_argument("--compose-storage", default="both", choices=["both", "f32", "bf16"],
                    help="pair storage of the composition measurement (fp32, bf16 or both)")
    ap.add_argument("--decay-only", action="store_true",
                    help="time only the decay-family builds (profiling aid; prints its own line)")
    ap.add_argument("--scan-heads", type=int, default=None,
                    help="heads of the scan measurement (default 960; fewer for counter captures)")
    ap.add_argument("--scan-only", action="store_true",
                    help="time only the affine scan (profiling aid; prints its own line)")
    ap.add_argument("--boundary-only", action="store_true",
                    help="time only the boundary patches (profiling aid; prints its own line)")
    ap.add_argument("--long-only", action="store_true",
                    help="time only the long mixed request (profiling aid; prints its own line)")
    ap.add_argument("--no-long", action="store_true", help="skip the long mixed request")
    ap.add_argument("--outputs-only", action="store_true",
                    help="time only the build with per-token outputs (profiling aid; prints its own line)")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    import workloads as W
    w = W.BUILD_32K

    if args.impl == "reference":
        return run_reference(args, w, rank, world)

    import torch
    import torch.distributed as dist
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device(dev))
    from linear_attention_state_gb300 import build as B
    if rank == 0 or world == 1:
        B.build_library()
    if world > 1:
        dist.barrier()
    import linear_attention_state_gb300 as hy
    hy.load()
    peaks = load_peaks()

    def sync_all():
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()

    if args.compose_only:
        res = compose_pool_measure(args.steps, args.warmup, dev, peaks, args.compose_pool, args.compose_n,
                                   args.compose_random, args.compose_storage, args.compose_layers)
        if rank == 0:
            print(json.dumps({"metric": "compositions/s", "value": res["compositions_per_s"] * world,
                              "unit": "compositions/s", "n_gpus": world, "steps": args.steps,
                              "warmup": args.warmup, "compose_pool": res}))
        return
    if args.decay_only or args.scan_only or args.boundary_only or args.outputs_only:
        fn, what = ((decay_build_measure, "decay-family builds") if args.decay_only else
                    (functools.partial(scan_measure, heads=args.scan_heads), "affine scan") if args.scan_only else
                    (build_outputs_measure, "build with outputs") if args.outputs_only else
                    (boundary_measure, "boundary patches"))
        res = fn(args.steps, args.warmup, dev, peaks)
        if rank == 0:
            print(json.dumps({"metric": what, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                              "result": res}))
        return
    if args.long_only:
        res = long_mixed_measure(args.steps, args.warmup, dev, peaks, os.cpu_count() or 1,
                                 cpu=rank == 0 and world == 1 and not args.no_cpu)
        if rank == 0:
            print(json.dumps({"metric": "long mixed request", "n_gpus": world, "steps": args.steps,
                              "warmup": args.warmup, "result": res}))
        return
    req = RequestStep(w, dev)
    status0 = hy.stream_status()
    if args.build_only:
        total_ms, k_build, k_asm = run_timed(req.step, args.steps, args.warmup, sync_all, finish=req.join)
        if rank == 0:
            print(json.dumps({"metric": "build and assembly loop", "n_gpus": world, "steps": args.steps,
                              "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
                              "build_ms": sum(k_build) / len(k_build), "assemble_ms": sum(k_asm) / len(k_asm),
                              "status": hy.stream_status()}))
        return
    clocks = ClockSampler(local)
    total_ms, k_build, k_asm = run_timed(req.step, args.steps, args.warmup, sync_all, finish=req.join)
    clk = clocks.stop()
    status = hy.stream_status()
    # what the timed loop wrote, kept for the parity check (the end-to-end loop below reuses the buffers)
    snap = types.SimpleNamespace(T=req.T.clone(), S=req.S.clone(), S_out=req.S_out.clone(), o=req.o.clone())
    t = torch.tensor([total_ms], device=dev)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    total_ms = float(t.item())
    step_s = total_ms / 1e3 / args.steps
    value = req.tokens * world / step_s

    # dominant kernel: the build
    avg_build_s = sum(k_build) / len(k_build) / 1e3
    avg_asm_s = sum(k_asm) / len(k_asm) / 1e3
    if os.environ.get("HYPIC_BUILD_PATH") == "recurrent":
        flops = FLOP_PER_HEAD_TOKEN_RECURRENT * req.body_head_tokens
        alu_peak = fp32_simt_peak_tflops(peaks["sm_max_mhz"])
        roof = {"bound": "alu", "achieved": flops / avg_build_s / 1e12, "peak": alu_peak, "unit": "TFLOP/s",
                "frac": flops / avg_build_s / 1e12 / alu_peak, "traffic": None,
                "kernel": "recurrent_kernel (build, fp32 SIMT)",
                "peak_source": "fp32 FMA: 152 SMs x 128 lanes x 2 FLOP x max SM clock",
                "flop_per_unit": FLOP_PER_HEAD_TOKEN_RECURRENT, "units_per_launch": req.body_head_tokens}
    else:
        flops = FLOP_PER_HEAD_TOKEN_WY * req.body_head_tokens
        pk = peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": flops / avg_build_s / 1e12, "peak": pk, "unit": "TFLOP/s",
                "frac": flops / avg_build_s / 1e12 / pk, "traffic": traffic("build_tc"),
                "kernel": "build: wy_prep_kernel + chain_tc_kernel (chunked WY, tcgen05)",
                "peak_source": f"{peaks['source']} dense bf16 (burst)",
                "flop_per_unit": FLOP_PER_HEAD_TOKEN_WY, "units_per_launch": req.body_head_tokens}

    # end to end through the API with host buffers
    host = req.host_copies()
    S_host = torch.empty(req.S_out.shape, pin_memory=True)
    o_host = torch.empty(req.o.shape, pin_memory=True)
    h2d = sum(x.numel() * x.element_size() for x in host.values())
    d2h = S_host.numel() * 4 + o_host.numel() * 4

    # The request's k, v and gates go through the host-input build, which copies segment groups on a
    # second stream while the earlier ones build; the seam tokens (0.7 MB) are copied first.  Two
    # sets of device input buffers alternate between requests, as in a serving loop: request i + 1's
    # inputs cross the host link while request i finishes (its last group, assembly and readback);
    # the copies of a set wait for the event recorded after the previous build that read it.
    bounds_host = torch.tensor(req.bounds_list, dtype=torch.int64)
    copy_stream = torch.cuda.Stream()
    seam_names = [n for n in host if n.startswith("seam_")]
    dev_sets = [(req.k, req.v, req.alpha, req.beta, req.bounds),
                tuple(torch.empty_like(t) for t in (req.k, req.v, req.alpha, req.beta, req.bounds))]
    set_free = [torch.cuda.Event(), torch.cuda.Event()]
    turn = [0]

    def e2e_step(ev):
        i = turn[0] % 2
        for n in seam_names:
            getattr(req, n).copy_(host[n], non_blocking=True)
        hy.segment_build_batched_host(host["k"], host["v"], bounds_host, host["alpha"], host["beta"],
                                      family=w.family, max_len=req.max_len, dev=dev_sets[i], out=(req.T, req.S),
                                      ws=req.ws, copy_stream=copy_stream,
                                      ready_event=set_free[i] if turn[0] >= 2 else None)
        set_free[i].record()
        turn[0] += 1
        hy.assemble(req.T, req.S, req.idx, req.seam_k, req.seam_v, req.seam_a, req.seam_b, seam_q=req.seam_q,
                    family=w.family, out=req.S_out, o_out=req.o)
        S_host.copy_(req.S_out, non_blocking=True)
        o_host.copy_(req.o, non_blocking=True)

    e2e_ms, _, _ = run_timed(e2e_step, args.steps, min(args.warmup, 3), sync_all, kernel_events=False)
    e2e_value = req.tokens * world / (e2e_ms / 1e3 / args.steps)
    del dev_sets, host

    threads = os.cpu_count() or 1
    decay = scan = bnd = outs = compose = longm = None
    if not args.no_compose:
        outs = build_outputs_measure(args.steps, args.warmup, dev, peaks)
        decay = decay_build_measure(args.steps, args.warmup, dev, peaks)
        scan = scan_measure(args.steps, args.warmup, dev, peaks)
        bnd = boundary_measure(args.steps, args.warmup, dev, peaks)
        compose = compose_pool_measure(args.steps, args.warmup, dev, peaks, args.compose_pool, args.compose_n,
                                       args.compose_random, args.compose_storage)
    if not args.no_long:
        longm = long_mixed_measure(args.steps, args.warmup, dev, peaks, threads,
                                   cpu=rank == 0 and world == 1 and not args.no_cpu)

    cpu = parity = t_par = None
    if rank == 0 and world == 1 and not args.no_cpu:
        n_heads = min(w.H, max(1, threads))
        torch.cuda.synchronize()
        # the device request's own inputs, so the oracle also checks what the timed loop computed
        host_tok = {"k": req.k[:, :n_heads].cpu(), "v": req.v[:, :n_heads].cpu(),
                    "alpha": req.alpha[:, :n_heads].cpu(), "beta": req.beta[:, :n_heads].cpu(),
                    "q": req.q_full[:, :n_heads].cpu()}
        v_cpu, dt, ref = cpu_baseline(w, n_heads, threads, tok=host_tok)
        parity = request_parity(snap, w, ref, 2e-3 if w.in_dtype == "bf16" else 1e-5)
        cpu = {"value": v_cpu, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"{n_heads} of {w.H} heads of the same request, all 8 segments (pairs, seams, compose), "
                         f"float64, {dt:.1f} s wall"}
        if os.environ.get("HYPIC_BUILD_PATH") != "recurrent":
            t_par = t_path_parity(dev, threads)

    dtype = "f32" if os.environ.get("HYPIC_BUILD_PATH") == "recurrent" else "bf16"
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": dtype, "data": "synthetic",
            "config": bench_config(w, world),
            "build": {"body_head_tokens_per_s": req.body_head_tokens / avg_build_s, "ms": avg_build_s * 1e3},
            "assemble": {"compositions_per_s": req.compositions / avg_asm_s,
                         "seam_head_tokens_per_s": req.seam_head_tokens / avg_asm_s, "ms": avg_asm_s * 1e3},
            "roofline": roof,
            "compose_pool": compose,
            "decay_builds": decay,
            "affine_scan": scan,
            "boundary_patches": bnd,
            "build_with_outputs": outs,
            "long_mixed": longm,
            "cpu_baseline": cpu,
            "parity": parity,
            "parity_t_path": t_par,
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": req.launches_per_step * args.steps,
            "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"],
                       "samples": clk["samples"], "window": "warm-up and timed steps"},
            "device_status": [status0, status],
        }
        line["summary"] = summary(line)
        print(json.dumps(line))
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def bench_config(w, world):
    """The workload of the headline line (both arms print the same)."""
    return {"workload": w.name, "layers": w.layers, "heads": w.heads, "d": w.d, "segments": w.n_seg,
            "segment_tokens": w.seg_len, "seam_w": w.w, "inputs": "bf16 q/k/v, fp32 gates and state",
            "l2": "inputs larger than L2 (k+v 537 MB per step), no flush",
            "parallelism": f"replicas x{world}",
            "pipelining": "request i's assembly runs on a second stream while request i+1 builds "
                          "(pairs double-buffered); every step builds and assembles a whole request"}


def summary(line):
    """The headline figures in a few hundred bytes, printed last in the JSON line."""
    def r(x, n=3):
        return None if x is None else float(f"{x:.{n}g}")

    def g(d, *keys):
        for k in keys:
            if d is None:
                return None
            d = d.get(k) if isinstance(d, dict) else None
        return d

    cp = line.get("compose_pool")
    dec = line.get("decay_builds") or {}
    lm = line.get("long_mixed")
    return {
        "tok_per_s": r(line["value"]), "e2e_tok_per_s": r(line["e2e"]["value"]),
        "build_ms": r(line["build"]["ms"]), "build_tensor_frac": r(line["roofline"]["frac"]),
        "assemble_ms": r(line["assemble"]["ms"]),
        "compose_f32": {"comp_per_s": r(g(cp, "compositions_per_s")), "hbm_frac": r(g(cp, "roofline", "frac")),
                        "dram_frac": r(g(cp, "roofline", "dram_frac"))},
        "compose_bf16": {"comp_per_s": r(g(cp, "bf16_pool", "compositions_per_s")),
                         "hbm_frac": r(g(cp, "bf16_pool", "roofline", "frac")),
                         "dram_frac": r(g(cp, "bf16_pool", "roofline", "dram_frac"))},
        "scan_hbm_frac": r(g(line.get("affine_scan"), "roofline", "frac")),
        "decay_frac": {f: r(g(dec, f, "roofline", "frac")) for f in dec},
        "outputs_build_tensor_frac": r(g(line.get("build_with_outputs"), "roofline", "frac")),
        "long_mixed": {"tok_per_s": r(g(lm, "request_tokens_per_s")),
                       "build_tensor_frac": r(g(lm, "build", "roofline", "frac")),
                       "assemble_hbm_frac": r(g(lm, "assemble", "roofline", "frac")),
                       "serial_tok_per_s": r(g(lm, "per_layer_serial", "request_tokens_per_s"))},
        "parity_ok": {"request": g(line.get("parity"), "ok"), "t_path": g(line.get("parity_t_path"), "ok"),
                      "long_mixed": g(lm, "parity", "ok")},
    }


def run_reference(args, w, rank, world):
    """Reference arm: the float64 oracle on every host core, K timed steps of a bounded sample of the
    same request (half the heads on 16 cores), in the headline line's format and config."""
    if rank != 0:
        return
    threads = os.cpu_count() or 1
    n_heads = min(w.H, max(1, threads))
    for _ in range(args.warmup):
        cpu_baseline(w, 1, 1)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        cpu_baseline(w, n_heads, threads)
    dt = (time.perf_counter() - t0) / args.steps
    value = w.n_seg * w.seg_len * w.layers * n_heads / w.H / dt
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": bench_config(w, world),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": f"{n_heads} of {w.H} heads of the request per step, {threads} threads; "
                                       "tokens/s scaled to the whole request"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
