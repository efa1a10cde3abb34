"""Pins for the float64 oracle: checks against what the pages and the mathematics fix.

Nothing here retypes the oracle's loops.  Each pin compares the oracle with an
independent statement of the same quantity:

* the page's worked example and Table 2 values (``tests/golden/``);
* closed forms (scalar and diagonal decay, the T_i = I reduction to a sum);
* brute force with dense matrices: T_i and u_i formed explicitly from Table 1
  and multiplied out with numpy, S_{C|0} taken as the explicit sum
  sum_t T_m...T_{t+1} u_t rather than a recurrence;
* algebraic laws: the composition law S(C1 C2) = T(C2) S(C1) + S(C2), paper
  Eq. (6) as a sum of products, associativity and non-commutativity;
* special cases of Table 1 (beta = 0, a = 1, idempotent erasure) and the
  spectral bound ||T_C||_2 <= prod a_t for beta in [0, 1], ||k|| = 1.

``test_pins_catch_planted_mistakes`` compiles mutated copies of the oracle
source (a dropped term, a sign flip, a transposed index, a misplaced gate ...)
and checks that every mutant fails at least one pin.

Source of every formula: HYPIC reading notes (HYPIC: Accelerating
Hybrid-Attention LLM Serving with Position-Independent Caching): Motivation 2
(paper Eqs. (2)-(5), Table 2), Method 2 (affine maps, composition, worked
example, Eq. (6)), Method 3 (Tables 1 and 3), Method 4 (two-pass build).
"""
from __future__ import annotations

import json
import math
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle as O

GOLD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
FAMS = ["scalar_const", "scalar", "diag", "delta", "gated_delta", "kda"]
DENSE = ("delta", "gated_delta", "kda")


def _softplus(z):
    return np.log1p(np.exp(-np.abs(z))) + np.maximum(z, 0)


def rand_inputs(rng, fam, L, dk, dv, gate_div=8.0):
    k = rng.standard_normal((L, dk))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    q = rng.standard_normal((L, dk))
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    v = rng.standard_normal((L, dv))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(L)))
    if fam in ("diag", "kda"):
        alpha = np.exp(-_softplus(rng.standard_normal((L, dk))) / gate_div)
    elif fam == "scalar_const":
        alpha = np.array([0.9 + 0.09 * rng.random()])
    else:
        alpha = np.exp(-_softplus(rng.standard_normal(L)) / gate_div)
    return k, q, v, alpha, beta


def rel(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


def as_dense_T(fam, T, dk):
    T = np.asarray(T)
    if fam in ("scalar_const", "scalar"):
        return float(T.reshape(-1)[0]) * np.eye(dk)
    if fam == "diag":
        return np.diag(T.reshape(-1))
    return T.reshape(dk, dk)


def slice_gates(fam, alpha, beta, a, b):
    if fam == "scalar_const":
        return alpha, beta[a:b]
    return alpha[a:b], beta[a:b]


# --- brute force straight from Table 1 -------------------------------------------------

def dense_step_matrices(fam, k, v, alpha, beta, t):
    dk = k.shape[1]
    kt, vt = k[t], v[t]
    eye = np.eye(dk)
    if fam == "scalar_const":
        return alpha[0] * eye, np.outer(kt, vt)
    if fam == "scalar":
        return alpha[t] * eye, np.outer(kt, vt)
    if fam == "diag":
        return np.diag(alpha[t]), np.outer(kt, vt)
    erase = eye - beta[t] * np.outer(kt, kt)
    if fam == "delta":
        return erase, beta[t] * np.outer(kt, vt)
    if fam == "kda":
        return erase @ np.diag(alpha[t]), beta[t] * np.outer(kt, vt)
    return alpha[t] * erase, beta[t] * np.outer(kt, vt)


def brute_pair(fam, k, v, alpha, beta):
    """T_C = T_m ... T_1 and S_{C|0} = sum_t (T_m ... T_{t+1}) u_t, both explicit."""
    L, dk = k.shape
    mats = [dense_step_matrices(fam, k, v, alpha, beta, t) for t in range(L)]
    T_C = np.eye(dk)
    for Ti, _ in mats:
        T_C = Ti @ T_C
    S = np.zeros((dk, v.shape[1]))
    for t in range(L):
        suffix = np.eye(dk)
        for s in range(t + 1, L):
            suffix = mats[s][0] @ suffix
        S += suffix @ mats[t][1]
    return T_C, S


def brute_outputs(fam, k, v, q, alpha, beta, S0):
    """o_t = q_t^T S_t with S_t = T_t S_{t-1} + u_t using dense T_t (paper Eq. (2))."""
    S = S0.copy()
    out = []
    for t in range(k.shape[0]):
        Ti, ui = dense_step_matrices(fam, k, v, alpha, beta, t)
        S = Ti @ S + ui
        out.append(q[t] @ S)
    return np.array(out), S


# --- the pins ---------------------------------------------------------------------------

def pin_worked_example(orc):
    g = json.load(open(os.path.join(GOLD, "worked_example_1d.json")))
    a = np.array([t["a"] for t in g["tokens"]])
    u = np.array([t["u"] for t in g["tokens"]])
    # u_t = k_t v_t^T with d_k = d_v = 1: k = 1, v = u.
    k = np.ones((len(a), 1))
    v = u.reshape(-1, 1)
    T, S = orc.segment_pair("scalar", k, v, a)
    assert abs(float(np.asarray(T).reshape(-1)[0]) - g["T_C"]) < 1e-15
    assert abs(float(S[0, 0]) - g["S_C_given_0"]) < 1e-15
    composed = orc.compose("scalar", np.asarray(T).reshape(1, -1), S[None], S_init=np.array([[g["prefix_state"]]]))
    assert abs(float(composed[0, 0]) - g["composed_end_state"]) < 1e-14
    ran, _ = orc.run("scalar", k, v, a, S0=np.array([[g["prefix_state"]]]))
    assert abs(float(ran[0, 0]) - g["composed_end_state"]) < 1e-14
    naive = g["prefix_state"] + float(S[0, 0])
    assert abs(naive - g["naive_addition_end_state"]) < 1e-14


def pin_table2(orc):
    g = json.load(open(os.path.join(GOLD, "table2_scalar_decay_error.json")))
    gamma = 1.0 - 2.0 ** -10
    rng = np.random.default_rng(7)
    d = 8
    for L, printed in zip(g["lengths"], g["relative_error_printed"]):
        k1, _, v1, _, _ = rand_inputs(rng, "scalar_const", 40, d, d)
        k2, _, v2, _, _ = rand_inputs(rng, "scalar_const", L, d, d)
        g1 = np.array([gamma])
        T1, S1 = orc.segment_pair("scalar_const", k1, v1, g1)
        T2, S2 = orc.segment_pair("scalar_const", k2, v2, g1)
        true = orc.compose("scalar_const", np.asarray(T2).reshape(1, -1), S2[None], S_init=S1)
        naive = S1 + S2
        delta = true - naive  # sign convention: true minus naive
        ratio = np.linalg.norm(delta) / np.linalg.norm(S1)
        assert round(ratio, g["printed_decimals"]) == printed
        assert abs(ratio - (1.0 - gamma ** L)) < 1e-12


def pin_composition_law(orc):
    rng = np.random.default_rng(11)
    for fam in FAMS:
        dk, dv, L = 5, 4, 23
        k, q, v, alpha, beta = rand_inputs(rng, fam, L, dk, dv)
        T12, S12 = orc.segment_pair(fam, k, v, alpha, beta)
        for cut in (0, 1, 9, L - 1, L):
            a1, b1 = slice_gates(fam, alpha, beta, 0, cut)
            a2, b2 = slice_gates(fam, alpha, beta, cut, L)
            T1, S1 = orc.segment_pair(fam, k[:cut], v[:cut], a1, b1)
            T2, S2 = orc.segment_pair(fam, k[cut:], v[cut:], a2, b2)
            # S(C1 C2) = T(C2) S(C1) + S(C2) and T(C1 C2) = T(C2) T(C1)
            D2 = as_dense_T(fam, T2, dk)
            assert rel(D2 @ S1 + S2, S12) < 1e-12
            assert rel(D2 @ as_dense_T(fam, T1, dk), as_dense_T(fam, T12, dk)) < 1e-12
            T3, S3 = orc.affine_combine(fam, T2, S2, T1, S1)
            assert rel(S3, S12) < 1e-12 and rel(as_dense_T(fam, T3, dk), as_dense_T(fam, T12, dk)) < 1e-12
        # F_C(X) = T_C X + S_{C|0} equals running the tokens from X.
        X = rng.standard_normal((dk, dv))
        ran, _ = orc.run(fam, k, v, alpha, beta, S0=X)
        assert rel(as_dense_T(fam, T12, dk) @ X + S12, ran) < 1e-12


def pin_eq6(orc):
    """Paper Eq. (6) as a sum of products equals n sequential compositions and the full run."""
    rng = np.random.default_rng(12)
    for fam in FAMS:
        dk, dv = 4, 6
        lens = [0, 1, 7, 3, 12]
        L = sum(lens)
        k, q, v, alpha, beta = rand_inputs(rng, fam, L, dk, dv)
        S_S = rng.standard_normal((dk, dv))
        Ts, Ss = [], []
        off = 0
        for n_ in lens:
            a_, b_ = slice_gates(fam, alpha, beta, off, off + n_)
            T, S = orc.segment_pair(fam, k[off:off + n_], v[off:off + n_], a_, b_)
            Ts.append(as_dense_T(fam, T, dk))
            Ss.append(S)
            off += n_
        n = len(lens)
        prod_all = np.eye(dk)
        for i in range(n):
            prod_all = Ts[i] @ prod_all
        eq6 = prod_all @ S_S
        for i in range(n):
            P = np.eye(dk)
            for j in range(i + 1, n):
                P = Ts[j] @ P
            eq6 += P @ Ss[i]
        ts = orc.t_size(fam, dk)
        Tstore = np.stack([(T if ts == dk * dk else (np.diag(T) if ts == dk else T[:1, :1])).reshape(-1)[:ts]
                           for T in Ts])
        comp = orc.compose(fam, Tstore, np.stack(Ss), S_init=S_S)
        full, _ = orc.run(fam, k, v, alpha, beta, S0=S_S)
        assert rel(comp, eq6) < 1e-12
        assert rel(full, eq6) < 1e-12


def pin_assoc_noncommut(orc):
    rng = np.random.default_rng(13)
    dk, dv = 5, 3
    pairs = []
    for _ in range(3):
        T = rng.standard_normal((dk, dk)) / math.sqrt(dk)
        S = rng.standard_normal((dk, dv))
        pairs.append((T, S))
    (Ta, Sa), (Tb, Sb), (Tc, Sc) = pairs
    Tba, Sba = orc.affine_combine("gated_delta", Tb, Sb, Ta, Sa)
    Tcb, Scb = orc.affine_combine("gated_delta", Tc, Sc, Tb, Sb)
    T1, S1 = orc.affine_combine("gated_delta", Tc, Sc, Tba, Sba)  # c o (b o a)
    T2, S2 = orc.affine_combine("gated_delta", Tcb, Scb, Ta, Sa)  # (c o b) o a
    assert rel(T1, T2) < 1e-12 and rel(S1, S2) < 1e-12
    # direct definition: (T_B T_A, T_B B_A + B_B)
    assert rel(Tba, Tb @ Ta) < 1e-12 and rel(Sba, Tb @ Sa + Sb) < 1e-12
    Tab, Sab = orc.affine_combine("gated_delta", Ta, Sa, Tb, Sb)
    assert rel(Sab, Sba) > 1e-3  # order matters


def pin_identity_reduction(orc):
    """With every T_i = I the zero-initial end states just add up (Motivation 2)."""
    rng = np.random.default_rng(14)
    dk, dv, L = 6, 5, 31
    k, _, v, _, _ = rand_inputs(rng, "scalar", L, dk, dv)
    ones = np.ones(L)
    T, S = orc.segment_pair("scalar", k, v, ones)
    assert float(np.asarray(T).reshape(-1)[0]) == 1.0
    assert rel(S, np.einsum("ti,tj->ij", k, v)) < 1e-13
    # and additivity of two segments holds exactly in that case
    T1, S1 = orc.segment_pair("scalar", k[:10], v[:10], ones[:10])
    T2, S2 = orc.segment_pair("scalar", k[10:], v[10:], ones[10:])
    assert rel(S1 + S2, S) < 1e-13


def pin_scalar_closed_form(orc):
    rng = np.random.default_rng(15)
    dk, dv, L = 4, 3, 300
    k, _, v, _, _ = rand_inputs(rng, "scalar_const", L, dk, dv)
    gamma = 1.0 - 2.0 ** -5.75
    T, S = orc.segment_pair("scalar_const", k, v, np.array([gamma]))
    assert abs(float(np.asarray(T).reshape(-1)[0]) / gamma ** L - 1.0) < 1e-13
    w = gamma ** (L - 1 - np.arange(L))
    assert rel(S, np.einsum("t,ti,tj->ij", w, k, v)) < 1e-13
    a = rng.uniform(0.5, 1.0, L)
    T, S = orc.segment_pair("scalar", k, v, a)
    assert abs(float(np.asarray(T).reshape(-1)[0]) / np.exp(np.sum(np.log(a))) - 1.0) < 1e-12
    suffix = np.exp(np.concatenate([np.cumsum(np.log(a)[::-1])[::-1][1:], [0.0]]))
    assert rel(S, np.einsum("t,ti,tj->ij", suffix, k, v)) < 1e-12


def pin_diag_closed_form(orc):
    rng = np.random.default_rng(16)
    dk, dv, L = 5, 4, 50
    k, _, v, alpha, _ = rand_inputs(rng, "diag", L, dk, dv, gate_div=16.0)
    T, S = orc.segment_pair("diag", k, v, alpha)
    assert rel(T, np.exp(np.sum(np.log(alpha), axis=0))) < 1e-13
    ref = np.zeros((dk, dv))
    for t in range(L):
        decay = np.exp(np.sum(np.log(alpha[t + 1:]), axis=0)) if t + 1 < L else np.ones(dk)
        ref += (decay * k[t])[:, None] * v[t][None, :]
    assert rel(S, ref) < 1e-12


def pin_dense_bruteforce(orc):
    rng = np.random.default_rng(17)
    for fam in FAMS:
        for (dk, dv, L) in [(3, 4, 6), (4, 2, 8), (2, 3, 1), (3, 3, 0)]:
            k, q, v, alpha, beta = rand_inputs(rng, fam, L, dk, dv)
            T, S = orc.segment_pair(fam, k, v, alpha, beta)
            Tb, Sb = brute_pair(fam, k, v, alpha, beta)
            assert rel(as_dense_T(fam, T, dk), Tb) < 1e-12
            if L > 0:
                assert rel(S, Sb) < 1e-12
            else:
                assert np.all(S == 0)
            S0 = rng.standard_normal((dk, dv))
            Sr, o = orc.run(fam, k, v, alpha, beta, q=q, S0=S0)
            ob, Sbend = brute_outputs(fam, k, v, q, alpha, beta, S0)
            assert rel(Sr, Sbend) < 1e-12
            if L > 0:
                assert rel(o, ob) < 1e-12


def pin_special_cases(orc):
    rng = np.random.default_rng(18)
    dk, dv, L = 6, 6, 20
    k, q, v, alpha, beta = rand_inputs(rng, "gated_delta", L, dk, dv)
    # beta = 0: GDN reduces to a_t I with no writes (Table 1, Mamba2 row with zero writes).
    T, S = orc.segment_pair("gated_delta", k, v, alpha, np.zeros(L))
    assert rel(T, np.prod(alpha) * np.eye(dk)) < 1e-13
    assert np.all(S == 0)
    # a = 1: GDN reduces to DeltaNet (Table 1).
    T1, S1 = orc.segment_pair("gated_delta", k, v, np.ones(L), beta)
    T2, S2 = orc.segment_pair("delta", k, v, None, beta)
    assert rel(T1, T2) < 1e-14 and rel(S1, S2) < 1e-14
    # beta = 1, ||k|| = 1: I - k k^T is a projector, a repeated erase changes nothing.
    kk = np.stack([k[0], k[0]])
    Ta = orc.transition("delta", kk[:1], None, np.ones(1))
    Tb = orc.transition("delta", kk, None, np.ones(2))
    assert rel(Ta, Tb) < 1e-13
    assert rel(Ta, np.eye(dk) - np.outer(k[0], k[0])) < 1e-13
    # KDA (Table 1): beta = 0 leaves the per-channel decay of GLA with no writes; g = 1 is
    # DeltaNet; a per-token gate repeated over the channels, g_t = a_t 1, is GDN.
    g = np.exp(-_softplus(rng.standard_normal((L, dk))) / 8.0)
    T, S = orc.segment_pair("kda", k, v, g, np.zeros(L))
    assert rel(T, np.diag(np.prod(g, axis=0))) < 1e-13
    assert np.all(S == 0)
    T1, S1 = orc.segment_pair("kda", k, v, np.ones((L, dk)), beta)
    assert rel(T1, T2) < 1e-14 and rel(S1, S2) < 1e-14
    T3, S3 = orc.segment_pair("kda", k, v, np.repeat(alpha[:, None], dk, axis=1), beta)
    T4, S4 = orc.segment_pair("gated_delta", k, v, alpha, beta)
    assert rel(T3, T4) < 1e-13 and rel(S3, S4) < 1e-13


def pin_spectral_bound(orc):
    rng = np.random.default_rng(19)
    for _ in range(5):
        dk, L = 7, 40
        k, _, v, alpha, beta = rand_inputs(rng, "gated_delta", L, dk, dk)
        T = orc.transition("gated_delta", k, alpha, beta)
        assert np.linalg.norm(T, 2) <= np.prod(alpha) * (1 + 1e-12)
        T = orc.transition("delta", k, None, beta)
        assert np.linalg.norm(T, 2) <= 1 + 1e-12


def pin_affine_scan(orc):
    rng = np.random.default_rng(20)
    for fam in FAMS:
        dk, dv = 4, 3
        lens = [5, 0, 3, 9, 1]
        L = sum(lens)
        k, _, v, alpha, beta = rand_inputs(rng, fam, L, dk, dv)
        Ts, Ss, off = [], [], 0
        for n_ in lens:
            a_, b_ = slice_gates(fam, alpha, beta, off, off + n_)
            T, S = orc.segment_pair(fam, k[off:off + n_], v[off:off + n_], a_, b_)
            Ts.append(np.asarray(T).reshape(-1))
            Ss.append(S)
            off += n_
        Tp, Sp = orc.affine_scan(fam, np.stack(Ts), np.stack(Ss))
        off = 0
        for i, n_ in enumerate(lens):
            off += n_
            a_, b_ = slice_gates(fam, alpha, beta, 0, off)
            Tr, Sr = orc.segment_pair(fam, k[:off], v[:off], a_, b_)
            assert rel(as_dense_T(fam, np.asarray(Tp[i]), dk), as_dense_T(fam, Tr, dk)) < 1e-12
            if off > 0:
                assert rel(Sp[i], Sr) < 1e-12


PINS = [pin_worked_example, pin_table2, pin_composition_law, pin_eq6, pin_assoc_noncommut,
        pin_identity_reduction, pin_scalar_closed_form, pin_diag_closed_form, pin_dense_bruteforce,
        pin_special_cases, pin_spectral_bound, pin_affine_scan]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(O.default())


# Mutations of the oracle source: each is a plausible mistake that some pin must catch.
MUTANTS = {
    "write_without_beta": ("TS + (with_write ? b * k[i] * v[j] : 0.0)", "TS + (with_write ? k[i] * v[j] : 0.0)"),
    "erase_sign_flipped": ("a * (S[i * dv + j] - b * k[i] * tmp[j])", "a * (S[i * dv + j] + b * k[i] * tmp[j])"),
    "gate_decays_write": ("TS + (with_write ? b * k[i] * v[j] : 0.0)", "TS + (with_write ? a * b * k[i] * v[j] : 0.0)"),
    "transposed_T_apply": ("acc += T[i * dk + l] * X[l * ncol + j]", "acc += T[l * dk + i] * X[l * ncol + j]"),
    "compose_order_swapped": ("mul_T(fam, dk, T2, T1, T3);", "mul_T(fam, dk, T1, T2, T3);"),
    "diag_gate_off_by_one": ("const double *g = alpha + t * dk;", "const double *g = alpha + (t > 0 ? t - 1 : 0) * dk;",
                             2),
    "transition_drops_token": ("for (t = 0; t < len; t++) p *= gate_scalar", "for (t = 1; t < len; t++) p *= gate_scalar"),
    "output_reads_k": ("acc += q[t * dk + i] * S[i * dv + j];", "acc += k[t * dk + i] * S[i * dv + j];"),
    "erase_uses_v": ("for (i = 0; i < dk; i++) acc += k[i] * S[i * dv + j];",
                     "for (i = 0; i < dk; i++) acc += (v ? v[i % dv] : k[i]) * S[i * dv + j];", 2),
    "kda_gate_on_value_index": ("for (j = 0; j < dv; j++) S[i * dv + j] *= g[i];",
                                "for (j = 0; j < dv; j++) S[i * dv + j] *= g[j % dk];"),
    "kda_erase_sign_flipped": ("S[i * dv + j] - b * k[i] * tmp[j] + (with_write", "S[i * dv + j] + b * k[i] * tmp[j] + (with_write"),
    "kda_gate_decays_write": ("+ (with_write ? b * k[i] * v[j] : 0.0);\n        return;",
                              "+ (with_write ? g[i] * b * k[i] * v[j] : 0.0);\n        return;"),
    "compose_drops_addend": ("S[i] = Y[i] + S0[(size_t)j * dk * dv + i];", "S[i] = Y[i];"),
}


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(name, tmp_path):
    src = open(os.path.join(os.path.dirname(O.__file__), "hypic_oracle.c")).read()
    old, new, count = (MUTANTS[name] + (1,))[:3]
    assert src.count(old) == count, f"mutation anchor for {name} not found exactly {count} times"
    path_c = tmp_path / "mutant.c"
    path_so = tmp_path / "mutant.so"
    path_c.write_text(src.replace(old, new))
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", str(path_so), str(path_c), "-lm"])
    mutant = O.Oracle(str(path_so))
    caught = []
    for pin in PINS:
        try:
            pin(mutant)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name}"
