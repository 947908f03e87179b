"""Pins for the CPU oracle: checks against facts fixed by the pages and by mathematics.

Every check takes an ``OracleLib`` so the same checks can be run on deliberately broken copies
of the oracle (``test_oracle_mutants.py``): each plausible mistake must fail at least one pin.

Pins (none of them re-types the recurrence loop):
  golden       hand-derived values of the recurrence definition (tests/golden/)
  quadratic    the semiseparable matrix form y = M x, M_ij = C_i^T Abar_{i:j} Bbar_j
               (youngju.dev Mamba article, "State Space Dualityの発見")
  a_zero       A = 0, N = 1, B = C = 1: the scan is a causal running sum,
               y = cumsum(dt x) + D x (SSM with trivial decay = causal linear attention,
               Qiita Mamba-2 article section 3.3)
  reset        huge dt: exp(dt A) underflows to 0 and the state restarts from Bbar_t x_t
               (youngju.dev article: large Delta resets the previous state)
  dt_zero      dt = 0 tokens leave the state unchanged (youngju.dev article, debugging
               checklist: padding tokens get Delta = 0 to block the state update)
  b_zero       B = 0: only the initial state, decayed, and the skip term remain
  retnet       constant decay gamma = exp(dt A): the output matrix is RetNet's D_ij = gamma^(i-j)
               (waylandz.com LLM book ch. 32, section 32.6.2)
  linearity    y is linear in (x, h0) jointly
  split        scan(0..L) = scan(0..L1) then scan(L1..L) with initial_state = final_state
               (youngju.dev article, "状態初期化とシーケンス境界": the state carries across calls)
  groups       G = H with B/C copied per head equals G < H (group sharing is only sharing)
  chunked      the chunk algorithm equals the recurrence at every chunk size, ragged tails too
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "hand_recurrence.json")


def _rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = max(float(np.max(np.abs(b))) if b.size else 0.0, 1e-300)
    return float(np.max(np.abs(a - b))) / den if a.size else 0.0


def _rand_inputs(rng, b=2, L=29, H=4, G=2, P=3, N=5, with_h0=True, with_D=True):
    x = rng.standard_normal((b, L, H, P))
    dt = np.log1p(np.exp(rng.standard_normal((b, L, H)) * 0.7 - 2.0))   # positive, softplus-like
    A = -np.exp(rng.uniform(0.0, math.log(16.0), H))
    B = rng.standard_normal((b, L, G, N)) / math.sqrt(N)
    C = rng.standard_normal((b, L, G, N)) / math.sqrt(N)
    D = rng.uniform(0.5, 1.5, H) if with_D else None
    h0 = rng.standard_normal((b, H, P, N)) * 0.3 if with_h0 else None
    return x, dt, A, B, C, D, h0


def pin_golden(lib):
    data = json.load(open(GOLDEN))
    for case in data["cases"]:
        x = np.array(case["x"])[None]
        dt = np.array(case["dt"])[None]
        B = np.array(case["B"])[None]
        C = np.array(case["C"])[None]
        h0 = np.array(case["h0"])[None]
        y, hT, _ = lib.scan_problems(x, dt, np.array([case["A"]]), B, C,
                                     np.array([case["D"]]), h0)
        assert _rel(y[0], case["y"]) <= 1e-14, (case["name"], y[0], case["y"])
        assert _rel(hT[0], case["final_state"]) <= 1e-14, (case["name"], hT[0])


def pin_quadratic(lib):
    rng = np.random.default_rng(11)
    for kw in (dict(), dict(with_h0=False, with_D=False), dict(L=1), dict(G=4, P=2, N=7, L=40)):
        x, dt, A, B, C, D, h0 = _rand_inputs(rng, **kw)
        y1, h1 = oracle.scan(x, dt, A, B, C, D, h0, lib=lib)
        y2, h2 = oracle.quadratic(x, dt, A, B, C, D, h0)
        assert _rel(y1, y2) <= 1e-12, ("quadratic y", _rel(y1, y2))
        assert _rel(h1, h2) <= 1e-12, ("quadratic final", _rel(h1, h2))


def pin_a_zero(lib):
    rng = np.random.default_rng(12)
    n, L, P = 3, 50, 4
    x = rng.standard_normal((n, L, P))
    dt = rng.uniform(0.0, 1.0, (n, L))
    D = rng.uniform(0.5, 1.5, n)
    ones = np.ones((n, L, 1))
    y, hT, _ = lib.scan_problems(x, dt, np.zeros(n), ones, ones, D, None)
    ref = np.cumsum(dt[:, :, None] * x, axis=1) + D[:, None, None] * x
    assert _rel(y, ref) <= 1e-13, ("A=0 running sum", _rel(y, ref))
    assert _rel(hT[:, :, 0], np.sum(dt[:, :, None] * x, axis=1)) <= 1e-13


def pin_reset(lib):
    rng = np.random.default_rng(13)
    n, L, P, N = 2, 17, 3, 6
    x = rng.standard_normal((n, L, P))
    dt = np.full((n, L), 1.0e3)
    A = np.array([-1.0, -4.0])
    B = rng.standard_normal((n, L, N))
    C = rng.standard_normal((n, L, N))
    D = np.array([0.75, 1.25])
    h0 = rng.standard_normal((n, P, N))
    y, hT, _ = lib.scan_problems(x, dt, A, B, C, D, h0)
    cb = np.einsum("itn,itn->it", C, B)
    ref = dt[:, :, None] * cb[:, :, None] * x + D[:, None, None] * x
    assert _rel(y, ref) <= 1e-13, ("reset", _rel(y, ref))
    ref_h = dt[:, -1, None, None] * x[:, -1, :, None] * B[:, -1, None, :]
    assert _rel(hT, ref_h) <= 1e-13


def pin_dt_zero(lib):
    rng = np.random.default_rng(14)
    x, dt, A, B, C, D, h0 = _rand_inputs(rng, b=1, L=30, H=2, G=1)
    dt[:, 10:20, :] = 0.0
    y_a, h_a = oracle.scan(x[:, :10], dt[:, :10], A, B[:, :10], C[:, :10], D, h0, lib=lib)
    y_b, h_b = oracle.scan(x[:, :20], dt[:, :20], A, B[:, :20], C[:, :20], D, h0, lib=lib)
    assert np.array_equal(h_a, h_b), "dt=0 tokens changed the state"
    # outputs on the frozen tokens read the frozen state
    g = C[:, 10:20, 0, :]                                   # [1, 10, N]
    ref = np.einsum("btn,bhpn->bthp", g, h_a) + D[None, None, :, None] * x[:, 10:20]
    assert _rel(y_b[:, 10:20], ref) <= 1e-13, ("dt=0 outputs", _rel(y_b[:, 10:20], ref))


def pin_b_zero(lib):
    rng = np.random.default_rng(15)
    x, dt, A, B, C, D, h0 = _rand_inputs(rng, b=2, L=23, H=3, G=1)
    B[:] = 0.0
    y, hT = oracle.scan(x, dt, A, B, C, D, h0, lib=lib)
    cum = np.cumsum(dt, axis=1) * A[None, None, :]          # [b, L, H]
    ch0 = np.einsum("btn,bhpn->bthp", C[:, :, 0, :], h0)    # C_t . h0
    ref = np.exp(cum)[..., None] * ch0 + D[None, None, :, None] * x
    assert _rel(y, ref) <= 1e-12, ("B=0", _rel(y, ref))
    ref_h = np.exp(cum[:, -1])[:, :, None, None] * h0
    assert _rel(hT, ref_h) <= 1e-12


def pin_retnet(lib):
    rng = np.random.default_rng(16)
    n, L, P = 2, 31, 3
    gamma = np.array([0.9, 0.5])
    x = rng.standard_normal((n, L, P))
    ones = np.ones((n, L, 1))
    y, _, _ = lib.scan_problems(x, np.ones((n, L)), np.log(gamma), ones, ones, np.zeros(n), None)
    i = np.arange(L)[:, None]
    j = np.arange(L)[None, :]
    for k in range(n):
        Dm = np.where(i >= j, np.power(gamma[k], np.maximum(i - j, 0)), 0.0)   # gamma^(i-j)
        assert _rel(y[k], Dm @ x[k]) <= 1e-12, ("retnet", k)


def pin_linearity(lib):
    rng = np.random.default_rng(17)
    x, dt, A, B, C, D, h0 = _rand_inputs(rng)
    x2 = rng.standard_normal(x.shape)
    h02 = rng.standard_normal(h0.shape)
    a = -2.5
    y1, f1 = oracle.scan(x, dt, A, B, C, D, h0, lib=lib)
    ya, fa = oracle.scan(a * x, dt, A, B, C, D, a * h0, lib=lib)
    assert _rel(ya, a * y1) <= 1e-12 and _rel(fa, a * f1) <= 1e-12, "homogeneity"
    y2, f2 = oracle.scan(x2, dt, A, B, C, D, h02, lib=lib)
    ys, fs = oracle.scan(x + x2, dt, A, B, C, D, h0 + h02, lib=lib)
    assert _rel(ys, y1 + y2) <= 1e-12 and _rel(fs, f1 + f2) <= 1e-12, "superposition"


def pin_split(lib):
    rng = np.random.default_rng(18)
    x, dt, A, B, C, D, h0 = _rand_inputs(rng, L=40)
    y, hT = oracle.scan(x, dt, A, B, C, D, h0, lib=lib)
    for L1 in (1, 17, 39):
        ya, ha = oracle.scan(x[:, :L1], dt[:, :L1], A, B[:, :L1], C[:, :L1], D, h0, lib=lib)
        yb, hb = oracle.scan(x[:, L1:], dt[:, L1:], A, B[:, L1:], C[:, L1:], D, ha, lib=lib)
        assert _rel(np.concatenate([ya, yb], axis=1), y) <= 1e-12, ("split y", L1)
        assert _rel(hb, hT) <= 1e-12, ("split final", L1)


def pin_groups(lib):
    rng = np.random.default_rng(19)
    x, dt, A, B, C, D, h0 = _rand_inputs(rng, H=6, G=2)
    y, hT = oracle.scan(x, dt, A, B, C, D, h0, lib=lib)
    rep = np.repeat(np.arange(2), 3)            # head h -> group h // 3
    y2, h2 = oracle.scan(x, dt, A, B[:, :, rep], C[:, :, rep], D, h0, lib=lib)
    assert np.array_equal(y, y2) and np.array_equal(hT, h2), "group sharing"
    # and the group really matters: another mapping gives another answer
    y3, _ = oracle.scan(x, dt, A, B[:, :, rep[::-1]], C[:, :, rep[::-1]], D, h0, lib=lib)
    assert _rel(y3, y) > 1e-3, "group mapping has no effect"


def pin_chunked(lib):
    rng = np.random.default_rng(20)
    x, dt, A, B, C, D, h0 = _rand_inputs(rng, L=70, G=1, H=2)
    y, hT = oracle.scan(x, dt, A, B, C, D, h0, lib=lib)
    for Q in (1, 4, 16, 23, 64, 70, 128):
        yc, hc = oracle.chunked(x, dt, A, B, C, D, h0, chunk_size=Q)
        assert _rel(yc, y) <= 1e-12, ("chunked y", Q, _rel(yc, y))
        assert _rel(hc, hT) <= 1e-12, ("chunked final", Q)


ALL_PINS = [pin_golden, pin_quadratic, pin_a_zero, pin_reset, pin_dt_zero, pin_b_zero,
            pin_retnet, pin_linearity, pin_split, pin_groups, pin_chunked]
