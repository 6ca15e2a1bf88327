"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle (``oracle/sd_oracle.cpp``) against something
other than itself: values the pages print for a worked example, closed
forms, the losslessness property (exact enumeration and a chi-square test),
library routines for special cases, brute force on tiny inputs, and a
second, independent Philox implementation plus published known-answer
vectors.
"""
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden")


def _softmax64(l, T):
    l = np.asarray(l, dtype=np.float64)
    z = l / T
    z = z - z.max()
    e = np.exp(z)
    return e / e.sum()


def _parse_golden(name):
    d = {}
    for line in open(os.path.join(GOLDEN, name), encoding="utf-8"):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, v = line.split(":", 1)
        d[k.strip()] = v.split()
    return d


# ------------------------------------------------------------- worked example
def _worked_example_inputs():
    g = _parse_golden("worked_example_greedy.txt")
    vocab = g["vocab"]
    V = 16                      # the page's words plus unused filler ids
    ids = {w: i for i, w in enumerate(vocab)}
    draft = [ids[w] for w in g["draft"]]
    top = [ids[w] for w in g["target_top"]]
    K = len(draft)
    target = np.zeros((K + 1, V), np.float32)
    rng = np.random.default_rng(7)
    target[:] = rng.integers(-8, 8, size=target.shape) / 8.0
    for j, t in enumerate(top):
        target[j, t] = 6.0
    target[K, V - 1] = 6.0       # the unshown bonus row: any peak will do
    draftl = np.zeros((K, V), np.float32)
    for j, t in enumerate(draft):
        draftl[j, t] = 6.0
    return g, ids, target, draftl, np.array(draft, np.int32)


def test_worked_example_greedy(oracle_lib):
    g, ids, target, draftl, tokens = _worked_example_inputs()
    K = tokens.size
    r = oracle_lib.verify_row_u(target, draftl, tokens, 0.0, np.full(K, 0.5), np.full(K + 1, 0.5))
    assert r["n_acc"] == int(g["expect_n_accepted"][0])
    assert r["tau"] == int(g["expect_tau"][0])
    assert r["out_tokens"][r["n_acc"]] == ids[g["expect_token"][0]]
    b = oracle_lib.verify(target[None], draftl[None], tokens[None], [0.0], seed=1)
    offsets, packed = oracle_lib.compact(b["out_tokens"], b["tau"])
    assert list(packed) == [ids[w] for w in g["expect_packed"]]
    assert list(offsets) == [0, int(g["expect_tau"][0])]


def test_bonus_when_all_greedy_drafts_match(oracle_lib):
    rng = np.random.default_rng(3)
    K, V = 5, 40
    target = rng.normal(size=(K + 1, V)).astype(np.float32)
    tokens = target[:K].argmax(-1).astype(np.int32)
    r = oracle_lib.verify_row_u(target, np.zeros((K, V), np.float32), tokens, 0.0,
                                np.full(K, 0.5), np.full(K + 1, 0.5))
    assert r["tau"] == K + 1 and r["n_acc"] == K
    assert list(r["out_tokens"][:K]) == list(tokens)
    assert r["out_tokens"][K] == int(target[K].argmax())


def test_greedy_argmax_ties_match_torch_first_occurrence(oracle_lib):
    # torch.argmax documents that it returns the first maximal index.
    rng = np.random.default_rng(11)
    K, V = 3, 64
    target = rng.integers(0, 4, size=(K + 1, V)).astype(np.float32)   # many ties
    amax = torch.argmax(torch.from_numpy(target), dim=-1).numpy()
    tokens = amax[:K].astype(np.int32).copy()
    tokens[2] = (tokens[2] + 1) % V
    r = oracle_lib.verify_row_u(target, np.zeros((K, V), np.float32), tokens, 0.0,
                                np.full(K, 0.5), np.full(K + 1, 0.5))
    assert list(r["argmax"]) == list(amax)
    assert r["n_acc"] == 2 and r["out_tokens"][2] == amax[2]


# ------------------------------------------------------- exact enumeration ----
def _slot_breakpoints(f, G=1024):
    """Breakpoints in (0,1] of a piecewise-constant black-box f(u)."""
    us = (np.arange(G) + 0.5) / G
    vals = [f(u) for u in us]
    bps = []
    for i in range(G - 1):
        if vals[i] != vals[i + 1]:
            lo, hi, vlo = us[i], us[i + 1], vals[i]
            for _ in range(64):
                mid = 0.5 * (lo + hi)
                if mid <= lo or mid >= hi:
                    break
                if f(mid) == vlo:
                    lo = mid
                else:
                    hi = mid
            bps.append(hi)
    return sorted(set(bps))


def _enumerate_law(oracle_lib, target, draft, tokens, T):
    """Exact law of the oracle's output over its uniforms for one draft
    sequence: every slot's breakpoints are found by bisection on the
    oracle itself, then the oracle is evaluated at the midpoint of every
    cell of the product partition and weighted by the cell's volume."""
    K = tokens.size
    tiny = 1e-300

    def run(ua, us):
        r = oracle_lib.verify_row_u(target, draft, tokens, T, ua, us)
        return tuple(r["out_tokens"][: r["tau"]])

    # settings that make each slot matter (others fixed)
    base_a = [0.5] * K
    base_s = [0.5] * (K + 1)
    parts_a, parts_s = [], []
    for j in range(K):
        def fa(u, j=j):
            ua = [tiny] * K
            ua[j] = u
            return run(ua, base_s)
        parts_a.append(_slot_breakpoints(fa))
    for j in range(K + 1):
        def fs(u, j=j):
            ua = [tiny] * K
            if j < K:
                ua[j] = 1.0
            us = list(base_s)
            us[j] = u
            return run(ua, us)
        parts_s.append(_slot_breakpoints(fs))

    def cells(bps):
        edges = [0.0] + list(bps) + [1.0]
        return [(0.5 * (a + b), b - a) for a, b in zip(edges[:-1], edges[1:]) if b > a]

    law = {}
    grids = [cells(b) for b in parts_a] + [cells(b) for b in parts_s]

    def rec(i, point, w):
        if i == len(grids):
            out = run(point[:K], point[K:])
            law[out] = law.get(out, 0.0) + w
            return
        for mid, length in grids[i]:
            rec(i + 1, point + [mid], w * length)

    rec(0, [], 1.0)
    return law


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_losslessness_exact_enumeration_V4_K2(oracle_lib, T):
    """[SD] FAQ / [D3D] 検証のまとめ: the emitted tokens follow exactly the
    target-only distribution.  Context-dependent toy target and draft
    (V=4, K=2); draft sequences enumerated with their draft probabilities."""
    V, K = 4, 2
    rng = np.random.default_rng(2024)
    q16 = lambda shape: (rng.integers(-24, 25, size=shape) / 16.0).astype(np.float32)
    a0 = q16(V)                 # target, first position
    a1 = q16((V, V))            # target second position given x0
    a2 = q16((V, V, V))         # target bonus position given x0, x1
    b0 = q16(V)                 # draft first position
    b1 = q16((V, V))            # draft second position given d0
    p0 = _softmax64(a0, T)
    p1 = np.stack([_softmax64(a1[x], T) for x in range(V)])
    p2 = np.stack([[_softmax64(a2[x, y], T) for y in range(V)] for x in range(V)])
    q0 = _softmax64(b0, T)
    q1 = np.stack([_softmax64(b1[x], T) for x in range(V)])

    law = {}
    reject0 = 0.0
    for d0 in range(V):
        for d1 in range(V):
            wd = q0[d0] * q1[d0, d1]
            target = np.stack([a0, a1[d0], a2[d0, d1]]).astype(np.float32)
            draft = np.stack([b0, b1[d0]]).astype(np.float32)
            sub = _enumerate_law(oracle_lib, target, draft, np.array([d0, d1], np.int32), T)
            for out, w in sub.items():
                law[out] = law.get(out, 0.0) + wd * w
                if len(out) == 1:
                    reject0 += wd * w
    total = sum(law.values())
    assert abs(total - 1.0) < 1e-12
    # first emitted token ~ p0
    m0 = np.zeros(V)
    for out, w in law.items():
        m0[out[0]] += w
    np.testing.assert_allclose(m0, p0, rtol=0, atol=1e-12)
    # second token given the first was an accepted draft ~ p1(.|x0)
    for x0 in range(V):
        m1 = np.zeros(V)
        for out, w in law.items():
            if len(out) >= 2 and out[0] == x0:
                m1[out[1]] += w
        if m1.sum() > 1e-9:
            np.testing.assert_allclose(m1 / m1.sum(), p1[x0], rtol=0, atol=1e-10)
    # bonus token given both drafts accepted ~ p2(.|x0, x1)
    for x0 in range(V):
        for x1 in range(V):
            m2 = np.zeros(V)
            for out, w in law.items():
                if len(out) == 3 and out[0] == x0 and out[1] == x1:
                    m2[out[2]] += w
            if m2.sum() > 1e-9:
                np.testing.assert_allclose(m2 / m2.sum(), p2[x0, x1], rtol=0, atol=1e-9)
    # closed form: the first draft is rejected with probability 1 - sum min(p0, q0)
    assert abs(reject0 - (1.0 - np.minimum(p0, q0).sum())) < 1e-12


def test_identical_models_accept_everything(oracle_lib):
    """p == q gives acceptance probability sum min(p,q) = 1: tau = K + 1."""
    rng = np.random.default_rng(5)
    K, V = 4, 50
    target = rng.normal(size=(K + 1, V)).astype(np.float32)
    draft = target[:K].copy()
    for trial in range(20):
        tokens = rng.integers(0, V, size=K).astype(np.int32)
        ua = rng.uniform(1e-9, 1.0, size=K)
        us = rng.uniform(1e-9, 1.0, size=K + 1)
        r = oracle_lib.verify_row_u(target, draft, tokens, 0.9, ua, us)
        assert r["tau"] == K + 1
        np.testing.assert_allclose(r["ratio"], 1.0, rtol=1e-12)


# --------------------------------------------------------------- chi-square ----
@pytest.mark.slow
def test_chi_square_V8_one_million_rounds(oracle_lib):
    """Monte-Carlo losslessness through the Philox path: 10^6 rounds at V=8,
    K=2, each token position tested against the target law (df = 7)."""
    from scipy.stats import chisquare
    V, K, T = 8, 2, 1.0
    rng = np.random.default_rng(99)
    a = rng.normal(scale=1.5, size=(K + 1, V)).astype(np.float32)
    b = (a[:K] + rng.normal(scale=0.8, size=(K, V))).astype(np.float32)
    p = np.stack([_softmax64(a[j], T) for j in range(K + 1)])
    q = np.stack([_softmax64(b[j], T) for j in range(K)])
    counts = [np.zeros(V) for _ in range(K + 1)]
    acc0 = 0
    n_total = 0
    rejected_equals_draft = 0
    for chunk in range(4):
        n = 250_000
        tokens = np.stack([rng.choice(V, size=n, p=q[j]) for j in range(K)], axis=1).astype(np.int32)
        target = np.broadcast_to(a, (n, K + 1, V))
        draft = np.broadcast_to(b, (n, K, V))
        r = oracle_lib.verify(target, draft, tokens, np.full(n, T, np.float32),
                              seed=0xC0FFEE + chunk)
        out, tau = r["out_tokens"], r["tau"]
        for t in range(K + 1):
            sel = tau >= t + 1
            counts[t] += np.bincount(out[sel, t], minlength=V)
        acc0 += int((r["num_accepted"] >= 1).sum())
        n_total += n
        rej = r["num_accepted"] < K
        idx = np.nonzero(rej)[0]
        rejected_equals_draft += int((out[idx, r["num_accepted"][idx]] ==
                                      tokens[idx, r["num_accepted"][idx]]).sum())
    for t in range(K + 1):
        c = counts[t]
        stat, pval = chisquare(c, c.sum() * p[t])
        assert pval > 1e-3, (t, pval, c / c.sum(), p[t])
    beta = np.minimum(p[0], q[0]).sum()
    sd = np.sqrt(beta * (1 - beta) / n_total)
    assert abs(acc0 / n_total - beta) < 5 * sd
    # a rejected draft token carries no residual mass, so it is never the correction
    assert rejected_equals_draft == 0


# ----------------------------------------------------- library special cases ----
def test_probabilities_match_torch_softmax_float64(oracle_lib):
    rng = np.random.default_rng(17)
    B, K, V = 3, 3, 333
    target = (rng.normal(size=(B, K + 1, V)) * 3).astype(np.float32)
    draft = (target[:, :K] + rng.normal(size=(B, K, V))).astype(np.float32)
    tokens = rng.integers(0, V, size=(B, K)).astype(np.int32)
    temps = np.array([0.7, 1.0, 1.3], np.float32)
    r = oracle_lib.verify(target, draft, tokens, temps, seed=3, stats=True)
    for b in range(B):
        T = float(temps[b])
        pt = torch.softmax(torch.from_numpy(target[b]).double() / T, dim=-1).numpy()
        qt = torch.softmax(torch.from_numpy(draft[b]).double() / T, dim=-1).numpy()
        for j in range(K):
            np.testing.assert_allclose(r["p_tok"][b, j], pt[j, tokens[b, j]], rtol=1e-12)
            np.testing.assert_allclose(r["q_tok"][b, j], qt[j, tokens[b, j]], rtol=1e-12)
        lse = torch.logsumexp(torch.from_numpy(target[b]).double() / T, dim=-1).numpy()
        np.testing.assert_allclose(r["Zt"][b], np.exp(lse - target[b].max(-1).astype(np.float64) / T),
                                   rtol=1e-12)


def test_bf16_inputs_are_widened_exactly(oracle_lib):
    rng = np.random.default_rng(23)
    B, K, V = 2, 2, 100
    t32 = torch.from_numpy((rng.normal(size=(B, K + 1, V)) * 2).astype(np.float32))
    d32 = torch.from_numpy((rng.normal(size=(B, K, V)) * 2).astype(np.float32))
    tb, db = t32.to(torch.bfloat16), d32.to(torch.bfloat16)
    bits = lambda x: x.view(torch.int16).numpy().view(np.uint16)
    tokens = rng.integers(0, V, size=(B, K)).astype(np.int32)
    temps = np.array([0.8, 0.0], np.float32)
    r1 = oracle_lib.verify(bits(tb), bits(db), tokens, temps, seed=9, stats=True)
    r2 = oracle_lib.verify(tb.float().numpy(), db.float().numpy(), tokens, temps, seed=9, stats=True)
    for k in ("out_tokens", "tau", "num_accepted", "argmax"):
        np.testing.assert_array_equal(r1[k], r2[k])
    np.testing.assert_array_equal(r1["ratio"][0], r2["ratio"][0])


# ----------------------------------------------------------------- top-F keys ----
def _brute_keys(draft, tokens, fanout, bonus=None):
    B, K, V = draft.shape
    n = int(sum(fanout))
    keys = np.full((B, n, 2), -1, np.int32)
    for b in range(B):
        s = 0
        for k in range(K + 1):
            if k < K:
                row, excl = torch.from_numpy(draft[b, k].astype(np.float64)), int(tokens[b, k])
            elif bonus is not None:
                row, excl = torch.from_numpy(bonus[b].astype(np.float64)), -1
            else:
                s += fanout[k]
                continue
            vals, idx = torch.sort(row, descending=True, stable=True)
            cand = [int(i) for v, i in zip(vals.tolist(), idx.tolist())
                    if i != excl and v != -np.inf]
            for f in range(fanout[k]):
                if f < len(cand):
                    keys[b, s] = (k, cand[f])
                s += 1
    return keys


def test_outcome_keys_match_stable_sort_brute_force(oracle_lib):
    rng = np.random.default_rng(31)
    B, K, V = 4, 6, 97
    draft = rng.integers(-6, 6, size=(B, K, V)).astype(np.float32)   # many ties
    draft[0, 1, :90] = -np.inf                                         # few candidates
    bonus = rng.integers(-6, 6, size=(B, V)).astype(np.float32)
    tokens = rng.integers(0, V, size=(B, K)).astype(np.int32)
    fanout = [4, 3, 2, 1, 1, 1, 1]
    keys = oracle_lib.outcome_predict(draft, tokens, fanout, bonus)
    np.testing.assert_array_equal(keys, _brute_keys(draft, tokens, fanout, bonus))
    keys_nb = oracle_lib.outcome_predict(draft, tokens, fanout, None)
    np.testing.assert_array_equal(keys_nb, _brute_keys(draft, tokens, fanout, None))
    assert (keys_nb[:, -1] == -1).all()


def test_key_counts_from_d3d_preparation_table(oracle_lib):
    """[D3D] preparation table: 11x2 -> 384 tokens, 15x2 -> 512, 11x5 -> 912,
    i.e. positions*candidates + 1 keys, (keys + 1) blocks of 16 tokens."""
    K, V, B = 15, 64, 2
    rng = np.random.default_rng(41)
    draft = rng.normal(size=(B, K, V)).astype(np.float32)
    bonus = rng.normal(size=(B, V)).astype(np.float32)
    tokens = draft.argmax(-1).astype(np.int32)
    for line in open(os.path.join(GOLDEN, "d3d_prep_table.txt")):
        if line.startswith("#") or not line.strip():
            continue
        positions, cands, tokens_prepared = map(int, line.split())
        fanout = [cands] * positions + [0] * (K - positions) + [1]
        keys = oracle_lib.outcome_predict(draft, tokens, fanout, bonus)
        n_keys = keys.shape[1]
        assert (n_keys + 1) * 16 == tokens_prepared
        # greedy drafting: the drafter's own 2nd, 3rd, ... candidates
        for k in range(positions):
            order = np.argsort(-draft[0, k], kind="stable")
            assert list(keys[0, k * cands:(k + 1) * cands, 1]) == list(order[1:cands + 1])


def test_hit_test_brute_force(oracle_lib):
    rng = np.random.default_rng(43)
    B, K, V = 64, 6, 50
    target = rng.normal(scale=2, size=(B, K + 1, V)).astype(np.float32)
    draft = (target[:, :K] + rng.normal(size=(B, K, V))).astype(np.float32)
    bonus = (target[:, K] + rng.normal(size=(B, V))).astype(np.float32)
    tokens = draft.argmax(-1).astype(np.int32)
    fanout = [4, 3, 2, 1, 1, 1, 1]
    keys = oracle_lib.outcome_predict(draft, tokens, fanout, bonus)
    r = oracle_lib.verify(target, draft, tokens, np.full(B, 0.7, np.float32), seed=5, keys=keys)
    for b in range(B):
        m = r["num_accepted"][b]
        tok = r["out_tokens"][b, m]
        expect = any(keys[b, i, 0] == m and keys[b, i, 1] == tok for i in range(keys.shape[1]))
        assert bool(r["hit"][b]) == expect
    assert 0 < r["hit"].sum() < B


# ---------------------------------------------------------------- compaction ----
def test_compaction_brute_force(oracle_lib):
    rng = np.random.default_rng(47)
    B, K = 37, 5
    tau = rng.integers(0, K + 2, size=B).astype(np.int32)
    out = np.full((B, K + 1), -1, np.int32)
    for b in range(B):
        out[b, : tau[b]] = rng.integers(0, 1000, size=tau[b])
    offsets, packed = oracle_lib.compact(out, tau)
    exp = [int(x) for b in range(B) for x in out[b, : tau[b]]]
    assert list(packed) == exp
    assert offsets[0] == 0 and offsets[-1] == tau.sum()
    assert list(np.diff(offsets)) == list(tau)


# -------------------------------------------------------------- edge cases ----
def test_invalid_rows_and_degenerate_K0(oracle_lib):
    rng = np.random.default_rng(53)
    B, K, V = 4, 3, 20
    target = rng.normal(size=(B, K + 1, V)).astype(np.float32)
    draft = rng.normal(size=(B, K, V)).astype(np.float32)
    tokens = rng.integers(0, V, size=(B, K)).astype(np.int32)
    tokens[1, 2] = V            # out of range
    temps = np.array([1.0, 1.0, -0.5, np.nan], np.float32)
    r = oracle_lib.verify(target, draft, tokens, temps, seed=1)
    assert r["invalid_rows"] == 3
    assert list(r["tau"][1:]) == [0, 0, 0]
    assert (r["out_tokens"][1:] == -1).all()
    # K = 0: a plain sampling step from the single target row
    t0 = target[:, :1]
    r0 = oracle_lib.verify(t0, np.zeros((B, 0, V), np.float32), np.zeros((B, 0), np.int32),
                           np.array([0.0, 1.0, 1.0, 1.0], np.float32), seed=2)
    assert list(r0["tau"]) == [1, 1, 1, 1]
    assert r0["out_tokens"][0, 0] == int(t0[0, 0].argmax())


def test_guard_flags_decisions_near_a_boundary(oracle_lib):
    rng = np.random.default_rng(59)
    K, V = 2, 10
    target = rng.normal(size=(K + 1, V)).astype(np.float32)
    draft = rng.normal(size=(K, V)).astype(np.float32)
    tokens = np.array([0, 1], np.int32)
    base = oracle_lib.verify_row_u(target, draft, tokens, 1.0, [1e-9, 1e-9], [0.5] * 3)
    r0 = base["ratio"][0]
    assert r0 < 1     # the seed gives a rejectable first draft
    for du, flagged in ((5e-7, True), (-5e-7, True), (2e-6, False), (-2e-6, False),
                        (5e-5, False), (-5e-5, False)):
        r = oracle_lib.verify_row_u(target, draft, tokens, 1.0, [r0 + du, 1e-9], [0.5] * 3)
        # u - r within 1e-6 flags position 0; further away nothing is flagged
        # (the draw at u = 0.5 is far from every CDF edge of these rows)
        assert r["guard_pos"] == (0 if flagged else -1), (du, r["guard_pos"])


def _cdf_case():
    """Sequence of one draft whose first position is rejected and whose
    residual max(0, p - q) has three equal bins: target row 0 uniform over
    four tokens, draft row 0 twice as likely on token 0.  Returns the inputs
    and the residual's unnormalised weights computed here in float64 from
    the float32 logits (softmax written out with numpy)."""
    target = np.zeros((2, 4), np.float32)
    draft = np.zeros((1, 4), np.float32)
    draft[0, 0] = np.float32(np.log(2.0))
    tokens = np.array([0], np.int32)
    p = np.exp(target[0].astype(np.float64))
    p /= p.sum()
    q = np.exp(draft[0].astype(np.float64))
    q /= q.sum()
    w = np.maximum(0.0, p - q)
    return target, draft, tokens, w


def test_guard_flags_draws_near_a_cdf_edge(oracle_lib):
    # The inverse-CDF draw picks the smallest i with C_i > u S; the guard
    # flags it when u S lies within 1e-6 S of either edge of bin i, and when
    # rounding leaves u S at or past the total.  Residual weights here:
    # (0, w, w, w) with S = 3w ~ 0.15, edges at S/3 and 2S/3.
    target, draft, tokens, w = _cdf_case()
    S = w.sum()
    C = np.cumsum(w)
    assert w[0] == 0 and np.allclose(w[1:], w[1]) and 0.14 < S < 0.16
    # accept uniform 1 > p/q(d_0) = 0.25 / 0.4: position 0 is rejected
    for edge in (1, 2):               # bins 1 | 2 and 2 | 3
        for d, flagged in ((5e-7, True), (-5e-7, True), (3e-6, False), (-3e-6, False),
                           (5e-5, False), (-5e-5, False)):
            # u S placed d S away from the edge C[edge] (d in units of S)
            u = C[edge] / S + d
            r = oracle_lib.verify_row_u(target, draft, tokens, 1.0, [1.0], [u, 0.5])
            assert r["n_acc"] == 0 and r["tau"] == 1
            assert r["out_tokens"][0] == (edge + 1 if d > 0 else edge), (edge, d)
            assert r["guard_pos"] == (0 if flagged else -1), (edge, d, r["guard_pos"])
    # u S exactly on the total: no bin passes it, the last weighted token is
    # taken and the draw is flagged
    r = oracle_lib.verify_row_u(target, draft, tokens, 1.0, [1.0], [1.0, 0.5])
    assert r["out_tokens"][0] == 3 and r["guard_pos"] == 0
    # the window is relative to S: 5e-7 of an absolute unit is 3.3e-6 S, far
    r = oracle_lib.verify_row_u(target, draft, tokens, 1.0, [1.0], [C[1] / S + 5e-7 / S, 0.5])
    assert r["out_tokens"][0] == 2 and r["guard_pos"] == -1
    # bonus draw (all accepted): over p of the last row, four equal bins of
    # 1/4; u = 1/2 + 5e-7 is flagged, u = 1/2 + 5e-5 is not
    same = target[:1].copy()
    for du, flagged in ((5e-7, True), (5e-5, False)):
        r = oracle_lib.verify_row_u(target, same, tokens, 1.0, [1e-9], [0.5, 0.5 + du])
        assert r["n_acc"] == 1 and r["out_tokens"][1] == 2
        assert r["guard_pos"] == (1 if flagged else -1)


def _row_bad(row):
    """NaN or +inf anywhere, or nothing but -inf: the check's definition."""
    row = np.asarray(row, np.float64)
    return bool(np.isnan(row).any() or np.isposinf(row).any() or np.isneginf(row).all())


def test_finite_check_flags_exactly_the_rows_read(oracle_lib):
    # The optional finiteness check makes a sequence invalid when a row the
    # step reads for it holds NaN or +inf, or only -inf.  Rows read: the K+1
    # target rows; draft row j when the sequence is sampled or keys are built
    # at j; the bonus draft row when keys are built at K.  Brute force over
    # planted values, against a numpy restatement of that rule.
    rng = np.random.default_rng(123)
    B, K, V = 40, 3, 12
    target = rng.normal(size=(B, K + 1, V)).astype(np.float32)
    draft = rng.normal(size=(B, K, V)).astype(np.float32)
    bonus = rng.normal(size=(B, V)).astype(np.float32)
    tokens = rng.integers(0, V, size=(B, K)).astype(np.int32)
    temps = np.where(np.arange(B) % 2 == 0, 0.0, 0.8).astype(np.float32)
    fan = np.array([2, 0, 1, 1], np.int32)       # keys at positions 0, 2 and K
    planted = [np.nan, np.inf, "allneg", -np.inf]  # the last one alone is allowed
    for b in range(B):
        kind = planted[b % 4]
        where = (b // 4) % 3                     # 0 target, 1 draft, 2 bonus
        arr = target[b] if where == 0 else draft[b] if where == 1 else bonus[b:b + 1]
        r = rng.integers(0, arr.shape[0])
        if kind == "allneg":
            arr[r, :] = -np.inf
        else:
            arr[r, rng.integers(0, V)] = kind
    ref = oracle_lib.verify(target, draft, tokens, temps, seed=5, fanout=fan, draft_bonus=bonus,
                            check_finite=True)
    plain = oracle_lib.verify(target, draft, tokens, temps, seed=5)
    for b in range(B):
        rows = [target[b, j] for j in range(K + 1)]
        rows += [draft[b, j] for j in range(K) if temps[b] > 0 or fan[j] > 0]
        if fan[K] > 0:
            rows.append(bonus[b])
        expect = any(_row_bad(x) for x in rows)
        assert bool(ref["nonfinite"][b]) == expect, b
        if expect:
            assert ref["tau"][b] == 0 and (ref["out_tokens"][b] == -1).all()
        else:
            assert ref["tau"][b] == plain["tau"][b]
            np.testing.assert_array_equal(ref["out_tokens"][b], plain["out_tokens"][b])
    assert ref["nonfinite"].sum() > 10 and ref["nonfinite"].sum() < B
    assert plain["nonfinite"].sum() == 0         # without the check nothing is flagged
    assert ref["invalid_rows"] == int(ref["nonfinite"].sum())


# ------------------------------------------------------------------- Philox ----
# Random123's published known-answer vectors for Philox4x32-10
# (Salmon et al., SC'11 distribution): (counter, key) -> output.
KAT = [
    ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF,) * 4, (0xFFFFFFFF,) * 2, (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


def test_philox_known_answers(oracle_lib):
    for ctr, key, out in KAT:
        assert tuple(int(x) for x in oracle_lib.philox4x32_10(ctr, key)) == out


@pytest.mark.slow
def test_philox_matches_triton_interpreter(oracle_lib):
    """An independent Philox4x32-10 (Triton's, run on the CPU interpreter)
    agrees bit for bit on random counters and keys."""
    pytest.importorskip("triton")
    rng = np.random.default_rng(61)
    n = 64
    ctr = rng.integers(0, 2 ** 32, size=(n, 4), dtype=np.uint64).astype(np.uint32)
    key = rng.integers(0, 2 ** 32, size=(n, 2), dtype=np.uint64).astype(np.uint32)
    script = textwrap.dedent(f"""
        import os, sys
        os.environ["TRITON_INTERPRET"] = "1"
        import numpy as np, torch, triton, triton.language as tl
        from triton.language.random import philox_impl
        @triton.jit
        def k(c_ptr, key_ptr, out_ptr, N: tl.constexpr):
            i = tl.arange(0, N)
            c = [tl.load(c_ptr + 4 * i + w) for w in range(4)]
            k0 = tl.load(key_ptr + 2 * i); k1 = tl.load(key_ptr + 2 * i + 1)
            o0, o1, o2, o3 = philox_impl(c[0], c[1], c[2], c[3], k0, k1, 10)
            tl.store(out_ptr + 4 * i + 0, o0); tl.store(out_ptr + 4 * i + 1, o1)
            tl.store(out_ptr + 4 * i + 2, o2); tl.store(out_ptr + 4 * i + 3, o3)
        ctr = torch.from_numpy(np.frombuffer(bytes.fromhex(sys.argv[1]), dtype=np.uint32).reshape({n}, 4).copy())
        key = torch.from_numpy(np.frombuffer(bytes.fromhex(sys.argv[2]), dtype=np.uint32).reshape({n}, 2).copy())
        out = torch.zeros(({n}, 4), dtype=torch.uint32)
        k[(1,)](ctr, key, out, {n})
        print(out.numpy().tobytes().hex())
    """)
    env = dict(os.environ, TRITON_INTERPRET="1")
    res = subprocess.run([sys.executable, "-c", script, ctr.tobytes().hex(), key.tobytes().hex()],
                         capture_output=True, text=True, env=env, timeout=600)
    if res.returncode != 0:
        pytest.skip("triton interpreter unavailable: " + res.stderr[-300:])
    tri = np.frombuffer(bytes.fromhex(res.stdout.strip().splitlines()[-1]), dtype=np.uint32).reshape(n, 4)
    mine = np.stack([oracle_lib.philox4x32_10(ctr[i], key[i]) for i in range(n)])
    np.testing.assert_array_equal(mine, tri)


def test_uniforms_are_uniform_and_exact(oracle_lib):
    from scipy.stats import chisquare
    us = np.array([oracle_lib.uniform(12345, r, p, s) for r in range(64) for p in range(16)
                   for s in range(4)])
    assert us.min() > 0 and us.max() <= 1
    assert np.all(us * 2 ** 24 == np.round(us * 2 ** 24))        # 24-bit grid
    _, pval = chisquare(np.histogram(us, bins=32, range=(0, 1))[0])
    assert pval > 1e-3
    # key (seed) and every counter word change the draw
    a = oracle_lib.uniform(1, 2, 3, 0)
    assert a != oracle_lib.uniform(2, 2, 3, 0) and a != oracle_lib.uniform(1, 3, 3, 0)
    assert a != oracle_lib.uniform(1, 2, 4, 0) and a != oracle_lib.uniform(1, 2, 3, 1)
    assert a != oracle_lib.uniform(1 << 32, 2, 3, 0)


# ------------------------------------------------------------ D3D packing --
def test_d3d_pack_worked_example(oracle_lib):
    """[D3D] worked example: the round confirms 今日 は いい 天気 and です
    replaces だ.  The continuation keyed (3, です) must start right after
    the confirmed text: block 0's first ctx tokens plus its anchor give
    exactly the anchor and the round's emitted tokens."""
    g, ids, target, draftl, tokens = _worked_example_inputs()
    K = tokens.size
    r = oracle_lib.verify(target[None], draftl[None], tokens[None], [0.0], seed=1)
    anchor, pos0, mask = ids[g["anchor"][0]], 40, -7
    keys = np.array([[[3, ids["です"]], [1, ids["ね"]], [-1, -1]]], np.int32)
    t, p, c = oracle_lib.d3d_pack(keys, tokens[None], [anchor], [pos0], mask)
    assert list(t[0, 0]) == [anchor] + list(tokens) and list(p[0, 0]) == list(range(40, 46))
    assert list(t[0, 1]) == [ids["です"]] + [mask] * K
    assert list(p[0, 1]) == list(range(44, 50)) and c[0, 1] == 4 == int(r["tau"][0])
    confirmed = list(t[0, 0, :c[0, 1]]) + [t[0, 1, 0]]
    assert confirmed == [anchor] + list(r["out_tokens"][0, :int(r["tau"][0])])
    assert [ids[w] for w in g["expect_packed"]] == confirmed[1:]
    assert c[0, 0] == 0 and c[0, 2] == 2 and list(p[0, 2]) == list(range(42, 48))
    assert list(t[0, 3]) == [-1] * (K + 1) and list(p[0, 3]) == [-1] * (K + 1) and c[0, 3] == -1


def test_d3d_pack_sizes_from_preparation_table(oracle_lib):
    """[D3D] パック: 23 continuations plus the block under verification are
    24 blocks of 16 = 384 tokens; the table's 512 and 912 likewise."""
    K, V, B = 15, 64, 2
    rng = np.random.default_rng(47)
    draft = rng.normal(size=(B, K, V)).astype(np.float32)
    bonus = rng.normal(size=(B, V)).astype(np.float32)
    tokens = draft.argmax(-1).astype(np.int32)
    for line in open(os.path.join(GOLDEN, "d3d_prep_table.txt")):
        if line.startswith("#") or not line.strip():
            continue
        positions, cands, prepared = map(int, line.split())
        fanout = [cands] * positions + [0] * (K - positions) + [1]
        keys = oracle_lib.outcome_predict(draft, tokens, fanout, bonus)
        t, p, c = oracle_lib.d3d_pack(keys, tokens, [5, 6], [100, 200], -1)
        assert t.shape[1:] == (prepared // 16, 16) and t[0].size == prepared
        assert (c >= 0).all()          # every key found a candidate: no empty block


def test_d3d_pack_hit_block_continues_confirmed_text(oracle_lib):
    """Over random rounds with keys: the block keyed by the real outcome (a
    hit) sees exactly tau tokens of block 0 and continues at the position
    after them; every block's positions are consecutive and start ctx after
    the anchor's."""
    rng = np.random.default_rng(53)
    B, K, V = 64, 6, 24
    target = rng.normal(0, 2, size=(B, K + 1, V)).astype(np.float32)
    draft = (target[:, :K] + rng.normal(0, 0.5, size=(B, K, V))).astype(np.float32)
    temps = rng.choice([0.0, 0.8], size=B).astype(np.float32)
    tokens = np.where(temps[:, None] == 0, draft.argmax(-1),
                      rng.integers(0, V, size=(B, K))).astype(np.int32)
    fanout = [3] * K + [2]
    keys = oracle_lib.outcome_predict(draft, tokens, fanout, target[:, K])
    r = oracle_lib.verify(target, draft, tokens, temps, seed=9, keys=keys)
    anchor = rng.integers(0, V, size=B).astype(np.int32)
    pos0 = rng.integers(0, 1000, size=B).astype(np.int32)
    t, p, c = oracle_lib.d3d_pack(keys, tokens, anchor, pos0, -3)
    hits = 0
    for b in range(B):
        assert c[b, 0] == 0
        for i in range(1, t.shape[1]):
            if c[b, i] < 0:
                continue
            assert list(p[b, i]) == list(range(p[b, i, 0], p[b, i, 0] + K + 1))
            assert p[b, i, 0] - pos0[b] == c[b, i]
        tau, tok = int(r["tau"][b]), int(r["out_tokens"][b, int(r["num_accepted"][b])])
        hit_blocks = [i for i in range(1, t.shape[1])
                      if c[b, i] == tau and t[b, i, 0] == tok]
        assert bool(hit_blocks) == bool(r["hit"][b])
        for i in hit_blocks:
            hits += 1
            confirmed = list(t[b, 0, :c[b, i]]) + [t[b, i, 0]]
            assert confirmed == [anchor[b]] + list(r["out_tokens"][b, :tau])
    assert hits > 0


# -------------------------------------------------- n-gram / prompt lookup --
def test_ngram_draft_worked_example(oracle_lib):
    """[SD] prompt-lookup drafting: the text ends with 1 2 3; its latest
    earlier occurrence (positions 6..8) is followed by 7 4 1 2, which become
    the drafts.  With n_max = 4 the 4-gram 4 1 2 3 has no earlier occurrence
    and the 3-gram is used."""
    h = np.array([[5, 1, 2, 3, 9, 9, 1, 2, 3, 7, 4, 1, 2, 3]], np.int32)
    d, c, pos, n = oracle_lib.ngram_draft(h, [14], 4, 4, 1)
    assert list(d[0]) == [7, 4, 1, 2] and c[0] == 4 and pos[0] == 6 and n[0] == 3
    # K beyond the copied span: truncated, the rest -1
    d, c, pos, n = oracle_lib.ngram_draft(h, [14], 8, 3, 1)
    assert list(d[0]) == [7, 4, 1, 2, 3, -1, -1, -1] and c[0] == 5
    # a history too short for any n-gram, and one with no repeat at all
    d, c, pos, n = oracle_lib.ngram_draft(np.array([[1, 2, 3, 4]], np.int32), [4], 3, 2, 1)
    assert c[0] == 0 and pos[0] == -1 and n[0] == -1 and list(d[0]) == [-1] * 3


def _ngram_by_rfind(h, n_tok, K, n_max, n_min):
    # independent restatement with Python's substring search: tokens become
    # characters, the pattern is searched in the text minus its last token
    s = "".join(chr(0x4E00 + int(t)) for t in h[:n_tok])
    for n in range(n_max, n_min - 1, -1):
        if n > n_tok:
            continue
        i = s.rfind(s[n_tok - n:], 0, n_tok - 1)
        if i >= 0:
            d = [int(t) for t in h[i + n:min(i + n + K, n_tok)]]
            return d + [-1] * (K - len(d)), len(d), i, n
    return [-1] * K, 0, -1, -1


def test_ngram_draft_matches_substring_search(oracle_lib):
    rng = np.random.default_rng(59)
    B, L = 300, 80
    h = rng.integers(0, 6, size=(B, L)).astype(np.int32)     # small vocabulary: many repeats
    h[::7] = rng.integers(0, 1000, size=(len(h[::7]), L))     # and rows with almost none
    lens = rng.integers(0, L + 1, size=B).astype(np.int32)
    for K, n_max, n_min in [(5, 4, 1), (8, 3, 3), (3, 6, 2)]:
        d, c, pos, n = oracle_lib.ngram_draft(h, lens, K, n_max, n_min)
        for b in range(B):
            want = _ngram_by_rfind(h[b], int(lens[b]), K, n_max, n_min)
            assert (list(d[b]), int(c[b]), int(pos[b]), int(n[b])) == want, (b, K, n_max, n_min)


# ------------------------------------------------------- KV-cache rollback --
def test_kv_rollback_worked_example(oracle_lib):
    """[D3D] worked example + [SD] rollback: the verify pass appended the
    anchor 今日 and the five drafts (entries 64..69 after a 64-entry
    prefix); the round confirms 今日 は いい 天気 (tau = 4), so entries 68
    and 69 (だ, よ) go and with them the last 4-entry page."""
    g, ids, target, draftl, tokens = _worked_example_inputs()
    r = oracle_lib.verify(target[None], draftl[None], tokens[None], [0.0], seed=1)
    tau = int(r["tau"][0])
    bt = np.arange(100, 120, dtype=np.int32)[None]          # page ids of the row
    bt2, new_len, freed, offs = oracle_lib.kv_rollback(bt, [70], [tau], 4, tokens.size + 1)
    assert tau == 4 and new_len[0] == 68
    assert list(freed) == [117] and list(offs) == [0, 1]
    assert bt2[0, 17] == -1 and (bt2[0, :17] == bt[0, :17]).all() and (bt2[0, 18:] == bt[0, 18:]).all()


def test_kv_rollback_matches_entry_sets(oracle_lib):
    """Restated with sets of entries and pages: the cache keeps the entries
    before the round plus the first min(tau, appended) appended ones; a page
    stays while it holds a kept entry."""
    rng = np.random.default_rng(61)
    for page, appended in [(16, 6), (1, 3), (7, 9), (32, 33)]:
        B, maxp = 50, 40
        bt = rng.permutation(B * maxp).astype(np.int32).reshape(B, maxp)
        kv = rng.integers(0, page * maxp + 1, size=B).astype(np.int32)
        tau = rng.integers(0, appended + 3, size=B).astype(np.int32)   # some past appended
        bt2, new_len, freed, offs = oracle_lib.kv_rollback(bt, kv, tau, page, appended)
        want_free = []
        for b in range(B):
            before = max(int(kv[b]) - appended, 0)
            kept = list(range(before)) + list(range(before, int(kv[b])))[:min(int(tau[b]), appended)]
            assert new_len[b] == len(kept)
            pages_kept = {e // page for e in kept}
            pages_all = {e // page for e in range(int(kv[b]))}
            gone = sorted(pages_all - pages_kept)
            assert list(freed[offs[b]:offs[b + 1]]) == [int(bt[b, p]) for p in gone]
            want_free += gone
            for p in range(maxp):
                assert bt2[b, p] == (-1 if p in gone else bt[b, p])
        assert offs[-1] == len(want_free)
