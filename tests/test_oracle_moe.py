"""Pins for the oracle's MoE region, independent of the oracle's own code.

* routing against a brute force written here: a stable sort of (-logit, expert)
  per token and a float64 softmax over the chosen logits; a hand-worked case
  with equal logits;
* the permutation against numpy's stable argsort of the expert ids;
* the down region with one expert and unit gates equals the dense region
  (pinned in test_oracle.py) bit for bit;
* exact scale law: doubling every gate doubles the region's sum z exactly;
* relabelling the experts (permuting We and the grouping) changes nothing;
* a float64 einsum over the rows on the CPU;
* a hand-worked 1-token, 2-expert case.
Runs on the CPU only.
"""
import numpy as np

import oracle
from synth import MOE_CONFIGS, Workload, f32_to_bf16_bits, make_inputs_moe


def _brute_route(logits, k):
    T, E = logits.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k))
    for t in range(T):
        order = np.lexsort((np.arange(E), -logits[t].astype(np.float64)))[:k]
        ids[t] = order
        sel = logits[t, order].astype(np.float64)
        ex = np.exp(sel - sel.max())
        w[t] = ex / ex.sum()
    return ids, w


def test_route_matches_brute_force():
    g = np.random.default_rng(3)
    for E, k in [(8, 2), (16, 4), (5, 5), (64, 8)]:
        logits = g.standard_normal((37, E)).astype(np.float32)
        logits[3, :] = 0.25  # all equal: experts 0..k-1 in order
        logits[5, 1] = logits[5, 4] = 9.0
        ids, w = oracle.moe_route(logits, k)
        bi, bw = _brute_route(logits, k)
        np.testing.assert_array_equal(ids, bi)
        np.testing.assert_allclose(w, bw, rtol=1e-15, atol=1e-16)
        np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=1e-15)


def test_route_hand_case():
    logits = np.array([[0.5, 2.0, 2.0, -1.0], [3.0, 1.0, 0.0, 3.0]], np.float32)
    ids, w = oracle.moe_route(logits, 2)
    np.testing.assert_array_equal(ids, [[1, 2], [0, 3]])
    np.testing.assert_array_equal(w, [[0.5, 0.5], [0.5, 0.5]])
    ids, w = oracle.moe_route(logits, 3)
    np.testing.assert_array_equal(ids, [[1, 2, 0], [0, 3, 1]])
    e = np.exp(-1.5)
    np.testing.assert_allclose(w[0], [1 / (2 + e), 1 / (2 + e), e / (2 + e)], rtol=1e-15)


def test_permute_matches_stable_argsort():
    g = np.random.default_rng(4)
    T, E, k = 50, 8, 3
    ids = np.stack([g.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    offsets, row_token, row_slot, row_of = oracle.moe_permute(ids, E)
    flat = ids.ravel()
    order = np.argsort(flat, kind="stable")  # pairs (t, j) in row-major order, stable by expert
    np.testing.assert_array_equal(row_token, order // k)
    np.testing.assert_array_equal(row_slot, order % k)
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
    inv = np.empty_like(order)
    inv[order] = np.arange(order.size)
    np.testing.assert_array_equal(row_of.ravel(), inv)


def _grouped(d, E):
    offsets, _, _, row_of = oracle.moe_permute(d["ids"], E)
    return offsets, row_of


def test_one_expert_equals_dense_region():
    wl = Workload("moe1", T=6, K=96, H=40, eps=1e-5, r_sigma=2.0, seed=7)
    d = make_inputs_moe(wl, 1, 1)
    offsets, row_of = _grouped(d, 1)
    wt = np.ones((6, 1), np.float32)
    for kind in (0, 1):
        a = oracle.moe_down_region(d["hg"], offsets, row_of, wt, d["We"], d["r0"], d["gamma"], wl.eps, kind)
        b = oracle.proj_add_rmsnorm(d["hg"], d["We"][0], d["r0"], d["gamma"], wl.eps, kind)
        for u, v in zip(a, b):
            assert np.array_equal(u, v)


def _r0(d):
    return (d["r0"].astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_gates_scale_the_sum_exactly():
    wl, E, k = MOE_CONFIGS["moe_tiny"]
    d = make_inputs_moe(wl, E, k)
    offsets, row_of = _grouped(d, E)
    zero = np.zeros_like(d["r0"])  # r = z exactly
    r1, _, _ = oracle.moe_down_region(d["hg"], offsets, row_of, d["wt"], d["We"], zero, d["gamma"], wl.eps, 0)
    r2, _, _ = oracle.moe_down_region(d["hg"], offsets, row_of, 2 * d["wt"], d["We"], zero, d["gamma"], wl.eps, 0)
    np.testing.assert_array_equal(r2, 2 * r1)


def test_expert_relabelling_changes_nothing():
    wl, E, k = MOE_CONFIGS["moe_tiny"]
    d = make_inputs_moe(wl, E, k)
    offsets, row_token, row_slot, row_of = oracle.moe_permute(d["ids"], E)
    a = oracle.moe_down_region(d["hg"], offsets, row_of, d["wt"], d["We"], d["r0"], d["gamma"], wl.eps, 0)
    # new label of expert e is p[e]; regroup the same activation rows under the new labels
    p = np.array([2, 0, 3, 1])
    ids2 = p[d["ids"]].astype(np.int32)
    off2, tok2, slot2, row_of2 = oracle.moe_permute(ids2, E)
    hg2 = np.empty_like(d["hg"])
    for r in range(hg2.shape[0]):
        hg2[r] = d["hg"][row_of[tok2[r], slot2[r]]]
    We2 = np.empty_like(d["We"])
    We2[p] = d["We"]
    b = oracle.moe_down_region(hg2, off2, row_of2, d["wt"], We2, d["r0"], d["gamma"], wl.eps, 0)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_against_float64_einsum():
    wl, E, k = MOE_CONFIGS["moe_tiny"]
    d = make_inputs_moe(wl, E, k)
    offsets, row_token, row_slot, row_of = oracle.moe_permute(d["ids"], E)
    f = lambda b: (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    hg, We = f(d["hg"]), f(d["We"])
    expert_of_row = np.repeat(np.arange(E), np.diff(offsets))
    y = np.einsum("rc,rhc->rh", hg, We[expert_of_row])
    z = np.zeros((wl.T, wl.H))
    for r in range(y.shape[0]):
        z[row_token[r]] += d["wt"][row_token[r], row_slot[r]].astype(np.float64) * y[r]
    r_, _, _ = oracle.moe_down_region(d["hg"], offsets, row_of, d["wt"], d["We"], d["r0"], d["gamma"], wl.eps, 0)
    np.testing.assert_allclose(r_, _r0(d) + z, rtol=1e-12, atol=1e-12)


def test_hand_worked_case():
    # one token, experts 0 and 1, gates 0.5 and 2; rows: expert 0 gets [1, 2], expert 1 gets [3, -1]
    # We[0] = [[1, 0], [0, 1]], We[1] = [[2, 1], [1, 1]] -> y0 = [1, 2], y1 = [5, 2]
    # z = 0.5 * [1, 2] + 2 * [5, 2] = [10.5, 5]
    hg = f32_to_bf16_bits(np.array([[1, 2], [3, -1]], np.float32))
    We = f32_to_bf16_bits(np.array([[[1, 0], [0, 1]], [[2, 1], [1, 1]]], np.float32))
    offsets = np.array([0, 1, 2], np.int32)
    row_of = np.array([[0, 1]], np.int32)
    wt = np.array([[0.5, 2.0]], np.float32)
    r0 = f32_to_bf16_bits(np.zeros((1, 2), np.float32))
    g = np.ones(2, np.float32)
    r, o, ms = oracle.moe_down_region(hg, offsets, row_of, wt, We, r0, g, 0.0, 0)
    np.testing.assert_array_equal(r, [[10.5, 5.0]])
    np.testing.assert_allclose(ms, [(10.5 ** 2 + 25) / 2], rtol=1e-15)


def test_gather_inverts_the_grouping():
    g = np.random.default_rng(8)
    T, E, k, H = 30, 6, 3, 16
    ids = np.stack([g.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    _, row_token, row_slot, row_of = oracle.moe_permute(ids, E)
    x = g.integers(0, 1 << 16, size=(T, H), dtype=np.uint16)
    xg = oracle.moe_gather(x, row_token)
    for t in range(T):
        for j in range(k):
            assert np.array_equal(xg[row_of[t, j]], x[t])
    assert np.array_equal(np.sort(row_token), np.repeat(np.arange(T), k))

