"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each ``pin_*`` function takes an :class:`oracle.oracle.Oracle` and raises
``AssertionError`` when the oracle disagrees with what the mathematics fixes:
exact integer arithmetic, hand-derived closed forms, brute force on tiny
inputs, library routines (torch / numpy fp64) in special cases, and
invariants. ``test_oracle_pins.py`` runs them on the oracle; the mutation
tests run them on copies of the oracle with a planted mistake and require
that at least one pin fails for every mistake.

The pages give no worked example of the layer, so nothing here is a value
printed by the pages; every expected value is derived in the comments.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from token_dispatch_grouped_moe_gb300.inputs import bf16_bits, make_inputs


def _bits(values) -> np.ndarray:
    """bf16 bits of values that bf16 holds exactly (checked)."""
    t = torch.tensor(np.asarray(values, dtype=np.float32))
    b = t.to(torch.bfloat16)
    assert torch.equal(b.float(), t), "value not exactly representable in bf16"
    return bf16_bits(b)


def _f(bits) -> np.ndarray:
    """bf16 bits -> float64 values."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def _rand_bits(shape, rng, sigma=1.0):
    return bf16_bits(torch.from_numpy((rng.standard_normal(shape) * sigma).astype(np.float32))
                     .to(torch.bfloat16))


# ------------------------------------------------------------------ logits --

def pin_logits_exact_integers(O):
    """Small-integer inputs: every partial sum is an exact fp32 integer, so in
    any order the logit equals the integer dot product (plus integer bias).
    H=200 is not a multiple of 8 or 256, so partial chunks are covered; Wg is
    not symmetric, so a transposed index changes the values."""
    rng = np.random.default_rng(1)
    T, H, E = 7, 200, 5
    xi = rng.integers(-4, 5, size=(T, H))
    wi = rng.integers(-4, 5, size=(H, E))
    bias = rng.integers(-8, 9, size=E).astype(np.float32)
    logits = O.logits(_bits(xi), _bits(wi), bias)
    exact = (xi.astype(np.int64) @ wi.astype(np.int64)) + bias.astype(np.int64)
    assert np.array_equal(logits.astype(np.int64), exact)
    assert np.array_equal(logits, exact.astype(np.float32))


def _one_hot_case(H, placements):
    """x = 1 at the given h, Wg[h, 0] = value; one token, one expert."""
    x = np.zeros((1, H), np.float32)
    w = np.zeros((H, 1), np.float32)
    for h, v in placements:
        x[0, h] = 1.0
        w[h, 0] = v
    return _bits(x), _bits(w)


def pin_logits_canonical_order(O):
    """The canonical order, pinned by cases whose fp32 result depends on it.
    Chunk c (h = 8c..8c+7) belongs to lane c mod 32; lanes reduce by the xor
    butterfly with s = 16, 8, 4, 2, 1. 2^24 + 1 is not an fp32 number and
    rounds (to even) back to 2^24, so adding 1 into a lane that holds 2^24
    loses it."""
    big = float(2 ** 24)
    # (a) +1 in chunk 1 (lane 1), -2^24 later in the same chunk: lane 1 holds
    #     1 - 2^24 exactly; lane 0 holds 2^24; total 1. A plain left-to-right
    #     sum over h would give (2^24 + 1) - 2^24 = 0.
    x, w = _one_hot_case(16, [(0, big), (8, 1.0), (9, -big)])
    assert O.logits(x, w)[0, 0] == 1.0
    # (b) butterfly order: lane 0 = 2^24 (chunk 0), lane 1 = 1 (chunk 1),
    #     lane 16 = -2^24 (chunk 16). s = 16 first pairs lanes 0 and 16 -> 0,
    #     then 0 + 1 = 1. Pairing lanes 0 and 1 first would lose the 1.
    x, w = _one_hot_case(256, [(0, big), (8, 1.0), (128, -big)])
    assert O.logits(x, w)[0, 0] == 1.0
    # (c) wrap-around: chunk 32 (h = 256) is lane 0 again, after chunk 0, so
    #     2^24 + 1 loses the 1 inside lane 0; lane 1 = -2^24; total 0.
    x, w = _one_hot_case(264, [(0, big), (256, 1.0), (8, -big)])
    assert O.logits(x, w)[0, 0] == 0.0
    # (d) within a chunk, h increases: lane 0 takes -2^24, then 1 (giving
    #     1 - 2^24, exact), then 2^24: 1. Decreasing h would add 2^24 + 1
    #     first, lose the 1, and give 0.
    x, w = _one_hot_case(8, [(0, -big), (1, 1.0), (2, big)])
    assert O.logits(x, w)[0, 0] == 1.0
    # (e) 32 lanes, not fewer: chunks 0 and 32 share lane 0 (2^24 + 1 -> 2^24),
    #     chunk 16 is lane 16 (-2^24); s = 16 then gives 0. With 16 lanes,
    #     chunk 16 would join lane 0 before chunk 32: (2^24 - 2^24) + 1 = 1.
    x, w = _one_hot_case(264, [(0, big), (128, -big), (256, 1.0)])
    assert O.logits(x, w)[0, 0] == 0.0


def pin_logits_vs_fp64(O):
    """Random bf16 inputs: the fp32 logit is within the forward error bound
    of its summation tree (depth H/256*8 + 5 adds, each rounding by at most
    2^-24 relative) of the fp64 dot product."""
    rng = np.random.default_rng(2)
    T, H, E = 33, 1024, 8
    x = _rand_bits((T, H), rng)
    w = _rand_bits((H, E), rng, 0.02)
    l = O.logits(x, w).astype(np.float64)
    xf, wf = _f(x), _f(w)
    exact = xf @ wf
    depth = (H + 255) // 256 * 8 + 5
    bound = depth * 2.0 ** -24 * (np.abs(xf) @ np.abs(wf)) * 1.01
    assert np.all(np.abs(l - exact) <= bound)


# ------------------------------------------------------------------- top-k --

def pin_topk_bruteforce(O):
    """Indices equal a full stable sort of all E logits by descending value."""
    rng = np.random.default_rng(3)
    for T, E, k in [(64, 8, 2), (40, 64, 6), (16, 5, 5), (9, 1, 1)]:
        H = 64
        x = _rand_bits((T, H), rng)
        w = _rand_bits((H, E), rng, 0.02)
        logits, idx, _ = O.route(x, w, k)
        for t in range(T):
            order = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))
            assert list(idx[t]) == order[:k]


def pin_topk_ties(O):
    """Equal logits go to the lower expert id, in selection order."""
    logits = np.array([[0.5, 0.5, 0.5, 0.5],
                       [1.0, 2.0, 2.0, 1.0],
                       [-1.0, -1.0, 3.0, 3.0]], np.float32)
    idx, w = O.topk(logits, 3)
    assert idx.tolist() == [[0, 1, 2], [1, 2, 0], [2, 3, 0]]
    # Equal logits have equal weights: 1/3 each in row 0.
    assert np.allclose(w[0], 1.0 / 3.0, rtol=0, atol=1e-7)


def pin_topk_vs_torch(O):
    """Without ties, the selected set and order equal torch.topk's."""
    rng = np.random.default_rng(4)
    logits = rng.standard_normal((200, 64)).astype(np.float32)
    idx, _ = O.topk(logits, 8)
    ref = torch.topk(torch.from_numpy(logits), 8, dim=1).indices.numpy()
    assert np.array_equal(idx, ref)


# ----------------------------------------------------------- gate weights --

def pin_gate_weights(O):
    """w = softmax over all E, renormalised over the k selected (numpy fp64);
    weights sum to 1; for k = 2, w0 = 1 / (1 + exp(l1 - l0))."""
    rng = np.random.default_rng(5)
    for E, k in [(8, 2), (64, 6), (64, 8), (3, 1)]:
        logits = (rng.standard_normal((50, E)) * 1.5).astype(np.float32)
        idx, w = O.topk(logits, k)
        l64 = logits.astype(np.float64)
        p = np.exp(l64 - l64.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        sel = np.take_along_axis(p, idx.astype(np.int64), axis=1)
        ref = sel / sel.sum(axis=1, keepdims=True)
        assert np.allclose(w, ref, rtol=1e-6, atol=1e-7)
        assert np.all(np.abs(w.astype(np.float64).sum(axis=1) - 1.0) <= 1e-6)
        if k == 2:
            l0 = np.take_along_axis(l64, idx[:, :1].astype(np.int64), 1)[:, 0]
            l1 = np.take_along_axis(l64, idx[:, 1:2].astype(np.int64), 1)[:, 0]
            assert np.allclose(w[:, 0], 1.0 / (1.0 + np.exp(l1 - l0)), rtol=1e-6)
        if k == 1:
            assert np.all(w == 1.0)


# ---------------------------------------------------------------- permute --

def _check_perm(idx_flat, E, counts, offsets, src_row, inv_pos):
    R = idx_flat.size
    order = sorted(range(R), key=lambda f: (int(idx_flat[f]), f))   # stable, by expert
    assert src_row.tolist() == order
    assert counts.tolist() == [int((idx_flat == e).sum()) for e in range(E)]
    assert offsets.tolist() == [0] + np.cumsum(counts).tolist()
    assert int(counts.sum()) == R
    assert np.array_equal(inv_pos[src_row], np.arange(R))
    for e in range(E):
        seg = src_row[offsets[e]:offsets[e + 1]]
        assert np.all(idx_flat[seg] == e)
        assert np.all(np.diff(seg) > 0)


def pin_permute_bruteforce(O):
    """Stable counting sort equals Python's stable sort; structural invariants."""
    rng = np.random.default_rng(6)
    for T, E, k in [(100, 8, 2), (37, 64, 6), (1, 4, 4), (0, 8, 2), (50, 1, 1)]:
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32) \
            if T else np.zeros((0, k), np.int32)
        counts, offsets, src_row, inv_pos = O.permute(idx, E)
        _check_perm(idx.reshape(-1), E, counts, offsets, src_row, inv_pos)
    # Skewed: most assignments to one expert, some experts empty.
    idx = np.where(rng.random((300, 1)) < 0.8, 3, rng.integers(0, 8, (300, 1))).astype(np.int32)
    _check_perm(idx.reshape(-1), 8, *O.permute(idx, 8))


def pin_permute_rejects_bad_ids(O):
    """An id outside [0, E) is an error, not a write out of bounds."""
    for bad in (8, -1):
        idx = np.array([[0, 1], [2, bad]], np.int32)
        try:
            O.permute(idx, 8)
        except ValueError:
            continue
        raise AssertionError("out-of-range id accepted")


# --------------------------------------------------------- FFN + combine --

def _swiglu_torch(x, W1, W3, W2):
    """Textbook SwiGLU FFN with torch's own silu, fp64."""
    return (torch.nn.functional.silu(x @ W1) * (x @ W3)) @ W2


def _t64(bits):
    return torch.from_numpy(_f(bits))


def pin_dense_E1(O):
    """E = 1, k = 1: the gate weight is exactly 1 and the layer is a dense
    SwiGLU FFN (torch fp64 on CPU)."""
    T, H, F = 12, 128, 96
    inp = make_inputs(T, H, F, 1, seed=11)
    b = {n: bf16_bits(v) for n, v in inp.items()}
    r = O.layer_forward(b["x"], b["Wg"], b["W1"], b["W3"], b["W2"], k=1)
    assert np.all(r["topk_idx"] == 0) and np.all(r["topk_w"] == 1.0)
    ref = _swiglu_torch(_t64(b["x"]), _t64(b["W1"][0]), _t64(b["W3"][0]), _t64(b["W2"][0]))
    scale = float(np.sqrt(np.mean(ref.numpy() ** 2)))
    assert np.max(np.abs(r["out"] - ref.numpy())) <= 1e-12 * scale * H


def pin_dense_all_experts(O):
    """Brute force: out = sum_e g_e * FFN_e(x) over ALL experts (numpy fp64
    matmuls), g_e the softmax renormalised over the top-k from a full sort,
    0 elsewhere. Independent of the oracle's permutation and combine loops."""
    T, H, F, E, k = 20, 64, 48, 6, 3
    inp = make_inputs(T, H, F, E, seed=12)
    b = {n: bf16_bits(v) for n, v in inp.items()}
    r = O.layer_forward(b["x"], b["Wg"], b["W1"], b["W3"], b["W2"], k=k)
    x = _f(b["x"])
    logits = r["logits"].astype(np.float64)
    g = np.zeros((T, E))
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-logits[t, e], e))[:k]
        p = np.exp(logits[t, order] - logits[t, order[0]])
        g[t, order] = p / p.sum()
    ref = np.zeros((T, H))
    for e in range(E):
        a = x @ _f(b["W1"][e])
        bb = x @ _f(b["W3"][e])
        y = (a / (1.0 + np.exp(-a)) * bb) @ _f(b["W2"][e])
        ref += g[:, e:e + 1] * y
    scale = float(np.sqrt(np.mean(ref ** 2)))
    assert np.max(np.abs(r["out"] - ref)) <= 1e-6 * scale


def pin_shared_expert(O):
    """The always-on shared expert adds a dense SwiGLU FFN with weight 1."""
    T, H, F, E, k, Fs = 10, 64, 32, 4, 2, 80
    inp = make_inputs(T, H, F, E, Fs=Fs, seed=13)
    b = {n: bf16_bits(v) for n, v in inp.items()}
    with_s = O.layer_forward(b["x"], b["Wg"], b["W1"], b["W3"], b["W2"], k=k,
                             W1s=b["W1s"], W3s=b["W3s"], W2s=b["W2s"])["out"]
    without = O.layer_forward(b["x"], b["Wg"], b["W1"], b["W3"], b["W2"], k=k)["out"]
    ref = _swiglu_torch(_t64(b["x"]), _t64(b["W1s"]), _t64(b["W3s"]), _t64(b["W2s"])).numpy()
    scale = float(np.sqrt(np.mean(ref ** 2)))
    assert np.max(np.abs((with_s - without) - ref)) <= 1e-9 * scale


def pin_row_independence(O):
    """out[t] depends on x[t] only: permuting the tokens permutes the routing
    and the output rows exactly, and any subset gives the same rows."""
    T, H, F, E, k = 16, 64, 32, 8, 2
    inp = make_inputs(T, H, F, E, seed=14)
    b = {n: bf16_bits(v) for n, v in inp.items()}
    full = O.layer_forward(b["x"], b["Wg"], b["W1"], b["W3"], b["W2"], k=k)
    perm = np.random.default_rng(7).permutation(T)
    pr = O.layer_forward(b["x"][perm], b["Wg"], b["W1"], b["W3"], b["W2"], k=k)
    assert np.array_equal(pr["topk_idx"], full["topk_idx"][perm])
    assert np.array_equal(pr["out"], full["out"][perm])
    sub = np.array([5, 0, 11], np.int64)
    rows = O.layer_rows(sub, full["topk_idx"], full["topk_w"], b["x"], b["W1"], b["W3"], b["W2"])
    assert np.array_equal(rows, full["out"][sub])


def pin_worked_example(O):
    """A hand-worked layer, T=2, H=8, F=2, E=3, k=2 (all values exact in bf16).

    x[0] = e_0, x[1] = e_1 (unit rows). Wg rows 0 and 1 are [1, 0, 2] and
    [0, 2, 1], so the logits are t0: [1, 0, 2] -> experts (2, 0); t1: [0, 2, 1]
    -> experts (1, 2). Both tokens have top-2 logits (2, 1), so the weights
    are (s, 1 - s) with s = 1 / (1 + e^-1).
    Every expert has W1 rows e_0, e_1 (so a = (x0, x1)), W3 = c_e * W1 with
    c = (1, 2, 4) (so b = c_e * a), and W2[f, n] = [f == n]. Hence
    FFN_e(x[0]) = silu(1) c_e e_0 and FFN_e(x[1]) = silu(1) c_e e_1, with
    silu(1) = s. So
      out[0, 0] = s (s c_2 + (1 - s) c_0) = s (4 s + (1 - s)),
      out[1, 1] = s (s c_1 + (1 - s) c_2) = s (2 s + 4 (1 - s)),
    and every other output is 0.
    """
    T, H, F, E = 2, 8, 2, 3
    x = np.zeros((T, H)); x[0, 0] = 1; x[1, 1] = 1
    Wg = np.zeros((H, E)); Wg[0] = [1, 0, 2]; Wg[1] = [0, 2, 1]
    c = [1.0, 2.0, 4.0]
    W1 = np.zeros((E, H, F)); W3 = np.zeros((E, H, F)); W2 = np.zeros((E, F, H))
    for e in range(E):
        W1[e, 0, 0] = 1; W1[e, 1, 1] = 1
        W3[e] = c[e] * W1[e]
        W2[e, 0, 0] = 1; W2[e, 1, 1] = 1
    r = O.layer_forward(_bits(x), _bits(Wg), _bits(W1), _bits(W3), _bits(W2), k=2)
    s = 1.0 / (1.0 + math.exp(-1.0))
    assert r["topk_idx"].tolist() == [[2, 0], [1, 2]]
    assert np.allclose(r["topk_w"], [[s, 1 - s], [s, 1 - s]], rtol=0, atol=1e-7)
    expect = np.zeros((T, H))
    expect[0, 0] = s * (4 * s + (1 - s))
    expect[1, 1] = s * (2 * s + 4 * (1 - s))
    # The weights are fp32-rounded router outputs: allow their rounding.
    assert np.allclose(r["out"], expect, rtol=1e-6, atol=0)
    assert r["counts"].tolist() == [1, 1, 2]
    assert r["src_row"].tolist() == [1, 2, 0, 3]      # f = t*k + j, grouped by expert


# ------------------------------------------------------- gating variants --

def pin_gate_weights_full(O):
    """Without renormalisation the weights are a softmax over all E experts
    (numpy fp64) at the selected ids; they sum to less than 1, and to 1 when
    k = E, where they equal the renormalised weights."""
    rng = np.random.default_rng(15)
    for E, k in [(8, 2), (64, 6), (5, 5)]:
        logits = (rng.standard_normal((40, E)) * 1.5).astype(np.float32)
        idx, w_renorm = O.topk(logits, k)
        w = O.gate_weights_full(logits, idx)
        l64 = logits.astype(np.float64)
        p = np.exp(l64 - l64.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        ref = np.take_along_axis(p, idx.astype(np.int64), axis=1)
        assert np.allclose(w, ref, rtol=1e-6, atol=1e-8)
        if k < E:
            assert np.all(w.astype(np.float64).sum(axis=1) < 1.0)
        else:
            assert np.allclose(w, w_renorm, rtol=1e-6, atol=1e-8)


def pin_shared_gate(O):
    """The sigmoid-gated shared expert: wsg = 0 gives exactly half the shared
    expert; random wsg scales it by torch's sigmoid(x @ wsg) (fp64)."""
    T, H, F, E, k, Fs = 10, 64, 32, 4, 2, 80
    inp = make_inputs(T, H, F, E, Fs=Fs, seed=16)
    b = {n: bf16_bits(v) for n, v in inp.items()}
    args = (b["x"], b["Wg"], b["W1"], b["W3"], b["W2"])
    without = O.layer_forward(*args, k=k)["out"]
    dense = _swiglu_torch(_t64(b["x"]), _t64(b["W1s"]), _t64(b["W3s"]), _t64(b["W2s"])).numpy()
    zero = np.zeros(H, np.uint16)
    half = O.layer_forward(*args, k=k, W1s=b["W1s"], W3s=b["W3s"], W2s=b["W2s"], wsg=zero)["out"]
    scale = float(np.sqrt(np.mean(dense ** 2)))
    assert np.max(np.abs((half - without) - 0.5 * dense)) <= 1e-9 * scale
    wsg = _rand_bits((H,), np.random.default_rng(17), 0.05)
    gated = O.layer_forward(*args, k=k, W1s=b["W1s"], W3s=b["W3s"], W2s=b["W2s"], wsg=wsg)["out"]
    s = torch.sigmoid(_t64(b["x"]) @ _t64(wsg)).numpy()
    assert np.max(np.abs((gated - without) - s[:, None] * dense)) <= 1e-9 * scale


ALL_PINS = [
    pin_logits_exact_integers,
    pin_logits_canonical_order,
    pin_logits_vs_fp64,
    pin_topk_bruteforce,
    pin_topk_ties,
    pin_topk_vs_torch,
    pin_gate_weights,
    pin_permute_bruteforce,
    pin_permute_rejects_bad_ids,
    pin_dense_E1,
    pin_dense_all_experts,
    pin_shared_expert,
    pin_row_independence,
    pin_worked_example,
    pin_gate_weights_full,
    pin_shared_gate,
]
