"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

Each test checks the oracle against brute force, exact rational arithmetic,
a closed form, an invariant of the method, or a library routine that a special
case reduces to -- never against a retyped copy of the oracle's own formula.
CPU only.
"""
from fractions import Fraction
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from sparse_moe_layer_router_gb300.synthetic import (CONFIGS, as_u16, normal_bf16,
                                                     quantize_w4)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers
def bf16_bits(values):
    """float values that are exactly bf16 -> uint16 bit patterns (asserts exactness)."""
    t = torch.tensor(np.asarray(values, np.float32))
    b = t.to(torch.bfloat16)
    assert torch.equal(b.to(torch.float32), t), "value not exactly representable in bf16"
    return as_u16(b)


def bits_to_fraction(u16):
    """Exact rational value of a bf16 bit pattern."""
    f = np.array([int(u16) << 16], np.uint32).view(np.float32)[0]
    return Fraction(float(f))


def exact_logits(x, wr, bias=None):
    """Exact rational logits from bf16 bit patterns (brute force, no rounding)."""
    T, D = x.shape
    E = wr.shape[0]
    xf = [[bits_to_fraction(v) for v in row] for row in x]
    wf = [[bits_to_fraction(v) for v in row] for row in wr]
    z = [[sum(xf[t][d] * wf[e][d] for d in range(D)) for e in range(E)] for t in range(T)]
    if bias is not None:
        z = [[z[t][e] + Fraction(float(bias[e])) for e in range(E)] for t in range(T)]
    return z


def brute_topk(zrow, k):
    """The k-subset whose every member beats every non-member under (z desc, index asc)."""
    E = len(zrow)

    def beats(a, b):
        return zrow[a] > zrow[b] or (zrow[a] == zrow[b] and a < b)

    found = [S for S in itertools.combinations(range(E), k)
             if all(beats(a, b) for a in S for b in range(E) if b not in S)]
    assert len(found) == 1
    return list(found[0])


def small_inputs(T, D, E, seed, wr_std=0.5):
    x = as_u16(normal_bf16((T, D), 1.0, seed, 11))
    wr = as_u16(normal_bf16((E, D), wr_std, seed, 12))
    return x, wr


# ---------------------------------------------------------------- routing
@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("k", [1, 2, 3, 6])
def test_route_matches_brute_force_exact(seed, k):
    """Top-k set equals exhaustive search over all k-subsets on exact logits."""
    T, D, E = 12, 8, 6
    x, wr = small_inputs(T, D, E, seed)
    ids, w = oracle.route(x, wr, k)
    z = exact_logits(x, wr)
    for t in range(T):
        assert ids[t].tolist() == brute_topk(z[t], k)


def test_route_ids_ascending_and_distinct():
    x, wr = small_inputs(40, 16, 12, 5)
    ids, _ = oracle.route(x, wr, 5)
    assert np.all(np.diff(ids, axis=1) > 0)


def test_route_with_bias_matches_brute_force():
    T, D, E, k = 10, 8, 7, 3
    x, wr = small_inputs(T, D, E, 9, wr_std=0.05)
    bias = np.array([0.0, -1.5, 2.25, -0.5, 0.75, -3.0, 1.0], np.float32)
    ids, _ = oracle.route(x, wr, k, bias)
    z = exact_logits(x, wr, bias)
    for t in range(T):
        assert ids[t].tolist() == brute_topk(z[t], k)


def test_route_zero_router_is_lowest_indices_uniform():
    """All logits equal: the tie rule picks experts 0..k-1, each with weight 1/k."""
    T, D, E, k = 5, 16, 9, 4
    x, _ = small_inputs(T, D, E, 1)
    wr = np.zeros((E, D), np.uint16)
    ids, w = oracle.route(x, wr, k)
    assert (ids == np.arange(k)).all()
    np.testing.assert_allclose(w, 1.0 / k, rtol=0, atol=1e-15)


def test_route_duplicate_router_rows_prefer_lower_index():
    """Two experts with identical router rows tie exactly; the lower index wins."""
    D = 4
    x = bf16_bits([[1.0, 0.5, -0.25, 2.0]])
    rows = [[0.0, 0.0, 0.0, 0.0], [1.0, 1.0, 0.0, 0.5], [0.0, 0.0, 0.0, 0.0],
            [1.0, 1.0, 0.0, 0.5], [-1.0, 0.0, 0.0, 0.0]]
    wr = bf16_bits(rows)
    ids, w = oracle.route(x, wr, 1)
    assert ids.tolist() == [[1]]
    ids, w = oracle.route(x, wr, 2)
    assert ids.tolist() == [[1, 3]]
    np.testing.assert_allclose(w, [[0.5, 0.5]], atol=1e-15)
    assert D == 4


def test_route_single_expert_and_top1():
    """E = 1: every token goes to expert 0 with weight 1.  k = 1: the argmax, weight 1
    (renormalising over one selected expert)."""
    T, D = 4, 8
    x, wr1 = small_inputs(T, D, 1, 9)
    ids, w = oracle.route(x, wr1, 1)
    assert (ids == 0).all() and (w == 1.0).all()
    x, wr = small_inputs(T, D, 7, 10)
    ids, w = oracle.route(x, wr, 1)
    z = np.array([[float(v) for v in row] for row in exact_logits(x, wr)])
    assert (ids[:, 0] == np.argmax(z, axis=1)).all()
    assert (w == 1.0).all()


def test_route_k_equals_E_is_dense_softmax():
    """k = E: renormalisation is a no-op and w is the softmax over all experts."""
    T, D, E = 6, 8, 5
    x, wr = small_inputs(T, D, E, 3)
    ids, w = oracle.route(x, wr, E)
    z = np.array([[float(v) for v in row] for row in exact_logits(x, wr)])
    assert (ids == np.arange(E)).all()
    np.testing.assert_allclose(w, scipy.special.softmax(z, axis=1), rtol=1e-13, atol=0)


def test_route_weights_are_renormalised_softmax_of_selected():
    """w_j = softmax(z)[id_j] / sum over the selected ids (scipy softmax)."""
    T, D, E, k = 20, 8, 9, 3
    x, wr = small_inputs(T, D, E, 4)
    ids, w = oracle.route(x, wr, k)
    z = np.array([[float(v) for v in row] for row in exact_logits(x, wr)])
    p = scipy.special.softmax(z, axis=1)
    sel = np.take_along_axis(p, ids.astype(np.int64), axis=1)
    np.testing.assert_allclose(w, sel / sel.sum(axis=1, keepdims=True), rtol=1e-13)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-15)


def test_route_hand_worked_example():
    """Golden fixture derived by hand (tests/golden/route_hand_example.json)."""
    with open(os.path.join(GOLDEN, "route_hand_example.json")) as f:
        g = json.load(f)
    x = bf16_bits(g["x"])
    wr = bf16_bits(g["w_router"])
    ids, w = oracle.route(x, wr, g["k"])
    assert ids.tolist() == g["ids"]
    np.testing.assert_allclose(w, g["weights"], rtol=1e-15, atol=1e-16)


BF16_NAN = np.uint16(0x7FC0)


def test_route_nan_logits_rank_below_every_number():
    """Reading R21: experts whose router row holds a NaN (NaN logits) are never
    chosen while k finite experts remain; the ids equal exhaustive search over
    the finite experts alone, and the weights equal the renormalised softmax of
    the selected exact logits (scipy), untouched by the unselected NaNs."""
    T, D, E, k = 9, 8, 7, 3
    x, wr = small_inputs(T, D, E, 21)
    nan_rows = [1, 4]
    wr_nan = wr.copy()
    for e in nan_rows:
        wr_nan[e, 3] = BF16_NAN
    ids, w = oracle.route(x, wr_nan, k)
    finite = [e for e in range(E) if e not in nan_rows]
    z = exact_logits(x, wr[finite])
    for t in range(T):
        sel = [finite[i] for i in brute_topk(z[t], k)]
        assert ids[t].tolist() == sel
        zsel = np.array([float(z[t][finite.index(e)]) for e in sel])
        np.testing.assert_allclose(w[t], scipy.special.softmax(zsel), rtol=1e-12, atol=0)


def test_route_fewer_finite_logits_than_k_fill_with_lowest_nan_indices():
    """Reading R21: with only two finite logits and k = 4, both finite experts
    and the two lowest-index NaN experts are chosen; a selected NaN makes the
    token's weights NaN."""
    T, D, E, k = 3, 8, 5, 4
    x, wr = small_inputs(T, D, E, 22)
    for e in (0, 2, 3):
        wr[e, 0] = BF16_NAN
    ids, w = oracle.route(x, wr, k)
    assert (ids == np.array([0, 1, 2, 4], np.int32)).all()
    assert np.isnan(w).all()


def test_route_nan_token_row_takes_lowest_indices_and_spares_other_tokens():
    """A token row with a NaN has NaN logits everywhere: ids 0..k-1 (reading
    R21), NaN weights; the other tokens route exactly as without it."""
    T, D, E, k = 6, 8, 9, 3
    x, wr = small_inputs(T, D, E, 23)
    ids0, w0 = oracle.route(x, wr, k)
    xn = x.copy()
    xn[2, 5] = BF16_NAN
    ids, w = oracle.route(xn, wr, k)
    assert ids[2].tolist() == list(range(k)) and np.isnan(w[2]).all()
    keep = [t for t in range(T) if t != 2]
    assert (ids[keep] == ids0[keep]).all()
    assert np.array_equal(w[keep], w0[keep])


def test_router_logits_index_order_sum():
    """Exact products summed left to right in fp64: check against exact rationals
    rounded after every addition (the definition's rounding sequence)."""
    T, D, E = 3, 64, 4
    x, wr = small_inputs(T, D, E, 8)
    z = oracle.router_logits(x, wr)
    for t in range(T):
        for e in range(E):
            acc = 0.0
            for d in range(D):
                prod = bits_to_fraction(x[t, d]) * bits_to_fraction(wr[e, d])
                acc = float(Fraction(acc) + prod)  # exact sum, one rounding
            assert z[t, e] == acc


# ---------------------------------------------------------------- blob
def test_blob_layout_and_roundtrip():
    ids = np.array([[3, 7], [0, 5]], np.int32)
    w = np.array([[0.25, 0.75], [0.5, 0.5]])
    blob = oracle.pack_blob(ids, w)
    assert blob.shape == (2, 2, 2)
    assert blob[0, 0].tolist() == [3, 7]
    assert blob[1, 1].view(np.float32).tolist() == [0.5, 0.5]
    assert blob[0, 1].tolist() == np.array([0.25, 0.75], np.float32).view(np.int32).tolist()
    ids2, w2 = oracle.unpack_blob(blob)
    assert (ids2 == ids).all() and (w2 == w.astype(np.float32)).all()


def test_blob_shape_matches_pages_metadata():
    """Per-device metadata: ids [1024,10] int and weights [1024,10] float -> one int32 array."""
    with open(os.path.join(GOLDEN, "page_shapes.json")) as f:
        g = json.load(f)
    T, k = g["routing_metadata_shape"]
    ids = np.zeros((T, k), np.int32)
    blob = oracle.pack_blob(ids, np.full((T, k), 0.1))
    assert blob.dtype == np.int32 and blob.size == 2 * T * k


# ---------------------------------------------------------------- permute
@pytest.mark.parametrize("T,E,k", [(1, 4, 1), (7, 5, 2), (64, 16, 2), (300, 33, 7)])
def test_permute_invariants(T, E, k):
    rng = np.random.default_rng(T * 100 + E)
    ids = np.stack([np.sort(rng.choice(E, size=k, replace=False)) for _ in range(T)]).astype(np.int32)
    counts, offsets, perm, inv = oracle.permute(ids, E)
    assert counts.sum() == T * k
    assert (counts == np.bincount(ids.ravel(), minlength=E)).all()
    assert offsets[0] == 0 and (np.diff(offsets) == counts).all()
    assert sorted(perm.tolist()) == list(range(T * k))          # bijection
    assert (inv[perm] == np.arange(T * k)).all()                # inverse
    # stable grouping by expert == a stable library sort of the flat ids
    assert (perm == np.argsort(ids.ravel(), kind="stable")).all()
    for e in range(E):
        rows = perm[offsets[e]:offsets[e + 1]]
        assert (ids.ravel()[rows] == e).all()


def test_permute_empty_experts_and_all_to_one():
    ids = np.zeros((9, 1), np.int32) + 2
    counts, offsets, perm, inv = oracle.permute(ids, 4)
    assert counts.tolist() == [0, 0, 9, 0]
    assert offsets.tolist() == [0, 0, 0, 9, 9]
    assert perm.tolist() == list(range(9))


# ---------------------------------------------------------------- expert FFN / layer
def numpy_layer(x, ids, w, gu, dn, sgu, sdn):
    """Independent fp64 layer with numpy matmuls and scipy's logistic function."""
    xf = x.astype(np.float64)
    out = np.zeros((x.shape[0], dn.shape[1]), np.float64)

    def ffn(X, GU, DN):
        I = GU.shape[0] // 2
        g = X @ GU[:I].T
        u = X @ GU[I:].T
        h = g * scipy.special.expit(g) * u
        return h @ DN.T

    for t in range(x.shape[0]):
        for j in range(ids.shape[1]):
            out[t] += w[t, j] * ffn(xf[t:t + 1], gu[ids[t, j]], dn[ids[t, j]])[0]
        out[t] += ffn(xf[t:t + 1], sgu, sdn)[0]
    return out


def u16_to_f64(a):
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def make_small_layer(T, D, E, I, Is, seed):
    x = as_u16(normal_bf16((T, D), 1.0, seed, 21))
    wr = as_u16(normal_bf16((E, D), 0.3, seed, 22))
    gu = as_u16(normal_bf16((E, 2 * I, D), D ** -0.5, seed, 23))
    dn = as_u16(normal_bf16((E, D, I), I ** -0.5, seed, 24))
    sgu = as_u16(normal_bf16((2 * Is, D), D ** -0.5, seed, 25))
    sdn = as_u16(normal_bf16((D, Is), Is ** -0.5, seed, 26))
    return x, wr, gu, dn, sgu, sdn


@pytest.mark.parametrize("k", [1, 2, 4])
def test_forward_matches_numpy_matmul_layer(k):
    T, D, E, I, Is = 9, 32, 6, 16, 24
    x, wr, gu, dn, sgu, sdn = make_small_layer(T, D, E, I, Is, k)
    experts = {e: (gu[e], dn[e]) for e in range(E)}
    y, ids, w = oracle.layer(x, wr, k, experts, (sgu, sdn), I=I, Is=Is)
    ref = numpy_layer(u16_to_f64(x), ids, w, u16_to_f64(gu), u16_to_f64(dn), u16_to_f64(sgu),
                      u16_to_f64(sdn))
    np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-12)


def test_forward_k_equals_E_is_dense_mixture():
    """k = E: y = sum_e softmax(z)_e * FFN_e(x) + FFN_shared(x)."""
    T, D, E, I = 5, 16, 4, 8
    x, wr, gu, dn, sgu, sdn = make_small_layer(T, D, E, I, I, 7)
    experts = {e: (gu[e], dn[e]) for e in range(E)}
    y, _, _ = oracle.layer(x, wr, E, experts, (sgu, sdn), I=I, Is=I)
    z = np.array([[float(v) for v in row] for row in exact_logits(x, wr)])
    p = scipy.special.softmax(z, axis=1)
    xf = u16_to_f64(x)
    ref = np.zeros_like(y)
    G, Dn = u16_to_f64(gu), u16_to_f64(dn)
    for e in range(E):
        g = xf @ G[e, :I].T
        u = xf @ G[e, I:].T
        ref += p[:, e:e + 1] * ((g * scipy.special.expit(g) * u) @ Dn[e].T)
    g = xf @ u16_to_f64(sgu)[:I].T
    u = xf @ u16_to_f64(sgu)[I:].T
    ref += (g * scipy.special.expit(g) * u) @ u16_to_f64(sdn).T
    np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-12)


def test_forward_identical_experts_collapse_to_one_ffn():
    """All routed experts equal: weights sum to 1, so y = FFN_0(x) + FFN_shared(x)."""
    T, D, E, I, k = 7, 16, 5, 8, 3
    x, wr, gu, dn, sgu, sdn = make_small_layer(T, D, E, I, I, 2)
    experts = {e: (gu[0], dn[0]) for e in range(E)}
    y, _, _ = oracle.layer(x, wr, k, experts, (sgu, sdn), I=I, Is=I)
    ids0 = np.zeros((T, 1), np.int32)
    y1 = oracle.forward(x, ids0, np.ones((T, 1)), {0: (gu[0], dn[0])}, (sgu, sdn), E=E, I=I, Is=I)
    np.testing.assert_allclose(y, y1, rtol=1e-13, atol=1e-14)


def test_forward_zero_input_gives_zero():
    T, D, E, I = 4, 16, 4, 8
    _, wr, gu, dn, sgu, sdn = make_small_layer(T, D, E, I, I, 3)
    x = np.zeros((T, D), np.uint16)
    y, _, _ = oracle.layer(x, wr, 2, {e: (gu[e], dn[e]) for e in range(E)}, (sgu, sdn), I=I, Is=I)
    assert (y == 0).all()


def test_forward_hand_closed_form():
    """D=4, I=2, E=3, k=1 with x = e_0: every dot product picks one column."""
    x = bf16_bits([[1.0, 0.0, 0.0, 0.0]])
    wr = bf16_bits([[0.5, 0, 0, 0], [2.0, 0, 0, 0], [-1.0, 0, 0, 0]])  # expert 1 wins
    a, b, c, d = 0.75, -1.5, 2.0, 0.5
    gu1 = bf16_bits([[a, 9, 9, 9], [b, 9, 9, 9], [c, 9, 9, 9], [d, 9, 9, 9]])
    dn1 = bf16_bits([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0], [0.25, -2.0]])
    zero_gu = np.zeros((4, 4), np.uint16)
    zero_dn = np.zeros((4, 2), np.uint16)
    sg, su = 1.0, 3.0
    sgu = bf16_bits([[sg, 0, 0, 0], [0, 0, 0, 0], [su, 0, 0, 0], [0, 0, 0, 0]])
    sdn = bf16_bits([[1.0, 0.0], [0.0, 0.0], [0.0, 0.0], [0.0, 0.0]])
    y, ids, w = oracle.layer(x, wr, 1, {0: (zero_gu, zero_dn), 1: (gu1, dn1), 2: (zero_gu, zero_dn)},
                             (sgu, sdn), I=2, Is=2)
    assert ids.tolist() == [[1]] and w.tolist() == [[1.0]]

    def silu(v):
        return v / (1.0 + math.exp(-v))

    h0, h1 = silu(a) * c, silu(b) * d
    shared = silu(sg) * su
    expect = [h0 + shared, h1, h0 + h1, 0.25 * h0 - 2.0 * h1]
    np.testing.assert_allclose(y[0], expect, rtol=1e-15, atol=1e-15)


# ---------------------------------------------------------------- W4A16
def pack_by_hand(q):
    """Pack a [R, C] array of ints in [-8, 7] with Python integers, pair order: value 2i
    of each 8 in bits 4i, value 2i+1 in bits 16+4i."""
    R, C = q.shape
    out = np.zeros((R, C // 8), np.int64)
    for r in range(R):
        for c8 in range(C // 8):
            word = 0
            for j in range(8):
                word |= (int(q[r, c8 * 8 + j]) & 0xF) << (4 * (j // 2) + 16 * (j % 2))
            out[r, c8] = word - (1 << 32) if word >= (1 << 31) else word
    return out.astype(np.int32)


def test_dequant_w4_literal_word():
    """0x86427531 holds, in pair order, the values 1..7 and -8: nibbles from bit 0 up are
    1 3 5 7 (values 0, 2, 4, 6) and 2 4 6 8 (values 1, 3, 5, 7; 0x8 is -8)."""
    word = np.array([[0x86427531 - (1 << 32)]], np.int32)
    s = bf16_bits(np.array([[0.5]]))
    out = oracle.dequant_w4(word, s, 8)
    assert out.tolist() == [[0.5, 1.0, 1.5, 2.0, 2.5, 3.0, 3.5, -4.0]]


def test_dequant_w4_nibble_order_sign_and_scales():
    rng = np.random.default_rng(0)
    R, C, G = 3, 32, 16
    q = rng.integers(-8, 8, size=(R, C))
    q[0, :16] = np.arange(-8, 8)
    s = bf16_bits(rng.choice([0.5, 0.25, 2.0, 0.125, 3.0], size=(R, C // G)))
    out = oracle.dequant_w4(pack_by_hand(q), s, G)
    sf = u16_to_f64(s)
    expect = q * np.repeat(sf, G, axis=1)
    assert (out == expect).all()


def test_w4a16_forward_equals_bf16_forward_on_dequantised_weights():
    """Power-of-two scales make q*s exactly bf16, so both oracle paths see the same
    numbers and must agree bit-for-bit."""
    T, D, E, I, Is, k, G = 6, 32, 4, 16, 16, 2, 16
    rng = np.random.default_rng(1)
    x = as_u16(normal_bf16((T, D), 1.0, 1, 31))
    wr = as_u16(normal_bf16((E, D), 0.3, 1, 32))

    def mat(R, C):
        q = rng.integers(-8, 8, size=(R, C))
        s = 2.0 ** rng.integers(-6, -2, size=(R, C // G))
        deq = q * np.repeat(s, G, axis=1)
        return pack_by_hand(q), bf16_bits(s), bf16_bits(deq)

    ex_q, ex_b = {}, {}
    for e in range(E):
        qg, sg, bg = mat(2 * I, D)
        qd, sd, bd = mat(D, I)
        ex_q[e] = (qg, sg, qd, sd)
        ex_b[e] = (bg, bd)
    qg, sg, bg = mat(2 * Is, D)
    qd, sd, bd = mat(D, Is)
    y4, ids4, _ = oracle.layer(x, wr, k, ex_q, (qg, sg, qd, sd), I=I, Is=Is, quant=1, group=G)
    yb, idsb, _ = oracle.layer(x, wr, k, ex_b, (bg, bd), I=I, Is=Is, quant=0)
    assert (ids4 == idsb).all()
    assert np.array_equal(y4, yb)


def test_dequant_w4_channel_scales():
    """group 0 (channel-wise): one scale per row, q * s_row exactly."""
    rng = np.random.default_rng(5)
    R, C = 5, 48
    q = rng.integers(-8, 8, size=(R, C))
    s = bf16_bits(rng.choice([0.5, 0.25, 2.0, 3.0, 0.0078125], size=R))
    out = oracle.dequant_w4(pack_by_hand(q), s, 0)
    assert (out == q * u16_to_f64(s)[:, None]).all()


def test_w4a16_channel_forward_equals_bf16_forward_on_dequantised_weights():
    """Channel-wise scales (group 0), power-of-two per row: the W4A16 oracle equals the
    bf16 oracle on the dequantised weights bit for bit."""
    T, D, E, I, Is, k = 6, 32, 4, 16, 16, 2
    rng = np.random.default_rng(3)
    x = as_u16(normal_bf16((T, D), 1.0, 1, 33))
    wr = as_u16(normal_bf16((E, D), 0.3, 1, 34))

    def mat(R, C):
        q = rng.integers(-8, 8, size=(R, C))
        s = 2.0 ** rng.integers(-6, -2, size=R)
        return pack_by_hand(q), bf16_bits(s), bf16_bits(q * s[:, None])

    ex_q, ex_b = {}, {}
    for e in range(E):
        qg, sg, bg = mat(2 * I, D)
        qd, sd, bd = mat(D, I)
        ex_q[e] = (qg, sg, qd, sd)
        ex_b[e] = (bg, bd)
    qg, sg, bg = mat(2 * Is, D)
    qd, sd, bd = mat(D, Is)
    y4, ids4, _ = oracle.layer(x, wr, k, ex_q, (qg, sg, qd, sd), I=I, Is=Is, quant=1, group=0)
    yb, idsb, _ = oracle.layer(x, wr, k, ex_b, (bg, bd), I=I, Is=Is, quant=0)
    assert (ids4 == idsb).all()
    assert np.array_equal(y4, yb)


def test_quantizer_channel_roundtrip_bounds():
    """Channel-wise quantiser: one scale per row, |w - q s| <= s/2, absmax maps to +-7."""
    w = normal_bf16((6, 256), 0.05, 0, 43)
    q, s = quantize_w4(w, 0)
    assert tuple(s.shape) == (6,)
    deq = oracle.dequant_w4(q.numpy(), as_u16(s), 0)
    wf = w.to(torch.float32).numpy().astype(np.float64)
    sf = u16_to_f64(as_u16(s))[:, None]
    assert np.all(np.abs(wf - deq) <= sf / 2 * (1 + 1e-12) + 1e-30)
    codes = np.rint(deq / sf)
    assert codes.min() >= -8 and codes.max() <= 7
    am = np.abs(wf).argmax(axis=1)
    assert all(abs(codes[r, am[r]]) == 7 for r in range(6))


def test_quantizer_roundtrip_bounds():
    """Input-side quantiser: codes in [-8, 7], |w - q s| <= s/2, absmax maps to +-7."""
    w = normal_bf16((8, 256), 0.05, 0, 41)
    q, s = quantize_w4(w, 128)
    deq = oracle.dequant_w4(q.numpy(), as_u16(s), 128)
    wf = w.to(torch.float32).numpy().astype(np.float64)
    sf = np.repeat(u16_to_f64(as_u16(s)), 128, axis=1)
    assert np.all(np.abs(wf - deq) <= sf / 2 * (1 + 1e-12) + 1e-30)
    codes = np.rint(deq / sf)
    assert codes.min() >= -8 and codes.max() <= 7
    am = np.abs(wf).reshape(8, 2, 128).argmax(axis=2)
    for r in range(8):
        for g in range(2):
            assert abs(codes[r, g * 128 + am[r, g]]) == 7


def test_config_presets_match_pages_shapes():
    with open(os.path.join(GOLDEN, "page_shapes.json")) as f:
        g = json.load(f)
    for name in ("decode", "prefill", "skewed", "w4a16"):
        c = CONFIGS[name]
        assert (c.D, c.E, c.I, c.k) == (g["hidden"], g["experts"], g["expert_intermediate"],
                                         g["top_k"])
    assert CONFIGS["prefill"].T == g["tokens_per_core_batch"]
    assert CONFIGS["w4a16"].group == 128


def test_expert_hidden_and_down_match_numpy():
    """The per-expert halves: numpy matmuls + scipy logistic (bf16 and int4 weights)."""
    D, I, n = 32, 16, 5
    x = as_u16(normal_bf16((n, D), 1.0, 5, 51))
    gu = as_u16(normal_bf16((2 * I, D), D ** -0.5, 5, 52))
    dn = as_u16(normal_bf16((D, I), I ** -0.5, 5, 53))
    h = oracle.expert_hidden(x, gu)
    xf, G, Dn = u16_to_f64(x), u16_to_f64(gu), u16_to_f64(dn)
    g, u = xf @ G[:I].T, xf @ G[I:].T
    np.testing.assert_allclose(h, g * scipy.special.expit(g) * u, rtol=1e-12, atol=1e-14)
    o = oracle.expert_down(h, dn)
    np.testing.assert_allclose(o, h @ Dn.T, rtol=1e-12, atol=1e-14)
    # int4 weights: the same against the hand-dequantised matrices
    rng = np.random.default_rng(3)
    qg = rng.integers(-8, 8, size=(2 * I, D))
    sg = bf16_bits(rng.choice([0.5, 0.25, 0.125], size=(2 * I, D // 16)))
    qd = rng.integers(-8, 8, size=(D, I))
    sd = bf16_bits(rng.choice([0.5, 0.25, 0.125], size=(D, I // 16)))
    Gq = qg * np.repeat(u16_to_f64(sg), 16, axis=1)
    Dq = qd * np.repeat(u16_to_f64(sd), 16, axis=1)
    h4 = oracle.expert_hidden(x, pack_by_hand(qg), sg, group=16)
    g, u = xf @ Gq[:I].T, xf @ Gq[I:].T
    np.testing.assert_allclose(h4, g * scipy.special.expit(g) * u, rtol=1e-12, atol=1e-14)
    o4 = oracle.expert_down(h4, pack_by_hand(qd), sd, group=16)
    np.testing.assert_allclose(o4, h4 @ Dq.T, rtol=1e-12, atol=1e-14)


def test_combine_matches_fancy_index_sum():
    rng = np.random.default_rng(7)
    T, D, k = 11, 8, 3
    o = rng.standard_normal((T * k, D))
    osh = rng.standard_normal((T, D))
    inv = rng.permutation(T * k).astype(np.int32)
    y = oracle.combine(o, osh, inv, k)
    np.testing.assert_allclose(y, osh + o[inv.reshape(T, k)].sum(axis=1), rtol=1e-14, atol=1e-14)
    y0 = oracle.combine(o, None, inv, k)
    np.testing.assert_allclose(y0, o[inv.reshape(T, k)].sum(axis=1), rtol=1e-14, atol=1e-14)
