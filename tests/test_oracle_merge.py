"""Pins for oracle.merge: composition of partial results over disjoint key sets."""

import numpy as np
import pytest

from oracle.attention import attention_fp64
from oracle.merge import merge_partials


def _qkv(seed, nq=37, nk=91, d=16):
    rng = np.random.default_rng(seed)
    return rng.normal(size=(nq, d)), rng.normal(size=(nk, d)) * 1.5, rng.normal(size=(nk, d))


@pytest.mark.parametrize("cuts", [[45], [10, 11, 60], [1, 2, 3, 4, 80]])
def test_chunked_softmax_merges_to_full(cuts):
    # attention over all keys == merge of attention over any partition of the keys
    q, k, v = _qkv(1)
    sm = 0.37
    o_full, lse_full = attention_fp64(q, k, v, sm, False)
    bounds = [0] + cuts + [k.shape[0]]
    parts = [attention_fp64(q, k[a:b], v[a:b], sm, False) for a, b in zip(bounds[:-1], bounds[1:])]
    o, lse = merge_partials([p[0] for p in parts], [p[1] for p in parts])
    np.testing.assert_allclose(o, o_full, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_full, rtol=0, atol=1e-12)


def test_single_part_is_identity():
    q, k, v = _qkv(2)
    o1, l1 = attention_fp64(q, k, v, 0.5, False)
    o, lse = merge_partials([o1], [l1])
    np.testing.assert_array_equal(o, o1)
    np.testing.assert_array_equal(lse, l1)


def test_order_invariant_and_empty_part_ignored():
    q, k, v = _qkv(3)
    a = attention_fp64(q, k[:50], v[:50], 0.3, False)
    b = attention_fp64(q, k[50:], v[50:], 0.3, False)
    empty_o = np.full_like(a[0], 123.0)              # any values: its weight is zero
    empty_l = np.full_like(a[1], -np.inf)
    o1, l1 = merge_partials([a[0], b[0]], [a[1], b[1]])
    o2, l2 = merge_partials([b[0], empty_o, a[0]], [b[1], empty_l, a[1]])
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)


def test_row_seen_by_no_part():
    o, lse = merge_partials([np.ones((2, 3))], [np.array([-np.inf, 0.0])])
    np.testing.assert_array_equal(o[0], 0.0)
    assert lse[0] == -np.inf
    np.testing.assert_array_equal(o[1], 1.0)
    assert lse[1] == 0.0


def test_two_equal_parts_closed_form():
    # two parts with equal lse and outputs x, y: o = (x + y) / 2, lse = lse + ln 2
    x, y = np.array([[1.0, -2.0]]), np.array([[3.0, 4.0]])
    o, lse = merge_partials([x, y], [np.array([0.25]), np.array([0.25])])
    np.testing.assert_allclose(o, [[2.0, 1.0]], atol=1e-15)
    np.testing.assert_allclose(lse, [0.25 + np.log(2.0)], atol=1e-15)
