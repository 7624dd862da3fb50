"""Pins of the oracle's sparse-attention key selection (scores and top-k) to things other than itself:
closed forms, numpy's own contraction and stable sort, the causal mask, ties, equivariance and linearity.
Each pin takes the oracle library handle (so that planted-mistake copies can be checked too)."""
from __future__ import annotations

import numpy as np

import harness as H
import oracle as O


def _bf16(a) -> np.ndarray:
    return H.to_bf16_bits(np.asarray(a, np.float32))


def _f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _random(rng, T, L, Hh, d):
    q = _bf16(rng.standard_normal((T, Hh, d)))
    w = rng.standard_normal((T, Hh)).astype(np.float32)
    k = _bf16(rng.standard_normal((L, d)))
    return q, w, k


def pin_scalar_closed_form(L=None):
    """d = 1, one head, q = 1, w = 1: the score of key s is max(0, k_s), exactly."""
    n = 40
    kv = np.arange(n, dtype=np.float32) - 20.0          # exact in bf16
    q = _bf16(np.ones((1, 1, 1)))
    w = np.ones((1, 1), np.float32)
    sc = O.indexer_scores(q, w, _bf16(kv.reshape(n, 1)), pos0=n, L=L)
    np.testing.assert_array_equal(sc[0], np.maximum(kv, 0.0))
    idx, gap = O.indexer_topk(sc, 5, L=L)
    np.testing.assert_array_equal(idx[0], np.arange(n - 5, n))     # the five largest keys, ascending
    assert gap[0] == 1.0


def pin_relu_per_head(L=None):
    """Two heads with opposite queries: the score is w0 * (v.k) where v.k > 0 and w1 * (-v.k) elsewhere."""
    rng = np.random.default_rng(1)
    d, n = 8, 30
    v = _f64(_bf16(rng.standard_normal(d)))
    q = _bf16(np.stack([v, -v]).reshape(1, 2, d))
    w = np.array([[0.75, 2.5]], np.float32)
    kb = _bf16(rng.standard_normal((n, d)))
    dots = _f64(kb) @ v
    want = np.where(dots > 0, 0.75 * dots, 2.5 * -dots)
    sc = O.indexer_scores(q, w, kb, pos0=n, L=L)
    np.testing.assert_allclose(sc[0], want, rtol=1e-12, atol=1e-12)


def pin_scores_match_einsum(L=None):
    """The contraction against numpy's einsum on random inputs (no mask)."""
    rng = np.random.default_rng(2)
    T, n, Hh, d = 3, 50, 4, 16
    q, w, k = _random(rng, T, n, Hh, d)
    dots = np.einsum("thi,si->ths", _f64(q), _f64(k))
    want = np.einsum("th,ths->ts", w.astype(np.float64), np.maximum(dots, 0.0))
    sc = O.indexer_scores(q, w, k, pos0=n, L=L)
    np.testing.assert_allclose(sc, want, rtol=1e-12, atol=1e-12)


def pin_topk_matches_stable_sort(L=None):
    """Selection against numpy's stable sort by (score descending, key ascending), with planted ties."""
    rng = np.random.default_rng(3)
    T, n, k = 4, 300, 37
    sc = np.round(rng.standard_normal((T, n)) * 8) / 8          # many equal scores
    idx, gap = O.indexer_topk(sc, k, L=L)
    for t in range(T):
        order = np.lexsort((np.arange(n), -sc[t]))
        np.testing.assert_array_equal(idx[t], np.sort(order[:k]))
        assert gap[t] == sc[t][order[k - 1]] - sc[t][order[k]]


def pin_causal_mask(L=None):
    """Query t at position pos0 + t sees keys s <= pos0 + t; with fewer visible keys than topk, all of them
    are selected and the rest is -1."""
    rng = np.random.default_rng(4)
    T, n, Hh, d = 3, 20, 2, 8
    q, w, k = _random(rng, T, n, Hh, d)
    pos0 = 5
    sc = O.indexer_scores(q, w, k, pos0=pos0, L=L)
    for t in range(T):
        assert np.all(np.isneginf(sc[t, pos0 + t + 1:]))
        assert np.all(np.isfinite(sc[t, :pos0 + t + 1]))
    idx, gap = O.indexer_topk(sc, 10, L=L)
    for t in range(T):
        vis = pos0 + t + 1
        np.testing.assert_array_equal(idx[t, :vis], np.arange(vis))
        assert np.all(idx[t, vis:] == -1) and gap[t] == np.inf


def pin_ties_go_to_lower_key(L=None):
    """Identical keys give identical scores: the selection is the lowest key indices."""
    rng = np.random.default_rng(5)
    d, n = 8, 64
    k = np.repeat(_bf16(rng.standard_normal((1, d))), n, axis=0)
    q, w, _ = _random(rng, 2, 1, 3, d)
    sc = O.indexer_scores(q, w, k, pos0=n, L=L)
    idx, gap = O.indexer_topk(sc, 9, L=L)
    np.testing.assert_array_equal(idx, np.tile(np.arange(9), (2, 1)))
    assert np.all(gap == 0.0)


def pin_key_permutation_equivariance(L=None):
    """Permuting the keys permutes the scores; the selected set maps along (no ties in the draw)."""
    rng = np.random.default_rng(6)
    T, n, Hh, d = 2, 80, 4, 16
    q, w, k = _random(rng, T, n, Hh, d)
    perm = rng.permutation(n)
    sc = O.indexer_scores(q, w, k, pos0=n, L=L)
    scp = O.indexer_scores(q, w, k[perm], pos0=n, L=L)
    np.testing.assert_array_equal(scp, sc[:, perm])
    idx, _ = O.indexer_topk(sc, 11, L=L)
    idxp, _ = O.indexer_topk(scp, 11, L=L)
    for t in range(T):
        assert set(perm[idxp[t]].tolist()) == set(idx[t].tolist())


def pin_linear_in_head_weights(L=None):
    """Scores are linear in w: I(w1 + w2) = I(w1) + I(w2) (weights on a dyadic grid, so w1 + w2 is exact)."""
    rng = np.random.default_rng(7)
    T, n, Hh, d = 2, 40, 5, 8
    q, _, k = _random(rng, T, n, Hh, d)
    w1 = (rng.integers(-16, 17, (T, Hh)) / 8).astype(np.float32)
    w2 = (rng.integers(-16, 17, (T, Hh)) / 8).astype(np.float32)
    s1 = O.indexer_scores(q, w1, k, pos0=n, L=L)
    s2 = O.indexer_scores(q, w2, k, pos0=n, L=L)
    s12 = O.indexer_scores(q, w1 + w2, k, pos0=n, L=L)
    np.testing.assert_allclose(s12, s1 + s2, rtol=1e-12, atol=1e-12)


ALL_PINS = [pin_scalar_closed_form, pin_relu_per_head, pin_scores_match_einsum, pin_topk_matches_stable_sort,
            pin_causal_mask, pin_ties_go_to_lower_key, pin_key_permutation_equivariance, pin_linear_in_head_weights]
