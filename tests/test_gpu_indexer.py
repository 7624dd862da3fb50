"""Sparse-attention key selection on the GPU vs the fp64 oracle, through the C ABI (needs a GB300).

Scores are compared element by element within a tolerance derived from the fp32 accumulation
(128 exact bf16 products per head, 64 weighted heads): 2e-5 of the query's largest score.  The
selection is checked two ways: bit-exact against a stable sort of the GPU's own scores (score
descending, key ascending), and against the oracle's scores for validity (every selected key scores
at least the oracle's topk-th value minus the tolerance, every other visible key at most that value
plus it; where the oracle's gap at the boundary exceeds twice the tolerance the sets are equal).
"""
from __future__ import annotations

import numpy as np
import pytest

import harness as H
import oracle as O

pytestmark = pytest.mark.gpu

TOL = 2e-5


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_expert_ffn_bias_gb300 as coli
    coli.build()
    return torch


def run_indexer(torch, q, w, keys, pos0, topk):
    import quantized_expert_ffn_bias_gb300 as coli
    from harness.device import to_dev
    T, Hh, d = q.shape
    L = keys.shape[0]
    nbytes = coli.colibri_indexer_workspace_size(T, L)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.full((T, topk), -7, dtype=torch.int32, device="cuda")
    qd, wd, kd = to_dev(q, "cuda"), to_dev(w, "cuda"), to_dev(keys, "cuda")
    st = torch.cuda.current_stream()
    coli.colibri_indexer_topk(T, L, pos0, Hh, d, topk, qd, wd, kd, out, ws, nbytes, st)
    torch.cuda.synchronize()
    assert coli.colibri_indexer_check_status(ws, st) == 0
    scores = ws[256:256 + T * L * 4].cpu().numpy().view(np.float32).reshape(T, L)
    return out.cpu().numpy(), scores


def check_indexer(q, w, keys, pos0, topk, idx, scores_gpu):
    T = q.shape[0]
    L = keys.shape[0]
    orc = O.indexer_scores(q, w, keys, pos0)
    sel_o, gap_o = O.indexer_topk(orc, topk)
    report = {"boundary_keys": 0, "sets_equal": 0}
    for t in range(T):
        vis = min(L, pos0 + t + 1)
        # scores: masked keys are -inf on both sides; visible ones within the tolerance
        assert np.all(np.isneginf(scores_gpu[t, vis:]))
        atol = TOL * max(np.abs(orc[t, :vis]).max(), 1e-30)
        err = np.abs(scores_gpu[t, :vis].astype(np.float64) - orc[t, :vis]).max()
        assert err <= atol, f"query {t}: score error {err:.3e} > {atol:.3e}"
        m = min(topk, vis)
        sel = idx[t]
        assert np.all(sel[m:] == -1), "padding"
        s = sel[:m]
        assert np.all(np.diff(s) > 0) and s[0] >= 0 and s[-1] < vis, "ascending distinct visible keys"
        # exact against the GPU's own scores (score descending, key ascending)
        g = scores_gpu[t, :vis]
        order = np.lexsort((np.arange(vis), -g.astype(np.float64)))
        np.testing.assert_array_equal(s, np.sort(order[:m]))
        if vis <= topk:
            report["sets_equal"] += 1
            continue
        # valid against the oracle's scores
        tau = np.sort(orc[t, :vis])[::-1][topk - 1]
        chosen = np.zeros(vis, bool)
        chosen[s] = True
        assert orc[t, :vis][chosen].min() >= tau - atol
        assert orc[t, :vis][~chosen].max() <= tau + atol
        report["boundary_keys"] += int(np.sum(np.abs(orc[t, :vis] - tau) <= atol))
        if gap_o[t] > 2 * atol:
            np.testing.assert_array_equal(s, sel_o[t, :m])
            report["sets_equal"] += 1
    return report


SMALL = [
    # (T, L, pos0, topk): several 128-key tiles and a ragged tail; two query groups (T = 6); queries that
    # see fewer keys than topk (causal, pos0 small); topk larger than L
    (1, 300, 299, 64),
    (3, 1000, 997, 100),
    (6, 4097, 4091, 2048),
    (4, 2000, 30, 64),
    (2, 129, 128, 2048),
]


@pytest.mark.parametrize("case", range(len(SMALL)))
def test_indexer_small(torch_cuda, case):
    T, L, pos0, topk = SMALL[case]
    w = H.INDEXER
    q, hw, keys = w.q(T, 10 + case), w.w(T, 10 + case), w.keys(L, 10 + case)
    idx, sc = run_indexer(torch_cuda, q, hw, keys, pos0, topk)
    rep = check_indexer(q, hw, keys, pos0, topk, idx, sc)
    print(f"indexer T={T} L={L} pos0={pos0} topk={topk}: {rep}")


@pytest.mark.parametrize("T", [1, 4])
def test_indexer_full_size(torch_cuda, T):
    """The workload: T queries at the end of a 65,536-key context, 64 heads of 128, top-2048."""
    w = H.INDEXER
    q, hw, keys = w.q(T, 0), w.w(T, 0), w.keys()
    idx, sc = run_indexer(torch_cuda, q, hw, keys, w.L - T, w.topk)
    rep = check_indexer(q, hw, keys, w.L - T, w.topk, idx, sc)
    print(f"indexer full size T={T}: {rep}")


def test_indexer_equal_scores_take_lowest_keys(torch_cuda):
    """Every key identical: all visible scores tie, the boundary holds more keys than the candidate buffer,
    and the selection is the lowest key indices (the long way through the selection kernel)."""
    w = H.INDEXER
    T, L, topk = 2, 6000, 2048
    q, hw = w.q(T, 20), w.w(T, 20)
    keys = np.repeat(w.keys(1, 20), L, axis=0)
    idx, sc = run_indexer(torch_cuda, q, hw, keys, L - T, topk)
    np.testing.assert_array_equal(idx, np.tile(np.arange(topk, dtype=np.int32), (T, 1)))
    check_indexer(q, hw, keys, L - T, topk, idx, sc)
