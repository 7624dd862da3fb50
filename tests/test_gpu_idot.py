"""Integer-dot (IDOT) expert inputs on the GPU against the oracle's IDOT layer (needs a GB300).

Checks, per forward:
  * routing and grouping: as with the default inputs (routing reads x itself);
  * the down projection's input (colibri_moe_debug_hidden), every row: each value lies on its block's grid
    q * 2^(e-6) with |q| <= 127, and equals the oracle's code exactly wherever the oracle's fp64 h is farther
    than tau code steps from a rounding boundary (elsewhere: within one step; a block whose maximum is
    within a relative tau/64 of a power of two: within 1.5 steps);
  * the output: |gpu - oracle_idot| <= base error + the oracle's near-tie bound for the same tau, where
    the base error is the fp32 accumulation of the decode kernels (rel-L2 1e-5, max 1e-4 x rms) or the
    fp16 operands of the tensor-core kernels (the default parity bar);
  * IDOT is really on: the output is closer to the IDOT oracle than to the default layer by a wide margin;
  * switching IDOT off again gives the default path's parity.
tau: decode 0.01 code steps (integer block sums are exact; only fp32 sums over blocks differ from fp64);
prefill int8 0.02 (fp16 codes and IDOT values are exact operands, fp32 accumulation); prefill int4 0.25
(each dequantised weight is rounded to fp16, up to 2^-12 relative, which moves h by a few hundredths of a
code step, with tails).
"""
from __future__ import annotations

import gc

import numpy as np
import pytest

import harness as H
import oracle as O
from tests import pins
from tests.gpu_parity import MAX_ABS_TOL, REL_L2_TOL, check_routing, rel_l2, run_layer_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_expert_ffn_bias_gb300 as coli
    coli.build()
    yield
    gc.collect()
    torch.cuda.empty_cache()


CASES = [
    # (qtype, d, F, E, k, F_shared, bias, T values)
    (H.Q_INT4_G128, 1024, 512, 16, 4, 256, "uniform:0.1", (1, 3, 8)),
    (H.Q_INT4_G128, 768, 1280, 64, 6, 0, "zipf:0.05:1.1", (2, 8)),
    (H.Q_INT8_PC, 640, 256, 32, 8, 384, "normal:0.5", (1, 5, 8)),
    (H.Q_INT4_G128, 1024, 512, 16, 4, 256, "uniform:0.1", (9, 130)),
    (H.Q_INT4_G128, 768, 1280, 64, 6, 512, "zipf:0.05:1.1", (300,)),
    (H.Q_INT8_PC, 640, 256, 32, 8, 384, "normal:0.5", (17, 200)),
]


def _tau(qtype: int, T: int) -> float:
    if T <= 8:
        return 0.01
    return 0.02 if qtype == H.Q_INT8_PC else 0.25


def check_hidden(layer, x, hg, idx, pt, ps, tau, rows=None):
    """The down kernels' input of the given rows (default: every row) against the oracle's IDOT hidden
    step."""
    T, k = idx.shape
    P = T * k
    xf = pins.x_as_f64(x)
    worst = 0.0
    n_near = 0
    for r in (range(hg.shape[0]) if rows is None else rows):
        if r < P:
            t, bank, e, F = int(pt[r]), layer.experts, int(idx[pt[r], ps[r]]), layer.F
        else:
            t, bank, e, F = r - P, layer.shared, 0, layer.shared.F
        h, hq, amb = O.idot_hidden(bank, e, xf[t], tau)
        g = hg[r, :F].astype(np.float64)
        assert not hg[r, F:].any(), f"row {r}: values past the FFN size"
        for b in range(0, F, 32):
            m = np.abs(h[b:b + 32]).max()
            eb = int(np.floor(np.log2(m))) if m > 0 else -100
            st = 2.0 ** (max(eb, -100) - 6)
            gb, qb, ab = g[b:b + 32], hq[b:b + 32], amb[b:b + 32]
            if not np.any(ab == 1.5 * st):     # the block's exponent is certain: g on its grid
                q = gb / st
                assert np.array_equal(q, np.round(q)) and np.abs(q).max() <= 127, f"row {r} block {b}: off grid"
            exact = ab == 0
            assert np.array_equal(gb[exact], qb[exact]), \
                f"row {r} block {b}: codes differ away from rounding boundaries ({np.flatnonzero(gb != qb)[:4]})"
            if (~exact).any():
                d_ = np.abs(gb[~exact] - qb[~exact]) / st
                worst = max(worst, float(d_.max()))
                assert np.all(np.abs(gb[~exact] - qb[~exact]) <= ab[~exact] * (1 + 1e-12)), f"row {r} block {b}"
                n_near += int((gb[~exact] != qb[~exact]).sum())
    return worst, n_near


def run_idot(dl, layer, x, base_rel, base_abs, tokens=None):
    """IDOT forward of x on the device layer, checked against the oracle on `tokens` (default: all): the
    hidden rows of those tokens' pairs and shared-expert rows, then their outputs."""
    import torch
    from harness.device import to_dev
    T = x.shape[0]
    tau = _tau(layer.qtype, T)
    dl.plan.set_idot(True)
    out = dl.forward(to_dev(x, dl.device))
    torch.cuda.synchronize()
    assert dl.plan.check_status(dl.ws) == 0, "device status word set"
    out = out.cpu().numpy().astype(np.float64)
    idx, w, nt, off, pt, ps = dl.routing(T)
    orc = O.Oracle(layer)
    ov, n_near, n_mis, _ = check_routing(orc, x, idx, w, nt, off, pt, ps, layer.E)
    rows = T * layer.k + (T if layer.shared is not None else 0)
    Fmax = max(layer.F, layer.shared.F if layer.shared is not None else 0)
    hbuf = torch.empty((rows, Fmax), dtype=torch.float32, device=dl.device)
    dl.plan.debug_hidden(dl.ws, T, hbuf)
    torch.cuda.synchronize()
    sel = np.arange(T) if tokens is None else np.asarray(tokens)
    P = T * layer.k
    rows = None
    if tokens is not None:
        mine = np.isin(pt[:P], sel)
        rows = list(np.flatnonzero(mine)) + ([P + int(t) for t in sel] if layer.shared is not None else [])
    check_hidden(layer, x, hbuf.cpu().numpy(), idx, pt, ps, tau, rows)
    # output, on the tokens whose expert set matches the oracle's
    tok = np.intersect1d(np.flatnonzero(ov[:, 0] < 0), sel).astype(np.int32)
    ref, bound = orc.forward_idot(x, tau, tokens=tok)
    err = np.abs(out[tok] - ref)
    excess = np.maximum(err - bound, 0.0)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    assert float(np.linalg.norm(excess)) <= base_rel * float(np.linalg.norm(ref)), \
        f"rel-L2 beyond the near-tie bound {np.linalg.norm(excess) / np.linalg.norm(ref):.3e}"
    assert float(excess.max()) <= base_abs * rms, f"max beyond the near-tie bound {excess.max() / rms:.3e}"
    exact = orc.forward(x, tokens=tok)
    assert rel_l2(out[tok], ref) * 3 < rel_l2(out[tok], exact), "output not closer to the IDOT layer"
    dl.plan.set_idot(False)
    return len(tok)


@pytest.mark.parametrize("case", range(len(CASES)))
def test_idot_parity(case):
    from harness.device import DeviceLayer
    qt, d, F, E, k, Fs, bias, Ts = CASES[case]
    layer = H.gen_layer(400 + case, 0, d=d, F=F, E=E, k=k, rho=2.5, qtype=qt, bias=bias, F_shared=Fs)
    dl = DeviceLayer(layer, max(Ts))
    for i, T in enumerate(Ts):
        x = H.gen_x(400 + case, i, T, d, H.X_BF16)
        base = (1e-5, 1e-4) if T <= 8 else (REL_L2_TOL, MAX_ABS_TOL)
        run_idot(dl, layer, x, *base)
        # IDOT off again: the default path's parity
        rep = run_layer_parity(dl, layer, x)
        assert rep.set_mismatch == 0 or rep.near_ties >= rep.set_mismatch
    dl.close()
