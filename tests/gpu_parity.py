"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI and compare with the oracle."""
from __future__ import annotations

import dataclasses

import numpy as np

import harness as H
import oracle as O

REL_L2_TOL = 2e-3          # output: relative L2 error
MAX_ABS_TOL = 1e-2         # output: max |err| <= MAX_ABS_TOL * rms(out)
GATE_W_RTOL = 1e-5         # gate weights of tokens whose expert set matches


@dataclasses.dataclass
class ParityReport:
    T: int
    near_ties: int            # tokens the oracle flags as near-tie
    set_mismatch: int         # tokens whose GPU expert set differs (all must be near-ties)
    rel_l2: float
    max_abs_over_rms: float
    max_w_rel: float
    n_out_checked: int


def rel_l2(a, b) -> float:
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def check_routing(orc: O.Oracle, x: np.ndarray, gpu_idx, gpu_w, gpu_nt, gpu_off, gpu_pt, gpu_ps, E: int):
    """Bit-exact routing except oracle near-ties; bit-exact grouping of the GPU's own routing.
    Returns (override array for forward, near-tie count, mismatch count, max weight rel err)."""
    idx_o, w_o, gap_o, s_o = orc.route(x)
    T, k = idx_o.shape
    near = gap_o < O.NEAR_TIE
    same = np.all(gpu_idx == idx_o, axis=1)
    bad = ~same & ~near
    assert not bad.any(), f"routing differs on {bad.sum()} non-near-tie tokens, e.g. t={np.flatnonzero(bad)[:5]}: " \
                          f"gpu={gpu_idx[bad][:2]} oracle={idx_o[bad][:2]} gap={gap_o[bad][:2]}"
    # gate weights where the set matches
    wrel = np.abs(gpu_w[same] - w_o[same]) / np.abs(w_o[same])
    max_w_rel = float(wrel.max()) if wrel.size else 0.0
    assert max_w_rel <= GATE_W_RTOL, f"gate weights rel err {max_w_rel}"
    # the GPU's grouping equals the oracle's grouping of the GPU's routing (bit-exact)
    off_o, pt_o, ps_o, _ = O.permute(gpu_idx, E)
    assert np.array_equal(gpu_off, off_o), "expert offsets differ"
    assert np.array_equal(gpu_pt, pt_o), "pair_token differs"
    assert np.array_equal(gpu_ps, ps_o), "pair_slot differs"
    # override: where the sets differ (near-ties), the oracle recomputes with the GPU's set
    ov = np.full((T, k), -1, np.int32)
    ov[~same] = gpu_idx[~same]
    ov[same, 0] = -1
    return ov, int(near.sum()), int((~same).sum()), max_w_rel


def check_output(out_gpu: np.ndarray, out_ref: np.ndarray):
    e = rel_l2(out_gpu, out_ref)
    rms = float(np.sqrt(np.mean(out_ref ** 2)))
    m = float(np.abs(out_gpu - out_ref).max() / max(rms, 1e-300))
    assert e <= REL_L2_TOL, f"rel-L2 {e:.3e} > {REL_L2_TOL}"
    assert m <= MAX_ABS_TOL, f"max-abs/rms {m:.3e} > {MAX_ABS_TOL}"
    return e, m


def run_layer_parity(dl, layer, x: np.ndarray, tokens=None, residual=None) -> ParityReport:
    """Forward x through the device layer `dl`, compare routing, grouping and (sampled) outputs."""
    import torch
    from harness.device import to_dev
    T = x.shape[0]
    xd = to_dev(x, dl.device)
    res_d = to_dev(residual.astype(np.float32), dl.device) if residual is not None else None
    out = dl.forward(xd, residual=res_d)
    torch.cuda.synchronize()
    assert dl.plan.check_status(dl.ws) == 0, "device status word set"
    out = out.cpu().numpy().astype(np.float64)
    idx, w, nt, off, pt, ps = dl.routing(T)
    orc = O.Oracle(layer)
    ov, n_near, n_mis, wrel = check_routing(orc, x, idx, w, nt, off, pt, ps, layer.E)
    tokens = np.arange(T, dtype=np.int32) if tokens is None else np.asarray(tokens, np.int32)
    ref = orc.forward(x, tokens=tokens, sel_override=ov[tokens])
    if residual is not None:
        ref = ref + residual[tokens].astype(np.float64)
    e, m = check_output(out[tokens], ref)
    return ParityReport(T, n_near, n_mis, e, m, wrel, len(tokens))
