"""Failure paths of the CUDA kernels, made to happen without any GPU fault (needs a GB300).

Every pipeline wait in the expert kernels is bounded; a test shortens the limit
to 2 ms and makes one TMA stage never arrive (colibri_moe_debug_inject), so the
waits run out.  The kernel must then record COLI_DEV_WAIT_TIMEOUT in the status
word, drain its copies, free its tensor memory and return; the next forward
without injection must be a normal one (parity with the oracle).  A planted
out-of-range expert id must be reported as COLI_DEV_BAD_EXPERT_ID, left out of
the output, and leave every other token's output unchanged.
"""
from __future__ import annotations

import time

import numpy as np
import pytest

import harness as H
import oracle as O
from tests.gpu_parity import check_output, run_layer_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_expert_ffn_bias_gb300 as coli
    coli.build()
    return torch


# decode (dequant-GEMV) and prefill (tensor-core) paths of a small int4 layer with a shared expert
CASES = [("decode", 4), ("prefill", 64)]


def _layer():
    return H.gen_layer(41, 0, d=1024, F=512, E=16, k=4, rho=2.5, qtype=H.Q_INT4_G128, bias="uniform:0.1",
                       F_shared=256)


@pytest.mark.parametrize("path,T", CASES)
def test_withheld_stage_times_out_and_the_next_forward_is_clean(torch_cuda, path, T):
    torch = torch_cuda
    import quantized_expert_ffn_bias_gb300 as coli
    from harness.device import DeviceLayer, to_dev
    layer = _layer()
    dl = DeviceLayer(layer, T)
    x = H.gen_x(41, 1, T, layer.d, H.X_BF16)
    xd = to_dev(x, dl.device)
    dl.plan.debug_inject(coli.COLI_INJECT_WITHHOLD_STAGE, 2.0)
    t0 = time.perf_counter()
    dl.forward(xd)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    status = dl.plan.check_status(dl.ws)
    assert status & coli.COLI_DEV_WAIT_TIMEOUT, f"status 0x{status:x}"
    assert dt < 5.0, f"the injected forward took {dt:.2f} s: the shortened wait limit did not end it"
    # injection off, fresh workspace: a normal forward, checked against the oracle
    dl.plan.debug_inject(0)
    dl.ws = torch.empty(dl.plan.workspace_bytes, dtype=torch.uint8, device=dl.device)
    rep = run_layer_parity(dl, layer, x)
    print(f"{path}: injected forward ended after {dt * 1e3:.1f} ms with status 0x{status:x}; "
          f"next forward rel_l2={rep.rel_l2:.2e}")
    dl.close()


@pytest.mark.parametrize("path,T", CASES)
def test_bad_expert_id_is_reported_and_left_out(torch_cuda, path, T):
    torch = torch_cuda
    import quantized_expert_ffn_bias_gb300 as coli
    from harness.device import DeviceLayer, to_dev
    layer = _layer()
    dl = DeviceLayer(layer, T)
    x = H.gen_x(41, 2, T, layer.d, H.X_BF16)
    xd = to_dev(x, dl.device)
    dl.plan.debug_inject(coli.COLI_INJECT_BAD_EXPERT_ID)
    out = dl.forward(xd)
    torch.cuda.synchronize()
    status = dl.plan.check_status(dl.ws)
    assert status == coli.COLI_DEV_BAD_EXPERT_ID, f"status 0x{status:x}"
    got = out.cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    # tokens 1..T-1 are untouched by the rejected pair of token 0
    orc = O.Oracle(layer)
    idx_o, _, gap, _ = orc.route(x)
    toks = np.array([t for t in range(1, T) if gap[t] >= O.NEAR_TIE], np.int32)
    check_output(got[toks], orc.forward(x, tokens=toks))
    # token 0 lost exactly its first chosen expert's contribution
    w0 = orc.route(x)[1][0]
    y0 = O.expert_ffn(layer.experts, int(idx_o[0, 0]), (x[0].astype(np.uint32) << 16).view(np.float32)
                      .astype(np.float64))
    if gap[0] >= O.NEAR_TIE:
        ref0 = orc.forward(x, tokens=np.array([0], np.int32))[0] - w0[0] * y0
        check_output(got[0], ref0)
    dl.plan.debug_inject(0)
    run_layer_parity(dl, layer, x)
    dl.close()
