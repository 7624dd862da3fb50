"""The forward pass that uses the library's static scratch instead of a caller workspace.

It exists for callers that cannot allocate device memory (a host framework that
owns every allocation, or code regions where allocating is not allowed).  The
test checks it against the ordinary forward (same kernels, caller workspace) on
two calls in a row, with the output tolerances of the parity tests, and that a
plan too large for the static scratch is refused.  This file is collected last
so that a failure here never hides the other tests.
"""
import numpy as np
import pytest

import harness as H
from tests.gpu_parity import MAX_ABS_TOL, REL_L2_TOL, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_expert_ffn_bias_gb300 as coli
    coli.build()
    return torch


def test_noalloc_forward_matches_workspace_forward(torch_cuda):
    torch = torch_cuda
    from harness.device import DeviceLayer, to_dev
    layer = H.gen_layer(31, 0, d=1024, F=512, E=16, k=4, rho=2.5, qtype=H.Q_INT4_G128, bias="uniform:0.1",
                        F_shared=256)
    dl = DeviceLayer(layer, 4)
    for call in range(2):                      # two calls in a row share (and reuse) the static scratch
        T = 4 - call
        x = to_dev(H.gen_x(31, call, T, 1024, H.X_BF16), dl.device)
        res = torch.randn((T, 1024), device=dl.device) if call == 1 else None
        ref = dl.forward(x, residual=res)
        out = torch.full((T, 1024), float("nan"), device=dl.device)
        dl.plan.forward_noalloc(T, x, dl.router_w, dl.bias, out, residual=res,
                                stream=torch.cuda.current_stream(dl.device))
        torch.cuda.synchronize()
        a = out.cpu().numpy().astype(np.float64)
        b = ref.cpu().numpy().astype(np.float64)
        assert np.isfinite(a).all()
        assert rel_l2(a, b) <= REL_L2_TOL
        assert np.abs(a - b).max() <= MAX_ABS_TOL * np.sqrt(np.mean(b ** 2))
    dl.close()


def test_noalloc_refuses_plans_beyond_the_static_scratch(torch_cuda):
    import quantized_expert_ffn_bias_gb300 as coli
    p = coli.Plan(T_max=2048, d=7168, d_ff=2048, E=256, k=8, routed_scale=2.5, qtype=coli.COLI_Q_INT4_G128,
                  xtype=coli.COLI_X_BF16)
    assert p.workspace_bytes > (8 << 20)
    with pytest.raises(coli.ColiError) as e:
        p.forward_noalloc(1, 16, 16, 16, 16)
    assert e.value.status == coli.COLI_EWORKSPACE
    assert "static scratch" in str(e.value)
    p.close()
