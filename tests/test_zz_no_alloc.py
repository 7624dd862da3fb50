"""The forward pass that uses the library's static scratch instead of a caller workspace.

It exists for callers that cannot allocate device memory (a host framework that
owns every allocation, or code regions where allocating is not allowed).  The
tests check it against the ordinary forward (same kernels, caller workspace) on
two calls in a row and against the oracle, with the output tolerances of the
parity tests; run a plan whose workspace is just under the 8 MiB limit (the
tensor-core path); and check that a plan too large for the static scratch is
refused.  This file is collected last
so that a failure here never hides the other tests.
"""
import numpy as np
import pytest

import harness as H
import oracle as O
from tests.gpu_parity import MAX_ABS_TOL, REL_L2_TOL, check_output, rel_l2

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
        # and against the oracle (tokens whose expert choice is not a near-tie)
        xn = H.gen_x(31, call, T, 1024, H.X_BF16)
        orc = O.Oracle(layer)
        gap = orc.route(xn)[2]
        toks = np.flatnonzero(gap >= O.NEAR_TIE).astype(np.int32)
        ref_o = orc.forward(xn, tokens=toks)
        if res is not None:
            ref_o = ref_o + res.cpu().numpy().astype(np.float64)[toks]
        check_output(a[toks], ref_o)
    # integer-dot inputs through the static scratch: the same kernels as the workspace forward
    dl.plan.set_idot(True)
    x = to_dev(H.gen_x(31, 7, 3, 1024, H.X_BF16), dl.device)
    ref = dl.forward(x).clone()
    out = torch.full((3, 1024), float("nan"), device=dl.device)
    dl.plan.forward_noalloc(3, x, dl.router_w, dl.bias, out, stream=torch.cuda.current_stream(dl.device))
    torch.cuda.synchronize()
    assert torch.equal(out, ref), "integer-dot forward through the static scratch differs"
    dl.plan.set_idot(False)
    dl.close()


def _largest_T_max_within(limit: int, **desc) -> int:
    import quantized_expert_ffn_bias_gb300 as coli
    lo, hi = 1, 1 << 14                 # plans are host-only: search the largest T_max that fits
    while lo < hi:
        mid = (lo + hi + 1) // 2
        p = coli.Plan(T_max=mid, **desc)
        fits = p.workspace_bytes <= limit
        p.close()
        lo, hi = (mid, hi) if fits else (lo, mid - 1)
    return lo


def test_noalloc_plan_at_the_scratch_limit(torch_cuda):
    """A plan whose workspace is just under 8 MiB (here a tensor-core sized token count), called after a
    workspace forward of another plan, matches the oracle on every token."""
    torch = torch_cuda
    import quantized_expert_ffn_bias_gb300 as coli
    from harness.device import DeviceLayer, to_dev
    layer = H.gen_layer(32, 0, d=1024, F=512, E=16, k=4, rho=2.5, qtype=H.Q_INT4_G128, bias="uniform:0.1",
                        F_shared=256)
    desc = dict(d=1024, d_ff=512, E=16, k=4, routed_scale=2.5, qtype=coli.COLI_Q_INT4_G128,
                xtype=coli.COLI_X_BF16, has_shared=True, shared_d_ff=256)
    T_max = _largest_T_max_within(8 << 20, **desc)
    assert T_max > 8                    # the limit is reached on the tensor-core path
    dl = DeviceLayer(layer, T_max)
    assert (8 << 20) - (1 << 16) < dl.plan.workspace_bytes <= (8 << 20)
    x = H.gen_x(32, 0, T_max, 1024, H.X_BF16)
    xd = to_dev(x, dl.device)
    dl.forward(xd)                      # leaves routing state of its own in the caller workspace
    out = torch.full((T_max, 1024), float("nan"), device=dl.device)
    dl.plan.forward_noalloc(T_max, xd, dl.router_w, dl.bias, out, stream=torch.cuda.current_stream(dl.device))
    torch.cuda.synchronize()
    a = out.cpu().numpy().astype(np.float64)
    orc = O.Oracle(layer)
    gap = orc.route(x)[2]
    toks = np.flatnonzero(gap >= O.NEAR_TIE).astype(np.int32)
    check_output(a[toks], orc.forward(x, tokens=toks))
    print(f"noalloc at T_max={T_max}: workspace {dl.plan.workspace_bytes} of {8 << 20} bytes")
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
