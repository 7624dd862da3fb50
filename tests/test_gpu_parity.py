"""CUDA path vs the fp64 oracle, through the C ABI (needs a GB300)."""
from __future__ import annotations

import gc

import numpy as np
import pytest

import harness as H
import oracle as O
from tests import pins
from tests.gpu_parity import check_output, run_layer_parity

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


def _dl(layer, T_max, xtype=H.X_BF16):
    from harness.device import DeviceLayer
    return DeviceLayer(layer, T_max, xtype=xtype)


# ------------------------------------------------------------------ medium shapes, every output checked

MEDIUM = [
    # (qtype, d, F, E, k, F_shared, bias, T values)
    (H.Q_INT4_G128, 1024, 512, 16, 4, 0, "uniform:0.1", (1, 3, 8)),
    (H.Q_INT4_G128, 1024, 512, 16, 4, 256, "normal:0.5", (1, 2, 5, 8)),
    (H.Q_INT8_PC, 512, 384, 12, 3, 0, "uniform:0.1", (1, 4, 7)),
    (H.Q_INT8_PC, 640, 256, 32, 8, 384, "zero", (3, 8)),
    (H.Q_INT4_G128, 768, 1280, 64, 6, 512, "zipf:0.05:1.1", (1, 6)),
]


# tensor-core (T > 8) path: every output checked.  Covers shared experts with d_ff below and above the
# routed one (the hidden row stride is the larger), int8 with a shared expert, int4 group counts that
# are not multiples of 8 (per-stage scale loads instead of 8-group batches), token counts that are not
# multiples of 16 (MMA N rounding) and experts with more than one 128-token chunk.
PREFILL = [
    # (qtype, d, F, E, k, F_shared, bias, T values)
    (H.Q_INT4_G128, 1024, 512, 16, 4, 256, "uniform:0.1", (9, 130)),
    (H.Q_INT4_G128, 768, 1280, 64, 6, 512, "zipf:0.05:1.1", (64, 300)),
    (H.Q_INT8_PC, 640, 256, 32, 8, 384, "normal:0.5", (17, 200)),
    (H.Q_INT4_G128, 2048, 1024, 8, 2, 1024, "spike:3:2.0", (257,)),
]


@pytest.mark.parametrize("case", range(len(PREFILL)))
def test_prefill_shapes(case):
    qt, d, F, E, k, Fs, bias, Ts = PREFILL[case]
    layer = H.gen_layer(200 + case, 0, d=d, F=F, E=E, k=k, rho=2.5, qtype=qt, bias=bias, F_shared=Fs)
    dl = _dl(layer, max(Ts))
    for i, T in enumerate(Ts):
        x = H.gen_x(200 + case, i, T, d, H.X_BF16)
        rep = run_layer_parity(dl, layer, x)
        assert rep.set_mismatch == 0 or rep.near_ties >= rep.set_mismatch
    dl.close()


@pytest.mark.parametrize("case", range(len(MEDIUM)))
def test_medium_shapes(case):
    qt, d, F, E, k, Fs, bias, Ts = MEDIUM[case]
    layer = H.gen_layer(100 + case, 0, d=d, F=F, E=E, k=k, rho=2.5, qtype=qt, bias=bias, F_shared=Fs)
    dl = _dl(layer, max(Ts))
    for i, T in enumerate(Ts):
        x = H.gen_x(100 + case, i, T, d, H.X_BF16)
        rep = run_layer_parity(dl, layer, x)
        assert rep.set_mismatch == 0 or rep.near_ties >= rep.set_mismatch
    dl.close()


def test_tiny_workload_f32_input():
    w = H.WORKLOADS["tiny"]
    layer = w.layer(0)
    x = w.x(16)
    dl = _dl(layer, 16, xtype=H.X_F32)
    run_layer_parity(dl, layer, x)
    # every token alone (T=1) gives the same routing and the same output within tolerance
    for t in (0, 7, 15):
        run_layer_parity(dl, layer, np.ascontiguousarray(x[t:t + 1]))
    dl.close()


# ------------------------------------------------------------------ edge cases

def test_all_tokens_to_one_expert():
    layer = H.gen_layer(7, 0, d=512, F=256, E=16, k=2, rho=1.0, qtype=H.Q_INT4_G128, bias="spike:5:10.0")
    dl = _dl(layer, 8)
    x = H.gen_x(7, 0, 8, 512, H.X_BF16)
    run_layer_parity(dl, layer, x)
    idx = dl.routing(8)[0]
    assert np.all((idx == 5).any(axis=1))
    dl.close()


def test_k_equals_E():
    layer = H.gen_layer(8, 0, d=256, F=256, E=8, k=8, rho=1.0, qtype=H.Q_INT8_PC, bias="uniform:0.1", F_shared=128)
    dl = _dl(layer, 5)
    x = H.gen_x(8, 0, 5, 256, H.X_BF16)
    run_layer_parity(dl, layer, x)
    dl.close()


def test_selection_experts_closed_form():
    """Experts whose weights select one input per row: the GPU output equals the closed form."""
    rng = np.random.default_rng(3)
    for qt in (H.Q_INT4_G128, H.Q_INT8_PC):
        layer, params, sparams = pins._selection_layer(rng, qt=qt, E=6, k=2, d=256, F=256, with_shared=True)
        dl = _dl(layer, 4)
        x = H.to_bf16_bits(rng.standard_normal((4, 256)).astype(np.float32))
        from harness.device import to_dev
        import torch
        out = dl.forward(to_dev(x, dl.device))
        torch.cuda.synchronize()
        out = out.cpu().numpy().astype(np.float64)
        idx, w = dl.routing(4)[:2]
        xf = pins.x_as_f64(x)
        want = np.stack([sum(float(w[t, j]) * pins.selection_ffn(params[idx[t, j]], xf[t]) for j in range(2)) +
                         pins.selection_ffn(sparams, xf[t]) for t in range(4)])
        check_output(out, want)
        dl.close()


def test_residual_input_and_output_alias():
    layer = H.gen_layer(9, 0, d=512, F=256, E=16, k=4, rho=2.5, qtype=H.Q_INT4_G128, bias="uniform:0.1")
    dl = _dl(layer, 4)
    x = H.gen_x(9, 0, 4, 512, H.X_BF16)
    res = H.normal(H.key(9, 50), 4 * 512).reshape(4, 512)
    run_layer_parity(dl, layer, x, residual=res)
    dl.close()


def test_argument_errors():
    import torch
    import quantized_expert_ffn_bias_gb300 as coli
    layer = H.gen_layer(10, 0, d=256, F=256, E=8, k=2, rho=1.0, qtype=H.Q_INT8_PC, bias="zero")
    dl = _dl(layer, 4)
    x = torch.zeros((4, 256), dtype=torch.int16, device="cuda")
    out = torch.empty((4, 256), dtype=torch.float32, device="cuda")
    p = dl.plan
    with pytest.raises(coli.ColiError) as e:
        p.forward(5, x, dl.router_w, dl.bias, out, dl.ws)              # T > T_max
    assert e.value.status == coli.COLI_EINVAL
    with pytest.raises(coli.ColiError) as e:
        p.forward(0, x, dl.router_w, dl.bias, out, dl.ws)              # T = 0
    assert e.value.status == coli.COLI_EINVAL
    with pytest.raises(coli.ColiError) as e:
        p.forward(4, x, dl.router_w, dl.bias, out, dl.ws, workspace_bytes=16)
    assert e.value.status == coli.COLI_EWORKSPACE
    with pytest.raises(coli.ColiError) as e:
        p.forward(4, x.data_ptr() + 2, dl.router_w, dl.bias, out, dl.ws)
    assert e.value.status == coli.COLI_EALIGN
    with pytest.raises(coli.ColiError) as e:
        p.forward(4, None, dl.router_w, dl.bias, out, dl.ws)
    assert e.value.status == coli.COLI_EINVAL
    # a misaligned weight pointer is refused at bind time
    bad = dl.experts.expert(0)
    bad.gate.q = bad.gate.q + 1
    with pytest.raises(coli.ColiError) as e:
        p.bind_experts([bad] + [dl.experts.expert(i) for i in range(1, 8)])
    assert e.value.status == coli.COLI_EALIGN
    # an unbound plan refuses to run
    q = coli.Plan(T_max=4, d=256, d_ff=256, E=8, k=2, routed_scale=1.0, qtype=coli.COLI_Q_INT8_PC,
                  xtype=coli.COLI_X_BF16)
    with pytest.raises(coli.ColiError) as e:
        q.forward(4, x, dl.router_w, dl.bias, out, dl.ws)
    assert e.value.status == coli.COLI_ESTATE
    # nothing above launched a kernel: the status word is clean
    dl.forward(x)
    torch.cuda.synchronize()
    assert p.check_status(dl.ws) == 0
    dl.close()
