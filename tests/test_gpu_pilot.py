"""Next-layer routing prediction with read-ahead on the GPU (needs a GB300): on a two-layer stack, the
experts predicted for layer 1 from layer 0's normalised input equal the oracle's routing of layer 1's
router on that input (routing is exact); they are prefetched into layer 1's cache on a side stream, layer
1's cached forward (after waiting for those copies) still equals the resident forward bit for bit, and the
predicted experts that layer 1 then uses count as hits."""
from __future__ import annotations

import numpy as np
import pytest

import harness as H
import oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_expert_ffn_bias_gb300 as coli
    coli.build()
    return torch


def test_pilot_predicts_and_prefetches(torch_cuda):
    torch = torch_cuda
    import quantized_expert_ffn_bias_gb300 as coli
    from harness.device import DeviceLayer, to_dev
    from tests.test_gpu_cache import pinned_bank
    E, k, d, T = 16, 4, 1024, 2
    layers = [H.gen_layer(61, l, d=d, F=512, E=E, k=k, rho=2.5, qtype=H.Q_INT4_G128, bias="uniform:0.1")
              for l in range(2)]
    dls = [DeviceLayer(L_, 8) for L_ in layers]
    keep1, host1 = pinned_bank(torch, layers[1].experts)
    sb = coli.colibri_moe_cache_slot_bytes(dls[1].plan)
    S = 8
    cache1 = coli.Cache(dls[1].plan, S, 1.0, host1, torch.empty(S * sb, dtype=torch.uint8, device="cuda"), S * sb)
    ws_pilot = torch.empty(dls[1].plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    ws1 = torch.empty(dls[1].plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    recall = []
    for step in range(6):
        x = H.gen_x(61, step, T, d, H.X_BF16)
        h0 = to_dev(x, "cuda").view(torch.bfloat16).float().contiguous()
        n0 = torch.empty((T, d), dtype=torch.int16, device="cuda")
        coli.colibri_moe_rmsnorm_bf16(h0, T, d, 1e-6, n0, main)
        torch.cuda.synchronize()
        # layer 1's experts predicted from layer 0's input, prefetched on the side stream
        cache1.reset_stats()
        pred = cache1.pilot(T, n0, dls[1].router_w, dls[1].bias, ws_pilot, stream=side)
        done = torch.cuda.Event()
        done.record(side)
        n0_np = n0.cpu().numpy().view(np.uint16)
        idx_o, _, gap, _ = O.Oracle(layers[1]).route(n0_np)
        if np.all(gap >= O.NEAR_TIE):
            assert pred == sorted(set(idx_o.ravel().tolist())), "prediction differs from the oracle's routing"
        # layer 0, then layer 1 on its real input
        h1 = dls[0].forward(n0, residual=h0)
        n1 = torch.empty_like(n0)
        coli.colibri_moe_rmsnorm_bf16(h1, T, d, 1e-6, n1, main)
        main.wait_event(done)
        ref = dls[1].forward(n1).clone()
        out = torch.full_like(ref, float("nan"))
        cache1.forward(T, n1, dls[1].router_w, dls[1].bias, out, ws1, stream=main)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"step {step}: cached layer 1 differs from the resident forward"
        actual = sorted(set(dls[1].routing(T)[0].ravel().tolist()))
        both = len(set(pred) & set(actual))
        s = cache1.stats()
        assert s["predicted"] == len(pred)
        assert s["hits"] >= both, "predicted experts that layer 1 used must be hits"
        recall.append(both / len(actual))
    print(f"pilot: mean recall of layer 1's experts {np.mean(recall):.2f}")
    cache1.close()
    for dl in dls:
        dl.close()
    del keep1
