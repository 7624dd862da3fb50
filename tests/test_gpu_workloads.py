"""The five workloads at full size on the GPU vs the oracle (routing of every token, sampled outputs).

Inputs follow the GLM-5.2-class shapes of the pages (d=7168, d_ff=2048, 256
experts, top-8, int4 group-128 / int8 per-channel), seeded and synthetic.
"""
from __future__ import annotations

import gc

import numpy as np
import pytest

import harness as H
import oracle as O
from tests.gpu_parity import check_output, rel_l2, run_layer_parity

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


def _sample(T, n, seed):
    if T <= n:
        return np.arange(T, dtype=np.int32)
    return np.sort(np.random.default_rng(seed).choice(T, size=n, replace=False)).astype(np.int32)


CHUNK = 128   # tokens per tensor-core chunk of one expert


def _chunk_cover(dl, T: int, has_shared: bool, seed: int, n_heavy: int = 2):
    """Tokens whose outputs reach every 128-token chunk of the n_heavy most loaded experts (one token of
    each chunk, from the GPU's own grouping of this input) and the shared expert's last chunk.  Returns
    (tokens, description of the chosen chunks)."""
    _, _, _, off, pt, _ = dl.routing(T)
    loads = np.diff(off)
    heavy = np.argsort(-loads, kind="stable")[:n_heavy]
    rng = np.random.default_rng(seed)
    toks, desc = set(), []
    for e in heavy:
        n_ch = (int(loads[e]) + CHUNK - 1) // CHUNK
        for c in range(n_ch):
            lo, hi = int(off[e]) + c * CHUNK, min(int(off[e + 1]), int(off[e]) + (c + 1) * CHUNK)
            toks.add(int(pt[rng.integers(lo, hi)]))
        desc.append(f"expert {int(e)}: {int(loads[e])} tokens, {n_ch} chunks")
    if has_shared:                 # the shared expert's rows are the tokens in order
        last = (T - 1) // CHUNK
        toks.add(int(rng.integers(last * CHUNK, T)))
        desc.append(f"shared expert: chunk {last} (tokens {last * CHUNK}..{T - 1})")
    return np.array(sorted(toks), np.int32), "; ".join(desc)


def _release(dl):
    import torch
    dl.close()
    del dl
    gc.collect()
    torch.cuda.empty_cache()


def test_decode_T1_T4():
    from harness.device import DeviceLayer
    w = H.WORKLOADS["decode"]
    layer = w.layer(0)
    dl = DeviceLayer(layer, 4)
    for T in (1, 4):
        for stream in range(3):
            x = w.x(T, stream)
            rep = run_layer_parity(dl, layer, x)
            print(f"decode T={T}: rel_l2={rep.rel_l2:.2e} max/rms={rep.max_abs_over_rms:.2e} near_ties={rep.near_ties}")
    # integer-dot inputs at full size, as the bench times them (T=1): every hidden row and the output
    from tests.test_gpu_idot import run_idot
    for stream in range(2):
        run_idot(dl, layer, w.x(1, 10 + stream), 1e-5, 1e-4)
    # the expert cache at the bench's configuration (every expert in pinned host memory, 32 device slots):
    # the cached forward equals the resident forward bit for bit
    import torch
    import quantized_expert_ffn_bias_gb300 as coli
    from harness.device import to_dev
    from tests.test_gpu_cache import pinned_bank
    keep, host = pinned_bank(torch, layer.experts)
    sb = coli.colibri_moe_cache_slot_bytes(dl.plan)
    S = 4 * layer.k
    cache = coli.Cache(dl.plan, S, 1.0, host, torch.empty(S * sb, dtype=torch.uint8, device=dl.device), S * sb)
    ws = torch.empty(dl.plan.workspace_bytes, dtype=torch.uint8, device=dl.device)
    for step in range(6):
        xd = to_dev(w.x(1, 20 + step), dl.device)
        ref = dl.forward(xd).clone()
        out = torch.full_like(ref, float("nan"))
        cache.forward(1, xd, dl.router_w, dl.bias, out, ws, stream=torch.cuda.current_stream(dl.device))
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"cached decode step {step} differs from the resident forward"
    s = cache.stats()
    assert s["lookups"] == 6 * layer.k and s["misses"] > 0
    cache.close()
    del keep
    _release(dl)


def test_mtp_verify_T3_shared_and_overlap():
    from harness.device import DeviceLayer
    w = H.WORKLOADS["mtp_verify"]
    layer = w.layer(0)
    dl = DeviceLayer(layer, 3)
    overlaps = []
    for stream in range(4):
        x = w.x(3, stream)
        rep = run_layer_parity(dl, layer, x)
        idx = dl.routing(3)[0]
        sets = [set(r) for r in idx]
        overlaps += [len(sets[a] & sets[b]) / layer.k for a in range(3) for b in range(a + 1, 3)]
        assert len(set().union(*sets)) < 3 * layer.k  # batch-union really merged something on average
    print(f"mtp verify: mean pairwise expert overlap {np.mean(overlaps):.2f}")
    _release(dl)


def test_prefill_T2048_skewed():
    from harness.device import DeviceLayer, to_dev
    w = H.WORKLOADS["prefill"]
    layer = w.layer(0)
    dl = DeviceLayer(layer, 2048)
    x = w.x(2048, 0)
    dl.forward(to_dev(x, dl.device))
    cover, desc = _chunk_cover(dl, 2048, True, 5)
    toks = np.union1d(_sample(2048, 48, 3), cover).astype(np.int32)
    rep = run_layer_parity(dl, layer, x, tokens=toks)
    off = dl.routing(2048)[3]
    loads = np.diff(off)
    print(f"prefill: loads min={loads.min()} max={loads.max()} idle={int((loads == 0).sum())} "
          f"rel_l2={rep.rel_l2:.2e} near_ties={rep.near_ties}; {len(toks)} outputs checked, covering {desc}")
    assert loads.max() > 400
    # integer-dot inputs at full size (the bench's IDOT prefill line): the chunk-covering sample of tokens
    from tests.gpu_parity import MAX_ABS_TOL, REL_L2_TOL
    from tests.test_gpu_idot import run_idot
    cover_i, _ = _chunk_cover(dl, 2048, True, 6)
    run_idot(dl, layer, x, REL_L2_TOL, MAX_ABS_TOL, tokens=np.union1d(_sample(2048, 16, 7), cover_i))
    _release(dl)


def test_stacked_six_layers_T256():
    """Six layers h <- h + MoE(bf16(RMSNorm(h))), alternating int4 / int8: each layer's GPU output
    matches the oracle fed the GPU's own layer input; RMSNorm matches to one bf16 rounding."""
    import torch
    import quantized_expert_ffn_bias_gb300 as coli
    from harness.device import DeviceLayer, to_dev
    w = H.WORKLOADS["stacked"]
    T, eps = 256, w.rmsnorm_eps
    x = w.x(T, 0)
    h = to_dev(x, "cuda").view(torch.bfloat16).float().contiguous()
    n = torch.empty((T, w.d), dtype=torch.int16, device="cuda")
    toks = _sample(T, 24, 4)
    for l in range(w.n_layers):
        layer = w.layer(l)
        dl = DeviceLayer(layer, T)
        coli.colibri_moe_rmsnorm_bf16(h, T, w.d, eps, n, torch.cuda.current_stream())
        torch.cuda.synchronize()
        n_np = n.cpu().numpy().view(np.uint16)
        h_np = h.cpu().numpy().astype(np.float64)
        n_ref = O.bf16_bits_of(O.rmsnorm_bf16(h_np, eps))
        diff = n_np != n_ref
        assert diff.mean() < 1e-3, f"layer {l}: rmsnorm differs on {diff.sum()} elements"
        if diff.any():
            assert np.all(np.abs(n_np[diff].astype(np.int32) - n_ref[diff].astype(np.int32)) == 1)
        dl.forward(n, residual=h)
        cover, desc = _chunk_cover(dl, T, False, 10 + l)
        lt = np.union1d(toks, cover).astype(np.int32)
        rep = run_layer_parity(dl, layer, n_np, tokens=lt, residual=h_np.astype(np.float32))
        print(f"stacked layer {l} ({'int4' if layer.qtype == 0 else 'int8'}): rel_l2={rep.rel_l2:.2e} "
              f"near_ties={rep.near_ties}; {len(lt)} outputs checked, covering {desc}")
        h_next = torch.empty_like(h)
        dl.forward(n, out=h_next, residual=h)
        torch.cuda.synchronize()
        h = h_next
        _release(dl)
