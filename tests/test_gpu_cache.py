"""Expert-slot cache with a host-memory tier on the GPU (needs a GB300): forwards whose experts come from
a small pool of device slots, filled from pinned host memory on misses, equal the resident forward bit for
bit (same kernels, same bytes); the hit / miss counts equal the host policy's on the same routing."""
from __future__ import annotations

import numpy as np
import pytest

import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_expert_ffn_bias_gb300 as coli
    coli.build()
    return torch


def pinned_bank(torch, bank):
    """Every expert of a bank in pinned host memory, as coli_expert descriptors (host pointers)."""
    import quantized_expert_ffn_bias_gb300 as coli

    def pin(a):
        a = np.ascontiguousarray(a)
        t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
        return t.pin_memory()

    keep = {n: tuple(pin(a) for a in (getattr(bank, n).q, getattr(bank, n).s, getattr(bank, n).z))
            for n in ("gate", "up", "down")}

    def qm(n, e):
        q, s, z = keep[n]
        return coli.qmat(q[e].data_ptr(), s[e].data_ptr(), z[e].data_ptr())

    return keep, [coli.coli_expert(qm("gate", e), qm("up", e), qm("down", e)) for e in range(bank.E)]


@pytest.mark.parametrize("qtype", [H.Q_INT4_G128, H.Q_INT8_PC])
def test_cached_forward_equals_resident(torch_cuda, qtype):
    torch = torch_cuda
    import quantized_expert_ffn_bias_gb300 as coli
    from harness.device import DeviceLayer, to_dev
    E, k = 16, 4
    layer = H.gen_layer(51, 0, d=1024, F=512, E=E, k=k, rho=2.5, qtype=qtype, bias="zipf:0.05:1.1", F_shared=256)
    dl = DeviceLayer(layer, 40)
    keep, host = pinned_bank(torch, layer.experts)
    sb = coli.colibri_moe_cache_slot_bytes(dl.plan)
    ws = torch.empty(dl.plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream()
    # decode: 8 slots for 16 experts (at most 8 distinct experts per forward at T <= 2, k = 4)
    S = 8
    slots = torch.empty(S * sb, dtype=torch.uint8, device="cuda")
    cache = coli.Cache(dl.plan, S, 1.0, host, slots, S * sb, shared=dl.shared.expert(0))
    sets = []
    for i, T in enumerate([1, 2, 2, 1, 2, 1, 1, 2, 2, 2, 1, 2, 2, 1, 2, 2]):
        xd = to_dev(H.gen_x(51, i, T, layer.d, H.X_BF16), "cuda")
        ref = dl.forward(xd).clone()
        out = torch.full_like(ref, float("nan"))
        cache.forward(T, xd, dl.router_w, dl.bias, out, ws, stream=st)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"forward {i} (T={T}) differs from the resident forward"
        sets.append(sorted(set(dl.routing(T)[0].ravel().tolist())))
    s = cache.stats()
    assert (s["hits"], s["misses"]) == coli.colibri_moe_cache_simulate(E, S, 1.0, sets)
    assert s["misses"] > 0 and s["evictions"] > 0 and s["lookups"] == sum(map(len, sets))
    assert s["bytes_copied"] == s["misses"] * sb
    print(f"cache (qtype {qtype}): {s}, hit rate {s['hits'] / s['lookups']:.2f}")
    # prefetch: an expert not resident is loaded ahead and then counts as a hit
    res = cache.resident(E)
    missing = [e for e in range(E) if res[e] < 0][:2]
    cache.reset_stats()
    cache.prefetch(missing, stream=st)
    assert cache.stats()["prefetched"] == len(missing)
    assert all(r >= 0 for r in (cache.resident(E)[e] for e in missing))
    # tensor-core path (T = 40): a cache with a slot for every expert
    cache2 = coli.Cache(dl.plan, E, 1.0, host, torch.empty(E * sb, dtype=torch.uint8, device="cuda"), E * sb,
                        shared=dl.shared.expert(0))
    for i, T in enumerate([40, 33]):
        xd = to_dev(H.gen_x(51, 100 + i, T, layer.d, H.X_BF16), "cuda")
        ref = dl.forward(xd).clone()
        out = torch.full_like(ref, float("nan"))
        cache2.forward(T, xd, dl.router_w, dl.bias, out, ws, stream=st)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"prefill forward {i} differs from the resident forward"
    # a forward that needs more experts than the cache has slots is refused
    small = coli.Cache(dl.plan, 2, 0.0, host, slots, S * sb, shared=dl.shared.expert(0))
    xd = to_dev(H.gen_x(51, 200, 2, layer.d, H.X_BF16), "cuda")
    with pytest.raises(coli.ColiError) as e:
        small.forward(2, xd, dl.router_w, dl.bias, torch.empty((2, layer.d), device="cuda"), ws, stream=st)
    assert e.value.status == coli.COLI_EUNSUPPORTED
    # host tier packed in the slot layout (one copy per miss)
    offs = coli.cache_slot_offsets(layer.d, layer.F, qtype)
    packed = torch.empty((E, sb), dtype=torch.uint8).pin_memory()
    pn = packed.numpy()
    for e in range(E):
        for j, (n, part) in enumerate((n, p) for n in ("gate", "up", "down") for p in ("q", "s", "z")):
            src = np.ascontiguousarray(getattr(getattr(layer.experts, n), part)[e]).view(np.uint8).ravel()
            pn[e, offs[j]:offs[j] + src.size] = src
    hp = []
    for e in range(E):
        b = packed.data_ptr() + e * sb
        q = [coli.qmat(b + offs[3 * m], b + offs[3 * m + 1], b + offs[3 * m + 2]) for m in range(3)]
        hp.append(coli.coli_expert(q[0], q[1], q[2]))
    cache3 = coli.Cache(dl.plan, S, 1.0, hp, slots, S * sb, shared=dl.shared.expert(0))
    for i, T in enumerate([2, 1, 2, 2]):
        xd = to_dev(H.gen_x(51, 300 + i, T, layer.d, H.X_BF16), "cuda")
        ref = dl.forward(xd).clone()
        out = torch.full_like(ref, float("nan"))
        cache3.forward(T, xd, dl.router_w, dl.bias, out, ws, stream=st)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"packed-tier forward {i} differs from the resident forward"
    assert cache3.stats()["bytes_copied"] == cache3.stats()["misses"] * sb
    # integer-dot inputs: the cached forward still runs the resident forward's kernels on slots
    dl.plan.set_idot(True)
    for i, (c, T) in enumerate([(cache3, 1), (cache3, 2), (cache2, 40)]):
        xd = to_dev(H.gen_x(51, 400 + i, T, layer.d, H.X_BF16), "cuda")
        ref = dl.forward(xd).clone()
        out = torch.full_like(ref, float("nan"))
        c.forward(T, xd, dl.router_w, dl.bias, out, ws, stream=st)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"integer-dot forward {i} (T={T}) differs from the resident forward"
    dl.plan.set_idot(False)
    for c in (cache, cache2, small, cache3):
        c.close()
    dl.close()
    del keep, packed
