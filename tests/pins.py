"""Checks that pin the fp64 oracle to something other than itself.

Every pin takes an oracle library handle `L` (None = the real build) so that
the planted-mistake tests can run the same pins against broken copies of the
oracle and show that each mistake is caught.

Kinds of pin used here:
  * exhaustive / brute force (all bit patterns of a format, all expert subsets),
  * closed forms (experts whose dequantised weights form a scaled selection
    matrix, so the FFN reduces to indexing; k = E routing),
  * library routines (numpy float16 decoding, numpy matmul, numpy stable argsort),
  * invariants (sum of gate weights = routed scale, token independence,
    permutation equivariance, quantiser error bounds).
"""
from __future__ import annotations

import itertools

import numpy as np

import harness as H
import oracle as O

# ----------------------------------------------------------------------------- helpers


def silu(a):
    return a / (1.0 + np.exp(-a))


def x_as_f64(x):
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


def dense_dequant(m: H.QMat) -> np.ndarray:
    """Dequantise a whole packed matrix with numpy (float16 decoding by numpy itself)."""
    if m.qtype == H.Q_INT4_G128:
        lo = (m.q & 15).astype(np.int64)
        hi = (m.q >> 4).astype(np.int64)
        codes = np.stack([lo, hi], axis=-1).reshape(m.q.shape[:-1] + (m.K,))
        zl = (m.z & 15).astype(np.int64)
        zh = (m.z >> 4).astype(np.int64)
        zeros = np.stack([zl, zh], axis=-1).reshape(m.z.shape[:-1] + (-1,))[..., : m.K // 128]
        scales = m.s.view(np.float16).astype(np.float64)
        return (codes - np.repeat(zeros, 128, axis=-1)) * np.repeat(scales, 128, axis=-1)
    return (m.q.astype(np.int64) - m.z.astype(np.int64)[..., None]) * m.s.astype(np.float64)[..., None]


def selection_qmat(qtype: int, N: int, K: int, rng: np.random.Generator):
    """A packed [N][K] matrix whose dequantised value is exactly c[n] at (n, col[n]) and 0 elsewhere.

    Scales and zero-points vary per group (int4) or per row (int8), so the
    closed form only holds if every index of the format is read correctly.
    Returns (QMat, col[N], c[N]).
    """
    col = rng.integers(0, K, size=N)
    m = H.empty_qmat(qtype, N, K)
    c = np.zeros(N)
    if qtype == H.Q_INT4_G128:
        G = K // 128
        scale_choices = np.array([0.25, 0.5, 1.0, 2.0, 0.125])
        sc = scale_choices[rng.integers(0, len(scale_choices), size=(N, G))]
        zp = rng.integers(6, 10, size=(N, G))            # mult in [-6, 6] always fits in [0, 15]
        codes = np.repeat(zp, 128, axis=1).astype(np.int64)
        mult = rng.integers(1, 7, size=N) * rng.choice([-1, 1], size=N)
        for n in range(N):
            g = col[n] // 128
            codes[n, col[n]] = zp[n, g] + mult[n]
            c[n] = mult[n] * sc[n, g]
        m.q[:] = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
        m.s[:] = sc.astype(np.float16).view(np.uint16)
        zpad = np.zeros((N, 2 * H.zp_bytes(K)), np.int64)
        zpad[:, :G] = zp
        m.z[:] = (zpad[:, 0::2] | (zpad[:, 1::2] << 4)).astype(np.uint8)
    else:
        sc = rng.choice([0.5, 0.25, 1.5, 0.75], size=N).astype(np.float32)
        zp = rng.integers(100, 156, size=N)
        codes = np.repeat(zp[:, None], K, axis=1)
        mult = rng.integers(1, 90, size=N) * rng.choice([-1, 1], size=N)
        codes[np.arange(N), col] = zp + mult
        c = mult * sc.astype(np.float64)
        m.q[:] = codes.astype(np.uint8)
        m.s[:] = sc
        m.z[:] = zp.astype(np.uint8)
    return m, col, c


def stack_banks(mats_per_expert, qtype, d, F):
    """Build an ExpertBank from a list of (gate, up, down) QMats."""
    E = len(mats_per_expert)

    def st(i):
        ms = [m[i] for m in mats_per_expert]
        return H.QMat(qtype, ms[0].N, ms[0].K, np.ascontiguousarray(np.stack([m.q for m in ms])),
                      np.ascontiguousarray(np.stack([m.s for m in ms])),
                      np.ascontiguousarray(np.stack([m.z for m in ms])))
    return H.ExpertBank(qtype, E, d, F, st(0), st(1), st(2))


def selection_bank(qtype, E, d, F, rng):
    """E experts built from selection matrices, with their closed-form parameters."""
    mats, params = [], []
    for _ in range(E):
        g, gc, gv = selection_qmat(qtype, F, d, rng)
        u, uc, uv = selection_qmat(qtype, F, d, rng)
        dn, dc, dv = selection_qmat(qtype, d, F, rng)
        mats.append((g, u, dn))
        params.append((gc, gv, uc, uv, dc, dv))
    return stack_banks(mats, qtype, d, F), params


def selection_ffn(params, x):
    """Closed form of a selection-matrix expert on x [d]: y[m] = cd[m] * h[col_d[m]]."""
    gc, gv, uc, uv, dc, dv = params
    h = silu(gv * x[gc]) * (uv * x[uc])
    return dv * h[dc]


def tiny_layer(seed=0, qtype=H.Q_INT8_PC, E=8, k=2, d=256, F=128, rho=1.0, bias="uniform:0.1", F_shared=0):
    return H.gen_layer(seed, 0, d=d, F=F, E=E, k=k, rho=rho, qtype=qtype, bias=bias, F_shared=F_shared)


# ----------------------------------------------------------------------------- number formats


def pin_f16_all_patterns(L=None):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([O.f16_to_double(int(b), L) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def pin_bf16_all_patterns(L=None):
    bits = np.arange(65536, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        ref = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    got = np.array([O.bf16_to_double(int(b), L) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def _bf16_neighbours(v: float):
    f = np.float32(v)
    b = int(f.view(np.uint32)) & 0xFFFF0000
    cands = []
    for delta in (-0x10000, 0, 0x10000, 0x20000):
        c = (b + delta) & 0xFFFFFFFF
        cands.append(float(np.uint32(c).view(np.float32)))
    return cands


def pin_round_to_bf16(L=None):
    rng = np.random.default_rng(7)
    vals = list(rng.standard_normal(2000) * 10.0 ** rng.integers(-30, 30, 2000))
    # exact midpoints between bf16 neighbours: ties go to the even mantissa
    for b in (0x3F80, 0x3F81, 0x4049, 0xC123, 0x0081):
        lo = float(np.uint32(b << 16).view(np.float32))
        hi = float(np.uint32((b + 1) << 16).view(np.float32))
        vals.append((lo + hi) / 2.0)
    for v in vals:
        r = O.round_to_bf16(float(v), L)
        f = np.float32(r)
        assert float(f) == r and (int(f.view(np.uint32)) & 0xFFFF) == 0, (v, r)   # representable
        best = min(abs(c - v) for c in _bf16_neighbours(v))
        assert abs(r - v) == best, (v, r)                                        # nearest
        ties = [c for c in _bf16_neighbours(v) if abs(c - v) == best]
        if len(set(ties)) > 1:                                                   # tie -> even
            assert (int(f.view(np.uint32)) >> 16) % 2 == 0, (v, r)


def pin_int4_unpack_all_bytes(L=None):
    """All 256 byte values: low nibble is the even input, high nibble the odd one."""
    K = 1024
    m = H.empty_qmat(H.Q_INT4_G128, 1, K)
    m.q[0, :256] = np.arange(256, dtype=np.uint8)
    m.q[0, 256:] = np.arange(256, dtype=np.uint8)[::-1]
    m.s[:] = np.float16(1.0).view(np.uint16)
    w = O.dequant_row(m, H.Q_INT4_G128, 0, L=L)
    b = m.q[0].astype(np.int64)
    assert np.array_equal(w[0::2], b & 15)
    assert np.array_equal(w[1::2], b >> 4)


def pin_int4_group_scales_and_zeros(L=None):
    """Each group of 128 inputs uses its own fp16 scale and its own zero nibble (low nibble = even group)."""
    K = 128 * 6
    m = H.empty_qmat(H.Q_INT4_G128, 1, K)
    m.q[0, :] = 0xFF                                  # every code 15
    scales = np.array([1.0, 0.5, 0.25, 2.0, 4.0, 0.125], np.float16)
    zeros = np.array([1, 2, 3, 4, 5, 6])
    m.s[0] = scales.view(np.uint16)
    m.z[0] = (zeros[0::2] | (zeros[1::2] << 4)).astype(np.uint8)
    w = O.dequant_row(m, H.Q_INT4_G128, 0, L=L)
    want = np.repeat((15 - zeros) * scales.astype(np.float64), 128)
    assert np.array_equal(w, want)


def pin_int8_per_row(L=None):
    rng = np.random.default_rng(3)
    m = H.empty_qmat(H.Q_INT8_PC, 3, 256)
    m.q[:] = rng.integers(0, 256, size=(3, 256), dtype=np.uint8)
    m.s[:] = np.array([0.5, 0.0625, 3.0], np.float32)
    m.z[:] = np.array([0, 128, 255], np.uint8)
    for n in range(3):
        w = O.dequant_row(m, H.Q_INT8_PC, n, L=L)
        assert np.array_equal(w, (m.q[n].astype(np.int64) - int(m.z[n])) * float(m.s[n]))


def pin_quantiser_roundtrip(L=None):
    """Quantise random rows with the generator's quantiser, dequantise with the oracle: error <= s/2 inside
    the representable range and <= s at the clipped ends."""
    rng = np.random.default_rng(11)
    w = (rng.standard_normal((8, 1024)) * 0.05).astype(np.float32)
    for qt in (H.Q_INT4_G128, H.Q_INT8_PC):
        m = H.quantize(w, qt)
        for n in range(8):
            deq = O.dequant_row(m, qt, n, L=L)
            if qt == H.Q_INT4_G128:
                s = np.repeat(m.s[n].view(np.float16).astype(np.float64), 128)
            else:
                s = np.full(1024, float(m.s[n]))
            err = np.abs(deq - w[n].astype(np.float64))
            assert np.all(err <= s * (1 + 1e-6)), (qt, n, err.max())
            assert np.mean(err <= 0.5 * s * (1 + 1e-6)) > 0.97, (qt, n)


# ----------------------------------------------------------------------------- routing


def _tiny_route(L, **kw):
    layer = tiny_layer(**kw)
    x = H.gen_x(0, 0, 16, layer.d, H.X_F32)
    return layer, x, O.Oracle(layer, L).route(x)


def pin_logits_match_matmul(L=None):
    layer, x, (idx, w, gap, s) = _tiny_route(L)
    z = x.astype(np.float64) @ layer.router_w.astype(np.float64).T
    assert np.allclose(s, 1.0 / (1.0 + np.exp(-z)), rtol=0, atol=1e-13)


def pin_topk_bruteforce(L=None):
    """The selected set maximises the sum of biased scores over all C(E,k) subsets."""
    for k in (1, 2, 3):
        layer, x, (idx, w, gap, s) = _tiny_route(L, k=k)
        u = s + layer.bias.astype(np.float64)
        for t in range(x.shape[0]):
            best = max(itertools.combinations(range(layer.E), k), key=lambda c: sum(u[t, list(c)]))
            assert tuple(idx[t]) == tuple(sorted(best)), (k, t, idx[t], best)


def pin_gate_weights(L=None):
    """g = rho * s / sum(s) over the selected set, with the UNBIASED s; so sum(g) = rho."""
    for rho in (1.0, 2.5):
        layer, x, (idx, w, gap, s) = _tiny_route(L, rho=rho, k=3)
        z = x.astype(np.float64) @ layer.router_w.astype(np.float64).T
        s_np = 1.0 / (1.0 + np.exp(-z))
        for t in range(x.shape[0]):
            sel = s_np[t, idx[t]]
            assert np.allclose(w[t], rho * sel / sel.sum(), rtol=1e-12, atol=0)
        assert np.allclose(w.sum(1), rho, rtol=1e-12, atol=0)


def pin_k_equals_E(L=None):
    layer, x, (idx, w, gap, s) = _tiny_route(L, k=8)
    assert np.array_equal(idx, np.tile(np.arange(8), (16, 1)))
    z = x.astype(np.float64) @ layer.router_w.astype(np.float64).T
    s_np = 1.0 / (1.0 + np.exp(-z))
    assert np.allclose(w, 1.0 * s_np / s_np.sum(1, keepdims=True), rtol=1e-12, atol=0)
    assert np.all(np.isinf(gap))


def pin_bias_selects_only(L=None):
    """A large bias forces an expert into every token's set but does not change its weight formula."""
    layer, x, (idx, w, gap, s) = _tiny_route(L, bias="spike:6:10.0", k=2, rho=2.5)
    z = x.astype(np.float64) @ layer.router_w.astype(np.float64).T
    s_np = 1.0 / (1.0 + np.exp(-z))
    for t in range(16):
        assert 6 in idx[t]
        j = list(idx[t]).index(6)
        assert np.isclose(w[t, j], 2.5 * s_np[t, 6] / s_np[t, idx[t]].sum(), rtol=1e-12, atol=0)


def pin_tie_goes_to_lower_id(L=None):
    layer = tiny_layer()
    layer.router_w[5] = layer.router_w[2]
    layer.bias[:] = 0.0
    layer.bias[2] = layer.bias[5] = 1.0
    x = H.gen_x(0, 0, 16, layer.d, H.X_F32)
    layer.k = 1
    idx, w, gap, s = O.Oracle(layer, L).route(x)
    assert np.all(idx[:, 0] == 2)
    assert np.all(gap == 0.0)


def pin_gap(L=None):
    layer, x, (idx, w, gap, s) = _tiny_route(L, k=3)
    u = np.sort(s + layer.bias.astype(np.float64), axis=1)[:, ::-1]
    assert np.array_equal(gap, u[:, 2] - u[:, 3])


def pin_permutation_vs_argsort(L=None):
    rng = np.random.default_rng(5)
    for T, k, E in ((16, 2, 8), (37, 8, 256), (1, 8, 256), (64, 4, 4)):
        idx = np.sort(np.array([rng.choice(E, size=k, replace=False) for _ in range(T)]), axis=1).astype(np.int32)
        off, pt, ps, po = O.permute(idx, E, L=L)
        flat = idx.reshape(-1)
        assert np.array_equal(off, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
        order = np.argsort(flat, kind="stable")
        assert np.array_equal(pt, order // k)
        assert np.array_equal(ps, order % k)
        inv = np.empty_like(order)
        inv[order] = np.arange(order.size)
        assert np.array_equal(po.reshape(-1), inv)


# ----------------------------------------------------------------------------- the expert FFN and the layer


def pin_selection_expert_closed_form(L=None):
    rng = np.random.default_rng(1)
    for qt, d, F in ((H.Q_INT4_G128, 512, 256), (H.Q_INT8_PC, 256, 384), (H.Q_INT4_G128, 256, 768)):
        bank, params = selection_bank(qt, 2, d, F, rng)
        for e in range(2):
            xt = rng.standard_normal(d)
            y = O.expert_ffn(bank, e, xt, L=L)
            assert np.allclose(y, selection_ffn(params[e], xt), rtol=1e-13, atol=1e-300)


def _selection_layer(rng, qt=H.Q_INT4_G128, E=6, k=2, d=256, F=256, rho=2.5, with_shared=True):
    bank, params = selection_bank(qt, E, d, F, rng)
    shared, sparams = (None, None)
    if with_shared:
        shared, sp = selection_bank(qt, 1, d, F, rng)
        sparams = sp[0]
    router = (rng.standard_normal((E, d)) / np.sqrt(d)).astype(np.float32)
    bias = (rng.standard_normal(E) * 0.1).astype(np.float32)
    layer = H.Layer(d, F, E, k, rho, qt, router, bias, bank, shared, F if with_shared else 0)
    return layer, params, sparams


def pin_layer_closed_form(L=None):
    """out[t] = sum_j g_j * FFN_{e_j}(x_t) + FFN_shared(x_t) with closed-form experts."""
    rng = np.random.default_rng(2)
    for with_shared in (False, True):
        layer, params, sparams = _selection_layer(rng, with_shared=with_shared)
        x = H.to_bf16_bits(rng.standard_normal((5, layer.d)).astype(np.float32))
        orc = O.Oracle(layer, L)
        idx, w, gap, s = orc.route(x)
        out = orc.forward(x)
        xf = x_as_f64(x)
        for t in range(5):
            want = sum(w[t, j] * selection_ffn(params[idx[t, j]], xf[t]) for j in range(layer.k))
            if with_shared:
                want = want + selection_ffn(sparams, xf[t])
            assert np.allclose(out[t], want, rtol=1e-12, atol=1e-14), (with_shared, t)


def pin_shared_only(L=None):
    """Routed experts whose codes all equal their zero-point contribute nothing: out = shared expert."""
    rng = np.random.default_rng(4)
    layer, params, sparams = _selection_layer(rng, qt=H.Q_INT8_PC, with_shared=True)
    for m in (layer.experts.gate, layer.experts.up, layer.experts.down):
        m.q[:] = m.z[..., None]
    x = H.to_bf16_bits(rng.standard_normal((3, layer.d)).astype(np.float32))
    out = O.Oracle(layer, L).forward(x)
    xf = x_as_f64(x)
    for t in range(3):
        assert np.allclose(out[t], selection_ffn(sparams, xf[t]), rtol=1e-13, atol=0)


def pin_dense_equivalence(L=None):
    """The grouped (batch-union) layer equals the dense sum over ALL experts with a 0/1 selection mask,
    computed with numpy matmuls on numpy-dequantised weights."""
    for qt in (H.Q_INT8_PC, H.Q_INT4_G128):
        layer = tiny_layer(qtype=qt, k=3, F_shared=128)
        x = H.gen_x(0, 1, 16, layer.d, H.X_BF16)
        orc = O.Oracle(layer, L)
        idx, w, gap, s = orc.route(x)
        out = orc.forward(x)
        xf = x_as_f64(x)
        Wg, Wu, Wd = (dense_dequant(m) for m in (layer.experts.gate, layer.experts.up, layer.experts.down))
        G = np.zeros((16, layer.E))
        for t in range(16):
            G[t, idx[t]] = w[t]
        want = np.zeros((16, layer.d))
        for e in range(layer.E):
            h = silu(xf @ Wg[e].T) * (xf @ Wu[e].T)
            want += G[:, e:e + 1] * (h @ Wd[e].T)
        Sg, Su, Sd = (dense_dequant(m)[0] for m in (layer.shared.gate, layer.shared.up, layer.shared.down))
        want += (silu(xf @ Sg.T) * (xf @ Su.T)) @ Sd.T
        assert np.allclose(out, want, rtol=1e-10, atol=1e-12), (qt, np.abs(out - want).max())


def pin_token_independence_and_equivariance(L=None):
    layer = tiny_layer(F_shared=128)
    x = H.gen_x(0, 2, 16, layer.d, H.X_BF16)
    orc = O.Oracle(layer, L)
    full = orc.forward(x)
    sub = np.array([13, 2, 7], np.int32)
    assert np.array_equal(orc.forward(x, tokens=sub), full[sub])
    one = np.stack([orc.forward(x[t:t + 1])[0] for t in range(16)])
    assert np.array_equal(one, full)
    perm = np.random.default_rng(9).permutation(16)
    assert np.array_equal(orc.forward(np.ascontiguousarray(x[perm])), full[perm])


def pin_override_uses_given_set(L=None):
    layer = tiny_layer(k=2)
    x = H.gen_x(0, 3, 4, layer.d, H.X_F32)
    orc = O.Oracle(layer, L)
    idx, w, gap, s = orc.route(x)
    ov = np.array([[0, 1], [-1, 0], [3, 7], [-1, 0]], np.int32)
    out = orc.forward(x, sel_override=ov)
    base = orc.forward(x)
    xf = x.astype(np.float64)
    for t in (0, 2):
        sel = ov[t]
        g = 1.0 * s[t, sel] / s[t, sel].sum()
        want = sum(g[j] * O.expert_ffn(layer.experts, sel[j], xf[t], L=L) for j in range(2))
        assert np.allclose(out[t], want, rtol=1e-13, atol=0)
    assert np.array_equal(out[[1, 3]], base[[1, 3]])


# ----------------------------------------------------------------------------- RMSNorm and stacked layers


def pin_rmsnorm(L=None):
    d = 64
    for c in (1.0, -3.0, 1e-3, 250.0):
        h = np.full((1, d), c)
        n = O.rmsnorm_bf16(h, 1e-6, L=L)
        want = float(np.float32(c / np.sqrt(c * c + 1e-6)))
        assert np.allclose(n, want, rtol=2 ** -8, atol=0)
    rng = np.random.default_rng(12)
    h = rng.standard_normal((4, d))
    n1 = O.rmsnorm_bf16(h, 0.0, L=L)
    for a in (0.25, 8.0, 1024.0):                    # scale invariance (exact for powers of two, eps = 0)
        assert np.array_equal(O.rmsnorm_bf16(h * a, 0.0, L=L), n1)
    want = h / np.sqrt((h * h).mean(1, keepdims=True))
    assert np.all(np.abs(n1 - want) <= np.abs(want) * 2 ** -8)
    assert np.abs(n1 - want).max() > 0                # and it really is rounded to bf16


def pin_stacked_zero_experts_keep_residual(L=None):
    layers = []
    for l in range(3):
        layer = tiny_layer(seed=l)
        for m in (layer.experts.gate, layer.experts.up, layer.experts.down):
            m.q[:] = m.z[..., None]
        layers.append(layer)
    x = H.gen_x(0, 4, 8, 256, H.X_BF16)
    h = O.stacked_forward(layers, x, 1e-6, L=L)
    assert np.array_equal(h, x_as_f64(x))


def pin_stacked_selection_layers(L=None):
    """Two stacked closed-form layers: h1 = x + MoE1(bf16(rms(x))), h2 = h1 + MoE2(bf16(rms(h1)))."""
    rng = np.random.default_rng(21)
    l1, p1, s1 = _selection_layer(rng, E=4, k=2, with_shared=True)
    l2, p2, s2 = _selection_layer(rng, E=4, k=2, with_shared=False)
    x = H.to_bf16_bits(rng.standard_normal((3, l1.d)).astype(np.float32))
    h = O.stacked_forward([l1, l2], x, 1e-6, L=L)
    hh = x_as_f64(x)
    for layer, params, sp in ((l1, p1, s1), (l2, p2, s2)):
        n = hh / np.sqrt((hh * hh).mean(1, keepdims=True) + 1e-6)
        n = np.array([[O.round_to_bf16(v) for v in row] for row in n])
        idx, w, gap, s = O.Oracle(layer).route(O.bf16_bits_of(n))
        out = np.zeros_like(hh)
        for t in range(3):
            out[t] = sum(w[t, j] * selection_ffn(params[idx[t, j]], n[t]) for j in range(layer.k))
            if sp is not None:
                out[t] += selection_ffn(sp, n[t])
        hh = hh + out
    assert np.allclose(h, hh, rtol=1e-12, atol=1e-14)


# ----------------------------------------------------------------------------- integer-dot (IDOT) inputs


def mx8_brute(v):
    """Brute force of the IDOT block rule: e by integer search (2^e <= max|v| < 2^(e+1), e >= -100), then for
    each value the code among all of -127..127 nearest to v / 2^(e-6), a tie going to the even code."""
    v = np.asarray(v, np.float64)
    m = float(np.abs(v).max())
    e = -100
    if m > 0.0:
        e = 0
        while 2.0 ** e > m:
            e -= 1
        while 2.0 ** (e + 1) <= m:
            e += 1
        e = max(e, -100)
    step = 2.0 ** (e - 6)
    codes = np.arange(-127, 128, dtype=np.float64)
    out = np.empty_like(v)
    for i, x in enumerate(v):
        dist = np.abs(codes * step - x)
        best = np.flatnonzero(dist == dist.min())
        pick = best[0] if len(best) == 1 else [b for b in best if int(codes[b]) % 2 == 0][0]
        out[i] = codes[pick] * step
    return out, e


def pin_mx8_closed_forms(L=None):
    # max |v| = 1: the step is 2^-6 and multiples of it are kept exactly
    v = np.array([1.0] + [k / 64.0 for k in range(-31, 31)][:31])
    vq, amb, e = O.mx8_block(v, L=L)
    assert e == 0 and np.array_equal(vq, v)
    # half steps go to the even code; negative values mirror positive ones
    v = np.array([1.0, 0.5 / 64, 1.5 / 64, 2.5 / 64, -2.5 / 64, -0.5 / 64, 126.5 / 64] + [0.0] * 25)
    vq, _, e = O.mx8_block(v, L=L)
    assert e == 0
    assert np.array_equal(vq[:7], np.array([64, 0, 2, 2, -2, 0, 126]) / 64.0)
    # codes saturate at +-127: 1.999 / 2^-6 rounds to 128
    vq, _, e = O.mx8_block(np.array([1.999, -1.999] + [0.25] * 30), L=L)
    assert e == 0 and vq[0] == 127 / 64.0 and vq[1] == -127 / 64.0 and vq[2] == 0.25
    # zeros, and blocks below 2^-100, become zeros
    vq, _, e = O.mx8_block(np.zeros(32), L=L)
    assert e == -100 and not vq.any()
    vq, _, e = O.mx8_block(np.full(32, 2.0 ** -110), L=L)
    assert e == -100 and not vq.any()
    # scaling the block by 2^j scales the result by 2^j
    rng = np.random.default_rng(21)
    v = rng.standard_normal(32)
    base, _, e0 = O.mx8_block(v, L=L)
    for j in (-9, -1, 1, 13):
        vq, _, e = O.mx8_block(v * 2.0 ** j, L=L)
        assert e == e0 + j and np.array_equal(vq, base * 2.0 ** j)


def pin_mx8_brute_force(L=None):
    """Random blocks (several magnitudes, exact ties and saturating maxima planted) against brute force; the
    error of every value is at most half a step, or one step where the code saturated."""
    rng = np.random.default_rng(22)
    for trial in range(120):
        scale = 2.0 ** rng.integers(-30, 30)
        v = rng.standard_normal(32) * scale
        if trial % 3 == 1:      # plant exact half steps
            m = float(np.abs(v).max())
            e = int(np.floor(np.log2(m)))
            st = 2.0 ** (e - 6)
            v[1:6] = (rng.integers(-120, 120, 5) + 0.5) * st
        if trial % 5 == 2:      # plant a maximum that saturates
            m = float(np.abs(v).max())
            e = int(np.floor(np.log2(m)))
            v[0] = 1.995 * 2.0 ** e
            v[1:] = np.clip(v[1:], -1.9 * 2.0 ** e, 1.9 * 2.0 ** e)
        vq, _, e = O.mx8_block(v, L=L)
        want, we = mx8_brute(v)
        assert e == we and np.array_equal(vq, want), trial
        st = 2.0 ** (e - 6)
        err = np.abs(vq - v)
        sat = np.abs(v) / st >= 127.5
        assert np.all(err[~sat] <= st / 2) and np.all(err[sat] <= st)


def pin_mx8_near_tie_allowance(L=None):
    """tau marks values within tau code steps of a half step (one step) and whole blocks whose maximum is
    within a relative tau/64 of a power of two (1.5 steps); nothing else."""
    st = 2.0 ** -6
    v = np.array([1.5, 3.5 * st, (3.5 + 0.01) * st, (10.5 - 0.004) * st, 0.3 * st, 7.0 * st] + [0.0] * 26)
    _, amb, e = O.mx8_block(v, tau=0.005, L=L)
    assert e == 0
    assert np.array_equal(amb[:6], np.array([0.0, st, 0.0, st, 0.0, 0.0])) and not amb[6:].any()
    # maximum exactly a power of two: the kernel's value may sit just below it (exponent one less)
    _, amb, _ = O.mx8_block(np.array([1.0, 0.3, -0.2] + [0.0] * 29), tau=0.005, L=L)
    assert np.all(amb == 1.5 * st)
    # maximum just under the next power of two
    _, amb, _ = O.mx8_block(np.array([2.0 * (1 - 1e-6), 0.3] + [0.0] * 30), tau=0.005, L=L)
    assert np.all(amb == 1.5 * st)
    # tau = 0: no allowance anywhere
    _, amb, _ = O.mx8_block(np.array([1.0, 3.5 * st] + [0.0] * 30), tau=0.0, L=L)
    assert not amb.any()


def pin_idot_expert_brute_force(L=None):
    """An IDOT expert against numpy matmuls on numpy-dequantised weights with brute-force block
    quantisation of x and of h; the near-tie bound against its definition."""
    rng = np.random.default_rng(23)
    for qt, d, F in ((H.Q_INT4_G128, 256, 128), (H.Q_INT8_PC, 256, 192)):
        layer = tiny_layer(qtype=qt, E=3, d=d, F=F)
        Wg, Wu, Wd = (dense_dequant(m) for m in (layer.experts.gate, layer.experts.up, layer.experts.down))
        for e in range(3):
            xt = x_as_f64(H.to_bf16_bits(rng.standard_normal(d).astype(np.float32)))
            tau = 0.01
            y, yb = O.expert_ffn_idot(layer.experts, e, xt, tau, L=L)
            xq = np.concatenate([mx8_brute(xt[b:b + 32])[0] for b in range(0, d, 32)])
            h = silu(Wg[e] @ xq) * (Wu[e] @ xq)
            hq, amb = [], []
            for b in range(0, F, 32):
                q, eb = mx8_brute(h[b:b + 32])
                hq.append(q)
                st = 2.0 ** (eb - 6)
                s = np.abs(h[b:b + 32]) / st
                a = np.where((np.abs(s - np.floor(s) - 0.5) < tau) & (s < 127.5), st, 0.0)
                r = np.abs(h[b:b + 32]).max() / 2.0 ** eb
                if r - 1 < tau / 64 or 2 - r < tau / 64:
                    a[:] = 1.5 * st
                amb.append(a)
            hq, amb = np.concatenate(hq), np.concatenate(amb)
            oh, ohq, oamb = O.idot_hidden(layer.experts, e, xt, tau, L=L)
            assert np.allclose(oh, h, rtol=1e-12, atol=1e-15), (qt, e)
            assert np.array_equal(ohq, hq) and np.array_equal(oamb, amb), (qt, e)
            assert np.allclose(y, Wd[e] @ hq, rtol=1e-11, atol=1e-13), (qt, e)
            assert np.allclose(yb, np.abs(Wd[e]) @ amb, rtol=1e-11, atol=1e-15), (qt, e)


def pin_idot_layer_combination(L=None):
    """The IDOT layer = routing of x itself (the exact layer's selection and gate weights) times the IDOT
    experts, plus the shared expert with weight 1; the bound combines with the same weights; and the IDOT
    layer stays within its quantisation error of the exact layer."""
    for qt in (H.Q_INT8_PC, H.Q_INT4_G128):
        layer = tiny_layer(qtype=qt, k=3, F_shared=128)
        x = H.gen_x(0, 4, 6, layer.d, H.X_BF16)
        orc = O.Oracle(layer, L)
        idx, w, gap, s = orc.route(x)
        out, bound = orc.forward_idot(x, 0.01)
        exact = orc.forward(x)
        xf = x_as_f64(x)
        for t in range(6):
            want = np.zeros(layer.d)
            wb = np.zeros(layer.d)
            for j in range(layer.k):
                y, yb = O.expert_ffn_idot(layer.experts, int(idx[t, j]), xf[t], 0.01, L=L)
                want += w[t, j] * y
                wb += w[t, j] * yb
            y, yb = O.expert_ffn_idot(layer.shared, 0, xf[t], 0.01, L=L)
            assert np.allclose(out[t], want + y, rtol=1e-12, atol=1e-14), (qt, t)
            assert np.allclose(bound[t], wb + yb, rtol=1e-12, atol=1e-16), (qt, t)
        # 8-bit inputs: a few per cent of the output's spread at most
        rel = np.abs(out - exact).max() / np.abs(exact).max()
        assert 1e-5 < rel < 0.05, (qt, rel)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
