"""The C ABI library loads and exports every symbol the headers declare; host-side plan validation (no GPU)."""
import ctypes
import glob
import os
import re

import pytest

import quantized_expert_ffn_bias_gb300 as coli

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    coli.build()
    return coli.lib()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names |= set(re.findall(r"COLI_API\s+[\w\s\*]+?\b(colibri_\w+)\s*\(", text))
    return sorted(names)


def test_headers_declare_functions():
    names = declared_functions()
    assert "colibri_moe_plan" in names and "colibri_moe_forward" in names
    assert len(names) >= 10


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), f"{name} declared in include/ but not exported"


def _desc(**kw):
    d = dict(T_max=4, d=512, d_ff=256, E=16, k=4, routed_scale=2.5, qtype=coli.COLI_Q_INT4_G128,
             xtype=coli.COLI_X_BF16, has_shared=0, shared_d_ff=0)
    d.update(kw)
    return coli.coli_moe_desc(**d)


def _plan(L, desc):
    h = ctypes.c_void_p()
    n = ctypes.c_size_t()
    rc = L.colibri_moe_plan(ctypes.byref(desc), ctypes.byref(h), ctypes.byref(n))
    return rc, h, n.value


def test_plan_valid_and_workspace_grows_with_T(L):
    rc, h, n1 = _plan(L, _desc(T_max=1))
    assert rc == coli.COLI_OK and n1 > 0
    L.colibri_moe_destroy(h)
    rc, h, n2 = _plan(L, _desc(T_max=64, has_shared=1, shared_d_ff=512))
    assert rc == coli.COLI_OK and n2 > n1
    L.colibri_moe_destroy(h)


def test_plan_reserves_split_router_weights_for_tensor_core_routing(L):
    """Plans that may run the tensor-core router (bf16 x, T_max >= 128) hold the router weights in three bf16
    parts, [3][E][d]; fp32-x plans and smaller T_max do not."""
    sizes = {}
    for xt in (coli.COLI_X_BF16, coli.COLI_X_F32):
        for T in (127, 128):
            rc, h, n = _plan(L, _desc(T_max=T, xtype=xt))
            assert rc == coli.COLI_OK
            L.colibri_moe_destroy(h)
            sizes[xt, T] = n
    grow_bf16 = sizes[coli.COLI_X_BF16, 128] - sizes[coli.COLI_X_BF16, 127]
    grow_f32 = sizes[coli.COLI_X_F32, 128] - sizes[coli.COLI_X_F32, 127]
    assert grow_bf16 - grow_f32 == 3 * 16 * 512 * 2
    assert sizes[coli.COLI_X_BF16, 127] == sizes[coli.COLI_X_F32, 127]


@pytest.mark.parametrize("bad,status", [
    (dict(k=0), coli.COLI_EINVAL),
    (dict(k=17), coli.COLI_EINVAL),            # k > E
    (dict(E=2048, k=4), coli.COLI_EUNSUPPORTED),
    (dict(T_max=0), coli.COLI_EINVAL),
    (dict(d=384), coli.COLI_EUNSUPPORTED),     # int4 needs multiples of 256
    (dict(qtype=7), coli.COLI_EUNSUPPORTED),
    (dict(xtype=5), coli.COLI_EUNSUPPORTED),
    (dict(has_shared=1, shared_d_ff=0), coli.COLI_EINVAL),
    (dict(has_shared=2, shared_d_ff=256), coli.COLI_EINVAL),
])
def test_plan_rejects(L, bad, status):
    rc, h, _ = _plan(L, _desc(**bad))
    assert rc == status
    assert L.colibri_moe_last_error()  # a message is set


def test_plan_null_arguments(L):
    h = ctypes.c_void_p()
    n = ctypes.c_size_t()
    assert L.colibri_moe_plan(None, ctypes.byref(h), ctypes.byref(n)) == coli.COLI_EINVAL
    assert L.colibri_moe_plan(ctypes.byref(_desc()), None, ctypes.byref(n)) == coli.COLI_EINVAL


def test_forward_refuses_unbound_plan_before_any_cuda_call(L):
    rc, h, n = _plan(L, _desc())
    assert rc == coli.COLI_OK
    rc = L.colibri_moe_forward(h, 1, 16, 16, 16, None, 16, 256, n, None)
    assert rc == coli.COLI_ESTATE
    L.colibri_moe_destroy(h)


def test_int8_allows_multiples_of_128(L):
    rc, h, _ = _plan(L, _desc(qtype=coli.COLI_Q_INT8_PC, d=384, d_ff=128))
    assert rc == coli.COLI_OK
    L.colibri_moe_destroy(h)
