"""fp64 CPU oracle of the quantized sparse MoE layer forward (ctypes wrapper).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  It shares no
code with the CUDA library: the arithmetic lives in ``oracle_moe.c`` and is
plain loops in double precision (see that file's header for the steps and the
page passages they follow).

Inputs are "layer-like" objects with the attributes produced by the seeded
generator (``d, F, E, k, rho, qtype, router_w, bias, experts, shared``), where
each expert bank holds ``gate/up/down`` packed matrices with a leading expert
axis.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_moe.c")
_SRC_INDEXER = os.path.join(_HERE, "oracle_indexer.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle_moe.so")
_lock = threading.Lock()
_lib = None

Q_INT4_G128, Q_INT8_PC = 0, 1
X_BF16, X_F32 = 0, 1
NEAR_TIE = 1e-5   # k-th minus (k+1)-th biased score below this counts as a near-tie


class _QMat(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("s", ctypes.c_void_p), ("z", ctypes.c_void_p)]


class _Expert(ctypes.Structure):
    _fields_ = [("gate", _QMat), ("up", _QMat), ("down", _QMat)]


class _Desc(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int), ("F", ctypes.c_int), ("E", ctypes.c_int), ("k", ctypes.c_int),
                ("rho", ctypes.c_double), ("qtype", ctypes.c_int), ("xtype", ctypes.c_int),
                ("has_shared", ctypes.c_int), ("F_shared", ctypes.c_int), ("qtype_shared", ctypes.c_int)]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP over tokens, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or \
            os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(_SRC), os.path.getmtime(_SRC_INDEXER)):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                               "-o", tmp, _SRC, _SRC_INDEXER, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(L):
    vp, i32, f64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
    L.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
    L.orc_bf16_to_double.restype = f64
    L.orc_f16_to_double.argtypes = [ctypes.c_uint16]
    L.orc_f16_to_double.restype = f64
    L.orc_round_to_bf16.argtypes = [f64]
    L.orc_round_to_bf16.restype = f64
    L.orc_dequant_row.argtypes = [ctypes.POINTER(_QMat), i32, i32, i32, vp]
    L.orc_expert_ffn.argtypes = [i32, i32, i32, ctypes.POINTER(_Expert), vp, vp, vp]
    L.orc_route.argtypes = [ctypes.POINTER(_Desc), i32, vp, vp, vp, vp, vp, vp, vp, i32]
    L.orc_route.restype = i32
    L.orc_permute.argtypes = [i32, i32, i32, vp, vp, vp, vp, vp]
    L.orc_permute.restype = i32
    L.orc_moe_forward.argtypes = [ctypes.POINTER(_Desc), vp, vp, vp, ctypes.POINTER(_Expert),
                                  ctypes.POINTER(_Expert), vp, i32, vp, vp, i32]
    L.orc_moe_forward.restype = i32
    L.orc_rmsnorm_bf16.argtypes = [i32, vp, f64, vp]
    if hasattr(L, "orc_mx8_block"):
        L.orc_mx8_block.argtypes = [i32, vp, f64, vp, vp]
        L.orc_mx8_block.restype = i32
        L.orc_expert_ffn_idot.argtypes = [i32, i32, i32, ctypes.POINTER(_Expert), vp, f64, vp, vp, vp]
        L.orc_idot_hidden.argtypes = [i32, i32, i32, ctypes.POINTER(_Expert), vp, f64, vp, vp, vp, vp]
        L.orc_moe_forward_idot.argtypes = [ctypes.POINTER(_Desc), vp, vp, vp, ctypes.POINTER(_Expert),
                                           ctypes.POINTER(_Expert), vp, i32, f64, vp, vp, i32]
        L.orc_moe_forward_idot.restype = i32
    if hasattr(L, "orc_indexer_scores"):
        L.orc_indexer_scores.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, i32]
        L.orc_indexer_scores.restype = i32
        L.orc_indexer_topk.argtypes = [i32, i32, i32, vp, vp, vp]
        L.orc_indexer_topk.restype = i32
    return L


def load(path: str):
    """Load an oracle build from `path` (the tests use this for deliberately broken copies)."""
    return _bind(ctypes.CDLL(path))


def compile_source(src_text: str, out_path: str) -> str:
    """Compile oracle C source text with the oracle's own flags (tests: planted-mistake copies)."""
    c_path = out_path + ".c"
    with open(c_path, "w") as f:
        f.write(src_text)
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                           "-o", out_path, c_path, "-lm"])
    return out_path


def source() -> str:
    with open(_SRC) as f:
        return f.read()


def lib(L=None):
    global _lib
    if L is not None:
        return L
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _p(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "arrays passed to the oracle must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _qmat(m, e: int) -> _QMat:
    return _QMat(m.q[e].ctypes.data, m.s[e].ctypes.data, m.z[e].ctypes.data)


def _experts(bank):
    arr = (_Expert * bank.E)()
    for e in range(bank.E):
        arr[e] = _Expert(_qmat(bank.gate, e), _qmat(bank.up, e), _qmat(bank.down, e))
    return arr


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


class Oracle:
    """The oracle bound to one layer's weights."""

    def __init__(self, layer, L=None):
        self.L = lib(L)
        self.layer = layer
        self.d, self.F, self.E, self.k = layer.d, layer.F, layer.E, layer.k
        shared = getattr(layer, "shared", None)
        self.desc = _Desc(layer.d, layer.F, layer.E, layer.k, float(layer.rho), layer.qtype, X_BF16,
                          1 if shared is not None else 0, shared.F if shared is not None else 0,
                          shared.qtype if shared is not None else layer.qtype)
        self._experts = _experts(layer.experts)
        self._shared = _experts(shared) if shared is not None else None
        self.router_w = np.ascontiguousarray(layer.router_w, np.float32)
        self.bias = np.ascontiguousarray(layer.bias, np.float32)

    def _desc_for(self, x: np.ndarray) -> _Desc:
        d = _Desc.from_buffer_copy(self.desc)
        d.xtype = X_BF16 if x.dtype == np.uint16 else X_F32
        if x.dtype not in (np.uint16, np.float32):
            raise TypeError("x must be bf16 bits (uint16) or float32")
        return d

    def route(self, x: np.ndarray, nthreads: int | None = None):
        """Returns (topk_idx int32 [T,k] ascending ids, topk_w f64 [T,k], gap f64 [T], s f64 [T,E])."""
        x = np.ascontiguousarray(x)
        T = x.shape[0]
        idx = np.zeros((T, self.k), np.int32)
        w = np.zeros((T, self.k), np.float64)
        gap = np.zeros(T, np.float64)
        s = np.zeros((T, self.E), np.float64)
        rc = self.L.orc_route(ctypes.byref(self._desc_for(x)), T, _p(x), _p(self.router_w), _p(self.bias), _p(idx),
                             _p(w), _p(gap), _p(s), nthreads or default_threads())
        if rc != 0:
            raise RuntimeError("orc_route failed")
        return idx, w, gap, s

    def forward(self, x: np.ndarray, tokens=None, sel_override: np.ndarray | None = None,
                nthreads: int | None = None) -> np.ndarray:
        """Layer output (float64) for `tokens` (default: all rows of x)."""
        x = np.ascontiguousarray(x)
        T = x.shape[0]
        tokens = np.arange(T, dtype=np.int32) if tokens is None else np.ascontiguousarray(tokens, np.int32)
        out = np.zeros((len(tokens), self.d), np.float64)
        ov = None
        if sel_override is not None:
            ov = np.ascontiguousarray(sel_override, np.int32)
            assert ov.shape == (len(tokens), self.k)
        rc = self.L.orc_moe_forward(ctypes.byref(self._desc_for(x)), _p(x), _p(self.router_w), _p(self.bias),
                                   self._experts, self._shared, _p(tokens), len(tokens), _p(ov), _p(out),
                                   nthreads or default_threads())
        if rc != 0:
            raise RuntimeError("orc_moe_forward failed")
        return out


    def forward_idot(self, x: np.ndarray, tau: float, tokens=None, nthreads: int | None = None):
        """The layer with integer-dot (IDOT) expert inputs: x and h in blocks of 32 int8 values sharing a
        power-of-two scale.  Returns (out f64 [n, d], bound f64 [n, d]): bound is the allowance of each output
        for h values within tau code steps of a rounding boundary (near ties, see orc_mx8_block)."""
        x = np.ascontiguousarray(x)
        T = x.shape[0]
        tokens = np.arange(T, dtype=np.int32) if tokens is None else np.ascontiguousarray(tokens, np.int32)
        out = np.zeros((len(tokens), self.d), np.float64)
        bound = np.zeros((len(tokens), self.d), np.float64)
        rc = self.L.orc_moe_forward_idot(ctypes.byref(self._desc_for(x)), _p(x), _p(self.router_w), _p(self.bias),
                                        self._experts, self._shared, _p(tokens), len(tokens), float(tau), _p(out),
                                        _p(bound), nthreads or default_threads())
        if rc != 0:
            raise RuntimeError("orc_moe_forward_idot failed")
        return out, bound


def mx8_block(v: np.ndarray, tau: float = 0.0, L=None):
    """One block of IDOT activations: (vq = q * 2^(e-6) f64 [n], amb f64 [n], e)."""
    v = np.ascontiguousarray(v, np.float64)
    vq = np.zeros_like(v)
    amb = np.zeros_like(v)
    e = lib(L).orc_mx8_block(len(v), _p(v), float(tau), _p(vq), _p(amb))
    return vq, amb, e


def expert_ffn_idot(bank, e: int, xt: np.ndarray, tau: float = 0.0, L=None):
    """One token through expert e of `bank` with IDOT inputs: (y f64 [d], ybound f64 [d])."""
    xt = np.ascontiguousarray(xt, np.float64)
    d, F = xt.shape[0], bank.F
    y = np.zeros(d, np.float64)
    yb = np.zeros(d, np.float64)
    mx = max(d, F)
    scratch = np.zeros(2 * mx + 3 * F, np.float64)
    ex = _Expert(_qmat(bank.gate, e), _qmat(bank.up, e), _qmat(bank.down, e))
    lib(L).orc_expert_ffn_idot(bank.qtype, d, F, ctypes.byref(ex), _p(xt), float(tau), _p(y), _p(yb), _p(scratch))
    return y, yb


def idot_hidden(bank, e: int, xt: np.ndarray, tau: float = 0.0, L=None):
    """The down projection's input of one token in expert e with IDOT inputs: (h f64 [F], hq f64 [F] (the
    values q * 2^(e-6)), amb f64 [F] (near-tie bounds))."""
    xt = np.ascontiguousarray(xt, np.float64)
    d, F = xt.shape[0], bank.F
    h, hq, amb = (np.zeros(F, np.float64) for _ in range(3))
    scratch = np.zeros(2 * max(d, F), np.float64)
    ex = _Expert(_qmat(bank.gate, e), _qmat(bank.up, e), _qmat(bank.down, e))
    lib(L).orc_idot_hidden(bank.qtype, d, F, ctypes.byref(ex), _p(xt), float(tau), _p(h), _p(hq), _p(amb),
                           _p(scratch))
    return h, hq, amb


def permute(topk_idx: np.ndarray, E: int, L=None):
    """Batch-union grouping: (offsets [E+1], pair_token [P], pair_slot [P], pair_of [T,k])."""
    topk_idx = np.ascontiguousarray(topk_idx, np.int32)
    T, k = topk_idx.shape
    offsets = np.zeros(E + 1, np.int32)
    pt = np.zeros(T * k, np.int32)
    ps = np.zeros(T * k, np.int32)
    po = np.zeros((T, k), np.int32)
    if lib(L).orc_permute(T, k, E, _p(topk_idx), _p(offsets), _p(pt), _p(ps), _p(po)) != 0:
        raise ValueError("expert id out of range")
    return offsets, pt, ps, po


def dequant_row(m, qtype: int, n: int, e: int | None = None, L=None) -> np.ndarray:
    """Row n of a packed matrix (leading expert index e if the bank is stacked) as float64."""
    q = _QMat(m.q[e].ctypes.data, m.s[e].ctypes.data, m.z[e].ctypes.data) if e is not None else \
        _QMat(m.q.ctypes.data, m.s.ctypes.data, m.z.ctypes.data)
    out = np.zeros(m.K, np.float64)
    lib(L).orc_dequant_row(ctypes.byref(q), qtype, m.K, n, _p(out))
    return out


def expert_ffn(bank, e: int, xt: np.ndarray, L=None) -> np.ndarray:
    """One token (float64 [d]) through expert e of a bank."""
    xt = np.ascontiguousarray(xt, np.float64)
    ex = _Expert(_qmat(bank.gate, e), _qmat(bank.up, e), _qmat(bank.down, e))
    y = np.zeros(bank.d, np.float64)
    scratch = np.zeros(max(bank.d, bank.F) + bank.F, np.float64)
    lib(L).orc_expert_ffn(bank.qtype, bank.d, bank.F, ctypes.byref(ex), _p(xt), _p(y), _p(scratch))
    return y


def f16_to_double(bits: int, L=None) -> float:
    return lib(L).orc_f16_to_double(bits)


def bf16_to_double(bits: int, L=None) -> float:
    return lib(L).orc_bf16_to_double(bits)


def round_to_bf16(v: float, L=None) -> float:
    return lib(L).orc_round_to_bf16(v)


def rmsnorm_bf16(h: np.ndarray, eps: float, L=None) -> np.ndarray:
    """Rows of h (float64 [T,d]) normalised and rounded to bf16 (float64 result)."""
    h = np.ascontiguousarray(h, np.float64)
    out = np.zeros_like(h)
    for t in range(h.shape[0]):
        lib(L).orc_rmsnorm_bf16(h.shape[1], _p(h[t]), eps, _p(out[t]))
    return out


def bf16_bits_of(v: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of values that are exactly representable in bf16."""
    f = np.ascontiguousarray(v, np.float64).astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def stacked_forward(layers, x: np.ndarray, eps: float, tokens=None, nthreads: int | None = None,
                    return_layer_inputs: bool = False, L=None):
    """Stacked layers: h0 = x; for each layer: n = bf16(RMSNorm(h)); h += MoE(n).  Rows `tokens` only."""
    x = np.ascontiguousarray(x)
    T = x.shape[0]
    tokens = np.arange(T, dtype=np.int32) if tokens is None else np.asarray(tokens, np.int32)
    if x.dtype == np.uint16:
        h = (x[tokens].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    else:
        h = x[tokens].astype(np.float64)
    inputs = []
    for layer in layers:
        n = rmsnorm_bf16(h, eps, L=L)
        nb = bf16_bits_of(n)
        inputs.append(nb)
        h = h + Oracle(layer, L=L).forward(nb, nthreads=nthreads)
    return (h, inputs) if return_layer_inputs else h


# --------------------------------------------------------------------------- sparse-attention key selection

def indexer_scores(q: np.ndarray, w: np.ndarray, keys: np.ndarray, pos0: int, nthreads: int | None = None,
                   L=None) -> np.ndarray:
    """I[t][s] = sum_j w[t][j] * relu(q[t][j] . k[s]) (float64 [T, L]); -inf where s > pos0 + t.
    q: bf16 bits [T, H, d]; w: float32 [T, H]; keys: bf16 bits [L, d]."""
    q = np.ascontiguousarray(q, np.uint16)
    w = np.ascontiguousarray(w, np.float32)
    keys = np.ascontiguousarray(keys, np.uint16)
    T, H, d = q.shape
    Lk = keys.shape[0]
    assert keys.shape[1] == d and w.shape == (T, H)
    out = np.zeros((T, Lk), np.float64)
    if lib(L).orc_indexer_scores(T, Lk, H, d, pos0, _p(q), _p(w), _p(keys), _p(out), nthreads or default_threads()):
        raise ValueError("orc_indexer_scores: bad sizes")
    return out


def indexer_topk(scores: np.ndarray, topk: int, L=None):
    """(selected keys int32 [T, topk] ascending, -1 padded; gap float64 [T] between the topk-th and the
    (topk+1)-th largest visible score) of float64 scores [T, L]."""
    scores = np.ascontiguousarray(scores, np.float64)
    T, Lk = scores.shape
    idx = np.zeros((T, topk), np.int32)
    gap = np.zeros(T, np.float64)
    if lib(L).orc_indexer_topk(T, Lk, topk, _p(scores), _p(idx), _p(gap)):
        raise ValueError("orc_indexer_topk failed")
    return idx, gap
