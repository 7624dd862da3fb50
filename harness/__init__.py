"""Seeded synthetic inputs for the quantized sparse MoE layer.

Test and benchmark infrastructure.  Both the fp64 oracle and the CUDA path
consume the byte arrays produced here; this module holds none of the layer's
forward arithmetic (see gen.c for the generator and quantiser definitions).

Workloads follow the shapes of the GLM-5.2-class model on the Colibri pages
(256 routed experts, 8 active per token, int4 weights; "GLM-5.2 in 25GB RAM"
page, sections 2 and 3.1) plus a tiny layer used for exhaustive checks.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libcoli_gen.so")
_lock = threading.Lock()
_lib = None

Q_INT4_G128 = 0
Q_INT8_PC = 1
X_BF16 = 0
X_F32 = 1

# stream tags
_TAG_X, _TAG_ROUTER, _TAG_BIAS, _TAG_GATE, _TAG_UP, _TAG_DOWN, _TAG_PERM = 1, 2, 3, 4, 5, 6, 7
_TAG_IDX_Q, _TAG_IDX_W, _TAG_IDX_K = 8, 9, 10
SHARED_ID = 1 << 20  # expert index used for the shared expert's streams


def build(force: bool = False) -> str:
    """Compile gen.c into a shared library (gcc, OpenMP, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O3", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                               "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            u64, i64, i32, f32, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_void_p
            L.gen_stream_key.argtypes = [u64, u64, u64, u64]
            L.gen_stream_key.restype = u64
            L.gen_normal_f32.argtypes = [u64, i64, f32, f32, vp]
            L.gen_uniform_f32.argtypes = [u64, i64, f32, f32, vp]
            L.gen_permutation.argtypes = [u64, i32, vp]
            L.gen_f32_to_bf16.argtypes = [vp, i64, vp]
            L.gen_f32_to_f16.argtypes = [vp, i64, vp]
            L.gen_quant_int4.argtypes = [vp, i32, i32, vp, vp, vp]
            L.gen_quant_int8.argtypes = [vp, i32, i32, vp, vp, vp]
            L.gen_quant_matrix.argtypes = [u64, i32, i32, i32, f32, vp, vp, vp]
            L.gen_quant_matrix.restype = i32
            _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


def key(seed: int, tag: int, a: int = 0, b: int = 0) -> int:
    return int(lib().gen_stream_key(seed & (2**64 - 1), tag, a, b))


def normal(k: int, n: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    out = np.empty(n, np.float32)
    lib().gen_normal_f32(k, n, mean, std, _p(out))
    return out


def uniform(k: int, n: int, lo: float, hi: float) -> np.ndarray:
    out = np.empty(n, np.float32)
    lib().gen_uniform_f32(k, n, lo, hi, _p(out))
    return out


def permutation(k: int, n: int) -> np.ndarray:
    out = np.empty(n, np.int32)
    lib().gen_permutation(k, n, _p(out))
    return out


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, np.float32)
    out = np.empty(a.shape, np.uint16)
    lib().gen_f32_to_bf16(_p(a), a.size, _p(out))
    return out


def to_f16_bits(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, np.float32)
    out = np.empty(a.shape, np.uint16)
    lib().gen_f32_to_f16(_p(a), a.size, _p(out))
    return out


# --------------------------------------------------------------------------- packed weights

def groups(K: int) -> int:
    return K // 128


def zp_bytes(K: int) -> int:
    return (K // 128 + 1) // 2


@dataclasses.dataclass
class QMat:
    """One quantised matrix W[N][K] in the library's packed layout."""
    qtype: int
    N: int
    K: int
    q: np.ndarray      # int4: uint8 [N, K/2]; int8: uint8 [N, K]
    s: np.ndarray      # int4: uint16 fp16 bits [N, K/128]; int8: float32 [N]
    z: np.ndarray      # int4: uint8 [N, ceil(K/256)]; int8: uint8 [N]

    @property
    def nbytes(self) -> int:
        return self.q.nbytes + self.s.nbytes + self.z.nbytes


def empty_qmat(qtype: int, N: int, K: int, lead=()) -> QMat:
    lead = tuple(lead)
    if qtype == Q_INT4_G128:
        return QMat(qtype, N, K, np.zeros(lead + (N, K // 2), np.uint8), np.zeros(lead + (N, groups(K)), np.uint16),
                    np.zeros(lead + (N, zp_bytes(K)), np.uint8))
    return QMat(qtype, N, K, np.zeros(lead + (N, K), np.uint8), np.zeros(lead + (N,), np.float32),
                np.zeros(lead + (N,), np.uint8))


def quantize(w: np.ndarray, qtype: int) -> QMat:
    """Quantise a dense float matrix with the min-max asymmetric quantiser of gen.c."""
    w = np.ascontiguousarray(w, np.float32)
    N, K = w.shape
    m = empty_qmat(qtype, N, K)
    if qtype == Q_INT4_G128:
        assert K % 128 == 0
        lib().gen_quant_int4(_p(w), N, K, _p(m.q), _p(m.s), _p(m.z))
    else:
        lib().gen_quant_int8(_p(w), N, K, _p(m.q), _p(m.s), _p(m.z))
    return m


def gen_qmat_into(k: int, qtype: int, N: int, K: int, std: float, q: np.ndarray, s: np.ndarray, z: np.ndarray):
    rc = lib().gen_quant_matrix(k, qtype, N, K, std, _p(q), _p(s), _p(z))
    if rc != 0:
        raise ValueError("gen_quant_matrix: unsupported K")


@dataclasses.dataclass
class ExpertBank:
    """E experts of one layer, each matrix stacked along a leading expert axis."""
    qtype: int
    E: int
    d: int
    F: int
    gate: QMat   # arrays [E, F, ...]
    up: QMat     # arrays [E, F, ...]
    down: QMat   # arrays [E, d, ...]

    def expert(self, e: int):
        def sl(m: QMat):
            return QMat(m.qtype, m.N, m.K, m.q[e], m.s[e], m.z[e])
        return sl(self.gate), sl(self.up), sl(self.down)

    @property
    def bytes_per_expert(self) -> int:
        return (self.gate.nbytes + self.up.nbytes + self.down.nbytes) // self.E


def gen_experts(seed: int, layer: int, qtype: int, E: int, d: int, F: int, first_id: int = 0) -> ExpertBank:
    """Expert weights W ~ N(0, 1/K) per matrix (K = fan-in), quantised; expert e uses stream id first_id+e."""
    gate, up, down = empty_qmat(qtype, F, d, (E,)), empty_qmat(qtype, F, d, (E,)), empty_qmat(qtype, d, F, (E,))
    for e in range(E):
        eid = first_id + e
        gen_qmat_into(key(seed, _TAG_GATE, layer, eid), qtype, F, d, d ** -0.5, gate.q[e], gate.s[e], gate.z[e])
        gen_qmat_into(key(seed, _TAG_UP, layer, eid), qtype, F, d, d ** -0.5, up.q[e], up.s[e], up.z[e])
        gen_qmat_into(key(seed, _TAG_DOWN, layer, eid), qtype, d, F, F ** -0.5, down.q[e], down.s[e], down.z[e])
    return ExpertBank(qtype, E, d, F, gate, up, down)


@dataclasses.dataclass
class Layer:
    d: int
    F: int
    E: int
    k: int
    rho: float
    qtype: int
    router_w: np.ndarray        # float32 [E, d]
    bias: np.ndarray            # float32 [E]
    experts: ExpertBank
    shared: ExpertBank | None   # E == 1 bank, or None
    F_shared: int = 0

    @property
    def has_shared(self) -> bool:
        return self.shared is not None


def gen_bias(seed: int, layer: int, kind: str, E: int) -> np.ndarray:
    """Router bias recipes: zero, uniform(a), normal(std), zipf(alpha, s), spike(e, value)."""
    name, *args = kind.split(":")
    k = key(seed, _TAG_BIAS, layer)
    if name == "zero":
        return np.zeros(E, np.float32)
    if name == "uniform":
        a = float(args[0])
        return uniform(k, E, -a, a)
    if name == "normal":          # N(0, std^2): the argument is the standard deviation
        return normal(k, E, 0.0, float(args[0]))
    if name == "zipf":            # b_e = -alpha * s * ln(rank_e), rank a seeded permutation of 1..E
        alpha, s = float(args[0]), float(args[1])
        rank = permutation(key(seed, _TAG_PERM, layer), E).astype(np.float64) + 1.0
        return (-alpha * s * np.log(rank)).astype(np.float32)
    if name == "spike":           # expert e gets +value, all others 0
        b = np.zeros(E, np.float32)
        b[int(args[0])] = float(args[1])
        return b
    raise ValueError(kind)


def gen_layer(seed: int, layer: int, *, d: int, F: int, E: int, k: int, rho: float, qtype: int,
              bias: str = "zero", F_shared: int = 0, qtype_shared: int | None = None) -> Layer:
    router_w = normal(key(seed, _TAG_ROUTER, layer), E * d, 0.0, d ** -0.5).reshape(E, d)
    b = gen_bias(seed, layer, bias, E)
    experts = gen_experts(seed, layer, qtype, E, d, F)
    shared = None
    if F_shared:
        shared = gen_experts(seed, layer, qtype if qtype_shared is None else qtype_shared, 1, d, F_shared,
                             first_id=SHARED_ID)
    return Layer(d, F, E, k, rho, qtype, router_w, b, experts, shared, F_shared)


def gen_x(seed: int, stream: int, T: int, d: int, xtype: int) -> np.ndarray:
    """Activations x[T][d] ~ N(0,1): bf16 bit patterns (uint16) or float32."""
    x = normal(key(seed, _TAG_X, stream), T * d).reshape(T, d)
    return to_bf16_bits(x) if xtype == X_BF16 else x


# --------------------------------------------------------------------------- the five workloads

@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    T: tuple
    d: int
    F: int
    E: int
    k: int
    rho: float
    qtypes: tuple          # one per layer
    xtype: int
    bias: str
    F_shared: int = 0
    rmsnorm_eps: float = 0.0  # > 0: stacked layers with residual + RMSNorm

    @property
    def n_layers(self) -> int:
        return len(self.qtypes)

    def layer(self, l: int) -> Layer:
        return gen_layer(self.seed, l, d=self.d, F=self.F, E=self.E, k=self.k, rho=self.rho, qtype=self.qtypes[l],
                         bias=self.bias, F_shared=self.F_shared)

    def x(self, T: int, stream: int = 0) -> np.ndarray:
        return gen_x(self.seed, stream, T, self.d, self.xtype)


WORKLOADS = {
    "tiny": Workload("tiny", 0, (16,), 256, 128, 8, 2, 1.0, (Q_INT8_PC,), X_F32, "uniform:0.1"),
    "decode": Workload("decode", 1, (1, 4), 7168, 2048, 256, 8, 2.5, (Q_INT4_G128,), X_BF16, "zero"),
    "mtp_verify": Workload("mtp_verify", 2, (3,), 7168, 2048, 256, 8, 2.5, (Q_INT4_G128,), X_BF16, "normal:0.5",
                           F_shared=2048),
    "prefill": Workload("prefill", 3, (2048,), 7168, 2048, 256, 8, 2.5, (Q_INT4_G128,), X_BF16, "zipf:0.05:1.1",
                        F_shared=2048),
    "stacked": Workload("stacked", 4, (256,), 7168, 2048, 256, 8, 2.5,
                        (Q_INT4_G128, Q_INT8_PC) * 3, X_BF16, "zero", rmsnorm_eps=1e-6),
}


# --------------------------------------------------------------------------- sparse-attention key selection

@dataclasses.dataclass(frozen=True)
class IndexerWorkload:
    """Inputs of the key-selection step of sparse attention: T query tokens at the end of a context of L
    cached keys; H indexer heads of dimension d; the topk highest-scoring causal keys are kept
    ("25GB RAM runs 744B GLM-5.2" page, section 3.3: top-2048 causal keys per layer).  The shapes H = 64,
    d = 128 follow the DeepSeek-V3.2 indexer that the page cites; q and k are bf16 N(0, 1), the per-head
    weights w fp32 N(0, 1/H)."""
    name: str
    seed: int
    T: tuple
    L: int
    H: int
    d: int
    topk: int

    def q(self, T: int, stream: int = 0) -> np.ndarray:
        return to_bf16_bits(normal(key(self.seed, _TAG_IDX_Q, stream), T * self.H * self.d).reshape(T, self.H, self.d))

    def w(self, T: int, stream: int = 0) -> np.ndarray:
        return normal(key(self.seed, _TAG_IDX_W, stream), T * self.H, 0.0, self.H ** -0.5).reshape(T, self.H)

    def keys(self, L: int | None = None, stream: int = 0) -> np.ndarray:
        L = self.L if L is None else L
        return to_bf16_bits(normal(key(self.seed, _TAG_IDX_K, stream), L * self.d).reshape(L, self.d))


INDEXER = IndexerWorkload("indexer", 5, (1, 4), 65536, 64, 128, 2048)
