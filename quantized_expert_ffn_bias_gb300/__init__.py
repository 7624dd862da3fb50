"""Python binding of the quantized sparse MoE layer library (libcolibri_moe.so).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Functions keep the C names (``colibri_moe_*``); the ``Plan`` class
wraps a plan handle.  Pointers are plain integers or objects with a
``data_ptr()`` method (for example torch tensors); streams are integers
(``torch.cuda.Stream.cuda_stream``) or objects with a ``cuda_stream`` attribute.

There is no CPU fallback: if the library has not been built, loading fails.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

COLI_OK, COLI_EINVAL, COLI_EALIGN, COLI_EUNSUPPORTED, COLI_EWORKSPACE, COLI_ECUDA, COLI_EDEVICE, COLI_ESTATE = range(8)
COLI_Q_INT4_G128, COLI_Q_INT8_PC = 0, 1
COLI_X_BF16, COLI_X_F32 = 0, 1
COLI_DEV_BAD_EXPERT_ID, COLI_DEV_WAIT_TIMEOUT = 1, 2
COLI_INJECT_WITHHOLD_STAGE, COLI_INJECT_BAD_EXPERT_ID = 1, 2

# the in-tree build, the only library this binding loads
LIB_PATH = _build.LIB
_lock = threading.Lock()
_lib = None


class ColiError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"colibri_moe error {status}: {msg}")
        self.status = status


class coli_qmat(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("zp", ctypes.c_void_p)]


class coli_expert(ctypes.Structure):
    _fields_ = [("gate", coli_qmat), ("up", coli_qmat), ("down", coli_qmat)]


class coli_moe_desc(ctypes.Structure):
    _fields_ = [("T_max", ctypes.c_int), ("d", ctypes.c_int), ("d_ff", ctypes.c_int), ("E", ctypes.c_int),
                ("k", ctypes.c_int), ("routed_scale", ctypes.c_float), ("qtype", ctypes.c_int),
                ("xtype", ctypes.c_int), ("has_shared", ctypes.c_int), ("shared_d_ff", ctypes.c_int)]


class coli_kernel_time(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("total_ms", ctypes.c_double), ("launches", ctypes.c_int)]


def build(force: bool = False) -> str:
    """Compile the CUDA library for sm_103a (in-tree)."""
    return _build.build(force=force)


def lib():
    """Load libcolibri_moe.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"CUDA library not built ({LIB_PATH}); run quantized_expert_ffn_bias_gb300.build()")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            st = ctypes.c_int
            L.colibri_moe_plan.argtypes = [ctypes.POINTER(coli_moe_desc), ctypes.POINTER(vp), ctypes.POINTER(sz)]
            L.colibri_moe_plan.restype = st
            L.colibri_moe_bind_experts.argtypes = [vp, ctypes.POINTER(coli_expert), ctypes.POINTER(coli_expert)]
            L.colibri_moe_bind_experts.restype = st
            L.colibri_moe_forward.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp, sz, vp]
            L.colibri_moe_forward.restype = st
            L.colibri_moe_forward_noalloc.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp]
            L.colibri_moe_forward_noalloc.restype = st
            L.colibri_moe_rmsnorm_bf16.argtypes = [vp, i32, i32, ctypes.c_float, vp, vp]
            L.colibri_moe_rmsnorm_bf16.restype = st
            L.colibri_moe_debug_routing.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, vp, vp]
            L.colibri_moe_debug_routing.restype = st
            L.colibri_moe_check_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int32), vp]
            L.colibri_moe_check_status.restype = st
            L.colibri_moe_profile_begin.argtypes = [vp, i32]
            L.colibri_moe_profile_begin.restype = st
            L.colibri_moe_profile_end.argtypes = [vp, ctypes.POINTER(coli_kernel_time), i32, ctypes.POINTER(i32)]
            L.colibri_moe_profile_end.restype = st
            L.colibri_moe_debug_inject.argtypes = [vp, i32, ctypes.c_double]
            L.colibri_moe_debug_inject.restype = st
            L.colibri_moe_set_idot.argtypes = [vp, i32]
            L.colibri_moe_debug_hidden.argtypes = [vp, vp, i32, vp, vp]
            L.colibri_moe_debug_hidden.restype = st
            L.colibri_moe_set_idot.restype = st
            L.colibri_indexer_workspace_size.argtypes = [i32, i32, ctypes.POINTER(sz)]
            L.colibri_indexer_workspace_size.restype = st
            L.colibri_indexer_topk.argtypes = [i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, sz, vp]
            L.colibri_indexer_topk.restype = st
            L.colibri_indexer_scores.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, sz, vp]
            L.colibri_indexer_scores.restype = st
            L.colibri_indexer_select.argtypes = [i32, i32, i32, i32, vp, vp, sz, vp]
            L.colibri_indexer_select.restype = st
            L.colibri_indexer_check_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int32), vp]
            L.colibri_indexer_check_status.restype = st
            L.colibri_moe_cache_slot_bytes.argtypes = [vp, ctypes.POINTER(sz)]
            L.colibri_moe_cache_slot_bytes.restype = st
            L.colibri_moe_cache_create.argtypes = [vp, i32, ctypes.c_double, ctypes.POINTER(coli_expert),
                                                   ctypes.POINTER(coli_expert), vp, sz, ctypes.POINTER(vp)]
            L.colibri_moe_cache_create.restype = st
            L.colibri_moe_forward_cached.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, vp, sz, vp]
            L.colibri_moe_forward_cached.restype = st
            L.colibri_moe_cache_prefetch.argtypes = [vp, vp, i32, vp]
            L.colibri_moe_cache_prefetch.restype = st
            L.colibri_moe_cache_stats.argtypes = [vp, vp]
            L.colibri_moe_cache_stats.restype = st
            L.colibri_moe_cache_reset_stats.argtypes = [vp]
            L.colibri_moe_cache_reset_stats.restype = st
            L.colibri_moe_cache_resident.argtypes = [vp, vp]
            L.colibri_moe_cache_resident.restype = st
            L.colibri_moe_cache_destroy.argtypes = [vp]
            L.colibri_moe_cache_destroy.restype = None
            L.colibri_moe_cache_pilot.argtypes = [vp, vp, i32, vp, vp, vp, vp, ctypes.POINTER(i32), vp, sz, vp]
            L.colibri_moe_cache_pilot.restype = st
            L.colibri_moe_cache_simulate.argtypes = [i32, i32, ctypes.c_double, vp, vp, i32, vp, vp]
            L.colibri_moe_cache_simulate.restype = st
            L.colibri_moe_last_launch_count.argtypes = [vp]
            L.colibri_moe_last_launch_count.restype = i32
            L.colibri_moe_last_error.argtypes = []
            L.colibri_moe_last_error.restype = ctypes.c_char_p
            L.colibri_moe_destroy.argtypes = [vp]
            L.colibri_moe_destroy.restype = None
            _lib = L
    return _lib


def _ptr(v) -> int | None:
    if v is None:
        return None
    if isinstance(v, int):
        return v
    return int(v.data_ptr())


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def _check(rc: int):
    if rc != COLI_OK:
        raise ColiError(rc, lib().colibri_moe_last_error().decode(errors="replace"))


def colibri_moe_last_error() -> str:
    return lib().colibri_moe_last_error().decode(errors="replace")


def colibri_moe_rmsnorm_bf16(h, T: int, d: int, eps: float, out, stream=None):
    _check(lib().colibri_moe_rmsnorm_bf16(_ptr(h), T, d, eps, _ptr(out), _stream(stream)))


def colibri_indexer_workspace_size(T_max: int, L_max: int) -> int:
    n = ctypes.c_size_t()
    _check(lib().colibri_indexer_workspace_size(T_max, L_max, ctypes.byref(n)))
    return n.value


def colibri_indexer_topk(T: int, L: int, pos0: int, H: int, d: int, topk: int, q, w, keys, topk_idx, workspace,
                         workspace_bytes: int, stream=None):
    """Sparse-attention key selection (see the header): scores in the workspace, selection in topk_idx."""
    _check(lib().colibri_indexer_topk(T, L, pos0, H, d, topk, _ptr(q), _ptr(w), _ptr(keys), _ptr(topk_idx),
                                      _ptr(workspace), workspace_bytes, _stream(stream)))


def colibri_indexer_scores(T: int, L: int, pos0: int, H: int, d: int, q, w, keys, workspace, workspace_bytes: int,
                           stream=None):
    _check(lib().colibri_indexer_scores(T, L, pos0, H, d, _ptr(q), _ptr(w), _ptr(keys), _ptr(workspace),
                                        workspace_bytes, _stream(stream)))


def colibri_indexer_select(T: int, L: int, pos0: int, topk: int, topk_idx, workspace, workspace_bytes: int,
                           stream=None):
    _check(lib().colibri_indexer_select(T, L, pos0, topk, _ptr(topk_idx), _ptr(workspace), workspace_bytes,
                                        _stream(stream)))


def colibri_indexer_check_status(workspace, stream=None) -> int:
    v = ctypes.c_int32()
    rc = lib().colibri_indexer_check_status(_ptr(workspace), ctypes.byref(v), _stream(stream))
    if rc not in (COLI_OK, COLI_EDEVICE):
        _check(rc)
    return v.value


class coli_cache_stats(ctypes.Structure):
    _fields_ = [("forwards", ctypes.c_longlong), ("lookups", ctypes.c_longlong), ("hits", ctypes.c_longlong),
                ("misses", ctypes.c_longlong), ("evictions", ctypes.c_longlong), ("prefetched", ctypes.c_longlong),
                ("bytes_copied", ctypes.c_longlong), ("predicted", ctypes.c_longlong)]


def colibri_moe_cache_simulate(E: int, n_slots: int, weight: float, expert_sets) -> tuple[int, int]:
    """(hits, misses) of the expert cache's policy over a trace: expert_sets is a sequence of per-forward
    collections of distinct expert ids (host only, no GPU)."""
    sets = [list(map(int, s)) for s in expert_sets]
    flat = (ctypes.c_int32 * max(1, sum(len(s) for s in sets)))(*[e for s in sets for e in s])
    sizes = (ctypes.c_int32 * max(1, len(sets)))(*[len(s) for s in sets])
    h, m = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().colibri_moe_cache_simulate(E, n_slots, weight, flat, sizes, len(sets), ctypes.byref(h),
                                            ctypes.byref(m)))
    return h.value, m.value


class Cache:
    """An expert-slot cache of a plan (colibri_moe_cache_create): slots in caller device memory, every routed
    expert in host memory."""

    def __init__(self, plan, n_slots: int, weight: float, host_experts, slot_memory, slot_memory_bytes: int,
                 shared=None):
        arr = (coli_expert * len(host_experts))(*host_experts)
        sh = ctypes.byref(shared) if shared is not None else None
        h = ctypes.c_void_p()
        _check(lib().colibri_moe_cache_create(plan.handle, n_slots, weight, arr, sh, _ptr(slot_memory),
                                              slot_memory_bytes, ctypes.byref(h)))
        self.handle = h.value
        self.plan = plan

    def forward(self, T: int, x, router_w, bias, out, workspace, workspace_bytes: int | None = None, residual=None,
                stream=None):
        wb = self.plan.workspace_bytes if workspace_bytes is None else workspace_bytes
        _check(lib().colibri_moe_forward_cached(self.plan.handle, self.handle, T, _ptr(x), _ptr(router_w), _ptr(bias),
                                                _ptr(residual), _ptr(out), _ptr(workspace), wb, _stream(stream)))

    def prefetch(self, experts, stream=None):
        ids = (ctypes.c_int32 * max(1, len(experts)))(*[int(e) for e in experts])
        _check(lib().colibri_moe_cache_prefetch(self.handle, ids, len(experts), _stream(stream)))

    def pilot(self, T: int, x, router_w, bias, workspace, workspace_bytes: int | None = None, stream=None) -> list:
        """Predict this cache's layer's experts from x (the previous layer's state) and prefetch them
        (colibri_moe_cache_pilot); returns the predicted expert ids."""
        wb = self.plan.workspace_bytes if workspace_bytes is None else workspace_bytes
        E = self.plan.desc.E
        buf = (ctypes.c_int32 * E)()
        n = ctypes.c_int()
        _check(lib().colibri_moe_cache_pilot(self.plan.handle, self.handle, T, _ptr(x), _ptr(router_w), _ptr(bias),
                                             buf, ctypes.byref(n), _ptr(workspace), wb, _stream(stream)))
        return list(buf[:n.value])

    def stats(self) -> dict:
        s = coli_cache_stats()
        _check(lib().colibri_moe_cache_stats(self.handle, ctypes.byref(s)))
        return {f: getattr(s, f) for f, _ in coli_cache_stats._fields_}

    def reset_stats(self):
        _check(lib().colibri_moe_cache_reset_stats(self.handle))

    def resident(self, E: int):
        arr = (ctypes.c_int32 * E)()
        _check(lib().colibri_moe_cache_resident(self.handle, arr))
        return list(arr)

    def close(self):
        if self.handle:
            lib().colibri_moe_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def cache_slot_offsets(d: int, d_ff: int, qtype: int) -> list[int]:
    """Byte offsets of the nine packed arrays (gate q, scale, zp, up ..., down ...) inside one cache slot,
    each 256-byte aligned (the layout colibri_moe_cache_slot_bytes sizes); host memory in this layout
    moves in one copy per miss."""
    offs, o = [], 0
    for m in range(3):
        N, K = (d_ff, d) if m < 2 else (d, d_ff)
        if qtype == COLI_Q_INT4_G128:
            parts = (N * K // 2, N * (K // 128) * 2, N * ((K // 128 + 1) // 2))
        else:
            parts = (N * K, N * 4, N)
        for p in parts:
            offs.append(o)
            o = (o + p + 255) // 256 * 256
    return offs


def colibri_moe_cache_slot_bytes(plan) -> int:
    n = ctypes.c_size_t()
    _check(lib().colibri_moe_cache_slot_bytes(plan.handle, ctypes.byref(n)))
    return n.value


def qmat(q, scale, zp) -> coli_qmat:
    return coli_qmat(_ptr(q), _ptr(scale), _ptr(zp))


class Plan:
    """A validated layer plan (colibri_moe_plan) with its bound experts."""

    def __init__(self, *, T_max: int, d: int, d_ff: int, E: int, k: int, routed_scale: float, qtype: int,
                 xtype: int, has_shared: bool = False, shared_d_ff: int = 0):
        self.desc = coli_moe_desc(T_max, d, d_ff, E, k, routed_scale, qtype, xtype, 1 if has_shared else 0,
                                  shared_d_ff)
        h = ctypes.c_void_p()
        nbytes = ctypes.c_size_t()
        _check(lib().colibri_moe_plan(ctypes.byref(self.desc), ctypes.byref(h), ctypes.byref(nbytes)))
        self.handle = h.value
        self.workspace_bytes = nbytes.value

    def colibri_moe_bind_experts(self, experts, shared=None):
        """experts: sequence of E coli_expert (device pointers); shared: coli_expert or None."""
        arr = (coli_expert * len(experts))(*experts)
        sh = ctypes.byref(shared) if shared is not None else None
        _check(lib().colibri_moe_bind_experts(self.handle, arr, sh))

    bind_experts = colibri_moe_bind_experts

    def colibri_moe_forward(self, T: int, x, router_w, bias, out, workspace, workspace_bytes: int | None = None,
                            residual=None, stream=None):
        wb = self.workspace_bytes if workspace_bytes is None else workspace_bytes
        _check(lib().colibri_moe_forward(self.handle, T, _ptr(x), _ptr(router_w), _ptr(bias), _ptr(residual),
                                         _ptr(out), _ptr(workspace), wb, _stream(stream)))

    forward = colibri_moe_forward

    def colibri_moe_forward_noalloc(self, T: int, x, router_w, bias, out, residual=None, stream=None):
        """Forward with the library's static scratch instead of a caller workspace (see the header)."""
        _check(lib().colibri_moe_forward_noalloc(self.handle, T, _ptr(x), _ptr(router_w), _ptr(bias),
                                                 _ptr(residual), _ptr(out), _stream(stream)))

    forward_noalloc = colibri_moe_forward_noalloc

    def colibri_moe_debug_routing(self, workspace, T: int, topk_idx=None, topk_w=None, near_tie=None,
                                  expert_offsets=None, pair_token=None, pair_slot=None, stream=None):
        _check(lib().colibri_moe_debug_routing(self.handle, _ptr(workspace), T, _ptr(topk_idx), _ptr(topk_w),
                                               _ptr(near_tie), _ptr(expert_offsets), _ptr(pair_token),
                                               _ptr(pair_slot), _stream(stream)))

    debug_routing = colibri_moe_debug_routing

    def colibri_moe_check_status(self, workspace, stream=None) -> int:
        v = ctypes.c_int32()
        rc = lib().colibri_moe_check_status(self.handle, _ptr(workspace), ctypes.byref(v), _stream(stream))
        if rc not in (COLI_OK, COLI_EDEVICE):
            _check(rc)
        return v.value

    check_status = colibri_moe_check_status

    def colibri_moe_profile_begin(self, max_calls: int):
        _check(lib().colibri_moe_profile_begin(self.handle, max_calls))

    profile_begin = colibri_moe_profile_begin

    def colibri_moe_profile_end(self):
        """Returns {kernel name: (total ms, launches)}."""
        buf = (coli_kernel_time * 32)()
        n = ctypes.c_int()
        _check(lib().colibri_moe_profile_end(self.handle, buf, 32, ctypes.byref(n)))
        return {buf[i].name.decode(): (buf[i].total_ms, buf[i].launches) for i in range(min(n.value, 32))}

    profile_end = colibri_moe_profile_end

    def colibri_moe_debug_inject(self, flags: int, wait_limit_ms: float = 0.0):
        """Failure-path testing: COLI_INJECT_* bits for the next forward calls (0 = off)."""
        _check(lib().colibri_moe_debug_inject(self.handle, flags, wait_limit_ms))

    debug_inject = colibri_moe_debug_inject

    def colibri_moe_set_idot(self, enable: bool):
        """Integer-dot expert inputs (int8 codes per block of 32 with a power-of-two scale) on or off."""
        _check(lib().colibri_moe_set_idot(self.handle, 1 if enable else 0))

    set_idot = colibri_moe_set_idot

    def colibri_moe_debug_hidden(self, workspace, T: int, h_out, stream=None):
        """The down projection's input of the last forward (device float [rows, Fmax], grouped row order)."""
        _check(lib().colibri_moe_debug_hidden(self.handle, _ptr(workspace), T, _ptr(h_out), _stream(stream)))

    debug_hidden = colibri_moe_debug_hidden

    def colibri_moe_last_launch_count(self) -> int:
        return lib().colibri_moe_last_launch_count(self.handle)

    last_launch_count = colibri_moe_last_launch_count

    def close(self):
        if self.handle:
            lib().colibri_moe_destroy(self.handle)
            self.handle = None

    colibri_moe_destroy = close

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
