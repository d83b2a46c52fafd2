"""Thin ctypes binding of librx (``include/rx.h``).

Argument marshalling only: every function here checks the tensors it is
given (device, dtype, contiguity), passes their data pointers and the current
CUDA stream to the library function of the same name, and turns a non-zero
status into ``RxError``.  No step of the path runs in Python, and there is no
fallback: if ``_build/librx.so`` is missing, importing this module raises.

Device tensors come from PyTorch (it owns device memory and streams); host
arrays are numpy.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import List, Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "librx.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"librx.so is not built ({LIB_PATH}); run __graft_entry__.build() or "
                      "python -m prefix_shared_kv_radixattention_gb300.build")
_lib = ctypes.CDLL(LIB_PATH)

RX_OK = 0
RX_ERR_INVALID = -1
RX_ERR_CAPACITY = -2
RX_ERR_NOMEM = -3
RX_ERR_NOT_ENOUGH = -4
RX_ERR_CUDA = -5
RX_ERR_UNSUPPORTED = -6
RX_SCHED_FCFS = 0
RX_SCHED_LPM = 1
RX_DEV_BAD_SLOT = 1
RX_DEV_BAD_LEN = 2
RX_DEV_TIMEOUT = 4
RX_DEV_FSM_DONE = 8
RX_DEV_BAD_STATE = 16
RX_PLAN_OPEN_END = -1


class RxError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


class KVPool(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("num_slots", ctypes.c_int64),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("num_layers", ctypes.c_int32), ("layer", ctypes.c_int32)]


class DecodePlan(ctypes.Structure):
    _fields_ = [("order", ctypes.c_void_p), ("nparts", ctypes.c_void_p), ("items", ctypes.c_void_p),
                ("n_items", ctypes.c_int32), ("max_parts", ctypes.c_int32), ("n_wide", ctypes.c_int32)]


class DecodePlanInfo(ctypes.Structure):
    _fields_ = [("n_items", ctypes.c_int32), ("max_parts", ctypes.c_int32),
                ("n_segments", ctypes.c_int32), ("kv_chunk", ctypes.c_int32),
                ("shared_tokens", ctypes.c_int64), ("tokens_read", ctypes.c_int64),
                ("buf_words", ctypes.c_int64), ("n_wide", ctypes.c_int32)]


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_PI64 = ctypes.POINTER(ctypes.c_int64)


def _sig(name, res, *args):
    f = getattr(_lib, name)
    f.restype = res
    f.argtypes = list(args)
    return f


_sig("rx_last_error", ctypes.c_char_p)
_sig("rx_version", ctypes.c_int)
_sig("rx_tree_create", ctypes.c_int, ctypes.POINTER(_P))
_sig("rx_tree_destroy", None, _P)
_sig("rx_match_prefix", ctypes.c_int, _P, _P, _I64, _P, _I64, _PI64)
_sig("rx_insert", ctypes.c_int, _P, _P, _P, _I64, _PI64)
_sig("rx_evict_lru", ctypes.c_int, _P, _I64, _P, _I64, _PI64)
_sig("rx_lock_prefix", ctypes.c_int, _P, _P, _I64, _I32, _PI64)
_sig("rx_tree_stats", ctypes.c_int, _P, _PI64, _PI64, _PI64)
_sig("rx_tree_dump", ctypes.c_int, _P, _P, _I64, _PI64)
_sig("rx_slot_alloc_create", ctypes.c_int, _P, _I64, _I64, ctypes.POINTER(_P))
_sig("rx_slot_alloc_destroy", None, _P)
_sig("rx_slot_alloc_take", ctypes.c_int, _P, _I64, _P)
_sig("rx_slot_alloc_give", ctypes.c_int, _P, _P, _I64)
_sig("rx_slot_alloc_free_count", _I64, _P)
_sig("rx_admit", ctypes.c_int, _P, _P, _P, _I64, _P, _PI64, _PI64)
_sig("rx_commit", ctypes.c_int, _P, _P, _P, _P, _I64, _I64)
_sig("rx_prefix_len", ctypes.c_int, _P, _P, _I64, _PI64)
_sig("rx_image_keys", ctypes.c_int, _P, _I64, _I64, _P)


class KVPoolFp8(ctypes.Structure):
    _fields_ = [("k", _P), ("v", _P), ("num_slots", ctypes.c_int64), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float),
                ("num_layers", ctypes.c_int32), ("layer", ctypes.c_int32)]


_sig("rx_kv_store_fp8", ctypes.c_int, ctypes.POINTER(KVPoolFp8), _P, _P, _P, _I64, _P, _P)
_sig("rx_attn_decode_fp8", ctypes.c_int, ctypes.POINTER(KVPoolFp8), _P, _P, _P, _I32, _P, _P, _P, _I64, _I32,
     _I32, _P, _P, ctypes.c_size_t, ctypes.c_float, _P, _P)
_sig("rx_attn_extend_fp8", ctypes.c_int, ctypes.POINTER(KVPoolFp8), _P, _P, _P, _I32, _P, _P, _P, _P, _P,
     _I64, _I32, _I32, _P, ctypes.c_size_t, ctypes.c_float, _P, _P)
_sig("rx_kv_store_rope_fp8", ctypes.c_int, ctypes.POINTER(KVPoolFp8), _P, _P, _P, _P, _I64, ctypes.c_double, _P, _P)


class FsmInfo(ctypes.Structure):
    _fields_ = [("n_edges", ctypes.c_int64), ("jump_tokens", ctypes.c_int64), ("n_singular", ctypes.c_int32),
                ("n_looped", ctypes.c_int32), ("longest_jump", ctypes.c_int32)]


class FsmStruct(ctypes.Structure):
    _fields_ = [("row_ptr", _P), ("tok", _P), ("nxt", _P), ("mask", _P), ("rank", _P), ("jump_len", _P),
                ("jump_off", _P), ("jump_end", _P), ("jump_tok", _P), ("n_states", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("max_jump", ctypes.c_int32)]


_sig("rx_fsm_compress", ctypes.c_int, _I32, _I32, _P, _P, _P, _I32, _P, _P, _P, _P, _P, _P, _I64,
     ctypes.POINTER(FsmInfo))
_sig("rx_fsm_step", ctypes.c_int, ctypes.POINTER(FsmStruct), _P, _I64, _I32, _P, _P, _P, _P, _P, _P)
_sig("rx_schedule", ctypes.c_int, _P, _P, _P, _I32, _I32, _P, _P)
_sig("rx_kv_store", ctypes.c_int, ctypes.POINTER(KVPool), _P, _P, _P, _I64, _P, _P)
_sig("rx_rope", ctypes.c_int, _P, _P, _I64, _I32, _I32, ctypes.c_double, _P)
_sig("rx_kv_store_rope", ctypes.c_int, ctypes.POINTER(KVPool), _P, _P, _P, _P, _I64, ctypes.c_double, _P, _P)
_sig("rx_attn_extend", ctypes.c_int, ctypes.POINTER(KVPool), _P, _P, _P, _I32, _P, _P, _P, _P, _P,
     _I64, _I32, _I32, _P, ctypes.c_size_t, ctypes.c_float, _P, _P)
_sig("rx_attn_extend_workspace", ctypes.c_size_t, _I64, _I32, _I32, _I32)
_sig("rx_decode_plan_build", ctypes.c_int, _P, _I64, _P, _P, _I32, _I32, _I32, _I32, _I32, _P, _I64,
     ctypes.POINTER(DecodePlanInfo))
_sig("rx_attn_decode_workspace", ctypes.c_size_t, _I32, _I32, _I32, _I32, _I32,
     ctypes.POINTER(DecodePlan))
_sig("rx_attn_decode", ctypes.c_int, ctypes.POINTER(KVPool), _P, _P, _P, _I32, _P, _P, _P, _I64, _I32,
     _I32, ctypes.POINTER(DecodePlan), _P, ctypes.c_size_t, ctypes.c_float, _P, _P)
_sig("rx_attn_decode_static", ctypes.c_int, ctypes.POINTER(KVPool), _P, _P, _P, _I32, _P, _P, _P, _I64,
     _I32, _I32, ctypes.POINTER(DecodePlan), ctypes.c_float, _P, _P)
RX_DECODE_STATIC_SCRATCH_BYTES = 16 << 20
_sig("rx_test_fail_alloc", ctypes.c_int, _I64)
_sig("rx_decode_set_wait_limit", ctypes.c_int, _I64)


def rx_test_fail_alloc(n: int) -> None:
    """The n-th next radix-tree node allocation fails (0: off); see rx.h."""
    _check(_lib.rx_test_fail_alloc(int(n)))


def rx_decode_set_wait_limit(cycles: int) -> None:
    """Bound on each decode pipeline wait, in SM cycles (<= 0: the default)."""
    _check(_lib.rx_decode_set_wait_limit(int(cycles)))


def library():
    """The loaded ctypes.CDLL (for symbol checks)."""
    return _lib


def version() -> int:
    return _lib.rx_version()


def last_error() -> str:
    return _lib.rx_last_error().decode()


def _check(rc: int, allow=()) -> int:
    if rc != RX_OK and rc not in allow:
        raise RxError(rc, last_error())
    return rc


def _np(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------------------
# radix tree and slot free list (host)
# ---------------------------------------------------------------------------


class RadixTree:
    """rx_tree: prefix match, insert, LRU eviction and locks over token ids."""

    def __init__(self):
        h = _P()
        _check(_lib.rx_tree_create(ctypes.byref(h)))
        self._h = h

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            _lib.rx_tree_destroy(h)
            self._h = None

    def match_prefix(self, tokens: Sequence[int]) -> Tuple[int, List[int]]:
        t, tp = _np(tokens, np.int64)
        out = np.empty(max(1, len(t)), np.int32)
        k = ctypes.c_int64()
        _check(_lib.rx_match_prefix(self._h, tp, len(t), out.ctypes.data_as(_P), len(t),
                                    ctypes.byref(k)))
        return k.value, out[:k.value].tolist()

    def insert(self, tokens: Sequence[int], slots: Sequence[int]) -> int:
        t, tp = _np(tokens, np.int64)
        s, sp = _np(slots, np.int32)
        assert len(t) == len(s)
        k = ctypes.c_int64()
        _check(_lib.rx_insert(self._h, tp, sp, len(t), ctypes.byref(k)))
        return k.value

    def evict(self, num_tokens: int, cap: Optional[int] = None) -> List[int]:
        """Freed slots; raises RxError(RX_ERR_CAPACITY) if ``cap`` is too small."""
        if cap is None:
            _, _, ev = self.stats()
            cap = max(ev, 1)
        out = np.empty(max(1, cap), np.int32)
        n = ctypes.c_int64()
        rc = _lib.rx_evict_lru(self._h, int(num_tokens), out.ctypes.data_as(_P), cap, ctypes.byref(n))
        _check(rc, allow=(RX_ERR_NOT_ENOUGH,))
        return out[:n.value].tolist()

    def lock(self, tokens: Sequence[int], delta: int) -> int:
        t, tp = _np(tokens, np.int64)
        k = ctypes.c_int64()
        _check(_lib.rx_lock_prefix(self._h, tp, len(t), int(delta), ctypes.byref(k)))
        return k.value

    def prefix_len(self, tokens: Sequence[int]) -> int:
        """Cached prefix length, without touching the LRU clock."""
        t, tp = _np(tokens, np.int64)
        k = ctypes.c_int64()
        _check(_lib.rx_prefix_len(self._h, tp, len(t), ctypes.byref(k)))
        return k.value

    def stats(self) -> Tuple[int, int, int]:
        a, b, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        _check(_lib.rx_tree_stats(self._h, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)))
        return a.value, b.value, c.value

    def dump(self) -> List[dict]:
        need = ctypes.c_int64()
        _check(_lib.rx_tree_dump(self._h, None, 0, ctypes.byref(need)), allow=(RX_ERR_CAPACITY,))
        buf = np.empty(max(1, need.value), np.int64)
        _check(_lib.rx_tree_dump(self._h, buf.ctypes.data_as(_P), len(buf), ctypes.byref(need)))
        out, i = [], 0
        while i < need.value:
            nid, par, last, n = buf[i:i + 4].tolist()
            i += 4
            toks = buf[i:i + n].tolist()
            slots = buf[i + n:i + 2 * n].tolist()
            locks = buf[i + 2 * n:i + 3 * n].tolist()
            i += 3 * n
            out.append(dict(id=nid, parent=par, last=last, tokens=toks, slots=slots, locks=locks))
        return out

    def nodes(self) -> List[Tuple[Tuple[int, ...], Tuple[int, ...]]]:
        """Every node as (token path before it, its own tokens), sorted."""
        recs = self.dump()
        path = {}
        out = []
        for r in recs:  # depth-first: parents come before children
            before = () if r["parent"] < 0 else path[r["parent"]]
            path[r["id"]] = before + tuple(r["tokens"])
            out.append((before, tuple(r["tokens"])))
        return sorted(out)


class SlotAllocator:
    """rx_slot_alloc: first-in first-out free list of pool slots."""

    def __init__(self, free_order: Sequence[int], num_slots: int):
        o, op = _np(free_order, np.int32)
        h = _P()
        _check(_lib.rx_slot_alloc_create(op, len(o), int(num_slots), ctypes.byref(h)))
        self._h = h

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            _lib.rx_slot_alloc_destroy(h)
            self._h = None

    def take(self, n: int) -> np.ndarray:
        out = np.empty(max(1, n), np.int32)
        _check(_lib.rx_slot_alloc_take(self._h, int(n), out.ctypes.data_as(_P)))
        return out[:n]

    def give(self, slots: Sequence[int]) -> None:
        s, sp = _np(slots, np.int32)
        _check(_lib.rx_slot_alloc_give(self._h, sp, len(s)))

    def free_count(self) -> int:
        return _lib.rx_slot_alloc_free_count(self._h)


def rx_admit(tree: RadixTree, alloc: SlotAllocator, tokens: Sequence[int]):
    """(slot row int32 [n], prefix_len, evicted tokens)."""
    t, tp = _np(tokens, np.int64)
    row = np.empty(max(1, len(t)), np.int32)
    k, ev = ctypes.c_int64(), ctypes.c_int64()
    _check(_lib.rx_admit(tree._h, alloc._h, tp, len(t), row.ctypes.data_as(_P), ctypes.byref(k),
                         ctypes.byref(ev)))
    return row[:len(t)], k.value, ev.value


def rx_commit(tree: RadixTree, alloc: SlotAllocator, tokens: Sequence[int], row: Sequence[int],
              prefix_len: int) -> None:
    t, tp = _np(tokens, np.int64)
    r, rp = _np(row, np.int32)
    _check(_lib.rx_commit(tree._h, alloc._h, tp, rp, len(t), int(prefix_len)))


def rx_image_keys(data: bytes, n_tokens: int) -> np.ndarray:
    """int64 keys of the n_tokens positions an image (its raw bytes) occupies."""
    buf = np.frombuffer(bytes(data), dtype=np.uint8)
    out = np.empty(max(1, n_tokens), np.int64)
    _check(_lib.rx_image_keys(buf.ctypes.data_as(_P) if len(buf) else None, len(buf), int(n_tokens),
                              out.ctypes.data_as(_P)))
    return out[:n_tokens]


def rx_schedule(tree: RadixTree, requests: Sequence[Sequence[int]], policy: int):
    """(order int32 [n], cached prefix lengths int64 [n]) for waiting requests."""
    n = len(requests)
    offs = np.zeros(n + 1, np.int64)
    for i, r in enumerate(requests):
        offs[i + 1] = offs[i] + len(r)
    toks = np.concatenate([np.asarray(r, np.int64) for r in requests]) if n else np.zeros(0, np.int64)
    toks = np.ascontiguousarray(toks, np.int64)
    order = np.empty(max(1, n), np.int32)
    plen = np.empty(max(1, n), np.int64)
    _check(_lib.rx_schedule(tree._h, toks.ctypes.data_as(_P), offs.ctypes.data_as(_P), n, int(policy),
                            order.ctypes.data_as(_P), plen.ctypes.data_as(_P)))
    return order[:n], plen[:n]


# ---------------------------------------------------------------------------
# device entry points
# ---------------------------------------------------------------------------


def _torch():
    import torch
    return torch


def _dev(t, dtype, name):
    torch = _torch()
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name}: expected a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    return t


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _pool_dims(k_pool, v_pool, layer: int):
    """(num_slots, kv heads, head_dim, num_layers) of a one-layer pool
    [S, Hkv, d] or a layered one [L, S, Hkv, d]."""
    if k_pool.shape != v_pool.shape or k_pool.dim() not in (3, 4):
        raise ValueError("k_pool and v_pool must both be [num_slots, num_kv_heads, head_dim] or "
                         "[num_layers, num_slots, num_kv_heads, head_dim]")
    if k_pool.dim() == 3:
        return (*k_pool.shape, 0)
    L, S, hkv, d = k_pool.shape
    return S, hkv, d, L


def make_pool(k_pool, v_pool, layer: int = 0) -> KVPool:
    """The C pool of k_pool / v_pool: one layer [S, Hkv, d], or layer `layer`
    of a layered pool [L, S, Hkv, d]."""
    torch = _torch()
    _dev(k_pool, torch.bfloat16, "k_pool")
    _dev(v_pool, torch.bfloat16, "v_pool")
    S, hkv, d, L = _pool_dims(k_pool, v_pool, layer)
    return KVPool(k_pool.data_ptr(), v_pool.data_ptr(), S, hkv, d, L, int(layer))


def rx_kv_store(k_pool, v_pool, k_new, v_new, slots, dev_status=None, stream=None, layer: int = 0) -> None:
    torch = _torch()
    pool = make_pool(k_pool, v_pool, layer)
    _dev(k_new, torch.bfloat16, "k_new")
    _dev(v_new, torch.bfloat16, "v_new")
    _dev(slots, torch.int32, "slots")
    _dev(dev_status, torch.int32, "dev_status")
    n = slots.numel()
    if k_new.numel() != n * pool.num_kv_heads * pool.head_dim or k_new.shape != v_new.shape:
        raise ValueError("k_new/v_new must be [n, num_kv_heads, head_dim]")
    _check(_lib.rx_kv_store(ctypes.byref(pool), _ptr(k_new), _ptr(v_new), _ptr(slots), n,
                            _ptr(dev_status), _stream(stream)))


def rx_rope(x, pos, base: float, stream=None) -> None:
    """In place on x (bf16 [n, heads, head_dim]) at positions pos (int32 [n])."""
    torch = _torch()
    _dev(x, torch.bfloat16, "x")
    _dev(pos, torch.int32, "pos")
    if x.dim() != 3 or pos.numel() != x.shape[0]:
        raise ValueError("x must be [n, heads, head_dim] and pos [n]")
    _check(_lib.rx_rope(_ptr(x), _ptr(pos), x.shape[0], x.shape[1], x.shape[2], float(base), _stream(stream)))


def rx_kv_store_rope(k_pool, v_pool, k_new, v_new, slots, pos, base: float, dev_status=None,
                     stream=None, layer: int = 0) -> None:
    torch = _torch()
    pool = make_pool(k_pool, v_pool, layer)
    _dev(k_new, torch.bfloat16, "k_new")
    _dev(v_new, torch.bfloat16, "v_new")
    _dev(slots, torch.int32, "slots")
    _dev(pos, torch.int32, "pos")
    _dev(dev_status, torch.int32, "dev_status")
    n = slots.numel()
    if k_new.numel() != n * pool.num_kv_heads * pool.head_dim or k_new.shape != v_new.shape or pos.numel() != n:
        raise ValueError("k_new/v_new must be [n, num_kv_heads, head_dim] and pos [n]")
    _check(_lib.rx_kv_store_rope(ctypes.byref(pool), _ptr(k_new), _ptr(v_new), _ptr(slots), _ptr(pos), n,
                                 float(base), _ptr(dev_status), _stream(stream)))


def rx_kv_store_rope_fp8(k_pool, v_pool, k_scale: float, v_scale: float, k_new, v_new, slots, pos, base: float,
                         dev_status=None, stream=None, layer: int = 0) -> None:
    """rx_kv_store_rope into uint8 E4M3 pools ([L,] S, Hkv, d) with per-pool scales."""
    torch = _torch()
    _dev(k_pool, torch.uint8, "k_pool")
    _dev(v_pool, torch.uint8, "v_pool")
    _dev(k_new, torch.bfloat16, "k_new")
    _dev(v_new, torch.bfloat16, "v_new")
    _dev(slots, torch.int32, "slots")
    _dev(pos, torch.int32, "pos")
    _dev(dev_status, torch.int32, "dev_status")
    S, hkv, d, L = _pool_dims(k_pool, v_pool, layer)
    n = slots.numel()
    if k_new.shape != (n, hkv, d) or v_new.shape != k_new.shape or pos.numel() != n:
        raise ValueError("k_new/v_new must be [n, num_kv_heads, head_dim] and pos [n]")
    pool = KVPoolFp8(k_pool.data_ptr(), v_pool.data_ptr(), S, hkv, d, float(k_scale), float(v_scale), L,
                     int(layer))
    _check(_lib.rx_kv_store_rope_fp8(ctypes.byref(pool), _ptr(k_new), _ptr(v_new), _ptr(slots), _ptr(pos), n,
                                     float(base), _ptr(dev_status), _stream(stream)))


def rx_attn_extend_workspace(total_ctx_tokens: int, batch: int, num_kv_heads: int, head_dim: int) -> int:
    """Workspace bytes for rx_attn_extend's staged path (contexts summing to at
    most total_ctx_tokens tokens)."""
    n = _lib.rx_attn_extend_workspace(int(total_ctx_tokens), int(batch), int(num_kv_heads), int(head_dim))
    if n == 0:
        raise RxError(last_error())
    return int(n)


def rx_attn_extend(k_pool, v_pool, q, o, lse, qo_indptr, req_idx, prefix_len, extend_len,
                   req_to_token, max_extend_len: int, sm_scale: float, dev_status=None,
                   stream=None, workspace=None, layer: int = 0) -> None:
    """Extend attention; `workspace` (a device uint8 tensor of at least
    rx_attn_extend_workspace(...) bytes) selects the staged path."""
    torch = _torch()
    pool = make_pool(k_pool, v_pool, layer)
    for t, n in ((q, "q"), (o, "o")):
        _dev(t, torch.bfloat16, n)
    _dev(lse, torch.float32, "lse")
    for t, n in ((qo_indptr, "qo_indptr"), (req_idx, "req_idx"), (prefix_len, "prefix_len"),
                 (extend_len, "extend_len"), (req_to_token, "req_to_token")):
        _dev(t, torch.int32, n)
    _dev(dev_status, torch.int32, "dev_status")
    _dev(workspace, torch.uint8, "workspace")
    if q.dim() != 3 or q.shape != o.shape:
        raise ValueError("q and o must be [tokens, num_q_heads, head_dim]")
    ws_bytes = 0 if workspace is None else workspace.numel()
    _check(_lib.rx_attn_extend(ctypes.byref(pool), _ptr(q), _ptr(o), _ptr(lse), q.shape[1],
                               _ptr(qo_indptr), _ptr(req_idx), _ptr(prefix_len), _ptr(extend_len),
                               _ptr(req_to_token), req_to_token.shape[1], req_idx.numel(),
                               int(max_extend_len), _ptr(workspace), ws_bytes, float(sm_scale),
                               _ptr(dev_status), _stream(stream)))


@dataclass
class DevicePlan:
    """A decode plan copied to the device; keeps its buffer alive."""

    buf: object          # torch int32 tensor on the device
    info: DecodePlanInfo
    batch: int
    struct: DecodePlan


def rx_decode_plan_build(req_to_token_host, req_idx_host, seq_len_host, num_q_heads: int,
                         num_kv_heads: int, kv_chunk: int = 0, min_shared: int = 16):
    """Host plan: (packed int32 numpy buffer, DecodePlanInfo)."""
    rtt, rp = _np(req_to_token_host, np.int32)
    ri, rip = _np(req_idx_host, np.int32)
    sl, slp = _np(seq_len_host, np.int32)
    info = DecodePlanInfo()
    # one call with room for the usual plan sizes; a second one only when the
    # library reports that more words are needed
    buf = np.empty(2 * len(ri) + 8 * max(8192, 64 * len(ri)), np.int32)
    rc = _lib.rx_decode_plan_build(rp, rtt.shape[1], rip, slp, len(ri), num_q_heads, num_kv_heads,
                                   kv_chunk, min_shared, buf.ctypes.data_as(_P), len(buf), ctypes.byref(info))
    if rc == RX_ERR_CAPACITY:
        buf = np.empty(max(1, info.buf_words), np.int32)
        rc = _lib.rx_decode_plan_build(rp, rtt.shape[1], rip, slp, len(ri), num_q_heads, num_kv_heads,
                                       kv_chunk, min_shared, buf.ctypes.data_as(_P), len(buf), ctypes.byref(info))
    _check(rc)
    return buf[:info.buf_words], info


def plan_to_device(buf: np.ndarray, info: DecodePlanInfo, batch: int, device="cuda") -> DevicePlan:
    torch = _torch()
    d = torch.from_numpy(np.ascontiguousarray(buf)).to(device)
    base = d.data_ptr()
    st = DecodePlan(base, base + 4 * batch, base + 8 * batch, info.n_items, info.max_parts, info.n_wide)
    return DevicePlan(d, info, batch, st)


def rx_attn_decode_workspace(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                             max_seq_len: int, plan: Optional[DevicePlan] = None) -> int:
    pp = ctypes.byref(plan.struct) if plan is not None else None
    return _lib.rx_attn_decode_workspace(batch, num_q_heads, num_kv_heads, head_dim, max_seq_len, pp)


def rx_attn_decode(k_pool, v_pool, q, o, lse, req_idx, seq_len, req_to_token, max_seq_len: int,
                   sm_scale: float, plan: Optional[DevicePlan] = None, workspace=None,
                   dev_status=None, stream=None, layer: int = 0) -> None:
    torch = _torch()
    pool = make_pool(k_pool, v_pool, layer)
    _dev(q, torch.bfloat16, "q")
    _dev(o, torch.bfloat16, "o")
    _dev(lse, torch.float32, "lse")
    for t, n in ((req_idx, "req_idx"), (seq_len, "seq_len"), (req_to_token, "req_to_token")):
        _dev(t, torch.int32, n)
    _dev(dev_status, torch.int32, "dev_status")
    if workspace is not None:
        _dev(workspace, workspace.dtype, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    pp = ctypes.byref(plan.struct) if plan is not None else None
    _check(_lib.rx_attn_decode(ctypes.byref(pool), _ptr(q), _ptr(o), _ptr(lse), q.shape[1],
                               _ptr(req_idx), _ptr(seq_len), _ptr(req_to_token),
                               req_to_token.shape[1], req_idx.numel(), int(max_seq_len), pp,
                               _ptr(workspace), ws_bytes, float(sm_scale), _ptr(dev_status),
                               _stream(stream)))


def rx_attn_decode_static(k_pool, v_pool, q, o, lse, req_idx, seq_len, req_to_token, max_seq_len: int,
                          sm_scale: float, plan: Optional[DevicePlan] = None, dev_status=None,
                          stream=None, layer: int = 0) -> None:
    """rx_attn_decode with the library's fixed scratch array instead of a
    workspace (for callers that cannot allocate device memory; see rx.h)."""
    torch = _torch()
    pool = make_pool(k_pool, v_pool, layer)
    _dev(q, torch.bfloat16, "q")
    _dev(o, torch.bfloat16, "o")
    _dev(lse, torch.float32, "lse")
    for t, n in ((req_idx, "req_idx"), (seq_len, "seq_len"), (req_to_token, "req_to_token")):
        _dev(t, torch.int32, n)
    _dev(dev_status, torch.int32, "dev_status")
    pp = ctypes.byref(plan.struct) if plan is not None else None
    _check(_lib.rx_attn_decode_static(ctypes.byref(pool), _ptr(q), _ptr(o), _ptr(lse), q.shape[1],
                                      _ptr(req_idx), _ptr(seq_len), _ptr(req_to_token),
                                      req_to_token.shape[1], req_idx.numel(), int(max_seq_len), pp,
                                      float(sm_scale), _ptr(dev_status), _stream(stream)))


# ---------------------------------------------------------------------------
# compressed finite-state machine (constrained decoding)
# ---------------------------------------------------------------------------


def rx_fsm_compress(n_states: int, vocab: int, row_ptr, tok, nxt, max_jump: int):
    """Host compression of a token automaton (CSR).  Returns (mask uint32
    [S, W], rank int32 [S, W] with W = ceil(V / 128) * 4, jump_len int32 [S],
    jump_off int64 [S], jump_end int32 [S], jump_tok int32 [total], info)."""
    rp, rpp = _np(row_ptr, np.int64)
    t, tp = _np(tok, np.int32)
    n, np_ = _np(nxt, np.int32)
    info = FsmInfo()
    _check(_lib.rx_fsm_compress(int(n_states), int(vocab), rpp, tp if len(t) else None, np_ if len(n) else None,
                                int(max_jump), None, None, None, None, None, None, 0, ctypes.byref(info)))
    W = (int(vocab) + 127) // 128 * 4   # mask words per state, rows padded to 16 bytes
    mask = np.empty((int(n_states), W), np.uint32)
    rank = np.empty((int(n_states), W), np.int32)
    jl = np.empty(int(n_states), np.int32)
    jo = np.empty(int(n_states), np.int64)
    je = np.empty(int(n_states), np.int32)
    jt = np.empty(max(1, int(info.jump_tokens)), np.int32)
    _check(_lib.rx_fsm_compress(int(n_states), int(vocab), rpp, tp if len(t) else None, np_ if len(n) else None,
                                int(max_jump), mask.ctypes.data_as(_P), rank.ctypes.data_as(_P),
                                jl.ctypes.data_as(_P), jo.ctypes.data_as(_P), je.ctypes.data_as(_P),
                                jt.ctypes.data_as(_P), len(jt), ctypes.byref(info)))
    return mask, rank, jl, jo, je, jt[:int(info.jump_tokens)], info


class Fsm:
    """A compressed machine resident on the current CUDA device: the
    automaton and its compression (rx_fsm_compress), as torch tensors."""

    def __init__(self, n_states: int, vocab: int, row_ptr, tok, nxt, max_jump: int):
        torch = _torch()
        mask, rank, jl, jo, je, jt, info = rx_fsm_compress(n_states, vocab, row_ptr, tok, nxt, max_jump)
        self.info = info
        self.n_states, self.vocab, self.max_jump = int(n_states), int(vocab), int(max_jump)

        def dev(a, dt):
            a = np.ascontiguousarray(a, dtype=dt)
            if a.size == 0:
                a = np.zeros(1, dt)
            return torch.from_numpy(a).cuda()

        self.row_ptr = dev(row_ptr, np.int64)
        self.tok = dev(tok, np.int32)
        self.nxt = dev(nxt, np.int32)
        self.mask = torch.from_numpy(mask.view(np.int32)).cuda()
        self.rank = torch.from_numpy(rank).cuda()
        self.jump_len, self.jump_off = dev(jl, np.int32), dev(jo, np.int64)
        self.jump_end, self.jump_tok = dev(je, np.int32), dev(jt, np.int32)
        self.struct = FsmStruct(self.row_ptr.data_ptr(), self.tok.data_ptr(), self.nxt.data_ptr(),
                                self.mask.data_ptr(), self.rank.data_ptr(), self.jump_len.data_ptr(),
                                self.jump_off.data_ptr(),
                                self.jump_end.data_ptr(), self.jump_tok.data_ptr(), self.n_states, self.vocab,
                                self.max_jump)


def fsm_workspace(batch: int):
    """The zeroed device workspace rx_fsm_step needs for `batch` requests:
    batch + 1 words (every call leaves it zero, so it can be kept and
    reused)."""
    torch = _torch()
    return torch.zeros(max(1, int(batch)) + 1, dtype=torch.int64, device="cuda")


def rx_fsm_step(fsm: Fsm, logits, state, out_tokens, out_count, workspace, dev_status=None,
                stream=None) -> None:
    """One constrained decoding step: logits fp32 [B, >= V] (rows 16-byte
    aligned), state int32 [B] (updated), out_tokens int32 [B, 1 + max_jump],
    out_count int32 [B], workspace from fsm_workspace(B)."""
    torch = _torch()
    _dev(workspace, torch.int64, "workspace")
    if workspace.numel() < state.numel():
        raise ValueError("rx_fsm_step: workspace smaller than the batch")
    _dev(logits, torch.float32, "logits")
    _dev(state, torch.int32, "state")
    _dev(out_tokens, torch.int32, "out_tokens")
    _dev(out_count, torch.int32, "out_count")
    _dev(dev_status, torch.int32, "dev_status")
    B = state.numel()
    if logits.dim() != 2 or logits.shape[0] != B or out_tokens.shape != (B, 1 + fsm.max_jump) or \
            out_count.numel() != B:
        raise ValueError("rx_fsm_step: logits [B, V], out_tokens [B, 1 + max_jump], out_count [B]")
    _check(_lib.rx_fsm_step(ctypes.byref(fsm.struct), _ptr(logits), logits.shape[1], B, _ptr(state),
                            _ptr(out_tokens), _ptr(out_count), _ptr(workspace), _ptr(dev_status),
                            _stream(stream)))


# ---------------------------------------------------------------------------
# FP8 key/value pools
# ---------------------------------------------------------------------------


def rx_kv_store_fp8(k_pool, v_pool, k_scale: float, v_scale: float, k_new, v_new, slots, dev_status=None,
                    stream=None, layer: int = 0) -> None:
    """Store bf16 rows into uint8 E4M3 pools ([L,] S, Hkv, d) with per-pool scales."""
    torch = _torch()
    _dev(k_pool, torch.uint8, "k_pool")
    _dev(v_pool, torch.uint8, "v_pool")
    _dev(k_new, torch.bfloat16, "k_new")
    _dev(v_new, torch.bfloat16, "v_new")
    _dev(slots, torch.int32, "slots")
    _dev(dev_status, torch.int32, "dev_status")
    S, hkv, d, L = _pool_dims(k_pool, v_pool, layer)
    n = slots.numel()
    if k_new.shape != (n, hkv, d) or v_new.shape != k_new.shape:
        raise ValueError("k_new/v_new must be [n, num_kv_heads, head_dim]")
    pool = KVPoolFp8(k_pool.data_ptr(), v_pool.data_ptr(), S, hkv, d, float(k_scale), float(v_scale), L,
                     int(layer))
    _check(_lib.rx_kv_store_fp8(ctypes.byref(pool), _ptr(k_new), _ptr(v_new), _ptr(slots), n,
                                _ptr(dev_status), _stream(stream)))


def rx_attn_extend_fp8(k_pool, v_pool, k_scale: float, v_scale: float, q, o, lse, qo_indptr, req_idx,
                       prefix_len, extend_len, req_to_token, max_extend_len: int, sm_scale: float, workspace,
                       dev_status=None, stream=None, layer: int = 0) -> None:
    """Extend attention over uint8 E4M3 pools ([L,] S, Hkv, d) with per-pool
    scales; `workspace` (at least rx_attn_extend_workspace(...) bytes, or
    None for the gather path) as in rx_attn_extend."""
    torch = _torch()
    _dev(k_pool, torch.uint8, "k_pool")
    _dev(v_pool, torch.uint8, "v_pool")
    for t, n in ((q, "q"), (o, "o")):
        _dev(t, torch.bfloat16, n)
    _dev(lse, torch.float32, "lse")
    for t, n in ((qo_indptr, "qo_indptr"), (req_idx, "req_idx"), (prefix_len, "prefix_len"),
                 (extend_len, "extend_len"), (req_to_token, "req_to_token")):
        _dev(t, torch.int32, n)
    _dev(dev_status, torch.int32, "dev_status")
    _dev(workspace, torch.uint8, "workspace")
    if q.dim() != 3 or q.shape != o.shape:
        raise ValueError("q and o must be [tokens, num_q_heads, head_dim]")
    S, hkv, d, L = _pool_dims(k_pool, v_pool, layer)
    pool = KVPoolFp8(k_pool.data_ptr(), v_pool.data_ptr(), S, hkv, d, float(k_scale), float(v_scale), L,
                     int(layer))
    ws_bytes = 0 if workspace is None else workspace.numel()
    _check(_lib.rx_attn_extend_fp8(ctypes.byref(pool), _ptr(q), _ptr(o), _ptr(lse), q.shape[1],
                                   _ptr(qo_indptr), _ptr(req_idx), _ptr(prefix_len), _ptr(extend_len),
                                   _ptr(req_to_token), req_to_token.shape[1], req_idx.numel(),
                                   int(max_extend_len), _ptr(workspace), ws_bytes, float(sm_scale),
                                   _ptr(dev_status), _stream(stream)))


def rx_attn_decode_fp8(k_pool, v_pool, k_scale: float, v_scale: float, q, o, lse, req_idx, seq_len, req_to_token,
                       max_seq_len: int, sm_scale: float, plan: DevicePlan, workspace, dev_status=None, stream=None,
                       layer: int = 0) -> None:
    """Decode attention over uint8 E4M3 pools ([L,] S, Hkv, d) with per-pool
    scales; the plan (or None) and the workspace (rx_attn_decode_workspace
    bytes, or None when no row is split) as in rx_attn_decode."""
    torch = _torch()
    _dev(k_pool, torch.uint8, "k_pool")
    _dev(v_pool, torch.uint8, "v_pool")
    _dev(q, torch.bfloat16, "q")
    _dev(o, torch.bfloat16, "o")
    _dev(lse, torch.float32, "lse")
    for t, n in ((req_idx, "req_idx"), (seq_len, "seq_len"), (req_to_token, "req_to_token")):
        _dev(t, torch.int32, n)
    _dev(dev_status, torch.int32, "dev_status")
    if workspace is not None:
        _dev(workspace, workspace.dtype, "workspace")
    S, hkv, d, L = _pool_dims(k_pool, v_pool, layer)
    pool = KVPoolFp8(k_pool.data_ptr(), v_pool.data_ptr(), S, hkv, d, float(k_scale), float(v_scale), L, int(layer))
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    pp = ctypes.byref(plan.struct) if plan is not None else None
    _check(_lib.rx_attn_decode_fp8(ctypes.byref(pool), _ptr(q), _ptr(o), _ptr(lse), q.shape[1], _ptr(req_idx),
                                   _ptr(seq_len), _ptr(req_to_token), req_to_token.shape[1], req_idx.numel(),
                                   int(max_seq_len), pp, _ptr(workspace), ws_bytes, float(sm_scale),
                                   _ptr(dev_status), _stream(stream)))
