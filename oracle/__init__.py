"""Oracle for the slot-indexed attention path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  It shares no code with the CUDA path: ``attn_fp64.c`` is plain C
compiled with gcc, ``tree_ref.py`` is plain Python, and nothing here imports
``prefix_shared_kv_radixattention_gb300`` except its ``inputs`` module, which
only draws seeded inputs.

Contents
  * ``kv_store``            -- definition of the pool scatter (attn_fp64.c)
  * ``attention``           -- fp64 softmax(q K^T * scale + causal) V gathered
                               through req_to_token (attn_fp64.c)
  * ``extend`` / ``decode`` -- the two query layouts of the path, mapped onto
                               ``attention``
  * ``merge_partials``      -- log-sum-exp combination of partial results
  * ``rope`` / ``rope_f64``  -- rotary position embedding (rotate-half form)
  * ``tree_ref.RadixTreeRef`` -- per-token trie with LRU eviction
  * ``tree_ref.schedule`` / ``tree_ref.optimal_hit_rate`` -- cache-aware
                               request order and the optimal cache hit rate
  * ``keys.image_keys``       -- radix-tree keys of an image's tokens
  * ``fp8.encode`` / ``fp8.quantize_rows`` -- E4M3 codes of FP8 key/value
                               pools (nearest, ties to even, saturating)
  * ``fsm.compress`` / ``fsm.step`` -- the compressed finite-state machine of
                               constrained decoding: jumps over fixed tokens,
                               and a masked-argmax decoding step with them

Every function here is pinned in ``tests/test_oracle_pins.py``,
``tests/test_tree_oracle.py``, ``tests/test_image_keys.py``,
``tests/test_fsm_oracle.py`` and ``tests/test_fp8_oracle.py``; none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle_attn.so")
_SRC = os.path.join(_HERE, "attn_fp64.c")
_lock = threading.Lock()
_lib = None


def build(src: str = _SRC, out: str = _LIB_PATH, extra=()) -> str:
    """Compile attn_fp64.c with gcc -O2 (no fast-math) into a shared library."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-std=c99", "-D_POSIX_C_SOURCE=200809L",
           *extra, src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _stale() -> bool:
    return (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)


def _bind(lib):
    P = ctypes.c_void_p
    i64 = ctypes.c_int64
    i32 = ctypes.c_int
    lib.oracle_kv_store.argtypes = [P, P, i64, i32, i32, P, P, P, i64]
    lib.oracle_kv_store.restype = i32
    lib.oracle_attention.argtypes = [P, i64, i32, P, P, i64, i32, i32, P, i64, P, P, P,
                                     ctypes.c_double, P, P, i32]
    lib.oracle_attention.restype = i32
    return lib


def load(path: str = None):
    """Load (building first if needed) the compiled oracle."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if _stale():
                build()
            _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------
# KV store
# ---------------------------------------------------------------------------


def kv_store(k_pool: np.ndarray, v_pool: np.ndarray, k_new: np.ndarray, v_new: np.ndarray,
             slots: np.ndarray, lib=None) -> None:
    """In place: pool[slots[i]] = new[i] for K and V (bf16 bits, [S, Hkv, d])."""
    lib = lib or load()
    S, hkv, d = k_pool.shape
    assert k_pool.dtype == np.uint16 and k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    k_new = np.ascontiguousarray(k_new, dtype=np.uint16)
    v_new = np.ascontiguousarray(v_new, dtype=np.uint16)
    slots = np.ascontiguousarray(slots, dtype=np.int32)
    rc = lib.oracle_kv_store(_ptr(k_pool), _ptr(v_pool), S, hkv, d, _ptr(k_new), _ptr(v_new),
                             _ptr(slots), len(slots))
    if rc != 0:
        raise ValueError(f"oracle_kv_store: status {rc}")


# ---------------------------------------------------------------------------
# Rotary position embedding (not from the pages, which do not reach inside
# the model: the position encoding the Llama-family models whose attention
# shapes the workloads use apply to q and k before attention)
# ---------------------------------------------------------------------------


def rope_f64(x: np.ndarray, pos, base: float) -> np.ndarray:
    """Rotate-half rotary embedding of x [n, heads, d] (fp64) at positions
    pos [n]: for c < d/2, with theta_c = base^(-2c/d) and a = pos * theta_c,
        x'[c]       = x[c] cos a - x[c + d/2] sin a
        x'[c + d/2] = x[c + d/2] cos a + x[c] sin a."""
    x = np.asarray(x, np.float64)
    n, h, d = x.shape
    half = d // 2
    theta = float(base) ** (-2.0 * np.arange(half, dtype=np.float64) / d)
    a = np.asarray(pos, np.float64).reshape(n, 1, 1) * theta.reshape(1, 1, half)
    c, s = np.cos(a), np.sin(a)
    lo, hi = x[..., :half], x[..., half:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


def rope(x_bf16: np.ndarray, pos, base: float) -> np.ndarray:
    """rope_f64 of bf16 bits (uint16 [n, heads, d]), widened exactly."""
    bits = np.ascontiguousarray(x_bf16, dtype=np.uint16).astype(np.uint32) << 16
    return rope_f64(bits.view(np.float32).astype(np.float64), pos, base)


# ---------------------------------------------------------------------------
# Attention
# ---------------------------------------------------------------------------


def attention(q, k_pool, v_pool, rtt, q_row, kbeg, kend, sm_scale, n_threads=None, lib=None):
    """fp64 attention of query rows over explicit key ranges of their rtt rows.

    q bf16 [n_q, Hq, d]; returns (o fp64 [n_q, Hq, d], lse fp64 [n_q, Hq]).
    """
    lib = lib or load()
    q = np.ascontiguousarray(q, dtype=np.uint16)
    n_q, hq, d = q.shape
    S, hkv, d2 = k_pool.shape
    assert d == d2
    rtt = np.ascontiguousarray(rtt, dtype=np.int32)
    q_row = np.ascontiguousarray(q_row, dtype=np.int32)
    kbeg = np.ascontiguousarray(kbeg, dtype=np.int32)
    kend = np.ascontiguousarray(kend, dtype=np.int32)
    o = np.empty((n_q, hq, d), dtype=np.float64)
    lse = np.empty((n_q, hq), dtype=np.float64)
    rc = lib.oracle_attention(_ptr(q), n_q, hq, _ptr(np.ascontiguousarray(k_pool)),
                              _ptr(np.ascontiguousarray(v_pool)), S, hkv, d, _ptr(rtt),
                              rtt.shape[1], _ptr(q_row), _ptr(kbeg), _ptr(kend), float(sm_scale),
                              _ptr(o), _ptr(lse), int(n_threads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle_attention: status {rc}")
    return o, lse


def extend(q, k_pool, v_pool, rtt, req_idx, prefix_len, extend_len, qo_indptr, sm_scale,
           n_threads=None, lib=None):
    """Extend rows: token i of request b sits at position P_b + i and sees keys 0..P_b+i."""
    n_q = int(qo_indptr[-1])
    q_row = np.empty(n_q, dtype=np.int32)
    kend = np.empty(n_q, dtype=np.int32)
    for b in range(len(req_idx)):
        s, e = int(qo_indptr[b]), int(qo_indptr[b + 1])
        assert e - s == int(extend_len[b])
        q_row[s:e] = req_idx[b]
        kend[s:e] = int(prefix_len[b]) + np.arange(1, e - s + 1)
    return attention(q, k_pool, v_pool, rtt, q_row, np.zeros(n_q, np.int32), kend, sm_scale,
                     n_threads, lib)


def decode(q, k_pool, v_pool, rtt, req_idx, seq_len, sm_scale, n_threads=None, lib=None):
    """Decode rows: one query per request at position L_b - 1, keys 0..L_b-1."""
    n = len(req_idx)
    return attention(q, k_pool, v_pool, rtt, np.asarray(req_idx, np.int32), np.zeros(n, np.int32),
                     np.asarray(seq_len, np.int32), sm_scale, n_threads, lib)


def merge_partials(o_parts: np.ndarray, lse_parts: np.ndarray):
    """Combine partial attention results over disjoint key sets.

    With m = max_s lse_s and w_s = exp(lse_s - m):
      o = sum_s w_s o_s / sum_s w_s,  lse = m + log(sum_s w_s).
    o_parts [..., P, d], lse_parts [..., P] (fp64).
    """
    m = np.max(lse_parts, axis=-1, keepdims=True)
    w = np.exp(lse_parts - m)
    tot = np.sum(w, axis=-1, keepdims=True)
    o = np.sum(w[..., None] * o_parts, axis=-2) / tot
    return o, (m + np.log(tot))[..., 0]
