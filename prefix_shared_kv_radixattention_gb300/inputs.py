"""Seeded synthetic inputs for the slot-indexed attention path.

This module only *draws* inputs: token ids, bf16 Q/K/V values, slot ids and
the per-request slot lists (``req_to_token``).  It holds none of the
method's arithmetic (no attention, no radix tree, no scatter), so both the
fp64 oracle and the CUDA path can be fed from it.

Workload families stand in for the ones the article "SGLang: Efficient
Execution of Structured Language Model Programs" (unite.ai) evaluates in its
section "Introducción a SGLang" (few-shot benchmarks, multi-turn chat) and
"SGLang: Modelo de programación y metodología" (fork/branching programs,
the radix-tree walkthrough).  None of those suites' items are used: token
ids are random integers and every value is N(0, 1).

Recipe (shared by every family):
  * ``rng = numpy.random.default_rng(seed)``; draws happen in a fixed order:
    token ids, slot permutation, cached K/V, new K/V, queries.
  * values ~ N(0, 1) drawn in float32 and rounded to bf16 round-to-nearest-
    even by ``bf16_round`` below.
  * slot ids: a seeded random permutation of ``[0, num_slots)``, handed out
    in order of first use (shared prefix tokens first, then each request's
    private tokens in request order, then the step's new tokens).
  * the long multi-turn chat instead comes as a ``Scenario``: token
    sequences and a free list only; its slot lists are whatever the radix
    cache hands out when the scenario's admissions are replayed through it
    (``problem_from_admission`` then draws the values).
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np

# -------------------------------------------------------------------------
# bf16 helpers (bit manipulation only)
# -------------------------------------------------------------------------


def bf16_round(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bits (uint16), round to nearest, ties to even: add
    0x7FFF plus the lowest kept bit to the float's bits, keep the top half."""
    u = np.array(x, dtype=np.float32, copy=True).view(np.uint32)
    lsb = u >> np.uint32(16)
    lsb &= np.uint32(1)
    u += lsb
    u += np.uint32(0x7FFF)
    u >>= np.uint32(16)
    return u.astype(np.uint16)


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    """bf16 bits (uint16) -> float32, exact."""
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def randn_bf16(rng: np.random.Generator, shape, chunk: int = 1 << 24) -> np.ndarray:
    """N(0,1) values rounded to bf16, drawn in float32 in fixed-size chunks."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = bf16_round(rng.standard_normal(e - s, dtype=np.float32))
    return out.reshape(shape)


# -------------------------------------------------------------------------
# Problem description
# -------------------------------------------------------------------------


@dataclasses.dataclass
class Problem:
    """One batch of the slot-indexed attention path.

    Pool rows ``cached_slots`` hold ``cached_k/v`` before the step; the step
    first stores ``new_k/v`` at ``new_slots`` and then runs attention:
      * extend rows: request ``ext_req_idx[b]`` (a row of ``req_to_token``)
        has ``ext_prefix_len[b]`` cached tokens and ``ext_extend_len[b]``
        new ones, queries packed along ``qo_indptr``;
      * decode rows: request ``dec_req_idx[b]`` has ``dec_seq_len[b]``
        tokens including its new one, one query each.
    """

    name: str
    hq: int
    hkv: int
    d: int
    num_slots: int
    req_to_token: np.ndarray          # int32 [R, stride]
    tokens: List[np.ndarray]          # int64 token ids per req_to_token row
    cached_slots: np.ndarray          # int32 [Nc]
    cached_k: np.ndarray              # uint16 (bf16) [Nc, hkv, d]
    cached_v: np.ndarray
    new_slots: np.ndarray             # int32 [Nn]
    new_k: np.ndarray                 # uint16 [Nn, hkv, d]
    new_v: np.ndarray
    ext_req_idx: np.ndarray           # int32 [Be]
    ext_prefix_len: np.ndarray        # int32 [Be]
    ext_extend_len: np.ndarray        # int32 [Be]
    qo_indptr: np.ndarray             # int32 [Be + 1]
    q_ext: np.ndarray                 # uint16 [sum E, hq, d]
    dec_req_idx: np.ndarray           # int32 [Bd]
    dec_seq_len: np.ndarray           # int32 [Bd]
    q_dec: np.ndarray                 # uint16 [Bd, hq, d]
    seed: int = 0

    @property
    def sm_scale(self) -> float:
        return 1.0 / float(np.sqrt(self.d))

    @property
    def rtt_stride(self) -> int:
        return int(self.req_to_token.shape[1])

    @property
    def kv_row_bytes(self) -> int:
        """Bytes of K plus V for one token (all kv heads)."""
        return 2 * self.hkv * self.d * 2

    def decode_unique_tokens(self) -> int:
        """Distinct pool slots that the decode rows read."""
        if len(self.dec_req_idx) == 0:
            return 0
        s = set()
        for r, L in zip(self.dec_req_idx, self.dec_seq_len):
            s.update(self.req_to_token[r, :L].tolist())
        return len(s)

    def decode_dense_tokens(self) -> int:
        return int(np.sum(self.dec_seq_len, dtype=np.int64))

    def extend_flops(self) -> int:
        """4*d per unmasked (query, key, q-head) triple: 2*d for QK^T, 2*d for PV."""
        pairs = 0
        for P, E in zip(self.ext_prefix_len.tolist(), self.ext_extend_len.tolist()):
            pairs += E * P + E * (E + 1) // 2
        return 4 * self.d * self.hq * pairs

    def decode_flops(self) -> int:
        return 4 * self.d * self.hq * self.decode_dense_tokens()


class _SlotSource:
    """Hands out a seeded permutation of [0, num_slots) in order of use."""

    def __init__(self, rng: np.random.Generator, num_slots: int):
        self.perm = rng.permutation(num_slots).astype(np.int32)
        self.next = 0

    def take(self, n: int) -> np.ndarray:
        if self.next + n > len(self.perm):
            raise ValueError("workload needs more slots than the pool holds")
        out = self.perm[self.next:self.next + n]
        self.next += n
        return out


def _tokens(rng: np.random.Generator, n: int, lo: int) -> np.ndarray:
    """n distinct-looking token ids from a disjoint range starting at lo."""
    return (lo + rng.permutation(n)).astype(np.int64)


def _empty_i32():
    return np.zeros(0, dtype=np.int32)


def _finish(name, seed, rng, hq, hkv, d, num_slots, rows, cached_slots, new_slots,
            ext, dec, draw_values=True) -> Problem:
    """Draw values and assemble a Problem.

    rows: list of (token ids int64, slot ids int32) per req_to_token row.
    ext:  list of (row, prefix_len, extend_len).
    dec:  list of (row, seq_len).
    With draw_values=False the value arrays have zero rows (structure only).
    """
    if not draw_values:
        def randn_bf16(_rng, shape):  # noqa: F811 - structure-only stand-in
            return np.zeros((0,) + tuple(shape[1:]), dtype=np.uint16)
    else:
        randn_bf16 = globals()["randn_bf16"]
    stride = max(len(s) for _, s in rows)
    stride = (stride + 15) // 16 * 16
    rtt = np.full((len(rows), stride), -1, dtype=np.int32)
    for i, (_, s) in enumerate(rows):
        rtt[i, :len(s)] = s
    cached_k = randn_bf16(rng, (len(cached_slots), hkv, d))
    cached_v = randn_bf16(rng, (len(cached_slots), hkv, d))
    new_k = randn_bf16(rng, (len(new_slots), hkv, d))
    new_v = randn_bf16(rng, (len(new_slots), hkv, d))
    ext_req = np.array([e[0] for e in ext], dtype=np.int32) if ext else _empty_i32()
    ext_P = np.array([e[1] for e in ext], dtype=np.int32) if ext else _empty_i32()
    ext_E = np.array([e[2] for e in ext], dtype=np.int32) if ext else _empty_i32()
    qo = np.zeros(len(ext) + 1, dtype=np.int32)
    if ext:
        qo[1:] = np.cumsum(ext_E)
    q_ext = randn_bf16(rng, (int(qo[-1]), hq, d))
    dec_req = np.array([x[0] for x in dec], dtype=np.int32) if dec else _empty_i32()
    dec_L = np.array([x[1] for x in dec], dtype=np.int32) if dec else _empty_i32()
    q_dec = randn_bf16(rng, (len(dec), hq, d))
    return Problem(name=name, hq=hq, hkv=hkv, d=d, num_slots=num_slots,
                   req_to_token=rtt, tokens=[t for t, _ in rows],
                   cached_slots=np.asarray(cached_slots, dtype=np.int32),
                   cached_k=cached_k, cached_v=cached_v,
                   new_slots=np.asarray(new_slots, dtype=np.int32), new_k=new_k, new_v=new_v,
                   ext_req_idx=ext_req, ext_prefix_len=ext_P, ext_extend_len=ext_E,
                   qo_indptr=qo, q_ext=q_ext, dec_req_idx=dec_req, dec_seq_len=dec_L,
                   q_dec=q_dec, seed=seed)


# -------------------------------------------------------------------------
# Workload families (defaults = the full-size configurations)
# -------------------------------------------------------------------------


def tiny_extend(seed: int = 1001, hq: int = 4, hkv: int = 4, d: int = 64, batch: int = 4,
                prefix: int = 64, extend: int = 16, num_slots: int = 512,
                draw_values: bool = True) -> Problem:
    """Requests sharing one cached prefix, each extending it causally.

    Full size: 4 q heads = 4 kv heads, head_dim 64, 4 requests on one
    64-token prefix, 16 new tokens each, 512-slot pool.
    """
    rng = np.random.default_rng(seed)
    shared_tok = _tokens(rng, prefix, 1_000_000)
    new_tok = [_tokens(rng, extend, 2_000_000 + 10_000 * b) for b in range(batch)]
    src = _SlotSource(rng, num_slots)
    shared_slots = src.take(prefix)
    rows, new_slots = [], []
    for b in range(batch):
        s_new = src.take(extend)
        new_slots.append(s_new)
        rows.append((np.concatenate([shared_tok, new_tok[b]]), np.concatenate([shared_slots, s_new])))
    ext = [(b, prefix, extend) for b in range(batch)]
    return _finish("tiny_extend", seed, rng, hq, hkv, d, num_slots, rows, shared_slots,
                   np.concatenate(new_slots), ext, [], draw_values)


def few_shot_decode(seed: int = 1002, hq: int = 32, hkv: int = 32, d: int = 128, batch: int = 64,
                    shared: int = 1024, private: int = 256, num_slots: int = 2 * 1024 * 1024,
                    draw_values: bool = True) -> Problem:
    """Few-shot batch: one shared example prefix, a private question each, one decode token.

    Full size: Llama-2-7B attention shape (32 = 32 heads, head_dim 128),
    64 requests of 1024 shared + 256 private + 1 new token, 2M-slot pool.
    """
    rng = np.random.default_rng(seed)
    shared_tok = _tokens(rng, shared, 1_000_000)
    priv_tok = [_tokens(rng, private + 1, 3_000_000 + 100_000 * b) for b in range(batch)]
    src = _SlotSource(rng, num_slots)
    shared_slots = src.take(shared)
    priv_slots = [src.take(private) for _ in range(batch)]
    new_slots = src.take(batch)
    rows = []
    for b in range(batch):
        rows.append((np.concatenate([shared_tok, priv_tok[b]]),
                     np.concatenate([shared_slots, priv_slots[b], new_slots[b:b + 1]])))
    cached = np.concatenate([shared_slots] + priv_slots)
    dec = [(b, shared + private + 1) for b in range(batch)]
    return _finish("few_shot_decode", seed, rng, hq, hkv, d, num_slots, rows, cached, new_slots, [], dec,
                   draw_values)


def cached_prefix_extend(seed: int = 1003, hq: int = 32, hkv: int = 8, d: int = 128,
                         n_prefix: int = 8, per_prefix: int = 4, prefix: int = 2048, extend: int = 512,
                         num_slots: int = 1024 * 1024, draw_values: bool = True) -> Problem:
    """Requests extending cached prefixes (several requests per prefix).

    Full size: Llama-3-8B GQA (32 q / 8 kv heads, head_dim 128), 8 distinct
    2048-token prefixes with 4 requests each, 512 new causal tokens per request.
    """
    rng = np.random.default_rng(seed)
    pre_tok = [_tokens(rng, prefix, 1_000_000 + 100_000 * i) for i in range(n_prefix)]
    new_tok = [_tokens(rng, extend, 50_000_000 + 100_000 * b) for b in range(n_prefix * per_prefix)]
    src = _SlotSource(rng, num_slots)
    pre_slots = [src.take(prefix) for _ in range(n_prefix)]
    rows, new_slots, ext = [], [], []
    for b in range(n_prefix * per_prefix):
        p = b // per_prefix
        s_new = src.take(extend)
        new_slots.append(s_new)
        rows.append((np.concatenate([pre_tok[p], new_tok[b]]), np.concatenate([pre_slots[p], s_new])))
        ext.append((b, prefix, extend))
    return _finish("cached_prefix_extend", seed, rng, hq, hkv, d, num_slots, rows,
                   np.concatenate(pre_slots), np.concatenate(new_slots), ext, [], draw_values)


def tree_of_thought_decode(seed: int = 1004, hq: int = 32, hkv: int = 8, d: int = 128, depth: int = 4,
                           fanout: int = 4, edge: int = 256, num_slots: int = 1024 * 1024,
                           draw_values: bool = True) -> Problem:
    """Branching program: a full tree of thoughts, one decode token per leaf.

    Full size: GQA 32/8, head_dim 128, depth 4, fanout 4, 256 tokens per edge
    (340 edges, 256 leaves with 1024-token contexts), shared ancestors' KV
    stored once.
    """
    rng = np.random.default_rng(seed)
    # edges in BFS order; edge e at level l (1-based) is child (e's index) of its parent
    levels = []
    n_edges = 0
    for lvl in range(1, depth + 1):
        cnt = fanout ** lvl
        levels.append(list(range(n_edges, n_edges + cnt)))
        n_edges += cnt
    edge_tok = [_tokens(rng, edge, 1_000_000 + 1_000 * e) for e in range(n_edges)]
    n_leaves = fanout ** depth
    leaf_new_tok = [_tokens(rng, 1, 900_000_000 + b) for b in range(n_leaves)]
    src = _SlotSource(rng, num_slots)
    edge_slots = [src.take(edge) for _ in range(n_edges)]
    new_slots = src.take(n_leaves)
    rows, dec = [], []
    for leaf in range(n_leaves):
        path = []
        idx = leaf
        for lvl in range(depth - 1, -1, -1):
            path.append(levels[lvl][idx])
            idx //= fanout
        path.reverse()
        toks = np.concatenate([edge_tok[e] for e in path] + [leaf_new_tok[leaf]])
        sl = np.concatenate([edge_slots[e] for e in path] + [new_slots[leaf:leaf + 1]])
        rows.append((toks, sl))
        dec.append((leaf, depth * edge + 1))
    return _finish("tree_of_thought_decode", seed, rng, hq, hkv, d, num_slots, rows,
                   np.concatenate(edge_slots), new_slots, [], dec, draw_values)


@dataclasses.dataclass
class Scenario:
    """A batch whose slot lists come out of the radix cache, as data only.

    The pool starts empty with ``free_order`` as its free list.  Every
    ``prefill`` sequence is admitted (prefix match, fresh slots) and then
    committed (inserted into the cache), in order; then every ``batch``
    request is admitted, in order, and not committed: its row of
    ``req_to_token`` is the admitted slot list.  The first ``n_dec`` batch
    requests decode one token (all but their last token must be cached); the
    others extend their cached prefix by their remaining tokens.  Replaying
    the admissions is the radix cache's job (the library's tree, or the
    oracle's); this object only says what is admitted and in which order.
    """

    name: str
    seed: int
    hq: int
    hkv: int
    d: int
    num_slots: int
    free_order: np.ndarray            # int32 [num_slots]
    prefill: List[np.ndarray]         # int64 token sequences, admitted then committed
    batch: List[np.ndarray]           # int64 token sequences of the step's requests
    n_dec: int
    notes: dict = dataclasses.field(default_factory=dict)


def _cold_families(rng: np.random.Generator, volume: int, lo: int, exact: bool) -> List[np.ndarray]:
    """Cold conversations that take ``volume`` fresh slots (at least, or
    exactly with ``exact``): families of a system prompt of 256 .. 2048
    tokens shared by 1 .. 6 continuations of 512 .. 8192 tokens each.
    Returned in admission order (a family's sequences one after another);
    token ids come from ranges starting at ``lo``, disjoint per family."""
    seqs, used, fam = [], 0, 0
    while used < volume:
        base = lo + fam * 1_000_000
        sys_tok = _tokens(rng, int(rng.integers(256, 2049)), base)
        n_kids = int(rng.integers(1, 7))
        for k in range(n_kids):
            fresh_sys = len(sys_tok) if k == 0 else 0
            n = int(rng.integers(512, 8193))
            left = volume - used
            if exact and fresh_sys + n >= left:
                if left - fresh_sys < 1:         # the shared part alone would not fit
                    break
                n = left - fresh_sys
            seqs.append(np.concatenate([sys_tok, _tokens(rng, n, base + 100_000 + 10_000 * k)]))
            used += fresh_sys + n
            if used >= volume:
                break
        fam += 1
        if exact and volume - used > 0 and volume - used < 257:
            # too little room for another family's system prompt: lengthen
            # the last continuation instead (its tokens are fresh)
            extra = volume - used
            tail = seqs[-1]
            seqs[-1] = np.concatenate([tail, _tokens(rng, extra, lo + 900_000_000 + fam)])
            used += extra
    return seqs


def mixed_chat_scenario(seed: int = 1005, hq: int = 64, hkv: int = 8, d: int = 128, n_dec: int = 16,
                        system: int = 8192, history: int = 24576, n_ext: int = 16, ext_prefix: int = 4096,
                        ext_new: int = 1024, num_slots: int = 1024 * 1024, cold_before: int = 131072,
                        fill: bool = True) -> Scenario:
    """Long multi-turn chat under a full pool: the admissions of one mixed batch.

    Full size: Llama-70B attention shape (64 q / 8 kv heads, head_dim 128).
      * warm cache: an 8192-token system prompt followed by 16 chat
        histories of 24576 tokens each (16 sessions on one system prompt),
        and 16 distinct 4096-token documents;
      * cold cache: seeded conversations (``_cold_families``), ``cold_before``
        tokens of them cached before the warm part and the rest after it, so
        that the 1M-slot pool is exactly full (``fill``);
      * the batch: 16 decode requests (a session's history plus one new
        token, 32769 tokens) and 16 extend requests (a document plus 1024 new
        tokens); admitting their 16 + 16 x 1024 fresh slots into the full
        pool evicts least-recently-used cold conversations.
    The free list is a seeded random permutation of the pool's slots.
    """
    rng = np.random.default_rng(seed)
    sys_tok = _tokens(rng, system, 1_000_000)
    hist_tok = [_tokens(rng, history + 1, 10_000_000 + 100_000 * b) for b in range(n_dec)]
    epre_tok = [_tokens(rng, ext_prefix, 100_000_000 + 10_000 * b) for b in range(n_ext)]
    enew_tok = [_tokens(rng, ext_new, 200_000_000 + 10_000 * b) for b in range(n_ext)]
    free_order = rng.permutation(num_slots).astype(np.int32)
    warm = [np.concatenate([sys_tok, hist_tok[b][:history]]) for b in range(n_dec)] + list(epre_tok)
    warm_slots = system + n_dec * history + n_ext * ext_prefix
    batch_new = n_dec + n_ext * ext_new
    if warm_slots + batch_new > num_slots:
        raise ValueError("the batch does not fit the pool")
    cold_after = num_slots - warm_slots - cold_before if fill else 0
    if fill and (cold_before < batch_new or cold_after < 0):
        raise ValueError("cold_before must cover the batch's fresh slots and fit the pool")
    before = _cold_families(rng, cold_before, 3_000_000_000, exact=True) if cold_before else []
    after = _cold_families(rng, cold_after, 5_000_000_000, exact=True) if cold_after else []
    batch = [np.concatenate([sys_tok, hist_tok[b]]) for b in range(n_dec)] + \
            [np.concatenate([epre_tok[b], enew_tok[b]]) for b in range(n_ext)]
    notes = {"warm_tokens": warm_slots, "cold_before": cold_before, "cold_after": cold_after,
             "batch_fresh_slots": batch_new, "cold_sequences": len(before) + len(after)}
    return Scenario(name="mixed_chat", seed=seed, hq=hq, hkv=hkv, d=d, num_slots=num_slots,
                    free_order=free_order, prefill=before + warm + after, batch=batch, n_dec=n_dec,
                    notes=notes)


def problem_from_admission(scn: Scenario, rows: List[np.ndarray], prefix_lens: List[int],
                           draw_values: bool = True) -> Problem:
    """The Problem of a scenario's batch, given the slot list and cached
    prefix length each batch request was admitted with.  Values are drawn
    from a generator seeded by (seed, 1): cached K/V for the distinct cached
    slots in order of first appearance, new K/V for the fresh slots in batch
    order, then the extend queries and the decode queries."""
    if len(rows) != len(scn.batch) or len(prefix_lens) != len(scn.batch):
        raise ValueError("one admitted row and prefix length per batch request")
    seen, cached, new, ext, dec, out_rows = set(), [], [], [], [], []
    for i, (toks, row, k) in enumerate(zip(scn.batch, rows, prefix_lens)):
        row = np.asarray(row, np.int32)
        k = int(k)
        if len(row) != len(toks) or not 0 <= k <= len(toks):
            raise ValueError(f"batch request {i}: bad admitted row")
        for s in row[:k].tolist():
            if s not in seen:
                seen.add(s)
                cached.append(s)
        new.append(row[k:])
        out_rows.append((toks, row))
        if i < scn.n_dec:
            if len(toks) - k != 1:
                raise ValueError(f"decode request {i}: {len(toks) - k} uncached tokens, expected 1")
            dec.append((i, len(toks)))
        else:
            ext.append((i, k, len(toks) - k))
    rng = np.random.default_rng([scn.seed, 1])
    return _finish(scn.name, scn.seed, rng, scn.hq, scn.hkv, scn.d, scn.num_slots, out_rows,
                   np.array(cached, np.int32), np.concatenate(new).astype(np.int32), ext, dec, draw_values)


def ragged(seed: int, hq: int, hkv: int, d: int, n_groups: int, per_group: int, shared_max: int,
           private_max: int, extend_max: int, decode: bool, num_slots: int,
           allow_empty_prefix: bool = True) -> Problem:
    """Random ragged batch: groups of requests sharing a random-length prefix,
    random private parts, either one decode token or a random extend each."""
    rng = np.random.default_rng(seed)
    src_tok = 1_000_000
    g_len = rng.integers(0 if allow_empty_prefix else 1, shared_max + 1, size=n_groups)
    B = n_groups * per_group
    p_len = rng.integers(0, private_max + 1, size=B)
    e_len = rng.integers(1, extend_max + 1, size=B)
    if decode:
        e_len = np.ones(B, dtype=np.int64)
    shared_tok = [_tokens(rng, int(n), src_tok + 1_000_000 * i) for i, n in enumerate(g_len)]
    own_tok = [_tokens(rng, int(p_len[b] + e_len[b]), 500_000_000 + 100_000 * b) for b in range(B)]
    src = _SlotSource(rng, num_slots)
    shared_slots = [src.take(int(n)) for n in g_len]
    priv_slots = [src.take(int(n)) for n in p_len]
    new_slots = [src.take(int(n)) for n in e_len]
    rows, ext, dec = [], [], []
    for b in range(B):
        g = b // per_group
        rows.append((np.concatenate([shared_tok[g], own_tok[b]]),
                     np.concatenate([shared_slots[g], priv_slots[b], new_slots[b]])))
        P = int(g_len[g] + p_len[b])
        if decode:
            dec.append((b, P + 1))
        else:
            ext.append((b, P, int(e_len[b])))
    cached = np.concatenate(shared_slots + priv_slots) if B else _empty_i32()
    return _finish("ragged", seed, rng, hq, hkv, d, num_slots, rows, cached,
                   np.concatenate(new_slots), ext, dec)


def random_tree(seed: int, hq: int, hkv: int, d: int, decode: bool, max_requests: int = 40,
                max_depth: int = 4, max_children: int = 4, edge_max: int = 300, private_max: int = 200,
                extend_max: int = 120, slack: int = 500) -> Problem:
    """Random radix forest: nested shared prefixes of random lengths (empty
    edges included) with random fan-outs; a request at every leaf and, at
    random, at inner nodes too (a context that ends inside another's shared
    prefix plus a tail of its own).  Each request adds a random private part
    and one decode token or a random causal extend; the batch lists the
    requests in a shuffled order, so batch index and req_to_token row differ.
    The pool holds every token plus `slack` unused rows."""
    rng = np.random.default_rng(seed)
    paths = []      # per request: the edge ids of its shared prefix, root first
    edge_len = []

    def grow(path, depth):
        if len(paths) >= max_requests:
            return
        lo = 2 if depth == 0 else 0   # a forest of at least two trees
        n_kids = 0 if depth >= max_depth else int(rng.integers(lo, max(lo, max_children) + 1))
        if n_kids == 0 or (path and rng.random() < 0.2):
            paths.append(list(path))
        for _ in range(n_kids):
            if len(paths) >= max_requests:
                break
            e = len(edge_len)
            edge_len.append(int(rng.integers(0, edge_max + 1)))
            grow(path + [e], depth + 1)

    grow([], 0)
    B = len(paths)
    p_len = rng.integers(0, private_max + 1, size=B)
    e_len = np.ones(B, np.int64) if decode else rng.integers(1, extend_max + 1, size=B)
    total = sum(edge_len) + int(p_len.sum()) + int(e_len.sum())
    src = _SlotSource(rng, total + slack)
    edge_tok = [_tokens(rng, n, 1_000_000 + 10_000 * e) for e, n in enumerate(edge_len)]
    edge_slots = [src.take(n) for n in edge_len]
    priv_slots = [src.take(int(n)) for n in p_len]
    new_slots = [src.take(int(n)) for n in e_len]
    rows = []
    for b in range(B):
        own = _tokens(rng, int(p_len[b] + e_len[b]), 900_000_000 + 100_000 * b)
        rows.append((np.concatenate([edge_tok[e] for e in paths[b]] + [own]).astype(np.int64),
                     np.concatenate([edge_slots[e] for e in paths[b]] + [priv_slots[b], new_slots[b]])
                     .astype(np.int32)))
    order = rng.permutation(B)
    ext, dec = [], []
    for b in order:
        P = len(rows[b][1]) - int(e_len[b])
        if decode:
            dec.append((int(b), P + 1))
        else:
            ext.append((int(b), P, int(e_len[b])))
    cached = np.concatenate(edge_slots + priv_slots) if total > int(e_len.sum()) else _empty_i32()
    return _finish("random_tree", seed, rng, hq, hkv, d, total + slack, rows, cached,
                   np.concatenate(new_slots), ext, dec)


FULL_SIZE = {
    "tiny_extend": tiny_extend,
    "few_shot_decode": few_shot_decode,
    "cached_prefix_extend": cached_prefix_extend,
    "tree_of_thought_decode": tree_of_thought_decode,
}


def token_stream(rng_seed: int, n: int, lo: int = 0, hi: int = 1 << 40) -> np.ndarray:
    """Uniform int64 token ids (for radix-tree operation sequences)."""
    rng = np.random.default_rng(rng_seed)
    return rng.integers(lo, hi, size=n, dtype=np.int64)
