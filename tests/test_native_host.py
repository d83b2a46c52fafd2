"""Host side of librx on the CPU: ABI surface, radix tree, admission, plans.

* the library loads and exports every function ``include/rx.h`` declares;
* the C++ radix tree matches the oracle trie bit for bit (prefix lengths, slot
  lists, freed-slot sequences, tree shape) on the nine-step walkthrough, on
  seeded random operation sequences with locks and on hypothesis sequences;
* rx_admit / rx_commit match the same steps composed from the oracle;
* decode plans partition every request's context exactly once, group only
  requests that really share slots, and find the radix structure of the
  workload families;
* error codes for bad arguments and short capacities.
"""
import os
import re

import numpy as np
import pytest

from oracle.tree_ref import RadixTreeRef
from prefix_shared_kv_radixattention_gb300 import admission
from prefix_shared_kv_radixattention_gb300 import binding as rx
from prefix_shared_kv_radixattention_gb300 import inputs
from tests import _walkthrough
from tests.serving_sim import OracleAdmission
from tests.test_tree_oracle import _apply, _random_ops

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "rx.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(rx_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_function():
    names = declared_functions()
    assert len(names) >= 20
    lib = rx.library()
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert rx.version() == 3


def test_layer_outside_the_pool_is_rejected_before_any_launch():
    """Every pool entry point resolves the call's layer first: a layer
    outside the pool is RX_ERR_INVALID, returned before any device work (the
    pointers here are never dereferenced)."""
    import ctypes
    lib = rx.library()
    fake = 0x100000
    for L, layer in ((2, 2), (0, 1), (1, 1), (3, -1), (-1, 0)):
        pool = rx.KVPool(fake, fake, 64, 2, 64, L, layer)
        p8 = rx.KVPoolFp8(fake, fake, 64, 2, 64, 1.0, 1.0, L, layer)
        P = ctypes.c_void_p(fake)
        calls = [
            lambda: lib.rx_kv_store(ctypes.byref(pool), P, P, P, 4, None, None),
            lambda: lib.rx_kv_store_fp8(ctypes.byref(p8), P, P, P, 4, None, None),
            lambda: lib.rx_kv_store_rope(ctypes.byref(pool), P, P, P, P, 4, 10000.0, None, None),
            lambda: lib.rx_kv_store_rope_fp8(ctypes.byref(p8), P, P, P, P, 4, 10000.0, None, None),
            lambda: lib.rx_attn_extend(ctypes.byref(pool), P, P, None, 2, P, P, P, P, P, 64, 1, 8, None, 0,
                                       ctypes.c_float(0.125), None, None),
            lambda: lib.rx_attn_decode(ctypes.byref(pool), P, P, None, 2, P, P, P, 64, 1, 8, None, None, 0,
                                       ctypes.c_float(0.125), None, None),
            lambda: lib.rx_attn_extend_fp8(ctypes.byref(p8), P, P, None, 2, P, P, P, P, P, 64, 1, 8, P, 1 << 20,
                                           ctypes.c_float(0.125), None, None),
            lambda: lib.rx_attn_decode_static(ctypes.byref(pool), P, P, None, 2, P, P, P, 64, 1, 8, None,
                                              ctypes.c_float(0.125), None, None),
        ]
        for call in calls:
            assert call() == rx.RX_ERR_INVALID, (L, layer)
            assert "layer" in rx.last_error()


def test_fp8_decode_rejects_bad_shapes_and_scales():
    """rx_attn_decode_fp8 takes the head counts and plans rx_attn_decode
    takes (no plan included) and checks its shapes, scales and plan before
    any device work (the pointers here are never dereferenced)."""
    import ctypes
    lib = rx.library()
    fake = 0x100000
    P = ctypes.c_void_p(fake)
    plan = rx.DecodePlan(fake, fake, fake, 4, 1, 4)

    def call(hq, hkv, d, ks=1.0, vs=1.0, pl=plan, batch=2):
        pool = rx.KVPoolFp8(fake, fake, 64, hkv, d, ks, vs, 0, 0)
        return lib.rx_attn_decode_fp8(ctypes.byref(pool), P, P, None, hq, P, P, P, 64, batch, 8,
                                      ctypes.byref(pl) if pl is not None else None, P, 1 << 20,
                                      ctypes.c_float(0.1), None, None)

    assert call(32, 8, 96) == rx.RX_ERR_UNSUPPORTED             # head_dim
    assert call(24, 8, 128) == rx.RX_ERR_UNSUPPORTED            # G = 3 does not divide 64
    assert call(32, 8, 128, ks=0.0) == rx.RX_ERR_INVALID
    assert call(32, 8, 128, vs=-1.0) == rx.RX_ERR_INVALID
    bad_plan = rx.DecodePlan(fake, fake, fake, 4, 0, 4)         # max_parts 0
    assert call(32, 8, 128, pl=bad_plan) == rx.RX_ERR_INVALID
    # valid shapes, with or without a plan, MHA included: an empty batch is a no-op
    for hq, hkv, pl in ((32, 32, plan), (32, 32, None), (8, 4, None), (32, 8, plan)):
        assert call(hq, hkv, 128, pl=pl, batch=0) == rx.RX_OK, (hq, hkv, rx.last_error())


def test_fp8_extend_checks_before_any_launch():
    """rx_attn_extend_fp8 needs valid scales, head_dim 64 or 128 and 8-byte
    aligned pools; each is refused before any device work (the pointers
    here are never dereferenced)."""
    import ctypes
    lib = rx.library()
    fake = 0x100000
    P = ctypes.c_void_p(fake)

    def call(pool, ws=P, ws_bytes=1 << 20, hq=4):
        return lib.rx_attn_extend_fp8(ctypes.byref(pool), P, P, None, hq, P, P, P, P, P, 64, 2, 8, ws, ws_bytes,
                                      ctypes.c_float(0.125), None, None)

    good = rx.KVPoolFp8(fake, fake, 64, 4, 128, 1.0, 1.0, 0, 0)
    assert call(rx.KVPoolFp8(fake, fake, 64, 4, 128, 0.0, 1.0, 0, 0)) == rx.RX_ERR_INVALID
    assert call(rx.KVPoolFp8(fake, fake, 64, 4, 128, 1.0, -1.0, 0, 0)) == rx.RX_ERR_INVALID
    assert call(rx.KVPoolFp8(fake, fake, 64, 4, 96, 1.0, 1.0, 0, 0)) == rx.RX_ERR_UNSUPPORTED
    assert call(rx.KVPoolFp8(fake + 4, fake, 64, 4, 128, 1.0, 1.0, 0, 0)) == rx.RX_ERR_INVALID
    assert call(good, hq=6) == rx.RX_ERR_UNSUPPORTED            # 6 q heads over 4 kv heads
    # an empty batch is a no-op once the arguments check out
    assert lib.rx_attn_extend_fp8(ctypes.byref(good), P, P, None, 4, P, P, P, P, P, 64, 0, 8, P, 1 << 20,
                                  ctypes.c_float(0.125), None, None) == rx.RX_OK


# ---------------------------------------------------------------------------
# radix tree
# ---------------------------------------------------------------------------


class _NativeAdapter:
    def __init__(self):
        self.t = rx.RadixTree()

    def match_prefix(self, toks):
        return self.t.match_prefix(toks)

    def insert(self, toks, slots):
        return self.t.insert(toks, slots)

    def evict(self, n):
        return self.t.evict(n)

    def lock(self, toks, delta):
        try:
            return self.t.lock(toks, delta)
        except rx.RxError as e:
            if e.code == rx.RX_ERR_INVALID:
                raise ValueError(str(e))
            raise

    def nodes(self):
        return self.t.nodes()


def test_walkthrough_native_matches_fixture():
    spec = _walkthrough.load()
    for step, ri, obs, exp in _walkthrough.run(_NativeAdapter(), spec):
        if ri is None:
            assert obs["nodes"] == exp["nodes"], f"step {step}"
        else:
            assert obs["matched"] == exp["matched"], f"step {step}"
            assert obs["cached"] == len(exp["matched"]), f"step {step}"
            assert obs["evicted_nodes"] == exp["evicted_nodes"], f"step {step}"


def test_walkthrough_native_equals_oracle_slots():
    spec = _walkthrough.load()
    a = list(_walkthrough.run(RadixTreeRef(), spec))
    b = list(_walkthrough.run(_NativeAdapter(), spec))
    for (sa, ra, oa, _), (sb, rb, ob, _) in zip(a, b):
        assert (sa, ra) == (sb, rb)
        if ra is not None:
            assert oa["freed"] == ob["freed"]


@pytest.mark.parametrize("seed", range(60))
def test_native_tree_vs_oracle_random(seed):
    ref, nat = RadixTreeRef(), _NativeAdapter()
    for op in _random_ops(seed, n_ops=80):
        a, b = _apply(ref, op), _apply(nat, op)
        if op[0] == "match":
            assert a[0] == b[0] and list(a[1]) == list(b[1]), op
        else:
            assert a == b, op
        assert ref.nodes() == nat.nodes(), op
    c, n, e = nat.t.stats()
    assert c == ref.cached_tokens and n == ref.num_nodes() and e == ref.evictable_tokens()


def test_native_tree_vs_oracle_hypothesis():
    hyp = pytest.importorskip("hypothesis")
    st = hyp.strategies
    op = st.one_of(
        st.tuples(st.just("insert"), st.lists(st.integers(0, 3), min_size=1, max_size=10)),
        st.tuples(st.just("match"), st.lists(st.integers(0, 3), min_size=0, max_size=10)),
        st.tuples(st.just("evict"), st.integers(0, 15)),
        st.tuples(st.just("lock"), st.lists(st.integers(0, 3), min_size=0, max_size=10)),
    )

    @hyp.settings(max_examples=200, deadline=None)
    @hyp.given(st.lists(op, max_size=50))
    def check(ops):
        ref, nat = RadixTreeRef(), _NativeAdapter()
        nxt, held = 0, []
        for o in ops:
            if o[0] == "insert":
                o = ("insert", o[1], list(range(nxt, nxt + len(o[1]))))
                nxt += len(o[1])
            elif o[0] == "lock":
                if held and len(o[1]) % 2 == 1:
                    o = ("unlock", held.pop(), -1)
                else:
                    k = ref.lock(o[1], 1)
                    ref.lock(o[1][:k], -1)   # probe the length, undo
                    held.append(o[1][:k])
                    o = ("lock", o[1][:k], 1)
            a, b = _apply(ref, o), _apply(nat, o)
            if o[0] == "match":
                assert a[0] == b[0] and list(a[1]) == list(b[1])
            else:
                assert a == b
            assert ref.nodes() == nat.nodes()

    check()


def test_evict_capacity_and_not_enough():
    t = rx.RadixTree()
    t.insert([1, 2, 3], [10, 11, 12])
    t.insert([4], [20])
    with pytest.raises(rx.RxError) as e:
        t.evict(4, cap=2)
    assert e.value.code == rx.RX_ERR_CAPACITY
    assert t.evict(100) == [10, 11, 12, 20]      # partial: NOT_ENOUGH reported as a list
    assert t.stats() == (0, 0, 0)


def test_locked_nodes_survive_eviction():
    t = rx.RadixTree()
    t.insert([1, 2, 3], [10, 11, 12])
    t.insert([5, 6], [20, 21])
    assert t.lock([1, 2, 3, 4], 1) == 3
    assert t.evict(10) == [20, 21]
    assert t.stats() == (3, 1, 0)
    t.insert([7, 8], [30, 31])
    with pytest.raises(rx.RxError) as e:
        t.lock([7], -1)                       # never locked
    assert e.value.code == rx.RX_ERR_INVALID
    assert t.lock([1, 2], -1) == 2            # tokens 1, 2 unlocked; 3 still locked
    assert t.evict(10) == [30, 31]            # the node [1 2 3] still holds a locked token
    assert t.lock([1, 2, 3], 1) == 3 and t.lock([1, 2, 3], -1) == 3
    assert t.lock([3], -1) == 0               # not a cached prefix: nothing to unlock
    assert t.lock([1, 2, 3][:0], -1) == 0


def test_match_capacity_error_code():
    t = rx.RadixTree()
    t.insert([1, 2, 3], [10, 11, 12])
    import ctypes
    toks = np.array([1, 2, 3], np.int64)
    out = np.zeros(1, np.int32)
    k = ctypes.c_int64()
    rc = rx.library().rx_match_prefix(t._h, toks.ctypes.data_as(ctypes.c_void_p), 3,
                                      out.ctypes.data_as(ctypes.c_void_p), 1, ctypes.byref(k))
    assert rc == rx.RX_ERR_CAPACITY and k.value == 3
    assert "capacity" in rx.last_error()


def test_extend_workspace_size():
    """Offsets [batch+1] int64, shared-tile sources and counts [batch] int32
    each, then K and V areas of (total + 127 batch) rows of num_kv_heads x
    head_dim bf16 (every context rounded up to whole 128-row tiles, none
    shared), each part rounded up to 256 bytes."""
    def up(x):
        return (x + 255) // 256 * 256
    for total, batch, hkv, d in ((1000, 3, 8, 128), (0, 1, 4, 64), (81920, 32, 8, 128), (5, 7, 1, 64)):
        rows = max(total + 127 * batch, 128)
        want = up((batch + 1) * 8) + 2 * up(batch * 4) + 2 * up(rows * hkv * d * 2)
        assert rx.rx_attn_extend_workspace(total, batch, hkv, d) == want


def test_invalid_arguments():
    lib = rx.library()
    import ctypes
    assert lib.rx_tree_create(None) == rx.RX_ERR_INVALID
    assert lib.rx_insert(None, None, None, 0, None) == rx.RX_ERR_INVALID
    assert lib.rx_kv_store(None, None, None, None, 0, None, None) == rx.RX_ERR_INVALID
    assert lib.rx_attn_decode(None, None, None, None, 0, None, None, None, 0, 0, 0, None, None, 0,
                              ctypes.c_float(1.0), None, None) == rx.RX_ERR_INVALID
    assert lib.rx_attn_extend(None, None, None, None, 0, None, None, None, None, None, 0, 0, 0,
                              None, 0, ctypes.c_float(1.0), None, None) == rx.RX_ERR_INVALID
    assert lib.rx_attn_extend_workspace(-1, 1, 8, 128) == 0
    assert lib.rx_attn_extend_workspace(100, 0, 8, 128) == 0
    assert lib.rx_attn_extend_workspace(100, 1, 8, 96) == 0
    base = ctypes.c_double(10000.0)
    assert lib.rx_rope(None, None, 0, 4, 96, base, None) == rx.RX_ERR_UNSUPPORTED
    assert lib.rx_rope(None, None, 0, 4, 64, ctypes.c_double(1.0), None) == rx.RX_ERR_UNSUPPORTED
    assert lib.rx_rope(None, None, 5, 4, 64, base, None) == rx.RX_ERR_INVALID
    assert lib.rx_rope(None, None, 0, 4, 64, base, None) == rx.RX_OK  # nothing to do
    assert lib.rx_kv_store_rope(None, None, None, None, None, 0, base, None, None) == rx.RX_ERR_INVALID
    with pytest.raises(rx.RxError):
        rx.SlotAllocator([0, 5], 3)
    a = rx.SlotAllocator([0, 1, 2], 3)
    with pytest.raises(rx.RxError) as e:
        a.take(4)
    assert e.value.code == rx.RX_ERR_NOT_ENOUGH and a.free_count() == 3


# ---------------------------------------------------------------------------
# admission
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("seed", range(12))
def test_admit_commit_vs_oracle(seed):
    rng = np.random.default_rng(seed)
    S = 60
    free = rng.permutation(S).astype(np.int32)
    nat_t, nat_a = rx.RadixTree(), rx.SlotAllocator(free, S)
    ref = OracleAdmission(free.tolist())
    pending = []
    for step in range(40):
        if pending and rng.random() < 0.5:
            toks, row, k = pending.pop(rng.integers(len(pending)))
            rx.rx_commit(nat_t, nat_a, toks, row, k)
            ref.commit(toks, list(row), k)
        else:
            base = [int(x) for x in rng.integers(0, 3, size=rng.integers(1, 4))]
            toks = base + [int(x) for x in rng.integers(0, 6, size=rng.integers(1, 12))]
            exp_row, exp_k, exp_ev = ref.admit(toks)
            try:
                row, k, ev = rx.rx_admit(nat_t, nat_a, toks)
            except rx.RxError as e:
                assert e.code == rx.RX_ERR_NOT_ENOUGH and exp_row is None
                continue
            assert exp_row is not None and row.tolist() == exp_row and k == exp_k and ev == exp_ev
            pending.append((toks, row, k))
        assert nat_t.nodes() == ref.t.nodes()
        assert nat_a.free_count() == len(ref.free)


# ---------------------------------------------------------------------------
# decode plans
# ---------------------------------------------------------------------------


def _plan(prob, kv_chunk=0, min_shared=16):
    buf, info = rx.rx_decode_plan_build(prob.req_to_token, prob.dec_req_idx, prob.dec_seq_len,
                                        prob.hq, prob.hkv, kv_chunk, min_shared)
    B = len(prob.dec_req_idx)
    order = buf[:B]
    nparts = buf[B:2 * B]
    items = buf[2 * B:].reshape(-1, 8)
    return order, nparts, items, info


def _plan_wide(prob):
    """Head counts for which the plan makes all-heads single-request items:
    one q head per kv head, or 8 kv heads with G = 2, 4, 8 or 16."""
    G = prob.hq // prob.hkv
    return G == 1 or (prob.hkv == 8 and G in (2, 4, 8, 16))


def check_plan(prob, order, nparts, items, info, auto=False):
    B = len(prob.dec_req_idx)
    G = prob.hq // prob.hkv
    assert sorted(order.tolist()) == list(range(B))
    cover = [np.zeros(int(L), np.int32) for L in prob.dec_seq_len]
    parts = [[] for _ in range(B)]
    open_end = [0] * B
    reads = 0
    for r0, nr, p0, p1, part, fin, row0, b0 in items.tolist():
        if p1 == rx.RX_PLAN_OPEN_END:
            # a request's own last piece ends at its length when the plan is used
            assert nr == 1
            p1 = int(prob.dec_seq_len[b0])
            open_end[b0] += 1
        assert 1 <= nr and nr * G <= 64 and p0 < p1
        assert b0 == order[r0] and row0 == prob.dec_req_idx[b0]
        # single-request items of an automatic plan for the all-heads kernel
        # follow their own length target (at most 4096 positions)
        wide_auto = nr == 1 and _plan_wide(prob) and auto
        assert p1 - p0 <= (4096 if wide_auto else info.kv_chunk)
        reqs = [int(order[r]) for r in range(r0, r0 + nr)]
        rows = [prob.req_to_token[prob.dec_req_idx[b], p0:p1] for b in reqs]
        for rr in rows[1:]:
            assert np.array_equal(rr, rows[0]), "grouped requests must share slots"
        for b in reqs:
            cover[b][p0:p1] += 1
            parts[b].append(part)
            assert bool(fin) == (nparts[b] == 1)
        reads += p1 - p0
    assert reads * 1 >= info.tokens_read
    assert open_end == [1] * B, "every request ends in one open-ended piece of its own"
    for b in range(B):
        assert np.all(cover[b] == 1), f"request {b} context not covered exactly once"
        assert sorted(parts[b]) == list(range(int(nparts[b])))
    assert info.max_parts == int(nparts.max())
    # per-head items first, then the n_wide all-heads ones: for the head
    # counts with an all-heads kernel every single-request item, and with
    # G > 1 also groups of up to 16 / G requests (16 query rows per kv head);
    # otherwise none.  Per-head items: those of several requests before
    # single-request ones, each of those longest first; all-heads items
    # (handed out first come first served): longest first.
    n_wide = int(info.n_wide)
    items = items.copy()
    is_open = items[:, 3] == rx.RX_PLAN_OPEN_END
    items[is_open, 3] = prob.dec_seq_len[items[is_open, 7]]
    head, tail = items[:len(items) - n_wide], items[len(items) - n_wide:]
    if not _plan_wide(prob):
        assert n_wide == 0
    else:
        assert not np.any(head[:, 1] == 1)
        assert np.all(tail[:, 1] * G <= 16) if G > 1 else np.all(tail[:, 1] == 1)
    single = head[:, 1] == 1
    k = int(single.sum())
    assert np.all(single[len(head) - k:]) and not np.any(single[:len(head) - k])
    for grp in (head[~single], head[single], tail):
        lens = grp[:, 3] - grp[:, 2]
        assert np.all(lens[:-1] >= lens[1:])


@pytest.mark.parametrize("seed", range(15))
def test_plan_partitions_ragged(seed):
    prob = inputs.ragged(100 + seed, hq=8, hkv=2, d=64, n_groups=3, per_group=int(2 + seed % 4),
                         shared_max=300, private_max=200, extend_max=1, decode=True, num_slots=5000)
    for kv_chunk, min_shared in ((64, 1), (128, 16), (0, 16), (4096, 64)):
        order, nparts, items, info = _plan(prob, kv_chunk, min_shared)
        check_plan(prob, order, nparts, items, info, auto=kv_chunk == 0)


def test_plan_structure_few_shot():
    prob = inputs.few_shot_decode(draw_values=False)
    order, nparts, items, info = _plan(prob)
    check_plan(prob, order, nparts, items, info, auto=True)
    assert info.n_segments == 1 and info.shared_tokens == 1024
    assert info.tokens_read == 1024 + 64 * 257 == prob.decode_unique_tokens()


def test_plan_structure_tree_of_thought():
    prob = inputs.tree_of_thought_decode(draw_values=False)
    order, nparts, items, info = _plan(prob)
    check_plan(prob, order, nparts, items, info, auto=True)
    assert info.n_segments == 4 + 16 + 64
    assert info.shared_tokens == 84 * 256
    assert info.tokens_read == prob.decode_unique_tokens() == 340 * 256 + 256
    # G = 4: groups of 4 requests.  Every segment goes to the all-heads
    # kernel: the 64 level-3 ones (4 requests: one group), the 16 level-2 ones
    # (16 requests: four groups) and the 4 level-1 ones (64 requests: sixteen
    # groups, the most one chunk is cut into); no per-head items remain.
    groups = items[items[:, 1] > 1]
    assert len(groups) == 64 + 16 * 4 + 4 * 16 and np.all(groups[:, 1] == 4)
    assert int(info.n_wide) == len(items)


def test_plan_structure_mixed_chat():
    prob = admission.mixed_chat(draw_values=False)
    order, nparts, items, info = _plan(prob)
    check_plan(prob, order, nparts, items, info, auto=True)
    assert info.n_segments == 1 and info.shared_tokens == 8192
    assert info.tokens_read == prob.decode_unique_tokens()


def test_plan_min_shared_folds_short_segments():
    prob = inputs.tree_of_thought_decode(depth=3, fanout=3, edge=8, draw_values=False)
    # edges of 8 tokens: level 1 spans [0, 8), level 2 [8, 16)
    order, nparts, items, info = _plan(prob, 64, min_shared=8)
    check_plan(prob, order, nparts, items, info)
    assert info.n_segments == 3 + 9 and info.shared_tokens == 12 * 8
    # level 1 is too short on its own and is folded into the level-2 segments
    order, nparts, items, info = _plan(prob, 64, min_shared=9)
    check_plan(prob, order, nparts, items, info)
    assert info.n_segments == 9 and info.shared_tokens == 9 * 16
    order, nparts, items, info = _plan(prob, 64, min_shared=17)
    check_plan(prob, order, nparts, items, info)
    assert info.n_segments == 0 and info.tokens_read == 27 * 25


def test_plan_identical_requests():
    prob = inputs.few_shot_decode(batch=3, shared=100, private=0, hq=4, hkv=4, d=64, num_slots=400,
                                  draw_values=False)
    rtt = prob.req_to_token.copy()
    rtt[1] = rtt[0]
    prob.req_to_token = rtt
    order, nparts, items, info = _plan(prob, 64, 1)
    check_plan(prob, order, nparts, items, info)


def test_plan_invalid():
    prob = inputs.few_shot_decode(batch=2, shared=10, private=5, hq=4, hkv=4, d=64, num_slots=100,
                                  draw_values=False)
    with pytest.raises(rx.RxError) as e:
        rx.rx_decode_plan_build(prob.req_to_token, prob.dec_req_idx, prob.dec_seq_len, 4, 4, 100, 1)
    assert e.value.code == rx.RX_ERR_INVALID
    with pytest.raises(rx.RxError) as e:
        rx.rx_decode_plan_build(prob.req_to_token, prob.dec_req_idx, prob.dec_seq_len, 128, 1, 64, 1)
    assert e.value.code == rx.RX_ERR_UNSUPPORTED


@pytest.mark.parametrize("hq,batch,all_heads", [(32, 64, True), (32, 68, False), (64, 32, True), (64, 34, False)])
def test_plan_group_limit(hq, batch, all_heads):
    """With 8 kv heads, a shared segment whose requests make at most 16
    groups of 16 / G requests goes to the all-heads kernel, one item per
    group; one more group sends it to the per-head kernel, in items of
    64 / G requests."""
    G = hq // 8
    prob = inputs.few_shot_decode(hq=hq, hkv=8, d=128, batch=batch, shared=128, private=8, num_slots=8192,
                                  draw_values=False)
    order, nparts, items, info = _plan(prob, 128, 16)
    check_plan(prob, order, nparts, items, info)
    shared = items[items[:, 2] == 0]                 # the items of the shared prefix (positions 0 ..)
    if all_heads:
        assert np.all(shared[:, 1] <= 16 // G) and len(shared) == -(-batch // (16 // G))
        assert info.n_items == info.n_wide
    else:
        assert np.all(shared[:, 1] <= 64 // G) and len(shared) == -(-batch // (64 // G))
        assert info.n_items - info.n_wide == len(shared)
