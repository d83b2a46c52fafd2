"""Pins for the reference radix tree (oracle/tree_ref.py).

* the nine-step walkthrough of "SGLang: Efficient Execution of Structured
  Language Model Programs" (unite.ai, es), section "SGLang: Modelo de
  programación y metodología", as a scripted fixture;
* a brute-force model over a prefix-closed set of token tuples with explicit
  node boundaries: longest cached prefix by exhaustive lookup, eviction by
  exhaustive search for the least recently used leaf node.
"""
import random
from collections import Counter

import pytest

from oracle.tree_ref import CapacityError, RadixTreeRef
from tests import _walkthrough


def test_walkthrough_oracle():
    tree = RadixTreeRef()
    spec = _walkthrough.load()
    toks = _walkthrough.segment_tokens(spec)
    freed_log = []
    for step, ri, obs, exp in _walkthrough.run(tree, spec):
        if ri is None:
            assert obs["nodes"] == exp["nodes"], f"step {step}: tree shape"
            continue
        assert obs["matched"] == exp["matched"], f"step {step}: matched prefix"
        assert obs["cached"] == len(exp["matched"]), f"step {step}: insert's cached length"
        assert obs["evicted_nodes"] == exp["evicted_nodes"], f"step {step}: evicted nodes"
        freed_log.append((step, obs["freed"]))
    # step 1: the tree starts empty; the final tree holds every token once
    assert RadixTreeRef().num_nodes() == 0


def test_walkthrough_eviction_order_and_slots():
    """Evicted slots come node by node, oldest node first, each in token order."""
    tree = RadixTreeRef()
    spec = _walkthrough.load()
    slot_of_token = {}
    orig_insert = tree.insert

    def insert(tokens, slots):
        k = orig_insert(tokens, slots)
        for t, s in zip(tokens[k:], slots[k:]):
            slot_of_token[t] = s
        return k

    tree.insert = insert
    for step, ri, obs, exp in _walkthrough.run(tree, spec):
        if ri is None or not exp["evicted_in_order"]:
            continue
        want = [slot_of_token[t] for node in exp["evicted_in_order"] for t in node]
        assert obs["freed"] == want, f"step {step}"


# ---------------------------------------------------------------------------
# brute-force model
# ---------------------------------------------------------------------------


class BruteTree:
    """Cached data as a prefix-closed set of token tuples.  ``start`` holds the
    tuples whose last token opens a radix node; ``last`` maps a node's first
    tuple to its last-access value."""

    def __init__(self):
        self.slot = {}
        self.locked = Counter()
        self.start = set()
        self.last = {}
        self.clock = 0

    def _node_start(self, p):
        while p not in self.start:
            p = p[:-1]
        return p

    def _matched(self, toks):
        k = 0
        while k < len(toks) and tuple(toks[:k + 1]) in self.slot:
            k += 1
        return k

    def _touch(self, toks, k):
        for i in range(k):
            p = tuple(toks[:i + 1])
            if p in self.start:
                self.last[p] = self.clock

    def match_prefix(self, toks):
        self.clock += 1
        k = self._matched(toks)
        self._touch(toks, k)
        return k, [self.slot[tuple(toks[:i + 1])] for i in range(k)]

    def _children(self, p):
        return [q for q in self.slot if len(q) == len(p) + 1 and q[:-1] == p]

    def insert(self, toks, slots):
        self.clock += 1
        k = self._matched(toks)
        if k < len(toks) and k > 0:
            end = tuple(toks[:k])
            kids = self._children(end)
            if len(kids) == 1 and kids[0] not in self.start:
                self.start.add(kids[0])
                self.last[kids[0]] = self.last[self._node_start(end)]
        self._touch(toks, k)
        for i in range(k, len(toks)):
            p = tuple(toks[:i + 1])
            self.slot[p] = slots[i]
        if k < len(toks):
            p = tuple(toks[:k + 1])
            self.start.add(p)
            self.last[p] = self.clock
        return k

    def lock(self, toks, delta):
        if delta > 0:
            self.clock += 1
        k = self._matched(toks)
        ps = [tuple(toks[:i + 1]) for i in range(k)]
        if delta < 0 and any(self.locked[p] == 0 for p in ps):
            raise ValueError("unlock without lock")
        if delta > 0:
            self._touch(toks, k)
        for p in ps:
            self.locked[p] += delta
        return k

    def evict(self, n):
        freed = []
        while len(freed) < n and self.slot:
            has_kid = Counter(p[:-1] for p in self.slot)
            leaves = [p for p in self.slot if has_kid[p] == 0]
            cands = {}
            for leaf in leaves:
                s = self._node_start(leaf)
                if all(self.locked[leaf[:L]] == 0 for L in range(len(s), len(leaf) + 1)):
                    cands[s] = leaf
            if not cands:
                break
            s = min(cands, key=lambda q: self.last[q])
            leaf = cands[s]
            for L in range(len(s), len(leaf) + 1):
                freed.append(self.slot.pop(leaf[:L]))
                self.start.discard(leaf[:L])
            self.last.pop(s)
        return freed

    def nodes(self):
        out = []
        for s in self.start:
            own = [s[-1]]
            p = s
            while True:
                kids = self._children(p)
                if len(kids) != 1 or kids[0] in self.start:
                    break
                p = kids[0]
                own.append(p[-1])
            out.append((s[:-1], tuple(own)))
        return sorted(out)


def _random_ops(seed, n_ops=60, alphabet=4, max_len=9):
    rng = random.Random(seed)
    next_slot = [0]
    ops = []
    held = []
    for _ in range(n_ops):
        kind = rng.choices(["insert", "match", "evict", "lock", "unlock"], weights=[5, 3, 2, 1, 1])[0]
        toks = [rng.randrange(alphabet) for _ in range(rng.randrange(1, max_len))]
        if kind == "lock":
            held.append(toks)
            ops.append(("lock", toks, 1))
        elif kind == "unlock":
            if held:
                ops.append(("unlock", held.pop(rng.randrange(len(held))), -1))
        elif kind == "evict":
            ops.append(("evict", rng.randrange(1, 12)))
        elif kind == "match":
            ops.append(("match", toks))
        else:
            slots = list(range(next_slot[0], next_slot[0] + len(toks)))
            next_slot[0] += len(toks)
            ops.append(("insert", toks, slots))
    return ops


def _apply(tree, op):
    if op[0] in ("lock", "unlock"):
        try:
            return tree.lock(op[1], op[2])
        except ValueError:
            return "unlock-error"
    if op[0] == "insert":
        return tree.insert(op[1], op[2])
    if op[0] == "match":
        return tree.match_prefix(op[1])
    return tree.evict(op[1])


@pytest.mark.parametrize("seed", range(40))
def test_oracle_vs_brute_force(seed):
    ref, brute = RadixTreeRef(), BruteTree()
    for op in _random_ops(seed):
        a, b = _apply(ref, op), _apply(brute, op)
        if op[0] == "match":
            assert a[0] == b[0] and list(a[1]) == list(b[1]), op
        else:
            assert a == b, op
        assert ref.nodes() == brute.nodes(), op


def test_oracle_vs_brute_force_hypothesis():
    hyp = pytest.importorskip("hypothesis")
    st = hyp.strategies

    op = st.one_of(
        st.tuples(st.just("insert"), st.lists(st.integers(0, 3), min_size=1, max_size=8)),
        st.tuples(st.just("match"), st.lists(st.integers(0, 3), min_size=0, max_size=8)),
        st.tuples(st.just("evict"), st.integers(0, 12)),
    )

    @hyp.settings(max_examples=150, deadline=None)
    @hyp.given(st.lists(op, max_size=40))
    def check(ops):
        ref, brute = RadixTreeRef(), BruteTree()
        nxt = 0
        for o in ops:
            if o[0] == "insert":
                o = ("insert", o[1], list(range(nxt, nxt + len(o[1]))))
                nxt += len(o[1])
            a, b = _apply(ref, o), _apply(brute, o)
            if o[0] == "match":
                assert a[0] == b[0] and list(a[1]) == list(b[1])
            else:
                assert a == b
            assert ref.nodes() == brute.nodes()

    check()


def test_match_is_longest_cached_prefix():
    t = RadixTreeRef()
    t.insert([1, 2, 3, 4], [10, 11, 12, 13])
    t.insert([1, 2, 5], [20, 21, 22])
    assert t.match_prefix([1, 2, 3, 9]) == (3, [10, 11, 12])
    assert t.match_prefix([1, 2, 5, 5]) == (3, [10, 11, 22])
    assert t.match_prefix([7]) == (0, [])
    assert t.match_prefix([]) == (0, [])


def test_insert_keeps_tree_slots_for_cached_part():
    t = RadixTreeRef()
    assert t.insert([1, 2, 3], [10, 11, 12]) == 0
    assert t.insert([1, 2, 3, 4], [90, 91, 92, 13]) == 3
    assert t.match_prefix([1, 2, 3, 4]) == (4, [10, 11, 12, 13])
    assert t.cached_tokens == 4


def test_evict_lru_leaf_first_and_cascade():
    t = RadixTreeRef()
    t.insert([1, 2, 3], [10, 11, 12])      # node A
    t.insert([5, 6], [20, 21])             # node B
    t.match_prefix([1, 2])                 # A used more recently than B
    assert t.evict(1) == [20, 21]          # B is the oldest leaf
    assert t.evict(100) == [10, 11, 12]    # then A; nothing left
    assert t.cached_tokens == 0 and t.evict(5) == []


def test_evict_capacity():
    t = RadixTreeRef()
    t.insert([1, 2, 3], [10, 11, 12])
    t.insert([4], [20])
    with pytest.raises(CapacityError) as e:
        t.evict(4, cap=2)
    assert e.value.args[0] == []
    assert t.evict(1, cap=3) == [10, 11, 12]
    assert t.evict(1) == [20]
