"""Host failure paths of the radix cache, driven without a failing allocator.

``rx_test_fail_alloc(n)`` makes the n-th next tree-node allocation throw as a
failing host allocator would.  Each entry point that needs a node must then
return RX_ERR_NOMEM with the tree, its locks and the free list exactly as
they were, and carry on normally once allocation works again (checked against
the oracle trie driven with the same successful operations).
"""
import numpy as np
import pytest

from oracle.tree_ref import Admission, RadixTreeRef
from prefix_shared_kv_radixattention_gb300 import binding as rx


@pytest.fixture(autouse=True)
def _hook_off():
    rx.rx_test_fail_alloc(0)
    yield
    rx.rx_test_fail_alloc(0)


def _nomem(fn, *a):
    with pytest.raises(rx.RxError) as e:
        fn(*a)
    assert e.value.code == rx.RX_ERR_NOMEM, e.value


def test_tree_create_fails_cleanly():
    rx.rx_test_fail_alloc(1)
    _nomem(rx.RadixTree)
    t = rx.RadixTree()                     # the hook fired once; the next works
    assert t.stats() == (0, 0, 0)


@pytest.mark.parametrize("fail_at", [1, 2])
def test_insert_that_splits_fails_without_a_trace(fail_at):
    """An insert that splits a node and adds a leaf needs two nodes; failing
    either allocation leaves the tree unchanged (structure, clock values,
    locks), and the same insert then succeeds as in the oracle."""
    nat, ref = rx.RadixTree(), RadixTreeRef()
    ops = [([1, 2, 3, 4, 5, 6], [10, 11, 12, 13, 14, 15]), ([1, 2, 3, 9, 9], [10, 11, 12, 20, 21])]
    for toks, slots in ops:
        nat.insert(toks, slots)
        ref.insert(toks, slots)
    nat.lock([1, 2, 3, 4], 1)
    ref.lock([1, 2, 3, 4], 1)
    before = (nat.dump(), nat.stats())
    rx.rx_test_fail_alloc(fail_at)
    _nomem(nat.insert, [1, 2, 3, 4, 7, 7], [10, 11, 12, 13, 30, 31])   # splits [4 5 6] after 4
    assert (nat.dump(), nat.stats()) == before
    rx.rx_test_fail_alloc(0)
    assert nat.insert([1, 2, 3, 4, 7, 7], [10, 11, 12, 13, 30, 31]) == 4
    ref.insert([1, 2, 3, 4, 7, 7], [10, 11, 12, 13, 30, 31])
    assert nat.nodes() == ref.nodes()
    assert nat.evict(100) == ref.evict(100)    # the locked path stays, the rest goes in LRU order


def test_commit_that_fails_keeps_the_request_admitted():
    """rx_commit needs a node for the request's new tokens.  When that
    allocation fails the request stays admitted: its prefix stays locked and
    its fresh slots stay its own; committing again works, and the whole
    sequence then matches the oracle's admission."""
    S = 64
    free = np.random.default_rng(5).permutation(S).astype(np.int32)
    tree, alloc = rx.RadixTree(), rx.SlotAllocator(free, S)
    ref = Admission(free.tolist())
    a = list(range(100, 130))
    b = a[:20] + list(range(200, 215))
    for toks in (a, b):
        row, k, ev = rx.rx_admit(tree, alloc, toks)
        rrow, rk, rev = ref.admit(toks)
        assert row.tolist() == rrow and k == rk and ev == rev
        if toks is b:
            before = (tree.dump(), tree.stats(), alloc.free_count())
            rx.rx_test_fail_alloc(1)
            _nomem(rx.rx_commit, tree, alloc, toks, row, k)
            assert (tree.dump(), tree.stats(), alloc.free_count()) == before
            rx.rx_test_fail_alloc(0)
        rx.rx_commit(tree, alloc, toks, row, k)
        ref.commit(toks, rrow, rk)
    c = list(range(300, 340))                                 # needs eviction of the unlocked nodes
    row, k, ev = rx.rx_admit(tree, alloc, c)
    rrow, rk, rev = ref.admit(c)
    assert row.tolist() == rrow and k == rk and ev == rev > 0
    assert tree.nodes() == ref.tree.nodes()
    assert alloc.free_count() == len(ref.free)


def test_hook_rejects_negative():
    with pytest.raises(rx.RxError) as e:
        rx.rx_test_fail_alloc(-1)
    assert e.value.code == rx.RX_ERR_INVALID
