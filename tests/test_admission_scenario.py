"""The long multi-turn chat batch admitted into a full 1M-slot pool.

The batch's slot lists are not written by hand: a seeded scenario
(``inputs.mixed_chat_scenario``) caches cold conversations, then 16 chat
sessions on one 8192-token system prompt and 16 documents, then more cold
conversations until the pool is exactly full; admitting the batch (16 decode
requests of 32769 tokens, 16 extend requests of 4096 cached + 1024 new) must
then evict least-recently-used cold conversations ("SGLang: Efficient
Execution of Structured Language Model Programs", unite.ai, es, "SGLang:
Modelo de programación y metodología", nine-step walkthrough, steps 5, 8 and
9).  The library's tree (``rx_admit`` / ``rx_commit``) and the oracle trie
(``oracle.tree_ref.replay``) replay the same scenario; everything they hand
out must agree bit for bit: every admitted slot list and prefix length, the
tokens evicted per admission, the whole sequence of freed slots, which
cached sequences survive, and the tree's counts.
"""
import numpy as np
import pytest

from oracle import tree_ref
from prefix_shared_kv_radixattention_gb300 import admission, inputs


def _native_freed(nat, scn):
    """The freed-slot sequence on the library's side: the free list is empty
    when the batch arrives, so the fresh slots the batch was handed are the
    first freed slots, in order, and what is left on the free list is the
    rest."""
    fresh = [row[k:] for row, k in zip(nat.rows, nat.prefix_lens)]
    rest = nat.alloc.take(nat.alloc.free_count())
    return np.concatenate(fresh + [rest]).astype(np.int64)


def _check(scn):
    nat = admission.replay(scn)
    adm, out = tree_ref.replay(scn.free_order, scn.prefill, scn.batch)
    assert nat.prefill_evicted == 0
    for i, ((row, k, ev), r, kk, e) in enumerate(zip(out, nat.rows, nat.prefix_lens, nat.evicted)):
        assert row is not None, f"batch request {i} refused by the oracle"
        assert kk == k, f"batch request {i}: prefix length"
        assert e == ev, f"batch request {i}: tokens evicted"
        assert np.array_equal(np.asarray(row, np.int64), r.astype(np.int64)), f"batch request {i}: slot list"
    # every sequence that was cached: same surviving prefix on both sides
    for i, toks in enumerate(scn.prefill):
        assert nat.tree.prefix_len(toks) == adm.tree.prefix_len(toks), f"prefill sequence {i}"
    cached, nodes, evictable = nat.tree.stats()
    assert cached == adm.tree.cached_tokens
    assert nodes == adm.tree.num_nodes()
    assert evictable == adm.tree.evictable_tokens()
    freed = _native_freed(nat, scn)
    assert np.array_equal(freed, np.asarray(adm.freed, np.int64))
    return nat, adm


def test_mixed_chat_full_size_admission_matches_oracle():
    scn = inputs.mixed_chat_scenario()
    nat, adm = _check(scn)
    # the configuration's shape: the pool was full, the batch evicted cold
    # conversations only, and every request found its cached prefix
    assert sum(len(t) for t in scn.prefill) >= scn.num_slots - 16
    assert sum(nat.evicted) >= scn.notes["batch_fresh_slots"] > 0
    assert nat.prefix_lens[:16] == [32768] * 16
    assert nat.prefix_lens[16:] == [4096] * 16
    assert len(adm.freed) == sum(nat.evicted)
    prob = inputs.problem_from_admission(scn, nat.rows, nat.prefix_lens, draw_values=False)
    assert prob.dec_seq_len.tolist() == [32769] * 16
    assert prob.ext_prefix_len.tolist() == [4096] * 16 and prob.ext_extend_len.tolist() == [1024] * 16
    assert len(np.unique(prob.new_slots)) == len(prob.new_slots) == 16 + 16 * 1024
    assert not np.isin(prob.new_slots, prob.cached_slots).any()
    assert len(prob.cached_slots) == 8192 + 16 * 24576 + 16 * 4096
    # the 16 sessions share the system prompt's slots; the documents share nothing
    rtt = prob.req_to_token
    assert (rtt[:16, :8192] == rtt[0, :8192]).all()
    assert len(np.unique(rtt[:16, 8192:32768])) == 16 * 24576


@pytest.mark.parametrize("seed", [21, 22])
def test_small_scenarios_match_oracle(seed):
    """The same recipe at a small size, other seeds: more of the batch's
    admissions evict, some cascading into cold system prompts."""
    scn = inputs.mixed_chat_scenario(seed=seed, n_dec=5, system=300, history=900, n_ext=6, ext_prefix=200,
                                     ext_new=700, num_slots=40_000, cold_before=9_000)
    nat, adm = _check(scn)
    assert sum(nat.evicted) >= scn.notes["batch_fresh_slots"]
    assert sum(1 for e in nat.evicted if e) >= 2


def test_scenario_rejects_a_pool_too_small():
    with pytest.raises(ValueError):
        inputs.mixed_chat_scenario(num_slots=400_000)
