"""GPU parity: the sm_103a kernels, called through the C ABI, against the fp64
oracle on the same seeded inputs.

Sizes span several 64-key tiles, several work items per request and ragged
tails; the tolerance is stated in tests/_gpu.py.
"""
import numpy as np
import pytest

import oracle
from prefix_shared_kv_radixattention_gb300 import inputs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _gpu():
    from tests import _gpu
    return _gpu


# ---------------------------------------------------------------------------
# KV store
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("hkv,d", [(4, 64), (8, 128), (32, 128)])
def test_kv_store_bit_exact(hkv, d):
    g = _gpu()
    prob = inputs.ragged(5, hq=hkv, hkv=hkv, d=d, n_groups=3, per_group=3, shared_max=40,
                         private_max=30, extend_max=50, decode=False, num_slots=2000)
    dev = g.Dev(prob)
    dev.kv_store()
    torch.cuda.synchronize()
    kp, vp, _ = dev.oracle_pools()
    assert np.array_equal(g.to_host_u16(dev.k_pool), kp)
    assert np.array_equal(g.to_host_u16(dev.v_pool), vp)
    assert dev.status_word() == 0


def test_kv_store_bad_slot_flagged_not_written():
    g = _gpu()
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    prob = inputs.tiny_extend()
    dev = g.Dev(prob)
    before_k = g.to_host_u16(dev.k_pool)
    slots = prob.new_slots.copy()
    slots[3] = prob.num_slots + 7
    slots[5] = -2
    rx.rx_kv_store(dev.k_pool, dev.v_pool, g.to_dev(prob.new_k), g.to_dev(prob.new_v), g.i32(slots),
                   dev.status)
    torch.cuda.synchronize()
    assert dev.status_word() & rx.RX_DEV_BAD_SLOT
    after_k = g.to_host_u16(dev.k_pool)
    ok = np.ones(len(slots), bool)
    ok[[3, 5]] = False
    assert np.array_equal(after_k[slots[ok]], prob.new_k[ok])
    untouched = np.setdiff1d(np.arange(prob.num_slots), slots[ok])
    assert np.array_equal(after_k[untouched], before_k[untouched])


def test_kv_store_empty_is_noop():
    g = _gpu()
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    prob = inputs.tiny_extend()
    dev = g.Dev(prob)
    before = g.to_host_u16(dev.k_pool)
    e = torch.empty((0, prob.hkv, prob.d), dtype=torch.bfloat16, device="cuda")
    rx.rx_kv_store(dev.k_pool, dev.v_pool, e, e, torch.empty(0, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert np.array_equal(g.to_host_u16(dev.k_pool), before)


# ---------------------------------------------------------------------------
# extend
# ---------------------------------------------------------------------------


def _check_extend(prob, g=None, staged=False):
    g = g or _gpu()
    dev = g.Dev(prob)
    dev.kv_store()
    o, lse = dev.extend(staged=staged)
    kp, vp, rtt = dev.oracle_pools()
    ro, rl = oracle.extend(prob.q_ext, kp, vp, rtt, prob.ext_req_idx, prob.ext_prefix_len,
                           prob.ext_extend_len, prob.qo_indptr, prob.sm_scale)
    g.compare(o, ro, prob.name)
    g.compare_lse(lse, rl, prob.name)
    assert dev.status_word() == 0
    return o, lse


@pytest.mark.parametrize("staged", [False, True])
def test_extend_tiny_full_config(staged):
    """The tiny-extend configuration at its full size, every output."""
    _check_extend(inputs.tiny_extend(), staged=staged)


@pytest.mark.parametrize("staged", [False, True])
@pytest.mark.parametrize("hq,hkv,d", [(4, 4, 64), (8, 2, 64), (32, 8, 128), (16, 2, 128), (4, 1, 128)])
def test_extend_ragged(hq, hkv, d, staged):
    prob = inputs.ragged(20 + hq + d, hq=hq, hkv=hkv, d=d, n_groups=3, per_group=2, shared_max=150,
                         private_max=90, extend_max=140, decode=False, num_slots=3000)
    _check_extend(prob, staged=staged)


@pytest.mark.parametrize("staged", [False, True])
def test_extend_cached_prefix_reduced(staged):
    _check_extend(inputs.cached_prefix_extend(n_prefix=2, per_prefix=2, prefix=300, extend=150,
                                              num_slots=4096), staged=staged)


@pytest.mark.parametrize("staged", [False, True])
def test_extend_edge_cases(staged):
    # prefix 0 (plain causal), extend 1 (a single new token), long prefix
    for P, E in ((0, 70), (0, 1), (5, 1), (333, 3), (64, 64), (1, 129)):
        prob = inputs.tiny_extend(seed=P * 1000 + E, hq=8, hkv=2, d=128, batch=2, prefix=P, extend=E,
                                  num_slots=1024)
        _check_extend(prob, staged=staged)


def test_extend_staged_equals_gathered_bitwise():
    """Staging the rows first changes where they are read from, not the arithmetic."""
    g = _gpu()
    prob = inputs.cached_prefix_extend(n_prefix=2, per_prefix=3, prefix=200, extend=130, num_slots=4096)
    dev = g.Dev(prob)
    dev.kv_store()
    o1, l1 = dev.extend(staged=False)
    o2, l2 = dev.extend(staged=True)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    assert dev.status_word() == 0


@pytest.mark.parametrize("prefix,extend", [(256, 100), (300, 70), (130, 200), (128, 1)])
def test_extend_staged_shares_prefix_tiles(prefix, extend):
    """Requests whose slot lists agree on whole leading 128-row prefix tiles
    stage those tiles once and read them from the first such request's
    rows: results bit-identical to the gather path and within tolerance of
    the oracle, for prefixes on and off tile boundaries; plus requests with
    a private prefix and one whose list departs from its group's inside the
    second tile."""
    g = _gpu()
    prob = inputs.cached_prefix_extend(seed=prefix + extend, hq=16, hkv=4, d=128, n_prefix=3, per_prefix=3,
                                       prefix=prefix, extend=extend, num_slots=8192)
    prob.req_to_token = prob.req_to_token.copy()
    if prefix >= 256:   # request 4 leaves its group at position 200 (inside the second tile)
        free = np.setdiff1d(np.arange(prob.num_slots), prob.req_to_token[prob.req_to_token >= 0])
        prob.req_to_token[4, 200:prefix] = free[:prefix - 200]
    dev = g.Dev(prob)
    dev.kv_store()
    o1, l1 = dev.extend(staged=False)
    o2, l2 = dev.extend(staged=True)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    assert dev.status_word() == 0
    kp, vp, rtt = dev.oracle_pools()
    ro, rl = oracle.extend(prob.q_ext, kp, vp, rtt, prob.ext_req_idx, prob.ext_prefix_len, prob.ext_extend_len,
                           prob.qo_indptr, prob.sm_scale)
    g.compare(o2, ro, "staged extend with shared tiles")
    g.compare_lse(l2, rl, "staged extend with shared tiles")


def test_extend_staged_workspace_too_small_is_flagged():
    g = _gpu()
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    prob = inputs.tiny_extend(seed=3, hq=8, hkv=2, d=128, batch=3, prefix=200, extend=40, num_slots=1024)
    dev = g.Dev(prob)
    dev.kv_store()
    # the three contexts need 512 packed rows even with their shared first
    # tile staged once; a workspace sized for 40 context tokens holds 421
    dev.extend(staged=True, ws_rows=40)
    assert dev.status_word() & rx.RX_DEV_BAD_LEN


def test_extend_staged_bad_slot_is_flagged():
    g = _gpu()
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    prob = inputs.tiny_extend(seed=4, hq=8, hkv=2, d=128, batch=2, prefix=100, extend=30, num_slots=1024)
    dev = g.Dev(prob)
    dev.kv_store()
    dev.rtt[1, 17] = prob.num_slots + 5
    o, _ = dev.extend(staged=True)
    assert dev.status_word() & rx.RX_DEV_BAD_SLOT
    assert np.isfinite(o).all()


# ---------------------------------------------------------------------------
# decode
# ---------------------------------------------------------------------------


def _check_decode(prob, plan, kv_chunk=0, min_shared=16, g=None):
    g = g or _gpu()
    dev = g.Dev(prob)
    dev.kv_store()
    o, lse = dev.decode(plan=plan, kv_chunk=kv_chunk, min_shared=min_shared)
    kp, vp, rtt = dev.oracle_pools()
    ro, rl = oracle.decode(prob.q_dec, kp, vp, rtt, prob.dec_req_idx, prob.dec_seq_len, prob.sm_scale)
    g.compare(o, ro, f"{prob.name} plan={plan}")
    g.compare_lse(lse, rl, f"{prob.name} plan={plan}")
    assert dev.status_word() == 0
    return o, lse


@pytest.mark.parametrize("plan", [False, True])
@pytest.mark.parametrize("hq,hkv,d", [(4, 4, 64), (32, 32, 128), (32, 8, 128), (64, 8, 128), (8, 1, 64),
                                      (16, 8, 64), (64, 8, 64)])
def test_decode_ragged(plan, hq, hkv, d):
    prob = inputs.ragged(40 + hq + d, hq=hq, hkv=hkv, d=d, n_groups=3, per_group=3, shared_max=400,
                         private_max=300, extend_max=1, decode=True, num_slots=5000)
    _check_decode(prob, plan, kv_chunk=128 if plan else 0, min_shared=8)


@pytest.mark.parametrize("plan", [False, True])
def test_decode_few_shot_reduced(plan):
    _check_decode(inputs.few_shot_decode(batch=12, shared=300, private=77, num_slots=8192), plan)


@pytest.mark.parametrize("hq", [8, 32])
@pytest.mark.parametrize("shared,private", [(300, 200), (700, 600)])
def test_decode_split_rows_merged(hq, shared, private):
    """Rows split into few (9) and many (21) parts, written by the per-head
    and the all-heads kernels (one and four q heads per kv head), combine to
    the oracle's result."""
    prob = inputs.few_shot_decode(hq=hq, hkv=8, d=128, batch=6, shared=shared, private=private, num_slots=8192)
    _check_decode(prob, plan=True, kv_chunk=64)


@pytest.mark.parametrize("hq,hkv,d,private,parts", [(8, 8, 64, 300, (13, 64)), (32, 8, 128, 900, (13, 64)),
                                                    (8, 8, 128, 3000, (65, 400)), (32, 8, 64, 2500, (65, 400))])
def test_decode_merge_part_counts(hq, hkv, d, private, parts):
    """The merge's three ways through a row's parts: the plan's automatic
    pieces give every row 13 to 64 parts (loaded in batches of 16) or more
    than 64 (the general loop), at d 64 and 128; the rows then match the
    oracle."""
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    prob = inputs.few_shot_decode(hq=hq, hkv=hkv, d=d, batch=2, shared=0, private=private, num_slots=8192)
    buf, info = rx.rx_decode_plan_build(prob.req_to_token, prob.dec_req_idx, prob.dec_seq_len, hq, hkv)
    nparts = np.asarray(buf[2:4])
    assert parts[0] <= nparts.min() and nparts.max() <= parts[1], nparts
    _check_decode(prob, plan=True)


def test_decode_tree_of_thought_reduced():
    prob = inputs.tree_of_thought_decode(depth=3, fanout=3, edge=70, num_slots=8192)
    _check_decode(prob, plan=True, kv_chunk=64, min_shared=16)
    _check_decode(prob, plan=True, kv_chunk=0, min_shared=16)
    _check_decode(prob, plan=False)


def test_decode_many_rows_per_segment():
    """A segment shared by more requests than one work item holds (row blocks)."""
    prob = inputs.few_shot_decode(hq=16, hkv=2, d=128, batch=40, shared=200, private=9,
                                  num_slots=4096)
    _check_decode(prob, plan=True, kv_chunk=64)


def test_decode_single_token_context():
    prob = inputs.few_shot_decode(hq=8, hkv=2, d=64, batch=5, shared=0, private=0, num_slots=64)
    for plan in (False, True):
        _check_decode(prob, plan)


@pytest.mark.parametrize("hq,hkv,d", [(32, 32, 128), (32, 8, 128), (64, 8, 128), (8, 2, 64), (4, 4, 64)])
def test_decode_plan_serves_later_steps(hq, hkv, d):
    """A plan built when every request was k tokens shorter serves the later
    step unchanged: each request's last piece ends at its length on the
    device (RX_PLAN_OPEN_END).  All-heads kernels (one and several q heads
    per kv head) and the per-head kernel (two kv heads) alike."""
    g = _gpu()
    prob = inputs.few_shot_decode(hq=hq, hkv=hkv, d=d, batch=9, shared=200, private=90, num_slots=8192)
    dev = g.Dev(prob)
    dev.kv_store()
    kp, vp, rtt = dev.oracle_pools()
    ro, rl = oracle.decode(prob.q_dec, kp, vp, rtt, prob.dec_req_idx, prob.dec_seq_len, prob.sm_scale)
    for k in (1, 5, 40):
        for chunk in (0, 64):
            o, lse = dev.decode(plan=True, kv_chunk=chunk, plan_seq_len=prob.dec_seq_len - k)
            g.compare(o, ro, f"plan built {k} tokens earlier, chunk {chunk}")
            g.compare_lse(lse, rl, f"plan built {k} tokens earlier, chunk {chunk}")
    assert dev.status_word() == 0


@pytest.mark.parametrize("hq,hkv", [(32, 32), (32, 8), (8, 2)])
def test_decode_open_end_past_the_slot_lists_is_flagged(hq, hkv):
    """A device length past the slot lists' stride, or one that no longer
    reaches a request's last piece, is flagged (RX_DEV_BAD_LEN); the outputs
    stay finite and nothing outside the buffers is read."""
    g = _gpu()
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    prob = inputs.few_shot_decode(hq=hq, hkv=hkv, d=128, batch=5, shared=64, private=40, num_slots=2048)
    dev = g.Dev(prob)
    dev.kv_store()
    for bad in (prob.rtt_stride + 3, 10):
        lens = prob.dec_seq_len.copy()
        lens[2] = bad
        dev.status.zero_()
        o, _ = dev.decode(plan=True, kv_chunk=64, seq_len=lens)
        assert dev.status_word() & rx.RX_DEV_BAD_LEN, bad
        assert np.isfinite(o).all()


@pytest.mark.parametrize("hq,hkv", [(32, 32), (32, 8), (8, 2)])
def test_decode_wait_that_runs_out_is_reported(hq, hkv):
    """With the decode kernels' wait limit cut to a few cycles, their first
    pipeline wait that is not already satisfied runs out: the call's status
    word gets RX_DEV_TIMEOUT, the kernels leave cleanly (copies in flight are
    waited for), and the context stays usable -- the next call with the
    default limit matches the oracle.  No GPU fault is involved: the waits
    are bounded by construction and simply give up early."""
    g = _gpu()
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    prob = inputs.few_shot_decode(hq=hq, hkv=hkv, d=128, batch=6, shared=300, private=200, num_slots=4096)
    dev = g.Dev(prob)
    dev.kv_store()
    try:
        rx.rx_decode_set_wait_limit(8)
        dev.decode(plan=True, kv_chunk=64)
        assert dev.status_word() & rx.RX_DEV_TIMEOUT
    finally:
        rx.rx_decode_set_wait_limit(0)
    dev.status.zero_()
    o, lse = dev.decode(plan=True, kv_chunk=64)
    assert dev.status_word() == 0
    kp, vp, rtt = dev.oracle_pools()
    ro, rl = oracle.decode(prob.q_dec, kp, vp, rtt, prob.dec_req_idx, prob.dec_seq_len, prob.sm_scale)
    g.compare(o, ro, "after a timed-out call")
    g.compare_lse(lse, rl, "after a timed-out call")


def test_decode_without_lse_output():
    g = _gpu()
    prob = inputs.few_shot_decode(hq=8, hkv=8, d=128, batch=6, shared=100, private=50, num_slots=1024)
    dev = g.Dev(prob)
    dev.kv_store()
    o, _ = dev.decode(plan=True, with_lse=False)
    kp, vp, rtt = dev.oracle_pools()
    ro, _ = oracle.decode(prob.q_dec, kp, vp, rtt, prob.dec_req_idx, prob.dec_seq_len, prob.sm_scale)
    g.compare(o, ro)


def test_decode_bad_slot_is_flagged():
    g = _gpu()
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    prob = inputs.few_shot_decode(hq=8, hkv=8, d=128, batch=4, shared=40, private=20, num_slots=512)
    prob.req_to_token = prob.req_to_token.copy()
    prob.req_to_token[2, 45] = prob.num_slots + 100
    dev = g.Dev(prob)
    dev.kv_store()
    o, _ = dev.decode(plan=False)
    assert dev.status_word() & rx.RX_DEV_BAD_SLOT
    assert np.isfinite(o).all()


@pytest.mark.parametrize("hq,hkv", [(8, 8), (32, 8)])
def test_decode_bad_slot_in_wide_item_is_flagged(hq, hkv):
    """A bad slot id inside a single-request item (the all-heads kernels, one
    and four q heads per kv head) is flagged and read as a zero row, like the
    per-head path does: the other rows match the oracle with that row's K
    and V set to zero."""
    g = _gpu()
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    prob = inputs.few_shot_decode(hq=hq, hkv=hkv, d=128, batch=4, shared=40, private=90, num_slots=512)
    buf, info = rx.rx_decode_plan_build(prob.req_to_token, prob.dec_req_idx, prob.dec_seq_len, prob.hq,
                                        prob.hkv, 64, 16)
    assert info.n_wide > 0
    good_slot = int(prob.req_to_token[1, 70])
    prob.req_to_token = prob.req_to_token.copy()
    prob.req_to_token[1, 70] = -3                      # inside request 1's private tail
    dev = g.Dev(prob)
    dev.kv_store()
    o, _ = dev.decode(plan=True, kv_chunk=64)
    assert dev.status_word() & rx.RX_DEV_BAD_SLOT
    assert np.isfinite(o).all()
    # the oracle with the bad position reading a zero row
    kp, vp, rtt = dev.oracle_pools()
    kp, vp = kp.copy(), vp.copy()
    rtt = rtt.copy()
    rtt[1, 70] = good_slot
    kp[good_slot] = 0
    vp[good_slot] = 0
    ro, _ = oracle.decode(prob.q_dec, kp, vp, rtt, prob.dec_req_idx, prob.dec_seq_len, prob.sm_scale)
    g.compare(o, ro, "bad slot as a zero row")


@pytest.mark.parametrize("hq", [16, 32, 64])
def test_decode_bad_slot_in_group_item_is_flagged(hq):
    """A bad slot id inside a shared segment read by a group item (several
    requests on the all-heads kernel with G = 2, 4, 8) is flagged and read as
    a zero row for every request of the group.  The id is planted in every
    request's list, so the segment stays shared."""
    g = _gpu()
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    prob = inputs.few_shot_decode(hq=hq, hkv=8, d=128, batch=5, shared=60, private=30, num_slots=1024)
    prob.req_to_token = prob.req_to_token.copy()
    good_slot = int(prob.req_to_token[0, 33])
    prob.req_to_token[:, 33] = prob.num_slots + 7
    buf, info = rx.rx_decode_plan_build(prob.req_to_token, prob.dec_req_idx, prob.dec_seq_len, prob.hq,
                                        prob.hkv, 64, 16)
    items = buf[2 * len(prob.dec_req_idx):].reshape(-1, 8)
    tail = items[len(items) - info.n_wide:]
    assert np.any(tail[:, 1] > 1) and len(items) == info.n_wide   # groups only, no per-head item
    dev = g.Dev(prob)
    dev.kv_store()
    o, _ = dev.decode(plan=True, kv_chunk=64)
    assert dev.status_word() & rx.RX_DEV_BAD_SLOT
    assert np.isfinite(o).all()
    kp, vp, rtt = dev.oracle_pools()
    kp, vp, rtt = kp.copy(), vp.copy(), rtt.copy()
    rtt[:, 33] = good_slot
    kp[good_slot] = 0
    vp[good_slot] = 0
    ro, _ = oracle.decode(prob.q_dec, kp, vp, rtt, prob.dec_req_idx, prob.dec_seq_len, prob.sm_scale)
    g.compare(o, ro, "bad slot in a group item as a zero row")


@pytest.mark.parametrize("hq", [8, 32])
def test_decode_wide_ctas_that_find_the_queue_empty(hq):
    """All-heads CTAs that start after the other CTAs have taken every
    single-request item end cleanly.  A 4096-position shared segment read as
    one chunk (three row blocks x eight kv heads: 24 per-head CTAs) holds 24
    SMs far longer than the 160 short private tails take on the rest, so the
    all-heads CTAs that wait for those SMs find the work queue empty."""
    g = _gpu()
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    prob = inputs.few_shot_decode(hq=hq, hkv=8, d=128, batch=160, shared=4096, private=20, num_slots=8192)
    buf, info = rx.rx_decode_plan_build(prob.req_to_token, prob.dec_req_idx, prob.dec_seq_len, prob.hq,
                                        prob.hkv, 4096, 16)
    # row blocks of 64 query rows: 64 requests at G = 1, 16 at G = 4
    assert info.n_wide == 160 and info.n_items - info.n_wide == (3 if hq == 8 else 10)
    for _ in range(3):
        _check_decode(prob, plan=True, kv_chunk=4096, g=g)


def test_decode_length_past_bound_is_flagged():
    g = _gpu()
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    prob = inputs.few_shot_decode(hq=8, hkv=8, d=64, batch=3, shared=400, private=200, num_slots=2048)
    dev = g.Dev(prob)
    dev.kv_store()
    p = prob
    q = g.to_dev(p.q_dec)
    o = torch.zeros_like(q)
    # claim max_seq_len far below the real lengths (601): the grid covers one
    # 64-position chunk, so the rows are skipped and flagged
    rx.rx_attn_decode(dev.k_pool, dev.v_pool, q, o, None, g.i32(p.dec_req_idx), g.i32(p.dec_seq_len),
                      dev.rtt, 10, p.sm_scale, None, None, dev.status)
    torch.cuda.synchronize()
    assert dev.status_word() & rx.RX_DEV_BAD_LEN


# ---------------------------------------------------------------------------
# invariants on the GPU
# ---------------------------------------------------------------------------


def test_grouped_equals_ungrouped():
    """Reading shared KV once per group gives the per-request result."""
    g = _gpu()
    prob = inputs.tree_of_thought_decode(depth=3, fanout=3, edge=90, num_slots=8192)
    dev = g.Dev(prob)
    dev.kv_store()
    o1, l1 = dev.decode(plan=False)
    o2, l2 = dev.decode(plan=True, kv_chunk=64, min_shared=1)
    assert np.max(np.abs(o1 - o2)) <= 2 * g.ATOL
    assert np.max(np.abs(l1 - l2)) <= 2 * g.LSE_ATOL


def test_slot_permutation_bit_identical():
    """Renaming pool rows (and req_to_token with them) changes no output bit."""
    g = _gpu()
    prob = inputs.few_shot_decode(hq=8, hkv=2, d=128, batch=6, shared=150, private=70, num_slots=2048)
    dev = g.Dev(prob)
    dev.kv_store()
    o1, l1 = dev.decode(plan=False)
    perm = np.random.default_rng(9).permutation(prob.num_slots).astype(np.int32)
    prob2 = inputs.few_shot_decode(hq=8, hkv=2, d=128, batch=6, shared=150, private=70, num_slots=2048)
    prob2.req_to_token = np.where(prob.req_to_token >= 0, perm[np.maximum(prob.req_to_token, 0)], -1)
    prob2.cached_slots = perm[prob.cached_slots]
    prob2.new_slots = perm[prob.new_slots]
    dev2 = g.Dev(prob2)
    dev2.kv_store()
    o2, l2 = dev2.decode(plan=False)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_decode_equals_last_extend_row():
    g = _gpu()
    prob = inputs.tiny_extend(seed=77, hq=8, hkv=2, d=128, batch=3, prefix=100, extend=40,
                              num_slots=1024)
    dev = g.Dev(prob)
    dev.kv_store()
    oe, le = dev.extend()
    last = prob.qo_indptr[1:] - 1
    prob.q_dec = prob.q_ext[last]
    prob.dec_req_idx = prob.ext_req_idx
    prob.dec_seq_len = prob.ext_prefix_len + prob.ext_extend_len
    od, ld = dev.decode(plan=False)
    assert np.max(np.abs(od - oe[last])) <= 2 * g.ATOL
