"""GPU parity at the workloads' full sizes, in the launch configuration that
bench.py times: the full pool, the decode plan with its automatic chunking,
extend on the staged path (and on the gather path).  The oracle computes
sampled rows one by one through the same slot lists: the first and last
request, the first and last token of each request, the tokens on both sides
of every 256-row CTA boundary of a sampled request, and seeded random rows.
Tolerance as in tests/_gpu.py.
"""
import numpy as np
import pytest

import oracle
from prefix_shared_kv_radixattention_gb300 import admission, inputs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _gpu():
    from tests import _gpu
    return _gpu


def _pick(rng, n, k, must=()):
    extra = rng.choice(n, size=min(k, n), replace=False)
    return np.array(sorted(set(int(i) for i in must) | set(int(i) for i in extra)), dtype=np.int64)


def _check_decode_rows(g, dev, prob, o, lse, rows):
    kp, vp, rtt = dev.oracle_pools()
    ro, rl = oracle.attention(prob.q_dec[rows], kp, vp, rtt, prob.dec_req_idx[rows],
                              np.zeros(len(rows), np.int32), prob.dec_seq_len[rows], prob.sm_scale)
    g.compare(o[rows], ro, f"{prob.name} decode")
    g.compare_lse(lse[rows], rl, f"{prob.name} decode")


def _extend_rows(rng, prob, per_req=6):
    """Packed token rows and their key ranges: boundary tokens plus random ones."""
    G = prob.hq // prob.hkv
    tb = 256 // G                       # tokens per CTA
    B = len(prob.ext_req_idx)
    reqs = _pick(rng, B, 4, must=(0, B - 1))
    rows, kend, rtt_row = [], [], []
    for b in reqs:
        E, P, q0 = int(prob.ext_extend_len[b]), int(prob.ext_prefix_len[b]), int(prob.qo_indptr[b])
        toks = {0, E - 1}
        for edge in range(tb, E, tb):
            toks |= {edge - 1, edge}
        toks |= set(int(t) for t in rng.choice(E, size=min(per_req, E), replace=False))
        for t in sorted(toks):
            rows.append(q0 + t)
            kend.append(P + t + 1)
            rtt_row.append(int(prob.ext_req_idx[b]))
    return np.array(rows), np.array(kend, np.int32), np.array(rtt_row, np.int32)


def _check_extend_rows(g, dev, prob, o, lse, rng):
    rows, kend, rtt_row = _extend_rows(rng, prob)
    kp, vp, rtt = dev.oracle_pools()
    ro, rl = oracle.attention(prob.q_ext[rows], kp, vp, rtt, rtt_row, np.zeros(len(rows), np.int32), kend,
                              prob.sm_scale)
    g.compare(o[rows], ro, f"{prob.name} extend")
    g.compare_lse(lse[rows], rl, f"{prob.name} extend")


@pytest.mark.parametrize("name", ["few_shot_decode", "tree_of_thought_decode"])
def test_decode_full_size(name):
    g = _gpu()
    prob = inputs.FULL_SIZE[name]()
    dev = g.Dev(prob)
    dev.kv_store()
    o, lse = dev.decode(plan=True)
    assert dev.status_word() == 0
    B = len(prob.dec_req_idx)
    rows = _pick(np.random.default_rng(11), B, 24, must=(0, B - 1))
    _check_decode_rows(g, dev, prob, o, lse, rows)


@pytest.mark.parametrize("staged", [True, False])
def test_extend_full_size_cached_prefix(staged):
    g = _gpu()
    prob = inputs.cached_prefix_extend()
    dev = g.Dev(prob)
    dev.kv_store()
    o, lse = dev.extend(staged=staged)
    assert dev.status_word() == 0
    _check_extend_rows(g, dev, prob, o, lse, np.random.default_rng(12))


def test_mixed_chat_full_size():
    """Long-context decode (32k, 8k shared) and extend rows of one batch,
    with the slot lists the radix cache handed out when the batch was
    admitted into the full 1M-slot pool (LRU eviction included)."""
    g = _gpu()
    prob = admission.mixed_chat()
    dev = g.Dev(prob)
    dev.kv_store()
    o_e, lse_e = dev.extend(staged=True)
    o_d, lse_d = dev.decode(plan=True)
    assert dev.status_word() == 0
    B = len(prob.dec_req_idx)
    _check_decode_rows(g, dev, prob, o_d, lse_d, np.arange(B))
    _check_extend_rows(g, dev, prob, o_e, lse_e, np.random.default_rng(13))
