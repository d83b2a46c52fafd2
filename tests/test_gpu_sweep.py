"""GPU parity on random radix forests: nested shared prefixes of random
lengths (empty edges included), random fan-outs, requests that end inside
another request's shared prefix, shuffled batch order (inputs.random_tree).

Each seed picks a head layout, a plan setting and the pool type, so the
sweep crosses every decode kernel (per-head, the one-q-head and GQA
all-heads kernels, the merge) and both extend operand paths with structures
no fixed workload has.  Tolerance as in tests/_gpu.py.
"""
import numpy as np
import pytest

import oracle
from oracle import fp8
from prefix_shared_kv_radixattention_gb300 import inputs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

# (q heads, kv heads, head_dim): one q head per kv head, 8 kv heads with
# G = 2 .. 16 (the GQA all-heads kernel), and other groupings (per-head only)
DECODE_HEADS = [(32, 32, 128), (32, 8, 128), (64, 8, 128), (16, 8, 64), (8, 2, 64), (4, 4, 64),
                (128, 8, 128), (64, 2, 64), (16, 16, 128), (32, 8, 64)]
EXTEND_HEADS = [(32, 8, 128), (8, 8, 64), (64, 8, 128), (16, 2, 128), (4, 1, 64), (32, 32, 128)]


def _setting(seed):
    rng = np.random.default_rng(77_000 + seed)
    kv_chunk = [0, 64, 128, 256][int(rng.integers(4))]
    min_shared = [1, 8, 32][int(rng.integers(3))]
    return kv_chunk, min_shared


@pytest.mark.parametrize("seed", range(16))
def test_decode_random_forest(seed):
    """bf16 pools: without a plan, with the automatic plan, and with the
    seed's chunk and minimum segment length."""
    from tests import _gpu as g
    hq, hkv, d = DECODE_HEADS[seed % len(DECODE_HEADS)]
    prob = inputs.random_tree(6100 + seed, hq, hkv, d, decode=True)
    kv_chunk, min_shared = _setting(seed)
    dev = g.Dev(prob)
    dev.kv_store()
    kp, vp, rtt = dev.oracle_pools()
    ro, rl = oracle.decode(prob.q_dec, kp, vp, rtt, prob.dec_req_idx, prob.dec_seq_len, prob.sm_scale)
    for plan, chunk, ms in ((False, 0, 16), (True, 0, 16), (True, kv_chunk, min_shared)):
        o, lse = dev.decode(plan=plan, kv_chunk=chunk, min_shared=ms)
        what = f"seed {seed} {hq}/{hkv}x{d} plan={plan} chunk={chunk} min_shared={ms}"
        g.compare(o, ro, what)
        g.compare_lse(lse, rl, what)
    assert dev.status_word() == 0


@pytest.mark.parametrize("seed", range(6))
def test_decode_fp8_random_forest(seed):
    """E4M3 pools with random scales, against the oracle over decoded codes."""
    from tests import _gpu as g
    from tests.test_gpu_fp8 import _decode_fp8, _fp8_problem
    hq, hkv, d = DECODE_HEADS[(3 * seed + 1) % len(DECODE_HEADS)]
    prob = inputs.random_tree(6300 + seed, hq, hkv, d, decode=True, max_requests=24)
    rng = np.random.default_rng(6300 + seed)
    ks, vs = float(rng.uniform(0.25, 2.0)), float(rng.uniform(0.25, 2.0))
    kd, vd, kc, vc, status = _fp8_problem(prob, ks, vs, seed)
    ro, rl = fp8.decode_rows(prob.q_dec, kc, vc, ks, vs, prob.req_to_token, prob.dec_req_idx, prob.dec_seq_len,
                             prob.sm_scale)
    kv_chunk, _ = _setting(seed)
    for use_plan, chunk in ((False, 0), (True, 0), (True, kv_chunk)):
        o, lse, _ = _decode_fp8(prob, kd, vd, ks, vs, status, kv_chunk=chunk, use_plan=use_plan)
        what = f"fp8 seed {seed} {hq}/{hkv}x{d} plan={use_plan} chunk={chunk}"
        g.compare(o, ro, what)
        g.compare_lse(lse, rl, what)
    assert int(status.item()) == 0


@pytest.mark.parametrize("seed", range(10))
def test_extend_random_forest(seed):
    """bf16 pools, both operand paths: the oracle's result, and the two
    paths bit for bit equal."""
    from tests import _gpu as g
    hq, hkv, d = EXTEND_HEADS[seed % len(EXTEND_HEADS)]
    prob = inputs.random_tree(6500 + seed, hq, hkv, d, decode=False, max_requests=16, edge_max=260,
                              private_max=150, extend_max=90)
    dev = g.Dev(prob)
    dev.kv_store()
    kp, vp, rtt = dev.oracle_pools()
    ro, rl = oracle.extend(prob.q_ext, kp, vp, rtt, prob.ext_req_idx, prob.ext_prefix_len,
                           prob.ext_extend_len, prob.qo_indptr, prob.sm_scale)
    outs = {}
    for staged in (False, True):
        o, lse = dev.extend(staged=staged)
        what = f"seed {seed} {hq}/{hkv}x{d} staged={staged}"
        g.compare(o, ro, what)
        g.compare_lse(lse, rl, what)
        outs[staged] = (o, lse)
    assert np.array_equal(outs[False][0], outs[True][0])
    assert np.array_equal(outs[False][1].view(np.uint32), outs[True][1].view(np.uint32))
    assert dev.status_word() == 0


@pytest.mark.parametrize("seed", range(4))
def test_extend_fp8_random_forest(seed):
    """E4M3 pools with random scales, both operand paths, against the oracle
    over decoded codes."""
    from tests import _gpu as g
    from tests.test_gpu_fp8 import _extend_fp8, _extend_rows, _fp8_problem
    hq, hkv, d = EXTEND_HEADS[(2 * seed + 1) % len(EXTEND_HEADS)]
    prob = inputs.random_tree(6700 + seed, hq, hkv, d, decode=False, max_requests=12, edge_max=200,
                              private_max=120, extend_max=80)
    rng = np.random.default_rng(6700 + seed)
    ks, vs = float(rng.uniform(0.25, 2.0)), float(rng.uniform(0.25, 2.0))
    kd, vd, kc, vc, status = _fp8_problem(prob, ks, vs, 100 + seed)
    q_row, kbeg, kend = _extend_rows(prob)
    ro, rl = fp8.attention(prob.q_ext, kc, vc, ks, vs, prob.req_to_token, q_row, kbeg, kend, prob.sm_scale)
    for staged in (True, False):
        o, lse = _extend_fp8(prob, kd, vd, ks, vs, status, staged=staged)
        what = f"fp8 seed {seed} {hq}/{hkv}x{d} staged={staged}"
        g.compare(o.float().cpu().numpy(), ro, what)
        g.compare_lse(lse.cpu().numpy(), rl, what)
    assert int(status.item()) == 0
