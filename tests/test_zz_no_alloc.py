"""rx_attn_decode_static: decode for callers that cannot allocate device memory.

Some callers of this library cannot hand it device scratch memory (all of
their device memory is committed at start-up, or allocator calls are not
allowed while serving).  rx_attn_decode_static keeps the partial results of
split work in a fixed device array inside the library instead of a caller
workspace.  This file checks, through the C ABI, that it returns what
rx_attn_decode returns with a workspace, on two calls in a row (the second
call finds the first call's data in the shared array), and that a batch too
big for the array is refused.  It sits last in collection order so that a
run stopping at the first failure has run every other test first.
"""
import numpy as np
import pytest

from prefix_shared_kv_radixattention_gb300 import inputs

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _setup(prob, kv_chunk):
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    from tests import _gpu as g
    dev = g.Dev(prob)
    dev.kv_store()
    B = len(prob.dec_req_idx)
    buf, info = rx.rx_decode_plan_build(prob.req_to_token, prob.dec_req_idx, prob.dec_seq_len, prob.hq,
                                        prob.hkv, kv_chunk, 16)
    plan = rx.plan_to_device(buf, info, B)
    return rx, g, dev, plan


def _with_workspace(rx, g, dev, plan, prob):
    B = len(prob.dec_req_idx)
    max_len = int(prob.dec_seq_len.max())
    q = g.to_dev(prob.q_dec)
    o = torch.empty_like(q)
    lse = torch.empty((B, prob.hq), dtype=torch.float32, device="cuda")
    ws_bytes = rx.rx_attn_decode_workspace(B, prob.hq, prob.hkv, prob.d, max_len, plan)
    assert ws_bytes > 0, "the case must split work, so that scratch memory is used"
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    rx.rx_attn_decode(dev.k_pool, dev.v_pool, q, o, lse, g.i32(prob.dec_req_idx), g.i32(prob.dec_seq_len),
                      dev.rtt, max_len, prob.sm_scale, plan, ws, dev.status)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def _static(rx, g, dev, plan, prob):
    B = len(prob.dec_req_idx)
    max_len = int(prob.dec_seq_len.max())
    q = g.to_dev(prob.q_dec)
    o = torch.empty_like(q)
    lse = torch.empty((B, prob.hq), dtype=torch.float32, device="cuda")
    rx.rx_attn_decode_static(dev.k_pool, dev.v_pool, q, o, lse, g.i32(prob.dec_req_idx),
                             g.i32(prob.dec_seq_len), dev.rtt, max_len, prob.sm_scale, plan, dev.status)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def test_static_scratch_matches_workspace_two_calls():
    """The static array and a workspace give bit-identical results (the same
    kernels run on the same plan; only where the partials live differs).
    The second call in a row is a smaller batch with other shapes than the
    first, so a partial read from the wrong offset, or one left over from
    the first call's data, would show.  Both also match the oracle."""
    import oracle
    cases = [
        (inputs.tree_of_thought_decode(seed=72, depth=3, fanout=3, edge=90, num_slots=8192), 64),
        (inputs.few_shot_decode(seed=71, hq=8, hkv=2, d=128, batch=10, shared=300, private=150,
                                num_slots=8192), 64),
    ]
    sizes = []
    for prob, kv_chunk in cases:   # two calls in a row on the shared array
        rx, g, dev, plan = _setup(prob, kv_chunk)
        sizes.append(rx.rx_attn_decode_workspace(len(prob.dec_req_idx), prob.hq, prob.hkv, prob.d,
                                                 int(prob.dec_seq_len.max()), plan))
        o_ws, l_ws = _with_workspace(rx, g, dev, plan, prob)
        o_st, l_st = _static(rx, g, dev, plan, prob)
        assert np.array_equal(o_st, o_ws), "static scratch and workspace outputs differ"
        assert np.array_equal(l_st, l_ws), "static scratch and workspace log-sum-exps differ"
        assert dev.status_word() == 0
        kp, vp, rtt = dev.oracle_pools()
        ro, rl = oracle.decode(prob.q_dec, kp, vp, rtt, prob.dec_req_idx, prob.dec_seq_len, prob.sm_scale)
        g.compare(o_st, ro, f"{prob.name} static scratch")
        g.compare_lse(l_st, rl, f"{prob.name} static scratch")
    assert sizes[1] < sizes[0], "the second call must use less of the array than the first"


def test_static_scratch_checks_arguments_before_capacity():
    """A malformed plan is reported as invalid, not as a batch too big for
    the array."""
    import ctypes
    prob = inputs.few_shot_decode(seed=73, hq=8, hkv=8, d=128, batch=4, shared=100, private=70, num_slots=1024)
    rx, g, dev, plan = _setup(prob, 64)
    bad = rx.DecodePlan.from_buffer_copy(plan.struct)
    bad.max_parts = 0
    q = g.to_dev(prob.q_dec)
    o = torch.empty_like(q)
    with pytest.raises(rx.RxError) as e:
        rx._check(rx._lib.rx_attn_decode_static(
            ctypes.byref(rx.make_pool(dev.k_pool, dev.v_pool)), rx._ptr(q), rx._ptr(o), None, prob.hq,
            rx._ptr(g.i32(prob.dec_req_idx)), rx._ptr(g.i32(prob.dec_seq_len)), rx._ptr(dev.rtt),
            dev.rtt.shape[1], len(prob.dec_req_idx), int(prob.dec_seq_len.max()), ctypes.byref(bad),
            ctypes.c_float(prob.sm_scale), None, rx._stream(None)))
    assert e.value.code == rx.RX_ERR_INVALID


def test_static_scratch_refuses_oversized_batch():
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    # 64 requests x 64 q heads split into 256 parts of 4096 positions need far
    # more partial-result space than the fixed array holds; the call is
    # refused on the host before anything is launched
    B, hq, hkv, d, max_len = 64, 64, 8, 128, 1 << 20
    need = rx.rx_attn_decode_workspace(B, hq, hkv, d, max_len, None)
    assert need > rx.RX_DECODE_STATIC_SCRATCH_BYTES
    k = torch.empty((1, hkv, d), dtype=torch.bfloat16, device="cuda")
    q = torch.empty((B, hq, d), dtype=torch.bfloat16, device="cuda")
    idx = torch.zeros(B, dtype=torch.int32, device="cuda")
    rtt = torch.zeros((1, max_len), dtype=torch.int32, device="cuda")
    with pytest.raises(rx.RxError) as e:
        rx.rx_attn_decode_static(k, k, q, q, None, idx, idx, rtt, max_len, 1.0 / d ** 0.5)
    assert e.value.code == rx.RX_ERR_CAPACITY
