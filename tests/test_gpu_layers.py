"""Layered pools: one allocation per K and V holding L layers, [L, S, Hkv, d].

A slot id names the same token in every layer, so one slot list (and one
decode plan) serves all layers; each call reads or writes one layer.  Two
layers with different values go through the same slot lists: the scatter
writes only its layer (bit for bit, the other layer untouched), and decode
and extend on each layer match the oracle on that layer's values.
"""
import numpy as np
import pytest

import oracle
from prefix_shared_kv_radixattention_gb300 import inputs

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _layered(prob, seed):
    """Host pools [2, S, Hkv, d] with the problem's cached rows in layer 0 and
    other values (same slots) in layer 1."""
    rng = np.random.default_rng(seed)
    S, hkv, d = prob.num_slots, prob.hkv, prob.d
    kp = inputs.randn_bf16(rng, (2, S, hkv, d))
    vp = inputs.randn_bf16(rng, (2, S, hkv, d))
    kp[0, prob.cached_slots], vp[0, prob.cached_slots] = prob.cached_k, prob.cached_v
    new1_k = inputs.randn_bf16(rng, prob.new_k.shape)
    new1_v = inputs.randn_bf16(rng, prob.new_v.shape)
    return kp, vp, (prob.new_k, new1_k), (prob.new_v, new1_v)


def _store_both(g, prob, kp, vp, new_k, new_v, rx):
    dk, dv = g.to_dev(kp), g.to_dev(vp)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots = g.i32(prob.new_slots)
    for layer in (0, 1):
        rx.rx_kv_store(dk, dv, g.to_dev(new_k[layer]), g.to_dev(new_v[layer]), slots, status, layer=layer)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for layer in (0, 1):   # the oracle's scatter, layer by layer
        k, v = kp[layer].copy(), vp[layer].copy()
        oracle.kv_store(k, v, new_k[layer], new_v[layer], prob.new_slots)
        kp[layer], vp[layer] = k, v
    assert np.array_equal(g.to_host_u16(dk), kp) and np.array_equal(g.to_host_u16(dv), vp)
    return dk, dv, status


def test_layers_decode_through_one_slot_list():
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    from tests import _gpu as g
    prob = inputs.few_shot_decode(hq=32, hkv=8, d=128, batch=7, shared=200, private=90, num_slots=4096)
    kp, vp, new_k, new_v = _layered(prob, 5)
    dk, dv, status = _store_both(g, prob, kp, vp, new_k, new_v, rx)
    B = len(prob.dec_req_idx)
    buf, info = rx.rx_decode_plan_build(prob.req_to_token, prob.dec_req_idx, prob.dec_seq_len, prob.hq, prob.hkv,
                                        64, 16)
    plan = rx.plan_to_device(buf, info, B)
    max_len = int(prob.dec_seq_len.max())
    ws = torch.empty(max(rx.rx_attn_decode_workspace(B, prob.hq, prob.hkv, prob.d, max_len, plan), 256),
                     dtype=torch.uint8, device="cuda")
    q = g.to_dev(prob.q_dec)
    rtt = g.i32(prob.req_to_token)
    outs = []
    for layer in (0, 1):
        o = torch.empty_like(q)
        lse = torch.empty((B, prob.hq), dtype=torch.float32, device="cuda")
        rx.rx_attn_decode(dk, dv, q, o, lse, g.i32(prob.dec_req_idx), g.i32(prob.dec_seq_len), rtt, max_len,
                          prob.sm_scale, plan, ws, status, layer=layer)
        torch.cuda.synchronize()
        ro, rl = oracle.decode(prob.q_dec, kp[layer], vp[layer], prob.req_to_token, prob.dec_req_idx,
                               prob.dec_seq_len, prob.sm_scale)
        g.compare(o.float().cpu().numpy(), ro, f"decode, layer {layer}")
        g.compare_lse(lse.cpu().numpy(), rl, f"decode, layer {layer}")
        outs.append(o.float().cpu().numpy())
    assert int(status.item()) == 0
    assert not np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("staged", [True, False])
def test_layers_extend_through_one_slot_list(staged):
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    from tests import _gpu as g
    prob = inputs.ragged(61, hq=16, hkv=4, d=64, n_groups=2, per_group=3, shared_max=150, private_max=90,
                         extend_max=150, decode=False, num_slots=4096)
    kp, vp, new_k, new_v = _layered(prob, 6)
    dk, dv, status = _store_both(g, prob, kp, vp, new_k, new_v, rx)
    q = g.to_dev(prob.q_ext)
    ws = None
    if staged:
        ctx = int((prob.ext_prefix_len + prob.ext_extend_len).sum())
        ws = torch.empty(rx.rx_attn_extend_workspace(ctx, len(prob.ext_req_idx), prob.hkv, prob.d),
                         dtype=torch.uint8, device="cuda")
    for layer in (1, 0):
        o = torch.empty_like(q)
        rx.rx_attn_extend(dk, dv, q, o, None, g.i32(prob.qo_indptr), g.i32(prob.ext_req_idx),
                          g.i32(prob.ext_prefix_len), g.i32(prob.ext_extend_len), g.i32(prob.req_to_token),
                          int(prob.ext_extend_len.max()), prob.sm_scale, status, workspace=ws, layer=layer)
        torch.cuda.synchronize()
        ro, _ = oracle.extend(prob.q_ext, kp[layer], vp[layer], prob.req_to_token, prob.ext_req_idx,
                              prob.ext_prefix_len, prob.ext_extend_len, prob.qo_indptr, prob.sm_scale)
        g.compare(o.float().cpu().numpy(), ro, f"extend, layer {layer}")
    assert int(status.item()) == 0
