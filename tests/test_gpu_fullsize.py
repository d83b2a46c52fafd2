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


# ---------------------------------------------------------------------------
# the same workloads over FP8 (E4M3) pools, as bench.py --kv-fp8 runs them
# ---------------------------------------------------------------------------

KS, VS = 0.5, 2.0       # pool scales (values N(0, 1): codes of N(0, 4) and N(0, 1/4))


def _fp8_setup(g, dev, prob):
    """Device code pools made by rx_kv_store_fp8 from the bf16 pools' used
    rows (cached and new slots); every other row holds the code of 448, so
    a read of an unused row shows.  Returns the device pools and the
    oracle's compact code pools with their slot lists."""
    from oracle import fp8
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    S, hkv, d = prob.num_slots, prob.hkv, prob.d
    k8 = torch.full((S, hkv, d), 0x7E, dtype=torch.uint8, device="cuda")
    v8 = torch.full((S, hkv, d), 0x7E, dtype=torch.uint8, device="cuda")
    used = np.unique(np.concatenate([prob.cached_slots, prob.new_slots])).astype(np.int64)
    idx = torch.from_numpy(used).cuda()
    for s in range(0, len(idx), 1 << 16):
        sl = idx[s:s + (1 << 16)]
        rx.rx_kv_store_fp8(k8, v8, KS, VS, dev.k_pool[sl], dev.v_pool[sl], sl.to(torch.int32), dev.status)
    kp, vp, rtt = dev.oracle_pools()
    kc = fp8.quantize_rows(inputs.bf16_to_f32(kp), KS)
    vc = fp8.quantize_rows(inputs.bf16_to_f32(vp), VS)
    torch.cuda.synchronize()
    return k8, v8, kc, vc, rtt


def _decode_fp8_full(g, dev, prob, k8, v8):
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    B = len(prob.dec_req_idx)
    buf, info = rx.rx_decode_plan_build(prob.req_to_token, prob.dec_req_idx, prob.dec_seq_len, prob.hq, prob.hkv)
    plan = rx.plan_to_device(buf, info, B)
    max_len = int(prob.dec_seq_len.max())
    ws = torch.empty(max(rx.rx_attn_decode_workspace(B, prob.hq, prob.hkv, prob.d, max_len, plan), 256),
                     dtype=torch.uint8, device="cuda")
    q = g.to_dev(prob.q_dec)
    og, lg = g.Guarded(q.shape, torch.bfloat16), g.Guarded((B, prob.hq), torch.float32)
    rx.rx_attn_decode_fp8(k8, v8, KS, VS, q, og.t, lg.t, g.i32(prob.dec_req_idx), g.i32(prob.dec_seq_len),
                          dev.rtt, max_len, prob.sm_scale, plan, ws, dev.status)
    torch.cuda.synchronize()
    og.check("fp8 decode o")
    lg.check("fp8 decode lse")
    return og.t.float().cpu().numpy(), lg.t.cpu().numpy()


def _extend_fp8_full(g, dev, prob, k8, v8):
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    B = len(prob.ext_req_idx)
    ctx = int((prob.ext_prefix_len + prob.ext_extend_len).sum())
    ws = torch.empty(rx.rx_attn_extend_workspace(ctx, B, prob.hkv, prob.d), dtype=torch.uint8, device="cuda")
    q = g.to_dev(prob.q_ext)
    og, lg = g.Guarded(q.shape, torch.bfloat16), g.Guarded(tuple(q.shape[:2]), torch.float32)
    rx.rx_attn_extend_fp8(k8, v8, KS, VS, q, og.t, lg.t, g.i32(prob.qo_indptr), g.i32(prob.ext_req_idx),
                          g.i32(prob.ext_prefix_len), g.i32(prob.ext_extend_len), dev.rtt,
                          int(prob.ext_extend_len.max()), prob.sm_scale, ws, dev.status)
    torch.cuda.synchronize()
    og.check("fp8 extend o")
    lg.check("fp8 extend lse")
    return og.t.float().cpu().numpy(), lg.t.cpu().numpy()


def _check_fp8_decode_rows(g, prob, kc, vc, rtt, o, lse, rows):
    from oracle import fp8
    ro, rl = fp8.attention(prob.q_dec[rows], kc, vc, KS, VS, rtt, prob.dec_req_idx[rows],
                           np.zeros(len(rows), np.int32), prob.dec_seq_len[rows], prob.sm_scale)
    g.compare(o[rows], ro, f"{prob.name} fp8 decode")
    g.compare_lse(lse[rows], rl, f"{prob.name} fp8 decode")


def _check_fp8_extend_rows(g, prob, kc, vc, rtt, o, lse, rng):
    from oracle import fp8
    rows, kend, rtt_row = _extend_rows(rng, prob)
    ro, rl = fp8.attention(prob.q_ext[rows], kc, vc, KS, VS, rtt, rtt_row, np.zeros(len(rows), np.int32), kend,
                           prob.sm_scale)
    g.compare(o[rows], ro, f"{prob.name} fp8 extend")
    g.compare_lse(lse[rows], rl, f"{prob.name} fp8 extend")


@pytest.mark.parametrize("name", ["few_shot_decode", "tree_of_thought_decode"])
def test_decode_full_size_fp8(name):
    """Few-shot (MHA: per-head and one-q-head FP8 kernels) and tree of
    thought (GQA FP8 kernel) at full size over code pools."""
    g = _gpu()
    prob = inputs.FULL_SIZE[name]()
    dev = g.Dev(prob)
    dev.kv_store()
    k8, v8, kc, vc, rtt = _fp8_setup(g, dev, prob)
    o, lse = _decode_fp8_full(g, dev, prob, k8, v8)
    assert dev.status_word() == 0
    B = len(prob.dec_req_idx)
    _check_fp8_decode_rows(g, prob, kc, vc, rtt, o, lse, _pick(np.random.default_rng(21), B, 24, must=(0, B - 1)))


def test_full_size_fp8_extend_and_mixed_chat():
    """The cached-prefix extend and the long multi-turn chat batch (decode and
    extend rows) over code pools at full size."""
    g = _gpu()
    prob = inputs.cached_prefix_extend()
    dev = g.Dev(prob)
    dev.kv_store()
    k8, v8, kc, vc, rtt = _fp8_setup(g, dev, prob)
    o, lse = _extend_fp8_full(g, dev, prob, k8, v8)
    assert dev.status_word() == 0
    _check_fp8_extend_rows(g, prob, kc, vc, rtt, o, lse, np.random.default_rng(22))
    del dev, k8, v8
    prob = admission.mixed_chat()
    dev = g.Dev(prob)
    dev.kv_store()
    k8, v8, kc, vc, rtt = _fp8_setup(g, dev, prob)
    o_e, lse_e = _extend_fp8_full(g, dev, prob, k8, v8)
    o_d, lse_d = _decode_fp8_full(g, dev, prob, k8, v8)
    assert dev.status_word() == 0
    _check_fp8_decode_rows(g, prob, kc, vc, rtt, o_d, lse_d, np.arange(len(prob.dec_req_idx)))
    _check_fp8_extend_rows(g, prob, kc, vc, rtt, o_e, lse_e, np.random.default_rng(23))
