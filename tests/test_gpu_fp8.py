"""GPU parity of the FP8 (E4M3) slot scatter (rx_kv_store_fp8) with the
oracle's quantizer (oracle/fp8.py), bit for bit: the same correctly rounded
fp32 division by the pool scale, then round to nearest even with
saturation."""
import numpy as np
import pytest

from oracle import fp8
from prefix_shared_kv_radixattention_gb300 import inputs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _rows(rng, n, hkv, d):
    """bf16 rows spanning E4M3's range: N(0, 1), large values that
    saturate, tiny ones that land on subnormals, and exact midpoints."""
    x = rng.standard_normal((n, hkv, d)).astype(np.float32)
    x[0::5] *= 900.0
    x[1::5] *= 1e-3
    x[2, 0, :4] = [1.0625, 1.1875, 200.0, -200.0]   # ties to even at scale 1 / 2
    return inputs.bf16_round(x)


@pytest.mark.parametrize("hkv,d,k_scale,v_scale", [(8, 128, 1.0, 0.5), (32, 128, 0.25, 2.0), (4, 64, 1.0, 1.0)])
def test_store_fp8_matches_oracle(hkv, d, k_scale, v_scale):
    from tests import _gpu as g
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    rng = np.random.default_rng(hkv * 7 + d)
    S, n = 2000, 301
    kp = rng.integers(0, 256, size=(S, hkv, d), dtype=np.uint8)
    vp = rng.integers(0, 256, size=(S, hkv, d), dtype=np.uint8)
    k_new, v_new = _rows(rng, n, hkv, d), _rows(rng, n, hkv, d)
    slots = rng.permutation(S)[:n].astype(np.int32)
    kd, vd = torch.from_numpy(kp).cuda(), torch.from_numpy(vp).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rx.rx_kv_store_fp8(kd, vd, k_scale, v_scale, g.to_dev(k_new), g.to_dev(v_new), g.i32(slots), status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    kg, vg = kd.cpu().numpy(), vd.cpu().numpy()
    want_k = fp8.quantize_rows(inputs.bf16_to_f32(k_new), k_scale)
    want_v = fp8.quantize_rows(inputs.bf16_to_f32(v_new), v_scale)
    assert np.array_equal(kg[slots], want_k) and np.array_equal(vg[slots], want_v)
    rest = np.setdiff1d(np.arange(S), slots)
    assert np.array_equal(kg[rest], kp[rest]) and np.array_equal(vg[rest], vp[rest])


def test_store_fp8_bad_slot_is_flagged():
    from tests import _gpu as g
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    rng = np.random.default_rng(9)
    S, hkv, d = 64, 2, 64
    kp = np.zeros((S, hkv, d), np.uint8)
    kd, vd = torch.from_numpy(kp).cuda(), torch.from_numpy(kp.copy()).cuda()
    rows = _rows(rng, 3, hkv, d)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rx.rx_kv_store_fp8(kd, vd, 1.0, 1.0, g.to_dev(rows), g.to_dev(rows), g.i32([5, S + 3, -1]), status)
    torch.cuda.synchronize()
    assert int(status.item()) & rx.RX_DEV_BAD_SLOT
    got = kd.cpu().numpy()
    assert np.array_equal(got[5], fp8.quantize_rows(inputs.bf16_to_f32(rows[0]), 1.0))
    assert not np.delete(got, 5, axis=0).any()


# ---------------------------------------------------------------------------
# decode over FP8 pools (rx_attn_decode_fp8)
# ---------------------------------------------------------------------------


def _fp8_problem(prob, k_scale, v_scale, seed):
    """Host code pools: every row the oracle's quantizer makes of N(0, 1)
    bf16 values (the cached rows here, the step's new rows as the store
    must); the device pools get the cached codes uploaded and the new rows
    through rx_kv_store_fp8."""
    from tests import _gpu as g
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    rng = np.random.default_rng(seed)
    S, hkv, d = prob.num_slots, prob.hkv, prob.d
    kc = fp8.quantize_rows(inputs.bf16_to_f32(inputs.randn_bf16(rng, (S, hkv, d))), k_scale)
    vc = fp8.quantize_rows(inputs.bf16_to_f32(inputs.randn_bf16(rng, (S, hkv, d))), v_scale)
    kd, vd = torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rx.rx_kv_store_fp8(kd, vd, k_scale, v_scale, g.to_dev(prob.new_k), g.to_dev(prob.new_v), g.i32(prob.new_slots),
                       status)
    kc[prob.new_slots] = fp8.quantize_rows(inputs.bf16_to_f32(prob.new_k), k_scale)
    vc[prob.new_slots] = fp8.quantize_rows(inputs.bf16_to_f32(prob.new_v), v_scale)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(kd.cpu().numpy(), kc) and np.array_equal(vd.cpu().numpy(), vc)
    return kd, vd, kc, vc, status


def _decode_fp8(prob, kd, vd, ks, vs, status, kv_chunk=0, plan_len=None, use_plan=True, bf16_pools=None):
    """Decode over the code pools (or, with bf16_pools = (k, v), the bf16
    path over those pools with the same plan) -> (o, lse, plan info)."""
    from tests import _gpu as g
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    B = len(prob.dec_req_idx)
    lens = prob.dec_seq_len if plan_len is None else plan_len
    plan, info = None, None
    if use_plan:
        buf, info = rx.rx_decode_plan_build(prob.req_to_token, prob.dec_req_idx, lens, prob.hq, prob.hkv,
                                            kv_chunk, 16)
        plan = rx.plan_to_device(buf, info, B)
    max_len = int(prob.dec_seq_len.max())
    ws = torch.empty(max(rx.rx_attn_decode_workspace(B, prob.hq, prob.hkv, prob.d, max_len, plan), 256),
                     dtype=torch.uint8, device="cuda")
    q = g.to_dev(prob.q_dec)
    og, lg = g.Guarded(q.shape, torch.bfloat16), g.Guarded((B, prob.hq), torch.float32)
    o, lse = og.t, lg.t
    if bf16_pools is None:
        rx.rx_attn_decode_fp8(kd, vd, ks, vs, q, o, lse, g.i32(prob.dec_req_idx), g.i32(prob.dec_seq_len),
                              g.i32(prob.req_to_token), max_len, prob.sm_scale, plan, ws, status)
    else:
        rx.rx_attn_decode(bf16_pools[0], bf16_pools[1], q, o, lse, g.i32(prob.dec_req_idx), g.i32(prob.dec_seq_len),
                          g.i32(prob.req_to_token), max_len, prob.sm_scale, plan, ws, status)
    torch.cuda.synchronize()
    og.check("fp8 decode o")
    lg.check("fp8 decode lse")
    return o.float().cpu().numpy(), lse.cpu().numpy(), info


@pytest.mark.parametrize("hq,d,ks,vs", [(16, 128, 1.0, 1.0), (32, 128, 0.37, 2.5), (64, 128, 1.5, 0.25),
                                        (128, 64, 0.5, 1.0), (32, 64, 2.0, 0.75)])
def test_decode_fp8_ragged_matches_oracle(hq, d, ks, vs):
    """Ragged batches with shared prefixes, 8 kv heads, G = 2 .. 16: grouped
    shared segments and single-request pieces, split rows merged."""
    from tests import _gpu as g
    prob = inputs.ragged(500 + hq + d, hq=hq, hkv=8, d=d, n_groups=3, per_group=3, shared_max=400,
                         private_max=300, extend_max=1, decode=True, num_slots=6000)
    kd, vd, kc, vc, status = _fp8_problem(prob, ks, vs, hq + d)
    for chunk in (64, 0):
        o, lse, info = _decode_fp8(prob, kd, vd, ks, vs, status, kv_chunk=chunk)
        ro, rl = fp8.decode_rows(prob.q_dec, kc, vc, ks, vs, prob.req_to_token, prob.dec_req_idx, prob.dec_seq_len,
                                 prob.sm_scale)
        g.compare(o, ro, f"fp8 decode G={hq // 8} d={d} chunk {chunk}")
        g.compare_lse(lse, rl, f"fp8 decode G={hq // 8} d={d} chunk {chunk}")
    assert int(status.item()) == 0


@pytest.mark.parametrize("shape", ["few_shot", "tree_of_thought"])
def test_decode_fp8_workload_shapes(shape):
    """The few-shot structure (one prefix shared by every request, long
    private parts) and the tree-of-thought one (nested shared segments),
    with GQA 32/8 heads; the plan built a token earlier serves the step."""
    from tests import _gpu as g
    if shape == "few_shot":
        prob = inputs.few_shot_decode(hq=32, hkv=8, d=128, batch=24, shared=512, private=200, num_slots=40000)
    else:
        prob = inputs.tree_of_thought_decode(depth=3, fanout=3, edge=120, num_slots=40000)
    kd, vd, kc, vc, status = _fp8_problem(prob, 0.8, 1.25, 17)
    for plan_len in (None, prob.dec_seq_len - 1):
        o, lse, info = _decode_fp8(prob, kd, vd, 0.8, 1.25, status, plan_len=plan_len)
        assert info.n_segments > 0 and info.n_wide == info.n_items
        ro, rl = fp8.decode_rows(prob.q_dec, kc, vc, 0.8, 1.25, prob.req_to_token, prob.dec_req_idx,
                                 prob.dec_seq_len, prob.sm_scale)
        g.compare(o, ro, f"fp8 decode {shape}")
        g.compare_lse(lse, rl, f"fp8 decode {shape}")
    assert int(status.item()) == 0


def _mha_shapes():
    return {
        # one prefix shared by every request (per-head kernel, FP8 copiers),
        # private pieces on the one-q-head all-heads kernel
        "few-shot MHA 32x128": lambda: inputs.few_shot_decode(hq=32, hkv=32, d=128, batch=12, shared=300,
                                                              private=150, num_slots=8000),
        "few-shot MHA 8x64": lambda: inputs.few_shot_decode(hq=8, hkv=8, d=64, batch=9, shared=200,
                                                            private=90, num_slots=4000),
        # G = 2 over 4 kv heads: the per-head kernel takes every item
        "ragged G=2": lambda: inputs.ragged(733, hq=8, hkv=4, d=128, n_groups=3, per_group=4, shared_max=300,
                                            private_max=200, extend_max=1, decode=True, num_slots=6000),
        # a prefix shared by 20 groups of 4: per-head FP8 items beside GQA FP8 ones
        "wide-shared GQA": lambda: inputs.few_shot_decode(hq=32, hkv=8, d=128, batch=80, shared=256,
                                                          private=70, num_slots=20000),
    }


@pytest.mark.parametrize("name", list(_mha_shapes()))
def test_decode_fp8_all_layouts_match_oracle(name):
    """FP8 decode on the layouts beyond 8 kv heads' all-heads kernel: one q
    head per kv head, G = 2 over 4 kv heads, a segment too widely shared for
    request groups; with and without a plan, against the oracle."""
    from tests import _gpu as g
    prob = _mha_shapes()[name]()
    kd, vd, kc, vc, status = _fp8_problem(prob, 0.6, 1.7, 29)
    ro, rl = fp8.decode_rows(prob.q_dec, kc, vc, 0.6, 1.7, prob.req_to_token, prob.dec_req_idx, prob.dec_seq_len,
                             prob.sm_scale)
    for use_plan in (True, False):
        o, lse, info = _decode_fp8(prob, kd, vd, 0.6, 1.7, status, use_plan=use_plan)
        g.compare(o, ro, f"fp8 decode {name} plan={use_plan}")
        g.compare_lse(lse, rl, f"fp8 decode {name} plan={use_plan}")
        if use_plan and name != "ragged G=2":
            assert info.n_items > info.n_wide > 0   # both kernels ran
    assert int(status.item()) == 0


@pytest.mark.parametrize("name", ["few-shot MHA 32x128", "few-shot MHA 8x64", "ragged G=2"])
def test_decode_fp8_unit_scales_equal_bf16_pool_bitwise(name):
    """Where the FP8 kernels widen codes exactly into the bf16 kernels'
    arithmetic (the per-head kernel's tiles, the one-q-head all-heads
    kernel's floats), unit scales give rx_attn_decode's result on a pool of
    the decoded values, bit for bit."""
    from tests import _gpu as g
    prob = _mha_shapes()[name]()
    kd, vd, kc, vc, status = _fp8_problem(prob, 1.0, 1.0, 31)
    pools = (g.to_dev(fp8.bf16_bits(kc)), g.to_dev(fp8.bf16_bits(vc)))
    for use_plan in (True, False):
        o8, l8, _ = _decode_fp8(prob, kd, vd, 1.0, 1.0, status, use_plan=use_plan)
        ob, lb, _ = _decode_fp8(prob, kd, vd, 1.0, 1.0, status, use_plan=use_plan, bf16_pools=pools)
        assert np.array_equal(o8.view(np.uint32), ob.view(np.uint32)), (name, use_plan)
        assert np.array_equal(l8.view(np.uint32), lb.view(np.uint32)), (name, use_plan)
    assert int(status.item()) == 0


def test_decode_fp8_bad_slot_is_flagged():
    from tests import _gpu as g
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    prob = inputs.few_shot_decode(hq=32, hkv=8, d=128, batch=5, shared=60, private=40, num_slots=1024)
    prob.req_to_token = prob.req_to_token.copy()
    prob.req_to_token[3, 80] = prob.num_slots + 9
    kd, vd, kc, vc, status = _fp8_problem(prob, 1.0, 1.0, 3)
    o, _, _ = _decode_fp8(prob, kd, vd, 1.0, 1.0, status, kv_chunk=64)
    assert int(status.item()) & rx.RX_DEV_BAD_SLOT
    assert np.isfinite(o).all()


# ---------------------------------------------------------------------------
# extend over FP8 pools (rx_attn_extend_fp8)
# ---------------------------------------------------------------------------


def _extend_fp8(prob, kd, vd, ks, vs, status, staged=True):
    from tests import _gpu as g
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    B = len(prob.ext_req_idx)
    ctx = int((prob.ext_prefix_len + prob.ext_extend_len).sum())
    ws = torch.empty(rx.rx_attn_extend_workspace(ctx, B, prob.hkv, prob.d), dtype=torch.uint8,
                     device="cuda") if staged else None
    q = g.to_dev(prob.q_ext)
    og, lg = g.Guarded(q.shape, torch.bfloat16), g.Guarded(tuple(q.shape[:2]), torch.float32)
    o, lse = og.t, lg.t
    rx.rx_attn_extend_fp8(kd, vd, ks, vs, q, o, lse, g.i32(prob.qo_indptr), g.i32(prob.ext_req_idx),
                          g.i32(prob.ext_prefix_len), g.i32(prob.ext_extend_len), g.i32(prob.req_to_token),
                          int(prob.ext_extend_len.max()), prob.sm_scale, ws, status)
    torch.cuda.synchronize()
    og.check("fp8 extend o")
    lg.check("fp8 extend lse")
    return o, lse


def _extend_rows(prob):
    """Query rows of the extend pass for the attention oracle: new token i of
    request b reads its slot list's positions 0 .. prefix_len[b] + i."""
    q_row, kend = [], []
    for b, r in enumerate(prob.ext_req_idx):
        P, E = int(prob.ext_prefix_len[b]), int(prob.ext_extend_len[b])
        q_row += [int(r)] * E
        kend += list(range(P + 1, P + E + 1))
    n = len(q_row)
    return np.asarray(q_row, np.int32), np.zeros(n, np.int32), np.asarray(kend, np.int32)


def _extend_problems():
    return {
        "tiny": lambda: inputs.tiny_extend(),
        "ragged GQA": lambda: inputs.ragged(611, hq=32, hkv=8, d=128, n_groups=3, per_group=3, shared_max=300,
                                            private_max=200, extend_max=300, decode=False, num_slots=8000),
        "shared prefixes": lambda: inputs.cached_prefix_extend(hq=16, hkv=4, d=64, n_prefix=2, per_prefix=3,
                                                               prefix=384, extend=200, num_slots=6000),
    }


@pytest.mark.parametrize("name,ks,vs", [("tiny", 1.0, 1.0), ("ragged GQA", 0.37, 2.5),
                                        ("shared prefixes", 1.5, 0.25)])
def test_extend_fp8_matches_oracle(name, ks, vs):
    """Extend over E4M3 pools against the oracle's attention over decoded
    codes with the pools' scales: several tiles, ragged tails, and requests
    whose shared prefix tiles are staged once."""
    from tests import _gpu as g
    prob = _extend_problems()[name]()
    kd, vd, kc, vc, status = _fp8_problem(prob, ks, vs, 41)
    o, lse = _extend_fp8(prob, kd, vd, ks, vs, status)
    assert int(status.item()) == 0
    q_row, kbeg, kend = _extend_rows(prob)
    ro, rl = fp8.attention(prob.q_ext, kc, vc, ks, vs, prob.req_to_token, q_row, kbeg, kend, prob.sm_scale)
    g.compare(o.float().cpu().numpy(), ro, f"fp8 extend {name}")
    g.compare_lse(lse.cpu().numpy(), rl, f"fp8 extend {name}")


@pytest.mark.parametrize("name,ks,vs", [("tiny", 0.8, 1.3), ("ragged GQA", 0.37, 2.5),
                                        ("shared prefixes", 1.5, 0.25)])
def test_extend_fp8_gather_path_equals_staged_bitwise(name, ks, vs):
    """Without a workspace the attention kernel's producer warps widen the
    code rows themselves: the same tiles, so the same result as the staged
    path bit for bit, and the oracle's."""
    from tests import _gpu as g
    prob = _extend_problems()[name]()
    kd, vd, kc, vc, status = _fp8_problem(prob, ks, vs, 47)
    o_s, l_s = _extend_fp8(prob, kd, vd, ks, vs, status, staged=True)
    o_g, l_g = _extend_fp8(prob, kd, vd, ks, vs, status, staged=False)
    assert int(status.item()) == 0
    assert np.array_equal(g.to_host_u16(o_g), g.to_host_u16(o_s))
    assert np.array_equal(l_g.cpu().numpy().view(np.uint32), l_s.cpu().numpy().view(np.uint32))
    q_row, kbeg, kend = _extend_rows(prob)
    ro, rl = fp8.attention(prob.q_ext, kc, vc, ks, vs, prob.req_to_token, q_row, kbeg, kend, prob.sm_scale)
    g.compare(o_g.float().cpu().numpy(), ro, f"fp8 extend gather {name}")
    g.compare_lse(l_g.cpu().numpy(), rl, f"fp8 extend gather {name}")


@pytest.mark.parametrize("name", ["ragged GQA", "shared prefixes"])
def test_extend_fp8_unit_scales_equal_bf16_pool_bitwise(name):
    """With both scales 1, extend over codes is rx_attn_extend over a bf16
    pool that holds the decoded codes, bit for bit: the staging copy widens
    codes exactly and the attention kernel is the same."""
    from tests import _gpu as g
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    prob = _extend_problems()[name]()
    kd, vd, kc, vc, status = _fp8_problem(prob, 1.0, 1.0, 43)
    o8, l8 = _extend_fp8(prob, kd, vd, 1.0, 1.0, status)
    kb, vb = g.to_dev(fp8.bf16_bits(kc)), g.to_dev(fp8.bf16_bits(vc))
    B = len(prob.ext_req_idx)
    ctx = int((prob.ext_prefix_len + prob.ext_extend_len).sum())
    ws = torch.empty(rx.rx_attn_extend_workspace(ctx, B, prob.hkv, prob.d), dtype=torch.uint8, device="cuda")
    q = g.to_dev(prob.q_ext)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    rx.rx_attn_extend(kb, vb, q, o, lse, g.i32(prob.qo_indptr), g.i32(prob.ext_req_idx), g.i32(prob.ext_prefix_len),
                      g.i32(prob.ext_extend_len), g.i32(prob.req_to_token), int(prob.ext_extend_len.max()),
                      prob.sm_scale, status, workspace=ws)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(g.to_host_u16(o8), g.to_host_u16(o))
    assert np.array_equal(l8.cpu().numpy().view(np.uint32), lse.cpu().numpy().view(np.uint32))


def test_extend_fp8_bad_slot_is_flagged():
    from tests import _gpu as g
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    prob = inputs.tiny_extend()
    prob.req_to_token = prob.req_to_token.copy()
    prob.req_to_token[int(prob.ext_req_idx[1]), 3] = prob.num_slots + 5
    kd, vd, kc, vc, status = _fp8_problem(prob, 1.0, 1.0, 5)
    o, _ = _extend_fp8(prob, kd, vd, 1.0, 1.0, status)
    assert int(status.item()) & rx.RX_DEV_BAD_SLOT
    assert torch.isfinite(o.float()).all()
