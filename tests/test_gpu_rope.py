"""GPU parity of the rotary position embedding (rx_rope, rx_kv_store_rope)
against the oracle's fp64 definition, and of a two-layer pool: stores and
attention on one layer leave the other alone.  Tolerance as in tests/_gpu.py
(the GPU rounds its fp32 rotation to bf16)."""
import numpy as np
import pytest

import oracle
from prefix_shared_kv_radixattention_gb300 import inputs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _g():
    from tests import _gpu
    return _gpu


def _positions(rng, n):
    """Positions of a long context, plus the ends of the int32 range: the
    angle is reduced exactly modulo 2 pi at any position, so rows at 10^7,
    2^31 - 1 and negative positions must match the fp64 definition too."""
    pos = rng.integers(0, 40000, size=n).astype(np.int32)
    pos[0] = 0
    pos[-1] = 32767
    pos[1:5] = [10_000_000, 2**31 - 1, -7, -(2**31)]
    return pos


@pytest.mark.parametrize("heads,d,base", [(4, 64, 10000.0), (32, 128, 10000.0), (8, 128, 500000.0)])
def test_rope_matches_oracle(heads, d, base):
    g = _g()
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    rng = np.random.default_rng(heads + d)
    n = 97
    x = inputs.randn_bf16(rng, (n, heads, d))
    pos = _positions(rng, n)
    xd = g.to_dev(x)
    rx.rx_rope(xd, g.i32(pos), base)
    got = xd.float().cpu().numpy()
    g.compare(got, oracle.rope(x, pos, base), f"rope {heads}x{d}")
    # position 0 rows are unchanged bit for bit
    assert np.array_equal(g.to_host_u16(xd)[0], x[0])


def test_rope_empty_is_noop():
    g = _g()
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    x = torch.zeros((0, 4, 64), dtype=torch.bfloat16, device="cuda")
    rx.rx_rope(x, torch.zeros(0, dtype=torch.int32, device="cuda"), 10000.0)


@pytest.mark.parametrize("hkv,d", [(8, 128), (4, 64)])
def test_kv_store_rope(hkv, d):
    g = _g()
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    rng = np.random.default_rng(7 + hkv)
    S, n, base = 3000, 211, 10000.0
    kp = inputs.randn_bf16(rng, (S, hkv, d))
    vp = inputs.randn_bf16(rng, (S, hkv, d))
    k_new = inputs.randn_bf16(rng, (n, hkv, d))
    v_new = inputs.randn_bf16(rng, (n, hkv, d))
    slots = rng.permutation(S)[:n].astype(np.int32)
    pos = _positions(rng, n)
    kd, vd = g.to_dev(kp), g.to_dev(vp)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rx.rx_kv_store_rope(kd, vd, g.to_dev(k_new), g.to_dev(v_new), g.i32(slots), g.i32(pos), base, status)
    assert int(status.item()) == 0
    k_got, v_got = g.to_host_u16(kd), g.to_host_u16(vd)
    g.compare(inputs.bf16_to_f32(k_got[slots]), oracle.rope(k_new, pos, base), "stored K")
    assert np.array_equal(v_got[slots], v_new)
    rest = np.setdiff1d(np.arange(S), slots)
    assert np.array_equal(k_got[rest], kp[rest]) and np.array_equal(v_got[rest], vp[rest])


@pytest.mark.parametrize("hkv,d,ks,vs", [(8, 128, 0.5, 2.0), (4, 64, 1.0, 1.0)])
def test_kv_store_rope_fp8_is_the_rope_store_then_the_fp8_store(hkv, d, ks, vs):
    """The rotary FP8 scatter stores, bit for bit, the codes rx_kv_store_fp8
    makes of the rows rx_kv_store_rope writes to a bf16 pool; other rows and
    bad slots are left alone."""
    g = _g()
    from oracle import fp8
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    rng = np.random.default_rng(19 + hkv)
    S, n, base = 3000, 211, 500000.0
    k_new = inputs.randn_bf16(rng, (n, hkv, d))
    v_new = inputs.randn_bf16(rng, (n, hkv, d))
    slots = rng.permutation(S)[:n].astype(np.int32)
    pos = _positions(rng, n)
    kb = g.to_dev(np.zeros((S, hkv, d), np.uint16))
    vb = g.to_dev(np.zeros((S, hkv, d), np.uint16))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rx.rx_kv_store_rope(kb, vb, g.to_dev(k_new), g.to_dev(v_new), g.i32(slots), g.i32(pos), base, status)
    init = rng.integers(0, 256, size=(S, hkv, d), dtype=np.uint8)
    k8, v8 = torch.from_numpy(init.copy()).cuda(), torch.from_numpy(init.copy()).cuda()
    rx.rx_kv_store_rope_fp8(k8, v8, ks, vs, g.to_dev(k_new), g.to_dev(v_new), g.i32(slots), g.i32(pos), base,
                            status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rotated = g.to_host_u16(kb)[slots]
    got_k, got_v = k8.cpu().numpy(), v8.cpu().numpy()
    assert np.array_equal(got_k[slots], fp8.quantize_rows(inputs.bf16_to_f32(rotated), ks))
    assert np.array_equal(got_v[slots], fp8.quantize_rows(inputs.bf16_to_f32(v_new), vs))
    rest = np.setdiff1d(np.arange(S), slots)
    assert np.array_equal(got_k[rest], init[rest]) and np.array_equal(got_v[rest], init[rest])


def test_kv_store_rope_bad_slot_is_flagged():
    g = _g()
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    rng = np.random.default_rng(3)
    S, hkv, d = 64, 2, 64
    kp = inputs.randn_bf16(rng, (S, hkv, d))
    kd, vd = g.to_dev(kp), g.to_dev(kp)
    k_new = inputs.randn_bf16(rng, (3, hkv, d))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rx.rx_kv_store_rope(kd, vd, g.to_dev(k_new), g.to_dev(k_new), g.i32([5, S + 2, -1]), g.i32([1, 2, 3]),
                        10000.0, status)
    assert int(status.item()) & rx.RX_DEV_BAD_SLOT
    got = g.to_host_u16(kd)
    assert np.array_equal(np.delete(got, 5, axis=0), np.delete(kp, 5, axis=0))


def test_two_layer_pool_store_and_decode():
    """Layer 1 of a [2, S, Hkv, d] pool: rotated K/V stored there, decode
    attention with rotated q over it; layer 0 is untouched.  The oracle
    rotates the same bf16 inputs in fp64 and rounds them to bf16 itself."""
    g = _g()
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    rng = np.random.default_rng(11)
    L, S, hq, hkv, d, base = 2, 1024, 16, 4, 128, 10000.0
    B, ctx = 3, 300
    pool_k = inputs.randn_bf16(rng, (L, S, hkv, d))
    pool_v = inputs.randn_bf16(rng, (L, S, hkv, d))
    k_new = inputs.randn_bf16(rng, (B * ctx, hkv, d))
    v_new = inputs.randn_bf16(rng, (B * ctx, hkv, d))
    q = inputs.randn_bf16(rng, (B, hq, d))
    slots = rng.permutation(S)[:B * ctx].astype(np.int32)
    rtt = slots.reshape(B, ctx).copy()
    pos_kv = np.tile(np.arange(ctx, dtype=np.int32), B)
    pos_q = np.full(B, ctx - 1, np.int32)
    kd, vd = g.to_dev(pool_k), g.to_dev(pool_v)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rx.rx_kv_store_rope(kd[1], vd[1], g.to_dev(k_new), g.to_dev(v_new), g.i32(slots), g.i32(pos_kv), base, status)
    qd = g.to_dev(q)
    rx.rx_rope(qd, g.i32(pos_q), base)
    o = torch.empty_like(qd)
    lse = torch.empty((B, hq), dtype=torch.float32, device="cuda")
    ws_bytes = rx.rx_attn_decode_workspace(B, hq, hkv, d, ctx, None)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    rx.rx_attn_decode(kd[1], vd[1], qd, o, lse, g.i32(np.arange(B)), g.i32(np.full(B, ctx)), g.i32(rtt), ctx,
                      1.0 / np.sqrt(d), None, ws if ws_bytes else None, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(g.to_host_u16(kd[0]), pool_k[0]) and np.array_equal(g.to_host_u16(vd[0]), pool_v[0])
    # the oracle: rotated, rounded bf16 rows in its own pools, then attention
    ok, ov = pool_k[1].copy(), pool_v[1].copy()
    ok[slots] = inputs.bf16_round(oracle.rope(k_new, pos_kv, base).astype(np.float32))
    ov[slots] = v_new
    oq = inputs.bf16_round(oracle.rope(q, pos_q, base).astype(np.float32))
    ro, rl = oracle.decode(oq, ok, ov, rtt, np.arange(B, dtype=np.int32), np.full(B, ctx, np.int32),
                           1.0 / np.sqrt(d))
    g.compare(o.float().cpu().numpy(), ro, "decode on layer 1")
    g.compare_lse(lse.cpu().numpy(), rl, "decode on layer 1")
