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
