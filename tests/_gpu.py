"""Helpers for the GPU parity tests: upload a Problem, run the C-ABI entry
points, build the oracle's pools, compare.

Tolerance (bf16 outputs): both readings of "max |err| <= 2e-2 absolute and
1e-2 relative" hold -- the allclose bound |gpu - oracle| <= 2e-2 + 1e-2 *
|oracle| per element, and the stricter max |gpu - oracle| <= 2e-2 over every
element; lse within 1e-3 absolute (fp32 sums in the kernel, fp64 in the
oracle).
"""
import numpy as np
import torch

import oracle
from prefix_shared_kv_radixattention_gb300 import binding as rx
from prefix_shared_kv_radixattention_gb300 import inputs

ATOL, RTOL, LSE_ATOL = 2e-2, 1e-2, 1e-3
FILL = 64.0  # unused pool rows hold this, so a wrong read shows

# Output canaries: every output tensor is the middle of a larger buffer whose
# every element -- the output's own included -- starts as a NaN bit pattern.
# After the call the regions before and after the output must still hold it
# bit for bit (no write out of bounds), and an output element the call did
# not write stays NaN, which no comparison with the oracle passes.
GUARD = 4096                      # canary elements on each side
CANARY_BF16 = -0x003F             # 0xFFC1: a bf16 NaN (exponent all ones)
CANARY_F32 = 0x7FC0DEAD           # an fp32 NaN


class Guarded:
    """An output tensor of `shape` inside canary-filled guard regions."""

    def __init__(self, shape, dtype, device="cuda"):
        self.n = int(np.prod(shape))
        self.dtype = dtype
        bits = torch.int16 if dtype == torch.bfloat16 else torch.int32
        fill = CANARY_BF16 if dtype == torch.bfloat16 else CANARY_F32
        self.buf = torch.full((self.n + 2 * GUARD,), fill, dtype=bits, device=device).view(dtype)
        self.fill, self.bits = fill, bits
        self.t = self.buf[GUARD:GUARD + self.n].view(shape)

    def check(self, what=""):
        raw = self.buf.view(self.bits).cpu().numpy()
        head, tail = raw[:GUARD], raw[GUARD + self.n:]
        assert (head == self.fill).all() and (tail == self.fill).all(), f"{what}: write outside the output"


def to_dev(a_u16: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a_u16).view(np.int16)).view(torch.bfloat16).cuda()


def to_host_u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def i32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


class Dev:
    """A Problem on the device: pools with cached rows placed, index arrays."""

    def __init__(self, prob: inputs.Problem, host_pools: bool = None, seed: int = 7):
        self.prob = prob
        S, hkv, d = prob.num_slots, prob.hkv, prob.d
        if host_pools is None:
            host_pools = S * hkv * d <= (1 << 24)
        self.host_pools = host_pools
        if host_pools:
            rng = np.random.default_rng(seed)
            kp = inputs.randn_bf16(rng, (S, hkv, d))
            vp = inputs.randn_bf16(rng, (S, hkv, d))
            kp[prob.cached_slots] = prob.cached_k
            vp[prob.cached_slots] = prob.cached_v
            self.kp_host, self.vp_host = kp, vp
            self.k_pool, self.v_pool = to_dev(kp), to_dev(vp)
        else:
            self.k_pool = torch.full((S, hkv, d), FILL, dtype=torch.bfloat16, device="cuda")
            self.v_pool = torch.full((S, hkv, d), FILL, dtype=torch.bfloat16, device="cuda")
            idx = torch.from_numpy(prob.cached_slots.astype(np.int64)).cuda()
            for pool, src in ((self.k_pool, prob.cached_k), (self.v_pool, prob.cached_v)):
                for s in range(0, len(idx), 1 << 16):
                    pool.index_copy_(0, idx[s:s + (1 << 16)], to_dev(src[s:s + (1 << 16)]))
        self.rtt = i32(prob.req_to_token)
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")

    # -- the path ------------------------------------------------------------
    def kv_store(self):
        p = self.prob
        rx.rx_kv_store(self.k_pool, self.v_pool, to_dev(p.new_k), to_dev(p.new_v), i32(p.new_slots),
                       self.status)

    def decode(self, plan: bool, kv_chunk: int = 0, min_shared: int = 16, with_lse: bool = True,
               plan_seq_len=None, seq_len=None):
        """Decode through the C ABI.  plan_seq_len: the lengths the plan is
        built for (default: the problem's); seq_len: the lengths the device
        call sees (default: the problem's)."""
        p = self.prob
        B = len(p.dec_req_idx)
        q = to_dev(p.q_dec)
        og = Guarded(q.shape, torch.bfloat16)
        lg = Guarded((B, p.hq), torch.float32) if with_lse else None
        o, lse = og.t, (lg.t if with_lse else None)
        dp = None
        if plan:
            lens = p.dec_seq_len if plan_seq_len is None else np.asarray(plan_seq_len, np.int32)
            buf, info = rx.rx_decode_plan_build(p.req_to_token, p.dec_req_idx, lens, p.hq,
                                                p.hkv, kv_chunk, min_shared)
            dp = rx.plan_to_device(buf, info, B)
        dev_len = p.dec_seq_len if seq_len is None else np.asarray(seq_len, np.int32)
        max_len = min(int(dev_len.max()), p.rtt_stride)
        ws_bytes = rx.rx_attn_decode_workspace(B, p.hq, p.hkv, p.d, max_len, dp)
        ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
        rx.rx_attn_decode(self.k_pool, self.v_pool, q, o, lse, i32(p.dec_req_idx), i32(dev_len),
                          self.rtt, max_len, p.sm_scale, dp, ws if ws_bytes else None, self.status)
        torch.cuda.synchronize()
        og.check("decode o")
        if with_lse:
            lg.check("decode lse")
        return o.float().cpu().numpy(), (lse.cpu().numpy() if with_lse else None)

    def extend(self, with_lse: bool = True, staged: bool = False, ws_rows=None):
        """Extend through the C ABI; staged=True passes a workspace sized for
        the problem's contexts (or for ws_rows context tokens)."""
        p = self.prob
        q = to_dev(p.q_ext)
        og = Guarded(q.shape, torch.bfloat16)
        lg = Guarded((q.shape[0], p.hq), torch.float32) if with_lse else None
        o, lse = og.t, (lg.t if with_lse else None)
        ws = None
        if staged:
            rows = int((p.ext_prefix_len + p.ext_extend_len).sum()) if ws_rows is None else int(ws_rows)
            nb = rx.rx_attn_extend_workspace(rows, len(p.ext_req_idx), p.hkv, p.d)
            ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
        rx.rx_attn_extend(self.k_pool, self.v_pool, q, o, lse, i32(p.qo_indptr), i32(p.ext_req_idx),
                          i32(p.ext_prefix_len), i32(p.ext_extend_len), self.rtt,
                          int(p.ext_extend_len.max()), p.sm_scale, self.status, workspace=ws)
        torch.cuda.synchronize()
        og.check("extend o")
        if with_lse:
            lg.check("extend lse")
        return o.float().cpu().numpy(), (lse.cpu().numpy() if with_lse else None)

    def status_word(self) -> int:
        return int(self.status.item())

    # -- the oracle's view ---------------------------------------------------
    def oracle_pools(self, rows=None):
        """Host pools after the step's KV store, and the matching req_to_token.

        Small pools: the full host pools plus the oracle's own kv_store.  Big
        pools: a compact pool of the cached rows (in the order they were
        drawn) and the new rows, placed by the oracle's kv_store, with
        req_to_token renamed to those rows (the slot-permutation invariance
        makes the renaming exact)."""
        p = self.prob
        if self.host_pools:
            kp, vp = self.kp_host.copy(), self.vp_host.copy()
            oracle.kv_store(kp, vp, p.new_k, p.new_v, p.new_slots)
            return kp, vp, p.req_to_token
        S = p.num_slots
        row_of = np.full(S, -1, np.int64)
        nc = len(p.cached_slots)
        row_of[p.cached_slots] = np.arange(nc)
        fresh = p.new_slots[row_of[p.new_slots] < 0]
        row_of[fresh] = nc + np.arange(len(fresh))
        kp = np.zeros((nc + len(fresh), p.hkv, p.d), np.uint16)
        vp = np.zeros_like(kp)
        kp[:nc], vp[:nc] = p.cached_k, p.cached_v
        oracle.kv_store(kp, vp, p.new_k, p.new_v, row_of[p.new_slots].astype(np.int32))
        rtt = p.req_to_token
        ok = (rtt >= 0) & (rtt < S)
        return kp, vp, np.where(ok, row_of[np.where(ok, rtt, 0)], -1).astype(np.int32)


def compare(gpu, ref, what=""):
    gpu = np.asarray(gpu, np.float64)
    err = np.abs(gpu - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    assert not np.isnan(gpu).any(), f"{what}: NaN in GPU output"
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; "
                           f"max abs err {err.max():.3e}")
    assert err.max() <= ATOL, f"{what}: max abs err {err.max():.3e} above {ATOL}"
    return float(err.max())


def compare_lse(gpu, ref, what=""):
    err = np.abs(np.asarray(gpu, np.float64) - ref)
    assert err.max() <= LSE_ATOL, f"{what}: lse max abs err {err.max():.3e}"
    return float(err.max())
