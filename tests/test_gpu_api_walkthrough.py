"""The public API as a serving loop drives it, step by step, checked against
the oracle: admit requests through the radix cache (shared prompt found
cached, LRU eviction when the pool runs short), store their new K/V rows,
extend, commit; then decode steps through one plan built for the batch.
The same walk is shown in README.md."""
import numpy as np
import pytest

import oracle
from prefix_shared_kv_radixattention_gb300 import inputs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


class HostPool:
    """The oracle's copy of the pool: bf16 bits, written where the GPU's is."""

    def __init__(self, S, hkv, d):
        self.k = np.zeros((S, hkv, d), np.uint16)
        self.v = np.zeros((S, hkv, d), np.uint16)

    def store(self, k_new, v_new, slots):
        oracle.kv_store(self.k, self.v, k_new, v_new, np.asarray(slots, np.int32))


def test_serving_loop_through_the_public_api():
    from tests import _gpu as g
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    rng = np.random.default_rng(4242)
    S, hq, hkv, d = 2048, 32, 8, 128
    scale = 1.0 / np.sqrt(d)
    k_pool = torch.zeros((S, hkv, d), dtype=torch.bfloat16, device="cuda")
    v_pool = torch.zeros_like(k_pool)
    host = HostPool(S, hkv, d)
    tree = rx.RadixTree()
    alloc = rx.SlotAllocator(rng.permutation(S).astype(np.int32), S)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def extend_batch(token_lists):
        """Admit, store, extend and commit a batch of prompts; returns the
        slot rows and prefix lengths the radix cache gave them."""
        rows, prefix = [], []
        for t in token_lists:
            row, k, _ = rx.rx_admit(tree, alloc, t)
            rows.append(row)
            prefix.append(k)
        ext = [len(t) - k for t, k in zip(token_lists, prefix)]
        new_slots = np.concatenate([r[k:] for r, k in zip(rows, prefix)]).astype(np.int32)
        k_new = inputs.randn_bf16(rng, (len(new_slots), hkv, d))
        v_new = inputs.randn_bf16(rng, (len(new_slots), hkv, d))
        rx.rx_kv_store(k_pool, v_pool, g.to_dev(k_new), g.to_dev(v_new), g.i32(new_slots), status)
        host.store(k_new, v_new, new_slots)
        stride = (max(len(t) for t in token_lists) + 15) // 16 * 16
        rtt = np.full((len(rows), stride), -1, np.int32)
        for i, r in enumerate(rows):
            rtt[i, :len(r)] = r
        qo = np.concatenate([[0], np.cumsum(ext)]).astype(np.int32)
        q = inputs.randn_bf16(rng, (int(qo[-1]), hq, d))
        o = torch.empty((int(qo[-1]), hq, d), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((int(qo[-1]), hq), dtype=torch.float32, device="cuda")
        req = np.arange(len(rows), dtype=np.int32)
        ws = torch.empty(rx.rx_attn_extend_workspace(int(sum(len(t) for t in token_lists)), len(rows), hkv, d),
                         dtype=torch.uint8, device="cuda")
        rx.rx_attn_extend(k_pool, v_pool, g.to_dev(q), o, lse, g.i32(qo), g.i32(req), g.i32(prefix),
                          g.i32(ext), g.i32(rtt), max(ext), scale, status, workspace=ws)
        torch.cuda.synchronize()
        ro, rl = oracle.extend(q, host.k, host.v, rtt, req, np.asarray(prefix, np.int32),
                               np.asarray(ext, np.int32), qo, scale)
        g.compare(o.float().cpu().numpy(), ro, "extend")
        g.compare_lse(lse.cpu().numpy(), rl, "extend")
        for t, r, k in zip(token_lists, rows, prefix):
            rx.rx_commit(tree, alloc, t, r, k)
        return rows, prefix

    prompt = list(range(1000, 1300))                   # a 300-token system prompt
    a = prompt + list(range(5000, 5120))
    rows_a, pre_a = extend_batch([a])
    assert pre_a == [0]
    # two more requests on the same prompt: found cached, their rows start
    # with A's prompt slots
    b = prompt + list(range(6000, 6090))
    c = prompt + list(range(7000, 7200))
    rows_bc, pre_bc = extend_batch([b, c])
    assert pre_bc == [300, 300]
    assert all(np.array_equal(r[:300], rows_a[0][:300]) for r in rows_bc)

    # decode: each request appends one token a step; the plan is built once
    # for the batch and serves every later step (its last pieces follow the
    # lengths on the device)
    toks = [a, b, c]
    rows = [np.asarray(r, np.int32) for r in rows_a + rows_bc]
    n_steps = 3
    stride = (max(len(t) for t in toks) + n_steps + 15) // 16 * 16
    rtt = np.full((3, stride), -1, np.int32)
    for i, r in enumerate(rows):
        rtt[i, :len(r)] = r
    lens = np.array([len(t) for t in toks], np.int32)
    plan = None
    for step in range(n_steps):
        new = alloc.take(3)
        for i in range(3):
            rtt[i, lens[i]] = new[i]
        lens = lens + 1
        k_new = inputs.randn_bf16(rng, (3, hkv, d))
        v_new = inputs.randn_bf16(rng, (3, hkv, d))
        rx.rx_kv_store(k_pool, v_pool, g.to_dev(k_new), g.to_dev(v_new), g.i32(new), status)
        host.store(k_new, v_new, new)
        if plan is None:
            buf, info = rx.rx_decode_plan_build(rtt, np.arange(3, dtype=np.int32), lens, hq, hkv)
            assert info.n_segments >= 1          # the shared prompt
            plan = rx.plan_to_device(buf, info, 3)
        max_len = int(lens.max())
        ws = torch.empty(max(rx.rx_attn_decode_workspace(3, hq, hkv, d, max_len, plan), 256),
                         dtype=torch.uint8, device="cuda")
        q = inputs.randn_bf16(rng, (3, hq, d))
        o = torch.empty((3, hq, d), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((3, hq), dtype=torch.float32, device="cuda")
        rx.rx_attn_decode(k_pool, v_pool, g.to_dev(q), o, lse, g.i32(np.arange(3)), g.i32(lens), g.i32(rtt),
                          max_len, scale, plan, ws, status)
        torch.cuda.synchronize()
        ro, rl = oracle.decode(q, host.k, host.v, rtt, np.arange(3, dtype=np.int32), lens, scale)
        g.compare(o.float().cpu().numpy(), ro, f"decode step {step}")
        g.compare_lse(lse.cpu().numpy(), rl, f"decode step {step}")
    assert int(status.item()) == 0

    # a request that no longer fits: admission evicts least recently used
    # leaves (unlocked ones) until its new slots are free
    free_before = alloc.free_count()
    big = list(range(90000, 90000 + free_before + 50))
    row, k, evicted = rx.rx_admit(tree, alloc, big)
    assert k == 0 and evicted >= 50 and len(row) == len(big)
