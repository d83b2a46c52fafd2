"""GPU parity of the constrained decoding step (rx_fsm_step) against the
oracle's step (oracle/fsm.py): chosen token, emitted jump, new state and
flags, bit for bit -- the argmax is a comparison of the same fp32 values on
both sides ("SGLang: Efficient Execution of Structured Language Model
Programs", unite.ai, es, "Introducción a SGLang", compressed-FSM bullet)."""
import numpy as np
import pytest

from oracle import fsm as ref
from prefix_shared_kv_radixattention_gb300 import fsm_inputs
from tests.test_fsm_native import random_automaton

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _rx():
    from prefix_shared_kv_radixattention_gb300 import binding as rx
    return rx


def _run(S, V, row_ptr, tok, nxt, max_jump, state, logits, stride=None):
    """One device step; returns (emitted lists, new states, status word) and
    the oracle's (emitted, states, per-request status)."""
    rx = _rx()
    m = rx.Fsm(S, V, row_ptr, tok, nxt, max_jump)
    B = len(state)
    stride = stride or (V + 3) // 4 * 4
    lg = torch.zeros((B, stride), dtype=torch.float32, device="cuda")
    lg[:, :V] = torch.from_numpy(np.ascontiguousarray(logits, np.float32)).cuda()
    st = torch.from_numpy(np.asarray(state, np.int32)).cuda()
    out = torch.full((B, 1 + max_jump), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = rx.fsm_workspace(B)
    rx.rx_fsm_step(m, lg, st, out, cnt, ws, status)
    torch.cuda.synchronize()
    assert not ws.any()   # left zero for the next call
    o, c, s2 = out.cpu().numpy(), cnt.cpu().numpy(), st.cpu().numpy()
    got = [o[b, :c[b]].tolist() for b in range(B)]
    jumps, ends, _ = ref.compress(S, row_ptr, tok, nxt, max_jump)
    em, ns, rst = ref.step(np.asarray(logits, np.float32), state, row_ptr, tok, nxt, jumps, ends)
    return (got, s2.tolist(), int(status.item())), (em, ns, rst)


@pytest.mark.parametrize("seed", range(8))
def test_step_matches_oracle_random(seed):
    rng = np.random.default_rng(100 + seed)
    S, V = int(rng.integers(2, 50)), int(rng.integers(1, 300))
    args = random_automaton(rng, S, V)
    live = [s for s in range(S) if args[0][s + 1] > args[0][s]]
    if not live:
        pytest.skip("no state with an edge")
    B = 37
    state = np.array([live[i % len(live)] for i in range(B)], np.int32)
    logits = rng.standard_normal((B, V)).astype(np.float32)
    (got, st, status), (em, ns, rst) = _run(S, V, *args, 5, state, logits)
    assert got == em and st == ns and status == 0


def test_ties_nan_and_inf():
    """Integer-valued logits tie often: the smallest id must win; NaN loses
    to any number; a row of -inf and NaN picks the smallest allowed id."""
    rng = np.random.default_rng(7)
    S, V = 30, 257
    args = random_automaton(rng, S, V, p_single=0.0)
    live = [s for s in range(S) if args[0][s + 1] > args[0][s]]
    B = 64
    state = np.array([live[i % len(live)] for i in range(B)], np.int32)
    logits = rng.integers(0, 3, size=(B, V)).astype(np.float32)
    logits[1::4] = np.nan
    logits[1::4, ::7] = 1.0
    logits[2::4] = -np.inf
    logits[3::4, ::3] = np.nan
    (got, st, status), (em, ns, _) = _run(S, V, *args, 3, state, logits)
    assert got == em and st == ns and status == 0


def test_signed_zero_ties():
    """-0 and +0 are equal values: where the largest allowed logit is zero,
    the smallest allowed id holding a zero of either sign wins."""
    rng = np.random.default_rng(11)
    S, V = 24, 300
    args = random_automaton(rng, S, V, p_single=0.0)
    live = [s for s in range(S) if args[0][s + 1] > args[0][s]]
    B = 48
    state = np.array([live[i % len(live)] for i in range(B)], np.int32)
    logits = np.full((B, V), -1.0, np.float32)
    logits[:, ::2] = -0.0
    logits[:, 1::4] = 0.0
    logits[::3, ::5] = np.nan
    (got, st, status), (em, ns, _) = _run(S, V, *args, 3, state, logits)
    assert got == em and st == ns and status == 0


def test_terminal_and_bad_states_are_flagged():
    rx = _rx()
    from tests.test_fsm_oracle import EX
    state = np.array([7, 5, 99, 1, -2], np.int32)      # terminal, live, out of range, live, out of range
    logits = np.zeros((5, 9), np.float32)
    logits[:, 5] = 1.0
    logits[3, 7] = 2.0
    m = rx.Fsm(8, 9, *EX, 16)
    lg = torch.zeros((5, 12), dtype=torch.float32, device="cuda")
    lg[:, :9] = torch.from_numpy(logits).cuda()
    s_dev = torch.from_numpy(state).cuda()
    out = torch.zeros((5, 17), dtype=torch.int32, device="cuda")
    cnt = torch.full((5,), -1, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rx.rx_fsm_step(m, lg, s_dev, out, cnt, rx.fsm_workspace(5), status)
    torch.cuda.synchronize()
    c, s2 = cnt.cpu().numpy(), s_dev.cpu().numpy()
    assert c.tolist() == [0, 2, 0, 3, 0]
    assert s2.tolist() == [7, 7, 99, 4, -2]
    assert out.cpu().numpy()[1, :2].tolist() == [5, 6] and out.cpu().numpy()[3, :3].tolist() == [7, 8, 2]
    assert int(status.item()) == rx.RX_DEV_FSM_DONE | rx.RX_DEV_BAD_STATE


# batches up to 512 finish in the scan kernel's last CTA; 700 takes the
# separate finish kernel
@pytest.mark.parametrize("vocab,batch", [(128256, 64), (32000, 300), (5003, 3), (5003, 512), (5003, 700)])
def test_json_workload_matches_oracle(vocab, batch):
    """The synthetic JSON constraint at a real vocabulary size: every slice
    split (cluster sizes 1 to 8 across these shapes) gives the oracle's
    answer; a padded row stride is honoured."""
    a = fsm_inputs.json_automaton(vocab=vocab, n_fields=6)
    state, logits = fsm_inputs.step_inputs(a, batch, seed=vocab + batch)
    (got, st, status), (em, ns, _) = _run(a.n_states, a.vocab, a.row_ptr, a.tok, a.nxt, 16, state, logits,
                                         stride=(vocab + 3) // 4 * 4 + 8)
    assert got == em and st == ns and status == 0


def test_decoding_loop_matches_oracle():
    """Twenty steps with the states fed back on the device: every request's
    text equals the oracle's decoding with jumps from the same start."""
    rx = _rx()
    a = fsm_inputs.json_automaton(vocab=20000, n_fields=6)
    B, steps, J = 24, 20, 16
    rng = np.random.default_rng(5)
    m = rx.Fsm(a.n_states, a.vocab, a.row_ptr, a.tok, a.nxt, J)
    jumps, ends, _ = ref.compress(a.n_states, a.row_ptr, a.tok, a.nxt, J)
    rows = rng.standard_normal((steps, B, a.vocab)).astype(np.float32)
    rows[:, :, 0] += 3.0   # end-of-sequence likely once allowed
    st = torch.full((B,), int(ends[a.start]), dtype=torch.int32, device="cuda")
    out = torch.zeros((B, 1 + J), dtype=torch.int32, device="cuda")
    cnt = torch.zeros(B, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    texts = [list(jumps[a.start]) for _ in range(B)]
    ws = rx.fsm_workspace(B)   # reused: every call leaves it zero
    for k in range(steps):
        lg = torch.from_numpy(rows[k]).cuda()
        rx.rx_fsm_step(m, lg, st, out, cnt, ws, status)
        o, c = out.cpu().numpy(), cnt.cpu().numpy()
        for b in range(B):
            texts[b].extend(o[b, :c[b]].tolist())
    for b in range(B):
        want, s_end, used = ref.decode_with_jumps(a.start, a.row_ptr, a.tok, a.nxt, jumps, ends, rows[:, b])
        assert texts[b] == want
        assert int(st[b].item()) == s_end
