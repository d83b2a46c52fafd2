"""The native compressed-FSM host step (rx_fsm_compress) against the oracle
(oracle/fsm.py), bit for bit, and the argument checks of both FSM entry
points ("SGLang: Efficient Execution of Structured Language Model Programs",
unite.ai, es, "Introducción a SGLang", compressed-FSM bullet)."""
import ctypes

import numpy as np
import pytest

from oracle import fsm as ref
from prefix_shared_kv_radixattention_gb300 import binding as rx
from prefix_shared_kv_radixattention_gb300 import fsm_inputs
from tests.test_fsm_oracle import EX, csr


def random_automaton(rng, n_states, vocab, p_single=0.3, loops=True):
    """Edge counts 0 to 6; single-edge states may point anywhere (loops of
    fixed tokens allowed) when ``loops``."""
    edges = {}
    for s in range(n_states):
        r = rng.random()
        if r < 0.1:
            continue
        if r < 0.1 + p_single:
            lo = 0 if loops else s + 1
            if lo >= n_states:
                continue
            edges[s] = [(int(rng.integers(vocab)), int(rng.integers(lo, n_states)))]
            continue
        k = int(rng.integers(2, min(7, vocab) + 1))
        ts = rng.choice(vocab, size=k, replace=False)
        edges[s] = [(int(t), int(rng.integers(n_states))) for t in ts]
    return csr(n_states, edges)


def _compare(S, V, row_ptr, tok, nxt, max_jump):
    mask, rank, jl, jo, je, jt, info = rx.rx_fsm_compress(S, V, row_ptr, tok, nxt, max_jump)
    jumps, ends, looped = ref.compress(S, row_ptr, tok, nxt, max_jump)
    length, offset, end, toks = ref.jump_table(jumps, ends)
    assert jl.tolist() == length.tolist() and jo.tolist() == offset.tolist()
    assert je.tolist() == end.tolist() and jt.tolist() == toks.tolist()
    W = (V + 127) // 128 * 4          # rows padded to 16 bytes
    assert mask.shape == (S, W)
    assert np.array_equal(mask[:, :(V + 31) // 32], ref.allowed_mask(S, V, row_ptr, tok))
    assert not mask[:, (V + 31) // 32:].any()
    # word ranks: edges of the state with a token below 32 w
    for s in range(S):
        t = np.asarray(tok[row_ptr[s]:row_ptr[s + 1]])
        assert rank[s].tolist() == [int(np.sum(t < 32 * w)) for w in range(W)]
    assert info.n_edges == len(tok) and info.jump_tokens == len(toks)
    assert info.n_singular == int(np.sum(np.diff(row_ptr) == 1))
    assert info.n_looped == sum(looped) and info.longest_jump == (max(length) if S else 0)


def test_worked_example():
    _compare(8, 9, *EX, 16)


@pytest.mark.parametrize("seed", range(16))
def test_compress_matches_oracle(seed):
    rng = np.random.default_rng(seed)
    S, V = int(rng.integers(1, 60)), int(rng.integers(1, 200))
    args = random_automaton(rng, S, V)
    for max_jump in (0, 1, 3, 64):
        _compare(S, V, *args, max_jump)


def test_json_automaton_matches_oracle():
    a = fsm_inputs.json_automaton(vocab=3000, n_fields=5)
    _compare(a.n_states, a.vocab, a.row_ptr, a.tok, a.nxt, 16)
    jumps, ends, _ = ref.compress(a.n_states, a.row_ptr, a.tok, a.nxt, 16)
    # the start fixes  {"  K0  ":   -- three tokens
    assert ["".join(a.strings[t] for t in jumps[a.start])] == ['{"K0": ']


def test_compress_rejects_bad_automata():
    lib = rx.library()
    P = ctypes.c_void_p
    info = rx.FsmInfo()

    def call(S, V, row_ptr, tok, nxt, max_jump=4, jt=None, cap=0):
        rp = np.asarray(row_ptr, np.int64)
        t = np.asarray(tok, np.int32)
        n = np.asarray(nxt, np.int32)
        return lib.rx_fsm_compress(S, V, rp.ctypes.data_as(P), t.ctypes.data_as(P), n.ctypes.data_as(P),
                                   max_jump, None, None, None, None, None,
                                   None if jt is None else jt.ctypes.data_as(P), cap, ctypes.byref(info))

    assert call(2, 4, [0, 2, 2], [1, 3], [1, 0]) == rx.RX_OK
    assert call(2, 3, [0, 2, 2], [1, 3], [1, 0]) == rx.RX_ERR_INVALID        # token >= vocab
    assert call(2, 4, [0, 2, 2], [3, 1], [1, 0]) == rx.RX_ERR_INVALID        # not increasing
    assert call(2, 4, [0, 2, 2], [1, 3], [1, 2]) == rx.RX_ERR_INVALID        # next >= S
    assert call(2, 4, [1, 2, 2], [1, 3], [1, 0]) == rx.RX_ERR_INVALID        # row_ptr[0] != 0
    assert call(2, 4, [0, 2, 1], [1, 3], [1, 0]) == rx.RX_ERR_INVALID        # decreasing
    assert call(2, 4, [0, 2, 2], [1, 3], [1, 0], max_jump=-1) == rx.RX_ERR_INVALID
    # a chain 0 -> 1 -> 2 needs 3 jump tokens (2 from state 0, 1 from state 1)
    small = np.zeros(2, np.int32)
    assert call(3, 4, [0, 1, 2, 2], [1, 2], [1, 2], jt=small, cap=2) == rx.RX_ERR_CAPACITY
    assert info.jump_tokens == 3


def test_step_argument_checks_without_a_gpu():
    """Host-side checks run before any CUDA call: a null machine, a negative
    batch; an empty batch is a no-op."""
    lib = rx.library()
    assert lib.rx_fsm_step(None, None, 8, 1, None, None, None, None, None, None) == rx.RX_ERR_INVALID
    st = rx.FsmStruct()
    st.n_states, st.vocab, st.max_jump = 2, 8, 4
    assert lib.rx_fsm_step(ctypes.byref(st), None, 8, -1, None, None, None, None, None, None) == rx.RX_ERR_INVALID
    assert lib.rx_fsm_step(ctypes.byref(st), None, 8, 0, None, None, None, None, None, None) == rx.RX_OK
    # a null pointer with a non-empty batch
    assert lib.rx_fsm_step(ctypes.byref(st), None, 8, 1, None, None, None, None, None, None) == rx.RX_ERR_INVALID


def test_json_decoding_emits_schema_text_and_saves_steps():
    """End to end on the synthetic JSON constraint (oracle only): with logits
    that favour short values, decoding with jumps reaches the terminal state,
    the text it emits matches the schema's regular expression, and it takes
    fewer model steps than tokens (the fixed keys and separators come as
    jumps)."""
    import re
    a = fsm_inputs.trim(fsm_inputs.json_automaton(vocab=6000, n_fields=6))
    ref.validate(a.n_states, a.vocab, a.row_ptr, a.tok, a.nxt)
    # trimmed: every reachable state but the terminal one has an edge
    assert all(a.row_ptr[s + 1] > a.row_ptr[s] for s in fsm_inputs.reachable_states(a) if s != a.terminal)
    jumps, ends, _ = ref.compress(a.n_states, a.row_ptr, a.tok, a.nxt, 16)
    rng = np.random.default_rng(3)
    rows = rng.standard_normal((400, a.vocab)).astype(np.float32)
    # prefer closing pieces and end-of-sequence once they are allowed
    closers = [t for t, w in enumerate(a.strings) if w in ("", ', "', '", "', "}", '"}')]
    rows[:, closers] += 6.0
    toks, state, used = ref.decode_with_jumps(a.start, a.row_ptr, a.tok, a.nxt, jumps, ends, rows)
    assert state == a.terminal and toks[-1] == 0           # ended by end-of-sequence
    text = "".join(a.strings[t] for t in toks)
    parts = []
    for i in range(6):
        parts.append(("{" if i == 0 else ", ") + f'"K{i}": ' + ("[0-9]+" if i % 2 == 0 else '"[a-z ]*"'))
    assert re.fullmatch("".join(parts) + "}", text), text
    assert used < len(toks)
