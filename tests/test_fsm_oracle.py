"""Pins of the compressed-FSM oracle (oracle/fsm.py): a worked example,
closed forms, the loop and cap rules, the allowed-token mask, and -- checked
against a decoder that never looks at the compression -- the fact that jumps
change how many steps decoding takes but not what it emits ("SGLang:
Efficient Execution of Structured Language Model Programs", unite.ai, es,
"Introducción a SGLang", compressed-FSM bullet)."""
import numpy as np
import pytest

from oracle import fsm


def csr(n_states, edges):
    """edges: {state: [(token, next), ...]} -> row_ptr, tok, nxt (tokens sorted)."""
    row_ptr, tok, nxt = [0], [], []
    for s in range(n_states):
        for t, n in sorted(edges.get(s, [])):
            tok.append(t)
            nxt.append(n)
        row_ptr.append(len(tok))
    return np.array(row_ptr, np.int64), np.array(tok, np.int32), np.array(nxt, np.int32)


# The worked example: text  {"name":"  then one or more of a / b, then  "}
# then end of sequence.  Vocabulary: 0 '{"', 1 'name', 2 '":"', 3 'a',
# 4 'b', 5 '"}', 6 <eos>, 7 'n', 8 'ame'.  "name" can be written as one
# token or as 'n' + 'ame', so state 1 has two edges.
EX_EDGES = {
    0: [(0, 1)],
    1: [(1, 3), (7, 2)],
    2: [(8, 3)],
    3: [(2, 4)],
    4: [(3, 5), (4, 5)],
    5: [(3, 5), (4, 5), (5, 6)],
    6: [(6, 7)],
}
EX = csr(8, EX_EDGES)


def test_worked_example_jumps():
    """By hand: the singular states are 0, 2, 3 and 6.
       0: '{"' -> 1 (two edges): jump [0], ends at 1.
       2: 'ame' -> 3, '":"' -> 4 (two edges): jump [8, 2], ends at 4.
       3: '":"' -> 4: jump [2], ends at 4.
       6: <eos> -> 7 (terminal, no edge): jump [6], ends at 7.
       1, 4, 5, 7: no jump."""
    fsm.validate(8, 9, *EX)
    jumps, ends, looped = fsm.compress(8, *EX, max_jump=16)
    assert jumps == [[0], [], [8, 2], [2], [], [], [6], []]
    assert ends == [1, 1, 4, 4, 4, 5, 7, 7]
    assert not any(looped)


def test_worked_example_steps():
    """From state 1, a model preferring 'n' emits n, ame, '":"' in one step
    and lands in state 4; one preferring 'name' emits name, '":"'.  From
    state 5, '"}' brings <eos> with it.  State 7 is terminal."""
    jumps, ends, _ = fsm.compress(8, *EX, max_jump=16)
    logits = np.full((4, 9), -1.0, np.float32)
    logits[0, 7] = 3.0           # 'n'
    logits[1, 1] = 2.0           # 'name'
    logits[1, 7] = 1.0
    logits[2, 5] = 0.5           # '"}' over a and b at -1
    em, ns, st = fsm.step(logits, [1, 1, 5, 7], *EX, jumps, ends)
    assert em == [[7, 8, 2], [1, 2], [5, 6], []]
    assert ns == [4, 4, 7, 7]
    assert st == [0, 0, 0, fsm.STATUS_TERMINAL]


def test_argmax_rules():
    """Only allowed tokens count; NaN is never chosen over a number; equal
    logits go to the smallest token id; all -inf / NaN gives the first
    allowed token."""
    tokens = np.array([2, 5, 9], np.int64)
    row = np.zeros(12, np.float32)
    row[0] = 100.0                      # not allowed
    row[[2, 5, 9]] = [1.0, 3.0, 3.0]
    assert fsm.choose(row, tokens) == 1
    row[5] = np.nan
    assert fsm.choose(row, tokens) == 2
    row[[2, 5, 9]] = [-np.inf, np.nan, -np.inf]
    assert fsm.choose(row, tokens) == 0


def test_linear_chain_closed_form():
    """A chain s0 -t0-> s1 -t1-> ... -> sn (terminal): every state jumps to
    the end, fixing the rest of the chain."""
    n = 9
    toks = [17 * i % 31 for i in range(n)]
    edges = {i: [(toks[i], i + 1)] for i in range(n)}
    row_ptr, tok, nxt = csr(n + 1, edges)
    jumps, ends, looped = fsm.compress(n + 1, row_ptr, tok, nxt, max_jump=64)
    for i in range(n + 1):
        assert jumps[i] == toks[i:] and ends[i] == n and not looped[i]


def test_cap_closed_form():
    """With max_jump = k a chain's jump stops after k tokens, at the k-th state."""
    n, k = 10, 4
    edges = {i: [(i, i + 1)] for i in range(n)}
    args = csr(n + 1, edges)
    jumps, ends, _ = fsm.compress(n + 1, *args, max_jump=k)
    for i in range(n + 1):
        m = min(k, n - i)
        assert jumps[i] == list(range(i, i + m)) and ends[i] == i + m


def test_loop_of_fixed_tokens():
    """0 -a-> 1 -b-> 0, both singular: the path stops on coming back."""
    args = csr(3, {0: [(5, 1)], 1: [(6, 0)], 2: [(5, 1), (7, 2)]})
    jumps, ends, looped = fsm.compress(3, *args, max_jump=32)
    assert jumps[0] == [5, 6] and ends[0] == 0 and looped[0]
    assert jumps[1] == [6, 5] and ends[1] == 1 and looped[1]
    assert jumps[2] == [] and ends[2] == 2 and not looped[2]


def test_no_singular_state_no_jump():
    args = csr(3, {0: [(0, 1), (1, 2)], 1: [(0, 0), (2, 2)], 2: []})
    jumps, ends, _ = fsm.compress(3, *args, max_jump=8)
    assert jumps == [[], [], []] and ends == [0, 1, 2]


def test_mask_bits():
    V = 70  # not a multiple of 32
    args = csr(3, {0: [(0, 1), (31, 2), (32, 2), (69, 0)], 1: [(33, 2)], 2: []})
    m = fsm.allowed_mask(3, V, args[0], args[1])
    assert m.shape == (3, 3) and m.dtype == np.uint32
    assert int(m[0, 0]) == (1 | (1 << 31)) and int(m[0, 1]) == 1 and int(m[0, 2]) == 1 << 5
    assert int(m[1, 1]) == 2 and not m[2].any()
    # popcount per state = out-degree
    pc = [sum(bin(int(w)).count("1") for w in row) for row in m]
    assert pc == [4, 1, 0]


def test_validation():
    row_ptr, tok, nxt = csr(2, {0: [(1, 1), (3, 0)]})
    fsm.validate(2, 4, row_ptr, tok, nxt)
    with pytest.raises(ValueError):
        fsm.validate(2, 3, row_ptr, tok, nxt)           # token 3 >= V
    with pytest.raises(ValueError):
        fsm.validate(2, 4, row_ptr, tok[::-1].copy(), nxt)  # not increasing
    with pytest.raises(ValueError):
        fsm.validate(2, 4, row_ptr, tok, np.array([1, 2], np.int32))  # next >= S


def _random_dfa(rng, n_states, vocab):
    """States with 0 to 4 edges; a fifth of them singular.  Singular edges
    only point to higher states (no loop of fixed tokens), other edges
    anywhere."""
    edges = {}
    for s in range(n_states):
        r = rng.random()
        if s == n_states - 1 or r < 0.1:
            continue
        if r < 0.3:
            edges[s] = [(int(rng.integers(vocab)), int(rng.integers(s + 1, n_states)))]
            continue
        k = int(rng.integers(2, 5))
        ts = rng.choice(vocab, size=k, replace=False)
        edges[s] = [(int(t), int(rng.integers(n_states))) for t in ts]
    return csr(n_states, edges)


@pytest.mark.parametrize("seed", range(12))
def test_jumps_emit_what_one_token_decoding_emits(seed):
    """Brute force on small machines: decoding with the compressed machine
    and decoding one token per step (which never looks at the jumps) emit
    the same tokens and end in the same state, using the same model rows;
    the compressed decoder takes one step per row, the other one step per
    token."""
    rng = np.random.default_rng(seed)
    S, V = int(rng.integers(5, 40)), int(rng.integers(8, 90))
    row_ptr, tok, nxt = _random_dfa(rng, S, V)
    fsm.validate(S, V, row_ptr, tok, nxt)
    jumps, ends, looped = fsm.compress(S, row_ptr, tok, nxt, max_jump=S + 1)
    assert not any(looped)
    for start in range(S):
        rows = rng.standard_normal((6, V)).astype(np.float32)
        a, sa, ua = fsm.decode_with_jumps(start, row_ptr, tok, nxt, jumps, ends, rows)
        b, sb, ub = fsm.decode_one_token_at_a_time(start, row_ptr, tok, nxt, rows[:ua], max_tokens=10 ** 6)
        assert a == b and sa == sb and ua == ub
        # every emitted token follows an edge
        s = start
        for t in a:
            lo, hi = row_ptr[s], row_ptr[s + 1]
            k = list(tok[lo:hi]).index(t)
            s = int(nxt[lo + k])
        assert s == sa


def test_jump_table_layout():
    jumps, ends, _ = fsm.compress(8, *EX, max_jump=16)
    length, offset, end, toks = fsm.jump_table(jumps, ends)
    assert length.tolist() == [1, 0, 2, 1, 0, 0, 1, 0]
    assert offset.tolist() == [0, 1, 1, 3, 4, 4, 4, 5]
    assert toks.tolist() == [0, 8, 2, 2, 6] and end.tolist() == ends
