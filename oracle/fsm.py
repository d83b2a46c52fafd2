"""Compressed finite-state machine for constrained decoding -- oracle.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may use it.
Plain Python and numpy; it imports nothing from the CUDA path.

Source: "SGLang: Efficient Execution of Structured Language Model Programs"
(unite.ai, es), "Introducción a SGLang", compressed-FSM bullet.  Systems that
follow an output constraint look only at the next token, so they decode one
token per step.  SGLang analyses the constraint, builds a compressed finite
state machine for it, and collapses a path of several tokens into one step
wherever it can, so that several tokens come out of one decoding step.

The pages give no algorithm; this module takes the plainest reading that
fits them:

* The constraint is a deterministic automaton over vocabulary token ids.
  It has states 0 .. S-1, and its edges (s, t) -> s' are stored per state in
  ascending token order: ``row_ptr`` [S+1], ``tok`` [E], ``nxt`` [E].  A
  state without edges is terminal: the constrained text is complete there.
* A state with exactly one edge is *singular*: the constraint fixes the
  next token.
* Compression gives every state s a *jump*: the tokens fixed along the path
  of singular states that starts at s, and the state where that path stops.
  It stops at the first state that is not singular, or at a state that the
  path has already passed through (a loop of fixed tokens), or after
  ``max_jump`` tokens.
* One decoding step of a request in state s with logits x over the
  vocabulary:
  - t = argmax of x over the tokens allowed at s; NaN counts as -inf, and
    ties go to the smallest token id;
  - s1 = the state the edge (s, t) leads to;
  - the jump of s1 is emitted in the same step: the step's tokens are t
    followed by the jump's tokens, and the request moves to the jump's end
    state.
  A request in a terminal state is flagged and left as it is.

Every function here is pinned in ``tests/test_fsm_oracle.py``.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

import numpy as np

STATUS_TERMINAL = 1  # a request's state has no edge (nothing left to decode)


def validate(n_states: int, vocab: int, row_ptr, tok, nxt) -> None:
    """The automaton's arrays as the reading above defines them: ValueError
    otherwise."""
    row_ptr = np.asarray(row_ptr, np.int64)
    tok = np.asarray(tok, np.int64)
    nxt = np.asarray(nxt, np.int64)
    if n_states < 1 or vocab < 1:
        raise ValueError("need at least one state and one token")
    if row_ptr.shape != (n_states + 1,) or row_ptr[0] != 0 or np.any(np.diff(row_ptr) < 0):
        raise ValueError("row_ptr must start at 0 and not decrease")
    E = int(row_ptr[-1])
    if tok.shape != (E,) or nxt.shape != (E,):
        raise ValueError("tok and nxt must hold row_ptr[S] edges")
    if E and (tok.min() < 0 or tok.max() >= vocab or nxt.min() < 0 or nxt.max() >= n_states):
        raise ValueError("token or next state out of range")
    for s in range(n_states):
        t = tok[row_ptr[s]:row_ptr[s + 1]]
        if np.any(np.diff(t) <= 0):
            raise ValueError(f"tokens of state {s} must be strictly increasing")


def compress(n_states: int, row_ptr, tok, nxt, max_jump: int):
    """The compressed machine: for every state its jump.

    Returns (jumps, ends, looped): jumps[s] is the list of fixed tokens,
    ends[s] the state where the path stops, looped[s] whether it stopped
    because it came back to a state it had passed."""
    row_ptr = [int(x) for x in row_ptr]
    tok = [int(x) for x in tok]
    nxt = [int(x) for x in nxt]
    jumps: List[List[int]] = []
    ends: List[int] = []
    looped: List[bool] = []
    for s in range(n_states):
        path: List[int] = []
        seen = set()
        u = s
        hit_loop = False
        while len(path) < max_jump and row_ptr[u + 1] - row_ptr[u] == 1:
            if u in seen:
                hit_loop = True
                break
            seen.add(u)
            e = row_ptr[u]
            path.append(tok[e])
            u = nxt[e]
        jumps.append(path)
        ends.append(u)
        looped.append(hit_loop)
    return jumps, ends, looped


def allowed_mask(n_states: int, vocab: int, row_ptr, tok) -> np.ndarray:
    """Bit t % 32 of word t // 32 of row s is set when token t is allowed at
    state s: uint32 [S, ceil(V / 32)]."""
    W = (vocab + 31) // 32
    mask = np.zeros((n_states, W), np.uint32)
    for s in range(n_states):
        for e in range(int(row_ptr[s]), int(row_ptr[s + 1])):
            t = int(tok[e])
            mask[s, t // 32] |= np.uint32(1 << (t % 32))
    return mask


def choose(logits_row: np.ndarray, tokens: np.ndarray) -> int:
    """Index (into ``tokens``, ascending ids) of the allowed token with the
    largest logit; NaN as -inf; the first (smallest id) of equal ones."""
    vals = np.asarray(logits_row, np.float32)[tokens].astype(np.float64)
    vals[np.isnan(vals)] = -np.inf
    return int(np.argmax(vals))


def step(logits: np.ndarray, state: Sequence[int], row_ptr, tok, nxt, jumps, ends):
    """One decoding step for a batch.

    logits: float32 [B, V].  Returns (emitted, new_state, status):
    emitted[b] is the list of tokens request b emits, new_state[b] its
    state afterwards, status[b] STATUS_TERMINAL or 0."""
    row_ptr = np.asarray(row_ptr, np.int64)
    tok = np.asarray(tok, np.int64)
    nxt = np.asarray(nxt, np.int64)
    emitted, new_state, status = [], [], []
    for b, s in enumerate(state):
        s = int(s)
        lo, hi = int(row_ptr[s]), int(row_ptr[s + 1])
        if hi == lo:
            emitted.append([])
            new_state.append(s)
            status.append(STATUS_TERMINAL)
            continue
        i = choose(logits[b], tok[lo:hi])
        t, s1 = int(tok[lo + i]), int(nxt[lo + i])
        emitted.append([t] + list(jumps[s1]))
        new_state.append(int(ends[s1]))
        status.append(0)
    return emitted, new_state, status


def decode_one_token_at_a_time(start: int, row_ptr, tok, nxt, choice_logits, max_tokens: int):
    """Constrained decoding without compression: one token per step.  A state
    with a single edge takes it without consulting the model; at every other
    state the next row of ``choice_logits`` (float32 [n, V]) picks the token.
    Stops at a terminal state, when the rows run out, or after max_tokens.
    Returns (tokens, state, rows used)."""
    row_ptr = np.asarray(row_ptr, np.int64)
    tok = np.asarray(tok, np.int64)
    nxt = np.asarray(nxt, np.int64)
    out: List[int] = []
    s, used = int(start), 0
    while len(out) < max_tokens:
        lo, hi = int(row_ptr[s]), int(row_ptr[s + 1])
        if hi == lo:
            break
        if hi - lo == 1:
            i = 0
        else:
            if used == len(choice_logits):
                break
            i = choose(choice_logits[used], tok[lo:hi])
            used += 1
        out.append(int(tok[lo + i]))
        s = int(nxt[lo + i])
    return out, s, used


def decode_with_jumps(start: int, row_ptr, tok, nxt, jumps, ends, choice_logits):
    """Constrained decoding with the compressed machine: the start state's
    jump first, then one ``step`` per row of ``choice_logits``, stopping at
    a terminal state.  Returns (tokens, state, rows used)."""
    out: List[int] = list(jumps[start])
    s = int(ends[start])
    used = 0
    row_ptr = np.asarray(row_ptr, np.int64)
    while used < len(choice_logits) and row_ptr[s + 1] > row_ptr[s]:
        em, ns, _ = step(choice_logits[used:used + 1], [s], row_ptr, tok, nxt, jumps, ends)
        out.extend(em[0])
        s = ns[0]
        used += 1
    return out, s, used


def jump_table(jumps, ends) -> Tuple[np.ndarray, np.ndarray, np.ndarray, np.ndarray]:
    """Packed form of the jumps: (length [S], offset [S] int64, end [S],
    tokens [sum of lengths]), offsets in state order."""
    n = len(jumps)
    length = np.array([len(j) for j in jumps], np.int32)
    offset = np.zeros(n, np.int64)
    if n:
        offset[1:] = np.cumsum(length[:-1], dtype=np.int64)
    toks = np.array([t for j in jumps for t in j], np.int32)
    return length, offset, np.asarray(ends, np.int32), toks
