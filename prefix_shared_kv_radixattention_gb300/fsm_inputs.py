"""Seeded synthetic inputs for constrained decoding: a vocabulary, a token
automaton for a JSON-object constraint over it, request states and logits.

This module only *draws* inputs.  It builds the constraint a caller would
hand to the library (a deterministic automaton over token ids), but none of
the method's arithmetic: no compression, no masked argmax, no jumps.  Both
the oracle (oracle/fsm.py) and the CUDA path are fed from it.

The workload stands in for the JSON-decoding runs of "SGLang: Efficient
Execution of Structured Language Model Programs" (unite.ai, es), "SGLang:
Evaluación y resultados".  No item of those runs is used: the vocabulary is
a seeded mix of strings and the schema is generated.

Recipe (``rng = numpy.random.default_rng(seed)``, draws in this order):
  * schema: ``n_fields`` keys ``K0 .. K{n-1}``, their values alternately an
    integer ``[0-9]+`` and a string ``"[a-z ]*"``; the text is
    ``{"K0": <v0>, "K1": "<v1>", ...}``;
  * vocabulary, like a tokenizer whose merges absorbed the schema's
    punctuation: id 0 is end-of-sequence (no text); then every printable
    ASCII character except ``{ } " : ,`` and the capitals; then the fixed
    text cut at its natural boundaries (``{"``, ``K0``, ``": ``, ``, "``,
    ``", "``, ``": "``, ``"}``, ...); the rest, in equal shares, digit runs
    (2 to 4), lower-case words of 2 to 8 letters (half with a leading
    space) and junk (2 to 6 characters from the single-character set);
  * the character automaton of that text, then the token automaton: token t
    leads from state q to the state its characters reach, if none of them
    is rejected; end-of-sequence leads from the state after ``}`` to a
    terminal state;
  * request states: uniform over the non-terminal states reachable from the
    start; logits: float32 N(0, 1).
"""
from __future__ import annotations

import dataclasses
from typing import List

import numpy as np

_PRINTABLE = [chr(c) for c in range(32, 127)]
_DIGITS = "0123456789"
_LETTERS = "abcdefghijklmnopqrstuvwxyz"


@dataclasses.dataclass
class TokenAutomaton:
    n_states: int
    vocab: int
    start: int
    terminal: int
    row_ptr: np.ndarray   # int64 [S+1]
    tok: np.ndarray       # int32 [E], ascending within a state
    nxt: np.ndarray       # int32 [E]
    strings: List[str]    # text of each token id ("" for end-of-sequence)
    schema_text: str      # the fixed text with value placeholders, for reading


_SINGLES = [c for c in _PRINTABLE if c not in '{}":,' and not c.isupper()]


def _pieces(n_fields: int) -> List[str]:
    """The schema's fixed text cut at its natural boundaries."""
    out = []
    for i in range(n_fields):
        is_int = i % 2 == 0
        if i == 0:
            out.append('{"')
        else:
            out.append(', "' if (i - 1) % 2 == 0 else '", "')
        out.append(f"K{i}")
        out.append('": ' if is_int else '": "')
    out.append("}" if (n_fields - 1) % 2 == 0 else '"}')
    return list(dict.fromkeys(out))  # each piece once


def _vocab(rng: np.random.Generator, size: int, n_fields: int) -> List[str]:
    words = [""] + _SINGLES + _pieces(n_fields)
    rest = size - len(words)
    if rest < 0:
        raise ValueError("vocabulary smaller than the single characters and the fixed pieces")
    kinds = rng.integers(0, 3, size=rest)
    for k in kinds:
        if k == 0:
            words.append("".join(rng.choice(list(_DIGITS), size=int(rng.integers(2, 5)))))
        elif k == 1:
            w = "".join(rng.choice(list(_LETTERS), size=int(rng.integers(2, 9))))
            words.append((" " + w) if rng.random() < 0.5 else w)
        else:
            words.append("".join(rng.choice(_SINGLES, size=int(rng.integers(2, 7)))))
    return words


def _char_automaton(n_fields: int):
    """Character automaton of {"K0": <int>, "K1": "<str>", ...}: dense table
    [Q, 128] of next states (-1 = rejected), the start and the final state."""
    trans: List[dict] = [{}]
    cur = 0
    pending = None  # state of an integer's digit loop, left on the next fixed character

    def new():
        trans.append({})
        return len(trans) - 1

    def literal(text):
        nonlocal cur, pending
        for j, ch in enumerate(text):
            nx = new()
            if j == 0 and pending is not None:
                trans[pending][ch] = nx
                pending = None
            else:
                trans[cur][ch] = nx
            cur = nx

    shown = []
    for i in range(n_fields):
        is_int = i % 2 == 0
        lead = ("{" if i == 0 else ", ") + f'"K{i}": ' + ("" if is_int else '"')
        literal(lead)
        if is_int:
            d = new()
            for c in _DIGITS:
                trans[cur][c] = d
                trans[d][c] = d
            cur = d
            pending = d
            shown.append(lead + "<int>")
        else:
            for c in _LETTERS + " ":
                trans[cur][c] = cur
            literal('"')
            shown.append(lead + '<str>"')
    literal("}")
    table = np.full((len(trans), 128), -1, np.int32)
    for q, d in enumerate(trans):
        for ch, nx in d.items():
            table[q, ord(ch)] = nx
    return table, 0, cur, "".join(shown) + "}"


def json_automaton(seed: int = 3001, vocab: int = 128256, n_fields: int = 8) -> TokenAutomaton:
    rng = np.random.default_rng(seed)
    table, start, final, shown = _char_automaton(n_fields)
    strings = _vocab(rng, vocab, n_fields)
    Q = table.shape[0]
    L = max(len(w) for w in strings)
    codes = np.full((vocab, L), -1, np.int32)
    for t, w in enumerate(strings):
        if w:
            codes[t, :len(w)] = [ord(c) for c in w]
    has_text = codes[:, 0] >= 0
    terminal = Q
    rows: List[np.ndarray] = []
    nexts: List[np.ndarray] = []
    for q in range(Q):
        cur = np.full(vocab, q, np.int32)
        alive = has_text.copy()
        for pos in range(L):
            c = codes[:, pos]
            act = alive & (c >= 0)
            if not act.any():
                break
            cur[act] = table[cur[act], c[act]]
            alive &= ~(act & (cur < 0))
        ids = np.nonzero(alive)[0].astype(np.int32)
        nx = cur[ids]
        if q == final:  # end-of-sequence closes the text
            ids = np.concatenate([np.zeros(1, np.int32), ids])
            nx = np.concatenate([np.full(1, terminal, np.int32), nx])
        rows.append(ids)
        nexts.append(nx.astype(np.int32))
    rows.append(np.zeros(0, np.int32))     # the terminal state
    nexts.append(np.zeros(0, np.int32))
    row_ptr = np.zeros(Q + 2, np.int64)
    row_ptr[1:] = np.cumsum([len(r) for r in rows])
    return TokenAutomaton(Q + 1, vocab, start, terminal, row_ptr, np.concatenate(rows), np.concatenate(nexts),
                          strings, shown)


def trim(a: TokenAutomaton) -> TokenAutomaton:
    """The automaton without its dead ends: edges into states from which
    the terminal state cannot be reached are dropped (a token that leads
    nowhere but a dead end is then not allowed).  ``json_automaton`` keeps
    them, as a plain character walk gives them; a request that reaches one
    is flagged as having no token left."""
    S = a.n_states
    # states that reach the terminal: backwards over the edges
    src = np.repeat(np.arange(S), np.diff(a.row_ptr))
    live = np.zeros(S, bool)
    live[a.terminal] = True
    changed = True
    while changed:
        new = live.copy()
        np.logical_or.at(new, src, live[a.nxt])
        changed = bool((new != live).any())
        live = new
    keep = live[a.nxt]
    counts = np.bincount(src[keep], minlength=S)
    row_ptr = np.zeros(S + 1, np.int64)
    row_ptr[1:] = np.cumsum(counts)
    return dataclasses.replace(a, row_ptr=row_ptr, tok=a.tok[keep].copy(), nxt=a.nxt[keep].copy())


def reachable_states(a: TokenAutomaton) -> np.ndarray:
    """States reachable from the start along token edges (breadth first)."""
    seen = np.zeros(a.n_states, bool)
    seen[a.start] = True
    frontier = [a.start]
    while frontier:
        nxt = []
        for s in frontier:
            for n in a.nxt[a.row_ptr[s]:a.row_ptr[s + 1]]:
                if not seen[n]:
                    seen[n] = True
                    nxt.append(int(n))
        frontier = nxt
    return np.nonzero(seen)[0]


def step_inputs(a: TokenAutomaton, batch: int, seed: int = 3002):
    """Request states (uniform over reachable non-terminal states) and
    float32 N(0, 1) logits [batch, vocab]."""
    rng = np.random.default_rng(seed)
    live = np.array([s for s in reachable_states(a) if a.row_ptr[s + 1] > a.row_ptr[s]], np.int32)
    state = live[rng.integers(0, len(live), size=batch)].astype(np.int32)
    logits = rng.standard_normal((batch, a.vocab), dtype=np.float32)
    return state, logits
