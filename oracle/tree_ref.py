"""Reference radix tree: a per-token trie that records radix-node boundaries.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Follows "SGLang: Efficient Execution of Structured Language Model Programs"
(unite.ai, es):
  * section "Introducción a SGLang", RadixAttention bullet: the KV cache of
    finished calls is kept as an LRU cache inside a radix tree that supports
    matching, insertion and eviction;
  * section "SGLang: Modelo de programación y metodología", the nine-step
    walkthrough: every edge carries a token sequence; a request that extends
    a cached sequence adds its new tokens as a new node (step 3) hung after
    the node it continues (step 5); a partial share splits a node in two
    (steps 4 and 7); under memory pressure least-recently-used nodes are
    evicted, one node or several (steps 5, 8, 9), and a request's own
    matched prefix is not among them (step 8 evicts the second session while
    the first session's system prompt is reused).

Storage is one trie node per token (page size 1).  Each trie node carries a
``head`` flag that is set on the first token of every radix node; a radix
node is a head token plus the run of non-head single children below it.  A
radix node's last-access value lives on its head.

Readings taken where the pages are silent:
  * a logical clock advances once per ``match_prefix`` or ``insert`` call;
    every radix node that holds at least one token of that call's matched
    path takes the new value (a partially matched node counts as used);
  * ``match_prefix`` never changes the structure;
  * ``insert`` splits a node only when new tokens diverge strictly inside it;
    the lower part keeps the node's value from before the call, the upper
    part is on the path and takes the new value; all new tokens form one new
    leaf node;
  * eviction removes whole leaf radix nodes, the one with the smallest
    last-access value first, one after another until at least the requested
    number of tokens is free or nothing is left (the last node may
    overshoot); a parent left without children becomes a leaf and competes
    in the same call.  Nodes holding a given value always lie on one root
    path (the path of the call that set it, and splits keep both parts on
    it), so two leaves never tie and no tie-break is needed;
  * freed slots are reported node by node, each node in token order;
  * locks: ``lock(tokens, +1)`` adds one to the lock count of every cached
    token of the matched prefix (and touches the clock like a match);
    ``lock(tokens, -1)`` takes one off again without touching the clock.  A
    node with any locked token is never evicted.  Locks sit on tokens, so a
    later split leaves each part exactly the locks of its own tokens.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence, Tuple


class _Tok:
    __slots__ = ("token", "slot", "head", "last", "parent", "children", "lock")

    def __init__(self, token, slot, parent, head, last):
        self.lock = 0
        self.token = token
        self.slot = slot
        self.head = head          # first token of a radix node
        self.last = last          # meaningful on heads only
        self.parent = parent
        self.children: Dict[int, "_Tok"] = {}


class CapacityError(Exception):
    """Raised when the caller's output capacity cannot hold the next node."""


class RadixTreeRef:
    def __init__(self):
        self.root = _Tok(None, -1, None, True, 0)
        self.clock = 0
        self.cached_tokens = 0

    # -- helpers ---------------------------------------------------------
    def _walk(self, tokens: Sequence[int]) -> List[_Tok]:
        node, path = self.root, []
        for t in tokens:
            nxt = node.children.get(int(t))
            if nxt is None:
                break
            path.append(nxt)
            node = nxt
        return path

    def _head_of(self, tok: _Tok) -> _Tok:
        while not tok.head:
            tok = tok.parent
        return tok

    def _tick(self, path: List[_Tok]) -> None:
        # every radix node on a root path starts on that path, so the heads
        # among the path's tokens are exactly the nodes it touches
        for t in path:
            if t.head:
                t.last = self.clock

    def _leaf_nodes(self) -> List[Tuple[_Tok, _Tok]]:
        """(head, last token) of every radix node without children."""
        out, stack = [], [self.root]
        while stack:
            n = stack.pop()
            if n.children:
                stack.extend(n.children.values())
            elif n is not self.root:
                out.append((self._head_of(n), n))
        return out

    # -- API ---------------------------------------------------------------
    def match_prefix(self, tokens: Sequence[int]) -> Tuple[int, List[int]]:
        """Longest cached prefix of ``tokens``: (length, its slot ids)."""
        self.clock += 1
        path = self._walk(tokens)
        self._tick(path)
        return len(path), [t.slot for t in path]

    def prefix_len(self, tokens: Sequence[int]) -> int:
        """Longest cached prefix length of ``tokens``, as a probe: the clock
        does not move and no node counts as used."""
        return len(self._walk(tokens))

    def insert(self, tokens: Sequence[int], slots: Sequence[int]) -> int:
        """Cache ``tokens`` with ``slots``; returns how many leading tokens
        were already cached (those keep the tree's slots)."""
        assert len(tokens) == len(slots)
        self.clock += 1
        path = self._walk(tokens)
        k = len(path)
        end = path[-1] if path else self.root
        if k < len(tokens) and end is not self.root and len(end.children) == 1:
            only = next(iter(end.children.values()))
            if not only.head:
                # new tokens leave a node strictly inside it: split there
                only.head = True
                only.last = self._head_of(end).last
        self._tick(path)
        node = end
        for i in range(k, len(tokens)):
            tok = _Tok(int(tokens[i]), int(slots[i]), node, i == k, self.clock)
            node.children[int(tokens[i])] = tok
            node = tok
            self.cached_tokens += 1
        return k

    def evict(self, num_tokens: int, cap: Optional[int] = None) -> List[int]:
        """Remove leaf radix nodes, least recently used first, until at least
        ``num_tokens`` slots are freed or the tree is empty.  Returns the
        freed slots.  If ``cap`` is given and the next node would not fit,
        raises CapacityError with the slots freed so far in ``err.args[0]``."""
        freed: List[int] = []
        while len(freed) < num_tokens:
            leaves = self._leaf_nodes()
            if not leaves:
                break
            runs = []
            for head, last_tok in leaves:
                run, n = [], last_tok
                while True:
                    run.append(n)
                    if n is head:
                        break
                    n = n.parent
                run.reverse()
                if all(t.lock == 0 for t in run):
                    runs.append((head.last, run))
            if not runs:
                break
            _, run = min(runs, key=lambda lr: lr[0])
            head = run[0]
            if cap is not None and len(freed) + len(run) > cap:
                raise CapacityError(freed)
            del head.parent.children[head.token]
            freed.extend(t.slot for t in run)
            self.cached_tokens -= len(run)
        return freed

    def lock(self, tokens: Sequence[int], delta: int) -> int:
        """Lock (+1) or unlock (-1) the cached prefix of ``tokens``; returns
        its length.  Unlocking a token whose count is zero raises ValueError
        and changes nothing."""
        assert delta in (1, -1)
        if delta > 0:
            self.clock += 1
        path = self._walk(tokens)
        if delta < 0 and any(t.lock == 0 for t in path):
            raise ValueError("unlock without lock")
        if delta > 0:
            self._tick(path)
        for t in path:
            t.lock += delta
        return len(path)

    def evictable_tokens(self) -> int:
        total, stack = 0, [self.root]
        while stack:
            n = stack.pop()
            for c in n.children.values():
                run, t = [c], c
                while len(t.children) == 1:
                    nxt = next(iter(t.children.values()))
                    if nxt.head:
                        break
                    run.append(nxt)
                    t = nxt
                if all(x.lock == 0 for x in run):
                    total += len(run)
                stack.append(t)
        return total

    # -- structure (for assertions) ----------------------------------------
    def nodes(self) -> List[Tuple[Tuple[int, ...], Tuple[int, ...]]]:
        """Every radix node as (token path before it, its own tokens), sorted."""
        out, stack = [], [(self.root, ())]
        while stack:
            n, before = stack.pop()
            for c in n.children.values():
                own, t = [c.token], c
                while len(t.children) == 1:
                    nxt = next(iter(t.children.values()))
                    if nxt.head:
                        break
                    own.append(nxt.token)
                    t = nxt
                out.append((before, tuple(own)))
                stack.append((t, before + tuple(own)))
        return sorted(out)

    def num_nodes(self) -> int:
        return len(self.nodes())

    def sequences(self) -> List[Tuple[int, ...]]:
        """All root-to-leaf token sequences."""
        out, stack = [], [(self.root, ())]
        while stack:
            n, acc = stack.pop()
            if not n.children and n is not self.root:
                out.append(acc)
            for t, c in n.children.items():
                stack.append((c, acc + (t,)))
        return sorted(out)


# ---------------------------------------------------------------------------
# admission into a token-slot pool
# ---------------------------------------------------------------------------
# "Introducción a SGLang", RadixAttention bullet (the cache of finished calls
# is reused by later calls that share a prefix) and the nine-step walkthrough
# of "SGLang: Modelo de programación y metodología" (steps 5, 8 and 9: under
# memory pressure, least-recently-used nodes are evicted to make room, and a
# request's own matched prefix is kept).  The composition, step by step:
#   admit(tokens):  match the cached prefix (a use: clock and path), lock it
#                   (+1), and when the free list holds fewer slots than the
#                   uncached tokens, evict least-recently-used unlocked leaves
#                   for the difference and append the freed slots to the free
#                   list's tail; then take the fresh slots from its head.  If
#                   the pool still cannot hold the request, unlock and refuse.
#   commit(tokens): unlock the admitted prefix, insert the whole sequence with
#                   its slot list, and return to the free list the fresh slots
#                   of tokens that another request cached in the meantime.


class Admission:
    """A radix cache over a pool whose free slots start as ``free_order``."""

    def __init__(self, free_order: Sequence[int]):
        from collections import deque
        self.tree = RadixTreeRef()
        self.free = deque(int(x) for x in free_order)
        self.freed: List[int] = []      # every evicted slot, in eviction order

    def admit(self, tokens: Sequence[int]):
        """(slot list, cached prefix length, tokens evicted); the slot list is
        None when the pool cannot hold the request."""
        k, slots = self.tree.match_prefix(tokens)
        self.tree.lock(tokens[:k], 1)
        need = len(tokens) - k
        ev = 0
        if len(self.free) < need:
            got = self.tree.evict(need - len(self.free))
            ev = len(got)
            self.freed.extend(got)
            self.free.extend(got)
        if len(self.free) < need:
            self.tree.lock(tokens[:k], -1)
            return None, k, ev
        fresh = [self.free.popleft() for _ in range(need)]
        return list(slots) + fresh, k, ev

    def commit(self, tokens: Sequence[int], row: Sequence[int], k: int) -> None:
        self.tree.lock(tokens[:k], -1)
        c = self.tree.insert(tokens, row)
        if c > k:
            self.free.extend(int(x) for x in row[k:c])


def replay(free_order: Sequence[int], prefill: Sequence[Sequence[int]], batch: Sequence[Sequence[int]]):
    """Admit and commit every prefill sequence in order, then admit every
    batch request in order (not committed).  Returns the Admission and, per
    batch request, (slot list, cached prefix length, tokens evicted)."""
    adm = Admission(free_order)
    for toks in prefill:
        toks = [int(t) for t in toks]
        row, k, _ = adm.admit(toks)
        if row is None:
            raise ValueError("a prefill sequence does not fit the pool")
        adm.commit(toks, row, k)
    out = []
    for toks in batch:
        out.append(adm.admit([int(t) for t in toks]))
    return adm, out


# ---------------------------------------------------------------------------
# cache-aware scheduling
# ---------------------------------------------------------------------------
# "SGLang: Evaluación y resultados": the cache-aware scheduling reaches about
# 96 % of the optimal cache hit rate on average.  The pages name no policy;
# the plain reading: waiting requests with the longest cached prefix run
# first, ties in arrival order.  The hit rate is the share of prompt tokens
# found cached at admission; the optimum computes every distinct prefix token
# exactly once (an unbounded cache, one request at a time).

SCHED_FCFS = 0  # arrival order
SCHED_LPM = 1   # longest cached prefix first


def schedule(tree: RadixTreeRef, requests: Sequence[Sequence[int]], policy: int) -> Tuple[List[int], List[int]]:
    """(order to run the waiting requests in, their cached prefix lengths)."""
    lens = [tree.prefix_len(r) for r in requests]
    order = list(range(len(requests)))
    if policy == SCHED_LPM:
        order.sort(key=lambda i: (-lens[i], i))
    return order, lens


def optimal_hit_rate(requests: Sequence[Sequence[int]]) -> float:
    """1 - (distinct prefix tokens) / (prompt tokens): a token is computed
    once per distinct prefix ending in it, i.e. once per node of the
    per-token trie of all requests."""
    root: dict = {}
    distinct = total = 0
    for r in requests:
        node = root
        for t in r:
            total += 1
            nxt = node.get(t)
            if nxt is None:
                nxt = node[t] = {}
                distinct += 1
            node = nxt
    return 0.0 if total == 0 else 1.0 - distinct / total
