"""A serving loop over the host radix tree, for cache hit rates under a
scheduling policy.  Test infrastructure: it drives the C ABI (rx_schedule,
rx_admit, rx_commit) and, side by side, the same loop on the oracle trie.

The loop follows the cache-aware scheduling of "SGLang: Efficient Execution of
Structured Language Model Programs" (unite.ai, es), "SGLang: Evaluación y
resultados" (cache-aware scheduling reaches about 96 % of the optimal hit
rate), in its plain reading:

  1. order the waiting requests by the policy (arrival order, or longest
     cached prefix first);
  2. admit them in that order, up to ``batch`` of them, stopping at the first
     one the pool cannot hold (admission locks its cached prefix, so later
     admissions in the round cannot evict it);
  3. commit the round's requests (their tokens become cached) and repeat.

A request's hits are its cached prefix length at admission; the hit rate is
hits over prompt tokens, and the optimum (oracle.tree_ref.optimal_hit_rate)
computes every distinct prefix token once.

    python -m tests.serving_sim        # prints the hit rates of the workloads below
"""
from __future__ import annotations

from typing import List, Sequence

import numpy as np

from oracle.tree_ref import SCHED_FCFS, SCHED_LPM, Admission, optimal_hit_rate, schedule


class OracleAdmission(Admission):
    """rx_admit / rx_commit composed from the oracle trie and a FIFO free
    list (``oracle.tree_ref.Admission``); ``t`` is its trie."""

    @property
    def t(self):
        return self.tree


class _Native:
    def __init__(self, num_slots):
        from prefix_shared_kv_radixattention_gb300 import binding as rx
        self.rx = rx
        self.tree = rx.RadixTree()
        self.alloc = rx.SlotAllocator(np.arange(num_slots, dtype=np.int32), num_slots)

    def order(self, reqs, policy):
        order, _ = self.rx.rx_schedule(self.tree, reqs, policy)
        return [int(x) for x in order]

    def admit(self, toks):
        try:
            row, k, _ = self.rx.rx_admit(self.tree, self.alloc, toks)
        except self.rx.RxError as e:
            if e.code != self.rx.RX_ERR_NOT_ENOUGH:
                raise
            return None, 0
        return row, k

    def commit(self, toks, row, k):
        self.rx.rx_commit(self.tree, self.alloc, toks, row, k)


class _Oracle:
    def __init__(self, num_slots):
        self.adm = OracleAdmission(range(num_slots))

    def order(self, reqs, policy):
        return schedule(self.adm.t, reqs, policy)[0]

    def admit(self, toks):
        row, k, _ = self.adm.admit(toks)
        return row, k

    def commit(self, toks, row, k):
        self.adm.commit(toks, list(row), k)


def run(requests: Sequence[Sequence[int]], num_slots: int, batch: int, policy: int, side: str = "native"):
    """Per-request hits (cached prefix at admission, by arrival index) and the hit rate."""
    eng = _Native(num_slots) if side == "native" else _Oracle(num_slots)
    reqs = [list(map(int, r)) for r in requests]
    waiting = list(range(len(reqs)))
    hits = [0] * len(reqs)
    while waiting:
        order = eng.order([reqs[i] for i in waiting], policy)
        done = []
        for o in order:
            if len(done) == batch:
                break
            i = waiting[o]
            row, k = eng.admit(reqs[i])
            if row is None:
                break
            done.append((i, row, k))
        if not done:
            raise RuntimeError(f"a request of {len(reqs[waiting[order[0]]])} tokens does not fit "
                               f"{num_slots} slots")
        for i, row, k in done:
            eng.commit(reqs[i], row, k)
            hits[i] = k
        gone = {i for i, _, _ in done}
        waiting = [i for i in waiting if i not in gone]
    total = sum(len(r) for r in reqs)
    return hits, (sum(hits) / total if total else 0.0)


# ---------------------------------------------------------------------------
# synthetic request streams shaped like the pages' workload families
# ---------------------------------------------------------------------------


def few_shot(seed=2001, prompts=8, examples=200, questions=12, qlen=40) -> List[List[int]]:
    """``prompts`` few-shot prompts of ``examples`` tokens, each followed by
    ``questions`` distinct questions; arrivals rotate over the prompts."""
    rng = np.random.default_rng(seed)
    heads = [list(rng.integers(1_000_000 * (p + 1), 1_000_000 * (p + 1) + 50_000, examples)) for p in range(prompts)]
    out = []
    for q in range(questions):
        for p in range(prompts):
            out.append(heads[p] + list(rng.integers(10**8 + 10**6 * p + 1000 * q, 10**8 + 10**6 * p + 1000 * q + 999, qlen)))
    return out


def multi_turn_chat(seed=2002, sessions=12, turns=5, system=100, msg=30) -> List[List[int]]:
    """``sessions`` chats sharing one system prompt; turn t's prompt is the
    session's history (system prompt and its earlier messages) plus a new
    message; arrivals go turn by turn over the sessions."""
    rng = np.random.default_rng(seed)
    sys_toks = list(rng.integers(1, 50_000, system))
    hist = [list(sys_toks) for _ in range(sessions)]
    out = []
    for t in range(turns):
        for s in range(sessions):
            hist[s] = hist[s] + list(rng.integers(10**7 * (s + 1) + 1000 * t, 10**7 * (s + 1) + 1000 * t + 999, msg))
            out.append(list(hist[s]))
    return out


def tree_of_thought(seed=2003, root=150, step=40, fanout=3, depth=3) -> List[List[int]]:
    """A question and its branches: every tree node is a request whose prompt
    is its root path; arrivals breadth first."""
    rng = np.random.default_rng(seed)
    level = [list(rng.integers(1, 50_000, root))]
    out = [list(level[0])]
    uid = 0
    for _ in range(depth):
        nxt = []
        for node in level:
            for _ in range(fanout):
                uid += 1
                nxt.append(node + list(rng.integers(10**7 * uid, 10**7 * uid + 999, step)))
        out.extend(list(n) for n in nxt)
        level = nxt
    return out


# workload, its requests, pool slots (below the distinct tokens: eviction
# happens), batch size
WORKLOADS = {
    "few-shot": (few_shot, 1200, 8),
    "multi-turn chat": (multi_turn_chat, 900, 4),
    "tree of thought": (tree_of_thought, 900, 4),
}


def report():
    rows = []
    for name, (make, slots, batch) in WORKLOADS.items():
        reqs = make()
        opt = optimal_hit_rate(reqs)
        _, fcfs = run(reqs, slots, batch, SCHED_FCFS)
        _, lpm = run(reqs, slots, batch, SCHED_LPM)
        rows.append((name, len(reqs), sum(len(r) for r in reqs), slots, batch, fcfs, lpm, opt))
    return rows


if __name__ == "__main__":
    print("| workload | requests | prompt tokens | pool slots | batch | arrival order | longest prefix first | optimum | longest prefix first / optimum |")
    print("|---|---:|---:|---:|---:|---:|---:|---:|---:|")
    for name, n, tot, slots, batch, fcfs, lpm, opt in report():
        print(f"| {name} | {n} | {tot} | {slots} | {batch} | {fcfs:.3f} | {lpm:.3f} | {opt:.3f} | {lpm / opt:.3f} |")
