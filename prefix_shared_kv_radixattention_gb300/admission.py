"""Replays an admission scenario (``inputs.Scenario``) through the library's
host radix cache, and builds the batch's Problem from what it hands out.

The cache is the one ``include/rx.h`` declares ("SGLang: Efficient Execution
of Structured Language Model Programs", unite.ai, es, "Introducción a
SGLang", RadixAttention bullet: an LRU cache of KV inside a radix tree; "SGLang:
Modelo de programación y metodología", nine-step walkthrough: under memory
pressure least-recently-used nodes are evicted).  Every step here is one C-ABI
call: ``rx_admit`` (prefix match, lock, fresh slots, eviction when the free
list is short) and ``rx_commit`` (insert, unlock).  This module only orders
the calls and collects their results.
"""
from __future__ import annotations

import dataclasses
from typing import List

import numpy as np

from . import binding as rx
from . import inputs


@dataclasses.dataclass
class Admitted:
    """What the cache handed out for a scenario's batch."""

    rows: List[np.ndarray]        # int32 slot list of each batch request
    prefix_lens: List[int]        # cached prefix length of each batch request
    evicted: List[int]            # tokens evicted while admitting each batch request
    prefill_evicted: int          # tokens evicted while admitting the prefill (0 when it fits)
    tree: rx.RadixTree
    alloc: rx.SlotAllocator


def replay(scn: inputs.Scenario) -> Admitted:
    """Admit and commit every prefill sequence, then admit the batch."""
    tree = rx.RadixTree()
    alloc = rx.SlotAllocator(scn.free_order, scn.num_slots)
    pre_ev = 0
    for toks in scn.prefill:
        row, k, ev = rx.rx_admit(tree, alloc, toks)
        pre_ev += ev
        rx.rx_commit(tree, alloc, toks, row, k)
    rows, ks, evs = [], [], []
    for toks in scn.batch:
        row, k, ev = rx.rx_admit(tree, alloc, toks)
        rows.append(np.array(row, np.int32))
        ks.append(int(k))
        evs.append(int(ev))
    return Admitted(rows, ks, evs, pre_ev, tree, alloc)


def mixed_chat(draw_values: bool = True, **kw) -> inputs.Problem:
    """The long multi-turn chat batch (``inputs.mixed_chat_scenario``) with
    the slot lists the library's radix cache hands out."""
    scn = inputs.mixed_chat_scenario(**kw)
    adm = replay(scn)
    return inputs.problem_from_admission(scn, adm.rows, adm.prefix_lens, draw_values)
