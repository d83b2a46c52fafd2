"""Drives the nine-step radix-tree walkthrough fixture against a tree.

The fixture is ``tests/golden/radix_walkthrough.json``.  A tree adapter
needs ``match_prefix(tokens) -> (k, slots)``, ``insert(tokens, slots) -> k``,
``evict(n) -> freed slots`` and ``nodes() -> [(before, own)]``.
"""
import json
import os

FIXTURE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "radix_walkthrough.json")


def load():
    with open(FIXTURE) as f:
        return json.load(f)


def segment_tokens(spec):
    toks, base = {}, 1000
    for name, n in spec["segments"].items():
        toks[name] = [base + i for i in range(n)]
        base += 1000
    return toks


def expand(toks, names):
    out = []
    for n in names:
        out.extend(toks[n])
    return out


def run(tree, spec=None):
    """Yields (step, request index or None, observed, expected) tuples; the
    caller asserts.  Observed/expected are dicts with matched, evicted, nodes."""
    spec = spec or load()
    toks = segment_tokens(spec)
    free = list(range(spec["capacity"]))
    for st in spec["steps"]:
        for ri, req in enumerate(st["requests"]):
            prompt = expand(toks, req["prompt"])
            full = prompt + expand(toks, req["gen"])
            k, slots = tree.match_prefix(prompt)
            need = len(full) - k
            freed = []
            if need > len(free):
                before = set(tree.nodes())
                freed = list(tree.evict(need - len(free)))
                gone = before - set(tree.nodes())
                free.extend(freed)
            else:
                gone = set()
            new = [free.pop(0) for _ in range(need)]
            cached = tree.insert(full, list(slots) + new)
            exp_evicted = [tuple(expand(toks, e)) for e in req["evicted"]]
            # freed slots arrive node by node in token order; rebuild the node
            # token runs from the order in which they were freed
            obs = {"matched": tuple(prompt[:k]), "slots_len": len(slots), "cached": cached,
                   "evicted_nodes": sorted(own for _, own in gone), "freed": freed}
            exp = {"matched": tuple(expand(toks, req["matched"])),
                   "evicted_nodes": sorted(exp_evicted), "evicted_in_order": exp_evicted}
            yield st["step"], ri, obs, exp
        exp_nodes = sorted((tuple(expand(toks, b)), tuple(expand(toks, o))) for b, o in st["nodes"])
        yield st["step"], None, {"nodes": sorted(tree.nodes())}, {"nodes": exp_nodes}
