"""Reference image keys for the radix tree.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

"SGLang: Efficient Execution of Structured Language Model Programs" (unite.ai,
es), "SGLang: Evaluación y resultados", multimodal results: RadixAttention uses
the hash of an input image as its key in the radix tree.  Reading taken (the
pages name no hash): the 64-bit FNV-1a hash of the image's bytes seeds a
SplitMix64 generator, and output i + 1, with the top bit set, is the key of the
image's token i.  Both are published definitions, written out here in plain
Python integers.
"""
from __future__ import annotations

from typing import List

_M64 = (1 << 64) - 1


def fnv1a64(data: bytes) -> int:
    """FNV-1a, 64 bits: start at the offset basis; per byte, xor it in, then
    multiply by the FNV prime (mod 2^64)."""
    h = 0xCBF29CE484222325
    for b in data:
        h ^= b
        h = (h * 0x100000001B3) & _M64
    return h


def splitmix64(seed: int, count: int) -> List[int]:
    """The first ``count`` outputs of SplitMix64 from ``seed``: the state
    advances by 0x9e3779b97f4a7c15 and each new state goes through the
    finaliser z ^= z >> 30; z *= 0xbf58476d1ce4e5b9; z ^= z >> 27;
    z *= 0x94d049bb133111eb; z ^= z >> 31 (mod 2^64)."""
    out, state = [], seed & _M64
    for _ in range(count):
        state = (state + 0x9E3779B97F4A7C15) & _M64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
        out.append(z ^ (z >> 31))
    return out


def image_keys(data: bytes, n_tokens: int) -> List[int]:
    """Keys (as signed int64 values) of an image's n_tokens positions."""
    keys = []
    for z in splitmix64(fnv1a64(data), n_tokens):
        z |= 1 << 63
        keys.append(z - (1 << 64))  # the same 64 bits read as int64
    return keys
