"""Pins for the fp64 attention oracle (oracle/attn_fp64.c).

The pages print no attention values, so the oracle is pinned by things
other than itself:
  * a library attention routine: torch's scaled_dot_product_attention in
    float64 on K/V gathered by numpy indexing, with an explicit causal mask
    over prefix + extend positions (the formula north of the path:
    softmax(q K^T / sqrt(d) + causal mask) V, GQA head h -> kv head h // G);
  * closed forms: one key -> o = v_0, lse = s_0; identical keys or q = 0 ->
    o = mean of the visible V rows and lse = s + ln(n); a single dominant
    logit -> o moves to that key's V row;
  * invariants: shared vs duplicated prefix slots, slot permutation, split +
    log-sum-exp merge, GQA vs replicated heads, batch order, decode = last
    extend row;
  * a mutation check: each of several plausible slips, planted in a copy of
    the oracle's source, fails at least one of the pins above.
"""
import os
import re
import shutil
import tempfile

import numpy as np
import pytest
import torch

import oracle
from prefix_shared_kv_radixattention_gb300 import inputs

TOL = 1e-12


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------


def make_pools(prob, rng_seed=7, lib=None):
    """Host pools filled with bf16 noise (so a wrong slot shows), cached rows
    placed, then the step's new rows stored by the oracle's kv_store."""
    rng = np.random.default_rng(rng_seed)
    shape = (prob.num_slots, prob.hkv, prob.d)
    kp = inputs.randn_bf16(rng, shape)
    vp = inputs.randn_bf16(rng, shape)
    kp[prob.cached_slots] = prob.cached_k
    vp[prob.cached_slots] = prob.cached_v
    oracle.kv_store(kp, vp, prob.new_k, prob.new_v, prob.new_slots, lib=lib)
    return kp, vp


def w(x):
    return inputs.bf16_to_f32(x).astype(np.float64)


def sdpa_extend(prob, kp, vp):
    """Library routine on gathered tensors: one call per request."""
    G = prob.hq // prob.hkv
    outs = []
    for b in range(len(prob.ext_req_idx)):
        P, E = int(prob.ext_prefix_len[b]), int(prob.ext_extend_len[b])
        slots = prob.req_to_token[prob.ext_req_idx[b], :P + E]
        k = torch.from_numpy(w(kp[slots])).permute(1, 0, 2).repeat_interleave(G, 0)
        v = torch.from_numpy(w(vp[slots])).permute(1, 0, 2).repeat_interleave(G, 0)
        q = torch.from_numpy(w(prob.q_ext[prob.qo_indptr[b]:prob.qo_indptr[b + 1]])).permute(1, 0, 2)
        mask = torch.arange(P + E)[None, :] <= (P + torch.arange(E))[:, None]
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask,
                                                             scale=prob.sm_scale)
        outs.append(o.permute(1, 0, 2).numpy())
    return np.concatenate(outs, 0)


def sdpa_decode(prob, kp, vp):
    G = prob.hq // prob.hkv
    outs = []
    for b in range(len(prob.dec_req_idx)):
        L = int(prob.dec_seq_len[b])
        slots = prob.req_to_token[prob.dec_req_idx[b], :L]
        k = torch.from_numpy(w(kp[slots])).permute(1, 0, 2).repeat_interleave(G, 0)
        v = torch.from_numpy(w(vp[slots])).permute(1, 0, 2).repeat_interleave(G, 0)
        q = torch.from_numpy(w(prob.q_dec[b:b + 1])).permute(1, 0, 2)
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=prob.sm_scale)
        outs.append(o.permute(1, 0, 2).numpy())
    return np.concatenate(outs, 0)


def run_extend(prob, kp, vp, lib=None):
    return oracle.extend(prob.q_ext, kp, vp, prob.req_to_token, prob.ext_req_idx,
                         prob.ext_prefix_len, prob.ext_extend_len, prob.qo_indptr, prob.sm_scale,
                         lib=lib)


def run_decode(prob, kp, vp, lib=None):
    return oracle.decode(prob.q_dec, kp, vp, prob.req_to_token, prob.dec_req_idx, prob.dec_seq_len,
                         prob.sm_scale, lib=lib)


def gqa_ext_problem(seed=11):
    return inputs.ragged(seed, hq=8, hkv=2, d=64, n_groups=2, per_group=2, shared_max=20,
                         private_max=9, extend_max=7, decode=False, num_slots=400)


def gqa_dec_problem(seed=12):
    return inputs.ragged(seed, hq=8, hkv=2, d=64, n_groups=2, per_group=3, shared_max=30,
                         private_max=12, extend_max=1, decode=True, num_slots=400)


# ---------------------------------------------------------------------------
# pin suites (shared with the mutation check)
# ---------------------------------------------------------------------------


def pin_library_routine(lib=None):
    for prob in (gqa_ext_problem(), inputs.tiny_extend(hq=2, hkv=2, batch=2, prefix=5, extend=6,
                                                       num_slots=64)):
        kp, vp = make_pools(prob, lib=lib)
        o, _ = run_extend(prob, kp, vp, lib)
        ref = sdpa_extend(prob, kp, vp)
        if not np.max(np.abs(o - ref)) <= TOL:
            return False
    prob = gqa_dec_problem()
    kp, vp = make_pools(prob, lib=lib)
    o, _ = run_decode(prob, kp, vp, lib)
    return bool(np.max(np.abs(o - sdpa_decode(prob, kp, vp))) <= TOL)


def _single_row_problem(L, hq=2, hkv=1, d=64, seed=5):
    """One decode row of length L over slots 3, 4, ... in a small pool."""
    rng = np.random.default_rng(seed)
    S = L + 8
    kp = inputs.randn_bf16(rng, (S, hkv, d))
    vp = inputs.randn_bf16(rng, (S, hkv, d))
    rtt = np.full((1, L + 4), -1, np.int32)
    rtt[0, :L] = 3 + np.arange(L)
    q = inputs.randn_bf16(rng, (1, hq, d))
    return kp, vp, rtt, q


def pin_closed_forms(lib=None):
    d = 64
    scale = 1.0 / np.sqrt(d)
    # one key: o = v_0 exactly, lse = s_0
    kp, vp, rtt, q = _single_row_problem(1)
    o, lse = oracle.decode(q, kp, vp, rtt, [0], [1], scale, lib=lib)
    s0 = np.sum(w(q[0]) * w(kp[3, 0])[None, :], axis=-1) * scale
    if not (np.array_equal(o[0], np.broadcast_to(w(vp[3, 0]), o[0].shape)) and
            np.max(np.abs(lse[0] - s0)) <= TOL):
        return False
    # identical keys: uniform weights -> mean of V, lse = s + ln n
    L = 37
    kp, vp, rtt, q = _single_row_problem(L)
    kp[:] = kp[3]
    o, lse = oracle.decode(q, kp, vp, rtt, [0], [L], scale, lib=lib)
    mean_v = np.mean(w(vp[3:3 + L, 0]), axis=0)
    s = np.sum(w(q[0]) * w(kp[3, 0])[None, :], axis=-1) * scale
    if not (np.max(np.abs(o[0] - mean_v[None, :])) <= TOL and
            np.max(np.abs(lse[0] - (s + np.log(L)))) <= TOL):
        return False
    # q = 0 -> mean of V, lse = ln n, whatever K holds
    kp, vp, rtt, q = _single_row_problem(L, seed=9)
    q[:] = 0
    o, lse = oracle.decode(q, kp, vp, rtt, [0], [L], scale, lib=lib)
    if not (np.max(np.abs(o[0] - np.mean(w(vp[3:3 + L, 0]), axis=0)[None, :])) <= TOL and
            np.max(np.abs(lse[0] - np.log(L))) <= TOL):
        return False
    # a dominant logit at key position jstar: q = e_0, k_jstar = 64 e_0, others 0
    # (all exact in bf16): s_jstar = 64 * scale, s_other = 0
    kp, vp, rtt, q = _single_row_problem(L, seed=13)
    jstar = 21
    q[:] = 0
    q[..., 0] = inputs.bf16_round(np.float32([1.0]))[0]
    kp[:] = 0
    kp[3 + jstar, 0, 0] = inputs.bf16_round(np.float32([64.0]))[0]
    o, lse = oracle.decode(q, kp, vp, rtt, [0], [L], scale, lib=lib)
    big = np.exp(64.0 * scale)
    V = w(vp[3:3 + L, 0])
    want = (big * V[jstar] + (V.sum(0) - V[jstar])) / (big + L - 1)
    return bool(np.max(np.abs(o[0] - want[None, :])) <= TOL and
                np.max(np.abs(lse[0] - np.log(big + L - 1))) <= TOL)


def pin_split_merge(lib=None):
    """Partials over a split of 0..L-1 merged by the LSE identity equal the whole."""
    prob = gqa_dec_problem()
    kp, vp = make_pools(prob, lib=lib)
    o, lse = run_decode(prob, kp, vp, lib)
    n = len(prob.dec_req_idx)
    cuts = []
    for L in prob.dec_seq_len:
        a = max(1, L // 3)
        b = max(a + 1, (2 * L) // 3) if L > 2 else a
        cuts.append([0, a, b, L] if L > 2 else [0, L])
    o_all, l_all = [], []
    for part in range(3):
        kb = np.array([c[min(part, len(c) - 2)] for c in cuts], np.int32)
        ke = np.array([c[min(part, len(c) - 2) + 1] for c in cuts], np.int32)
        op, lp = oracle.attention(prob.q_dec, kp, vp, prob.req_to_token, prob.dec_req_idx, kb, ke,
                                  prob.sm_scale, lib=lib)
        o_all.append(op)
        l_all.append(lp)
    # rows with L <= 2 repeated the single part; keep only distinct parts
    om, lm = np.empty_like(o), np.empty_like(lse)
    for r in range(n):
        k = len(cuts[r]) - 1
        parts_o = np.stack([o_all[i][r] for i in range(k)], axis=-2)
        parts_l = np.stack([l_all[i][r] for i in range(k)], axis=-1)
        om[r], lm[r] = oracle.merge_partials(parts_o, parts_l)
    return bool(np.max(np.abs(om - o)) <= TOL and np.max(np.abs(lm - lse)) <= TOL)


PIN_SUITES = [pin_library_routine, pin_closed_forms, pin_split_merge]


# ---------------------------------------------------------------------------
# the pins as tests
# ---------------------------------------------------------------------------


def test_library_routine():
    assert pin_library_routine()


def test_closed_forms():
    assert pin_closed_forms()


def test_split_merge():
    assert pin_split_merge()


def test_sharing_equals_duplication():
    """I1: a shared prefix gives bit-identical output to private copies of it."""
    prob = inputs.ragged(21, hq=4, hkv=2, d=64, n_groups=1, per_group=3, shared_max=25,
                         private_max=5, extend_max=6, decode=False, num_slots=300,
                         allow_empty_prefix=False)
    kp, vp = make_pools(prob)
    o1, l1 = run_extend(prob, kp, vp)
    # copy every request's prefix rows into fresh slots of a bigger pool
    rtt = prob.req_to_token.copy()
    extra = sum(int(P) for P in prob.ext_prefix_len)
    S2 = prob.num_slots + extra
    kp2 = np.zeros((S2, prob.hkv, prob.d), np.uint16)
    vp2 = np.zeros_like(kp2)
    kp2[:prob.num_slots], vp2[:prob.num_slots] = kp, vp
    nxt = prob.num_slots
    for b, P in enumerate(prob.ext_prefix_len):
        for j in range(int(P)):
            kp2[nxt], vp2[nxt] = kp[rtt[b, j]], vp[rtt[b, j]]
            rtt[b, j] = nxt
            nxt += 1
    o2, l2 = oracle.extend(prob.q_ext, kp2, vp2, rtt, prob.ext_req_idx, prob.ext_prefix_len,
                           prob.ext_extend_len, prob.qo_indptr, prob.sm_scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_slot_permutation():
    """I2: permuting pool rows and remapping req_to_token changes nothing."""
    prob = gqa_ext_problem(31)
    kp, vp = make_pools(prob)
    o1, l1 = run_extend(prob, kp, vp)
    perm = np.random.default_rng(3).permutation(prob.num_slots)
    kp2, vp2 = np.empty_like(kp), np.empty_like(vp)
    kp2[perm], vp2[perm] = kp, vp          # row s moves to perm[s]
    rtt = np.where(prob.req_to_token >= 0, perm[np.maximum(prob.req_to_token, 0)], -1).astype(np.int32)
    o2, l2 = oracle.extend(prob.q_ext, kp2, vp2, rtt, prob.ext_req_idx, prob.ext_prefix_len,
                           prob.ext_extend_len, prob.qo_indptr, prob.sm_scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_gqa_equals_replicated_heads():
    """I4: GQA equals MHA with each kv head replicated over its q-head group."""
    prob = gqa_dec_problem(41)
    kp, vp = make_pools(prob)
    o1, l1 = run_decode(prob, kp, vp)
    G = prob.hq // prob.hkv
    kp2 = np.ascontiguousarray(np.repeat(kp, G, axis=1))
    vp2 = np.ascontiguousarray(np.repeat(vp, G, axis=1))
    o2, l2 = oracle.decode(prob.q_dec, kp2, vp2, prob.req_to_token, prob.dec_req_idx,
                           prob.dec_seq_len, prob.sm_scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_batch_order():
    """I6: permuting the batch permutes the output rows."""
    prob = gqa_dec_problem(51)
    kp, vp = make_pools(prob)
    o1, l1 = run_decode(prob, kp, vp)
    p = np.random.default_rng(1).permutation(len(prob.dec_req_idx))
    o2, l2 = oracle.decode(prob.q_dec[p], kp, vp, prob.req_to_token, prob.dec_req_idx[p],
                           prob.dec_seq_len[p], prob.sm_scale)
    assert np.array_equal(o1[p], o2) and np.array_equal(l1[p], l2)


def test_decode_is_last_extend_row():
    prob = gqa_ext_problem(61)
    kp, vp = make_pools(prob)
    o, lse = run_extend(prob, kp, vp)
    last = prob.qo_indptr[1:] - 1
    od, ld = oracle.decode(prob.q_ext[last], kp, vp, prob.req_to_token, prob.ext_req_idx,
                           prob.ext_prefix_len + prob.ext_extend_len, prob.sm_scale)
    assert np.array_equal(o[last], od) and np.array_equal(lse[last], ld)


def test_prefix_zero_is_standard_causal():
    """P = 0: plain causal self-attention (library is_causal path)."""
    prob = inputs.tiny_extend(seed=3, hq=4, hkv=4, d=64, batch=1, prefix=0, extend=33, num_slots=64)
    kp, vp = make_pools(prob)
    o, _ = run_extend(prob, kp, vp)
    slots = prob.req_to_token[0, :33]
    q = torch.from_numpy(w(prob.q_ext)).permute(1, 0, 2)
    k = torch.from_numpy(w(kp[slots])).permute(1, 0, 2)
    v = torch.from_numpy(w(vp[slots])).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True,
                                                           scale=prob.sm_scale)
    assert np.max(np.abs(o - ref.permute(1, 0, 2).numpy())) <= TOL


def test_thread_count_does_not_change_result():
    prob = gqa_ext_problem(71)
    kp, vp = make_pools(prob)
    a = oracle.extend(prob.q_ext, kp, vp, prob.req_to_token, prob.ext_req_idx, prob.ext_prefix_len,
                      prob.ext_extend_len, prob.qo_indptr, prob.sm_scale, n_threads=1)
    b = oracle.extend(prob.q_ext, kp, vp, prob.req_to_token, prob.ext_req_idx, prob.ext_prefix_len,
                      prob.ext_extend_len, prob.qo_indptr, prob.sm_scale, n_threads=5)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_kv_store_definition():
    rng = np.random.default_rng(2)
    kp = inputs.randn_bf16(rng, (50, 3, 16))
    vp = inputs.randn_bf16(rng, (50, 3, 16))
    kn = inputs.randn_bf16(rng, (7, 3, 16))
    vn = inputs.randn_bf16(rng, (7, 3, 16))
    slots = rng.permutation(50)[:7].astype(np.int32)
    ek, ev = kp.copy(), vp.copy()
    ek[slots], ev[slots] = kn, vn          # numpy's indexed assignment
    oracle.kv_store(kp, vp, kn, vn, slots)
    assert np.array_equal(kp, ek) and np.array_equal(vp, ev)
    with pytest.raises(ValueError):
        oracle.kv_store(kp, vp, kn[:1], vn[:1], np.array([50], np.int32))
    with pytest.raises(ValueError):
        oracle.kv_store(kp, vp, kn[:2], vn[:2], np.array([4, 4], np.int32))
    oracle.kv_store(kp, vp, kn[:0], vn[:0], np.zeros(0, np.int32))
    assert np.array_equal(kp, ek)


def test_merge_single_part_is_identity():
    rng = np.random.default_rng(0)
    o = rng.standard_normal((3, 1, 8))
    lse = rng.standard_normal((3, 1))
    om, lm = oracle.merge_partials(o, lse)
    assert np.array_equal(om, o[:, 0]) and np.array_equal(lm, lse[:, 0])


# ---------------------------------------------------------------------------
# mutation check: plausible slips in the oracle must be caught by the pins
# ---------------------------------------------------------------------------

MUTANTS = {
    "dropped_scale": ("s[j - j0] = dot * J->sm_scale;", "s[j - j0] = dot;"),
    "wrong_gqa_map": ("int g = h / G; ", "int g = h % J->hkv; "),
    "q_head_index": ("(t * J->hq + h) * (int64_t)J->d", "(t * J->hq + g) * (int64_t)J->d"),
    "v_from_k_pool": ("const uint16_t *v = J->v_pool", "const uint16_t *v = J->k_pool"),
    "drops_diagonal": ("j1 = J->kend[t];", "j1 = J->kend[t] - (J->kend[t] - J->kbeg[t] > 1);"),
    "lse_without_max": ("J->lse[item] = m + log(wsum);", "J->lse[item] = log(wsum);"),
    "unshifted_weights": ("double w = exp(s[j - j0] - m);", "double w = exp(s[j - j0] - m * 0.5);"),
    "first_key_skipped": ("double m = s[0]; ", "double m = s[0]; s[0] = -1e300; "),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name):
    src = open(oracle._SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"anchor for {name} not unique in oracle source"
    tmp = tempfile.mkdtemp()
    try:
        path = os.path.join(tmp, "mut.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        lib = oracle.load(oracle.build(path, os.path.join(tmp, "libmut.so")))
        caught = []
        for suite in PIN_SUITES:
            try:
                caught.append(not suite(lib))
            except Exception:
                caught.append(True)
        assert any(caught), f"mutant {name} survived every pin"
    finally:
        shutil.rmtree(tmp)


# ---------------------------------------------------------------------------
# rotary position embedding
# ---------------------------------------------------------------------------


def test_rope_position_zero_is_identity():
    x = np.random.default_rng(1).standard_normal((3, 2, 8))
    assert np.array_equal(oracle.rope_f64(x, [0, 0, 0], 10000.0), x)


def test_rope_worked_example():
    """d = 4, base 100: pairs (0, 2) and (1, 3) turn by theta_0 = 1 and
    theta_1 = 100^(-1/2) = 0.1 radians per position.  At position 1 the unit
    vector e0 goes to (cos 1, 0, sin 1, 0) and e1 to (0, cos 0.1, 0, sin 0.1);
    at position 2, e2 goes to (-sin 2, 0, cos 2, 0)."""
    e = np.eye(4).reshape(4, 1, 4)
    out = oracle.rope_f64(e, [1, 1, 2, 0], 100.0)
    assert np.allclose(out[0, 0], [np.cos(1), 0, np.sin(1), 0], atol=1e-15)
    assert np.allclose(out[1, 0], [0, np.cos(0.1), 0, np.sin(0.1)], atol=1e-15)
    assert np.allclose(out[2, 0], [-np.sin(2), 0, np.cos(2), 0], atol=1e-15)
    assert np.allclose(out[3, 0], [0, 0, 0, 1], atol=1e-15)


def test_rope_keeps_pair_norms_and_composes():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((5, 3, 16))
    pos = np.array([0, 7, 100, 4095, 32768])
    y = oracle.rope_f64(x, pos, 10000.0)
    half = 8
    assert np.allclose(x[..., :half] ** 2 + x[..., half:] ** 2, y[..., :half] ** 2 + y[..., half:] ** 2)
    # rotations compose: turning by a then by b is turning by a + b
    z = oracle.rope_f64(oracle.rope_f64(x, pos, 10000.0), [3, 3, 3, 3, 3], 10000.0)
    assert np.allclose(z, oracle.rope_f64(x, pos + 3, 10000.0), atol=1e-9)


def test_rope_scores_depend_on_relative_position():
    """q at position p and k at position p - r give the same score for every
    p: the property that makes the embedding relative."""
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 1, 32))
    k = rng.standard_normal((1, 1, 32))
    r = 5
    scores = [float(np.sum(oracle.rope_f64(q, [p], 500000.0) * oracle.rope_f64(k, [p - r], 500000.0)))
              for p in (5, 40, 1000, 30000)]
    assert np.allclose(scores, scores[0], rtol=0, atol=1e-9)


def test_rope_from_bf16_bits():
    x = np.array([[[0x3F80, 0x0000, 0x4000, 0xBF80]]], np.uint16)  # 1, 0, 2, -1
    out = oracle.rope(x, [0], 10000.0)
    assert np.array_equal(out, np.array([[[1.0, 0.0, 2.0, -1.0]]]))
