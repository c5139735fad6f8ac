"""Pins for the fp64 oracle: checks against what the definitions fix, independent of the oracle itself.

Every pin is a closed form, an invariant, a special case that reduces to a plain mean, or brute force
on a tiny input.  ``test_mutations_are_caught`` compiles deliberately broken copies of the oracle's C
source (a dropped scale, a wrong sign, a shifted causal limit, an interleaved head mapping, a reversed
tie-break, ...) and checks that at least one pin fails for each, so a plausible slip anywhere in the
oracle cannot pass unnoticed.
"""
import itertools
import os
import shutil
import subprocess
import sys
import tempfile

import numpy as np
import pytest
import torch

import oracle
import synth
from tests import golden_util as gu

TOL = 1e-12


def _rand_bf16(shape, seed, stream):
    return synth.normal_bf16(seed, synth.stream_id(901, stream), shape)


# ----------------------------------------------------------------------------------------------
# pins (each takes an optional oracle library handle so mutated builds can be checked)

def pin_golden_focal(lib=None):
    for case in gu.load()["focal_cases"]:
        q, k, v, length = gu.focal_case_tensors(case)
        out, sc = oracle.focal(k, v, length, q, q_pos0=case["q_pos0"], cand=tuple(case["cand"]), lib=lib)
        for key, dim, expr in case["out"]:
            b, g, i = (int(x) for x in key.split(","))
            assert abs(out[b, g, i, dim] - gu.ev(expr)) < TOL, (case["name"], key, dim)
        for key, j, expr in case["scores"]:
            b, h = (int(x) for x in key.split(","))
            assert abs(sc[b, h, j] - gu.ev(expr)) < TOL, (case["name"], key, j)


def pin_golden_topk(lib=None):
    for case in gu.load()["topk_cases"]:
        got = oracle.topk(np.array([case["scores"]]), case["k"], lib=lib)[0]
        assert got.tolist() == case["expect"], case["name"]


def pin_golden_sparse(lib=None):
    d = 128
    for case in gu.load()["sparse_cases"]:
        T = case["T"]
        k = torch.zeros((1, 1, T, d), dtype=torch.bfloat16)
        v = torch.zeros((1, 1, T, d), dtype=torch.float32)
        v[0, 0, :, 0] = torch.tensor(case["v_row_value"])
        v = v.to(torch.bfloat16)
        q = torch.zeros((1, 1, 1, d), dtype=torch.bfloat16)
        q[0, 0, 0, 0] = 1.0
        idx = torch.tensor(case["idx"], dtype=torch.int32).view(1, 1, -1)
        out = oracle.sparse_decode(k, v, torch.tensor(case["len"], dtype=torch.int32), q, idx,
                                   case["tail_lo"], lib=lib)
        assert abs(out[0, 0, 0, 0] - gu.ev(case["expect_dim0"])) < TOL, case["name"]


def pin_golden_shared_prefix(lib=None):
    d = 128
    for case in gu.load()["shared_prefix_cases"]:
        P, off, Mq = case["P"], case["off"], case["Mq"]
        Br = len(off) - 1
        pk = torch.zeros((1, P, d), dtype=torch.bfloat16)
        pv = torch.zeros((1, P, d))
        pv[0, :, 0] = torch.tensor(case["prefix_v"])
        S = off[-1]
        sk = torch.zeros((1, S, d), dtype=torch.bfloat16)
        sv = torch.zeros((1, S, d))
        sv[0, :, 0] = torch.tensor(case["suffix_v"])
        dk = torch.zeros((Br, Mq, 1, d), dtype=torch.bfloat16)
        dv = torch.zeros((Br, Mq, 1, d))
        dv[:, :, 0, 0] = torch.tensor(case["draft_v"])
        q = torch.zeros((Br, 1, Mq, d), dtype=torch.bfloat16)
        out = oracle.shared_prefix(pk, pv.bfloat16(), sk, sv.bfloat16(), torch.tensor(off), dk,
                                   dv.bfloat16(), q, lib=lib)
        for key, expr in case["expect_dim0"].items():
            b, i = (int(x) for x in key.split(","))
            assert abs(out[b, 0, i, 0] - gu.ev(expr)) < TOL, (case["name"], key)


def pin_uniform_keys_give_mean(lib=None):
    """Identical keys make every softmax uniform: out = mean of the visible V rows, s_j = R / len."""
    B, Hkv, G, T, d = 3, 2, 2, 37, 128
    row = _rand_bf16((d,), 1, 1)
    k = row.view(1, 1, 1, d).expand(B, Hkv, T, d).contiguous()
    v = _rand_bf16((B, Hkv, T, d), 1, 2)
    q = _rand_bf16((B, Hkv * G, 1, d), 1, 3)
    length = torch.tensor([37, 1, 20], dtype=torch.int32)
    out, sc = oracle.focal(k, v, length, q, lib=lib)
    vf = v.double().numpy()
    for b in range(B):
        n = int(length[b])
        for g in range(Hkv * G):
            mean = vf[b, g // G, :n].mean(axis=0)
            assert np.max(np.abs(out[b, g, 0] - mean)) < TOL
        for h in range(Hkv):
            assert np.max(np.abs(sc[b, h, :n] - G / n)) < TOL
            assert np.all(sc[b, h, n:] == 0.0)


def pin_importance_sums_to_rows(lib=None):
    """Each query row's probabilities sum to 1, so the importance summed over all tokens is R = G*Mq."""
    B, Hkv, G, Mq, T, d = 2, 2, 4, 3, 50, 128
    k = _rand_bf16((B, Hkv, T, d), 2, 1)
    v = _rand_bf16((B, Hkv, T, d), 2, 2)
    q = _rand_bf16((B, Hkv * G, Mq, d), 2, 3)
    length = torch.tensor([50, 33], dtype=torch.int32)
    for pos0 in (-1, 10):
        _, sc = oracle.focal(k, v, length, q, q_pos0=pos0, lib=lib)
        assert np.max(np.abs(sc.sum(axis=-1) - G * Mq)) < 1e-12


def pin_single_key_and_dominant_key(lib=None):
    B, Hkv, G, T, d = 1, 1, 2, 8, 128
    v = _rand_bf16((B, Hkv, T, d), 3, 2)
    q = torch.zeros((B, G, 1, d), dtype=torch.bfloat16)
    q[..., 0] = 1.0
    k = torch.zeros((B, Hkv, T, d), dtype=torch.bfloat16)
    out, sc = oracle.focal(k, v, torch.tensor([1], dtype=torch.int32), q, lib=lib)
    assert np.array_equal(out[0, 0, 0], v[0, 0, 0].double().numpy())
    assert sc[0, 0, 0] == pytest.approx(G, abs=1e-15)
    k[0, 0, 5, 0] = 64.0 * 11.3125          # logit = 64*11.3125/sqrt(128) ~ 64
    _, sc = oracle.focal(k, v, torch.tensor([T], dtype=torch.int32), q, lib=lib)
    assert sc[0, 0, 5] == pytest.approx(G, rel=1e-20, abs=1e-20) or abs(sc[0, 0, 5] - G) < 1e-20
    assert np.all(sc[0, 0, [0, 1, 2, 3, 4, 6, 7]] < 1e-26)


def pin_topk_brute_force(lib=None):
    rng = np.random.default_rng(7)
    for n in (1, 2, 5, 9, 16):
        for trial in range(4):
            s = rng.integers(0, 4, size=(3, n)).astype(np.float64) * 0.25   # many ties
            for k in range(1, n + 1):
                got = oracle.topk(s, k, lib=lib)
                for r in range(3):
                    order = sorted(range(n), key=lambda j: (-s[r, j], j))
                    assert got[r].tolist() == sorted(order[:k]), (n, k, r)


def pin_sparse_full_set_equals_dense(lib=None):
    B, Hkv, G, T, d = 2, 2, 2, 41, 128
    k = _rand_bf16((B, Hkv, T, d), 4, 1)
    v = _rand_bf16((B, Hkv, T, d), 4, 2)
    q = _rand_bf16((B, Hkv * G, 1, d), 4, 3)
    length = torch.tensor([T, T], dtype=torch.int32)
    dense, _ = oracle.focal(k, v, length, q, want_scores=False, lib=lib)
    full = torch.arange(T, dtype=torch.int32).view(1, 1, T).expand(B, Hkv, T).contiguous()
    a = oracle.sparse_decode(k, v, length, q, full, T, lib=lib)
    assert np.max(np.abs(a - dense)) < TOL
    b = oracle.sparse_decode(k, v, length, q, None, 0, lib=lib)
    assert np.max(np.abs(b - dense)) < TOL
    split = torch.arange(17, dtype=torch.int32).view(1, 1, 17).expand(B, Hkv, 17).contiguous()
    c = oracle.sparse_decode(k, v, length, q, split, 17, lib=lib)
    assert np.max(np.abs(c - dense)) < TOL
    perm = torch.from_numpy(np.random.default_rng(1).permutation(T).astype(np.int32))
    shuffled = perm.view(1, 1, T).expand(B, Hkv, T).contiguous()
    e = oracle.sparse_decode(k, v, length, q, shuffled, T, lib=lib)
    assert np.max(np.abs(e - dense)) < 1e-13


def pin_compaction_equals_sparse(lib=None):
    """Attention over the compacted cache equals attention over the same index set in place."""
    B, Hkv, G, T, d = 2, 3, 2, 30, 128
    k = _rand_bf16((B, Hkv, T, d), 5, 1)
    v = _rand_bf16((B, Hkv, T, d), 5, 2)
    q = _rand_bf16((B, Hkv * G, 1, d), 5, 3)
    length = torch.tensor([30, 26], dtype=torch.int32)
    kk, tail_lo = 6, 22
    idx = torch.stack([torch.stack([torch.sort(torch.from_numpy(
        np.random.default_rng(b * 10 + h).choice(tail_lo, kk, replace=False).astype(np.int32))).values
        for h in range(Hkv)]) for b in range(B)])
    ck, cv, cl = oracle.kv_compact(k, v, length, idx, tail_lo, cap=kk + T - tail_lo, lib=lib)
    assert cl.tolist() == [kk + 8, kk + 4]
    for b in range(B):
        for h in range(Hkv):
            rows = idx[b, h].tolist() + list(range(tail_lo, int(length[b])))
            assert torch.equal(ck[b, h, :len(rows)], k[b, h, rows])
            assert torch.equal(cv[b, h, :len(rows)], v[b, h, rows])
    a = oracle.sparse_decode(k, v, length, q, idx, tail_lo, lib=lib)
    c = oracle.sparse_decode(ck, cv, cl, q, None, 0, lib=lib)
    assert np.array_equal(a, c)


def _concat_branch(pk, pv, sk, sv, off, dk, dv, b, prefix_idx=None):
    Hkv = pk.shape[0]
    ks, vs = [], []
    for h in range(Hkv):
        rows = prefix_idx[b, h].long() if prefix_idx is not None else torch.arange(pk.shape[1])
        ks.append(torch.cat([pk[h, rows], sk[h, off[b]:off[b + 1]], dk[b, :, h]]))
        vs.append(torch.cat([pv[h, rows], sv[h, off[b]:off[b + 1]], dv[b, :, h]]))
    return torch.stack(ks).unsqueeze(0).contiguous(), torch.stack(vs).unsqueeze(0).contiguous()


def pin_shared_prefix_equals_concatenation(lib=None):
    Hkv, G, P, Mq, Br, d = 2, 2, 12, 3, 3, 128
    lens = [0, 5, 2]
    off = [0]
    for L in lens:
        off.append(off[-1] + L)
    pk, pv = _rand_bf16((Hkv, P, d), 6, 1), _rand_bf16((Hkv, P, d), 6, 2)
    sk, sv = _rand_bf16((Hkv, off[-1], d), 6, 3), _rand_bf16((Hkv, off[-1], d), 6, 4)
    dk, dv = _rand_bf16((Br, Mq, Hkv, d), 6, 5), _rand_bf16((Br, Mq, Hkv, d), 6, 6)
    q = _rand_bf16((Br, Hkv * G, Mq, d), 6, 7)
    pidx = torch.stack([torch.stack([torch.sort(torch.from_numpy(np.random.default_rng(b * 7 + h).choice(
        P, 4, replace=False).astype(np.int32))).values for h in range(Hkv)]) for b in range(Br)])
    offt = torch.tensor(off, dtype=torch.int32)
    for pi in (None, pidx):
        got = oracle.shared_prefix(pk, pv, sk, sv, offt, dk, dv, q, pi, lib=lib)
        for b in range(Br):
            ck, cv = _concat_branch(pk, pv, sk, sv, off, dk, dv, b, pi)
            n = ck.shape[2]
            ref, _ = oracle.focal(ck, cv, torch.tensor([n], dtype=torch.int32), q[b:b + 1].contiguous(),
                                  q_pos0=n - Mq, want_scores=False, lib=lib)
            assert np.max(np.abs(got[b] - ref[0])) < TOL, (b, pi is None)


def pin_forked_branches_equal_concatenation(lib=None):
    """Branches forked at different prefix positions (HPD-Parsing part 2: a content branch sees the
    shared context up to its fork position) with suffixes in fixed, non-adjacent slots equal attention
    over each branch's explicitly concatenated cache."""
    Hkv, G, P, Mq, Br, d, slot = 2, 2, 15, 2, 4, 128, 6
    pre_len = [15, 4, 0, 9]
    suf_len = [0, 6, 3, 1]
    off = [b * slot for b in range(Br)]
    pk, pv = _rand_bf16((Hkv, P, d), 8, 1), _rand_bf16((Hkv, P, d), 8, 2)
    sk, sv = _rand_bf16((Hkv, Br * slot, d), 8, 3), _rand_bf16((Hkv, Br * slot, d), 8, 4)
    dk, dv = _rand_bf16((Br, Mq, Hkv, d), 8, 5), _rand_bf16((Br, Mq, Hkv, d), 8, 6)
    q = _rand_bf16((Br, Hkv * G, Mq, d), 8, 7)
    got = oracle.shared_prefix(pk, pv, sk, sv, torch.tensor(off, dtype=torch.int32), dk, dv, q,
                               pre_len=torch.tensor(pre_len, dtype=torch.int32),
                               suf_len=torch.tensor(suf_len, dtype=torch.int32), lib=lib)
    for b in range(Br):
        ck = torch.stack([torch.cat([pk[h, :pre_len[b]], sk[h, off[b]:off[b] + suf_len[b]], dk[b, :, h]])
                          for h in range(Hkv)]).unsqueeze(0).contiguous()
        cv = torch.stack([torch.cat([pv[h, :pre_len[b]], sv[h, off[b]:off[b] + suf_len[b]], dv[b, :, h]])
                          for h in range(Hkv)]).unsqueeze(0).contiguous()
        n = ck.shape[2]
        ref, _ = oracle.focal(ck, cv, torch.tensor([n], dtype=torch.int32), q[b:b + 1].contiguous(),
                              q_pos0=n - Mq, want_scores=False, lib=lib)
        assert np.max(np.abs(got[b] - ref[0])) < TOL, b


# Focal-layer profiling (FastOCR, Focal-Guided Pruning: Focal Layer Selection), pinned without
# reference to how focal_mass / choose_focal_layers are written.

def pin_focal_mass_whole_range_is_one(lib=None, mass_fn=None):
    """With every visible token a candidate, each of the R softmax rows puts all of its attention on the
    candidates: the share is exactly 1."""
    mass_fn = mass_fn or oracle.focal_mass
    B, Hkv, G, Mq, T = 2, 2, 2, 3, 37
    k, v = _rand_bf16((B, Hkv, T, 128), 31, 1), _rand_bf16((B, Hkv, T, 128), 31, 2)
    q = _rand_bf16((B, Hkv * G, Mq, 128), 31, 3)
    length = torch.tensor([T, 20], dtype=torch.int32)
    _, sc = oracle.focal(k, v, length, q, cand=(0, T), want_out=False, lib=lib)
    m = mass_fn(sc, G * Mq)
    assert np.all(np.abs(m - 1.0) < 1e-12), m


def pin_focal_mass_uniform_attention(lib=None, mass_fn=None):
    """q = 0 gives uniform attention over the len visible tokens: the share of the first n_img of them
    is n_img / len."""
    mass_fn = mass_fn or oracle.focal_mass
    B, Hkv, G, Mq, T, n_img = 1, 2, 4, 2, 50, 30
    k, v = _rand_bf16((B, Hkv, T, 128), 32, 1), _rand_bf16((B, Hkv, T, 128), 32, 2)
    q = torch.zeros((B, Hkv * G, Mq, 128), dtype=torch.bfloat16)
    length = torch.tensor([40], dtype=torch.int32)
    _, sc = oracle.focal(k, v, length, q, cand=(0, n_img), want_out=False, lib=lib)
    m = mass_fn(sc, G * Mq)
    assert np.all(np.abs(m - n_img / 40.0) < 1e-12), m


def pin_choose_focal_layers_brute_force(lib=None, choose_fn=None):
    """Every chosen layer outranks every other layer (higher ratio, or equal ratio and lower index);
    exhaustive over small ratio vectors with ties."""
    choose_fn = choose_fn or oracle.choose_focal_layers
    levels = (0.1, 0.4, 0.4, 0.7)
    for n in range(1, 6):
        for ratio in itertools.product(levels, repeat=n):
            for C in range(1, n + 1):
                got = choose_fn(list(ratio), C)
                assert len(got) == C and got == sorted(got) and len(set(got)) == C, (ratio, C, got)
                rest = [l for l in range(n) if l not in got]
                for i in got:
                    for j in rest:
                        assert ratio[i] > ratio[j] or (ratio[i] == ratio[j] and i < j), (ratio, C, got)


PROFILE_PINS = [pin_focal_mass_whole_range_is_one, pin_focal_mass_uniform_attention,
                pin_choose_focal_layers_brute_force]


@pytest.mark.parametrize("pin", PROFILE_PINS, ids=[p.__name__ for p in PROFILE_PINS])
def test_profile_pin(pin, oracle_mod):
    pin()


def test_profile_pins_catch_planted_mistakes(oracle_mod):
    """Plausible mistakes in the profiling functions each fail a pin (planted here, on the CPU)."""
    wrong_mass = [lambda s, R: np.asarray(s, np.float64).sum(axis=-1),            # R not divided out
                  lambda s, R: np.asarray(s, np.float64).mean(axis=-1),           # mean over tokens
                  lambda s, R: np.asarray(s, np.float64).max(axis=-1) / R]        # max instead of sum
    for fn in wrong_mass:
        with pytest.raises(AssertionError):
            pin_focal_mass_whole_range_is_one(mass_fn=fn)
            pin_focal_mass_uniform_attention(mass_fn=fn)
    wrong_choose = [lambda r, C: sorted(sorted(range(len(r)), key=lambda l: (r[l], l))[:C]),      # smallest
                    lambda r, C: sorted(sorted(range(len(r)), key=lambda l: (-r[l], -l))[:C]),    # ties high
                    lambda r, C: sorted(range(len(r)), key=lambda l: (-r[l], l))[:C]]            # unsorted
    for fn in wrong_choose:
        with pytest.raises(AssertionError):
            pin_choose_focal_layers_brute_force(choose_fn=fn)


# Decode-step append (FastKV 3.2 and FastOCR decoding: the step's new K/V row joins the cache), pinned
# by rebuilding the expected cache with explicit concatenation and by the attention it feeds.

def pin_append_equals_concatenation(lib=None, append_fn=None):
    """Row pos[b] of every (layer, b, h) becomes the new row: the result equals the cache cut at pos,
    the new row, and the rest, concatenated; a position outside [0, T) leaves that sequence as it was."""
    append_fn = append_fn or oracle.kv_append
    L, B, Hkv, T = 2, 3, 2, 9
    k, v = _rand_bf16((L, B, Hkv, T, 128), 41, 1), _rand_bf16((L, B, Hkv, T, 128), 41, 2)
    kn, vn = _rand_bf16((L, B, Hkv, 128), 41, 3), _rand_bf16((L, B, Hkv, 128), 41, 4)
    pos = torch.tensor([0, 8, -1], dtype=torch.int32)
    gk, gv = append_fn(k, v, kn, vn, pos)
    for src, new, got in ((k, kn, gk), (v, vn, gv)):
        for b, t in enumerate(pos.tolist()):
            if 0 <= t < T:
                want = torch.cat([src[:, b, :, :t], new[:, b, :, None], src[:, b, :, t + 1:]], dim=2)
            else:
                want = src[:, b]
            assert torch.equal(got[:, b].view(torch.int16), want.view(torch.int16)), (b, t)


def pin_decode_after_append_sees_the_new_row(lib=None, append_fn=None):
    """A new key far along the query direction takes almost all of the attention once appended at
    row len-1 (and the cache's length then covers it): the output is that row's value."""
    append_fn = append_fn or oracle.kv_append
    B, Hkv, G, T = 1, 1, 2, 12
    k, v = _rand_bf16((B, Hkv, T, 128), 42, 1), _rand_bf16((B, Hkv, T, 128), 42, 2)
    q = _rand_bf16((B, Hkv * G, 1, 128), 42, 3)
    u = q[0, :, 0].float().sum(dim=0)
    kn = (u / u.norm() * 60.0).to(torch.bfloat16).view(B, Hkv, 128)
    vn = _rand_bf16((B, Hkv, 128), 42, 4)
    pos = torch.tensor([7], dtype=torch.int32)
    k2, v2 = append_fn(k, v, kn, vn, pos)
    out = oracle.sparse_decode(k2, v2, pos + 1, q, None, 0, lib=lib)
    assert np.max(np.abs(np.asarray(out)[0, :, 0] - vn[0, 0].double().numpy())) < 1e-6


APPEND_PINS = [pin_append_equals_concatenation, pin_decode_after_append_sees_the_new_row]


@pytest.mark.parametrize("pin", APPEND_PINS, ids=[p.__name__ for p in APPEND_PINS])
def test_append_pin(pin, oracle_mod):
    pin()


def test_append_pins_catch_planted_mistakes(oracle_mod):
    """Plausible mistakes in the append each fail a pin (planted here, on the CPU)."""
    def shifted(k, v, kn, vn, pos):            # writes one row later
        return oracle.kv_append(k, v, kn, vn, pos + 1)

    def k_only(k, v, kn, vn, pos):             # forgets the V row
        k2, _ = oracle.kv_append(k, v, kn, vn, pos)
        return k2, v.clone()

    def swapped(k, v, kn, vn, pos):            # K and V rows exchanged
        return oracle.kv_append(k, v, vn, kn, pos)

    for fn in (shifted, k_only, swapped):
        with pytest.raises(AssertionError):
            pin_append_equals_concatenation(append_fn=fn)
            pin_decode_after_append_sees_the_new_row(append_fn=fn)


PINS = [pin_golden_focal, pin_golden_topk, pin_golden_sparse, pin_golden_shared_prefix,
        pin_uniform_keys_give_mean, pin_importance_sums_to_rows, pin_single_key_and_dominant_key,
        pin_topk_brute_force, pin_sparse_full_set_equals_dense, pin_compaction_equals_sparse,
        pin_shared_prefix_equals_concatenation, pin_forked_branches_equal_concatenation]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin, oracle_mod):
    pin()


# ----------------------------------------------------------------------------------------------
# planted mistakes: each must make at least one pin fail

MUTATIONS = {
    "dropped_scale": ("        l *= scale;\n", "\n"),
    "softmax_sign": ("p[j] = exp(p[j] - m);", "p[j] = exp(m - p[j]);"),
    "interleaved_heads": ("int g = h * G + gi;", "int g = gi * c->Hkv + h;"),
    "causal_off_by_one": ("int lim = c->q_pos0 + i + 1;", "int lim = c->q_pos0 + i;"),
    "candidate_offset": ("s[j - c->cand_lo] += p[j];", "s[j - c->cand_lo] += p[j] / c->Mq;"),
    "tie_break_reversed": ("return (x->j > y->j) - (x->j < y->j);", "return (x->j < y->j) - (x->j > y->j);"),
    "output_unsorted": ("qsort(sel, (size_t)k, sizeof(int), cmp_int);", ";"),
    "tail_skips_first": ("for (int t = c->tail_lo; t < c->len[b]; ++t, ++m) {",
                         "for (int t = c->tail_lo + 1; t < c->len[b]; ++t, ++m) {"),
    "compact_tail_shift": ("tail_lo + (r - kk);", "tail_lo + (r - kk) + (r > kk);"),
    "draft_not_causal": ("attend(qrow, d, c->scale, m + i + 1, kr, vr, p, orow);",
                         "attend(qrow, d, c->scale, m + c->Mq, kr, vr, p, orow);"),
    "suffix_wrong_branch": ("int s0 = c->off[b];", "int s0 = c->off[b > 0 ? b - 1 : 0];"),
    "fork_position_ignored": ("int np = c->pidx ? c->kp : (c->pre_len ? c->pre_len[b] : c->P);",
                              "int np = c->pidx ? c->kp : c->P;"),
    "value_uses_key": ("out[c] += p[j] * bf(v[c]);", "out[c] += p[j] * bf(kr[j][c]);"),
    "normaliser_dropped": ("for (int j = 0; j < n; ++j) p[j] /= z;", ";"),
    "len_ignored": ("int visible = n;", "int visible = c->Tcap;"),
}


@pytest.fixture(scope="module")
def mutant_dir():
    d = tempfile.mkdtemp(prefix="oracle_mut_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


def run_pins_on(lib_path):
    """Run every pin against the oracle built at lib_path; print the failing pins (used by the
    mutation test in a child process, so a mutant that crashes cannot take pytest down)."""
    lib = oracle.open_library(lib_path)
    failed = []
    for pin in PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
    print("FAILED:" + ",".join(failed))


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutations_are_caught(name, mutant_dir, oracle_mod):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "fx_oracle.c")).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path = os.path.join(mutant_dir, f"{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    so = oracle.compile_source(path, os.path.join(mutant_dir, f"lib{name}.so"))
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    proc = subprocess.run([sys.executable, "-c",
                           f"import tests.test_oracle_pins as t; t.run_pins_on({so!r})"],
                          cwd=root, capture_output=True, text=True, timeout=300)
    caught_by_crash = proc.returncode != 0
    line = [l for l in proc.stdout.splitlines() if l.startswith("FAILED:")]
    failed = line[-1][len("FAILED:"):].split(",") if line else []
    failed = [f for f in failed if f]
    assert caught_by_crash or failed, f"no pin catches the planted mistake {name}"


# ----------------------------------------------------------------------------------------------
# Cross-step fixation reuse: the layer schedule of a decode step, pinned by the FastOCR configuration
# written out by hand (28 layers, focal layers 3 and 14) and by small cases.
def test_csfr_schedule_fastocr_configuration():
    later = [("previous", 14)] * 3 + [("focal", 3)] + [("current", 3)] * 10 + [("focal", 14)] + [("current", 14)] * 13
    first = [("dense", -1)] * 3 + later[3:]
    assert oracle.csfr_schedule(28, (3, 14), first_step=False) == later
    assert oracle.csfr_schedule(28, (14, 3), first_step=True) == first


def test_csfr_schedule_small_cases():
    # a focal first layer: nothing reuses an older set
    assert oracle.csfr_schedule(4, (0,), first_step=False) == [("focal", 0), ("current", 0), ("current", 0),
                                                                ("current", 0)]
    # every layer focal
    assert oracle.csfr_schedule(3, (0, 1, 2), first_step=False) == [("focal", 0), ("focal", 1), ("focal", 2)]
    # the deepest focal layer is the last one: layers before the first reuse it
    assert oracle.csfr_schedule(5, (2, 4), first_step=False) == [("previous", 4), ("previous", 4), ("focal", 2),
                                                                 ("current", 2), ("focal", 4)]
