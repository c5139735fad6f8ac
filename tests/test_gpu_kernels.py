"""GPU parity of every entry point against the fp64 oracle on small seeded cases.

Sizes span several key tiles and splits and end on ragged tails; edge cases cover empty rows,
single keys, k = n, ties, warm starts and bad device-side data.  All calls go through the C ABI
(the ctypes binding only marshals arguments).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests import parity_util as pu

pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module")
def fx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kv_cache_token_fx_gb300 as fxm
    fxm.load_library()
    return fxm


def rnd(shape, seed, stream):
    return synth.normal_bf16(seed, synth.stream_id(777, stream), shape)


def dev(t):
    return t.to("cuda")


def kv_case(B, Hkv, T, seed):
    return rnd((B, Hkv, T, D), seed, 1), rnd((B, Hkv, T, D), seed, 2)


# ----------------------------------------------------------------------------------------------
@pytest.mark.parametrize("G,Mq,q_pos0", [(1, 1, -1), (2, 1, -1), (4, 1, -1), (8, 1, -1), (2, 3, 500), (4, 8, 690),
                                         (16, 2, -1)])
def test_focal_matches_oracle(fx, G, Mq, q_pos0):
    B, Hkv, T = 3, 2, 700
    k, v = kv_case(B, Hkv, T, 10 + G + Mq)
    q = rnd((B, Hkv * G, Mq, D), 10 + G, 3)
    length = torch.tensor([700, 333, 17], dtype=torch.int32)
    cand = (5, 650)
    ref_out, ref_sc = oracle.focal(k, v, length, q, q_pos0=q_pos0, cand=cand)
    out, sc = fx.fx_focal_attn_scores(dev(k), dev(v), dev(length), dev(q), q_pos0=q_pos0, cand=cand)
    torch.cuda.synchronize()
    assert fx.fx_device_errors() == 0
    vmax = float(v.float().abs().max())
    pu.assert_out_close(out, ref_out, vmax)
    pu.assert_scores_close(sc, ref_sc)


def test_focal_edge_cases(fx):
    B, Hkv, G, T = 4, 1, 2, 40
    k, v = kv_case(B, Hkv, T, 3)
    q = rnd((B, Hkv * G, 1, D), 3, 3)
    length = torch.tensor([0, 1, 40, 16], dtype=torch.int32)   # empty, single key, full, one tile
    ref_out, ref_sc = oracle.focal(k, v, length, q)
    out, sc = fx.fx_focal_attn_scores(dev(k), dev(v), dev(length), dev(q))
    pu.assert_out_close(out, ref_out, float(v.float().abs().max()))
    pu.assert_scores_close(sc, ref_sc)
    assert torch.all(out[0] == 0) and torch.all(sc[0] == 0)
    assert torch.equal(out[1, :, 0].cpu(), v[1, 0, 0].float().expand(G, D))
    # scores only / output only
    o2, s2 = fx.fx_focal_attn_scores(dev(k), dev(v), dev(length), dev(q), want_out=False)
    assert o2 is None
    pu.assert_scores_close(s2, ref_sc)
    o3, s3 = fx.fx_focal_attn_scores(dev(k), dev(v), dev(length), dev(q), want_scores=False)
    assert s3 is None
    pu.assert_out_close(o3, ref_out, float(v.float().abs().max()))


def test_focal_strided_cache(fx):
    """A cache view with padding between heads and rows (strides, not shapes, address the rows)."""
    B, Hkv, G, T = 2, 3, 2, 300
    big_k = rnd((B, Hkv + 1, T + 20, D + 64), 4, 1)
    big_v = rnd((B, Hkv + 1, T + 20, D + 64), 4, 2)
    k, v = big_k[:, 1:, 10:10 + T, 64:], big_v[:, 1:, 10:10 + T, 64:]
    q = rnd((B, Hkv * G, 1, D), 4, 3)
    length = torch.tensor([300, 211], dtype=torch.int32)
    ref_out, ref_sc = oracle.focal(k.contiguous(), v.contiguous(), length, q)
    dk, dv = dev(big_k)[:, 1:, 10:10 + T, 64:], dev(big_v)[:, 1:, 10:10 + T, 64:]
    out, sc = fx.fx_focal_attn_scores(dk, dv, dev(length), dev(q))
    pu.assert_out_close(out, ref_out, float(v.float().abs().max()))
    pu.assert_scores_close(sc, ref_sc)


@pytest.mark.parametrize("G,Mq,q_pos0", [(4, 8, 690), (2, 12, 650), (8, 6, -1), (2, 4, 690), (4, 3, -1)])
def test_focal_scores_only_matches_oracle(fx, G, Mq, q_pos0):
    """Scoring-only focal calls (no output rows: V is not read; more than 16 rows use the 32-row
    layout) give the oracle's importance scores."""
    B, Hkv, T = 3, 2, 700
    k, v = kv_case(B, Hkv, T, 40 + G * Mq)
    q = rnd((B, Hkv * G, Mq, D), 41 + G * Mq, 3)
    length = torch.tensor([700, 523, 64], dtype=torch.int32)
    cand = (5, 600)
    _, ref_sc = oracle.focal(k, v, length, q, q_pos0=q_pos0, cand=cand, want_out=False)
    _, sc = fx.fx_focal_attn_scores(dev(k), dev(v), dev(length), dev(q), q_pos0=q_pos0, cand=cand, want_out=False)
    torch.cuda.synchronize()
    assert fx.fx_device_errors() == 0
    pu.assert_scores_close(sc, ref_sc)


@pytest.mark.parametrize("G,Mq,T,lens,q_off,cand,scale", [
    (4, 8, 5000, [5000, 3001, 0, 129], 8, (0, 4992), None),      # 32 rows: 5 ranges of 1024 keys, causal window
    (8, 8, 4000, [4000, 3999, 513, 1], None, (17, 3333), 1.0),   # 64 rows: 8 ranges of 512, sharp softmax
    (2, 8, 4500, [4500, 2049, 2047, 4500], 8, (0, 4492), None),  # 16 rows: 3 ranges of 2048 (a boundary at 2048)
    (3, 16, 3000, [3000, 1280, 641, 640], None, (0, 3000), 0.5),  # 48 rows: 5 ranges of 640
    (1, 9, 2100, [2100, 7, 2048, 2049], 3, (100, 2090), None),   # 9 rows in a 16-column tile, window past len
])
def test_scores_only_on_tensor_cores_matches_oracle(fx, G, Mq, T, lens, q_off, cand, scale):
    """Scores-only calls with more than 8 rows per KV head keep their logits in tensor memory and merge
    the per-range row maxima and sums across CTAs: several ranges per (sequence, KV head), ragged and
    empty sequences, a causal window, a candidate range.  Equal to the oracle, and to the split-KV path
    (taken when output rows are wanted, which writes its logits out) on the same inputs."""
    B, Hkv = len(lens), 2
    k, v = kv_case(B, Hkv, T, 300 + G * Mq)
    q = rnd((B, Hkv * G, Mq, D), 301 + G * Mq, 3)
    length = torch.tensor(lens, dtype=torch.int32)
    q_pos0 = -1 if q_off is None else T - q_off
    _, ref_sc = oracle.focal(k, v, length, q, q_pos0=q_pos0, cand=cand, want_out=False, scale=scale)
    dk, dv, dl, dq = dev(k), dev(v), dev(length), dev(q)
    _, sc = fx.fx_focal_attn_scores(dk, dv, dl, dq, q_pos0=q_pos0, cand=cand, want_out=False, scale=scale)
    _, sc_split = fx.fx_focal_attn_scores(dk, dv, dl, dq, q_pos0=q_pos0, cand=cand, scale=scale)
    # back to back on the same workspace, as a programmatic dependent launch: the counters were reset
    _, sc2 = fx.fx_focal_attn_scores(dk, dv, dl, dq, q_pos0=q_pos0, cand=cand, want_out=False, scale=scale,
                                     flags=fx.FX_LAUNCH_PDL)
    torch.cuda.synchronize()
    assert fx.fx_device_errors() == 0
    pu.assert_scores_close(sc, ref_sc)
    pu.assert_scores_close(sc, sc_split, "tensor-core vs split-KV scores")
    assert torch.equal(sc, sc2)
    assert torch.all(sc[lens.index(min(lens))][:, max(0, min(lens) - cand[0]):] == 0)


def test_scores_only_on_tensor_cores_shared_cache(fx):
    """A cache shared by every sequence (batch stride 0, as in shared-prefix scoring) with per-sequence
    lengths and queries."""
    B, Hkv, G, Mq, T = 3, 2, 4, 4, 2600
    k1, v1 = kv_case(1, Hkv, T, 321)
    q = rnd((B, Hkv * G, Mq, D), 322, 3)
    length = torch.tensor([2600, 1500, 1024], dtype=torch.int32)
    k, v = k1.expand(B, -1, -1, -1), v1.expand(B, -1, -1, -1)
    _, ref_sc = oracle.focal(k.contiguous(), v.contiguous(), length, q, want_out=False)
    _, sc = fx.fx_focal_attn_scores(dev(k1).expand(B, -1, -1, -1), dev(v1).expand(B, -1, -1, -1), dev(length),
                                    dev(q), want_out=False)
    torch.cuda.synchronize()
    assert fx.fx_device_errors() == 0
    pu.assert_scores_close(sc, ref_sc)


# ----------------------------------------------------------------------------------------------
def _quantised_scores(rows, n, seed, levels):
    g = np.random.default_rng(seed)
    return torch.from_numpy((g.integers(0, levels, size=(rows, n)) / levels).astype(np.float32))


@pytest.mark.parametrize("rows,n,k,levels", [(3, 1, 1, 4), (4, 5, 3, 3), (8, 1024, 64, 1 << 20), (5, 4097, 205, 50),
                                             (3, 4096, 4096, 7), (2, 33000, 2040, 1 << 22), (2, 60000, 2048, 1000),
                                             (2, 131072, 2048, 1 << 24)])
def test_topk_matches_oracle_exactly(fx, rows, n, k, levels):
    s = _quantised_scores(rows, n, rows * n + k, levels)
    ref = oracle.topk(s.numpy(), k)
    got = fx.fx_topk_select(dev(s), k)
    torch.cuda.synchronize()
    assert fx.fx_device_errors() == 0
    assert np.array_equal(got.cpu().numpy(), ref)


@pytest.mark.parametrize("n,k", [(4096, 205), (2304, 256), (50000, 100)])
def test_topk_warm_start_is_exact(fx, n, k):
    rows = 6
    s = _quantised_scores(rows, n, n + k, 1 << 16)
    prev_scores = s + torch.from_numpy(np.random.default_rng(5).normal(0, 0.05, size=s.shape).astype(np.float32))
    prev = torch.from_numpy(oracle.topk(prev_scores.numpy(), k))
    ref = oracle.topk(s.numpy(), k)
    got = fx.fx_topk_select(dev(s), k, prev=dev(prev))
    assert np.array_equal(got.cpu().numpy(), ref)
    # the previous set read before the dependency wait (programmatic dependent launch, inputs ready)
    got_early = fx.fx_topk_select(dev(s), k, prev=dev(prev), flags=fx.FX_LAUNCH_PDL | fx.FX_LAUNCH_INPUTS_READY)
    assert np.array_equal(got_early.cpu().numpy(), ref)
    # a previous set that is the exact answer, and one with repeated entries, change nothing
    got2 = fx.fx_topk_select(dev(s), k, prev=dev(torch.from_numpy(ref)))
    assert np.array_equal(got2.cpu().numpy(), ref)
    rep = torch.zeros_like(prev)
    got3 = fx.fx_topk_select(dev(s), k, prev=dev(rep))
    assert np.array_equal(got3.cpu().numpy(), ref)
    assert fx.fx_device_errors() == 0


def test_topk_long_rows_stop_early_or_run_every_pass(fx):
    """Long rows (a cluster of CTAs per row, or one CTA per row when there are many): the passes stop once
    the chosen bin holds exactly the keys still needed, and run to the last byte when the k-th key is
    tied.  Exact against the oracle."""
    g = np.random.default_rng(11)
    cases = []
    cases.append((g.normal(size=(3, 32760)).astype(np.float32), 2040))      # distinct keys
    cases.append((g.random(size=(2, 20000)).astype(np.float32), 20000))     # k = n: every key
    two = np.full((2, 32760), 0.5, np.float32)
    two[:, :5000] = 1.0
    g.shuffle(two[1])
    cases.append((two, 5000))    # the bin of 1.0 holds exactly k keys (same top byte as 0.5)
    cases.append((two, 5001))    # one 0.5 is needed: the lowest index among the tied ones
    many = np.full((40, 20000), 0.25, np.float32)   # 40 long rows: one CTA per row
    many[:, ::7] = g.normal(size=(40, (20000 + 6) // 7)).astype(np.float32)
    cases.append((many, 1500))
    cases.append((many, 2858))   # every key above 0.25 and the first tied 0.25s
    for s, k in cases:
        ref = oracle.topk(s, k)
        got = fx.fx_topk_select(dev(torch.from_numpy(s)), k)
        torch.cuda.synchronize()
        assert fx.fx_device_errors() == 0
        assert np.array_equal(got.cpu().numpy(), ref), (s.shape, k)


def test_topk_many_rows_too_long_for_shared_memory(fx):
    """Many long rows (one CTA per row reading global memory): the candidates move to shared memory in
    the first scan (a sampled threshold), once a chosen bin fits (after the first or a later pass), or
    never (every key tied, or k = n); a sample that lets too few or too many keys through; rows not
    16-byte aligned; a warm start; rows past the bitmap limit.  Exact against the oracle."""
    g = np.random.default_rng(12)
    rows = 40   # more than a cluster launch takes
    cases = []
    # long-context shaped importance: lognormal bulk, a few planted high keys (bin fits after pass 1)
    ln = np.exp(g.normal(size=(rows, 131072))).astype(np.float32) * 1e-5
    ln[:, g.integers(0, 131072, size=1024)] += 0.01
    cases.append((ln, 2048))
    # distinct normal keys: the first chosen bin is too large, a later one fits
    cases.append((g.normal(size=(rows, 50000)).astype(np.float32) * 1e-3 + 1.0, 2048))
    # odd row length (rows not 16-byte aligned), ties at the boundary
    cases.append(((g.integers(0, 300, size=(rows, 50001)) / 300).astype(np.float32), 2048))
    # every key tied: no bin ever fits, the first need_eq = k indices are taken
    cases.append((np.full((rows, 60000), 0.75, np.float32), 100))
    # k = n: the first pass takes every key
    cases.append((g.random(size=(rows, 45057)).astype(np.float32), 45057))
    # the bin of 1.0 holds exactly k keys
    two = np.full((rows, 50000), 0.5, np.float32)
    two[:, :3000] = 1.0
    for r in range(1, rows):
        g.shuffle(two[r])
    cases.append((two, 3000))
    cases.append((two, 3001))
    # k = 1 and a negative row
    cases.append((-np.abs(g.normal(size=(rows, 46000))).astype(np.float32), 1))
    # the row's largest keys sit exactly at the positions the kernel samples (4 keys at each 16-byte group
    # t * n / 4096, t < 1024), so fewer than k keys reach the sampled threshold and the row is counted
    # again without it; and the unaligned rows' sampled positions (t * n / 4096, t < 4096)
    adv = g.random(size=(rows, 65536)).astype(np.float32)
    pos = (np.arange(1024)[:, None] * 64 + np.arange(4)[None, :]).reshape(-1)
    adv[:, pos] = 10.0 + 100.0 * g.random(size=(rows, pos.size)).astype(np.float32)
    cases.append((adv, 100))
    adv_odd = g.random(size=(rows, 65537)).astype(np.float32)
    pos_odd = (np.arange(4096, dtype=np.int64) * 65537) // 4096
    adv_odd[:, pos_odd] = 10.0 + 100.0 * g.random(size=(rows, pos_odd.size)).astype(np.float32)
    cases.append((adv_odd, 100))
    # longer than the bitmaps allow: every pass reads global memory
    cases.append((g.normal(size=(rows, 270000)).astype(np.float32), 1000))
    for s, k in cases:
        ref = oracle.topk(s, k)
        got = fx.fx_topk_select(dev(torch.from_numpy(s)), k)
        torch.cuda.synchronize()
        assert fx.fx_device_errors() == 0
        assert np.array_equal(got.cpu().numpy(), ref), (s.shape, k)
    # warm start: a previous set from perturbed scores, read early and late
    s = cases[1][0]
    prev_scores = s + g.normal(0, 2e-4, size=s.shape).astype(np.float32)
    prev = torch.from_numpy(oracle.topk(prev_scores, 2048))
    ref = oracle.topk(s, 2048)
    got = fx.fx_topk_select(dev(torch.from_numpy(s)), 2048, prev=dev(prev))
    got_early = fx.fx_topk_select(dev(torch.from_numpy(s)), 2048, prev=dev(prev),
                                  flags=fx.FX_LAUNCH_PDL | fx.FX_LAUNCH_INPUTS_READY)
    torch.cuda.synchronize()
    assert fx.fx_device_errors() == 0
    assert np.array_equal(got.cpu().numpy(), ref) and np.array_equal(got_early.cpu().numpy(), ref)


def test_topk_negative_and_signed_zero(fx):
    s = torch.tensor([[-1.0, 0.0, -0.0, 2.0, -3.0, 2.0, -0.5]], dtype=torch.float32)
    for k in range(1, 8):
        got = fx.fx_topk_select(dev(s), k).cpu().numpy()
        order = sorted(range(7), key=lambda j: (-float(s[0, j]), j))
        # -0.0 compares equal to +0.0 in the oracle's ordering; the library orders -0.0 below +0.0,
        # which only matters when both straddle the boundary (k = 3 here): accept either.
        exp = sorted(order[:k])
        if k == 3:
            assert got[0].tolist() in ([1, 3, 5], [2, 3, 5])
        else:
            assert got[0].tolist() == exp, k


# ----------------------------------------------------------------------------------------------
def _sorted_subsets(B, Hkv, pool, kk, seed):
    g = np.random.default_rng(seed)
    return torch.from_numpy(np.stack([np.stack([np.sort(g.choice(pool, kk, replace=False)) for _ in range(Hkv)])
                                      for _ in range(B)]).astype(np.int32))


@pytest.mark.parametrize("G,kk,tail_lo", [(1, 64, 1000), (2, 205, 4096), (4, 2048, 6000), (8, 37, 500), (2, 0, 0),
                                          (4, 300, 300), (16, 205, 4096)])
def test_sparse_matches_oracle(fx, G, kk, tail_lo):
    B, Hkv = 3, 2
    T = max(tail_lo + 513, 700)
    k, v = kv_case(B, Hkv, T, 20 + G)
    q = rnd((B, Hkv * G, 1, D), 20 + G, 3)
    length = torch.tensor([T, tail_lo + 77, tail_lo], dtype=torch.int32)
    idx = _sorted_subsets(B, Hkv, max(tail_lo, 1), kk, kk + G) if kk else None
    ref = oracle.sparse_decode(k, v, length, q, idx, tail_lo)
    out = fx.fx_sparse_gqa_decode(dev(k), dev(v), dev(length), dev(q), dev(idx) if idx is not None else None, tail_lo)
    torch.cuda.synchronize()
    assert fx.fx_device_errors() == 0
    pu.assert_out_close(out, ref, float(v.float().abs().max()))
    # same call again (the merge counters must have been reset)
    out2 = fx.fx_sparse_gqa_decode(dev(k), dev(v), dev(length), dev(q), dev(idx) if idx is not None else None, tail_lo)
    assert torch.equal(out, out2)


def test_sparse_full_set_equals_dense(fx):
    B, Hkv, G, T = 2, 2, 4, 900
    k, v = kv_case(B, Hkv, T, 31)
    q = rnd((B, Hkv * G, 1, D), 31, 3)
    length = torch.tensor([T, T], dtype=torch.int32)
    full = torch.arange(T, dtype=torch.int32).view(1, 1, T).expand(B, Hkv, T).contiguous()
    a = fx.fx_sparse_gqa_decode(dev(k), dev(v), dev(length), dev(q), dev(full), T)
    b = fx.fx_sparse_gqa_decode(dev(k), dev(v), dev(length), dev(q), None, 0)
    c, _ = fx.fx_focal_attn_scores(dev(k), dev(v), dev(length), dev(q), want_scores=False)
    ref = oracle.sparse_decode(k, v, length, q, None, 0)
    for x in (a, b, c):
        pu.assert_out_close(x, ref, float(v.float().abs().max()))


def test_sparse_bad_index_is_flagged_not_read(fx):
    B, Hkv, G, T = 1, 2, 2, 64
    k, v = kv_case(B, Hkv, T, 41)
    q = rnd((B, Hkv * G, 1, D), 41, 3)
    length = torch.tensor([50], dtype=torch.int32)
    idx = torch.tensor([[[1, 2, 3, 49], [4, 5, 50, 1 << 30]]], dtype=torch.int32)   # 50 >= len, huge
    fx.fx_device_errors()
    out = fx.fx_sparse_gqa_decode(dev(k), dev(v), dev(length), dev(q), dev(idx), 50)
    bits = fx.fx_device_errors()
    assert bits & fx.FX_DEVERR_INDEX
    ok = torch.tensor([[[1, 2, 3, 49], [4, 5, 4, 5]]], dtype=torch.int32)[:, :, :4]
    ref0 = oracle.sparse_decode(k, v, length, q, ok, 50)
    pu.assert_out_close(out[:, :2], ref0[:, :2], float(v.float().abs().max()))
    # KV head 1 kept rows 4, 5 only
    ref1 = oracle.sparse_decode(k, v, length, q, torch.tensor([[[1, 2], [4, 5]]], dtype=torch.int32), 50)
    pu.assert_out_close(out[:, 2:], ref1[:, 2:], float(v.float().abs().max()))


def test_bad_length_is_flagged(fx):
    B, Hkv, G, T = 2, 1, 2, 64
    k, v = kv_case(B, Hkv, T, 43)
    q = rnd((B, Hkv * G, 1, D), 43, 3)
    fx.fx_device_errors()
    length = torch.tensor([64, 65], dtype=torch.int32)
    out, _ = fx.fx_focal_attn_scores(dev(k), dev(v), dev(length), dev(q))
    assert fx.fx_device_errors() & fx.FX_DEVERR_LEN
    ref, _ = oracle.focal(k, v, torch.tensor([64, 64], dtype=torch.int32), q)
    pu.assert_out_close(out, ref, float(v.float().abs().max()))


def test_host_argument_errors(fx):
    k = torch.zeros((1, 1, 16, D), dtype=torch.bfloat16, device="cuda")
    ln = torch.tensor([16], dtype=torch.int32, device="cuda")
    q = torch.zeros((1, 3, 1, D), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fx.FxError) as e:
        fx.fx_topk_select(torch.zeros((2, 5), device="cuda"), 6)
    assert e.value.status == 1
    k65 = torch.zeros((1, 1, 16, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fx.FxError) as e:
        fx.fx_sparse_gqa_decode(k65, k65, ln, q[:, :1, :, :64].contiguous(), None, 0)
    assert e.value.status == 2
    q3 = torch.zeros((1, 3, 1, D), dtype=torch.bfloat16, device="cuda")
    k2 = torch.zeros((1, 2, 16, D), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fx.FxError) as e:
        fx.fx_sparse_gqa_decode(k2, k2, ln, q3, None, 0)   # 3 query heads over 2 KV heads
    assert e.value.status == 1


# ----------------------------------------------------------------------------------------------
@pytest.mark.parametrize("n_layers,kk,tail_lo", [(1, 40, 90), (3, 2040, 4000), (2, 0, 0)])
def test_compaction_is_bit_exact(fx, n_layers, kk, tail_lo):
    B, Hkv = 2, 3
    T = tail_lo + 100
    ks = torch.stack([rnd((B, Hkv, T, D), 50 + l, 1) for l in range(n_layers)])
    vs = torch.stack([rnd((B, Hkv, T, D), 50 + l, 2) for l in range(n_layers)])
    length = torch.tensor([T, tail_lo + 3], dtype=torch.int32)
    idx = _sorted_subsets(B, Hkv, max(tail_lo, 1), kk, 9) if kk else None
    cap = kk + 100
    dk = torch.full((n_layers, B, Hkv, cap, D), 7.0, dtype=torch.bfloat16, device="cuda")
    dv = torch.full_like(dk, 7.0)
    dl = torch.zeros(B, dtype=torch.int32, device="cuda")
    fx.fx_kv_compact(dev(ks), dev(vs), dev(length), dev(idx) if idx is not None else None, tail_lo, dk, dv, dl)
    torch.cuda.synchronize()
    assert fx.fx_device_errors() == 0
    for l in range(n_layers):
        rk, rv, rl = oracle.kv_compact(ks[l], vs[l], length, idx if idx is not None else torch.zeros((B, Hkv, 0), dtype=torch.int32),
                                       tail_lo, cap)
        assert torch.equal(dl.cpu(), rl)
        for b in range(B):
            n = int(rl[b])
            assert torch.equal(dk[l, b, :, :n].cpu().view(torch.int16), rk[b, :, :n].view(torch.int16))
            assert torch.equal(dv[l, b, :, :n].cpu().view(torch.int16), rv[b, :, :n].view(torch.int16))
            assert torch.all(dk[l, b, :, n:].float() == 7.0)   # rows past the new length untouched


def test_compaction_with_per_layer_sets(fx):
    """A [L, B, Hkv, k] index array gives every layer its own set."""
    n_layers, B, Hkv, kk, tail_lo = 3, 2, 2, 25, 300
    T = tail_lo + 40
    ks = torch.stack([rnd((B, Hkv, T, D), 150 + l, 1) for l in range(n_layers)])
    vs = torch.stack([rnd((B, Hkv, T, D), 150 + l, 2) for l in range(n_layers)])
    length = torch.tensor([T, tail_lo + 7], dtype=torch.int32)
    idx = torch.stack([_sorted_subsets(B, Hkv, tail_lo, kk, 20 + l) for l in range(n_layers)])
    cap = kk + 64
    dk = torch.zeros((n_layers, B, Hkv, cap, D), dtype=torch.bfloat16, device="cuda")
    dv = torch.zeros_like(dk)
    dl = torch.zeros(B, dtype=torch.int32, device="cuda")
    fx.fx_kv_compact(dev(ks), dev(vs), dev(length), dev(idx), tail_lo, dk, dv, dl)
    torch.cuda.synchronize()
    assert fx.fx_device_errors() == 0
    for l in range(n_layers):
        rk, rv, rl = oracle.kv_compact(ks[l], vs[l], length, idx[l], tail_lo, cap)
        assert torch.equal(dl.cpu(), rl)
        for b in range(B):
            n = int(rl[b])
            assert torch.equal(dk[l, b, :, :n].cpu().view(torch.int16), rk[b, :, :n].view(torch.int16))
            assert torch.equal(dv[l, b, :, :n].cpu().view(torch.int16), rv[b, :, :n].view(torch.int16))


def test_per_layer_retention_matches_oracle(fx):
    """fx_kv_retain_per_layer: each layer's window scores (causal window of the last Mq positions),
    its own top-k, and the compaction of every layer with its own set plus the window tail."""
    n_layers, B, Hkv, G, Mq, T, keep = 3, 2, 2, 2, 4, 600, 37
    cand = T - Mq
    ks = torch.stack([rnd((B, Hkv, T, D), 160 + l, 1) for l in range(n_layers)])
    vs = torch.stack([rnd((B, Hkv, T, D), 160 + l, 2) for l in range(n_layers)])
    qs = torch.stack([rnd((B, Hkv * G, Mq, D), 160 + l, 3) for l in range(n_layers)])
    length = torch.tensor([T, 500], dtype=torch.int32)
    cap = keep + Mq + 8
    dk = torch.zeros((n_layers, B, Hkv, cap, D), dtype=torch.bfloat16, device="cuda")
    dv = torch.zeros_like(dk)
    dl = torch.zeros(B, dtype=torch.int32, device="cuda")
    idx = fx.fx_kv_retain_per_layer(dev(ks), dev(vs), dev(length), dev(qs), keep, cand, cand, dk, dv, dl,
                                    q_pos0=cand)
    torch.cuda.synchronize()
    assert fx.fx_device_errors() == 0
    assert tuple(idx.shape) == (n_layers, B, Hkv, keep)
    for l in range(n_layers):
        _, sc = oracle.focal(ks[l], vs[l], length, qs[l], q_pos0=cand, cand=(0, cand), want_out=False)
        ref_idx = oracle.topk(sc, keep)
        pu.check_index_sets(idx[l], ref_idx, sc, keep)
        # the compaction, checked on the sets the GPU chose
        rk, rv, rl = oracle.kv_compact(ks[l], vs[l], length, idx[l].cpu(), cand, cap)
        assert torch.equal(dl.cpu(), rl)
        for b in range(B):
            n = int(rl[b])
            assert torch.equal(dk[l, b, :, :n].cpu().view(torch.int16), rk[b, :, :n].view(torch.int16))
            assert torch.equal(dv[l, b, :, :n].cpu().view(torch.int16), rv[b, :, :n].view(torch.int16))


def test_retention_on_tensor_cores_matches_calls_and_captures(fx):
    """FastKV retention with 32 window rows per KV head: the scoring takes the tensor-core route, eight
    layers per launch (11 layers: a batch of 8, then one of 3).  Equal to the individual calls (scores of
    one layer, top-k, compaction) and to the oracle; the same call captured in a CUDA graph and replayed
    gives the same result."""
    n_layers, B, Hkv, G, Mq, T, keep = 11, 2, 2, 4, 8, 3000, 300
    cand = T - Mq
    ks = torch.stack([rnd((B, Hkv, T, D), 190 + l, 1) for l in range(n_layers)])
    vs = torch.stack([rnd((B, Hkv, T, D), 190 + l, 2) for l in range(n_layers)])
    qs = torch.stack([rnd((B, Hkv * G, Mq, D), 190 + l, 3) for l in range(n_layers)])
    length = torch.tensor([T, 2100], dtype=torch.int32)
    cap = keep + Mq + 8
    dks, dvs, dls, dl = dev(ks), dev(vs), dev(length), torch.zeros(B, dtype=torch.int32, device="cuda")
    dk = torch.zeros((n_layers, B, Hkv, cap, D), dtype=torch.bfloat16, device="cuda")
    dv = torch.zeros_like(dk)
    idx = fx.fx_kv_retain_per_layer(dks, dvs, dls, dev(qs), keep, cand, cand, dk, dv, dl, q_pos0=cand,
                                    flags=fx.FX_LAUNCH_PDL)
    torch.cuda.synchronize()
    assert fx.fx_device_errors() == 0
    for l in range(n_layers):
        _, sc = fx.fx_focal_attn_scores(dks[l], dvs[l], dls, dev(qs[l]), q_pos0=cand, cand=(0, cand), want_out=False)
        ref_gpu = fx.fx_topk_select(sc.reshape(B * Hkv, cand), keep).reshape(B, Hkv, keep)
        assert torch.equal(idx[l], ref_gpu), l
        if l in (0, n_layers - 1):
            _, osc = oracle.focal(ks[l], vs[l], length, qs[l], q_pos0=cand, cand=(0, cand), want_out=False)
            pu.check_index_sets(idx[l], oracle.topk(osc, keep), osc, keep)
        rk, rv, rl = oracle.kv_compact(ks[l], vs[l], length, idx[l].cpu(), cand, cap)
        assert torch.equal(dl.cpu(), rl)
        for b in range(B):
            n = int(rl[b])
            assert torch.equal(dk[l, b, :, :n].cpu().view(torch.int16), rk[b, :, :n].view(torch.int16))
    # captured in a CUDA graph and replayed
    idx2 = torch.full_like(idx, -1)
    dk2, dv2 = torch.zeros_like(dk), torch.zeros_like(dv)
    dl2 = torch.zeros_like(dl)
    dq = dev(qs)
    ws = fx.Workspace(torch.device("cuda", 0),
                      fx.load_library().fx_retain_workspace_bytes(B, Hkv, Hkv * G, Mq, T, cand))
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        fx.fx_kv_retain_per_layer(dks, dvs, dls, dq, keep, cand, cand, dk2, dv2, dl2, q_pos0=cand, idx_out=idx2, ws=ws,
                                  stream=s)
    graph.replay()
    torch.cuda.synchronize()
    assert fx.fx_device_errors() == 0
    assert torch.equal(idx2, idx) and torch.equal(dk2, dk) and torch.equal(dl2, dl)


def test_focal_layer_profiling_matches_oracle(fx):
    """Warm-up profiling of the image-attention ratio per layer (fx_focal_mass over each layer's image
    scores, accumulated over the warm-up steps) and the choice of the C focal layers."""
    n_layers, B, Hkv, G, T, n_img, steps, C = 4, 2, 2, 2, 300, 200, 2, 2
    boost = (0.0, 0.5, 0.15, 0.9)   # how strongly each layer's image keys align with the queries
    length = torch.tensor([T, 260], dtype=torch.int32)
    qs = [[rnd((B, Hkv * G, 1, D), 170 + t, 10 + l) for l in range(n_layers)] for t in range(steps)]
    ks, vs = [], []
    for l in range(n_layers):
        k = rnd((B, Hkv, T, D), 180 + l, 1).float()
        u = sum(qs[t][l].float().sum(dim=2) for t in range(steps))          # [B, Hq, D]
        u = u.view(B, Hkv, G, D).sum(dim=2)
        u = u / u.norm(dim=-1, keepdim=True)
        k[:, :, :n_img] += boost[l] * 4.0 * u[:, :, None, :]
        ks.append(k.to(torch.bfloat16))
        vs.append(rnd((B, Hkv, T, D), 180 + l, 2))
    mass = [torch.zeros((B, Hkv), dtype=torch.float32, device="cuda") for _ in range(n_layers)]
    ref = [np.zeros((B, Hkv)) for _ in range(n_layers)]
    for t in range(steps):
        for l in range(n_layers):
            _, sc = fx.fx_focal_attn_scores(dev(ks[l]), dev(vs[l]), dev(length), dev(qs[t][l]), cand=(0, n_img),
                                            want_out=False)
            fx.fx_focal_mass(sc, G, mass=mass[l], accumulate=t > 0)
            _, rsc = oracle.focal(ks[l], vs[l], length, qs[t][l], cand=(0, n_img), want_out=False)
            ref[l] += oracle.focal_mass(rsc, G)
    torch.cuda.synchronize()
    assert fx.fx_device_errors() == 0
    for l in range(n_layers):
        got = mass[l].cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - ref[l]) <= 1e-4 * np.abs(ref[l]) + 1e-7), (l, got, ref[l])
    ratio = [float(mass[l].mean()) / steps for l in range(n_layers)]
    ref_ratio = [float(ref[l].mean()) / steps for l in range(n_layers)]
    assert fx.fx_choose_focal_layers(ratio, C) == oracle.choose_focal_layers(ref_ratio, C) == [1, 3]


def test_kv_append_matches_oracle(fx):
    """Decode-step append into the caches of 3 layers (strided layer views of one buffer), rows at the
    first and last capacity positions and in between; then a dense decode over the grown cache equals
    the oracle's decode over the oracle's appended cache."""
    L, B, Hkv, T, G = 3, 3, 2, 40, 2
    full_k, full_v = rnd((L, B, Hkv, T + 8, D), 400, 1), rnd((L, B, Hkv, T + 8, D), 400, 2)
    buf_k, buf_v = full_k[:, :, :, :T], full_v[:, :, :, :T]   # caches of capacity T in padded rows
    k_new, v_new = rnd((L, B, Hkv, D), 400, 3), rnd((L, B, Hkv, D), 400, 4)
    pos = torch.tensor([0, T - 1, 17], dtype=torch.int32)
    ref_k, ref_v = oracle.kv_append(buf_k, buf_v, k_new, v_new, pos)
    gk_full, gv_full = dev(full_k), dev(full_v)
    gk, gv = gk_full[:, :, :, :T], gv_full[:, :, :, :T]
    fx.fx_kv_append(gk, gv, dev(k_new), dev(v_new), dev(pos))
    torch.cuda.synchronize()
    assert fx.fx_device_errors() == 0
    assert torch.equal(gk.cpu().view(torch.int16), ref_k.view(torch.int16))
    assert torch.equal(gv.cpu().view(torch.int16), ref_v.view(torch.int16))
    assert torch.equal(gk_full[:, :, :, T:].cpu().view(torch.int16), full_k[:, :, :, T:].view(torch.int16))
    # decode over len = pos + 1 on layer 1 of both caches
    length = pos + 1
    q = rnd((B, Hkv * G, 1, D), 400, 5)
    ref = oracle.sparse_decode(ref_k[1], ref_v[1], length, q, None, 0)
    out = fx.fx_sparse_gqa_decode(gk[1], gv[1], dev(length), dev(q), None, 0)
    pu.assert_out_close(out, ref, float(ref_v[1].float().abs().max()))


def test_kv_append_rejects_positions_past_capacity(fx):
    B, Hkv, T = 2, 2, 16
    k, v = kv_case(B, Hkv, T, 401)
    k_new, v_new = rnd((B, Hkv, D), 401, 3), rnd((B, Hkv, D), 401, 4)
    gk, gv = dev(k), dev(v)
    fx.fx_device_errors()
    fx.fx_kv_append(gk, gv, dev(k_new), dev(v_new), dev(torch.tensor([T, 5], dtype=torch.int32)))
    torch.cuda.synchronize()
    assert fx.fx_device_errors() & fx.FX_DEVERR_LEN
    ref_k, ref_v = oracle.kv_append(k, v, k_new, v_new, torch.tensor([-1, 5], dtype=torch.int32))
    assert torch.equal(gk.cpu().view(torch.int16), ref_k.view(torch.int16))
    assert torch.equal(gv.cpu().view(torch.int16), ref_v.view(torch.int16))


def test_compaction_capacity_is_flagged(fx):
    B, Hkv, T = 1, 1, 50
    k, v = kv_case(B, Hkv, T, 60)
    length = torch.tensor([50], dtype=torch.int32)
    dk = torch.zeros((B, Hkv, 30, D), dtype=torch.bfloat16, device="cuda")
    dv = torch.zeros_like(dk)
    dl = torch.zeros(B, dtype=torch.int32, device="cuda")
    fx.fx_device_errors()
    fx.fx_kv_compact(dev(k), dev(v), dev(length), None, 10, dk, dv, dl)
    assert fx.fx_device_errors() & fx.FX_DEVERR_CAPACITY
    assert int(dl[0]) == 30
    assert torch.equal(dk[0, 0].cpu().view(torch.int16), k[0, 0, 10:40].view(torch.int16))


# ----------------------------------------------------------------------------------------------
@pytest.mark.parametrize("sparse", [False, True])
def test_shared_prefix_matches_oracle(fx, sparse):
    Hkv, G, P, Mq, Br = 2, 2, 300, 7, 5
    lens = [0, 130, 1, 77, 200]
    off = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32)
    S = int(off[-1])
    pk, pv = rnd((Hkv, P, D), 70, 1), rnd((Hkv, P, D), 70, 2)
    sk, sv = rnd((Hkv, S, D), 70, 3), rnd((Hkv, S, D), 70, 4)
    dk, dv = rnd((Br, Mq, Hkv, D), 70, 5), rnd((Br, Mq, Hkv, D), 70, 6)
    q = rnd((Br, Hkv * G, Mq, D), 70, 7)
    pidx = _sorted_subsets(Br, Hkv, P, 48, 3) if sparse else None
    ref = oracle.shared_prefix(pk, pv, sk, sv, off, dk, dv, q, pidx)
    out = fx.fx_shared_prefix_decode(dev(pk), dev(pv), dev(sk), dev(sv), dev(off), dev(dk), dev(dv), dev(q),
                                     max_suffix=256, prefix_idx=dev(pidx) if sparse else None)
    torch.cuda.synchronize()
    assert fx.fx_device_errors() == 0
    vmax = max(float(t.float().abs().max()) for t in (pv, sv, dv))
    pu.assert_out_close(out, ref, vmax)


@pytest.mark.parametrize("sparse", [False, True])
def test_forked_branches_from_pool_match_oracle(fx, sparse):
    """Branches forked from a growing shared prefix (branch pool: fork positions, fixed suffix slots)
    verified in one fx_shared_prefix_decode call, against the oracle with the same fork positions."""
    Hkv, G, Mq, slot, cap = 2, 2, 3, 40, 300
    pool = fx.BranchPool(prefix_cap=cap, max_branches=6, slot_rows=slot)
    pool.extend_prefix(120)
    ids = [pool.fork(), pool.fork()]
    pool.extend_prefix(60)
    ids.append(pool.fork())
    pool.extend_prefix(100)
    ids.append(pool.fork())
    pool.release(ids[1])                       # a finished branch leaves a hole
    for b, n in zip((ids[0], ids[2], ids[3]), (25, 0, 40)):
        if n:
            pool.append(b, n)
    live, start, slen, plen = pool.batch()
    Br = live.numel()
    P = pool.prefix_len()
    pk, pv = rnd((Hkv, P, D), 190, 1), rnd((Hkv, P, D), 190, 2)
    sk, sv = rnd((Hkv, 6 * slot, D), 190, 3), rnd((Hkv, 6 * slot, D), 190, 4)
    dk, dv = rnd((Br, Mq, Hkv, D), 190, 5), rnd((Br, Mq, Hkv, D), 190, 6)
    q = rnd((Br, Hkv * G, Mq, D), 190, 7)
    pidx = None
    if sparse:
        # each branch picks 16 prefix positions among the ones it can see
        g = np.random.default_rng(190)
        pidx = torch.from_numpy(np.stack([np.stack([np.sort(g.choice(int(plen[b]), 16, replace=False))
                                                    for _ in range(Hkv)]) for b in range(Br)]).astype(np.int32))
    ref = oracle.shared_prefix(pk, pv, sk, sv, start, dk, dv, q, pidx, pre_len=plen, suf_len=slen)
    out = fx.fx_shared_prefix_decode(dev(pk), dev(pv), dev(sk), dev(sv), dev(start), dev(dk), dev(dv), dev(q),
                                     max_suffix=slot, prefix_idx=dev(pidx) if sparse else None,
                                     prefix_len=dev(plen), suf_len=dev(slen))
    torch.cuda.synchronize()
    assert fx.fx_device_errors() == 0
    vmax = max(float(t.float().abs().max()) for t in (pv, sv, dv))
    pu.assert_out_close(out, ref, vmax)


@pytest.mark.parametrize("fork", [False, True])
def test_dense_prefix_on_tensor_cores_matches_oracle(fx, fork):
    """A dense prefix of at least one 128-key tile with at least 128 query rows per KV head takes the
    tensor-core route (S = Q K^T and O = P V per 128 x 128 tile, partials folded into the verify
    merge): 168 rows (one full and one ragged row tile), 700 prefix keys (a ragged last key tile), and
    with fork positions 0, 1, 127, 128, 129, 640 and 700 (empty, one key, both sides of a tile edge)."""
    Hkv, G, Mq, Br, P = 2, 2, 7, 12, 700
    lens = [3, 0, 9, 1, 0, 12, 5, 7, 2, 0, 4, 6]
    off = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32)
    S = int(off[-1])
    pk, pv = rnd((Hkv, P, D), 75, 1), rnd((Hkv, P, D), 75, 2)
    sk, sv = rnd((Hkv, S, D), 75, 3), rnd((Hkv, S, D), 75, 4)
    dk, dv = rnd((Br, Mq, Hkv, D), 75, 5), rnd((Br, Mq, Hkv, D), 75, 6)
    q = rnd((Br, Hkv * G, Mq, D), 75, 7)
    plen = torch.tensor([0, 1, 127, 128, 129, 640, 700, 700, 3, 255, 256, 511], dtype=torch.int32) if fork else None
    ref = oracle.shared_prefix(pk, pv, sk, sv, off, dk, dv, q, None, pre_len=plen)
    out = fx.fx_shared_prefix_decode(dev(pk), dev(pv), dev(sk), dev(sv), dev(off), dev(dk), dev(dv), dev(q),
                                     max_suffix=16, prefix_len=dev(plen) if fork else None)
    torch.cuda.synchronize()
    assert fx.fx_device_errors() == 0
    vmax = max(float(t.float().abs().max()) for t in (pv, sv, dv))
    pu.assert_out_close(out, ref, vmax)


@pytest.mark.parametrize("G,Mq,Br,P", [(4, 3, 11, 128), (1, 8, 17, 129), (2, 7, 10, 256), (8, 2, 9, 383)])
def test_dense_prefix_tile_edges_on_tensor_cores(fx, G, Mq, Br, P):
    """Tensor-core prefix route at tile edges: one full key tile (128), one key past it (129), two full
    tiles (256), a ragged third (383); 132 to 144 query rows (a second, nearly empty row tile) with
    group sizes 1 to 8 and 2 to 8 draft positions."""
    Hkv = 2
    lens = [(3 * b) % 11 for b in range(Br)]
    off = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32)
    S = max(1, int(off[-1]))
    seed = 300 + P
    pk, pv = rnd((Hkv, P, D), seed, 1), rnd((Hkv, P, D), seed, 2)
    sk, sv = rnd((Hkv, S, D), seed, 3), rnd((Hkv, S, D), seed, 4)
    dk, dv = rnd((Br, Mq, Hkv, D), seed, 5), rnd((Br, Mq, Hkv, D), seed, 6)
    q = rnd((Br, Hkv * G, Mq, D), seed, 7)
    assert Br * G * Mq >= 128
    ref = oracle.shared_prefix(pk, pv, sk, sv, off, dk, dv, q, None)
    out = fx.fx_shared_prefix_decode(dev(pk), dev(pv), dev(sk), dev(sv), dev(off), dev(dk), dev(dv), dev(q),
                                     max_suffix=16)
    torch.cuda.synchronize()
    assert fx.fx_device_errors() == 0
    vmax = max(float(t.float().abs().max()) for t in (pv, sv, dv))
    pu.assert_out_close(out, ref, vmax)


def test_sparse_long_dense_tail(fx):
    """70000 keys in one row (one (b, h) pair): 16 splits of about 4400 keys, each CTA's ring cycling
    hundreds of times, merged inside one cluster."""
    B, Hkv, G, T = 1, 1, 2, 70000
    k, v = kv_case(B, Hkv, T, 81)
    q = rnd((B, Hkv * G, 1, D), 81, 3)
    length = torch.tensor([T - 5], dtype=torch.int32)
    idx = torch.tensor([[[3, 17, 40000]]], dtype=torch.int32)
    ref = oracle.sparse_decode(k, v, length, q, idx, 50)
    out = fx.fx_sparse_gqa_decode(dev(k), dev(v), dev(length), dev(q), dev(idx), 50)
    torch.cuda.synchronize()
    assert fx.fx_device_errors() == 0
    pu.assert_out_close(out, ref, float(v.float().abs().max()))


@pytest.mark.parametrize("n_keys", [1, 63, 64, 65, 130, 1000, 1023, 1025])
def test_sparse_split_counts(fx, n_keys):
    """Key counts around tile and cluster boundaries (1 to 16 splits of one cluster)."""
    B, Hkv, G = 2, 2, 2
    T = n_keys + 3
    k, v = kv_case(B, Hkv, T, 90 + n_keys % 7)
    q = rnd((B, Hkv * G, 1, D), 91, 3)
    length = torch.tensor([n_keys, max(1, n_keys // 2)], dtype=torch.int32)
    ref = oracle.sparse_decode(k, v, length, q, None, 0)
    out = fx.fx_sparse_gqa_decode(dev(k), dev(v), dev(length), dev(q), None, 0)
    pu.assert_out_close(out, ref, float(v.float().abs().max()))


def test_programmatic_dependent_launch_chain_is_identical(fx):
    """The same focal -> top-k -> sparse -> sparse chain launched plainly and as programmatic dependent
    launches (with and without early input reads) gives bit-identical results."""
    B, Hkv, G, T, kk = 2, 2, 2, 900, 40
    k, v = kv_case(B, Hkv, T, 101)
    q1, q2, q3 = (rnd((B, Hkv * G, 1, D), 101, s) for s in (3, 4, 5))
    length = torch.tensor([T, 777], dtype=torch.int32)
    dk, dv, dl = dev(k), dev(v), dev(length)

    def chain(flags_focal, flags_topk, flags_sp1, flags_sp2):
        out0, sc = fx.fx_focal_attn_scores(dk, dv, dl, dev(q1), cand=(0, 700), flags=flags_focal)
        idx = fx.fx_topk_select(sc, kk, flags=flags_topk)
        o1 = fx.fx_sparse_gqa_decode(dk, dv, dl, dev(q2), idx, 700, flags=flags_sp1)
        o2 = fx.fx_sparse_gqa_decode(dk, dv, dl, dev(q3), idx, 700, flags=flags_sp2)
        torch.cuda.synchronize()
        return [t.clone() for t in (out0, sc, idx, o1, o2)]

    P, R = fx.FX_LAUNCH_PDL, fx.FX_LAUNCH_INPUTS_READY
    plain = chain(0, 0, 0, 0)
    for variant in ((P, P, P, P), (P | R, P, P, P | R)):
        got = chain(*variant)
        for a, b in zip(plain, got):
            assert torch.equal(a, b)
    assert fx.fx_device_errors() == 0
    ref = oracle.sparse_decode(k, v, length, q3, plain[2].cpu(), 700)
    pu.assert_out_close(plain[4], ref, float(v.float().abs().max()))


def test_sparse_pdl_chain_of_layers_is_identical(fx):
    """Twelve decode layers back to back as programmatic dependent launches that read their lengths,
    index lists and K/V early (the next layer's CTAs are resident and loading while the previous layer
    runs) give bit-identical results to plain launches, and match the oracle."""
    B, Hkv, G, T, kk, L = 8, 8, 2, 1200, 205, 12
    ks = torch.stack([rnd((B, Hkv, T, D), 120 + l, 1) for l in range(L)]).to("cuda")
    vs = torch.stack([rnd((B, Hkv, T, D), 120 + l, 2) for l in range(L)]).to("cuda")
    qs = torch.stack([rnd((B, Hkv * G, 1, D), 140 + l, 3) for l in range(L)]).to("cuda")
    length = torch.tensor([T - 3 * b for b in range(B)], dtype=torch.int32)
    idx = _sorted_subsets(B, Hkv, 800, kk, 7)
    dl, di = dev(length), dev(idx)
    outs = torch.zeros((2, L, B, Hkv * G, 1, D), dtype=torch.float32, device="cuda")
    P, R = fx.FX_LAUNCH_PDL, fx.FX_LAUNCH_INPUTS_READY
    for v_, fl in enumerate((0, P | R)):
        for l in range(L):
            fx.fx_sparse_gqa_decode(ks[l], vs[l], dl, qs[l], di, 800, out=outs[v_, l], flags=fl)
    torch.cuda.synchronize()
    assert fx.fx_device_errors() == 0
    assert torch.equal(outs[0], outs[1])
    for l in (0, 5, 11):
        ref = oracle.sparse_decode(ks[l].cpu(), vs[l].cpu(), length, qs[l].cpu(), idx, 800)
        pu.assert_out_close(outs[1, l], ref, float(vs[l].float().abs().max()))


def test_bounded_wait_runs_out_and_is_reported(fx):
    """A device-side wait that nothing completes gives up after its poll limit: the call returns, the
    context stays usable, the result is unaffected and FX_DEVERR_TIMEOUT is reported."""
    B, Hkv, G, T = 2, 2, 2, 500
    k, v = kv_case(B, Hkv, T, 61)
    q = rnd((B, Hkv * G, 1, D), 61, 3)
    length = torch.tensor([T, 321], dtype=torch.int32)
    ref = oracle.sparse_decode(k, v, length, q, None, 0)
    fx.fx_device_errors()
    lib = fx.load_library()
    lib.fx_test_stall_wait(2000)
    try:
        out = fx.fx_sparse_gqa_decode(dev(k), dev(v), dev(length), dev(q), None, 0)
        torch.cuda.synchronize()
        bits = fx.fx_device_errors()
    finally:
        lib.fx_test_stall_wait(0)
    assert bits & fx.FX_DEVERR_TIMEOUT
    pu.assert_out_close(out, ref, float(v.float().abs().max()))
    again = fx.fx_sparse_gqa_decode(dev(k), dev(v), dev(length), dev(q), None, 0)
    torch.cuda.synchronize()
    assert fx.fx_device_errors() == 0
    assert torch.equal(out, again)


def test_sparse_without_tensor_maps_matches_oracle(fx):
    """A cache view whose batch stride is 0 (every sequence reads the same rows) cannot be described by a
    TMA tensor map; the decode kernel then copies the contiguous tail rows with cp.async as well.  Same
    results as the oracle over the broadcast cache."""
    B, Hkv, G, T, kk = 4, 2, 2, 900, 61
    k1, v1 = kv_case(1, Hkv, T, 131)
    kb = dev(k1).expand(B, Hkv, T, D)
    vb = dev(v1).expand(B, Hkv, T, D)
    assert kb.stride(0) == 0
    q = rnd((B, Hkv * G, 1, D), 131, 3)
    length = torch.tensor([T, 800, 517, 300], dtype=torch.int32)
    idx = _sorted_subsets(B, Hkv, 300, kk, 5)
    out = fx.fx_sparse_gqa_decode(kb, vb, dev(length), dev(q), dev(idx), 300)
    torch.cuda.synchronize()
    assert fx.fx_device_errors() == 0
    ref = oracle.sparse_decode(k1.expand(B, Hkv, T, D).contiguous(), v1.expand(B, Hkv, T, D).contiguous(), length, q,
                               idx, 300)
    pu.assert_out_close(out, ref, float(v1.float().abs().max()))

