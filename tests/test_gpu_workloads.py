"""Parity at the full workload sizes, on sampled rows.

The device runs each workload end to end through the library at its full size; the fp64 oracle then
recomputes sampled (sequence / branch, KV head) rows from host-regenerated inputs (the generator is
bit-identical on both devices, checked first) and the two are compared:
  outputs      max |gpu - oracle| <= 2e-3 * max|V|
  importance   relative 1e-4
  index sets   exact on rows whose oracle rank-k / rank-(k+1) gap is >= 1e-3; otherwise the
               tie-tolerant check
  compaction   bit-exact
Every sampled output is compared.  An output that depends on a selected set is compared with the
oracle run on the library's set once that set has passed the index-set check: on a gapped row it is
the oracle's own set; on a row where a near-tie resolved the other way the library's set is an equally
valid top-k, and the oracle then attends over it.  Each test counts the rows it compared and the
gapped rows, and asserts that nothing sampled went uncompared.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth.workloads import D, HpdBranch, KvSelect, LongCtx, OcrDecode
from tests import parity_util as pu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kv_cache_token_fx_gb300 as fx
    fx.load_library()


def _as_kv(rows):
    return rows.view(1, 1, *rows.shape).contiguous()


def _validated_set(gpu_set, ref_set, ref_scores, k, stats):
    """The set the oracle attends over for an output that depends on a selection: the library's set,
    after the index-set check (exact on gapped rows, tie-tolerant otherwise).  Counts rows where the
    two sets differ (near-ties resolved the other way)."""
    g = np.asarray(gpu_set).reshape(-1)
    pu.check_index_sets(g.reshape(1, -1), np.asarray(ref_set).reshape(1, -1),
                        np.asarray(ref_scores).reshape(1, -1), k)
    if not np.array_equal(g, np.asarray(ref_set).reshape(-1)):
        stats["tie_sets"] = stats.get("tie_sets", 0) + 1
    return g.astype(np.int32)


def test_generator_is_bit_identical_across_devices():
    s = synth.stream_id(3, 9)
    a = synth.normal_bf16(7, s, (3, 1000), device="cuda", offset=123456789012).cpu()
    b = synth.normal_bf16(7, s, (3, 1000), device="cpu", offset=123456789012)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    w = OcrDecode()
    tab = w.fourier_table(5)
    k, v = w.layer_kv(5, device="cuda", table=tab)
    kr, vr = w.layer_kv_rows(5, 3, 6, table=tab)
    assert torch.equal(k[3, 6].cpu().view(torch.int16), kr.view(torch.int16))
    assert torch.equal(v[3, 6].cpu().view(torch.int16), vr.view(torch.int16))
    assert torch.equal(w.query(9, 5, device="cuda", table=tab).cpu().view(torch.int16),
                       w.query(9, 5, table=tab).view(torch.int16))
    ks = KvSelect()
    k15, _ = ks.layer_kv(ks.switch_layer, device="cuda")
    r15, _ = ks.layer_kv_rows(ks.switch_layer, 2, 3)
    assert torch.equal(k15[2, 3].cpu().view(torch.int16), r15.view(torch.int16))


# ----------------------------------------------------------------------------------------------
def test_ocr_decode_full_run_sampled():
    from tests.workload_runs import ocr_decode_run
    w = OcrDecode()
    keep = (0, 1, 2, 131, 255)
    gpu = ocr_decode_run(w, set(keep))
    G = w.Hq // w.Hkv
    pairs = [(0, 0), (3, 5), (7, 7)]
    layers_check = (0, 2, 3, 5, 14, 20, 27)
    tables = {}
    stats = dict(rows=0, gapped=0, exact=0, sparse_checked=0)
    for t in keep:
        L_t = w.length_at(t)
        ln = torch.tensor([L_t], dtype=torch.int32)
        for b, h in pairs:
            # the oracle's own sets at this step (and layer 14's at the previous step)
            own = {}
            for (l, tt) in ((3, t), (14, t)) + (((14, t - 1),) if t > 0 else ()):
                tab = tables.setdefault(l, w.fourier_table(l))
                kr, vr = w.layer_kv_rows(l, b, h, table=tab)
                q = w.query(tt, l, table=tab)[b:b + 1, h * G:(h + 1) * G].contiguous()
                lnt = torch.tensor([w.length_at(tt)], dtype=torch.int32)
                out, sc = oracle.focal(_as_kv(kr), _as_kv(vr), lnt, q, cand=(0, w.n_vis))
                own[(l, tt)] = (oracle.topk(sc, w.k_keep)[0, 0], sc[0, 0], out)
            for l in layers_check:
                tab = tables.setdefault(l, w.fourier_table(l))
                kr, vr = w.layer_kv_rows(l, b, h, table=tab)
                q = w.query(t, l, table=tab)[b:b + 1, h * G:(h + 1) * G].contiguous()
                vmax = float(vr.float().abs().max())
                g_out = gpu[t]["out"][l, b, h * G:(h + 1) * G]
                if l in w.focal_layers:
                    ref_idx, ref_sc, ref_out = own[(l, t)]
                    pu.assert_out_close(g_out, ref_out[0], vmax, f"t{t} l{l} focal out")
                    pu.assert_scores_close(gpu[t]["scores"][l][b, h], ref_sc, f"t{t} l{l} scores")
                    r, gp, ex = pu.check_index_sets(gpu[t]["sets"][l][b, h].view(1, -1), ref_idx.reshape(1, -1),
                                                     ref_sc.reshape(1, -1), w.k_keep)
                    stats["rows"] += r
                    stats["gapped"] += gp
                    stats["exact"] += ex
                    continue
                kind, src = oracle.csfr_schedule(w.n_layers, w.focal_layers, first_step=(t == 0))[l]
                if kind == "dense":
                    ref = oracle.sparse_decode(_as_kv(kr), _as_kv(vr), ln, q, None, 0)
                    pu.assert_out_close(g_out, ref[0], vmax, f"t{t} l{l} dense")
                    stats["sparse_checked"] += 1
                    continue
                if kind == "previous":
                    src_layer, src_t, gpu_set = src, t - 1, gpu[t]["prev14"][b, h]
                else:
                    src_layer, src_t, gpu_set = src, t, gpu[t]["sets"][src][b, h]
                ref_set, ref_sc = own[(src_layer, src_t)][0], own[(src_layer, src_t)][1]
                use = _validated_set(gpu_set, ref_set, ref_sc, w.k_keep, stats)
                ref = oracle.sparse_decode(_as_kv(kr), _as_kv(vr), ln, q, torch.from_numpy(use).view(1, 1, -1),
                                           w.n_vis)
                pu.assert_out_close(g_out, ref[0], vmax, f"t{t} l{l} sparse")
                stats["sparse_checked"] += 1
    n_sparse = len(pairs) * sum(5 for t in keep)   # layers 0, 2, 5, 20, 27 of every sampled step
    assert stats["sparse_checked"] == n_sparse, stats
    assert stats["rows"] == len(keep) * len(pairs) * 2, stats
    print("ocr_decode sampled:", stats)


# ----------------------------------------------------------------------------------------------
def test_kv_select_full_sampled():
    from tests.workload_runs import kv_select_run
    w = KvSelect()
    sample_layers = (0, w.switch_layer, w.n_layers - 1)
    steps = (0, 1, w.decode_steps - 1)
    gpu = kv_select_run(w, steps, sample_layers)
    T, G, ncand = w.T, w.Hq // w.Hkv, w.T - w.window
    assert gpu["clen"].tolist() == [w.keep] * w.B
    qw = w.window_queries("cpu")
    appended = {l: w.appended_kv(l) for l in sample_layers}
    stats = dict(rows=0, gapped=0, compacted=0, decoded=0)
    pairs = [(0, 0), (2, 5), (3, 7)]
    for b, h in pairs:
        kr, vr = w.layer_kv_rows(w.switch_layer, b, h)
        q = qw[b:b + 1, h * G:(h + 1) * G].contiguous()
        _, sc = oracle.focal(_as_kv(kr), _as_kv(vr), torch.tensor([T], dtype=torch.int32), q, q_pos0=T - w.window,
                             cand=(0, ncand), want_out=False)
        pu.assert_scores_close(gpu["scores"][b, h], sc[0, 0], f"scores b{b} h{h}")
        ref_idx = oracle.topk(sc[0, 0], w.k_select)
        _, gp, _ = pu.check_index_sets(gpu["idx"][b, h].view(1, -1), ref_idx.reshape(1, -1),
                                       sc[0, 0].reshape(1, -1), w.k_select)
        stats["rows"] += 1
        stats["gapped"] += gp
        use = _validated_set(gpu["idx"][b, h].numpy(), ref_idx, sc[0, 0], w.k_select, stats)
        for l in sample_layers:
            krl, vrl = w.layer_kv_rows(l, b, h)
            ck, cv, cl = oracle.kv_compact(_as_kv(krl), _as_kv(vrl), torch.tensor([T], dtype=torch.int32),
                                           torch.from_numpy(use).view(1, 1, -1), ncand, w.compact_cap)
            assert int(cl[0]) == w.keep
            gk, gv = gpu["compact"][l]
            assert torch.equal(gk[b, h, :w.keep].view(torch.int16), ck[0, 0, :w.keep].view(torch.int16))
            assert torch.equal(gv[b, h, :w.keep].view(torch.int16), cv[0, 0, :w.keep].view(torch.int16))
            stats["compacted"] += 1
            ak, av = appended[l]
            for t in steps:
                full_k = torch.cat([ck[0, 0, :w.keep], ak[b, h, :t + 1]])
                full_v = torch.cat([cv[0, 0, :w.keep], av[b, h, :t + 1]])
                q = w.decode_query(t, l)[b:b + 1, h * G:(h + 1) * G].contiguous()
                n = full_k.shape[0]
                ref = oracle.sparse_decode(_as_kv(full_k), _as_kv(full_v), torch.tensor([n], dtype=torch.int32), q,
                                           None, 0)
                pu.assert_out_close(gpu["decode"][(t, l)][b, h * G:(h + 1) * G], ref[0],
                                    float(full_v.float().abs().max()), f"decode t{t} l{l} b{b} h{h}")
                stats["decoded"] += 1
    assert stats["compacted"] == len(pairs) * len(sample_layers), stats
    assert stats["decoded"] == len(pairs) * len(sample_layers) * len(steps), stats
    print("kv_select sampled:", stats)


def test_kv_select_per_layer_retention_full_sampled():
    """FastKV per-layer retention at the full kv_select size, launched as the bench launches it (the 32
    layers' window scores in one tensor-core launch, one top-k over their 1024 rows, one compaction;
    programmatic dependent launches).  Sampled (layer, sequence, KV head) rows against the oracle's window
    scores and top-k; the compaction bit for bit on the validated set."""
    import kv_cache_token_fx_gb300 as fx
    w = KvSelect()
    L, B, Hkv, Hq, T, win = w.n_layers, w.B, w.Hkv, w.Hq, w.T, w.window
    G, ncand, cap = Hq // Hkv, T - win, w.compact_cap
    dev = torch.device("cuda", 0)
    K = torch.empty((L, B, Hkv, T, D), dtype=torch.bfloat16, device=dev)
    V = torch.empty_like(K)
    QW = torch.empty((L, B, Hq, win, D), dtype=torch.bfloat16, device=dev)
    for l in range(L):
        k, v = w.layer_kv_salient(l, device=dev)
        K[l].copy_(k)
        V[l].copy_(v)
        QW[l].copy_(w.window_queries_at(l, device=dev))
        del k, v
    ln = torch.full((B,), T, dtype=torch.int32, device=dev)
    CK = torch.zeros((L, B, Hkv, cap, D), dtype=torch.bfloat16, device=dev)
    CV = torch.zeros_like(CK)
    clen = torch.zeros(B, dtype=torch.int32, device=dev)
    idx = fx.fx_kv_retain_per_layer(K, V, ln, QW, w.k_select, ncand, ncand, CK, CV, clen, q_pos0=ncand,
                                    flags=fx.FX_LAUNCH_PDL)
    torch.cuda.synchronize()
    assert fx.fx_device_errors() == 0
    assert clen.tolist() == [w.keep] * B
    del K, V
    samples = [(0, 0, 0), (7, 1, 3), (w.switch_layer, 2, 5), (16, 3, 7), (24, 0, 6), (L - 1, 3, 1)]
    stats = dict(rows=0, gapped=0, compacted=0)
    lt = torch.tensor([T], dtype=torch.int32)
    for l, b, h in samples:
        kr, vr = w.layer_kv_salient_rows(l, b, h)
        q = w.window_queries_at(l)[b:b + 1, h * G:(h + 1) * G].contiguous()
        _, sc = oracle.focal(_as_kv(kr), _as_kv(vr), lt, q, q_pos0=ncand, cand=(0, ncand), want_out=False)
        ref_idx = oracle.topk(sc[0, 0], w.k_select)
        g_idx = idx[l, b, h].cpu().numpy()
        _, gp, _ = pu.check_index_sets(g_idx.reshape(1, -1), ref_idx.reshape(1, -1), sc[0, 0].reshape(1, -1),
                                       w.k_select)
        stats["rows"] += 1
        stats["gapped"] += gp
        use = _validated_set(g_idx, ref_idx, sc[0, 0], w.k_select, stats)
        ck, cv, cl = oracle.kv_compact(_as_kv(kr), _as_kv(vr), lt, torch.from_numpy(use).view(1, 1, -1), ncand, cap)
        assert int(cl[0]) == w.keep
        assert torch.equal(CK[l, b, h, :w.keep].cpu().view(torch.int16), ck[0, 0, :w.keep].view(torch.int16))
        assert torch.equal(CV[l, b, h, :w.keep].cpu().view(torch.int16), cv[0, 0, :w.keep].view(torch.int16))
        stats["compacted"] += 1
    assert stats["rows"] == len(samples) and stats["compacted"] == len(samples), stats
    print("kv_select per-layer retention sampled:", stats)


# ----------------------------------------------------------------------------------------------
def test_long_ctx_full_sampled():
    from tests.workload_runs import long_ctx_run
    w = LongCtx()
    gpu = long_ctx_run(w)
    G = w.Hq // w.Hkv
    q0 = w.query(0, "cpu")
    q1 = w.query(1, "cpu")
    ln = torch.tensor([w.T], dtype=torch.int32)
    # 16 (sequence, KV head) rows spread over the batch and the heads
    pairs = [(b, (5 * i + 3) % w.Hkv) for i, b in enumerate(range(0, w.B, 4))]
    assert len(pairs) == 16 and len({h for _, h in pairs}) == w.Hkv
    stats = dict(rows=0, gapped=0, sparse_checked=0)
    for b, h in pairs:
        kr, vr = w.layer_kv_rows(0, b, h)
        vmax = float(vr.float().abs().max())
        out, sc = oracle.focal(_as_kv(kr), _as_kv(vr), ln, q0[b:b + 1, h * G:(h + 1) * G].contiguous())
        pu.assert_out_close(gpu["out"][b, h * G:(h + 1) * G], out[0], vmax, f"focal out b{b} h{h}")
        pu.assert_scores_close(gpu["scores"][b, h].cpu(), sc[0, 0], f"scores b{b} h{h}")
        ref_idx = oracle.topk(sc[0, 0], w.k)
        _, gp, _ = pu.check_index_sets(gpu["idx"][b, h].view(1, -1), ref_idx.reshape(1, -1),
                                       sc[0, 0].reshape(1, -1), w.k)
        stats["rows"] += 1
        stats["gapped"] += gp
        use = _validated_set(gpu["idx"][b, h].numpy(), ref_idx, sc[0, 0], w.k, stats)
        ref = oracle.sparse_decode(_as_kv(kr), _as_kv(vr), ln, q1[b:b + 1, h * G:(h + 1) * G].contiguous(),
                                   torch.from_numpy(use).view(1, 1, -1), w.T)
        pu.assert_out_close(gpu["sparse"][b, h * G:(h + 1) * G], ref[0], vmax, f"sparse b{b} h{h}")
        stats["sparse_checked"] += 1
    assert stats["sparse_checked"] == stats["rows"] == len(pairs), stats
    print("long_ctx sampled:", stats)


# ----------------------------------------------------------------------------------------------
def test_hpd_branch_full_sampled():
    from tests.workload_runs import hpd_run
    w = HpdBranch()
    gpu = hpd_run(w)
    d = w.small_inputs(0, device="cpu")
    off = w.offsets().tolist()
    G = w.Hq // w.Hkv
    branches = (0, 100, 511)
    stats = dict(rows=0, gapped=0, dense_checked=0, sparse_checked=0)
    for b in branches:
        sk, sv = w.suffix_rows(0, b)
        vmax = max(float(t.float().abs().max()) for t in (d["pv"], sv, d["dv"]))
        o1 = torch.tensor([0, off[b + 1] - off[b]], dtype=torch.int32)
        dk, dv, q = d["dk"][b:b + 1], d["dv"][b:b + 1], d["q"][b:b + 1]
        ref = oracle.shared_prefix(d["pk"], d["pv"], sk, sv, o1, dk, dv, q)
        pu.assert_out_close(gpu["dense"][b], ref[0], vmax, f"dense branch {b}")
        stats["dense_checked"] += 1
        # sparse variant: the oracle's own prefix selection
        _, psc = oracle.focal(d["pk"].unsqueeze(0), d["pv"].unsqueeze(0), torch.tensor([w.P], dtype=torch.int32), q,
                              want_out=False)
        pu.assert_scores_close(gpu["pscores"][b], psc[0], f"prefix scores branch {b}")
        ref_idx = oracle.topk(psc[0], w.kp)
        _, gp, _ = pu.check_index_sets(gpu["pidx"][b], ref_idx, psc[0], w.kp)
        stats["rows"] += w.Hkv
        stats["gapped"] += gp
        use = np.stack([_validated_set(gpu["pidx"][b, h].numpy(), ref_idx[h], psc[0, h], w.kp, stats)
                        for h in range(w.Hkv)])
        ref_s = oracle.shared_prefix(d["pk"], d["pv"], sk, sv, o1, dk, dv, q,
                                     torch.from_numpy(use).view(1, w.Hkv, w.kp))
        pu.assert_out_close(gpu["sparse"][b], ref_s[0], vmax, f"sparse branch {b}")
        stats["sparse_checked"] += w.Hkv
    assert stats["dense_checked"] == len(branches) and stats["sparse_checked"] == len(branches) * w.Hkv, stats
    print("hpd_branch sampled:", stats)
