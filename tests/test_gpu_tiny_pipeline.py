"""The tiny single-step workload end to end on the GPU: focal scores over 1024 tokens, top-64 per KV
head, then sparse decode over the chosen set -- each stage compared with the oracle."""
import numpy as np
import pytest
import torch

import oracle
from synth.workloads import Tiny
from tests import parity_util as pu

pytestmark = pytest.mark.gpu


def enforce_gaps(k, v, length, q, kk, max_iter=60):
    """Make every row's rank-k / rank-(k+1) gap at least 2e-3 (relative) by halving the keys of the
    near-boundary losers, as ranked by the oracle's scores.  Halving a bf16 row is exact."""
    k = k.clone()
    for _ in range(max_iter):
        _, sc = oracle.focal(k, v, length, q)
        changed = False
        for b in range(sc.shape[0]):
            for h in range(sc.shape[1]):
                s = sc[b, h]
                order = np.lexsort((np.arange(s.size), -s))
                sk = s[order[kk - 1]]
                losers = [j for j in order[kk:] if s[j] >= sk * (1 - 2e-3)]
                for j in losers:
                    k[b, h, j] = (k[b, h, j].float() * 0.5).to(torch.bfloat16)
                    changed = True
        if not changed:
            return k, sc
    raise AssertionError("could not separate the boundary")


@pytest.fixture(scope="module")
def tiny():
    w = Tiny()
    d = w.build()
    k, sc = enforce_gaps(d["k"], d["v"], d["len"], d["q"], w.k)
    d["k"] = k
    return w, d


def test_tiny_pipeline(tiny):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kv_cache_token_fx_gb300 as fx
    w, d = tiny
    k, v, q, length = d["k"], d["v"], d["q"], d["len"]
    ref_out, ref_sc = oracle.focal(k, v, length, q)
    ref_idx = oracle.topk(ref_sc, w.k)
    assert np.all(pu.row_gaps(ref_sc.reshape(-1, w.T), w.k) >= pu.GAP)
    ref_sparse = oracle.sparse_decode(k, v, length, q, torch.from_numpy(ref_idx), w.T)

    dk, dv, dq, dl = (t.cuda() for t in (k, v, q, length))
    out, sc = fx.fx_focal_attn_scores(dk, dv, dl, dq)
    idx = fx.fx_topk_select(sc, w.k)
    sp = fx.fx_sparse_gqa_decode(dk, dv, dl, dq, idx, w.T)
    torch.cuda.synchronize()
    assert fx.fx_device_errors() == 0
    vmax = float(v.float().abs().max())
    pu.assert_out_close(out, ref_out, vmax, "focal out")
    pu.assert_scores_close(sc, ref_sc)
    rows, gapped, exact = pu.check_index_sets(idx, ref_idx, ref_sc, w.k)
    assert gapped == rows == exact == w.B * w.Hkv
    assert sp.shape == (1, 16, 1, 128)
    pu.assert_out_close(sp, ref_sparse, vmax, "sparse out")
    # every planted salient key is among the selected tokens of its head
    sel = idx.cpu().numpy()
    hits = np.mean([np.isin(d["salient"][0, h].numpy(), sel[0, h]).mean() for h in range(w.Hkv)])
    assert hits > 0.5
