"""Runs of the full-size workloads through the library (GPU side only), for the parity tests.

Each function drives the public calls exactly as a user would and returns the device results the
tests then compare, on sampled rows, with the fp64 oracle run on host-regenerated slices.
"""
import torch

import kv_cache_token_fx_gb300 as fx
from synth.workloads import D, HpdBranch, KvSelect, LongCtx, OcrDecode


def ocr_decode_run(w: OcrDecode, steps_to_keep, n_steps=None, device="cuda"):
    """All decode steps 0..n_steps-1 of the FastOCR-shaped workload (CSFR schedule, warm-started
    top-k).  Returns {t: dict(out=[L,B,Hq,1,D], sets={layer: [B,Hkv,k]}, scores={layer: [B,Hkv,n_vis]})}
    for the steps in `steps_to_keep`."""
    n_steps = w.steps if n_steps is None else n_steps
    L, B, Hkv, Hq, T = w.n_layers, w.B, w.Hkv, w.Hq, w.tcap
    K = torch.empty((L, B, Hkv, T, D), dtype=torch.bfloat16, device=device)
    V = torch.empty_like(K)
    tables = []
    for l in range(L):
        tab = w.fourier_table(l)
        tables.append(tab)
        k, v = w.layer_kv(l, device=device, table=tab)
        K[l].copy_(k)
        V[l].copy_(v)
        del k, v
    sets = {l: torch.zeros((2, B, Hkv, w.k_keep), dtype=torch.int32, device=device) for l in w.focal_layers}
    scores = {l: torch.empty((B, Hkv, w.n_vis), dtype=torch.float32, device=device) for l in w.focal_layers}
    out = torch.empty((L, B, Hq, 1, D), dtype=torch.float32, device=device)
    ws = fx.Workspace(torch.device(device))
    kept = {}
    f_last = w.focal_layers[-1]
    for t in range(n_steps):
        p = t % 2
        ln = torch.full((B,), w.length_at(t), dtype=torch.int32, device=device)
        # FastOCR's cross-step fixation reuse, as the library schedules it
        kinds, srcs = fx.fx_csfr_schedule(L, w.focal_layers, first_step=(t == 0))
        for l in range(L):
            q = w.query(t, l, device=device, table=tables[l])
            if kinds[l] == fx.FX_CSFR_FOCAL:
                fx.fx_focal_attn_scores(K[l], V[l], ln, q, cand=(0, w.n_vis), out=out[l], scores=scores[l], ws=ws)
                prev = sets[l][1 - p] if t > 0 else None
                fx.fx_topk_select(scores[l], w.k_keep, prev=prev, out=sets[l][p])
                continue
            if kinds[l] == fx.FX_CSFR_DENSE:
                sel = None
            else:
                sel = sets[srcs[l]][p if kinds[l] == fx.FX_CSFR_CURRENT else 1 - p]
            fx.fx_sparse_gqa_decode(K[l], V[l], ln, q, sel, w.n_vis if sel is not None else 0, out=out[l], ws=ws)
        if t in steps_to_keep:
            torch.cuda.synchronize()
            kept[t] = dict(out=out.cpu(), sets={l: sets[l][p].cpu() for l in w.focal_layers},
                           scores={l: scores[l].cpu() for l in w.focal_layers},
                           prev14=(sets[f_last][1 - p].cpu() if t > 0 else None))
    torch.cuda.synchronize()
    return kept


def kv_select_run(w: KvSelect, decode_steps_to_keep, sample_layers, device="cuda"):
    """Scoring at the switch layer (window queries, causal), top-(keep - window) selection, compaction of
    every layer, then dense decode on the compacted caches for the kept steps."""
    L, B, Hkv, Hq, T = w.n_layers, w.B, w.Hkv, w.Hq, w.T
    K = torch.empty((L, B, Hkv, T, D), dtype=torch.bfloat16, device=device)
    V = torch.empty_like(K)
    for l in range(L):
        k, v = w.layer_kv(l, device=device)
        K[l].copy_(k)
        V[l].copy_(v)
        del k, v
    ln = torch.full((B,), T, dtype=torch.int32, device=device)
    qw = w.window_queries(device)
    ncand = T - w.window
    _, scores = fx.fx_focal_attn_scores(K[w.switch_layer], V[w.switch_layer], ln, qw, q_pos0=T - w.window,
                                        cand=(0, ncand), want_out=False)
    idx = fx.fx_topk_select(scores, w.k_select)
    cap = w.compact_cap
    CK = torch.zeros((L, B, Hkv, cap, D), dtype=torch.bfloat16, device=device)
    CV = torch.zeros_like(CK)
    clen = torch.zeros(B, dtype=torch.int32, device=device)
    fx.fx_kv_compact(K, V, ln, idx, ncand, CK, CV, clen)
    torch.cuda.synchronize()
    res = dict(scores=scores.cpu(), idx=idx.cpu(), clen=clen.cpu(),
               compact={l: (CK[l].cpu(), CV[l].cpu()) for l in sample_layers})
    del K, V
    # decode: step t appends its K/V row at position keep + t of every layer, then attends densely
    app = {l: w.appended_kv(l, device) for l in range(L)}
    for l in range(L):
        CK[l, :, :, w.keep:w.keep + w.decode_steps] = app[l][0]
        CV[l, :, :, w.keep:w.keep + w.decode_steps] = app[l][1]
    out = torch.empty((B, Hq, 1, D), dtype=torch.float32, device=device)
    dec = {}
    for t in decode_steps_to_keep:
        dl = torch.full((B,), w.keep + t + 1, dtype=torch.int32, device=device)
        for l in sample_layers:
            q = w.decode_query(t, l, device)
            fx.fx_sparse_gqa_decode(CK[l], CV[l], dl, q, None, 0, out=out)
            dec[(t, l)] = out.cpu().clone()
    torch.cuda.synchronize()
    res["decode"] = dec
    return res


def long_ctx_run(w: LongCtx, device="cuda"):
    """One focal pass over 131072 tokens per sequence, top-2048 per KV head, sparse decode over them."""
    k, v = w.layer_kv(0, device=device)
    ln = torch.full((w.B,), w.T, dtype=torch.int32, device=device)
    q = w.query(0, device)
    out, scores = fx.fx_focal_attn_scores(k, v, ln, q)
    idx = fx.fx_topk_select(scores, w.k)
    q2 = w.query(1, device)
    sp = fx.fx_sparse_gqa_decode(k, v, ln, q2, idx, w.T)
    torch.cuda.synchronize()
    return dict(out=out.cpu(), scores=scores, idx=idx.cpu(), sparse=sp.cpu())


def hpd_run(w: HpdBranch, device="cuda"):
    """Dense shared-prefix draft verification, then the sparse variant: the prefix tokens of each
    (branch, KV head) are scored with that branch's draft queries over the prefix and the top kp kept."""
    d = w.layer_inputs(0, device=device)
    dense = fx.fx_shared_prefix_decode(d["pk"], d["pv"], d["sk"], d["sv"], d["off"], d["dk"], d["dv"], d["q"],
                                       max_suffix=w.max_suffix)
    # prefix scoring: every branch sees the same prefix rows (batch stride 0)
    P = w.P
    pk4 = d["pk"].unsqueeze(0).expand(w.Br, w.Hkv, P, D)
    pv4 = d["pv"].unsqueeze(0).expand(w.Br, w.Hkv, P, D)
    plen = torch.full((w.Br,), P, dtype=torch.int32, device=device)
    _, pscores = fx.fx_focal_attn_scores(pk4, pv4, plen, d["q"], want_out=False)
    pidx = fx.fx_topk_select(pscores, w.kp)
    sparse = fx.fx_shared_prefix_decode(d["pk"], d["pv"], d["sk"], d["sv"], d["off"], d["dk"], d["dv"], d["q"],
                                        max_suffix=w.max_suffix, prefix_idx=pidx)
    torch.cuda.synchronize()
    return dict(dense=dense.cpu(), sparse=sparse.cpu(), pscores=pscores.cpu(), pidx=pidx.cpu())
