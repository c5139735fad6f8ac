"""Seeded synthetic workloads shaped like the pages' settings.  No method arithmetic lives here.

Every tensor comes from the counter-based generator in ``synth`` (bit-identical on CPU and GPU).
Planted structure (salient tokens, a drifting fixation window, high-affinity tokens) is added with
elementwise float32 operations only -- a bf16 value widened to fp32, plus an fp32 table or an fp32
sum of query rows taken in a fixed order, then rounded back to bf16 -- so a slice rebuilt on the host
matches the device tensor bit for bit.  Small tables (cos/sin of random frequencies) are computed on
the host in float64 and rounded to float32 once.

Workloads (names describe what they are):
  tiny        1 sequence, 16 q / 8 KV heads, 1024 tokens, 32 planted salient keys per head, k = 64
  ocr_decode  FastOCR-shaped decode: 8 sequences x 28 layers, 4096 visual + 512 text tokens, a 64-token
              salient window drifting +4 tokens per step, focal layers 3 and 14, k = 205 (5% of 4096)
  kv_select   FastKV-shaped: 4 sequences x 32768 prompt tokens, 32 q / 8 KV heads, 8-query window at
              switch layer 15, 1% planted high-affinity tokens, keep 2040 + 8 window rows, then decode
  long_ctx    64 sequences x 131072 tokens, 32 q / 8 KV heads, 64 planted clusters of 16 tokens, k = 2048
  hpd_branch  512 branches over one 2048 + 256 token prefix, private suffixes of U[0, 1024] tokens,
              7-token causal drafts, 16 q / 8 KV heads; sparse variant keeps 256 prefix tokens
"""
from __future__ import annotations

import math

import numpy as np
import torch

from . import distinct_positions, normal_bf16, normal_bf16_at, normal_f32_at, stream_id, uint32_at

D = 128

# stream kinds
_K, _V, _Q, _THETA, _POS, _APPK, _APPV, _DRK, _DRV, _SUFK, _SUFV, _PREK, _PREV, _LEN = range(1, 15)


def _rows_of(seed, stream, full_shape, b, h, device):
    """K/V rows of (b, h) of a [B, Hkv, T, D] tensor generated with normal_bf16(seed, stream, full_shape)."""
    B, H, T, d = full_shape
    base = (b * H + h) * T * d
    ctr = torch.arange(base, base + T * d, dtype=torch.int64, device=device)
    return normal_bf16_at(seed, stream, ctr).view(T, d)


def _add_f32(x_bf16: torch.Tensor, add_f32: torch.Tensor) -> torch.Tensor:
    """bf16(fp32(x) + add): the one rounding step used for every planted structure."""
    return (x_bf16.to(torch.float32) + add_f32).to(torch.bfloat16)


# ----------------------------------------------------------------------------------------------
# tiny: one layer, 16 q / 8 KV heads, T = 1024, top-64
class Tiny:
    seed = 1
    B, Hq, Hkv, T, k, n_salient = 1, 16, 8, 1024, 64, 32

    def build(self):
        """All tensors on the host (the case is small).  The salient rule: for KV head h let
        u = normalize(q_{2h} + q_{2h+1}); for each of 32 hashed positions, the key's component along
        u, a = k.u, is replaced by 4|a| (k <- k + (4|a| - a) u), computed in float64, rounded to bf16."""
        B, Hq, Hkv, T = self.B, self.Hq, self.Hkv, self.T
        k = normal_bf16(self.seed, stream_id(_K), (B, Hkv, T, D))
        v = normal_bf16(self.seed, stream_id(_V), (B, Hkv, T, D))
        q = normal_bf16(self.seed, stream_id(_Q), (B, Hq, 1, D))
        kd = k.double().numpy()
        qd = q.double().numpy()
        G = Hq // Hkv
        salient = np.zeros((B, Hkv, self.n_salient), np.int64)
        for b in range(B):
            for h in range(Hkv):
                u = qd[b, h * G:(h + 1) * G, 0].sum(axis=0)
                u /= np.linalg.norm(u)
                pos = distinct_positions(self.seed, stream_id(_POS, b, h), T, self.n_salient).numpy()
                salient[b, h] = pos
                for t in pos:
                    a = float(kd[b, h, t] @ u)
                    kd[b, h, t] = kd[b, h, t] + (4.0 * abs(a) - a) * u
        k = torch.from_numpy(kd).to(torch.bfloat16)
        length = torch.full((B,), T, dtype=torch.int32)
        return dict(k=k, v=v, q=q, len=length, salient=torch.from_numpy(salient), kk=self.k)


# ----------------------------------------------------------------------------------------------
# ocr_decode: FastOCR-shaped decode
class OcrDecode:
    seed = 2
    B, Hq, Hkv = 8, 16, 8
    n_layers = 28
    focal_layers = (3, 14)
    n_vis, n_text = 4096, 512
    steps = 256
    k_keep = 205               # ceil(5% of 4096)
    n_freq = 32
    gamma = math.sqrt(2.1)
    freq_sigma = 1.0 / 16.0

    @property
    def tcap(self):
        return self.n_vis + self.n_text + self.steps

    def length_at(self, t):
        """Cache length while decoding step t (the step's own token is already appended)."""
        return self.n_vis + self.n_text + t + 1

    def centers(self, t):
        """Centre of each sequence's salient window at step t, in raster order of the visual tokens."""
        return [32 + 4 * t + 256 * b for b in range(self.B)]

    def _theta(self, layer):
        c = torch.arange(self.Hkv * self.n_freq, dtype=torch.int64)
        z = normal_f32_at(self.seed, stream_id(_THETA, layer), c).double().numpy()
        return (z * self.freq_sigma).reshape(self.Hkv, self.n_freq)

    def fourier_table(self, layer):
        """fp32 [Hkv, n_vis, 64]: gamma * (cos(theta_f j), sin(theta_f j)) for every visual position j.
        The dot product of two such codes is gamma^2 sum_f cos(theta_f (j - c)), an RBF-like bump of
        width ~1/sigma around j = c (random Fourier features)."""
        th = self._theta(layer)
        j = np.arange(self.n_vis, dtype=np.float64)
        ang = th[:, None, :] * j[None, :, None]
        tab = np.concatenate([np.cos(ang), np.sin(ang)], axis=-1) * self.gamma
        return torch.from_numpy(tab.astype(np.float32))

    def kv_shape(self):
        return (self.B, self.Hkv, self.tcap, D)

    def layer_kv(self, layer, device="cpu", table=None):
        """Full K, V of one layer on `device`."""
        shape = self.kv_shape()
        k = normal_bf16(self.seed, stream_id(_K, layer), shape, device=device)
        v = normal_bf16(self.seed, stream_id(_V, layer), shape, device=device)
        tab = (self.fourier_table(layer) if table is None else table).to(device)
        k[:, :, :self.n_vis, :2 * self.n_freq] = _add_f32(k[:, :, :self.n_vis, :2 * self.n_freq], tab[None])
        return k, v

    def layer_kv_rows(self, layer, b, h, table=None):
        """K, V rows of one (b, h) of one layer, on the host ([tcap, 128] each)."""
        shape = self.kv_shape()
        k = _rows_of(self.seed, stream_id(_K, layer), shape, b, h, "cpu").clone()
        v = _rows_of(self.seed, stream_id(_V, layer), shape, b, h, "cpu")
        tab = self.fourier_table(layer) if table is None else table
        k[:self.n_vis, :2 * self.n_freq] = _add_f32(k[:self.n_vis, :2 * self.n_freq], tab[h])
        return k, v

    def query(self, t, layer, device="cpu", table=None):
        """q [B, Hq, 1, 128] of one layer at step t (base normal + the code of the window centre)."""
        q = normal_bf16(self.seed, stream_id(_Q, layer, t), (self.B, self.Hq, 1, D), device=device)
        tab = self.fourier_table(layer) if table is None else table
        G = self.Hq // self.Hkv
        c = self.centers(t)
        add = torch.stack([torch.stack([tab[g // G, c[b]] for g in range(self.Hq)]) for b in range(self.B)])
        q[:, :, 0, :2 * self.n_freq] = _add_f32(q[:, :, 0, :2 * self.n_freq], add.to(device))
        return q


# ----------------------------------------------------------------------------------------------
# kv_select: FastKV-shaped prefill selection + compaction + decode
class KvSelect:
    seed = 3
    B, Hq, Hkv = 4, 32, 8
    T = 32768
    n_layers = 32
    switch_layer = 15
    window = 8
    keep = 2048
    decode_steps = 512
    planted_frac = 0.01
    alpha = 0.25

    @property
    def n_planted(self):
        return int(round(self.planted_frac * self.T))   # 328

    @property
    def k_select(self):
        return self.keep - self.window                  # 2040 chosen from [0, T - window)

    @property
    def compact_cap(self):
        return self.keep + self.decode_steps

    def window_queries(self, device="cpu"):
        """q of the last `window` prompt positions at the switch layer: [B, Hq, window, 128]."""
        return normal_bf16(self.seed, stream_id(_Q, self.switch_layer, 999999), (self.B, self.Hq, self.window, D),
                           device=device)

    def planted_positions(self, b, h):
        return distinct_positions(self.seed, stream_id(_POS, b, h), self.T - self.window, self.n_planted)

    # Per-layer retention (each layer selects its own tokens): every layer gets its own window queries
    # and its own planted high-affinity tokens; at the switch layer both equal the ones above.
    def window_queries_at(self, layer, device="cpu"):
        """q of the last `window` prompt positions at `layer`: [B, Hq, window, 128]."""
        return normal_bf16(self.seed, stream_id(_Q, layer, 999999), (self.B, self.Hq, self.window, D), device=device)

    def planted_positions_at(self, layer, b, h):
        if layer == self.switch_layer:
            return self.planted_positions(b, h)
        return distinct_positions(self.seed, stream_id(_POS, b, h, layer), self.T - self.window, self.n_planted)

    def layer_kv_salient(self, layer, device="cpu"):
        """Layer `layer` with its own planted tokens (equals layer_kv at the switch layer)."""
        shape = (self.B, self.Hkv, self.T, D)
        k = normal_bf16(self.seed, stream_id(_K, layer), shape, device=device)
        v = normal_bf16(self.seed, stream_id(_V, layer), shape, device=device)
        aff = self._affinity(self.window_queries_at(layer, device))
        for b in range(self.B):
            for h in range(self.Hkv):
                pos = self.planted_positions_at(layer, b, h).to(device)
                k[b, h, pos] = _add_f32(k[b, h, pos], aff[b, h][None])
        return k, v

    def layer_kv_salient_rows(self, layer, b, h):
        shape = (self.B, self.Hkv, self.T, D)
        k = _rows_of(self.seed, stream_id(_K, layer), shape, b, h, "cpu").clone()
        v = _rows_of(self.seed, stream_id(_V, layer), shape, b, h, "cpu")
        aff = self._affinity(self.window_queries_at(layer, "cpu"))
        pos = self.planted_positions_at(layer, b, h)
        k[pos] = _add_f32(k[pos], aff[b, h][None])
        return k, v

    def _affinity(self, qw):
        """fp32 [B, Hkv, 128]: alpha * (sum of the group's window query rows, added in a fixed order)."""
        G = self.Hq // self.Hkv
        w = torch.zeros((self.B, self.Hkv, D), dtype=torch.float32, device=qw.device)
        for gi in range(G):
            for i in range(self.window):
                w = w + qw[:, torch.arange(self.Hkv) * G + gi, i, :].to(torch.float32)
        return w * self.alpha

    def layer_kv(self, layer, device="cpu"):
        shape = (self.B, self.Hkv, self.T, D)
        k = normal_bf16(self.seed, stream_id(_K, layer), shape, device=device)
        v = normal_bf16(self.seed, stream_id(_V, layer), shape, device=device)
        if layer == self.switch_layer:
            aff = self._affinity(self.window_queries(device))
            for b in range(self.B):
                for h in range(self.Hkv):
                    pos = self.planted_positions(b, h).to(device)
                    k[b, h, pos] = _add_f32(k[b, h, pos], aff[b, h][None])
        return k, v

    def layer_kv_rows(self, layer, b, h):
        shape = (self.B, self.Hkv, self.T, D)
        k = _rows_of(self.seed, stream_id(_K, layer), shape, b, h, "cpu").clone()
        v = _rows_of(self.seed, stream_id(_V, layer), shape, b, h, "cpu")
        if layer == self.switch_layer:
            aff = self._affinity(self.window_queries("cpu"))
            pos = self.planted_positions(b, h)
            k[pos] = _add_f32(k[pos], aff[b, h][None])
        return k, v

    def appended_kv(self, layer, device="cpu"):
        """K, V rows appended during decode: [B, Hkv, decode_steps, 128] each."""
        shape = (self.B, self.Hkv, self.decode_steps, D)
        return (normal_bf16(self.seed, stream_id(_APPK, layer), shape, device=device),
                normal_bf16(self.seed, stream_id(_APPV, layer), shape, device=device))

    def decode_query(self, t, layer, device="cpu"):
        return normal_bf16(self.seed, stream_id(_Q, layer, t), (self.B, self.Hq, 1, D), device=device)


# ----------------------------------------------------------------------------------------------
# long_ctx: long-context focal pass + sparse decode
class LongCtx:
    seed = 4
    B, Hq, Hkv = 64, 32, 8
    T = 131072
    n_layers = 16
    k = 2048
    n_clusters, cluster_len = 64, 16
    alpha = 0.25

    def query(self, layer, device="cpu", B=None):
        B = self.B if B is None else B
        return normal_bf16(self.seed, stream_id(_Q, layer), (self.B, self.Hq, 1, D), device=device)[:B].contiguous()

    def cluster_starts(self, b, h):
        c = torch.arange(self.n_clusters, dtype=torch.int64)
        return uint32_at(self.seed, stream_id(_POS, b, h), c) % (self.T - self.cluster_len)

    def _affinity(self, q):
        G = self.Hq // self.Hkv
        w = torch.zeros((q.shape[0], self.Hkv, D), dtype=torch.float32, device=q.device)
        for gi in range(G):
            w = w + q[:, torch.arange(self.Hkv) * G + gi, 0, :].to(torch.float32)
        return w * self.alpha

    def planted_positions(self, b, h):
        s = self.cluster_starts(b, h)
        pos = (s[:, None] + torch.arange(self.cluster_len)[None, :]).reshape(-1)
        return torch.unique(pos)

    def layer_kv(self, layer, device="cpu", B=None):
        """K, V of one layer for the first B sequences (default: all 64)."""
        B = self.B if B is None else B
        shape = (self.B, self.Hkv, self.T, D)
        k = torch.empty((B, self.Hkv, self.T, D), dtype=torch.bfloat16, device=device)
        v = torch.empty_like(k)
        per_b = self.Hkv * self.T * D
        for b in range(B):
            normal_bf16(self.seed, stream_id(_K, layer), (self.Hkv, self.T, D), device=device, offset=b * per_b, out=k[b])
            normal_bf16(self.seed, stream_id(_V, layer), (self.Hkv, self.T, D), device=device, offset=b * per_b, out=v[b])
        aff = self._affinity(self.query(layer, device))
        for b in range(B):
            for h in range(self.Hkv):
                pos = self.planted_positions(b, h).to(device)
                k[b, h, pos] = _add_f32(k[b, h, pos], aff[b, h][None])
        return k, v

    def layer_kv_rows(self, layer, b, h):
        shape = (self.B, self.Hkv, self.T, D)
        k = _rows_of(self.seed, stream_id(_K, layer), shape, b, h, "cpu").clone()
        v = _rows_of(self.seed, stream_id(_V, layer), shape, b, h, "cpu")
        aff = self._affinity(self.query(layer, "cpu"))
        pos = self.planted_positions(b, h)
        k[pos] = _add_f32(k[pos], aff[b, h][None])
        return k, v


# ----------------------------------------------------------------------------------------------
# hpd_branch: shared-prefix draft verification
class HpdBranch:
    seed = 5
    Br, Hq, Hkv = 512, 16, 8
    n_vis, n_layout = 2048, 256
    max_suffix = 1024
    Mq = 7
    n_layers = 28
    kp = 256

    @property
    def P(self):
        return self.n_vis + self.n_layout

    def suffix_lengths(self, Br=None):
        Br = self.Br if Br is None else Br
        u = uint32_at(self.seed, stream_id(_LEN), torch.arange(Br, dtype=torch.int64))
        return (u % (self.max_suffix + 1)).to(torch.int32)

    def offsets(self, Br=None):
        L = self.suffix_lengths(Br).to(torch.int64)
        off = torch.zeros(L.numel() + 1, dtype=torch.int64)
        off[1:] = torch.cumsum(L, 0)
        return off.to(torch.int32)

    def suffix_rows(self, layer, b, device="cpu"):
        """Suffix K, V rows of branch b only: [Hkv, L_b, 128] each (same values as layer_inputs)."""
        off = self.offsets()
        o0, o1 = int(off[b]), int(off[b + 1])
        smax = self.Br * self.max_suffix
        ks, vs = [], []
        for h in range(self.Hkv):
            ks.append(normal_bf16(self.seed, stream_id(_SUFK, layer), (o1 - o0, D), device=device,
                                  offset=(h * smax + o0) * D))
            vs.append(normal_bf16(self.seed, stream_id(_SUFV, layer), (o1 - o0, D), device=device,
                                  offset=(h * smax + o0) * D))
        return torch.stack(ks), torch.stack(vs)

    def small_inputs(self, layer, device="cpu"):
        """Everything but the suffixes: prefix [Hkv, P, 128], draft [Br, Mq, Hkv, 128], q [Br, Hq, Mq, 128]."""
        return dict(
            pk=normal_bf16(self.seed, stream_id(_PREK, layer), (self.Hkv, self.P, D), device=device),
            pv=normal_bf16(self.seed, stream_id(_PREV, layer), (self.Hkv, self.P, D), device=device),
            dk=normal_bf16(self.seed, stream_id(_DRK, layer), (self.Br, self.Mq, self.Hkv, D), device=device),
            dv=normal_bf16(self.seed, stream_id(_DRV, layer), (self.Br, self.Mq, self.Hkv, D), device=device),
            q=normal_bf16(self.seed, stream_id(_Q, layer), (self.Br, self.Hq, self.Mq, D), device=device))

    def layer_inputs(self, layer, device="cpu", Br=None):
        """prefix K/V [Hkv, P, 128]; suffix K/V [Hkv, S, 128]; offsets [Br+1]; draft K/V [Br, Mq, Hkv, 128];
        q [Br, Hq, Mq, 128].  Br defaults to all 512 branches; a smaller Br takes the first branches."""
        Br = self.Br if Br is None else Br
        off = self.offsets(Br)
        S = int(off[-1])
        pk = normal_bf16(self.seed, stream_id(_PREK, layer), (self.Hkv, self.P, D), device=device)
        pv = normal_bf16(self.seed, stream_id(_PREV, layer), (self.Hkv, self.P, D), device=device)
        sk = torch.empty((self.Hkv, S, D), dtype=torch.bfloat16, device=device)
        sv = torch.empty_like(sk)
        smax = self.Br * self.max_suffix      # counters laid out as [Hkv, smax, D]: independent of Br
        for h in range(self.Hkv):
            normal_bf16(self.seed, stream_id(_SUFK, layer), (S, D), device=device, offset=h * smax * D, out=sk[h])
            normal_bf16(self.seed, stream_id(_SUFV, layer), (S, D), device=device, offset=h * smax * D, out=sv[h])
        dk = normal_bf16(self.seed, stream_id(_DRK, layer), (self.Br, self.Mq, self.Hkv, D), device=device)[:Br]
        dv = normal_bf16(self.seed, stream_id(_DRV, layer), (self.Br, self.Mq, self.Hkv, D), device=device)[:Br]
        q = normal_bf16(self.seed, stream_id(_Q, layer), (self.Br, self.Hq, self.Mq, D), device=device)[:Br]
        return dict(pk=pk, pv=pv, sk=sk, sv=sv, off=off.to(device), dk=dk.contiguous(), dv=dv.contiguous(),
                    q=q.contiguous())
