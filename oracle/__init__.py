"""CPU fp64 oracle for the KV token selection + sparse GQA decode path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It does not import the CUDA library's package and the library
does not import it; the two share no code.  The arithmetic lives in ``fx_oracle.c`` (plain C loops in
double precision); this module only compiles it with gcc and marshals arguments through ctypes.

Inputs are CPU torch tensors: bf16 caches/queries (read through their 16-bit patterns, decoded
exactly to double by the C code) and int32 lengths/indices.  Outputs are numpy float64 arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fx_oracle.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

c_i64 = ctypes.c_int64
c_int = ctypes.c_int
c_dbl = ctypes.c_double
c_vp = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile fx_oracle.c into oracle/_lib/liboracle.so (gcc, fp contraction off)."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    return compile_source(_SRC, _LIB)


def compile_source(src_path: str, out_path: str) -> str:
    """Compile an oracle C source (this package's, or a mutated copy made by a test) into a .so."""
    tmp = out_path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, src_path,
           "-lpthread", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out_path)
    return out_path


def open_library(path: str):
    """Load a compiled oracle and declare its argument types."""
    lib = ctypes.CDLL(path)
    lib.oracle_set_threads.argtypes = [c_int]
    lib.oracle_set_threads.restype = c_int
    lib.oracle_get_threads.argtypes = []
    lib.oracle_get_threads.restype = c_int
    kv = [c_vp, c_vp, c_vp, c_i64, c_i64, c_i64]
    lib.oracle_focal.argtypes = kv + [c_int, c_int, c_int, c_int, c_vp, c_int, c_int, c_int,
                                      c_dbl, c_int, c_int, c_vp, c_vp]
    lib.oracle_focal.restype = None
    lib.oracle_topk.argtypes = [c_vp, c_int, c_int, c_int, c_vp]
    lib.oracle_topk.restype = None
    lib.oracle_sparse_decode.argtypes = kv + [c_int, c_int, c_int, c_vp, c_int, c_vp, c_int,
                                              c_int, c_dbl, c_vp]
    lib.oracle_sparse_decode.restype = None
    lib.oracle_kv_compact.argtypes = kv + [c_int, c_int, c_int, c_vp, c_int, c_int, c_vp, c_vp,
                                           c_i64, c_i64, c_i64, c_vp]
    lib.oracle_kv_compact.restype = None
    lib.oracle_shared_prefix.argtypes = [c_vp, c_vp, c_i64, c_i64, c_int, c_vp, c_vp, c_i64,
                                         c_i64, c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, c_vp,
                                         c_int, c_int, c_int, c_int, c_int, c_vp, c_int, c_vp, c_vp,
                                         c_dbl, c_vp]
    lib.oracle_shared_prefix.restype = None
    return lib


def _load(lib=None):
    global _lib
    if lib is not None:
        return lib
    with _lock:
        if _lib is None:
            build()
            _lib = open_library(_LIB)
    return _lib


def set_threads(n: int = 0) -> int:
    """Worker threads for the oracle (0: every online core).  Returns the count in use."""
    return _load().oracle_set_threads(int(n))


def get_threads() -> int:
    return _load().oracle_get_threads()


def _bits(t: torch.Tensor) -> torch.Tensor:
    if t.device.type != "cpu" or t.dtype != torch.bfloat16:
        raise TypeError("oracle expects CPU bfloat16 tensors")
    return t.view(torch.int16)


def _i32(t) -> torch.Tensor:
    t = torch.as_tensor(t, dtype=torch.int32)
    if t.device.type != "cpu":
        raise TypeError("oracle expects CPU tensors")
    return t.contiguous()


def _kv_strides(k: torch.Tensor):
    if k.dim() != 4 or k.stride(3) != 1:
        raise ValueError("KV cache must be [B, Hkv, Tcap, d] with unit stride over d")
    return k.stride(0), k.stride(1), k.stride(2)


def default_scale(d: int) -> float:
    return 1.0 / float(np.sqrt(d))


def focal(k, v, length, q, *, scale=None, q_pos0: int = -1, cand=None, want_out=True, want_scores=True, lib=None):
    """Focal-layer attention + importance.

    k, v   : bf16 [B, Hkv, Tcap, d] (same strides);  length: int32 [B];  q: bf16 [B, Hq, Mq, d]
    cand   : (lo, hi) candidate token range for the importance scores (default: 0 .. Tcap)
    returns (out [B, Hq, Mq, d] float64 or None, scores [B, Hkv, hi - lo] float64 or None)
    """
    lib = _load(lib)
    B, Hkv, Tcap, d = k.shape
    _, Hq, Mq, _ = q.shape
    if v.stride() != k.stride():
        raise ValueError("k and v must share strides")
    sb, sh, st = _kv_strides(k)
    kb, vb, qb = _bits(k), _bits(v), _bits(q.contiguous())
    ln = _i32(length)
    lo, hi = cand if cand is not None else (0, Tcap)
    scale = default_scale(d) if scale is None else float(scale)
    out = np.zeros((B, Hq, Mq, d), np.float64) if want_out else None
    sc = np.zeros((B, Hkv, hi - lo), np.float64) if want_scores else None
    lib.oracle_focal(kb.data_ptr(), vb.data_ptr(), ln.data_ptr(), sb, sh, st, B, Hkv, Tcap, d,
                     qb.data_ptr(), Hq, Mq, int(q_pos0), scale, int(lo), int(hi),
                     out.ctypes.data if out is not None else None,
                     sc.ctypes.data if sc is not None else None)
    return out, sc


def focal_mass(scores, R: int) -> np.ndarray:
    """FastOCR, Focal-Guided Pruning (Focal Layer Selection): the share of attention the R query rows of
    one (b, KV head) group put on the image tokens.  scores [..., n] are the group's softmax rows summed
    over R (focal() with the image tokens as candidates), so the share is their sum over the tokens
    divided by R.  Returns float64 [...]."""
    s = np.asarray(scores, dtype=np.float64)
    return s.sum(axis=-1) / float(R)


def choose_focal_layers(ratio, C: int) -> list:
    """FastOCR, Focal-Guided Pruning: the C layers with the highest image-attention ratio (ties go to
    the lower layer index), listed in ascending layer order."""
    r = [float(x) for x in ratio]
    order = sorted(range(len(r)), key=lambda l: (-r[l], l))
    return sorted(order[:C])


def csfr_schedule(n_layers: int, focal_layers, first_step: bool) -> list:
    """FastOCR, Focal-Guided Pruning and Cross-Step Fixation Reuse: where each layer of one decode step
    takes its attention set from.  A focal layer makes its own ("focal", l).  A layer below a focal layer
    attends to this step's set of the nearest focal layer above it ("current", f).  A layer above the
    first focal layer reuses the set the deepest focal layer chose at the previous step ("previous",
    f_last); at the first step there is none and it attends to the whole cache ("dense", -1)."""
    focal = sorted(int(f) for f in focal_layers)
    out = []
    for l in range(n_layers):
        if l in focal:
            out.append(("focal", l))
        elif l < focal[0]:
            out.append(("dense", -1) if first_step else ("previous", focal[-1]))
        else:
            out.append(("current", max(f for f in focal if f < l)))
    return out


def topk(scores, k: int, *, lib=None) -> np.ndarray:
    """scores [..., n] (any float type, compared in double) -> int32 [..., k]: the k best by
    (score descending, index ascending), written in ascending index order."""
    s = np.ascontiguousarray(np.asarray(scores, dtype=np.float64))
    n = s.shape[-1]
    rows = int(np.prod(s.shape[:-1])) if s.ndim > 1 else 1
    out = np.zeros(s.shape[:-1] + (k,), np.int32)
    _load(lib).oracle_topk(s.ctypes.data, rows, n, int(k), out.ctypes.data)
    return out


def sparse_decode(k, v, length, q, idx, tail_lo: int, *, scale=None, lib=None):
    """Decode attention of q [B, Hq, 1, d] over rows idx[b, h, :] plus the tail [tail_lo, len[b]).
    idx may be None (k = 0).  Returns float64 [B, Hq, 1, d]."""
    lib = _load(lib)
    B, Hkv, Tcap, d = k.shape
    _, Hq, Mq, _ = q.shape
    if Mq != 1:
        raise ValueError("sparse decode takes one query position per sequence")
    sb, sh, st = _kv_strides(k)
    kb, vb, qb = _bits(k), _bits(v), _bits(q.contiguous())
    ln = _i32(length)
    if idx is None:
        kk, ip = 0, None
    else:
        it = _i32(idx)
        kk, ip = it.shape[-1], it
    scale = default_scale(d) if scale is None else float(scale)
    out = np.zeros((B, Hq, 1, d), np.float64)
    lib.oracle_sparse_decode(kb.data_ptr(), vb.data_ptr(), ln.data_ptr(), sb, sh, st, B, Hkv, d,
                             qb.data_ptr(), Hq, ip.data_ptr() if ip is not None else None, kk,
                             int(tail_lo), scale, out.ctypes.data)
    return out


def kv_compact(k, v, length, idx, tail_lo: int, cap: int, *, lib=None):
    """Gather rows idx[b, h, :] then the tail [tail_lo, len[b]) into a new contiguous cache of
    capacity ``cap``.  Returns (k', v', len') as CPU tensors (unwritten rows are zero)."""
    lib = _load(lib)
    B, Hkv, Tcap, d = k.shape
    sb, sh, st = _kv_strides(k)
    kb, vb = _bits(k), _bits(v)
    ln = _i32(length)
    it = _i32(idx)
    kk = it.shape[-1]
    dk = torch.zeros((B, Hkv, cap, d), dtype=torch.bfloat16)
    dv = torch.zeros_like(dk)
    dl = torch.zeros(B, dtype=torch.int32)
    lib.oracle_kv_compact(kb.data_ptr(), vb.data_ptr(), ln.data_ptr(), sb, sh, st, B, Hkv, d,
                          it.data_ptr(), kk, int(tail_lo), dk.view(torch.int16).data_ptr(),
                          dv.view(torch.int16).data_ptr(), dk.stride(0), dk.stride(1), dk.stride(2),
                          dl.data_ptr())
    return dk, dv, dl


def kv_append(k, v, k_new, v_new, pos):
    """Decode-step append (FastKV 3.2, decoding over the compacted cache; FastOCR, decoding): every
    (layer, sequence, KV head) cache gains the new token's row at position pos[b].  k, v [..., B, Hkv,
    T, d]; k_new, v_new [..., B, Hkv, d]; a position outside [0, T) writes nothing.  Returns new CPU
    tensors (the inputs are not modified)."""
    k2, v2 = k.clone().cpu(), v.clone().cpu()
    kn, vn = k_new.cpu(), v_new.cpu()
    T = k2.shape[-2]
    for b, t in enumerate(pos.tolist()):
        if 0 <= t < T:
            k2[..., b, :, t, :] = kn[..., b, :, :]
            v2[..., b, :, t, :] = vn[..., b, :, :]
    return k2, v2


def shared_prefix(pk, pv, sk, sv, off, dk, dv, q, prefix_idx=None, *, pre_len=None, suf_len=None, scale=None,
                  lib=None):
    """Shared-prefix draft verification.

    pk, pv : bf16 [Hkv, P, d]            one prefix shared by every branch
    sk, sv : bf16 [Hkv, S, d]            private suffixes; branch b owns rows off[b] .. off[b]+L_b-1
    off    : int32 [Br + 1] (L_b = off[b+1] - off[b]), or [Br] starts when suf_len gives the L_b
    pre_len: int32 [Br] or None          rows of the prefix branch b sees (its fork position); None: all P
    suf_len: int32 [Br] or None
    dk, dv : bf16 [Br, Mq, Hkv, d]       draft rows; draft position i sees draft rows 0 .. i
    q      : bf16 [Br, Hq, Mq, d]
    prefix_idx : int32 [Br, Hkv, kp] or None (dense prefix)
    returns float64 [Br, Hq, Mq, d]
    """
    lib = _load(lib)
    Hkv, P, d = pk.shape
    Br, Hq, Mq, _ = q.shape
    for t in (pk, pv, sk, sv, dk, dv):
        if t.stride(-1) != 1:
            raise ValueError("rows must have unit stride over d")
    if pk.stride() != pv.stride() or sk.stride() != sv.stride() or dk.stride() != dv.stride():
        raise ValueError("paired K and V tensors must share strides")
    o = _i32(off)
    pi = _i32(prefix_idx) if prefix_idx is not None else None
    kp = pi.shape[-1] if pi is not None else 0
    scale = default_scale(d) if scale is None else float(scale)
    out = np.zeros((Br, Hq, Mq, d), np.float64)
    qb = _bits(q.contiguous())
    pl = _i32(pre_len) if pre_len is not None else None
    sl = _i32(suf_len) if suf_len is not None else None
    lib.oracle_shared_prefix(_bits(pk).data_ptr(), _bits(pv).data_ptr(), pk.stride(0), pk.stride(1), P,
                             _bits(sk).data_ptr(), _bits(sv).data_ptr(), sk.stride(0), sk.stride(1),
                             o.data_ptr(), _bits(dk).data_ptr(), _bits(dv).data_ptr(), dk.stride(0),
                             dk.stride(1), dk.stride(2), qb.data_ptr(), Br, Hkv, Hq, Mq, d,
                             pi.data_ptr() if pi is not None else None, kp,
                             pl.data_ptr() if pl is not None else None, sl.data_ptr() if sl is not None else None,
                             scale, out.ctypes.data)
    return out


__all__ = ["build", "set_threads", "get_threads", "focal", "topk", "sparse_decode", "kv_compact",
           "shared_prefix", "default_scale"]
