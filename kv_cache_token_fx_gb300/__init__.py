"""Python binding of libfx (include/fx.h): argument marshalling only.

Every function here checks tensor dtypes/devices, allocates outputs and workspaces with PyTorch, and
calls the C entry point of the same name; all arithmetic runs in the library's CUDA kernels.  There is
no fallback: if libfx.so has not been built, or a CUDA tensor is missing, the call raises.

Build the library with ``python -m kv_cache_token_fx_gb300.build`` (or ``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from . import build as _build

__all__ = [
    "FxError", "load_library", "library_path", "Workspace", "fx_focal_attn_scores", "fx_topk_select",
    "fx_focal_mass", "fx_choose_focal_layers", "fx_csfr_schedule", "FX_CSFR_FOCAL", "FX_CSFR_CURRENT",
    "FX_CSFR_PREVIOUS", "FX_CSFR_DENSE",
    "fx_sparse_gqa_decode", "fx_kv_compact", "fx_kv_append", "fx_kv_retain_per_layer", "fx_shared_prefix_decode",
    "fx_device_errors", "fx_focal_workspace_bytes", "fx_sparse_workspace_bytes", "fx_shared_prefix_workspace_bytes",
    "FX_DEVERR_LEN", "FX_DEVERR_INDEX", "FX_DEVERR_OFFSETS", "FX_DEVERR_CAPACITY", "FX_DEVERR_TIMEOUT",
    "FX_LAUNCH_PDL", "FX_LAUNCH_INPUTS_READY", "BranchPool",
]

FX_OK, FX_ERR_INVALID_ARG, FX_ERR_UNSUPPORTED, FX_ERR_WORKSPACE, FX_ERR_CUDA, FX_ERR_DEVICE = range(6)
FX_DEVERR_LEN, FX_DEVERR_INDEX, FX_DEVERR_OFFSETS, FX_DEVERR_CAPACITY, FX_DEVERR_TIMEOUT = 1, 2, 4, 8, 16
FX_LAUNCH_PDL, FX_LAUNCH_INPUTS_READY = 1, 2
FX_CSFR_FOCAL, FX_CSFR_CURRENT, FX_CSFR_PREVIOUS, FX_CSFR_DENSE = range(4)
_STATUS = {0: "FX_OK", 1: "FX_ERR_INVALID_ARG", 2: "FX_ERR_UNSUPPORTED", 3: "FX_ERR_WORKSPACE",
           4: "FX_ERR_CUDA", 5: "FX_ERR_DEVICE"}

c_vp, c_i64, c_i32, c_int, c_float, c_size = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int,
                                              ctypes.c_float, ctypes.c_size_t)


class FxError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS.get(status, status)}: {message}")
        self.status = status
        self.message = message


class KVDesc(ctypes.Structure):
    _fields_ = [("k", c_vp), ("v", c_vp), ("len", c_vp), ("stride_b", c_i64), ("stride_h", c_i64),
                ("stride_t", c_i64), ("B", c_i32), ("Hkv", c_i32), ("Tcap", c_i32), ("d", c_i32)]


KVOutDesc = type("KVOutDesc", (ctypes.Structure,), {"_fields_": KVDesc._fields_})


class PrefixDesc(ctypes.Structure):
    _fields_ = [("k", c_vp), ("v", c_vp), ("stride_h", c_i64), ("stride_t", c_i64), ("P", c_i32),
                ("Hkv", c_i32), ("d", c_i32), ("len", c_vp)]


class BranchDesc(ctypes.Structure):
    _fields_ = [("suf_k", c_vp), ("suf_v", c_vp), ("suf_stride_h", c_i64), ("suf_stride_t", c_i64),
                ("suf_off", c_vp), ("suf_rows", c_i32), ("max_suffix", c_i32), ("draft_k", c_vp),
                ("draft_v", c_vp), ("draft_stride_b", c_i64), ("draft_stride_i", c_i64),
                ("draft_stride_h", c_i64), ("Br", c_i32), ("Mq", c_i32), ("suf_len", c_vp)]


_lib = None
_lib_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB


def load_library():
    """Load libfx.so (must have been built).  Raises FxError if it is missing."""
    global _lib
    with _lib_lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise FxError(FX_ERR_CUDA, f"{path} is not built; run `python -m kv_cache_token_fx_gb300.build`")
        lib = ctypes.CDLL(path)
        lib.fx_last_error.restype = ctypes.c_char_p
        lib.fx_abi_version.restype = c_int
        lib.fx_device_errors.argtypes = [ctypes.POINTER(ctypes.c_uint), c_vp]
        lib.fx_test_stall_wait.argtypes = [ctypes.c_uint]
        lib.fx_test_stall_wait.restype = None
        lib.fx_workspace_init.argtypes = [c_vp, c_size, c_vp]
        lib.fx_focal_workspace_bytes.argtypes = [c_int] * 5
        lib.fx_focal_workspace_bytes.restype = c_size
        c_uint = ctypes.c_uint
        lib.fx_focal_attn_scores.argtypes = [ctypes.POINTER(KVDesc), c_vp, c_int, c_int, c_int, c_float, c_int,
                                             c_int, c_vp, c_vp, c_vp, c_size, c_uint, c_vp]
        lib.fx_topk_select.argtypes = [c_vp, c_int, c_int, c_int, c_vp, c_vp, c_uint, c_vp]
        lib.fx_focal_mass.argtypes = [c_vp, c_int, c_int, c_int, c_int, c_vp, c_uint, c_vp]
        lib.fx_choose_focal_layers.argtypes = [ctypes.POINTER(ctypes.c_float), c_int, c_int,
                                               ctypes.POINTER(ctypes.c_int32)]
        lib.fx_csfr_schedule.argtypes = [c_int, ctypes.POINTER(ctypes.c_int32), c_int, c_int,
                                         ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]
        lib.fx_sparse_workspace_bytes.argtypes = [c_int] * 6
        lib.fx_sparse_workspace_bytes.restype = c_size
        lib.fx_sparse_gqa_decode.argtypes = [ctypes.POINTER(KVDesc), c_vp, c_int, c_vp, c_int, c_int, c_float,
                                             c_vp, c_vp, c_size, c_uint, c_vp]
        lib.fx_kv_compact.argtypes = [ctypes.POINTER(KVDesc), c_i64, c_vp, c_i64, c_int, c_int,
                                      ctypes.POINTER(KVOutDesc), c_i64, c_int, c_uint, c_vp]
        lib.fx_kv_append.argtypes = [ctypes.POINTER(KVOutDesc), c_i64, c_int, c_vp, c_vp, c_vp, c_uint, c_vp]
        lib.fx_retain_workspace_bytes.argtypes = [c_int] * 6
        lib.fx_retain_workspace_bytes.restype = c_size
        lib.fx_kv_retain_per_layer.argtypes = [ctypes.POINTER(KVDesc), c_i64, c_int, c_vp, c_int, c_int, c_int,
                                               c_float, c_int, c_int, c_int, c_vp, ctypes.POINTER(KVOutDesc), c_i64,
                                               c_vp, c_size, ctypes.c_uint, c_vp]
        lib.fx_branch_pool_create.argtypes = [c_int, c_int, c_int]
        lib.fx_branch_pool_create.restype = c_vp
        lib.fx_branch_pool_destroy.argtypes = [c_vp]
        lib.fx_branch_pool_destroy.restype = None
        for name, args in (("extend_prefix", [c_vp, c_int]), ("fork", [c_vp]), ("append", [c_vp, c_int, c_int]),
                           ("release", [c_vp, c_int]), ("release_parent", [c_vp]), ("prefix_refs", [c_vp]),
                           ("prefix_len", [c_vp]), ("batch", [c_vp] + [ctypes.POINTER(ctypes.c_int32)] * 4)):
            f = getattr(lib, "fx_branch_pool_" + name)
            f.argtypes = args
            f.restype = c_int
        lib.fx_shared_prefix_workspace_bytes.argtypes = [c_int] * 6
        lib.fx_shared_prefix_workspace_bytes.restype = c_size
        lib.fx_shared_prefix_decode.argtypes = [ctypes.POINTER(PrefixDesc), ctypes.POINTER(BranchDesc), c_vp, c_int,
                                                c_vp, c_int, c_float, c_vp, c_vp, c_size, c_uint, c_vp]
        for name in ("fx_device_errors", "fx_workspace_init", "fx_focal_attn_scores", "fx_topk_select",
                     "fx_focal_mass", "fx_choose_focal_layers", "fx_csfr_schedule",
                     "fx_sparse_gqa_decode", "fx_kv_compact", "fx_kv_append", "fx_kv_retain_per_layer",
                     "fx_shared_prefix_decode"):
            getattr(lib, name).restype = c_int
        _lib = lib
        return lib


def _check(status: int):
    if status != FX_OK:
        msg = load_library().fx_last_error().decode(errors="replace")
        raise FxError(status, msg)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need_cuda(t, name, dtype):
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise FxError(FX_ERR_INVALID_ARG, f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise FxError(FX_ERR_INVALID_ARG, f"{name} must be {dtype}, got {t.dtype}")


def _kv_desc(k, v, length):
    _need_cuda(k, "k", torch.bfloat16)
    _need_cuda(v, "v", torch.bfloat16)
    _need_cuda(length, "len", torch.int32)
    if k.dim() != 4 or k.shape != v.shape or k.stride() != v.stride() or k.stride(3) != 1:
        raise FxError(FX_ERR_INVALID_ARG, "k and v must be [B, Hkv, Tcap, d] views with equal strides, unit last stride")
    B, Hkv, Tcap, d = k.shape
    return KVDesc(k.data_ptr(), v.data_ptr(), length.data_ptr(), k.stride(0), k.stride(1), k.stride(2), B, Hkv,
                  Tcap, d)


def _default_scale(d):
    return 1.0 / math.sqrt(d)


class Workspace:
    """A zero-initialised device scratch buffer reused across calls on one stream.

    ``ensure(nbytes)`` grows it (allocating a fresh zeroed buffer) when needed; a buffer that a CUDA
    graph has captured must not be grown afterwards, so size it before capture.
    """

    def __init__(self, device=None, nbytes: int = 0):
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        self.buf = None
        if nbytes:
            self.ensure(nbytes)

    def ensure(self, nbytes: int, stream=None):
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=self.device)
            _check(load_library().fx_workspace_init(_ptr(self.buf), self.buf.numel(), _stream(stream)))
        return self.buf


_default_ws = {}


def _workspace(ws, nbytes, device, stream):
    if ws is None:
        key = device.index if device.index is not None else torch.cuda.current_device()
        ws = _default_ws.get(key)
        if ws is None:
            ws = _default_ws[key] = Workspace(torch.device("cuda", key))
    buf = ws.ensure(nbytes, stream)
    return buf


def fx_focal_workspace_bytes(B, Hkv, Hq, Mq, Tcap) -> int:
    return int(load_library().fx_focal_workspace_bytes(B, Hkv, Hq, Mq, Tcap))


def fx_sparse_workspace_bytes(B, Hkv, Hq, k, tail_lo, Tcap) -> int:
    return int(load_library().fx_sparse_workspace_bytes(B, Hkv, Hq, k, tail_lo, Tcap))


def fx_shared_prefix_workspace_bytes(Br, Hkv, Hq, Mq, np_, max_suffix) -> int:
    return int(load_library().fx_shared_prefix_workspace_bytes(Br, Hkv, Hq, Mq, np_, max_suffix))


def fx_focal_attn_scores(k, v, length, q, *, q_pos0: int = -1, scale=None, cand=None, want_out=True,
                         want_scores=True, out=None, scores=None, ws=None, stream=None, flags: int = 0):
    """Focal layer: full attention + per-token importance.  Returns (out, scores) (None if not wanted).

    k, v [B, Hkv, Tcap, 128] bf16; length int32 [B]; q [B, Hq, Mq, 128] bf16 (contiguous).
    cand = (lo, hi) candidate range for the scores (default: the whole capacity).
    """
    lib = load_library()
    desc = _kv_desc(k, v, length)
    _need_cuda(q, "q", torch.bfloat16)
    if not q.is_contiguous() or q.dim() != 4:
        raise FxError(FX_ERR_INVALID_ARG, "q must be a contiguous [B, Hq, Mq, 128] tensor")
    B, Hkv, Tcap, d = k.shape
    _, Hq, Mq, _ = q.shape
    lo, hi = cand if cand is not None else (0, Tcap)
    if want_out and out is None:
        out = torch.empty((B, Hq, Mq, d), dtype=torch.float32, device=k.device)
    if want_scores and scores is None:
        scores = torch.empty((B, Hkv, hi - lo), dtype=torch.float32, device=k.device)
    if not want_out:
        out = None
    if not want_scores:
        scores = None
    nbytes = lib.fx_focal_workspace_bytes(B, Hkv, Hq, Mq, Tcap)
    buf = _workspace(ws, nbytes, k.device, stream)
    sc = _default_scale(d) if scale is None else float(scale)
    _check(lib.fx_focal_attn_scores(ctypes.byref(desc), _ptr(q), Hq, Mq, int(q_pos0), sc, int(lo), int(hi),
                                    _ptr(out), _ptr(scores), _ptr(buf), buf.numel(), int(flags), _stream(stream)))
    return out, scores


def fx_focal_mass(scores, R: int, *, mass=None, accumulate=False, stream=None, flags: int = 0):
    """Image-attention share per row: mass[r] (+)= sum_j scores[r, j] / R.  scores [..., n] fp32
    (contiguous, from fx_focal_attn_scores over the image tokens); returns mass [...] fp32."""
    lib = load_library()
    _need_cuda(scores, "scores", torch.float32)
    if not scores.is_contiguous():
        raise FxError(FX_ERR_INVALID_ARG, "scores must be contiguous")
    n = scores.shape[-1]
    rows = scores.numel() // n if n else 0
    if mass is None:
        if accumulate:
            raise FxError(FX_ERR_INVALID_ARG, "accumulate needs a mass tensor")
        mass = torch.empty(scores.shape[:-1], dtype=torch.float32, device=scores.device)
    _need_cuda(mass, "mass", torch.float32)
    if mass.numel() != rows or not mass.is_contiguous():
        raise FxError(FX_ERR_INVALID_ARG, "mass must be a contiguous tensor of one value per row")
    _check(lib.fx_focal_mass(_ptr(scores), rows, n, int(R), int(bool(accumulate)), _ptr(mass), int(flags),
                             _stream(stream)))
    return mass


def fx_choose_focal_layers(ratio, C: int):
    """The C layers with the largest image-attention ratio (ties: the lower layer), ascending."""
    lib = load_library()
    r = (ctypes.c_float * len(ratio))(*[float(x) for x in ratio])
    out = (ctypes.c_int32 * int(C))()
    _check(lib.fx_choose_focal_layers(r, len(ratio), int(C), out))
    return [int(x) for x in out]


def fx_topk_select(scores, k: int, *, prev=None, out=None, stream=None, flags: int = 0):
    """Top-k of each row of ``scores`` [..., n] (fp32, contiguous): int32 [..., k], ascending indices."""
    lib = load_library()
    _need_cuda(scores, "scores", torch.float32)
    if not scores.is_contiguous():
        raise FxError(FX_ERR_INVALID_ARG, "scores must be contiguous")
    n = scores.shape[-1]
    rows = scores.numel() // n if n else 0
    if out is None:
        out = torch.empty(scores.shape[:-1] + (k,), dtype=torch.int32, device=scores.device)
    if prev is not None:
        _need_cuda(prev, "prev", torch.int32)
        if prev.numel() != rows * k or not prev.is_contiguous():
            raise FxError(FX_ERR_INVALID_ARG, "prev must be a contiguous [rows, k] int32 tensor")
    _check(lib.fx_topk_select(_ptr(scores), rows, n, int(k), _ptr(prev), _ptr(out), int(flags), _stream(stream)))
    return out


def fx_csfr_schedule(n_layers: int, focal_layers, first_step: bool):
    """Per layer of one decode step: (kind, src) -- FX_CSFR_FOCAL (src = the layer), FX_CSFR_CURRENT /
    FX_CSFR_PREVIOUS (attend over this / the previous step's set of focal layer src) or FX_CSFR_DENSE
    (src = -1).  Host only."""
    lib = load_library()
    f = [int(x) for x in focal_layers]
    kind = (ctypes.c_int32 * n_layers)()
    src = (ctypes.c_int32 * n_layers)()
    _check(lib.fx_csfr_schedule(int(n_layers), (ctypes.c_int32 * len(f))(*f), len(f), 1 if first_step else 0,
                                kind, src))
    return list(kind), list(src)


def fx_sparse_gqa_decode(k, v, length, q, idx, tail_lo: int, *, scale=None, out=None, ws=None, stream=None,
                         flags: int = 0):
    """Decode attention of q [B, Hq, 1, 128] over idx [B, Hkv, kk] (or None) plus the tail [tail_lo, len)."""
    lib = load_library()
    desc = _kv_desc(k, v, length)
    _need_cuda(q, "q", torch.bfloat16)
    if not q.is_contiguous() or q.dim() != 4 or q.shape[2] != 1:
        raise FxError(FX_ERR_INVALID_ARG, "q must be a contiguous [B, Hq, 1, 128] tensor")
    B, Hkv, Tcap, d = k.shape
    Hq = q.shape[1]
    kk = 0
    if idx is not None:
        _need_cuda(idx, "idx", torch.int32)
        if not idx.is_contiguous() or idx.dim() != 3 or tuple(idx.shape[:2]) != (B, Hkv):
            raise FxError(FX_ERR_INVALID_ARG, "idx must be a contiguous [B, Hkv, k] int32 tensor")
        kk = idx.shape[2]
    if out is None:
        out = torch.empty((B, Hq, 1, d), dtype=torch.float32, device=k.device)
    nbytes = lib.fx_sparse_workspace_bytes(B, Hkv, Hq, kk, int(tail_lo), Tcap)
    buf = _workspace(ws, nbytes, k.device, stream)
    sc = _default_scale(d) if scale is None else float(scale)
    _check(lib.fx_sparse_gqa_decode(ctypes.byref(desc), _ptr(q), Hq, _ptr(idx) if kk else None, kk, int(tail_lo),
                                    sc, _ptr(out), _ptr(buf), buf.numel(), int(flags), _stream(stream)))
    return out


def fx_kv_compact(k, v, length, idx, tail_lo: int, dst_k, dst_v, dst_len, *, stream=None, flags: int = 0):
    """Compact the retained rows of one layer ([B, Hkv, T, 128]) or of L layers ([L, B, Hkv, T, 128]).

    idx: [B, Hkv, k] (one set for every layer) or, for L layers, [L, B, Hkv, k] (a set per layer)."""
    lib = load_library()
    if k.dim() == 5:
        n_layers = k.shape[0]
        if dst_k.dim() != 5 or dst_k.shape[0] != n_layers:
            raise FxError(FX_ERR_INVALID_ARG, "dst must have the same number of layers")
        s_layer, d_layer = k.stride(0), dst_k.stride(0)
        if v.stride(0) != s_layer or dst_v.stride(0) != d_layer:
            raise FxError(FX_ERR_INVALID_ARG, "k/v layer strides must match")
        src = _kv_desc(k[0], v[0], length)
        dst = _kv_desc(dst_k[0], dst_v[0], dst_len)
    else:
        n_layers, s_layer, d_layer = 1, 0, 0
        src = _kv_desc(k, v, length)
        dst = _kv_desc(dst_k, dst_v, dst_len)
    kk, i_layer = 0, 0
    if idx is not None:
        _need_cuda(idx, "idx", torch.int32)
        if not idx.is_contiguous():
            raise FxError(FX_ERR_INVALID_ARG, "idx must be contiguous [B, Hkv, k] or [L, B, Hkv, k]")
        kk = idx.shape[-1]
        if idx.dim() == 4:
            if k.dim() != 5 or idx.shape[0] != n_layers:
                raise FxError(FX_ERR_INVALID_ARG, "a per-layer idx [L, B, Hkv, k] needs L-layer caches")
            i_layer = idx.stride(0)
    dst_out = KVOutDesc(*[getattr(dst, f) for f, _ in KVDesc._fields_])
    _check(lib.fx_kv_compact(ctypes.byref(src), s_layer, _ptr(idx) if kk else None, i_layer, kk, int(tail_lo),
                             ctypes.byref(dst_out), d_layer, n_layers, int(flags), _stream(stream)))
    return dst_k, dst_v, dst_len


def fx_kv_append(k, v, k_new, v_new, pos, *, stream=None, flags: int = 0):
    """Write one new key/value row per (layer, sequence, KV head) into the caches: row pos[b] of
    k, v ([B, Hkv, T, 128], or [L, B, Hkv, T, 128] for L layers) takes k_new, v_new ([B, Hkv, 128] or
    [L, B, Hkv, 128], contiguous).  pos: int32 [B] on the device."""
    lib = load_library()
    if k.dim() == 5:
        n_layers, s_layer = k.shape[0], k.stride(0)
        if v.stride(0) != s_layer:
            raise FxError(FX_ERR_INVALID_ARG, "k/v layer strides must match")
        cache = _kv_desc(k[0], v[0], pos)
    else:
        n_layers, s_layer = 1, 0
        cache = _kv_desc(k, v, pos)
    for t, name in ((k_new, "k_new"), (v_new, "v_new")):
        _need_cuda(t, name, torch.bfloat16)
        if not t.is_contiguous() or t.numel() != n_layers * cache.B * cache.Hkv * cache.d:
            raise FxError(FX_ERR_INVALID_ARG, f"{name} must be a contiguous [L, B, Hkv, 128] tensor")
    out = KVOutDesc(*[getattr(cache, f) for f, _ in KVDesc._fields_])
    _check(lib.fx_kv_append(ctypes.byref(out), s_layer, n_layers, _ptr(k_new), _ptr(v_new), _ptr(pos), int(flags),
                            _stream(stream)))
    return k, v


def fx_kv_retain_per_layer(k, v, length, q, keep_k: int, cand_hi: int, tail_lo: int, dst_k, dst_v, dst_len, *,
                           q_pos0: int = -1, scale=None, idx_out=None, ws=None, stream=None, flags: int = 0):
    """FastKV retention with a selection per layer: window scores of every layer, its top keep_k, and
    the compaction of every layer with its own set plus the tail [tail_lo, len).

    k, v [L, B, Hkv, T, 128]; q [L, B, Hq, Mq, 128] (each layer's window queries); dst_k, dst_v
    [L, B, Hkv, cap, 128]; dst_len int32 [B].  Returns idx [L, B, Hkv, keep_k] (ascending rows)."""
    lib = load_library()
    if k.dim() != 5 or dst_k.dim() != 5 or q.dim() != 5 or not (k.shape[0] == dst_k.shape[0] == q.shape[0]):
        raise FxError(FX_ERR_INVALID_ARG, "k, v, dst and q need a leading layer dimension of the same size")
    L, B, Hkv, T, d = k.shape
    _need_cuda(q, "q", torch.bfloat16)
    if not q.is_contiguous():
        raise FxError(FX_ERR_INVALID_ARG, "q must be a contiguous [L, B, Hq, Mq, 128] tensor")
    s_layer, d_layer = k.stride(0), dst_k.stride(0)
    if v.stride(0) != s_layer or dst_v.stride(0) != d_layer:
        raise FxError(FX_ERR_INVALID_ARG, "k/v layer strides must match")
    src = _kv_desc(k[0], v[0], length)
    dst = _kv_desc(dst_k[0], dst_v[0], dst_len)
    dst_out = KVOutDesc(*[getattr(dst, f) for f, _ in KVDesc._fields_])
    _, _, Hq, Mq, _ = q.shape
    if idx_out is None:
        idx_out = torch.empty((L, B, Hkv, int(keep_k)), dtype=torch.int32, device=k.device)
    _need_cuda(idx_out, "idx_out", torch.int32)
    if idx_out.numel() != L * B * Hkv * int(keep_k) or not idx_out.is_contiguous():
        raise FxError(FX_ERR_INVALID_ARG, "idx_out must be a contiguous [L, B, Hkv, keep_k] int32 tensor")
    nbytes = lib.fx_retain_workspace_bytes(B, Hkv, Hq, Mq, T, int(cand_hi))
    buf = _workspace(ws, nbytes, k.device, stream)
    sc = _default_scale(d) if scale is None else float(scale)
    _check(lib.fx_kv_retain_per_layer(ctypes.byref(src), s_layer, L, _ptr(q), Hq, Mq, int(q_pos0), sc, int(cand_hi),
                                      int(keep_k), int(tail_lo), _ptr(idx_out), ctypes.byref(dst_out), d_layer,
                                      _ptr(buf), buf.numel(), int(flags), _stream(stream)))
    return idx_out


def fx_shared_prefix_decode(pk, pv, sk, sv, off, dk, dv, q, *, max_suffix: int, prefix_idx=None, scale=None,
                            prefix_len=None, suf_len=None, out=None, ws=None, stream=None, flags: int = 0):
    """Draft verification of Br branches over one shared prefix.

    pk, pv [Hkv, P, 128]; sk, sv [Hkv, S, 128]; dk, dv [Br, Mq, Hkv, 128]; q [Br, Hq, Mq, 128];
    prefix_idx [Br, Hkv, kp] or None.  Branch b owns suffix rows off[b]..off[b+1]-1 (off int32 [Br+1]),
    or off[b]..off[b]+suf_len[b]-1 when suf_len [Br] is given; it sees the first prefix_len[b] prefix
    rows (its fork position; all P when prefix_len is None).
    """
    lib = load_library()
    for t, n in ((pk, "pk"), (pv, "pv"), (sk, "sk"), (sv, "sv"), (dk, "dk"), (dv, "dv"), (q, "q")):
        _need_cuda(t, n, torch.bfloat16)
    _need_cuda(off, "off", torch.int32)
    if pk.stride() != pv.stride() or sk.stride() != sv.stride() or dk.stride() != dv.stride():
        raise FxError(FX_ERR_INVALID_ARG, "paired K/V tensors must share strides")
    if not q.is_contiguous():
        raise FxError(FX_ERR_INVALID_ARG, "q must be contiguous")
    Hkv, P, d = pk.shape
    Br, Hq, Mq, _ = q.shape
    for t, n in ((prefix_len, "prefix_len"), (suf_len, "suf_len")):
        if t is not None:
            _need_cuda(t, n, torch.int32)
            if t.numel() != Br or not t.is_contiguous():
                raise FxError(FX_ERR_INVALID_ARG, f"{n} must be a contiguous [Br] int32 tensor")
    if off.numel() != (Br if suf_len is not None else Br + 1):
        raise FxError(FX_ERR_INVALID_ARG, "off must hold Br + 1 offsets (or Br starts with suf_len)")
    pre = PrefixDesc(pk.data_ptr(), pv.data_ptr(), pk.stride(0), pk.stride(1), P, Hkv, d,
                     prefix_len.data_ptr() if prefix_len is not None else None)
    brd = BranchDesc(sk.data_ptr(), sv.data_ptr(), sk.stride(0), sk.stride(1), off.data_ptr(), sk.shape[1],
                     int(max_suffix), dk.data_ptr(), dv.data_ptr(), dk.stride(0), dk.stride(1), dk.stride(2), Br, Mq,
                     suf_len.data_ptr() if suf_len is not None else None)
    kp = 0
    if prefix_idx is not None:
        _need_cuda(prefix_idx, "prefix_idx", torch.int32)
        if not prefix_idx.is_contiguous():
            raise FxError(FX_ERR_INVALID_ARG, "prefix_idx must be contiguous [Br, Hkv, kp]")
        kp = prefix_idx.shape[-1]
    if out is None:
        out = torch.empty((Br, Hq, Mq, d), dtype=torch.float32, device=q.device)
    np_ = kp if prefix_idx is not None else P
    nbytes = lib.fx_shared_prefix_workspace_bytes(Br, Hkv, Hq, Mq, np_, int(max_suffix))
    buf = _workspace(ws, nbytes, q.device, stream)
    sc = _default_scale(d) if scale is None else float(scale)
    _check(lib.fx_shared_prefix_decode(ctypes.byref(pre), ctypes.byref(brd), _ptr(q), Hq, _ptr(prefix_idx), kp, sc,
                                       _ptr(out), _ptr(buf), buf.numel(), int(flags), _stream(stream)))
    return out


class BranchPool:
    """Host bookkeeping of content branches forked from one shared prefix (include/fx.h: branch pool).
    Thin wrapper: every method is one C call; errors raise FxError."""

    def __init__(self, prefix_cap: int, max_branches: int, slot_rows: int):
        lib = load_library()
        self._lib = lib
        self._h = lib.fx_branch_pool_create(int(prefix_cap), int(max_branches), int(slot_rows))
        if not self._h:
            _check(FX_ERR_INVALID_ARG)
        self.max_branches = int(max_branches)
        self.slot_rows = int(slot_rows)

    def _int(self, r):
        if r < 0:
            raise FxError(FX_ERR_INVALID_ARG, self._lib.fx_last_error().decode(errors="replace"))
        return int(r)

    def extend_prefix(self, n: int) -> int:
        return self._int(self._lib.fx_branch_pool_extend_prefix(self._h, int(n)))

    def fork(self) -> int:
        return self._int(self._lib.fx_branch_pool_fork(self._h))

    def append(self, branch: int, n: int) -> int:
        return self._int(self._lib.fx_branch_pool_append(self._h, int(branch), int(n)))

    def release(self, branch: int) -> int:
        return self._int(self._lib.fx_branch_pool_release(self._h, int(branch)))

    def release_parent(self) -> int:
        return self._int(self._lib.fx_branch_pool_release_parent(self._h))

    def prefix_refs(self) -> int:
        return self._int(self._lib.fx_branch_pool_prefix_refs(self._h))

    def prefix_len(self) -> int:
        return self._int(self._lib.fx_branch_pool_prefix_len(self._h))

    def batch(self):
        """(ids, suf_start, suf_len, prefix_len) of the live branches, as int32 CPU tensors."""
        m = self.max_branches
        arrs = [(ctypes.c_int32 * m)() for _ in range(4)]
        n = self._int(self._lib.fx_branch_pool_batch(self._h, *arrs))
        return tuple(torch.tensor(list(a)[:n], dtype=torch.int32) for a in arrs)

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h:
            self._lib.fx_branch_pool_destroy(h)


def fx_device_errors(stream=None) -> int:
    """Synchronise the stream and return (and clear) the FX_DEVERR_* bits of the current device."""
    bits = ctypes.c_uint(0)
    st = load_library().fx_device_errors(ctypes.byref(bits), _stream(stream))
    if st not in (FX_OK, FX_ERR_DEVICE):
        _check(st)
    return int(bits.value)
