"""The C ABI library builds, loads and exports every entry point declared in include/fx.h; host-side
argument checks answer without touching a GPU."""
import ctypes
import os
import re
import shutil

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fx.h")


def declared_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^FX_API\s+[\w\s\*]+?\b(fx_\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from kv_cache_token_fx_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_five_calls():
    names = declared_functions()
    for n in ("fx_focal_attn_scores", "fx_topk_select", "fx_sparse_gqa_decode", "fx_kv_compact",
              "fx_shared_prefix_decode"):
        assert n in names
    assert len(names) >= 12


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_host_argument_checks_without_gpu(lib):
    lib.fx_last_error.restype = ctypes.c_char_p
    lib.fx_abi_version.restype = ctypes.c_int
    assert lib.fx_abi_version() == 3
    lib.fx_topk_select.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                   ctypes.c_void_p, ctypes.c_uint, ctypes.c_void_p]
    assert lib.fx_topk_select(None, 1, 4, 2, None, None, 0, None) == 1
    assert b"non-NULL" in lib.fx_last_error()
    fake = ctypes.c_void_p(256)
    assert lib.fx_topk_select(fake, 1, 4, 5, None, fake, 0, None) == 1       # k > n
    assert b"k (5) <= n (4)" in lib.fx_last_error()
    assert lib.fx_topk_select(fake, 1, 4, 2, None, fake, 0x80, None) == 1    # unknown launch flag
    assert b"unknown launch flags" in lib.fx_last_error()
    lib.fx_focal_attn_scores.restype = ctypes.c_int
    assert lib.fx_focal_attn_scores(None, None, 1, 1, -1, ctypes.c_float(1.0), 0, 0, None, None, None,
                                    ctypes.c_size_t(0), ctypes.c_uint(0), None) == 1
    # per-layer retention: argument checks before any device work
    from kv_cache_token_fx_gb300 import KVDesc, KVOutDesc
    kv = KVDesc(256, 512, 768, 2 * 600 * 128, 600 * 128, 128, 2, 2, 600, 128)
    dst = KVOutDesc(1024, 1280, 1536, 2 * 64 * 128, 64 * 128, 128, 2, 2, 64, 128)
    lib.fx_kv_retain_per_layer.restype = ctypes.c_int
    lib.fx_retain_workspace_bytes.restype = ctypes.c_size_t
    retain = lambda n_layers, cand_hi, keep: lib.fx_kv_retain_per_layer(
        ctypes.byref(kv), ctypes.c_int64(2 * 2 * 600 * 128), n_layers, ctypes.c_void_p(256), 4, 4, 596,
        ctypes.c_float(1.0), cand_hi, keep, 596, ctypes.c_void_p(256), ctypes.byref(dst), ctypes.c_int64(0), None,
        ctypes.c_size_t(0), ctypes.c_uint(0), None)
    assert retain(0, 596, 37) == 1 and b"n_layers" in lib.fx_last_error()
    assert retain(3, 601, 37) == 1 and b"cand_hi" in lib.fx_last_error()
    assert retain(3, 596, 597) == 1 and b"keep_k" in lib.fx_last_error()
    assert retain(3, 596, 37) == 3    # no workspace
    # the window queries and the softmax are checked before any device work too
    retain_q = lambda hq, q, q_pos0, scale: lib.fx_kv_retain_per_layer(
        ctypes.byref(kv), ctypes.c_int64(2 * 2 * 600 * 128), 3, q, hq, 4, q_pos0, ctypes.c_float(scale), 596, 37, 596,
        ctypes.c_void_p(256), ctypes.byref(dst), ctypes.c_int64(0), None, ctypes.c_size_t(0), ctypes.c_uint(0), None)
    assert retain_q(3, ctypes.c_void_p(256), 596, 1.0) != 0                       # 3 query heads over 2 KV heads
    assert retain_q(4, ctypes.c_void_p(264), 596, 1.0) == 1 and b"16-byte" in lib.fx_last_error()
    assert retain_q(4, ctypes.c_void_p(256), -2, 1.0) == 1 and b"q_pos0" in lib.fx_last_error()
    assert retain_q(4, ctypes.c_void_p(256), 596, float("nan")) == 1 and b"scale" in lib.fx_last_error()
    assert retain_q(4, ctypes.c_void_p(256), 596, 1.0) == 3                       # valid: only the workspace is missing
    # the workspace holds the scores of a batch of layers and the scoring scratch of all of them
    assert lib.fx_retain_workspace_bytes(2, 2, 4, 4, 600, 596) > 2 * 2 * 596 * 4
    lib.fx_focal_workspace_bytes.restype = ctypes.c_size_t
    assert lib.fx_retain_workspace_bytes(4, 8, 32, 8, 32768, 32760) >= \
        lib.fx_focal_workspace_bytes(4, 8, 32, 8, 32768) + 32 * 4 * 8 * 32760 * 4
    # decode-step append: argument checks before any device work
    lib.fx_kv_append.restype = ctypes.c_int
    append = lambda n_layers, knew, pos, flags=0: lib.fx_kv_append(
        ctypes.byref(dst), ctypes.c_int64(2 * 2 * 64 * 128), n_layers, knew, ctypes.c_void_p(2048), pos,
        ctypes.c_uint(flags), None)
    assert append(0, ctypes.c_void_p(256), ctypes.c_void_p(256)) == 1 and b"n_layers" in lib.fx_last_error()
    assert append(2, ctypes.c_void_p(256), None) == 1 and b"pos" in lib.fx_last_error()
    assert append(2, None, ctypes.c_void_p(256)) == 1 and b"k_new" in lib.fx_last_error()
    assert append(2, ctypes.c_void_p(264), ctypes.c_void_p(256)) == 1 and b"aligned" in lib.fx_last_error()
    assert append(2, ctypes.c_void_p(256), ctypes.c_void_p(256), 0x40) == 1
    # the focal-layer choice is host code: it runs here, and agrees with the oracle's rule
    import oracle
    lib.fx_choose_focal_layers.restype = ctypes.c_int
    g = np.random.default_rng(4)
    for n in (1, 3, 7, 28):
        ratio = g.integers(0, 4, size=n).astype(np.float32) / 4
        for C in range(1, n + 1, max(1, n // 5)):
            out = (ctypes.c_int32 * C)()
            assert lib.fx_choose_focal_layers((ctypes.c_float * n)(*ratio), n, C, out) == 0
            assert list(out) == oracle.choose_focal_layers(ratio.tolist(), C)
    assert lib.fx_choose_focal_layers((ctypes.c_float * 2)(0.1, 0.2), 2, 3, (ctypes.c_int32 * 3)()) == 1
    # the cross-step reuse schedule is host code too: every small configuration against the oracle's rule
    import itertools
    lib.fx_csfr_schedule.restype = ctypes.c_int
    names = {0: "focal", 1: "current", 2: "previous", 3: "dense"}
    for n in range(1, 7):
        for C in range(1, n + 1):
            for focal in itertools.combinations(range(n), C):
                for first in (0, 1):
                    kind, src = (ctypes.c_int32 * n)(), (ctypes.c_int32 * n)()
                    assert lib.fx_csfr_schedule(n, (ctypes.c_int32 * C)(*focal), C, first, kind, src) == 0
                    got = [(names[k], s_) for k, s_ in zip(kind, src)]
                    assert got == oracle.csfr_schedule(n, focal, bool(first)), (n, focal, first)
    bad = (ctypes.c_int32 * 2)(5, 3)
    assert lib.fx_csfr_schedule(8, bad, 2, 0, (ctypes.c_int32 * 8)(), (ctypes.c_int32 * 8)()) == 1
    assert b"ascending" in lib.fx_last_error()
    # shared-prefix workspace: a dense prefix of a full 128 x 128 tile or more (and at least 128 query
    # rows per KV head) also needs room for the tensor-core prefix partials (O, m, l per row)
    lib.fx_shared_prefix_workspace_bytes.restype = ctypes.c_size_t
    sp = lambda Br, Hkv, Hq, Mq, np_, ms: lib.fx_shared_prefix_workspace_bytes(Br, Hkv, Hq, Mq, np_, ms)
    assert sp(512, 8, 16, 7, 2304, 1024) >= 8 * 512 * 14 * 130 * 4          # tensor-core route
    assert sp(512, 8, 16, 7, 2304, 1024) >= sp(512, 8, 16, 7, 0, 1024)
    assert sp(4, 8, 16, 7, 2304, 1024) > 0                                     # 56 rows: no tensor cores
    assert sp(0, 8, 16, 7, 2304, 1024) == 0 and sp(4, 8, 4, 7, 2304, 1024) == 0   # Br < 1, Hq < Hkv
    lib.fx_sparse_workspace_bytes.restype = ctypes.c_size_t
    # decode shapes (at most 8 query heads per KV head) merge their splits inside a cluster: no
    # workspace; wider groups keep split partials in the workspace
    assert lib.fx_sparse_workspace_bytes(8, 8, 16, 205, 4096, 4864) == 0
    assert lib.fx_sparse_workspace_bytes(8, 1, 16, 205, 4096, 4864) > 0
    assert lib.fx_sparse_workspace_bytes(0, 8, 16, 205, 4096, 4864) == 0
    lib.fx_focal_workspace_bytes.restype = ctypes.c_size_t
    assert lib.fx_focal_workspace_bytes(8, 8, 16, 1, 4864) >= 8 * 8 * 2 * 4864 * 4


def test_binding_refuses_cpu_tensors():
    import torch
    import kv_cache_token_fx_gb300 as fx
    try:
        fx.load_library()
    except fx.FxError:
        pytest.skip("library not built")
    with pytest.raises(fx.FxError):
        fx.fx_topk_select(torch.zeros((2, 8)), 3)


def test_product_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "kv_cache_token_fx_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".h", ".cuh", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"\boracle\b", text.replace("oracle-free", "")) or f.endswith(".md"), \
                    f"{f} mentions the oracle"
