"""The allocation-free focal call against the ordinary one.

fx_focal_attn_scores_noalloc exists for callers that cannot allocate device memory -- code running
during CUDA graph capture, real-time loops that allow no allocator calls after start-up, hosts that
only have the C interface.  It keeps its scratch in a fixed array inside the library instead of a
caller workspace.  This test calls it through the C ABI, twice in a row with different inputs, and
checks each result against fx_focal_attn_scores with a caller workspace and against the fp64 oracle,
within the tolerances used by every parity test here.  The file name makes pytest collect it last.
"""
import ctypes

import pytest
import torch

import oracle
import synth
from tests import parity_util as pu

pytestmark = pytest.mark.gpu

D = 128


def _inputs(seed, B, Hkv, G, T, device):
    k = synth.normal_bf16(seed, synth.stream_id(555, 1), (B, Hkv, T, D), device=device)
    v = synth.normal_bf16(seed, synth.stream_id(555, 2), (B, Hkv, T, D), device=device)
    q = synth.normal_bf16(seed, synth.stream_id(555, 3), (B, Hkv * G, 1, D), device=device)
    return k, v, q


def test_noalloc_focal_matches_workspace_call_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kv_cache_token_fx_gb300 as fx

    lib = fx.load_library()
    lib.fx_focal_attn_scores_noalloc.argtypes = [ctypes.POINTER(fx.KVDesc), ctypes.c_void_p, ctypes.c_int,
                                                 ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_int,
                                                 ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint,
                                                 ctypes.c_void_p]
    lib.fx_focal_attn_scores_noalloc.restype = ctypes.c_int
    lib.fx_noalloc_scratch_bytes.restype = ctypes.c_size_t
    assert lib.fx_noalloc_scratch_bytes() == 16 << 20

    dev = torch.device("cuda", 0)
    B, Hkv, G, T = 4, 8, 2, 2100
    length = torch.tensor([2100, 1500, 64, 999], dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    for call, seed in enumerate((11, 12)):
        k, v, q = _inputs(seed, B, Hkv, G, T, dev)
        ref_out, ref_sc = fx.fx_focal_attn_scores(k, v, length, q, cand=(0, T), ws=fx.Workspace(dev))
        out = torch.full((B, Hkv * G, 1, D), float("nan"), dtype=torch.float32, device=dev)
        sc = torch.full((B, Hkv, T), float("nan"), dtype=torch.float32, device=dev)
        desc = fx.KVDesc(k.data_ptr(), v.data_ptr(), length.data_ptr(), k.stride(0), k.stride(1), k.stride(2),
                         B, Hkv, T, D)
        st = lib.fx_focal_attn_scores_noalloc(ctypes.byref(desc), ctypes.c_void_p(q.data_ptr()), Hkv * G, 1, -1,
                                              ctypes.c_float(D ** -0.5), 0, T, ctypes.c_void_p(out.data_ptr()),
                                              ctypes.c_void_p(sc.data_ptr()), 0,
                                              ctypes.c_void_p(stream.cuda_stream))
        assert st == 0, lib.fx_last_error()
        torch.cuda.synchronize()
        assert fx.fx_device_errors() == 0
        vmax = float(v.float().abs().max())
        pu.assert_out_close(out, ref_out, vmax, what=f"call {call} out")
        pu.assert_scores_close(sc, ref_sc, what=f"call {call} scores")
        # and against the oracle on the same inputs
        orc_out, orc_sc = oracle.focal(k.cpu(), v.cpu(), length.cpu(), q.cpu(), cand=(0, T))
        pu.assert_out_close(out, orc_out, vmax, what=f"call {call} out vs oracle")
        pu.assert_scores_close(sc, orc_sc, what=f"call {call} scores vs oracle")

    # a call needing more scratch than the fixed array is refused before anything is launched
    # (the descriptor claims 64 x 8 x 32768 rows; the call is refused before anything reads them)
    small = torch.zeros((1, 1, 8, D), dtype=torch.bfloat16, device=dev)
    big_len = torch.full((64,), 32768, dtype=torch.int32, device=dev)
    qb = torch.zeros((64, 16, 1, D), dtype=torch.bfloat16, device=dev)
    desc = fx.KVDesc(small.data_ptr(), small.data_ptr(), big_len.data_ptr(), 8 * 32768 * D, 32768 * D, D,
                     64, 8, 32768, D)
    st = lib.fx_focal_attn_scores_noalloc(ctypes.byref(desc), ctypes.c_void_p(qb.data_ptr()), 16, 1, -1,
                                          ctypes.c_float(1.0), 0, 32768, None, None, 0,
                                          ctypes.c_void_p(stream.cuda_stream))
    assert st == fx.FX_ERR_UNSUPPORTED
    assert b"16 MiB" in lib.fx_last_error()
