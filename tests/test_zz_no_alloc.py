"""The decode call that needs no workspace (idx_score_topk_decode_static).

It exists for callers that cannot allocate device memory, for example a
plug-in running inside another framework's process (where device memory
belongs to that framework's allocator) or code on a path where cudaMalloc /
cudaFree are not allowed because they may synchronise the device.  Its
scratch is a fixed area of the library's own device memory, shared by every
call, so this test calls it twice in a row (the second call starts from what
the first left behind) and compares both results with the regular
workspace-based decode call on the same inputs.

The file name sorts last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from sparse_attention_top_idx_gb300 import dsaidx
from sparse_attention_top_idx_gb300 import workloads as wl
from tests.parity import TOL, build_cache, decode_inputs, run_decode

pytestmark = pytest.mark.gpu


def _static_call(cache, ins, W, oi, osc):
    L = dsaidx.load()
    return L.idx_score_topk_decode_static(
        cache.handle, ctypes.c_void_p(ins["q"].data_ptr()), ctypes.c_void_p(ins["w"].data_ptr()),
        ctypes.c_void_p(ins["block_table"].data_ptr()), ins["block_table"].shape[1],
        ctypes.c_void_p(ins["seq_lens"].data_ptr()), W.batch, W.max_seq_len, W.H, W.topk,
        ctypes.c_void_p(oi.data_ptr()), ctypes.c_void_p(osc.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("mode", [dsaidx.FP8, dsaidx.BF16])
def test_static_scratch_decode_matches_workspace_decode(mode):
    W = wl.make_workload("noalloc", [4500, 10000, 700, 129, 3000, 1], [1] * 6, topk=512, seed=61 + mode)
    cache = build_cache(W, mode)
    ref = run_decode(W, mode, cache=cache)            # regular entry point, own workspace
    ins = decode_inputs(W)
    for call in range(2):
        oi = torch.full((W.batch, W.topk), -7, dtype=torch.int32, device="cuda")
        osc = torch.full((W.batch, W.topk), float("nan"), dtype=torch.float32, device="cuda")
        assert _static_call(cache, ins, W, oi, osc) == 0
        torch.cuda.synchronize()
        gi, gs = oi.cpu().numpy(), osc.cpu().numpy()
        assert np.array_equal(gi, ref["idx"]), "call %d: indices differ" % call
        valid = gi >= 0
        assert np.array_equal(np.isneginf(gs), ~valid)
        r, g = ref["score"][valid].astype(np.float64), gs[valid].astype(np.float64)
        assert np.all(np.abs(g - r) <= TOL * np.abs(r) + 1e-6 * np.abs(r).max()), "call %d: scores" % call


def test_static_scratch_rejects_oversized_shape():
    W = wl.make_workload("noalloc_big", [1000], [1], topk=2048, seed=7)
    cache = build_cache(W, dsaidx.FP8)
    ins = decode_inputs(W)
    oi = torch.empty((1, 2048), dtype=torch.int32, device="cuda")
    osc = torch.empty((1, 2048), dtype=torch.float32, device="cuda")
    # a bound of 128M keys with top-2048 needs per sequence a sorted top-k run
    # for each of its 2048 segments of 65536 keys (32 MiB) besides the slow-path
    # scratch: more than the 32 MiB area, so the call is refused before
    # anything is launched
    need = dsaidx.workspace_bytes_decode(cache, 1, 1 << 27, 64, 2048)
    assert need > 32 << 20
    big = dsaidx.load().idx_score_topk_decode_static(
        cache.handle, ctypes.c_void_p(ins["q"].data_ptr()), ctypes.c_void_p(ins["w"].data_ptr()),
        ctypes.c_void_p(ins["block_table"].data_ptr()), ins["block_table"].shape[1],
        ctypes.c_void_p(ins["seq_lens"].data_ptr()), 1, 1 << 27, 64, 2048,
        ctypes.c_void_p(oi.data_ptr()), ctypes.c_void_p(osc.data_ptr()), None)
    assert big == 4     # IDX_ERR_WORKSPACE_TOO_SMALL
