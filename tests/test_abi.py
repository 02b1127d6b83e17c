"""The C ABI library loads on any host and exports every function that
include/dsaidx.h declares; host-side argument checks answer before any CUDA
call (no GPU needed for these)."""
import ctypes

import pytest

from sparse_attention_top_idx_gb300 import build, dsaidx


@pytest.fixture(scope="module")
def lib():
    build.build()
    return dsaidx.load()


def test_exports_every_declared_function(lib):
    names = dsaidx.header_functions()
    assert len(names) == 21, names
    for n in names:
        assert hasattr(lib, n), n


def test_block_bytes(lib):
    assert lib.idx_block_bytes(0, 64, 128) == 8448
    assert lib.idx_block_bytes(0, 32, 128) == 4224
    assert lib.idx_block_bytes(1, 64, 128) == 16384
    assert lib.idx_block_bytes(1, 32, 128) == 8192
    assert lib.idx_block_bytes(0, 16, 128) == 0
    assert lib.idx_block_bytes(0, 64, 64) == 0
    assert lib.idx_block_bytes(2, 64, 128) == 0


def test_host_argument_checks(lib):
    h = ctypes.c_void_p()
    # null pool, bad block size, bad dtype, misaligned pool -> invalid argument
    assert lib.idx_cache_create(ctypes.byref(h), None, 4, 64, 128, 0) == 1
    assert lib.idx_cache_create(ctypes.byref(h), ctypes.c_void_p(4096), 4, 48, 128, 0) == 1
    assert lib.idx_cache_create(ctypes.byref(h), ctypes.c_void_p(4096), 4, 64, 128, 5) == 1
    assert lib.idx_cache_create(ctypes.byref(h), ctypes.c_void_p(4100), 4, 64, 128, 0) == 1
    assert lib.idx_cache_create(ctypes.byref(h), ctypes.c_void_p(4096), 0, 64, 128, 0) == 1
    # head_dim other than 128 is a valid request the library does not build
    assert lib.idx_cache_create(ctypes.byref(h), ctypes.c_void_p(4096), 4, 64, 96, 0) == 2
    # calls on a null handle
    assert lib.idx_store_keys(None, None, None, 1, None, None) == 1
    assert lib.idx_store_keys_rotated(None, None, None, 1, None, None) == 1
    assert lib.idx_store_keys_ex(None, None, None, 1, 2, None, None) == 1
    assert lib.idx_gather_blocks(None, None, 1, None, 1, None, None, None) == 1
    assert lib.idx_score_topk_decode(None, None, None, None, 1, None, 1, 1, 64, 8, None, None,
                                     None, 0, None) == 1
    assert lib.idx_score_topk_prefill(None, None, None, None, None, None, 1, 1, 1, 1, 64, 8, None,
                                      None, None, 0, None) == 1
    assert lib.idx_workspace_bytes_decode(None, 1, 1, 64, 8) == 0
    assert lib.idx_workspace_init(None, 1024, None) == 1
    v = ctypes.c_int32()
    assert lib.idx_read_device_status(None, None, ctypes.byref(v)) == 1
    assert lib.idx_test_set_wait_limit(0) == 0     # restores the normal limit
    assert lib.idx_kernel_timing(0) == 0            # timing off: no events
    assert lib.idx_kernel_times(None, 0) == 0
    assert lib.idx_copy(None, None, 16, None) == 1   # null pointers
    assert lib.idx_copy(ctypes.c_void_p(16), ctypes.c_void_p(32), 8, None) == 1   # size not a multiple of 16
    assert dsaidx.status_str(0) == "ok"
    assert dsaidx.status_str(4) == "workspace too small"
