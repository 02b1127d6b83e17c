"""Thin ctypes binding of libdsaidx.so (the C ABI in include/dsaidx.h).

Argument marshalling only: torch tensors are checked for device, dtype and
contiguity and passed as raw pointers with the current CUDA stream; every step
of the indexer path runs in the library's CUDA kernels.  There is no fallback:
if the library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsaidx.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "dsaidx.h")

FP8 = 0   # IDX_KEY_FP8_E4M3
BF16 = 1  # IDX_KEY_BF16
HEAD_DIM = 128
MAX_TOPK = 2048

STATUS = {0: "IDX_OK", 1: "IDX_ERR_INVALID_ARG", 2: "IDX_ERR_UNSUPPORTED", 3: "IDX_ERR_CUDA",
          4: "IDX_ERR_WORKSPACE_TOO_SMALL", 5: "IDX_ERR_DEVICE_CHECK", 6: "IDX_ERR_TIMEOUT"}


class IdxError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__("%s: %s (%d)" % (what, STATUS.get(code, "?"), code))
        self.code = code


_lib = None


def load(path: Optional[str] = None):
    """Load libdsaidx.so (built by sparse_attention_top_idx_gb300.build)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError("libdsaidx.so not built (%s); run sparse_attention_top_idx_gb300.build.build()" % p)
    L = ctypes.CDLL(p)
    P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    L.idx_block_bytes.argtypes = [I, I, I]
    L.idx_block_bytes.restype = SZ
    L.idx_cache_create.argtypes = [ctypes.POINTER(P), P, I64, I, I, I]
    L.idx_cache_create.restype = I
    L.idx_cache_destroy.argtypes = [P]
    L.idx_cache_destroy.restype = None
    L.idx_store_keys.argtypes = [P, P, P, I64, P, P]
    L.idx_store_keys.restype = I
    L.idx_store_keys_rotated.argtypes = [P, P, P, I64, P, P]
    L.idx_store_keys_rotated.restype = I
    L.idx_store_keys_ex.argtypes = [P, P, P, I64, ctypes.c_uint, P, P]
    L.idx_store_keys_ex.restype = I
    L.idx_gather_blocks.argtypes = [P, P, I, P, I, P, P, P]
    L.idx_gather_blocks.restype = I
    L.idx_workspace_bytes_decode.argtypes = [P, I, I, I, I]
    L.idx_workspace_bytes_decode.restype = SZ
    L.idx_workspace_init.argtypes = [P, SZ, P]
    L.idx_workspace_init.restype = I
    L.idx_score_topk_decode.argtypes = [P, P, P, P, I, P, I, I, I, I, P, P, P, SZ, P]
    L.idx_score_topk_decode.restype = I
    L.idx_score_topk_decode_slots.argtypes = [P, P, P, P, I, P, I, I, I, I, P, P, P, P, SZ, P]
    L.idx_score_topk_decode_slots.restype = I
    L.idx_score_topk_decode_static.argtypes = [P, P, P, P, I, P, I, I, I, I, P, P, P]
    L.idx_score_topk_decode_static.restype = I
    L.idx_workspace_bytes_prefill.argtypes = [P, I, I, I, I, I]
    L.idx_workspace_bytes_prefill.restype = SZ
    L.idx_score_topk_prefill.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, P, P, P, SZ, P]
    L.idx_score_topk_prefill.restype = I
    L.idx_score_topk_prefill_slots.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, P, P, P, P, SZ, P]
    L.idx_score_topk_prefill_slots.restype = I
    L.idx_read_device_status.argtypes = [P, P, ctypes.POINTER(ctypes.c_int32)]
    L.idx_read_device_status.restype = I
    L.idx_status_str.argtypes = [I]
    L.idx_status_str.restype = ctypes.c_char_p
    L.idx_test_set_wait_limit.argtypes = [ctypes.c_ulonglong]
    L.idx_test_set_wait_limit.restype = I
    L.idx_kernel_timing.argtypes = [ctypes.c_int]
    L.idx_kernel_timing.restype = ctypes.c_int
    L.idx_copy.argtypes = [P, P, SZ, P]
    L.idx_copy.restype = I
    L.idx_kernel_times.argtypes = [ctypes.c_void_p, ctypes.c_int]
    L.idx_kernel_times.restype = ctypes.c_int
    if path is None:
        _lib = L
    return L


def header_functions():
    """Names of the functions include/dsaidx.h declares."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(idx_[a-z_]+)\s*\(", src)))


def _check(code: int, what: str):
    if code != 0:
        raise IdxError(code, what)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t: torch.Tensor, dtype, name: str, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))


def block_bytes(key_dtype: int, block_size: int, head_dim: int = HEAD_DIM) -> int:
    return int(load().idx_block_bytes(key_dtype, block_size, head_dim))


def status_str(code: int) -> str:
    return load().idx_status_str(code).decode()


class IndexCache:
    """A caller-owned paged pool (uint8 CUDA tensor) bound to an idx_cache handle."""

    def __init__(self, pool: torch.Tensor, block_size: int, key_dtype: int):
        _need(pool, torch.uint8, "pool")
        bb = block_bytes(key_dtype, block_size)
        if bb == 0 or pool.numel() % bb:
            raise ValueError("pool size must be a multiple of the block bytes")
        self.pool = pool
        self.block_size = block_size
        self.key_dtype = key_dtype
        self.num_blocks = pool.numel() // bb
        h = ctypes.c_void_p()
        with torch.cuda.device(pool.device):
            _check(load().idx_cache_create(ctypes.byref(h), _ptr(pool), self.num_blocks, block_size,
                                           HEAD_DIM, key_dtype), "idx_cache_create")
        self.handle = h

    @staticmethod
    def allocate(num_blocks: int, block_size: int, key_dtype: int, device="cuda", fill: int = 0):
        pool = torch.full((num_blocks * block_bytes(key_dtype, block_size),), fill, dtype=torch.uint8,
                          device=device)
        return IndexCache(pool, block_size, key_dtype)

    def close(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            load().idx_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


STORE_ROTATE = 1
STORE_FP4_ROUNDTRIP = 2


def store_keys(cache: IndexCache, k_bf16: torch.Tensor, slot_mapping: torch.Tensor,
               status: Optional[torch.Tensor] = None, stream=None, rotate: bool = False, fp4: bool = False):
    """idx_store_keys: quantise (fp8) or copy (bf16) n keys into their slots;
    rotate=True: idx_store_keys_rotated (Walsh-Hadamard rotation first);
    fp4=True: idx_store_keys_ex with the fp4 round trip (after the rotation)."""
    n = k_bf16.shape[0]
    _need(k_bf16, torch.bfloat16, "k_bf16", (n, HEAD_DIM))
    _need(slot_mapping, torch.int64, "slot_mapping", (n,))
    if status is not None:
        _need(status, torch.int32, "status")
    L = load()
    if fp4:
        flags = STORE_FP4_ROUNDTRIP | (STORE_ROTATE if rotate else 0)
        _check(L.idx_store_keys_ex(cache.handle, _ptr(k_bf16), _ptr(slot_mapping), n, flags, _ptr(status),
                                   _stream(stream)), "idx_store_keys_ex")
        return
    fn = L.idx_store_keys_rotated if rotate else L.idx_store_keys
    name = "idx_store_keys_rotated" if rotate else "idx_store_keys"
    _check(fn(cache.handle, _ptr(k_bf16), _ptr(slot_mapping), n, _ptr(status), _stream(stream)), name)


def gather_blocks(cache: IndexCache, block_table: torch.Tensor, seq_lens: torch.Tensor, dst: torch.Tensor,
                  status: Optional[torch.Tensor] = None, stream=None):
    """idx_gather_blocks: copy every sequence's blocks, in logical order, into
    the dense grid dst ([batch * max_blocks_per_seq] blocks, uint8)."""
    _need(block_table, torch.int32, "block_table")
    _need(seq_lens, torch.int32, "seq_lens")
    _need(dst, torch.uint8, "dst")
    B, mbps = block_table.shape
    if dst.numel() < B * mbps * block_bytes(cache.key_dtype, cache.block_size):
        raise ValueError("dst must hold batch * max_blocks_per_seq blocks")
    if status is not None:
        _need(status, torch.int32, "status")
    _check(load().idx_gather_blocks(cache.handle, _ptr(block_table), mbps, _ptr(seq_lens), B, _ptr(dst),
                                    _ptr(status), _stream(stream)), "idx_gather_blocks")


def workspace_bytes_decode(cache: IndexCache, batch: int, max_seq_len: int, heads: int, topk: int) -> int:
    return int(load().idx_workspace_bytes_decode(cache.handle, batch, max_seq_len, heads, topk))


def score_topk_decode_static(cache: IndexCache, q: torch.Tensor, w: torch.Tensor, block_table: torch.Tensor,
                             seq_lens: torch.Tensor, max_seq_len: int, topk: int, out_idx: torch.Tensor,
                             out_score: Optional[torch.Tensor] = None, stream=None):
    """idx_score_topk_decode_static: decode without a workspace (the library's
    own fixed 32 MiB scratch per GPU; calls must not overlap on the GPU)."""
    B, H = q.shape[0], q.shape[1]
    _need(q, torch.bfloat16, "q", (B, H, HEAD_DIM))
    _need(w, torch.float32, "w", (B, H))
    _need(block_table, torch.int32, "block_table")
    _need(seq_lens, torch.int32, "seq_lens", (B,))
    _need(out_idx, torch.int32, "out_idx", (B, topk))
    if out_score is not None:
        _need(out_score, torch.float32, "out_score", (B, topk))
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be [batch, max_blocks_per_seq]")
    _check(load().idx_score_topk_decode_static(cache.handle, _ptr(q), _ptr(w), _ptr(block_table),
                                               block_table.shape[1], _ptr(seq_lens), B, max_seq_len, H, topk,
                                               _ptr(out_idx), _ptr(out_score), _stream(stream)),
           "idx_score_topk_decode_static")


def workspace_bytes_prefill(cache: IndexCache, batch: int, total_q: int, max_seq_len: int, heads: int,
                            topk: int) -> int:
    return int(load().idx_workspace_bytes_prefill(cache.handle, batch, total_q, max_seq_len, heads, topk))


def new_workspace(nbytes: int, device="cuda", stream=None) -> torch.Tensor:
    """Allocate (through PyTorch) and zero a workspace of nbytes."""
    ws = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    workspace_init(ws, stream)
    return ws


def workspace_init(ws: torch.Tensor, stream=None):
    _need(ws, torch.uint8, "workspace")
    _check(load().idx_workspace_init(_ptr(ws), ws.numel(), _stream(stream)), "idx_workspace_init")


def score_topk_decode(cache: IndexCache, q: torch.Tensor, w: torch.Tensor, block_table: torch.Tensor,
                      seq_lens: torch.Tensor, max_seq_len: int, topk: int, out_idx: torch.Tensor,
                      workspace: torch.Tensor, out_score: Optional[torch.Tensor] = None, stream=None,
                      out_slot: Optional[torch.Tensor] = None):
    """idx_score_topk_decode: one query per sequence, all its keys visible;
    with out_slot ([batch, topk] int64) idx_score_topk_decode_slots, which
    also writes each selected key's physical pool slot."""
    B, H = q.shape[0], q.shape[1]
    _need(q, torch.bfloat16, "q", (B, H, HEAD_DIM))
    _need(w, torch.float32, "w", (B, H))
    _need(block_table, torch.int32, "block_table")
    _need(seq_lens, torch.int32, "seq_lens", (B,))
    _need(out_idx, torch.int32, "out_idx", (B, topk))
    if out_score is not None:
        _need(out_score, torch.float32, "out_score", (B, topk))
    _need(workspace, torch.uint8, "workspace")
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be [batch, max_blocks_per_seq]")
    if out_slot is not None:
        _need(out_slot, torch.int64, "out_slot", (B, topk))
        _check(load().idx_score_topk_decode_slots(cache.handle, _ptr(q), _ptr(w), _ptr(block_table),
                                                  block_table.shape[1], _ptr(seq_lens), B, max_seq_len, H, topk,
                                                  _ptr(out_idx), _ptr(out_score), _ptr(out_slot), _ptr(workspace),
                                                  workspace.numel(), _stream(stream)), "idx_score_topk_decode_slots")
        return
    _check(load().idx_score_topk_decode(cache.handle, _ptr(q), _ptr(w), _ptr(block_table),
                                        block_table.shape[1], _ptr(seq_lens), B, max_seq_len, H, topk,
                                        _ptr(out_idx), _ptr(out_score), _ptr(workspace), workspace.numel(),
                                        _stream(stream)), "idx_score_topk_decode")


def score_topk_prefill(cache: IndexCache, q: torch.Tensor, w: torch.Tensor, cu_seqlens_q: torch.Tensor,
                       seq_lens: torch.Tensor, block_table: torch.Tensor, max_seq_len: int, topk: int,
                       out_idx: torch.Tensor, workspace: torch.Tensor,
                       out_score: Optional[torch.Tensor] = None, stream=None,
                       out_slot: Optional[torch.Tensor] = None):
    """idx_score_topk_prefill: causal query chunks (queries at each sequence's
    last positions); with out_slot ([total_q, topk] int64)
    idx_score_topk_prefill_slots."""
    T, H = q.shape[0], q.shape[1]
    B = seq_lens.shape[0]
    _need(q, torch.bfloat16, "q", (T, H, HEAD_DIM))
    _need(w, torch.float32, "w", (T, H))
    _need(cu_seqlens_q, torch.int32, "cu_seqlens_q", (B + 1,))
    _need(seq_lens, torch.int32, "seq_lens", (B,))
    _need(block_table, torch.int32, "block_table")
    _need(out_idx, torch.int32, "out_idx", (T, topk))
    if out_score is not None:
        _need(out_score, torch.float32, "out_score", (T, topk))
    _need(workspace, torch.uint8, "workspace")
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be [batch, max_blocks_per_seq]")
    if out_slot is not None:
        _need(out_slot, torch.int64, "out_slot", (T, topk))
        _check(load().idx_score_topk_prefill_slots(cache.handle, _ptr(q), _ptr(w), _ptr(cu_seqlens_q),
                                                   _ptr(seq_lens), _ptr(block_table), block_table.shape[1], B, T,
                                                   max_seq_len, H, topk, _ptr(out_idx), _ptr(out_score),
                                                   _ptr(out_slot), _ptr(workspace), workspace.numel(),
                                                   _stream(stream)), "idx_score_topk_prefill_slots")
        return
    _check(load().idx_score_topk_prefill(cache.handle, _ptr(q), _ptr(w), _ptr(cu_seqlens_q), _ptr(seq_lens),
                                         _ptr(block_table), block_table.shape[1], B, T, max_seq_len, H, topk,
                                         _ptr(out_idx), _ptr(out_score), _ptr(workspace), workspace.numel(),
                                         _stream(stream)), "idx_score_topk_prefill")


def read_device_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronise the stream and return the workspace's device status word."""
    v = ctypes.c_int32(0)
    _check(load().idx_read_device_status(_ptr(workspace), _stream(stream), ctypes.byref(v)),
           "idx_read_device_status")
    return int(v.value)


def test_set_wait_limit(limit_ns: int = 0):
    """idx_test_set_wait_limit: shorten the decode kernel's pipeline waits (and
    withhold one MMA signal) so that the timeout path runs; 0 restores."""
    _check(load().idx_test_set_wait_limit(int(limit_ns)), "idx_test_set_wait_limit")


def copy(dst: torch.Tensor, src: torch.Tensor, stream=None):
    """idx_copy: copy src into dst (same byte size, contiguous; device or
    pinned host tensors) with the library's copy kernel."""
    if not (dst.is_contiguous() and src.is_contiguous()):
        raise ValueError("copy wants contiguous tensors")
    nb = dst.numel() * dst.element_size()
    if nb != src.numel() * src.element_size():
        raise ValueError("copy wants equal byte sizes")
    _check(load().idx_copy(_ptr(dst), _ptr(src), nb, _stream(stream)), "idx_copy")


def kernel_timing(capacity: int) -> int:
    """idx_kernel_timing: record CUDA events around each kernel of the next
    score calls (up to `capacity` kernels); 0 stops."""
    r = load().idx_kernel_timing(int(capacity))
    if r < 0:
        raise RuntimeError("idx_kernel_timing failed")
    return r


def kernel_times(max_kernels: int = 4096):
    """idx_kernel_times: durations (ms) of the kernels recorded since the last
    read, in launch order; starts a new record."""
    buf = (ctypes.c_float * max_kernels)()
    n = load().idx_kernel_times(ctypes.cast(buf, ctypes.c_void_p), max_kernels)
    if n < 0:
        raise RuntimeError("idx_kernel_times failed")
    return [buf[i] for i in range(n)]
