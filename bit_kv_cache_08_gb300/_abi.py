"""ctypes binding of libkvarn.so (include/kvarn.h): argument marshalling only.

Every function takes torch CUDA tensors, checks dtypes and shapes, passes raw
pointers and the current CUDA stream to the C ABI, and raises KVarNError on a
non-zero status. There is no fallback: if the library is missing the first
call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkvarn.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "kvarn.h")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_WORKSPACE = 0, -1, -2, -3, -4
DEVERR_BLOCK_ID, DEVERR_POSITION, DEVERR_NONFINITE, DEVERR_WAIT_TIMEOUT = 0x1, 0x2, 0x4, 0x8
BF16, FP32 = 0, 1
KIND_K, KIND_V = 0, 1
FLAG_NO_ROTATION, FLAG_NO_TOKEN_PASS, FLAG_NO_CHANNEL_PASS = 0x1, 0x2, 0x4
FLAG_TEST_WAIT_TIMEOUT = 0x100   # test only: the decode kernel's first copy waits give up at once


class KVarNError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: status {status} ({status_string(status)})")
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("group_size", ctypes.c_int32), ("bits", ctypes.c_int32),
                ("varn_iters", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("sm_scale", ctypes.c_float),
                ("sign_bits", ctypes.c_uint32 * 4), ("flags", ctypes.c_uint32)]


def make_config(n_q_heads: int, n_kv_heads: int, block_size: int, varn_iters: int,
                sign_bits: Sequence[int], sm_scale: float = 0.0, head_dim: int = 128,
                group_size: int = 32, bits: int = 2, flags: int = 0) -> Config:
    c = Config()
    c.flags = flags
    c.head_dim, c.block_size, c.group_size, c.bits = head_dim, block_size, group_size, bits
    c.varn_iters, c.n_q_heads, c.n_kv_heads, c.sm_scale = varn_iters, n_q_heads, n_kv_heads, sm_scale
    for i in range(4):
        c.sign_bits[i] = int(sign_bits[i]) & 0xFFFFFFFF
    return c


_lib = None
_vp = ctypes.c_void_p
_i32, _i64, _sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
_cfgp = ctypes.POINTER(Config)

_SIGS = {
    "kvarn_version": (ctypes.c_char_p, []),
    "kvarn_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "kvarn_head_block_bytes": (_sz, [_cfgp]),
    "kvarn_block_bytes": (_sz, [_cfgp]),
    "kvarn_staging_bytes": (_sz, [_cfgp, _i32]),
    "kvarn_workspace_bytes": (_sz, [_cfgp, _i32, _i32]),
    "kvarn_prefill_workspace_bytes": (_sz, [_cfgp, _i32, _i32, _i32]),
    "kvarn_quantize_block": (ctypes.c_int, [_cfgp, _i32, _vp, _i32, _i64, _i64, _i64, _vp, _vp, _vp, _vp]),
    "kvarn_append": (ctypes.c_int, [_cfgp, _vp, _i64, _vp, _vp, _i32, _vp, _vp, _vp, _i32, _vp, _vp]),
    "kvarn_decode_attn": (ctypes.c_int, [_cfgp, _vp, _i32, _vp, _i64, _vp, _vp, _i32, _vp, _i32, _vp, _vp,
                                         _sz, _vp]),
    "kvarn_prefill_attn": (ctypes.c_int, [_cfgp, _vp, _i32, _vp, _i64, _vp, _vp, _i32, _vp, _i32, _i32, _vp,
                                          _vp, _sz, _vp]),
    "kvarn_dequantize": (ctypes.c_int, [_cfgp, _i32, _vp, _vp, _i64, _i32, _vp, _vp]),
    "kvarn_decode_attn_bf16": (ctypes.c_int, [_cfgp, _vp, _i32, _vp, _i64, _vp, _i32, _vp, _i32, _vp, _vp,
                                              _sz, _vp]),
    "kvarn_decode_attn_noalloc": (ctypes.c_int, [_cfgp, _vp, _i32, _vp, _i64, _vp, _vp, _i32, _vp, _i32, _vp,
                                                 _vp, _vp]),
    "kvarn_error_decomposition": (ctypes.c_int, [_cfgp, _i32, _vp, _i32, _i64, _i64, _i64, _vp, _vp, _vp, _vp]),
    "kvarn_read_error": (ctypes.c_int, [_vp, ctypes.POINTER(ctypes.c_uint32), _vp]),
    "kvarn_clear_error": (ctypes.c_int, [_vp, _vp]),
}


def lib():
    """Load libkvarn.so (built by bit_kv_cache_08_gb300.build.build())."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with bit_kv_cache_08_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def header_symbols() -> list:
    """Names of the functions include/kvarn.h declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(kvarn_[a-z0-9_]+)\s*\(", text)))


def status_string(status: int) -> str:
    return lib().kvarn_status_string(status).decode()


def version() -> str:
    return lib().kvarn_version().decode()


def _check(status: int, what: str):
    if status != OK:
        raise KVarNError(status, what)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _need_cuda(t: torch.Tensor, name: str, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# ------------------------------------------------------------------ sizes

def head_block_bytes(cfg: Config) -> int:
    return int(lib().kvarn_head_block_bytes(ctypes.byref(cfg)))


def block_bytes(cfg: Config) -> int:
    return int(lib().kvarn_block_bytes(ctypes.byref(cfg)))


def staging_bytes(cfg: Config, max_seqs: int) -> int:
    return int(lib().kvarn_staging_bytes(ctypes.byref(cfg), max_seqs))


def workspace_bytes(cfg: Config, batch: int, max_blocks_per_seq: int) -> int:
    return int(lib().kvarn_workspace_bytes(ctypes.byref(cfg), batch, max_blocks_per_seq))


# ------------------------------------------------------------------ buffers

def prefill_workspace_bytes(cfg: Config, batch: int, chunk: int, max_blocks_per_seq: int) -> int:
    return int(lib().kvarn_prefill_workspace_bytes(ctypes.byref(cfg), batch, chunk, max_blocks_per_seq))


def alloc_prefill_workspace(cfg: Config, batch: int, chunk: int, max_blocks_per_seq: int,
                            device="cuda") -> torch.Tensor:
    n = prefill_workspace_bytes(cfg, batch, chunk, max_blocks_per_seq)
    if n == 0:
        raise ValueError("kvarn_prefill_workspace_bytes: invalid config or sizes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def alloc_workspace(cfg: Config, batch: int, max_blocks_per_seq: int, device="cuda") -> torch.Tensor:
    n = workspace_bytes(cfg, batch, max_blocks_per_seq)
    if n == 0:
        raise KVarNError(ERR_CUDA, "kvarn_workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def alloc_pool(cfg: Config, n_blocks: int, device="cuda") -> torch.Tensor:
    return torch.zeros(n_blocks, block_bytes(cfg), dtype=torch.uint8, device=device)


def alloc_staging(cfg: Config, max_seqs: int, device="cuda") -> torch.Tensor:
    return torch.zeros(max_seqs, cfg.n_kv_heads, 2, cfg.block_size, 128, dtype=torch.bfloat16,
                       device=device)


# ------------------------------------------------------------------ entry points

def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return FP32
    raise ValueError(f"unsupported dtype {t.dtype}")


def _blocks_in(src: torch.Tensor, cfg: Config, n_head_blocks: Optional[int], block_stride: Optional[int],
               token_stride: int):
    """(n, block stride) for a source of head-blocks read from src's first
    element at the given strides (elements); n defaults to every whole block a
    contiguous src holds. Raises if block n-1 would read past src's storage."""
    B = cfg.block_size
    explicit = block_stride is not None or token_stride != 128
    if not explicit and not src.is_contiguous():
        raise ValueError("src must be contiguous unless its strides are given")
    bstride = B * 128 if block_stride is None else block_stride
    if n_head_blocks is None:
        if explicit:
            raise ValueError("n_head_blocks is required with explicit strides")
        n = src.numel() // (B * 128)
    else:
        n = n_head_blocks
    room = src.untyped_storage().nbytes() // src.element_size() - src.storage_offset()
    if n > 0 and (n - 1) * bstride + (B - 1) * token_stride + 128 > room:
        raise ValueError("src holds fewer elements than n_head_blocks blocks at these strides")
    return n, bstride


def quantize_block(cfg: Config, kind: int, src: torch.Tensor, dst_base: torch.Tensor,
                   workspace: torch.Tensor, dst_offsets: Optional[torch.Tensor] = None,
                   n_head_blocks: Optional[int] = None, block_stride: Optional[int] = None,
                   token_stride: int = 128):
    """src: contiguous bf16|fp32 values, head-block i at element i * block_stride
    (default B * 128) with token rows token_stride apart; n_head_blocks defaults
    to the whole blocks src holds. dst_base: uint8 buffer."""
    _need_cuda(dst_base, "dst_base", torch.uint8)
    if not src.is_cuda:
        raise ValueError("src must be a CUDA tensor")
    n, bstride = _blocks_in(src, cfg, n_head_blocks, block_stride, token_stride)
    if dst_offsets is not None:
        _need_cuda(dst_offsets, "dst_offsets", torch.int64)
    _check(lib().kvarn_quantize_block(ctypes.byref(cfg), kind, _ptr(src), _dtype_code(src), n, bstride,
                                      token_stride, _ptr(dst_base), _ptr(dst_offsets), _ptr(workspace),
                                      _stream()), "kvarn_quantize_block")


def append(cfg: Config, pool: torch.Tensor, staging: torch.Tensor, block_table: torch.Tensor,
           pos: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, workspace: torch.Tensor):
    _need_cuda(pool, "pool", torch.uint8)
    _need_cuda(staging, "staging", torch.bfloat16)
    _need_cuda(block_table, "block_table", torch.int32)
    _need_cuda(pos, "pos", torch.int32)
    _need_cuda(k_new, "k_new", torch.bfloat16)
    _need_cuda(v_new, "v_new", torch.bfloat16)
    batch = pos.shape[0]
    _check(lib().kvarn_append(ctypes.byref(cfg), _ptr(pool), pool.shape[0], _ptr(staging), _ptr(block_table),
                              block_table.shape[1], _ptr(pos), _ptr(k_new), _ptr(v_new), batch,
                              _ptr(workspace), _stream()), "kvarn_append")


def decode_attn(cfg: Config, q: torch.Tensor, pool: torch.Tensor, staging: torch.Tensor,
                block_table: torch.Tensor, seq_lens: torch.Tensor, out: torch.Tensor,
                workspace: torch.Tensor):
    _need_cuda(q, "q")
    _need_cuda(pool, "pool", torch.uint8)
    _need_cuda(staging, "staging", torch.bfloat16)
    _need_cuda(block_table, "block_table", torch.int32)
    _need_cuda(seq_lens, "seq_lens", torch.int32)
    _need_cuda(out, "out", torch.float32)
    _need_cuda(workspace, "workspace", torch.uint8)
    _check(lib().kvarn_decode_attn(ctypes.byref(cfg), _ptr(q), _dtype_code(q), _ptr(pool), pool.shape[0],
                                   _ptr(staging), _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
                                   q.shape[0], _ptr(out), _ptr(workspace), workspace.numel(), _stream()),
           "kvarn_decode_attn")


def prefill_attn(cfg: Config, q: torch.Tensor, pool: torch.Tensor, staging: torch.Tensor,
                 block_table: torch.Tensor, seq_lens: torch.Tensor, out: torch.Tensor, workspace: torch.Tensor):
    """q: [batch][chunk][n_q][128] (bf16|fp32) queries of each sequence's last
    chunk tokens; out: fp32 [batch][chunk][n_q][128]."""
    _need_cuda(q, "q")
    _need_cuda(pool, "pool", torch.uint8)
    _need_cuda(staging, "staging", torch.bfloat16)
    _need_cuda(block_table, "block_table", torch.int32)
    _need_cuda(seq_lens, "seq_lens", torch.int32)
    _need_cuda(out, "out", torch.float32)
    _need_cuda(workspace, "workspace", torch.uint8)
    if q.dim() != 4 or out.shape != q.shape:
        raise ValueError("q and out must be [batch][chunk][n_q][128]")
    _check(lib().kvarn_prefill_attn(ctypes.byref(cfg), _ptr(q), _dtype_code(q), _ptr(pool), pool.shape[0],
                                    _ptr(staging), _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
                                    q.shape[0], q.shape[1], _ptr(out), _ptr(workspace), workspace.numel(),
                                    _stream()),
           "kvarn_prefill_attn")


def decode_attn_bf16(cfg: Config, q: torch.Tensor, kv_pool: torch.Tensor, block_table: torch.Tensor,
                     seq_lens: torch.Tensor, out: torch.Tensor, workspace: torch.Tensor):
    """kv_pool: bf16 [n_blocks][n_kv][2][B][128]."""
    _need_cuda(q, "q")
    _need_cuda(kv_pool, "kv_pool", torch.bfloat16)
    _need_cuda(block_table, "block_table", torch.int32)
    _need_cuda(seq_lens, "seq_lens", torch.int32)
    _need_cuda(out, "out", torch.float32)
    _need_cuda(workspace, "workspace", torch.uint8)
    _check(lib().kvarn_decode_attn_bf16(ctypes.byref(cfg), _ptr(q), _dtype_code(q), _ptr(kv_pool),
                                        kv_pool.shape[0], _ptr(block_table), block_table.shape[1],
                                        _ptr(seq_lens), q.shape[0], _ptr(out), _ptr(workspace),
                                        workspace.numel(), _stream()), "kvarn_decode_attn_bf16")


def decode_attn_noalloc(cfg: Config, q: torch.Tensor, pool: torch.Tensor, staging: torch.Tensor,
                        block_table: torch.Tensor, seq_lens: torch.Tensor, out: torch.Tensor,
                        error_word: Optional[torch.Tensor] = None):
    """kvarn_decode_attn with the library's built-in scratch (no workspace):
    for callers that cannot allocate device memory."""
    _need_cuda(q, "q")
    _need_cuda(pool, "pool", torch.uint8)
    _need_cuda(staging, "staging", torch.bfloat16)
    _need_cuda(block_table, "block_table", torch.int32)
    _need_cuda(seq_lens, "seq_lens", torch.int32)
    _need_cuda(out, "out", torch.float32)
    if error_word is not None:
        _need_cuda(error_word, "error_word", torch.int32)
    _check(lib().kvarn_decode_attn_noalloc(ctypes.byref(cfg), _ptr(q), _dtype_code(q), _ptr(pool),
                                           pool.shape[0], _ptr(staging), _ptr(block_table),
                                           block_table.shape[1], _ptr(seq_lens), q.shape[0], _ptr(out),
                                           _ptr(error_word), _stream()), "kvarn_decode_attn_noalloc")


def dequantize(cfg: Config, kind: int, src_base: torch.Tensor, out: torch.Tensor, rotated: bool,
               src_offsets: Optional[torch.Tensor] = None, n_head_blocks: Optional[int] = None):
    _need_cuda(src_base, "src_base", torch.uint8)
    _need_cuda(out, "out", torch.float32)
    n = out.shape[0] if n_head_blocks is None else n_head_blocks
    if src_offsets is not None:
        _need_cuda(src_offsets, "src_offsets", torch.int64)
    _check(lib().kvarn_dequantize(ctypes.byref(cfg), kind, _ptr(src_base), _ptr(src_offsets), n,
                                  1 if rotated else 0, _ptr(out), _stream()), "kvarn_dequantize")


def error_decomposition(cfg: Config, kind: int, src: torch.Tensor, packed_base: torch.Tensor, out: torch.Tensor,
                        packed_offsets: Optional[torch.Tensor] = None, n_head_blocks: Optional[int] = None,
                        block_stride: Optional[int] = None, token_stride: int = 128):
    """src: the n head-blocks' values before quantisation, block i at element
    i * block_stride (default B * 128), token rows token_stride apart; out:
    fp32 [n][B][4] = (|x|, |x^|, |E_M|, |E_D|) per token. n defaults to
    out.shape[0]."""
    _need_cuda(packed_base, "packed_base", torch.uint8)
    _need_cuda(out, "out", torch.float32)
    if not src.is_cuda:
        raise ValueError("src must be a CUDA tensor")
    n, bstride = _blocks_in(src, cfg, out.shape[0] if n_head_blocks is None else n_head_blocks, block_stride,
                            token_stride)
    if out.numel() < n * cfg.block_size * 4:
        raise ValueError("out holds fewer than n_head_blocks x B x 4 values")
    if packed_offsets is not None:
        _need_cuda(packed_offsets, "packed_offsets", torch.int64)
    _check(lib().kvarn_error_decomposition(ctypes.byref(cfg), kind, _ptr(src), _dtype_code(src), n, bstride,
                                           token_stride, _ptr(packed_base), _ptr(packed_offsets), _ptr(out),
                                           _stream()), "kvarn_error_decomposition")


def read_error(workspace: torch.Tensor) -> int:
    code = ctypes.c_uint32(0)
    _check(lib().kvarn_read_error(_ptr(workspace), ctypes.byref(code), _stream()), "kvarn_read_error")
    return code.value


def clear_error(workspace: torch.Tensor):
    _check(lib().kvarn_clear_error(_ptr(workspace), _stream()), "kvarn_clear_error")
