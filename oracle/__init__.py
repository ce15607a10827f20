"""fp64 CPU oracle for the KVarN 2-bit KV-cache path: ctypes glue around
``kvarn_oracle.c``.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s cpu_baseline / reference leg may import this package. It shares
no code with the CUDA library ``bit_kv_cache_08_gb300`` and never imports it.

Every function restates one step of the method (see the C file's header for
the pages and sections it follows); arrays are float64 numpy arrays unless
stated otherwise.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvarn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libkvarn_oracle.so")
_lock = threading.Lock()
_lib = None

D = 128
NG = 4
GS = 32
KIND_K, KIND_V = 0, 1
# ablation switches (the pages' 消融 study): no rotation, VarN without the
# token pass, VarN without the channel pass
NO_ROTATION, NO_TOKEN_PASS, NO_CHANNEL_PASS = 1, 2, 4
_u32 = ctypes.c_uint32


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-fopenmp", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_f64p = ctypes.POINTER(ctypes.c_double)
_i32p = ctypes.POINTER(ctypes.c_int32)
_u32p = ctypes.POINTER(ctypes.c_uint32)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_i = ctypes.c_int
_i64 = ctypes.c_int64
_d = ctypes.c_double


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            sig = {
                "orc_f16_rn": (_d, [_d]), "orc_f16_rd": (_d, [_d]), "orc_f16_ru": (_d, [_d]),
                "orc_f16_bits": (ctypes.c_uint16, [_d]),
                "orc_f16_value": (_d, [ctypes.c_uint16]),
                "orc_bf16_value": (_d, [ctypes.c_uint16]),
                "orc_hadamard": (None, [_i, _i32p]),
                "orc_rotate": (None, [_f64p, _u32p, _f64p]),
                "orc_unrotate": (None, [_f64p, _u32p, _f64p]),
                "orc_varn": (None, [_i, _i, ctypes.c_uint32, _f64p, _f64p, _f64p, _f64p, _f64p]),
                "orc_round_factor": (_d, [_d]),
                "orc_group_params": (None, [_f64p, _i, _i, _f64p, _f64p, _f64p, _f64p]),
                "orc_code": (_i, [_d, _d, _d, _i]),
                "orc_step_for": (_d, [_d, _d, _i]),
                "orc_code_position": (None, [_i, _i, _i, _i, _i32p, _i32p]),
                "orc_head_block_bytes": (ctypes.c_size_t, [_i, _i]),
                "orc_pack": (None, [_i, _i, _i, _i32p, _f64p, _f64p, _f64p, _f64p, _u8p]),
                "orc_unpack": (None, [_i, _i, _i, _u8p, _i32p, _f64p, _f64p, _f64p, _f64p]),
                "orc_quantize_block": (None, [_i, _i, _i, ctypes.c_uint32, _i, _u32p, _f64p, _u8p, _f64p, _f64p,
                                              _f64p, _f64p, _f64p, _f64p, _f64p, _f64p,
                                              _i32p, _f64p]),
                "orc_quantize_blocks": (None, [_i64, _i, _i, _i, ctypes.c_uint32, _i, _u32p, _f64p, _u8p]),
                "orc_decode_block": (None, [_i, _i, ctypes.c_uint32, _i, _u32p, _u8p, _i, _f64p]),
                "orc_decode_blocks": (None, [_i64, _i, _i, ctypes.c_uint32, _i, _u32p, _u8p, _i, _f64p]),
                "orc_attention": (None, [_f64p, _f64p, _f64p, _i64, _d, _f64p]),
                "orc_attention_rotated": (None, [_f64p, _f64p, _f64p, _i64, _d, _u32p, _f64p]),
                "orc_decode_attention": (None, [_i, _i, ctypes.c_uint32, _i, _i, _u32p, _d, _f64p, _u8p, _u16p,
                                                _i32p, _i, _i32p, _i, _f64p]),
                "orc_prefill_attention": (None, [_i, _i, ctypes.c_uint32, _i, _i, _u32p, _d, _f64p, _u8p, _u16p,
                                                 _i32p, _i, _i32p, _i, _i, _f64p]),
                "orc_code_high_position": (None, [_i, _i, _i, ctypes.POINTER(_i), ctypes.POINTER(_i)]),
                "orc_error_split": (None, [_f64p, _f64p, _f64p]),
                "orc_error_decomposition": (None, [_i, _i, ctypes.c_uint32, _i, _u32p, _f64p, _u8p, _f64p]),
                "orc_normalise": (None, [_i, _f64p, _f64p, _f64p, _f64p]),
                "orc_group_params_all": (None, [_i, _i, _f64p, _f64p, _f64p, _f64p, _f64p]),
                "orc_codes_given": (None, [_i, _i, _f64p, _f64p, _f64p, _i32p, _f64p]),
                "orc_set_threads": (None, [_i]),
                "orc_max_threads": (_i, []),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def set_threads(n: int) -> None:
    """Threads of the oracle's OpenMP loops from now on (n >= 1)."""
    lib().orc_set_threads(int(n))


def max_threads() -> int:
    return int(lib().orc_max_threads())


# --------------------------------------------------------------------------
# array plumbing
# --------------------------------------------------------------------------

def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a, ct):
    return a.ctypes.data_as(ct)


def _signs(sign_bits):
    s = np.ascontiguousarray(np.asarray(sign_bits, dtype=np.uint32).reshape(4))
    return s


def sigma(sign_bits) -> np.ndarray:
    """The 128 signs (+1/-1) encoded by ``sign_bits`` (bit c set => -1)."""
    s = _signs(sign_bits)
    c = np.arange(D)
    bits = (s[c // 32] >> (c % 32).astype(np.uint32)) & 1
    return np.where(bits == 1, -1.0, 1.0)


def head_block_bytes(B: int, bits: int = 2) -> int:
    return int(lib().orc_head_block_bytes(B, bits))


# --------------------------------------------------------------------------
# fp16 / bf16 grid
# --------------------------------------------------------------------------

def f16_rn(v: float) -> float:
    return lib().orc_f16_rn(float(v))


def f16_rd(v: float) -> float:
    return lib().orc_f16_rd(float(v))


def f16_ru(v: float) -> float:
    return lib().orc_f16_ru(float(v))


def f16_bits(h: float) -> int:
    return int(lib().orc_f16_bits(float(h)))


def f16_value(b: int) -> float:
    return lib().orc_f16_value(int(b) & 0xFFFF)


def bf16_value(b: int) -> float:
    return lib().orc_bf16_value(int(b) & 0xFFFF)


def bf16_array_to_f64(u16: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 values: the top half of an fp32."""
    u = np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# rotation
# --------------------------------------------------------------------------

def hadamard(n: int = D) -> np.ndarray:
    H = np.zeros((n, n), dtype=np.int32)
    lib().orc_hadamard(n, _p(H, _i32p))
    return H


def rotate(x, sign_bits) -> np.ndarray:
    x = _f64(x).reshape(-1, D)
    out = np.empty_like(x)
    s = _signs(sign_bits)
    for i in range(x.shape[0]):
        lib().orc_rotate(_p(x[i], _f64p), _p(s, _u32p), _p(out[i], _f64p))
    return out


def unrotate(y, sign_bits) -> np.ndarray:
    y = _f64(y).reshape(-1, D)
    out = np.empty_like(y)
    s = _signs(sign_bits)
    for i in range(y.shape[0]):
        lib().orc_unrotate(_p(y[i], _f64p), _p(s, _u32p), _p(out[i], _f64p))
    return out


# --------------------------------------------------------------------------
# VarN and quantisation
# --------------------------------------------------------------------------

def varn(Xr, iters: int, flags: int = 0):
    """Returns (Y, R, C, trace[iters][3]) for one head-block of rotated values."""
    Xr = _f64(Xr)
    B = Xr.shape[0]
    Y = np.empty_like(Xr)
    R = np.empty(B)
    C = np.empty(D)
    tr = np.empty((max(iters, 1), 3))
    lib().orc_varn(B, iters, flags, _p(Xr, _f64p), _p(Y, _f64p), _p(R, _f64p), _p(C, _f64p),
                   _p(tr, _f64p))
    return Y, R, C, tr[:iters]


def round_factor(f: float) -> float:
    return lib().orc_round_factor(float(f))


def group_params(y, bits: int = 2):
    y = _f64(y)
    z = ctypes.c_double()
    s = ctypes.c_double()
    m = ctypes.c_double()
    M = ctypes.c_double()
    lib().orc_group_params(_p(y, _f64p), y.size, (1 << bits) - 1, ctypes.byref(z), ctypes.byref(s),
                           ctypes.byref(m), ctypes.byref(M))
    return z.value, s.value, m.value, M.value


def step_for(z16: float, M: float, bits: int = 2) -> float:
    """Least fp16 s >= 0 with z16 + (2^bits - 1) s >= M."""
    return lib().orc_step_for(float(z16), float(M), (1 << bits) - 1)


def code(y: float, z16: float, s16: float, bits: int = 2) -> int:
    return int(lib().orc_code(float(y), float(z16), float(s16), (1 << bits) - 1))


def code_position(kind: int, t: int, c: int, bits: int = 2):
    w = ctypes.c_int32()
    b = ctypes.c_int32()
    lib().orc_code_position(kind, bits, t, c, ctypes.byref(w), ctypes.byref(b))
    return w.value, b.value


def code_high_position(kind: int, t: int, c: int):
    """(word, bit) of the high bit of a 3-bit code (its low two bits sit at
    code_position(kind, t, c, bits=3))."""
    w, b = ctypes.c_int(), ctypes.c_int()
    lib().orc_code_high_position(kind, t, c, ctypes.byref(w), ctypes.byref(b))
    return w.value, b.value


def pack(B, kind, codes, s16, z16, R16, C16, bits: int = 2) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.int32).reshape(B, D)
    s16, z16 = _f64(s16).reshape(B, NG), _f64(z16).reshape(B, NG)
    R16, C16 = _f64(R16).reshape(B), _f64(C16).reshape(D)
    out = np.zeros(head_block_bytes(B, bits), dtype=np.uint8)
    lib().orc_pack(B, bits, kind, _p(codes, _i32p), _p(s16, _f64p), _p(z16, _f64p), _p(R16, _f64p),
                   _p(C16, _f64p), _p(out, _u8p))
    return out


def unpack(B, kind, hb_bytes, bits: int = 2):
    hb = np.ascontiguousarray(hb_bytes, dtype=np.uint8).reshape(-1)
    codes = np.empty((B, D), dtype=np.int32)
    s16 = np.empty((B, NG))
    z16 = np.empty((B, NG))
    R16 = np.empty(B)
    C16 = np.empty(D)
    lib().orc_unpack(B, bits, kind, _p(hb, _u8p), _p(codes, _i32p), _p(s16, _f64p), _p(z16, _f64p),
                     _p(R16, _f64p), _p(C16, _f64p))
    return dict(codes=codes, s16=s16, z16=z16, R16=R16, C16=C16)


def quantize_block(X, iters: int, kind: int, sign_bits, flags: int = 0, bits: int = 2) -> dict:
    """All intermediate results of one head-block (X: [B][128] values)."""
    X = _f64(X)
    B = X.shape[0]
    s = _signs(sign_bits)
    r = dict(bytes=np.zeros(head_block_bytes(B, bits), dtype=np.uint8), Xr=np.empty((B, D)),
             R=np.empty(B), C=np.empty(D), R16=np.empty(B), C16=np.empty(D),
             y=np.empty((B, D)), z16=np.empty((B, NG)), s16=np.empty((B, NG)),
             codes=np.empty((B, D), dtype=np.int32), trace=np.empty((max(iters, 1), 3)))
    lib().orc_quantize_block(B, bits, iters, flags, kind, _p(s, _u32p), _p(X, _f64p), _p(r["bytes"], _u8p),
                             _p(r["Xr"], _f64p), _p(r["R"], _f64p), _p(r["C"], _f64p),
                             _p(r["R16"], _f64p), _p(r["C16"], _f64p), _p(r["y"], _f64p),
                             _p(r["z16"], _f64p), _p(r["s16"], _f64p), _p(r["codes"], _i32p),
                             _p(r["trace"], _f64p))
    r["trace"] = r["trace"][:iters]
    return r


def quantize_blocks(X, iters: int, kind: int, sign_bits, flags: int = 0, bits: int = 2) -> np.ndarray:
    """X: [n][B][128] -> packed bytes [n][head_block_bytes(B)]."""
    X = _f64(X)
    n, B = X.shape[0], X.shape[1]
    out = np.zeros((n, head_block_bytes(B, bits)), dtype=np.uint8)
    s = _signs(sign_bits)
    lib().orc_quantize_blocks(n, B, bits, iters, flags, kind, _p(s, _u32p), _p(X, _f64p), _p(out, _u8p))
    return out


def decode_blocks(hb_bytes, B: int, kind: int, sign_bits, rotated: bool, flags: int = 0,
                  bits: int = 2) -> np.ndarray:
    """Packed head-blocks [n][bytes] -> values [n][B][128]."""
    hb = np.ascontiguousarray(hb_bytes, dtype=np.uint8).reshape(-1, head_block_bytes(B, bits))
    n = hb.shape[0]
    out = np.empty((n, B, D))
    s = _signs(sign_bits)
    lib().orc_decode_blocks(n, B, bits, flags, kind, _p(s, _u32p), _p(hb, _u8p), 1 if rotated else 0,
                            _p(out, _f64p))
    return out


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------

def attention(q, K, V, sm_scale: float) -> np.ndarray:
    q, K, V = _f64(q).reshape(D), _f64(K).reshape(-1, D), _f64(V).reshape(-1, D)
    out = np.empty(D)
    lib().orc_attention(_p(q, _f64p), _p(K, _f64p), _p(V, _f64p), K.shape[0], float(sm_scale),
                        _p(out, _f64p))
    return out


def attention_rotated(q, K, V, sm_scale: float, sign_bits) -> np.ndarray:
    q, K, V = _f64(q).reshape(D), _f64(K).reshape(-1, D), _f64(V).reshape(-1, D)
    out = np.empty(D)
    s = _signs(sign_bits)
    lib().orc_attention_rotated(_p(q, _f64p), _p(K, _f64p), _p(V, _f64p), K.shape[0],
                                float(sm_scale), _p(s, _u32p), _p(out, _f64p))
    return out


def decode_attention(B, n_q, n_kv, sign_bits, sm_scale, q, pool, staging, block_table,
                     seq_lens, flags: int = 0, bits: int = 2) -> np.ndarray:
    """Attention of every (sequence, query head) over the paged 2-bit cache.

    q: [batch][n_q][128] values; pool: raw bytes of the physical blocks;
    staging: bf16 bit patterns [batch][n_kv][2][B][128]; block_table:
    int32 [batch][max_blocks]; seq_lens: int32 [batch].
    """
    q = _f64(q)
    batch = q.shape[0]
    pool = np.ascontiguousarray(pool, dtype=np.uint8).reshape(-1)
    staging = np.ascontiguousarray(staging, dtype=np.uint16)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32).reshape(batch)
    out = np.zeros((batch, n_q, D))
    s = _signs(sign_bits)
    lib().orc_decode_attention(B, bits, flags, n_q, n_kv, _p(s, _u32p), float(sm_scale), _p(q, _f64p),
                               _p(pool, _u8p), _p(staging, _u16p), _p(bt, _i32p), bt.shape[1],
                               _p(sl, _i32p), batch, _p(out, _f64p))
    return out


def prefill_attention(B, n_q, n_kv, sign_bits, sm_scale, q, pool, staging, block_table,
                      seq_lens, flags: int = 0, bits: int = 2) -> np.ndarray:
    """Chunked prefill attention over the paged cache: q is [batch][chunk][n_q][128];
    query row r of sequence b sits at position seq_lens[b] - chunk + r and sees
    the tokens up to it, read from the cache as it stands (zeros for a row at a
    negative position). Returns [batch][chunk][n_q][128]."""
    q = _f64(q)
    batch, chunk = q.shape[0], q.shape[1]
    pool = np.ascontiguousarray(pool, dtype=np.uint8).reshape(-1)
    staging = np.ascontiguousarray(staging, dtype=np.uint16)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32).reshape(batch)
    out = np.zeros((batch, chunk, n_q, D))
    s = _signs(sign_bits)
    lib().orc_prefill_attention(B, bits, flags, n_q, n_kv, _p(s, _u32p), float(sm_scale), _p(q, _f64p),
                                _p(pool, _u8p), _p(staging, _u16p), _p(bt, _i32p), bt.shape[1],
                                _p(sl, _i32p), batch, chunk, _p(out, _f64p))
    return out


# --------------------------------------------------------------------------
# error decomposition (magnitude / direction)
# --------------------------------------------------------------------------

def error_split(x, xh) -> np.ndarray:
    """(|x|, |x^|, |E_M|, |E_D|) of one token vector and its quantised version."""
    x, xh = _f64(x).reshape(D), _f64(xh).reshape(D)
    out = np.empty(4)
    lib().orc_error_split(_p(x, _f64p), _p(xh, _f64p), _p(out, _f64p))
    return out


def error_decomposition(X, packed, B: int, kind: int, sign_bits, flags: int = 0, bits: int = 2) -> np.ndarray:
    """X: [n][B][128] values before quantisation, packed: [n][bytes] -> [n][B][4]."""
    X = _f64(X).reshape(-1, B, D)
    pk = np.ascontiguousarray(packed, dtype=np.uint8).reshape(X.shape[0], -1)
    out = np.empty((X.shape[0], B, 4))
    s = _signs(sign_bits)
    for i in range(X.shape[0]):
        lib().orc_error_decomposition(B, bits, flags, kind, _p(s, _u32p), _p(X[i], _f64p), _p(pk[i], _u8p),
                                      _p(out[i], _f64p))
    return out


# --------------------------------------------------------------------------
# staged hand-off helpers
# --------------------------------------------------------------------------

def normalise(Xr, R16, C16) -> np.ndarray:
    Xr = _f64(Xr)
    B = Xr.shape[0]
    R16, C16 = _f64(R16).reshape(B), _f64(C16).reshape(D)
    y = np.empty_like(Xr)
    lib().orc_normalise(B, _p(Xr, _f64p), _p(R16, _f64p), _p(C16, _f64p), _p(y, _f64p))
    return y


def group_params_all(y, bits: int = 2):
    y = _f64(y)
    B = y.shape[0]
    z, s, m, M = (np.empty((B, NG)) for _ in range(4))
    lib().orc_group_params_all(B, bits, _p(y, _f64p), _p(z, _f64p), _p(s, _f64p), _p(m, _f64p),
                               _p(M, _f64p))
    return z, s, m, M


def codes_given(y, z16, s16, bits: int = 2):
    y = _f64(y)
    B = y.shape[0]
    z16, s16 = _f64(z16).reshape(B, NG), _f64(s16).reshape(B, NG)
    codes = np.empty((B, D), dtype=np.int32)
    dist = np.empty((B, D))
    lib().orc_codes_given(B, bits, _p(y, _f64p), _p(z16, _f64p), _p(s16, _f64p), _p(codes, _i32p),
                          _p(dist, _f64p))
    return codes, dist
