"""The C ABI library builds, loads and exports every symbol include/kvarn.h
declares; size queries and host-side argument validation work without a GPU
(no compute is launched here)."""
import ctypes

import pytest

import bit_kv_cache_08_gb300 as kv
import oracle
import synth


@pytest.fixture(scope="module", autouse=True)
def built():
    kv.build()


def _cfg(**kw):
    base = dict(n_q_heads=32, n_kv_heads=8, block_size=32, varn_iters=3, sign_bits=synth.sign_bits(1))
    base.update(kw)
    return kv.make_config(**base)


def test_library_exports_every_declared_symbol():
    names = kv.header_symbols()
    assert len(names) >= 13
    L = kv.lib()
    for n in names:
        assert hasattr(L, n), n
    assert kv.version().startswith("kvarn")


def test_sizes_match_the_format():
    c32, c64 = _cfg(), _cfg(block_size=64)
    assert kv.head_block_bytes(c32) == 1856 and kv.head_block_bytes(c64) == 3456
    assert kv.block_bytes(c32) == 8 * 2 * 1856
    assert kv.staging_bytes(c32, 16) == 16 * 8 * 2 * 32 * 128 * 2
    assert kv.workspace_bytes(c32, 0, 0) == 256


def test_prefill_workspace_query_without_a_device():
    c = _cfg()
    assert kv.prefill_workspace_bytes(c, 0, 4, 0) == 256
    assert kv.prefill_workspace_bytes(c, 2, 0, 4) == 0          # chunk >= 1
    assert kv.prefill_workspace_bytes(c, -1, 4, 4) == 0


def test_wide_code_sizes_match_the_oracle_format():
    """3- and 4-bit codes: records of 48 / 64 bytes, then the same s, z, R, C sections."""
    for B in (32, 64):
        for bits in (3, 4):
            c = _cfg(block_size=B, bits=bits)
            hb = (16 * bits + 18) * B + 256
            assert kv.head_block_bytes(c) == hb == oracle.head_block_bytes(B, bits=bits)
            assert kv.block_bytes(c) == 8 * 2 * hb


@pytest.mark.parametrize("field,value", [("head_dim", 64), ("block_size", 16), ("bits", 5),
                                         ("bits", 1), ("bits", 8),
                                         ("group_size", 64), ("n_q_heads", 48)])
def test_unsupported_configs_are_rejected(field, value):
    c = _cfg()
    setattr(c, field, value)
    assert kv.head_block_bytes(c) == 0
    r = kv.lib().kvarn_quantize_block(ctypes.byref(c), 0, None, 0, 1, 4096, 128, None, None, None, None)
    assert r == kv._abi.ERR_UNSUPPORTED


def test_invalid_arguments_are_rejected_before_any_launch():
    L = kv.lib()
    c = _cfg()
    INV = -1
    assert L.kvarn_quantize_block(None, 0, None, 0, 1, 4096, 128, None, None, None, None) == INV
    assert L.kvarn_quantize_block(ctypes.byref(c), 2, None, 0, 1, 4096, 128, None, None, None, None) == INV
    assert L.kvarn_quantize_block(ctypes.byref(c), 0, None, 0, 1, 4096, 128, None, None, None, None) == INV
    # zero blocks is a no-op
    assert L.kvarn_quantize_block(ctypes.byref(c), 0, None, 0, 0, 4096, 128, None, None, None, None) == 0
    # misaligned pointers
    p = ctypes.c_void_p(0x1000 + 2)
    assert L.kvarn_append(ctypes.byref(c), p, 10, p, p, 4, p, p, p, 1, p, None) == INV
    assert L.kvarn_decode_attn(ctypes.byref(c), None, 0, None, 1, None, None, 4, None, 1, None, None, 0,
                               None) == INV
    bad = _cfg(varn_iters=0)
    assert L.kvarn_dequantize(ctypes.byref(bad), 0, None, None, 1, 0, None, None) == INV
    assert kv.status_string(-4) == "workspace too small"


def test_ablation_flags_and_zero_iterations_are_validated():
    L = kv.lib()
    assert kv.head_block_bytes(_cfg(varn_iters=0)) == 1856                  # Hadamard only
    assert kv.head_block_bytes(_cfg(flags=kv.FLAG_NO_ROTATION | kv.FLAG_NO_TOKEN_PASS)) == 1856
    for bad in (_cfg(varn_iters=-1), _cfg(varn_iters=9), _cfg(flags=8)):
        assert kv.head_block_bytes(bad) == 0
        assert L.kvarn_quantize_block(ctypes.byref(bad), 0, None, 0, 1, 4096, 128, None, None, None,
                                      None) == kv._abi.ERR_INVALID_ARG


def test_source_extent_checks_in_the_binding():
    """The binding counts whole blocks of a contiguous source and refuses a
    block count or strides that would read past the source's storage."""
    import torch
    c = _cfg()
    src = torch.zeros(2, 2, 64, 128, dtype=torch.bfloat16)
    assert kv._abi._blocks_in(src, c, None, None, 128) == (8, 32 * 128)
    with pytest.raises(ValueError):
        kv._abi._blocks_in(src, c, 9, None, 128)
    with pytest.raises(ValueError):
        kv._abi._blocks_in(src, c, None, 64 * 128, 128)          # strides need an explicit count
    inter = torch.zeros(3, 32, 2, 128)                             # [n][B][2][128], V rows interleaved
    view = inter[:, :, 1]
    assert kv._abi._blocks_in(view, c, 3, 32 * 256, 256) == (3, 32 * 256)
    with pytest.raises(ValueError):
        kv._abi._blocks_in(view, c, 4, 32 * 256, 256)
    with pytest.raises(ValueError):
        kv._abi._blocks_in(view, c, None, None, 128)               # non-contiguous without strides
