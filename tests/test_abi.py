"""CPU checks of the C-ABI library: it builds, loads, exports every symbol the
header declares, and its host-side argument checks answer without a GPU."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mlaq.h")


@pytest.fixture(scope="module")
def lib():
    from bit_mla_kv_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mlaq_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("mlaq_append", "mlaq_decode", "mlaq_buffer_sizes", "mlaq_cache_create", "mlaq_export_tokens"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_covers_the_exports():
    import bit_mla_kv_gb300.mlaq as m
    assert sorted(m.EXPORTED) == declared_functions()


def test_binding_status_bits_match_the_header():
    import bit_mla_kv_gb300.mlaq as m
    text = open(HEADER).read()
    bits = dict(re.findall(r"#define MLAQ_DEV_([A-Z_]+) (0x[0-9a-fA-F]+)", text))
    assert len(bits) >= 6
    for name, val in bits.items():
        assert getattr(m, "DEV_" + name) == int(val, 16), name
    assert len(set(bits.values())) == len(bits)   # distinct bits


def test_buffer_sizes_host_logic(lib):
    import bit_mla_kv_gb300.mlaq as m
    cb, mb, rb, wb = m.buffer_sizes("C4R4", 10, 3, 16)
    assert cb == 10 * 64 * 288 and mb == 10 * 64 * 36 and rb == 3 * 132 * 576 * 2
    cb, mb, rb, wb2 = m.buffer_sizes("C2R4", 10, 3, 16)
    assert cb == 10 * 64 * 160 and mb == 10 * 64 * 36 and wb2 == wb
    cb, mb, rb, _ = m.buffer_sizes("BF16", 10, 3, 16)
    assert cb == 10 * 64 * 1152 and mb == 0 and rb == 0
    with pytest.raises(m.MlaqError):
        m.buffer_sizes("C4R4", 10, 3, 24)   # heads not a multiple of 16
    with pytest.raises(m.MlaqError):
        m.buffer_sizes("C4R4", 0, 3, 16)


def test_host_argument_errors(lib):
    lib.mlaq_status_string.restype = ctypes.c_char_p
    assert lib.mlaq_status_string(0) == b"ok"
    out = ctypes.c_void_p()
    # bad mode / sizes / NULL buffers are rejected before any CUDA call
    assert lib.mlaq_cache_create(ctypes.byref(out), 7, 1, 1, 1, 16, None, None, None, None, ctypes.c_size_t(0)) == -2
    assert lib.mlaq_cache_create(ctypes.byref(out), 0, 0, 1, 1, 16, None, None, None, None, ctypes.c_size_t(0)) == -3
    assert lib.mlaq_cache_create(ctypes.byref(out), 0, 1, 1, 1, 16, None, None, None, None, ctypes.c_size_t(0)) == -1
    # plan cost sums would overflow 32 bits: 16384 * (32 * 5000 + 512) >= 2^31
    assert lib.mlaq_cache_create(ctypes.byref(out), 0, 1, 16384, 5000, 16, None, None, None, None, ctypes.c_size_t(0)) == -3
    buf = ctypes.create_string_buffer(64)
    addr = (ctypes.addressof(buf) + 15) // 16 * 16
    mis = ctypes.c_void_p(addr + 4)
    assert lib.mlaq_cache_create(ctypes.byref(out), 0, 1, 1, 1, 16, mis, mis, mis, mis, ctypes.c_size_t(0)) == -4
    assert lib.mlaq_decode(None, None, None, None, None, 1, 16, ctypes.c_float(1.0), None, None, None) == -1
    assert lib.mlaq_append(None, None, None, 1, None, None, 1, None, 0, None) == -1
    assert lib.mlaq_timing_enable(None, 4) == -1
    assert lib.mlaq_set_plan_costs(None, 8, 19, 40) == -1
    # multi-token decode: Q * H <= 128, H a multiple of 16
    assert lib.mlaq_decode_mtp(None, None, None, None, None, 1, 2, 16, ctypes.c_float(1.0), None, None, None) == -1
    # the bounded-wait test hook checks its arguments before any launch
    assert lib.mlaq_debug_wait_probe(None, 1000, 0, None) == -1
    assert lib.mlaq_debug_wait_probe(mis, 0, 0, None) == -3
    assert lib.mlaq_debug_wait_probe(mis, 100001, 0, None) == -3
    assert lib.mlaq_debug_wait_probe(mis, 1000, 2, None) == -3


def test_code_layout_is_a_bijection():
    # The physical nibble/crumb positions of the 64 channels of a group must
    # be distinct and fill the group's bytes (checked through the export
    # path's inverse on the GPU; here the formula itself, mirrored in Python
    # from the header comment, is checked for collisions).
    def content_bit(c, bits):
        kk, bi, i, ln = c >> 4, (c >> 3) & 1, (c >> 1) & 3, c & 1
        if bits == 4:
            word, p = 2 * i + (kk >> 1), 2 * (kk & 1) + bi
            return word * 32 + 16 * ln + 4 * (p & 1) + 8 * (p >> 1)
        word, p = i, 2 * kk + bi
        return word * 32 + 16 * ln + 2 * (p & 3) + 8 * (p >> 2)

    def rope_bit(c):
        kk, bi, i, ln = c >> 4, (c >> 3) & 1, (c >> 1) & 3, c & 1
        return (2 * kk + (i >> 1)) * 32 + 16 * ln + 8 * (i & 1) + 4 * bi

    for bits in (4, 2):
        cells = sorted(content_bit(c, bits) // bits for c in range(64))
        assert cells == list(range(64))
        assert all(content_bit(c, bits) % bits == 0 for c in range(64))
    assert sorted(rope_bit(c) // 4 for c in range(64)) == list(range(64))


def test_bf16_row_chunk_permutation():
    # The binding's inverse of the stored BF16 row order (header: channel e of
    # row r at ((e / 8) ^ (r % 8)) * 8 + e % 8) undoes a forward scatter, and
    # the 8 rows of one fragment read one channel from 8 distinct chunks mod 8.
    import torch
    from bit_mla_kv_gb300.mlaq import _bf16_rows_in_channel_order
    rows = 132
    logical = torch.arange(rows * 576, dtype=torch.float32).view(1, rows, 576)
    stored = torch.empty_like(logical)
    for r in range(rows):
        for e in range(576):
            stored[0, r, ((e // 8) ^ (r % 8)) * 8 + e % 8] = logical[0, r, e]
    assert torch.equal(_bf16_rows_in_channel_order(stored), logical)
    for e in range(0, 576, 8):
        assert sorted((((e // 8) ^ r) * 8) // 8 % 8 for r in range(8)) == list(range(8))
