"""The allocation-free decode entry point (mlaq_decode_noalloc).

Some callers cannot allocate device memory (code inside another runtime's
allocator, plugins that must not call cudaMalloc during stream capture,
hosts that reserve all of HBM). For them the split-KV scratch lives in a
fixed array inside the library. This test calls that entry point through the
C ABI and checks it against mlaq_decode on the same cache, twice in a row
(the second call reuses the array the first one left behind), and against
the oracle. It sits in a
file collected last so that a stop-at-first-failure run has already run every
other test; it passes alone in a fresh process as well.
"""

import ctypes

import pytest
import torch

from mlaq_testlib import Case, assert_close_out

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode,lens,H", [("C4R4", [5, 140, 1000, 5000, 12000], 16),
                                         ("C2R4", [300, 2048], 128)])
def test_noalloc_matches_decode_twice(mode, lens, H):
    import bit_mla_kv_gb300.mlaq as m
    case = Case(mode, lens, H, seed=21)
    case.build()
    ql, qr = case.ql.cuda().contiguous(), case.qr.cuda().contiguous()
    ref_out, ref_lse = case.cache.decode(ql, qr, case.pt_d, case.seq_d, case.scale)
    ref_out, ref_lse = ref_out.clone(), ref_lse.clone()
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        c = case.cache
        rc = m._lib.mlaq_decode_noalloc(
            m.MODES[mode], ctypes.c_void_p(c.codes.data_ptr()), ctypes.c_void_p(c.meta.data_ptr()),
            ctypes.c_void_p(c.ring.data_ptr()), c.num_pages, c.max_pages_per_seq,
            ctypes.c_void_p(ql.data_ptr()), ctypes.c_void_p(qr.data_ptr()), ctypes.c_void_p(case.pt_d.data_ptr()),
            ctypes.c_void_p(case.seq_d.data_ptr()), case.B, H, ctypes.c_float(case.scale),
            ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()), ctypes.c_void_p(st.data_ptr()),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == 0, m._lib.mlaq_status_string(rc)
        torch.cuda.synchronize()
        assert int(st.item()) == 0, f"call {call}: device status {int(st.item())}"
        for b in range(case.B):
            assert_close_out(out[b], lse[b], ref_out[b].float().cpu().double().numpy(),
                             ref_lse[b].cpu().double().numpy(), f"call {call} seq {b}")
    # and directly against the oracle, so that a fault shared by both entry
    # points (planner, attention kernel, combine) cannot pass unseen
    for b in range(case.B):
        ro, rl = case.oracle_seq(b)
        assert_close_out(out[b], lse[b], ro, rl, f"oracle seq {b}")


def _noalloc(m, cache, mode, ql, qr, pt, seq, B, H, scale, out, lse, st):
    return m._lib.mlaq_decode_noalloc(
        m.MODES[mode], ctypes.c_void_p(cache.codes.data_ptr()), ctypes.c_void_p(cache.meta.data_ptr()),
        ctypes.c_void_p(cache.ring.data_ptr()), cache.num_pages, cache.max_pages_per_seq,
        ctypes.c_void_p(ql.data_ptr()), ctypes.c_void_p(qr.data_ptr()), ctypes.c_void_p(pt.data_ptr()),
        ctypes.c_void_p(seq.data_ptr()), B, H, ctypes.c_float(scale), ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(lse.data_ptr()), ctypes.c_void_p(st.data_ptr()) if st is not None else None,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _largest_batch_that_fits(m, H):
    """The largest B whose split-KV scratch (the workspace mlaq_buffer_sizes
    asks for at max_seqs = B, max_heads = H) fits the fixed 64 MiB array."""
    lo, hi = 1, 16384
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if m.buffer_sizes("C4R4", 1, mid, H)[3] <= 64 << 20:
            lo = mid
        else:
            hi = mid - 1
    return lo


def test_noalloc_capacity_edge():
    # Just under the limit the call runs and agrees with mlaq_decode and the
    # oracle; one sequence more is refused before anything is launched.
    import bit_mla_kv_gb300.mlaq as m
    H = 128
    B = _largest_batch_that_fits(m, H)
    assert 240 <= B <= 260, B   # the documented capacity at H = 128
    lens = [(1, 5, 64, 133, 300)[b % 5] for b in range(B)]
    case = Case("C4R4", lens, H, seed=24, gen_device="cuda")
    case.build()
    ql, qr = case.ql.cuda().contiguous(), case.qr.cuda().contiguous()
    ref_out, ref_lse = case.cache.decode(ql, qr, case.pt_d, case.seq_d, case.scale)
    out = torch.full_like(ref_out, float("nan"))
    lse = torch.full_like(ref_lse, float("nan"))
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    rc = _noalloc(m, case.cache, "C4R4", ql, qr, case.pt_d, case.seq_d, B, H, case.scale, out, lse, st)
    assert rc == 0, m._lib.mlaq_status_string(rc)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for b in range(B):
        assert_close_out(out[b], lse[b], ref_out[b].float().cpu().double().numpy(),
                         ref_lse[b].cpu().double().numpy(), f"seq {b}")
    for b in (0, 3, 4, B - 1):
        ro, rl = case.oracle_seq(b)
        assert_close_out(out[b], lse[b], ro, rl, f"oracle seq {b}")
    rc = _noalloc(m, case.cache, "C4R4", ql, qr, case.pt_d, case.seq_d, B + 1, H, case.scale, out, lse, None)
    assert rc == -5   # MLAQ_ERR_CAPACITY


def test_noalloc_rejects_oversized_batch():
    import bit_mla_kv_gb300.mlaq as m
    case = Case("C4R4", [10], 16, seed=22)
    case.build()
    big_b, H = 8192, 128   # needs far more than the fixed scratch holds
    rc = m._lib.mlaq_decode_noalloc(
        0, ctypes.c_void_p(case.cache.codes.data_ptr()), ctypes.c_void_p(case.cache.meta.data_ptr()),
        ctypes.c_void_p(case.cache.ring.data_ptr()), case.cache.num_pages, case.cache.max_pages_per_seq,
        ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16), big_b, H,
        ctypes.c_float(1.0), ctypes.c_void_p(16), ctypes.c_void_p(16), None, None)
    assert rc == -5   # MLAQ_ERR_CAPACITY, returned before anything is launched
