"""GPU parity of libmlaq against the CPU oracle (codes bit-exact, outputs
within the stated tolerances), called through the C ABI."""

import math

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from mlaq_testlib import Case, assert_close_out, expected_codes

pytestmark = pytest.mark.gpu

EDGE_LENS = [0, 1, 3, 4, 5, 63, 64, 65, 131, 132, 133, 200, 257, 1000, 4097]


def _export_all(case):
    bs, ts = [], []
    for b, L in enumerate(case.seq_lens):
        bs += [b] * L
        ts += list(range(L))
    tb = torch.tensor(bs, dtype=torch.int32, device="cuda")
    tt = torch.tensor(ts, dtype=torch.int32, device="cuda")
    codes, meta = case.cache.export_tokens(case.pt_d, tb, tt)
    return codes.cpu().numpy(), meta.cpu().numpy()


@pytest.mark.parametrize("mode", ["C4R4", "C2R4"])
def test_writer_codes_meta_ring_bit_exact(mode):
    case = Case(mode, EDGE_LENS, 16, seed=11)
    case.build()
    assert case.cache.device_status() == 0
    assert case.seq_d.cpu().tolist() == case.seq_lens
    codes, meta = _export_all(case)
    off = 0
    ring = case.cache.ring_view().float().cpu().numpy()
    for b, L in enumerate(case.seq_lens):
        if L == 0:
            continue
        ec, em = expected_codes(case, b)
        np.testing.assert_array_equal(codes[off:off + L], ec, err_msg=f"codes seq {b} L={L}")
        np.testing.assert_array_equal(meta[off:off + L].view(np.uint16), em.view(np.uint16),
                                      err_msg=f"meta seq {b} L={L}")
        off += L
        er, valid = O.expected_ring(case.tokens(b), L)
        np.testing.assert_array_equal(ring[b][valid], er[valid], err_msg=f"ring seq {b} L={L}")


@pytest.mark.parametrize("mode", ["C4R4", "C2R4"])
def test_writer_exact_ties_round_half_to_even(mode):
    # Groups with a power-of-two scale whose values sit on code midpoints, so
    # (x - mn) / s = k + 1/2 exactly and the code must round half to even like
    # the oracle's fp32 quantizer; 1000 rows in one call take the bulk writer.
    case = Case(mode, [700, 300], 16, seed=31)
    n = sum(case.seq_lens)
    rng = np.random.default_rng(31)
    c = np.empty((n, 512), np.float32)
    k = np.empty((n, 64), np.float32)
    for arr, bits in ((c, 4 if mode == "C4R4" else 2), (k, 4)):
        qmax = (1 << bits) - 1
        for g in range(arr.shape[1] // 64):
            s0 = rng.choice([0.25, 0.5, 1.0], size=n)
            mn = rng.integers(-4, 4, size=n) * 0.5
            vals = rng.integers(0, qmax, size=(n, 64)) + 0.5
            exact = rng.random((n, 64)) < 0.25  # some entries exactly on a code
            vals[exact] = np.floor(vals[exact])
            vals[:, 0] = 0.0   # the group minimum
            vals[:, 1] = qmax  # the group maximum: s = s0 exactly
            arr[:, 64 * g:64 * g + 64] = mn[:, None] + vals * s0[:, None]
    case.c = torch.from_numpy(c).to(torch.bfloat16)
    case.k = torch.from_numpy(k).to(torch.bfloat16)
    assert np.array_equal(case.c.float().numpy(), c) and np.array_equal(case.k.float().numpy(), k)
    case.build()
    assert case.cache.device_status() == 0
    codes, meta = _export_all(case)
    off = 0
    for b, L in enumerate(case.seq_lens):
        ec, em = expected_codes(case, b)
        np.testing.assert_array_equal(codes[off:off + L], ec, err_msg=f"codes seq {b}")
        np.testing.assert_array_equal(meta[off:off + L].view(np.uint16), em.view(np.uint16), err_msg=f"meta seq {b}")
        off += L


@pytest.mark.parametrize("mode", ["C4R4", "C2R4"])
def test_writer_odd_scale_midpoints_bit_exact(mode):
    # Scales with an odd mantissa (3, 5 or 7 times a power of two, so 1/s is
    # not exact in fp32) and values on code midpoints (x - mn)/s = k + 1/2, or
    # one bf16 ulp beside them: the fp32 quotient must round exactly as the
    # oracle's IEEE division does; 1000 rows take the bulk writer.
    case = Case(mode, [600, 400], 16, seed=37)
    n = sum(case.seq_lens)
    rng = np.random.default_rng(37)
    c = np.empty((n, 512), np.float32)
    k = np.empty((n, 64), np.float32)
    for arr, bits in ((c, 4 if mode == "C4R4" else 2), (k, 4)):
        qmax = (1 << bits) - 1
        for g in range(arr.shape[1] // 64):
            s0 = rng.choice([3.0, 5.0, 7.0], size=n) * 2.0 ** rng.integers(-9, -2, size=n)
            mn = rng.integers(-8, 8, size=n) * s0 / 2
            vals = rng.integers(0, qmax, size=(n, 64)) + 0.5
            x = mn[:, None] + vals * s0[:, None]
            # one bf16 ulp away from the midpoint (away from or towards zero)
            bits = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
            nudge = rng.random((n, 64))
            step = np.where(nudge < 0.2, 1, np.where(nudge > 0.8, -1, 0)).astype(np.int16)
            bits = np.where(x != 0, bits + step, bits).astype(np.int16)
            x = torch.from_numpy(bits).view(torch.bfloat16).float().numpy().astype(np.float64)
            x[:, 0] = mn               # the group minimum
            x[:, 1] = mn + qmax * s0   # the group maximum: s = s0 exactly
            arr[:, 64 * g:64 * g + 64] = x
    case.c = torch.from_numpy(c).to(torch.bfloat16)
    case.k = torch.from_numpy(k).to(torch.bfloat16)
    case.build()
    assert case.cache.device_status() == 0
    codes, meta = _export_all(case)
    off = 0
    for b, L in enumerate(case.seq_lens):
        ec, em = expected_codes(case, b)
        np.testing.assert_array_equal(codes[off:off + L], ec, err_msg=f"codes seq {b}")
        np.testing.assert_array_equal(meta[off:off + L].view(np.uint16), em.view(np.uint16), err_msg=f"meta seq {b}")
        off += L


@pytest.mark.parametrize("mode", ["C4R4", "C2R4", "BF16"])
def test_writer_bulk_varlen_gaps_then_uniform(mode):
    # Two bulk appends on top of each other: a varlen call whose counts
    # include empty sequences between non-empty ones, then a uniform call of
    # 64 rows per sequence starting at those lengths (both above the
    # small-append threshold of 4 rows per SM).
    first = [300, 0, 0, 517, 3, 130, 0, 64, 1, 0, 200, 63, 65, 0, 4, 700]
    n2 = 64
    case = Case(mode, [a + n2 for a in first], 16, seed=19)
    from bit_mla_kv_gb300.mlaq import Cache
    case.cache = Cache(mode, case.num_pages, case.B, case.page_table.shape[1], max_heads=16)
    case.pt_d = case.page_table.cuda()
    case.seq_d = torch.zeros(case.B, dtype=torch.int32, device="cuda")
    cu0 = torch.zeros(case.B + 1, dtype=torch.int32)
    cu0[1:] = torch.cumsum(torch.tensor(first), 0)
    rows = torch.cat([torch.arange(int(case.cu[b]), int(case.cu[b]) + first[b]) for b in range(case.B)])
    case.cache.append(case.pt_d, case.seq_d, case.c[rows].cuda().contiguous(), case.k[rows].cuda().contiguous(),
                      cu_new=cu0.cuda())
    assert case.seq_d.cpu().tolist() == first
    rows = torch.cat([torch.arange(int(case.cu[b]) + first[b], int(case.cu[b]) + first[b] + n2)
                      for b in range(case.B)])
    case.cache.append(case.pt_d, case.seq_d, case.c[rows].view(case.B, n2, 512).cuda().contiguous(),
                      case.k[rows].view(case.B, n2, 64).cuda().contiguous())
    assert case.cache.device_status() == 0
    assert case.seq_d.cpu().tolist() == case.seq_lens
    if mode == "BF16":
        pages = case.cache.bf16_pages_view().cpu()
        for b, L in enumerate(case.seq_lens):
            tok = torch.from_numpy(case.tokens(b))
            for t in range(L):
                p = int(case.page_table[b, t // 64])
                assert torch.equal(pages[p, t % 64].float(), tok[t]), (b, t)
        return
    codes, meta = _export_all(case)
    ring = case.cache.ring_view().float().cpu().numpy()
    off = 0
    for b, L in enumerate(case.seq_lens):
        ec, em = expected_codes(case, b)
        np.testing.assert_array_equal(codes[off:off + L], ec, err_msg=f"codes seq {b} L={L}")
        np.testing.assert_array_equal(meta[off:off + L].view(np.uint16), em.view(np.uint16),
                                      err_msg=f"meta seq {b} L={L}")
        off += L
        er, valid = O.expected_ring(case.tokens(b), L)
        np.testing.assert_array_equal(ring[b][valid], er[valid], err_msg=f"ring seq {b} L={L}")


@pytest.mark.parametrize("lens", [[100, 50], [700, 300]])
@pytest.mark.parametrize("extra", [20, -30])
def test_writer_flags_rows_cu_new_does_not_cover(lens, extra):
    # total_new must equal cu_new[B]. More rows than cu_new places (extra >
    # 0) or fewer (extra < 0) set MLAQ_DEV_BAD_ROWS instead of reading past
    # cu_new and seq_lens; with more rows every placed row is still stored
    # bit-exact. 150 rows take the one-CTA-per-row writer, 1000 the bulk one.
    from bit_mla_kv_gb300.mlaq import Cache, DEV_BAD_ROWS
    case = Case("C4R4", lens, 16, seed=43)
    case.cache = Cache("C4R4", case.num_pages, case.B, case.page_table.shape[1], max_heads=16)
    case.pt_d = case.page_table.cuda()
    case.seq_d = torch.zeros(case.B, dtype=torch.int32, device="cuda")
    n = sum(lens)
    total = n + extra
    gen = torch.Generator().manual_seed(43)
    pad_c = torch.randn(max(extra, 0), 512, generator=gen).to(torch.bfloat16)
    pad_k = torch.randn(max(extra, 0), 64, generator=gen).to(torch.bfloat16)
    c = torch.cat([case.c, pad_c])[:total].cuda().contiguous()
    k = torch.cat([case.k, pad_k])[:total].cuda().contiguous()
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32, device="cuda")
    case.cache.append(case.pt_d, case.seq_d, c, k, cu_new=cu)
    assert case.cache.device_status() & DEV_BAD_ROWS
    case.cache.clear_status()
    if extra > 0:
        assert case.seq_d.cpu().tolist() == lens
        codes, meta = _export_all(case)
        off = 0
        for b, L in enumerate(case.seq_lens):
            ec, em = expected_codes(case, b)
            np.testing.assert_array_equal(codes[off:off + L], ec, err_msg=f"codes seq {b}")
            np.testing.assert_array_equal(meta[off:off + L].view(np.uint16), em.view(np.uint16),
                                          err_msg=f"meta seq {b}")
            off += L
    assert case.cache.device_status() == 0


def test_positions_beyond_the_page_table_are_flagged():
    # A page table with room for 128 tokens per sequence: the writer skips the
    # rows of sequence 1 past position 127 and sets MLAQ_DEV_SEQ_OVERFLOW
    # (the rows inside stay bit-exact); the planner clamps a length beyond the
    # table, sets the same bit, and the other sequence decodes as usual.
    from bit_mla_kv_gb300.mlaq import Cache, DEV_SEQ_OVERFLOW
    lens = [100, 200]
    case = Case("C4R4", lens, 16, seed=47)
    pt = case.page_table[:, :2].contiguous()
    case.cache = Cache("C4R4", case.num_pages, case.B, 2, max_heads=16)
    case.pt_d = pt.cuda()
    case.seq_d = torch.zeros(case.B, dtype=torch.int32, device="cuda")
    case.cache.append(case.pt_d, case.seq_d, case.c.cuda().contiguous(), case.k.cuda().contiguous(),
                      cu_new=case.cu.cuda())
    assert case.cache.device_status() & DEV_SEQ_OVERFLOW
    case.cache.clear_status()
    for b, L in ((0, 100), (1, 128)):
        tb = torch.full((L,), b, dtype=torch.int32, device="cuda")
        tt = torch.arange(L, dtype=torch.int32, device="cuda")
        codes, meta = case.cache.export_tokens(case.pt_d, tb, tt)
        ec, em = expected_codes(case, b)
        np.testing.assert_array_equal(codes.cpu().numpy(), ec[:L], err_msg=f"codes seq {b}")
        np.testing.assert_array_equal(meta.cpu().numpy().view(np.uint16), em[:L].view(np.uint16),
                                      err_msg=f"meta seq {b}")
    assert case.cache.device_status() == 0
    out, lse = case.decode()
    assert case.cache.device_status() & DEV_SEQ_OVERFLOW
    ro, rl = case.oracle_seq(0)
    assert_close_out(out[0], lse[0], ro, rl, "sequence inside the table")


@pytest.mark.parametrize("lens", [[700, 300], [1, 1]])
def test_nonfinite_groups_are_flagged(lens):
    # A NaN in one RoPE group and an infinity in one content group give
    # non-finite (scale, min) metadata: MLAQ_DEV_NONFINITE, no fault, and
    # every other token is still stored bit-exact (bulk and one-CTA writers).
    from bit_mla_kv_gb300.mlaq import DEV_NONFINITE
    case = Case("C4R4", lens, 16, seed=53)
    a0, a1 = int(case.cu[0]) + lens[0] - 1, int(case.cu[1]) + lens[1] - 1   # last row of each sequence
    case.k[a0, 7] = float("nan")
    case.c[a1, 200] = float("inf")
    case.build()
    assert case.cache.device_status() & DEV_NONFINITE
    case.cache.clear_status()
    codes, meta = _export_all(case)
    off = 0
    for b, L in enumerate(case.seq_lens):
        if L > 1:
            tok = case.tokens(b)[:L - 1]   # the finite rows
            ec, em = O.quantize_tokens(tok[:, :512], tok[:, 512:], case.mode)
            np.testing.assert_array_equal(codes[off:off + L - 1], ec, err_msg=f"codes seq {b}")
            np.testing.assert_array_equal(meta[off:off + L - 1].view(np.uint16), em.view(np.uint16),
                                          err_msg=f"meta seq {b}")
        off += L
    assert case.cache.device_status() == 0


def _extreme_groups(n, ncols, rng):
    """Rows whose 64-channel groups stress the quantizer's edge cases: tiny
    values (fp16-subnormal scales and minima that round), constant and
    two-valued groups, large magnitudes and large offsets with small spread."""
    x = np.empty((n, ncols), np.float32)
    for g in range(ncols // 64):
        kind = rng.integers(0, 7, size=n)
        base = rng.standard_normal((n, 64)).astype(np.float32)
        sc = np.ones(n, np.float32)
        off = np.zeros(n, np.float32)
        sc[kind == 1] = 10.0 ** rng.uniform(-8, -5, size=(kind == 1).sum())
        off[kind == 2] = 10.0 ** rng.uniform(-6, -4.5, size=(kind == 2).sum())
        sc[kind == 2] = 10.0 ** rng.uniform(-8, -6, size=(kind == 2).sum())
        sc[kind == 5] = 10.0 ** rng.uniform(2, 3.8, size=(kind == 5).sum())
        off[kind == 6] = rng.choice([-1, 1], size=(kind == 6).sum()) * 10.0 ** rng.uniform(1, 4, size=(kind == 6).sum())
        sc[kind == 6] = 10.0 ** rng.uniform(-2, 1, size=(kind == 6).sum())
        blk = off[:, None] + sc[:, None] * base
        blk[kind == 3] = rng.standard_normal(((kind == 3).sum(), 1))  # constant: scale 0
        two = kind == 4
        a, b = rng.standard_normal(two.sum()), rng.standard_normal(two.sum())
        blk[two] = np.where(rng.random((two.sum(), 64)) < 0.5, a[:, None], b[:, None])
        x[:, 64 * g:64 * g + 64] = np.clip(blk, -60000, 60000)
    return x


@pytest.mark.parametrize("mode", ["C4R4", "C2R4"])
@pytest.mark.parametrize("lens", [[500, 200], [60, 40, 1, 100]])
def test_writer_extreme_groups_bit_exact(mode, lens):
    # 700 rows take the bulk writer, 201 rows the small-append kernel; both
    # must match the oracle's fp32 quantizer bit for bit on groups whose
    # codes leave [0, qmax] before clamping or whose scale is an fp16
    # subnormal or zero.
    case = Case(mode, lens, 16, seed=41)
    n = sum(lens)
    rng = np.random.default_rng(41)
    case.c = torch.from_numpy(_extreme_groups(n, 512, rng)).to(torch.bfloat16)
    case.k = torch.from_numpy(_extreme_groups(n, 64, rng)).to(torch.bfloat16)
    case.build()
    assert case.cache.device_status() == 0
    codes, meta = _export_all(case)
    ring = case.cache.ring_view().float().cpu().numpy()
    off = 0
    for b, L in enumerate(case.seq_lens):
        ec, em = expected_codes(case, b)
        np.testing.assert_array_equal(codes[off:off + L], ec, err_msg=f"codes seq {b}")
        np.testing.assert_array_equal(meta[off:off + L].view(np.uint16), em.view(np.uint16), err_msg=f"meta seq {b}")
        off += L
        er, valid = O.expected_ring(case.tokens(b), L)
        np.testing.assert_array_equal(ring[b][valid], er[valid], err_msg=f"ring seq {b}")


def test_writer_bf16_pages_hold_tokens():
    case = Case("BF16", [1, 64, 65, 300], 16, seed=12)
    case.build()
    pages = case.cache.bf16_pages_view().cpu()
    for b, L in enumerate(case.seq_lens):
        tok = torch.from_numpy(case.tokens(b))
        for t in range(L):
            p = int(case.page_table[b, t // 64])
            assert torch.equal(pages[p, t % 64].float(), tok[t]), (b, t)


@pytest.mark.parametrize("mode", ["C4R4", "C2R4", "BF16"])
def test_decode_tiny_workload(mode):
    wl = W.workload("tiny_c4r4")
    case = Case(mode, wl.seq_lens, wl.H, seed=wl.seed)
    case.build()
    out, lse = case.decode()
    for b in range(case.B):
        ro, rl = case.oracle_seq(b)
        assert_close_out(out[b], lse[b], ro, rl, f"{mode} seq {b}")
    assert case.cache.device_status() == 0


@pytest.mark.parametrize("mode", ["C4R4", "C2R4", "BF16"])
def test_decode_edge_lengths(mode):
    case = Case(mode, EDGE_LENS, 16, seed=13)
    case.build()
    out, lse = case.decode()
    for b, L in enumerate(case.seq_lens):
        ro, rl = case.oracle_seq(b)
        assert_close_out(out[b], lse[b], ro, rl, f"{mode} L={L}")


@pytest.mark.parametrize("mode,H", [("C4R4", 32), ("C4R4", 48), ("C4R4", 64), ("C4R4", 128), ("C2R4", 64),
                                    ("BF16", 64)])
def test_decode_more_heads(mode, H):
    # 32 heads per CTA when H is a multiple of 32 (one head block at H=32,
    # two at 64, four at 128), 16 otherwise (three blocks at H=48); forced
    # single-item and many-item splits exercise the final and partial epilogues.
    case = Case(mode, [5, 140, 777, 2048], H, seed=14)
    case.build()
    for ctas in (None, 1, 600):
        if ctas is not None:
            case.cache.set_decode_ctas(ctas)
        out, lse = case.decode()
        for b in range(case.B):
            ro, rl = case.oracle_seq(b)
            assert_close_out(out[b], lse[b], ro, rl, f"{mode} H={H} ctas={ctas} seq {b}")


@pytest.mark.parametrize("seed", range(8))
def test_random_append_schedules_bit_exact(seed):
    # Each sequence's tokens arrive in a random schedule of varlen appends
    # (zero, one or many rows per sequence per call: both the one-CTA-per-row
    # and the bulk writer, ring retirement, page edges); afterwards every
    # code, meta word and ring slot equals the oracle's for the whole
    # sequence, as if it had been appended at once.
    from bit_mla_kv_gb300.mlaq import Cache
    rng = np.random.default_rng(3000 + seed)
    mode = ["C4R4", "C2R4"][seed % 2]
    B = int(rng.integers(1, 16))
    ncalls = int(rng.integers(2, 6))
    counts = rng.integers(0, 400, size=(ncalls, B)) * (rng.random((ncalls, B)) < 0.8)
    counts[rng.random((ncalls, B)) < 0.2] = 1
    lens = [int(x) for x in counts.sum(0)]
    case = Case(mode, lens, 16, seed=4000 + seed)
    case.cache = Cache(mode, case.num_pages, case.B, case.page_table.shape[1], max_heads=16)
    case.pt_d = case.page_table.cuda()
    case.seq_d = torch.zeros(case.B, dtype=torch.int32, device="cuda")
    done = [0] * B
    for call in range(ncalls):
        cnt = [int(x) for x in counts[call]]
        if sum(cnt) == 0:
            continue
        rows = torch.cat([torch.arange(int(case.cu[b]) + done[b], int(case.cu[b]) + done[b] + cnt[b])
                          for b in range(B)])
        cu = torch.zeros(B + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(cnt), 0)
        case.cache.append(case.pt_d, case.seq_d, case.c[rows].cuda().contiguous(), case.k[rows].cuda().contiguous(),
                          cu_new=cu.cuda())
        done = [d + c for d, c in zip(done, cnt)]
    assert case.cache.device_status() == 0
    assert case.seq_d.cpu().tolist() == lens
    codes, meta = _export_all(case)
    ring = case.cache.ring_view().float().cpu().numpy()
    off = 0
    for b, L in enumerate(lens):
        if L == 0:
            continue
        ec, em = expected_codes(case, b)
        np.testing.assert_array_equal(codes[off:off + L], ec, err_msg=f"seed {seed} codes seq {b}")
        np.testing.assert_array_equal(meta[off:off + L].view(np.uint16), em.view(np.uint16),
                                      err_msg=f"seed {seed} meta seq {b}")
        off += L
        er, valid = O.expected_ring(case.tokens(b), L)
        np.testing.assert_array_equal(ring[b][valid], er[valid], err_msg=f"seed {seed} ring seq {b}")


@pytest.mark.parametrize("seed", range(24))
def test_random_batches_against_oracle(seed):
    # Seeded random batches: mode, head count (every blocking: 16-head and
    # 32-head CTAs), kernel variant, CTA count and a mix of empty, short,
    # ring-only, page-edge and longer sequences; every sequence is checked.
    rng = np.random.default_rng(1000 + seed)
    mode = ["C4R4", "C2R4", "BF16"][seed % 3]
    H = int(rng.choice([16, 32, 48, 64, 128]))
    B = int(rng.integers(1, 24))
    pool = [0, 1, 3, 4, 5, 63, 64, 65, 127, 131, 132, 133, 200, 256, 257, 700, 1000, 2049, 4097]
    lens = [int(rng.choice(pool)) if rng.random() < 0.7 else int(rng.integers(1, 6000)) for _ in range(B)]
    case = Case(mode, lens, H, seed=2000 + seed)
    case.build()
    ctas = [None, 1, int(rng.integers(2, 1025))][int(rng.integers(0, 3))]
    if ctas is not None:
        case.cache.set_decode_ctas(ctas)
    variant = int(rng.choice([0, 0, 2]))
    case.cache.set_decode_variant(variant)
    out, lse = case.decode()
    assert case.cache.device_status() == 0
    for b in range(case.B):
        ro, rl = case.oracle_seq(b)
        assert_close_out(out[b], lse[b], ro, rl, f"seed {seed} {mode} H={H} ctas={ctas} v={variant} seq {b} L={lens[b]}")


@pytest.mark.parametrize("mode,where", [("C4R4", "ring"), ("C4R4", "packed"), ("C2R4", "ring_small_append"),
                                        ("BF16", "page")])
def test_fp16_range_is_checked_for_tokens(mode, where):
    # A cached value beyond the fp16 range (a ring copy, a packed-only token,
    # a token of the all-BF16 cache; bulk and one-token appends) sets
    # MLAQ_DEV_RANGE in the writer; decoding the batch leaves the other
    # sequences exact.
    from bit_mla_kv_gb300.mlaq import DEV_RANGE
    lens = [300, 500, 700]
    case = Case(mode, [L + 1 for L in lens] if where == "ring_small_append" else lens, 16, seed=33)
    b_bad, t_bad = {"ring": (0, 299), "packed": (1, 100), "ring_small_append": (0, 300), "page": (1, 100)}[where]
    case.c[int(case.cu[b_bad]) + t_bad, 7] = 1e5
    if where == "ring_small_append":
        last = torch.tensor([int(case.cu[b + 1]) - 1 for b in range(case.B)])
        keep = torch.ones(int(case.cu[-1]), dtype=torch.bool)
        keep[last] = False
        full_c, full_k, full_cu = case.c, case.k, case.cu
        case.c, case.k = full_c[keep], full_k[keep]
        case.cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32)
        case.build()
        assert case.cache.device_status() == 0
        case.cache.append(case.pt_d, case.seq_d, full_c[last].view(case.B, 1, 512).cuda().contiguous(),
                          full_k[last].view(case.B, 1, 64).cuda().contiguous())
        case.c, case.k, case.cu = full_c, full_k, full_cu
    else:
        case.build()
    assert case.cache.device_status() & DEV_RANGE
    case.cache.clear_status()
    out, lse = case.decode()
    for b in range(case.B):
        if b != b_bad:
            ro, rl = case.oracle_seq(b)
            assert_close_out(out[b], lse[b], ro, rl, f"{mode} {where} seq {b}")


def test_fp16_range_is_checked_for_queries():
    from bit_mla_kv_gb300.mlaq import DEV_RANGE
    case = Case("C4R4", [300, 500, 700], 32, seed=34)
    case.ql[2, 21, 17] = 1e5   # one element of one head (in the second 16-head half)
    case.build()
    assert case.cache.device_status() == 0
    out, lse = case.decode()
    assert case.cache.device_status() & DEV_RANGE
    for b in (0, 1):
        ro, rl = case.oracle_seq(b)
        assert_close_out(out[b], lse[b], ro, rl, f"seq {b}")


def test_error_response_through_the_library():
    """The pages' error-response diagnosis (reading R8; ai.info "Methodology
    in Plain English" and "Main Findings": perturb one path's cache to NMSE
    0.01 and measure the output's NMSE per unit of cache NMSE), computed with
    the library: the perturbed tokens go through mlaq_append into an all-BF16
    cache, mlaq_decode runs on the clean and the perturbed cache, and the
    response is NMSE(out_perturbed, out_clean) / 0.01 over all heads. It must
    agree with the oracle's path_response within 3% (the cache and the outputs
    are rounded to bf16: about 0.4% per element, well under the 10%
    per-element perturbation)."""
    from bit_mla_kv_gb300.mlaq import Cache
    lens = [1024, 4096]
    base = Case("BF16", lens, 16, seed=5)
    rng = np.random.default_rng(5)
    for path, lo, hi in (("content", 0, 512), ("rope", 512, 576)):
        noises = [rng.standard_normal((L, hi - lo)) for L in lens]
        pert = base.c.float().clone(), base.k.float().clone()
        for b, L in enumerate(lens):
            a = int(base.cu[b])
            x = torch.cat([pert[0], pert[1]], -1)[a:a + L, lo:hi].double()
            n = torch.from_numpy(noises[b])
            d = n * torch.sqrt(0.01 * (x * x).sum() / (n * n).sum())   # ||d||^2 / ||x||^2 = 0.01
            if path == "content":
                pert[0][a:a + L] = (x + d).float()
            else:
                pert[1][a:a + L] = (x + d).float()
        outs = []
        for c, k in ((base.c, base.k), (pert[0].to(torch.bfloat16), pert[1].to(torch.bfloat16))):
            cache = Cache("BF16", base.num_pages, base.B, base.page_table.shape[1], max_heads=16)
            pt = base.page_table.cuda()
            seq = torch.zeros(base.B, dtype=torch.int32, device="cuda")
            cache.append(pt, seq, c.cuda().contiguous(), k.cuda().contiguous(), cu_new=base.cu.cuda())
            out, _ = cache.decode(base.ql.cuda().contiguous(), base.qr.cuda().contiguous(), pt, seq, base.scale)
            assert cache.device_status() == 0
            outs.append(out.double().cpu())
        for b, L in enumerate(lens):
            got = float(((outs[1][b] - outs[0][b]) ** 2).sum() / (outs[0][b] ** 2).sum()) / 0.01
            want = O.path_response(base.ql[b].float().numpy(), base.qr[b].float().numpy(), base.tokens(b),
                                   base.scale, path, noises[b])
            assert abs(got - want) <= 0.03 * want, (path, b, got, want)


@pytest.mark.parametrize("mode", ["C4R4", "C2R4", "BF16"])
def test_cache_bytes_matches_oracle(mode):
    """The library's persistent-cache accounting (mlaq_cache_bytes: BF16
    buffers + packed copies + page mapping, onedev.kr system-efficiency
    paragraph) equals the oracle's for single lengths and a mixed batch, and
    the C4R4 ratios sit within 2% of the pages' 3.22x (4K) and 3.59x (128K)."""
    import json
    import os
    from bit_mla_kv_gb300.mlaq import Cache
    cache = Cache(mode, 1, 16, 2048, max_heads=16)
    for lens in ([1], [132], [4096], [131072], [0, 1, 63, 64, 65, 132, 133, 4096, 131072, 7777]):
        assert cache.cache_bytes(lens) == O.cache_bytes(lens, mode), (mode, lens)
    if mode == "C4R4":
        g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "compression.json")))
        for L, published in g["ratios"].items():
            pol, ref = cache.cache_bytes([int(L)])
            assert abs(ref / pol - published) / published < 0.02, (L, ref / pol, published)


@pytest.mark.parametrize("H,lens", [(32, [32768, 30000]), (128, [20000] * 4)])
def test_decode_max_ctas_fills_partial_rows(H, lens):
    # 1024 decode CTAs over sequences long enough that the plan makes about
    # one item per CTA: the split partials reach the workspace's row bound
    # (items * H up to B * H + 32768 + H), which must hold them all.
    case = Case("C4R4", lens, H, seed=17)
    case.build()
    case.cache.set_decode_ctas(1024)
    out, lse = case.decode()
    assert case.cache.device_status() == 0
    for b in range(case.B):
        ro, rl = case.oracle_seq(b)
        assert_close_out(out[b], lse[b], ro, rl, f"H={H} seq {b}")


@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("mode,H", [("C4R4", 16), ("C4R4", 64), ("C4R4", 128), ("C2R4", 32), ("C2R4", 128),
                                    ("BF16", 48), ("BF16", 64)])
def test_decode_kernel_variants(mode, H, variant):
    # Both attention kernels on every head blocking: register scores
    # (variant 1) and tcgen05 scores (variant 2, 64 / 32 / 16 heads per CTA),
    # with the default, a single and many splits per sequence.
    case = Case(mode, [5, 140, 777, 2048, 4097], H, seed=51)
    case.build()
    case.cache.set_decode_variant(variant)
    for ctas in (None, 1, 600):
        if ctas is not None:
            case.cache.set_decode_ctas(ctas)
        out, lse = case.decode()
        assert case.cache.device_status() == 0
        for b in range(case.B):
            ro, rl = case.oracle_seq(b)
            assert_close_out(out[b], lse[b], ro, rl, f"{mode} H={H} variant {variant} ctas={ctas} seq {b}")


@pytest.mark.parametrize("mode,Q,H,variant", [("C4R4", 2, 16, 0), ("C4R4", 4, 16, 0), ("C2R4", 2, 32, 0),
                                              ("BF16", 3, 16, 0), ("C4R4", 4, 16, 2), ("C4R4", 2, 64, 0),
                                              ("C2R4", 2, 32, 2), ("BF16", 3, 16, 2)])
def test_decode_multi_token_causal(mode, Q, H, variant):
    # Q query tokens per sequence after their Q tokens were appended: query j
    # sees t < L - (Q - 1 - j). The lengths put the hidden tokens among the
    # sink slots (L <= 6), the recent ring and, in BF16 mode, the last page.
    case = Case(mode, [1, 2, 3, 6, 133, 140, 700, 3000], H, seed=40 + Q)
    case.build(max_heads=Q * H)
    case.cache.set_decode_variant(variant)
    ql, qr = W.make_queries(case.B, Q * H, W.generator(90 + Q, "cpu"), "cpu")
    ql = ql.view(case.B, Q, H, 512).contiguous()
    qr = qr.view(case.B, Q, H, 64).contiguous()
    for ctas in (None, 1, 600):
        if ctas is not None:
            case.cache.set_decode_ctas(ctas)
        out, lse = case.cache.decode_mtp(ql.cuda(), qr.cuda(), case.pt_d, case.seq_d, case.scale)
        assert case.cache.device_status() == 0
        for b, L in enumerate(case.seq_lens):
            tok = case.tokens(b)
            codes = meta = None
            if mode != "BF16":
                codes, meta = O.quantize_tokens(tok[:, :512], tok[:, 512:], mode)
            for j in range(Q):
                ro, rl = O.decode_sequence(ql[b, j].float().numpy(), qr[b, j].float().numpy(), tok, codes, meta, L,
                                           case.scale, mode, n_attend=L - (Q - 1 - j))
                assert_close_out(out[b, j], lse[b, j], ro, rl, f"{mode} Q={Q} ctas={ctas} seq {b} query {j}")


@pytest.mark.parametrize("mode,H,variant", [("C4R4", 16, 0), ("C2R4", 16, 0), ("BF16", 16, 0), ("C4R4", 64, 2),
                                            ("C2R4", 16, 2), ("BF16", 64, 2)])
def test_decode_running_max_rescale(mode, H, variant):
    # Later tokens carry larger latents, so the running max of every head
    # rises by far more than the lazy-rescale threshold partway through each
    # sequence: the accumulated output (TMEM or registers) must be rescaled
    # mid-item, in full-page and 16-token steps and across splits.
    case = Case(mode, [700, 3000, 5000], H, seed=22)
    for b, L in enumerate(case.seq_lens):
        a = int(case.cu[b])
        for lo, f in ((L // 3, 3.0), (2 * L // 3, 6.0)):
            case.c[a + lo:a + L] = (case.c[a + lo:a + L].float() * f).to(torch.bfloat16)
    case.build()
    case.cache.set_decode_variant(variant)
    for ctas in (1, 300):
        case.cache.set_decode_ctas(ctas)
        out, lse = case.decode()
        for b in range(case.B):
            ro, rl = case.oracle_seq(b)
            assert_close_out(out[b], lse[b], ro, rl, f"{mode} H={H} variant {variant} ctas={ctas} seq {b}")


@pytest.mark.parametrize("costs", [(8, 19, 40), (1, 50, 0), (8, 1, 500), (3, 7, 100)])
def test_plan_costs_change_only_the_split(costs):
    # The planner's costs move the CTA boundaries (and so the split points and
    # the combine), never the result; out-of-range costs are refused.
    case = Case("C4R4", [700, 1500, 3000, 133, 65], 16, seed=21)
    case.build()
    from bit_mla_kv_gb300.mlaq import MlaqError
    with pytest.raises(MlaqError):
        case.cache.set_plan_costs(9, 19, 40)   # 4 * step > 32
    with pytest.raises(MlaqError):
        case.cache.set_plan_costs(8, 60, 0)    # item + 9 * ring > 512
    case.cache.set_plan_costs(*costs)
    out, lse = case.decode()
    for b in range(case.B):
        ro, rl = case.oracle_seq(b)
        assert_close_out(out[b], lse[b], ro, rl, f"costs {costs} seq {b}")


@pytest.mark.parametrize("B", [1000, 1100])
def test_many_short_sequences_plan(B):
    # Many short and empty sequences (around and above a thousand) put many
    # items and empty sequences in one CTA range; forced CTA counts move every
    # boundary. Empty sequences give out = 0 and lse = -inf.
    rng = np.random.default_rng(40 + B)
    lens = rng.choice([0, 0, 1, 3, 4, 5, 64, 65, 131, 132, 133, 200, 333], size=B)
    lens[:3] = 0        # empty sequences first
    lens[-2:] = 0       # and last
    case = Case("C4R4", lens, 16, seed=41)
    case.build()
    check = sorted(set(rng.choice(B, size=40, replace=False).tolist()) | {0, 3, B - 3, B - 1})
    for ctas in (None, 7, 600):
        if ctas is not None:
            case.cache.set_decode_ctas(ctas)
        out, lse = case.decode()
        assert case.cache.device_status() == 0
        empty = torch.tensor(lens == 0, device=out.device)
        assert torch.all(out[empty] == 0) and torch.all(torch.isneginf(lse[empty]))
        for b in check:
            if lens[b] == 0:
                continue
            ro, rl = case.oracle_seq(b)
            assert_close_out(out[b], lse[b], ro, rl, f"B={B} ctas={ctas} seq {b} L={lens[b]}")


def test_split_invariance():
    case = Case("C4R4", [3000, 9000, 133, 640], 16, seed=15)
    case.build()
    case.cache.set_decode_ctas(1)
    o1, l1 = case.decode()
    o1, l1 = o1.clone(), l1.clone()
    case.cache.set_decode_ctas(600)
    o2, l2 = case.decode()
    for b in range(case.B):
        ro, rl = case.oracle_seq(b)
        assert_close_out(o1[b], l1[b], ro, rl, f"1 split seq {b}")
        assert_close_out(o2[b], l2[b], ro, rl, f"many splits seq {b}")
    assert torch.allclose(l1, l2, atol=1e-4)


def test_incremental_append_retires_without_requant():
    # Append one token per step across the sink/recent boundary; every
    # token's stored codes equal the bulk quantization (no re-quantization),
    # and decode matches the oracle at several lengths.
    L0 = [100, 130, 2000]
    steps = 40
    case = Case("C4R4", [L + steps for L in L0], 16, seed=16)
    from bit_mla_kv_gb300.mlaq import Cache
    cache = Cache("C4R4", case.num_pages, case.B, case.page_table.shape[1], max_heads=16)
    case.cache = cache
    case.pt_d = case.page_table.cuda()
    case.seq_d = torch.zeros(case.B, dtype=torch.int32, device="cuda")
    # prefill the first L0 tokens of each sequence
    cu0 = torch.zeros(case.B + 1, dtype=torch.int32)
    cu0[1:] = torch.cumsum(torch.tensor(L0), 0)
    rows = torch.cat([torch.arange(int(case.cu[b]), int(case.cu[b]) + L0[b]) for b in range(case.B)])
    cache.append(case.pt_d, case.seq_d, case.c[rows].cuda().contiguous(), case.k[rows].cuda().contiguous(),
                 cu_new=cu0.cuda())
    for s in range(steps):
        rows = torch.tensor([int(case.cu[b]) + L0[b] + s for b in range(case.B)])
        cache.append(case.pt_d, case.seq_d, case.c[rows].view(case.B, 1, 512).cuda().contiguous(),
                     case.k[rows].view(case.B, 1, 64).cuda().contiguous())
        if s in (0, 2, 31, 39):
            out, lse = case.decode()
            for b in range(case.B):
                ro, rl = case.oracle_seq(b, L=L0[b] + s + 1)
                assert_close_out(out[b], lse[b], ro, rl, f"step {s} seq {b}")
    assert case.seq_d.cpu().tolist() == case.seq_lens
    codes, meta = _export_all(case)
    off = 0
    for b, L in enumerate(case.seq_lens):
        ec, em = expected_codes(case, b)
        np.testing.assert_array_equal(codes[off:off + L], ec)
        np.testing.assert_array_equal(meta[off:off + L].view(np.uint16), em.view(np.uint16))
        off += L


def test_device_status_reports_bad_page_without_fault():
    case = Case("C4R4", [500, 700], 16, seed=17)
    case.build()
    bad = case.page_table.clone()
    bad[1, 3] = case.num_pages + 5   # outside the pool: masked out by the kernel's bounds check
    out, lse = case.cache.decode(case.ql.cuda(), case.qr.cuda(), bad.cuda(), case.seq_d, case.scale)
    st = case.cache.device_status()
    assert st & 0x1
    ro, rl = case.oracle_seq(0)
    assert_close_out(out[0], lse[0], ro, rl, "untouched sequence")
    assert torch.isfinite(out[1].float()).all()
    case.cache.clear_status()
    assert case.cache.device_status() == 0


def test_bounded_wait_runs_out_and_reports_status():
    # A wait on an mbarrier that nothing completes ends after its limit with
    # the timeout status (no trap, no hang), and the context stays usable.
    import time
    from bit_mla_kv_gb300.mlaq import DEV_TIMEOUT, debug_wait_probe
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    debug_wait_probe(st, 5000, arrive=False)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert int(st.item()) == DEV_TIMEOUT
    assert waited >= 0.004  # the 5 ms limit, measured on the device timer
    st.fill_(-1)
    debug_wait_probe(st, 5000, arrive=True)
    assert int(st.item()) == 0
    case = Case("C4R4", [700], 16, seed=3)
    case.build()
    out, lse = case.decode()
    ro, rl = case.oracle_seq(0)
    assert_close_out(out[0], lse[0], ro, rl, "decode after a timed-out wait")
    assert case.cache.device_status() == 0


@pytest.mark.parametrize("name,sample", [("v2lite_c4r4", [0, 7, 19, 31]), ("v2lite_c2r4", [3, 30]),
                                         ("v2lite_bf16", [5]), ("v3_c4r4", [0, 63]),
                                         ("long_c2r4", [2]), ("long_c4r4", [1]), ("long_bf16", [3])])
def test_full_size_sampled(name, sample):
    """Full workload sizes in the benchmark's launch configuration (the whole
    workload through the bulk writer in one varlen call, then one decode); the
    oracle checks whole sampled sequences: every code and meta word bit for
    bit, and the decode output."""
    wl = W.workload(name)
    case = Case(wl.mode, wl.seq_lens, wl.H, seed=wl.seed, gen_device="cuda")
    case.build()
    out, lse = case.decode()
    assert case.cache.device_status() == 0
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    for b in sample:
        ro, rl = case.oracle_seq(b)
        assert_close_out(out[b], lse[b], ro, rl, f"{name} seq {b}")
        if wl.mode == "BF16":
            continue
        L = case.seq_lens[b]
        tb = torch.full((L,), b, dtype=torch.int32, device="cuda")
        tt = torch.arange(L, dtype=torch.int32, device="cuda")
        codes, meta = case.cache.export_tokens(case.pt_d, tb, tt)
        ec, em = expected_codes(case, b)
        np.testing.assert_array_equal(codes.cpu().numpy(), ec, err_msg=f"{name} codes seq {b}")
        np.testing.assert_array_equal(meta.cpu().numpy().view(np.uint16), em.view(np.uint16),
                                      err_msg=f"{name} meta seq {b}")


@pytest.mark.parametrize("mode", ["C4R4", "BF16"])
def test_many_short_sequences(mode):
    """A large batch of short and empty sequences: the planner's multi-pass
    scans, CTAs that hold many whole sequences, and sequences split across CTA
    boundaries all at once; every sequence is checked."""
    rng = np.random.default_rng(23)
    lens = [int(x) for x in rng.choice([0, 1, 4, 5, 64, 65, 131, 133, 200, 300, 700], size=3000)]
    case = Case(mode, lens, 16, seed=23, gen_device="cuda")
    case.build()
    out, lse = case.decode()
    assert case.cache.device_status() == 0
    for b in range(case.B):
        ro, rl = case.oracle_seq(b)
        assert_close_out(out[b], lse[b], ro, rl, f"{mode} seq {b} L={lens[b]}")


def test_serving_loop_sampled():
    """Serving loop at full size: B=128, H=16, L0~U[2K,16K], 256 steps of
    mlaq_append (one token per sequence) + mlaq_decode. Appended codes are
    checked bit-exactly at steps {0,1,127,128,255}; decode outputs of sampled
    sequences at steps {0,128,255} against the oracle."""
    wl = W.workload("serving_c4r4")
    steps = wl.steps
    final = [L + steps for L in wl.seq_lens]
    case = Case("C4R4", final, wl.H, seed=wl.seed, gen_device="cuda")
    from bit_mla_kv_gb300.mlaq import Cache
    cache = Cache("C4R4", case.num_pages, case.B, case.page_table.shape[1], max_heads=16)
    case.cache = cache
    case.pt_d = case.page_table.cuda()
    case.seq_d = torch.zeros(case.B, dtype=torch.int32, device="cuda")
    cu = case.cu.long()
    first = torch.cat([torch.arange(int(cu[b]), int(cu[b]) + wl.seq_lens[b]) for b in range(case.B)]).cuda()
    cu0 = torch.zeros(case.B + 1, dtype=torch.int32)
    cu0[1:] = torch.cumsum(torch.tensor(wl.seq_lens), 0)
    cache.append(case.pt_d, case.seq_d, case.c[first].contiguous(), case.k[first].contiguous(), cu_new=cu0.cuda())
    sample_b = [0, 37, 127]
    for s in range(steps):
        rows = torch.tensor([int(cu[b]) + wl.seq_lens[b] + s for b in range(case.B)], device="cuda")
        cache.append(case.pt_d, case.seq_d, case.c[rows].view(case.B, 1, 512).contiguous(),
                     case.k[rows].view(case.B, 1, 64).contiguous())
        if s in (0, 1, 127, 128, 255):
            tb = torch.arange(case.B, dtype=torch.int32, device="cuda")
            tt = torch.tensor([wl.seq_lens[b] + s for b in range(case.B)], dtype=torch.int32, device="cuda")
            codes, meta = cache.export_tokens(case.pt_d, tb, tt)
            tok = torch.cat([case.c[rows], case.k[rows]], -1).float().cpu().numpy()
            ec, em = O.quantize_tokens(tok[:, :512], tok[:, 512:], "C4R4")
            np.testing.assert_array_equal(codes.cpu().numpy(), ec, err_msg=f"step {s}")
            np.testing.assert_array_equal(meta.cpu().numpy().view(np.uint16), em.view(np.uint16))
        if s in (0, 128, 255):
            out, lse = case.decode()
            for b in sample_b:
                ro, rl = case.oracle_seq(b, L=wl.seq_lens[b] + s + 1)
                assert_close_out(out[b], lse[b], ro, rl, f"step {s} seq {b}")
    assert case.seq_d.cpu().tolist() == final
    assert cache.device_status() == 0


def test_cuda_graph_capture_of_append_decode():
    """One serving step (append + decode) captured in a CUDA graph and replayed
    gives the same results as eager execution."""
    case = Case("C4R4", [700, 1500, 3000], 16, seed=18, extra_capacity=64)
    case.build()
    dev = "cuda"
    ql, qr = case.ql.to(dev).contiguous(), case.qr.to(dev).contiguous()
    g = W.generator(99, dev)
    newc, newk = W.make_tokens(case.B * 8, case.stats, g, dev)
    newc, newk = newc.view(8, case.B, 1, 512), newk.view(8, case.B, 1, 64)
    # eager reference on a copy of the cache state
    ref_cache = Case("C4R4", [700, 1500, 3000], 16, seed=18, extra_capacity=64)
    ref_cache.build()
    outs_ref = []
    for s in range(8):
        ref_cache.cache.append(ref_cache.pt_d, ref_cache.seq_d, newc[s].contiguous(), newk[s].contiguous())
        o, l = ref_cache.cache.decode(ql, qr, ref_cache.pt_d, ref_cache.seq_d, case.scale)
        outs_ref.append((o.clone(), l.clone()))
    # graph: static input buffers
    bc = torch.empty_like(newc[0])
    bk = torch.empty_like(newk[0])
    out = torch.empty(case.B, 16, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(case.B, 16, dtype=torch.float32, device=dev)
    # warm the attribute setting outside capture
    s0 = torch.cuda.Stream()
    s0.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s0):
        case.cache.decode(ql, qr, case.pt_d, case.seq_d, case.scale, out=out, lse=lse)
    torch.cuda.current_stream().wait_stream(s0)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        case.cache.append(case.pt_d, case.seq_d, bc, bk)
        case.cache.decode(ql, qr, case.pt_d, case.seq_d, case.scale, out=out, lse=lse)
    for s in range(8):
        bc.copy_(newc[s])
        bk.copy_(newk[s])
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, outs_ref[s][0]), s
        assert torch.equal(lse, outs_ref[s][1]), s
    assert case.seq_d.cpu().tolist() == ref_cache.seq_d.cpu().tolist()
