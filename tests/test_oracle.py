"""Pins of the CPU oracle to facts other than itself (CPU only).

Each test checks the oracle against a closed form, a brute-force search, an
independent library routine, an invariant, or a number printed on the pages.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(x):
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def _rand_groups(n, seed, outliers=True):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, 64)).astype(np.float32)
    if outliers:
        x[:, rng.integers(0, 64, 3)] *= 10
    x[n // 2:] *= rng.uniform(1e-3, 30, size=(n - n // 2, 1)).astype(np.float32)
    return _bf16(x)


# ---------------------------------------------------------------- quantizer

@pytest.mark.parametrize("bits", [2, 4])
def test_quantizer_integer_ramp_is_identity(bits):
    # values 0..qmax repeated: min 0, max qmax, scale exactly 1 -> codes = values
    qmax = 2 ** bits - 1
    x = np.tile(np.arange(qmax + 1, dtype=np.float32), 64 // (qmax + 1))[None]
    q, s, m = O.quantize_groups(x, bits)
    assert float(s[0]) == 1.0 and float(m[0]) == 0.0
    np.testing.assert_array_equal(q[0], x[0].astype(np.uint8))


@pytest.mark.parametrize("bits", [2, 4])
def test_quantizer_shifted_scaled_ramp(bits):
    # x = -3 + 0.25*k for k in codes: exactly representable, codes recovered
    qmax = 2 ** bits - 1
    rng = np.random.default_rng(5)
    k = rng.integers(0, qmax + 1, 64)
    k[0], k[1] = 0, qmax
    x = (-3.0 + 0.25 * k).astype(np.float32)[None]
    q, s, m = O.quantize_groups(x, bits)
    assert float(s[0]) == 0.25 and float(m[0]) == -3.0
    np.testing.assert_array_equal(q[0], k)


@pytest.mark.parametrize("bits", [2, 4])
def test_quantizer_constant_group(bits):
    x = np.full((1, 64), 1.234375, dtype=np.float32)
    q, s, m = O.quantize_groups(x, bits)
    assert float(s[0]) == 0.0
    assert np.all(q == 0)
    deq = O.dequantize_tokens(np.zeros((1, 576), np.uint8),
                              np.stack([np.zeros(9, np.float16), np.full(9, m[0])], -1)[None])
    assert np.all(deq == float(np.float16(1.234375)))


@pytest.mark.parametrize("bits", [2, 4])
def test_quantizer_two_valued_group_hits_both_ends(bits):
    x = np.where(np.arange(64) % 3 == 0, -0.75, 2.5).astype(np.float32)[None]
    q, s, m = O.quantize_groups(x, bits)
    np.testing.assert_array_equal(q[0], np.where(np.arange(64) % 3 == 0, 0, 2 ** bits - 1))


@pytest.mark.parametrize("bits", [2, 4])
def test_quantizer_brute_force_nearest_level(bits):
    # Every code is the nearest of the 2^b levels q*s+m (fp64), except at
    # near-ties where fp32 rounding of the quotient may pick either neighbour.
    x = _rand_groups(400, 11 + bits)
    q, s, m = O.quantize_groups(x, bits)
    levels = np.arange(2 ** bits)[None, None, :] * s.astype(np.float64)[:, None, None] \
        + m.astype(np.float64)[:, None, None]
    dist = np.abs(x.astype(np.float64)[..., None] - levels)
    best = dist.argmin(-1)
    srt = np.sort(dist, -1)
    near_tie = (srt[..., 1] - srt[..., 0]) <= 1e-5 * s.astype(np.float64)[:, None] + 1e-12
    mism = (best != q) & ~near_tie
    assert not mism.any(), np.argwhere(mism)[:5]
    # and the chosen level is never farther than the best by more than a tie
    chosen = np.take_along_axis(dist, q[..., None].astype(np.int64), -1)[..., 0]
    assert np.all(chosen <= srt[..., 0] + 1e-5 * s.astype(np.float64)[:, None] + 1e-12)


@pytest.mark.parametrize("mode", ["C4R4", "C2R4"])
def test_dequant_error_bound(mode):
    # Whole 576-channel tokens through quantize_tokens and dequantize_tokens:
    # |x - c_hat| <= s/2 per element, widened by the fp16 rounding of the
    # stored meta (ai.info "Methodology in Plain English": asymmetric affine
    # quantizer, group 64).
    n = 300
    x = _rand_groups(9 * n, 23 + len(mode)).reshape(n, 576)
    codes, meta = O.quantize_tokens(x[:, :512], x[:, 512:], mode)
    deq = O.dequantize_tokens(codes, meta)
    bc, br = O.mode_bits(mode)
    qmax = np.array([2 ** bc - 1] * 8 + [2 ** br - 1], np.float64)      # per group
    xg = x.astype(np.float64).reshape(n, 9, 64)
    s = meta[..., 0].astype(np.float64)
    m = meta[..., 1].astype(np.float64)
    s32 = (xg.max(-1) - xg.min(-1)) / qmax
    err = np.abs(deq.reshape(n, 9, 64) - xg)
    bound = 0.5 * s + qmax * np.abs(s32 - s) + np.abs(xg.min(-1) - m) + 1e-6 * np.abs(xg).max(-1)
    assert np.all(err <= bound[..., None])
    # without the meta rounding slack the plain s/2 bound holds for most groups
    assert np.mean(err <= 0.5 * s[..., None] + 1e-9) > 0.99


def test_dequantize_tokens_hand_written():
    # Two tokens whose nine groups carry distinct metadata: token 0, group g
    # has s = 2^-g, min = g - 4 and codes j mod 16 (j = channel within the
    # group); token 1 reverses both (s = 2^-(8-g), min = 4 - g, codes 15 - j
    # mod 16). A group- or token-axis mix-up, a swapped (scale, min) or a
    # dropped min changes the values below.
    j = np.arange(64)
    codes = np.stack([np.tile(j % 16, 9), np.tile(15 - j % 16, 9)]).astype(np.uint8)
    meta = np.zeros((2, 9, 2), np.float16)
    for g in range(9):
        meta[0, g] = (2.0 ** -g, g - 4)
        meta[1, g] = (2.0 ** -(8 - g), 4 - g)
    deq = O.dequantize_tokens(codes, meta)
    assert deq.shape == (2, 576) and deq.dtype == np.float64
    # values written out by hand: (token, channel) -> q * s + min
    written = {(0, 0): -4.0, (0, 5): 1.0, (0, 67): -1.5, (0, 130): -1.5, (0, 511): 3.1171875,
               (0, 527): 4.05859375, (0, 575): 4.05859375, (0, 448): 3.0, (0, 463): 3.1171875,
               (1, 0): 4.05859375, (1, 15): 4.0, (1, 64): 3.1171875, (1, 79): 3.0,
               (1, 512): 11.0, (1, 527): -4.0, (1, 448): 4.5}
    for (t, c), v in written.items():
        assert deq[t, c] == v, (t, c, deq[t, c], v)
    # every element, group by group
    for t in range(2):
        for g in range(9):
            sc = 2.0 ** -g if t == 0 else 2.0 ** -(8 - g)
            mn = g - 4.0 if t == 0 else 4.0 - g
            for jj in range(64):
                qq = jj % 16 if t == 0 else 15 - jj % 16
                assert deq[t, 64 * g + jj] == qq * sc + mn


def test_quantize_tokens_group_layout_and_modes():
    rng = np.random.default_rng(3)
    c = _bf16(rng.standard_normal((5, 512)))
    k = _bf16(rng.standard_normal((5, 64)) * 3)
    for mode in ("C4R4", "C2R4"):
        codes, meta = O.quantize_tokens(c, k, mode)
        assert codes.shape == (5, 576) and meta.shape == (5, 9, 2)
        bc, br = O.mode_bits(mode)
        assert codes[:, :512].max() <= 2 ** bc - 1 and codes[:, 512:].max() <= 2 ** br - 1
        # group g of the content is channels [64g, 64g+64); RoPE is group 8
        for g in range(8):
            qg, sg, mg = O.quantize_groups(c[:, 64 * g:64 * g + 64], bc)
            np.testing.assert_array_equal(codes[:, 64 * g:64 * g + 64], qg)
            np.testing.assert_array_equal(meta[:, g, 0], sg)
            np.testing.assert_array_equal(meta[:, g, 1], mg)
        assert np.all(meta[:, 8, 1] == k.min(-1).astype(np.float16))
        # the RoPE group uses the RoPE width (4 bits in both modes), not the content width
        assert br == 4
        qr, sr, mr = O.quantize_groups(k, br)
        np.testing.assert_array_equal(codes[:, 512:], qr)
        np.testing.assert_array_equal(meta[:, 8, 0], sr)
        np.testing.assert_array_equal(meta[:, 8, 1], mr)


def test_quantization_is_per_token_no_requant():
    # A token's codes do not depend on which other tokens are quantized with
    # it, nor on when it was appended: bulk == one at a time.
    rng = np.random.default_rng(9)
    c = _bf16(rng.standard_normal((40, 512)) * 2)
    k = _bf16(rng.standard_normal((40, 64)))
    bulk_codes, bulk_meta = O.quantize_tokens(c, k, "C4R4")
    for t in range(40):
        ct, mt = O.quantize_tokens(c[t:t + 1], k[t:t + 1], "C4R4")
        np.testing.assert_array_equal(ct[0], bulk_codes[t])
        np.testing.assert_array_equal(mt[0], bulk_meta[t])


# ---------------------------------------------------------------- packing

@pytest.mark.parametrize("mode", ["C4R4", "C2R4"])
def test_pack_roundtrip_all_bytes(mode):
    # every byte value survives unpack -> pack
    nb = O.packed_bytes_per_token(mode)
    assert nb == (288 if mode == "C4R4" else 160)
    allb = np.arange(256, dtype=np.uint8)
    packed = np.resize(allb, (3, nb))
    packed[1] = np.roll(packed[1], 7)
    np.testing.assert_array_equal(O.pack_canonical(O.unpack_canonical(packed, mode), mode), packed)


def test_pack_known_bytes():
    codes = np.zeros(576, np.uint8)
    codes[0], codes[1] = 1, 2           # INT4: code 0 low nibble, code 1 high nibble
    codes[512], codes[513] = 15, 3      # RoPE INT4 after the content bytes
    p = O.pack_canonical(codes, "C4R4")
    assert p[0] == 0x21 and p[256] == 0x3F
    codes2 = np.zeros(576, np.uint8)
    codes2[:4] = [1, 2, 3, 0]           # INT2: 4 codes per byte, code i at bits 2i
    p2 = O.pack_canonical(codes2, "C2R4")
    assert p2[0] == 0b00111001 and p2.shape == (160,)


# ---------------------------------------------------------------- selection

def test_selection_rule_exhaustive():
    for L in range(0, 301):
        mask = O.bf16_token_mask(L)
        assert mask.sum() == min(L, 132)
        for t in range(L):
            assert mask[t] == ((t < 4) or (t >= L - 128)) == O.is_bf16_token(t, L)


def test_ring_holds_exactly_the_bf16_tokens():
    tok = np.arange(400, dtype=np.float32)[:, None] * np.ones((1, 576), np.float32)
    for L in list(range(0, 140)) + [200, 255, 256, 257, 399, 400]:
        ring, valid = O.expected_ring(tok, L)
        held = sorted(int(ring[j, 0]) for j in range(132) if valid[j])
        want = [t for t in range(L) if O.is_bf16_token(t, L)]
        assert held == want, L


def test_ring_incremental_writer_matches():
    # appending one token at a time into slot (t if t<4 else 4 + t%128)
    # reproduces expected_ring at every length: retirement = overwrite
    tok = np.random.default_rng(1).standard_normal((300, 576)).astype(np.float32)
    ring = np.zeros((132, 576), np.float32)
    for L in range(1, 301):
        t = L - 1
        ring[t if t < 4 else 4 + t % 128] = tok[t]
        exp, valid = O.expected_ring(tok, L)
        np.testing.assert_array_equal(ring[valid], exp[valid])


# ---------------------------------------------------------------- attention

def _torch_reference(q_lat, q_rope, kv, scale):
    q = torch.tensor(np.concatenate([q_lat, q_rope], -1), dtype=torch.float64)[None, :, None, :]
    k = torch.tensor(kv, dtype=torch.float64)[None, None].expand(1, q.shape[1], -1, -1)
    v = torch.tensor(kv[:, :512], dtype=torch.float64)[None, None].expand(1, q.shape[1], -1, -1)
    out = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=scale)[0, :, 0]
    z = torch.einsum("hd,ld->hl", q[0, :, 0], k[0, 0]) * scale
    lse = torch.logsumexp(z, dim=-1)
    return out.numpy(), lse.numpy()


def test_attend_all_bf16_equals_sdpa():
    rng = np.random.default_rng(0)
    H, L = 16, 300
    ql = _bf16(rng.standard_normal((H, 512)))
    qr = _bf16(rng.standard_normal((H, 64)))
    kv = _bf16(rng.standard_normal((L, 576)))
    out, lse = O.decode_sequence(ql, qr, kv, None, None, L, 1 / math.sqrt(192), "BF16")
    ref_out, ref_lse = _torch_reference(ql, qr, kv.astype(np.float64), 1 / math.sqrt(192))
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_attend_tiny_bruteforce_no_max_subtraction():
    rng = np.random.default_rng(2)
    for L in range(1, 9):
        ql = rng.standard_normal((3, 512)) * 0.05
        qr = rng.standard_normal((3, 64)) * 0.05
        kv = rng.standard_normal((L, 576))
        out, lse = O.attend(ql, qr, kv, 0.5)
        for h in range(3):
            z = [0.5 * (math.fsum(ql[h, i] * kv[t, i] for i in range(512))
                        + math.fsum(qr[h, j] * kv[t, 512 + j] for j in range(64))) for t in range(L)]
            e = [math.exp(v) for v in z]
            tot = math.fsum(e)
            assert abs(lse[h] - math.log(tot)) < 1e-12
            o = [math.fsum(e[t] * kv[t, c] for t in range(L)) / tot for c in range(512)]
            np.testing.assert_allclose(out[h], o, rtol=0, atol=1e-12)


def test_attend_empty_sequence():
    out, lse = O.attend(np.ones((4, 512)), np.ones((4, 64)), np.zeros((0, 576)), 0.1)
    assert np.all(out == 0) and np.all(lse == -np.inf)


def test_split_combine_invariance():
    rng = np.random.default_rng(4)
    H, L = 8, 257
    ql, qr = rng.standard_normal((H, 512)), rng.standard_normal((H, 64))
    kv = rng.standard_normal((L, 576)) * 2
    full_out, full_lse = O.attend(ql, qr, kv, 0.2)
    for cuts in ([0, 257], [0, 1, 257], [0, 64, 128, 200, 257], sorted({0, 257, *rng.integers(1, 257, 6)})):
        parts = [O.attend(ql, qr, kv[a:b], 0.2) for a, b in zip(cuts[:-1], cuts[1:])]
        out, lse = O.combine_partials([p[0] for p in parts], [p[1] for p in parts])
        np.testing.assert_allclose(out, full_out, atol=1e-12)
        np.testing.assert_allclose(lse, full_lse, atol=1e-12)
    # an empty partial (-inf lse, zero out) changes nothing
    out, lse = O.combine_partials([full_out, np.zeros_like(full_out)], [full_lse, np.full(H, -np.inf)])
    np.testing.assert_allclose(out, full_out, atol=1e-15)


def test_decode_uses_exactly_one_representation():
    # Changing the packed copy of a protected token, or the BF16 copy of an
    # unprotected one, must not change the result; the other way round must.
    rng = np.random.default_rng(6)
    L, H = 400, 4
    c = _bf16(rng.standard_normal((L, 512)))
    k = _bf16(rng.standard_normal((L, 64)))
    tok = np.concatenate([c, k], -1)
    codes, meta = O.quantize_tokens(c, k, "C4R4")
    ql, qr = rng.standard_normal((H, 512)), rng.standard_normal((H, 64))
    base = O.decode_sequence(ql, qr, tok, codes, meta, L, 0.1, "C4R4")
    for t, protected in ((0, True), (3, True), (4, False), (271, False), (272, True), (399, True)):
        c2, t2 = codes.copy(), tok.copy()
        c2[t] = 15 - c2[t]
        t2[t] = -t2[t] + 1
        a = O.decode_sequence(ql, qr, tok, c2, meta, L, 0.1, "C4R4")
        b = O.decode_sequence(ql, qr, t2, codes, meta, L, 0.1, "C4R4")
        if protected:
            assert np.array_equal(a[0], base[0]) and not np.allclose(b[0], base[0])
        else:
            assert np.array_equal(b[0], base[0]) and not np.allclose(a[0], base[0])


def test_short_sequence_is_all_bf16():
    rng = np.random.default_rng(8)
    L = 132
    c = _bf16(rng.standard_normal((L, 512)))
    k = _bf16(rng.standard_normal((L, 64)))
    tok = np.concatenate([c, k], -1)
    codes, meta = O.quantize_tokens(c, k, "C2R4")
    ql, qr = rng.standard_normal((2, 512)), rng.standard_normal((2, 64))
    a = O.decode_sequence(ql, qr, tok, codes, meta, L, 0.1, "C2R4")
    b = O.decode_sequence(ql, qr, tok, None, None, L, 0.1, "BF16")
    np.testing.assert_array_equal(a[0], b[0])


# ---------------------------------------------------------------- accounting

def test_compression_accounting_near_published():
    g = json.load(open(os.path.join(GOLDEN, "compression.json")))
    for L, published in g["ratios"].items():
        pol, ref = O.cache_bytes([int(L)], "C4R4")
        ratio = ref / pol
        # our metadata is 36 B/token vs ~32 implied by the pages: within 2%
        assert abs(ratio - published) / published < 0.02, (L, ratio, published)
    # closed forms: 4096 tokens = 64 pages; C4R4 keeps 288 + 36 B per token,
    # the 132-token BF16 ring and a 4-byte page entry per page; the all-BF16
    # cache is its own reference (1152 B per token + the page entries)
    assert O.cache_bytes([4096], "C4R4") == (64 * 64 * 324 + 132 * 1152 + 64 * 4, 64 * 64 * 1152 + 64 * 4)
    assert O.cache_bytes([4096], "BF16") == (64 * 64 * 1152 + 64 * 4, 64 * 64 * 1152 + 64 * 4)
    assert O.cache_bytes([65], "C2R4")[0] == 2 * 64 * 196 + 132 * 1152 + 2 * 4


def test_decode_causal_attended_prefix():
    """Reading R7: a query that sees only tokens t < n keeps each token in the
    representation of the length-L cache. Pinned against the selection rule
    restated here (BF16 iff t < 4 or t >= L - 128) and the plain definition of
    softmax attention over the chosen rows."""
    rng = np.random.default_rng(7)
    L = 300
    tok = rng.standard_normal((L, 576)).astype(np.float32)
    codes, meta = O.quantize_tokens(tok[:, :512], tok[:, 512:], "C4R4")
    deq = O.dequantize_tokens(codes, meta)
    ql = rng.standard_normal((2, 512))
    qr = rng.standard_normal((2, 64))
    scale = 1 / math.sqrt(192)
    full = O.decode_sequence(ql, qr, tok, codes, meta, L, scale, "C4R4")
    same = O.decode_sequence(ql, qr, tok, codes, meta, L, scale, "C4R4", n_attend=L)
    np.testing.assert_array_equal(full[0], same[0])
    np.testing.assert_array_equal(full[1], same[1])
    for n in (1, 4, 5, 100, 171, 172, 173, 299):
        rows = np.array([tok[t] if (t < 4 or t >= L - 128) else deq[t] for t in range(n)], dtype=np.float64)
        z = scale * (ql @ rows[:, :512].T + qr @ rows[:, 512:].T)
        w = np.exp(z - z.max(axis=1, keepdims=True))
        want_out = (w / w.sum(axis=1, keepdims=True)) @ rows[:, :512]
        want_lse = z.max(axis=1) + np.log(w.sum(axis=1))
        got_out, got_lse = O.decode_sequence(ql, qr, tok, codes, meta, L, scale, "C4R4", n_attend=n)
        np.testing.assert_allclose(got_out, want_out, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(got_lse, want_lse, rtol=1e-12, atol=1e-12)
    # the all-BF16 cache has no selection: a prefix is a shorter sequence
    a = O.decode_sequence(ql, qr, tok, None, None, L, scale, "BF16", n_attend=57)
    b = O.decode_sequence(ql, qr, tok[:57], None, None, 57, scale, "BF16")
    np.testing.assert_allclose(a[0], b[0], rtol=1e-13, atol=1e-13)
    out0, lse0 = O.decode_sequence(ql, qr, tok, codes, meta, L, scale, "C4R4", n_attend=0)
    assert np.all(out0 == 0) and np.all(np.isneginf(lse0))


def test_path_response_closed_forms():
    """Reading R8 pinned by cases with closed forms: the rescaled noise has the
    requested NMSE; with one token the softmax weight is 1, so a content
    perturbation moves the output by exactly the cache error (response 1) and
    a RoPE perturbation not at all (response 0); with q_rope = 0 the RoPE key
    never reaches the output."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((50, 64))
    n = rng.standard_normal((50, 64))
    y = O.perturb_to_nmse(x, n, 0.01)
    assert abs(np.sum((y - x) ** 2) / np.sum(x * x) - 0.01) < 1e-14
    ql, qr = rng.standard_normal((4, 512)), rng.standard_normal((4, 64))
    one = rng.standard_normal((1, 576))
    assert abs(O.path_response(ql, qr, one, 0.07, "content", rng.standard_normal((1, 512))) - 1.0) < 1e-12
    assert O.path_response(ql, qr, one, 0.07, "rope", rng.standard_normal((1, 64))) < 1e-24
    many = rng.standard_normal((300, 576))
    assert O.path_response(ql, np.zeros_like(qr), many, 0.07, "rope", rng.standard_normal((300, 64))) == 0.0


def test_path_response_on_synthetic_caches():
    """A report, not a pin (the closed-form test above pins reading R8): the
    diagnosis on the synthetic cache distribution (no model weights), content
    and RoPE responses at cache NMSE 0.01 over whole sequences, printed for
    the record. The pages' per-model numbers come from trained models and are
    not a target; this only checks the values are finite and positive."""
    import workloads as W
    stats = W.CacheStats(5)
    g = W.generator(5)
    lens = [1024, 4096]
    c, k, cu = W.make_sequences(lens, stats, g)
    ql, qr = W.make_queries(len(lens), 16, g)
    rng = np.random.default_rng(5)
    res = {"content": [], "rope": []}
    for b, L in enumerate(lens):
        a, e = int(cu[b]), int(cu[b + 1])
        tok = torch.cat([c[a:e], k[a:e]], -1).float().numpy()
        for path, width in (("content", 512), ("rope", 64)):
            r = O.path_response(ql[b].float().numpy(), qr[b].float().numpy(), tok, W.SOFTMAX_SCALE, path,
                                rng.standard_normal((L, width)))
            assert np.isfinite(r) and r > 0
            res[path].append(r)
    rc, rr = float(np.mean(res["content"])), float(np.mean(res["rope"]))
    print(f"synthetic caches: content response {rc:.3f}, RoPE response {rr:.3f}, ratio {rr / rc:.3f}")
