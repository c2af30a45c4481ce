"""Plain CPU restatement of the QuantMLA low-bit MLA decode path (test oracle).

TEST INFRASTRUCTURE ONLY: imported by tests/, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py``; never by the library.

Sources (five web summaries of "QuantMLA: Function-Aligned Dual-Path
Quantization for Low-Bit MLA KV Caching", arXiv 2609.36760):
  [AIS]  ai.info "AI summary" -- sections "Key Contributions" (item 4) and
         "Methodology in Plain English".
  [ODK]  onedev.kr summary -- sections "어떻게 쓰나" (how to use: the fused
         writer, sink/recent BF16 copies, one global softmax) and
         "전제와 한계" (per-token asymmetric quantizer, group size 64).
  [SLN]  slinene.github.io daily summary -- section "方法关键点" (4 sink +
         128 recent tokens kept in BF16; unpack/dequant fused into attention).
  [TDH]  tokendh.com article -- section "从实验室到实际部署" (sink/recent
         protection zone, 27.9% / 3.59x persistent cache at 128K).

Readings taken where the pages are silent:
  R1  quantizer arithmetic: mn = min(x); s32 = (max(x) - mn) / (2^b - 1) in
      IEEE fp32; the stored metadata are s = fp16_rn(s32), m = fp16_rn(mn);
      codes use the STORED (s, m): q = clamp(rint_even((x - m) / s), 0, 2^b-1)
      with fp32 subtract and fp32 IEEE division; s == 0 gives q = 0.
  R2  content groups are channels [64g, 64g+64), g = 0..7; the RoPE key is one
      group of 64 channels.
  R3  canonical packing: code i of a segment sits in bits [b*(i mod k), +b) of
      byte floor(i/k), k = 8/b; content segment first, then the RoPE segment.
  R4  token t of a length-L sequence is read in BF16 iff t < 4 or t >= L-128,
      otherwise from its packed copy; L counts every appended token.
  R5  scores are softmax_scale * (q_lat . c + q_rope . k_r); lse is the natural
      log of the sum of exp(score); out = sum_t softmax_t * c_t (512-d latent).
  R6  every token gets a packed copy (sink and recent ones too); the ring slot
      of a non-sink token t is 4 + (t mod 128); sink token t uses slot t.
  R8  error response (the pages' diagnosis, [AIS] "Methodology in Plain
      English" and Main Findings): one path's cache (content latent or RoPE
      key) gets additive noise rescaled to NMSE ||d||^2 / ||x||^2 = 0.01
      exactly; the response is the attention output's NMSE divided by that
      cache NMSE; the noise is an input (drawn by the caller).
  R7  several query tokens per sequence (the pages describe one): with Q new
      tokens appended (length L), query j = 0..Q-1 attends to tokens
      t < L - (Q - 1 - j), causally, and every token keeps the representation
      (BF16 or packed) that the length-L cache gives it.

Parity pins for every function live in tests/test_oracle.py.
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "SINK", "RECENT", "GROUP", "D_LATENT", "D_ROPE", "D_QK", "N_GROUPS", "RING_SLOTS",
    "MODES", "mode_bits", "packed_bytes_per_token", "quantize_groups", "quantize_tokens",
    "pack_canonical", "unpack_canonical", "dequantize_tokens", "is_bf16_token",
    "bf16_token_mask", "assemble_kv", "attend", "decode_sequence",
    "combine_partials", "expected_ring", "cache_bytes", "perturb_to_nmse", "path_response",
]

SINK = 4            # [SLN] 方法关键点 / [ODK] 어떻게 쓰나: first 4 tokens kept in BF16
RECENT = 128        # same passages: most recent 128 tokens kept in BF16
GROUP = 64          # [AIS] Methodology / [ODK] 전제와 한계: group size 64
D_LATENT = 512      # MLA content latent width
D_ROPE = 64         # MLA decoupled RoPE key width
D_QK = D_LATENT + D_ROPE
N_GROUPS = D_QK // GROUP  # 8 content groups + 1 RoPE group
RING_SLOTS = SINK + RECENT

# (content bits, rope bits); C4R4 / C2R4 are named in [AIS] Key Contributions 3.
MODES = {"C4R4": (4, 4), "C2R4": (2, 4), "BF16": None}


def mode_bits(mode: str):
    """(content bits, RoPE bits) of a packed mode; None for the all-BF16 cache."""
    return MODES[mode]


def packed_bytes_per_token(mode: str) -> int:
    """Bytes of codes per token under canonical packing (no metadata)."""
    bc, br = MODES[mode]
    return D_LATENT * bc // 8 + D_ROPE * br // 8


def quantize_groups(x, bits: int):
    """Per-group asymmetric affine quantizer (reading R1).

    x: array [..., 64] of bf16 values held as float32. Returns
    (codes uint8 [..., 64], scale float16 [...], minimum float16 [...]).

    Source: [AIS] "Methodology in Plain English" and [ODK] "전제와 한계" --
    every quantized cache uses the same per-token asymmetric affine quantizer
    with group size 64. The fp32/fp16 arithmetic is reading R1.
    """
    x = np.asarray(x, dtype=np.float32)
    assert x.shape[-1] == GROUP
    qmax = np.float32(2 ** bits - 1)
    mn = x.min(axis=-1)
    mx = x.max(axis=-1)
    s32 = np.divide(np.subtract(mx, mn, dtype=np.float32), qmax, dtype=np.float32)
    s_h = s32.astype(np.float16)
    mn_h = mn.astype(np.float16)
    s_f = s_h.astype(np.float32)[..., None]
    mn_f = mn_h.astype(np.float32)[..., None]
    zero = s_f == 0
    diff = np.subtract(x, mn_f, dtype=np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = np.divide(diff, np.where(zero, np.float32(1), s_f), dtype=np.float32)
    q = np.clip(np.rint(t), np.float32(0), qmax)
    q = np.where(zero, np.float32(0), q)
    return q.astype(np.uint8), s_h, mn_h


def quantize_tokens(c_latent, k_rope, mode: str):
    """Quantize whole tokens: 8 content groups + 1 RoPE group (reading R2).

    c_latent [..., 512], k_rope [..., 64] (bf16 values as float32).
    Returns codes uint8 [..., 576] (one code per element, content then RoPE)
    and meta float16 [..., 9, 2] holding (scale, minimum) per group.
    """
    bc, br = MODES[mode]
    c = np.asarray(c_latent, dtype=np.float32)
    k = np.asarray(k_rope, dtype=np.float32)
    lead = c.shape[:-1]
    qc, sc, mc = quantize_groups(c.reshape(*lead, D_LATENT // GROUP, GROUP), bc)
    qr, sr, mr = quantize_groups(k.reshape(*lead, 1, GROUP), br)
    codes = np.concatenate([qc.reshape(*lead, D_LATENT), qr.reshape(*lead, D_ROPE)], axis=-1)
    scale = np.concatenate([sc, sr], axis=-1)
    mins = np.concatenate([mc, mr], axis=-1)
    meta = np.stack([scale, mins], axis=-1)
    return codes, meta


def _pack_segment(codes, bits):
    k = 8 // bits
    n = codes.shape[-1]
    c = codes.reshape(*codes.shape[:-1], n // k, k).astype(np.uint16)
    out = np.zeros(c.shape[:-1], dtype=np.uint16)
    for j in range(k):
        out |= c[..., j] << (bits * j)
    return out.astype(np.uint8)


def _unpack_segment(packed, bits):
    k = 8 // bits
    p = packed.astype(np.uint16)
    mask = (1 << bits) - 1
    parts = [(p >> (bits * j)) & mask for j in range(k)]
    return np.stack(parts, axis=-1).reshape(*packed.shape[:-1], packed.shape[-1] * k).astype(np.uint8)


def pack_canonical(codes, mode: str):
    """Canonical packing (reading R3): [..., 576] codes -> [..., bytes/token]."""
    bc, br = MODES[mode]
    codes = np.asarray(codes, dtype=np.uint8)
    return np.concatenate([_pack_segment(codes[..., :D_LATENT], bc),
                           _pack_segment(codes[..., D_LATENT:], br)], axis=-1)


def unpack_canonical(packed, mode: str):
    """Inverse of pack_canonical."""
    bc, br = MODES[mode]
    nb = D_LATENT * bc // 8
    packed = np.asarray(packed, dtype=np.uint8)
    return np.concatenate([_unpack_segment(packed[..., :nb], bc),
                           _unpack_segment(packed[..., nb:], br)], axis=-1)


def dequantize_tokens(codes, meta):
    """c_hat = q * s + m per group, exactly in fp64 (s, m the stored fp16 meta).

    Source: the affine dequantization implied by [AIS] Methodology (asymmetric
    affine quantizer) with the stored (scale, minimum) of reading R1.
    """
    codes = np.asarray(codes)
    meta = np.asarray(meta)
    lead = codes.shape[:-1]
    q = codes.astype(np.float64).reshape(*lead, N_GROUPS, GROUP)
    s = meta[..., 0].astype(np.float64)[..., None]
    m = meta[..., 1].astype(np.float64)[..., None]
    return (q * s + m).reshape(*lead, D_QK)


def is_bf16_token(t: int, L: int) -> bool:
    """Reading R4 of [SLN] 方法关键点 / [ODK] 어떻게 쓰나: sink or recent."""
    return t < SINK or t >= L - RECENT


def bf16_token_mask(L: int):
    """Boolean [L]: True where token t is served from its BF16 copy."""
    t = np.arange(L)
    return (t < SINK) | (t >= L - RECENT)


def assemble_kv(tokens_bf16, codes, meta, L: int, mode: str):
    """The [L, 576] fp64 matrix attention sees: exactly one representation per
    token ([ODK] 어떻게 쓰나) -- the BF16 value for sink/recent tokens, the
    dequantized packed copy for every other token. mode 'BF16' uses the BF16
    value for all tokens (the uncompressed comparison cache)."""
    x = np.asarray(tokens_bf16[:L], dtype=np.float64)
    if mode == "BF16" or L == 0:
        return x
    deq = dequantize_tokens(codes[:L], meta[:L])
    sel = bf16_token_mask(L)[:, None]
    return np.where(sel, x, deq)


def attend(q_lat, q_rope, kv, scale: float):
    """Single global softmax MLA decode attention in fp64 (readings R5).

    q_lat [H, 512], q_rope [H, 64], kv [L, 576]. Returns (out [H, 512], lse [H]).
    One softmax covers every valid token ([AIS] Key Contributions 4: a single
    global softmax over all valid tokens). L == 0 gives out = 0, lse = -inf.
    """
    q_lat = np.asarray(q_lat, dtype=np.float64)
    q_rope = np.asarray(q_rope, dtype=np.float64)
    kv = np.asarray(kv, dtype=np.float64)
    H = q_lat.shape[0]
    if kv.shape[0] == 0:
        return np.zeros((H, D_LATENT)), np.full(H, -np.inf)
    z = scale * (q_lat @ kv[:, :D_LATENT].T + q_rope @ kv[:, D_LATENT:].T)
    m = z.max(axis=1, keepdims=True)
    e = np.exp(z - m)
    ssum = e.sum(axis=1, keepdims=True)
    lse = (m + np.log(ssum))[:, 0]
    out = (e / ssum) @ kv[:, :D_LATENT]
    return out, lse


def decode_sequence(q_lat, q_rope, tokens_bf16, codes, meta, L, scale, mode, n_attend=None):
    """Decode one sequence: token selection, then one softmax (fp64).

    n_attend (reading R7): the query sees only tokens t < n_attend, each in the
    representation the length-L cache gives it; None means all L tokens."""
    kv = assemble_kv(tokens_bf16, codes, meta, L, mode)
    if n_attend is not None:
        kv = kv[:max(0, min(int(n_attend), L))]
    return attend(q_lat, q_rope, kv, scale)


def combine_partials(outs, lses):
    """Merge split partial results (each normalized over its own token range)
    into the single global softmax: lse = log sum_i exp(lse_i),
    out = sum_i exp(lse_i - lse) out_i. Empty input / all -inf gives 0, -inf."""
    lses = np.asarray(lses, dtype=np.float64)
    outs = np.asarray(outs, dtype=np.float64)
    if lses.shape[0] == 0:
        raise ValueError("no partials")
    m = lses.max(axis=0)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.exp(lses - m_safe[None])
    tot = w.sum(axis=0)
    lse = np.where(finite, m_safe + np.log(np.where(finite, tot, 1.0)), -np.inf)
    wn = np.where(finite[None], w / np.where(finite, tot, 1.0)[None], 0.0)
    out = np.einsum("s...,s...d->...d", wn, outs)
    return out, lse


def expected_ring(tokens_bf16, L: int):
    """Contents of the BF16 sink/recent ring after L tokens (reading R6).

    Returns (ring [132, 576] float32, valid [132] bool). Slot j < 4 holds sink
    token j; slot 4 + r holds the newest token t < L with t mod 128 == r and
    t >= 4 (a token leaving the recent window is overwritten by its successor
    128 positions later, which is how it retires to its packed copy:
    [ODK] 어떻게 쓰나).
    """
    tok = np.asarray(tokens_bf16, dtype=np.float32)
    ring = np.zeros((RING_SLOTS, D_QK), dtype=np.float32)
    valid = np.zeros(RING_SLOTS, dtype=bool)
    for j in range(min(SINK, L)):
        ring[j] = tok[j]
        valid[j] = True
    for t in range(max(SINK, L - RECENT), L):
        ring[SINK + t % RECENT] = tok[t]
        valid[SINK + t % RECENT] = True
    return ring, valid


def cache_bytes(seq_lens, mode: str, page_tokens: int = 64, meta_bytes_per_token: int = N_GROUPS * 4,
                page_entry_bytes: int = 4):
    """Persistent cache bytes under the mixed-precision policy, counted the way
    [ODK] 시스템 효율 paragraph counts them: BF16 buffers + packed copies of all
    tokens + page mapping. Returns (packed_policy_bytes, bf16_cache_bytes).
    Mode 'BF16' is the paged all-BF16 cache the paragraph compares against, so
    its policy bytes are its BF16 bytes (no ring, no packed copies)."""
    bf16 = MODES[mode] is None
    packed_tok = D_QK * 2 if bf16 else packed_bytes_per_token(mode) + meta_bytes_per_token
    ring = 0 if bf16 else RING_SLOTS * D_QK * 2
    pol = 0
    ref = 0
    for L in seq_lens:
        pages = math.ceil(L / page_tokens)
        pol += pages * page_tokens * packed_tok + ring + pages * page_entry_bytes
        ref += pages * page_tokens * D_QK * 2 + pages * page_entry_bytes
    return pol, ref


def perturb_to_nmse(x, noise, nmse: float):
    """x + d with d = noise rescaled so that ||d||^2 / ||x||^2 == nmse (reading R8)."""
    x = np.asarray(x, dtype=np.float64)
    noise = np.asarray(noise, dtype=np.float64)
    d = noise * math.sqrt(nmse * float(np.sum(x * x)) / float(np.sum(noise * noise)))
    return x + d


def path_response(q_lat, q_rope, tokens, scale: float, path: str, noise, nmse: float = 0.01):
    """Output damage per unit cache error of one path (reading R8).

    tokens [L, 576] (content latent then RoPE key, full precision); path
    'content' perturbs the latent (it enters the logits and the values),
    'rope' the RoPE key (logits only). Returns NMSE(out') / nmse over all
    heads of q_lat [H, 512], q_rope [H, 64]."""
    tok = np.asarray(tokens, dtype=np.float64)
    out, _ = attend(q_lat, q_rope, tok, scale)
    pert = tok.copy()
    if path == "content":
        pert[:, :D_LATENT] = perturb_to_nmse(tok[:, :D_LATENT], noise, nmse)
    elif path == "rope":
        pert[:, D_LATENT:] = perturb_to_nmse(tok[:, D_LATENT:], noise, nmse)
    else:
        raise ValueError(path)
    out2, _ = attend(q_lat, q_rope, pert, scale)
    return float(np.sum((out2 - out) ** 2) / np.sum(out * out)) / nmse

