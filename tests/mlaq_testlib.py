"""Test helpers: build a cache through the library from seeded inputs, and
compute the oracle's answer for the same inputs (test infrastructure)."""

from __future__ import annotations

import math

import numpy as np
import torch

import oracle as O
import workloads as W


class Case:
    """Seeded inputs for one batch: tokens per sequence, queries, page table."""

    def __init__(self, mode, seq_lens, H, seed, extra_capacity=0, gen_device="cpu"):
        self.mode, self.H, self.seed = mode, H, seed
        self.seq_lens = [int(x) for x in seq_lens]
        self.B = len(self.seq_lens)
        self.stats = W.CacheStats(seed)
        g = W.generator(seed, gen_device)
        self.c, self.k, self.cu = W.make_sequences(self.seq_lens, self.stats, g, gen_device)
        self.ql, self.qr = W.make_queries(self.B, H, g, gen_device)
        cap = [L + extra_capacity for L in self.seq_lens]
        self.page_table, self.num_pages = W.make_page_table(cap, seed, extra_pages=3)
        self.scale = W.SOFTMAX_SCALE

    # -- oracle side -------------------------------------------------------
    def tokens(self, b):
        a, e = int(self.cu[b]), int(self.cu[b + 1])
        return torch.cat([self.c[a:e], self.k[a:e]], -1).float().cpu().numpy()

    def oracle_seq(self, b, L=None):
        tok = self.tokens(b)
        L = tok.shape[0] if L is None else L
        codes = meta = None
        if self.mode != "BF16":
            codes, meta = O.quantize_tokens(tok[:, :512], tok[:, 512:], self.mode)
        return O.decode_sequence(self.ql[b].float().cpu().numpy(), self.qr[b].float().cpu().numpy(),
                                 tok, codes, meta, L, self.scale, self.mode)

    # -- library side ------------------------------------------------------
    def build(self, device="cuda", max_heads=None):
        from bit_mla_kv_gb300.mlaq import Cache
        self.cache = Cache(self.mode, self.num_pages, self.B, self.page_table.shape[1],
                           max_heads=max_heads or max(self.H, 16), device=device)
        self.pt_d = self.page_table.to(device)
        self.seq_d = torch.zeros(self.B, dtype=torch.int32, device=device)
        self.cache.append(self.pt_d, self.seq_d, self.c.to(device).contiguous(), self.k.to(device).contiguous(),
                          cu_new=self.cu.to(device))
        return self.cache

    def decode(self, device="cuda"):
        return self.cache.decode(self.ql.to(device).contiguous(), self.qr.to(device).contiguous(), self.pt_d,
                                 self.seq_d, self.scale)


def assert_close_out(out_gpu, lse_gpu, out_ref, lse_ref, what=""):
    """Tolerances: out max abs error <= 1e-2 * max|ref| (per sequence), lse max
    abs error <= 1e-3; empty sequences must give exactly 0 and -inf."""
    o = out_gpu.float().cpu().numpy().astype(np.float64)
    l = lse_gpu.float().cpu().numpy().astype(np.float64)
    if np.all(np.isneginf(lse_ref)):
        assert np.all(np.isneginf(l)), what
        assert np.all(o == 0), what
        return
    scale = np.abs(out_ref).max()
    err = np.abs(o - out_ref).max()
    assert np.isfinite(o).all(), what
    assert err <= 1e-2 * scale, f"{what}: out err {err:.3e} > 1e-2 * {scale:.3e}"
    lerr = np.abs(l - lse_ref).max()
    assert lerr <= 1e-3, f"{what}: lse err {lerr:.3e}"
    return err / scale, lerr


def expected_codes(case, b):
    tok = case.tokens(b)
    return O.quantize_tokens(tok[:, :512], tok[:, 512:], case.mode)
