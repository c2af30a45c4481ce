"""Thin ctypes binding of libmlaq (argument marshalling only).

Every step of the decode path runs in the CUDA kernels behind the C ABI
declared in include/mlaq.h; the functions here check tensor dtypes and
shapes, pass device pointers and the current CUDA stream, and turn status
codes into exceptions. There is no fallback: if libmlaq.so is missing or
cannot be loaded, importing this module raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

from . import MODES

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmlaq.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        "libmlaq.so not built: run `python -c 'import __graft_entry__ as g; g.build()'` "
        "or `python -m bit_mla_kv_gb300.build` first")
_lib = ctypes.CDLL(LIB_PATH)

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_sz = ctypes.c_size_t
_szp = ctypes.POINTER(ctypes.c_size_t)

EXPORTED = [
    "mlaq_buffer_sizes", "mlaq_cache_create", "mlaq_cache_destroy", "mlaq_append", "mlaq_decode",
    "mlaq_export_tokens", "mlaq_cache_bytes", "mlaq_get_device_status", "mlaq_clear_device_status",
    "mlaq_timing_enable", "mlaq_timing_read", "mlaq_set_decode_ctas", "mlaq_set_plan_costs", "mlaq_status_string",
    "mlaq_decode_noalloc", "mlaq_debug_wait_probe", "mlaq_decode_mtp", "mlaq_set_decode_variant",
]

_lib.mlaq_status_string.restype = ctypes.c_char_p
_lib.mlaq_status_string.argtypes = [ctypes.c_int]
_lib.mlaq_buffer_sizes.argtypes = [ctypes.c_int, _i32, _i32, _i32, _szp, _szp, _szp, _szp]
_lib.mlaq_cache_create.argtypes = [ctypes.POINTER(_vp), ctypes.c_int, _i32, _i32, _i32, _i32,
                                   _vp, _vp, _vp, _vp, _sz]
_lib.mlaq_cache_destroy.argtypes = [_vp]
_lib.mlaq_append.argtypes = [_vp, _vp, _vp, _i32, _vp, _vp, _i32, _vp, _i32, _vp]
_lib.mlaq_decode.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _i32, ctypes.c_float, _vp, _vp, _vp]
_lib.mlaq_export_tokens.argtypes = [_vp, _vp, _i32, _vp, _vp, _i32, _vp, _vp, _vp]
_lib.mlaq_cache_bytes.argtypes = [_vp, ctypes.POINTER(_i32), _i32, _szp, _szp]
_lib.mlaq_get_device_status.argtypes = [_vp, _vp, ctypes.POINTER(_i32)]
_lib.mlaq_clear_device_status.argtypes = [_vp, _vp]
_lib.mlaq_timing_enable.argtypes = [_vp, _i32]
_lib.mlaq_timing_read.argtypes = [_vp, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(_i32)]
_lib.mlaq_set_decode_ctas.argtypes = [_vp, _i32]
_lib.mlaq_set_plan_costs.argtypes = [_vp, _i32, _i32, _i32]
_lib.mlaq_set_decode_variant.argtypes = [_vp, _i32]
_lib.mlaq_decode_noalloc.argtypes = [ctypes.c_int, _vp, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _i32, _i32,
                                     ctypes.c_float, _vp, _vp, _vp, _vp]
_lib.mlaq_debug_wait_probe.argtypes = [_vp, _i32, _i32, _vp]
_lib.mlaq_decode_mtp.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, ctypes.c_float, _vp, _vp, _vp]
for _name in EXPORTED:
    if _name != "mlaq_status_string":
        getattr(_lib, _name).restype = ctypes.c_int

DEV_PAGE_OOB, DEV_SEQ_OVERFLOW, DEV_NONFINITE, DEV_TIMEOUT, DEV_RANGE, DEV_BAD_ROWS = 0x1, 0x2, 0x4, 0x8, 0x10, 0x20


class MlaqError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {_lib.mlaq_status_string(code).decode()} ({code})")
        self.code = code


def _check(code: int, what: str):
    if code != 0:
        raise MlaqError(code, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, dtype, shape=None, name="tensor"):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")


def buffer_sizes(mode: str, num_pages: int, max_seqs: int, max_heads: int):
    out = [ctypes.c_size_t() for _ in range(4)]
    _check(_lib.mlaq_buffer_sizes(MODES[mode], num_pages, max_seqs, max_heads, *[ctypes.byref(o) for o in out]),
           "mlaq_buffer_sizes")
    return tuple(o.value for o in out)


def debug_wait_probe(status, wait_us: int, arrive: bool, stream=None):
    """Runs the bounded-wait test hook into `status` (int32 CUDA tensor of one
    element): MLAQ_DEV_TIMEOUT when the wait ran out, 0 when it completed."""
    _need(status, torch.int32, (1,), "status")
    _check(_lib.mlaq_debug_wait_probe(_ptr(status), int(wait_us), 1 if arrive else 0, _stream(stream)),
           "mlaq_debug_wait_probe")


def _bf16_rows_in_channel_order(raw):
    """Undo the stored chunk permutation of BF16 rows: channel e of row r
    sits at element ((e // 8) ^ (r % 8)) * 8 + e % 8 of the row."""
    rows = raw.shape[-2]
    e = torch.arange(576)
    r = torch.arange(rows)[:, None]
    idx = (((e // 8) ^ (r % 8)) * 8 + e % 8).to(raw.device)
    return torch.gather(raw, -1, idx.expand(raw.shape))


class Cache:
    """A paged QuantMLA cache: the code pool, fp16 meta pool, BF16 sink/recent
    ring and workspace are torch device tensors owned by this object."""

    def __init__(self, mode: str, num_pages: int, max_seqs: int, max_pages_per_seq: int,
                 max_heads: int = 128, device="cuda"):
        self.mode = mode
        self.num_pages, self.max_seqs = num_pages, max_seqs
        self.max_pages_per_seq, self.max_heads = max_pages_per_seq, max_heads
        cb, mb, rb, wb = buffer_sizes(mode, num_pages, max_seqs, max_heads)
        self.codes = torch.zeros(cb, dtype=torch.uint8, device=device)
        self.meta = torch.zeros(max(mb, 16), dtype=torch.uint8, device=device)
        self.ring = torch.zeros(max(rb, 16), dtype=torch.uint8, device=device)
        self.workspace = torch.zeros(wb, dtype=torch.uint8, device=device)
        h = ctypes.c_void_p()
        with torch.cuda.device(self.codes.device):
            _check(_lib.mlaq_cache_create(ctypes.byref(h), MODES[mode], num_pages, max_seqs, max_pages_per_seq,
                                          max_heads, _ptr(self.codes), _ptr(self.meta), _ptr(self.ring),
                                          _ptr(self.workspace), wb), "mlaq_cache_create")
        self._h = h

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            _lib.mlaq_cache_destroy(h)
            self._h = None

    @property
    def handle(self):
        return self._h

    def ring_view(self):
        """The BF16 ring as [max_seqs, 132, 576] bfloat16 in channel order
        (slots 0-3 sink, slot 4 + t % 128 for recent token t); a copy, with
        the stored chunk permutation undone."""
        raw = self.ring[: self.max_seqs * 132 * 576 * 2].view(torch.bfloat16).view(self.max_seqs, 132, 576)
        return _bf16_rows_in_channel_order(raw)

    def bf16_pages_view(self):
        """BF16 mode: the page pool as [num_pages, 64, 576] bfloat16 in
        channel order (a copy)."""
        assert self.mode == "BF16"
        raw = self.codes[: self.num_pages * 64 * 576 * 2].view(torch.bfloat16).view(self.num_pages, 64, 576)
        return _bf16_rows_in_channel_order(raw)

    def append(self, page_table, seq_lens, c_latent, k_rope, cu_new=None, stream=None):
        """Append tokens. Without cu_new: c_latent [B, n_new, 512], k_rope
        [B, n_new, 64]. With cu_new (int32 [B+1] device prefix sum):
        c_latent [N, 512], k_rope [N, 64]. seq_lens is advanced in place."""
        B = seq_lens.shape[0]
        _need(page_table, torch.int32, (B, self.max_pages_per_seq), "page_table")
        _need(seq_lens, torch.int32, (B,), "seq_lens")
        _need(c_latent, torch.bfloat16, None, "c_latent")
        _need(k_rope, torch.bfloat16, None, "k_rope")
        if cu_new is None:
            if c_latent.dim() != 3 or c_latent.shape[0] != B or c_latent.shape[2] != 512:
                raise ValueError("c_latent must be [B, n_new, 512]")
            n_new = c_latent.shape[1]
            _need(k_rope, torch.bfloat16, (B, n_new, 64), "k_rope")
            total = B * n_new
        else:
            _need(cu_new, torch.int32, (B + 1,), "cu_new")
            total = c_latent.shape[0]
            _need(c_latent, torch.bfloat16, (total, 512), "c_latent")
            _need(k_rope, torch.bfloat16, (total, 64), "k_rope")
            n_new = 0
        _check(_lib.mlaq_append(self._h, _ptr(page_table), _ptr(seq_lens), B, _ptr(c_latent), _ptr(k_rope),
                                n_new, _ptr(cu_new), total, _stream(stream)), "mlaq_append")

    def decode(self, q_latent, q_rope, page_table, seq_lens, softmax_scale, out=None, lse=None, stream=None):
        """Decode attention; returns (out_latent [B, H, 512] bf16, lse [B, H] fp32)."""
        B, H = q_latent.shape[0], q_latent.shape[1]
        _need(q_latent, torch.bfloat16, (B, H, 512), "q_latent")
        _need(q_rope, torch.bfloat16, (B, H, 64), "q_rope")
        _need(page_table, torch.int32, (B, self.max_pages_per_seq), "page_table")
        _need(seq_lens, torch.int32, (B,), "seq_lens")
        if out is None:
            out = torch.empty(B, H, 512, dtype=torch.bfloat16, device=q_latent.device)
        if lse is None:
            lse = torch.empty(B, H, dtype=torch.float32, device=q_latent.device)
        _need(out, torch.bfloat16, (B, H, 512), "out")
        _need(lse, torch.float32, (B, H), "lse")
        _check(_lib.mlaq_decode(self._h, _ptr(q_latent), _ptr(q_rope), _ptr(page_table), _ptr(seq_lens), B, H,
                                float(softmax_scale), _ptr(out), _ptr(lse), _stream(stream)), "mlaq_decode")
        return out, lse

    def decode_mtp(self, q_latent, q_rope, page_table, seq_lens, softmax_scale, out=None, lse=None, stream=None):
        """Decode attention for Q query tokens per sequence, causal over the Q
        newest tokens (query j sees t < L - (Q - 1 - j)); q_latent [B, Q, H, 512],
        q_rope [B, Q, H, 64]; returns (out [B, Q, H, 512] bf16, lse [B, Q, H] fp32)."""
        B, Q, H = q_latent.shape[0], q_latent.shape[1], q_latent.shape[2]
        _need(q_latent, torch.bfloat16, (B, Q, H, 512), "q_latent")
        _need(q_rope, torch.bfloat16, (B, Q, H, 64), "q_rope")
        _need(page_table, torch.int32, (B, self.max_pages_per_seq), "page_table")
        _need(seq_lens, torch.int32, (B,), "seq_lens")
        if out is None:
            out = torch.empty(B, Q, H, 512, dtype=torch.bfloat16, device=q_latent.device)
        if lse is None:
            lse = torch.empty(B, Q, H, dtype=torch.float32, device=q_latent.device)
        _need(out, torch.bfloat16, (B, Q, H, 512), "out")
        _need(lse, torch.float32, (B, Q, H), "lse")
        _check(_lib.mlaq_decode_mtp(self._h, _ptr(q_latent), _ptr(q_rope), _ptr(page_table), _ptr(seq_lens), B, Q, H,
                                    float(softmax_scale), _ptr(out), _ptr(lse), _stream(stream)), "mlaq_decode_mtp")
        return out, lse

    def export_tokens(self, page_table, token_b, token_t, stream=None):
        """Canonical codes [n, 576] uint8 and meta [n, 9, 2] fp16 of stored tokens."""
        n = token_b.shape[0]
        _need(token_b, torch.int32, (n,), "token_b")
        _need(token_t, torch.int32, (n,), "token_t")
        codes = torch.empty(n, 576, dtype=torch.uint8, device=token_b.device)
        meta = torch.empty(n, 9, 2, dtype=torch.float16, device=token_b.device)
        _check(_lib.mlaq_export_tokens(self._h, _ptr(page_table), page_table.shape[0], _ptr(token_b),
                                       _ptr(token_t), n, _ptr(codes), _ptr(meta), _stream(stream)),
               "mlaq_export_tokens")
        return codes, meta

    def cache_bytes(self, seq_lens):
        arr = (ctypes.c_int32 * len(seq_lens))(*[int(x) for x in seq_lens])
        pol, ref = ctypes.c_size_t(), ctypes.c_size_t()
        _check(_lib.mlaq_cache_bytes(self._h, arr, len(seq_lens), ctypes.byref(pol), ctypes.byref(ref)),
               "mlaq_cache_bytes")
        return pol.value, ref.value

    def device_status(self, stream=None) -> int:
        v = ctypes.c_int32()
        _check(_lib.mlaq_get_device_status(self._h, _stream(stream), ctypes.byref(v)), "mlaq_get_device_status")
        return v.value

    def clear_status(self, stream=None):
        _check(_lib.mlaq_clear_device_status(self._h, _stream(stream)), "mlaq_clear_device_status")

    def timing_enable(self, max_calls: int):
        _check(_lib.mlaq_timing_enable(self._h, max_calls), "mlaq_timing_enable")

    def timing_read(self):
        buf = (ctypes.c_float * 65536)()
        n = ctypes.c_int32()
        _check(_lib.mlaq_timing_read(self._h, buf, ctypes.byref(n)), "mlaq_timing_read")
        return [buf[k] for k in range(n.value)]

    def decode_noalloc(self, q_latent, q_rope, page_table, seq_lens, softmax_scale, out=None, lse=None,
                       dev_status=None, stream=None):
        """mlaq_decode_noalloc over this cache's pools: the split-KV scratch
        comes from the library's fixed device array instead of the workspace."""
        B, H = q_latent.shape[0], q_latent.shape[1]
        _need(q_latent, torch.bfloat16, (B, H, 512), "q_latent")
        _need(q_rope, torch.bfloat16, (B, H, 64), "q_rope")
        _need(page_table, torch.int32, (B, self.max_pages_per_seq), "page_table")
        _need(seq_lens, torch.int32, (B,), "seq_lens")
        if out is None:
            out = torch.empty(B, H, 512, dtype=torch.bfloat16, device=q_latent.device)
        if lse is None:
            lse = torch.empty(B, H, dtype=torch.float32, device=q_latent.device)
        _check(_lib.mlaq_decode_noalloc(MODES[self.mode], _ptr(self.codes), _ptr(self.meta), _ptr(self.ring),
                                        self.num_pages, self.max_pages_per_seq, _ptr(q_latent), _ptr(q_rope),
                                        _ptr(page_table), _ptr(seq_lens), B, H, float(softmax_scale), _ptr(out),
                                        _ptr(lse), _ptr(dev_status), _stream(stream)), "mlaq_decode_noalloc")
        return out, lse

    def set_decode_ctas(self, ctas: int):
        _check(_lib.mlaq_set_decode_ctas(self._h, ctas), "mlaq_set_decode_ctas")

    def set_decode_variant(self, variant: int):
        """0 automatic, 1 register-score kernel, 2 tcgen05-score kernel."""
        _check(_lib.mlaq_set_decode_variant(self._h, variant), "mlaq_set_decode_variant")

    def set_plan_costs(self, step: int, ring: int, item: int):
        _check(_lib.mlaq_set_plan_costs(self._h, step, ring, item), "mlaq_set_plan_costs")
