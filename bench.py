"""Benchmark of the QuantMLA decode path (libmlaq) on synthetic inputs.

One step = the whole hot path for one batch: the fused writer appends one new
token to every sequence (mlaq_append), then split-KV decode attention runs
over the mixed-precision paged cache (mlaq_decode: planner, attention kernel,
combine). Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl mlaq|reference]

value = effective cache GB/s = algorithmic bytes per step / device time per
step (inputs resident in HBM, L2 flushed between timed steps). The algorithmic
bytes of a decode step are sum_b [min(L_b,132) * 1152 + max(0, L_b-132) * P]
+ B*H*(1152 + 1024 + 4), P = packed bytes + fp16 meta per token (C4R4 324,
C2R4 196, BF16 1152); the append adds B * (1152 read + P + 1152) bytes.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "decode-attn µs/step & effective cache GB/s (C4R4/C2R4), % of roofline"
PACKED_TOKEN_BYTES = {"C4R4": 288 + 36, "C2R4": 160 + 36, "BF16": 1152}
L2_FLUSH_BYTES = 256 << 20


def decode_bytes(seq_lens, mode, B, H):
    P = PACKED_TOKEN_BYTES[mode]
    tot = 0
    for L in seq_lens:
        if mode == "BF16":
            tot += L * 1152
        else:
            tot += min(L, 132) * 1152 + max(0, L - 132) * P
    return tot + B * H * (1152 + 1024 + 4)


def append_bytes(B, mode):
    P = PACKED_TOKEN_BYTES[mode]
    return B * (1152 + P + (0 if mode == "BF16" else 1152))


def prefill_bytes(seq_lens, mode):
    """Writer traffic of appending whole sequences: every token's bf16 row read,
    its packed codes and meta (or its bf16 page copy) written, and the BF16
    sink/recent copies of the packed modes."""
    ring = 0 if mode == "BF16" else sum(min(L, 132) for L in seq_lens) * 1152
    return sum(seq_lens) * (1152 + PACKED_TOKEN_BYTES[mode]) + ring


def decode_flops(seq_lens, H):
    return sum(seq_lens) * 2 * H * (576 + 512)


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return pk["hbm_gbs"], pk["bf16_tflops"], pk.get("bf16_tflops_sustained", pk["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def kernel_source_sha():
    h = hashlib.sha256()
    for f in ("mlaq_decode.cu", "mlaq_internal.cuh"):
        with open(os.path.join(ROOT, "bit_mla_kv_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per launch of the decode kernel from a committed ncu summary,
    or None when absent or taken on a different kernel source."""
    path = os.path.join(ROOT, "profiles", "decode_kernel_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    ent = rec.get(workload)
    if not ent or ent.get("kernel_source_sha") != kernel_source_sha():
        return None
    return ent.get("traffic_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
            # the tool's start-up (driver queries) must not overlap the timed
            # steps: wait until its first sample is written (at most 5 s)
            t_end = time.time() + 5.0
            time.sleep(0.3)
            while time.time() < t_end and os.path.getsize(self.path) == 0 and self.proc.poll() is None:
                time.sleep(0.05)
            time.sleep(0.15)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 7:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[3 + k].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def dist_setup(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "mlaq" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws, device):
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, ws, device):
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def oracle_sample(case_tokens, seq_lens, queries, mode, budget_s):
    """Time the oracle (as it stands) on whole sequences until ~budget_s of CPU
    work, going over the workload's sequences again when one pass is shorter.
    case_tokens(b) -> [L, 576] float32. Returns (bytes, seconds, desc)."""
    import oracle as O
    done_bytes, t_total, n_seq, toks, passes = 0, 0.0, 0, 0, 0
    order = sorted(range(len(seq_lens)), key=lambda b: seq_lens[b])
    order = order[len(order) // 2:] + order[:len(order) // 2]  # start near the median length
    ql, qr = queries
    while t_total < budget_s and passes < 64:  # the pass cap only matters for near-empty workloads
        passes += 1
        for b in order:
            L = seq_lens[b]
            tok = case_tokens(b)
            codes = meta = None
            if mode != "BF16":
                codes, meta = O.quantize_tokens(tok[:, :512], tok[:, 512:], mode)  # cache state, not timed
            t0 = time.perf_counter()
            O.decode_sequence(ql[b], qr[b], tok, codes, meta, L, W.SOFTMAX_SCALE, mode)
            t_total += time.perf_counter() - t0
            done_bytes += decode_bytes([L], mode, 1, ql.shape[1])
            n_seq += 1
            toks += L
            if t_total >= budget_s:
                break
    return done_bytes, t_total, (f"{n_seq} whole sequences in {passes} pass(es) over the workload "
                                 f"({toks} tokens, H={ql.shape[1]})")


def cores_used():
    try:
        n = len(os.sched_getaffinity(0))
    except Exception:
        n = os.cpu_count() or 1
    return n


def build_inputs(wl, rank, device, total_steps):
    """Seeded inputs on the device for one replica."""
    seed = wl.seed + 1000 * rank
    stats = W.CacheStats(seed)
    g = W.generator(seed, device)
    c, k, cu = W.make_sequences(wl.seq_lens, stats, g, device)
    ql, qr = W.make_queries(wl.B, wl.H, g, device)
    cn, kn = W.make_tokens(wl.B * total_steps, stats, g, device)
    cn = cn.view(total_steps, wl.B, 1, 512)
    kn = kn.view(total_steps, wl.B, 1, 64)
    pt, num_pages = W.make_page_table([L + total_steps + 64 for L in wl.seq_lens], seed)
    return dict(c=c, k=k, cu=cu, ql=ql, qr=qr, cn=cn, kn=kn, pt=pt.to(device), num_pages=num_pages, seed=seed)


def make_l2_flush(device):
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    clean = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    sink = torch.empty(1, dtype=torch.float32, device=device)

    def l2_flush():
        # Write a buffer twice the L2 size (evicts the step's inputs), then
        # read a second one of the same size, so that the flush's own dirty
        # lines are written back here and not inside the timed decode.
        flush.zero_()
        torch.sum(clean, dim=0, keepdim=True, out=sink)
    return l2_flush


class Workbench:
    """One workload on one device: its seeded inputs, a cache filled by the
    fused writer, and the step (append one token per sequence + decode)."""

    def __init__(self, wl, rank, device, total_steps, variant=0):
        from bit_mla_kv_gb300.mlaq import Cache
        self.wl, self.device = wl, device
        self.inp = build_inputs(wl, rank, device, total_steps)
        self.cache = Cache(wl.mode, self.inp["num_pages"], wl.B, self.inp["pt"].shape[1], max_heads=max(wl.H, 16),
                           device=device)
        self.cache.set_decode_variant(variant)
        self.seq = torch.zeros(wl.B, dtype=torch.int32, device=device)
        self.cu_d = self.inp["cu"].to(device)
        self.out = torch.empty(wl.B, wl.H, 512, dtype=torch.bfloat16, device=device)
        self.lse = torch.empty(wl.B, wl.H, dtype=torch.float32, device=device)

    def prefill(self):
        """The whole workload through the fused writer in one varlen call
        (inputs far larger than L2); the second of two identical calls (same
        tokens at the same positions, the same bytes written) is timed."""
        inp = self.inp
        self.cache.append(inp["pt"], self.seq, inp["c"], inp["k"], cu_new=self.cu_d)
        self.seq.zero_()
        torch.cuda.synchronize()
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        p0.record()
        self.cache.append(inp["pt"], self.seq, inp["c"], inp["k"], cu_new=self.cu_d)
        p1.record()
        torch.cuda.synchronize()
        assert self.cache.device_status() == 0, "writer reported a device error"
        ms = p0.elapsed_time(p1)
        pf = prefill_bytes(self.wl.seq_lens, self.wl.mode)
        return {"tokens": int(sum(self.wl.seq_lens)), "us": ms * 1e3, "bytes": pf, "GB/s": pf / (ms * 1e-3) / 1e9,
                "how": "varlen mlaq_append of every sequence in one call (the second of two identical calls), "
                       "CUDA events"}

    def append(self, i):
        self.cache.append(self.inp["pt"], self.seq, self.inp["cn"][i], self.inp["kn"][i])

    def decode(self):
        self.cache.decode(self.inp["ql"], self.inp["qr"], self.inp["pt"], self.seq, W.SOFTMAX_SCALE, out=self.out,
                          lse=self.lse)

    def step(self, i):
        self.append(i)
        self.decode()

    def lens(self):
        return [int(x) for x in self.seq.cpu().tolist()]

    def release(self):
        for name in ("inp", "cache", "seq", "cu_d", "out", "lse"):
            setattr(self, name, None)
        torch.cuda.empty_cache()


# GB300 datasheet figures (context beside the measured peaks): HBM3e bandwidth
# and dense bf16 tensor throughput per GPU.
NOMINAL_HBM_GBS = 7900.0
NOMINAL_BF16_TFLOPS = 2250.0


def roofline_for(wl, mean_lens, kern_ms):
    """Roofline of one mlaq_decode call (plan + decode + combine) for the
    workload at the given (mean) sequence lengths."""
    dec_bytes = decode_bytes(mean_lens, wl.mode, wl.B, wl.H)
    hbm, tf_burst, tf_sus, peak_src = load_peaks()
    flops = decode_flops(mean_lens, wl.H)
    t_mem = dec_bytes / (hbm * 1e9)
    t_ten = flops / (tf_burst * 1e12)
    if t_mem >= t_ten:
        achieved = dec_bytes / (kern_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "peak_source": f"{peak_src} hbm_gbs (copy)",
                "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": achieved / NOMINAL_HBM_GBS}
    else:
        achieved = flops / (kern_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": tf_burst, "unit": "TFLOP/s",
                "frac": achieved / tf_burst, "peak_source": f"{peak_src} bf16_tflops (burst)",
                "nominal_peak": NOMINAL_BF16_TFLOPS, "frac_of_nominal": achieved / NOMINAL_BF16_TFLOPS}
    roof["kernel_ms"] = kern_ms
    roof["roofline_us"] = max(t_mem, t_ten) * 1e6
    roof["algorithmic_bytes"] = dec_bytes
    roof["algorithmic_flops"] = flops
    return roof


def measure_steps(wb, K, Wm, l2_flush, ws, device, first_step=0):
    """Wm warm-up steps, K timed steps (events at step boundaries only, L2
    flushed between steps outside the events), then K instrumented steps
    (an event after the append, the library's events around mlaq_decode)."""
    for i in range(Wm):
        l2_flush()
        wb.step(first_step + i)
    torch.cuda.synchronize()
    lens_at_start = wb.lens()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    barrier(ws)
    torch.cuda.synchronize()
    for j in range(K):
        l2_flush()
        evs[j][0].record()
        wb.step(first_step + Wm + j)
        evs[j][1].record()
    torch.cuda.synchronize()
    barrier(ws)
    ms = sum(a.elapsed_time(b) for a, b in evs) / K
    ms_max = max_over_ranks(ms, ws, device)
    wl = wb.wl
    mean_lens = [L + (K - 1) / 2.0 for L in lens_at_start]
    bytes_step = decode_bytes(mean_lens, wl.mode, wl.B, wl.H) + append_bytes(wl.B, wl.mode)
    bytes_all = sum_over_ranks(bytes_step, ws, device)
    lens_inst = wb.lens()
    wb.cache.timing_enable(K)
    ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    mid = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    torch.cuda.synchronize()
    for j in range(K):
        l2_flush()
        ev2[j][0].record()
        wb.append(first_step + Wm + K + j)
        mid[j].record()
        wb.decode()
        ev2[j][1].record()
    torch.cuda.synchronize()
    append_ms = sum(a.elapsed_time(m) for (a, _), m in zip(ev2, mid)) / K
    inst_step_ms = sum(a.elapsed_time(b) for a, b in ev2) / K
    kern_ms = wb.cache.timing_read()
    wb.cache.timing_enable(0)
    kern_avg = sum(kern_ms) / max(len(kern_ms), 1)
    roof = roofline_for(wl, [L + (K - 1) / 2.0 for L in lens_inst], kern_avg)
    assert wb.cache.device_status() == 0, "device error during the benchmark"
    return {"ms_max": ms_max, "bytes_all": bytes_all, "value": bytes_all / (ms_max * 1e-3) / 1e9,
            "lens_at_start": lens_at_start, "append_ms": append_ms, "inst_step_ms": inst_step_ms,
            "kern_avg": kern_avg, "roof": roof}


PER_CONFIG_DEFAULT = "v2lite_c2r4,v2lite_bf16,v3_c4r4,long_c2r4,long_c4r4,long_bf16,serving_c4r4"


def run_per_config(names, K, Wm, l2_flush, ws, rank, device, local, variant=0):
    """The other workloads, each with its own cache, K timed steps and its own
    clock record; one line of numbers per workload."""
    res = {}
    for name in names:
        wl = W.workload(name)
        wb = Workbench(wl, rank, device, Wm + 2 * K, variant)
        pre = wb.prefill()
        sampler = ClockSampler(local)
        sampler.start()
        m = measure_steps(wb, K, Wm, l2_flush, ws, device)
        clocks = sampler.stop()
        roof = m["roof"]
        res[name] = {"workload": wl.description, "steps": K, "warmup": Wm,
                     "step_us": m["ms_max"] * 1e3, "GB/s": m["value"],
                     "decode_call_us": m["kern_avg"] * 1e3, "append_us": m["append_ms"] * 1e3,
                     "roofline": {k: roof[k] for k in ("bound", "achieved", "peak", "unit", "frac", "roofline_us", "frac_of_nominal")},
                     "writer_prefill_GB/s": pre["GB/s"], "clocks": clocks}
        wb.release()
    return res


def compression_record(cache, mode, seq_lens):
    """Persistent-cache accounting through the library (mlaq_cache_bytes):
    policy bytes vs the same sequences in a paged all-BF16 cache."""
    rec = {"how": "mlaq_cache_bytes: BF16 sink/recent ring + packed copies of all tokens + page mapping, "
                  "against a paged all-BF16 cache (onedev.kr system-efficiency paragraph)", "mode": mode}
    for label, lens in (("workload", seq_lens), ("4K", [4096]), ("128K", [131072])):
        pol, ref = cache.cache_bytes(lens)
        rec[label] = {"policy_bytes": pol, "bf16_bytes": ref, "ratio": ref / pol}
    rec["pages_quote"] = {"4K": 3.22, "128K": 3.59}
    return rec


def run_mlaq(args, ws, rank, local):
    from bit_mla_kv_gb300 import build as B
    B.build()

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    wl = W.workload(args.workload)
    K, Wm = args.steps, args.warmup
    wb = Workbench(wl, rank, device, Wm + 3 * K, args.decode_variant)  # warmup + timed + instrumented + e2e steps
    prefill = wb.prefill()
    l2_flush = make_l2_flush(device)
    inp, cache, seq, out, lse = wb.inp, wb.cache, wb.seq, wb.out, wb.lse

    # The clock sampler starts before the warm-up, so that neither its
    # start-up nor an idle GPU sits right before the timed steps.
    sampler = ClockSampler(local)
    sampler.start()
    m = measure_steps(wb, K, Wm, l2_flush, ws, device)
    clocks = sampler.stop()
    ms_max, bytes_all, value = m["ms_max"], m["bytes_all"], m["value"]
    lens_at_start, kern_avg = m["lens_at_start"], m["kern_avg"]
    roof = dict(m["roof"])
    roof["traffic"] = recorded_traffic(args.workload)
    roof["kernel"] = "mlaq_decode: plan_kernel + decode_kernel (split-KV attention) + combine_kernel"
    roof["frac_of_roofline_kernel"] = roof["roofline_us"] * 1e-3 / kern_avg

    # ---- end to end through the public API with host buffers
    # A step's inputs (queries and the new token of every sequence) travel in
    # one pinned buffer and its results (out, lse) in another: one copy each
    # way per step. The copies run on their own streams into double buffers,
    # ordered by events, so step j + 1's inputs move while step j computes
    # (every copy is still inside the timed region). The library is called on
    # views into the device buffers (every view starts 16-byte aligned).
    def as_bytes(t):
        return t.contiguous().view(torch.uint8).reshape(-1)

    parts = [inp["ql"], inp["qr"], inp["cn"][0], inp["kn"][0]]
    sizes = [as_bytes(t).numel() for t in parts]
    offs = [sum(sizes[:i]) for i in range(len(sizes))]
    assert all(o % 16 == 0 for o in offs)
    n_in = sum(sizes)
    n_out = out.numel() * 2
    n_res = n_out + lse.numel() * 4
    h_in = torch.empty(K, n_in, dtype=torch.uint8).pin_memory()
    for j in range(K):
        step_parts = [inp["ql"], inp["qr"], inp["cn"][Wm + 2 * K + j], inp["kn"][Wm + 2 * K + j]]
        h_in[j].copy_(torch.cat([as_bytes(t).cpu() for t in step_parts]))
    h_res = torch.empty(K, n_res, dtype=torch.uint8).pin_memory()
    NBUF = 2
    d_in = [torch.empty(n_in, dtype=torch.uint8, device=device) for _ in range(NBUF)]
    d_res = [torch.empty(n_res, dtype=torch.uint8, device=device) for _ in range(NBUF)]

    def view(buf, i, like):
        return buf[offs[i]:offs[i] + sizes[i]].view(like.dtype).view(like.shape)

    v_ql = [view(d, 0, inp["ql"]) for d in d_in]
    v_qr = [view(d, 1, inp["qr"]) for d in d_in]
    v_cn = [view(d, 2, inp["cn"][0]) for d in d_in]
    v_kn = [view(d, 3, inp["kn"][0]) for d in d_in]
    v_out = [d[:n_out].view(torch.bfloat16).view(out.shape) for d in d_res]
    v_lse = [d[n_out:].view(torch.float32).view(lse.shape) for d in d_res]
    main = torch.cuda.current_stream(device)
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev_in = [torch.cuda.Event() for _ in range(K)]
    ev_done = [torch.cuda.Event() for _ in range(K)]
    ev_out = [torch.cuda.Event() for _ in range(K)]
    h2d = n_in
    d2h = n_res
    # the host-side setup above leaves the GPU idle: a few decode calls (they
    # read the cache and change nothing) keep it busy up to the timed steps
    for _ in range(3):
        wb.decode()
    barrier(ws)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    # The host enqueues every step without waiting for the previous one, as a
    # serving loop would; the time ends when the last step's result is on the
    # host.
    for j in range(K):
        u = j % NBUF
        with torch.cuda.stream(s_in):
            if j >= NBUF:
                s_in.wait_event(ev_done[j - NBUF])  # step j - 2 no longer reads d_in[u]
            d_in[u].copy_(h_in[j], non_blocking=True)
            ev_in[j].record(s_in)
        main.wait_event(ev_in[j])
        if j >= NBUF:
            main.wait_event(ev_out[j - NBUF])  # step j - 2's results left d_res[u]
        cache.append(inp["pt"], seq, v_cn[u], v_kn[u])
        cache.decode(v_ql[u], v_qr[u], inp["pt"], seq, W.SOFTMAX_SCALE, out=v_out[u], lse=v_lse[u])
        ev_done[j].record(main)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[j])
            h_res[j].copy_(d_res[u], non_blocking=True)
            ev_out[j].record(s_out)
    torch.cuda.synchronize()
    e2e_s = (time.perf_counter() - t0) / K
    barrier(ws)
    e2e_s = max_over_ranks(e2e_s, ws, device)
    e2e_val = bytes_all / e2e_s / 1e9
    assert cache.device_status() == 0, "device error during the benchmark"
    compression = compression_record(cache, wl.mode, wl.seq_lens)
    wb.release()
    del d_in, d_res, v_ql, v_qr, v_cn, v_kn, v_out, v_lse

    per_config = None
    names = [n for n in args.per_config.split(",") if n and n != "none" and n != args.workload]
    if names:
        per_config = run_per_config(names, args.per_config_steps, 3, l2_flush, ws, rank, device, local,
                                    args.decode_variant)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        c_host, k_host, cu = inp["c"], inp["k"], inp["cu"]

        def tokens(b):
            a, e = int(cu[b]), int(cu[b + 1])
            return torch.cat([c_host[a:e], k_host[a:e]], -1).float().cpu().numpy()

        qs = (inp["ql"].float().cpu().numpy(), inp["qr"].float().cpu().numpy())
        nb, secs, desc = oracle_sample(tokens, wl.seq_lens, qs, wl.mode, args.cpu_budget)
        cpu = {"value": nb / secs / 1e9, "unit": "GB/s", "cores": cores_used(), "kind": "oracle",
               "sample": desc + f", {secs:.1f} s of fp64 NumPy decode (BLAS threads: default)"}

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": K, "warmup": Wm,
        "ms_per_step": ms_max, "us_per_step": ms_max * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16 MMA operands (int4/int2 codes exact), f32 accumulate",
        "data": "synthetic (seeded; N(0,1) latent with 8 outlier channels x10, RoPE pairs x10^U(-1,1))",
        "config": {"workload": f"{wl.name}: {wl.description}", "mode": wl.mode, "B": wl.B, "H": wl.H,
                   "decode_variant": args.decode_variant,
                   "tokens_at_start": sum(lens_at_start), "step": "mlaq_append (1 token/seq) + mlaq_decode",
                   "l2": "flushed between timed steps, outside the step events: 256 MiB written, then 256 MiB of another buffer read so the flush leaves no dirty lines",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_val, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_s * 1e3,
                "how": "host wall time over K steps; each step copies its inputs (queries and new tokens) "
                       "from one pinned buffer, runs mlaq_append + mlaq_decode on views of that copy and copies "
                       "out/lse back into one pinned buffer; copies on their own streams into double buffers, "
                       "ordered by events, overlap the neighbouring steps' kernels; one synchronize at the end"},
        "gpu_launches": 4 * K,  # per step: append, plan, decode, combine
        "step_breakdown": {"append_us": m["append_ms"] * 1e3, "decode_call_us": kern_avg * 1e3,
                           "step_us": m["inst_step_ms"] * 1e3,
                           "how": "K more steps with an event after the append and the library's events "
                                  "around mlaq_decode (these break the launch overlap the timed steps keep)"},
        "writer_prefill": prefill,
        "compression": compression,
        "per_config": per_config,
        "clocks": clocks,
        "impl": "mlaq",
    }
    if rank == 0:
        print(json.dumps(line))


def run_reference(args, ws, rank):
    """The oracle, as it stands, on the host cores: each step decodes a bounded
    sample of the workload's sequences."""
    if rank != 0:
        return
    wl = W.workload(args.workload)
    g = W.generator(wl.seed, "cpu")
    stats = W.CacheStats(wl.seed)
    # generate only the sampled sequences (the oracle never sees the rest)
    order = sorted(range(wl.B), key=lambda b: wl.seq_lens[b])
    ql, qr = W.make_queries(wl.B, wl.H, g)
    qs = (ql.float().numpy(), qr.float().numpy())
    cache = {}

    def tokens(b):
        if b not in cache:
            gb = W.generator(wl.seed * 7 + b, "cpu")
            c, k = W.make_tokens(wl.seq_lens[b], stats, gb)
            cache[b] = torch.cat([c, k], -1).float().numpy()
        return cache[b]

    per = []
    for i in range(args.warmup + args.steps):
        nb, secs, desc = oracle_sample(tokens, wl.seq_lens, qs, wl.mode, args.ref_budget)
        if i >= args.warmup:
            per.append((nb, secs))
    nb = sum(x for x, _ in per)
    secs = sum(s for _, s in per)
    val = nb / secs / 1e9
    ms = secs / len(per) * 1e3
    line = {
        "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, same distributions)",
        "config": {"workload": f"{wl.name}: {wl.description}", "mode": wl.mode, "B": wl.B, "H": wl.H,
                   "step": "oracle decode of a bounded sample of the batch's sequences"},
        "impl": "reference",
        "cpu_baseline": {"value": val, "unit": "GB/s", "cores": cores_used(), "kind": "oracle",
                         "sample": desc + " per step"},
        "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="v2lite_c4r4")
    ap.add_argument("--impl", default="mlaq", choices=["mlaq", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--ref-budget", type=float, default=2.0, help="seconds of oracle work per reference step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--per-config", default=PER_CONFIG_DEFAULT,
                    help="comma-separated other workloads measured after the headline ('none' to skip)")
    ap.add_argument("--per-config-steps", type=int, default=10)
    ap.add_argument("--decode-variant", type=int, default=0, choices=[0, 1, 2],
                    help="attention kernel: 0 automatic, 1 register scores, 2 tcgen05 scores")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    ws, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, ws, rank)
    else:
        run_mlaq(args, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
