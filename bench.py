#!/usr/bin/env python
"""Benchmark of the NVFP4 paged-KV hot path on GB300; prints one JSON line.

A step is one pass of the whole path over one batch of synthetic input:
  * page round-trip workload (4096 pages x 32 tokens x 8 KV heads x 128, K and V BF16 ~ N(0,1)
    with 1% of blocks x1e3 and 1% x1e-3): tensor amax -> global scale, encode to NVFP4,
    decode to BF16, decode to FP8 E4M3 (output scale amax/448), for K and for V;
  * long-context decode workload (8 sequences of 32K-128K tokens, 64 query / 8 KV heads,
    head_dim 128, 64-token pages, split-KV): paged GQA decode attention over the NVFP4 cache.
`value` is the algorithmic HBM bytes of the step (what each kernel must read and write at
minimum) divided by the step time, in GB/s, summed over ranks. Inputs are larger than the
129 MB L2 and are not reused between kernels of a step except where the path itself reuses
them. Inside the step a launch also pays for writing back the dirty output lines its
predecessors left in L2 (the decode follows the FP8 decode of V); `roofline.achieved` is that
in-step time. Per-kernel numbers are taken separately with an L2 flush before each launch (a
512 MB buffer written, then half of it read back, so that the flush's own write-back is done
before the timed launch), which is the kernel's own time; `roofline.achieved_isolated` is the
decode's.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs its own batch (weak scaling, no data-path collective).
"""
from __future__ import annotations

import argparse
import datetime
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GB = 1e9
# ncu summary of the decode call whose DRAM traffic is reported, valid while the decode
# sources hash to the value recorded in it
DECODE_PROFILE = os.path.join(ROOT, "profiles", "decode_split_kernel_long_context.md")
DECODE_SOURCES = [os.path.join(ROOT, "nvfp4_paged_kv_gb300", "csrc", f)
                  for f in ("decode.cu", "common.cuh")]
METRIC = "NVFP4 paged decode-attn KV GB/s + quant/dequant GB/s, % of GB300 HBM peak"
WORKLOAD = ("page round-trip 4096x32x8x128 K+V (amax, encode, decode->BF16, decode->FP8) + "
            "long-context decode 8 seqs U[32K,128K] 64q/8kv d128 page64 split-KV")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay timing")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-kernels", action="store_true", help="skip per-kernel timings")
    ap.add_argument("--clock-window", type=float, default=1.0,
                    help="seconds of untimed steps under the clock sampler before timing")
    ap.add_argument("--ref-pages", type=int, default=256,
                    help="reference arm: page round-trip pages per step")
    ap.add_argument("--ref-max-tokens", type=int, default=0,
                    help="reference arm: cap on the sampled sequence length (0 = none)")
    ap.add_argument("--profile-case", default="",
                    help="run only one kernel family a few times (for ncu): decode_batch | "
                         "long_context | decode_head_dim_64 | decode_head_dim_256 | "
                         "extend_step | quantize | dequantize | dequantize_fp8 | amax | codec")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------------------- distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def dist_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() \
        else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling during the timed region (SM clock, throttle reasons)."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None
        self.t_load = None

    def mark_load(self):
        """Samples taken before this moment (sampler start-up, idle) are dropped."""
        self.t_load = time.time()

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    t = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    t = None
                if self.t_load is not None and t is not None and t < self.t_load:
                    continue
                rows.append(parts[1:])
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")
        sm = [num(r[1]) for r in rows]
        smax = [num(r[2]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].lower().startswith("active")})
        loaded = [s for s in sm if math.isfinite(s)]
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(x for x in smax if math.isfinite(x)) if smax else None,
                "reasons": reasons, "samples": len(rows)}


def decode_traffic():
    """DRAM bytes (read + write) of one long-context decode call from the committed ncu
    summary, or None when the decode sources changed since that capture."""
    import hashlib
    try:
        h = hashlib.sha256()
        for f in DECODE_SOURCES:
            with open(f, "rb") as fh:
                h.update(fh.read())
        fields = {}
        with open(DECODE_PROFILE) as fh:
            for line in fh:
                if ":" in line and line.startswith(("traffic_bytes_per_call", "sources_sha256")):
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip().strip("`")
        if fields.get("sources_sha256") == h.hexdigest():
            return int(fields["traffic_bytes_per_call"])
    except (OSError, KeyError, ValueError):
        pass
    return None


# ---------------------------------------------------------------------------- the path

class Path:
    """Device buffers of both workloads and the launches of one step."""

    def __init__(self, kv, dev, seed):
        import torch
        import synthetic
        self.kv, self.dev = kv, dev
        # page round-trip workload
        rt = synthetic.RoundTripWorkload(seed=seed)
        self.rt = rt
        self.k, self.v = rt.make(device=dev)
        P, H, T, D = rt.P, rt.H, rt.T, rt.D
        self.lay_rt = kv.Layout(H, D, T)
        # K pages in the dim-pair packing, V pages in the token-pair packing (what decode reads)
        self.lay_rt_kv = (self.lay_rt, self.lay_rt.with_packing(kv.PACK_TOKEN_PAIRS))
        u8 = torch.uint8
        self.rt_out = []
        for _ in range(2):
            self.rt_out.append(dict(
                g=torch.empty(1, dtype=torch.float32, device=dev),
                data=torch.empty((P, H, T, D // 2), dtype=u8, device=dev),
                scales=torch.empty((P, H, T, D // 16), dtype=u8, device=dev),
                bf16=torch.empty((P, H, T, D), dtype=torch.bfloat16, device=dev),
                fp8=torch.empty((P, H, T, D), dtype=u8, device=dev),
                fp8_scale=torch.empty(1, dtype=torch.float32, device=dev)))
        self.gs_ws = torch.empty(kv.nvfp4_kv_global_scale_workspace_size(), dtype=u8,
                                 device=dev)
        for src, o in zip((self.k, self.v), self.rt_out):
            # FP8 workspace scale amax / 448 (= 6 g), fixed per tensor at set-up
            o["fp8_scale"].copy_(src.float().abs().max() / 448.0)
        n_rt = P * H * T * D
        self.bytes_rt = {
            "amax": 2 * n_rt * 2,
            "quantize": 2 * n_rt * (2 + 0.5625),
            "dequantize_bf16": 2 * n_rt * (0.5625 + 2),
            "dequantize_fp8": 2 * n_rt * (0.5625 + 1),
        }
        # long-context decode workload: NVFP4 cache built once by the encoder
        wl = synthetic.long_context(seed=seed)
        self.wl = wl
        q, k, v, pt, sl = wl.make(device=dev)
        self.lay_lc = kv.Layout(wl.H, wl.D, wl.T)
        self.q, self.pt, self.sl = q, pt, sl
        Pl = wl.pool_pages
        mk = lambda w: torch.empty((Pl, wl.H, wl.T, w), dtype=u8, device=dev)  # noqa: E731
        self.c_kd, self.c_ks, self.c_vd, self.c_vs = mk(wl.D // 2), mk(wl.D // 16), \
            mk(wl.D // 2), mk(wl.D // 16)
        self.c_gk = torch.empty(1, dtype=torch.float32, device=dev)
        self.c_gv = torch.empty(1, dtype=torch.float32, device=dev)
        kv.nvfp4_kv_compute_global_scale(self.lay_lc, k, self.c_gk, workspace=self.gs_ws)
        kv.nvfp4_kv_compute_global_scale(self.lay_lc, v, self.c_gv, workspace=self.gs_ws)
        kv.nvfp4_kv_quantize_pages(self.lay_lc, k, self.c_gk, self.c_kd, self.c_ks)
        kv.nvfp4_kv_quantize_pages(self.lay_lc.with_packing(kv.PACK_TOKEN_PAIRS), v, self.c_gv,
                                   self.c_vd, self.c_vs)
        del k, v
        self.out = torch.empty((wl.B, wl.Hq, wl.D), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((wl.B, wl.Hq), dtype=torch.float32, device=dev)
        wsb = kv.nvfp4_paged_decode_workspace_size(self.lay_lc, wl.B, wl.Hq, pt.shape[1], 0)
        self.dec_ws = torch.empty(wsb, dtype=u8, device=dev)
        kv_tokens = wl.kv_tokens
        # per (token, KV head): K and V packed data D/2 each + K and V scales D/16 each
        self.bytes_decode = (kv_tokens * wl.H * (wl.D + wl.D // 8)          # K+V data+scales
                             + wl.B * wl.Hq * wl.D * 2 * 2                   # q in, out
                             + pt.numel() * 4 + wl.B * 4 + wl.B * wl.Hq * 4)  # table, lens, lse
        self.decode_tokens = wl.B
        self.launches_per_step = 2 + 2 + 4 + 1   # amax x2, quantize x2, dequantize x4, decode 1
        torch.cuda.synchronize()

    # individual launches --------------------------------------------------------------
    def amax(self, i):
        src = (self.k, self.v)[i]
        self.kv.nvfp4_kv_compute_global_scale(self.lay_rt, src, self.rt_out[i]["g"],
                                              workspace=self.gs_ws)

    def quantize(self, i):
        o = self.rt_out[i]
        self.kv.nvfp4_kv_quantize_pages(self.lay_rt_kv[i], (self.k, self.v)[i], o["g"],
                                        o["data"], o["scales"])

    def dequantize_bf16(self, i):
        o = self.rt_out[i]
        self.kv.nvfp4_kv_dequantize_pages(self.lay_rt_kv[i], o["data"], o["scales"], o["g"],
                                          o["bf16"])

    def dequantize_fp8(self, i):
        o = self.rt_out[i]
        self.kv.nvfp4_kv_dequantize_pages(self.lay_rt_kv[i], o["data"], o["scales"], o["g"],
                                          o["fp8"], dst_dtype=self.kv.FP8_E4M3,
                                          dst_scale=o["fp8_scale"])

    def decode(self):
        wl = self.wl
        self.kv.nvfp4_paged_decode_attention(
            self.lay_lc, self.q, self.c_kd, self.c_ks, self.c_gk, self.c_vd, self.c_vs,
            self.c_gv, self.pt, self.sl, wl.sm_scale, self.out, lse=self.lse,
            workspace=self.dec_ws)

    def step(self, dec_events=None):
        for i in range(2):
            self.amax(i)
            self.quantize(i)
            self.dequantize_bf16(i)
            self.dequantize_fp8(i)
        if dec_events is not None:
            dec_events[0].record()
        self.decode()
        if dec_events is not None:
            dec_events[1].record()

    @property
    def step_bytes(self):
        return sum(self.bytes_rt.values()) + self.bytes_decode


def time_kernel(fn, flush, reps=25):
    """CUDA-event time (ms) of fn() with an L2 flush before each launch: the flush buffer (4x L2)
    is written, then its first half is read back, so that the write-back of the dirty flush
    lines happens before the timed launch and the launch starts on an L2 holding only clean
    lines of another buffer. CUDA event times come in steps of about 2 us, so the figure is the
    mean of the middle 60 % of the launches (finer than one step) rather than their median (a
    whole number of steps)."""
    import torch
    ts = []
    half = flush[: flush.numel() // 2]
    for _ in range(reps):
        flush.fill_(1)
        half.max()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    ts.sort()
    k = len(ts) // 5
    mid = ts[k:len(ts) - k]
    return sum(mid) / len(mid)


def error_vs_unquantized(q, k, v, pt, sl, out, sm_scale):
    """What NVFP4 costs in accuracy: the decode output (NVFP4 K/V) against attention over the
    unquantized BF16 K/V pages, computed here in plain PyTorch fp32 on the device (a reporting
    reference, not part of the path)."""
    import torch
    B, Hq, D = q.shape
    H, T = k.shape[1], k.shape[2]
    G = Hq // H
    diffs, refs = [], []
    for b in range(B):
        L = int(sl[b])
        n = (L + T - 1) // T
        ids = pt[b, :n].long()
        kb = k[ids].permute(1, 0, 2, 3).reshape(H, n * T, D)[:, :L].float()
        vb = v[ids].permute(1, 0, 2, 3).reshape(H, n * T, D)[:, :L].float()
        qb = q[b].float().reshape(H, G, D)
        s = torch.einsum("hgd,htd->hgt", qb, kb) * sm_scale
        ref = torch.einsum("hgt,htd->hgd", torch.softmax(s, dim=-1), vb).reshape(Hq, D)
        diffs.append((out[b].float() - ref).flatten())
        refs.append(ref.flatten())
    d = torch.cat(diffs)
    rf = torch.cat(refs)
    return {"vs": "attention over the unquantized BF16 K/V (PyTorch fp32)",
            "max_abs": round(float(d.abs().max()), 6), "mean_abs": round(float(d.abs().mean()), 6),
            "rel_rmse": round(float(d.pow(2).mean().sqrt() / rf.pow(2).mean().sqrt()), 6)}


def kernel_table(path, peak):
    """Per-kernel achieved GB/s (L2 flushed before every launch), plus the decode-batch
    workload and the extend workload as extra single-kernel cases."""
    import torch
    import synthetic
    kv, dev = path.kv, path.dev
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    res = {}

    def add(name, fn, nbytes, launches, extra=None):
        ms = time_kernel(fn, flush)
        gbs = nbytes / (ms * 1e-3) / GB
        d = {"ms": round(ms, 4), "bytes": int(nbytes), "GB_s": round(gbs, 1),
             "frac_of_peak": round(gbs / peak, 4), "launches": launches}
        if extra:
            d.update(extra)
        res[name] = d

    n = path.rt.P * path.rt.H * path.rt.T * path.rt.D
    add("amax_K (page round-trip)", lambda: path.amax(0), n * 2, 1)
    add("quantize_K dim pairs (page round-trip)", lambda: path.quantize(0), n * 2.5625, 1)
    add("quantize_V token pairs (page round-trip)", lambda: path.quantize(1), n * 2.5625, 1)
    add("dequantize_K_bf16 (page round-trip)", lambda: path.dequantize_bf16(0), n * 2.5625, 1)
    add("dequantize_V_bf16 token pairs (page round-trip)", lambda: path.dequantize_bf16(1),
        n * 2.5625, 1)
    add("dequantize_K_fp8 (page round-trip)", lambda: path.dequantize_fp8(0), n * 1.5625, 1)
    add("dequantize_V_fp8 token pairs (page round-trip)", lambda: path.dequantize_fp8(1),
        n * 1.5625, 1)
    wl = path.wl
    add("decode (long context)", path.decode, path.bytes_decode, 1,
        {"kv_tokens": wl.kv_tokens})
    res["decode (long context)"]["kv_tokens_per_s"] = round(
        wl.kv_tokens / (res["decode (long context)"]["ms"] * 1e-3), 1)
    # decode batch workload (32 x 8192 tokens, GQA 4)
    db = synthetic.decode_batch(seed=1)
    q, k, v, pt, sl = db.make(device=dev)
    lay = kv.Layout(db.H, db.D, db.T)
    u8 = torch.uint8
    P = db.pool_pages
    kd = torch.empty((P, db.H, db.T, db.D // 2), dtype=u8, device=dev)
    ks = torch.empty((P, db.H, db.T, db.D // 16), dtype=u8, device=dev)
    vd, vs = torch.empty_like(kd), torch.empty_like(ks)
    gk = torch.empty(1, dtype=torch.float32, device=dev)
    gv = torch.empty(1, dtype=torch.float32, device=dev)
    kv.nvfp4_kv_compute_global_scale(lay, k, gk)
    kv.nvfp4_kv_compute_global_scale(lay, v, gv)
    kv.nvfp4_kv_quantize_pages(lay, k, gk, kd, ks)
    kv.nvfp4_kv_quantize_pages(lay.with_packing(kv.PACK_TOKEN_PAIRS), v, gv, vd, vs)
    out = torch.empty((db.B, db.Hq, db.D), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(kv.nvfp4_paged_decode_workspace_size(lay, db.B, db.Hq, pt.shape[1], 0),
                     dtype=u8, device=dev)
    kv.nvfp4_paged_decode_attention(lay, q, kd, ks, gk, vd, vs, gv, pt, sl, db.sm_scale, out,
                                    workspace=ws)
    qerr = error_vs_unquantized(q, k, v, pt, sl, out, db.sm_scale)
    del k, v
    nbytes = db.kv_tokens * db.H * (db.D + db.D // 8) + db.B * db.Hq * db.D * 4 + \
        pt.numel() * 4 + db.B * 4
    add("decode (decode batch 32x8192, GQA 4)",
        lambda: kv.nvfp4_paged_decode_attention(lay, q, kd, ks, gk, vd, vs, gv, pt, sl,
                                                db.sm_scale, out, workspace=ws),
        nbytes, 1)
    r = res["decode (decode batch 32x8192, GQA 4)"]
    r["decode_tokens_per_s"] = round(db.B / (r["ms"] * 1e-3), 1)
    r["kv_tokens_per_s"] = round(db.kv_tokens / (r["ms"] * 1e-3), 1)
    r["error_vs_unquantized_bf16"] = qerr
    del kd, ks, vd, vs, q, out, ws
    # extend workload: gather + dequantize a 1024-page prefix into FP8, encode a 128-page chunk
    ex = synthetic.ExtendWorkload(seed=2)
    prefix, ept, chunk, chunk_dst = ex.make(device=dev)
    lay = kv.Layout(ex.H, ex.D, ex.T)
    pool = prefix.shape[0]
    pd = torch.empty((pool, ex.H, ex.T, ex.D // 2), dtype=u8, device=dev)
    ps = torch.empty((pool, ex.H, ex.T, ex.D // 16), dtype=u8, device=dev)
    g = torch.empty(1, dtype=torch.float32, device=dev)
    kv.nvfp4_kv_compute_global_scale(lay, prefix, g)
    kv.nvfp4_kv_quantize_pages(lay, prefix, g, pd, ps)
    ids = ept.reshape(-1).contiguous()
    wsp = torch.empty((ids.numel(), ex.H, ex.T, ex.D), dtype=u8, device=dev)
    per = ex.H * ex.T * ex.D
    add("extend prefix gather->FP8 (1024 pages)",
        lambda: kv.nvfp4_kv_dequantize_pages(lay, pd, ps, g, wsp, dst_dtype=kv.FP8_E4M3,
                                             src_page_ids=ids),
        ids.numel() * per * 1.5625 + ids.numel() * 4, 1)
    add("extend chunk encode (128 pages)",
        lambda: kv.nvfp4_kv_quantize_pages(lay, chunk, g, pd, ps, dst_page_ids=chunk_dst),
        chunk.shape[0] * per * 2.5625 + chunk.shape[0] * 4, 1)
    # fused extend write: the chunk read once, NVFP4 pages + its FP8 workspace copy written
    wsc = torch.empty((chunk.shape[0], ex.H, ex.T, ex.D), dtype=u8, device=dev)
    add("extend chunk write NVFP4 + FP8 workspace (128 pages)",
        lambda: kv.nvfp4_kv_extend_write(lay, chunk, g, pd, ps, wsc, dst_page_ids=chunk_dst),
        chunk.shape[0] * per * 3.5625 + chunk.shape[0] * 4, 1)
    # the same two chunk calls as a serving loop issues them, back to back over 12 rotating
    # chunks (the K and V chunks of 6 layers: 201 MB of inputs, more than L2), per launch
    nrot = 12
    chunks = [synthetic.kv_pages_bf16(chunk.shape[0], ex.H, ex.T, ex.D,
                                      synthetic.gen(50 + r, device=dev), device=dev)
              for r in range(nrot)]
    wss = [torch.empty_like(wsc) for _ in range(nrot)]
    for name, fn, bpv in (
            ("extend chunk encode (128 pages, 12 chunks back to back)",
             lambda r: kv.nvfp4_kv_quantize_pages(lay, chunks[r], g, pd, ps,
                                                  dst_page_ids=chunk_dst), 2.5625),
            ("extend chunk write NVFP4 + FP8 workspace (128 pages, 12 chunks back to back)",
             lambda r: kv.nvfp4_kv_extend_write(lay, chunks[r], g, pd, ps, wss[r],
                                                dst_page_ids=chunk_dst), 3.5625)):
        ms = time_kernel(lambda: [fn(r) for r in range(nrot)], flush) / nrot
        nbytes = chunk.shape[0] * per * bpv + chunk.shape[0] * 4
        gbs = nbytes / (ms * 1e-3) / GB
        res[name] = {"ms": round(ms, 4), "bytes": int(nbytes), "GB_s": round(gbs, 1),
                     "frac_of_peak": round(gbs / peak, 4), "launches": nrot}
    del chunks, wss
    extend_step_table(path, flush, peak, res)
    decode_extra_table(path, flush, peak, res)
    res.update(cold_table(path, flush, time_kernel))
    del flush
    # codec throughput in tokens: a launch encodes or decodes P pages of T tokens of one tensor
    tok = path.rt.P * path.rt.T
    for name, r in res.items():
        if name.startswith(("quantize_", "dequantize_", "amax_")):
            r["tokens_per_s"] = round(tok / (r["ms"] * 1e-3), 1)
    return res


def per_config(result, peak):
    """Fractions of the measured copy peak for each workload the targets name, from the kernel
    table (each call timed alone after an L2 flush) and, where a serving loop issues the call
    back to back, from that timing too."""
    k = result["kernels"]
    pick = lambda name: {key: k[name][key] for key in  # noqa: E731
                         ("ms", "GB_s", "frac_of_peak", "bytes") if key in k[name]}
    out = {
        "page_roundtrip_quantize": {n: pick(n) for n in k if n.startswith("quantize_")},
        "page_roundtrip_dequantize": {n: pick(n) for n in k if n.startswith("dequantize_")},
        "decode_batch": dict(pick("decode (decode batch 32x8192, GQA 4)"),
                             back_to_back=pick("decode (decode batch 32x8192, GQA 4), back to back")),
        "long_context": dict(pick("decode (long context)"),
                             in_step={"ms": result["roofline"]["launch_ms"],
                                      "frac_of_peak": result["roofline"]["frac"]}),
        "extend_step": dict(pick("extend step: K+V prefix gather -> FP8 + K+V chunk write "
                                 "(one launch)"),
                            four_launches=pick("extend step: K+V prefix gather -> FP8 + K+V "
                                               "chunk write (4 launches back to back)")),
        "decode_head_dim_64": pick("decode (32x8192, GQA 4, head_dim 64)"),
        "decode_head_dim_256": pick("decode (32x8192, GQA 4, head_dim 256)"),
    }
    out["peak_GB_s"] = peak
    return out


def decode_cache(kv, dev, wl, seed_shift=0):
    """NVFP4 K (dim pairs) and V (token pairs) pools of a decode workload, encoded on the GPU,
    with its queries, page table and lengths; the BF16 sources are dropped."""
    import torch
    q, k, v, pt, sl = wl.make(device=dev)
    lay = kv.Layout(wl.H, wl.D, wl.T)
    u8 = torch.uint8
    P = wl.pool_pages
    c = dict(lay=lay, q=q, pt=pt, sl=sl)
    c["kd"] = torch.empty((P, wl.H, wl.T, wl.D // 2), dtype=u8, device=dev)
    c["ks"] = torch.empty((P, wl.H, wl.T, wl.D // 16), dtype=u8, device=dev)
    c["vd"], c["vs"] = torch.empty_like(c["kd"]), torch.empty_like(c["ks"])
    c["gk"] = torch.empty(1, dtype=torch.float32, device=dev)
    c["gv"] = torch.empty(1, dtype=torch.float32, device=dev)
    kv.nvfp4_kv_compute_global_scale(lay, k, c["gk"])
    kv.nvfp4_kv_compute_global_scale(lay, v, c["gv"])
    kv.nvfp4_kv_quantize_pages(lay, k, c["gk"], c["kd"], c["ks"])
    kv.nvfp4_kv_quantize_pages(lay.with_packing(kv.PACK_TOKEN_PAIRS), v, c["gv"], c["vd"], c["vs"])
    c["out"] = torch.empty((wl.B, wl.Hq, wl.D), dtype=torch.bfloat16, device=dev)
    c["ws"] = torch.empty(kv.nvfp4_paged_decode_workspace_size(lay, wl.B, wl.Hq, pt.shape[1], 0),
                          dtype=u8, device=dev)
    del k, v
    return c


def decode_call(kv, wl, c):
    return lambda: kv.nvfp4_paged_decode_attention(
        c["lay"], c["q"], c["kd"], c["ks"], c["gk"], c["vd"], c["vs"], c["gv"], c["pt"], c["sl"],
        wl.sm_scale, c["out"], workspace=c["ws"])


def decode_bytes(wl, pt):
    return (wl.kv_tokens * wl.H * (wl.D + wl.D // 8) + wl.B * wl.Hq * wl.D * 4 +
            pt.numel() * 4 + wl.B * 4)


def decode_extra_table(path, flush, peak, res):
    """The decode batch issued back to back as a serving loop issues decode steps (two NVFP4
    caches of 302 MB used in turn, so no call finds its inputs in the 129 MB L2; launches overlap
    through programmatic dependent launch), and the decode batch at head_dim 64 and 256."""
    import torch
    import synthetic
    kv, dev = path.kv, path.dev
    wl = synthetic.decode_batch(seed=1)
    caches = [decode_cache(kv, dev, wl), decode_cache(kv, dev, synthetic.decode_batch(seed=11))]
    calls = [decode_call(kv, wl, c) for c in caches]
    nbytes = decode_bytes(wl, caches[0]["pt"])
    n = 20
    for cl in calls * 2:
        cl()
    torch.cuda.synchronize()
    ts = []
    for _ in range(5):
        flush.fill_(1)
        flush[: flush.numel() // 2].max()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for i in range(n):
            calls[i % 2]()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b) / n)
    ms = statistics.median(ts)
    gbs = nbytes / (ms * 1e-3) / GB
    res["decode (decode batch 32x8192, GQA 4), back to back"] = {
        "ms": round(ms, 4), "bytes": int(nbytes), "GB_s": round(gbs, 1),
        "frac_of_peak": round(gbs / peak, 4), "launches": n,
        "decode_tokens_per_s": round(wl.B / (ms * 1e-3), 1),
        "kv_tokens_per_s": round(wl.kv_tokens / (ms * 1e-3), 1),
        "method": "20 calls back to back over two caches used in turn (each 302 MB, above L2)"}
    del caches, calls
    for D in (64, 256):
        wl = synthetic.DecodeWorkload(f"decode batch head_dim {D}", B=32, Hq=32, H=8, D=D, T=64,
                                      seq_lens=[8192] * 32, pool_pages=4096, seed=1)
        c = decode_cache(kv, dev, wl)
        nbytes = decode_bytes(wl, c["pt"])
        ms = time_kernel(decode_call(kv, wl, c), flush)
        gbs = nbytes / (ms * 1e-3) / GB
        res[f"decode (32x8192, GQA 4, head_dim {D})"] = {
            "ms": round(ms, 4), "bytes": int(nbytes), "GB_s": round(gbs, 1),
            "frac_of_peak": round(gbs / peak, 4), "launches": 1,
            "kv_tokens_per_s": round(wl.kv_tokens / (ms * 1e-3), 1)}
        del c


def extend_step_table(path, flush, peak, res):
    """The extend workload as one step: for K and for V, the 4096-token NVFP4 prefix of each of
    16 sequences gathered and dequantized into the FP8 workspace, and the 512-token BF16 chunk
    written as NVFP4 pages and as its FP8 workspace copy: four launches back to back (K gather,
    V gather, K chunk write, V chunk write), timed as one after an L2 flush."""
    kv, dev = path.kv, path.dev
    ex, tens, step, parts = extend_setup(kv, dev)

    def fused():
        kv.nvfp4_kv_extend_step(parts)
    H, T, D = ex.H, ex.T, ex.D
    vals = H * T * D
    gather = 2 * ex.prefix_pages * vals * 1.5625 + 2 * ex.prefix_pages * 4
    write = 2 * ex.chunk_pages * vals * (2 + 0.5625 + 1) + 2 * ex.chunk_pages * 4
    for name, fn, launches in (
            ("extend step: K+V prefix gather -> FP8 + K+V chunk write (4 launches back to back)",
             step, 4),
            ("extend step: K+V prefix gather -> FP8 + K+V chunk write (one launch)", fused, 1)):
        ms = time_kernel(fn, flush)
        gbs = (gather + write) / (ms * 1e-3) / GB
        res[name] = {
            "ms": round(ms, 4), "bytes": int(gather + write), "GB_s": round(gbs, 1),
            "frac_of_peak": round(gbs / peak, 4), "launches": launches,
            "bytes_gather": int(gather), "bytes_chunk_write": int(write),
            "tokens_per_s": round(ex.B * (ex.prefix + ex.chunk) / (ms * 1e-3), 1)}
    del tens, parts


def extend_setup(kv, dev):
    """The extend workload's K and V tensors (NVFP4 prefix pools encoded on the GPU, BF16
    chunks, FP8 workspaces), the four-launch step and the fused call's parts."""
    import torch
    import synthetic
    ex = synthetic.ExtendWorkload(seed=2)
    H, T, D = ex.H, ex.T, ex.D
    lay = kv.Layout(H, D, T)
    u8 = torch.uint8
    per_seq = ex.prefix // T + ex.chunk // T          # workspace slots of one sequence
    slots = torch.arange(ex.B * per_seq, dtype=torch.int32, device=dev).view(ex.B, per_seq)
    ws_prefix = slots[:, :ex.prefix // T].reshape(-1).contiguous()
    ws_chunk = slots[:, ex.prefix // T:].reshape(-1).contiguous()
    tens = []
    for t, (packing, seed) in enumerate(((kv.PACK_DIM_PAIRS, 2), (kv.PACK_TOKEN_PAIRS, 3))):
        exs = synthetic.ExtendWorkload(seed=seed)
        prefix, ept, chunk, chunk_dst = exs.make(device=dev)
        ly = lay.with_packing(packing)
        pool = prefix.shape[0]
        d = dict(lay=ly, ids=ept.reshape(-1).contiguous(), chunk=chunk, chunk_dst=chunk_dst)
        d["pd"] = torch.empty((pool, H, T, D // 2), dtype=u8, device=dev)
        d["ps"] = torch.empty((pool, H, T, D // 16), dtype=u8, device=dev)
        d["g"] = torch.empty(1, dtype=torch.float32, device=dev)
        kv.nvfp4_kv_compute_global_scale(ly, prefix, d["g"])
        kv.nvfp4_kv_quantize_pages(ly, prefix, d["g"], d["pd"], d["ps"])
        d["ws"] = torch.empty((ex.B * per_seq, H, T, D), dtype=u8, device=dev)
        del prefix
        tens.append(d)

    def step():
        for d in tens:
            kv.nvfp4_kv_dequantize_pages(d["lay"], d["pd"], d["ps"], d["g"], d["ws"],
                                         dst_dtype=kv.FP8_E4M3, src_page_ids=d["ids"],
                                         dst_page_ids=ws_prefix)
        for d in tens:
            kv.nvfp4_kv_extend_write(d["lay"], d["chunk"], d["g"], d["pd"], d["ps"], d["ws"],
                                     dst_page_ids=d["chunk_dst"], ws_page_ids=ws_chunk)
    parts = [dict(layout=d["lay"], global_scale=d["g"], data=d["pd"], scales=d["ps"],
                  prefix_page_ids=d["ids"], ws=d["ws"], ws_prefix_ids=ws_prefix,
                  ws_chunk_ids=ws_chunk, chunk=d["chunk"], chunk_dst_ids=d["chunk_dst"])
             for d in tens]
    return ex, tens, step, parts


def cold_table(path, flush, timer, pages=2048):
    """Cold-page codec over the host link: offload (encode fused with the write of the cold
    blocks into pinned host memory) and onboard (decode fused with the read back), for `pages`
    pages of the round-trip workload (K and V, 32 tokens x 8 heads x 128 dims per page), with
    the RoPE part of K (head dims 64..127) quantized like the rest, kept at 16 bits, or stored
    as two NVFP4 components. Each line carries the measured time of a plain copy of the same
    cold bytes over the same link (the bound) and of a plain copy of the uncompressed 16-bit
    pages (what a codec that only concatenates the pools would move)."""
    import torch
    kv, rt = path.kv, path.rt
    H, T, D = rt.H, rt.T, rt.D
    lay = kv.Layout(H, D, T)
    n = min(pages, rt.P)
    hk, hv = path.k[:n], path.v[:n]
    gk, gv = path.rt_out[0]["g"], path.rt_out[1]["g"]
    hot_h = torch.empty((2, n, H, T, D), dtype=torch.bfloat16).pin_memory()
    back_k, back_v = torch.empty_like(hk), torch.empty_like(hv)
    hot_bytes = 2 * n * H * T * D * 2
    t_d2h_hot = timer(lambda: (hot_h[0].copy_(hk, non_blocking=True),
                               hot_h[1].copy_(hv, non_blocking=True)), flush)
    t_h2d_hot = timer(lambda: (back_k.copy_(hot_h[0], non_blocking=True),
                               back_v.copy_(hot_h[1], non_blocking=True)), flush)
    out = {}
    for label, rope in (("", None), (", RoPE dims kept 16-bit", kv.ColdRope(kv.ROPE_SKIP, 64, 64)),
                        (", RoPE dims 2FP4", kv.ColdRope(kv.ROPE_2FP4, 64, 64))):
        bl = kv.nvfp4_kv_cold_block_layout(lay, 0, rope)
        cold_h = torch.empty((n, bl.bytes), dtype=torch.uint8).pin_memory()
        cold_d = torch.empty((n, bl.bytes), dtype=torch.uint8, device=path.dev)
        cold_bytes = n * bl.bytes
        t_off = timer(lambda: kv.nvfp4_kv_offload_pages(lay, hk, hv, cold_h, k_global_scale=gk,
                                                        v_global_scale=gv, rope=rope), flush)
        t_on = timer(lambda: kv.nvfp4_kv_onboard_pages(lay, cold_h, back_k, back_v,
                                                       k_global_scale=gk, v_global_scale=gv,
                                                       rope=rope), flush)
        t_d2h = timer(lambda: cold_h.copy_(cold_d, non_blocking=True), flush)
        t_h2d = timer(lambda: cold_d.copy_(cold_h, non_blocking=True), flush)
        for name, t, t_copy, t_hot, direction in (
                ("cold offload K+V -> pinned host (%d pages%s)" % (n, label), t_off, t_d2h,
                 t_d2h_hot, "d2h"),
                ("cold onboard pinned host -> K+V (%d pages%s)" % (n, label), t_on, t_h2d,
                 t_h2d_hot, "h2d")):
            out[name] = {
                "ms": round(t, 4), "bound": "host link (" + direction + ")",
                "link_bytes": int(cold_bytes), "hbm_bytes": int(hot_bytes),
                "bits_per_value": round(cold_bytes * 8 / (2 * n * H * T * D), 4),
                "link_GB_s": round(cold_bytes / (t * 1e-3) / GB, 1),
                "plain_copy_ms": round(t_copy, 4),
                "plain_copy_GB_s": round(cold_bytes / (t_copy * 1e-3) / GB, 1),
                "frac_of_plain_copy": round(t_copy / t, 4),
                "uncompressed_copy_ms": round(t_hot, 4),
                "speedup_vs_uncompressed_copy": round(t_hot / t, 3),
                "launches": 1}
        del cold_h, cold_d
    del hot_h, back_k, back_v
    return out


def scale_stats(kv, lay, x, g_t):
    """Encode BF16 pages x ([P, H, T, D]) with the global scale in g_t (device scalar) and decode
    them back to BF16, both through the library; return the error and the scale-range counts:
    blocks whose E4M3 scale rounds to 0 (every value of the block decodes to 0), blocks whose
    scale is subnormal (below 2^-6: fewer than 4 significant bits), blocks whose scale saturates
    (amax / (6 g) above 464, the midpoint between 448 and the next E4M3 step, so rounding alone
    would not bring it to 448), and the values the range clips (|x| above 7 * 448 g, the
    midpoint beyond the largest code 6 at the largest scale)."""
    import torch
    P, H, T, D = x.shape
    u8 = torch.uint8
    data = torch.empty((P, H, T, D // 2), dtype=u8, device=x.device)
    scales = torch.empty((P, H, T, D // 16), dtype=u8, device=x.device)
    kv.nvfp4_kv_quantize_pages(lay, x, g_t, data, scales)
    y = torch.empty_like(x)
    kv.nvfp4_kv_dequantize_pages(lay, data, scales, g_t, y)
    g = float(g_t.item())
    xf, yf = x.float().view(-1, 16), y.float().view(-1, 16)
    err = xf - yf
    amax = xf.abs().amax(1)
    s = scales.view(-1).to(torch.int32)
    nz = amax > 0
    lim = 7.0 * 448.0 * g
    rel_blk = (err.abs().amax(1)[nz] / amax[nz])
    return {
        "g": g,
        "blocks": int(xf.shape[0]),
        "rel_rmse": float(err.pow(2).sum().sqrt() / xf.pow(2).sum().sqrt()),
        "mean_block_rel_max_err": float(rel_blk.mean()),
        "blocks_zero_scale": int(((s == 0) & nz).sum()),
        "blocks_subnormal_scale": int((((s & 0x78) == 0) & (s != 0)).sum()),
        "blocks_saturated_scale": int((amax / (6.0 * g) > 464.0).sum()),
        "values_clipped": int((xf.abs() > lim).sum()),
    }


def global_scale_study(path):
    """Error and scale-range counts of the unit global scale (g = 1) against the calibrated one
    (g = amax / 2688) on the synthetic distributions."""
    import torch
    import synthetic
    kv, dev = path.kv, path.dev
    cases = {}
    rt = path.rt
    lay = kv.Layout(rt.H, rt.D, rt.T)
    gen = synthetic.gen(7, device=dev)
    cases["N(0,1), 1% blocks x1e3, 1% x1e-3 (round-trip K, 4096 pages)"] = (path.k, lay)
    db = synthetic.decode_batch()
    cases["N(0,1), K channels 13/42/77/118 x20 (decode K, 1024 pages)"] = (
        synthetic.kv_pages_bf16(1024, db.H, db.T, db.D, gen, k_outliers=True, device=dev),
        kv.Layout(db.H, db.D, db.T))
    cases["N(0,1) (V, 1024 pages)"] = (
        synthetic.kv_pages_bf16(1024, db.H, db.T, db.D, gen, device=dev),
        kv.Layout(db.H, db.D, db.T))
    out = {}
    for name, (x, ly) in cases.items():
        g_cal = torch.empty(1, dtype=torch.float32, device=dev)
        kv.nvfp4_kv_compute_global_scale(ly, x, g_cal)
        g_one = torch.ones(1, dtype=torch.float32, device=dev)
        out[name] = {"unit": scale_stats(kv, ly, x, g_one),
                     "calibrated": scale_stats(kv, ly, x, g_cal)}
    torch.cuda.synchronize()
    return out


# ---------------------------------------------------------------------------- CPU baseline

def oracle_sample(seed=0, pages=1024, decode_seqs=1, max_tokens=None):
    """Run the oracle on a bounded sample of the same workload; returns (bytes, seconds,
    threads, description)."""
    import numpy as np
    import torch
    import oracle
    import synthetic
    rt = synthetic.RoundTripWorkload(P=pages, seed=seed)
    k, _ = rt.make()
    kb = synthetic.bf16_bits(k)
    H, D, T = rt.H, rt.D, rt.T
    n = kb.size
    t0 = time.perf_counter()
    g = oracle.global_scale(kb, oracle.BF16, H, D, T)
    d, s = oracle.quantize_pages(kb, oracle.BF16, H, D, T, g)
    oracle.dequantize_pages(d, s, H, D, T, g, oracle.BF16)
    oracle.dequantize_pages(d, s, H, D, T, g, oracle.FP8_E4M3, out_scale=6 * g)
    t_codec = time.perf_counter() - t0
    codec_bytes = n * (2 + 2.5625 + 2.5625 + 1.5625)
    # decode: the first `decode_seqs` sequences of the long-context workload, all 64 heads
    wl = synthetic.long_context(seed=seed)
    lens = wl.seq_lens[:decode_seqs]
    if max_tokens:
        lens = [min(L, max_tokens) for L in lens]
    T2 = wl.T
    dpages = sum(-(-L // T2) for L in lens)
    g2 = synthetic.gen(seed + 7)
    q = synthetic.randn_bf16((decode_seqs, wl.Hq, wl.D), g2)
    kd = np.random.default_rng(seed).integers(0, 256, (dpages, wl.H, T2, wl.D // 2), np.uint8)
    ks = np.random.default_rng(seed + 1).integers(0x20, 0x48, (dpages, wl.H, T2, wl.D // 16),
                                                  np.uint8)
    vd = np.random.default_rng(seed + 2).integers(0, 256, kd.shape, np.uint8)
    vs = np.random.default_rng(seed + 3).integers(0x20, 0x48, ks.shape, np.uint8)
    maxp = max(-(-L // T2) for L in lens)
    pt = np.zeros((decode_seqs, maxp), np.int32)
    off = 0
    for b, L in enumerate(lens):
        npg = -(-L // T2)
        pt[b, :npg] = np.arange(off, off + npg)
        off += npg
    t0 = time.perf_counter()
    oracle.paged_decode_attention(synthetic.bf16_bits(q), kd, ks, 0.01, vd, vs, 0.01, pt,
                                  np.array(lens, np.int32), wl.sm_scale, wl.H, T2)
    t_dec = time.perf_counter() - t0
    dec_bytes = sum(lens) * wl.H * (wl.D + wl.D // 8)
    desc = (f"oracle on {rt.P} page round-trip pages of K (amax, encode, decode BF16 + FP8) and "
            f"{decode_seqs} long-context sequence(s) ({sum(lens)} tokens, {wl.Hq} query heads) "
            f"over random NVFP4 K/V bytes of the cache's shape (the oracle's time does not "
            f"depend on the values)")
    return codec_bytes + dec_bytes, t_codec + t_dec, oracle.max_threads(), desc


def workload_config(seed):
    """The `config` object of both arms' lines: what the step runs on, nothing measured."""
    import synthetic
    return {"workload": WORKLOAD,
            "l2": "inputs larger than L2 (129 MB); kernel table: L2 flushed before each launch "
                  "(512 MB written, then 256 MB of it read)",
            "long_context_seq_lens": synthetic.long_context_lengths(seed)}


def run_reference(args):
    """The oracle as the reference arm: each step is a bounded sample of the workload."""
    world, rank, local = dist_setup()
    if rank != 0:
        return
    import oracle
    oracle.build()
    kw = dict(pages=args.ref_pages, decode_seqs=1, max_tokens=args.ref_max_tokens or None)
    for _ in range(args.warmup):
        oracle_sample(args.seed, **kw)
    tot_b, tot_t = 0.0, 0.0
    desc, thr = "", 1
    for _ in range(args.steps):
        b, t, thr, desc = oracle_sample(args.seed, **kw)
        tot_b += b
        tot_t += t
    v = tot_b / tot_t / GB
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot_t / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args.seed),
        "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": thr,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}))


# ---------------------------------------------------------------------------- main

def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    import torch
    world, rank, local = dist_setup()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the NVFP4 KV path has no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import nvfp4_paged_kv_gb300 as kv
    from nvfp4_paged_kv_gb300 import build
    build.build()
    kv.load()
    peak, peak_kind = peaks()

    if args.profile_case:
        profile_case(kv, dev, args.profile_case)
        return

    path = Path(kv, dev, args.seed + 1000 * rank)
    for _ in range(args.warmup):
        path.step()
    torch.cuda.synchronize()
    barrier(world)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        # keep the GPU loaded for about a second of sampling before the timed region, so the
        # nvidia-smi samples (every 200 ms) see the clocks under this load
        clk.mark_load()
        t_end = time.time() + args.clock_window
        while time.time() < t_end:
            for _ in range(8):
                path.step()
            torch.cuda.synchronize()
        start.record()
        for i in range(args.steps):
            path.step(ev[i])
        end.record()
        torch.cuda.synchronize()
    barrier(world)
    ms_total = dist_max(start.elapsed_time(end), world)
    ms_step = ms_total / args.steps
    dec_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    step_bytes = path.step_bytes
    value = step_bytes * world / (ms_step * 1e-3) / GB
    clocks = clk.summary()
    clocks["window"] = f"{args.clock_window:g} s of untimed steps, then the timed steps"

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp32",
        "dtype_detail": ("NVFP4 storage (E2M1 codes, E4M3 block scales, FP32 tensor scale); "
                         "encode arithmetic in FP32; decode attention on FP16 tensor-core "
                         "operands (exact dequantized K/V) with FP32 accumulation"),
        "data": "synthetic",
        "config": workload_config(args.seed),
        "bytes_per_step_per_gpu": int(step_bytes),
        "peak": {"GB_s": peak, "kind": peak_kind, "frac": round(value / world / peak, 4)},
        "roofline": {"bound": "hbm", "kernel": "decode_split_kernel (nvfp4_paged_decode_attention, one launch)",
                     "achieved": round(path.bytes_decode / (dec_ms * 1e-3) / GB, 1),
                     "peak": peak, "unit": "GB/s",
                     "frac": round(path.bytes_decode / (dec_ms * 1e-3) / GB / peak, 4),
                     "traffic": decode_traffic(), "peak_kind": peak_kind,
                     "launch_ms": round(dec_ms, 4), "algorithmic_bytes": int(path.bytes_decode)},
        "clocks": clocks,
        "gpu_launches": path.launches_per_step * args.steps,
    }
    if not args.no_graph:
        result["graph"] = graph_replay(path, args, world, step_bytes, peak)
    if not args.no_kernels and rank == 0:
        result["kernels"] = kernel_table(path, peak)
        result["global_scale_study"] = global_scale_study(path)
        iso = result["kernels"]["decode (long context)"]
        result["roofline"]["achieved_isolated"] = iso["GB_s"]
        result["roofline"]["frac_isolated"] = iso["frac_of_peak"]
        result["roofline"]["launch_ms_isolated"] = iso["ms"]
        result["roofline"]["per_config"] = per_config(result, peak)
    if not args.no_e2e:
        result["e2e"] = e2e(path, args, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        b, t, thr, desc = oracle_sample(args.seed, pages=4096, decode_seqs=8)
        result["cpu_baseline"] = {"value": round(b / t / GB, 4), "unit": "GB/s", "cores": thr,
                                  "kind": "oracle", "sample": desc,
                                  "seconds": round(t, 2)}
    if rank == 0:
        print(json.dumps(result))


def graph_replay(path, args, world, step_bytes, peak):
    """The same step captured once in a CUDA graph and replayed (the 9 launches of a step go
    to the GPU as one graph launch); reported beside the eager number, not instead of it."""
    import torch
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        path.step()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    barrier(world)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(args.steps):
        graph.replay()
    end.record()
    torch.cuda.synchronize()
    barrier(world)
    ms = dist_max(start.elapsed_time(end), world) / args.steps
    value = step_bytes * world / (ms * 1e-3) / GB
    del graph
    return {"value": round(value, 2), "unit": "GB/s", "ms_per_step": round(ms, 4),
            "frac_of_peak": round(value / world / peak, 4)}


def e2e(path, args, world):
    """Same metric through the public API with host buffers: every step copies its inputs from
    pinned host memory and reads every result back. The inputs of a step are the 16-bit K/V
    pages of the round trip and the decode's queries, page table and lengths; the NVFP4 cache the
    decode reads is state that stays in HBM from step to step (the encoder fills it once, as a
    serving loop keeps its cache on the GPU). Steps are pipelined over two sets of device
    buffers and three streams (host->device copies of step i+1 and device->host copies of step
    i-1 run while step i computes), as a serving loop would."""
    import torch
    dev = path.dev
    sets = [path, Path(path.kv, dev, args.seed + 1000 * int(os.environ.get("RANK", "0")))]

    def ins_of(pth):
        return [pth.k, pth.v, pth.q, pth.pt, pth.sl]

    def outs_of(pth):
        return [pth.rt_out[i][key] for i in range(2)
                for key in ("g", "data", "scales", "bf16", "fp8")] + [pth.out, pth.lse]

    h_in = [t.cpu().pin_memory() for t in ins_of(path)]
    h_out = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs_of(pth)]
             for pth in sets]
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = sum(t.numel() * t.element_size() for t in h_out[0])
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def launch(i):
        j = i % 2
        pth = sets[j]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_comp[j])   # step i-2 is done reading this set's inputs
            for h, d in zip(h_in, ins_of(pth)):
                d.copy_(h, non_blocking=True)
            ev_in[j].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(ev_in[j])
            if i >= 2:
                s_comp.wait_event(ev_out[j])  # step i-2's results are copied out
            pth.step()
            ev_comp[j].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[j])
            for h, d in zip(h_out[j], outs_of(pth)):
                h.copy_(d, non_blocking=True)
            ev_out[j].record(s_out)

    for i in range(max(2, args.warmup)):
        launch(i)
    torch.cuda.synchronize()
    barrier(world)
    n = max(4, args.steps // 2)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for i in range(n):
        launch(i)
    b.record(s_out)  # the last device->host copy is the last work of the timed steps
    torch.cuda.synchronize()
    barrier(world)
    ms = dist_max(a.elapsed_time(b), world) / n

    # the host link as these pinned buffers see it, alone: one copy each way of the largest
    # input and output buffers (context for the figure above, which is bound by this link)
    def link_gbs(stream, dst, src):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            dst.copy_(src, non_blocking=True)    # warm
            e0.record(stream)
            dst.copy_(src, non_blocking=True)
            e1.record(stream)
        torch.cuda.synchronize()
        return round(src.numel() * src.element_size() / (e0.elapsed_time(e1) * 1e-3) / GB, 1)

    big_in = max(range(len(h_in)), key=lambda i: h_in[i].numel() * h_in[i].element_size())
    big_out = max(range(len(h_out[0])), key=lambda i: h_out[0][i].numel() * h_out[0][i].element_size())
    h2d_gbs = link_gbs(s_in, ins_of(path)[big_in], h_in[big_in])
    d2h_gbs = link_gbs(s_out, h_out[0][big_out], outs_of(path)[big_out])
    return {"value": round(path.step_bytes * world / (ms * 1e-3) / GB, 2), "unit": "GB/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": round(ms, 3), "pipelined": "2 buffer sets, 3 streams",
            "resident": "the long-context NVFP4 cache (filled once by the encoder)",
            "link_alone_GB_s": {"h2d": h2d_gbs, "d2h": d2h_gbs}}


def profile_case(kv, dev, case):
    """A few launches of one kernel family on one workload, for ncu captures."""
    import torch
    import synthetic
    u8 = torch.uint8
    if case == "extend_step":
        _, _, _, parts = extend_setup(kv, dev)
        for _ in range(4):
            kv.nvfp4_kv_extend_step(parts)
    elif case in ("decode_batch", "long_context", "decode_head_dim_64", "decode_head_dim_256"):
        if case == "decode_batch":
            wl = synthetic.decode_batch()
        elif case == "long_context":
            wl = synthetic.long_context()
        else:
            D = int(case.rsplit("_", 1)[1])
            wl = synthetic.DecodeWorkload(f"decode batch head_dim {D}", B=32, Hq=32, H=8, D=D,
                                          T=64, seq_lens=[8192] * 32, pool_pages=4096, seed=1)
        q, k, v, pt, sl = wl.make(device=dev)
        lay = kv.Layout(wl.H, wl.D, wl.T)
        P = wl.pool_pages
        kd = torch.empty((P, wl.H, wl.T, wl.D // 2), dtype=u8, device=dev)
        ks = torch.empty((P, wl.H, wl.T, wl.D // 16), dtype=u8, device=dev)
        vd, vs = torch.empty_like(kd), torch.empty_like(ks)
        gk = torch.empty(1, dtype=torch.float32, device=dev)
        gv = torch.empty(1, dtype=torch.float32, device=dev)
        kv.nvfp4_kv_compute_global_scale(lay, k, gk)
        kv.nvfp4_kv_compute_global_scale(lay, v, gv)
        kv.nvfp4_kv_quantize_pages(lay, k, gk, kd, ks)
        kv.nvfp4_kv_quantize_pages(lay.with_packing(kv.PACK_TOKEN_PAIRS), v, gv, vd, vs)
        del k, v
        out = torch.empty((wl.B, wl.Hq, wl.D), dtype=torch.bfloat16, device=dev)
        for _ in range(4):
            kv.nvfp4_paged_decode_attention(lay, q, kd, ks, gk, vd, vs, gv, pt, sl,
                                            wl.sm_scale, out)
    else:
        rt = synthetic.RoundTripWorkload()
        k, _ = rt.make(device=dev)
        lay = kv.Layout(rt.H, rt.D, rt.T)
        g = torch.empty(1, dtype=torch.float32, device=dev)
        d = torch.empty((rt.P, rt.H, rt.T, rt.D // 2), dtype=u8, device=dev)
        s = torch.empty((rt.P, rt.H, rt.T, rt.D // 16), dtype=u8, device=dev)
        kv.nvfp4_kv_compute_global_scale(lay, k, g)
        kv.nvfp4_kv_quantize_pages(lay, k, g, d, s)
        if case == "codec":
            # after the 2 set-up launches: one launch of each codec kernel on the K pages
            o8 = torch.empty(k.shape, dtype=u8, device=dev)
            kb = torch.empty_like(k)
            kv.nvfp4_kv_compute_global_scale(lay, k, g)
            kv.nvfp4_kv_quantize_pages(lay, k, g, d, s)
            kv.nvfp4_kv_dequantize_pages(lay, d, s, g, kb)
            kv.nvfp4_kv_dequantize_pages(lay, d, s, g, o8, dst_dtype=kv.FP8_E4M3)
        for _ in range(4 if case != "codec" else 0):
            if case == "quantize":
                kv.nvfp4_kv_quantize_pages(lay, k, g, d, s)
            elif case == "dequantize":
                kv.nvfp4_kv_dequantize_pages(lay, d, s, g, k)
            elif case == "dequantize_fp8":
                o = torch.empty(k.shape, dtype=u8, device=dev)
                kv.nvfp4_kv_dequantize_pages(lay, d, s, g, o, dst_dtype=kv.FP8_E4M3)
            else:
                kv.nvfp4_kv_compute_global_scale(lay, k, g)
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": case, "ok": True}))


if __name__ == "__main__":
    main()
