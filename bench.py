#!/usr/bin/env python
"""Benchmark: one displaced denoising step of the whole hot path per step.

A step runs, through the C ABI, on the SDXL-3840px-with-guidance workload
(latent 480x480, batch 2 = conditional + unconditional, 8 bands):
  1. displaced 3x3 conv 320->320 on [2,480,480,320], its
     epilogue also summing the output per band and group  (dpp_conv3x3_gn)
  2. displaced GroupNorm (32 groups) on the conv output,
     one pass on those sums                                (dpp_groupnorm_apply)
  3. displaced self-attention, 2 x 57600 tokens, C=640,
     10 heads of 64: QKV projection writing the fresh K/V
     state, attention core, output projection             (dpp_self_attn)
  4. cross-attention of the result over 77 x 2048 text
     context tokens, whose K/V were projected once per
     prompt at set-up                                      (dpp_cross_attn_cached)
  5. guidance combine + rel-MAE sums, 2 x [4,480,480] fp32 (dpp_cfg_combine)
  6. refresh of the conv's stale buffer with this step's
     input (the all_gather)                                (dpp_refresh_stale)
The GroupNorm statistics and attention K/V states ping-pong between two
buffers, as consecutive denoising steps do.

Printed metric: tensor TFLOP/s of the step (conv + self-attention core and
projections + cross-attention; the bandwidth ops add time but no FLOPs),
with per-op numbers and roofline fractions (of the measured burst bf16 peak,
and of the sustained one) alongside.  The step's inputs and working set
(~2.5 GB) exceed the 126 MB L2; GroupNorm, refresh and guidance are also
timed alone with L2 flushed before every rep, and `per_config` times every
op of every workload that way (contractions warm, bandwidth ops cold).  A
run whose kernels recorded a timeout (dpp_device_status) exits 1.

After the step, `block_chain` reports one level of the U-Net stepped the same
way (ResNet block + transformer block at 2 x 240 x 240 x 640, 8 bands;
14 ops per step through the same library), timed per displaced step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--no-chain] [--no-cpu-baseline]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as wl  # noqa: E402

METRIC = "displaced-patch conv/attn TFLOP/s, GroupNorm GB/s; % of B300 roofline"
WORKLOAD = "sdxl_3840_cfg"
# adaptive switching controller of the end-to-end loop: relative-drop and
# rise tolerances and patience (the pages give no values)
SWITCH_FLAT_TOL, SWITCH_RISE_TOL, SWITCH_PATIENCE = 0.02, 0.05, 2
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


# ------------------------------------------------------------------ work model
def work_model(w):
    """Algorithmic FLOPs / bytes per step (counting rules of the method's ops:
    tensor-core MMAs only; GroupNorm = read x + write y; refresh = read +
    write the band; guidance = read u, c + write out)."""
    c, a = w.conv, w.attn
    conv = 2.0 * c.B * c.H * c.W * c.C * 9 * c.C
    core = 4.0 * a.B * a.N * a.N * a.head_dim * a.heads
    proj = 2.0 * a.B * a.N * a.C * 3 * a.C + 2.0 * a.B * a.N * a.C * a.C
    cross = a.n_ctx > 0
    xq_o = 2.0 * 2.0 * a.B * a.N * a.C * a.C if cross else 0.0
    # the context's K/V are projected once per prompt (dpp_cross_attn_kv),
    # not per denoising step: counted apart
    xkv = 2.0 * a.B * a.n_ctx * a.c_ctx * 2 * a.C
    xcore = 4.0 * a.B * a.N * a.n_ctx * a.head_dim * a.heads
    act_bytes = c.B * c.H * c.W * c.C * 2
    n_cfg = int(np.prod(w.cfg_shape)) if w.cfg_shape else 0
    return {
        "conv_flop": conv, "self_core_flop": core, "self_proj_flop": proj,
        "cross_flop": xq_o + xcore, "cross_core_flop": xcore, "cross_kv_flop_per_prompt": xkv,
        "gn_bytes": 2.0 * act_bytes, "refresh_bytes": 2.0 * act_bytes,
        "cfg_bytes": 3.0 * 4 * n_cfg,
        "step_flop": conv + core + proj + xq_o + xcore,
    }


def attn_traffic():
    """DRAM bytes per launch of the attention core from the committed ncu
    summary, or None when the kernel sources have changed since it was taken
    (the summary records a SHA-256 of k_attn_tc.cu + tc_common.cuh)."""
    import hashlib
    here = os.path.dirname(os.path.abspath(__file__))
    try:
        text = open(os.path.join(here, "profiles", "dram_bytes_sdxl_3840_cfg.md")).read()
        rec = dict(l.strip().split(": ", 1) for l in text.splitlines()
                   if l.strip().startswith("attn_tc_"))
        h = hashlib.sha256()
        for f in ("k_attn_tc.cu", "tc_common.cuh"):
            with open(os.path.join(here, "displaced_patch_parallelism_02_b300", "csrc", f),
                      "rb") as fh:
                h.update(fh.read())
        if h.hexdigest() != rec["attn_tc_source_sha256"]:
            return None
        return int(rec["attn_tc_dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device_index: int):
        self.dev = self._gpu_id(device_index)
        self.proc = None
        self.lines = []

    @staticmethod
    def _gpu_id(idx):
        try:
            u = str(torch.cuda.get_device_properties(idx).uuid)
            return u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            return vis.split(",")[idx] if vis else str(idx)

    def start(self):
        cmd = ["nvidia-smi", "-i", self.dev, "--query-gpu=" + ",".join(self.FIELDS),
               "--format=csv,noheader,nounits", "-lms", "100"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
                pw.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------ per-op timing
def l2_flusher(dev):
    """A call that evicts L2: it writes a buffer of twice the L2 size (a torch
    fill, run outside the timed events)."""
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 << 20))
    buf = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)

    def flush():
        buf.fill_(1.0)
    return flush, 2 * l2


def timed(call, stream, reps, warmup=3, flush=None, core=None):
    """Median milliseconds of `reps` calls, each between two CUDA events on
    `stream` (after `warmup` untimed calls); `flush` runs before every timed
    call, outside its events.  With `core` (the stream on which to create the
    events the library records around the attention core,
    dpp_set_attn_core_events) every rep gets its own pair of core events, so
    the reps are queued back to back as in a step -- no host synchronisation,
    and no host launch time, between them -- and the median of the core's own
    times is returned as well."""
    import displaced_patch_parallelism_02_b300 as dpp
    for _ in range(warmup):
        call()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    cores = [core_event_pair(core) for _ in range(reps)] if core is not None else None
    for i in range(reps):
        if flush:
            flush()
        if cores:
            dpp.dpp_set_attn_core_events(*cores[i])
        evs[i][0].record(stream)
        call()
        evs[i][1].record(stream)
        if cores:
            dpp.dpp_set_attn_core_events(None, None)
    torch.cuda.synchronize()
    ms = statistics.median(a.elapsed_time(b) for a, b in evs)
    if cores:
        return ms, statistics.median(a.elapsed_time(b) for a, b in cores)
    return ms


def core_event_pair(stream):
    """Two timing events for dpp_set_attn_core_events; recording them once
    creates the CUDA events, which the library then re-records."""
    pair = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    for e in pair:
        e.record(stream)
    return pair


class ConfigOps:
    """Every op of one workload timed on its own, through the C ABI: the conv
    (plain and with the GroupNorm band sums), GroupNorm (single pass on the
    conv's sums, and the two-read entry point), the stale refresh,
    self-attention (whole call and its core), cross-attention and the
    guidance combine.  Contractions run warm, back to back; the bandwidth
    ops (GroupNorm, refresh, guidance) run with L2 flushed before every
    rep, so their GB/s are cold-cache figures."""

    def __init__(self, w, dev):
        import displaced_patch_parallelism_02_b300 as dpp
        self.dpp, self.w, self.dev = dpp, w, dev
        self.s = torch.cuda.current_stream(dev)
        self.code = dpp.DPP_BF16 if w.dtype == "bf16" else dpp.DPP_F32
        tdt = wl.torch_dtype(w.dtype)
        put = lambda t: t.contiguous().to(dev)
        self.c = c = w.conv
        if c:
            shape = (c.B, c.H, c.W, c.C)
            F = wl.normal(shape, wl.seed_of(w.index, 0, wl.T_FRESH), dtype=w.dtype)
            self.x = put(F)
            self.stale = put(wl.perturbed(F, wl.seed_of(w.index, 1, wl.T_STALE_NOISE),
                                          w.stale_scale))
            del F
            self.wconv = put(wl.conv_weight(c.C, c.C, wl.seed_of(w.index, 0, wl.T_CONV_W),
                                            w.dtype).permute(0, 2, 3, 1))
            self.y1 = torch.empty(shape, dtype=tdt, device=dev)
            self.y2 = torch.empty(shape, dtype=tdt, device=dev)
            g, b = wl.gn_affine(c.C, w.index)
            self.gamma, self.beta = put(g), put(b)
            self.cd = dpp.dpp_conv_desc(c.B, c.H, c.W, c.C, c.C, c.P, self.code, 0)
            self.gd = dpp.dpp_gn_desc(c.B, c.H, c.W, c.C, w.groups, c.P, w.eps, self.code)
            self.gws_n = dpp.dpp_groupnorm_workspace_bytes(self.gd)
            self.gws = torch.empty(max(self.gws_n, 16), dtype=torch.uint8, device=dev)
            self.stats = [torch.zeros((c.P, c.B, w.groups, 2), device=dev) for _ in range(2)]
            self.sums = torch.zeros((c.P, c.B, w.groups, 2), dtype=torch.float64, device=dev)
            self.act_bytes = c.B * c.H * c.W * c.C * self.y1.element_size()
        self.a = a = w.attn
        if a:
            X = wl.normal((a.B, a.N, a.C), wl.seed_of(w.index, 0, wl.T_ATTN_X), dtype=w.dtype)
            self.xa = put(X)
            del X
            self.aw = {k: put(v) for k, v in wl.attn_weights(a, w.index, w.dtype).items()}
            kvt = torch.float16 if w.dtype == "bf16" else torch.float32
            self.kv = [torch.empty((a.B, a.N, 2, a.C), dtype=kvt, device=dev) for _ in range(2)]
            self.ya = torch.empty((a.B, a.N, a.C), dtype=tdt, device=dev)
            self.ad = dpp.dpp_attn_desc(a.B, a.H, a.W, a.C, a.heads, a.head_dim, a.P, 0, 0,
                                        self.code)
            self.aws_n = dpp.dpp_self_attn_workspace_bytes(self.ad)
            self.aws = torch.empty(self.aws_n, dtype=torch.uint8, device=dev)
            self.cross = a.n_ctx > 0
            if self.cross:
                self.xw = {k: put(v) for k, v in wl.cross_weights(a, w.index, w.dtype).items()}
                self.ctx = put(wl.context(a, w.index, w.dtype))
                self.xd = dpp.dpp_attn_desc(a.B, a.H, a.W, a.C, a.heads, a.head_dim, 1, a.n_ctx,
                                            a.c_ctx, self.code)
                self.xcws_n = dpp.dpp_cross_attn_cached_workspace_bytes(self.xd)
                self.xcws = torch.empty(self.xcws_n, dtype=torch.uint8, device=dev)
                self.yc = torch.empty_like(self.ya)
                self.kvc = torch.empty((a.B, a.n_ctx, 2, a.C), dtype=kvt, device=dev)
                dpp.dpp_cross_attn_kv(self.xd, self.ctx, self.xw["wk"], self.xw["wv"], self.kvc,
                                      stream=self.s)
            # K/V state of the previous step: a synchronous call fills it
            dpp.dpp_self_attn(self.ad, self.xa, self.aw["wq"], self.aw["wk"], self.aw["wv"],
                              self.aw["wo"], None, self.kv[0], self.ya, self.aws, self.aws_n,
                              stream=self.s)
        self.has_cfg = w.cfg_shape is not None
        if self.has_cfg:
            u, cc = wl.guidance_maps(w.cfg_shape, w.index)
            self.u, self.cm = put(u), put(cc)
            self.n_cfg = u.numel()
            self.cfg_out = torch.empty_like(self.u)
            self.csums = torch.zeros(3, dtype=torch.float64, device=dev)
            self.cws_n = dpp.dpp_cfg_workspace_bytes(self.n_cfg)
            self.cws = torch.zeros(self.cws_n, dtype=torch.uint8, device=dev)
        torch.cuda.synchronize(dev)

    def run(self, reps, peaks, flush):
        dpp, s, w, c, a = self.dpp, self.s, self.w, self.c, self.a
        out = {"workload": w.name, "dtype": w.dtype}
        tf = lambda f, ms: f / (ms / 1e3) / 1e12
        gb = lambda b, ms: b / (ms / 1e3) / 1e9
        burst, hbm = peaks["bf16_tflops"], peaks["hbm_gbs"]

        def tensor_op(flop, ms, **kw):
            d = {"ms": ms, "tflops": tf(flop, ms)}
            if w.dtype == "bf16":
                d["frac_of_burst_bf16"] = d["tflops"] / burst
            d.update(kw)
            return d

        def hbm_op(nbytes, ms, **kw):
            d = {"ms": ms, "gbs": gb(nbytes, ms), "frac_of_hbm": gb(nbytes, ms) / hbm,
                 "l2": "flushed before every rep"}
            d.update(kw)
            return d

        if c:
            conv_f = 2.0 * c.B * c.H * c.W * c.C * 9 * c.C
            ms = timed(lambda: dpp.dpp_conv3x3(self.cd, self.x, self.stale, self.wconv, None,
                                               self.y1, stream=s), s, reps)
            out["conv"] = tensor_op(conv_f, ms, entry="dpp_conv3x3")
            if w.dtype == "bf16":
                ms = timed(lambda: dpp.dpp_conv3x3_gn(self.cd, self.x, self.stale, self.wconv,
                                                      None, self.y1, w.groups, self.sums,
                                                      stream=s), s, reps)
                out["conv_gn_sums"] = tensor_op(conv_f, ms, entry="dpp_conv3x3_gn")
                ms = timed(lambda: dpp.dpp_groupnorm_apply(self.gd, self.y1, self.stats[0],
                                                           self.sums, self.stats[1], self.gamma,
                                                           self.beta, self.y2, stream=s),
                           s, reps, flush=flush)
                out["groupnorm_apply"] = hbm_op(2.0 * self.act_bytes, ms,
                                                entry="dpp_groupnorm_apply (one pass)")
            ms = timed(lambda: dpp.dpp_groupnorm(self.gd, self.y1, self.stats[0], self.stats[1],
                                                 self.gamma, self.beta, self.y2, self.gws,
                                                 self.gws_n, stream=s), s, reps, flush=flush)
            out["groupnorm"] = hbm_op(2.0 * self.act_bytes, ms,
                                      entry="dpp_groupnorm (sums its own input)")
            ms = timed(lambda: dpp.dpp_refresh_stale(self.x, self.stale, c.B, c.H,
                                                     c.W * c.C * self.x.element_size(), c.P,
                                                     stream=s), s, reps, flush=flush)
            out["refresh"] = hbm_op(2.0 * self.act_bytes, ms, entry="dpp_refresh_stale")
        if a:
            core_f = 4.0 * a.B * a.N * a.N * a.head_dim * a.heads
            proj_f = 2.0 * a.B * a.N * a.C * 4 * a.C
            ms, cms = timed(lambda: dpp.dpp_self_attn(
                self.ad, self.xa, self.aw["wq"], self.aw["wk"], self.aw["wv"], self.aw["wo"],
                self.kv[0], self.kv[1], self.ya, self.aws, self.aws_n, stream=s),
                s, max(3, reps // 2), core=s)
            out["self_attn"] = tensor_op(core_f + proj_f, ms, entry="dpp_self_attn")
            out["self_attn_core"] = tensor_op(core_f, cms, entry="attention core alone")
            out["self_attn_projections"] = tensor_op(proj_f, ms - cms,
                                                     entry="QKV + output projections")
            if self.cross:
                xf = (2.0 * 2.0 * a.B * a.N * a.C * a.C
                      + 4.0 * a.B * a.N * a.n_ctx * a.head_dim * a.heads)
                kvf = 2.0 * a.B * a.n_ctx * a.c_ctx * 2 * a.C
                ms, cms = timed(lambda: dpp.dpp_cross_attn_cached(
                    self.xd, self.ya, self.kvc, self.xw["wq"], self.xw["wo"], self.yc,
                    self.xcws, self.xcws_n, stream=s), s, reps, core=s)
                out["cross_attn"] = tensor_op(xf, ms, entry="dpp_cross_attn_cached (per step)")
                out["cross_attn_core"] = tensor_op(4.0 * a.B * a.N * a.n_ctx * a.head_dim * a.heads,
                                                   cms, entry="attention core over 77 keys")
                ms = timed(lambda: dpp.dpp_cross_attn_kv(self.xd, self.ctx, self.xw["wk"],
                                                         self.xw["wv"], self.kvc, stream=s),
                           s, reps)
                out["cross_attn_kv"] = tensor_op(kvf, ms, entry="dpp_cross_attn_kv (per prompt)")
        if self.has_cfg:
            ms = timed(lambda: dpp.dpp_cfg_combine(self.u, self.cm, w.cfg_scale, self.n_cfg,
                                                   self.cfg_out, self.csums, self.cws,
                                                   self.cws_n, stream=s), s, reps, flush=flush)
            out["cfg"] = hbm_op(3.0 * 4 * self.n_cfg, ms, entry="dpp_cfg_combine")
        return out


def per_config(dev, reps, peaks, names):
    """ConfigOps over the named workloads, one at a time (buffers freed in
    between).  Returns {workload name: per-op figures}."""
    flush, _ = l2_flusher(dev)
    res = {}
    for name in names:
        ops = ConfigOps(wl.WORKLOADS[name], dev)
        res[name] = ops.run(reps, peaks, flush)
        del ops
        torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------------ our step
class Step:
    """Device buffers and one displaced step of the hot path through the C ABI."""

    def __init__(self, w, dev):
        import displaced_patch_parallelism_02_b300 as dpp
        self.dpp = dpp
        self.w = w
        c, a = w.conv, w.attn
        bf = torch.bfloat16
        self.stream = torch.cuda.current_stream(dev)
        put = lambda t: t.contiguous().to(dev)
        shape = (c.B, c.H, c.W, c.C)
        F = wl.normal(shape, wl.seed_of(w.index, 0, wl.T_FRESH), dtype=w.dtype)
        S = wl.perturbed(F, wl.seed_of(w.index, 1, wl.T_STALE_NOISE), w.stale_scale)
        self.host_x = F.pin_memory()
        self.x, self.stale = put(F), put(S)
        del F, S
        self.wconv = put(wl.conv_weight(c.C, c.C, wl.seed_of(w.index, 0, wl.T_CONV_W),
                                        w.dtype).permute(0, 2, 3, 1))
        self.y1 = torch.empty(shape, dtype=bf, device=dev)
        self.y2 = torch.empty(shape, dtype=bf, device=dev)
        g, b = wl.gn_affine(c.C, w.index)
        self.gamma, self.beta = put(g), put(b)
        self.gn_desc = dpp.dpp_gn_desc(c.B, c.H, c.W, c.C, w.groups, c.P, w.eps, dpp.DPP_BF16)
        self.gn_ws_n = dpp.dpp_groupnorm_workspace_bytes(self.gn_desc)
        self.gn_ws = torch.empty(self.gn_ws_n, dtype=torch.uint8, device=dev)
        self.stats = [torch.empty((c.P, c.B, w.groups, 2), device=dev) for _ in range(2)]
        # band sums of the conv output, written by the conv's epilogue
        self.gn_sums = torch.empty((c.P, c.B, w.groups, 2), dtype=torch.float64, device=dev)
        self.conv_desc = dpp.dpp_conv_desc(c.B, c.H, c.W, c.C, c.C, c.P, dpp.DPP_BF16, 0)
        # attention level
        X = wl.normal((a.B, a.N, a.C), wl.seed_of(w.index, 0, wl.T_ATTN_X), dtype=w.dtype)
        Xs = wl.perturbed(X, wl.seed_of(w.index, 1, wl.T_ATTN_X), w.stale_scale)
        self.host_xa = X.pin_memory()
        self.xa = put(X)
        xs = put(Xs)
        del X, Xs
        self.aw = {k: put(v) for k, v in wl.attn_weights(a, w.index, w.dtype).items()}
        self.cross = a.n_ctx > 0
        self.xw = ({k: put(v) for k, v in wl.cross_weights(a, w.index, w.dtype).items()}
                   if self.cross else {})
        ctx = wl.context(a, w.index, w.dtype) if self.cross else torch.zeros(16)
        self.host_ctx = ctx.pin_memory()
        self.ctx = put(ctx)
        self.attn_desc = dpp.dpp_attn_desc(a.B, a.H, a.W, a.C, a.heads, a.head_dim, a.P, 0, 0,
                                           dpp.DPP_BF16)
        self.cross_desc = dpp.dpp_attn_desc(a.B, a.H, a.W, a.C, a.heads, a.head_dim, 1,
                                            a.n_ctx, a.c_ctx, dpp.DPP_BF16)
        self.sa_ws_n = dpp.dpp_self_attn_workspace_bytes(self.attn_desc)
        self.sa_ws = torch.empty(self.sa_ws_n, dtype=torch.uint8, device=dev)
        self.xa_ws_n = (dpp.dpp_cross_attn_cached_workspace_bytes(self.cross_desc)
                        if self.cross else 0)
        self.xa_ws = torch.empty(max(self.xa_ws_n, 16), dtype=torch.uint8, device=dev)
        # the prompt's context K/V, projected once (the context is the same
        # at every denoising step)
        self.kv_ctx = torch.empty((a.B, max(a.n_ctx, 1), 2, a.C), dtype=torch.float16, device=dev)
        if self.cross:
            dpp.dpp_cross_attn_kv(self.cross_desc, self.ctx, self.xw["wk"], self.xw["wv"],
                                  self.kv_ctx, stream=self.stream)
        self.kv = [torch.empty((a.B, a.N, 2, a.C), dtype=torch.float16, device=dev)
                   for _ in range(2)]  # fp16 K/V state of a bf16 attention layer
        self.ya = torch.empty((a.B, a.N, a.C), dtype=bf, device=dev)
        self.yc = torch.empty((a.B, a.N, a.C), dtype=bf, device=dev)
        # guidance maps
        self.has_cfg = w.cfg_shape is not None
        u, cc = wl.guidance_maps(w.cfg_shape or (4,), w.index)
        self.host_u, self.host_c = u.pin_memory(), cc.pin_memory()
        self.u, self.c = put(u), put(cc)
        self.n_cfg = u.numel()
        self.cfg_out = torch.empty_like(self.u)
        self.sums = torch.zeros(3, dtype=torch.float64, device=dev)
        self.cfg_ws_n = dpp.dpp_cfg_workspace_bytes(self.n_cfg)
        self.cfg_ws = torch.zeros(self.cfg_ws_n, dtype=torch.uint8, device=dev)
        # step "t-1": synchronous calls on the stale inputs seed the states
        s = self.stream
        dpp.dpp_conv3x3(self.conv_desc, self.stale, None, self.wconv, None, self.y1, stream=s)
        dpp.dpp_groupnorm(self.gn_desc, self.y1, None, self.stats[0], self.gamma, self.beta,
                          self.y2, self.gn_ws, self.gn_ws_n, stream=s)
        dpp.dpp_self_attn(self.attn_desc, xs, self.aw["wq"], self.aw["wk"], self.aw["wv"],
                          self.aw["wo"], None, self.kv[0], self.ya, self.sa_ws, self.sa_ws_n,
                          stream=s)
        torch.cuda.synchronize(dev)
        del xs
        self.i = 0
        c_ = w.conv
        self.row_bytes = c_.W * c_.C * 2
        self.ops = ["conv", "groupnorm", "self_attn", "cross_attn", "cfg", "refresh"]

    def run(self, events=None, core_events=None, waits=None):
        """One displaced step; events (len 7) bracket the six ABI calls;
        waits maps a call's index (0 conv, 2 self-attention, 4 guidance) to
        an event the stream waits for before that call (its input copied
        in)."""
        dpp, s, w = self.dpp, self.stream, self.w
        c = w.conv
        k0, k1 = self.i % 2, (self.i + 1) % 2
        rec = (lambda j: events[j].record(s)) if events else (lambda j: None)
        pre = (lambda j: s.wait_event(waits[j]) if j in waits else None) if waits else \
            (lambda j: None)
        pre(0)
        rec(0)
        # conv whose epilogue also sums each band of its output for the GroupNorm
        dpp.dpp_conv3x3_gn(self.conv_desc, self.x, self.stale, self.wconv, None, self.y1,
                           w.groups, self.gn_sums, stream=s)
        rec(1)
        dpp.dpp_groupnorm_apply(self.gn_desc, self.y1, self.stats[k0], self.gn_sums,
                                self.stats[k1], self.gamma, self.beta, self.y2, stream=s)
        rec(2)
        pre(2)
        if core_events:
            dpp.dpp_set_attn_core_events(*core_events)
        dpp.dpp_self_attn(self.attn_desc, self.xa, self.aw["wq"], self.aw["wk"], self.aw["wv"],
                          self.aw["wo"], self.kv[k0], self.kv[k1], self.ya, self.sa_ws,
                          self.sa_ws_n, stream=s)
        if core_events:
            dpp.dpp_set_attn_core_events(None, None)
        rec(3)
        if self.cross:  # the prompt's context K/V from set-up
            dpp.dpp_cross_attn_cached(self.cross_desc, self.ya, self.kv_ctx, self.xw["wq"],
                                      self.xw["wo"], self.yc, self.xa_ws, self.xa_ws_n, stream=s)
        rec(4)
        pre(4)
        if self.has_cfg:
            dpp.dpp_cfg_combine(self.u, self.c, w.cfg_scale, self.n_cfg, self.cfg_out,
                                self.sums, self.cfg_ws, self.cfg_ws_n, stream=s)
        rec(5)
        dpp.dpp_refresh_stale(self.x, self.stale, c.B, c.H, self.row_bytes, c.P, stream=s)
        rec(6)
        self.i += 1

    def time_two_pass_groupnorm(self, reps=5):
        """The workspace entry point dpp_groupnorm (sums its input itself: two
        reads of x) on the conv output: `reps` calls back to back between two
        events (so host launch time overlaps the GPU's work), ms per call."""
        dpp, s = self.dpp, self.stream
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        for _ in range(reps):
            dpp.dpp_groupnorm(self.gn_desc, self.y1, self.stats[0], self.stats[1], self.gamma,
                              self.beta, self.y2, self.gn_ws, self.gn_ws_n, stream=s)
        b.record(s)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    # The step's inputs copied in and results copied out each end-to-end step;
    # two device sets, so one step's copies overlap the other set's compute.
    IO = ("x", "xa", "u", "c", "y2", "yc", "cfg_out", "sums")

    def make_io_sets(self):
        self._sets = [{n: getattr(self, n) for n in self.IO},
                      {n: torch.empty_like(getattr(self, n)) for n in self.IO}]

    def select(self, i):
        for n, t in self._sets[i].items():
            setattr(self, n, t)

    def h2d(self, stream, marks=None):
        """Copies the step's inputs in; marks (3 events), if given, are
        recorded after the conv input, the attention input and the guidance
        maps."""
        with torch.cuda.stream(stream):
            self.x.copy_(self.host_x, non_blocking=True)
            if marks:
                marks[0].record(stream)
            self.xa.copy_(self.host_xa, non_blocking=True)
            if marks:
                marks[1].record(stream)
            self.u.copy_(self.host_u, non_blocking=True)
            self.c.copy_(self.host_c, non_blocking=True)
            if marks:
                marks[2].record(stream)
        return sum(t.numel() * t.element_size() for t in
                   (self.host_x, self.host_xa, self.host_u, self.host_c))

    def alloc_d2h(self):
        self.out_host = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                         for t in (self.y2, self.yc, self.cfg_out, self.sums)]
        return sum(t.numel() * t.element_size() for t in self.out_host)

    def d2h(self, stream, after=None):
        """Copies the step's results out; after (3 events), if given, are
        waited for before the GroupNorm output, the cross-attention output
        and the guidance results respectively."""
        with torch.cuda.stream(stream):
            for k, (h, d) in enumerate(zip(self.out_host,
                                           (self.y2, self.yc, self.cfg_out, self.sums))):
                if after and k < 3:
                    stream.wait_event(after[k])
                h.copy_(d, non_blocking=True)


# ------------------------------------------------------------------ oracle arm
class OracleSample:
    """Times the fp64 oracle on a bounded sample of the workload: conv output
    rows at band edges and inside, and queries of one band of self- and
    cross-attention (keys/values of that band's composite are projected in
    full).  The full-size fp64 inputs are drawn once, outside the timing."""

    def __init__(self, w):
        import oracle
        self.oracle, self.w = oracle, w
        c, a = w.conv, w.attn
        shape = (c.B, c.H, c.W, c.C)
        self.F = wl.to_f64(wl.normal(shape, wl.seed_of(w.index, 0, wl.T_FRESH), dtype=w.dtype))
        self.S = wl.to_f64(wl.perturbed(wl.normal(shape, wl.seed_of(w.index, 0, wl.T_FRESH),
                                                  dtype=w.dtype),
                                        wl.seed_of(w.index, 1, wl.T_STALE_NOISE), w.stale_scale))
        self.Wt = wl.to_f64(wl.conv_weight(c.C, c.C, wl.seed_of(w.index, 0, wl.T_CONV_W),
                                           w.dtype))
        X = wl.normal((a.B, a.N, a.C), wl.seed_of(w.index, 0, wl.T_ATTN_X), dtype=w.dtype)
        self.X = wl.to_f64(X[:1])
        self.Xs = wl.to_f64(wl.perturbed(X, wl.seed_of(w.index, 1, wl.T_ATTN_X),
                                         w.stale_scale)[:1])
        self.aw = {k: wl.to_f64(v) for k, v in wl.attn_weights(a, w.index, w.dtype).items()}
        self.xw = {k: wl.to_f64(v) for k, v in wl.cross_weights(a, w.index, w.dtype).items()}
        self.ctx = wl.to_f64(wl.context(a, w.index, w.dtype)[:1])
        self.rng = np.random.default_rng(7)

    def run(self, sample_rows=8, sample_queries=48):
        """Returns (tensor FLOPs of the sampled outputs, seconds, description)."""
        o, w, rng = self.oracle, self.w, self.rng
        c, a = w.conv, w.attn
        Hp, Np = c.H // c.P, a.N // a.P
        rows = sorted(set([Hp, 2 * Hp - 1] + list(rng.integers(0, c.H, sample_rows - 2))))
        p = int(rng.integers(0, a.P))
        qs = np.sort(rng.choice(np.arange(p * Np, (p + 1) * Np), sample_queries, replace=False))
        t0 = time.perf_counter()
        o.displaced_conv3x3(self.F, self.S, self.Wt, None, c.P, out_rows=rows)
        o.displaced_self_attention(self.X, self.Xs, self.aw["wq"], self.aw["wk"], self.aw["wv"],
                                   self.aw["wo"], a.heads, a.P, queries=qs)
        o.cross_attention(self.X, self.ctx, self.xw["wq"], self.xw["wk"], self.xw["wv"],
                          self.xw["wo"], a.heads, queries=qs)
        secs = time.perf_counter() - t0
        conv_f = 2.0 * c.B * len(rows) * c.W * c.C * 9 * c.C
        nq = len(qs)
        self_f = (4.0 * nq * a.N * a.head_dim * a.heads    # core for the sampled queries
                  + 2.0 * a.N * a.C * 2 * a.C               # K/V of the band's composite
                  + 2.0 * 2.0 * nq * a.C * a.C)             # Q and O projections
        cross_f = (4.0 * nq * a.n_ctx * a.head_dim * a.heads + 2.0 * a.n_ctx * a.c_ctx * 2 * a.C
                   + 2.0 * 2.0 * nq * a.C * a.C)
        desc = (f"{len(rows)} conv output rows x batch {c.B}; {nq} queries of one band, "
                f"batch 0, for self-attention (K/V of the band's composite projected in "
                f"full) and cross-attention; fp64 numpy; per-step sample")
        return conv_f + self_f + cross_f, secs, desc

    def run_bandwidth(self):
        """The bandwidth ops on the host: displaced GroupNorm of one band of
        image 0 (its statistics span the whole composite image), the stale
        refresh of image 0, and the guidance combine with its sums over the
        full maps.  Returns {op: {"gbs", "seconds", "sample"}}, GB/s counted
        in the GPU's algorithmic bytes of the sampled part (bf16 activations,
        fp32 maps)."""
        o, w = self.oracle, self.w
        c = w.conv
        res = {}
        g, b = (wl.to_f64(t) for t in wl.gn_affine(c.C, w.index))
        band = int(self.rng.integers(0, c.P))
        t0 = time.perf_counter()
        o.displaced_groupnorm(self.F[:1], self.S[:1], w.groups, w.eps, g, b, c.P, bands=[band])
        dt = time.perf_counter() - t0
        nb = 2.0 * (c.H // c.P) * c.W * c.C * 2
        res["groupnorm"] = {"gbs": nb / dt / 1e9, "seconds": dt,
                            "sample": f"band {band} of image 0 (composite statistics in full)"}
        t0 = time.perf_counter()
        o.refresh_stale(self.F[:1], self.S[:1], c.P)
        dt = time.perf_counter() - t0
        nb = 2.0 * c.H * c.W * c.C * 2
        res["refresh"] = {"gbs": nb / dt / 1e9, "seconds": dt, "sample": "image 0, all bands"}
        if w.cfg_shape:
            u, cc = wl.guidance_maps(w.cfg_shape, w.index)
            u, cc = wl.to_f64(u), wl.to_f64(cc)
            t0 = time.perf_counter()
            o.cfg_combine(u, cc, w.cfg_scale)
            dt = time.perf_counter() - t0
            res["cfg"] = {"gbs": 3.0 * 4 * u.size / dt / 1e9, "seconds": dt,
                          "sample": "full maps"}
        return res


def time_chain(dev, steps, warmup=2):
    """One level of the U-Net (ResNet block + transformer block) stepped
    with displaced patch parallelism at 3840px: latent 2 x 240 x 240 x 640 in
    8 bands, 10 heads, text context 77 x 2048.  Times `steps` displaced steps
    back to back, then the same number again with an event pair around every
    op, then the chain with the GroupNorm -> SiLU applied in the convs' loads
    (for comparison with the default, which stores the normalised tensors),
    then the two guidance branches as chains of batch 1 run serially and on
    two streams; returns the per-step figures."""
    import displaced_patch_parallelism_02_b300 as dpp
    from displaced_patch_parallelism_02_b300.chain import OPS, BlockChain
    ch = wl.CHAINS["sdxl_3840_level2"]
    wts = {}
    for k, v in wl.chain_weights(ch).items():
        if k.startswith("conv") and k.endswith("_w"):
            v = v.permute(0, 2, 3, 1)  # channels-last [C, 3, 3, C]
        wts[k] = v.contiguous().to(dev)
    xs, ctx = wl.chain_inputs(ch, 0)
    x, ctx = xs[0].to(dev), ctx.to(dev)
    del xs
    chain = BlockChain(ch.B, ch.H, ch.W, ch.C, ch.heads, ch.P, ch.G, ch.n_ctx, ch.c_ctx, wts, dev,
                       ff_mult=ch.ff_mult)
    s = torch.cuda.current_stream(dev)
    for _ in range(max(warmup, 1)):  # the first step is the synchronous one
        chain.step(x, ctx, stream=s)
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n0 = dpp.dpp_launch_count()
    a.record(s)
    for _ in range(steps):
        chain.step(x, ctx, stream=s)
    b.record(s)
    torch.cuda.synchronize(dev)
    launches = (dpp.dpp_launch_count() - n0) // max(steps, 1)
    ms = a.elapsed_time(b) / max(steps, 1)
    evs = []

    def hook(name, when, tensors):
        e = torch.cuda.Event(enable_timing=True)
        e.record(s)
        evs.append((name, when, e))

    for _ in range(steps):
        chain.step(x, ctx, stream=s, hook=hook)
    torch.cuda.synchronize(dev)
    op_ms = {n: 0.0 for n in OPS}
    for (n, w1, e1), (_, w2, e2) in zip(evs[0::2], evs[1::2]):
        op_ms[n] += e1.elapsed_time(e2) / max(steps, 1)
    ok = dpp.dpp_device_status() == dpp.DPP_OK and bool(torch.isfinite(x.float()).all())
    flop = chain.flops()
    del chain
    torch.cuda.empty_cache()
    # the same chain with the ResNet block's GroupNorm -> SiLU applied by the
    # convs as they load their inputs (never stored), for comparison
    fused = BlockChain(ch.B, ch.H, ch.W, ch.C, ch.heads, ch.P, ch.G, ch.n_ctx, ch.c_ctx, wts,
                        dev, ff_mult=ch.ff_mult, fuse_norm=True)
    xs_ = x.clone()
    for _ in range(max(warmup, 1)):
        fused.step(xs_, ctx, stream=s)
    torch.cuda.synchronize(dev)
    a.record(s)
    for _ in range(steps):
        fused.step(xs_, ctx, stream=s)
    b.record(s)
    torch.cuda.synchronize(dev)
    ms_fused = a.elapsed_time(b) / max(steps, 1)
    ok = ok and dpp.dpp_device_status() == dpp.DPP_OK
    del fused, xs_
    torch.cuda.empty_cache()
    # the guided pair as two branches of batch 1 (condition-based partition):
    # serially on one stream, and on two streams (the parallel stage)
    from displaced_patch_parallelism_02_b300.chain import BranchPair
    pair = BranchPair(ch.H, ch.W, ch.C, ch.heads, ch.P, ch.G, ch.n_ctx, ch.c_ctx, wts, dev,
                      ff_mult=ch.ff_mult)
    xb = [x[b:b + 1].contiguous() for b in range(2)]
    cb = [ctx[b:b + 1].contiguous() for b in range(2)]
    sched = {}
    for name, par in (("branches_serial", False), ("branches_two_stream", True)):
        for _ in range(max(warmup, 1)):
            pair.step(xb, cb, par, stream=s)
        torch.cuda.synchronize(dev)
        a.record(s)
        for _ in range(steps):
            pair.step(xb, cb, par, stream=s)
        b.record(s)
        torch.cuda.synchronize(dev)
        sched[name] = a.elapsed_time(b) / max(steps, 1)
    ok = ok and dpp.dpp_device_status() == dpp.DPP_OK
    del pair, wts, x, ctx, xb, cb
    torch.cuda.empty_cache()
    return {"workload": ch.name, "latent": [ch.B, ch.H, ch.W, ch.C], "P": ch.P,
            "heads": ch.heads, "context": [ch.n_ctx, ch.c_ctx], "steps": steps,
            "ms_per_step": ms, "tflops": flop / (ms / 1e3) / 1e12, "step_flop": flop,
            "launches_per_step": launches, "ok": ok,
            "norm_in_conv": False, "ms_per_step_norm_in_conv": ms_fused,
            "ops_ms": {n: round(v, 4) for n, v in op_ms.items()},
            "schedules_ms_per_step": {"batched": ms, **sched}}


def cpu_cores():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("internal_api") in
             ("openblas", "mkl", "blis")]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


# ------------------------------------------------------------------ main
def max_over_ranks(pg, ms, device):
    """The slowest rank's time (every rank returns the same value); ms as is
    when there is no process group."""
    if pg is None:
        return float(ms)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flop_per_step_per_rank, world_size, steps, ms):
    """Throughput of the whole job: the work every rank did over the slowest
    rank's time (the replicas are independent and equal in size)."""
    return flop_per_step_per_rank * world_size * steps / (ms / 1e3) / 1e12


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_reference(args, w, ws, rank):
    if rank != 0:
        return 0
    model = work_model(w)
    sample = OracleSample(w)
    for _ in range(args.warmup):
        sample.run(4, 16)
    flops, secs = 0.0, 0.0
    desc = ""
    for _ in range(args.steps):
        f, t, desc = sample.run(4, 16)
        flops += f
        secs += t
    val = flops / secs / 1e12
    bw = sample.run_bandwidth()
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "step_tflop_full": model["step_flop"] / 1e12},
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": desc, "bandwidth_ops": bw},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-chain", action="store_true",
                    help="skip the ResNet + transformer block chain timing")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload op timings")
    ap.add_argument("--workload", default=WORKLOAD, choices=["sdxl_3840_cfg", "sdxl_2048"],
                    help="sdxl_2048 (no guidance maps or text context) is the smaller case "
                         "used for profiler captures")
    args = ap.parse_args()
    w = wl.WORKLOADS[args.workload]
    ws, rank, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, w, ws, rank)

    assert torch.cuda.is_available(), "bench.py needs a CUDA device"
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    import displaced_patch_parallelism_02_b300 as dpp
    model = work_model(w)
    peaks, peak_src = load_peaks()

    step = Step(w, dev)
    s = step.stream
    for _ in range(max(args.warmup, 0)):
        step.run()
    torch.cuda.synchronize(dev)

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(K)]
    core = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(K)]
    for a_, b_ in core:  # create the CUDA events now; the library re-records them
        a_.record(s)
        b_.record(s)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    launches0 = dpp.dpp_launch_count()
    t_start.record(s)
    for k in range(K):
        step.run(evs[k], core[k])
    t_end.record(s)
    torch.cuda.synchronize(dev)
    launches = dpp.dpp_launch_count() - launches0
    # a bounded wait that gave up records DPP_ERR_TIMEOUT on the device; a
    # run that saw one publishes no number
    status = dpp.dpp_device_status()
    if pg:
        pg.barrier()
    clocks = sampler.stop()
    total_ms = max_over_ranks(pg, t_start.elapsed_time(t_end), dev)
    ms_step = total_ms / K
    value = whole_job_tflops(model["step_flop"], ws, K, total_ms)

    op_ms = {op: sum(evs[k][j].elapsed_time(evs[k][j + 1]) for k in range(K)) / K
             for j, op in enumerate(step.ops)}
    gn2_ms = step.time_two_pass_groupnorm()
    core_ms = sum(a.elapsed_time(b) for a, b in core) / K
    tf = lambda f, ms: f / (ms / 1e3) / 1e12 if f and ms > 0 else None
    gb = lambda b, ms: b / (ms / 1e3) / 1e9 if b and ms > 0 else None
    sus, burst = peaks["bf16_tflops_sustained"], peaks["bf16_tflops"]
    ops = {
        "conv": {"ms": op_ms["conv"], "tflops": tf(model["conv_flop"], op_ms["conv"]),
                 "entry": "dpp_conv3x3_gn (epilogue also sums the output per band and group)"},
        "groupnorm": {"ms": op_ms["groupnorm"], "gbs": gb(model["gn_bytes"], op_ms["groupnorm"]),
                      "entry": "dpp_groupnorm_apply (band sums from the conv epilogue)"},
        "groupnorm_two_pass": {"ms": gn2_ms, "gbs": gb(model["gn_bytes"], gn2_ms),
                               "entry": "dpp_groupnorm (sums its own input), timed alone"},
        "self_attn": {"ms": op_ms["self_attn"],
                      "tflops": tf(model["self_core_flop"] + model["self_proj_flop"],
                                   op_ms["self_attn"])},
        "self_attn_core": {"ms": core_ms, "tflops": tf(model["self_core_flop"], core_ms)},
        "cross_attn": {"ms": op_ms["cross_attn"],
                       "tflops": tf(model["cross_flop"], op_ms["cross_attn"])},
        "cfg": {"ms": op_ms["cfg"], "gbs": gb(model["cfg_bytes"], op_ms["cfg"])},
        "refresh": {"ms": op_ms["refresh"], "gbs": gb(model["refresh_bytes"], op_ms["refresh"])},
    }
    for k, v in ops.items():
        if v.get("tflops") is not None:
            v["frac_of_burst_bf16"] = v["tflops"] / burst
            v["frac_of_sustained_bf16"] = v["tflops"] / sus
        elif v.get("gbs") is not None:
            v["frac_of_hbm"] = v["gbs"] / peaks["hbm_gbs"]
            v["l2"] = "in the step: may read what the previous op left in L2"

    # end to end: pinned host inputs -> device, step, results -> host
    bi = bo = 0
    e2e_val = None
    stages = []
    if K > 0:
        bo = step.alloc_d2h()
        torch.cuda.synchronize(dev)
        if pg:
            pg.barrier()
        # Every step copies its inputs in from pinned host memory and its
        # results out, all inside the timed region.  With two device sets the
        # copies of one step overlap the other set's compute, and the two
        # directions run on two copy streams (PCIe is full duplex: one stream
        # would serialise them): step k+1's inputs are copied in once step
        # k-1, the last reader of that set, is done; each op of a step starts
        # once its own input has landed, and each result is copied out as
        # soon as its op is done (the GroupNorm output while the attention
        # runs); step k+2 overwrites step k's result buffers only after they
        # are copied out.
        step.make_io_sets()
        cs_in, cs_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        marks = [[torch.cuda.Event() for _ in range(3)] for _ in range(2)]  # inputs landed
        op_ev = [[torch.cuda.Event() for _ in range(7)] for _ in range(2)]  # ops done
        done = [torch.cuda.Event() for _ in range(2)]
        out_done = [torch.cuda.Event() for _ in range(2)]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        cs_in.wait_stream(s)
        cs_out.wait_stream(s)
        e0.record(cs_in)
        step.select(0)
        bi = step.h2d(cs_in, marks[0])
        # The sampler's side of each step: once a step's results are on the
        # host, its discrepancy (rel-MAE from the guidance sums) goes to the
        # adaptive switching controller, which names the stage of the steps
        # to come.  The host waits for step k-1's results only after step k
        # is queued, so the device never idles on it.
        sw = dpp.dpp_switch_state()
        dpp.dpp_switch_init(sw, SWITCH_FLAT_TOL, SWITCH_RISE_TOL, SWITCH_PATIENCE)
        stages = []

        def observe(k):
            out_done[k % 2].synchronize()
            h = step.out_host[3]
            stages.append(dpp.dpp_switch_update(sw, float(h[0] / h[1])))

        for k in range(K):
            i, j = k % 2, 1 - k % 2
            step.select(i)
            if k >= 2:
                s.wait_event(out_done[i])  # step k-2's results are out of this set
            step.run(events=op_ev[i], waits={0: marks[i][0], 2: marks[i][1], 4: marks[i][2]})
            done[i].record(s)
            if k >= 1:
                observe(k - 1)
            if k + 1 < K:
                if k >= 1:
                    cs_in.wait_event(done[j])
                step.select(j)
                step.h2d(cs_in, marks[j])
                step.select(i)
            step.d2h(cs_out, (op_ev[i][2], op_ev[i][4], op_ev[i][5]))
            out_done[i].record(cs_out)
        observe(K - 1)
        cs_out.wait_stream(cs_in)
        e1.record(cs_out)
        torch.cuda.synchronize(dev)
        step.select(0)
        e2e_ms = max_over_ranks(pg, e0.elapsed_time(e1), dev)
        e2e_val = whole_job_tflops(model["step_flop"], ws, K, e2e_ms)

    del step
    torch.cuda.empty_cache()
    status2 = dpp.dpp_device_status()  # the end-to-end loop's waits
    if status == dpp.DPP_OK:
        status = status2

    chain = None
    if not args.no_chain and K > 0:
        chain = time_chain(dev, K)
        chain["ms_per_step"] = max_over_ranks(pg, chain["ms_per_step"], dev)
        chain["tflops"] = whole_job_tflops(chain["step_flop"], ws, 1, chain["ms_per_step"])
        chain["frac_of_burst_bf16"] = chain["tflops"] / (burst * ws)
        chain["frac_of_sustained_bf16"] = chain["tflops"] / (sus * ws)

    # every workload's ops on their own; the bandwidth ops cold (L2 flushed)
    configs = None
    if not args.no_configs and K > 0:
        configs = per_config(dev, max(5, min(K, 20)), peaks, list(wl.WORKLOADS))
        for nm, k in (("groupnorm", "groupnorm_apply"), ("groupnorm_two_pass", "groupnorm"),
                      ("refresh", "refresh"), ("cfg", "cfg")):
            cold = (configs.get(w.name) or {}).get(k)
            if cold:
                ops[nm].update({"in_step_ms": ops[nm]["ms"], "ms": cold["ms"],
                                "gbs": cold["gbs"], "frac_of_hbm": cold["frac_of_hbm"],
                                "l2": cold["l2"]})
        if dpp.dpp_device_status() != dpp.DPP_OK:
            status = dpp.DPP_ERR_TIMEOUT

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        sample = OracleSample(w)
        f, secs, desc = sample.run()
        cpu = {"value": f / secs / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(),
               "kind": "oracle", "sample": desc, "seconds": secs,
               "bandwidth_ops": sample.run_bandwidth()}
        del sample

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) activations, N(0,1/fan_in) weights)",
            "config": {"workload": w.name,
                       "latent": [w.conv.B, w.conv.H, w.conv.W, w.conv.C], "bands": w.conv.P,
                       "attn_tokens": [w.attn.B, w.attn.N], "attn_channels": w.attn.C,
                       "heads": w.attn.heads,
                       "text_ctx": [w.attn.n_ctx, w.attn.c_ctx] if w.attn.n_ctx else None,
                       "cfg_maps": [2] + list(w.cfg_shape) if w.cfg_shape else None,
                       "parallelism": f"replicas{ws}",
                       "l2": ("step: inputs and working set exceed the 126 MB L2, no flush; "
                              "GroupNorm, refresh and guidance also timed alone with L2 "
                              "flushed before every rep (ops.*.gbs are those cold figures)")},
            "roofline": {"kernel": "self-attention core", "bound": "tensor",
                         "achieved": ops["self_attn_core"]["tflops"], "peak": burst,
                         "unit": "TFLOP/s", "frac": ops["self_attn_core"]["tflops"] / burst,
                         "peak_source": f"{peak_src} bf16 burst (the kernel runs in a short "
                                        f"timed region at near-maximum clocks: see clocks)",
                         "frac_of_sustained": ops["self_attn_core"]["tflops"] / sus,
                         "traffic": attn_traffic() if w.name == "sdxl_3840_cfg" else None,
                         "traffic_unit": "bytes per launch (ncu dram read + write)"},
            "ops": ops,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": bi,
                    "d2h_bytes_per_step": bo, "switch_stages": stages},
            "gpu_launches": launches,
            "block_chain": chain,
            "per_config": configs,
            "device_status": dpp.dpp_status_string(status),
            "clocks": clocks,
        }
        print(json.dumps(line))
    if pg:
        pg.destroy_process_group()
    return 0 if status == dpp.DPP_OK else 1


if __name__ == "__main__":
    sys.exit(main())
