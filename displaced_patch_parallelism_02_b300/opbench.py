"""Times one library call at a given shape: the single-kernel view that
profiling needs (ncu -k ... -s <warm-up launches> -c ...).

    python -m displaced_patch_parallelism_02_b300.opbench linear --M 65536 --K 2560 --N 640 \
        --bias --accumulate
    python -m displaced_patch_parallelism_02_b300.opbench cfg --n 921600
    python -m displaced_patch_parallelism_02_b300.opbench conv_gn --H 512 --W 512 --C 320 --P 8
    python -m displaced_patch_parallelism_02_b300.opbench layernorm --T 262144 --C 640
    python -m displaced_patch_parallelism_02_b300.opbench attn --B 2 --H 240 --W 240 --P 8
    python -m displaced_patch_parallelism_02_b300.opbench groupnorm --B 2 --H 480 --W 480 \
        --C 320 --P 8 --flush
    python -m displaced_patch_parallelism_02_b300.opbench cross --B 2 --H 240 --W 240 \
        --heads 10 --n_ctx 77 --c_ctx 2048

`attn` is one displaced self-attention call (QKV projection, core, output
projection); its figure is the attention core alone, timed by the events the
library records around the core launch (dpp_set_attn_core_events), FLOPs
4 * B * N^2 * 64 * heads.  `cross` is one cross-attention call against a
prompt's context K/V projected once beforehand (dpp_cross_attn_cached); its
figure is again the core alone, FLOPs 4 * B * N * n_ctx * 64 * heads.

Inputs are seeded random device tensors (bf16 activations, weights scaled by
1/sqrt(fan_in), fp32 guidance maps); `--warmup` calls run first, then `--reps`
calls between two CUDA events (with `--flush`, each rep between its own
events after a write of twice the L2 size, and the median is reported).  Prints one JSON line with the time per call
and the achieved TFLOP/s (contractions) or GB/s (read x + write y).
Every call is the library's own entry point; nothing here computes anything.
"""
from __future__ import annotations

import argparse
import json

import torch

from . import (DPP_ACT_SILU, DPP_BF16, DPP_EPI_GEGLU, DPP_EPI_NONE, dpp_attn_desc,
               dpp_cfg_combine, dpp_cfg_workspace_bytes, dpp_conv3x3, dpp_conv3x3_gn,
               dpp_conv3x3_norm, dpp_conv_desc,
               dpp_cross_attn_cached, dpp_cross_attn_cached_workspace_bytes, dpp_cross_attn_kv,
               dpp_device_status, dpp_gn_desc, dpp_groupnorm, dpp_groupnorm_apply,
               dpp_groupnorm_workspace_bytes, dpp_layernorm, dpp_linear, dpp_linear_desc,
               dpp_ln_desc, dpp_self_attn, dpp_self_attn_workspace_bytes,
               dpp_set_attn_core_events)


def _randn(shape, gen, scale=1.0, dtype=torch.bfloat16):
    return (torch.randn(shape, generator=gen, device="cuda") * scale).to(dtype)


def setup(args, gen):
    """Returns (call, work, unit) for the op: call() makes one library call,
    work is the FLOPs or bytes of one call."""
    if args.op == "linear":
        M, K, N = args.M, args.K, args.N
        rows = 2 * N if args.geglu else N
        x = _randn((M, K), gen)
        w = _randn((rows, K), gen, K ** -0.5)
        b = _randn((rows,), gen, 0.1, torch.float32) if args.bias else None
        y = _randn((M, N), gen)
        d = dpp_linear_desc(M, K, N, DPP_BF16, DPP_EPI_GEGLU if args.geglu else DPP_EPI_NONE,
                            int(args.accumulate))
        return (lambda: dpp_linear(d, x, w, b, y)), 2.0 * M * K * rows, "TFLOP/s"
    if args.op == "cfg":
        n = args.n
        u, c = _randn((n,), gen, dtype=torch.float32), _randn((n,), gen, dtype=torch.float32)
        out = torch.empty_like(u)
        sums = torch.zeros(3, dtype=torch.float64, device="cuda")
        nws = dpp_cfg_workspace_bytes(n)
        ws = torch.zeros(nws, dtype=torch.uint8, device="cuda")
        return (lambda: dpp_cfg_combine(u, c, 7.5, n, out, sums, ws, nws)), 12.0 * n, "GB/s"
    if args.op == "conv_gn":
        B, H, W, C, P, G = args.B, args.H, args.W, args.C, args.P, args.G
        x = _randn((B, H, W, C), gen)
        stale = _randn((B, H, W, C), gen)
        w = _randn((C, 3, 3, C), gen, (9 * C) ** -0.5)
        y, y2 = torch.empty_like(x), torch.empty_like(x)
        sums = torch.empty((P, B, G, 2), dtype=torch.float64, device="cuda")
        st_prev = torch.zeros((P, B, G, 2), device="cuda")
        st_next = torch.empty_like(st_prev)
        gamma, beta = torch.ones(C, device="cuda"), torch.zeros(C, device="cuda")
        cd = dpp_conv_desc(B, H, W, C, C, P, DPP_BF16, 0, 0)
        gd = dpp_gn_desc(B, H, W, C, G, P, 1e-5, DPP_BF16, 0, 0)

        def call():
            dpp_conv3x3_gn(cd, x, stale, w, None, y, G, sums)
            dpp_groupnorm_apply(gd, y, st_prev, sums, st_next, gamma, beta, y2)
        return call, 2.0 * B * H * W * C * 9 * C, "TFLOP/s"
    if args.op in ("conv", "normconv"):  # displaced conv; normconv: GroupNorm + SiLU on load
        B, H, W, C, P = args.B, args.H, args.W, args.C, args.P
        x = _randn((B, H, W, C), gen)
        stale = _randn((B, H, W, C), gen)
        w = _randn((C, 3, 3, C), gen, (9 * C) ** -0.5)
        y = torch.empty_like(x)
        cd = dpp_conv_desc(B, H, W, C, C, P, DPP_BF16, 0, 0)
        if args.op == "conv":
            return (lambda: dpp_conv3x3(cd, x, stale, w, None, y)), 2.0 * B * H * W * C * 9 * C, \
                "TFLOP/s"
        aff = [torch.rand((P, B, C, 2), generator=gen, device="cuda") for _ in range(2)]
        return (lambda: dpp_conv3x3_norm(cd, x, stale, aff[0], aff[1], DPP_ACT_SILU, w, None, y)), \
            2.0 * B * H * W * C * 9 * C, "TFLOP/s"
    if args.op == "layernorm":
        T, C = args.T, args.C
        x = _randn((T, C), gen)
        y = torch.empty_like(x)
        g, b = torch.ones(C, device="cuda"), torch.zeros(C, device="cuda")
        d = dpp_ln_desc(T, C, 1e-5, DPP_BF16)
        return (lambda: dpp_layernorm(d, x, g, b, y)), 2.0 * 2 * T * C, "GB/s"
    if args.op == "attn":
        B, H, W, P, heads = args.B, args.H, args.W, args.P, args.heads
        C, N = 64 * heads, args.H * args.W
        x = _randn((B, N, C), gen)
        wq, wk, wv, wo = (_randn((C, C), gen, C ** -0.5) for _ in range(4))
        kv = [torch.empty((B, N, 2, C), dtype=torch.float16, device="cuda") for _ in range(2)]
        y = torch.empty_like(x)
        d = dpp_attn_desc(B, H, W, C, heads, 64, P, 0, 0, DPP_BF16, 0, 0)
        nws = dpp_self_attn_workspace_bytes(d)
        ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
        dpp_self_attn(d, x, wq, wk, wv, wo, None, kv[0], y, ws, nws)  # synchronous step
        ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        for e in ev:  # creates the CUDA events; the library re-records them
            e.record()

        def call():
            dpp_set_attn_core_events(*ev)
            dpp_self_attn(d, x, wq, wk, wv, wo, kv[0], kv[1], y, ws, nws)
            dpp_set_attn_core_events(None, None)
        call.core_events = ev
        return call, 4.0 * B * N * N * 64 * heads, "TFLOP/s"
    if args.op == "cross":  # cross-attention against a prompt's context K/V
        B, H, W, heads, L, Cc = args.B, args.H, args.W, args.heads, args.n_ctx, args.c_ctx
        C, N = 64 * heads, args.H * args.W
        x = _randn((B, N, C), gen)
        ctx = _randn((B, L, Cc), gen)
        wq, wo = (_randn((C, C), gen, C ** -0.5) for _ in range(2))
        wk, wv = (_randn((C, Cc), gen, Cc ** -0.5) for _ in range(2))
        d = dpp_attn_desc(B, H, W, C, heads, 64, 1, L, Cc, DPP_BF16, 0, 0)
        kv = torch.empty((B, L, 2, C), dtype=torch.float16, device="cuda")
        dpp_cross_attn_kv(d, ctx, wk, wv, kv)  # once per prompt
        nws = dpp_cross_attn_cached_workspace_bytes(d)
        ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
        y = torch.empty_like(x)
        ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        for e in ev:  # creates the CUDA events; the library re-records them
            e.record()

        def call():
            dpp_set_attn_core_events(*ev)
            dpp_cross_attn_cached(d, x, kv, wq, wo, y, ws, nws)
            dpp_set_attn_core_events(None, None)
        call.core_events = ev
        return call, 4.0 * B * N * L * 64 * heads, "TFLOP/s"
    if args.op == "groupnorm":  # the displaced step, sums of its own input
        B, H, W, C, P, G = args.B, args.H, args.W, args.C, args.P, args.G
        x = _randn((B, H, W, C), gen)
        y = torch.empty_like(x)
        gamma, beta = torch.ones(C, device="cuda"), torch.zeros(C, device="cuda")
        d = dpp_gn_desc(B, H, W, C, G, P, 1e-5, DPP_BF16, 0, 0)
        nws = dpp_groupnorm_workspace_bytes(d)
        ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
        st = [torch.empty((P, B, G, 2), device="cuda") for _ in range(2)]
        dpp_groupnorm(d, x, None, st[0], gamma, beta, y, ws, nws)  # synchronous step
        return (lambda: dpp_groupnorm(d, x, st[0], st[1], gamma, beta, y, ws, nws),
                2.0 * B * H * W * C * 2, "GB/s")
    raise ValueError(args.op)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("op", choices=["linear", "cfg", "conv", "normconv", "conv_gn", "layernorm",
                                   "attn", "groupnorm", "cross"])
    ap.add_argument("--M", type=int, default=115200)
    ap.add_argument("--K", type=int, default=640)
    ap.add_argument("--N", type=int, default=640)
    ap.add_argument("--bias", action="store_true")
    ap.add_argument("--accumulate", action="store_true")
    ap.add_argument("--geglu", action="store_true")
    ap.add_argument("--n", type=int, default=4 * 480 * 480)
    ap.add_argument("--B", type=int, default=1)
    ap.add_argument("--H", type=int, default=512)
    ap.add_argument("--W", type=int, default=512)
    ap.add_argument("--C", type=int, default=320)
    ap.add_argument("--P", type=int, default=8)
    ap.add_argument("--G", type=int, default=32)
    ap.add_argument("--T", type=int, default=262144)
    ap.add_argument("--heads", type=int, default=10)
    ap.add_argument("--n_ctx", type=int, default=77)
    ap.add_argument("--c_ctx", type=int, default=2048)
    ap.add_argument("--warmup", type=int, default=2)
    ap.add_argument("--reps", type=int, default=1)
    ap.add_argument("--flush", action="store_true",
                    help="evict L2 before every timed call (cold-cache figure)")
    args = ap.parse_args(argv)
    assert torch.cuda.is_available(), "opbench needs a CUDA device"
    gen = torch.Generator(device="cuda").manual_seed(1234)
    call, work, unit = setup(args, gen)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    if args.flush:
        import statistics
        l2 = int(getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 128 << 20))
        buf = torch.empty(2 * l2 // 4, dtype=torch.float32, device="cuda")
        times = []
        for _ in range(max(args.reps, 1)):
            buf.fill_(1.0)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            call()
            b.record()
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b))
        ms = statistics.median(times)
    else:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.reps):
            call()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / max(args.reps, 1)
    core = getattr(call, "core_events", None)
    if core is not None and args.reps > 0:  # the last call's attention core alone
        ms = core[0].elapsed_time(core[1])
    rate = work / (ms / 1e3) / (1e12 if unit == "TFLOP/s" else 1e9)
    out = {k: v for k, v in vars(args).items()}
    out.update(ms_per_call=ms, achieved=rate, unit=unit, status=dpp_device_status())
    print(json.dumps(out))
    return 0 if out["status"] == 0 else 1


if __name__ == "__main__":
    raise SystemExit(main())
