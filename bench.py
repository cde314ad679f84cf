#!/usr/bin/env python3
"""Benchmark of the Wan2.2-TI2V-5B VAE decode on GB300.

One step = one whole 720p clip: latents [1, 48, 31, 44, 80] (device-resident
when the timed region starts) decoded to a [1, 3, 121, 704, 1280] bf16 video
through the library's stream API (causal chunks of --chunk latent frames).
Weights are seeded random init of the full-width TI2V-5B decoder, latents
~ N(0, 1); weight packing happens before the timed region.

Prints one JSON line.  The decode runs on one GPU: its conv kernels share
weight tiles between the two CTAs of a cluster with multicast TMA loads,
which this library issues only in one-GPU processes, so `--gpus N` with
N > 1 (or a torchrun launch with WORLD_SIZE > 1) stops with an error before
any GPU work.  `--impl reference` times the CPU oracle instead, on a bounded
crop of the same workload, on this machine's host cores; under torchrun only
rank 0 runs it.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import wan_synth  # noqa: E402

WORKLOAD = wan_synth.CONFIGS["720p"]
B, Z, T, H_LAT, W_LAT = WORKLOAD["latents"]
FRAMES = 4 * T - 3
H_OUT, W_OUT = 16 * H_LAT, 16 * W_LAT
METRIC = "decoded frames/s (704x1280, bf16)"
UNIT = "frames/s"
# bounded sample for the CPU oracle: the first 2 latent frames of a 11x20 crop
# of the 720p latents (1/16 of the area): 5 video frames of 176x320
CPU_SAMPLE = dict(T=2, h=11, w=20)


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d["bf16_tflops"], d["bf16_tflops_sustained"], d["hbm_gbs"], "measured"
    except Exception:
        return 1900.0, 1700.0, 6800.0, "fallback"


def _sustained_peak_mhz():
    """Median SM clock under load while the sustained bf16 peak was measured."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["clocks_under_load"]["sm_mhz_median"])
    except Exception:
        return None


def clock_note(clocks):
    """The sustained peak's clock next to this run's: a fraction above 1 of a
    peak measured at a lower clock is a clock effect, not more work per cycle."""
    ref = _sustained_peak_mhz()
    run = clocks.get("sm_mhz") if clocks else None
    if not ref or not run:
        return None
    return {"sustained_peak_sm_mhz": ref, "this_run_sm_mhz": run, "ratio": run / ref}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


ONE_GPU_ONLY = ("the decode runs on one GPU: its conv kernels use cluster-multicast TMA loads, which this "
                "library issues only in one-GPU processes")


def check_one_gpu(gpus: int, world: int) -> None:
    """Stops (before any CUDA call) unless this is a one-GPU, one-process run."""
    if gpus != 1 or world != 1:
        raise SystemExit(f"bench.py --gpus {gpus} (WORLD_SIZE {world}): {ONE_GPU_ONLY}")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
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
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        reasons = sorted({n for r in rows for n, v in zip(self.NAMES, r[5:9]) if v.lower() == "active"})
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(power) if power else None}


def cpu_oracle_sample(z_full):
    """The CPU oracle (fp32 NumPy, frame loop) on the bounded crop; returns
    (seconds, 720p-equivalent frames, description)."""
    import oracle
    s = CPU_SAMPLE
    z = np.ascontiguousarray(z_full[:, :, :s["T"], :s["h"], :s["w"]])
    w = wan_synth.make_weights(base=WORKLOAD["base"], seed=WORKLOAD["weight_seed"])
    t0 = time.perf_counter()
    v = oracle.decode(z, w)
    dt = time.perf_counter() - t0
    frames_equiv = v.shape[2] * (v.shape[3] * v.shape[4]) / float(H_OUT * W_OUT)
    desc = (f"oracle frame loop on latents [:, :, :{s['T']}, :{s['h']}, :{s['w']}] of the 720p latents "
            f"-> {v.shape[2]} frames of {v.shape[3]}x{v.shape[4]} = {frames_equiv:.4f} frames of 704x1280")
    return dt, frames_equiv, desc


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    z = wan_synth.make_latents(WORKLOAD["latents"], WORKLOAD["latent_seed"])
    times, fe, desc = [], 0.0, ""
    for i in range(args.warmup + args.steps):
        dt, fe, desc = cpu_oracle_sample(z)
        if i >= args.warmup:
            times.append(dt)
    ms = 1000.0 * statistics.mean(times)
    value = fe / (ms / 1000.0)
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "720p: latents [1,48,31,44,80] -> video [1,3,121,704,1280]; each step a bounded crop",
                   "sample": desc},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def run_attention(args):
    """The isolated attention block: RMS norm, qkv 1x1 conv, softmax(q k^T / sqrt(C)) v over
    the frame's positions (one head, d = C), proj, + x; bf16.  Default: 8 frames of 44x80 at
    C = 1024 (the TI2V-5B mid block at 720p); --attn-shape N,C,H,W for others (e.g.
    4,384,90,160: the Wan2.1 mid block at 720p).  Head dims up to 384 run the one-CTA flash
    kernel, 512 and 1024 the flash kernel with C / 256 CTAs per 128 queries (each computes the
    scores: (C / 256 + 1) / 2 times the nominal attention-core FLOPs run on the tensor cores).
    Weights are packed once, before the timed region (wan_attention_create)."""
    import torch
    from video_vae_decoding_gb300 import build as _build
    _build.build()
    import video_vae_decoding_gb300 as wv
    cfg = wan_synth.CONFIGS["attention"]
    N, C, H, W = (int(v) for v in args.attn_shape.split(",")) if args.attn_shape else cfg["x"]
    HW = H * W
    r = np.random.default_rng(cfg["weight_seed"])
    bound = np.float32(1.0 / np.sqrt(C))
    name = "a"
    wnp = {f"{name}.norm.gamma": 1 + 0.1 * r.standard_normal(C, dtype=np.float32),
           f"{name}.to_qkv.weight": (r.random((3 * C, C, 1, 1), dtype=np.float32) * 2 - 1) * bound,
           f"{name}.to_qkv.bias": (r.random(3 * C, dtype=np.float32) * 2 - 1) * bound,
           f"{name}.proj.weight": (r.random((C, C, 1, 1), dtype=np.float32) * 2 - 1) * bound,
           f"{name}.proj.bias": (r.random(C, dtype=np.float32) * 2 - 1) * bound}
    wd = {k: torch.from_numpy(v).cuda() for k, v in wnp.items()}
    x = torch.from_numpy(wan_synth.make_normal((N, C, H, W), cfg["x_seed"])).cuda()
    x = x.permute(0, 2, 3, 1).reshape(N, HW, C).contiguous().to(torch.bfloat16)
    block = wv.AttentionBlock(wd, N, H, W, C)
    out = torch.empty_like(x)
    for _ in range(args.warmup):
        block(x, out)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        block(x, out)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    flops = 2.0 * N * HW * (3 * C * C + 2 * HW * C + C * C)
    core = 4.0 * N * HW * HW * C
    exec_flops = flops - core + core * ((C // 256 + 1) / 2.0 if C in (512, 1024) else 1.0)
    burst, sustained, _, src = _peaks()
    tf = flops / (ms / 1000.0) / 1e12
    print(json.dumps({
        "metric": f"attention block TFLOP/s (x [{N},{C},{H},{W}], bf16)", "value": tf, "unit": "TFLOP/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "dtype": "bf16", "data": "synthetic", "config": {
            "workload": f"isolated mid-block attention, {N} frames of {H}x{W}, C {C}",
            "kernel": ("flash (one CTA per 128 queries)" if C <= 384 and C % 64 == 0 else
                       "flash (C / 256 CTAs per 128 queries, scores computed by each)" if C in (512, 1024) else
                       "score GEMM + row softmax + P V GEMM"),
            "weights": "packed before the timed region"},
        "nominal_gflop_per_step": flops / 1e9, "executed_gflop_per_step": exec_flops / 1e9,
        "tflops_executed": exec_flops / (ms / 1000.0) / 1e12, "frac_of_bf16_peak": {"burst": tf / burst, "sustained": tf / sustained,
                                                                    "source": src}}))
    block.close()
    return 0


def _tile_origins(n, tile, stride):
    return [(s, min(tile, n - s)) for s in range(0, n, stride)]


def run_tiled(args):
    """The 720p clip decoded as overlapping spatial tiles (wan_vae_decode_tiled),
    default tiles of 256x256 pixels at a stride of 192; the untiled decode of
    the same clip is timed beside it."""
    import torch
    from video_vae_decoding_gb300 import build as _build
    _build.build()
    import video_vae_decoding_gb300 as wv
    th, tw = (int(v) for v in args.tile.split(","))
    sh, sw = (int(v) for v in args.stride.split(","))
    w = wan_synth.make_weights(base=WORKLOAD["base"], seed=WORKLOAD["weight_seed"])
    wdev = {k: torch.from_numpy(np.array(v)).cuda() for k, v in w.items()}
    model = wv.Model(wdev, dtype=torch.bfloat16)
    del wdev
    z = torch.from_numpy(wan_synth.make_latents((B, Z, T, H_LAT, W_LAT), WORKLOAD["latent_seed"])).cuda()
    rows = _tile_origins(H_LAT, th // 16, sh // 16)
    cols = _tile_origins(W_LAT, tw // 16, sw // 16)
    shapes = {}
    for _, rh in rows:
        for _, cw in cols:
            shapes[(rh, cw)] = shapes.get((rh, cw), 0) + 1
    # nominal FLOPs of the tile decodes, counted by the library's profiler
    flops = 0.0
    for (rh, cw), n in shapes.items():
        st = wv.DecodeStream(model, n * B, rh, cw, max_chunk=args.chunk)
        st.profile_begin()
        st.decode_clip(torch.zeros((n * B, Z, T, rh, cw), device="cuda"), out_dtype=torch.bfloat16)
        flops += st.profile_end()["tc_flops"]
        st.close()
    torch.cuda.synchronize()

    def tiled():
        return model.decode_tiled(z, tile=(th, tw), stride=(sh, sw), max_chunk=args.chunk)

    for _ in range(args.warmup):
        tiled()
    torch.cuda.synchronize()
    gpu_uuid = str(torch.cuda.get_device_properties(0).uuid)
    sampler = ClockSampler(gpu_uuid if gpu_uuid.startswith("GPU-") else f"GPU-{gpu_uuid}")
    sampler.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        tiled()
    e1.record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1) / args.steps
    # the untiled decode of the same clip, same chunking
    st = wv.DecodeStream(model, B, H_LAT, W_LAT, max_chunk=args.chunk)
    out = torch.empty((B, 3, FRAMES, H_OUT, W_OUT), device="cuda", dtype=torch.bfloat16)
    st.decode_clip(z, out)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(args.steps):
        st.decode_clip(z, out)
    e1.record()
    torch.cuda.synchronize()
    ms_untiled = e0.elapsed_time(e1) / args.steps
    burst, sustained, _, src = _peaks()
    tf = flops / (ms / 1000.0) / 1e12
    area = sum(rh * cw * n for (rh, cw), n in shapes.items()) / (H_LAT * W_LAT)
    print(json.dumps({
        "metric": f"tiled decode frames/s (704x1280, bf16, tiles {th}x{tw} stride {sh}x{sw})",
        "value": B * FRAMES / (ms / 1000.0), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16",
        "data": "synthetic: seeded random-init TI2V-5B decoder weights, N(0,1) latents",
        "config": {"workload": "720p: latents [1,48,31,44,80] -> video [1,3,121,704,1280] bf16, tiled",
                   "tiles": f"{len(rows)}x{len(cols)}", "tile_shapes_latents": {f"{a}x{b}": n for (a, b), n in
                                                                              sorted(shapes.items())},
                   "tile_area_over_frame": area, "chunk_latent_frames": args.chunk},
        "nominal_tflop_per_step": flops / 1e12, "tflops_nominal": tf,
        "frac_of_bf16_peak": {"burst": tf / burst, "sustained": tf / sustained, "source": src},
        "untiled_ms_per_step": ms_untiled, "tiled_over_untiled_time": ms / ms_untiled, "clocks": clocks}))
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--chunk", type=int, default=4, help="latent frames per causal chunk")
    ap.add_argument("--latents", default=None,
                    help="B,T,h,w of the latents (default: the 720p workload 1,31,44,80); other shapes are "
                         "for profiling and report frames of their own size")
    ap.add_argument("--workload", choices=("decode", "attention", "tiled"), default="decode",
                    help="attention: the isolated mid-block attention (x [8, 1024, 44, 80]) instead of the decode; "
                         "tiled: the 720p clip decoded as overlapping spatial tiles")
    ap.add_argument("--model", choices=("ti2v", "wan21"), default="ti2v",
                    help="wan21: the Wan2.1 VAE decode at 720p (latents [1,16,21,90,160]) instead of TI2V-5B's")
    ap.add_argument("--attn-shape", default=None,
                    help="attention workload: N,C,H,W (default 8,1024,44,80; 4,384,90,160 is Wan2.1's at 720p)")
    ap.add_argument("--tile", default="256,256", help="tiled workload: tile height,width in pixels")
    ap.add_argument("--stride", default="192,192", help="tiled workload: tile stride height,width in pixels")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    check_one_gpu(args.gpus, _dist()[0])
    if args.workload == "attention":
        return run_attention(args)
    if args.workload == "tiled":
        return run_tiled(args)
    global B, Z, T, H_LAT, W_LAT, FRAMES, H_OUT, W_OUT, METRIC, WORKLOAD
    wan21 = args.model == "wan21"
    if wan21:
        # the Wan2.1 VAE at 720p: latents [1, 16, 21, 90, 160] -> [1, 3, 81, 720, 1280]
        WORKLOAD = wan_synth.CONFIGS["wan21_720p"]
        B, Z, T, H_LAT, W_LAT = WORKLOAD["latents"]
        FRAMES, H_OUT, W_OUT = 4 * T - 3, 8 * H_LAT, 8 * W_LAT
        METRIC = f"decoded frames/s ({H_OUT}x{W_OUT}, bf16, Wan2.1 VAE)"
    custom = args.latents is not None
    if custom:
        B, T, H_LAT, W_LAT = (int(v) for v in args.latents.split(","))
        k = 8 if wan21 else 16
        FRAMES, H_OUT, W_OUT = 4 * T - 3, k * H_LAT, k * W_LAT
        METRIC = f"decoded frames/s ({H_OUT}x{W_OUT}, bf16{', Wan2.1 VAE' if wan21 else ''})"

    import torch
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)

    from video_vae_decoding_gb300 import build as _build
    _build.build()
    import video_vae_decoding_gb300 as wv

    stream = torch.cuda.current_stream()
    w = wan_synth.make_weights(base=WORKLOAD["base"], seed=WORKLOAD["weight_seed"],
                               variant=WORKLOAD.get("variant", "ti2v"))
    wdev = {k: torch.from_numpy(np.array(v)).to(dev) for k, v in w.items()}
    torch.cuda.synchronize()
    t_pack = time.perf_counter()
    model = wv.Model(wdev, dtype=torch.bfloat16)  # weight packing: outside the timed region
    torch.cuda.synchronize()
    pack_ms = (time.perf_counter() - t_pack) * 1000.0
    del wdev
    z_np = wan_synth.make_latents((B, Z, T, H_LAT, W_LAT), WORKLOAD["latent_seed"])
    z = torch.from_numpy(z_np).to(dev)
    st = wv.DecodeStream(model, B, H_LAT, W_LAT, max_chunk=args.chunk)
    out = torch.empty((B, 3, FRAMES, H_OUT, W_OUT), device=dev, dtype=torch.bfloat16)

    for _ in range(args.warmup):
        st.decode_clip(z, out)
    st.sync_status()
    free_b, total_b = torch.cuda.mem_get_info()
    mem_used_gb = (total_b - free_b) / 1e9  # all of the device in use: packed weights, workspace, I/O, context
    gpu_uuid = str(torch.cuda.get_device_properties(dev).uuid)
    sampler = ClockSampler(gpu_uuid if gpu_uuid.startswith("GPU-") else f"GPU-{gpu_uuid}")

    # ---- timed region: K clips, device-resident inputs
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    st.profile_begin()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        st.decode_clip(z, out)
    e1.record(stream)
    torch.cuda.synchronize()
    prof = st.profile_end()
    clocks = sampler.stop()
    st.sync_status()
    ms = e0.elapsed_time(e1) / args.steps
    value = B * FRAMES / (ms / 1000.0)
    burst, sustained, hbm, peak_src = _peaks()
    flops_step = prof["tc_flops"] / args.steps
    # dominant kernel: conv_gemm_kernel on the causal 3x3x3 convs (conv_in and
    # the 28 residual-block convs), timed per launch with CUDA events
    dom = prof["kinds"]["conv3x3x3"]
    achieved = dom["flops"] / (dom["ms"] / 1000.0) / 1e12 if dom["ms"] > 0 else 0.0

    # ---- end to end: host latents in, host video out, through the C ABI
    e2e = None
    if not args.no_e2e:
        z_host = torch.from_numpy(z_np).pin_memory()
        v_host = torch.empty((B, 3, FRAMES, H_OUT, W_OUT), dtype=torch.bfloat16).pin_memory()
        st.decode_clip_host(z_host, v_host)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            st.decode_clip_host(z_host, v_host)
        e2e_s = (time.perf_counter() - t0) / args.steps
        e2e = {"value": B * FRAMES / e2e_s, "unit": UNIT,
               "h2d_bytes_per_step": z_host.numel() * z_host.element_size(),
               "d2h_bytes_per_step": v_host.numel() * v_host.element_size()}

    cpu = None
    if not args.no_cpu_baseline and not custom and not wan21:
        dt, fe, desc = cpu_oracle_sample(z_np)
        cpu = {"value": fe / dt, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle", "sample": desc}

    kinds = {}
    for k, v in prof["kinds"].items():
        row = {"ms_per_step": v["ms"] / args.steps, "launches_per_step": v["launches"] / args.steps}
        if "flops" in v:
            row["tflops"] = v["flops"] / (v["ms"] / 1000.0) / 1e12 if v["ms"] > 0 else None
            # executed: the sub-pixel upsample runs 4/9 of its nominal FLOPs
            row["tflops_executed"] = v["exec_flops"] / (v["ms"] / 1000.0) / 1e12 if v["ms"] > 0 else None
            row["frac_of_sustained_executed"] = (row["tflops_executed"] / sustained
                                                 if row["tflops_executed"] else None)
        else:
            row["gbs"] = v["bytes"] / (v["ms"] / 1000.0) / 1e9 if v["ms"] > 0 else None
            row["frac_of_hbm"] = row["gbs"] / hbm if row["gbs"] else None
        kinds[k] = row
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": (f"synthetic: seeded random-init {'Wan2.1' if wan21 else 'TI2V-5B'} decoder weights, "
                 "N(0,1) latents"),
        "config": {"workload": (f"latents [{B},48,{T},{H_LAT},{W_LAT}] -> video [{B},3,{FRAMES},{H_OUT},{W_OUT}] bf16"
                                if custom or wan21 else
                                "720p: latents [1,48,31,44,80] -> video [1,3,121,704,1280] bf16"),
                   "chunk_latent_frames": args.chunk, "batch_per_gpu": B,
                   "l2": "working set larger than L2 (1.1 GB packed weights; GB-scale activations per chunk)"},
        "mpix_per_s": value * H_OUT * W_OUT / 1e6,
        "nominal_tflop_per_step": flops_step / 1e12,
        "executed_tflop_per_step": prof["tc_exec_flops"] / args.steps / 1e12,
        "tflops_nominal": flops_step / (ms / 1000.0) / 1e12,
        "frac_of_bf16_peak": {"burst": flops_step / (ms / 1000.0) / 1e12 / burst,
                              "sustained": flops_step / (ms / 1000.0) / 1e12 / sustained, "source": peak_src},
        "roofline": {"bound": "tensor",
                     "kernel": "conv_gemm_kernel<256, store, pairs, band>: causal 3x3x3 convs (implicit GEMM, tcgen05)",
                     "achieved": achieved, "peak": sustained, "unit": "TFLOP/s",
                     "frac": achieved / sustained, "peak_kind": f"bf16 sustained ({peak_src})",
                     "frac_of_burst": achieved / burst,
                     "clock_note": clock_note(clocks),
                     "launches_per_step": dom["launches"] / args.steps,
                     "flop_per_step": dom["flops"] / args.steps,
                     # DRAM bytes of one level-D 256->256 launch of 4 output frames from the
                     # ncu capture in profiles/ (algorithmic bytes of that launch: 1.156e9)
                     "traffic": None if wan21 else 1.124e9,
                     "traffic_case": None if wan21 else "level-D 256->256 causal conv, 4 frames"},
        "tensor_core_tflops": prof["tc_flops"] / (prof["tc_ms"] / 1000.0) / 1e12 if prof["tc_ms"] > 0 else None,
        "tensor_core_ms_per_step": prof["tc_ms"] / args.steps,
        "by_kind": kinds,
        "gpu_launches": prof["launches"],
        "workspace_gb": st.workspace_bytes / 1e9,
        "weight_pack_ms": pack_ms,
        "device_memory_used_gb": mem_used_gb,
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())
