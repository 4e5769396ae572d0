#!/usr/bin/env python
"""Benchmark: S2-Pro Dual-AR frame decode (one step = one frame = main draw + 9 Fast-AR calls with
their draws + one Slow-AR step) on synthetic bf16 weights of the full S2-Pro shape, batch 1.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line (rank 0).  Multi-GPU: replicas only (streams are independent; no collective):
each rank decodes its own stream; value = frames of all ranks / max rank time.
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

METRIC = "codec frames/sec per stream & aggregate (S2-Pro shapes); HBM GB/s vs 8 TB/s"
# DRAM bytes (read + write) over algorithmic bytes for one frame_kernel launch, from an ncu capture
# of the same kernel on a smaller case (S2-Pro widths, 4 Slow-AR layers, 2 frames: 16.649 GB
# measured against 16.611 GB algorithmic; the capture's summary is committed with the profiles).  Traffic grows
# with the weights and KV streamed, so the full launch's traffic is this ratio times its
# algorithmic bytes.  Set to None when the kernel changes until a new capture is taken.
NCU_TRAFFIC_RATIO = 1.0023
WORKLOAD = "full-frame Dual-AR decode, S2-Pro shapes (36+4 layers, dim 2560, vocab 155776), batch 1"
PROMPT_LEN = 512


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-frames", type=int, default=2, help="frames in the CPU-oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batched", default="serving,longctx",
                    help="comma-separated batched workloads to measure as well (serving, longctx; 'none')")
    ap.add_argument("--batched-steps", type=int, default=None,
                    help="frames per stream of the batched workloads (default: the workload's own count)")
    ap.add_argument("--no-extra", dest="extra", action="store_false",
                    help="skip the tiny-model, Fast-AR-alone and long-prompt prefill measurements")
    ap.add_argument("--no-fp8", dest="fp8", action="store_false",
                    help="skip the fp8 e4m3 weight-streaming measurements")
    ap.add_argument("--batched-streams", type=int, default=None,
                    help="profiling captures only: the first N streams of the batched workload")
    ap.add_argument("--slow-layers", type=int, default=None,
                    help="profiling captures only: Slow-AR layer count (S2-Pro widths kept); the bench line "
                         "then describes that smaller model")
    return ap.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def frame_bytes(d, ctx_avg):
    """Algorithmic HBM bytes of one frame at batch 1: every weight the frame needs, read once
    per use (Fast-AR weights once per call), admissible tied-logit rows, embedding rows gathered,
    KV cache read over the context and the new slot written."""
    e = 2  # bf16
    fp8 = bool(d.get("weight_fp8", 0))
    # projection matrices: bf16, or e4m3 codes + one fp32 scale per row when streamed as fp8
    mat = (lambda r, c: r * c + 4 * r) if fp8 else (lambda r, c: r * c * e)
    D, F, hd = d["dim"], d["ffn"], d["head_dim"]
    lay = lambda D_, H, Hk, h, F_: mat((H + 2 * Hk) * h, D_) + mat(D_, H * h) + 2 * mat(F_, D_) + mat(D_, F_)
    slow = d["n_layer"] * lay(D, d["n_head"], d["n_kv_head"], hd, F)
    logits = (d["codebook_size"] + 1) * D * e
    gathers = (1 + d["n_codebooks"]) * D * e + (d["n_codebooks"] - 1) * d["fast_dim"] * e
    fast = (d["n_codebooks"] - 1) * (d["fast_n_layer"] * lay(d["fast_dim"], d["fast_n_head"], d["fast_n_kv_head"],
                                                             d["fast_head_dim"], d["fast_ffn"])
                                     + mat(d["codebook_size"], d["fast_dim"]))
    proj = mat(d["fast_dim"], D)
    kv_per_slot = d["n_layer"] * d["n_kv_head"] * hd * 2 * 2  # K and V, fp16
    kv = kv_per_slot * (ctx_avg + 1)  # read slots 0..pos, the new one written
    return slow + logits + gathers + fast + proj + kv, dict(slow=slow, logits=logits, fast=fast + proj, kv=kv)


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                mhz.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(mhz)}


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def batched_measure(pkg, d, dev_w, cfg_name, steps, warmup, peak, local, n_streams=None):
    """Aggregate frames/s of a batched workload: every stream of the workload decoded in one call
    (weights read once per step for the whole batch).  Each stream's decode state (its context's
    fp16 K/V, its last residual) is imported from seeded device-side random values: the KV
    contents do not change the work of a decode step, and a prefill of these contexts is not part
    of the timed step.  Returns the dict reported under 'batched'."""
    import numpy as np
    import torch
    import synth
    cfg = synth.CONFIGS[cfg_name]
    n, slots, seed = cfg["streams"], cfg["kv_slots"], cfg["input_seed"]
    steps = steps or cfg["frames"]
    lengths = synth.prompt_lengths(cfg_name)
    if n_streams:
        n = min(n, n_streams)
        lengths = lengths[:n]
    kmax = max(lengths)
    dec = pkg.Decoder(d, dev_w, max_streams=n, kv_slots=slots)
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    shape = (d["n_layer"], d["n_kv_head"], kmax, d["head_dim"])
    k = torch.randn(shape, generator=g, device="cuda", dtype=torch.float32).half()
    v = torch.randn(shape, generator=g, device="cuda", dtype=torch.float32).half()
    for i, L in enumerate(lengths):
        x = torch.randn(d["dim"], generator=g, device="cuda", dtype=torch.float32)
        dec.import_stream(i, k[:, :, :L].contiguous(), v[:, :, :L].contiguous(), x)
    del k, v
    s = synth.sampling(cfg_name, min_tokens_before_end=warmup + steps + 1)
    ex = np.stack([synth.expo(seed, i, warmup + steps) for i in range(n)])
    expo_w = torch.from_numpy(np.ascontiguousarray(ex[:, :warmup])).cuda()
    expo_t = torch.from_numpy(np.ascontiguousarray(ex[:, warmup:])).cuda()
    dec.decode(warmup, s, expo_w)
    torch.cuda.synchronize()
    assert dec.sync_status() == pkg.S2_OK, pkg.s2_last_error(dec.ctx)
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        ev0.record(stream)
        out = dec.decode(steps, s, expo_t)
        ev1.record(stream)
        torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    assert dec.sync_status() == pkg.S2_OK, pkg.s2_last_error(dec.ctx)
    assert (out["n_out"].cpu().numpy() == steps).all()
    dec.close()
    w_bytes, parts = frame_bytes(d, 0)
    w_bytes -= parts["kv"]
    kv_slot = d["n_layer"] * d["n_kv_head"] * d["head_dim"] * 2 * 2
    ctx_avg = [L + warmup + (steps - 1) / 2.0 for L in lengths]
    step_bytes = w_bytes + sum(kv_slot * (c + 1) for c in ctx_avg)
    t = ms / 1000.0
    achieved = step_bytes * steps / t / 1e9
    wname = "fp8 e4m3 projections (per-row scales)" if d.get("weight_fp8") else "bf16 weights"
    return {"workload": f"{cfg_name}: {n} streams, contexts {min(lengths)}..{kmax}, {wname}, fp16 KV "
                        f"(decode state imported, see docstring)",
            "streams": n, "frames_per_stream": steps, "warmup": warmup,
            "value": n * steps / t, "unit": "frames/s (aggregate)", "per_stream_fps": steps / t,
            "ms_per_step": ms / steps, "algorithmic_gb_per_step": step_bytes / 1e9,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak},
            "clocks": clk.summary()}


def fp8_measure(pkg, d, dev_w, prompt, args, peak, local):
    """The same two measurements with the projection matrices streamed as fp8 e4m3 (quantised by
    the library at init): one stream (the frame workload, decoded by the batched engine) and the
    batched workload."""
    import torch
    import synth
    d8 = dict(d, weight_fp8=1)
    K, W = args.steps, args.warmup
    s = synth.sampling("frame", min_tokens_before_end=W + K + 1)
    dec = pkg.Decoder(d8, dev_w, max_streams=1, kv_slots=PROMPT_LEN + W + K + 8)
    dec.prefill([prompt])
    expo_w = torch.from_numpy(synth.expo(100, 0, W)).cuda()[None]
    dec.decode(W, s, expo_w)
    torch.cuda.synchronize()
    assert dec.sync_status() == pkg.S2_OK, pkg.s2_last_error(dec.ctx)
    expo = torch.from_numpy(synth.expo(200, 0, K)).cuda()[None]
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        ev0.record(stream)
        out = dec.decode(K, s, expo)
        ev1.record(stream)
        torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    assert dec.sync_status() == pkg.S2_OK, pkg.s2_last_error(dec.ctx)
    assert int(out["n_out"][0]) == K
    dec.close()
    torch.cuda.empty_cache()
    fb, parts = frame_bytes(d8, PROMPT_LEN + W + (K - 1) / 2.0)
    achieved = fb * K / (ms / 1000.0) / 1e9
    res = {"weights": "projections e4m3 + fp32 row scales; embeddings, norms and tied logits bf16",
           "batch1": {"workload": "frame: 1 stream, context 512, batched engine", "value": K / (ms / 1000.0),
                      "unit": "frames/s", "ms_per_step": ms / K, "algorithmic_gb_per_frame": fb / 1e9,
                      "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                                   "frac": achieved / peak},
                      "clocks": clk.summary()}}
    work = batched_workloads(args)
    if work:
        res["batched"] = batched_measure(pkg, d8, dev_w, work[0], args.batched_steps, W, peak, local,
                                         args.batched_streams)
    return res


def batched_workloads(args):
    return [w for w in args.batched.split(",") if w and w != "none"]


def tiny_measure(pkg, args):
    """The tiny Dual-AR model (fp32, L2-resident weights): frames/s of its 16-frame decode."""
    import torch
    import synth
    cfg = synth.CONFIGS["tiny"]
    d = cfg["dims"]
    dec = pkg.Decoder(d, pkg.upload_weights(synth.make_weights(d, 0)), max_streams=1, kv_slots=cfg["kv_slots"])
    n = cfg["frames"]
    s = synth.sampling("tiny")
    best = None
    for rep in range(4):
        dec.prefill([synth.prompt("tiny")])
        expo = torch.from_numpy(synth.expo(cfg["input_seed"], 0, n)).cuda()[None]
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record()
        out = dec.decode(n, s, expo)
        ev1.record()
        torch.cuda.synchronize()
        assert dec.sync_status() == pkg.S2_OK
        ms = ev0.elapsed_time(ev1)
        if rep > 0:  # the first call is a warm-up
            best = ms if best is None else min(best, ms)
    produced = int(out["n_out"][0])
    dec.close()
    return {"workload": "tiny Dual-AR (dim 256, 4+2 layers, fp32), 32-position prompt, one call of 16 frames",
            "value": produced / (best / 1000.0), "unit": "frames/s", "ms_per_frame": best / produced,
            "roofline": "n/a (weights L2-resident, latency-bound)"}


def fast_measure(pkg, d_full, dev_w, peak, args):
    """Fast-AR alone at S2-Pro shapes, batch 1: 1000 teacher-forced frames x 9 windows."""
    import torch
    import synth
    cfg = synth.CONFIGS["fast"]
    d = cfg["dims"]
    by = dict(zip([nm for nm, _, _ in synth.weight_specs(d_full)], dev_w))
    w = [None if nm in ("embeddings", "codebook_embeddings", "norm") else by[nm] for nm, _, _ in synth.weight_specs(d)]
    dec = pkg.Decoder(d, w, max_streams=1, kv_slots=0)
    n = cfg["frames"]
    hid, pre = synth.fast_inputs(cfg["input_seed"], n, d)
    h, p = torch.from_numpy(hid).cuda(), torch.from_numpy(pre).cuda()
    dec.fast_logits(h[:8].contiguous(), p[:8].contiguous())
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    dec.fast_logits(h, p)
    ev1.record()
    torch.cuda.synchronize()
    assert dec.sync_status() == pkg.S2_OK
    ms = ev0.elapsed_time(ev1)
    dec.close()
    _, parts = frame_bytes(d_full, 0)
    fb = parts["fast"]
    achieved = fb * n / (ms / 1000.0) / 1e9
    return {"workload": "Fast-AR alone, S2-Pro shapes (4 layers, dim 2560), batch 1, 1000 frames x 9 windows",
            "value": n / (ms / 1000.0), "unit": "frames/s", "ms_per_frame": ms / n,
            "algorithmic_gb_per_frame": fb / 1e9,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak}}


def prefill_long_measure(pkg, d, dev_w):
    """Prefill of the 30000-position long-context prompt (1000 text ids, 29000 reference positions)."""
    import torch
    import synth
    prompt = synth.prompt("longctx", stream=0)
    dec = pkg.Decoder(d, dev_w, max_streams=1, kv_slots=len(prompt) + 8)
    dec.prefill([prompt[:512]])
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    dec.prefill([prompt])
    ev1.record()
    torch.cuda.synchronize()
    assert dec.sync_status() == pkg.S2_OK
    ms = ev0.elapsed_time(ev1)
    dec.close()
    return {"positions": len(prompt), "ms": ms, "positions_per_s": len(prompt) / (ms / 1000.0)}


def cpu_oracle_sample(d, host_w, n_frames, s):
    """Oracle (plain fp32 C + OpenMP) on the host cores: n_frames whole frames timed from a decode
    state of the bench's context (PROMPT_LEN positions).  The state is seeded synthetic fp16 K/V
    and a last residual (the oracle's own prefill of the prompt takes minutes; the contents of the
    cache do not change the work of a frame).  Returns (frames/s, cores, description)."""
    import oracle
    import synth
    sess = oracle.Session(d, host_w, PROMPT_LEN + n_frames + 1)
    k16, v16, x = synth.kv_state(9, 0, d, PROMPT_LEN)
    logits, hidden = sess.import_state(k16, v16, x)
    expo = synth.expo(9, 0, n_frames)
    t = time.perf_counter()
    oracle.run_frames(sess, logits, hidden, n_frames, dict(s, min_tokens_before_end=n_frames), expo, trace=False)
    dt = time.perf_counter() - t
    sess.close()
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count()))
    return n_frames / dt, cores, (f"{n_frames} whole frames (main draw over the full vocabulary, 9 Fast-AR calls "
                                  f"recomputed per window, Slow-AR step) at a {PROMPT_LEN}-position context "
                                  f"(seeded fp16 K/V state); S2-Pro shapes, bf16 weights widened to fp32")


def bench_config(world, K, fb=None):
    c = {"workload": WORKLOAD, "global_batch": world, "seq_len": PROMPT_LEN,
         "parallelism": f"replicas{world}" if world > 1 else "none", "frames_per_call": K}
    c["l2"] = "inputs larger than L2 (about 14.8 GB of weights and KV streamed per frame)"
    return c


def run_reference(args):
    """The oracle as the reference arm (the pages ship no runnable code)."""
    import synth
    world, rank, _ = dist_setup(args)
    if rank != 0:
        return 0
    d = synth.CONFIGS["frame"]["dims"]
    host_w = synth.make_weights(d, 0)
    s = synth.sampling("frame")
    frames = max(1, min(args.cpu_frames, 4))
    t0 = time.perf_counter()
    vals = []
    for _ in range(max(1, min(args.steps, 2))):
        v, cores, sample = cpu_oracle_sample(d, host_w, frames, s)
        vals.append(v)
    v = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "frames/s", "n_gpus": args.gpus,
            "steps": len(vals), "warmup": 0, "ms_per_step": 1000.0 / v, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": bench_config(args.gpus, args.steps),
            "cpu_baseline": {"kind": "oracle", "value": v, "unit": "frames/s", "cores": cores, "sample": sample},
            "e2e": {"value": v, "unit": "frames/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": time.perf_counter() - t0}
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    import numpy as np
    import torch

    import dual_ar_tts_gb300 as pkg
    import synth

    world, rank, local = dist_setup(args)
    torch.cuda.set_device(local)
    if args.warmup < 3:
        args.warmup = 3
    d = synth.CONFIGS["frame"]["dims"]
    workload = WORKLOAD
    if args.slow_layers is not None:
        d = dict(d, n_layer=args.slow_layers)
        workload = WORKLOAD.replace("36+4 layers", f"{args.slow_layers}+4 layers (profiling case)")
    s = synth.sampling("frame", min_tokens_before_end=args.warmup + args.steps + 1)
    t_setup = time.perf_counter()
    host_w = synth.make_weights(d, 0)
    dev_w = pkg.upload_weights(host_w)
    kv_slots = PROMPT_LEN + args.warmup + 2 * args.steps + 8
    dec = pkg.Decoder(d, dev_w, max_streams=1, kv_slots=kv_slots)
    prompt = synth.prompt("frame", stream=rank)
    dec.prefill([prompt])  # first prefill: one-time setup (tensor maps, caches)
    torch.cuda.synchronize()
    pe0, pe1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pe0.record()
    dec.prefill([prompt])  # timed: the stream is reset and the prompt run again
    pe1.record()
    torch.cuda.synchronize()
    prefill_ms = pe0.elapsed_time(pe1)
    assert dec.sync_status() == pkg.S2_OK, pkg.s2_last_error(dec.ctx)
    setup_s = time.perf_counter() - t_setup

    stream = torch.cuda.current_stream()
    expo_w = torch.from_numpy(synth.expo(100 + rank, 0, args.warmup)).cuda()[None]
    out = dec.decode(args.warmup, s, expo_w)
    torch.cuda.synchronize()
    assert dec.sync_status() == pkg.S2_OK, pkg.s2_last_error(dec.ctx)
    assert int(out["n_out"][0]) == args.warmup

    # ---- device-timed: one call decoding K frames (inputs resident in HBM)
    expo = torch.from_numpy(synth.expo(200 + rank, 0, args.steps)).cuda()[None]
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        ev0.record(stream)
        out = dec.decode(args.steps, s, expo)
        ev1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    dev_ms = ev0.elapsed_time(ev1)
    st = dec.sync_status()
    if st != pkg.S2_OK:
        raise RuntimeError(pkg.s2_last_error(dec.ctx))
    produced = int(out["n_out"][0])
    assert produced == args.steps, (produced, args.steps)
    t_max = max_over_ranks(dev_ms, world)

    # ---- end to end through the C ABI with host buffers (pinned): H2D of the step's variates,
    # decode, D2H of the emitted codes and frame count
    K = args.steps
    expo_h = torch.from_numpy(synth.expo(300 + rank, 0, K)).pin_memory()
    expo_d = torch.empty_like(expo_h, device="cuda")
    codes_h = torch.empty((1, d["n_codebooks"] * K), dtype=torch.int32).pin_memory()
    nout_h = torch.empty(1, dtype=torch.int32).pin_memory()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    expo_d.copy_(expo_h, non_blocking=True)
    o2 = dec.decode(K, s, expo_d[None])
    codes_h.copy_(o2["codes"], non_blocking=True)
    nout_h.copy_(o2["n_out"], non_blocking=True)
    torch.cuda.synchronize()
    e2e_s = time.perf_counter() - t0
    barrier(world)
    e2e_max = max_over_ranks(e2e_s, world)
    assert int(nout_h[0]) == K

    # codec front on the frames just produced: latent = Σ_cb quantizer_cb[code] (synthetic codebooks)
    qs = synth.codec_quantizers(11, d["n_codebooks"], d["codebook_size"])
    dq = [torch.from_numpy(q.view(np.int16)).cuda() for q in qs]
    lat = torch.empty((K, synth.CODEC_DIM), device="cuda")
    codes_d = o2["codes"][0].contiguous()
    args_q = [t.data_ptr() for t in dq]
    for _ in range(3):
        pkg.s2_codec_latent(d["n_codebooks"], d["codebook_size"], synth.CODEC_DIM, args_q, K, codes_d.data_ptr(),
                            lat.data_ptr())
    ce0, ce1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ce0.record()
    for _ in range(10):
        pkg.s2_codec_latent(d["n_codebooks"], d["codebook_size"], synth.CODEC_DIM, args_q, K, codes_d.data_ptr(),
                            lat.data_ptr())
    ce1.record()
    torch.cuda.synchronize()
    codec_us = ce0.elapsed_time(ce1) * 100.0
    codec_bytes = K * synth.CODEC_DIM * (2 * d["n_codebooks"] + 4)
    pk, pk_kind = peaks()
    ctx_avg = PROMPT_LEN + args.warmup + (K - 1) / 2.0
    fb, parts = frame_bytes(d, ctx_avg)
    achieved = fb * K / (dev_ms / 1000.0) / 1e9
    value = world * K / (t_max / 1000.0)
    line = {
        "metric": METRIC, "value": value, "unit": "frames/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": t_max / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded random weights of the S2-Pro shape, synthetic prompt/variates)",
        "config": dict(bench_config(world, K), workload=workload),
        "per_stream_fps": K / (dev_ms / 1000.0),
        "hbm": {"algorithmic_gb_per_frame": fb / 1e9, "achieved_gbs": achieved, "frac_of_8tbs": achieved / 8000.0,
                "frac_of_measured": achieved / pk, "parts_gb": {k: v / 1e9 for k, v in parts.items()}},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk, "unit": "GB/s", "frac": achieved / pk,
                     "traffic": NCU_TRAFFIC_RATIO * fb * K if NCU_TRAFFIC_RATIO else None,
                     "traffic_unit": "bytes per launch", "algorithmic_bytes": fb * K, "kernel": "frame_kernel", "peak_kind": pk_kind},
        "e2e": {"value": world * K / e2e_max, "unit": "frames/s", "h2d_bytes_per_step": int(expo_h[0].numel() * 4),
                "d2h_bytes_per_step": int(d["n_codebooks"] * 4)},
        "prefill": {"positions": len(prompt), "ms": prefill_ms, "positions_per_s": len(prompt) / (prefill_ms / 1000.0),
                    "projections": "tcgen05" if d["weight_dtype"] == synth.BF16 else "fp32 tiles"},
        "codec_latent": {"frames": K, "us": codec_us, "frames_per_s": K / (codec_us / 1e6),
                         "gb_s": codec_bytes / (codec_us * 1e3)},
        "gpu_launches": 2,
        "clocks": clk.summary(),
        "setup_s": setup_s,
    }
    work = batched_workloads(args)
    if work:
        dec.close()
        torch.cuda.empty_cache()
        line["batched"] = batched_measure(pkg, d, dev_w, work[0], args.batched_steps, args.warmup, pk, local,
                                          args.batched_streams)
        for wname in work[1:]:
            torch.cuda.empty_cache()
            line[f"batched_{wname}"] = batched_measure(pkg, d, dev_w, wname, args.batched_steps, args.warmup, pk,
                                                       local, args.batched_streams)
    if args.extra and args.slow_layers is None:
        dec.close()
        torch.cuda.empty_cache()
        line["tiny"] = tiny_measure(pkg, args)
        line["fast_alone"] = fast_measure(pkg, d, dev_w, pk, args)
        line["prefill_longctx"] = prefill_long_measure(pkg, d, dev_w)
    if args.fp8:
        dec.close()
        torch.cuda.empty_cache()
        line["fp8"] = fp8_measure(pkg, d, dev_w, prompt, args, pk, local)
    if rank == 0 and not args.no_cpu_baseline and args.slow_layers is None:
        try:
            v, cores, sample = cpu_oracle_sample(d, host_w, args.cpu_frames, s)
            line["cpu_baseline"] = {"value": v, "unit": "frames/s", "cores": cores, "kind": "oracle", "sample": sample}
        except Exception as e:  # pragma: no cover
            line["cpu_baseline"] = {"value": None, "unit": "frames/s", "cores": os.cpu_count(), "kind": "oracle",
                                    "sample": f"failed: {e}"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    dec.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
