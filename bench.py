"""Throughput of the V-JEPA 2 ViT-L/16 encoder forward on GB300.

Workload: ViT-L/16 (D 1024, 24 layers, 16 heads, FFN 4096), bf16 weights and
activations with fp32 accumulation and fp32 residual stream, tiled 3-D RoPE,
clips of 16 frames x 256 x 256 (2048 tokens each), batch 8 per GPU.  Weights
N(0, 0.02) and uniform uint8 clips from the seeded generator (synthetic: the
pages' real clips and checkpoints are not available).

One step = one jepa_encode call over the batch (patch embed, 24 blocks, final
LayerNorm), inputs already resident in HBM.  The L2 cache (129 MB) is flushed
between timed steps by writing a 256 MB buffer outside the timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--workload vitl16-16f256 | vitb16-img384]

--workload vitb16-img384 measures the V-JEPA 2.1 native image path instead
(ViT-B/16, 32 images of 384 x 384, 576 tokens each) and prints the same line
for that workload; --workload vitl16-16f256-ssv2 adds the SSv2 attentive-pool
head and 174-class classifier to every step.

Under torchrun (N > 1) every rank runs its own replica (weak scaling, no
collective on the data path); rank 0 prints one JSON line.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

UNIT = "tokens/s"
# name -> (seeded config, metric, workload description, fraction of tokens kept or None)
WORKLOADS = {
    "vitl16-16f256": ("vitl16-16f256", "encoder tokens/sec (ViT-L/16, 16f 256px, bf16) and % of bf16 tensor peak",
                      "ViT-L/16 24L D1024 h16 FFN4096, bf16, tiled RoPE, 16f x 256x256 (2048 tokens/clip), "
                      "batch 8 per GPU", None),
    "vitl16-16f256-masked50": ("vitl16-16f256", "masked-encoder kept tokens/sec (ViT-L/16, 16f 256px, half the "
                               "tokens kept, bf16) and % of bf16 tensor peak",
                               "ViT-L/16 24L D1024 h16 FFN4096, bf16, tiled RoPE, 16f x 256x256, masked encoder "
                               "forward keeping a seeded random 1024 of each clip's 2048 tokens, batch 8 per GPU", 0.5),
    "vitb16-img384": ("img384", "encoder tokens/sec (V-JEPA 2.1 ViT-B/16 native image path, 384px, bf16) and % of "
                      "bf16 tensor peak",
                      "ViT-B/16 12L D768 h12 FFN3072, bf16, 2.1 native image path (tubelet 1, patch_embed_img), "
                      "interleaved interpolated RoPE, 1f x 384x384 (576 tokens/image), batch 32 per GPU", None),
    "vitl16-16f256-ssv2": ("vitl16-16f256", "classified tokens/sec (ViT-L/16 encoder + SSv2 attentive-pool head "
                           "and 174-class classifier, 16f 256px, bf16) and % of bf16 tensor peak",
                           "ViT-L/16 24L D1024 h16 FFN4096, bf16, tiled RoPE, 16f x 256x256 (2048 tokens/clip), then the "
                           "attentive-pool head (3 pool blocks, 16 heads, single-query cross-attention, 174 classes), "
                           "batch 8 per GPU", None),
    "vitl16-64f256": ("vitl16-64f256-pred", "encoder tokens/sec (ViT-L/16, 64f 256px, bf16) and % of bf16 tensor "
                      "peak",
                      "ViT-L/16 24L D1024 h16 FFN4096, bf16, tiled RoPE, 64f x 256x256 (8192 tokens/clip), "
                      "batch 1 per GPU", None),
    "vitb16-64f384": ("vitb16-64f384", "encoder tokens/sec (V-JEPA 2.1 ViT-B/16, 64f 384px, bf16) and % of bf16 "
                      "tensor peak",
                      "ViT-B/16 12L D768 h12 FFN3072, bf16, interleaved interpolated RoPE, 64f x 384x384 "
                      "(18432 tokens/clip), batch 1 per GPU", None),
}
# Workloads whose step also runs the SSv2 attentive-pool head and classifier
# on the encoder's output (the conversion notes' classifier checkpoint geometry).
HEAD_WORKLOADS = {"vitl16-16f256-ssv2"}
# The oracle holds each head's full score matrix in float64; above this many
# tokens per clip one of its blocks no longer fits a bounded CPU sample.
CPU_BASELINE_MAX_TOKENS = 8192
DEFAULT_WORKLOAD = "vitl16-16f256"
CLASSES = ["patch_embed", "layernorm", "qkv_gemm", "attention", "out_proj_gemm", "ffn_up_gemm", "ffn_down_gemm",
           "other"]


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"bf16_burst": d["bf16_tflops"], "bf16_sustained": d["bf16_tflops_sustained"],
                "hbm_gbs": d["hbm_gbs"], "source": "measured"}
    return {"bf16_burst": 1900.0, "bf16_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


def _patch_k(cfg):
    """Width of one token's unfolded pixels: 3 x tubelet x 16 x 16 (tubelet 1 on the image path)."""
    tub = 1 if (cfg.n_frames == 1 and cfg.has_image_path) else cfg.tubelet
    return 3 * tub * cfg.patch * cfg.patch


def flops_per_clip(cfg, n_tok):
    """Algorithmic FLOPs of one clip: per token L*(24 D^2 + 4 N D) + 2*K_patch*D."""
    D, L, F = cfg.embed_dim, cfg.n_layer, cfg.ffn_dim
    per_tok_layer = 2 * (3 * D * D + D * D + 2 * D * F) + 4 * n_tok * D
    return n_tok * (L * per_tok_layer + 2 * _patch_k(cfg) * D)


def head_flops_per_clip(hc, n_tok):
    """Algorithmic FLOPs of the attentive-pool head on one clip: the pool blocks
    like encoder blocks (no patch embed), the cross-attention's k/v projections
    of every token and its single-query scores and sums, and the per-clip MLP and
    classifier."""
    D, F, L, C = hc.embed_dim, hc.ffn_dim, hc.n_layer, hc.n_classes
    blocks = n_tok * L * (2 * (3 * D * D + D * D + 2 * D * F) + 4 * n_tok * D)
    xattn = 2 * n_tok * 2 * D * D + 4 * n_tok * D + 2 * D * D
    tail = 2 * (D * D + 2 * D * F + C * D)
    return blocks + xattn + tail


def class_flops_per_launch(cfg, batch, n_tok):
    D, F, H = cfg.embed_dim, cfg.ffn_dim, cfg.n_head
    M = batch * n_tok
    return {"patch_embed": 2 * M * _patch_k(cfg) * D, "qkv_gemm": 2 * M * D * 3 * D, "attention": 4 * batch * H * n_tok * n_tok * (D // H),
            "out_proj_gemm": 2 * M * D * D, "ffn_up_gemm": 2 * M * D * F, "ffn_down_gemm": 2 * M * F * D}


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.5)   # nvidia-smi is sampling before the timed region starts
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def _source_sha(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _traffic_for(kernel_class, launch_key):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current source of that kernel; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel_class)
    if not e or e.get("launch") != launch_key:
        return None
    if e.get("source_sha") != _source_sha(e.get("sources", [])):
        return None
    return e.get("dram_bytes_per_launch")


def first_clip_for_rank(rank: int, batch: int) -> int:
    """Replicas encode disjoint clips: rank r takes clip streams r*B .. r*B+B-1."""
    return rank * batch


def max_over_ranks(value: float, dist=None, device="cpu") -> float:
    """The slowest rank's value (the job's time), or value itself on one rank."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _host_threads():
    """(host cores, threads the oracle's BLAS uses)."""
    try:
        host = len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        host = os.cpu_count() or 1
    try:
        from threadpoolctl import threadpool_info
        blas = max((i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"), default=host)
    except Exception:
        blas = host
    return host, blas


def _oracle_blocks(cfg, weights, x, COS, SIN, l0, l1):
    import oracle
    for i in range(l0, l1):
        x = oracle.block_forward(x, weights, i, cfg.n_head, cfg.ln_eps, COS, SIN)
    return x


def cpu_baseline(cfg, weights, clip, whole=True, head=None):
    """The oracle, as it stands, on the host cores: one clip's forward timed
    end to end (patch embed, every block, final norm) when ``whole``; else
    (clips too long for a bounded sample) the patch embed and one block timed
    and the clip time extrapolated as embed + n_layer x block + norm."""
    import oracle
    T, H, W, _ = clip.shape
    host, blas = _host_threads()
    t0 = time.perf_counter()
    x = oracle.encoder_embed(cfg, weights, clip)
    COS, SIN = oracle.encoder_rope(cfg, T, H, W)
    t_embed = time.perf_counter() - t0
    n_run = cfg.n_layer if whole else 1
    t0 = time.perf_counter()
    x = _oracle_blocks(cfg, weights, x, COS, SIN, 0, n_run)
    t_blocks = time.perf_counter() - t0
    t0 = time.perf_counter()   # the final norm (and the head)
    out = oracle.layer_norm(x, weights["norm.weight"], weights["norm.bias"], cfg.ln_eps)
    if head is not None:   # whole clips only: the head on the oracle's own tokens
        import synth
        oracle.attentive_pool_forward(head, synth.head_weights(head, cfg.seed, cfg.dtype), out)
    t_tail = time.perf_counter() - t0
    n_tok = x.shape[0]
    if whole:
        sec = t_embed + t_blocks + t_tail
        sample = (f"1 clip ({n_tok} tokens): patch embed + {cfg.n_layer} of {cfg.n_layer} blocks + final norm"
                  f"{' + attentive-pool head' if head is not None else ''}, timed end to end in float64: {sec:.2f} s")
    else:
        sec = t_embed + cfg.n_layer * t_blocks + t_tail
        sample = (f"1 clip ({n_tok} tokens): patch embed + 1 of {cfg.n_layer} blocks + final norm timed in float64, "
                  f"extrapolated to {cfg.n_layer} blocks: {sec:.2f} s")
    return {"value": n_tok / sec, "unit": UNIT, "cores": blas, "host_cores": host, "kind": "oracle",
            "sample": sample, "seconds_per_clip": sec}


def run_reference(args):
    """--impl reference: the CPU oracle, timed on the host cores.

    A step is a bounded sample of the workload: half of one clip's forward
    (the patch embed and the first n_layer/2 blocks, or the remaining blocks
    and the final norm), the halves alternating on the carried residual, so
    every two consecutive steps encode one whole clip and each step's time is
    what it measured.  Warm-up steps run the patch embed and one block."""
    import synth
    import oracle
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    key, metric, workload, keep_frac = WORKLOADS[args.workload]
    if keep_frac is not None or args.workload in HEAD_WORKLOADS:
        print(json.dumps({"impl": "reference", "unavailable": "the oracle arm times the encoder-only unmasked workloads"}))
        return 0
    cfg = synth.CONFIGS[key]
    if synth.tokens_per_clip(cfg) > CPU_BASELINE_MAX_TOKENS:
        print(json.dumps({"impl": "reference", "unavailable": f"one oracle block at {synth.tokens_per_clip(cfg)} "
                          "tokens per clip takes minutes on the host cores (float64 score matrices)"}))
        return 0
    w = synth.encoder_weights(cfg)
    clip = synth.clip_u8(cfg, batch=1)[0]
    T, H, W, _ = clip.shape
    COS, SIN = oracle.encoder_rope(cfg, T, H, W)
    L, half = cfg.n_layer, cfg.n_layer // 2
    for _ in range(args.warmup):
        x = oracle.encoder_embed(cfg, w, clip)
        _oracle_blocks(cfg, w, x, COS, SIN, 0, 1)
    times = []
    x = None
    for i in range(args.steps):
        t0 = time.perf_counter()
        if i % 2 == 0:
            x = oracle.encoder_embed(cfg, w, clip)
            x = _oracle_blocks(cfg, w, x, COS, SIN, 0, half)
        else:
            x = _oracle_blocks(cfg, w, x, COS, SIN, half, L)
            oracle.layer_norm(x, w["norm.weight"], w["norm.bias"], cfg.ln_eps)
        times.append(time.perf_counter() - t0)
    n_tok = synth.tokens_per_clip(cfg)
    total = sum(times)
    v = n_tok * (args.steps / 2.0) / total
    host, blas = _host_threads()
    whole = [times[j] + times[j + 1] for j in range(0, args.steps - 1, 2)]
    sample = (f"each step half of one clip's forward in float64 ({half} of {L} blocks, with the patch embed or the "
              f"final norm), halves alternating, so every two steps encode one whole clip of {n_tok} tokens"
              + (f"; whole-clip times {min(whole):.2f}-{max(whole):.2f} s" if whole else ""))
    line = {"impl": "reference", "metric": metric, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total * 1000.0 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload, "global_batch": cfg.batch, "seq_len": n_tok,
                       "parallelism": "none",
                       "note": "CPU oracle on the host cores; each step half of one of the batch's clips"},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": blas, "host_cores": host, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    import numpy as np
    import torch

    import synth
    import video_vit_encoder_gb300 as jg

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    key, metric, workload, keep_frac = WORKLOADS[args.workload]
    cfg = synth.CONFIGS[key]
    B = cfg.batch
    n_grid = synth.tokens_per_clip(cfg)
    # tokens per clip that pass through the blocks (all, or the kept ones)
    n_tok = n_grid if keep_frac is None else int(n_grid * keep_frac)
    weights = synth.encoder_weights(cfg)
    # each rank encodes its own clips (clip streams rank*B .. rank*B+B-1)
    clip_np = synth.clip_u8(cfg, batch=B, first_clip=first_clip_for_rank(rank, B))
    enc = jg.Encoder(cfg, weights, device=local)
    clip = torch.from_numpy(clip_np).cuda()
    out = torch.empty((B, n_tok, cfg.embed_dim), dtype=torch.float32, device="cuda")
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    head = None
    if args.workload in HEAD_WORKLOADS:
        hc = synth.HEAD_SSV2
        head = jg.Head(hc, synth.head_weights(hc, cfg.seed, cfg.dtype), cfg.dtype, device=local)
        logits = torch.empty((B, hc.n_classes), dtype=torch.float32, device="cuda")

        def step():
            enc.encode(clip, out=out)
            head.forward(out, out=logits)
    elif keep_frac is None:
        def step():
            enc.encode(clip, out=out)
    else:
        keep = torch.from_numpy(np.stack([np.random.default_rng(1000 + b).choice(n_grid, n_tok, replace=False)
                                          for b in range(B)]).astype(np.int32)).cuda()

        def step():
            return enc.encode_masked(clip, keep, out=out)["out"]

    for _ in range(args.warmup):
        step()
    enc.sync()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        for i in range(args.steps):
            flush.fill_(float(i))                     # L2 flush, outside the timed region
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
    enc.sync()
    if dist:
        dist.barrier()
    # Per-class times come from separate profiled steps: the events around
    # every kernel class cost about 5 % of a step, so the timed steps above
    # run without them.
    n_prof = min(args.steps, 10)
    enc.profile(reset=True)
    enc.set_profiling(True)
    for i in range(n_prof):
        flush.fill_(float(i))
        step()
    enc.sync()
    enc.set_profiling(False)
    prof = enc.profile(reset=True)
    total_ms = max_over_ranks(sum(s.elapsed_time(e) for s, e in zip(starts, ends)), dist, "cuda")
    ms_step = total_ms / args.steps
    tokens = world * B * n_tok * args.steps
    value = tokens / (total_ms / 1e3)
    fl_step = B * flops_per_clip(cfg, n_tok)
    if head is not None:
        fl_step += B * head_flops_per_clip(synth.HEAD_SSV2, n_tok)
    peaks = _peaks()
    tflops = fl_step / (ms_step / 1e3) / 1e12

    # dominant kernel class and its roofline
    dom = max((k for k in prof if k in class_flops_per_launch(cfg, B, n_tok)), key=lambda k: prof[k][0])
    t_ms, launches = prof[dom]
    avg_ms = t_ms / max(launches, 1)
    fl = class_flops_per_launch(cfg, B, n_tok)[dom]
    achieved = fl / (avg_ms / 1e3) / 1e12
    launch_key = f"B{B} N{n_tok} D{cfg.embed_dim}"
    roof = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": peaks["bf16_sustained"],
            "unit": "TFLOP/s", "frac": achieved / peaks["bf16_sustained"],
            "traffic": _traffic_for(dom, launch_key),
            "peak_note": f"{peaks['source']} sustained bf16 (kernel timed inside a long step)",
            "avg_launch_ms": avg_ms, "flops_per_launch": fl}
    kernels = {k: {"ms_per_step": v[0] / n_prof, "launches_per_step": v[1] / n_prof} for k, v in prof.items()}
    kernels["_note"] = f"per-class CUDA-event times from {n_prof} separate profiled steps"
    # kernels per timed step (the unfold kernel inside patch_embed counted too), x the timed steps
    gpu_launches = int(round((sum(v[1] for v in prof.values()) / n_prof + 1) * args.steps))

    # end to end through the host-buffer entry point (pinned host memory)
    hclip = torch.from_numpy(clip_np).pin_memory()
    hout = torch.empty((B, n_tok, cfg.embed_dim), dtype=torch.float32).pin_memory()

    if head is not None:
        hlogits = torch.empty((B, synth.HEAD_SSV2.n_classes), dtype=torch.float32).pin_memory()

    def e2e_serial_step():
        if head is not None:   # pinned clip in, encoder + head on the device, logits out
            clip.copy_(hclip, non_blocking=True)
            step()
            hlogits.copy_(logits, non_blocking=True)
            torch.cuda.current_stream().synchronize()
        elif keep_frac is None:
            enc.encode_host(hclip, hout)
        else:   # the masked forward has no host entry point: copies around jepa_encode_masked
            clip.copy_(hclip, non_blocking=True)
            hout.copy_(step(), non_blocking=True)
            torch.cuda.current_stream().synchronize()

    def e2e_run(n, streaming):
        """Wall time per step of n steps, each copying its clip in and its
        tokens out; with streaming, one step's copies overlap its neighbours'
        encodes and the run ends when the last copy-out has landed."""
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(n):
            if streaming:
                enc.encode_host_async(hclip, hout)
            else:
                e2e_serial_step()
        if streaming:
            enc.sync()
        return max_over_ranks((time.perf_counter() - t0) / n, dist, "cuda")

    streaming = keep_frac is None and head is None
    e2e_run(2, False)
    if streaming:
        e2e_run(2, True)      # both staging slots and their graphs warm
    e2e_serial_s = e2e_run(args.e2e_steps, False)
    e2e_s = e2e_run(args.e2e_steps, True) if streaming else e2e_serial_s
    e2e_val = world * B * n_tok / e2e_s

    line = {
        "metric": metric, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,0.02) weights, uniform uint8 clips)",
        "config": {"workload": workload, "global_batch": B * world, "seq_len": n_tok,
                   "parallelism": f"replicas x{world}" if world > 1 else "none",
                   "l2": "flushed between timed steps (256 MB write outside the timed region)"},
        "clips_per_s": value / n_tok,
        "tflops": tflops, "pct_bf16_peak": {"burst": tflops / peaks["bf16_burst"],
                                            "sustained": tflops / peaks["bf16_sustained"], "source": peaks["source"]},
        "roofline": roof,
        "kernels": kernels,
        "gpu_launches": gpu_launches,
        "e2e": {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": int(hclip.numel()),
                "d2h_bytes_per_step": int(hlogits.numel() * 4) if head is not None else int(hout.numel() * 4),
                "api": "jepa_encode_host_async per step + jepa_encoder_sync at the end (pinned host buffers; "
                       "copies overlap the neighbouring steps' encodes)" if streaming else
                       ("pinned host clip -> device, jepa_encode + jepa_head_forward, device -> pinned host logits"
                        if head is not None else
                        "pinned host clip -> device, jepa_encode_masked, device -> pinned host tokens"),
                "serial_value": world * B * n_tok / e2e_serial_s,
                "serial_api": "jepa_encode_host per step (copy in, encode, copy out, synchronise)" if streaming else
                              "as api"},
        "clocks": clocks.summary(),
    }
    if args.workload == DEFAULT_WORKLOAD:
        line["context_baseline"] = {"value": 2048 / 0.0465, "unit": UNIT,
                                    "what": "pages' ggml-CUDA f16 ViT-L/16 16f 256px, batch 1, RTX 4500 Ada "
                                            "(context only)"}
    if rank == 0 and not args.no_cpu_baseline:
        if synth.tokens_per_clip(cfg) > CPU_BASELINE_MAX_TOKENS:
            line["cpu_baseline"] = {"value": None, "unit": UNIT, "kind": "oracle",
                                    "sample": "not run: one oracle block at this clip length takes minutes "
                                              "on the host cores (float64 score matrices)"}
        else:
            # a whole clip up to 2048 tokens (about 17 s for the ViT-L clip); longer clips are extrapolated
            line["cpu_baseline"] = cpu_baseline(cfg, weights, clip_np[0], whole=synth.tokens_per_clip(cfg) <= 2048,
                                                head=synth.HEAD_SSV2 if head is not None else None)
            line["cpu_baseline"].pop("seconds_per_clip", None)
    if head is not None:
        line["config"]["head"] = "SSv2 attentive-pool head: 3 pool blocks, 16 heads, 174 classes"
        head.close()
    enc.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
