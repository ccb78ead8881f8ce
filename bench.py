"""Benchmark: DiT forward tokens/s and ms/forward on GB300, with the roofline of the dominant kernel.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step = one DiT forward (every block: norm+modulate, QKV GEMM with RoPE, varlen attention,
out-projection with gated residual, FFN up with SiLU gate, FFN down with gated residual, final
norm) over the packed sequence of the workload, inputs already resident in HBM.  The denoise_loop
workload's step is one denoise step (forward + Euler step).  Prints ONE JSON line on rank 0.

--impl reference times the CPU oracle (the plain double-precision statement of the same forward)
on the host cores on a bounded sample of the workload, scaled to the same metric.
"""
from __future__ import annotations

import argparse
import hashlib
import re
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

METRIC = "DiT forward tokens/s & ms/forward on 1 GB300; % of bf16 tensor-pipe peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
SAMPLE_SECONDS = 10.0   # target CPU work of the oracle baseline sample
KINDS = ["gemm_qkv", "attention", "gemm_out", "gemm_ffn_up", "gemm_ffn_down", "norm_modulate", "other", "latent_io"]

# DRAM traffic per launch from ncu captures (dram__bytes_read.sum + dram__bytes_write.sum), keyed by
# kernel kind and workload, with the hash of the kernel source's code (source_hash: comments left
# out) the capture was taken on; the figure is reported only while that code is unchanged.
TRAFFIC = {
    # C2 block kernels, captured on the one-block slice video_audio_bf16_l1 (the same launch shapes)
    ("attention", "video_audio_bf16"): {"bytes": 409211648, "src_sha": "092678d55769e8ae"},
    ("gemm_qkv", "video_audio_bf16"): {"bytes": 884737024, "src_sha": "0bff13141c90176c"},
    ("gemm_out", "video_audio_bf16"): {"bytes": 508703488, "src_sha": "0bff13141c90176c"},
    ("gemm_ffn_up", "video_audio_bf16"): {"bytes": 939630848, "src_sha": "0bff13141c90176c"},
    ("gemm_ffn_down", "video_audio_bf16"): {"bytes": 1246642688, "src_sha": "0bff13141c90176c"},
    ("norm_modulate", "video_audio_bf16"): {"bytes": 288434480, "src_sha": "ffcb4dee053268dc"},
    # C3 block kernels, captured on the one-block slice long_doc_bf16_l1
    ("attention", "long_doc_bf16"): {"bytes": 1369731840, "src_sha": "092678d55769e8ae"},
    ("gemm_qkv", "long_doc_bf16"): {"bytes": 6321965312, "src_sha": "0bff13141c90176c"},
    ("gemm_out", "long_doc_bf16"): {"bytes": 3178683392, "src_sha": "0bff13141c90176c"},
    ("gemm_ffn_up", "long_doc_bf16"): {"bytes": 10245911040, "src_sha": "0bff13141c90176c"},
    ("gemm_ffn_down", "long_doc_bf16"): {"bytes": 8454970624, "src_sha": "0bff13141c90176c"},
    ("norm_modulate", "long_doc_bf16"): {"bytes": 1004406016, "src_sha": "ffcb4dee053268dc"},
    # fp32 path, captured on the two-block slice music_fp32_l2 (the same launch shapes)
    ("gemm_qkv", "music_fp32"): {"bytes": 51839488, "src_sha": "8f478e2ee86c66d3"},
    ("gemm_out", "music_fp32"): {"bytes": 18276352, "src_sha": "8f478e2ee86c66d3"},
    ("gemm_ffn_up", "music_fp32"): {"bytes": 135834112, "src_sha": "8f478e2ee86c66d3"},
    ("gemm_ffn_down", "music_fp32"): {"bytes": 73186560, "src_sha": "8f478e2ee86c66d3"},
    ("attention", "music_fp32"): {"bytes": 4259584, "src_sha": "8f478e2ee86c66d3"},
}


def traffic_src(kind: str, m: dict) -> str:
    """The source file of the kernels behind a kind (a TRAFFIC entry holds while its hash matches)."""
    if m["dtype"] == "fp32":
        return "fp32.cu"
    return "attention.cu" if kind == "attention" else ("gemm.cu" if kind.startswith("gemm") else "elementwise.cu")


# ------------------------------------------------------------------------------------------------
# host logic shared with the multi-process tests
# ------------------------------------------------------------------------------------------------

def rank_documents(docs: list, rank: int, world: int) -> list:
    """Weak scaling: every rank runs its own copy of the workload's documents (independent requests,
    no data-path exchange).  Returns this rank's document list."""
    assert 0 <= rank < world
    return [dict(d) for d in docs]


def rank_seed(seed: int, rank: int) -> int:
    return seed + 1000 * rank


def reduce_max_ms(ms: float, dist=None) -> float:
    """Max of a per-rank time over the process group (identity without one)."""
    if dist is None or not dist.is_initialized():
        return ms
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([ms], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def step_flops(m: dict, cu) -> dict:
    """Algorithmic FLOPs of one forward, per kernel kind (per launch x L)."""
    N = int(cu[-1])
    d, F, L = m["hidden"], m["ffn_hidden"], m["n_blocks"]
    s2 = sum(int(cu[j + 1] - cu[j]) ** 2 for j in range(len(cu) - 1))
    per = {"gemm_qkv": 2.0 * N * 3 * d * d, "attention": 4.0 * s2 * d, "gemm_out": 2.0 * N * d * d,
           "gemm_ffn_up": 2.0 * N * 2 * F * d, "gemm_ffn_down": 2.0 * N * d * F}
    return {"per_launch": per, "total": L * sum(per.values())}


def norm_bytes(m: dict, N: int) -> float:
    """Algorithmic HBM bytes of one norm+modulate launch: fp32 row in, bf16 row out, one tag byte."""
    return N * m["hidden"] * (4 + 2) + N


def fp32_alu_peak_tflops(peaks: dict, n_sms: int) -> float:
    """FP32 FMA peak derived from unit counts: SMs x 128 FP32 lanes x 2 FLOP x the maximum SM clock."""
    return n_sms * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12


def fp32_weight_bytes(m: dict) -> dict:
    """Bytes of weights one launch of each fp32 GEMM kind streams: f16 hi and lo parts, 4 per weight."""
    d, F = m["hidden"], m["ffn_hidden"]
    return {"gemm_qkv": 3 * d * d * 4, "gemm_out": d * d * 4, "gemm_ffn_up": 2 * F * d * 4,
            "gemm_ffn_down": d * F * 4}


def fp32_3xf16_peak_tflops(peaks: dict) -> float:
    """fp32-equivalent peak of the 3xF16 GEMM: the f16 tensor rate (the measured sustained bf16
    figure; kind::f16 runs f16 and bf16 at one rate) over the three f16 products it spends per fp32
    product."""
    return peaks["bf16_tflops_sustained"] / 3.0


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return FALLBACK_PEAKS, "fallback"


def source_hash(name: str) -> str:
    """sha256 prefix of a kernel source's code: comments and blank space are left out, so that a
    comment edit does not retire a traffic figure while any change to the code does."""
    with open(os.path.join(ROOT, "video_audio_gen_gb300", "csrc", name), encoding="utf-8") as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return hashlib.sha256(" ".join(text.split()).encode()).hexdigest()[:16]


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample of the workload
# ------------------------------------------------------------------------------------------------

def sample_rows(w: dict, lay: dict, seconds: float) -> int:
    """Rows of the oracle sample that take about `seconds` of CPU work (calibrated on a few rows)."""
    threads = len(os.sched_getaffinity(0))
    _, dt0, r0, _ = oracle_sample(w, lay, budget_rows=2 * threads)
    return int(min(4096, max(r0, r0 * seconds / max(dt0, 1e-3))))


def oracle_sample(w: dict, lay: dict, budget_rows: int | None = None, seconds: float = SAMPLE_SECONDS):
    """Time the oracle computing one block for a sample of R query rows of the workload: norm and
    modulate, the QKV projection and RoPE of those rows, attention of those rows over the full
    document (keys/values of the document are seeded inputs), the output projection with gated
    residual and the gated FFN.  Scaled to tokens/s of the whole forward: R rows x 1 block per
    sample; the forward is N rows x L blocks.  Returns (tokens_per_s, seconds, rows, threads)."""
    import oracle
    import synth
    m = w["model"]
    d, F, H, Dh = m["hidden"], m["ffn_hidden"], m["n_heads"], m["head_dim"]
    threads = len(os.sched_getaffinity(0))
    oracle.set_threads(threads)
    if not m["adaln"] and not m.get("vit_positions"):
        # small token counts (the music DiT): whole blocks over every token, repeated until about
        # `seconds` of CPU work, scaled by L
        sub = dict(m, n_blocks=1)
        W = synth.make_weights(dict(w, model=sub))
        x = synth.normal(w["seed"], "sample.x", (lay["n_tokens"], d), 1.0)
        cs, sn = oracle.rope_cos_sin(sub, lay["pos"])
        reps, dt = 0, 0.0
        t0 = time.perf_counter()
        while reps == 0 or dt < seconds:
            oracle.block_forward(sub, W, 0, None, x, lay, cs, sn)
            reps += 1
            dt = time.perf_counter() - t0
        oracle.set_threads(1)
        return lay["n_tokens"] * reps / (dt * m["n_blocks"]), dt, lay["n_tokens"] * reps, threads
    if budget_rows is None:
        R = sample_rows(w, lay, seconds)
        oracle.set_threads(threads)
    else:
        R = budget_rows
    cu = lay["cu_seqlens"]
    # the sample's rows: spread over the longest document
    j = int(np.argmax(np.diff(cu)))
    a, b = int(cu[j]), int(cu[j + 1])
    R = min(R, b - a)
    rows = np.linspace(a, b - 1, R).astype(np.int64)
    seed = w["seed"]
    x = synth.normal(seed, "sample.x", (R, d), 1.0)
    wq, _ = synth.normal(seed, "block0.w_qkv", (3 * d, d), w["w_std"], bf16=True)
    wo, _ = synth.normal(seed, "block0.w_o", (d, d), w["w_std"], bf16=True)
    wi, _ = synth.normal(seed, "block0.w_in", (2 * F, d), w["w_std"], bf16=True)
    wd, _ = synth.normal(seed, "block0.w_down", (d, F), w["w_std"], bf16=True)
    S = b - a
    kdoc = synth.normal(seed, "sample.k", (S, d), 1.0)
    vdoc = synth.normal(seed, "sample.v", (S, d), 1.0)
    shift = synth.normal(seed, "sample.mod", (6, d), 0.1)
    tags = np.zeros(R, dtype=np.uint8)
    sub = dict(m, n_blocks=1)
    t0 = time.perf_counter()
    y = oracle.modulate(oracle.rms_norm(x, m["norm_eps"]), tags, shift[0:1], shift[1:2])
    qkv = oracle.linear(y, wq, None)
    cs, sn = oracle.rope_cos_sin(sub, lay["pos"][rows])
    q = oracle.rope_apply(qkv[:, :d], H, Dh, m["rotary_dim"], cs, sn)
    # attention of the sampled rows over the whole document: the rows are placed first in a local
    # sequence whose keys/values are the document's
    qfull = np.zeros((S, d))
    qfull[:R] = q
    o = oracle.attention_rows(qfull, kdoc, vdoc, np.array([0, S], dtype=np.int32), H, Dh, np.arange(R))
    xo = x + shift[2] * oracle.linear(o, wo, None)
    y2 = oracle.modulate(oracle.rms_norm(xo, m["norm_eps"]), tags, shift[3:4], shift[4:5])
    hh = oracle.swiglu(oracle.linear(y2, wi, None))
    _ = xo + shift[5] * oracle.linear(hh, wd, None)
    dt = time.perf_counter() - t0
    oracle.set_threads(1)
    per_token_block = dt / R
    tokens_per_s = 1.0 / (per_token_block * m["n_blocks"])
    return tokens_per_s, dt, R, threads


# ------------------------------------------------------------------------------------------------
# GPU arm
# ------------------------------------------------------------------------------------------------

def run_gpu(args, w, dist, rank, world):
    import torch

    import synth
    from tests import gpu_util
    from video_audio_gen_gb300 import dit

    dev = torch.cuda.current_device()
    m = w["model"]
    docs = rank_documents(w["docs"], rank, world)
    lay = synth.build_layout(docs)
    if m.get("vit_positions"):  # RotaryEmbeddingND's normalised grid, from the library
        lay = dict(lay, pos=np.concatenate([dit.vit_positions(*dd["video"]) for dd in docs]))
    wr = dict(w, seed=rank_seed(w["seed"], rank))
    W = synth.make_weights(wr)
    if m.get("nvfp4"):  # the four linear maps come as NVFP4 weights; their bf16 matrices are not bound
        for b, bb in zip(W["blocks"], W["bits"]["blocks"]):
            for n in ("w_qkv", "w_o", "w_in", "w_down"):
                b[n] = bb[n] = None
    h = gpu_util.make_handle(m, lay, W)
    del W
    if m.get("nvfp4"):
        h.bind_nvfp4([{n: (torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), g) for n, (q, s, g) in b.items()}
                      for b in synth.make_nvfp4_linears(wr)])
    N, D = lay["n_tokens"], lay["n_docs"]
    dl = gpu_util.dev_layout(lay)
    x_host = synth.make_tokens(wr, lay)
    x = gpu_util.dev_f32(x_host)
    out = torch.empty_like(x)
    ws = gpu_util.workspace(h, N, D)
    t_step = synth.timestep(w) if w["t"] != "schedule" else 1.0
    loop = w["t"] == "schedule"
    sig = synth.sigmas(w.get("steps", 50))
    stream = torch.cuda.current_stream()
    latent = w.get("latent", False)
    if latent:
        # the loop state is each modality's latent tokens; per-modality shifted schedules
        widths = synth.latent_widths()
        io = synth.make_latent_io(rank_seed(w["seed"], rank) + 50, m["hidden"], widths)
        h.bind_latent_io({k: [None if a is None else gpu_util.dev_f32(a) for a in v] for k, v in io.items()})
        del io
        z_host = synth.make_latents(rank_seed(w["seed"], rank) + 50, lay, widths)
        zd = [gpu_util.dev_f32(a) for a in z_host]
        vd = [torch.empty_like(a) for a in zd]
        ws = torch.empty(h.workspace_bytes_latent(N, D), dtype=torch.uint8, device="cuda")
        sv, sa = ([dit.time_shift(float(a), sh) for a in sig] for sh in w["shifts"])

    def one_step(i):
        if latent:
            k = i % (len(sig) - 1)
            h.forward_latent(zd, dl["cu"], dl["ids"], dl["tags"], dl["pos"], [sv[k], sa[k]], vd, ws)
            dit.euler_step(zd[0], vd[0], sv[k], sv[k + 1])
            dit.euler_step(zd[1], vd[1], sa[k], sa[k + 1])
        elif loop:
            k = i % (len(sig) - 1)
            h.forward(x, dl["cu"], dl["ids"], dl["tags"], dl["pos"], float(sig[k]), out, ws)
            dit.euler_step(x, out, float(sig[k]), float(sig[k + 1]))
        else:
            h.forward(x, dl["cu"], dl["ids"], dl["tags"], dl["pos"], t_step, out, ws)

    for i in range(args.warmup):
        one_step(i)
    assert h.sync_status(ws) == 0, "device status after warm-up"
    torch.cuda.synchronize()
    launches0 = h.stats()["kernels_launched"]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev) as clk:
        # the timed region: K steps, nothing but the forward's own launches on the stream
        e0.record(stream)
        for i in range(args.steps):
            one_step(args.warmup + i)
        e1.record(stream)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        launches = h.stats()["kernels_launched"] - launches0
        # a second timed pass of K steps with a CUDA event pair around every kernel kind on the
        # launching stream: the per-kernel durations the roofline divides by
        h.set_kernel_timing(True)
        for i in range(args.steps):
            one_step(args.warmup + args.steps + i)
        torch.cuda.synchronize()
        kt = h.kernel_times()
        h.set_kernel_timing(False)
    ms_total = e0.elapsed_time(e1)
    assert h.sync_status(ws) == 0, "device status after the timed region"
    ms_total = reduce_max_ms(ms_total, dist)
    ms_step = ms_total / args.steps

    # roofline of the dominant kernel kind (largest summed time), from its CUDA-event durations
    fl = step_flops(m, lay["cu_seqlens"])
    peaks, peak_src = load_peaks()
    alu_peak = fp32_alu_peak_tflops(peaks, torch.cuda.get_device_properties(dev).multi_processor_count)
    f16x3_peak = fp32_3xf16_peak_tflops(peaks)
    kernels = {}
    for k in KINDS:
        ms, n = kt[k]
        if n == 0:
            continue
        avg = ms / n
        entry = {"launches": n, "avg_ms": round(avg, 4), "share": None}
        if k in fl["per_launch"]:
            tf = fl["per_launch"][k] / (avg * 1e-3) / 1e12
            if m["dtype"] == "fp32" and k == "attention":
                entry.update(bound="alu", achieved_tflops=round(tf, 1), frac=round(tf / alu_peak, 3))
            elif m["dtype"] == "fp32":
                entry.update(bound="tensor", achieved_tflops=round(tf, 1), frac=round(tf / f16x3_peak, 3))
                # the other bound of these small-M GEMMs: the weight stream, 4 bytes per weight
                # (the f16 hi and lo parts), read once per launch
                wb = fp32_weight_bytes(m).get(k)
                if wb:
                    gbs = wb / (avg * 1e-3) / 1e9
                    entry.update(weight_gbs=round(gbs, 1), hbm_frac=round(gbs / peaks["hbm_gbs"], 3))
            else:
                entry.update(bound="tensor", achieved_tflops=round(tf, 1),
                             frac=round(tf / peaks["bf16_tflops_sustained"], 3))
        elif k == "norm_modulate":
            gbs = norm_bytes(m, N) / (avg * 1e-3) / 1e9
            entry.update(bound="hbm", achieved_gbs=round(gbs, 1), frac=round(gbs / peaks["hbm_gbs"], 3))
        tr = TRAFFIC.get((k, args.workload))
        if tr:
            entry["traffic"] = tr["bytes"] if tr["src_sha"] == source_hash(traffic_src(k, m)) else None
        kernels[k] = entry
    tot = sum(kt[k][0] for k in KINDS)
    for k in kernels:
        kernels[k]["share"] = round(kt[k][0] / tot, 3) if tot else None
    top = max((k for k in kernels if k in fl["per_launch"]), key=lambda k: kt[k][0])
    tr = TRAFFIC.get((top, args.workload))
    traffic = tr["bytes"] if tr and tr["src_sha"] == source_hash(traffic_src(top, m)) else None
    if m["dtype"] == "fp32" and top == "attention":
        roofline = {"bound": "alu", "kernel": top, "achieved": kernels[top]["achieved_tflops"],
                    "peak": round(alu_peak, 1), "unit": "TFLOP/s", "frac": kernels[top]["frac"], "traffic": traffic,
                    "peak_source": "derived: SMs x 128 FP32 lanes x 2 FLOP x sm_max_mhz (FFMA)",
                    "algorithmic_flops_per_launch": fl["per_launch"][top]}
    elif m["dtype"] == "fp32":
        roofline = {"bound": "tensor", "kernel": top, "achieved": kernels[top]["achieved_tflops"],
                    "hbm": {"achieved_gbs": kernels[top].get("weight_gbs"), "peak_gbs": peaks["hbm_gbs"],
                            "frac": kernels[top].get("hbm_frac"),
                            "bytes_per_launch": fp32_weight_bytes(m).get(top)},
                    "peak": round(f16x3_peak, 1), "unit": "TFLOP/s", "frac": kernels[top]["frac"], "traffic": traffic,
                    "peak_source": f"3xF16: bf16_tflops_sustained of {peak_src} (the f16 rate) / 3 f16 products "
                                   "per fp32 product",
                    "algorithmic_flops_per_launch": fl["per_launch"][top]}
    else:
        roofline = {"bound": "tensor", "kernel": top, "achieved": kernels[top]["achieved_tflops"],
                    "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s", "frac": kernels[top]["frac"],
                    "traffic": traffic, "peak_source": f"bf16_tflops_sustained of {peak_src}",
                    "algorithmic_flops_per_launch": fl["per_launch"][top]}

    if args.no_e2e:
        return dict(ms_step=ms_step, tokens=N, world=world, kernels=kernels, roofline=roofline, clocks=clk.summary(),
                    launches=launches, e2e_ms=None, h2d=0, d2h=0, flops=fl["total"], docs=D, lay=lay)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    if latent:
        # end to end: each step copies the latent tokens and the layout in from pinned host memory,
        # runs the latent forward and both Euler steps, and reads the new latent tokens back
        hz = [pin(a) for a in z_host]
        hcu, hids = pin(lay["cu_seqlens"].astype(np.int32)), pin(lay["doc_ids"].astype(np.int32))
        htags, hpos = pin(lay["tags"]), pin(lay["pos"])
        hback = [torch.empty_like(a) for a in hz]

        def e2e_step(i):
            for dst, src in zip(zd, hz):
                dst.copy_(src, non_blocking=True)
            for key, src in (("cu", hcu), ("ids", hids), ("tags", htags), ("pos", hpos)):
                dl[key].copy_(src, non_blocking=True)
            one_step(i)
            for dst, src in zip(hback, zd):
                dst.copy_(src, non_blocking=True)
            torch.cuda.current_stream().synchronize()

        for i in range(2):
            e2e_step(i)
        e2e_steps = max(3, min(args.steps, 10))
        if dist is not None:
            dist.barrier()
        t0 = time.perf_counter()
        for i in range(e2e_steps):
            e2e_step(i)
        e2e_ms = reduce_max_ms((time.perf_counter() - t0) * 1e3 / e2e_steps, dist)
        h2d = sum(a.numel() * 4 for a in hz) + hcu.numel() * 4 + hids.numel() * 4 + htags.numel() + hpos.numel() * 8
        d2h = sum(a.numel() * 4 for a in hback)
        return dict(ms_step=ms_step, tokens=N, world=world, kernels=kernels, roofline=roofline, clocks=clk.summary(),
                    launches=launches, e2e_ms=e2e_ms, h2d=h2d, d2h=d2h, flops=fl["total"], docs=D, lay=lay)
    # end to end through the C ABI from pinned host buffers (copies inside the timed region)
    hx, hcu = pin(x_host), pin(lay["cu_seqlens"].astype(np.int32))
    hids, htags, hpos = pin(lay["doc_ids"].astype(np.int32)), pin(lay["tags"]), pin(lay["pos"])
    hout = torch.empty(x_host.shape, dtype=torch.float32).pin_memory()
    wsh = gpu_util.workspace(h, N, D, host=True)
    for _ in range(2):
        h.forward_host(hx, hcu, hids, htags, hpos, t_step, hout, wsh)
    e2e_steps = max(3, min(args.steps, 10))
    if dist is not None:
        dist.barrier()
    with ClockSampler(dev) as eclk:  # the e2e leg's own clocks: it runs after the timed passes
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            h.forward_host(hx, hcu, hids, htags, hpos, t_step, hout, wsh)
        e2e_ms = reduce_max_ms((time.perf_counter() - t0) * 1e3 / e2e_steps, dist)
    h2d = hx.numel() * 4 + hcu.numel() * 4 + hids.numel() * 4 + htags.numel() + hpos.numel() * 8
    d2h = hout.numel() * 4
    return dict(ms_step=ms_step, tokens=N, world=world, kernels=kernels, roofline=roofline, clocks=clk.summary(),
                launches=launches, e2e_ms=e2e_ms, h2d=h2d, d2h=d2h, flops=fl["total"], docs=D, lay=lay,
                e2e_clocks=eclk.summary())


def run_loop_figures(args, dist, rank, world):
    """The 50-step denoise loop on the video+audio model (requests of 17,408 and 9,216 tokens packed in
    one sequence), measured beside the default workload's forward: ms per step (forward + Euler step,
    inputs resident) over one whole 50-step loop, and the loop end to end, from the initial noise in
    pinned host memory to the final x read back (the copies inside the timed region)."""
    import torch

    import synth
    from tests import gpu_util
    from video_audio_gen_gb300 import dit

    w = synth.WORKLOADS["denoise_loop"]
    m = w["model"]
    lay = synth.build_layout(rank_documents(w["docs"], rank, world))
    wr = dict(w, seed=rank_seed(w["seed"], rank))
    W = synth.make_weights(wr)
    if m.get("nvfp4"):  # the four linear maps come as NVFP4 weights; their bf16 matrices are not bound
        for b, bb in zip(W["blocks"], W["bits"]["blocks"]):
            for n in ("w_qkv", "w_o", "w_in", "w_down"):
                b[n] = bb[n] = None
    h = gpu_util.make_handle(m, lay, W)
    del W
    if m.get("nvfp4"):
        h.bind_nvfp4([{n: (torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), g) for n, (q, s, g) in b.items()}
                      for b in synth.make_nvfp4_linears(wr)])
    N, D = lay["n_tokens"], lay["n_docs"]
    dl = gpu_util.dev_layout(lay)
    x_host = synth.make_tokens(wr, lay)
    x0 = gpu_util.dev_f32(x_host)
    x = torch.empty_like(x0)
    v = torch.empty_like(x0)
    ws = gpu_util.workspace(h, N, D)
    sig = [float(a) for a in synth.sigmas(w["steps"])]
    steps = len(sig) - 1
    stream = torch.cuda.current_stream()

    def loop():
        for i in range(steps):
            h.forward(x, dl["cu"], dl["ids"], dl["tags"], dl["pos"], sig[i], v, ws)
            dit.euler_step(x, v, sig[i], sig[i + 1])

    x.copy_(x0)
    for i in range(args.warmup):
        h.forward(x, dl["cu"], dl["ids"], dl["tags"], dl["pos"], sig[i], v, ws)
    x.copy_(x0)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    loop()
    e1.record(stream)
    torch.cuda.synchronize()
    loop_ms = reduce_max_ms(e0.elapsed_time(e1), dist)
    assert h.sync_status(ws) == 0, "device status after the timed loop"
    hx = torch.from_numpy(np.ascontiguousarray(x_host)).pin_memory()
    hout = torch.empty(x_host.shape, dtype=torch.float32).pin_memory()
    if dist is not None:
        dist.barrier()
    t0 = time.perf_counter()
    x.copy_(hx, non_blocking=True)
    loop()
    hout.copy_(x, non_blocking=True)
    stream.synchronize()
    e2e_ms = reduce_max_ms((time.perf_counter() - t0) * 1e3, dist)
    assert h.sync_status(ws) == 0, "device status after the end-to-end loop"
    h.close()
    return {"workload": f"denoise_loop: the {m['n_blocks']}-block video+audio model, {N} tokens in {D} requests "
                        f"({', '.join(synth_doc(d) for d in w['docs'])}), {steps} Euler steps, sigmas 1 -> 0",
            "steps": steps, "ms_per_step": round(loop_ms / steps, 3), "loop_ms": round(loop_ms, 1),
            "tokens_per_s": round(N * world / (loop_ms / steps * 1e-3), 1),
            "e2e_loop_ms": round(e2e_ms, 1), "h2d_bytes": int(hx.numel() * 4), "d2h_bytes": int(hout.numel() * 4)}


def run_nvfp4_gemm(args):
    """The four linear maps of one block of the video+audio model at its full 17,408-token sequence,
    with NVFP4 weights (E2M1 codes, an E4M3 scale per 16 along K, fp32 global scale; f16
    activations) and, on the same shapes, with bf16 weights through the bf16 engine.  A step is one
    pass over the four NVFP4 GEMMs; the bf16 GEMMs run in a second pass for the comparison."""
    import torch

    import synth
    from video_audio_gen_gb300 import dit

    dev = torch.cuda.current_device()
    m = synth.WORKLOADS["video_audio_bf16"]["model"]
    d, F = m["hidden"], m["ffn_hidden"]
    M = synth.build_layout(synth.WORKLOADS["video_audio_bf16"]["docs"])["n_tokens"]
    shapes = {"gemm_qkv": (3 * d, d), "gemm_out": (d, d), "gemm_ffn_up": (2 * F, d), "gemm_ffn_down": (d, F)}
    ops = {}
    for k, (N, K) in shapes.items():
        q, sc, g = synth.make_nvfp4(5, f"bench.{k}", N, K)
        packed = torch.empty(dit.nvfp4_packed_bytes(N, K), dtype=torch.uint8, device="cuda")
        dit.pack_nvfp4(torch.from_numpy(q).cuda(), torch.from_numpy(sc).cuda(), packed)
        a16 = torch.from_numpy(synth.normal(5, f"bench.a.{k}", (M, K), 1.0).astype(np.float16)).cuda()
        wbf = torch.from_numpy(synth.normal(5, f"bench.w.{k}", (N, K), 0.02)).cuda().bfloat16()
        out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        ops[k] = dict(N=N, K=K, packed=packed, g=g, a16=a16, abf=a16.bfloat16(), wbf=wbf, out=out)
    stream = torch.cuda.current_stream()

    def timed(fn_for):
        ev = {k: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for k in ops}
        tot = {k: 0.0 for k in ops}
        for _ in range(args.steps):
            for k, o in ops.items():
                ev[k][0].record(stream)
                fn_for(o)
                ev[k][1].record(stream)
            torch.cuda.synchronize()
            for k in ops:
                tot[k] += ev[k][0].elapsed_time(ev[k][1])
        return {k: v / args.steps for k, v in tot.items()}

    nv = lambda o: dit.gemm_nvfp4(o["a16"], o["packed"], o["g"], None, o["N"], o["out"], 0)
    bf = lambda o: dit.gemm(o["abf"], o["wbf"], None, o["out"], 0)
    for _ in range(args.warmup):
        for o in ops.values():
            nv(o)
            bf(o)
    torch.cuda.synchronize()
    with ClockSampler(dev) as clk:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            for o in ops.values():
                nv(o)
        e1.record(stream)
        torch.cuda.synchronize()
        t_nv = timed(nv)
        t_bf = timed(bf)
    ms_step = e0.elapsed_time(e1) / args.steps
    flops = {k: 2.0 * M * o["N"] * o["K"] for k, o in ops.items()}
    peaks, peak_src = load_peaks()
    peak = peaks["bf16_tflops_sustained"]  # f16 and bf16 share the tensor rate
    kernels = {}
    for k in ops:
        tf_nv = flops[k] / (t_nv[k] * 1e-3) / 1e12
        tf_bf = flops[k] / (t_bf[k] * 1e-3) / 1e12
        kernels[k] = {"M": M, "N": ops[k]["N"], "K": ops[k]["K"], "nvfp4_ms": round(t_nv[k], 4),
                      "nvfp4_tflops": round(tf_nv, 1), "frac": round(tf_nv / peak, 3),
                      "bf16_ms": round(t_bf[k], 4), "bf16_tflops": round(tf_bf, 1),
                      "weight_bytes_nvfp4": ops[k]["N"] * ops[k]["K"] * 9 // 16,
                      "weight_bytes_bf16": ops[k]["N"] * ops[k]["K"] * 2}
    top = max(kernels, key=lambda k: t_nv[k])
    value = sum(flops.values()) / (ms_step * 1e-3) / 1e12
    line = {"metric": "NVFP4-weight GEMM TFLOP/s on the four linear maps of one video+audio block (1 GB300)",
            "value": round(value, 1), "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f16 x nvfp4", "data": "synthetic (random valid NVFP4 codes, N(0, 1) f16 activations)",
            "config": {"workload": f"nvfp4_gemm: M={M} tokens; QKV {3 * d}x{d}, out {d}x{d}, FFN up {2 * F}x{d}, "
                                   f"FFN down {d}x{F}", "l2": "activations and outputs (>400 MB) larger than L2; "
                                                            "weights L2-resident as in the forward"},
            "roofline": {"bound": "tensor", "kernel": f"{top} (nvfp4)", "achieved": kernels[top]["nvfp4_tflops"],
                         "peak": peak, "unit": "TFLOP/s", "frac": kernels[top]["frac"], "traffic": None,
                         "peak_source": f"bf16_tflops_sustained of {peak_src} (f16 runs at the bf16 rate)",
                         "algorithmic_flops_per_launch": flops[top]},
            "kernels": kernels, "gpu_launches": args.steps * len(ops), "clocks": clk.summary()}
    print(json.dumps(line))


def run_nvfp4_reference(args):
    """The oracle's NVFP4 linear (double precision) on a bounded sample of rows of the QKV shape,
    scaled to TFLOP/s."""
    import oracle
    import synth
    d = synth.WORKLOADS["video_audio_bf16"]["model"]["hidden"]
    N, K = 3 * d, d
    q, sc, g = synth.make_nvfp4(5, "bench.gemm_qkv", N, K)
    threads = os.cpu_count() or 1
    oracle.set_threads(threads)
    vals = []
    R = 4
    for _ in range(args.steps):
        a = synth.normal(5, "bench.a.sample", (R, K), 1.0).astype(np.float16).astype(np.float64)
        t0 = time.perf_counter()
        oracle.nvfp4_linear(a, q, sc, g)
        dt = time.perf_counter() - t0
        vals.append(2.0 * R * N * K / dt / 1e12)
    oracle.set_threads(1)
    v = statistics.median(vals)
    line = {"impl": "reference", "metric": "NVFP4-weight GEMM TFLOP/s on the four linear maps of one video+audio "
            "block (1 GB300)", "value": round(v, 6), "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"nvfp4_gemm: the oracle's NVFP4 linear on {R} rows of the {N}x{K} QKV shape"},
            "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": f"{R} rows x {N} outputs x {K} per step, dequantisation included"},
            "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


L2_BYTES = 129 * 1024 * 1024


def l2_note(m: dict, lay: dict) -> str:
    """How the timed steps relate to the 129 MB L2: the bytes one forward streams (weights once,
    the fp32 residual and the bf16 activations of every block) against the cache size."""
    d, F, L, N = m["hidden"], m["ffn_hidden"], m["n_blocks"], lay["n_tokens"]
    wb = 4 if m["dtype"] == "fp32" else 2
    weights = L * (4 * d * d + 3 * d * F) * wb
    acts = L * N * (4 * d * 4 + 2 * F * 2)
    total = weights + acts
    if total > L2_BYTES:
        return f"inputs larger than L2: about {total / 1e9:.2f} GB of weights and activations stream each step"
    return f"working set about {total / 1e6:.0f} MB, within L2 (no flush): a parity-size case, not a bench workload"


def workload_config(name, w, lay, extra=None):
    m = w["model"]
    docs = ", ".join(f"{synth_doc(d)}" for d in w["docs"])
    cond = ("rmsnorm + modality AdaLN" if m["adaln"] else
            f"{m['norm']}norm, ungated residuals, 1x1 convs {m['io_channels']}->{m['hidden']}->{m['io_channels']}")
    if m.get("vit_positions"):
        cond = (f"RMSNorm gains, interleaved qkv, per-head q/k RMS norm, per-channel residual scales, "
                f"RotaryEmbeddingND (base {m['rope_base']:g}, {m['rotary_dim']} of {m['head_dim']} dims), final LayerNorm")
    c = {"workload": f"{name}: {m['n_blocks']} blocks, d={m['hidden']}, {m['n_heads']}x{m['head_dim']} heads, "
                     f"FFN {m['ffn_hidden']} (value*silu(gate)), {cond}; "
                     f"{lay['n_tokens']} packed tokens in {lay['n_docs']} documents ({docs})",
         "tokens": int(lay["n_tokens"]), "documents": int(lay["n_docs"]),
         "cu_seqlens": [int(v) for v in lay["cu_seqlens"]],
         "l2": l2_note(m, lay)}
    if w.get("latent"):
        import synth
        widths = synth.latent_widths()
        c["latent_io"] = (f"fp32 patch projections and output heads per modality: video {widths[0]} features "
                          f"({synth.VIDEO_LATENT['channels']} channels, patch {synth.VIDEO_LATENT['patch']}), "
                          f"audio {widths[1]}; sigma shifts video {w['shifts'][0]:g}, audio {w['shifts'][1]:g}")
    if extra:
        c.update(extra)
    return c


def synth_doc(d):
    if "frames" in d:
        return f"{d['frames']} frames"
    t, hh, ww = d.get("video", (0, 0, 0))
    return f"video {t}x{hh}x{ww}" + (f" + {d['audio']} audio" if d.get("audio") else "")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="long_doc_bf16",
                    choices=["video_audio_bf16", "long_doc_bf16", "denoise_loop", "t2va_loop", "music_fp32",
                             "video_audio_bf16_l1", "long_doc_bf16_l1", "video_audio_nvfp4", "tiny", "ragged", "music_small", "music_fp32_l2", "nvfp4_gemm", "vit3d_decoder",
                             "vit3d_small"])
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-loop", action="store_true",
                    help="skip the denoise-loop figures that the default workload's line carries")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    import synth
    if args.workload == "nvfp4_gemm":
        if int(os.environ.get("RANK", "0")) == 0:
            (run_nvfp4_reference if args.impl == "reference" else run_nvfp4_gemm)(args)
        return
    w = synth.WORKLOADS[args.workload]
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    is_loop = w["t"] == "schedule"
    metric = METRIC if not is_loop else "DiT denoise step ms/step (forward + Euler) and tokens/s on 1 GB300"
    if w.get("latent"):
        metric = ("DiT t2va denoise step ms/step (latent forward: patch projections, blocks, heads; Euler per "
                  "modality) and tokens/s on 1 GB300")
    if w["model"].get("vit_positions"):
        metric = "video-VAE ViT3D decoder forward tokens/s & ms/forward on 1 GB300; % of bf16 tensor-pipe peak"

    if args.impl == "reference":
        if rank != 0:
            return
        lay = synth.build_layout(w["docs"])
        if w["model"].get("vit_positions"):
            import oracle
            lay = dict(lay, pos=np.concatenate([oracle.vit_positions(*dd["video"]) for dd in w["docs"]]))
        vals, secs = [], []
        # each step a bounded sample: the whole run stays within a couple of minutes
        per_step = max(1.0, min(SAMPLE_SECONDS, 120.0 / max(1, args.steps)))
        rows = sample_rows(w, lay, per_step) if (w["model"]["adaln"] or w["model"].get("vit_positions")) else None
        for _ in range(args.steps):
            tps, dt, R, threads = oracle_sample(w, lay, budget_rows=rows, seconds=per_step)
            vals.append(tps)
            secs.append(dt)
        tps = statistics.median(vals)
        ms_step = lay["n_tokens"] / tps * 1e3
        sample = (f"{R} query rows x 1 block of the workload per step ({args.steps} steps, median), "
                  f"scaled by N={lay['n_tokens']} rows x L={w['model']['n_blocks']} blocks")
        if not w["model"]["adaln"] and not w["model"].get("vit_positions"):
            sample = (f"whole blocks over {R} tokens per step ({args.steps} steps, median), "
                      f"scaled by L={w['model']['n_blocks']} blocks")
        line = {"impl": "reference", "metric": metric, "value": round(tps, 4), "unit": "tokens/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 1),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": workload_config(args.workload, w, lay),
                "cpu_baseline": {"value": round(tps, 4), "unit": "tokens/s", "cores": threads, "kind": "oracle",
                                 "sample": sample},
                "e2e": {"value": round(tps, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    dist = None
    if world > 1:
        import torch.distributed as tdist
        local = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl")
        dist = tdist
    r = run_gpu(args, w, dist, rank, world)
    m_dtype = "f32" if w["model"]["dtype"] == "fp32" else "bf16"
    if rank == 0:
        tokens_total = r["tokens"] * world
        value = tokens_total / (r["ms_step"] * 1e-3)
        tflops = r["flops"] / (r["ms_step"] * 1e-3) / 1e12
        peaks, peak_src = load_peaks()
        line = {"metric": metric, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(r["ms_step"], 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": m_dtype,
                "data": (f"synthetic (seeded N(0, 0.02) {'fp32' if m_dtype == 'f32' else 'bf16'} weights, "
                         "N(0, 1) fp32 tokens)"),
                "config": workload_config(args.workload, w, r["lay"], {
                    "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                    "forward_tflop": round(r["flops"] / 1e12, 3),
                    "step_tflops": round(tflops, 1),
                    "step_frac_of_bf16_peak": round(tflops / peaks["bf16_tflops_sustained"], 3),
                    "kernel_timing": "per-kernel CUDA events in a second timed pass of the same K steps, "
                                     "so value carries no event overhead"}),
                "roofline": r["roofline"], "kernels": r["kernels"],
                "e2e": (None if r["e2e_ms"] is None else
                        {"value": round(tokens_total / (r["e2e_ms"] * 1e-3), 1), "unit": "tokens/s",
                         "ms_per_step": round(r["e2e_ms"], 3), "h2d_bytes_per_step": int(r["h2d"]),
                         "d2h_bytes_per_step": int(r["d2h"]), "clocks": r.get("e2e_clocks")}),
                "gpu_launches": int(r["launches"]), "clocks": r["clocks"]}
        if m_dtype == "f32":
            # the fp32 path's own reference point: the FP32 FFMA rate of the device (the forward runs
            # its contractions as three f16 tensor-core products per fp32 product instead)
            import torch
            ffma = fp32_alu_peak_tflops(peaks, torch.cuda.get_device_properties(torch.cuda.current_device())
                                        .multi_processor_count)
            line["config"]["step_frac_of_fp32_ffma_peak"] = round(tflops / ffma, 3)
            line["config"]["fp32_ffma_peak_tflops"] = round(ffma, 1)
        if not args.no_cpu_baseline:
            lay_cpu = r["lay"]
            if w["model"].get("vit_positions"):  # the oracle's own positions
                import oracle
                lay_cpu = dict(lay_cpu, pos=np.concatenate([oracle.vit_positions(*dd["video"]) for dd in w["docs"]]))
            tps, dt, R, threads = oracle_sample(w, lay_cpu)
            whole = not w["model"]["adaln"] and not w["model"].get("vit_positions")
            what = f"whole blocks over {R} tokens in all" if whole else f"{R} query rows x 1 block"
            line["cpu_baseline"] = {"value": round(tps, 4), "unit": "tokens/s", "cores": threads, "kind": "oracle",
                                    "sample": f"{what} ({dt:.1f} s on {threads} threads), "
                                              f"scaled by N={r['tokens']} rows x L={w['model']['n_blocks']} blocks"}
    loop = None
    if args.workload == "long_doc_bf16" and not args.no_loop:
        loop = run_loop_figures(args, dist, rank, world)
    if rank == 0:
        if loop is not None:
            line["denoise_loop"] = loop
        print(json.dumps(line))
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
