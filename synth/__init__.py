"""Seeded synthetic inputs: the one module both the CUDA path and the oracle are fed from.

It holds the workload recipes (model shapes, document mixes, seeds) and the generators that turn
them into arrays.  It holds none of the DiT's arithmetic: no norm, projection, rotary, attention or
sampler step lives here.  The packed-layout builder and the fp64 position grid are *inputs* of the
forward (the caller builds them; the forward only reads them), so they live here too, written from
the page "feat(minimax-h3): port the MiniMax-H3 omni-modal video+audio DiT", section "Correctness
gates": the grid is numpy.linspace(endpoint=False) evaluated in the order i*step + start.

Random numbers come from ``synth_gen.c`` (FNV-1a keyed, counter-based splitmix64 + Box-Muller).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ``libsynth.so`` next to its source with the host C compiler."""
    src = os.path.join(_HERE, "synth_gen.c")
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", src, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.synth_fnv1a64.restype = ctypes.c_uint64
            lib.synth_fnv1a64.argtypes = [ctypes.c_char_p]
            lib.synth_normal.restype = None
            lib.synth_normal.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_double,
                                         ctypes.c_void_p, ctypes.c_void_p]
            lib.synth_uniform.restype = None
            lib.synth_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_double,
                                          ctypes.c_double, ctypes.c_void_p]
            _lib = lib
    return _lib


def key(seed: int, name: str) -> int:
    return int(_load().synth_fnv1a64(f"seed={seed}/{name}".encode()))


def normal(seed: int, name: str, shape, std: float = 1.0, bf16: bool = False):
    """N(0, std^2) as float32; with ``bf16=True`` the values are rounded to bf16 (RNE) and the
    function returns ``(float32 values, uint16 bf16 bits)`` holding the same numbers."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(shape, dtype=np.float32)
    bits = np.empty(shape, dtype=np.uint16) if bf16 else None
    if n:
        _load().synth_normal(key(seed, name), n, float(std), out.ctypes.data,
                             bits.ctypes.data if bf16 else None)
    return (out, bits) if bf16 else out


def uniform(seed: int, name: str, n: int, lo: float = 0.0, hi: float = 1.0) -> np.ndarray:
    out = np.empty((n,), dtype=np.float64)
    if n:
        _load().synth_uniform(key(seed, name), n, float(lo), float(hi), out.ctypes.data)
    return out


# ----------------------------------------------------------------------------------------------
# Packed layout and fp64 position grid (inputs of the forward)
# ----------------------------------------------------------------------------------------------

def grid_axis(start: float, stop: float, n: int) -> np.ndarray:
    """linspace(start, stop, n, endpoint=False) evaluated as i*step + start, step = (stop-start)/n."""
    step = (float(stop) - float(start)) / n
    out = np.empty((n,), dtype=np.float64)
    for i in range(n):
        out[i] = float(i) * step + float(start)
    return out


def doc_tokens(doc: dict) -> int:
    if "frames" in doc:
        return int(doc["frames"])
    t, h, w = doc.get("video", (0, 0, 0))
    return t * h * w + int(doc.get("audio", 0))


def build_layout(docs) -> dict:
    """Pack documents into one varlen sequence.

    Within a document: video tokens first, flattened (t, h, w) with w fastest, then audio tokens.
    Tags: 0 = video, 1 = audio.  ``frames`` documents (the music DiT) are one-axis sequences with
    tag 0 whose position is the frame index.  Every document's positions start at 0.
    """
    sizes = [doc_tokens(d) for d in docs]
    n = int(sum(sizes))
    cu = np.zeros((len(docs) + 1,), dtype=np.int32)
    cu[1:] = np.cumsum(sizes)
    doc_ids = np.empty((n,), dtype=np.int32)
    tags = np.zeros((n,), dtype=np.uint8)
    pos = np.zeros((n, 3), dtype=np.float64)
    for j, d in enumerate(docs):
        a = int(cu[j])
        doc_ids[a:a + sizes[j]] = j
        if "frames" in d:
            pos[a:a + sizes[j], 0] = grid_axis(0.0, d["frames"], d["frames"])
            continue
        T, H, W = d.get("video", (0, 0, 0))
        nv = T * H * W
        if nv:
            gt, gh, gw = grid_axis(0.0, T, T), grid_axis(0.0, H, H), grid_axis(0.0, W, W)
            r = a
            for it in range(T):
                for ih in range(H):
                    for iw in range(W):
                        pos[r] = (gt[it], gh[ih], gw[iw])
                        r += 1
        na = int(d.get("audio", 0))
        if na:
            span = T if T > 0 else na
            pos[a + nv:a + nv + na, 0] = grid_axis(0.0, span, na)
            tags[a + nv:a + nv + na] = 1
    return dict(cu_seqlens=cu, doc_ids=doc_ids, tags=tags, pos=pos, n_tokens=n, n_docs=len(docs))


# ----------------------------------------------------------------------------------------------
# Workload recipes
# ----------------------------------------------------------------------------------------------

def _model(**kw):
    m = dict(n_blocks=2, hidden=256, n_heads=4, head_dim=64, ffn_hidden=1024, norm="rms", norm_eps=1e-6,
             adaln=True, n_mod=2, t_dim=256, rope_axes=3, rope_dims=(16, 24, 24), rotary_dim=64,
             rope_base=10000.0, io_channels=0, dtype="bf16")
    m.update(kw)
    return m


# The video-VAE decoder's block: no AdaLN, RMS gains, per-head q/k RMS norm, interleaved qkv,
# per-channel residual scales, final LayerNorm; READINGS: ffn_hidden 5632 (the usual 8/3 d rounded
# to 256; the pages give none), norm eps 1e-6, 48 rotary dims split 16/16/16 over (t, h, w).
VIT_MODEL = _model(n_blocks=36, hidden=2048, n_heads=32, head_dim=64, ffn_hidden=5632, adaln=False, n_mod=1,
                   rope_dims=(16, 16, 16), rotary_dim=48, rope_base=100.0, qk_norm=True, qkv_interleaved=True,
                   final_norm="ln", res_scale=True, norm_affine=True, vit_positions=True)

C2_MODEL = _model(n_blocks=8, hidden=3072, n_heads=24, head_dim=128, ffn_hidden=8192,
                  rope_dims=(32, 48, 48), rotary_dim=128)

WORKLOADS = {
    # Tiny DiT: 2 documents, 96 + (128 video + 32 audio) tokens.
    "tiny": dict(model=_model(), seed=0, docs=[dict(video=(2, 6, 8)), dict(video=(2, 8, 8), audio=32)],
                 t=0.5, w_std=0.02, bias_std=0.0, x_std=1.0),
    # Music-DiT shape: fp32, LayerNorm, partial rotary on 64 of 128 dims, 1x1 pre/post convs
    # 128 -> 2048 -> 128, two CFG branches of 86 frames each.
    "music_fp32": dict(model=_model(n_blocks=24, hidden=2048, n_heads=16, head_dim=128, ffn_hidden=8192,
                                    norm="ln", norm_eps=1e-5, adaln=False, n_mod=1, rope_axes=1,
                                    rope_dims=(64, 0, 0), rotary_dim=64, io_channels=128, dtype="fp32"),
                       seed=1, docs=[dict(frames=86), dict(frames=86)], t=0.0, w_std=0.02, bias_std=0.02,
                       x_std=1.0),
    # Video+audio DiT, bf16: 2 x (8192 video + 512 audio) = 17,408 tokens.
    "video_audio_bf16": dict(model=C2_MODEL, seed=2,
                             docs=[dict(video=(8, 32, 32), audio=512), dict(video=(8, 32, 32), audio=512)],
                             t="uniform", w_std=0.02, bias_std=0.0, x_std=1.0),
    # Long single document: 32,768 video + 1,024 audio = 33,792 tokens.
    "long_doc_bf16": dict(model=_model(n_blocks=4, hidden=5120, n_heads=40, head_dim=128, ffn_hidden=13824,
                                       rope_dims=(32, 48, 48), rotary_dim=128),
                          seed=3, docs=[dict(video=(16, 32, 64), audio=1024)], t="uniform", w_std=0.02,
                          bias_std=0.0, x_std=1.0),
    # 50-step Euler loop on the video+audio model: requests of 17,408 and 9,216 tokens.
    "denoise_loop": dict(model=C2_MODEL, seed=4,
                         docs=[dict(video=(8, 32, 64), audio=1024), dict(video=(4, 32, 64), audio=1024)],
                         t="schedule", steps=50, w_std=0.02, bias_std=0.0, x_std=1.0),
    # The same two requests as the joint loop in latent token space: per-modality fp32 patch
    # projections and output heads around the block stack, video sigmas shifted by 12 and audio by 3.
    "t2va_loop": dict(model=C2_MODEL, seed=4,
                      docs=[dict(video=(8, 32, 64), audio=1024), dict(video=(4, 32, 64), audio=1024)],
                      t="schedule", steps=50, latent=True, shifts=(12.0, 3.0), w_std=0.02, bias_std=0.0,
                      x_std=1.0),
    # The video-VAE ViT3D decoder stack ([H3] "Update: video-VAE ViT3D decoder complete": 36 blocks,
    # 32 x 64 heads, rms_norm affine, q/k rms_norm without affine, gated SiLU, rope_theta 100,
    # rope_dim_ratio 0.75) on one 8 x 32 x 32 latent grid; positions are RotaryEmbeddingND's.
    "vit3d_decoder": dict(model=VIT_MODEL, seed=6, docs=[dict(video=(8, 32, 32))], t=0.0, w_std=0.02,
                          bias_std=0.02, x_std=1.0, affine_std=0.1),
    # The same block at parity size: two grids (one ragged), 2 blocks of width 256.
    "vit3d_small": dict(model=dict(VIT_MODEL, n_blocks=2, hidden=256, n_heads=4, ffn_hidden=768), seed=7,
                        docs=[dict(video=(2, 8, 16)), dict(video=(1, 6, 10))], t=0.0, w_std=0.02,
                        bias_std=0.02, x_std=1.0, affine_std=0.1),
    # One block of the video+audio model on its full 17,408-token sequence: every kernel launch has
    # exactly the full workload's shape, with a few GB on the device (profiling captures).
    "video_audio_bf16_l1": dict(model=dict(C2_MODEL, n_blocks=1), seed=2,
                                docs=[dict(video=(8, 32, 32), audio=512), dict(video=(8, 32, 32), audio=512)],
                                t="uniform", w_std=0.02, bias_std=0.0, x_std=1.0),
    # The video+audio model with NVFP4 weights in its four linear maps per block ([H3] "What this
    # push adds": the NVFP4 checkpoint), everything else as in video_audio_bf16.
    "video_audio_nvfp4": dict(model=dict(C2_MODEL, nvfp4=True), seed=2,
                              docs=[dict(video=(8, 32, 32), audio=512), dict(video=(8, 32, 32), audio=512)],
                              t="uniform", w_std=0.02, bias_std=0.0, x_std=1.0),
    # One block of the long-document model on its full 33,792-token sequence (profiling captures of
    # the same launch shapes with a few GB on the device).
    "long_doc_bf16_l1": dict(model=_model(n_blocks=1, hidden=5120, n_heads=40, head_dim=128, ffn_hidden=13824,
                                          rope_dims=(32, 48, 48), rotary_dim=128),
                             seed=3, docs=[dict(video=(16, 32, 64), audio=1024)], t="uniform", w_std=0.02,
                             bias_std=0.0, x_std=1.0),
    # Parity cases that span several 128-row tiles with ragged document ends, a 1-token document and
    # non-zero biases (the oracle finishes them in seconds).
    "ragged": dict(model=_model(n_blocks=2, hidden=512, n_heads=4, head_dim=128, ffn_hidden=1536,
                                rope_dims=(32, 48, 48), rotary_dim=128),
                   seed=11, docs=[dict(video=(2, 5, 7), audio=13), dict(video=(3, 8, 9), audio=41),
                                  dict(video=(1, 1, 1)), dict(video=(4, 12, 10), audio=37)],
                   t=0.37, w_std=0.02, bias_std=0.02, x_std=1.0),
    # Parity case for the tile schedule and the key masking: 13 documents whose lengths sit on and
    # around the 128-token tile (1, 2, 127, 128, 129, 255, 256, 257, 300, ...), none starting on a
    # tile boundary after the first, head_dim 64, non-zero biases.
    "many_docs": dict(model=_model(), seed=13,
                      docs=[dict(video=(1, 1, 1)), dict(video=(2, 8, 8)), dict(video=(2, 8, 8), audio=1),
                            dict(video=(4, 8, 8)), dict(video=(1, 9, 14), audio=1), dict(video=(1, 1, 2)),
                            dict(video=(3, 5, 17)), dict(video=(1, 8, 8)), dict(video=(2, 10, 15)),
                            dict(video=(1, 1, 1), audio=5), dict(video=(5, 5, 5), audio=3),
                            dict(video=(1, 3, 3)), dict(video=(2, 16, 8), audio=1)],
                      t=0.61, w_std=0.02, bias_std=0.02, x_std=1.0),
    # Two blocks of the music model on its full 172-frame batch: every launch has the full workload's
    # shape, with about 0.6 GB on the device (profiling captures).
    "music_fp32_l2": dict(model=_model(n_blocks=2, hidden=2048, n_heads=16, head_dim=128, ffn_hidden=8192,
                                       norm="ln", norm_eps=1e-5, adaln=False, n_mod=1, rope_axes=1,
                                       rope_dims=(64, 0, 0), rotary_dim=64, io_channels=128, dtype="fp32"),
                          seed=1, docs=[dict(frames=86), dict(frames=86)], t=0.0, w_std=0.02, bias_std=0.02,
                          x_std=1.0),
    "music_small": dict(model=_model(n_blocks=2, hidden=256, n_heads=2, head_dim=128, ffn_hidden=1024,
                                     norm="ln", norm_eps=1e-5, adaln=False, n_mod=1, rope_axes=1,
                                     rope_dims=(64, 0, 0), rotary_dim=64, io_channels=128, dtype="fp32"),
                        seed=12, docs=[dict(frames=37), dict(frames=37)], t=0.0, w_std=0.02,
                        bias_std=0.02, x_std=1.0),
}


def timestep(w: dict) -> float:
    t = w["t"]
    if t == "uniform":
        return float(np.float32(uniform(w["seed"], "timestep", 1)[0]))
    if t == "schedule":
        return 1.0
    return float(t)


def sigmas(steps: int) -> np.ndarray:
    """Linear sigmas from 1.0 to 0.0 (steps + 1 values), fp32 of the double value 1 - i/steps."""
    return np.array([np.float32(1.0 - i / steps) for i in range(steps + 1)], dtype=np.float32)


def weight_shapes(m: dict) -> dict:
    """Per-block and global weight tensor shapes (row-major [out, in] for every linear map)."""
    d, F, L = m["hidden"], m["ffn_hidden"], m["n_blocks"]
    blk = dict(w_qkv=(3 * d, d), b_qkv=(3 * d,), w_o=(d, d), b_o=(d,), w_in=(2 * F, d), b_in=(2 * F,),
               w_down=(d, F), b_down=(d,))
    glob = {}
    if m["adaln"]:
        blk.update(w_ada=(m["n_mod"] * 6 * d, m["t_dim"]), b_ada=(m["n_mod"] * 6 * d,))
        glob.update(w_ada_final=(m["n_mod"] * 2 * d, m["t_dim"]), b_ada_final=(m["n_mod"] * 2 * d,))
    if m["norm"] == "ln":
        blk.update(ln1_g=(d,), ln1_b=(d,), ln2_g=(d,), ln2_b=(d,))
        glob.update(lnf_g=(d,), lnf_b=(d,))
    if m.get("norm_affine"):  # RMSNorm with a per-channel gain
        blk.update(ln1_g=(d,), ln2_g=(d,))
    if m.get("final_norm") == "ln":
        glob.update(lnf_g=(d,), lnf_b=(d,))
    if m.get("res_scale"):  # per-channel residual scales
        blk.update(res1=(d,), res2=(d,))
    if m["io_channels"]:
        c = m["io_channels"]
        glob.update(w_pre=(d, c), b_pre=(d,), w_post=(c, d), b_post=(c,))
    return dict(block=blk, glob=glob, n_blocks=L)


def make_weights(w: dict, bf16: bool | None = None):
    """Seeded weights for workload ``w``.  Matrices ~ N(0, w_std^2); biases ~ N(0, bias_std^2)
    (all-zero when bias_std == 0); LayerNorm gains 1 and shifts 0.

    Returns ``{"blocks": [ {name: float32 array}, ...], "glob": {...}, "bits": same with bf16 bits or None}``.
    """
    m = w["model"]
    if bf16 is None:
        bf16 = m["dtype"] == "bf16"
    shapes = weight_shapes(m)
    seed = w["seed"]

    def gen(name, shp):
        base = name.split(".")[-1]  # "block3.b_qkv" -> "b_qkv"
        # gains, shifts and residual scales: fp32 vectors (no bf16 bits); 1 / 0 unless the workload
        # asks for spread (affine_std) so that their paths are exercised
        spread = w.get("affine_std", 0.0)
        if (base.startswith("ln") and base.endswith("_g")) or base.startswith("res"):
            v = np.ones(shp, dtype=np.float32)
            if spread:
                v = v + normal(seed, name, shp, spread)
            return v, None
        if base.startswith("ln") and base.endswith("_b"):
            v = normal(seed, name, shp, spread) if spread else np.zeros(shp, dtype=np.float32)
            return v, None
        std = w["bias_std"] if base.startswith("b_") else w["w_std"]
        if std == 0.0:
            return np.zeros(shp, dtype=np.float32), (np.zeros(shp, dtype=np.uint16) if bf16 else None)
        if bf16:
            return normal(seed, name, shp, std, bf16=True)
        return normal(seed, name, shp, std), None

    blocks, bblocks = [], []
    for l in range(shapes["n_blocks"]):
        fb, bb = {}, {}
        for name, shp in shapes["block"].items():
            fb[name], bb[name] = gen(f"block{l}.{name}", shp)
        blocks.append(fb)
        bblocks.append(bb)
    glob, bglob = {}, {}
    for name, shp in shapes["glob"].items():
        glob[name], bglob[name] = gen(name, shp)
    return dict(blocks=blocks, glob=glob, bits=dict(blocks=bblocks, glob=bglob) if bf16 else None)


def make_tokens(w: dict, layout: dict, name: str = "x") -> np.ndarray:
    """Input latent.  Token-major [N, d] for the DiT configs; channel-major per document
    ([io_channels, len_doc] blocks, concatenated) for a model with 1x1 pre/post convolutions."""
    m = w["model"]
    n = layout["n_tokens"]
    width = m["io_channels"] if m["io_channels"] else m["hidden"]
    return normal(w["seed"], name, (n, width) if not m["io_channels"] else (width * n,), w["x_std"])


# ---------------------------------------------------------------------------------------------
# Latent I/O recipe.  The audio latent is 32 channels wide (the DiT emits a 32-wide audio latent,
# [H3] "Milestone: the whole t2va path composes end to end"); the pages give no video latent
# width or patch, so the stand-in is 48 channels with a (1, 2, 2) patch: 192 features per token.
# Tokens of each modality are rows [rows_m, width_m] in packed order; projections N(0, 1/fan_in)
# so activations keep unit scale, biases N(0, bias_std).
# ---------------------------------------------------------------------------------------------

VIDEO_LATENT = dict(channels=48, patch=(1, 2, 2))
AUDIO_LATENT = dict(channels=32)


def latent_widths() -> list[int]:
    pt, ph, pw = VIDEO_LATENT["patch"]
    return [VIDEO_LATENT["channels"] * pt * ph * pw, AUDIO_LATENT["channels"]]


def make_latent_io(seed: int, d: int, widths, bias_std: float = 0.02) -> dict:
    """Per-modality fp32 patch projections [d, width] and output heads [width, d] with biases."""
    return dict(w_patch=[normal(seed, f"w_patch{m}", (d, k), 1.0 / np.sqrt(k)) for m, k in enumerate(widths)],
                b_patch=[normal(seed, f"b_patch{m}", (d,), bias_std) for m in range(len(widths))],
                w_head=[normal(seed, f"w_head{m}", (k, d), 1.0 / np.sqrt(d)) for m, k in enumerate(widths)],
                b_head=[normal(seed, f"b_head{m}", (k,), bias_std) for m, k in enumerate(widths)])


def make_latents(seed: int, layout: dict, widths, name: str = "z") -> list:
    """Initial noise in token form: one N(0, 1) array [rows_m, width_m] per modality."""
    return [normal(seed, f"{name}{m}", (int((layout["tags"] == m).sum()), k), 1.0) for m, k in enumerate(widths)]


# ---------------------------------------------------------------------------------------------
# NVFP4 weights: random valid codes, no quantisation arithmetic.  Two FP4 (E2M1) codes per byte,
# uniform over all 16; one E4M3 scale per 16 along K with exponent field 4..6 (2^-3 .. 2^-1) and a
# random mantissa; the fp32 global scale 2^-6, so the dequantised weight has RMS near 0.02 (and,
# the global scale being a power of two, code * scale * global is exact in fp32).
# ---------------------------------------------------------------------------------------------

NVFP4_GLOBAL = 2.0 ** -6


def nvfp4_shapes(m: dict) -> dict:
    """[N, K] of the four linear maps of a block (the logical weight shapes)."""
    d, F = m["hidden"], m["ffn_hidden"]
    return {"qkv": (3 * d, d), "o": (d, d), "in": (2 * F, d), "down": (d, F)}


def make_nvfp4_linears(w: dict) -> list:
    """Per block {name: (q, s, g)} NVFP4 weights of the four linear maps of workload w."""
    shapes = nvfp4_shapes(w["model"])
    return [{n: make_nvfp4(w["seed"], f"block{l}.nvfp4.{n}", N, K) for n, (N, K) in shapes.items()}
            for l in range(w["model"]["n_blocks"])]


def make_nvfp4(seed: int, name: str, N: int, K: int):
    """(q [N, K/2] u8, scales [N, K/16] u8 E4M3 codes, global scale) for an [N, K] weight."""
    assert K % 16 == 0
    q = np.minimum(uniform(seed, name + ".q", N * K // 2) * 256, 255).astype(np.uint8).reshape(N, K // 2)
    e = 4 + np.minimum(uniform(seed, name + ".se", N * K // 16) * 3, 2).astype(np.uint8)
    m = np.minimum(uniform(seed, name + ".sm", N * K // 16) * 8, 7).astype(np.uint8)
    s = ((e << 3) | m).astype(np.uint8).reshape(N, K // 16)
    return q, s, NVFP4_GLOBAL
