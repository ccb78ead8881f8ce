"""Python face of the CPU oracle (``oracle.cpp``): ctypes marshalling only.

TEST INFRASTRUCTURE ONLY.  The oracle is the plain double-precision statement of the DiT forward;
only the tests, the package smoke check and the bench's CPU-baseline leg may import it.  It shares
no code with the CUDA library and never imports it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()

_c_dp = ctypes.POINTER(ctypes.c_double)
_c_fp = ctypes.POINTER(ctypes.c_float)


class OrcConfig(ctypes.Structure):
    _fields_ = [("n_blocks", ctypes.c_int), ("hidden", ctypes.c_int), ("n_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("ffn_hidden", ctypes.c_int), ("norm", ctypes.c_int),
                ("norm_eps", ctypes.c_double), ("adaln", ctypes.c_int), ("n_mod", ctypes.c_int),
                ("t_dim", ctypes.c_int), ("rope_axes", ctypes.c_int), ("rope_dims", ctypes.c_int * 3),
                ("rotary_dim", ctypes.c_int), ("rope_base", ctypes.c_double), ("io_channels", ctypes.c_int),
                ("qk_norm", ctypes.c_int), ("qkv_interleaved", ctypes.c_int), ("final_norm", ctypes.c_int)]


_BLOCK_NAMES = ["w_qkv", "b_qkv", "w_o", "b_o", "w_in", "b_in", "w_down", "b_down", "w_ada", "b_ada",
                "ln1_g", "ln1_b", "ln2_g", "ln2_b", "res1", "res2"]
_GLOB_NAMES = ["w_ada_final", "b_ada_final", "lnf_g", "lnf_b", "w_pre", "b_pre", "w_post", "b_post"]


class OrcBlock(ctypes.Structure):
    _fields_ = [(n, _c_fp) for n in _BLOCK_NAMES]


class OrcWeights(ctypes.Structure):
    _fields_ = [("blocks", ctypes.POINTER(OrcBlock))] + [(n, _c_fp) for n in _GLOB_NAMES]


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` beside its source (g++, OpenMP, no FMA contraction, no fast-math)."""
    src = os.path.join(_HERE, "oracle.cpp")
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", src, "-o", tmp])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            _lib.orc_forward.restype = ctypes.c_int
            _lib.orc_forward_mod.restype = ctypes.c_int
            _lib.orc_forward_latent.restype = ctypes.c_int
            _lib.orc_time_shift.restype = ctypes.c_double
            _lib.orc_span_sum_sequential.restype = ctypes.c_double
            _lib.orc_span_sum_pairwise.restype = ctypes.c_double
            _lib.orc_e2m1_decode.restype = ctypes.c_double
            _lib.orc_e4m3_decode.restype = ctypes.c_double
            _lib.orc_check_layout.restype = ctypes.c_int
            _lib.orc_count_q_tiles.restype = ctypes.c_int
            _lib.orc_get_threads.restype = ctypes.c_int
    return _lib


def set_threads(n: int) -> None:
    lib().orc_set_threads(int(n))


def _d(a):
    return a.ctypes.data_as(_c_dp)


def _p(a):
    return ctypes.c_void_p(a.ctypes.data)


def _f(a):
    return a.ctypes.data_as(_c_fp) if a is not None else None


def _dbl(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _flt(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


def config(m: dict) -> OrcConfig:
    c = OrcConfig()
    c.n_blocks, c.hidden, c.n_heads = m["n_blocks"], m["hidden"], m["n_heads"]
    c.head_dim, c.ffn_hidden = m["head_dim"], m["ffn_hidden"]
    c.norm = 0 if m["norm"] == "rms" else 1
    c.norm_eps = m["norm_eps"]
    c.adaln = 1 if m["adaln"] else 0
    c.n_mod, c.t_dim, c.rope_axes = m["n_mod"], m["t_dim"], m["rope_axes"]
    for i in range(3):
        c.rope_dims[i] = m["rope_dims"][i]
    c.rotary_dim, c.rope_base, c.io_channels = m["rotary_dim"], m["rope_base"], m["io_channels"]
    c.qk_norm = 1 if m.get("qk_norm") else 0
    c.qkv_interleaved = 1 if m.get("qkv_interleaved") else 0
    c.final_norm = {"same": 0, "rms": 1, "ln": 2}[m.get("final_norm", "same")]
    return c


class _Weights:
    """Keeps the float32 arrays alive while the ctypes view of them is in use."""

    def __init__(self, m: dict, weights: dict):
        self.keep = []
        self.blocks = (OrcBlock * m["n_blocks"])()
        for l, bw in enumerate(weights["blocks"]):
            for n in _BLOCK_NAMES:
                a = _flt(bw.get(n))
                self.keep.append(a)
                setattr(self.blocks[l], n, _f(a))
        self.w = OrcWeights()
        self.w.blocks = ctypes.cast(self.blocks, ctypes.POINTER(OrcBlock))
        for n in _GLOB_NAMES:
            a = _flt(weights["glob"].get(n))
            self.keep.append(a)
            setattr(self.w, n, _f(a))


# ------------------------------------------------------------------------------------------------
# op-level entry points
# ------------------------------------------------------------------------------------------------

def linspace(start: float, stop: float, n: int) -> np.ndarray:
    out = np.empty((n,), dtype=np.float64)
    lib().orc_linspace(ctypes.c_double(start), ctypes.c_double(stop), ctypes.c_int(n), _d(out))
    return out


def check_layout(cu, doc_ids, tags, n_tokens: int, n_mod: int) -> int:
    cu = np.ascontiguousarray(cu, dtype=np.int32)
    doc_ids = np.ascontiguousarray(doc_ids, dtype=np.int32)
    tags = np.ascontiguousarray(tags, dtype=np.uint8)
    return int(lib().orc_check_layout(_p(cu), len(cu) - 1, _p(doc_ids), _p(tags),
                                      int(n_tokens), int(n_mod)))


def span_sum_sequential(x) -> float:
    """Left-to-right sum of the spans, each add rounded ([H3] "Correctness gates")."""
    x = _dbl(np.asarray(x).reshape(-1))
    return float(lib().orc_span_sum_sequential(_d(x), ctypes.c_int(x.size)))


def span_sum_pairwise(x) -> float:
    """The spans summed in numpy's pairwise order ([H3] "Correctness gates")."""
    x = _dbl(np.asarray(x).reshape(-1))
    return float(lib().orc_span_sum_pairwise(_d(x), ctypes.c_int(x.size)))


def count_q_tiles(cu, tile: int = 128) -> int:
    cu = np.ascontiguousarray(cu, dtype=np.int32)
    return int(lib().orc_count_q_tiles(_p(cu), len(cu) - 1, int(tile)))


def timestep_embedding(t: float, t_dim: int) -> np.ndarray:
    out = np.empty((t_dim,), dtype=np.float64)
    lib().orc_timestep_embedding(ctypes.c_double(t), ctypes.c_int(t_dim), _d(out))
    return out


def adaln(m: dict, weights: dict, t):
    """Returns (mod [L, n_mod, 6, d], mod_final [n_mod, 2, d]) in float64.  t is one timestep, or
    one per modality (the per-modality sigma schedules)."""
    c = config(m)
    w = _Weights(m, weights)
    d, L, nm = m["hidden"], m["n_blocks"], m["n_mod"]
    mod = np.empty((L, nm, 6, d), dtype=np.float64)
    modf = np.empty((nm, 2, d), dtype=np.float64)
    if np.ndim(t) == 0:
        lib().orc_adaln(ctypes.byref(c), ctypes.byref(w.w), ctypes.c_double(t), _d(mod), _d(modf))
    else:
        tm = np.ascontiguousarray(t, dtype=np.float64)
        assert tm.shape == (nm,)
        lib().orc_adaln_mod(ctypes.byref(c), ctypes.byref(w.w), _d(tm), _d(mod), _d(modf))
    return mod, modf


def vit_positions(T: int, H: int, W: int) -> np.ndarray:
    """RotaryEmbeddingND positions [T*H*W, 3] (fp64) of the video-VAE decoder's T x H x W grid."""
    pos = np.empty((T * H * W, 3), dtype=np.float64)
    lib().orc_vit_positions(ctypes.c_int(T), ctypes.c_int(H), ctypes.c_int(W), _d(pos))
    return pos


def time_shift(sigma: float, shift: float) -> float:
    """The rectified-flow time shift of one sigma, in double (the oracle's formula)."""
    return float(lib().orc_time_shift(ctypes.c_double(sigma), ctypes.c_double(shift)))


def sigmas_shifted(base, shift: float) -> np.ndarray:
    """fp32 shifted schedule: each fp32 base sigma shifted in double, then rounded to fp32."""
    return np.array([time_shift(float(s), shift) for s in np.asarray(base, dtype=np.float32)], dtype=np.float32)


def rope_inv_freq(m: dict) -> np.ndarray:
    c = config(m)
    out = np.empty((m["rotary_dim"] // 2,), dtype=np.float32)
    lib().orc_rope_inv_freq(ctypes.byref(c), _f(out))
    return out


def rope_cos_sin(m: dict, pos) -> tuple[np.ndarray, np.ndarray]:
    c = config(m)
    pos = _dbl(pos)
    n = pos.shape[0]
    half = m["rotary_dim"] // 2
    cs = np.empty((n, half), dtype=np.float64)
    sn = np.empty((n, half), dtype=np.float64)
    lib().orc_rope_cos_sin(ctypes.byref(c), _d(pos), ctypes.c_int(n), _d(cs), _d(sn))
    return cs, sn


def rope_apply(x, n_heads: int, head_dim: int, rotary_dim: int, cs, sn) -> np.ndarray:
    x = _dbl(x).copy()
    n = x.shape[0]
    lib().orc_rope_apply(_d(x), ctypes.c_int(n), ctypes.c_int(n_heads), ctypes.c_int(head_dim),
                         ctypes.c_int(rotary_dim), _d(_dbl(cs)), _d(_dbl(sn)))
    return x


def rms_norm(x, eps: float) -> np.ndarray:
    x = _dbl(x)
    y = np.empty_like(x)
    lib().orc_rms_norm(_d(x), ctypes.c_int(x.shape[0]), ctypes.c_int(x.shape[1]), ctypes.c_double(eps), _d(y))
    return y


def layer_norm(x, eps: float, g=None, b=None) -> np.ndarray:
    x = _dbl(x)
    y = np.empty_like(x)
    g, b = _flt(g), _flt(b)
    lib().orc_layer_norm(_d(x), ctypes.c_int(x.shape[0]), ctypes.c_int(x.shape[1]), ctypes.c_double(eps),
                         _f(g), _f(b), _d(y))
    return y


def modulate(nrm, tags, shift, scale) -> np.ndarray:
    """shift, scale: [n_mod, d]."""
    nrm = _dbl(nrm)
    tags = np.ascontiguousarray(tags, dtype=np.uint8)
    shift, scale = _dbl(shift), _dbl(scale)
    y = np.empty_like(nrm)
    lib().orc_modulate(_d(nrm), ctypes.c_int(nrm.shape[0]), ctypes.c_int(nrm.shape[1]), _p(tags),
                       _d(shift), _d(scale), ctypes.c_size_t(shift.shape[1]), _d(y))
    return y


def linear(x, W, b=None) -> np.ndarray:
    x = _dbl(x)
    W = _flt(W)
    b = _flt(b)
    m, k = x.shape
    n_out = W.shape[0]
    y = np.empty((m, n_out), dtype=np.float64)
    lib().orc_linear(_d(x), ctypes.c_int(m), ctypes.c_int(k), _f(W), _f(b), ctypes.c_int(n_out), _d(y))
    return y


def conv1x1(x, W, b=None) -> np.ndarray:
    """x: [ci, T] channel-major; W: [co, ci]."""
    x = _dbl(x)
    W = _flt(W)
    b = _flt(b)
    ci, T = x.shape
    co = W.shape[0]
    y = np.empty((co, T), dtype=np.float64)
    lib().orc_conv1x1(_d(x), ctypes.c_int(ci), ctypes.c_int(T), _f(W), _f(b), ctypes.c_int(co), _d(y))
    return y


def attention(q, k, v, cu, n_heads: int, head_dim: int) -> np.ndarray:
    """q, k, v: [N, H*Dh]; returns [N, H*Dh]."""
    q, k, v = _dbl(q), _dbl(k), _dbl(v)
    cu = np.ascontiguousarray(cu, dtype=np.int32)
    o = np.empty_like(q)
    lib().orc_attention(_d(q), _d(k), _d(v), ctypes.c_int(q.shape[0]), ctypes.c_int(n_heads),
                        ctypes.c_int(head_dim), _p(cu), ctypes.c_int(len(cu) - 1), _d(o))
    return o


def attention_rows(q, k, v, cu, n_heads: int, head_dim: int, rows) -> np.ndarray:
    q, k, v = _dbl(q), _dbl(k), _dbl(v)
    cu = np.ascontiguousarray(cu, dtype=np.int32)
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    o = np.empty((len(rows), q.shape[1]), dtype=np.float64)
    lib().orc_attention_rows(_d(q), _d(k), _d(v), ctypes.c_int(q.shape[0]), ctypes.c_int(n_heads),
                             ctypes.c_int(head_dim), _p(cu), ctypes.c_int(len(cu) - 1), _p(rows),
                             ctypes.c_int(len(rows)), _d(o))
    return o


def swiglu(uv) -> np.ndarray:
    uv = _dbl(uv)
    n, f2 = uv.shape
    h = np.empty((n, f2 // 2), dtype=np.float64)
    lib().orc_swiglu(_d(uv), ctypes.c_int(n), ctypes.c_int(f2 // 2), _d(h))
    return h


def euler_step(x, v, sigma: float, sigma_next: float) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32).copy()
    v = np.ascontiguousarray(v, dtype=np.float32)
    lib().orc_euler_step(_f(x), _f(v), ctypes.c_int64(x.size), ctypes.c_float(sigma), ctypes.c_float(sigma_next))
    return x


def e2m1_decode(codes) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8).reshape(-1)
    return np.array([lib().orc_e2m1_decode(ctypes.c_uint8(int(v))) for v in c], dtype=np.float64)


def e4m3_decode(codes) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8).reshape(-1)
    return np.array([lib().orc_e4m3_decode(ctypes.c_uint8(int(v))) for v in c], dtype=np.float64)


def nvfp4_linear(x, q, scales, g: float, b=None) -> np.ndarray:
    """y = x W^T + b with the NVFP4 weight W = fp4(q) * e4m3(scales) * g; q [N, K/2] u8 (even k in the
    low nibble), scales [N, K/16] u8 (E4M3 codes), g the fp32 global scale.  Double precision."""
    x = _dbl(x)
    q = np.ascontiguousarray(q, dtype=np.uint8)
    sc = np.ascontiguousarray(scales, dtype=np.uint8)
    M, K = x.shape
    N = q.shape[0]
    assert q.shape == (N, K // 2) and sc.shape == (N, K // 16)
    y = np.empty((M, N), dtype=np.float64)
    lib().orc_nvfp4_linear(_d(x), ctypes.c_int(M), ctypes.c_int(K), _p(q), _p(sc), ctypes.c_float(g), _f(_flt(b)),
                           ctypes.c_int(N), _d(y))
    return y


def nvfp4_dequant(q, scales, g: float) -> np.ndarray:
    """The logical weight [N, K] of NVFP4 codes: e2m1(code) * e4m3(scale) * g, from the oracle's
    decoders, in double; returned as float32, which holds it exactly when g is a power of two (an E2M1
    value times an E4M3 scale has at most 6 significant bits)."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    sc = np.ascontiguousarray(scales, dtype=np.uint8)
    N = q.shape[0]
    K = q.shape[1] * 2
    codes = np.empty((N, K), dtype=np.uint8)
    codes[:, 0::2] = q & 15
    codes[:, 1::2] = q >> 4
    t2 = e2m1_decode(np.arange(16))
    t4 = e4m3_decode(np.arange(256))
    w = t2[codes] * np.repeat(t4[sc], 16, axis=1) * float(g)
    w32 = w.astype(np.float32)
    assert np.array_equal(w32.astype(np.float64), w), "not exact in fp32 (global scale not a power of two?)"
    return w32


def patchify(lat, pt: int, ph: int, pw: int) -> np.ndarray:
    """Latent [C, T*pt, H*ph, W*pw] -> tokens [T*H*W, C*pt*ph*pw] (exact)."""
    lat = np.ascontiguousarray(lat, dtype=np.float32)
    C, Tf, Hf, Wf = lat.shape
    T, H, W = Tf // pt, Hf // ph, Wf // pw
    assert T * pt == Tf and H * ph == Hf and W * pw == Wf
    tok = np.empty((T * H * W, C * pt * ph * pw), dtype=np.float32)
    lib().orc_patchify(_f(lat), C, T, H, W, pt, ph, pw, _f(tok))
    return tok


def unpatchify(tok, C: int, T: int, H: int, W: int, pt: int, ph: int, pw: int) -> np.ndarray:
    """Tokens [T*H*W, C*pt*ph*pw] -> latent [C, T*pt, H*ph, W*pw] (exact)."""
    tok = np.ascontiguousarray(tok, dtype=np.float32)
    assert tok.shape == (T * H * W, C * pt * ph * pw)
    lat = np.empty((C, T * pt, H * ph, W * pw), dtype=np.float32)
    lib().orc_unpatchify(_f(tok), C, T, H, W, pt, ph, pw, _f(lat))
    return lat


def audio_pack(lat) -> np.ndarray:
    """Audio latent [C, T] -> tokens [T, C]: patchify of a [C, T, 1, 1] latent with a 1x1x1 patch."""
    lat = np.ascontiguousarray(lat, dtype=np.float32)
    return patchify(lat.reshape(lat.shape[0], lat.shape[1], 1, 1), 1, 1, 1)


def audio_unpack(tok) -> np.ndarray:
    tok = np.ascontiguousarray(tok, dtype=np.float32)
    T, C = tok.shape
    return unpatchify(tok, C, T, 1, 1, 1, 1, 1).reshape(C, T)


def forward_latent(m: dict, weights: dict, io: dict, z, layout: dict, t, dumps: bool = False):
    """The forward between latent tokens: per-modality patch projection into the packed rows of that
    modality, the forward, per-modality output heads.  io = dict(w_patch, b_patch, w_head, b_head), one
    entry per modality; z[m] [rows_m, width_m] fp32.  Returns ([v_m float64], dumps or None)."""
    c = config(m)
    w = _Weights(m, weights)
    n_mod = len(z)
    n = layout["n_tokens"]
    zs = [np.ascontiguousarray(a, dtype=np.float32) for a in z]
    wp = [np.ascontiguousarray(a, dtype=np.float32) for a in io["w_patch"]]
    wh = [np.ascontiguousarray(a, dtype=np.float32) for a in io["w_head"]]
    bp = [None if a is None else np.ascontiguousarray(a, dtype=np.float32) for a in io["b_patch"]]
    bh = [None if a is None else np.ascontiguousarray(a, dtype=np.float32) for a in io["b_head"]]
    widths = [a.shape[1] for a in zs]
    vs = [np.empty((a.shape[0], widths[i]), dtype=np.float64) for i, a in enumerate(zs)]
    FP = _c_fp * n_mod
    DP = _c_dp * n_mod
    IA = ctypes.c_int * n_mod
    opt = lambda a: _f(a) if a is not None else None
    tm = np.ascontiguousarray([t] * n_mod if np.ndim(t) == 0 else t, dtype=np.float64)
    dm = np.empty((m["n_blocks"], n, m["hidden"]), dtype=np.float64) if dumps else None
    rc = lib().orc_forward_latent(
        ctypes.byref(c), ctypes.byref(w.w), ctypes.c_int(n_mod), FP(*[_f(a) for a in zs]),
        IA(*[a.shape[0] for a in zs]), IA(*widths), FP(*[_f(a) for a in wp]), FP(*[opt(a) for a in bp]),
        FP(*[_f(a) for a in wh]), FP(*[opt(a) for a in bh]), ctypes.c_int(n),
        _p(np.ascontiguousarray(layout["cu_seqlens"], dtype=np.int32)), ctypes.c_int(layout["n_docs"]),
        _p(np.ascontiguousarray(layout["doc_ids"], dtype=np.int32)),
        _p(np.ascontiguousarray(layout["tags"], dtype=np.uint8)), _d(_dbl(layout["pos"])), _d(tm),
        DP(*[_d(a) for a in vs]), _d(dm) if dumps else None)
    if rc:
        raise ValueError(f"oracle: invalid packed layout (code {rc})")
    return vs, dm


def euler_step_tagged(x, v, tags, sigma, sigma_next) -> np.ndarray:
    """Euler step of x [N, d] with each row's modality sigma pair (sigma[tags[r]], sigma_next[tags[r]])."""
    x = np.ascontiguousarray(x, dtype=np.float32).copy()
    v = np.ascontiguousarray(v, dtype=np.float32)
    tags = np.ascontiguousarray(tags, dtype=np.uint8)
    st = np.ascontiguousarray(sigma, dtype=np.float32)
    sn = np.ascontiguousarray(sigma_next, dtype=np.float32)
    lib().orc_euler_step_tagged(_f(x), _f(v), ctypes.c_int(x.shape[0]), ctypes.c_int(x.shape[1]),
                                _p(tags), _f(st), _f(sn))
    return x


def block_forward(m: dict, weights: dict, l: int, mod_block, x, layout: dict, cs, sn) -> np.ndarray:
    """One block in place on a float64 copy of x [N, d]; mod_block [n_mod, 6, d] or None."""
    c = config(m)
    w = _Weights(m, weights)
    x = _dbl(x).copy()
    mb = _dbl(mod_block) if mod_block is not None else None
    lib().orc_block_forward(ctypes.byref(c), ctypes.byref(w.blocks[l]), _d(mb) if mb is not None else None,
                            _d(x), ctypes.c_int(x.shape[0]),
                            _p(np.ascontiguousarray(layout["cu_seqlens"], dtype=np.int32)),
                            ctypes.c_int(layout["n_docs"]),
                            _p(np.ascontiguousarray(layout["tags"], dtype=np.uint8)),
                            _d(_dbl(cs)), _d(_dbl(sn)))
    return x


def block_rows(m: dict, weights: dict, l: int, mod_block, x, layout: dict, rows) -> np.ndarray:
    """Block ``l`` of the modality-AdaLN DiT on a subset of query rows: the output rows ``rows`` of
    orc_block_forward for the block input x [N, d], without computing the other rows' outputs.

    The attention of a row reads every key and value of its own document, so those are computed for
    every row of the documents the sampled rows fall in; everything after the attention is per row.
    The steps are orc_block_forward's ([H3] "The device-resident forward (W2b)"):
      y = RMS(x) (1 + scale1[tag]) + shift1[tag];   k, v = y W_{k,v}^T + b;   k <- RoPE(k)
      q = RoPE(y W_q^T + b) on the sampled rows;    o = softmax(q k^T / sqrt(Dh)) v per document
      x' = x + gate1[tag] (o W_o^T + b_o);          y2 = RMS(x') (1 + scale2) + shift2
      out = x' + gate2[tag] ((u * silu(g)) W_down^T + b_down),  [u | g] = y2 W_in^T + b_in
    every step in double.  The key/value projection of whole documents is the one step done with a
    library primitive (numpy's float64 matmul) rather than the oracle's naive loop, so that documents
    of tens of thousands of tokens finish in seconds; the other steps are the oracle's own functions.
    mod_block: [n_mod, 6, d] (this block's AdaLN rows).  Returns [len(rows), d] float64."""
    assert m["adaln"] and m["norm"] == "rms" and not m.get("qk_norm") and not m.get("qkv_interleaved")
    d, H, Dh, R, eps = m["hidden"], m["n_heads"], m["head_dim"], m["rotary_dim"], m["norm_eps"]
    bw = weights["blocks"][l]
    x = np.asarray(x)
    rows = np.asarray(rows, dtype=np.int64)
    cu = np.asarray(layout["cu_seqlens"], dtype=np.int64)
    tags = np.asarray(layout["tags"], dtype=np.uint8)
    mod = _dbl(mod_block)
    docs = np.unique(np.asarray(layout["doc_ids"])[rows])
    keys = np.concatenate([np.arange(cu[j], cu[j + 1]) for j in docs])
    lens = np.array([cu[j + 1] - cu[j] for j in docs], dtype=np.int64)
    cu_loc = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    first = {int(j): int(cu_loc[i]) - int(cu[j]) for i, j in enumerate(docs)}
    loc = np.array([r + first[int(layout["doc_ids"][r])] for r in rows], dtype=np.int64)

    y = modulate(rms_norm(x[keys], eps), tags[keys], mod[:, 0], mod[:, 1])
    w_qkv = np.asarray(bw["w_qkv"], dtype=np.float64)
    b_qkv = bw.get("b_qkv")
    b_qkv = None if b_qkv is None else np.asarray(b_qkv, dtype=np.float64)
    k = y @ w_qkv[d:2 * d].T
    v = y @ w_qkv[2 * d:].T
    if b_qkv is not None:
        k += b_qkv[d:2 * d]
        v += b_qkv[2 * d:]
    cs, sn = rope_cos_sin(m, np.asarray(layout["pos"])[keys])
    k = rope_apply(k, H, Dh, R, cs, sn)
    q = linear(y[loc], bw["w_qkv"][:d], None if b_qkv is None else bw["b_qkv"][:d])
    q = rope_apply(q, H, Dh, R, cs[loc], sn[loc])
    q_all = np.zeros_like(k)  # only the sampled rows' queries are read
    q_all[loc] = q
    o = attention_rows(q_all, k, v, cu_loc, H, Dh, loc)
    tg = tags[rows]
    xm = _dbl(x[rows]) + mod[tg, 2] * linear(o, bw["w_o"], bw.get("b_o"))
    y2 = modulate(rms_norm(xm, eps), tg, mod[:, 3], mod[:, 4])
    hh = swiglu(linear(y2, bw["w_in"], bw.get("b_in")))
    return xm + mod[tg, 5] * linear(hh, bw["w_down"], bw.get("b_down"))


def final_rows(m: dict, mod_final, x, tags) -> np.ndarray:
    """The final layer of the AdaLN DiT on given rows: RMS(x) (1 + scale_f[tag]) + shift_f[tag]
    (orc_forward's last step).  mod_final [n_mod, 2, d]; x [n, d]; tags [n]."""
    mf = _dbl(mod_final)
    return modulate(rms_norm(x, m["norm_eps"]), tags, mf[:, 0], mf[:, 1])


def forward(m: dict, weights: dict, x_in, layout: dict, t, dumps: bool = False):
    """Whole forward.  Returns (out float64 shaped like x_in, block dumps [L, N, d] or None).
    t is one timestep, or one per modality."""
    c = config(m)
    w = _Weights(m, weights)
    x_in = np.ascontiguousarray(x_in, dtype=np.float32)
    n = layout["n_tokens"]
    out = np.empty(x_in.shape, dtype=np.float64)
    dm = np.empty((m["n_blocks"], n, m["hidden"]), dtype=np.float64) if dumps else None
    cu = np.ascontiguousarray(layout["cu_seqlens"], dtype=np.int32)
    ids = np.ascontiguousarray(layout["doc_ids"], dtype=np.int32)
    tags = np.ascontiguousarray(layout["tags"], dtype=np.uint8)
    pos = _dbl(layout["pos"])
    if np.ndim(t) == 0:
        rc = lib().orc_forward(ctypes.byref(c), ctypes.byref(w.w), _f(x_in), ctypes.c_int(n), _p(cu),
                               ctypes.c_int(layout["n_docs"]), _p(ids), _p(tags), _d(pos),
                               ctypes.c_double(t), _d(out), _d(dm) if dumps else None)
    else:
        tm = np.ascontiguousarray(t, dtype=np.float64)
        rc = lib().orc_forward_mod(ctypes.byref(c), ctypes.byref(w.w), _f(x_in), ctypes.c_int(n), _p(cu),
                                   ctypes.c_int(layout["n_docs"]), _p(ids), _p(tags), _d(pos),
                                   _d(tm), _d(out), _d(dm) if dumps else None)
    if rc:
        raise ValueError(f"oracle: invalid packed layout (code {rc})")
    return out, dm
