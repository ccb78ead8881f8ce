"""Thin Python binding of libdit.so (include/dit.h): argument marshalling only.

Every step of the forward runs in the library's CUDA kernels; this module only turns torch tensors
into device pointers and calls the C ABI with the same names.  It raises if the library is missing:
there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdit.so")

DIT_OK, DIT_ERR_INVALID_ARG, DIT_ERR_CONFIG, DIT_ERR_UNBOUND, DIT_ERR_MISSING_WEIGHT, DIT_ERR_LAYOUT, \
    DIT_ERR_CAPACITY, DIT_ERR_CUDA, DIT_ERR_DEVICE_TIMEOUT, DIT_ERR_UNSUPPORTED, DIT_ERR_RANGE = range(11)
STATUS_NAMES = {0: "DIT_OK", 1: "DIT_ERR_INVALID_ARG", 2: "DIT_ERR_CONFIG", 3: "DIT_ERR_UNBOUND",
                4: "DIT_ERR_MISSING_WEIGHT", 5: "DIT_ERR_LAYOUT", 6: "DIT_ERR_CAPACITY", 7: "DIT_ERR_CUDA",
                8: "DIT_ERR_DEVICE_TIMEOUT", 9: "DIT_ERR_UNSUPPORTED", 10: "DIT_ERR_RANGE"}
DIT_RMSNORM, DIT_LAYERNORM = 0, 1
DIT_BF16, DIT_FP32 = 0, 1
DIT_ELEM_BF16, DIT_ELEM_F16 = 0, 1
KERNEL_KINDS = ["gemm_qkv", "attention", "gemm_out", "gemm_ffn_up", "gemm_ffn_down", "norm_modulate", "other",
                "latent_io"]
MAX_LATENT_MODALITIES = 8

EXPORTS = ["dit_create", "dit_destroy", "dit_last_error", "dit_workspace_bytes", "dit_bind_weights", "dit_bind_nvfp4",
           "dit_forward",
           "dit_forward_modal", "dit_workspace_bytes_host", "dit_forward_host", "dit_euler_step",
           "dit_euler_step_modal", "dit_time_shift", "dit_vit_positions", "dit_bind_latent_io", "dit_workspace_bytes_latent",
           "dit_forward_latent", "dit_patchify", "dit_unpatchify", "dit_audio_pack", "dit_audio_unpack", "dit_get_stats", "dit_sync_status",
           "dit_set_dump", "dit_set_kernel_timing", "dit_get_kernel_times", "dit_op_norm_modulate",
           "dit_op_rope_cache", "dit_op_adaln", "dit_op_gemm", "dit_op_gemm_qkv_rope", "dit_op_gemm_gated_residual",
           "dit_op_gemm_swiglu", "dit_nvfp4_packed_bytes", "dit_op_pack_nvfp4", "dit_op_gemm_nvfp4",
           "dit_gemm_f32_workspace_bytes", "dit_op_gemm_f32", "dit_op_pack_ffn_in", "dit_attention_workspace_bytes", "dit_op_attention",
           "dit_attention_block_rows",
           "dit_op_attention_noalloc", "dit_op_attention_noalloc_status", "dit_selftest_wait_timeout"]


class DitLatentIO(ctypes.Structure):
    _fields_ = [("n_modalities", ctypes.c_int), ("width", ctypes.c_int * MAX_LATENT_MODALITIES)] + \
               [(n, ctypes.c_void_p * MAX_LATENT_MODALITIES) for n in ("w_patch", "b_patch", "w_head", "b_head")]


class DitError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class DitConfig(ctypes.Structure):
    _fields_ = [("n_blocks", ctypes.c_int), ("hidden", ctypes.c_int), ("n_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("ffn_hidden", ctypes.c_int), ("norm", ctypes.c_int),
                ("norm_eps", ctypes.c_float), ("adaln", ctypes.c_int), ("n_modalities", ctypes.c_int),
                ("t_embed_dim", ctypes.c_int), ("rope_axes", ctypes.c_int), ("rope_dims", ctypes.c_int * 3),
                ("rotary_dim", ctypes.c_int), ("rope_base", ctypes.c_double), ("io_channels", ctypes.c_int),
                ("dtype", ctypes.c_int), ("max_tokens", ctypes.c_int), ("max_docs", ctypes.c_int),
                ("qk_norm", ctypes.c_int), ("qkv_interleaved", ctypes.c_int), ("final_norm", ctypes.c_int),
                ("act_bf16", ctypes.c_int), ("nvfp4", ctypes.c_int)]


class DitNvfp4Linear(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("s", ctypes.c_void_p), ("g", ctypes.c_float)]


NVFP4_LINEARS = ["qkv", "o", "in", "down"]


class DitNvfp4Block(ctypes.Structure):
    _fields_ = [(n, DitNvfp4Linear) for n in NVFP4_LINEARS]


BLOCK_FIELDS = ["w_qkv", "b_qkv", "w_o", "b_o", "w_in", "b_in", "w_down", "b_down", "w_ada", "b_ada",
                "ln1_g", "ln1_b", "ln2_g", "ln2_b", "res1", "res2"]
GLOB_FIELDS = ["w_ada_final", "b_ada_final", "lnf_g", "lnf_b", "w_pre", "b_pre", "w_post", "b_post"]


class DitBlockWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in BLOCK_FIELDS]


class DitWeights(ctypes.Structure):
    _fields_ = [("n_blocks", ctypes.c_int), ("blocks", ctypes.POINTER(DitBlockWeights))] + \
        [(n, ctypes.c_void_p) for n in GLOB_FIELDS]


class DitStats(ctypes.Structure):
    _fields_ = [("forwards", ctypes.c_int64), ("kernels_launched", ctypes.c_int64),
                ("gemm_launches", ctypes.c_int64), ("attention_launches", ctypes.c_int64),
                ("norm_launches", ctypes.c_int64), ("other_launches", ctypes.c_int64),
                ("attention_tiles", ctypes.c_int64), ("bound_bytes", ctypes.c_int64),
                ("device_status", ctypes.c_int32), ("last_layout_error", ctypes.c_int32)]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


_lib = None


def lib():
    """Load libdit.so from the package directory (built by ``video_audio_gen_gb300.build``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libdit.so is not built ({LIB_PATH}); run video_audio_gen_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, f32, f64, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_double,
                                      ctypes.c_size_t)
        sig = {
            "dit_create": (i32, [ctypes.POINTER(DitConfig), ctypes.POINTER(vp)]),
            "dit_destroy": (i32, [vp]),
            "dit_last_error": (ctypes.c_char_p, [vp]),
            "dit_workspace_bytes": (sz, [ctypes.POINTER(DitConfig), i32, i32]),
            "dit_workspace_bytes_host": (sz, [ctypes.POINTER(DitConfig), i32, i32]),
            "dit_bind_weights": (i32, [vp, ctypes.POINTER(DitWeights), vp]),
            "dit_bind_nvfp4": (i32, [vp, ctypes.POINTER(DitNvfp4Block), vp]),
            "dit_forward": (i32, [vp, vp, vp, i32, vp, vp, vp, i32, f32, vp, vp, sz, vp]),
            "dit_forward_host": (i32, [vp, vp, vp, i32, vp, vp, vp, i32, f32, vp, vp, sz, vp]),
            "dit_forward_modal": (i32, [vp, vp, vp, i32, vp, vp, vp, i32, ctypes.POINTER(ctypes.c_float), vp, vp,
                                        sz, vp]),
            "dit_euler_step": (i32, [vp, vp, i64, f32, f32, vp]),
            "dit_euler_step_modal": (i32, [vp, vp, i32, i32, vp, ctypes.POINTER(ctypes.c_float),
                                           ctypes.POINTER(ctypes.c_float), i32, vp]),
            "dit_time_shift": (f32, [f32, f32]),
            "dit_vit_positions": (i32, [i32, i32, i32, vp]),
            "dit_bind_latent_io": (i32, [vp, ctypes.POINTER(DitLatentIO), vp]),
            "dit_workspace_bytes_latent": (sz, [vp, i32, i32]),
            "dit_forward_latent": (i32, [vp, ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_int), vp, i32, vp,
                                         vp, vp, i32, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_void_p),
                                         vp, sz, vp]),
            "dit_patchify": (i32, [vp, i32, i32, i32, i32, i32, i32, i32, vp, vp]),
            "dit_unpatchify": (i32, [vp, i32, i32, i32, i32, i32, i32, i32, vp, vp]),
            "dit_audio_pack": (i32, [vp, i32, i32, vp, vp]),
            "dit_audio_unpack": (i32, [vp, i32, i32, vp, vp]),
            "dit_get_stats": (i32, [vp, ctypes.POINTER(DitStats)]),
            "dit_sync_status": (i32, [vp, vp, vp]),
            "dit_set_dump": (i32, [vp, vp]),
            "dit_set_kernel_timing": (i32, [vp, i32]),
            "dit_get_kernel_times": (i32, [vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64)]),
            "dit_op_norm_modulate": (i32, [vp, i32, i32, i32, f32, vp, vp, vp, vp, vp, i64, vp, i32, vp]),
            "dit_op_rope_cache": (i32, [vp, i32, i32, ctypes.POINTER(ctypes.c_int), f64, vp, vp, vp]),
            "dit_op_adaln": (i32, [vp, vp, i32, i32, f32, vp, vp]),
            "dit_op_gemm": (i32, [vp, vp, vp, i32, i32, i32, vp, i32, i32, vp]),
            "dit_op_gemm_qkv_rope": (i32, [vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, i32, i32,
                                           vp]),
            "dit_op_gemm_gated_residual": (i32, [vp, vp, vp, i32, i32, i32, vp, vp, i64, vp, i32, vp]),
            "dit_op_gemm_swiglu": (i32, [vp, vp, vp, i32, i32, i32, vp, i32, vp]),
            "dit_op_pack_ffn_in": (i32, [vp, vp, i32, i32, vp, vp, vp]),
            "dit_attention_workspace_bytes": (sz, [i32, i32]),
            "dit_attention_block_rows": (i32, []),
            "dit_gemm_f32_workspace_bytes": (sz, [i32, i32, i32]),
            "dit_nvfp4_packed_bytes": (sz, [i32, i32]),
            "dit_op_pack_nvfp4": (i32, [vp, vp, i32, i32, vp, vp]),
            "dit_op_gemm_nvfp4": (i32, [vp, vp, f32, vp, i32, i32, i32, vp, i32, vp]),
            "dit_op_gemm_f32": (i32, [vp, vp, vp, i32, i32, i32, vp, vp, vp]),
            "dit_op_attention": (i32, [vp, vp, vp, i32, vp, i32, i32, i32, i32, vp, vp, i32, vp]),
            "dit_op_attention_noalloc": (i32, [vp, vp, vp, i32, vp, i32, i32, i32, i32, vp, i32, vp]),
            "dit_op_attention_noalloc_status": (i32, [vp, vp]),
            "dit_selftest_wait_timeout": (i32, [ctypes.c_uint64, vp, vp]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(st: int, handle=None):
    if st != DIT_OK:
        msg = lib().dit_last_error(handle)
        raise DitError(st, msg.decode() if msg else "")


def make_config(m: dict, max_tokens: int, max_docs: int) -> DitConfig:
    """dit_config from a model description (the dict layout of the workload recipes)."""
    c = DitConfig()
    c.n_blocks, c.hidden, c.n_heads, c.head_dim = m["n_blocks"], m["hidden"], m["n_heads"], m["head_dim"]
    c.ffn_hidden = m["ffn_hidden"]
    c.norm = DIT_RMSNORM if m["norm"] == "rms" else DIT_LAYERNORM
    c.norm_eps = m["norm_eps"]
    c.adaln = 1 if m["adaln"] else 0
    c.n_modalities, c.t_embed_dim, c.rope_axes = m["n_mod"], m["t_dim"], m["rope_axes"]
    for i in range(3):
        c.rope_dims[i] = m["rope_dims"][i]
    c.rotary_dim, c.rope_base, c.io_channels = m["rotary_dim"], m["rope_base"], m["io_channels"]
    c.dtype = DIT_BF16 if m["dtype"] == "bf16" else DIT_FP32
    c.max_tokens, c.max_docs = max_tokens, max_docs
    c.qk_norm = 1 if m.get("qk_norm") else 0
    c.qkv_interleaved = 1 if m.get("qkv_interleaved") else 0
    c.final_norm = {"same": 0, "rms": 1, "ln": 2}[m.get("final_norm", "same")]
    c.act_bf16 = 1 if m.get("act_bf16") else 0
    c.nvfp4 = 1 if m.get("nvfp4") else 0
    return c


class Dit:
    """One dit_handle: create, bind once, forward many times."""

    def __init__(self, model: dict, max_tokens: int, max_docs: int):
        self.model = model
        self.cfg = make_config(model, max_tokens, max_docs)
        h = ctypes.c_void_p()
        _check(lib().dit_create(ctypes.byref(self.cfg), ctypes.byref(h)))
        self.h = h
        self._keep = None

    def close(self):
        if self.h:
            lib().dit_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def workspace_bytes(self, n_tokens: int, n_docs: int, host: bool = False) -> int:
        f = lib().dit_workspace_bytes_host if host else lib().dit_workspace_bytes
        return int(f(ctypes.byref(self.cfg), n_tokens, n_docs))

    def bind_weights(self, blocks: list[dict], glob: dict, stream=None):
        """blocks / glob: dicts of device tensors (names as in dit_block_weights / dit_weights)."""
        arr = (DitBlockWeights * len(blocks))()
        for l, b in enumerate(blocks):
            for n in BLOCK_FIELDS:
                t = b.get(n)
                setattr(arr[l], n, t.data_ptr() if t is not None else None)
        w = DitWeights()
        w.n_blocks = len(blocks)
        w.blocks = ctypes.cast(arr, ctypes.POINTER(DitBlockWeights))
        for n in GLOB_FIELDS:
            t = glob.get(n)
            setattr(w, n, t.data_ptr() if t is not None else None)
        self._keep = (blocks, glob)
        _check(lib().dit_bind_weights(self.h, ctypes.byref(w), _stream(stream)), self.h)

    def bind_nvfp4(self, blocks: list[dict], stream=None):
        """dit_bind_nvfp4: per block a dict {name: (q, s, g)} for name in qkv, o, in, down, with q, s
        device uint8 tensors (E2M1 codes two per byte, E4M3 scales) and g the fp32 global scale."""
        arr = (DitNvfp4Block * len(blocks))()
        for l, b in enumerate(blocks):
            for n in NVFP4_LINEARS:
                q, s, g = b[n]
                lin = getattr(arr[l], n)
                lin.q, lin.s, lin.g = _ptr(q), _ptr(s), float(g)
        self._keep_nvfp4 = blocks
        _check(lib().dit_bind_nvfp4(self.h, arr, _stream(stream)), self.h)

    def forward(self, x, cu_seqlens, doc_ids, tags, pos, t: float, out, workspace, stream=None):
        n_docs = cu_seqlens.numel() - 1
        n_tokens = doc_ids.numel()
        _check(lib().dit_forward(self.h, _ptr(x), _ptr(cu_seqlens), n_docs, _ptr(doc_ids), _ptr(tags), _ptr(pos),
                                 n_tokens, float(t), _ptr(out), _ptr(workspace), workspace.numel(),
                                 _stream(stream)), self.h)

    def forward_modal(self, x, cu_seqlens, doc_ids, tags, pos, ts, out, workspace, stream=None):
        """dit_forward_modal: `ts` holds one flow time per modality (tag order)."""
        n_docs = cu_seqlens.numel() - 1
        n_tokens = doc_ids.numel()
        arr = (ctypes.c_float * len(ts))(*[float(t) for t in ts])
        _check(lib().dit_forward_modal(self.h, _ptr(x), _ptr(cu_seqlens), n_docs, _ptr(doc_ids), _ptr(tags),
                                       _ptr(pos), n_tokens, arr, _ptr(out), _ptr(workspace), workspace.numel(),
                                       _stream(stream)), self.h)

    def bind_latent_io(self, io: dict, stream=None):
        """io: dict of per-modality lists of fp32 device tensors w_patch [d, width], b_patch [d] (or None),
        w_head [width, d], b_head [width] (or None).  The library keeps its own copies."""
        n = len(io["w_patch"])
        s = DitLatentIO()
        s.n_modalities = n
        for m in range(n):
            s.width[m] = io["w_patch"][m].shape[1]
            for name in ("w_patch", "b_patch", "w_head", "b_head"):
                t = io[name][m]
                getattr(s, name)[m] = t.data_ptr() if t is not None else None
        _check(lib().dit_bind_latent_io(self.h, ctypes.byref(s), _stream(stream)), self.h)

    def workspace_bytes_latent(self, n_tokens: int, n_docs: int) -> int:
        return int(lib().dit_workspace_bytes_latent(self.h, n_tokens, n_docs))

    def forward_latent(self, z, cu_seqlens, doc_ids, tags, pos, ts, v, workspace, stream=None):
        """z, v: per-modality lists of device tensors [rows_m, width_m]; ts one flow time per modality."""
        n = len(z)
        zp = (ctypes.c_void_p * n)(*[a.data_ptr() if a is not None and a.numel() else None for a in z])
        vp_ = (ctypes.c_void_p * n)(*[a.data_ptr() if a is not None and a.numel() else None for a in v])
        rows = (ctypes.c_int * n)(*[0 if a is None else int(a.shape[0]) for a in z])
        tt = (ctypes.c_float * n)(*[float(t) for t in ts])
        _check(lib().dit_forward_latent(self.h, zp, rows, _ptr(cu_seqlens), cu_seqlens.numel() - 1, _ptr(doc_ids),
                                        _ptr(tags), _ptr(pos), doc_ids.numel(), tt, vp_, _ptr(workspace),
                                        workspace.numel(), _stream(stream)), self.h)

    def forward_host(self, x, cu_seqlens, doc_ids, tags, pos, t: float, out, workspace, stream=None):
        """Host (preferably pinned) CPU tensors in and out; device workspace."""
        n_docs = cu_seqlens.numel() - 1
        n_tokens = doc_ids.numel()
        _check(lib().dit_forward_host(self.h, _ptr(x), _ptr(cu_seqlens), n_docs, _ptr(doc_ids), _ptr(tags),
                                      _ptr(pos), n_tokens, float(t), _ptr(out), _ptr(workspace), workspace.numel(),
                                      _stream(stream)), self.h)

    def stats(self) -> dict:
        s = DitStats()
        _check(lib().dit_get_stats(self.h, ctypes.byref(s)), self.h)
        return s.as_dict()

    def sync_status(self, workspace, stream=None) -> int:
        return int(lib().dit_sync_status(self.h, _ptr(workspace), _stream(stream)))

    def set_dump(self, dump):
        _check(lib().dit_set_dump(self.h, _ptr(dump)), self.h)

    def set_kernel_timing(self, enable: bool):
        _check(lib().dit_set_kernel_timing(self.h, 1 if enable else 0), self.h)

    def kernel_times(self) -> dict:
        ms = (ctypes.c_double * len(KERNEL_KINDS))()
        n = (ctypes.c_int64 * len(KERNEL_KINDS))()
        _check(lib().dit_get_kernel_times(self.h, ms, n), self.h)
        return {k: (ms[i], n[i]) for i, k in enumerate(KERNEL_KINDS)}


# ------------------------------------------------------------------------------------------------
# op-level calls
# ------------------------------------------------------------------------------------------------

def selftest_wait_timeout(limit_ns: int, status_word, stream=None) -> int:
    """Run the bounded-wait self-test; returns the dit_status (DIT_ERR_DEVICE_TIMEOUT when the wait ran
    out and was reported, as it should)."""
    return int(lib().dit_selftest_wait_timeout(int(limit_ns), _ptr(status_word), _stream(stream)))


def euler_step(x, v, sigma: float, sigma_next: float, stream=None):
    _check(lib().dit_euler_step(_ptr(x), _ptr(v), x.numel(), float(sigma), float(sigma_next), _stream(stream)))


def euler_step_modal(x, v, tags, sigma, sigma_next, stream=None):
    """dit_euler_step_modal: row r of x [N, d] steps with (sigma[tags[r]], sigma_next[tags[r]])."""
    n, d = x.shape
    if len(sigma) != len(sigma_next):
        raise ValueError("sigma and sigma_next differ in length")
    st = (ctypes.c_float * len(sigma))(*[float(a) for a in sigma])
    sn = (ctypes.c_float * len(sigma_next))(*[float(a) for a in sigma_next])
    _check(lib().dit_euler_step_modal(_ptr(x), _ptr(v), n, d, _ptr(tags), st, sn, len(sigma), _stream(stream)))


def vit_positions(T: int, H: int, W: int):
    """dit_vit_positions: RotaryEmbeddingND positions [T*H*W, 3] (numpy fp64) of a T x H x W grid."""
    import numpy as np
    pos = np.empty((T * H * W, 3), dtype=np.float64)
    _check(lib().dit_vit_positions(T, H, W, pos.ctypes.data))
    return pos


def time_shift(sigma: float, shift: float) -> float:
    """dit_time_shift: shift * sigma / (1 + (shift - 1) * sigma) in double, rounded to fp32."""
    return float(lib().dit_time_shift(float(sigma), float(shift)))


def patchify(latent, pt: int, ph: int, pw: int, tokens, stream=None):
    """dit_patchify: latent [C, T*pt, H*ph, W*pw] -> tokens [T*H*W, C*pt*ph*pw] (device fp32)."""
    C, Tf, Hf, Wf = latent.shape
    _check(lib().dit_patchify(_ptr(latent), C, Tf // pt, Hf // ph, Wf // pw, pt, ph, pw, _ptr(tokens),
                              _stream(stream)))


def unpatchify(tokens, C: int, T: int, H: int, W: int, pt: int, ph: int, pw: int, latent, stream=None):
    _check(lib().dit_unpatchify(_ptr(tokens), C, T, H, W, pt, ph, pw, _ptr(latent), _stream(stream)))


def audio_pack(latent, tokens, stream=None):
    """dit_audio_pack: [C, T] -> [T, C]."""
    C, T = latent.shape
    _check(lib().dit_audio_pack(_ptr(latent), C, T, _ptr(tokens), _stream(stream)))


def audio_unpack(tokens, latent, stream=None):
    T, C = tokens.shape
    _check(lib().dit_audio_unpack(_ptr(tokens), C, T, _ptr(latent), _stream(stream)))


def norm_modulate(x, norm: int, eps: float, y, out_kind: int, tags=None, shift=None, scale=None, mod_stride=0,
                  ln_g=None, ln_b=None, stream=None):
    n, d = x.shape
    _check(lib().dit_op_norm_modulate(_ptr(x), n, d, norm, float(eps), _ptr(ln_g), _ptr(ln_b), _ptr(tags),
                                      _ptr(shift), _ptr(scale), int(mod_stride), _ptr(y), out_kind, _stream(stream)))


def rope_cache(pos, n_axes: int, dims, base: float, cos_out, sin_out, stream=None):
    arr = (ctypes.c_int * 3)(*list(dims) + [0] * (3 - len(dims)))
    _check(lib().dit_op_rope_cache(_ptr(pos), pos.shape[0], n_axes, arr, float(base), _ptr(cos_out), _ptr(sin_out),
                                   _stream(stream)))


def adaln(w, b, t: float, mod, stream=None):
    rows, t_dim = w.shape
    _check(lib().dit_op_adaln(_ptr(w), _ptr(b), rows, t_dim, float(t), _ptr(mod), _stream(stream)))


def elem_of(t) -> int:
    """DIT_ELEM_F16 for a torch.float16 tensor, DIT_ELEM_BF16 for a torch.bfloat16 one."""
    import torch
    if t.dtype == torch.float16:
        return DIT_ELEM_F16
    if t.dtype == torch.bfloat16:
        return DIT_ELEM_BF16
    raise TypeError(f"16-bit operand expected, got {t.dtype}")


def gemm(a, b, bias, out, out_kind: int, stream=None):
    M, K = a.shape
    N = b.shape[0]
    _check(lib().dit_op_gemm(_ptr(a), _ptr(b), _ptr(bias), M, N, K, _ptr(out), out_kind, elem_of(a), _stream(stream)))


def nvfp4_packed_bytes(N: int, K: int) -> int:
    return int(lib().dit_nvfp4_packed_bytes(N, K))


def pack_nvfp4(q, scales, packed, stream=None):
    """dit_op_pack_nvfp4: q u8 [N, K/2], scales u8 [N, K/16] (device) -> packed (device bytes)."""
    N = q.shape[0]
    K = scales.shape[1] * 16
    _check(lib().dit_op_pack_nvfp4(_ptr(q), _ptr(scales), N, K, _ptr(packed), _stream(stream)))


def gemm_nvfp4(a_f16, packed, w_scale: float, bias, N: int, out, out_kind: int, stream=None):
    """dit_op_gemm_nvfp4: out = A W^T + bias, A f16 [M, K], W the packed NVFP4 weight [N, K]."""
    M, K = a_f16.shape
    _check(lib().dit_op_gemm_nvfp4(_ptr(a_f16), _ptr(packed), float(w_scale), _ptr(bias), M, N, K, _ptr(out),
                                   out_kind, _stream(stream)))


def gemm_f32_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(lib().dit_gemm_f32_workspace_bytes(M, N, K))


def gemm_f32(x, w, bias, y, workspace, stream=None):
    """dit_op_gemm_f32: y = x w^T + bias in fp32 (3xTF32 on the tensor cores)."""
    M, K = x.shape
    N = w.shape[0]
    _check(lib().dit_op_gemm_f32(_ptr(x), _ptr(w), _ptr(bias), M, N, K, _ptr(y), _ptr(workspace), _stream(stream)))


def gemm_qkv_rope(a, b, bias, n_heads, head_dim, rotary_dim, cos_c, sin_c, q, k, vt, n_pad, stream=None):
    M, K = a.shape
    d = b.shape[0] // 3
    _check(lib().dit_op_gemm_qkv_rope(_ptr(a), _ptr(b), _ptr(bias), M, d, K, n_heads, head_dim, rotary_dim,
                                      _ptr(cos_c), _ptr(sin_c), _ptr(q), _ptr(k), _ptr(vt), n_pad, elem_of(a),
                                      _stream(stream)))


def gemm_gated_residual(a, b, bias, x, gate=None, gate_stride=0, tags=None, stream=None):
    M, K = a.shape
    N = b.shape[0]
    _check(lib().dit_op_gemm_gated_residual(_ptr(a), _ptr(b), _ptr(bias), M, N, K, _ptr(x), _ptr(gate),
                                            int(gate_stride), _ptr(tags), elem_of(a), _stream(stream)))


def gemm_swiglu(a, b_packed, bias_packed, h, stream=None):
    M, K = a.shape
    F = b_packed.shape[0] // 2
    _check(lib().dit_op_gemm_swiglu(_ptr(a), _ptr(b_packed), _ptr(bias_packed), M, F, K, _ptr(h), elem_of(a),
                                    _stream(stream)))


def pack_ffn_in(w_in, b_in, w_packed, b_packed, stream=None):
    F2, d = w_in.shape
    _check(lib().dit_op_pack_ffn_in(_ptr(w_in), _ptr(b_in), F2 // 2, d, _ptr(w_packed), _ptr(b_packed),
                                    _stream(stream)))


def attention_workspace_bytes(n_docs: int, n_tokens: int) -> int:
    return int(lib().dit_attention_workspace_bytes(n_docs, n_tokens))


def attention_block_rows() -> int:
    return int(lib().dit_attention_block_rows())


def attention(q, k, vt, n_pad, cu_seqlens, n_heads, head_dim, o, workspace, stream=None):
    n_tokens = q.shape[0]
    _check(lib().dit_op_attention(_ptr(q), _ptr(k), _ptr(vt), n_pad, _ptr(cu_seqlens), cu_seqlens.numel() - 1,
                                  n_tokens, n_heads, head_dim, _ptr(o), _ptr(workspace), elem_of(q), _stream(stream)))


def attention_noalloc(q, k, vt, n_pad, cu_seqlens, n_heads, head_dim, o, stream=None):
    """dit_op_attention_noalloc: the attention with its scratch in the library's fixed device array
    (for callers that cannot allocate); calls whose device work overlaps must be serialised."""
    n_tokens = q.shape[0]
    _check(lib().dit_op_attention_noalloc(_ptr(q), _ptr(k), _ptr(vt), n_pad, _ptr(cu_seqlens),
                                          cu_seqlens.numel() - 1, n_tokens, n_heads, head_dim, _ptr(o), elem_of(q),
                                          _stream(stream)))


def attention_noalloc_status(stream=None) -> tuple[int, int]:
    """dit_op_attention_noalloc_status: (status, layout code) of the last no-allocation attention call
    in this context; synchronises the stream."""
    code = ctypes.c_int(0)
    st = int(lib().dit_op_attention_noalloc_status(ctypes.byref(code), _stream(stream)))
    return st, int(code.value)
