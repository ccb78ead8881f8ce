"""The C ABI without a GPU: libdit.so loads, exports every entry point include/dit.h declares, and its
host-side validation answers with status codes before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _lib():
    from video_audio_gen_gb300 import build, dit
    build.build()
    return dit


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "dit.h")).read()
    return sorted(set(re.findall(r"^DIT_API [^(]*?\b(dit_\w+)\(", src, flags=re.M)))


def test_header_declares_the_boundary_calls():
    names = declared_symbols()
    for required in ("dit_create", "dit_bind_weights", "dit_forward", "dit_euler_step", "dit_destroy"):
        assert required in names
    assert len(names) >= 20


def test_library_exports_every_declared_symbol():
    dit = _lib()
    lib = dit.lib()
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)
    assert set(declared_symbols()) == set(dit.EXPORTS)


def _model(**kw):
    import synth
    m = dict(synth.WORKLOADS["video_audio_bf16"]["model"])
    m.update(kw)
    return m


def test_create_accepts_the_vit_decoder_block():
    import synth
    dit = _lib()
    h = dit.Dit(synth.WORKLOADS["vit3d_decoder"]["model"], 8192, 1)
    assert h.workspace_bytes(8192, 1) > 8192 * 2048 * 4
    h.h = None


def test_create_validates_config():
    dit = _lib()
    h = dit.Dit(_model(), 17408, 2)  # a supported model: no device memory is touched
    assert h.workspace_bytes(17408, 2) > 17408 * 3072 * 4
    h.h = None  # nothing was allocated; skip dit_destroy's device synchronisation here
    bad = [(dict(n_heads=23), dit.DIT_ERR_CONFIG), (dict(rope_dims=(32, 48, 40)), dit.DIT_ERR_CONFIG),
           (dict(hidden=3200, n_heads=25), dit.DIT_ERR_UNSUPPORTED), (dict(dtype="fp32"), dit.DIT_ERR_UNSUPPORTED),
           (dict(dtype="fp32", adaln=False, io_channels=96), dit.DIT_ERR_UNSUPPORTED),
           (dict(head_dim=96, n_heads=32, rope_dims=(32, 32, 32), rotary_dim=96), dit.DIT_ERR_UNSUPPORTED), (dict(n_blocks=0), dit.DIT_ERR_CONFIG),
           (dict(final_norm="ln"), dit.DIT_ERR_CONFIG),  # AdaLN's final layer is RMSNorm + modulate
           (dict(dtype="fp32", adaln=False, qk_norm=True), dit.DIT_ERR_UNSUPPORTED),
           (dict(rope_dims=(12, 16, 16), rotary_dim=44, n_heads=48, head_dim=64), dit.DIT_ERR_UNSUPPORTED),
           (dict(nvfp4=True, act_bf16=True), dit.DIT_ERR_UNSUPPORTED),  # NVFP4 GEMMs take f16 activations
           (dict(nvfp4=True, qkv_interleaved=True), dit.DIT_ERR_UNSUPPORTED)]
    for kw, st in bad:
        with pytest.raises(dit.DitError) as e:
            dit.Dit(_model(**kw), 100, 1)
        assert e.value.status == st, kw
        assert str(e.value)


def test_workspace_bytes_grows_with_tokens_and_rejects_bad_sizes():
    dit = _lib()
    cfg = dit.make_config(_model(), 40000, 4)
    f = dit.lib().dit_workspace_bytes
    a, b = f(ctypes.byref(cfg), 1000, 1), f(ctypes.byref(cfg), 2000, 1)
    assert 0 < a < b
    assert f(ctypes.byref(cfg), 0, 1) == 0 and f(ctypes.byref(cfg), 10, 0) == 0
    assert dit.lib().dit_workspace_bytes_host(ctypes.byref(cfg), 1000, 1) > a


def test_op_argument_checks_need_no_device():
    dit = _lib()
    L = dit.lib()
    assert L.dit_euler_step(None, None, 5, 1.0, 0.5, None) == dit.DIT_ERR_INVALID_ARG
    assert L.dit_euler_step(None, None, 0, 0.0, 0.5, None) == dit.DIT_ERR_INVALID_ARG  # sigma must be > 0
    assert L.dit_op_gemm(None, None, None, 10, 256, 64, None, 0, 0, None) == dit.DIT_ERR_INVALID_ARG
    p = ctypes.c_void_p(256)
    assert L.dit_op_gemm(p, p, None, 10, 200, 64, p, 0, 0, None) == dit.DIT_ERR_UNSUPPORTED
    assert L.dit_op_attention(p, p, p, 16, p, 1, 10, 2, 96, p, p, 0, None) == dit.DIT_ERR_UNSUPPORTED
    assert L.dit_op_attention(p, p, p, 16, p, 1, 10, 2, 128, p, p, 2, None) == dit.DIT_ERR_INVALID_ARG
    assert dit.attention_workspace_bytes(2, 17408) > 0 and dit.attention_workspace_bytes(0, 5) == 0
