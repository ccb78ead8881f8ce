"""The video-VAE ViT3D decoder block as a second workload of the bf16 kernels, through the C ABI
against the oracle: per-head interleaved qkv (repacked at bind), per-head q/k RMS norm, RMS gains,
per-channel residual scales, RotaryEmbeddingND positions, a final LayerNorm."""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from tests.parity import GATE, forward_gates  # noqa: E402


def _gu():
    from tests import gpu_util
    return gpu_util


def _dit():
    from video_audio_gen_gb300 import dit
    return dit


def _positions(fn, docs):
    """Each document's own normalised grid, concatenated in packed order."""
    return np.concatenate([fn(*d["video"]) for d in docs])


def test_vit_positions_match_the_oracle_bit_for_bit():
    dit = _dit()
    for grid in [(1, 1, 1), (2, 8, 16), (8, 32, 32), (3, 5, 7)]:
        a = dit.vit_positions(*grid)
        b = oracle.vit_positions(*grid)
        assert np.array_equal(a.view(np.uint64), b.view(np.uint64)), grid


def test_vit_block_forward_matches_oracle():
    gu = _gu()
    w = synth.WORKLOADS["vit3d_small"]
    m = w["model"]
    lay = dict(synth.build_layout(w["docs"]))
    W = synth.make_weights(w)
    x = synth.make_tokens(w, lay)
    lay_gpu = dict(lay, pos=_positions(_dit().vit_positions, w["docs"]))
    run = gu.run_forward(w, dumps=True, layout=lay_gpu, weights=W, x=x, t=0.0)
    assert run["status"] == 0
    lay_orc = dict(lay, pos=_positions(oracle.vit_positions, w["docs"]))
    oracle.set_threads(8)
    ref, dumps = oracle.forward(m, W, x, lay_orc, 0.0, dumps=True)
    oracle.set_threads(1)
    fails = forward_gates(x, run["dumps"], dumps, run["out"], ref)
    assert not fails, fails


def test_vit_block_reading_the_weight_the_dit_way_fails_the_gate():
    """The trap the pages record: the same weights read as [q_all | k_all | v_all] give a
    plausible-but-wrong result, which the gate catches."""
    gu = _gu()
    w = synth.WORKLOADS["vit3d_small"]
    m = w["model"]
    lay = dict(synth.build_layout(w["docs"]))
    W = synth.make_weights(w)
    x = synth.make_tokens(w, lay)
    lay_gpu = dict(lay, pos=_positions(_dit().vit_positions, w["docs"]))
    wrong = dict(w, model=dict(m, qkv_interleaved=False))
    run = gu.run_forward(wrong, dumps=True, layout=lay_gpu, weights=W, x=x, t=0.0)
    assert run["status"] == 0 and np.isfinite(run["out"]).all()
    lay_orc = dict(lay, pos=_positions(oracle.vit_positions, w["docs"]))
    ref, dumps = oracle.forward(m, W, x, lay_orc, 0.0, dumps=True)
    assert forward_gates(x, run["dumps"], dumps, run["out"], ref)


@pytest.mark.slow
def test_vit_decoder_full_size_zero_residual_scales_is_final_layer_norm():
    """All 36 blocks at the full 8,192-token grid with zero residual scales: every block is the
    identity, so the output is the final LayerNorm of the input, checked on sampled rows."""
    gu = _gu()
    w = synth.WORKLOADS["vit3d_decoder"]
    m = w["model"]
    lay = dict(synth.build_layout(w["docs"]), pos=_positions(_dit().vit_positions, w["docs"]))
    W = synth.make_weights(w)
    for b in W["blocks"]:
        b["res1"] = np.zeros_like(b["res1"])
        b["res2"] = np.zeros_like(b["res2"])
    run = gu.run_forward(w, layout=lay, weights=W, t=0.0)
    assert run["status"] == 0
    rows = np.unique(np.concatenate([[0, lay["n_tokens"] - 1],
                                     (synth.uniform(400, "rows", 64) * lay["n_tokens"]).astype(np.int64)]))
    G = W["glob"]
    ref = oracle.layer_norm(run["x"][rows], m["norm_eps"], G["lnf_g"], G["lnf_b"])
    assert np.abs(run["out"][rows] - ref).max() <= 1e-5 * np.sqrt((ref ** 2).mean())
    run["handle"].close()
