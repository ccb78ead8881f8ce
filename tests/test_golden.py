"""Pins against values the pages print (tests/golden/, each file citing its passage)."""
import os

import synth

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _table(name):
    rows = {}
    for line in open(os.path.join(HERE, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            parts = line.split()
            rows[parts[0]] = parts[1:]
    return rows


def test_nvfp4_layout_matches_the_printed_checkpoint_shapes():
    """Two codes per byte and one E4M3 scale per 16 along K: the packed and scale shapes the pages
    print for the logical [21504, 5376] qkv weight, and the library's tile repack holds exactly the
    codes and scales."""
    t = _table("nvfp4_qkv_block0_shapes.txt")
    N, K = (int(v) for v in t["logical"][1:])
    assert [int(v) for v in t["weight"][1:]] == [N, K // 2]
    assert [int(v) for v in t["weight_scale"][1:]] == [N, K // 16]
    from video_audio_gen_gb300 import build, dit
    build.build()
    assert dit.nvfp4_packed_bytes(N, K) == N * (K // 2) + N * (K // 16)
    q, s, _ = synth.make_nvfp4(1, "shape", 256, 64)
    assert q.shape == (256, 64 // 2) and s.shape == (256, 64 // 16)


def test_vit3d_block_reading_matches_the_printed_manifest():
    """Twelve tensors per block (the four linears with biases, two RMS gains, two residual scales),
    the final LayerNorm's two, and the six surround tensors add up to the 440 the manifest lists."""
    t = _table("vit3d_decoder_manifest.txt")
    m = synth.VIT_MODEL
    shapes = synth.weight_shapes(m)
    assert m["n_blocks"] == int(t["blocks"][0]) and m["n_heads"] == int(t["heads"][0])
    assert m["head_dim"] == int(t["head_dim"][0]) and m["rope_base"] == float(t["rope_theta"][0])
    assert m["rotary_dim"] == float(t["rope_dim_ratio"][0]) * m["head_dim"]
    total = m["n_blocks"] * len(shapes["block"]) + len(shapes["glob"]) + int(t["surround"][0])
    assert len(shapes["block"]) == 12 and total == int(t["tensors"][0])


def test_audio_latent_width_matches_the_printed_width():
    t = _table("audio_latent_width.txt")
    c = int(t["audio_latent_channels"][0])
    assert synth.AUDIO_LATENT["channels"] == c == int(t["dec_in_proj"][0])
    assert synth.latent_widths()[1] == c  # audio pack: one token per latent frame, c features
