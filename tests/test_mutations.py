"""The gates discriminate: each plausible mistake, planted in the oracle's inputs on the CPU, fails the
gate the GPU path is held to, while the unmutated oracle and bf16-level noise pass.

Whole-forward gates (tests/parity.py) catch mistakes in the block structure.  They cannot catch RoPE
mistakes at these weight scales: with N(0, 0.02) weights the attention logits are ~0.1, the softmax is
nearly uniform and any rotation leaves the forward almost unchanged.  RoPE is therefore held to the
op-level gate of the QKV + RoPE kernel test (one bf16 rounding of q and k), where its mistakes fail."""
import numpy as np
import pytest

import oracle
import synth
from tests.parity import forward_gates

W0 = synth.WORKLOADS["tiny"]


@pytest.fixture(scope="module")
def base():
    lay = synth.build_layout(W0["docs"])
    W = synth.make_weights(W0)
    x = synth.make_tokens(W0, lay)
    oracle.set_threads(4)
    out, dumps = oracle.forward(W0["model"], W, x, lay, 0.5, dumps=True)
    return lay, W, x, out, dumps


def _copy(W):
    return dict(blocks=[{k: (v.copy() if v is not None else None) for k, v in b.items()} for b in W["blocks"]],
                glob={k: (v.copy() if v is not None else None) for k, v in W["glob"].items()})


def _run(W, x, lay, m=None):
    return oracle.forward(m or W0["model"], W, x, lay, 0.5, dumps=True)


def test_gates_pass_for_the_oracle_itself_and_for_bf16_level_noise(base):
    lay, W, x, out, dumps = base
    assert forward_gates(x, dumps, dumps, out, out) == []
    # perturb every block output by one bf16 rounding of its update: must still pass
    rng = np.random.default_rng(0)
    noisy = dumps.copy()
    prev = x.astype(np.float64)
    for l in range(len(dumps)):
        upd = dumps[l] - prev
        noisy[l] = prev + upd * (1 + rng.uniform(-2 ** -9, 2 ** -9, upd.shape))
        prev = dumps[l]
    assert forward_gates(x, noisy, dumps, out, out) == []


def _mutations():
    m = W0["model"]
    d, F, H, Dh = m["hidden"], m["ffn_hidden"], m["n_heads"], m["head_dim"]

    def swap_value_gate(W, lay):
        for b in W["blocks"]:
            b["w_in"] = np.concatenate([b["w_in"][F:], b["w_in"][:F]])
            b["b_in"] = np.concatenate([b["b_in"][F:], b["b_in"][:F]])
        return W, lay

    def swap_q_k(W, lay):
        for b in W["blocks"]:
            b["w_qkv"] = np.concatenate([b["w_qkv"][d:2 * d], b["w_qkv"][:d], b["w_qkv"][2 * d:]])
        return W, lay

    def drop_document_boundary(W, lay):
        lay = dict(lay, cu_seqlens=np.array([0, lay["n_tokens"]], dtype=np.int32),
                   doc_ids=np.zeros(lay["n_tokens"], dtype=np.int32), n_docs=1)
        return W, lay

    def wrong_modality_row(W, lay):
        return W, dict(lay, tags=(1 - lay["tags"]).astype(np.uint8))

    def ungated_residual(W, lay):
        for b in W["blocks"]:
            wa = b["w_ada"].reshape(2, 6, d, -1)
            ba = b["b_ada"].reshape(2, 6, d)
            for c in (2, 5):
                wa[:, c] = 0.0
                ba[:, c] = 1.0
        return W, lay

    return [swap_value_gate, swap_q_k, drop_document_boundary, wrong_modality_row, ungated_residual]


@pytest.mark.parametrize("mutate", _mutations(), ids=lambda f: f.__name__)
def test_planted_mistake_fails_the_gates(base, mutate):
    lay, W, x, out, dumps = base
    W2, lay2 = mutate(_copy(W), dict(lay))
    out2, dumps2 = _run(W2, x, lay2)
    assert forward_gates(x, dumps2, dumps, out2, out) != []


# ------------------------------------------------------------------------------------------------
# RoPE mistakes against the op-level gate of the QKV + RoPE kernel
# ------------------------------------------------------------------------------------------------

BF16_REL = 2.0 ** -8


def _qk_after_rope(m, lay, qk, pos=None, perm=None):
    cs, sn = oracle.rope_cos_sin(m, lay["pos"] if pos is None else pos)
    H, Dh = m["n_heads"], m["head_dim"]
    if perm is not None:  # rotate pairs (perm[j], perm[j + Dh/2]) instead of (j, j + Dh/2)
        idx = np.concatenate([h * Dh + perm for h in range(H)])
        inv = np.argsort(idx)
        return oracle.rope_apply(qk[:, idx], H, Dh, m["rotary_dim"], cs, sn)[:, inv]
    return oracle.rope_apply(qk, H, Dh, m["rotary_dim"], cs, sn)


def _rope_mutations():
    Dh = W0["model"]["head_dim"]
    inter = np.empty(Dh, dtype=np.int64)
    inter[:Dh // 2] = np.arange(0, Dh, 2)
    inter[Dh // 2:] = np.arange(1, Dh, 2)
    return {
        "interleaved_pairs": lambda m, lay, qk: _qk_after_rope(m, lay, qk, perm=inter),
        "wrong_direction": lambda m, lay, qk: _qk_after_rope(m, lay, qk, pos=-lay["pos"]),
        "audio_after_video": lambda m, lay, qk: _qk_after_rope(
            m, lay, qk, pos=lay["pos"] + np.outer(lay["tags"] == 1, [2.0, 0.0, 0.0])),
        "axes_swapped": lambda m, lay, qk: _qk_after_rope(m, lay, qk, pos=lay["pos"][:, [1, 0, 2]]),
    }


@pytest.mark.parametrize("name", list(_rope_mutations()))
def test_planted_rope_mistake_fails_the_qkv_op_gate(base, name):
    lay, W, x, out, dumps = base
    m = W0["model"]
    y = oracle.rms_norm(x, m["norm_eps"])
    qk = oracle.linear(y, W["blocks"][0]["w_qkv"][:m["hidden"]], None)
    ref = _qk_after_rope(m, lay, qk)
    mut = _rope_mutations()[name](m, lay, qk)
    tol = BF16_REL * np.abs(ref) + 1e-5
    assert np.any(np.abs(mut - ref) > tol)
    # and the unmutated rotation passes the same gate under one bf16 rounding
    assert np.all(np.abs(ref * (1 + 2 ** -9) - ref) <= tol)


# ------------------------------------------------------------------------------------------------
# per-modality timesteps and the latent I/O, against the gates they are held to
# ------------------------------------------------------------------------------------------------

def test_swapped_modality_timesteps_fail_the_forward_gates(base):
    lay, W, x, _, _ = base
    ref, rd = oracle.forward(W0["model"], W, x, lay, [0.8, 0.3], dumps=True)
    mut, md = oracle.forward(W0["model"], W, x, lay, [0.3, 0.8], dumps=True)
    assert forward_gates(x, md, rd, mut, ref) != []


def test_latent_rows_in_the_wrong_packed_places_fail_the_head_gate(base):
    """A row map that sends the r-th video token to another video row: the per-modality v gate
    (3e-3 of RMS) fails."""
    from tests.parity import GATE
    lay, W, _, _, _ = base
    widths = synth.latent_widths()
    io = synth.make_latent_io(5, W0["model"]["hidden"], widths)
    z = synth.make_latents(5, lay, widths)
    ref, _ = oracle.forward_latent(W0["model"], W, io, z, lay, [0.6, 0.2])
    perm = np.roll(np.arange(z[0].shape[0]), 7)
    mut, _ = oracle.forward_latent(W0["model"], W, io, [z[0][perm], z[1]], lay, [0.6, 0.2])
    mut_back = np.empty_like(mut[0])
    mut_back[perm] = mut[0]  # undo the permutation on the output rows: only the packed places differ
    rms = np.sqrt((ref[0] ** 2).mean())
    assert np.abs(mut_back - ref[0]).max() > GATE * rms


# ------------------------------------------------------------------------------------------------
# NVFP4 format mistakes against the NVFP4 GEMM's gate (fp32 accumulation bound, see test_gpu_ops)
# ------------------------------------------------------------------------------------------------

def _nvfp4_case():
    M, N, K = 16, 32, 128
    q, s, g = synth.make_nvfp4(90, "w", N, K)
    a = synth.normal(90, "a", (M, K), 1.0).astype(np.float16).astype(np.float64)
    ref = oracle.nvfp4_linear(a, q, s, g)
    bound = (K + 2) * 2.0 ** -23 * oracle.nvfp4_linear(np.abs(a), (q & 0x77).astype(np.uint8), s, g)
    return a, q, s, g, ref, bound


@pytest.mark.parametrize("mistake", ["nibbles_swapped", "scale_group_shifted", "global_divides", "scale_bias_6"])
def test_planted_nvfp4_mistake_fails_the_gemm_gate(mistake):
    a, q, s, g, ref, bound = _nvfp4_case()
    if mistake == "nibbles_swapped":       # odd k in the low nibble
        got = oracle.nvfp4_linear(a, ((q >> 4) | (q << 4)).astype(np.uint8), s, g)
    elif mistake == "scale_group_shifted":  # group index off by one along K
        got = oracle.nvfp4_linear(a, q, np.roll(s, 1, axis=1), g)
    elif mistake == "global_divides":       # code * scale / global
        got = oracle.nvfp4_linear(a, q, s, 1.0 / g)
    else:                                   # E4M3 decoded with exponent bias 6 instead of 7: every scale x2
        got = oracle.nvfp4_linear(a, q, s, g) * 2.0
    assert np.any(np.abs(got - ref) > bound)
    # the unmutated linear passes it under fp32-level noise
    assert np.all(np.abs(ref * (1 + 2.0 ** -24) - ref) <= bound + 1e-30)
