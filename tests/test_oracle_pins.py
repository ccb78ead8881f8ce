"""Pins for the CPU oracle, independent of the oracle itself.

Each test checks the oracle against something it does not compute: numpy.linspace, closed forms,
invariants of the mathematics, textbook special cases, library routines (numpy matmul / einsum),
and brute force by an independent numpy forward on 8-token inputs.
"""
import numpy as np
import pytest

import oracle
import synth
from tests import numpy_dit

# ---------------------------------------------------------------------------------------------
# small models used by brute force
# ---------------------------------------------------------------------------------------------

TINY_RMS = dict(n_blocks=2, hidden=16, n_heads=2, head_dim=8, ffn_hidden=24, norm="rms", norm_eps=1e-6,
                adaln=True, n_mod=2, t_dim=16, rope_axes=3, rope_dims=(2, 2, 4), rotary_dim=8,
                rope_base=10000.0, io_channels=0, dtype="fp32")
TINY_LN = dict(n_blocks=2, hidden=16, n_heads=2, head_dim=8, ffn_hidden=24, norm="ln", norm_eps=1e-5,
               adaln=False, n_mod=1, t_dim=16, rope_axes=1, rope_dims=(4, 0, 0), rotary_dim=4,
               rope_base=10000.0, io_channels=6, dtype="fp32")
DOCS8 = [dict(video=(1, 2, 2), audio=1), dict(video=(1, 1, 2), audio=1)]


def _workload(m, seed, docs, w_std=0.3, bias_std=0.2):
    return dict(model=m, seed=seed, docs=docs, t=0.3, w_std=w_std, bias_std=bias_std, x_std=1.0)


def _ln_params_random(W, seed):
    """Give LayerNorm gains/shifts non-trivial values so the affine path is exercised."""
    for l, b in enumerate(W["blocks"]):
        for n in ("ln1_g", "ln2_g"):
            b[n] = 1.0 + synth.normal(seed, f"{l}{n}", b[n].shape, 0.2)
        for n in ("ln1_b", "ln2_b"):
            b[n] = synth.normal(seed, f"{l}{n}", b[n].shape, 0.2)
    W["glob"]["lnf_g"] = 1.0 + synth.normal(seed, "lnf_g", W["glob"]["lnf_g"].shape, 0.2)
    W["glob"]["lnf_b"] = synth.normal(seed, "lnf_b", W["glob"]["lnf_b"].shape, 0.2)


# ---------------------------------------------------------------------------------------------
# fp64 grid: bit-exact against numpy.linspace(endpoint=False)
# ---------------------------------------------------------------------------------------------

PROBES = [(0.0, 3.0, 7), (0.1, 5.3, 17), (0.0, 8.0, 512), (0.0, 16.0, 1024), (0.0, 2.0, 32), (-1.7, 2.9, 33),
          (0.0, 1.0, 16), (3.3, 3.4, 100), (0.0, 86.0, 86), (1e-3, 7.0, 1000)]


@pytest.mark.parametrize("start,stop,n", PROBES)
def test_linspace_bit_exact_vs_numpy(start, stop, n):
    ref = np.linspace(start, stop, n, endpoint=False)
    assert np.array_equal(oracle.linspace(start, stop, n).view(np.uint64), ref.view(np.uint64))
    assert np.array_equal(synth.grid_axis(start, stop, n).view(np.uint64), ref.view(np.uint64))


def test_linspace_order_matters():
    """The pin discriminates: a different arithmetic order misses numpy on some probe."""
    miss = 0
    for start, stop, n in PROBES:
        alt = np.array([i * (stop - start) / n + start for i in range(n)])
        miss += int(not np.array_equal(alt, np.linspace(start, stop, n, endpoint=False)))
    assert miss > 0


SPAN_SETS = {
    "uniform": lambda n: synth.uniform(41, "spans", n, 0.0, 3.0),
    "one third": lambda n: np.full(n, 1.0 / 3.0),
    "steps of 1/17": lambda n: np.arange(n) / 17.0,
    "normal x 1e3": lambda n: synth.normal(42, "spans", (n,), 1e3).astype(np.float64) / 7.0,
}


@pytest.mark.parametrize("name", list(SPAN_SETS))
def test_span_sums_bit_exact_vs_numpy_and_python(name):
    """The pairwise span sum equals numpy's sum of a float64 array bit for bit, and the sequential
    one a Python left-to-right loop, from n = 0 through several recursion levels of the pairwise
    split."""
    for n in list(range(0, 300)) + [511, 512, 513, 1000, 1024, 1031, 4097]:
        x = SPAN_SETS[name](n)
        assert oracle.span_sum_pairwise(x) == float(np.sum(x)), n
        seq = 0.0
        for v in x:
            seq = seq + float(v)
        assert oracle.span_sum_sequential(x) == seq, n


@pytest.mark.parametrize("span", [1.0 / 3.0, 2.0 / 3.0, 0.3])
def test_span_sums_part_in_the_last_ulp_from_n_16(span):
    """[H3] "Correctness gates": the numpy-pairwise and the Python-sequential span sums diverge in
    the last ulp from n = 16.  For these spans they agree below 16 terms and part by one ulp at 16."""
    for n in range(1, 16):
        x = np.full(n, span)
        assert oracle.span_sum_pairwise(x) == oracle.span_sum_sequential(x), n
    x = np.full(16, span)
    a, b = oracle.span_sum_pairwise(x), oracle.span_sum_sequential(x)
    assert a != b and abs(a - b) == np.spacing(max(abs(a), abs(b)))


def test_layout_sizes_and_grid():
    expect = {"tiny": [96, 160], "video_audio_bf16": [8704, 8704], "long_doc_bf16": [33792],
              "denoise_loop": [17408, 9216], "music_fp32": [86, 86]}
    for name, sizes in expect.items():
        lay = synth.build_layout(synth.WORKLOADS[name]["docs"])
        assert list(np.diff(lay["cu_seqlens"])) == sizes
        assert lay["n_tokens"] == sum(sizes)
        assert oracle.check_layout(lay["cu_seqlens"], lay["doc_ids"], lay["tags"], lay["n_tokens"], 2) == 0
    lay = synth.build_layout(synth.WORKLOADS["tiny"]["docs"])
    # doc A: 96 video tokens on T2,H6,W8, w fastest; doc B: 128 video then 32 audio
    assert np.array_equal(lay["pos"][:96], np.array([(t, h, w) for t in range(2) for h in range(6)
                                                      for w in range(8)], dtype=np.float64))
    assert (lay["tags"][96:224] == 0).all() and (lay["tags"][224:] == 1).all()
    assert np.array_equal(lay["pos"][224:, 0], np.linspace(0, 2, 32, endpoint=False))
    assert (lay["pos"][224:, 1:] == 0).all()


def test_layout_check_rejects():
    lay = synth.build_layout(synth.WORKLOADS["tiny"]["docs"])
    cu, ids, tags, n = lay["cu_seqlens"], lay["doc_ids"], lay["tags"], lay["n_tokens"]
    assert oracle.check_layout(cu, ids, tags, n, 2) == 0
    bad = cu.copy(); bad[0] = 1
    assert oracle.check_layout(bad, ids, tags, n, 2) == 2
    bad = cu.copy(); bad[1] = 0
    assert oracle.check_layout(bad, ids, tags, n, 2) == 3
    assert oracle.check_layout(cu, ids, tags, n + 1, 2) == 4
    bad = ids.copy(); bad[95] = 1
    assert oracle.check_layout(cu, bad, tags, n, 2) == 5
    bad = tags.copy(); bad[3] = 2
    assert oracle.check_layout(cu, ids, bad, n, 2) == 6
    assert oracle.count_q_tiles(np.array([0, 96, 256])) == 1 + 2
    assert oracle.count_q_tiles(np.array([0, 8704, 17408])) == 2 * 68


# ---------------------------------------------------------------------------------------------
# timestep embedding, AdaLN, norms
# ---------------------------------------------------------------------------------------------

def test_timestep_embedding_closed_form_at_zero():
    e = oracle.timestep_embedding(0.0, 256)
    assert (e[:128] == 1.0).all() and (e[128:] == 0.0).all()


def test_timestep_embedding_invariants_and_quarter_turn():
    """Closed forms and invariants of the sinusoid [cos(1000 t f_k) | sin(1000 t f_k)] at t != 0:
    each (cos, sin) pair lies on the unit circle; f_0 = 1 puts the first pair a quarter and a half
    turn round at t = pi / 2000 and pi / 1000; the recovered angles fall geometrically by
    10000^(-1 / half) from 1000 t (so a swapped cos/sin, a missing 1000 or an endpoint-style
    exponent k / (half - 1) each fail)."""
    half = 128
    for t in (0.37, 0.9731, 1.0):
        e = oracle.timestep_embedding(t, 2 * half)
        assert np.allclose(e[:half] ** 2 + e[half:] ** 2, 1.0, rtol=0, atol=1e-15)
    e = oracle.timestep_embedding(np.pi / 2000, 2 * half)
    assert abs(e[0]) < 1e-15 and abs(e[half] - 1.0) < 1e-15
    e = oracle.timestep_embedding(np.pi / 1000, 2 * half)
    assert abs(e[0] + 1.0) < 1e-15 and abs(e[half]) < 1e-15
    t = 1e-3  # every angle below pi: atan2 recovers it without wrapping
    e = oracle.timestep_embedding(t, 2 * half)
    ang = np.arctan2(e[half:], e[:half])
    assert abs(ang[0] - 1000 * t) < 1e-14
    ratio = ang[1:] / ang[:-1]
    assert np.allclose(ratio, 10000.0 ** (-1.0 / half), rtol=1e-12, atol=0)


def test_adaln_is_matvec_of_silu_embedding():
    w = _workload(TINY_RMS, 5, DOCS8)
    W = synth.make_weights(w)
    mod, modf = oracle.adaln(TINY_RMS, W, 0.3)
    e = oracle.timestep_embedding(0.3, 16)
    se = e / (1 + np.exp(-e))
    for l in range(2):
        ref = W["blocks"][l]["w_ada"].astype(np.float64) @ se + W["blocks"][l]["b_ada"]
        assert np.allclose(mod[l].reshape(-1), ref, rtol=0, atol=1e-14)
    ref = W["glob"]["w_ada_final"].astype(np.float64) @ se + W["glob"]["b_ada_final"]
    assert np.allclose(modf.reshape(-1), ref, rtol=0, atol=1e-14)


def test_rms_norm_closed_form():
    x = synth.normal(7, "rms", (5, 64), 3.0).astype(np.float64)
    y = oracle.rms_norm(x, 1e-6)
    m = (x * x).mean(axis=1)
    assert np.allclose((y * y).mean(axis=1), m / (m + 1e-6), rtol=1e-14, atol=0)
    c = np.full((1, 32), 0.25)
    assert np.allclose(oracle.rms_norm(c, 1e-6), 0.25 / np.sqrt(0.0625 + 1e-6), rtol=1e-15)
    # direction is preserved
    assert np.allclose(y / np.linalg.norm(y, axis=1, keepdims=True), x / np.linalg.norm(x, axis=1, keepdims=True))


def test_layer_norm_closed_form():
    x = synth.normal(7, "ln", (5, 64), 3.0).astype(np.float64) + 4.0
    y = oracle.layer_norm(x, 1e-5)
    v = x.var(axis=1)
    assert np.allclose(y.mean(axis=1), 0.0, atol=1e-14)
    assert np.allclose((y * y).mean(axis=1), v / (v + 1e-5), rtol=1e-13)
    g = np.full(64, 2.0, dtype=np.float32)
    b = np.full(64, 3.0, dtype=np.float32)
    y2 = oracle.layer_norm(x, 1e-5, g, b)
    assert np.allclose(y2, 2 * y + 3, rtol=1e-15, atol=1e-15)


def test_modulate_zero_is_bare_norm_bit_exact():
    x = synth.normal(8, "m", (6, 32), 1.0)
    nrm = oracle.rms_norm(x, 1e-6)
    tags = np.array([0, 1, 1, 0, 1, 0], dtype=np.uint8)
    z = np.zeros((2, 32))
    assert np.array_equal(oracle.modulate(nrm, tags, z, z), nrm)
    sh = np.stack([np.full(32, 1.0), np.full(32, -2.0)])
    sc = np.stack([np.full(32, 0.5), np.full(32, 1.0)])
    y = oracle.modulate(nrm, tags, sh, sc)
    assert np.allclose(y[0], nrm[0] * 1.5 + 1.0) and np.allclose(y[1], nrm[1] * 2.0 - 2.0)


# ---------------------------------------------------------------------------------------------
# RoPE
# ---------------------------------------------------------------------------------------------

M3AX = dict(TINY_RMS, rope_dims=(2, 2, 4), rotary_dim=8, head_dim=8)


def test_rope_identity_at_origin_bit_exact():
    pos = np.zeros((3, 3))
    cs, sn = oracle.rope_cos_sin(M3AX, pos)
    x = synth.normal(9, "x", (3, 16), 1.0)
    assert np.array_equal(oracle.rope_apply(x, 2, 8, 8, cs, sn), x.astype(np.float64))


def test_rope_norm_preserving_and_rotation_matrix():
    lay = synth.build_layout([dict(video=(3, 4, 5), audio=7)])
    cs, sn = oracle.rope_cos_sin(M3AX, lay["pos"])
    x = synth.normal(9, "y", (lay["n_tokens"], 16), 1.0).astype(np.float64)
    y = oracle.rope_apply(x, 2, 8, 8, cs, sn)
    for h in range(2):
        a, b = np.linalg.norm(x[:, 8 * h:8 * h + 8], axis=1), np.linalg.norm(y[:, 8 * h:8 * h + 8], axis=1)
        assert np.allclose(a, b, rtol=1e-14)
    # one pair = a 2-D rotation by +theta (textbook [[c, -s], [s, c]])
    th = 0.7
    R = np.array([[np.cos(th), -np.sin(th)], [np.sin(th), np.cos(th)]])
    v = np.array([[0.3, -1.1]])
    out = oracle.rope_apply(v, 1, 2, 2, np.array([[np.cos(th)]]), np.array([[np.sin(th)]]))
    assert np.allclose(out[0], R @ v[0], rtol=0, atol=1e-15)


def test_rope_pairs_are_rotate_half():
    """A unit vector in dim j moves only within the pair (j, j + R/2)."""
    pos = np.array([[1.0, 2.0, 3.0]])
    cs, sn = oracle.rope_cos_sin(M3AX, pos)
    for j in range(8):
        e = np.zeros((1, 8)); e[0, j] = 1.0
        y = oracle.rope_apply(e, 1, 8, 8, cs, sn)
        partner = j + 4 if j < 4 else j - 4
        nz = set(np.nonzero(np.abs(y[0]) > 1e-15)[0].tolist())
        assert nz <= {j, partner} and partner in nz


def test_rope_axis_blocks_concatenate_t_h_w():
    """Position (p,0,0) turns only the t block; (0,p,0) only h; (0,0,p) only w.  Pair 0 of each block
    has inverse frequency exactly 1, so its angle is the position itself."""
    m = dict(TINY_RMS, rope_dims=(4, 6, 6), rotary_dim=16, head_dim=16)
    blocks = [(0, 2), (2, 5), (5, 8)]
    for a, (lo, hi) in enumerate(blocks):
        pos = np.zeros((1, 3)); pos[0, a] = 2.5
        cs, sn = oracle.rope_cos_sin(m, pos)
        moved = np.nonzero(cs[0] != 1.0)[0]
        assert lo in moved and all(lo <= j < hi for j in moved)
        assert cs[0, lo] == np.cos(2.5) and sn[0, lo] == np.sin(2.5)


def test_rope_relative_position_invariance():
    """Shifting every position of a document by an integer leaves its attention output unchanged."""
    m = TINY_RMS
    lay = synth.build_layout([dict(video=(2, 2, 3), audio=3)])
    n = lay["n_tokens"]
    q, k, v = (synth.normal(10, nm, (n, 16), 1.0).astype(np.float64) for nm in "qkv")
    outs = []
    for shift in (0.0, 5.0):
        pos = lay["pos"] + shift
        cs, sn = oracle.rope_cos_sin(m, pos)
        qr, kr = oracle.rope_apply(q, 2, 8, 8, cs, sn), oracle.rope_apply(k, 2, 8, 8, cs, sn)
        outs.append(oracle.attention(qr, kr, v, lay["cu_seqlens"], 2, 8))
    assert np.allclose(outs[0], outs[1], rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------------------------
# linear map, 1x1 conv, gated FFN
# ---------------------------------------------------------------------------------------------

def test_linear_matches_numpy_matmul():
    x = synth.normal(11, "x", (7, 33), 1.0).astype(np.float64)
    W = synth.normal(11, "W", (19, 33), 0.5)
    b = synth.normal(11, "b", (19,), 0.5)
    assert np.allclose(oracle.linear(x, W, b), x @ W.astype(np.float64).T + b, rtol=1e-13, atol=1e-13)


def test_conv1x1_equals_matmulbt_on_transposed_activation():
    x = synth.normal(12, "x", (6, 9), 1.0).astype(np.float64)  # [ci, T]
    W = synth.normal(12, "W", (5, 6), 0.5)
    b = synth.normal(12, "b", (5,), 0.5)
    direct = oracle.conv1x1(x, W, b)
    via_gemm = oracle.linear(x.T, W, b).T
    assert np.allclose(direct, via_gemm, rtol=1e-14, atol=1e-14)


def test_swiglu_value_first_gate_second():
    uv = np.array([[1.0, 2.0]])
    assert np.isclose(oracle.swiglu(uv)[0, 0], 1.0 * 2.0 / (1.0 + np.exp(-2.0)), rtol=1e-15)
    uv = np.array([[3.0, 0.0]])
    assert oracle.swiglu(uv)[0, 0] == 0.0


# ---------------------------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------------------------

def test_attention_identical_keys_give_mean_of_v():
    lay = synth.build_layout([dict(video=(1, 3, 4)), dict(video=(1, 1, 5))])
    n = lay["n_tokens"]
    q = synth.normal(13, "q", (n, 16), 1.0)
    k = np.tile(synth.normal(13, "k", (1, 16), 1.0), (n, 1))
    v = synth.normal(13, "v", (n, 16), 1.0).astype(np.float64)
    o = oracle.attention(q, k, v, lay["cu_seqlens"], 2, 8)
    cu = lay["cu_seqlens"]
    for j in range(2):
        assert np.allclose(o[cu[j]:cu[j + 1]], v[cu[j]:cu[j + 1]].mean(axis=0), rtol=0, atol=1e-14)


def test_attention_block_diagonal_equals_docs_alone_and_one_token_doc():
    lay = synth.build_layout([dict(video=(1, 3, 4), audio=2), dict(video=(1, 1, 1)), dict(video=(1, 2, 3))])
    n, cu = lay["n_tokens"], lay["cu_seqlens"]
    q, k, v = (synth.normal(14, nm, (n, 16), 1.0).astype(np.float64) for nm in "qkv")
    o = oracle.attention(q, k, v, cu, 2, 8)
    for j in range(3):
        a, b = cu[j], cu[j + 1]
        alone = oracle.attention(q[a:b], k[a:b], v[a:b], np.array([0, b - a]), 2, 8)
        assert np.array_equal(o[a:b], alone)
    assert np.allclose(o[cu[1]], v[cu[1]], rtol=0, atol=1e-15)  # a 1-token document returns its v


def test_attention_matches_numpy_softmax_and_rows():
    lay = synth.build_layout([dict(video=(1, 3, 4), audio=2), dict(video=(1, 2, 3))])
    n, cu = lay["n_tokens"], lay["cu_seqlens"]
    q, k, v = (synth.normal(15, nm, (n, 16), 1.0).astype(np.float64) for nm in "qkv")
    o = oracle.attention(q, k, v, cu, 2, 8)
    assert np.allclose(o, numpy_dit.attention(q, k, v, cu, 2, 8), rtol=0, atol=1e-13)
    rows = np.array([0, 5, 13, n - 1])
    assert np.array_equal(oracle.attention_rows(q, k, v, cu, 2, 8, rows), o[rows])


def test_attention_permutation_equivariance():
    lay = synth.build_layout([dict(video=(1, 3, 4))])
    n, cu = lay["n_tokens"], lay["cu_seqlens"]
    q, k, v = (synth.normal(16, nm, (n, 16), 1.0).astype(np.float64) for nm in "qkv")
    perm = np.random.default_rng(0).permutation(n)
    o = oracle.attention(q, k, v, cu, 2, 8)
    op = oracle.attention(q[perm], k[perm], v[perm], cu, 2, 8)
    assert np.allclose(op, o[perm], rtol=0, atol=1e-14)


# ---------------------------------------------------------------------------------------------
# Euler step (fp32, exact order)
# ---------------------------------------------------------------------------------------------

def _numpy_euler(x, v, s, sn):
    s, sn = np.float32(s), np.float32(sn)
    x0 = x - s * v
    return x0 + (sn * (x - x0)) / s


def test_euler_bit_exact_vs_numpy_float32():
    x = synth.normal(17, "x", (4099,), 1.0)
    v = synth.normal(17, "v", (4099,), 1.0)
    sig = synth.sigmas(50)
    for i in (0, 1, 17, 48, 49):
        got = oracle.euler_step(x, v, sig[i], sig[i + 1])
        ref = _numpy_euler(x, v, sig[i], sig[i + 1])
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), i


def test_euler_last_step_lands_on_x0_and_constant_velocity_telescopes():
    x = synth.normal(18, "x", (1000,), 1.0)
    v = synth.normal(18, "v", (1000,), 1.0)
    got = oracle.euler_step(x, v, np.float32(0.02), np.float32(0.0))
    assert np.array_equal(got, x - np.float32(0.02) * v)
    sig = synth.sigmas(50)
    assert sig[0] == 1.0 and sig[50] == 0.0 and sig[25] == np.float32(0.5)
    z = x.copy()
    for i in range(50):
        z = oracle.euler_step(z, v, sig[i], sig[i + 1])
    assert np.allclose(z, x - v, rtol=0, atol=2e-5)


# ---------------------------------------------------------------------------------------------
# whole forward: brute force on 8 tokens, invariants
# ---------------------------------------------------------------------------------------------

def test_forward_brute_force_rms_adaln():
    w = _workload(TINY_RMS, 21, DOCS8)
    lay = synth.build_layout(DOCS8)
    assert lay["n_tokens"] == 8 and lay["tags"].tolist().count(1) == 2
    W = synth.make_weights(w, bf16=False)
    x = synth.make_tokens(w, lay)
    out, _ = oracle.forward(TINY_RMS, W, x, lay, 0.3)
    ref = numpy_dit.forward(TINY_RMS, W, x, lay, 0.3)
    assert np.abs(out - ref).max() <= 1e-12 * np.abs(ref).max()


def test_forward_brute_force_layernorm_partial_rotary_conv():
    w = _workload(TINY_LN, 22, [dict(frames=5), dict(frames=3)])
    lay = synth.build_layout(w["docs"])
    W = synth.make_weights(w, bf16=False)
    _ln_params_random(W, 22)
    x = synth.make_tokens(w, lay)
    out, _ = oracle.forward(TINY_LN, W, x, lay, 0.0)
    ref = numpy_dit.forward(TINY_LN, W, x, lay, 0.0)
    assert out.shape == (6 * 8,)
    assert np.abs(out - ref).max() <= 1e-12 * np.abs(ref).max()


def test_forward_gate_zero_block_is_identity_bit_exact():
    w = _workload(TINY_RMS, 23, DOCS8)
    lay = synth.build_layout(DOCS8)
    W = synth.make_weights(w, bf16=False)
    d = TINY_RMS["hidden"]
    for b in W["blocks"]:
        wa = b["w_ada"].reshape(2, 6, d, -1)
        wa[:, 2] = 0.0; wa[:, 5] = 0.0
        ba = b["b_ada"].reshape(2, 6, d)
        ba[:, 2] = 0.0; ba[:, 5] = 0.0
    x = synth.make_tokens(w, lay)
    _, dumps = oracle.forward(TINY_RMS, W, x, lay, 0.3, dumps=True)
    assert np.array_equal(dumps[0], x.astype(np.float64)) and np.array_equal(dumps[1], x.astype(np.float64))


def test_forward_modality_swap_symmetry():
    """Swapping every tag together with the two modalities' AdaLN rows gives the same result."""
    w = _workload(TINY_RMS, 24, DOCS8)
    lay = synth.build_layout(DOCS8)
    W = synth.make_weights(w, bf16=False)
    x = synth.make_tokens(w, lay)
    out, _ = oracle.forward(TINY_RMS, W, x, lay, 0.3)
    d = TINY_RMS["hidden"]
    for b in W["blocks"]:
        b["w_ada"] = b["w_ada"].reshape(2, -1)[::-1].reshape(b["w_ada"].shape).copy()
        b["b_ada"] = b["b_ada"].reshape(2, -1)[::-1].reshape(-1).copy()
    W["glob"]["w_ada_final"] = W["glob"]["w_ada_final"].reshape(2, -1)[::-1].reshape(2 * 2 * d, -1).copy()
    W["glob"]["b_ada_final"] = W["glob"]["b_ada_final"].reshape(2, -1)[::-1].reshape(-1).copy()
    lay2 = dict(lay, tags=(1 - lay["tags"]).astype(np.uint8))
    out2, _ = oracle.forward(TINY_RMS, W, x, lay2, 0.3)
    assert np.array_equal(out, out2)


def test_block_rows_equals_the_whole_block_on_its_rows():
    """The teacher-forcing block (the keys and values of whole documents, everything else on the
    sampled rows only) against the oracle's whole block: every sampled row agrees to rounding.
    Rows: document ends, 128-row tile edges, a 1-token document, audio rows; non-zero biases."""
    w = synth.WORKLOADS["ragged"]
    m = dict(w["model"], n_blocks=1)
    wl = dict(w, model=m)
    lay = synth.build_layout(w["docs"])
    W = synth.make_weights(wl)
    x = synth.make_tokens(wl, lay).astype(np.float64) * 1.5
    mod, _ = oracle.adaln(m, W, 0.37)
    cs, sn = oracle.rope_cos_sin(m, lay["pos"])
    oracle.set_threads(4)
    full = oracle.block_forward(m, W, 0, mod[0], x, lay, cs, sn)
    cu = lay["cu_seqlens"]
    rows = np.unique([0, 1, int(cu[1]) - 1, int(cu[1]), 127, 128, 129, int(cu[2]), int(cu[3]) - 1,
                      int(cu[3]), 300, lay["n_tokens"] - 1] + list(np.nonzero(lay["tags"] == 1)[0][::9]))
    got = oracle.block_rows(m, W, 0, mod[0], x, lay, rows)
    # rows of only some documents: the others' keys are not needed
    one = oracle.block_rows(m, W, 0, mod[0], x, lay, [int(cu[3]) + 5])
    oracle.set_threads(1)
    scale = np.abs(full[rows]).max()
    assert np.abs(got - full[rows]).max() <= 1e-12 * scale
    assert np.abs(one[0] - full[int(cu[3]) + 5]).max() <= 1e-12 * scale
    # and the block did move these rows (the comparison is not of the residual alone)
    assert np.abs(full[rows] - x[rows]).max() > 1e-3


def test_block_rows_reads_only_its_own_document():
    """Changing another document's inputs leaves a sampled row's block output unchanged (bit for bit):
    the keys and values it attends over are its own document's."""
    w = synth.WORKLOADS["ragged"]
    m = dict(w["model"], n_blocks=1)
    wl = dict(w, model=m)
    lay = synth.build_layout(w["docs"])
    W = synth.make_weights(wl)
    x = synth.make_tokens(wl, lay).astype(np.float64)
    mod, _ = oracle.adaln(m, W, 0.37)
    cu = lay["cu_seqlens"]
    r = [int(cu[1]) + 3]
    a = oracle.block_rows(m, W, 0, mod[0], x, lay, r)
    x2 = x.copy()
    x2[cu[3]:cu[4]] += 1.0
    b = oracle.block_rows(m, W, 0, mod[0], x2, lay, r)
    assert np.array_equal(a, b)


def test_forward_thread_count_does_not_change_bits():
    w = synth.WORKLOADS["ragged"]
    w = dict(w, model=dict(w["model"], n_blocks=1))
    lay = synth.build_layout(w["docs"][:2])
    W = synth.make_weights(w)
    x = synth.make_tokens(w, lay)
    oracle.set_threads(1)
    a, _ = oracle.forward(w["model"], W, x, lay, 0.37)
    oracle.set_threads(4)
    b, _ = oracle.forward(w["model"], W, x, lay, 0.37)
    oracle.set_threads(1)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------------------------------------
# per-modality sigma schedules ([H3] "Milestone: the whole t2va path composes end to end": video
# shift 12, audio 3): the time shift, per-modality AdaLN timesteps, the tagged Euler step
# ---------------------------------------------------------------------------------------------

def test_time_shift_closed_forms_and_group_law():
    sig = np.linspace(0.0, 1.0, 41)
    for s in (1.0, 3.0, 12.0):
        assert oracle.time_shift(0.0, s) == 0.0 and oracle.time_shift(1.0, s) == 1.0
    assert all(oracle.time_shift(float(x), 1.0) == float(x) for x in sig)  # shift 1 is the identity
    assert oracle.time_shift(0.5, 3.0) == 0.75
    assert abs(oracle.time_shift(0.5, 12.0) - 12.0 / 13.0) <= 1e-16
    for s in (3.0, 12.0):  # increasing in sigma, and above the identity for s > 1
        v = [oracle.time_shift(float(x), s) for x in sig]
        assert all(b > a for a, b in zip(v, v[1:]))
        assert all(vi >= float(x) for vi, x in zip(v, sig))
    # the shifts form a group under composition: shift(shift(sigma, a), b) = shift(sigma, a b)
    for x in sig:
        assert abs(oracle.time_shift(oracle.time_shift(float(x), 3.0), 4.0) - oracle.time_shift(float(x), 12.0)) <= 1e-15


def test_shifted_schedule_is_the_base_schedule_rounded_once():
    base = synth.sigmas(50)
    sv = oracle.sigmas_shifted(base, 12.0)
    assert sv.dtype == np.float32 and sv[0] == 1.0 and sv[-1] == 0.0
    assert np.array_equal(sv, np.float32([12.0 * float(b) / (1.0 + 11.0 * float(b)) for b in base]))


def test_adaln_per_modality_rows_come_from_their_own_timestep():
    w = _workload(TINY_RMS, 23, DOCS8)
    W = synth.make_weights(w, bf16=False)
    mod2, modf2 = oracle.adaln(TINY_RMS, W, [0.3, 0.8])
    modv, modfv = oracle.adaln(TINY_RMS, W, 0.3)
    moda, modfa = oracle.adaln(TINY_RMS, W, 0.8)
    assert np.array_equal(mod2[:, 0], modv[:, 0]) and np.array_equal(mod2[:, 1], moda[:, 1])
    assert np.array_equal(modf2[0], modfv[0]) and np.array_equal(modf2[1], modfa[1])
    eq, eqf = oracle.adaln(TINY_RMS, W, [0.3, 0.3])
    assert np.array_equal(eq, modv) and np.array_equal(eqf, modfv)


def test_euler_tagged_is_the_scalar_step_row_by_row():
    x = synth.normal(24, "x", (9, 16), 1.0)
    v = synth.normal(24, "v", (9, 16), 1.0)
    tags = np.array([0, 1, 1, 0, 0, 1, 0, 1, 0], dtype=np.uint8)
    st, sn = np.float32([0.9, 0.7]), np.float32([0.85, 0.6])
    got = oracle.euler_step_tagged(x, v, tags, st, sn)
    for r in range(9):
        assert np.array_equal(got[r], oracle.euler_step(x[r], v[r], st[tags[r]], sn[tags[r]]))
    same = oracle.euler_step_tagged(x, v, tags, np.float32([0.9, 0.9]), np.float32([0.85, 0.85]))
    assert np.array_equal(same, oracle.euler_step(x, v, 0.9, 0.85))


def test_forward_per_modality_timesteps_brute_force():
    w = _workload(TINY_RMS, 25, DOCS8)
    lay = synth.build_layout(DOCS8)
    W = synth.make_weights(w, bf16=False)
    x = synth.make_tokens(w, lay)
    out, _ = oracle.forward(TINY_RMS, W, x, lay, [0.3, 0.8])
    ref = numpy_dit.forward(TINY_RMS, W, x, lay, [0.3, 0.8])
    assert np.abs(out - ref).max() <= 1e-12 * np.abs(ref).max()
    one, _ = oracle.forward(TINY_RMS, W, x, lay, 0.3)
    same, _ = oracle.forward(TINY_RMS, W, x, lay, [0.3, 0.3])
    assert np.array_equal(one, same)
    assert np.abs(out - one).max() > 1e-3 * np.abs(one).max()  # the audio rows really changed


# ---------------------------------------------------------------------------------------------
# latent <-> token packing and the fp32 islands around the block stack
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("C,T,H,W,pt,ph,pw", [(3, 2, 3, 2, 2, 2, 2), (5, 3, 2, 4, 1, 2, 3), (2, 1, 1, 1, 1, 1, 1),
                                              (4, 2, 5, 3, 1, 1, 1)])
def test_patchify_is_the_reshape_transpose(C, T, H, W, pt, ph, pw):
    """numpy's view of the same map: split each axis into (grid, patch), move the grid axes out front,
    flatten the patch in (c, a, b, e) order."""
    lat = synth.normal(30, "lat", (C, T * pt, H * ph, W * pw), 1.0)
    want = lat.reshape(C, T, pt, H, ph, W, pw).transpose(1, 3, 5, 0, 2, 4, 6).reshape(T * H * W, C * pt * ph * pw)
    got = oracle.patchify(lat, pt, ph, pw)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_unpatchify_inverts_patchify_and_both_are_permutations():
    C, T, H, W, pt, ph, pw = 3, 2, 4, 3, 1, 2, 2
    n = C * T * pt * H * ph * W * pw
    lat = np.arange(n, dtype=np.float32).reshape(C, T * pt, H * ph, W * pw)
    tok = oracle.patchify(lat, pt, ph, pw)
    assert np.array_equal(np.sort(tok.reshape(-1)), np.arange(n, dtype=np.float32))
    assert np.array_equal(oracle.unpatchify(tok, C, T, H, W, pt, ph, pw), lat)
    tok2 = synth.normal(31, "tok", tok.shape, 1.0)
    back = oracle.patchify(oracle.unpatchify(tok2, C, T, H, W, pt, ph, pw), pt, ph, pw)
    assert np.array_equal(back.view(np.uint32), tok2.view(np.uint32))
    # token (t, h, w) holds the patch whose corner is (t*pt, h*ph, w*pw)
    t, h, w = 1, 2, 1
    r = (t * H + h) * W + w
    assert tok[r, 0] == lat[0, t * pt, h * ph, w * pw]


def test_audio_pack_is_the_transpose():
    lat = synth.normal(32, "alat", (32, 37), 1.0)
    tok = oracle.audio_pack(lat)
    assert np.array_equal(tok, lat.T)
    assert np.array_equal(oracle.audio_unpack(tok), lat)


def test_patch_projection_is_a_strided_conv3d():
    """Kernel == stride: a direct Conv3d loop equals the linear map on the patchified latent with the
    conv weight flattened as [d, C*pt*ph*pw]."""
    C, T, H, W, pt, ph, pw, d = 3, 2, 2, 3, 1, 2, 2, 5
    lat = synth.normal(33, "lat", (C, T * pt, H * ph, W * pw), 1.0)
    Wc = synth.normal(33, "w", (d, C, pt, ph, pw), 0.5)
    b = synth.normal(33, "b", (d,), 0.5)
    conv = np.zeros((d, T, H, W))
    for o in range(d):
        for t in range(T):
            for h in range(H):
                for w in range(W):
                    acc = float(b[o])
                    for c in range(C):
                        for a in range(pt):
                            for bb in range(ph):
                                for e in range(pw):
                                    acc += float(Wc[o, c, a, bb, e]) * float(lat[c, t * pt + a, h * ph + bb, w * pw + e])
                    conv[o, t, h, w] = acc
    got = oracle.linear(oracle.patchify(lat, pt, ph, pw), Wc.reshape(d, -1), b)
    assert np.abs(got - conv.reshape(d, -1).T).max() <= 1e-13


def _latent_io(seed, d, widths, std=0.3):
    return dict(w_patch=[synth.normal(seed, f"wp{m}", (d, k), std) for m, k in enumerate(widths)],
                b_patch=[synth.normal(seed, f"bp{m}", (d,), std) for m in range(len(widths))],
                w_head=[synth.normal(seed, f"wh{m}", (k, d), std) for m, k in enumerate(widths)],
                b_head=[synth.normal(seed, f"bh{m}", (k,), std) for m, k in enumerate(widths)])


def test_forward_latent_brute_force():
    """Per-modality patch projection into that modality's packed rows, the forward, per-modality
    heads: against numpy matmuls around the independent numpy forward on 8 tokens."""
    w = _workload(TINY_RMS, 34, DOCS8)
    lay = synth.build_layout(DOCS8)
    W = synth.make_weights(w, bf16=False)
    widths = [12, 5]
    io = _latent_io(34, TINY_RMS["hidden"], widths)
    rows = [np.nonzero(lay["tags"] == m)[0] for m in range(2)]
    z = [synth.normal(34, f"z{m}", (len(rows[m]), widths[m]), 1.0) for m in range(2)]
    vs, _ = oracle.forward_latent(TINY_RMS, W, io, z, lay, [0.7, 0.2])
    f64 = lambda a: np.asarray(a, dtype=np.float64)
    x = np.zeros((lay["n_tokens"], TINY_RMS["hidden"]))
    for m in range(2):
        x[rows[m]] = f64(z[m]) @ f64(io["w_patch"][m]).T + f64(io["b_patch"][m])
    out = numpy_dit.forward(TINY_RMS, W, x, lay, [0.7, 0.2])
    for m in range(2):
        ref = out[rows[m]] @ f64(io["w_head"][m]).T + f64(io["b_head"][m])
        assert vs[m].shape == (len(rows[m]), widths[m])
        assert np.abs(vs[m] - ref).max() <= 1e-12 * np.abs(ref).max()


def test_forward_latent_with_identity_islands_is_the_forward():
    """Width d, identity projections, zero biases: the latent forward is the plain forward row by row."""
    w = _workload(TINY_RMS, 35, DOCS8)
    lay = synth.build_layout(DOCS8)
    W = synth.make_weights(w, bf16=False)
    d = TINY_RMS["hidden"]
    x = synth.make_tokens(w, lay)
    eye = np.eye(d, dtype=np.float32)
    io = dict(w_patch=[eye, eye], b_patch=[None, None], w_head=[eye, eye], b_head=[None, None])
    rows = [np.nonzero(lay["tags"] == m)[0] for m in range(2)]
    vs, _ = oracle.forward_latent(TINY_RMS, W, io, [x[rows[0]], x[rows[1]]], lay, [0.4, 0.9])
    out, _ = oracle.forward(TINY_RMS, W, x, lay, [0.4, 0.9])
    for m in range(2):
        assert np.array_equal(vs[m], out[rows[m]])


def test_forward_latent_rejects_row_counts_that_disagree_with_tags():
    w = _workload(TINY_RMS, 36, DOCS8)
    lay = synth.build_layout(DOCS8)
    W = synth.make_weights(w, bf16=False)
    io = _latent_io(36, TINY_RMS["hidden"], [4, 4])
    z = [synth.normal(36, "z0", (5, 4), 1.0), synth.normal(36, "z1", (3, 4), 1.0)]  # tags say 6 and 2
    with pytest.raises(ValueError, match="code 8"):
        oracle.forward_latent(TINY_RMS, W, io, z, lay, 0.5)


# ---------------------------------------------------------------------------------------------
# NVFP4 weights
# ---------------------------------------------------------------------------------------------

def test_e2m1_decodes_to_the_fp4_grid():
    """E2M1: 1 sign, 2 exponent bits (bias 1), 1 mantissa bit; exponent 0 subnormal.  The eight
    magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6 and the high bit is the sign."""
    v = oracle.e2m1_decode(np.arange(16))
    assert list(v[:8]) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert np.array_equal(v[8:], -v[:8]) and np.signbit(v[8])


def test_e4m3_decodes_like_torch_float8_e4m3fn():
    torch = pytest.importorskip("torch")
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = oracle.e4m3_decode(np.arange(256))
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[0x08] == 2.0 ** -6 and got[0x01] == 2.0 ** -9 and got[0x38] == 1.0


def test_nvfp4_linear_against_numpy_dequantisation():
    torch = pytest.importorskip("torch")
    M, N, K = 5, 7, 64
    q, s, g = synth.make_nvfp4(60, "w", N, K)
    x = synth.normal(60, "x", (M, K), 1.0)
    b = synth.normal(60, "b", (N,), 0.1)
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    codes = np.empty((N, K), dtype=np.int64)
    codes[:, 0::2] = q & 15
    codes[:, 1::2] = q >> 4
    fp4 = np.where(codes >= 8, -1.0, 1.0) * grid[codes & 7]
    sc = torch.from_numpy(s.copy()).view(torch.float8_e4m3fn).double().numpy()
    W = fp4 * np.repeat(sc, 16, axis=1) * np.float64(np.float32(g))
    ref = x.astype(np.float64) @ W.T + b
    got = oracle.nvfp4_linear(x, q, s, g, b)
    assert np.abs(got - ref).max() <= 1e-13 * np.abs(ref).max()


def test_nvfp4_even_k_sits_in_the_low_nibble():
    """A weight whose only nonzero code is the high nibble of byte 0 reads x[:, 1]."""
    K = 32
    q = np.zeros((1, K // 2), dtype=np.uint8)
    q[0, 0] = 0x20  # code 2 (= 1.0) at k = 1, code 0 at k = 0
    s = np.full((1, K // 16), 0x38, dtype=np.uint8)  # scale 1.0
    x = synth.normal(61, "x", (3, K), 1.0)
    y = oracle.nvfp4_linear(x, q, s, 1.0)
    assert np.array_equal(y[:, 0], x[:, 1].astype(np.float64))


def test_nvfp4_dequant_is_the_linear_maps_weight():
    """The dequantised weight fed to the oracle's forward is the weight of the oracle's NVFP4 linear:
    x W^T with W = nvfp4_dequant(q, s, g) equals nvfp4_linear(x, q, s, g), and with a power-of-two
    global scale W is exact in fp32."""
    q, s, g = synth.make_nvfp4(63, "w", 256, 192)
    assert g == 2.0 ** -6
    x = synth.normal(63, "x", (5, 192), 1.0).astype(np.float64)
    W = oracle.nvfp4_dequant(q, s, g)
    ref = oracle.nvfp4_linear(x, q, s, g)
    assert np.abs(x @ W.astype(np.float64).T - ref).max() <= 1e-12 * np.abs(ref).max()
    with pytest.raises(AssertionError):
        oracle.nvfp4_dequant(q, s, 0.015)  # not a power of two: not exact in fp32


def test_synthetic_nvfp4_weights_have_the_intended_scale():
    q, s, g = synth.make_nvfp4(62, "w", 256, 1024)
    e = (s >> 3) & 15
    assert e.min() == 4 and e.max() == 6 and (s >> 7).max() == 0
    vals = oracle.e2m1_decode(np.arange(16))
    codes = np.concatenate([q & 15, q >> 4], axis=1).reshape(-1)
    assert np.bincount(codes, minlength=16).min() > 0.8 * codes.size / 16  # all 16 codes, near uniform
    rms = np.sqrt((vals[codes] ** 2).mean()) * np.sqrt((oracle.e4m3_decode(s) ** 2).mean()) * g
    assert 0.01 < rms < 0.04


# ---------------------------------------------------------------------------------------------
# the video-VAE ViT3D decoder block
# ---------------------------------------------------------------------------------------------

TINY_VIT = dict(n_blocks=2, hidden=32, n_heads=2, head_dim=16, ffn_hidden=24, norm="rms", norm_eps=1e-6,
                adaln=False, n_mod=1, t_dim=16, rope_axes=3, rope_dims=(4, 4, 4), rotary_dim=12,
                rope_base=100.0, io_channels=0, dtype="fp32", qk_norm=True, qkv_interleaved=True,
                final_norm="ln", res_scale=True, norm_affine=True)


def _vit_case(seed, m=TINY_VIT, grid=(2, 2, 2)):
    docs = [dict(video=grid)]
    w = dict(model=m, seed=seed, docs=docs, t=0.0, w_std=0.3, bias_std=0.2, x_std=1.0, affine_std=0.2)
    lay = dict(synth.build_layout(docs))
    lay["pos"] = oracle.vit_positions(*grid)
    return w, lay, synth.make_weights(w, bf16=False), synth.make_tokens(w, lay)


def test_vit_positions_closed_form():
    """(i + 0.5) / n mapped into [-1, 1), times 2 pi: symmetric about 0, spacing 4 pi / n, w fastest."""
    T, H, W = 3, 4, 5
    pos = oracle.vit_positions(T, H, W).reshape(T, H, W, 3)
    for a, n in enumerate((T, H, W)):
        ax = np.moveaxis(pos[..., a], a, 0).reshape(n, -1)
        assert (ax == ax[:, :1]).all()  # depends on its own axis id only
        v = ax[:, 0]
        assert np.allclose(v, 2 * np.pi * (np.arange(n) * 2 + 1 - n) / n, rtol=0, atol=1e-14)
        assert np.allclose(v + v[::-1], 0.0, atol=1e-14) and np.all(np.abs(v) < 2 * np.pi)


def test_forward_brute_force_vit_block():
    """Interleaved qkv, per-head q/k RMS norm, RMS gains, per-channel residual scales, 3-axis RoPE
    on the normalised grid (base 100, 12 of 16 dims) and a final LayerNorm: against the numpy forward."""
    w, lay, W, x = _vit_case(37)
    out, _ = oracle.forward(TINY_VIT, W, x, lay, 0.0)
    ref = numpy_dit.forward(TINY_VIT, W, x, lay, 0.0)
    assert np.abs(out - ref).max() <= 1e-12 * np.abs(ref).max()


def test_vit_interleaved_qkv_is_a_row_permutation_of_the_dit_order():
    """qkv.view(S, H, 3 Dh).chunk(3) == the [q_all | k_all | v_all] order with W's rows permuted."""
    w, lay, W, x = _vit_case(38)
    H, Dh = TINY_VIT["n_heads"], TINY_VIT["head_dim"]
    perm = np.array([h * 3 * Dh + s * Dh + j for s in range(3) for h in range(H) for j in range(Dh)])
    W2 = dict(blocks=[dict(b) for b in W["blocks"]], glob=W["glob"])
    for b in W2["blocks"]:
        b["w_qkv"] = b["w_qkv"][perm]
        b["b_qkv"] = b["b_qkv"][perm]
    a, _ = oracle.forward(TINY_VIT, W, x, lay, 0.0)
    b, _ = oracle.forward(dict(TINY_VIT, qkv_interleaved=False), W2, x, lay, 0.0)
    assert np.array_equal(a, b)
    c, _ = oracle.forward(dict(TINY_VIT, qkv_interleaved=False), W, x, lay, 0.0)
    assert np.abs(a - c).max() > 1e-3  # reading the interleaved weight the DiT way is wrong


def test_vit_zero_residual_scales_make_the_blocks_the_identity():
    w, lay, W, x = _vit_case(39)
    for b in W["blocks"]:
        b["res1"] = np.zeros_like(b["res1"])
        b["res2"] = np.zeros_like(b["res2"])
    out, dumps = oracle.forward(TINY_VIT, W, x, lay, 0.0, dumps=True)
    for l in range(TINY_VIT["n_blocks"]):
        assert np.array_equal(dumps[l], x.astype(np.float64))
    G = W["glob"]
    assert np.allclose(out, oracle.layer_norm(x, TINY_VIT["norm_eps"], G["lnf_g"], G["lnf_b"]), rtol=0, atol=1e-13)
