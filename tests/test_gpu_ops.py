"""Kernel-level parity: each CUDA op of the forward, called through the C ABI, against the oracle
on the same seeded inputs.  Sizes span several tiles with ragged tails; bounds are derived from the
arithmetic (fp32 accumulation, one bf16 rounding of the stored result)."""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

BF16_REL = 2.0 ** -8   # one bf16 rounding (2^-9) with a factor 2 of headroom
F16_REL = 2.0 ** -10   # one f16 rounding (2^-11) with a factor 2 of headroom
REL = {"bf16": BF16_REL, "f16": F16_REL}
ELEMS = ["bf16", "f16"]


def _dit():
    from video_audio_gen_gb300 import dit
    return dit


def _gu():
    from tests import gpu_util
    return gpu_util


def bf16_to_f64(t):
    return t.float().double().cpu().numpy()


def dev16(vals, bits, elem):
    """(device tensor, the float32 values it holds): the seeded bf16 values as a bf16 tensor (from
    their bits), or rounded to f16 (exact except below 2^-17, where f16 is subnormal)."""
    from tests import gpu_util
    if elem == "bf16":
        return gpu_util.dev_bf16(bits), np.asarray(vals, dtype=np.float32)
    t = torch.from_numpy(np.ascontiguousarray(vals, dtype=np.float32)).cuda().half()
    return t, t.float().cpu().numpy()


def tdt(elem):
    return torch.bfloat16 if elem == "bf16" else torch.float16


def fp32_sum_bound(a, b):
    """Elementwise bound on the error of an fp32-accumulated dot product: K * 2^-23 * sum|a||b|."""
    K = a.shape[1]
    return K * 2.0 ** -23 * (np.abs(a) @ np.abs(b).T)


# ------------------------------------------------------------------------------------------------
# norm + modulate
# ------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("n,d", [(1, 256), (333, 512), (130, 3072), (77, 5120)])
def test_rms_norm_modulate_matches_oracle(n, d):
    dit, gu = _dit(), _gu()
    x = synth.normal(31, "x", (n, d), 2.0)
    tags = (synth.uniform(31, "tags", n) < 0.3).astype(np.uint8)
    shift = synth.normal(31, "sh", (2, d), 0.2)
    scale = synth.normal(31, "sc", (2, d), 0.2)
    ref = oracle.modulate(oracle.rms_norm(x, 1e-6), tags, shift, scale)
    xd = gu.dev_f32(x)
    y = torch.empty((n, d), dtype=torch.bfloat16, device="cuda")
    dit.norm_modulate(xd, dit.DIT_RMSNORM, 1e-6, y, 0, tags=torch.from_numpy(tags).cuda(),
                      shift=gu.dev_f32(shift), scale=gu.dev_f32(scale), mod_stride=d)
    got = bf16_to_f64(y)
    assert np.all(np.abs(got - ref) <= BF16_REL * np.abs(ref) + 1e-5)
    yf = torch.empty((n, d), dtype=torch.float32, device="cuda")
    dit.norm_modulate(xd, dit.DIT_RMSNORM, 1e-6, yf, 1, tags=torch.from_numpy(tags).cuda(),
                      shift=gu.dev_f32(shift), scale=gu.dev_f32(scale), mod_stride=d)
    gotf = yf.double().cpu().numpy()
    assert np.abs(gotf - ref).max() <= 1e-5 * np.abs(ref).max()
    yh = torch.empty((n, d), dtype=torch.float16, device="cuda")
    dit.norm_modulate(xd, dit.DIT_RMSNORM, 1e-6, yh, 2, tags=torch.from_numpy(tags).cuda(),
                      shift=gu.dev_f32(shift), scale=gu.dev_f32(scale), mod_stride=d)
    assert np.all(np.abs(bf16_to_f64(yh) - ref) <= F16_REL * np.abs(ref) + 1e-5)


def test_norm_without_modulation_is_bare_rms():
    dit, gu = _dit(), _gu()
    x = synth.normal(32, "x", (200, 768), 1.5)
    yf = torch.empty((200, 768), dtype=torch.float32, device="cuda")
    dit.norm_modulate(gu.dev_f32(x), dit.DIT_RMSNORM, 1e-6, yf, 1)
    ref = oracle.rms_norm(x, 1e-6)
    assert np.abs(yf.double().cpu().numpy() - ref).max() <= 1e-5 * np.abs(ref).max()


def test_layer_norm_affine_matches_oracle():
    dit, gu = _dit(), _gu()
    x = synth.normal(33, "x", (150, 2048), 1.0) + 0.5
    g = 1.0 + synth.normal(33, "g", (2048,), 0.1)
    b = synth.normal(33, "b", (2048,), 0.1)
    yf = torch.empty((150, 2048), dtype=torch.float32, device="cuda")
    dit.norm_modulate(gu.dev_f32(x), dit.DIT_LAYERNORM, 1e-5, yf, 1, ln_g=gu.dev_f32(g), ln_b=gu.dev_f32(b))
    ref = oracle.layer_norm(x, 1e-5, g, b)
    assert np.abs(yf.double().cpu().numpy() - ref).max() <= 2e-5 * np.abs(ref).max()


# ------------------------------------------------------------------------------------------------
# cos/sin cache, AdaLN conditioning
# ------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "video_audio_bf16", "ragged"])
def test_rope_cache_matches_oracle(name):
    dit, gu = _dit(), _gu()
    w = synth.WORKLOADS[name]
    m = w["model"]
    lay = synth.build_layout(w["docs"])
    half = m["rotary_dim"] // 2
    cs = torch.empty((lay["n_tokens"], half), dtype=torch.float32, device="cuda")
    sn = torch.empty_like(cs)
    dit.rope_cache(gu.dev_layout(lay)["pos"], m["rope_axes"], m["rope_dims"], m["rope_base"], cs, sn)
    rc, rs = oracle.rope_cos_sin(m, lay["pos"])
    gc, gs = cs.cpu().numpy(), sn.cpu().numpy()
    # fp64 cos/sin rounded once to fp32: equal to the oracle's rounding, up to one fp32 ulp where the
    # two fp64 libraries round the last bit differently
    ulp = np.spacing(np.float32(1.0))
    assert np.abs(gc - rc).max() <= ulp and np.abs(gs - rs).max() <= ulp
    assert (gc == rc.astype(np.float32)).mean() > 0.999 and (gs == rs.astype(np.float32)).mean() > 0.999


def test_adaln_matches_oracle():
    dit, gu = _dit(), _gu()
    w = synth.WORKLOADS["tiny"]
    m = w["model"]
    W = synth.make_weights(w)
    # give the projection non-zero biases so the bias path is exercised
    for l, b in enumerate(W["blocks"]):
        b["b_ada"] = synth.normal(34, f"b{l}", b["b_ada"].shape, 0.05)
    W["glob"]["b_ada_final"] = synth.normal(34, "bf", W["glob"]["b_ada_final"].shape, 0.05)
    for t in (0.0, 0.5, 0.9731):
        mod, modf = oracle.adaln(m, W, float(np.float32(t)))
        wall = np.concatenate([b["w_ada"] for b in W["bits"]["blocks"]] + [W["bits"]["glob"]["w_ada_final"]])
        ball = np.concatenate([b["b_ada"] for b in W["blocks"]] + [W["glob"]["b_ada_final"]])
        out = torch.empty((wall.shape[0],), dtype=torch.float32, device="cuda")
        dit.adaln(gu.dev_bf16(wall), gu.dev_f32(ball), t, out)
        ref = np.concatenate([mod.reshape(-1), modf.reshape(-1)])
        assert np.abs(out.double().cpu().numpy() - ref).max() <= 2e-5, t


# ------------------------------------------------------------------------------------------------
# GEMM engine and its epilogues
# ------------------------------------------------------------------------------------------------

def _ab(M, N, K, seed, std_b=0.05):
    a, abits = synth.normal(seed, "A", (M, K), 1.0, bf16=True)
    b, bbits = synth.normal(seed, "B", (N, K), std_b, bf16=True)
    bias = synth.normal(seed, "bias", (N,), 0.1)
    return a, abits, b, bbits, bias


@pytest.mark.parametrize("elem", ELEMS)
@pytest.mark.parametrize("M,N,K", [(1, 256, 64), (333, 512, 512), (128, 768, 256), (1000, 1024, 1536),
                                   (257, 256, 4096), (4224, 2560, 128)])
def test_gemm_store_matches_oracle(M, N, K, elem):
    """Row tiles run in pairs of 128-row blocks: one row (the second block of the pair past M), an
    odd number of row blocks (the last pair's second block wholly past M), one K-block and one
    N-tile, a K of 64 blocks (the stage ring wraps ten times), and 170 pair tiles (every pair of
    the persistent grid takes two or three, so both accumulator buffers and their phases turn)."""
    dit, gu = _dit(), _gu()
    a, abits, b, bbits, bias = _ab(M, N, K, 40 + M)
    (A, a), (B, b) = dev16(a, abits, elem), dev16(b, bbits, elem)
    ref = oracle.linear(a, b, bias)
    bound = fp32_sum_bound(a.astype(np.float64), b.astype(np.float64))
    out = torch.empty((M, N), dtype=torch.float32, device="cuda")
    dit.gemm(A, B, gu.dev_f32(bias), out, 1)
    got = out.double().cpu().numpy()
    assert np.all(np.abs(got - ref) <= bound + 1e-6)
    outb = torch.empty((M, N), dtype=tdt(elem), device="cuda")
    dit.gemm(A, B, None, outb, 0 if elem == "bf16" else 2)
    refb = oracle.linear(a, b, None)
    assert np.all(np.abs(bf16_to_f64(outb) - refb) <= REL[elem] * np.abs(refb) + bound + 1e-6)


@pytest.mark.parametrize("elem", ELEMS)
@pytest.mark.parametrize("name", ["tiny", "ragged"])
def test_gemm_qkv_rope_matches_oracle(name, elem):
    dit, gu = _dit(), _gu()
    w = synth.WORKLOADS[name]
    m = w["model"]
    lay = synth.build_layout(w["docs"])
    M, d, H, Dh, R = lay["n_tokens"], m["hidden"], m["n_heads"], m["head_dim"], m["rotary_dim"]
    a, abits, b, bbits, bias = _ab(M, 3 * d, d, 50)
    (A, a), (B, b) = dev16(a, abits, elem), dev16(b, bbits, elem)
    cs, sn = oracle.rope_cos_sin(m, lay["pos"])
    qkv = oracle.linear(a, b, bias)
    qr = oracle.rope_apply(qkv[:, :d], H, Dh, R, cs, sn)
    kr = oracle.rope_apply(qkv[:, d:2 * d], H, Dh, R, cs, sn)
    vr = qkv[:, 2 * d:]
    n_pad = (M + 7) // 8 * 8
    q = torch.empty((M, d), dtype=tdt(elem), device="cuda")
    k = torch.empty_like(q)
    vt = torch.full((d, n_pad), float("nan"), dtype=tdt(elem), device="cuda")  # garbage on entry
    gcs = torch.empty((M, R // 2), dtype=torch.float32, device="cuda")
    gsn = torch.empty_like(gcs)
    dit.rope_cache(gu.dev_layout(lay)["pos"], m["rope_axes"], m["rope_dims"], m["rope_base"], gcs, gsn)
    dit.gemm_qkv_rope(A, B, gu.dev_f32(bias), H, Dh, R, gcs, gsn, q, k, vt, n_pad)
    bound = fp32_sum_bound(a.astype(np.float64), b.astype(np.float64))
    # rotation mixes two accumulators: bound both, plus fp32 cos/sin (2^-24) and the 16-bit store
    bq = bound[:, :d] + np.roll(bound[:, :d], 1, axis=1)  # generous pair bound
    for got, ref, bb in ((bf16_to_f64(q), qr, bq), (bf16_to_f64(k), kr, bq)):
        err = np.abs(got - ref)
        assert np.all(err <= REL[elem] * np.abs(ref) + 2 * bb.max() + 1e-5), err.max()
    gv = bf16_to_f64(vt)[:, :M].T
    assert np.all(np.abs(gv - vr) <= REL[elem] * np.abs(vr) + bound[:, 2 * d:] + 1e-6)
    assert (bf16_to_f64(vt)[:, M:] == 0).all()  # padding columns are written as zeros


@pytest.mark.parametrize("Dh,R", [(32, 32), (128, 128), (128, 96), (256, 256), (256, 128)])
def test_gemm_qkv_rope_head_dims(Dh, R):
    """The QKV epilogue at other head dims than the models': the tile's 256 columns are split between
    two epilogue warps per TMEM lane quarter, a head never between them (at head_dim 256 the first
    warp takes the whole head).  d = 512, a ragged M of three row tiles, random cos/sin caches."""
    dit, gu = _dit(), _gu()
    d, M, K = 512, 300, 256
    H = d // Dh
    a, abits, b, bbits, bias = _ab(M, 3 * d, K, 70 + Dh + R)
    (A, a), (B, b) = dev16(a, abits, "bf16"), dev16(b, bbits, "bf16")
    ang = synth.uniform(71 + Dh + R, "angles", M * (R // 2)).reshape(M, R // 2) * 6.283185307179586
    cs = np.cos(ang).astype(np.float32).astype(np.float64)
    sn = np.sin(ang).astype(np.float32).astype(np.float64)
    qkv = oracle.linear(a, b, bias)
    qr = oracle.rope_apply(qkv[:, :d], H, Dh, R, cs, sn)
    kr = oracle.rope_apply(qkv[:, d:2 * d], H, Dh, R, cs, sn)
    vr = qkv[:, 2 * d:]
    n_pad = (M + 7) // 8 * 8
    q = torch.empty((M, d), dtype=torch.bfloat16, device="cuda")
    k = torch.empty_like(q)
    vt = torch.full((d, n_pad), float("nan"), dtype=torch.bfloat16, device="cuda")
    gcs = gu.dev_f32(cs.astype(np.float32))
    gsn = gu.dev_f32(sn.astype(np.float32))
    dit.gemm_qkv_rope(A, B, gu.dev_f32(bias), H, Dh, R, gcs, gsn, q, k, vt, n_pad)
    bound = fp32_sum_bound(a.astype(np.float64), b.astype(np.float64))
    bq = bound[:, :d] + np.roll(bound[:, :d], 1, axis=1)
    for got, ref in ((bf16_to_f64(q), qr), (bf16_to_f64(k), kr)):
        err = np.abs(got - ref)
        assert np.all(err <= REL["bf16"] * np.abs(ref) + 2 * bq.max() + 1e-5), err.max()
    gv = bf16_to_f64(vt)[:, :M].T
    assert np.all(np.abs(gv - vr) <= REL["bf16"] * np.abs(vr) + bound[:, 2 * d:] + 1e-6)
    assert (bf16_to_f64(vt)[:, M:] == 0).all()


@pytest.mark.parametrize("elem", ELEMS)
@pytest.mark.parametrize("M", [1, 129, 555])
def test_gemm_gated_residual_matches_oracle(M, elem):
    """One row, one row past a tile, and several ragged tiles: the residual epilogue stages each
    column group through shared memory and writes only the rows below M."""
    dit, gu = _dit(), _gu()
    N, K = 512, 1024
    a, abits, b, bbits, bias = _ab(M, N, K, 60 + M)
    (A, a), (B, b) = dev16(a, abits, elem), dev16(b, bbits, elem)
    x = synth.normal(60 + M, "x", (M, N), 1.0)
    gate = synth.normal(60 + M, "gate", (2, N), 0.3)
    tags = (synth.uniform(60 + M, "tags", M) < 0.5).astype(np.uint8)
    ref = x.astype(np.float64) + gate[tags].astype(np.float64) * oracle.linear(a, b, bias)
    xd = gu.dev_f32(x)
    dit.gemm_gated_residual(A, B, gu.dev_f32(bias), xd, gate=gu.dev_f32(gate), gate_stride=N,
                            tags=torch.from_numpy(tags).cuda())
    bound = fp32_sum_bound(a.astype(np.float64), b.astype(np.float64)) * np.abs(gate[tags]) + 2 ** -23 * 4
    assert np.all(np.abs(xd.double().cpu().numpy() - ref) <= bound + 1e-6)
    # gate = NULL: plain residual add
    xd2 = gu.dev_f32(x)
    dit.gemm_gated_residual(A, B, None, xd2)
    ref2 = x.astype(np.float64) + oracle.linear(a, b, None)
    assert np.abs(xd2.double().cpu().numpy() - ref2).max() <= 1e-4


def tf32x3_bound(x, w, ref):
    """Elementwise bound for the 3xTF32 fp32 GEMM, from its arithmetic: the split drops about
    3 x 2^-22 of |x w| per product; each 32-deep TMEM chunk (12 accumulating MMAs) adds at most
    4e-6 of its sum of |x w| (the accumulation is biased, so this is linear, not a random walk);
    the chunk sums and the K-split reduction are fp32 round-to-nearest adds (one 2^-24 of the sum of
    |x w| each); the store rounds once."""
    K = x.shape[1]
    P = np.abs(x) @ np.abs(w).T
    return (5e-6 + (K / 32 + 16) * 2.0 ** -24) * P + 2.0 ** -23 * np.abs(ref)


@pytest.mark.parametrize("M,N,K", [(1, 128, 32), (17, 128, 4096), (74, 256, 1024), (300, 384, 96),
                                   (172, 2048, 8192)])
def test_gemm_f32_matches_oracle(M, N, K):
    """The fp32 forward's linear map (3xTF32 on the tensor cores): token counts below, at and above
    one 256-wide token tile, ragged M, the music DiT's deepest K; against the oracle's fp64 linear."""
    dit, gu = _dit(), _gu()
    x = synth.normal(140, "x", (M, K), 1.0)
    w = synth.normal(140, "w", (N, K), 0.02)
    b = synth.normal(140, "b", (N,), 0.02)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ws = torch.empty(dit.gemm_f32_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
    ws.fill_(0xFF)  # stale NaN bytes: nothing may read scratch it did not write
    dit.gemm_f32(gu.dev_f32(x), gu.dev_f32(w), gu.dev_f32(b), y, ws)
    torch.cuda.synchronize()
    oracle.set_threads(16)
    ref = oracle.linear(x.astype(np.float64), w, b)
    oracle.set_threads(1)
    got = y.double().cpu().numpy()
    bound = tf32x3_bound(x.astype(np.float64), w.astype(np.float64), ref)
    assert np.all(np.abs(got - ref) <= bound), float((np.abs(got - ref) / bound).max())
    # a single tf32 product would miss by ~1e-3 relative: the bound is far tighter than that
    P = np.abs(x).astype(np.float64) @ np.abs(w).astype(np.float64).T
    assert np.abs(got - ref).max() <= 2e-5 * P.max()


def test_gemm_f32_rejects_bad_shapes():
    dit, gu = _dit(), _gu()
    x = gu.dev_f32(np.zeros((4, 48), np.float32))
    w = gu.dev_f32(np.zeros((128, 48), np.float32))
    y = torch.empty((4, 128), dtype=torch.float32, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(dit.DitError):
        dit.gemm_f32(x, w, None, y, ws)  # K = 48 is not a multiple of 32


@pytest.mark.parametrize("elem", ELEMS)
def test_gemm_swiglu_matches_oracle(elem):
    dit, gu = _dit(), _gu()
    M, F, d = 300, 768, 512
    a, abits, _, _, _ = _ab(M, 256, d, 70)
    win, wbits = synth.normal(70, "win", (2 * F, d), 0.05, bf16=True)
    (A, a), (Win, win) = dev16(a, abits, elem), dev16(win, wbits, elem)
    bin_ = synth.normal(70, "bin", (2 * F,), 0.1)
    ref = oracle.swiglu(oracle.linear(a, win, bin_))
    wp = torch.empty((2 * F, d), dtype=tdt(elem), device="cuda")
    bp = torch.empty((2 * F,), dtype=torch.float32, device="cuda")
    dit.pack_ffn_in(Win, gu.dev_f32(bin_), wp, bp)
    h = torch.empty((M, F), dtype=tdt(elem), device="cuda")
    dit.gemm_swiglu(A, wp, bp, h)
    got = bf16_to_f64(h)
    uv_bound = fp32_sum_bound(a.astype(np.float64), win.astype(np.float64))
    # |d(u silu g)| <= |silu g| du + |u| |silu'| dg with |silu'| <= 1.1
    uv = oracle.linear(a, win, bin_)
    u, g = uv[:, :F], uv[:, F:]
    prop = np.abs(g) * uv_bound[:, :F] + 1.1 * np.abs(u) * uv_bound[:, F:]
    assert np.all(np.abs(got - ref) <= REL[elem] * np.abs(ref) + prop + 1e-5 * np.abs(u) + 1e-6)


# ------------------------------------------------------------------------------------------------
# attention
# ------------------------------------------------------------------------------------------------

def _attn_inputs(lay, H, Dh, seed, same_keys=False):
    n = lay["n_tokens"]
    q, qb = synth.normal(seed, "q", (n, H * Dh), 1.0, bf16=True)
    k, kb = synth.normal(seed, "k", (n, H * Dh), 1.0, bf16=True)
    if same_keys:
        k = np.tile(k[:1], (n, 1))
        kb = np.tile(kb[:1], (n, 1))
    v, vb = synth.normal(seed, "v", (n, H * Dh), 1.0, bf16=True)
    return q, qb, k, kb, v, vb


def _run_attention(lay, H, Dh, qb, kb, vb, elem="bf16"):
    """qb, kb, vb: bf16 bits of the inputs; with elem "f16" the same values run as f16."""
    dit, gu = _dit(), _gu()
    n = lay["n_tokens"]
    n_pad = (n + 7) // 8 * 8
    vt = np.zeros((H * Dh, n_pad), dtype=np.uint16)
    vt[:, :n] = vb.T
    def dev(bits):
        t = gu.dev_bf16(bits)
        return t if elem == "bf16" else t.half()  # bf16 values are exact in f16 at these magnitudes
    o = torch.empty((n, H * Dh), dtype=tdt(elem), device="cuda")
    ws = torch.empty(dit.attention_workspace_bytes(lay["n_docs"], n), dtype=torch.uint8, device="cuda")
    dit.attention(dev(qb), dev(kb), dev(vt), n_pad, gu.dev_layout(lay)["cu"], H, Dh, o, ws)
    torch.cuda.synchronize()
    return bf16_to_f64(o)


def attn_tol(ref, v, elem="bf16"):
    """P is rounded to the 16-bit type before P.V (relative 2^-9 or 2^-11 per weight) and O is stored
    in it."""
    return REL[elem] * np.abs(ref) + REL[elem] * np.abs(v).max()


DOCSETS = {
    "tiny": synth.WORKLOADS["tiny"]["docs"],
    "ragged": synth.WORKLOADS["ragged"]["docs"],
    "edges": [dict(video=(1, 1, 1)), dict(video=(1, 1, 127)), dict(video=(1, 1, 128)), dict(video=(1, 1, 129)),
              dict(video=(1, 5, 51)), dict(video=(1, 1, 1), audio=1)],
}


@pytest.mark.parametrize("elem", ELEMS)
@pytest.mark.parametrize("docs", list(DOCSETS))
@pytest.mark.parametrize("Dh", [64, 128])
def test_attention_matches_oracle(docs, Dh, elem):
    lay = synth.build_layout(DOCSETS[docs])
    H = 2
    q, qb, k, kb, v, vb = _attn_inputs(lay, H, Dh, 80 + Dh)
    ref = oracle.attention(q, k, v, lay["cu_seqlens"], H, Dh)
    got = _run_attention(lay, H, Dh, qb, kb, vb, elem)
    assert np.all(np.abs(got - ref) <= attn_tol(ref, v, elem))


def test_attention_identical_keys_gives_mean_of_v():
    lay = synth.build_layout(DOCSETS["ragged"])
    H, Dh = 2, 128
    q, qb, k, kb, v, vb = _attn_inputs(lay, H, Dh, 90, same_keys=True)
    got = _run_attention(lay, H, Dh, qb, kb, vb)
    cu = lay["cu_seqlens"]
    for j in range(lay["n_docs"]):
        mean = v[cu[j]:cu[j + 1]].astype(np.float64).mean(axis=0)
        assert np.all(np.abs(got[cu[j]:cu[j + 1]] - mean) <= BF16_REL * np.abs(mean) + 2 ** -8 * np.abs(v).max())


def test_attention_one_token_doc_returns_v_and_docs_do_not_mix():
    lay = synth.build_layout(DOCSETS["edges"])
    H, Dh = 2, 128
    q, qb, k, kb, v, vb = _attn_inputs(lay, H, Dh, 91)
    got = _run_attention(lay, H, Dh, qb, kb, vb)
    assert np.array_equal(got[0], v[0].astype(np.float64))  # the 1-token document: softmax weight exactly 1
    # perturb document 3: every other document's rows stay bit-identical
    cu = lay["cu_seqlens"]
    qb2, kb2, vb2 = qb.copy(), kb.copy(), vb.copy()
    a, b = cu[3], cu[4]
    qb2[a:b] ^= 0x0040
    kb2[a:b] ^= 0x0040
    vb2[a:b] ^= 0x0040
    got2 = _run_attention(lay, H, Dh, qb2, kb2, vb2)
    mask = np.ones(lay["n_tokens"], dtype=bool)
    mask[a:b] = False
    assert np.array_equal(got[mask], got2[mask])
    assert not np.array_equal(got[~mask], got2[~mask])


@pytest.mark.parametrize("elem", ELEMS)
@pytest.mark.parametrize("Dh", [64, 128])
def test_attention_nonfinite_document_is_isolated(Dh, elem):
    """NaN and +-Inf in one document's q, k and v: every other document's output rows stay
    bit-identical to the clean run, including the neighbours that share its 128-token boundary
    tiles (their keys are masked and their V^T columns zeroed before the P.V product)."""
    lay = synth.build_layout(DOCSETS["edges"] + [dict(video=(1, 3, 70)), dict(video=(1, 1, 50))])
    H = 2
    q, qb, k, kb, v, vb = _attn_inputs(lay, H, Dh, 93)
    clean = _run_attention(lay, H, Dh, qb, kb, vb, elem)
    cu = lay["cu_seqlens"]
    j = 6                                  # tokens [642, 852): both ends inside tiles shared with neighbours
    a, b = int(cu[j]), int(cu[j + 1])
    assert a % 128 and b % 128
    NAN, PINF, NINF = np.uint16(0x7FC0), np.uint16(0x7F80), np.uint16(0xFF80)
    qb2, kb2, vb2 = qb.copy(), kb.copy(), vb.copy()
    qb2[a:b:3, 5] = NAN
    kb2[a + 1:b:4, 7] = PINF
    kb2[a + 2:b:5, 1] = NAN
    vb2[a:b:2, 3] = NAN
    vb2[a + 1:b:7, Dh + 9] = NINF
    vb2[b - 1, :] = PINF
    got = _run_attention(lay, H, Dh, qb2, kb2, vb2, elem)
    mask = np.ones(lay["n_tokens"], dtype=bool)
    mask[a:b] = False
    assert np.isfinite(got[mask]).all()
    assert np.array_equal(got[mask].view(np.uint64), clean[mask].view(np.uint64))


@pytest.mark.slow
def test_attention_full_size_sampled_rows():
    """The 17,408-token, 24-head launch the forward uses, checked on sampled query rows."""
    w = synth.WORKLOADS["video_audio_bf16"]
    m = w["model"]
    lay = synth.build_layout(w["docs"])
    H, Dh = m["n_heads"], m["head_dim"]
    q, qb, k, kb, v, vb = _attn_inputs(lay, H, Dh, 92)
    got = _run_attention(lay, H, Dh, qb, kb, vb)
    n = lay["n_tokens"]
    rows = np.unique(np.concatenate([[0, 127, 128, 8703, 8704, n - 1],
                                     (synth.uniform(92, "rows", 26) * n).astype(np.int64)]))
    oracle.set_threads(8)
    ref = oracle.attention_rows(q, k, v, lay["cu_seqlens"], H, Dh, rows)
    oracle.set_threads(1)
    assert np.all(np.abs(got[rows] - ref) <= attn_tol(ref, v))


# ------------------------------------------------------------------------------------------------
# Euler step: bit-exact
# ------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 7, 4096, 1_000_003])
def test_euler_step_bit_exact(n):
    dit, gu = _dit(), _gu()
    x = synth.normal(100, "x", (n,), 1.0)
    v = synth.normal(100, "v", (n,), 1.0)
    sig = synth.sigmas(50)
    for i in (0, 13, 49):
        xd = gu.dev_f32(x)
        dit.euler_step(xd, gu.dev_f32(v), float(sig[i]), float(sig[i + 1]))
        ref = oracle.euler_step(x, v, sig[i], sig[i + 1])
        assert np.array_equal(xd.cpu().numpy().view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("n_tokens,d,n_mod", [(1, 1, 1), (1001, 7, 3), (4096, 256, 2), (17, 3072, 8)])
def test_euler_step_modal_bit_exact(n_tokens, d, n_mod):
    """Each row stepped with its own modality's sigma pair, bit for bit the oracle's fp32 sequence;
    rows whose tag is out of range are left as they were."""
    dit, gu = _dit(), _gu()
    x = synth.normal(102, "x", (n_tokens, d), 1.0)
    v = synth.normal(102, "v", (n_tokens, d), 1.0)
    tags = (synth.uniform(102, "tags", n_tokens) * (n_mod + 1)).astype(np.uint8)  # includes tag n_mod
    base = synth.sigmas(50)
    shifts = [1.0, 12.0, 3.0, 0.5, 2.0, 7.0, 1.5, 4.0][:n_mod]
    for i in (0, 31, 49):
        sg = [float(oracle.sigmas_shifted(base[i:i + 2], s)[0]) for s in shifts]
        sn = [float(oracle.sigmas_shifted(base[i:i + 2], s)[1]) for s in shifts]
        xd = gu.dev_f32(x)
        dit.euler_step_modal(xd, gu.dev_f32(v), gu.dev_u8(tags), sg, sn)
        got = xd.cpu().numpy()
        ok = tags < n_mod
        ref = oracle.euler_step_tagged(x[ok], v[ok], tags[ok], sg, sn)
        assert np.array_equal(got[ok].view(np.uint32), ref.view(np.uint32))
        assert np.array_equal(got[~ok].view(np.uint32), x[~ok].view(np.uint32))


def test_euler_step_modal_rejects_bad_arguments():
    dit, gu = _dit(), _gu()
    xd = gu.dev_f32(np.ones((4, 8), dtype=np.float32))
    tags = gu.dev_u8(np.zeros(4, dtype=np.uint8))
    for sg, sn in (([0.0], [0.0]), ([0.5] * 9, [0.4] * 9), ([], [])):
        with pytest.raises(dit.DitError):
            dit.euler_step_modal(xd, xd, tags, sg, sn)
    assert (xd == 1.0).all()


def test_time_shift_matches_oracle():
    """dit_time_shift on the fp32 base schedule gives the oracle's shifted schedule bit for bit."""
    dit = _dit()
    base = synth.sigmas(50)
    for shift in (1.0, 3.0, 12.0, 0.25, 5.5):
        got = np.array([dit.time_shift(float(s), shift) for s in base], dtype=np.float32)
        assert np.array_equal(got.view(np.uint32), oracle.sigmas_shifted(base, shift).view(np.uint32)), shift


def test_euler_unaligned_view_bit_exact():
    dit, gu = _dit(), _gu()
    x = synth.normal(101, "x", (1001,), 1.0)
    v = synth.normal(101, "v", (1001,), 1.0)
    xd = gu.dev_f32(x)
    vd = gu.dev_f32(v)
    dit.euler_step(xd[1:], vd[1:], 0.5, 0.48)
    ref = oracle.euler_step(x[1:], v[1:], np.float32(0.5), np.float32(0.48))
    got = xd.cpu().numpy()
    assert got[0] == x[0] and np.array_equal(got[1:].view(np.uint32), ref.view(np.uint32))


# ------------------------------------------------------------------------------------------------
# NVFP4 weights
# ------------------------------------------------------------------------------------------------

def _nvfp4_tiles(q, s, N, K):
    """The tile-contiguous layout, built independently on the host: per (256-row block, 64-column
    block) the 256 rows' 32 code bytes, then their 4 scale bytes."""
    out = []
    for nb in range(N // 256):
        for kb in range(K // 64):
            out.append(q[nb * 256:(nb + 1) * 256, kb * 32:(kb + 1) * 32].reshape(-1))
            out.append(s[nb * 256:(nb + 1) * 256, kb * 4:(kb + 1) * 4].reshape(-1))
    return np.concatenate(out)


def test_pack_nvfp4_layout_is_exact():
    dit, gu = _dit(), _gu()
    N, K = 512, 192
    q, s, g = synth.make_nvfp4(70, "w", N, K)
    packed = torch.zeros(dit.nvfp4_packed_bytes(N, K), dtype=torch.uint8, device="cuda")
    dit.pack_nvfp4(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), packed)
    assert np.array_equal(packed.cpu().numpy(), _nvfp4_tiles(q, s, N, K))


@pytest.mark.parametrize("M,N,K,out_kind", [(1, 256, 64, 1), (200, 512, 1024, 1), (300, 768, 3072, 0),
                                            (1000, 256, 128, 2), (129, 9216, 3072, 1)])
def test_gemm_nvfp4_matches_oracle(M, N, K, out_kind):
    """out = A W^T + bias with W = E2M1 code * E4M3 scale * global: the products are exact in f16,
    so the only error is fp32 accumulation, bounded by (K + 2) 2^-23 sum|a||w|, plus the output
    rounding (bf16 2^-8, f16 2^-11 relative)."""
    dit, gu = _dit(), _gu()
    q, s, g = synth.make_nvfp4(71, f"w{N}x{K}", N, K)
    a = synth.normal(71, f"a{M}x{K}", (M, K), 1.0).astype(np.float16)
    bias = synth.normal(71, f"b{N}", (N,), 0.1)
    packed = torch.empty(dit.nvfp4_packed_bytes(N, K), dtype=torch.uint8, device="cuda")
    dit.pack_nvfp4(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), packed)
    odt = {0: torch.bfloat16, 1: torch.float32, 2: torch.float16}[out_kind]
    out = torch.full((M, N), float("nan"), dtype=odt, device="cuda")
    dit.gemm_nvfp4(torch.from_numpy(a).cuda(), packed, g, gu.dev_f32(bias), N, out, out_kind)
    got = out.double().cpu().numpy()
    oracle.set_threads(8)
    ref = oracle.nvfp4_linear(a.astype(np.float64), q, s, g, bias)
    # sum|a||w|: the same linear with |A| and the codes' sign bits cleared (the scales are positive)
    sumabs = oracle.nvfp4_linear(np.abs(a.astype(np.float64)), (q & 0x77).astype(np.uint8), s, g)
    oracle.set_threads(1)
    rel = {0: 2.0 ** -8, 1: 0.0, 2: 2.0 ** -11}[out_kind]
    bound = (K + 2) * 2.0 ** -23 * sumabs + rel * np.abs(ref) + 1e-30
    assert np.isfinite(got).all()
    assert np.all(np.abs(got - ref) <= bound), np.abs(got - ref).max()


def test_gemm_nvfp4_rejects_bad_shapes():
    dit = _dit()
    lib = dit.lib()
    a = torch.zeros((4, 64), dtype=torch.float16, device="cuda")
    p = torch.zeros(dit.nvfp4_packed_bytes(256, 64), dtype=torch.uint8, device="cuda")
    o = torch.zeros((4, 256), dtype=torch.float32, device="cuda")
    assert lib.dit_op_gemm_nvfp4(a.data_ptr(), p.data_ptr(), 1.0, None, 4, 128, 64, o.data_ptr(), 1, None) != 0
    assert lib.dit_op_gemm_nvfp4(a.data_ptr(), p.data_ptr(), 1.0, None, 4, 256, 48, o.data_ptr(), 1, None) != 0
    assert lib.dit_op_gemm_nvfp4(a.data_ptr(), p.data_ptr(), 1.0, None, 4, 256, 64, o.data_ptr(), 3, None) != 0
    assert dit.nvfp4_packed_bytes(100, 64) == 0


def test_gemm_nvfp4_zero_codes_give_the_bias():
    """Every code +0 or -0: the weight is zero whatever the scales, so out = bias exactly."""
    dit, gu = _dit(), _gu()
    M, N, K = 70, 256, 128
    _, s, g = synth.make_nvfp4(73, "wz", N, K)
    q = np.where(synth.uniform(73, "sign", N * K // 2).reshape(N, K // 2) < 0.5, 0x00, 0x88).astype(np.uint8)
    a = synth.normal(73, "az", (M, K), 1.0).astype(np.float16)
    bias = synth.normal(73, "bz", (N,), 0.5)
    packed = torch.empty(dit.nvfp4_packed_bytes(N, K), dtype=torch.uint8, device="cuda")
    dit.pack_nvfp4(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), packed)
    out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    dit.gemm_nvfp4(torch.from_numpy(a).cuda(), packed, g, gu.dev_f32(bias), N, out, 1)
    assert np.array_equal(out.cpu().numpy(), np.broadcast_to(bias, (M, N)))


def test_euler_step_modal_with_no_tokens_is_a_no_op():
    dit, gu = _dit(), _gu()
    x = torch.zeros((0, 16), dtype=torch.float32, device="cuda")
    t = torch.zeros((0,), dtype=torch.uint8, device="cuda")
    dit.euler_step_modal(x, x, t, [0.5, 0.4], [0.4, 0.3])  # returns DIT_OK, launches nothing
    torch.cuda.synchronize()
