"""Full-size checks in the launch configurations the bench times: the oracle computes sampled
outputs one by one (attention rows, GEMM rows), and whole forwards are checked through properties
that hold at any size (zero gates make every block the identity, determinism)."""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.slow]

BF16_REL = 2.0 ** -8


def _gu():
    from tests import gpu_util
    return gpu_util


def _dit():
    from video_audio_gen_gb300 import dit
    return dit


def _rows(n, seed, extra=()):
    r = (synth.uniform(seed, "rows", 24) * n).astype(np.int64)
    return np.unique(np.concatenate([np.array(extra, dtype=np.int64), r]))


@pytest.mark.parametrize("name", ["long_doc_bf16", "denoise_loop"])
def test_attention_full_size_sampled_rows(name):
    """33,792-token single document x 40 heads; the loop's 17,408 + 9,216-token pair x 24 heads."""
    dit, gu = _dit(), _gu()
    w = synth.WORKLOADS[name]
    m = w["model"]
    lay = synth.build_layout(w["docs"])
    n, H, Dh = lay["n_tokens"], m["n_heads"], m["head_dim"]
    d = H * Dh
    q, qb = synth.normal(300, "q", (n, d), 1.0, bf16=True)
    k, kb = synth.normal(300, "k", (n, d), 1.0, bf16=True)
    v, vb = synth.normal(300, "v", (n, d), 1.0, bf16=True)
    n_pad = (n + 7) // 8 * 8
    vt = np.zeros((d, n_pad), dtype=np.uint16)
    vt[:, :n] = vb.T
    o = torch.empty((n, d), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(dit.attention_workspace_bytes(lay["n_docs"], n), dtype=torch.uint8, device="cuda")
    dit.attention(gu.dev_bf16(qb), gu.dev_bf16(kb), gu.dev_bf16(vt), n_pad, gu.dev_layout(lay)["cu"], H, Dh, o, ws)
    torch.cuda.synchronize()
    cu = lay["cu_seqlens"]
    rows = _rows(n, 301, [0, 127, int(cu[1]) - 1, int(cu[1]) % n, n - 1])
    oracle.set_threads(16)
    ref = oracle.attention_rows(q, k, v, cu, H, Dh, rows)
    oracle.set_threads(1)
    got = o.float().double().cpu().numpy()[rows]
    assert np.all(np.abs(got - ref) <= BF16_REL * np.abs(ref) + 2.0 ** -8 * np.abs(v).max())


@pytest.mark.parametrize("which", ["qkv", "ffn_up", "ffn_down"])
def test_long_doc_gemms_sampled_rows(which):
    """The long-document model's GEMM shapes (M = 33,792, d = 5120, F = 13,824) on sampled rows."""
    dit, gu = _dit(), _gu()
    w = synth.WORKLOADS["long_doc_bf16"]
    m = w["model"]
    lay = synth.build_layout(w["docs"])
    M, d, F, H, Dh = lay["n_tokens"], m["hidden"], m["ffn_hidden"], m["n_heads"], m["head_dim"]
    K = F if which == "ffn_down" else d
    a, ab = synth.normal(310, "a", (M, K), 1.0, bf16=True)
    rows = _rows(M, 311, [0, 1, 127, 128, M - 1])
    oracle.set_threads(16)
    if which == "qkv":
        W, Wb = synth.normal(310, "w", (3 * d, d), 0.02, bf16=True)
        R = m["rotary_dim"]
        n_pad = (M + 7) // 8 * 8
        cs = torch.empty((M, R // 2), dtype=torch.float32, device="cuda")
        sn = torch.empty_like(cs)
        dit.rope_cache(gu.dev_layout(lay)["pos"], 3, m["rope_dims"], m["rope_base"], cs, sn)
        q = torch.empty((M, d), dtype=torch.bfloat16, device="cuda")
        k = torch.empty_like(q)
        vt = torch.empty((d, n_pad), dtype=torch.bfloat16, device="cuda")
        dit.gemm_qkv_rope(gu.dev_bf16(ab), gu.dev_bf16(Wb), None, H, Dh, R, cs, sn, q, k, vt, n_pad)
        torch.cuda.synchronize()
        qkv = oracle.linear(a[rows], W, None)
        c, s = oracle.rope_cos_sin(m, lay["pos"][rows])
        refq = oracle.rope_apply(qkv[:, :d], H, Dh, R, c, s)
        refk = oracle.rope_apply(qkv[:, d:2 * d], H, Dh, R, c, s)
        refv = qkv[:, 2 * d:]
        gq = q.float().double().cpu().numpy()[rows]
        gk = k.float().double().cpu().numpy()[rows]
        gv = vt[:, torch.from_numpy(rows).cuda()].float().double().cpu().numpy().T
        bound = 2 * d * 2.0 ** -23 * (np.abs(a[rows]).astype(np.float64) @ np.abs(W).astype(np.float64).T).max()
        for g, r in ((gq, refq), (gk, refk), (gv, refv)):
            assert np.all(np.abs(g - r) <= BF16_REL * np.abs(r) + bound + 1e-5)
    elif which == "ffn_up":
        W, Wb = synth.normal(312, "w", (2 * F, d), 0.02, bf16=True)
        wp = torch.empty((2 * F, d), dtype=torch.bfloat16, device="cuda")
        bp = torch.empty((2 * F,), dtype=torch.float32, device="cuda")
        dit.pack_ffn_in(gu.dev_bf16(Wb), None, wp, bp)
        h = torch.empty((M, F), dtype=torch.bfloat16, device="cuda")
        dit.gemm_swiglu(gu.dev_bf16(ab), wp, bp, h)
        torch.cuda.synchronize()
        uv = oracle.linear(a[rows], W, None)
        ref = oracle.swiglu(uv)
        got = h.float().double().cpu().numpy()[rows]
        bound = d * 2.0 ** -23 * (np.abs(a[rows]).astype(np.float64) @ np.abs(W).astype(np.float64).T)
        prop = np.abs(uv[:, F:]) * bound[:, :F] + 1.1 * np.abs(uv[:, :F]) * bound[:, F:]
        assert np.all(np.abs(got - ref) <= BF16_REL * np.abs(ref) + prop + 1e-5)
    else:
        W, Wb = synth.normal(313, "w", (d, F), 0.02, bf16=True)
        x0 = synth.normal(313, "x", (M, d), 1.0)
        gate = synth.normal(313, "gate", (2, d), 0.2)
        tags = lay["tags"]
        x = gu.dev_f32(x0)
        dit.gemm_gated_residual(gu.dev_bf16(ab), gu.dev_bf16(Wb), None, x, gate=gu.dev_f32(gate), gate_stride=d,
                                tags=torch.from_numpy(tags).cuda())
        torch.cuda.synchronize()
        ref = x0[rows].astype(np.float64) + gate[tags[rows]].astype(np.float64) * oracle.linear(a[rows], W, None)
        got = x.double().cpu().numpy()[rows]
        bound = F * 2.0 ** -23 * (np.abs(a[rows]).astype(np.float64) @ np.abs(W).astype(np.float64).T)
        assert np.all(np.abs(got - ref) <= bound * np.abs(gate[tags[rows]]) + 1e-5)
    oracle.set_threads(1)


@pytest.mark.parametrize("name", ["video_audio_bf16", "long_doc_bf16"])
def test_full_forward_zero_gates_is_final_norm(name):
    """With every block's gate rows zero, each block is the identity, so the full-size forward must
    return the final norm + modulate of the input, row by row (checked on sampled rows)."""
    gu = _gu()
    w = synth.WORKLOADS[name]
    m = w["model"]
    d = m["hidden"]
    lay = synth.build_layout(w["docs"])
    W = synth.make_weights(w)
    for b, bb in zip(W["blocks"], W["bits"]["blocks"]):
        for arr in (b["w_ada"], bb["w_ada"], b["b_ada"], bb["b_ada"]):
            v = arr.reshape(m["n_mod"], 6, d, -1)
            v[:, 2] = 0
            v[:, 5] = 0
    run = gu.run_forward(w, layout=lay, weights=W)
    assert run["status"] == 0
    out = run["out"]
    assert np.isfinite(out).all()
    rows = _rows(lay["n_tokens"], 320, [0, lay["n_tokens"] - 1])
    _, modf = oracle.adaln(m, W, run["t"])
    x = run["x"][rows]
    ref = oracle.modulate(oracle.rms_norm(x, m["norm_eps"]), lay["tags"][rows], modf[:, 0], modf[:, 1])
    rms = np.sqrt((ref ** 2).mean())
    assert np.abs(out[rows] - ref).max() <= 3e-3 * rms
    run["handle"].close()


def test_full_latent_forward_zero_gates_sampled_rows():
    """The latent forward at the full 17,408-token size with every block's gate rows zero: each block
    is the identity, so v_m[r] = head_m(final norm + modulate(patch_m(z_m[r]))), all fp32, checked row
    by row against the oracle on sampled rows of each modality (row maps, scatter, gather, padding)."""
    gu = _gu()
    w = synth.WORKLOADS["video_audio_bf16"]
    m = w["model"]
    d = m["hidden"]
    lay = synth.build_layout(w["docs"])
    W = synth.make_weights(w)
    for b, bb in zip(W["blocks"], W["bits"]["blocks"]):
        for arr in (b["w_ada"], bb["w_ada"], b["b_ada"], bb["b_ada"]):
            v = arr.reshape(m["n_mod"], 6, d, -1)
            v[:, 2] = 0
            v[:, 5] = 0
    widths = synth.latent_widths()
    io = synth.make_latent_io(77, d, widths)
    z = synth.make_latents(77, lay, widths)
    h = gu.make_handle(m, lay, W)
    h.bind_latent_io({k: [None if a is None else gu.dev_f32(a) for a in v] for k, v in io.items()})
    dl = gu.dev_layout(lay)
    zd = [gu.dev_f32(a) for a in z]
    vd = [torch.full((a.shape[0], widths[k]), float("nan"), dtype=torch.float32, device="cuda")
          for k, a in enumerate(z)]
    ws = torch.empty(h.workspace_bytes_latent(lay["n_tokens"], lay["n_docs"]), dtype=torch.uint8, device="cuda")
    ts = [float(np.float32(0.91)), float(np.float32(0.47))]
    h.forward_latent(zd, dl["cu"], dl["ids"], dl["tags"], dl["pos"], ts, vd, ws)
    assert h.sync_status(ws) == 0
    _, modf = oracle.adaln(m, W, ts)
    oracle.set_threads(8)
    for k in range(2):
        got = vd[k].double().cpu().numpy()
        assert np.isfinite(got).all()
        sel = _rows(z[k].shape[0], 160, [0, z[k].shape[0] - 1])
        xk = oracle.linear(z[k][sel], io["w_patch"][k], io["b_patch"][k])
        tags = np.full(len(sel), k, dtype=np.uint8)
        yk = oracle.modulate(oracle.rms_norm(xk, m["norm_eps"]), tags, modf[:, 0], modf[:, 1])
        ref = oracle.linear(yk, io["w_head"][k], io["b_head"][k])
        # fp32 end to end here (no bf16 operand touches these rows): far inside the bf16 gate
        assert np.abs(got[sel] - ref).max() <= 1e-4 * np.sqrt((ref ** 2).mean()), k
    oracle.set_threads(1)
    h.close()


def test_full_forward_is_deterministic_and_counts_tiles():
    gu = _gu()
    w = synth.WORKLOADS["video_audio_bf16"]
    r1 = gu.run_forward(w)
    r2 = gu.run_forward(w, layout=r1["layout"], weights=r1["weights"], x=r1["x"], handle=r1["handle"])
    assert np.array_equal(r1["out"], r2["out"])
    assert r2["stats"]["attention_tiles"] == oracle.count_q_tiles(r1["layout"]["cu_seqlens"], _dit().attention_block_rows()) * w["model"]["n_heads"]
    r1["handle"].close()
