"""Latent I/O through the C ABI against the oracle: patchify / unpatchify / audio pack bit for bit,
the forward between latent tokens (fp32 patch projections and output heads around the block
stack), and the joint denoise loop run in latent token space with per-modality schedules."""
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


def _bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


# ------------------------------------------------------------------------------------------------
# packing: exact
# ------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("C,T,H,W,pt,ph,pw", [
    (48, 2, 4, 70, 1, 2, 2),    # the video recipe; W = 70 > the 63 patches one CTA stages: two runs per row
    (3, 2, 3, 2, 2, 2, 2),
    (1, 1, 1, 1, 1, 1, 1),
    (16, 3, 5, 50, 2, 4, 4),    # 512 features per token: runs of 23 patches
    (5, 1, 7, 9, 1, 3, 2),      # odd patch sizes
])
def test_patchify_and_unpatchify_bit_exact(C, T, H, W, pt, ph, pw):
    dit, gu = _dit(), _gu()
    lat = synth.normal(40, "lat", (C, T * pt, H * ph, W * pw), 1.0)
    ref = oracle.patchify(lat, pt, ph, pw)
    tok = torch.full(ref.shape, float("nan"), dtype=torch.float32, device="cuda")
    dit.patchify(gu.dev_f32(lat), pt, ph, pw, tok)
    got = tok.cpu().numpy()
    assert np.array_equal(_bits(got), _bits(ref))
    tok2 = synth.normal(40, "tok", ref.shape, 1.0)
    back = torch.full(lat.shape, float("nan"), dtype=torch.float32, device="cuda")
    dit.unpatchify(gu.dev_f32(tok2), C, T, H, W, pt, ph, pw, back)
    assert np.array_equal(_bits(back.cpu().numpy()), _bits(oracle.unpatchify(tok2, C, T, H, W, pt, ph, pw)))
    # the round trip on the device
    again = torch.empty_like(tok)
    dit.patchify(back, pt, ph, pw, again)
    assert np.array_equal(_bits(again.cpu().numpy()), _bits(tok2))


@pytest.mark.parametrize("C,T", [(32, 1000), (32, 1), (7, 3)])
def test_audio_pack_and_unpack_bit_exact(C, T):
    dit, gu = _dit(), _gu()
    lat = synth.normal(41, "alat", (C, T), 1.0)
    tok = torch.empty((T, C), dtype=torch.float32, device="cuda")
    dit.audio_pack(gu.dev_f32(lat), tok)
    assert np.array_equal(_bits(tok.cpu().numpy()), _bits(oracle.audio_pack(lat)))
    back = torch.empty((C, T), dtype=torch.float32, device="cuda")
    dit.audio_unpack(tok, back)
    assert np.array_equal(_bits(back.cpu().numpy()), _bits(lat))


def test_patchify_rejects_bad_arguments():
    dit = _dit()
    buf = torch.zeros(4 * 4 * 4, dtype=torch.float32, device="cuda")
    lib = dit.lib()
    p = buf.data_ptr()
    # each case is refused on the host, before any launch
    assert lib.dit_patchify(p, 1, 1, 1, 1, 1, 1, 1, p, None) == dit.DIT_ERR_INVALID_ARG          # overlap
    assert lib.dit_patchify(p, 0, 1, 1, 1, 1, 1, 1, p + 128, None) == dit.DIT_ERR_INVALID_ARG    # empty
    assert lib.dit_patchify(p, 4096, 1, 1, 1, 1, 2, 2, p + 128, None) == dit.DIT_ERR_UNSUPPORTED  # P too wide
    assert lib.dit_patchify(None, 1, 1, 1, 1, 1, 1, 1, p, None) == dit.DIT_ERR_INVALID_ARG


# ------------------------------------------------------------------------------------------------
# the forward between latent tokens
# ------------------------------------------------------------------------------------------------

def _latent_setup(w, seed_off=0):
    gu = _gu()
    lay = synth.build_layout(w["docs"])
    W = synth.make_weights(w)
    widths = synth.latent_widths()
    io = synth.make_latent_io(w["seed"] + 50 + seed_off, w["model"]["hidden"], widths)
    z = synth.make_latents(w["seed"] + 50 + seed_off, lay, widths)
    h = gu.make_handle(w["model"], lay, W)
    h.bind_latent_io({k: [None if a is None else gu.dev_f32(a) for a in v] for k, v in io.items()})
    return lay, W, widths, io, z, h


def _run_latent(h, lay, z, ts, widths, dump=None):
    gu = _gu()
    dl = gu.dev_layout(lay)
    zd = [gu.dev_f32(a) for a in z]
    vd = [torch.full((a.shape[0], widths[m]), float("nan"), dtype=torch.float32, device="cuda")
          for m, a in enumerate(z)]
    ws = torch.empty(h.workspace_bytes_latent(lay["n_tokens"], lay["n_docs"]), dtype=torch.uint8, device="cuda")
    ws.fill_(255)
    if dump is not None:
        h.set_dump(dump)
    h.forward_latent(zd, dl["cu"], dl["ids"], dl["tags"], dl["pos"], ts, vd, ws)
    st = h.sync_status(ws)
    if dump is not None:
        h.set_dump(None)
    return [a.double().cpu().numpy() for a in vd], st


@pytest.mark.parametrize("name", ["tiny", "ragged", "many_docs"])
def test_forward_latent_matches_oracle(name):
    w = synth.WORKLOADS[name]
    m = w["model"]
    lay, W, widths, io, z, h = _latent_setup(w)
    ts = [float(np.float32(0.83)), float(np.float32(0.31))]
    dump = torch.empty((m["n_blocks"], lay["n_tokens"], m["hidden"]), dtype=torch.float32, device="cuda")
    vs, st = _run_latent(h, lay, z, ts, widths, dump)
    assert st == 0
    oracle.set_threads(8)
    ref, ref_dumps = oracle.forward_latent(m, W, io, z, lay, ts, dumps=True)
    oracle.set_threads(1)
    # the residual after each block: the forward's gates, from the embedded input
    rows = [np.nonzero(lay["tags"] == k)[0] for k in range(2)]
    x_ref = np.zeros((lay["n_tokens"], m["hidden"]))
    for k in range(2):
        x_ref[rows[k]] = oracle.linear(z[k], io["w_patch"][k], io["b_patch"][k])
    fails = forward_gates(x_ref, dump.double().cpu().numpy(), ref_dumps, np.zeros(1), np.zeros(1))
    assert not fails, fails
    for k in range(2):
        rms = np.sqrt((ref[k] ** 2).mean())
        err = np.abs(vs[k] - ref[k]).max()
        assert np.isfinite(vs[k]).all() and err <= GATE * rms, (k, err / rms)


def test_forward_latent_counts_its_launches():
    w = synth.WORKLOADS["tiny"]
    lay, W, widths, io, z, h = _latent_setup(w)
    s0 = h.stats()
    h.set_kernel_timing(True)
    _, st = _run_latent(h, lay, z, [0.5, 0.5], widths)
    kt = h.kernel_times()
    h.set_kernel_timing(False)
    assert st == 0
    L = w["model"]["n_blocks"]
    s1 = h.stats()
    assert s1["forwards"] - s0["forwards"] == 1
    assert s1["gemm_launches"] - s0["gemm_launches"] == 4 * L
    # one row-map launch group, then a projection and a head per modality
    assert kt["latent_io"][1] == 1 + 2 + 2


def test_forward_latent_row_counts_must_match_the_tags():
    """n_rows that add up to n_tokens but disagree with the tags: the device check flags the layout
    (code 8) and the heads write nothing."""
    dit, gu = _dit(), _gu()
    w = synth.WORKLOADS["tiny"]
    lay, W, widths, io, z, h = _latent_setup(w)
    nv = z[0].shape[0]
    z_bad = [synth.normal(1, "zb0", (nv - 1, widths[0]), 1.0), synth.normal(1, "zb1", (z[1].shape[0] + 1, widths[1]),
                                                                             1.0)]
    vs, st = _run_latent(h, lay, z_bad, [0.5, 0.5], widths)
    assert st == dit.DIT_ERR_LAYOUT
    assert h.stats()["last_layout_error"] == 8
    assert all(np.isnan(v).all() for v in vs)


def test_forward_latent_rejects_bad_arguments():
    dit, gu = _dit(), _gu()
    w = synth.WORKLOADS["tiny"]
    lay, W, widths, io, z, h = _latent_setup(w)
    dl = gu.dev_layout(lay)
    ws = torch.empty(h.workspace_bytes_latent(lay["n_tokens"], lay["n_docs"]), dtype=torch.uint8, device="cuda")
    zd = [gu.dev_f32(a) for a in z]
    vd = [torch.empty_like(a) for a in zd]
    short = [zd[0][:-1], zd[1]]  # rows add up to n_tokens - 1
    with pytest.raises(dit.DitError) as e:
        h.forward_latent(short, dl["cu"], dl["ids"], dl["tags"], dl["pos"], [0.5, 0.5], vd, ws)
    assert e.value.status == dit.DIT_ERR_INVALID_ARG
    with pytest.raises(dit.DitError) as e:
        h.forward_latent(zd, dl["cu"], dl["ids"], dl["tags"], dl["pos"], [0.5, 0.5], vd, ws[:-256])
    assert e.value.status == dit.DIT_ERR_CAPACITY
    h2 = gu.make_handle(w["model"], lay, W)
    assert h2.workspace_bytes_latent(lay["n_tokens"], lay["n_docs"]) == 0
    with pytest.raises(dit.DitError) as e:
        h2.forward_latent(zd, dl["cu"], dl["ids"], dl["tags"], dl["pos"], [0.5, 0.5], vd, ws)
    assert e.value.status == dit.DIT_ERR_UNBOUND


# ------------------------------------------------------------------------------------------------
# the joint loop in latent token space
# ------------------------------------------------------------------------------------------------

LOOP_LATENT = dict(model=dict(synth.WORKLOADS["ragged"]["model"], hidden=256, n_heads=2, ffn_hidden=1024),
                   seed=45, docs=[dict(video=(2, 8, 16), audio=64), dict(video=(1, 8, 16), audio=64)],
                   t="schedule", steps=50, w_std=0.02, bias_std=0.0, x_std=1.0)


@pytest.mark.slow
def test_latent_denoise_loop_matches_oracle():
    """50 steps from noise: each step one latent forward at (sigma_v, sigma_a) and an Euler step of each
    modality's latent tokens on its own schedule (video shift 12, audio 3); GPU against the oracle."""
    dit, gu = _dit(), _gu()
    w = LOOP_LATENT
    lay, W, widths, io, z0, h = _latent_setup(w)
    base = synth.sigmas(50)
    sv = np.array([dit.time_shift(float(a), 12.0) for a in base], dtype=np.float32)
    sa = np.array([dit.time_shift(float(a), 3.0) for a in base], dtype=np.float32)
    dl = gu.dev_layout(lay)
    zd = [gu.dev_f32(a) for a in z0]
    vd = [torch.empty_like(a) for a in zd]
    ws = torch.empty(h.workspace_bytes_latent(lay["n_tokens"], lay["n_docs"]), dtype=torch.uint8, device="cuda")
    for i in range(50):
        h.forward_latent(zd, dl["cu"], dl["ids"], dl["tags"], dl["pos"], [sv[i], sa[i]], vd, ws)
        dit.euler_step(zd[0], vd[0], float(sv[i]), float(sv[i + 1]))
        dit.euler_step(zd[1], vd[1], float(sa[i]), float(sa[i + 1]))
    assert h.sync_status(ws) == 0
    zg = [a.cpu().numpy() for a in zd]
    oracle.set_threads(8)
    zo = [a.copy() for a in z0]
    for i in range(50):
        v, _ = oracle.forward_latent(w["model"], W, io, zo, lay, [float(sv[i]), float(sa[i])])
        zo[0] = oracle.euler_step(zo[0], v[0].astype(np.float32), sv[i], sv[i + 1])
        zo[1] = oracle.euler_step(zo[1], v[1].astype(np.float32), sa[i], sa[i + 1])
    oracle.set_threads(1)
    # each modality's decrements sum to 1, so the loop inherits the per-forward bound on v's scale
    for k in range(2):
        rms_z0 = np.sqrt((z0[k].astype(np.float64) ** 2).mean())
        err = np.abs(zg[k].astype(np.float64) - zo[k]).max()
        print(f"latent loop, modality {k}: max error {err:.3e}; gate GATE * RMS(z0) = {GATE * rms_z0:.3e}; "
              f"GATE * RMS(final z) = {GATE * np.sqrt((zo[k] ** 2).mean()):.3e}")
        assert err <= GATE * rms_z0, k


def test_forward_latent_with_an_empty_modality():
    """Documents without audio: the audio modality has no rows, its z / v pointers are NULL, and the
    video rows match the oracle."""
    gu = _gu()
    w = dict(synth.WORKLOADS["tiny"], docs=[dict(video=(2, 6, 8)), dict(video=(1, 4, 4))])
    m = w["model"]
    lay = synth.build_layout(w["docs"])
    assert (lay["tags"] == 0).all()
    W = synth.make_weights(w)
    widths = synth.latent_widths()
    io = synth.make_latent_io(52, m["hidden"], widths)
    z = synth.make_latents(52, lay, widths)
    assert z[1].shape[0] == 0
    h = gu.make_handle(m, lay, W)
    h.bind_latent_io({k: [None if a is None else gu.dev_f32(a) for a in v] for k, v in io.items()})
    dl = gu.dev_layout(lay)
    zd = [gu.dev_f32(z[0]), None]
    vd = [torch.full((z[0].shape[0], widths[0]), float("nan"), dtype=torch.float32, device="cuda"), None]
    ws = torch.empty(h.workspace_bytes_latent(lay["n_tokens"], lay["n_docs"]), dtype=torch.uint8, device="cuda")
    ts = [float(np.float32(0.6)), float(np.float32(0.2))]
    h.forward_latent(zd, dl["cu"], dl["ids"], dl["tags"], dl["pos"], ts, vd, ws)
    assert h.sync_status(ws) == 0
    ref, _ = oracle.forward_latent(m, W, io, z, lay, ts)
    got = vd[0].double().cpu().numpy()
    rms = np.sqrt((ref[0] ** 2).mean())
    assert np.isfinite(got).all() and np.abs(got - ref[0]).max() <= GATE * rms


def test_patchify_at_the_widest_token():
    """C*pt*ph*pw = 12287, the widest token one CTA stages: one patch per run."""
    dit, gu = _dit(), _gu()
    C, T, H, W, pt, ph, pw = 12287, 1, 1, 3, 1, 1, 1
    lat = synth.normal(42, "wide", (C, T * pt, H * ph, W * pw), 1.0)
    tok = torch.empty((T * H * W, C), dtype=torch.float32, device="cuda")
    dit.patchify(gu.dev_f32(lat), pt, ph, pw, tok)
    assert np.array_equal(_bits(tok.cpu().numpy()), _bits(oracle.patchify(lat, pt, ph, pw)))
