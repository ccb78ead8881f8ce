"""Whole-forward parity through the C ABI, against the oracle on the same seeded inputs, plus the
forward's invariants and its error paths."""
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


def check_against_oracle(w, run, ref_out, ref_dumps):
    fails = forward_gates(run["x"], run["dumps"], ref_dumps, run["out"], ref_out)
    assert not fails, fails


@pytest.mark.parametrize("name", ["tiny", "ragged", "many_docs"])
def test_forward_matches_oracle(name):
    gu = _gu()
    w = synth.WORKLOADS[name]
    run = gu.run_forward(w, dumps=True)
    assert run["status"] == 0
    oracle.set_threads(8)
    ref, dumps = oracle.forward(w["model"], run["weights"], run["x"], run["layout"], run["t"], dumps=True)
    oracle.set_threads(1)
    check_against_oracle(w, run, ref, dumps)


def _modal_t(seed):
    """Two different fp32 flow times (video, audio) drawn from the workload's seed."""
    u = synth.uniform(seed, "modal timesteps", 2)
    return [float(np.float32(u[0])), float(np.float32(0.5 * u[1]))]


@pytest.mark.parametrize("name", ["tiny", "ragged"])
def test_forward_modal_matches_oracle(name):
    """Video and audio at different flow times: every AdaLN row takes its own modality's timestep."""
    gu = _gu()
    w = synth.WORKLOADS[name]
    t = _modal_t(w["seed"] + 7)
    assert t[0] != t[1]
    run = gu.run_forward(w, dumps=True, t=t)
    assert run["status"] == 0
    oracle.set_threads(8)
    ref, dumps = oracle.forward(w["model"], run["weights"], run["x"], run["layout"], t, dumps=True)
    oracle.set_threads(1)
    check_against_oracle(w, run, ref, dumps)
    # Against the single-t forward at the video time: documents without audio never read an audio
    # AdaLN row and stay bit-identical; the audio rows differ.
    lay = run["layout"]
    one = gu.run_forward(w, layout=lay, weights=run["weights"], x=run["x"], t=t[0], handle=run["handle"])
    audio = lay["tags"] == 1
    has_audio = np.bincount(lay["doc_ids"][audio], minlength=lay["n_docs"]) > 0
    video_only = ~has_audio[lay["doc_ids"]]
    assert video_only.any() and audio.any()
    assert np.array_equal(one["out"][video_only].view(np.uint64), run["out"][video_only].view(np.uint64))
    assert not np.array_equal(one["out"][audio], run["out"][audio])


def test_forward_modal_equal_timesteps_is_forward():
    """All modalities at one t: bit-identical to dit_forward at that t."""
    gu = _gu()
    w = synth.WORKLOADS["ragged"]
    t = synth.timestep(w)
    r1 = gu.run_forward(w)
    r2 = gu.run_forward(w, layout=r1["layout"], weights=r1["weights"], x=r1["x"], t=[t, t], handle=r1["handle"])
    assert np.array_equal(r1["out"].view(np.uint64), r2["out"].view(np.uint64))


def test_forward_modal_rejects_bad_timesteps():
    dit, gu = _dit(), _gu()
    w = synth.WORKLOADS["tiny"]
    run = gu.run_forward(w)
    h, lay = run["handle"], run["layout"]
    dl = gu.dev_layout(lay)
    x = gu.dev_f32(run["x"])
    out = torch.full_like(x, 3.0)
    ws = gu.workspace(h, lay["n_tokens"], lay["n_docs"])
    for bad in ([0.5, 1.5], [-0.1, 0.5], [float("nan"), 0.5]):
        with pytest.raises(dit.DitError) as e:
            h.forward_modal(x, dl["cu"], dl["ids"], dl["tags"], dl["pos"], bad, out, ws)
        assert e.value.status == dit.DIT_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert (out == 3.0).all()


def test_forward_counters_and_tiles():
    """The CUDA path ran: launch counters and the device tile count are asserted, not printed."""
    gu = _gu()
    w = synth.WORKLOADS["ragged"]
    run = gu.run_forward(w)
    st = run["stats"]
    L = w["model"]["n_blocks"]
    assert st["forwards"] == 1
    assert st["gemm_launches"] == 4 * L and st["attention_launches"] == L and st["norm_launches"] == 2 * L + 1
    assert st["attention_tiles"] == oracle.count_q_tiles(run["layout"]["cu_seqlens"], _dit().attention_block_rows()) * w["model"]["n_heads"]
    assert st["device_status"] == 0 and st["last_layout_error"] == 0


def test_forward_is_deterministic():
    """Two forwards of the same inputs give the same bits (no race, no order-dependent reduction)."""
    gu = _gu()
    w = synth.WORKLOADS["ragged"]
    r1 = gu.run_forward(w)
    r2 = gu.run_forward(w, layout=r1["layout"], weights=r1["weights"], x=r1["x"], handle=r1["handle"])
    diff = np.nonzero((r1["out"] != r2["out"]).any(axis=1))[0]
    assert diff.size == 0, f"rows differing between identical forwards: {diff[:20].tolist()} ({diff.size})"


def test_segmentation_bit_identity():
    """Perturbing one document's tokens leaves every output row of the other documents bit-identical."""
    gu = _gu()
    w = synth.WORKLOADS["ragged"]
    lay = synth.build_layout(w["docs"])
    W = synth.make_weights(w)
    x = synth.make_tokens(w, lay)
    r1 = gu.run_forward(w, layout=lay, weights=W, x=x)
    cu = lay["cu_seqlens"]
    x2 = x.copy()
    x2[cu[1]:cu[2]] += synth.normal(5, "perturb", (cu[2] - cu[1], x.shape[1]), 0.5)
    r2 = gu.run_forward(w, layout=lay, weights=W, x=x2, handle=r1["handle"])
    other = np.ones(lay["n_tokens"], dtype=bool)
    other[cu[1]:cu[2]] = False
    bad = np.nonzero(other & (r1["out"] != r2["out"]).any(axis=1))[0]
    assert bad.size == 0, f"rows of unperturbed documents changed: {bad[:20].tolist()} ({bad.size})"
    assert not np.array_equal(r1["out"][~other], r2["out"][~other])


def test_nonfinite_document_does_not_reach_the_others():
    """NaN and Inf in one document's input tokens: every row of the other documents, including the
    neighbours that share its 128-token attention tiles, is finite and bit-identical to the clean run
    (the forward has no other cross-document step)."""
    gu = _gu()
    w = synth.WORKLOADS["many_docs"]
    lay = synth.build_layout(w["docs"])
    W = synth.make_weights(w)
    x = synth.make_tokens(w, lay)
    r1 = gu.run_forward(w, layout=lay, weights=W, x=x)
    cu = lay["cu_seqlens"]
    j = int(np.argmax([(cu[i] % 128 != 0) and (cu[i + 1] % 128 != 0) and cu[i + 1] - cu[i] > 100
                       for i in range(lay["n_docs"] - 1)]))
    a, b = int(cu[j]), int(cu[j + 1])
    assert a % 128 and b % 128 and j + 1 < lay["n_docs"]
    x2 = x.copy()
    x2[a:b:5, 3] = np.nan
    x2[a + 1:b:7, 11] = np.inf
    x2[b - 1, :] = -np.inf
    r2 = gu.run_forward(w, layout=lay, weights=W, x=x2, handle=r1["handle"])
    other = np.ones(lay["n_tokens"], dtype=bool)
    other[a:b] = False
    assert np.isfinite(r2["out"][other]).all()
    assert np.array_equal(r1["out"][other].view(np.uint64), r2["out"][other].view(np.uint64))
    assert not np.isfinite(r2["out"][a:b]).all()


def test_bf16_operand_forward_matches_oracle():
    """The act_bf16 configuration (bf16 operands throughout instead of f16) on the ragged case: the
    same gates at this width (its rounding only misses the tolerance on the full-width models)."""
    gu = _gu()
    w = synth.WORKLOADS["ragged"]
    wb = dict(w, model=dict(w["model"], act_bf16=True))
    run = gu.run_forward(wb, dumps=True)
    assert run["status"] == 0
    oracle.set_threads(8)
    ref, dumps = oracle.forward(w["model"], run["weights"], run["x"], run["layout"], run["t"], dumps=True)
    oracle.set_threads(1)
    check_against_oracle(wb, run, ref, dumps)
    # and the f16 operands are the more accurate of the two on the same inputs
    r16 = gu.run_forward(w, dumps=True, layout=run["layout"], weights=run["weights"], x=run["x"], t=run["t"])
    e16 = max(np.abs(r16["dumps"][l] - dumps[l]).max() for l in range(len(dumps)))
    e_bf = max(np.abs(run["dumps"][l] - dumps[l]).max() for l in range(len(dumps)))
    print(f"ragged: max block error f16 operands {e16:.3e}, bf16 operands {e_bf:.3e}")
    assert e16 < e_bf


def test_forward_host_equals_device_forward():
    gu = _gu()
    w = synth.WORKLOADS["tiny"]
    run = gu.run_forward(w)
    h, lay = run["handle"], run["layout"]
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    out = torch.empty(run["x"].shape, dtype=torch.float32).pin_memory()
    ws = gu.workspace(h, lay["n_tokens"], lay["n_docs"], host=True)
    h.forward_host(pin(run["x"]), pin(lay["cu_seqlens"].astype(np.int32)), pin(lay["doc_ids"].astype(np.int32)),
                   pin(lay["tags"]), pin(lay["pos"]), run["t"], out, ws)
    assert np.array_equal(out.double().numpy(), run["out"])


def test_device_validator_rejects_bad_layout():
    """A doc id that disagrees with cu_seqlens: the forward's kernels skip their work and the status
    word reads DIT_ERR_LAYOUT with the same code the oracle's layout check gives."""
    dit, gu = _dit(), _gu()
    w = synth.WORKLOADS["tiny"]
    lay = synth.build_layout(w["docs"])
    W = synth.make_weights(w)
    h = gu.make_handle(w["model"], lay, W)
    bad = dict(lay)
    bad["doc_ids"] = lay["doc_ids"].copy()
    bad["doc_ids"][100] = 0
    code = oracle.check_layout(bad["cu_seqlens"], bad["doc_ids"], bad["tags"], lay["n_tokens"], 2)
    assert code == 5
    dl = gu.dev_layout(bad)
    x = gu.dev_f32(synth.make_tokens(w, lay))
    out = torch.full_like(x, 7.0)
    ws = gu.workspace(h, lay["n_tokens"], lay["n_docs"])
    h.forward(x, dl["cu"], dl["ids"], dl["tags"], dl["pos"], 0.5, out, ws)
    assert h.sync_status(ws) == dit.DIT_ERR_LAYOUT
    assert h.stats()["last_layout_error"] == code
    assert (out == 7.0).all()  # nothing was written
    bad_tags = dict(lay)
    bad_tags["tags"] = lay["tags"].copy()
    bad_tags["tags"][5] = 9
    dl = gu.dev_layout(bad_tags)
    h.forward(x, dl["cu"], dl["ids"], dl["tags"], dl["pos"], 0.5, out, ws)
    assert h.sync_status(ws) == dit.DIT_ERR_LAYOUT and h.stats()["last_layout_error"] == 6
    # and a good layout afterwards runs normally on the same handle and workspace
    dl = gu.dev_layout(lay)
    h.forward(x, dl["cu"], dl["ids"], dl["tags"], dl["pos"], 0.5, out, ws)
    assert h.sync_status(ws) == dit.DIT_OK


def test_host_validation_errors_launch_nothing():
    dit, gu = _dit(), _gu()
    w = synth.WORKLOADS["tiny"]
    lay = synth.build_layout(w["docs"])
    W = synth.make_weights(w)
    h = gu.make_handle(w["model"], lay, W)
    dl = gu.dev_layout(lay)
    x = gu.dev_f32(synth.make_tokens(w, lay))
    out = torch.empty_like(x)
    ws = gu.workspace(h, lay["n_tokens"], lay["n_docs"])
    before = h.stats()["kernels_launched"]
    with pytest.raises(dit.DitError) as e:
        h.forward(x, dl["cu"], dl["ids"], dl["tags"], dl["pos"], 0.5, out, ws[:1024])
    assert e.value.status == dit.DIT_ERR_CAPACITY
    with pytest.raises(dit.DitError) as e:
        h.forward(x, dl["cu"], dl["ids"], dl["tags"], dl["pos"], 0.5, x, ws)
    assert e.value.status == dit.DIT_ERR_INVALID_ARG
    assert h.stats()["kernels_launched"] == before


def test_missing_weight_is_named():
    dit, gu = _dit(), _gu()
    w = synth.WORKLOADS["tiny"]
    W = synth.make_weights(w)
    blocks, glob = gu.upload_weights(W, True)
    blocks[1]["w_down"] = None
    h = dit.Dit(w["model"], 256, 2)
    with pytest.raises(dit.DitError) as e:
        h.bind_weights(blocks, glob)
    assert e.value.status == dit.DIT_ERR_MISSING_WEIGHT and "blocks[1].w_down" in str(e.value)
    x = torch.zeros((256, 256), device="cuda")
    with pytest.raises(dit.DitError) as e:
        h.forward(x, torch.zeros(3, dtype=torch.int32, device="cuda"), torch.zeros(256, dtype=torch.int32, device="cuda"),
                  torch.zeros(256, dtype=torch.uint8, device="cuda"), torch.zeros((256, 3), dtype=torch.float64,
                                                                                device="cuda"),
                  0.5, torch.empty_like(x), torch.empty(1 << 20, dtype=torch.uint8, device="cuda"))
    assert e.value.status == dit.DIT_ERR_UNBOUND


# ------------------------------------------------------------------------------------------------
# the denoise loop
# ------------------------------------------------------------------------------------------------

LOOP_SMALL = dict(model=dict(synth.WORKLOADS["ragged"]["model"], hidden=256, n_heads=2, ffn_hidden=1024),
                  seed=44, docs=[dict(video=(2, 8, 16), audio=64), dict(video=(1, 8, 16), audio=64)],
                  t="schedule", steps=50, w_std=0.02, bias_std=0.0, x_std=1.0)


def _loop_gate(xg, xo, x0, what):
    """The loop's gate, GATE x the RMS of the initial noise x0, printed beside the measured error and
    beside the RMS of the oracle's final x (the gate's scale before it was tied to the noise)."""
    err = float(np.abs(xg.astype(np.float64) - xo).max())
    rms_x0 = float(np.sqrt((x0.astype(np.float64) ** 2).mean()))
    rms_final = float(np.sqrt((xo ** 2).mean()))
    print(f"loop ({what}): max|x_gpu - x_oracle| = {err:.3e}; gate GATE * RMS(x0) = {GATE * rms_x0:.3e}; "
          f"GATE * RMS(final x) = {GATE * rms_final:.3e}; error / RMS(x0) = {err / rms_x0:.2e}")
    assert err <= GATE * rms_x0


def _gpu_loop(h, lay, x0, sig, start=0, stop=None, x_from=None):
    dit, gu = _dit(), _gu()
    dl = gu.dev_layout(lay)
    x = gu.dev_f32(x0 if x_from is None else x_from)
    v = torch.empty_like(x)
    ws = gu.workspace(h, lay["n_tokens"], lay["n_docs"])
    stop = len(sig) - 1 if stop is None else stop
    for i in range(start, stop):
        h.forward(x, dl["cu"], dl["ids"], dl["tags"], dl["pos"], float(sig[i]), v, ws)
        dit.euler_step(x, v, float(sig[i]), float(sig[i + 1]))
    assert h.sync_status(ws) == 0
    return x.cpu().numpy()


@pytest.mark.slow
def test_denoise_loop_matches_oracle_reduced():
    """50 Euler steps on a reduced copy of the two-request loop, every forward and step on the GPU,
    against the same 50 steps in the oracle."""
    gu = _gu()
    w = LOOP_SMALL
    lay = synth.build_layout(w["docs"])
    W = synth.make_weights(w)
    x0 = synth.make_tokens(w, lay)
    sig = synth.sigmas(50)
    h = gu.make_handle(w["model"], lay, W)
    xg = _gpu_loop(h, lay, x0, sig)
    oracle.set_threads(8)
    xo = x0.copy()
    for i in range(50):
        v, _ = oracle.forward(w["model"], W, xo, lay, float(sig[i]))
        xo = oracle.euler_step(xo, v.astype(np.float32), sig[i], sig[i + 1])
    oracle.set_threads(1)
    # Each step moves x by (sigma_next - sigma) * v, and the steps' sigma decrements sum to 1, so the
    # loop inherits the per-forward bound on v's scale, which is the initial noise's RMS; the final x
    # itself nearly cancels (x0 - sum dsigma v) and is no scale to measure against.
    _loop_gate(xg, xo, x0, "single schedule")


def _gpu_loop_modal(h, lay, x0, sig_v, sig_a):
    dit, gu = _dit(), _gu()
    dl = gu.dev_layout(lay)
    x = gu.dev_f32(x0)
    v = torch.empty_like(x)
    ws = gu.workspace(h, lay["n_tokens"], lay["n_docs"])
    for i in range(len(sig_v) - 1):
        h.forward_modal(x, dl["cu"], dl["ids"], dl["tags"], dl["pos"], [sig_v[i], sig_a[i]], v, ws)
        dit.euler_step_modal(x, v, dl["tags"], [sig_v[i], sig_a[i]], [sig_v[i + 1], sig_a[i + 1]])
    assert h.sync_status(ws) == 0
    return x.cpu().numpy()


@pytest.mark.slow
def test_denoise_loop_shifted_modal_schedules_match_oracle():
    """The joint loop with separate schedules: video sigmas shifted by 12, audio by 3 (tag 0 = video,
    1 = audio), each forward at the pair (sigma_v, sigma_a) and each token stepped on its own
    modality's pair; 50 steps on the GPU against the same 50 in the oracle."""
    dit, gu = _dit(), _gu()
    w = LOOP_SMALL
    lay = synth.build_layout(w["docs"])
    W = synth.make_weights(w)
    x0 = synth.make_tokens(w, lay)
    base = synth.sigmas(50)
    sv = np.array([dit.time_shift(float(s), 12.0) for s in base], dtype=np.float32)
    sa = np.array([dit.time_shift(float(s), 3.0) for s in base], dtype=np.float32)
    assert np.array_equal(sv.view(np.uint32), oracle.sigmas_shifted(base, 12.0).view(np.uint32))
    assert np.array_equal(sa.view(np.uint32), oracle.sigmas_shifted(base, 3.0).view(np.uint32))
    h = gu.make_handle(w["model"], lay, W)
    xg = _gpu_loop_modal(h, lay, x0, [float(a) for a in sv], [float(a) for a in sa])
    oracle.set_threads(8)
    xo = x0.copy()
    for i in range(50):
        v, _ = oracle.forward(w["model"], W, xo, lay, [float(sv[i]), float(sa[i])])
        xo = oracle.euler_step_tagged(xo, v.astype(np.float32), lay["tags"], [sv[i], sa[i]], [sv[i + 1], sa[i + 1]])
    oracle.set_threads(1)
    # the same bound as the single-schedule loop: each modality's decrements still sum to 1
    _loop_gate(xg, xo, x0, "shifted schedules")


def test_denoise_loop_resume_is_bit_identical():
    """The loop state is x alone: stopping after step k and resuming from the saved x reproduces the
    uninterrupted run bit for bit."""
    gu = _gu()
    w = LOOP_SMALL
    lay = synth.build_layout(w["docs"])
    W = synth.make_weights(w)
    x0 = synth.make_tokens(w, lay)
    sig = synth.sigmas(50)
    h = gu.make_handle(w["model"], lay, W)
    full = _gpu_loop(h, lay, x0, sig, 0, 6)
    part = _gpu_loop(h, lay, x0, sig, 0, 3)
    resumed = _gpu_loop(h, lay, x0, sig, 3, 6, x_from=part)
    assert np.array_equal(full.view(np.uint32), resumed.view(np.uint32))


# ------------------------------------------------------------------------------------------------
# the fp32 forward (music DiT shape)
# Gates: every layer output within 1e-5 of its RMS with a 1e-6 absolute floor,
# max|g - r| <= max(1e-5 * RMS(r), 1e-6), and the per-element form |g - r| <= 1e-5 |r| + 1e-6.
# The per-element form is asserted on the small case.  On the full 24-block shape each layer's count
# of elements outside it and its worst ratio |g - r| / (1e-5 |r| + 1e-6) are printed: there the
# elements whose value is near zero carry the absolute rounding of K = 8192 fp32 sums.
# ------------------------------------------------------------------------------------------------

FP32_REL, FP32_ABS = 1e-5, 1e-6


def _fp32_check(w, run, ref_out, ref_dumps, per_element):
    layers = [(run["dumps"][l], ref_dumps[l]) for l in range(w["model"]["n_blocks"])] + [(run["out"], ref_out)]
    worst = 0.0
    for i, (g, o) in enumerate(layers):
        err = np.abs(g - o).max()
        rms = np.sqrt((o ** 2).mean())
        ratio = np.abs(g - o) / (FP32_REL * np.abs(o) + FP32_ABS)
        bad = ratio > 1.0
        name = f"block {i}" if i < len(layers) - 1 else "output"
        print(f"{w['model']['n_blocks']}-block fp32 {name}: max|g - r| / RMS = {err / rms:.3e}; per-element "
              f"violations {int(bad.sum())} of {bad.size} ({bad.mean():.2e}), worst ratio {ratio.max():.3f}, at "
              f"|r| = {np.abs(o).reshape(-1)[int(ratio.argmax())]:.3e}")
        assert err <= max(FP32_REL * rms, FP32_ABS), (i, float(err), float(rms))
        worst = max(worst, float(err / rms))
        if per_element:
            assert not bad.any(), (i, int(bad.sum()), float(err))
    return worst


@pytest.mark.parametrize("name", ["music_small", pytest.param("music_fp32", marks=pytest.mark.slow)])
def test_fp32_forward_matches_oracle(name):
    """LayerNorm, partial rotary, ungated residuals, value * silu(gate), 1x1 pre/post convolutions as
    frame-major GEMMs, fp32 throughout; the music-DiT shape runs its full 24 blocks on 172 tokens."""
    gu = _gu()
    w = synth.WORKLOADS[name]
    run = gu.run_forward(w, dumps=True)
    assert run["status"] == 0
    assert run["out"].shape == run["x"].shape
    oracle.set_threads(16)
    ref, dumps = oracle.forward(w["model"], run["weights"], run["x"], run["layout"], run["t"], dumps=True)
    oracle.set_threads(1)
    worst = _fp32_check(w, run, ref, dumps, per_element=(name == "music_small"))
    print(f"{name}: worst max|g - r| / RMS over the layer outputs = {worst:.3e}")


# ------------------------------------------------------------------------------------------------
# failure detection without a GPU fault
# ------------------------------------------------------------------------------------------------

def test_bounded_wait_runs_out_reports_and_leaves_context_usable():
    """A wait on an mbarrier that nothing arrives at (the flag nobody sets) ends after its limit with
    the timeout recorded in the status word; the next forward on the same context runs normally."""
    dit, gu = _dit(), _gu()
    word = torch.zeros(1, dtype=torch.int32, device="cuda")
    import time
    t0 = time.perf_counter()
    assert dit.selftest_wait_timeout(1_000_000, word) == dit.DIT_ERR_DEVICE_TIMEOUT  # 1 ms limit
    assert time.perf_counter() - t0 < 5.0
    assert int(word.item()) & 1  # kDevTimeout
    run = gu.run_forward(synth.WORKLOADS["tiny"])
    assert run["status"] == 0 and np.isfinite(run["out"]).all()
