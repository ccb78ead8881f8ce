"""Full-size parity with live gates, by per-layer teacher forcing.

The real forward runs at the full sizes the bench times (17,408 and 33,792 tokens; the loop's
17,408 + 9,216), with every AdaLN gate live.  For the first, middle and last block the oracle is fed
the GPU's own fp32 input to that block (so errors do not compound across blocks and each block is
judged alone) and computes that block's output on sampled query rows: every key and value of the
rows' documents, then the rows' attention, out-projection, gated residual and FFN.  The rows include
each document's first and last rows, the rows either side of the 128-row tiles where a document
starts or ends, the last video and first audio row, and seeded random rows.  Gates, on those rows:
the block output within 3e-3 of its RMS, and the block's update (output minus input) within 8% of
its largest and 2% of its RMS value.  The final layer is teacher-forced the same way from the GPU's
last block output.  The loop runs its 50 steps on the GPU; at steps 0, 25 and 49 its forward is
checked like this, and every step's Euler update is compared bit for bit with the oracle's fp32 step
on the GPU's own x and v."""
import os

import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.slow]

from tests.parity import DELTA_MAX, DELTA_RMS, GATE  # noqa: E402


def _gu():
    from tests import gpu_util
    return gpu_util


def _dit():
    from video_audio_gen_gb300 import dit
    return dit


def sample_rows(lay: dict, seed: int, per_doc: int = 48) -> np.ndarray:
    """Query rows to check: per document its ends, the rows around the 128-row tiles it starts and
    ends in, the video/audio boundary and seeded random rows."""
    cu, tags = lay["cu_seqlens"], lay["tags"]
    rows = []
    for j in range(lay["n_docs"]):
        a, b = int(cu[j]), int(cu[j + 1])
        cand = [a, a + 1, b - 2, b - 1]
        for edge in (a, b):
            t0 = edge // 128 * 128
            cand += [t0 - 1, t0, t0 + 127, t0 + 128]
        audio = np.nonzero(tags[a:b] == 1)[0]
        if audio.size:
            cand += [a + int(audio[0]) - 1, a + int(audio[0]), a + int(audio[-1])]
        cand += list(a + (synth.uniform(seed + j, "teacher rows", per_doc) * (b - a)).astype(np.int64))
        rows += [r for r in cand if a <= r < b]
    return np.unique(np.array(rows, dtype=np.int64))


def block_gate_failures(x_in, got, ref, what: str) -> list:
    """The bf16 stream's gates on sampled rows of one block: x_in, got, ref [rows, d]."""
    fails = []
    rms = np.sqrt((ref ** 2).mean())
    e = np.abs(got - ref).max() / rms
    dg, do = got - x_in, ref - x_in
    err = dg - do
    r1 = np.abs(err).max() / np.abs(do).max()
    r2 = np.sqrt((err ** 2).mean()) / np.sqrt((do ** 2).mean())
    print(f"{what}: max|dx| = {e:.2e} RMS; update error max {r1:.2e}, rms {r2:.2e}")
    if not e <= GATE:
        fails.append(f"{what}: max|dx| = {e:.2e} RMS")
    if not r1 <= DELTA_MAX:
        fails.append(f"{what}: update max error {r1:.2e} of max|update|")
    if not r2 <= DELTA_RMS:
        fails.append(f"{what}: update rms error {r2:.2e} of rms(update)")
    return fails


def _threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def check_forward_teacher_forced(m, W, lay, x_in, dump, out, t, rows, label):
    """Blocks 0, L/2 and L-1 and the final layer of one forward, each from the GPU's own input."""
    L = m["n_blocks"]
    mod, modf = oracle.adaln(m, W, t)
    fails = []
    oracle.set_threads(_threads())
    try:
        for l in sorted({0, L // 2, L - 1}):
            xb = x_in if l == 0 else dump[l - 1].cpu().numpy()
            got = dump[l][torch.from_numpy(rows).cuda()].double().cpu().numpy()
            ref = oracle.block_rows(m, W, l, mod[l], xb, lay, rows)
            assert np.isfinite(got).all(), f"{label} block {l}: non-finite rows"
            fails += block_gate_failures(xb[rows].astype(np.float64), got, ref, f"{label} block {l}")
        xl = dump[L - 1][torch.from_numpy(rows).cuda()].double().cpu().numpy()
        ref = oracle.final_rows(m, modf, xl, lay["tags"][rows])
        g = out[rows]
        e = np.abs(g - ref).max() / np.sqrt((ref ** 2).mean())
        print(f"{label} final layer: max|dv| = {e:.2e} RMS")
        if not e <= GATE:
            fails.append(f"{label} final layer: max|dv| = {e:.2e} RMS")
    finally:
        oracle.set_threads(1)
    return fails


@pytest.mark.parametrize("name", ["video_audio_bf16", "long_doc_bf16"])
def test_full_size_forward_teacher_forced(name):
    """17,408 tokens in 2 documents x 8 blocks, and one 33,792-token document x 4 blocks."""
    gu = _gu()
    w = synth.WORKLOADS[name]
    m = w["model"]
    L, d = m["n_blocks"], m["hidden"]
    lay = synth.build_layout(w["docs"])
    N, D = lay["n_tokens"], lay["n_docs"]
    W = synth.make_weights(w)
    x = synth.make_tokens(w, lay)
    t = synth.timestep(w)
    h = gu.make_handle(m, lay, W)
    dl = gu.dev_layout(lay)
    xd = gu.dev_f32(x)
    outd = torch.empty_like(xd)
    ws = gu.workspace(h, N, D)
    dump = torch.empty((L, N, d), dtype=torch.float32, device="cuda")
    h.set_dump(dump)
    h.forward(xd, dl["cu"], dl["ids"], dl["tags"], dl["pos"], t, outd, ws)
    st = h.sync_status(ws)
    h.set_dump(None)
    assert st == 0
    rows = sample_rows(lay, 900 + w["seed"])
    out = outd.double().cpu().numpy()
    fails = check_forward_teacher_forced(m, W, lay, x, dump, out, t, rows, name)
    h.close()
    assert not fails, fails


def test_full_size_denoise_loop_teacher_forced():
    """The 50-step loop on the two requests (17,408 + 9,216 tokens): the forwards of steps 0, 25 and
    49 teacher-forced block by block from the GPU's x_k, and all 50 Euler steps bit-exact against the
    oracle's fp32 step applied to the GPU's own x_k and v_k."""
    dit, gu = _dit(), _gu()
    w = synth.WORKLOADS["denoise_loop"]
    m = w["model"]
    L, d = m["n_blocks"], m["hidden"]
    lay = synth.build_layout(w["docs"])
    N, D = lay["n_tokens"], lay["n_docs"]
    W = synth.make_weights(w)
    x0 = synth.make_tokens(w, lay)
    sig = synth.sigmas(w["steps"])
    h = gu.make_handle(m, lay, W)
    dl = gu.dev_layout(lay)
    x = gu.dev_f32(x0)
    v = torch.empty_like(x)
    ws = gu.workspace(h, N, D)
    dump = torch.empty((L, N, d), dtype=torch.float32, device="cuda")
    rows = sample_rows(lay, 940)
    fails, euler_bad = [], []
    for i in range(w["steps"]):
        check = i in (0, 25, 49)
        if check:
            h.set_dump(dump)
        h.forward(x, dl["cu"], dl["ids"], dl["tags"], dl["pos"], float(sig[i]), v, ws)
        if check:
            h.set_dump(None)
        assert h.sync_status(ws) == 0, f"step {i}"
        xk, vk = x.cpu().numpy(), v.cpu().numpy()
        if check:
            fails += check_forward_teacher_forced(m, W, lay, xk, dump, vk.astype(np.float64), float(sig[i]), rows,
                                                  f"step {i}")
        dit.euler_step(x, v, float(sig[i]), float(sig[i + 1]))
        ref = oracle.euler_step(xk, vk, sig[i], sig[i + 1])
        if not np.array_equal(x.cpu().numpy().view(np.uint32), ref.view(np.uint32)):
            euler_bad.append(i)
    h.close()
    assert not euler_bad, f"Euler steps not bit-exact: {euler_bad}"
    assert not fails, fails
