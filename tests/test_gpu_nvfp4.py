"""The whole forward with NVFP4 weights ([H3] "What this push adds": the NVFP4 checkpoint's
projections carry E2M1 codes two per byte, an E4M3 scale per 16 along K and an fp32 global scale).
The four linear maps of every block run on the NVFP4 GEMM (codes * scales expanded to f16 in shared
memory, f16 activations, the global scale on the accumulator); everything else is the bf16 model.
The oracle runs its forward on the dequantised weights (exact in fp32 with a power-of-two global
scale), so the gates are those of the bf16 stream."""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from tests.parity import forward_gates  # noqa: E402


def _gu():
    from tests import gpu_util
    return gpu_util


def nvfp4_model(w):
    return dict(w, model=dict(w["model"], nvfp4=True))


def dequantised_weights(W, nv):
    """The oracle's weights: the four linear maps of every block replaced by their NVFP4 values."""
    names = {"qkv": "w_qkv", "o": "w_o", "in": "w_in", "down": "w_down"}
    blocks = []
    for b, lin in zip(W["blocks"], nv):
        b = dict(b)
        for n, (q, s, g) in lin.items():
            b[names[n]] = oracle.nvfp4_dequant(q, s, g)
        blocks.append(b)
    return dict(W, blocks=blocks)


def run_nvfp4(w, dumps=True):
    gu = _gu()
    wn = nvfp4_model(w)
    lay = synth.build_layout(w["docs"])
    W = synth.make_weights(w)
    nv = synth.make_nvfp4_linears(w)
    h = gu.make_handle(wn["model"], lay, W)
    dev = [{n: (torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), g) for n, (q, s, g) in b.items()} for b in nv]
    h.bind_nvfp4(dev)
    run = gu.run_forward(wn, dumps=dumps, layout=lay, weights=W, handle=h)
    return run, W, nv


@pytest.mark.parametrize("name", ["tiny", "ragged", "many_docs"])
def test_nvfp4_forward_matches_oracle(name):
    w = synth.WORKLOADS[name]
    run, W, nv = run_nvfp4(w)
    assert run["status"] == 0
    oracle.set_threads(8)
    ref, dumps = oracle.forward(w["model"], dequantised_weights(W, nv), run["x"], run["layout"], run["t"], dumps=True)
    oracle.set_threads(1)
    fails = forward_gates(run["x"], run["dumps"], dumps, run["out"], ref)
    assert not fails, fails
    st = run["stats"]
    assert st["gemm_launches"] == 4 * w["model"]["n_blocks"]


def test_nvfp4_forward_differs_from_the_bf16_weights_it_does_not_use():
    """The bf16 matrices passed to dit_bind_weights are ignored with nvfp4 = 1: zeroing them changes
    nothing, bit for bit (the NVFP4 weights are the ones that run)."""
    gu = _gu()
    w = synth.WORKLOADS["tiny"]
    run, W, nv = run_nvfp4(w, dumps=False)
    W0 = {"blocks": [dict(b) for b in W["blocks"]], "glob": W["glob"],
          "bits": {"blocks": [dict(b) for b in W["bits"]["blocks"]], "glob": W["bits"]["glob"]}}
    for b, bb in zip(W0["blocks"], W0["bits"]["blocks"]):
        for n in ("w_qkv", "w_o", "w_in", "w_down"):
            b[n] = np.zeros_like(b[n])
            bb[n] = np.zeros_like(bb[n])
    wn = nvfp4_model(w)
    h = gu.make_handle(wn["model"], run["layout"], W0)
    h.bind_nvfp4([{n: (torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), g) for n, (q, s, g) in b.items()}
                  for b in nv])
    r2 = gu.run_forward(wn, layout=run["layout"], weights=W0, x=run["x"], t=run["t"], handle=h)
    assert np.array_equal(run["out"].view(np.uint64), r2["out"].view(np.uint64))


def test_nvfp4_forward_before_bind_is_refused():
    gu = _gu()
    from video_audio_gen_gb300 import dit
    w = synth.WORKLOADS["tiny"]
    wn = nvfp4_model(w)
    lay = synth.build_layout(w["docs"])
    W = synth.make_weights(w)
    h = gu.make_handle(wn["model"], lay, W)
    with pytest.raises(dit.DitError) as e:
        gu.run_forward(wn, layout=lay, weights=W, handle=h)
    assert e.value.status == dit.DIT_ERR_UNBOUND
