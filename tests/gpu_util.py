"""Helpers shared by the GPU tests, the smoke check and the bench: upload seeded inputs, run the
library's forward through the C ABI, read results back.  No arithmetic of the method lives here."""
from __future__ import annotations

import numpy as np
import torch

import synth
from video_audio_gen_gb300 import dit


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev_f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def dev_u8(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def dev_layout(lay: dict) -> dict:
    return dict(cu=torch.from_numpy(lay["cu_seqlens"].astype(np.int32)).cuda(),
                ids=torch.from_numpy(lay["doc_ids"].astype(np.int32)).cuda(),
                tags=torch.from_numpy(lay["tags"].astype(np.uint8)).cuda(),
                pos=torch.from_numpy(lay["pos"].astype(np.float64)).cuda())


def upload_weights(W: dict, bf16: bool):
    """Device copies of the seeded weights in the model dtype (biases too)."""
    def up(name, f, b):
        if f is None:
            return None
        # matrices and biases in the model dtype; gains, shifts and residual scales (no bf16 bits) fp32
        return dev_bf16(b) if (bf16 and b is not None) else dev_f32(f)
    blocks = []
    for l, fb in enumerate(W["blocks"]):
        bb = W["bits"]["blocks"][l] if bf16 else {}
        blocks.append({n: up(n, fb[n], bb.get(n)) for n in fb})
    gb = W["bits"]["glob"] if bf16 else {}
    glob = {n: up(n, f, gb.get(n)) for n, f in W["glob"].items()}
    return blocks, glob


def make_handle(model: dict, lay: dict, W: dict, max_tokens=None, max_docs=None):
    h = dit.Dit(model, max_tokens or lay["n_tokens"], max_docs or lay["n_docs"])
    blocks, glob = upload_weights(W, model["dtype"] == "bf16")
    h.bind_weights(blocks, glob)
    return h


def workspace(h: dit.Dit, n_tokens: int, n_docs: int, host: bool = False, poison: bool = True) -> torch.Tensor:
    """Device workspace for a forward.  Poisoned with 0xFF bytes (NaN in every float format) by
    default: the forward must not depend on what the workspace held on entry."""
    nbytes = h.workspace_bytes(n_tokens, n_docs, host=host)
    assert nbytes > 0
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    if poison:
        ws.fill_(255)
    return ws


def run_forward(w: dict, dumps: bool = False, layout=None, weights=None, x=None, t=None, handle=None):
    """One forward of workload ``w`` (seeded inputs unless given).  ``t`` may be one flow time or a
    sequence with one per modality (the per-modality forward).  Returns numpy results."""
    lay = layout or synth.build_layout(w["docs"])
    W = weights or synth.make_weights(w)
    xin = synth.make_tokens(w, lay) if x is None else x
    tt = synth.timestep(w) if t is None else t
    m = w["model"]
    h = handle or make_handle(m, lay, W)
    dl = dev_layout(lay)
    xd = dev_f32(xin)
    out = torch.empty_like(xd)
    ws = workspace(h, lay["n_tokens"], lay["n_docs"])
    dump = None
    if dumps:
        dump = torch.empty((m["n_blocks"], lay["n_tokens"], m["hidden"]), dtype=torch.float32, device="cuda")
        h.set_dump(dump)
    if np.ndim(tt) == 0:
        h.forward(xd, dl["cu"], dl["ids"], dl["tags"], dl["pos"], tt, out, ws)
    else:  # one flow time per modality
        h.forward_modal(xd, dl["cu"], dl["ids"], dl["tags"], dl["pos"], list(tt), out, ws)
    st = h.sync_status(ws)
    torch.cuda.synchronize()
    if dumps:
        h.set_dump(None)
    return dict(out=out.double().cpu().numpy(), dumps=None if dump is None else dump.double().cpu().numpy(),
                status=st, stats=h.stats(), layout=lay, weights=W, x=xin, t=tt, handle=h)
