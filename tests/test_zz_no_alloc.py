"""dit_op_attention_noalloc against dit_op_attention, through the C ABI.

The no-allocation variant exists for callers that cannot call cudaMalloc (a plugin inside another
framework's executor with no allocator handed to it, a latency-critical serving thread that cannot
take cudaMalloc's implicit device synchronisation): its scratch lives in a fixed array inside the
library.  Two calls in a row with different layouts check that the shared array is reset between
calls: their results equal dit_op_attention's bit for bit.  This file is collected last so a failure here cannot hide any other test's result; it also
passes on its own in a fresh process.
"""
import numpy as np
import pytest

import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

BF16_REL = 2.0 ** -8


def _attention_inputs(docs, H, Dh, seed):
    from tests import gpu_util as gu
    lay = synth.build_layout(docs)
    n = lay["n_tokens"]
    n_pad = (n + 7) // 8 * 8
    _, qb = synth.normal(seed, "q", (n, H * Dh), 1.0, bf16=True)
    _, kb = synth.normal(seed, "k", (n, H * Dh), 1.0, bf16=True)
    v, vb = synth.normal(seed, "v", (n, H * Dh), 1.0, bf16=True)
    vt = np.zeros((H * Dh, n_pad), dtype=np.uint16)
    vt[:, :n] = vb.T
    return lay, n_pad, gu.dev_bf16(qb), gu.dev_bf16(kb), gu.dev_bf16(vt), gu.dev_layout(lay)["cu"], v


def test_attention_noalloc_matches_workspace_entry_point():
    from video_audio_gen_gb300 import build, dit
    build.build()
    cases = [(synth.WORKLOADS["ragged"]["docs"], 2, 128, 201),   # 4 documents, ragged ends
             (synth.WORKLOADS["tiny"]["docs"], 4, 64, 202)]      # then 2 documents, head dim 64
    for docs, H, Dh, seed in cases:                              # two calls in a row
        lay, n_pad, q, k, vt, cu, v = _attention_inputs(docs, H, Dh, seed)
        n = lay["n_tokens"]
        ws = torch.empty(dit.attention_workspace_bytes(lay["n_docs"], n), dtype=torch.uint8, device="cuda")
        ref = torch.empty((n, H * Dh), dtype=torch.bfloat16, device="cuda")
        dit.attention(q, k, vt, n_pad, cu, H, Dh, ref, ws)
        got = torch.full((n, H * Dh), float("nan"), dtype=torch.bfloat16, device="cuda")
        dit.attention_noalloc(q, k, vt, n_pad, cu, H, Dh, got)
        torch.cuda.synchronize()
        # the same kernels on the same inputs: the results agree bit for bit (a stale entry left in
        # the shared array by the previous call would show here)
        assert torch.equal(got, ref)
        assert dit.attention_noalloc_status() == (dit.DIT_OK, 0)
        g = got.float().double().cpu().numpy()
        assert np.isfinite(g).all() and np.abs(g).max() <= np.abs(v).max() * (1 + BF16_REL)


def test_attention_noalloc_reports_a_rejected_layout():
    """cu_seqlens that is not strictly increasing is rejected on the device: the output is left as it
    was, the call itself returns DIT_OK (its work is asynchronous), and the status reader returns
    DIT_ERR_LAYOUT with the validator's code 3; a valid call afterwards reads DIT_OK again."""
    from video_audio_gen_gb300 import build, dit
    build.build()
    lay, n_pad, q, k, vt, cu, _ = _attention_inputs(synth.WORKLOADS["tiny"]["docs"], 4, 64, 203)
    n = lay["n_tokens"]
    bad = torch.tensor([0, 160, 96], dtype=torch.int32, device="cuda")  # same sizes, decreasing
    o = torch.full((n, 4 * 64), 5.0, dtype=torch.bfloat16, device="cuda")
    dit.attention_noalloc(q, k, vt, n_pad, bad, 4, 64, o)
    assert dit.attention_noalloc_status() == (dit.DIT_ERR_LAYOUT, 3)
    assert (o == 5.0).all()
    dit.attention_noalloc(q, k, vt, n_pad, cu, 4, 64, o)
    assert dit.attention_noalloc_status() == (dit.DIT_OK, 0)
    assert torch.isfinite(o.float()).all() and not (o == 5.0).all()


def test_attention_noalloc_rejects_sizes_beyond_its_scratch():
    """More work items than the fixed array holds: rejected before any work is enqueued.  The inputs
    are real, correctly sized buffers, so nothing could be out of bounds even if it were not."""
    from video_audio_gen_gb300 import build, dit
    build.build()
    n_docs = 9000  # one token each: at least 9000 (document, q block) items > 8192
    n = n_docs
    n_pad = (n + 7) // 8 * 8
    q = torch.zeros((n, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros_like(q)
    vt = torch.zeros((128, n_pad), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    cu = torch.arange(n + 1, dtype=torch.int32, device="cuda")
    st = dit.lib().dit_op_attention_noalloc(q.data_ptr(), k.data_ptr(), vt.data_ptr(), n_pad, cu.data_ptr(), n_docs,
                                            n, 1, 128, o.data_ptr(), dit.DIT_ELEM_BF16, None)
    assert st == dit.DIT_ERR_CAPACITY
    assert b"fixed scratch" in dit.lib().dit_last_error(None)
