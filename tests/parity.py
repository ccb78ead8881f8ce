"""Whole-forward parity gates shared by the GPU forward tests and the CPU mutation tests."""
import numpy as np

# Every block output within 3e-3 of its RMS (the bf16 stream's tolerance).
GATE = 3e-3
# The residual dwarfs each block's update x_out - x_in, so the update gets its own gate: bf16 GEMM
# operands put ~2^-9 relative noise on every product, so the update may differ by a few percent of its
# own magnitude, never by its size.
DELTA_MAX = 0.08
DELTA_RMS = 0.02


def forward_gates(x_in, dumps, ref_dumps, out, ref_out):
    """Return a list of failed gates (empty when the candidate passes)."""
    fails = []
    prev_g = prev_o = np.asarray(x_in, dtype=np.float64)
    for l in range(len(ref_dumps)):
        g, o = dumps[l], ref_dumps[l]
        rms = np.sqrt((o ** 2).mean())
        e = np.abs(g - o).max() / rms
        if not e <= GATE:
            fails.append(f"block {l}: max|dx| = {e:.2e} RMS")
        dg, do = g - prev_g, o - prev_o
        err = dg - do
        r1 = np.abs(err).max() / np.abs(do).max()
        r2 = np.sqrt((err ** 2).mean()) / np.sqrt((do ** 2).mean())
        if not r1 <= DELTA_MAX:
            fails.append(f"block {l}: update max error {r1:.2e} of max|update|")
        if not r2 <= DELTA_RMS:
            fails.append(f"block {l}: update rms error {r2:.2e} of rms(update)")
        prev_g, prev_o = g, o
    rms = np.sqrt((ref_out ** 2).mean())
    if not np.isfinite(out).all():
        fails.append("non-finite output")
    elif not np.abs(out - ref_out).max() <= GATE * rms:
        fails.append(f"output: max err {np.abs(out - ref_out).max() / rms:.2e} RMS")
    return fails
