"""Acceptance checker for GPU outputs against the oracle's bf16-rounded reference.

Per launch (all computed on the host, in binary64):
  * element-wise  |c - ref| <= 0.02 |ref| + 0.01 rms(ref)   (rms over all of ref)
  * relL2         ||c - ref|| / ||ref|| <= 3e-3
  * no NaN in c   (outputs are NaN-poisoned before each launch)
The element-wise bound is the one that catches a band of rows computed with one
K tile missing or repeated; relL2 alone can miss it (ROCm/mori PR 785, Test).
"""
import numpy as np

REL_TOL = 0.02
RMS_TOL = 0.01
RELL2_TOL = 3e-3


def bf16_bits_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def check(c_bits, ref_bits, rms_ref=None):
    """Compare GPU bf16 bits with oracle bf16 bits.  Returns a dict; ``ok`` is the verdict.

    ``rms_ref`` overrides the rms of ``ref`` (for sampled checks of a large
    output, where it is estimated from the sample).
    """
    c = bf16_bits_to_f64(c_bits).ravel()
    r = bf16_bits_to_f64(ref_bits).ravel()
    nan = int(np.isnan(c).sum())
    if rms_ref is None:
        rms_ref = float(np.sqrt(np.mean(r * r))) if r.size else 0.0
    with np.errstate(invalid="ignore"):
        diff = np.abs(c - r)
        bound = REL_TOL * np.abs(r) + RMS_TOL * rms_ref
        bad = int(np.count_nonzero(~(diff <= bound)))  # NaN counts as bad
    nr = float(np.linalg.norm(r))
    if nan:
        rel = float("inf")
    else:
        rel = float(np.linalg.norm(c - r) / nr) if nr > 0 else float(np.linalg.norm(c))
    ok = nan == 0 and bad == 0 and rel <= RELL2_TOL
    worst = None
    if bad:
        with np.errstate(invalid="ignore"):
            excess = np.where(np.isnan(diff), np.inf, diff - bound)
        i = int(np.argmax(excess))
        worst = (i, float(c[i]), float(r[i]))
    return {"ok": ok, "bad": bad, "nan": nan, "rel_l2": rel, "rms_ref": rms_ref, "worst": worst}
