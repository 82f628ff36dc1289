"""Error metrics and tolerances for GPU-vs-oracle parity.

Tolerances (fp16/bf16 inputs, fp32 accumulation):
  O    max |x - y| <= 1e-2 and ||x - y||_2 / ||y||_2 <= 5e-3
  L    max |x - y| <= 1e-3
  dQ, dK, dV   ||x - y||_2 / ||y||_2 <= 2e-2
with y the fp64 oracle.
"""
import json
import os

import numpy as np

O_MAX_ABS = 1e-2
O_REL_L2 = 5e-3
LSE_MAX_ABS = 1e-3
GRAD_REL_L2 = 2e-2


def to_np(t):
    if hasattr(t, "detach"):
        return t.detach().double().cpu().numpy()
    return np.asarray(t, dtype=np.float64)


def max_abs(x, ref) -> float:
    x, ref = to_np(x), to_np(ref)
    return float(np.abs(x - ref).max()) if x.size else 0.0


def rel_l2(x, ref) -> float:
    x, ref = to_np(x), to_np(ref)
    den = float(np.linalg.norm(ref))
    return float(np.linalg.norm(x - ref)) / (den if den > 0 else 1.0)


def record(what, **errs):
    """Append the measured errors to $FA_PARITY_LOG (JSON lines), if set."""
    path = os.environ.get("FA_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"case": what, **errs}) + "\n")


def check_forward(o, lse, o_ref, lse_ref, what=""):
    e1, e2, e3 = max_abs(o, o_ref), rel_l2(o, o_ref), max_abs(lse, lse_ref)
    record(what, o_max_abs=e1, o_rel_l2=e2, lse_max_abs=e3)
    assert np.isfinite(to_np(o)).all(), f"{what}: non-finite O"
    assert e1 <= O_MAX_ABS and e2 <= O_REL_L2 and e3 <= LSE_MAX_ABS, \
        f"{what}: O max_abs {e1:.3e} rel_l2 {e2:.3e}, LSE max_abs {e3:.3e}"
    return e1, e2, e3


def check_grads(pairs, what=""):
    errs = {}
    for name, x, ref in pairs:
        assert np.isfinite(to_np(x)).all(), f"{what}: non-finite {name}"
        errs[name] = rel_l2(x, ref)
    record(what, **{f"{k}_rel_l2": v for k, v in errs.items()})
    bad = {k: v for k, v in errs.items() if v > GRAD_REL_L2}
    assert not bad, f"{what}: gradient rel_l2 over {GRAD_REL_L2}: {errs}"
    return errs


def check_grads_tiled(pairs, tile=128, what=""):
    """Each (name, x, ref) of shape [heads, rows, d]: the rel_L2 bound of the
    gradients applied to every (head, 128-row tile) block on its own, so that
    one wrong tile cannot hide inside the norm of the whole tensor."""
    worst = {}
    for name, x, ref in pairs:
        x, ref = to_np(x), to_np(ref)
        assert x.shape == ref.shape and x.ndim == 3, (name, x.shape, ref.shape)
        w = 0.0
        for h in range(x.shape[0]):
            for r0 in range(0, x.shape[1], tile):
                e = rel_l2(x[h, r0:r0 + tile], ref[h, r0:r0 + tile])
                assert e <= GRAD_REL_L2, f"{what}: {name} head {h} rows {r0}.. rel_l2 {e:.3e}"
                w = max(w, e)
        worst[name] = w
    record(what + " (worst tile)", **{f"{k}_rel_l2": v for k, v in worst.items()})
    return worst
