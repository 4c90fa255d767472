"""Comparison helpers shared by the GPU parity tests."""
import numpy as np
import torch

# Attention tolerance for BF16 inputs/outputs with fp32 accumulation, against the fp64
# oracle: every element within 1e-2 absolute, and every element whose reference
# magnitude is at least 1e-2 within 2e-2 relative (below 1e-2 the absolute bound rules).
ATOL = 1e-2
RTOL = 2e-2
REL_FLOOR = 1e-2


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def attention_errors(got, ref):
    got = to_f64(got) if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    d = np.abs(got - ref)
    big = np.abs(ref) >= REL_FLOOR
    max_abs = float(d.max()) if d.size else 0.0
    max_rel = float((d[big] / np.abs(ref[big])).max()) if big.any() else 0.0
    rel_l2 = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))
    return dict(max_abs=max_abs, max_rel=max_rel, rel_l2=rel_l2,
                finite=bool(np.isfinite(got).all()))


def assert_attention_close(got, ref, what=""):
    e = attention_errors(got, ref)
    assert e["finite"], f"{what}: non-finite output"
    assert e["max_abs"] <= ATOL and e["max_rel"] <= RTOL, f"{what}: {e}"
    return e
