"""Shared helpers for the parity tests (comparison rules, device setup)."""
import numpy as np
import pytest
import torch

from oracle import formats as F

REL_L2_MAX = 5e-3        # layer outputs vs the oracle
COS_MIN = 0.9999
FP8_FLIP_FRAC = 1e-3     # FP8 intermediates: at most 0.1% of elements differ ...
FP8_MAX_STEPS = 1        # ... and by at most one E4M3 code step


def rel_l2(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def cosine(got, ref):
    got = np.asarray(got, np.float64).ravel()
    ref = np.asarray(ref, np.float64).ravel()
    return float(got @ ref / max(np.linalg.norm(got) * np.linalg.norm(ref), 1e-300))


def assert_close_layer(got, ref, what="output"):
    r, c = rel_l2(got, ref), cosine(got, ref)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    assert r <= REL_L2_MAX and c >= COS_MIN, f"{what}: rel_l2={r:.3e} cos={c:.7f}"
    return r, c


def _signed_step(codes):
    """E4M3 code -> signed position on the ordered grid (0 = zero)."""
    c = np.asarray(codes, np.int64)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def assert_mx_close(q_got, s_got, q_ref, s_ref, what="fp8"):
    """MXFP8 tensors [rows, C] / [rows, C/32]: a scale mismatch counts its whole
    block as differing; elements of matching blocks may differ by one code
    step; the differing elements stay below 0.1%."""
    q_got, q_ref = np.asarray(q_got), np.asarray(q_ref)
    s_got, s_ref = np.asarray(s_got), np.asarray(s_ref)
    rows, C = q_ref.shape
    blk_bad = (s_got != s_ref)
    step = np.abs(_signed_step(q_got) - _signed_step(q_ref)).reshape(rows, C // 32, 32)
    step = np.where(blk_bad[..., None], 0, step)
    assert step.max(initial=0) <= FP8_MAX_STEPS, f"{what}: element off by {step.max()} code steps"
    differing = blk_bad.sum() * 32 + (step > 0).sum()
    frac = differing / max(q_ref.size, 1)
    assert frac <= FP8_FLIP_FRAC, f"{what}: {differing} of {q_ref.size} elements differ ({frac:.2e})"
    return frac


def cuda_device():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return torch.device("cuda:0")


def np_(t):
    return t.detach().cpu().numpy()
