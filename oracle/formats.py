"""Number formats of the routed-MoE layer, decoded exactly in fp64.

TEST INFRASTRUCTURE ONLY: this package is the CPU oracle. Only the tests,
the smoke check and the benchmark's CPU-baseline leg may import it; the
product path never does.

The pages name the formats without defining them (NVIDIA blog "Boosting MoE
training throughput with advanced fusion kernels", section on fusing MXFP8 /
NVFP4 quantisation; GC-MoE summary, key contributions: FP8 x FP4 grouped
GEMM). The definitions used here are the OCP Microscaling (MX) v1.0 element
and scale formats, which those names refer to:

* E2M1 (FP4): sign bit 3, exponent bits 2..1 with bias 1, mantissa bit 0;
  exponent 0 is subnormal (m * 0.5). Magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6.
* E4M3 (FP8, "FN" variant): sign bit 7, exponent bits 6..3 with bias 7,
  mantissa bits 2..0; exponent 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN,
  there is no infinity; the largest finite magnitude is 448.
* E8M0 (MX scale): the byte c means 2^(c-127); 0xFF is NaN.

Activation quantisation (MXFP8, blocks of 32): the pages give no rule for the
block scale. Reading taken: the block exponent e is the smallest integer with
amax <= 448 * 2^e (so no element ever saturates), clamped to [-127, 127], and
e = -127 for an all-zero block; elements are E4M3 round-to-nearest-even of
v / 2^e.

Parity pins for everything here live in tests/test_oracle_formats.py.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def _e2m1_value(code: int) -> float:
    s = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return s * m * 0.5
    return s * 2.0 ** (e - 1) * (1.0 + m / 2.0)


def _e4m3_value(code: int) -> float:
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * 2.0 ** (e - 7) * (1.0 + m / 8.0)


def _e8m0_value(code: int) -> float:
    if code == 0xFF:
        return float("nan")
    return 2.0 ** (code - 127)


E2M1_TABLE = np.array([_e2m1_value(c) for c in range(16)], dtype=np.float64)
E4M3_TABLE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)
E8M0_TABLE = np.array([_e8m0_value(c) for c in range(256)], dtype=np.float64)

# non-negative finite E4M3 magnitudes in code order 0x00..0x7E (increasing)
_E4M3_POS = E4M3_TABLE[:0x7F].copy()


def decode_e2m1_packed(b: np.ndarray) -> np.ndarray:
    """Bytes [..., K/2] holding two E2M1 codes each -> fp64 [..., K].
    Element 2i sits in the low nibble of byte i (reading taken: the pages do
    not say which nibble comes first)."""
    b = np.asarray(b, dtype=np.uint8)
    lo = E2M1_TABLE[b & 0xF]
    hi = E2M1_TABLE[b >> 4]
    out = np.empty(b.shape[:-1] + (b.shape[-1] * 2,), dtype=np.float64)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def decode_e4m3(c: np.ndarray) -> np.ndarray:
    return E4M3_TABLE[np.asarray(c, dtype=np.uint8)]


def decode_e8m0(c: np.ndarray) -> np.ndarray:
    return E8M0_TABLE[np.asarray(c, dtype=np.uint8)]


def rne_e4m3(x: np.ndarray) -> np.ndarray:
    """E4M3 code of the representable value nearest to x (fp64 in).

    Ties go to the code with an even mantissa (round-half-to-even); beyond
    448 the result saturates to +-448. The sign of x is kept, so a negative
    value that rounds to zero gives 0x80. NaN maps to 0x7F.
    """
    x = np.asarray(x, dtype=np.float64)
    mag = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.searchsorted(_E4M3_POS, mag, side="left")     # first value >= mag
    hi = np.clip(hi, 0, len(_E4M3_POS) - 1)
    lo = np.clip(hi - 1, 0, len(_E4M3_POS) - 1)
    d_hi = _E4M3_POS[hi] - mag
    d_lo = mag - _E4M3_POS[lo]
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))
    code = np.where(pick_lo, lo, hi).astype(np.uint8)
    neg = np.signbit(x)
    code = np.where(neg, code | 0x80, code).astype(np.uint8)
    code = np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)
    return code


def mx_block_exponent(amax: np.ndarray) -> np.ndarray:
    """Smallest integer e with amax <= 448 * 2^e, clamped to [-127, 127];
    -127 for amax == 0. Found by exact fp64 comparisons around a log2 guess."""
    amax = np.asarray(amax, dtype=np.float64)
    out = np.full(amax.shape, -127, dtype=np.int64)
    flat_a = amax.reshape(-1)
    flat_o = out.reshape(-1)
    for i, a in enumerate(flat_a):
        if not a > 0.0:
            continue
        e = int(np.floor(np.log2(a / E4M3_MAX)))
        while a > E4M3_MAX * 2.0 ** e:
            e += 1
        while a <= E4M3_MAX * 2.0 ** (e - 1):
            e -= 1
        flat_o[i] = min(max(e, -127), 127)
    return out


def mx_quantize(v: np.ndarray):
    """MXFP8-quantise v [..., K] along its last axis in blocks of 32.
    Returns (E4M3 codes uint8 [..., K], E8M0 scale codes uint8 [..., K/32])."""
    v = np.asarray(v, dtype=np.float64)
    K = v.shape[-1]
    assert K % 32 == 0, K
    blk = v.reshape(v.shape[:-1] + (K // 32, 32))
    e = mx_block_exponent(np.abs(blk).max(axis=-1))
    scaled = blk / np.exp2(e.astype(np.float64))[..., None]
    codes = rne_e4m3(scaled).reshape(v.shape)
    return codes, (e + 127).astype(np.uint8)


def mx_dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Inverse of mx_quantize's encoding: E4M3 value * 2^(scale-127)."""
    q = decode_e4m3(codes)
    K = q.shape[-1]
    s = decode_e8m0(scales)
    return (q.reshape(q.shape[:-1] + (K // 32, 32)) * s[..., None]).reshape(q.shape)


def nvfp4_dequantize(packed: np.ndarray, scales: np.ndarray, gs: float) -> np.ndarray:
    """NVFP4 matrix [N, K/2] bytes + E4M3 scales [N, K/16] + fp32 per-tensor
    scale -> fp64 [N, K] = E2M1 * E4M3 scale (blocks of 16 along K) * gs."""
    q = decode_e2m1_packed(packed)
    N, K = q.shape[-2], q.shape[-1]
    s = decode_e4m3(scales)
    w = q.reshape(q.shape[:-1] + (K // 16, 16)) * s[..., None]
    return w.reshape(q.shape) * float(gs)


def mxfp4_dequantize(packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """MXFP4 matrix [N, K/2] bytes (two E2M1 codes each, element 2i in the low
    nibble) + E8M0 scales [N, K/32] -> fp64 [N, K] = E2M1 value * 2^(s - 127)
    per block of 32 along K (OCP MX: the FP4 element format with the shared
    E8M0 scale, the GC-MoE summary's "(1,1,32)" scale recipe)."""
    q = decode_e2m1_packed(packed)
    K = q.shape[-1]
    s = decode_e8m0(scales)
    return (q.reshape(q.shape[:-1] + (K // 32, 32)) * s[..., None]).reshape(q.shape)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Raw bfloat16 bit patterns (uint16/int16) -> exact fp64 values."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16(v: np.ndarray) -> np.ndarray:
    """fp64 -> nearest bfloat16 (ties to even), returned as uint16 patterns.
    Rounds from fp64 directly (no double rounding through fp32)."""
    v = np.asarray(v, dtype=np.float64)
    out = np.zeros(v.shape, dtype=np.uint16)
    flat_v = v.reshape(-1)
    flat_o = out.reshape(-1)
    # candidate truncation in fp32 then exact neighbour comparison in fp64
    f = flat_v.astype(np.float32)
    bits = f.view(np.uint32) & np.uint32(0xFFFF0000)
    lo = bits.view(np.float32).astype(np.float64)
    sign = np.where(np.signbit(flat_v), -1.0, 1.0)
    # neighbour one bf16 step further from zero
    step_bits = bits + np.uint32(0x10000)
    hi = step_bits.view(np.float32).astype(np.float64)
    # make lo the bf16 value toward zero from v, hi the one away from zero
    too_big = np.abs(lo) > np.abs(flat_v)
    prev_bits = bits - np.uint32(0x10000)
    lo = np.where(too_big, prev_bits.view(np.float32).astype(np.float64), lo)
    lo_bits = np.where(too_big, prev_bits, bits)
    hi = np.where(too_big, bits.view(np.float32).astype(np.float64), hi)
    hi_bits = np.where(too_big, bits, step_bits)
    d_lo = np.abs(flat_v - lo)
    d_hi = np.abs(hi - flat_v)
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & ((lo_bits >> 16) % 2 == 0))
    res = np.where(pick_lo, lo_bits, hi_bits) >> 16
    res = np.where(flat_v == 0.0, np.where(np.signbit(flat_v), 0x8000, 0), res)
    flat_o[:] = res.astype(np.uint16)
    del sign
    return out
