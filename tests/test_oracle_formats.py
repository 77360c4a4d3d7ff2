"""Pins for the oracle's number formats (no GPU).

Each check ties oracle/formats.py to something outside itself: the OCP
format tables (tests/golden), torch's float8_e4m3fn / bfloat16 conversions
(library routines), brute-force nearest search, and the defining inequality
of the MX block exponent.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import formats as F


def _read_table(path):
    rows = []
    for line in open(path):
        line = line.split("#")[0].strip()
        if not line:
            continue
        c, v = line.split()
        rows.append((int(c, 0), float(v)))
    return rows


def test_e2m1_table_matches_spec(golden_dir):
    for code, val in _read_table(os.path.join(golden_dir, "e2m1_table.txt")):
        got = F.E2M1_TABLE[code]
        assert got == val and math.copysign(1, got) == math.copysign(1, val), (code, got, val)


def test_e4m3_points_match_spec(golden_dir):
    for code, val in _read_table(os.path.join(golden_dir, "e4m3_points.txt")):
        got = F.E4M3_TABLE[code]
        if math.isnan(val):
            assert math.isnan(got), code
        else:
            assert got == val and math.copysign(1, got) == math.copysign(1, val), (hex(code), got, val)


def test_e4m3_table_matches_torch_decode():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    both_nan = np.isnan(ref) & np.isnan(F.E4M3_TABLE)
    assert (both_nan | (ref == F.E4M3_TABLE)).all()
    assert np.isnan(F.E4M3_TABLE).sum() == 2
    pos = F.E4M3_TABLE[:0x7F]
    assert (np.diff(pos) > 0).all()          # codes 0x00..0x7E increase


def test_e8m0_table():
    assert F.E8M0_TABLE[127] == 1.0
    assert F.E8M0_TABLE[0] == 2.0 ** -127
    assert F.E8M0_TABLE[254] == 2.0 ** 127
    assert math.isnan(F.E8M0_TABLE[255])
    assert (F.E8M0_TABLE[1:255] / F.E8M0_TABLE[0:254] == 2.0).all()


def test_e2m1_nibble_order():
    # byte 0x21: low nibble 1 (0.5) is element 0, high nibble 2 (1.0) element 1
    b = np.array([[0x21, 0xF8]], np.uint8)
    assert F.decode_e2m1_packed(b).tolist() == [[0.5, 1.0, -0.0, -6.0]]


def test_nvfp4_dequantize_by_hand():
    # one row, 16 elements: codes 0..15 in order, scale 0x38 (1.0), gs 0.5
    codes = np.arange(16, dtype=np.uint8)
    packed = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)[None]
    w = F.nvfp4_dequantize(packed, np.array([[0x40]], np.uint8), 0.5)   # scale 2.0
    expect = [v * 2.0 * 0.5 for v in [0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6]]
    assert w[0].tolist() == expect


def test_mxfp4_dequantize_by_hand():
    # one row, 64 elements (two blocks of 32): block 0 holds codes 0..15
    # twice with scale 0x80 (2^1), block 1 the code 0x7 (6.0) everywhere
    # with scale 0x7C (2^-3)
    codes = np.concatenate([np.arange(16), np.arange(16), np.full(32, 7)]).astype(np.uint8)
    packed = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)[None]
    w = F.mxfp4_dequantize(packed, np.array([[0x80, 0x7C]], np.uint8))
    mag = [0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6]
    assert w[0, :32].tolist() == [2.0 * v for v in mag * 2]
    assert w[0, 32:].tolist() == [0.75] * 32


def _brute_e4m3(x):
    best, bestd = None, None
    for c in range(256):
        v = F.E4M3_TABLE[c]
        if math.isnan(v):
            continue
        if (c & 0x80) != (0x80 if math.copysign(1, x) < 0 else 0):
            continue
        d = abs(v - max(min(x, 448.0), -448.0))
        if bestd is None or d < bestd or (d == bestd and (c & 1) == 0 and (best & 1) == 1):
            best, bestd = c, d
    return best


def test_rne_e4m3_brute_force():
    rng = np.random.default_rng(1)
    xs = np.concatenate([rng.normal(0, 1, 300), rng.normal(0, 100, 100),
                         rng.normal(0, 0.01, 100), [500.0, -1000.0, 0.0, -0.0, 1e-9, -1e-9]])
    got = F.rne_e4m3(xs)
    for x, c in zip(xs, got):
        assert c == _brute_e4m3(float(x)), (x, c)


def test_rne_e4m3_matches_torch_including_ties():
    pos = F.E4M3_TABLE[:0x7F]
    mids = (pos[1:] + pos[:-1]) / 2            # exact ties (representable in fp32)
    rng = np.random.default_rng(2)
    pts = np.concatenate([mids, -mids, pos, -pos,
                          np.nextafter(mids, 0), np.nextafter(mids, 1000),
                          rng.uniform(-448, 448, 2000), rng.normal(0, 1e-2, 2000),
                          [448.0, 449.0, 463.99, 464.0, -464.0]])
    pts32 = pts.astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(pts32).to(torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = F.rne_e4m3(pts32)
    bad = np.nonzero(got != ref)[0]
    assert len(bad) == 0, [(pts32[i], got[i], ref[i]) for i in bad[:10]]


def test_mx_block_exponent_definition():
    rng = np.random.default_rng(3)
    amax = np.abs(np.concatenate([rng.lognormal(0, 8, 4000), [448.0, 448.0 * 2 ** -5, 896.0, 1.0]]))
    e = F.mx_block_exponent(amax)
    for a, ee in zip(amax, e):
        if -127 < ee < 127:
            assert a <= 448.0 * 2.0 ** ee and a > 448.0 * 2.0 ** (ee - 1), (a, ee)
    assert F.mx_block_exponent(np.array([0.0]))[0] == -127
    assert F.mx_block_exponent(np.array([1e-300]))[0] == -127
    assert F.mx_block_exponent(np.array([448.0]))[0] == 0
    assert F.mx_block_exponent(np.array([448.0001]))[0] == 1


def test_mx_quantize_properties():
    rng = np.random.default_rng(4)
    v = rng.normal(0, 1, (8, 256)) * np.exp2(rng.integers(-20, 20, (8, 1)))
    q, s = F.mx_quantize(v)
    dq = F.mx_dequantize(q, s)
    e = s.astype(np.int64) - 127
    blk = np.abs(v.reshape(8, 8, 32))
    # never saturates; the block maximum lands in the top binade [224, 448] * 2^e
    assert (np.abs(F.decode_e4m3(q)) <= 448).all()
    assert (blk.max(-1) > 224.0 * np.exp2(e)).all()
    # error within half an E4M3 step (relative 2^-4) for normal elements
    rel = np.abs(dq - v) / np.maximum(np.abs(v), 1e-300)
    normal = np.abs(v) >= (2.0 ** -6) * np.exp2(np.repeat(e, 32, axis=1))
    assert (rel[normal] <= 2.0 ** -4 + 1e-12).all()
    # values already on the grid come back unchanged
    q2, s2 = F.mx_quantize(dq)
    assert (F.mx_dequantize(q2, s2) == dq).all()


def test_bf16_roundtrip_matches_torch():
    rng = np.random.default_rng(5)
    v32 = np.concatenate([rng.normal(0, 1, 5000), rng.normal(0, 1e-30, 100), [0.0, -0.0, 1.0]]).astype(np.float32)
    ref = torch.from_numpy(v32).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = F.f64_to_bf16(v32.astype(np.float64))
    assert (got == ref).all()
    back = F.bf16_to_f64(ref)
    assert (back == torch.from_numpy(v32).to(torch.bfloat16).to(torch.float64).numpy()).all()
