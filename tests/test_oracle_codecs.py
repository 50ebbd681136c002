"""Pins for the oracle's e4m3 and bf16 codecs (CPU only).

The codecs are checked against the OCP OFP8 E4M3 definition (golden table of
specific codes), against PyTorch's own float8_e4m3fn / bfloat16 conversions
(library routines), exhaustively over every code, and on hand-chosen rounding
midpoints.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle.codecs import (E4M3_TABLE, bf16_decode, bf16_encode, e4m3_decode,
                           e4m3_encode)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_e4m3_golden_codes():
    with open(os.path.join(GOLDEN, "e4m3_codes.json")) as f:
        spec = json.load(f)
    for entry in spec["codes"]:
        v = e4m3_decode(entry["code"])
        if entry["value"] == "nan":
            assert math.isnan(v)
        else:
            assert v == entry["value"], entry
            assert math.copysign(1.0, v) == math.copysign(1.0, entry["value"])


def test_e4m3_decode_matches_torch_exhaustively():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = e4m3_decode(np.arange(256))
    both_nan = np.isnan(ref) & np.isnan(ours)
    assert np.array_equal(both_nan, np.isnan(ref))
    assert np.array_equal(ref[~both_nan], ours[~both_nan])


def test_e4m3_table_shape():
    finite = E4M3_TABLE[np.isfinite(E4M3_TABLE)]
    assert finite.size == 254
    assert np.nanmax(E4M3_TABLE) == 448.0
    pos = E4M3_TABLE[:127]
    assert np.all(np.diff(pos) > 0), "codes 0..126 must be strictly increasing"
    assert np.array_equal(E4M3_TABLE[128:255], -pos)


def test_e4m3_roundtrip_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    assert np.array_equal(e4m3_encode(e4m3_decode(codes)), codes.astype(np.uint8))


def test_e4m3_rne_midpoints():
    # (value, expected code): exact midpoints go to the even code
    cases = [
        (1.0625, 0x38),        # between 1.0 (0x38) and 1.125 (0x39): tie -> even 0x38
        (1.1875, 0x3A),        # between 1.125 (0x39) and 1.25 (0x3A): tie -> even 0x3A
        (2.0 ** -10, 0x00),    # half of the smallest subnormal: tie -> +0
        (1.5 * 2.0 ** -9, 0x02),  # between codes 1 and 2: tie -> even 0x02
        (0.75 * 2.0 ** -9, 0x01),
        (0.25 * 2.0 ** -9, 0x00),
        (464.0, 0x7E),         # above 448 saturates (satfinite)
        (1e9, 0x7E),
        (-1e9, 0xFE),
        (float("inf"), 0x7E),
        (-0.0, 0x80),
        (-(2.0 ** -12), 0x80),  # tiny negative keeps its sign
    ]
    for v, code in cases:
        assert int(e4m3_encode(np.float64(v))) == code, (v, hex(code))
    assert int(e4m3_encode(np.float64("nan"))) == 0x7F


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(200_000) * 50.0,
        rng.uniform(-448, 448, 50_000),
        rng.standard_normal(50_000) * 2.0 ** -8,
        # every midpoint between consecutive finite codes
        (E4M3_TABLE[:126] + E4M3_TABLE[1:127]) / 2.0,
        -(E4M3_TABLE[:126] + E4M3_TABLE[1:127]) / 2.0,
    ]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(e4m3_encode(x), ref)


def test_bf16_decode_exhaustive_vs_torch():
    u = np.arange(65536, dtype=np.uint32).astype(np.int32)
    ref = torch.from_numpy(u.astype(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    ours = bf16_decode(np.arange(65536))
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(ref[~nan].view(np.uint32), ours[~nan].view(np.uint32))


def test_bf16_encode_vs_torch_and_midpoints():
    rng = np.random.default_rng(11)
    x = rng.standard_normal(300_000).astype(np.float32) * np.float32(3.0)
    bits = rng.integers(0, 2**32, 100_000, dtype=np.uint64).astype(np.uint32)
    y = bits.view(np.float32)
    y = y[np.isfinite(y)]
    # exact midpoints: low half 0x8000 over both even and odd upper halves
    mids = ((rng.integers(0, 0x7F00, 1000).astype(np.uint32) << 16) | 0x8000).view(np.float32)
    allx = np.concatenate([x, y, mids])
    ref = torch.from_numpy(allx).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bf16_encode(allx), ref)
    # hand-worked ties: 1 + 2^-8 lies half-way between 1.0 (0x3F80) and 1+2^-7 (0x3F81)
    assert int(bf16_encode(np.float32(1.0 + 2.0 ** -8))) == 0x3F80
    assert int(bf16_encode(np.float32(1.0 + 3 * 2.0 ** -8))) == 0x3F82
    assert int(bf16_encode(np.float32("nan"))) & 0x7FC0 == 0x7FC0
