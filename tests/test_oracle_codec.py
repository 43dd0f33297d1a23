"""Pins for the oracle's E4M3 codec, quantize and scale (CPU only).

Each test checks the oracle against something other than itself: values
worked by hand from the E4M3 definition (tests/golden), an independent
nearest-value encoder over every fp32 bit pattern, torch's float8_e4m3fn
conversion (a library routine) and numpy's IEEE fp32 division.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _parse_value(tok):
    tok = tok.strip()
    if tok == "nan":
        return float("nan")
    if tok in ("inf", "-inf"):
        return float(tok)
    neg = tok.startswith("-")
    t = tok[1:] if neg else tok
    if "*2^" in t:
        m, e = t.split("*2^")
        v = float(m) * 2.0 ** int(e)
    elif t.startswith("2^"):
        v = 2.0 ** int(t[2:])
    else:
        v = float(t)
    return -v if neg else v


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                yield line.split()


def test_decode_closed_forms():
    for code_hex, val in ((r[0], r[1]) for r in _rows("e4m3_closed_form.txt")):
        code = int(code_hex, 16)
        want = _parse_value(val)
        got = float(oracle.e4m3_decode(code))
        if math.isnan(want):
            assert math.isnan(got), code_hex
        else:
            assert got == want and math.copysign(1, got) == math.copysign(1, want), (code_hex, got, want)


def test_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    assert np.array_equal(np.signbit(ref[~nan]), np.signbit(got[~nan]))


def test_encode_worked_rounding_cases():
    for inp, code_hex in ((r[0], r[1]) for r in _rows("e4m3_rounding_cases.txt")):
        y = np.float32(_parse_value(inp))
        want = int(code_hex, 16)
        assert int(oracle.e4m3_encode(np.array([y]))[0]) == want, (inp, code_hex)
        assert int(oracle.e4m3_encode_nearest(np.array([y]))[0]) == want, (inp, code_hex)


def test_roundtrip_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def test_encode_matches_independent_nearest_on_all_fp32():
    """Exhaustive: every one of the 2^32 fp32 bit patterns."""
    n_bad, first = oracle.e4m3_sweep(0, 1 << 32)
    assert n_bad == 0, f"{n_bad} disagreements, first bits 0x{first:08x}"


def test_encode_matches_torch_in_range():
    rng = np.random.default_rng(5)
    y = np.concatenate([
        rng.uniform(-448, 448, 200000),
        rng.standard_normal(200000) * 4,
        rng.standard_normal(200000) * 2.0 ** -7,  # subnormal region
    ]).astype(np.float32)
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(y)
    assert np.array_equal(ref, got)


def test_quantize_uses_ieee_fp32_division():
    rng = np.random.default_rng(6)
    from paged_fp8_kv_quantize_gb300.synth import bf16_bits, bf16_to_f32

    x = bf16_bits(rng.standard_normal(20000).astype(np.float32) * 3)
    s = (rng.uniform(0.001, 0.05, 20000)).astype(np.float32)
    y = bf16_to_f32(x) / s  # numpy: correctly rounded fp32 division
    assert y.dtype == np.float32
    in_range = np.abs(y) <= 448
    want = torch.from_numpy(y[in_range]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.quantize(int(a), float(b)) for a, b in zip(x[in_range], s[in_range])], dtype=np.uint8)
    assert np.array_equal(want, got)
    # out of range saturates (R1)
    sat = np.array([oracle.quantize(int(a), float(b)) for a, b in zip(x[~in_range], s[~in_range])], dtype=np.uint8)
    assert np.all((sat & 0x7F) == 0x7E)


def test_scale_from_amax():
    rng = np.random.default_rng(7)
    for a in rng.uniform(1e-3, 1e3, 2000).astype(np.float32):
        assert oracle.scale_from_amax(float(a)) == float(np.float32(a) / np.float32(448.0))
    assert oracle.scale_from_amax(0.0) == 1.0  # R5
    assert oracle.scale_from_amax(448.0) == 1.0


def test_calibrate_per_head_is_amax_over_head():
    rng = np.random.default_rng(8)
    from paged_fp8_kv_quantize_gb300.synth import bf16_bits, bf16_to_f32

    x = bf16_bits(rng.standard_normal((300, 3, 16)).astype(np.float32))
    x[:, 2, :] = 0  # an all-zero head takes scale 1 (R5)
    s = oracle.calibrate_per_head(x)
    f = bf16_to_f32(x)
    for h in range(2):
        assert s[h] == np.float32(np.abs(f[:, h, :]).max()) / np.float32(448.0)
    assert s[2] == 1.0
