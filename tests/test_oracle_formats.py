"""Pins for the oracle's number formats: bf16 rounding, E4M3 codec, E8M0 block
exponent and the 1x32 / group-aware 32x1 MXFP8 block quantisers.

The independent references are torch's own bfloat16 and float8_e4m3fn
conversions (library routines), exhaustive enumeration of the 256 E4M3 codes,
closed forms at exact powers of two, and error bounds.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O


def _torch_bf16_bits(x_f32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x_f32, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _torch_e4m3_bits(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def _torch_e4m3_values() -> np.ndarray:
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(1)
    parts = [
        rng.standard_normal(4000).astype(np.float32),
        (rng.standard_normal(2000) * 1e30).astype(np.float32),
        (rng.standard_normal(2000) * 1e-38).astype(np.float32),      # bf16 subnormals
        np.array([0.0, -0.0, 1.0, -1.0, 3.3895314e38, -3.3895314e38, 3.4e38,
                  1.00390625, 1.01171875, 1.0078125 + 2 ** -9], np.float32),
    ]
    # exact midpoints between neighbouring bf16 values: ties to even
    base = rng.standard_normal(2000).astype(np.float32)
    bits = base.view(np.uint32) & np.uint32(0xFFFF0000)
    parts.append((bits | np.uint32(0x8000)).view(np.float32))
    x = np.concatenate(parts)
    ours = O.f64_to_bf16(x.astype(np.float64))
    assert np.array_equal(ours, _torch_bf16_bits(x))


def test_bf16_decode_roundtrip():
    codes = np.arange(0, 65536, 7, dtype=np.uint16)
    vals = O.bf16_to_f64(codes)
    finite = np.isfinite(vals)
    assert np.array_equal(O.f64_to_bf16(vals[finite]), codes[finite])


def test_e4m3_decode_all_codes_match_torch():
    ours = O.e4m3_decode(np.arange(256, dtype=np.uint8))
    ref = _torch_e4m3_values()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(ours[~nan], ref[~nan])
    # signs of zero and extreme codes
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6
    assert math.copysign(1.0, ours[0x80]) == -1.0


def test_e4m3_encode_roundtrip_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = O.e4m3_decode(codes)
    assert np.array_equal(O.e4m3_encode(vals), codes)


def test_e4m3_encode_ties_to_even_and_saturation():
    pos = np.array([c for c in range(0, 0x7F)], np.uint8)
    v = O.e4m3_decode(pos)
    mids = (v[:-1] + v[1:]) / 2
    enc = O.e4m3_encode(mids)
    lo, hi = pos[:-1], pos[1:]
    want = np.where(lo % 2 == 0, lo, hi)          # even mantissa LSB wins
    assert np.array_equal(enc, want)
    assert np.array_equal(O.e4m3_encode(-mids), want | 0x80)
    sat = O.e4m3_encode(np.array([448.0, 449.0, 463.9, 464.0, 500.0, 1e9, np.inf]))
    assert np.all(sat == 0x7E)
    assert np.all(O.e4m3_encode(np.array([-449.0, -1e9, -np.inf])) == 0xFE)
    assert O.e4m3_encode(np.array([-1e-30]))[0] == 0x80   # rounds to -0
    assert O.e4m3_encode(np.array([2.0 ** -10]))[0] == 0x00   # tie to even (0)
    assert O.e4m3_encode(np.array([1.5 * 2.0 ** -10]))[0] == 0x01


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.uniform(-463.0, 463.0, 5000),
                        rng.standard_normal(5000) * 2.0 ** rng.integers(-12, 8, 5000)])
    x = x.astype(np.float32)
    assert np.array_equal(O.e4m3_encode(x.astype(np.float64)), _torch_e4m3_bits(x))


@pytest.mark.parametrize("k", [-133, -127, -126, -20, -9, -1, 0, 1, 8, 9, 100, 127])
def test_e8m0_scale_byte_powers_of_two(k):
    lo = 2.0 ** k
    hi = 2.0 ** k * (2 - 2.0 ** -40)
    want = min(254, max(0, k - 8 + 127))
    assert O.e8m0_scale_byte(lo) == want
    assert O.e8m0_scale_byte(hi) == want
    assert O.e8m0_scale_byte(2.0 ** k * (1 - 2.0 ** -40)) == min(254, max(0, k - 9 + 127))


def test_e8m0_zero_block():
    assert O.e8m0_scale_byte(0.0) == 127


def _dequant_rows(q, s):
    vals = _torch_e4m3_values()[q]
    return vals * np.exp2(np.repeat(s.astype(np.float64) - 127, 32, axis=1))


def test_quant_rows_payload_matches_torch_and_error_bound():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((64, 256)) * 0.02).astype(np.float32)
    x[3, :32] = 0.0                                   # zero block
    x[5, 32:64] *= 1e6                                # large block
    x[7, 64:96] = 2.0 ** 7                            # exact power of two block
    x[9, 96:128] = -(x[9, 96:128] ** 2)
    xb = _torch_bf16_bits(x)
    q, s = O.quant_rows(xb)
    xv = O.bf16_to_f64(xb)
    # scale bytes: floor(log2(amax)) - 8 + 127 (pinned above), payloads: torch's RNE of x / 2^e
    amax = np.abs(xv).reshape(64, 8, 32).max(axis=2)
    assert np.array_equal(s, np.vectorize(O.e8m0_scale_byte)(amax).astype(np.uint8))
    scaled = xv / np.exp2(np.repeat(s.astype(np.float64) - 127, 32, axis=1))
    assert np.all(np.abs(scaled) < 512)
    assert np.array_equal(q, _torch_e4m3_bits(np.clip(scaled, -448, 448).astype(np.float32)))
    assert np.all(q[3, :32] == 0) and s[3, 0] == 127
    # error bound: half an E4M3 ulp (relative 2^-4) or half the subnormal quantum,
    # except for elements above 448 * 2^e which saturate
    deq = _dequant_rows(q, s)
    err = np.abs(deq - xv)
    bound = np.maximum(np.abs(xv) * 2.0 ** -4,
                       np.exp2(np.repeat(s.astype(np.float64) - 127, 32, axis=1)) * 2.0 ** -10)
    sat = np.abs(scaled) > 448
    assert np.all(err[~sat] <= bound[~sat])
    assert np.all(np.abs(deq[sat]) == 448 * np.exp2(np.repeat(s.astype(np.float64) - 127, 32, axis=1))[sat])


def test_quant_cols_grouped_blocks_restart_at_groups():
    rng = np.random.default_rng(4)
    cols = 64
    sizes = np.array([0, 40, 32, 1, 0, 70, 5], np.int32)      # ragged, empty, tiny groups
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    R = int(off[-1])
    R_cap = R + 13
    x = (rng.standard_normal((R_cap, cols)) * 0.02).astype(np.float32)
    # give each group its own magnitude so that a block leaking across a group
    # boundary would pick up a wrong amax
    for e in range(sizes.size):
        x[off[e]:off[e + 1]] *= 4.0 ** e
    xb = _torch_bf16_bits(x)
    q, s = O.quant_cols_grouped(xb, off)
    xv = O.bf16_to_f64(xb)
    E = sizes.size
    seen_rows = set()
    for e in range(E):
        for b in range((int(sizes[e]) + 31) // 32):
            r0 = off[e] + 32 * b
            r1 = min(off[e + 1], r0 + 32)
            srow = e + off[e] // 32 + b
            assert srow not in seen_rows
            seen_rows.add(srow)
            blk = xv[r0:r1]
            want_s = np.array([O.e8m0_scale_byte(a) for a in np.abs(blk).max(axis=0)], np.uint8)
            assert np.array_equal(s[srow], want_s)
            scaled = blk / np.exp2(want_s.astype(np.float64) - 127)
            assert np.array_equal(q[r0:r1], _torch_e4m3_bits(np.clip(scaled, -448, 448)))
    assert max(seen_rows) < O.colwise_scale_rows(R_cap, E)
    assert np.all(q[R:] == 0)


def test_quant_cols_equals_rows_of_transpose_when_groups_are_whole_blocks():
    rng = np.random.default_rng(5)
    sizes = np.array([64, 32, 96], np.int32)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    x = _torch_bf16_bits((rng.standard_normal((192, 96)) * 0.3).astype(np.float32))
    qc, sc = O.quant_cols_grouped(x, off)
    qr, sr = O.quant_rows(np.ascontiguousarray(x.T))
    assert np.array_equal(qc, qr.T)
    # block b of group e sits at scale row e + off[e]/32 + b
    srows = [e + off[e] // 32 + b for e in range(3) for b in range(sizes[e] // 32)]
    assert np.array_equal(sc[srows], sr.T)
