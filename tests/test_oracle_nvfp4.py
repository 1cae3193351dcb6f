"""Pins of the oracle's NVFP4 codec and row quantiser (E2M1 elements, 1x16 E4M3 block scales, an
fp32 tensor encode scale 448 * 6 / amax) and of its grouped matmul, against what is fixed
independently of the oracle's code: the E2M1 value set of the format's definition, exhaustive
round trips, ties swept through every midpoint against a search-based encoder, torch's E4M3
conversion (a library routine) for the block scales, brute force over the 16 codes for every
element, the nibble order, the tensor-amax element decoding to itself, an error bound, and
explicit loops for the grouped matmul."""
import numpy as np
import pytest
import torch

import oracle as O

# E2M1: 1 sign, 2 exponent bits (bias 1), 1 mantissa bit; no infinities or NaN
E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _bf(a):
    return O.f64_to_bf16(np.asarray(a, np.float64))


def test_e2m1_value_set_and_sign():
    assert [O.e2m1_decode(c) for c in range(8)] == E2M1_MAGNITUDES
    for c in range(8):
        neg = O.e2m1_decode(c | 8)
        assert neg == -E2M1_MAGNITUDES[c] and np.signbit(neg)


def test_e2m1_round_trip_and_saturation():
    for c in range(16):
        assert O.e2m1_encode(O.e2m1_decode(c)) == c
    for v in (6.0001, 7.0, 1e30, np.inf):
        assert O.e2m1_encode(v) == 7 and O.e2m1_encode(-v) == 15
    assert O.e2m1_encode(-0.0) == 8 and O.e2m1_encode(-1e-9) == 8


def _nearest_even(v):
    """Search-based reference: the grid neighbours of |v| by searchsorted; the nearer one, and
    on an exact midpoint the one whose code has an even mantissa bit (even code)."""
    g = np.array(E2M1_MAGNITUDES)
    a = min(abs(v), 6.0)
    i = int(np.searchsorted(g, a))
    if i < len(g) and g[i] == a:
        c = i
    else:
        lo, hi = i - 1, i
        dl, dh = a - g[lo], g[hi] - a
        c = lo if dl < dh else hi if dh < dl else (lo if lo % 2 == 0 else hi)
    return c | (8 if np.signbit(v) else 0)


def test_e2m1_ties_and_sweep():
    g = E2M1_MAGNITUDES
    mids = [(g[i] + g[i + 1]) / 2 for i in range(7)]
    # exact midpoints go to the even code: 0.25->0, 0.75->1.0, 1.25->1.0, 1.75->2, 2.5->2, 3.5->4, 5->4
    assert [O.e2m1_encode(m) for m in mids] == [0, 2, 2, 4, 4, 6, 6]
    for v in np.concatenate([np.linspace(-7, 7, 4001), mids, np.nextafter(mids, 0), np.nextafter(mids, 9)]):
        assert O.e2m1_encode(v) == _nearest_even(v), v


def _codes(q):
    """Unpacked codes of a packed [rows, cols/2] array: element 2i from the low nibble."""
    out = np.empty((q.shape[0], q.shape[1] * 2), np.uint8)
    out[:, 0::2] = q & 0x0F
    out[:, 1::2] = q >> 4
    return out


def test_encode_scale_closed_forms():
    assert O.nvfp4_encode_scale(0.0) == 1.0
    assert O.nvfp4_encode_scale(1.0) == 2688.0
    assert O.nvfp4_encode_scale(448.0) == 6.0
    assert O.nvfp4_encode_scale(1e-38) == np.finfo(np.float32).max      # clamped, never inf


@pytest.mark.parametrize("seed,scale", [(0, 1.0), (1, 0.02), (2, 300.0)])
def test_quant_rows_block_scales_and_codes_brute_force(seed, scale):
    rng = np.random.default_rng(seed)
    rows, cols = 6, 96
    x = _bf(rng.standard_normal((rows, cols)) * scale * np.exp(rng.uniform(-4, 4, (rows, 1))))
    q, s, S = O.quant_rows_nvfp4(x)
    xv = O.bf16_to_f64(x)
    S32 = np.float32(S)
    assert S32 == np.float32(2688.0) / np.float32(np.abs(xv).max())
    amax_b = np.abs(xv).reshape(rows, cols // 16, 16).max(-1).astype(np.float32)
    sbf = (amax_b / np.float32(6.0)) * S32                                     # fp32 operations
    ref_s = torch.from_numpy(np.minimum(sbf, 448.0)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(s, ref_s)
    ds = torch.from_numpy(s).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    codes = _codes(q)
    for r in range(rows):
        for c in range(cols):
            d = ds[r, c // 16]
            if d == 0:
                assert codes[r, c] == 0
                continue
            v = np.float32(xv[r, c]) * (S32 / d)                               # fp32 operations
            assert codes[r, c] == _nearest_even(float(v)), (r, c)


def test_nibble_order_and_amax_element_decodes_to_itself():
    x = np.zeros((2, 32), np.float64)
    x[0, 0] = 3.0                              # the tensor amax: scale 448, code 6 (0x7)
    x[1, 17] = -1.5
    q, s, S = O.quant_rows_nvfp4(_bf(x))
    assert q[0, 0] == 0x07                     # element 0 in the low nibble
    assert q[1, 8] == (_nearest_even(-1.5 * S / float(O.e4m3_decode(s[1, 1]))) << 4)
    dec = O.nvfp4_decode(q, s, S)
    assert abs(dec[0, 0] - 3.0) <= 3.0 * 2.0 ** -22


@pytest.mark.parametrize("seed", [3, 4])
def test_decode_error_bound(seed):
    """In the block's scaled units v = x S / ds the E2M1 error is at most max(1/4, |v| / 4)
    (half the grid step; codes are chosen from v in fp32), |v| <= 6 / (1 - 2^-4) after the
    E4M3 rounding of the block scale."""
    rng = np.random.default_rng(seed)
    x = _bf(rng.standard_normal((16, 256)) * np.exp(rng.uniform(-6, 6, (16, 1))))
    q, s, S = O.quant_rows_nvfp4(x)
    xv = O.bf16_to_f64(x)
    dec = O.nvfp4_decode(q, s, S)
    ds = np.repeat(torch.from_numpy(s).view(torch.float8_e4m3fn).to(torch.float64).numpy(), 16, axis=1)
    v = xv * S / np.where(ds > 0, ds, 1)
    assert np.abs(v[ds > 0]).max() <= 6.0 / (1 - 2 ** -4) + 1e-9
    err_v = np.abs(dec - xv) * S / np.where(ds > 0, ds, 1)
    # + the fp32 rounding of the scaled value the code is chosen from (a few ulp)
    slack = 1e-6 * np.maximum(1.0, np.abs(v[ds > 0]))
    assert np.all(err_v[ds > 0] <= np.maximum(0.25, np.abs(v[ds > 0]) / 4) + slack)


def test_all_zero_tensor():
    q, s, S = O.quant_rows_nvfp4(np.zeros((3, 64), np.uint16))
    assert S == 1.0 and not q.any() and not s.any()


def test_grouped_matmul_against_loops():
    rng = np.random.default_rng(5)
    off = np.array([0, 3, 3, 7, 8])
    a = rng.standard_normal((10, 5))
    b = rng.standard_normal((4, 6, 5))
    out = O.grouped_matmul(a, b, off)
    ref = np.zeros((10, 6))
    for e in range(4):
        for r in range(off[e], off[e + 1]):
            for n in range(6):
                ref[r, n] = sum(a[r, k] * b[e, n, k] for k in range(5))
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)
    assert not out[8:].any()
