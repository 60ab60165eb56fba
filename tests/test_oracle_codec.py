"""Pins for the oracle's quantizer and codecs (CPU only).

Each check compares the oracle with something other than itself: torch's
float8_e4m3fn format, a brute-force search over the code set, IEEE fp32
division done by NumPy, closed-form bounds, or hand-worked bytes.
"""
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32_to_bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- e4m3 codec

def test_e4m3_decode_all_codes_match_torch(orc):
    codes = np.arange(256, dtype=np.uint8)
    mine = orc.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert (np.isnan(mine) == nan).all()
    assert set(np.flatnonzero(nan)) == {0x7F, 0xFF}
    assert np.array_equal(mine[~nan], ref[~nan])
    assert mine[0x7E] == 448.0 and mine[0x01] == 2.0 ** -9 and mine[0x08] == 2.0 ** -6


def test_e4m3_encode_matches_torch_dense_sweep(orc):
    # every fp32 bit pattern with the low 8 mantissa bits stepped by 37, over
    # |x| <= 464 (torch's cast is round-to-nearest-even there; above 464 it
    # gives NaN where the reading saturates, checked separately)
    bits = np.arange(0, 0x43E80000 + 1, 37, dtype=np.uint32)
    x = bits.view(np.float32)
    x = np.concatenate([x, -x])
    mine = orc.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mine, ref)


def _brute_e4m3(v, table):
    """Nearest finite e4m3 value by exhaustive search; ties to the even code."""
    finite = [c for c in range(256) if not np.isnan(table[c])]
    best = None
    for c in finite:
        d = abs(float(table[c]) - float(v))
        key = (d, c & 1, 0 if (c & 0x80) == (0x80 if np.signbit(v) else 0) else 1)
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


def test_e4m3_encode_brute_force_and_saturation(orc):
    table = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    rng = np.random.default_rng(7)
    vals = np.concatenate([
        rng.standard_normal(300) * 50,
        rng.uniform(-2 ** -6, 2 ** -6, 100),                    # subnormal range
        np.array([0.0, 2 ** -10, 3 * 2 ** -10, 5 * 2 ** -10, 448.0, 460.0, 464.0, 1e5, -1e30]),
        (table[np.isfinite(table)][:-1] + np.diff(table[np.isfinite(table)]) / 2)[::3],  # midpoints
    ]).astype(np.float32)
    mine = orc.e4m3_encode(vals)
    for v, c in zip(vals, mine):
        if abs(float(v)) >= 448.0:
            assert c == (0xFE if v < 0 else 0x7E), v        # reading R7: saturate to +-448
            continue
        b = _brute_e4m3(v, table)
        # +0 and -0 both decode to zero: accept either sign of zero
        if table[b] == 0 and table[c] == 0:
            continue
        assert c == b, (v, c, b)


# ------------------------------------------------------------ quantize row

@pytest.mark.parametrize("dtype,qmax", [(1, 127.0), (3, 7.0), (2, 448.0)])
def test_per_row_scale_is_fp32_absmax_over_qmax(orc, dtype, qmax):
    rng = np.random.default_rng(dtype)
    for _ in range(50):
        D = int(rng.choice([1, 2, 3, 63, 64, 128, 256]))
        x = f32_to_bf16_bits(rng.standard_normal(D) * np.exp(rng.uniform(-20, 20)))
        _, s = orc.quantize_row(x, dtype, orc.PER_ROW)
        amax = np.abs(orc.bf16_bits_to_f64(x)).max().astype(np.float32)
        assert np.float32(s) == np.float32(amax) / np.float32(qmax)       # IEEE fp32 division


def _decoded(orc, codes, dtype, D):
    return orc.code_values(codes, dtype, D)


@pytest.mark.parametrize("dtype", [1, 3, 2])
@pytest.mark.parametrize("mode", [1, 2, 3])
def test_append_round_trip_within_half_step(orc, dtype, mode):
    """kv-quant-attn page, "Correctness": appends round-trip within half a
    quantization step.  int8/int4: |x - code*s| <= s/2 (1 + qmax 2^-23) for
    every element not clamped; e4m3: within half an e4m3 ulp at x/s."""
    rng = np.random.default_rng(10 * dtype + mode)
    qmax = orc.QMAX[dtype]
    for trial in range(40):
        D = int(rng.choice([2, 3, 64, 128, 256]))
        xf = rng.standard_normal(D) * np.exp(rng.uniform(-8, 8))
        x = f32_to_bf16_bits(xf)
        xd = orc.bf16_bits_to_f64(x)
        if mode == orc.PER_ROW:
            st = None
        elif mode == orc.PER_TENSOR:
            st = np.array([np.abs(xd).max() / qmax * rng.uniform(0.7, 1.5)], np.float32)
        else:
            st = (np.abs(xd) / qmax * rng.uniform(0.7, 1.5, D) + 1e-30).astype(np.float32)
        codes, s_row = orc.quantize_row(x, dtype, mode, st)
        c = _decoded(orc, codes, dtype, D)
        s = (np.full(D, s_row) if mode == orc.PER_ROW else np.broadcast_to(st, (D,)).astype(np.float64))
        v = xd / s
        if dtype == 2:
            # half ulp of e4m3 at |v|: ulp 2^(e-3) in the normal range, 2^-9 below 2^-6
            e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -6)))
            half_ulp = np.where(np.abs(v) < 2.0 ** -6, 2.0 ** -10, 2.0 ** (e - 4))
            ok = np.abs(v) <= 448.0
            assert (np.abs(v - c)[ok] <= half_ulp[ok] * (1 + 2 ** -20) + 1e-300).all()
            assert (np.abs(c[~ok]) == 448.0).all()
        else:
            ok = np.abs(v) <= qmax
            err = np.abs(xd - c * s)
            assert (err[ok] <= s[ok] / 2 * (1 + qmax * 2.0 ** -23)).all()
            assert (np.abs(c[~ok]) == qmax).all()
            assert (np.abs(c) <= qmax).all()            # reading R3: -128 / -8 never produced


@pytest.mark.parametrize("dtype", [1, 3])
def test_integer_codes_brute_force_nearest_even(orc, dtype):
    """The code is the integer in [-qmax, qmax] nearest to fl32(x / s), ties to
    the even integer (reading R1), found by exhaustive search."""
    qmax = int(orc.QMAX[dtype])
    rng = np.random.default_rng(3 + dtype)
    for _ in range(30):
        D = 8
        # include exact ties: x = (k + 1/2) * s with s a power of two
        s = np.float32(2.0 ** rng.integers(-6, 6))
        k = rng.integers(-qmax - 2, qmax + 2, D)
        frac = rng.choice([0.0, 0.5, 0.25, 0.75, 0.5], D)
        xf = ((k + frac) * s).astype(np.float32)
        x = f32_to_bf16_bits(xf)
        codes, _ = orc.quantize_row(x, dtype, orc.PER_TENSOR, np.array([s], np.float32))
        c = _decoded(orc, codes, dtype, D)
        xd = orc.bf16_bits_to_f64(x).astype(np.float32)
        for d in range(D):
            v = float(np.float32(xd[d]) / np.float32(s))
            cands = sorted(range(-qmax, qmax + 1), key=lambda z: (abs(z - v), z % 2))
            assert c[d] == cands[0], (v, c[d], cands[:2])


def test_all_zero_row_has_zero_scale_and_codes(orc):
    """Reading R4: an all-zero row stores scale 0 and zero codes."""
    for dtype in (1, 2, 3):
        codes, s = orc.quantize_row(np.zeros(64, np.uint16), dtype, orc.PER_ROW)
        assert s == 0.0 and not codes.any()


def test_tiny_static_scale_uses_division(orc):
    """INT4 PR #32515 review: tiny cache-write scales must not overflow a
    reciprocal.  With s = 1e-40 (subnormal) a zero input stays code 0 and any
    other input saturates; nothing becomes NaN-driven garbage."""
    x = f32_to_bf16_bits(np.array([0.0, 1.0, -1.0, 1e-30], np.float32))
    for dtype in (1, 3, 2):
        codes, _ = orc.quantize_row(x, dtype, orc.PER_TENSOR, np.array([1e-40], np.float32))
        c = _decoded(orc, codes, dtype, 4)
        q = orc.QMAX[dtype]
        assert list(c) == [0.0, q, -q, q]


def _read_int4_golden():
    rows = []
    with open(os.path.join(GOLDEN, "int4_pack.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            lhs, rhs = line.split("->")
            rows.append(([int(t) for t in lhs.split()], bytes.fromhex(rhs.replace(" ", ""))))
    return rows


def test_int4_packing_golden(orc):
    rows = _read_int4_golden()
    assert len(rows) >= 5
    for codes, packed in rows:
        x = f32_to_bf16_bits(np.array(codes, np.float32))
        got, _ = orc.quantize_row(x, 3, orc.PER_TENSOR, np.array([1.0], np.float32))
        assert bytes(got) == packed, (codes, got.tobytes().hex(), packed.hex())
        assert list(orc.code_values(got, 3, len(codes))) == codes
