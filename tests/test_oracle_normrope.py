"""Pins for the oracle's QK-RMSNorm + RoPE prologue (CPU only).

The prologue follows onnxruntime PR #29912, Summary of Changes (q_norm_weight /
k_norm_weight, qk_norm_epsilon default 1e-6, rotary_offset; QkNormRotaryTNH
fuses QK-RMSNorm and RoPE in that order).  Each check compares the oracle with
something other than itself: torch's bf16 cast, torch's fp64 RMSNorm routine,
closed forms (a constant row, a quarter-turn rotation), and the invariants a
rotation must keep (pair norms, relative-position dot products, the channel
permutation between the two pair layouts).  The oracle evaluates the
definitions in fp64, so against an fp64 reference its bf16 rows are the
round-to-nearest-even of that reference, exactly, except for a value lying so
close to a bf16 tie (within 2^-40 of it, relative) that the two fp64
evaluation orders may round to different sides; those are counted and must be
rare.
"""
import math

import numpy as np
import pytest
import torch

from decode_attention_quantized_gb300 import synth


def bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(u):
    return (np.asarray(u, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_neighbours(v):
    """(lower, upper) bf16 values around each fp64 value v (finite, normal
    range) and the midpoint between them, exactly in fp64."""
    v = np.asarray(v, np.float64)
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -126)))
    q = np.ldexp(1.0, (e - 7).astype(int))  # bf16 spacing in v's binade
    lo = np.floor(v / q) * q
    return lo, lo + q, lo + q / 2


def assert_rne_of(got_bits, ref, rel=2.0 ** -40, max_near=0):
    """got (bf16 bits) equals the nearest-even bf16 of the fp64 reference at
    every element whose reference lies farther than rel * |ref| from a bf16
    tie; at the others it is one of the two neighbours.  Returns how many were
    that close (at most max_near)."""
    got = bits_to_f64(got_bits).reshape(-1)
    ref = np.asarray(ref, np.float64).reshape(-1)
    lo, hi, mid = bf16_neighbours(ref)
    tie = ref == mid  # an exact tie (exact fp64 sums of bf16 values): nearest even on both sides
    near = (np.abs(ref - mid) <= rel * np.abs(ref)) & ~tie
    exact = ~near
    lo_even = (bf16_bits(lo.astype(np.float32)) & 1) == 0  # lo, hi are bf16 values: exact in float32
    want = np.where(tie, np.where(lo_even, lo, hi), np.where(ref - lo < hi - ref, lo, hi))
    assert np.array_equal(got[exact], want[exact]), \
        f"{np.count_nonzero(got[exact] != want[exact])} values are not the nearest bf16 of the reference"
    assert np.isin(got[near], np.stack([lo[near], hi[near]])).all() if near.any() else True
    assert near.sum() <= max_near, near.sum()
    return int(near.sum())


def rows(shape, *parts):
    return bf16_bits(synth.randn_bf16(shape, "cpu", *parts).float().numpy())


# ------------------------------------------------------------- bf16 rounding

def test_f64_to_bf16_matches_torch_on_float32_values(orc):
    # for values that are float32 numbers, one rounding from double equals
    # torch's float32 -> bf16 cast (round to nearest even); the sweep covers
    # ties, subnormals, the overflow edge and both signs
    rng = np.random.default_rng(5)
    u = rng.integers(0, 1 << 32, 20000, dtype=np.uint64).astype(np.uint32)
    x = u.view(np.float32)
    x = x[np.isfinite(x)]
    ties = (np.arange(1, 2000, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    edge = np.array([3.3895313892515355e38, 3.3961e38, 3.4e38, 2.0 ** -126, 2.0 ** -130, 2.0 ** -133,
                     1.5 * 2.0 ** -133, 2.0 ** -134, 0.0, -0.0], np.float32)
    x = np.concatenate([x, ties, -ties, edge, -edge])
    mine = np.array([orc.f64_to_bf16(float(v)) for v in x], np.uint16)
    assert np.array_equal(mine, bf16_bits(x))


def test_f64_to_bf16_rounds_once_from_double(orc):
    # 1 + 2^-8 + 2^-30 is above the tie: a single rounding gives 1 + 2^-7,
    # while rounding to float32 first would land on the tie and round to 1
    assert orc.f64_to_bf16(1.0 + 2.0 ** -8 + 2.0 ** -30) == 0x3F81
    assert orc.f64_to_bf16(1.0 + 2.0 ** -8) == 0x3F80
    assert orc.f64_to_bf16(-(1.0 + 3 * 2.0 ** -8)) == 0xBF82


# ------------------------------------------------------------------ RMSNorm

def test_rms_norm_of_a_constant_row_is_closed_form(orc):
    D, eps = 128, 1e-6
    for c in (0.5, -3.0, 1e-3):
        x = np.full((1, 1, D), bf16_bits(np.float32(c)), np.uint16)
        w = bf16_bits(np.linspace(0.5, 1.5, D).astype(np.float32))
        out, bad = orc.norm_rope(x, norm_weight=w, eps=eps)
        cf = float(bits_to_f64(x[0, 0, 0]))
        ref = cf / math.sqrt(cf * cf + np.float64(np.float32(eps))) * bits_to_f64(w)
        assert bad == 0
        assert_rne_of(out[0, 0], ref)


def test_rms_norm_matches_torch_fp64(orc):
    N, H, D = 5, 3, 256
    x = rows((N, H, D), "normrope", "x")
    w = bf16_bits(synth.norm_weight_bf16(D, "cpu", "normrope", "w").float().numpy())
    for eps in (1e-6, 1e-2):
        out, _ = orc.norm_rope(x, norm_weight=w, eps=eps)
        ref = torch.nn.functional.rms_norm(torch.from_numpy(bits_to_f64(x)), (D,),
                                           torch.from_numpy(bits_to_f64(w)), float(np.float32(eps))).numpy()
        assert_rne_of(out, ref)


def test_rms_norm_is_scale_invariant_and_has_unit_rms(orc):
    D = 64
    x = rows((1, 4, D), "normrope", "scale")
    out1, _ = orc.norm_rope(x, norm_weight=np.full(D, 0x3F80, np.uint16), eps=0.0)
    x2 = bf16_bits(bits_to_f64(x) * 8.0)  # exact: a power of two
    out2, _ = orc.norm_rope(x2, norm_weight=np.full(D, 0x3F80, np.uint16), eps=0.0)
    assert np.array_equal(out1, out2)
    y = bits_to_f64(out1)
    rms = np.sqrt((y * y).mean(axis=-1))
    assert np.allclose(rms, 1.0, rtol=2 ** -8)


# --------------------------------------------------------------------- RoPE

def test_quarter_turn_is_exact_and_touches_only_the_rotated_channels(orc):
    # cos = 0, sin = 1: the pair (a, b) -> (-b, a), exactly; channels outside
    # [offset, offset + rotary_dim) pass through unchanged
    D, rd, off = 64, 8, 6
    x = rows((1, 2, D), "normrope", "quarter")
    cos = np.zeros((1, rd // 2), np.float32)
    sin = np.ones((1, rd // 2), np.float32)
    for inter in (False, True):
        out, bad = orc.norm_rope(x, rotary_dim=rd, rotary_offset=off, interleaved=inter, cos=cos, sin=sin,
                                 positions=np.zeros(1, np.int64))
        assert bad == 0
        exp = x.copy()
        for i in range(rd // 2):
            a, b = (off + 2 * i, off + 2 * i + 1) if inter else (off + i, off + i + rd // 2)
            exp[..., a] = x[..., b] ^ 0x8000
            exp[..., b] = x[..., a]
        assert np.array_equal(out, exp)


def test_position_zero_is_the_identity(orc):
    D, rd = 128, 128
    x = rows((3, 2, D), "normrope", "ident")
    cos, sin = synth.rope_tables(16, rd)
    out, _ = orc.norm_rope(x, rotary_dim=rd, cos=cos, sin=sin, positions=np.zeros(3, np.int64))
    assert np.array_equal(out, x)


def test_rotation_keeps_pair_norms(orc):
    D, rd, off = 256, 64, 64
    x = rows((6, 2, D), "normrope", "norms")
    cos, sin = synth.rope_tables(1000, rd)
    pos = np.array([1, 7, 99, 500, 998, 3], np.int64)
    out, _ = orc.norm_rope(x, rotary_dim=rd, rotary_offset=off, cos=cos, sin=sin, positions=pos)
    xa, ya = bits_to_f64(x), bits_to_f64(out)
    a = np.arange(off, off + rd // 2)
    n0 = np.hypot(xa[..., a], xa[..., a + rd // 2])
    n1 = np.hypot(ya[..., a], ya[..., a + rd // 2])
    assert np.allclose(n1, n0, rtol=2 ** -7, atol=1e-30)


def test_dot_products_depend_only_on_relative_position(orc):
    # <R_m q, R_n k> = <R_(m+s) q, R_(n+s) k> for tables of angles pos * theta_i
    D, rd = 128, 128
    q = rows((1, 1, D), "normrope", "q")
    k = rows((1, 1, D), "normrope", "k")
    cos, sin = synth.rope_tables(4096, rd)

    def rot(x, p):
        return bits_to_f64(orc.norm_rope(x, rotary_dim=rd, cos=cos, sin=sin, positions=np.array([p], np.int64))[0])

    d0 = float((rot(q, 40) * rot(k, 13)).sum())
    for s in (1, 100, 2000):
        d1 = float((rot(q, 40 + s) * rot(k, 13 + s)).sum())
        assert abs(d1 - d0) <= 2 ** -6 * (np.abs(bits_to_f64(q)).sum() * np.abs(bits_to_f64(k)).max())


def test_interleaved_layout_is_the_half_split_layout_permuted(orc):
    D, rd, off = 64, 32, 16
    x = rows((4, 3, D), "normrope", "perm")
    cos, sin = synth.rope_tables(64, rd)
    pos = np.array([3, 0, 63, 17], np.int64)
    perm = np.arange(D)
    half = rd // 2
    perm[off:off + half] = off + 2 * np.arange(half)       # half-split slot i <- interleaved 2i
    perm[off + half:off + rd] = off + 2 * np.arange(half) + 1
    a, _ = orc.norm_rope(x, rotary_dim=rd, rotary_offset=off, interleaved=True, cos=cos, sin=sin, positions=pos)
    b, _ = orc.norm_rope(x[..., perm], rotary_dim=rd, rotary_offset=off, interleaved=False, cos=cos, sin=sin,
                         positions=pos)
    assert np.array_equal(a[..., perm], b)


def test_norm_then_rope_order_and_bad_positions(orc):
    # RMSNorm commutes with a rotation when the weight is uniform (rotations keep
    # the row's norm), so the order shows only through a non-uniform weight:
    # the oracle must equal rotate(normalize(x)), computed here in fp64
    D, rd = 64, 64
    x = rows((3, 1, D), "normrope", "order")
    w = bf16_bits(synth.norm_weight_bf16(D, "cpu", "normrope", "w2").float().numpy())
    cos, sin = synth.rope_tables(8, rd)
    pos = np.array([5, 8, -1], np.int64)  # two of them outside the 8-row tables
    out, bad = orc.norm_rope(x, norm_weight=w, eps=1e-6, rotary_dim=rd, cos=cos, sin=sin, positions=pos)
    assert bad == 2
    assert not out[1:].any()  # skipped rows untouched (zero)
    xf = bits_to_f64(x[0, 0])
    y = xf * (1.0 / math.sqrt((xf * xf).mean() + np.float64(np.float32(1e-6)))) * bits_to_f64(w)
    c, s = cos[5].astype(np.float64), sin[5].astype(np.float64)
    z = y.copy()
    z[:32] = y[:32] * c - y[32:] * s
    z[32:] = y[32:] * c + y[:32] * s
    assert_rne_of(out[0, 0], z)
    # the other order (rotate, then normalize) is a different row
    zr = xf.copy()
    zr[:32] = xf[:32] * c - xf[32:] * s
    zr[32:] = xf[32:] * c + xf[:32] * s
    zr = zr * (1.0 / math.sqrt((zr * zr).mean() + np.float64(np.float32(1e-6)))) * bits_to_f64(w)
    assert not np.array_equal(bits_to_f64(out[0, 0]), bits_to_f64(bf16_bits(zr.astype(np.float32))))


# ---------------------------------------------------------- Hadamard rotation

def test_hadamard_matches_scipys_matrix(orc):
    """The rotation is scipy's Sylvester Hadamard matrix over sqrt(D), then one
    bf16 rounding (also after a norm and a rotation, the order the pages
    name)."""
    from scipy.linalg import hadamard
    for D in (64, 128, 256):
        x = rows((3, 2, D), "normrope", "had", D)
        out, _ = orc.norm_rope(x, hadamard=True)
        ref = bits_to_f64(x) @ (hadamard(D).astype(np.float64) / math.sqrt(D)).T
        assert_rne_of(out, ref)
        # the transposed orientation (H^T = H for Sylvester order) and a
        # missing 1/sqrt(D) would both differ: pin the scale separately
        raw = bits_to_f64(x) @ hadamard(D).astype(np.float64).T
        assert not np.allclose(bits_to_f64(out), raw)
    D, rd = 128, 128
    x = rows((2, 3, D), "normrope", "had-full")
    w = bf16_bits(synth.norm_weight_bf16(D, "cpu", "normrope", "w3").float().numpy())
    cos, sin = synth.rope_tables(64, rd)
    pos = np.array([9, 61], np.int64)
    out, _, out64 = orc.norm_rope(x, norm_weight=w, eps=1e-6, rotary_dim=rd, cos=cos, sin=sin, positions=pos,
                                  hadamard=True, return_f64=True)
    pre, _, pre64 = orc.norm_rope(x, norm_weight=w, eps=1e-6, rotary_dim=rd, cos=cos, sin=sin, positions=pos,
                                  return_f64=True)
    assert_rne_of(out, pre64 @ (hadamard(D).astype(np.float64) / math.sqrt(D)).T)
    assert_rne_of(out, out64)


def test_hadamard_of_a_basis_vector_is_a_signed_row(orc):
    # H e_j = column j: entries (-1)^popcount(i & j) / sqrt(D), exact for D = 64, 256
    for D in (64, 256):
        for j in (0, 1, 5, D - 1):
            x = np.zeros((1, 1, D), np.uint16)
            x[0, 0, j] = 0x3F80
            out, _ = orc.norm_rope(x, hadamard=True)
            sign = np.array([(-1) ** bin(i & j).count("1") for i in range(D)], np.float64)
            assert np.array_equal(bits_to_f64(out[0, 0]), sign / math.sqrt(D))


def test_hadamard_keeps_dot_products_and_is_its_own_inverse(orc):
    D = 128
    x = rows((4, 1, D), "normrope", "had-dot")
    y = rows((4, 1, D), "normrope", "had-dot2")
    hx, _ = orc.norm_rope(x, hadamard=True)
    hy, _ = orc.norm_rope(y, hadamard=True)
    d0 = (bits_to_f64(x) * bits_to_f64(y)).sum(-1)
    d1 = (bits_to_f64(hx) * bits_to_f64(hy)).sum(-1)
    scale = np.linalg.norm(bits_to_f64(x), axis=-1) * np.linalg.norm(bits_to_f64(y), axis=-1)
    assert (np.abs(d1 - d0) <= 2 ** -7 * scale).all()
    hhx, _ = orc.norm_rope(hx, hadamard=True)
    assert np.allclose(bits_to_f64(hhx), bits_to_f64(x), rtol=2 ** -6, atol=2 ** -6 * np.abs(bits_to_f64(x)).max())


def test_hadamard_spreads_an_outlier_channel_and_narrows_int4_error(orc):
    """The reason for the rotation: a row with one large channel quantizes
    badly per-row at int4 (every other channel rounds to zero); rotated, the
    energy spreads over all channels and the dequantized row is closer."""
    D = 128
    x = rows((32, 1, D), "normrope", "had-outlier").astype(np.uint16)
    xf = bits_to_f64(x)
    xf[:, 0, 7] = 40.0
    x = bf16_bits(xf.astype(np.float32))
    hx, _ = orc.norm_rope(x, hadamard=True)

    def err(rows_bits):
        e = 0.0
        for r in rows_bits[:, 0]:
            codes, sc = orc.quantize_row(r, orc.INT4, orc.PER_ROW)
            deq = orc.code_values(codes, orc.INT4, D) * sc
            e += float(((deq - bits_to_f64(r)) ** 2).sum())
        return e

    # both in the rotated frame's norm (the rotation is orthonormal)
    assert err(hx) < 0.5 * err(x)
