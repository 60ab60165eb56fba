"""Pins for the oracle's group-wise scales (CPU only).

Group-wise scaling is what the kv-quant-attn page lists under "Requirements
and limits" as not done there (per-row absmax only, "no group-wise scaling or
outlier channels"); the reading here is the per-row rule applied to each run
of group_size consecutive channels.  Every check reduces it to something
pinned elsewhere or fixed by arithmetic: the per-row quantizer (pinned in
test_oracle_codec.py) on the group's own values, IEEE fp32 division by NumPy,
the half-step bound, and per-row caches of head_dim = group_size.
"""
import numpy as np
import pytest
import torch

DTYPES = [1, 3, 2]  # int8, int4, e4m3


def f32_to_bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def rows(rng, n, D):
    """bf16 rows with per-channel magnitudes spread over several binades."""
    out = []
    for _ in range(n):
        mag = np.exp(rng.uniform(-6, 6, D)) if rng.random() < 0.5 else np.exp(rng.uniform(-3, 3))
        out.append(f32_to_bf16_bits(rng.standard_normal(D) * mag))
    return out


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("D", [64, 128, 256])
def test_one_group_of_the_whole_row_is_per_row(orc, dtype, D):
    rng = np.random.default_rng(D + dtype)
    for x in rows(rng, 20, D):
        c_row, s_row = orc.quantize_row(x, dtype, orc.PER_ROW)
        c_grp, s_grp = orc.quantize_row(x, dtype, orc.PER_GROUP, group_size=D)
        assert np.array_equal(c_row, c_grp)
        assert s_grp.shape == (1,) and np.float32(s_grp[0]) == np.float32(s_row)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("D,G", [(64, 32), (128, 32), (128, 64), (256, 32), (256, 128), (12, 4), (8, 2)])
def test_each_group_is_its_own_per_row_quantization(orc, dtype, D, G):
    """Group g's codes and scale are the per-row quantization of its G values
    alone, and its scale is fl32(absmax) / fl32(qmax) of those values."""
    rng = np.random.default_rng(7 * D + G + dtype)
    qmax = np.float32(orc.QMAX[dtype])
    for x in rows(rng, 15, D):
        codes, s = orc.quantize_row(x, dtype, orc.PER_GROUP, group_size=G)
        assert s.shape == (D // G,)
        vals = orc.code_values(codes, dtype, D)
        xd = orc.bf16_bits_to_f64(x)
        for g in range(D // G):
            part = x[g * G:(g + 1) * G]
            c1, s1 = orc.quantize_row(part, dtype, orc.PER_ROW)
            assert np.float32(s[g]) == np.float32(s1)
            assert np.float32(s[g]) == np.float32(np.abs(xd[g * G:(g + 1) * G]).max()) / qmax
            assert np.array_equal(vals[g * G:(g + 1) * G], orc.code_values(c1, dtype, G))


@pytest.mark.parametrize("dtype", [1, 3])
def test_group_round_trip_within_half_its_own_step(orc, dtype):
    """|x - code * s_g| <= s_g / 2 (1 + qmax 2^-23) for every element, with s_g
    the scale of its own group: an outlier in one group does not coarsen the
    others (the int4 gap the page says group-wise scaling would narrow)."""
    rng = np.random.default_rng(40 + dtype)
    qmax = orc.QMAX[dtype]
    D, G = 128, 32
    worse = 0
    for trial in range(30):
        xf = rng.standard_normal(D)
        xf[rng.integers(0, D)] = 100.0 * np.abs(xf).max()  # one outlier channel
        x = f32_to_bf16_bits(xf)
        xd = orc.bf16_bits_to_f64(x)
        codes, s = orc.quantize_row(x, dtype, orc.PER_GROUP, group_size=G)
        c = orc.code_values(codes, dtype, D)
        sg = np.repeat(s.astype(np.float64), G)
        err = np.abs(xd - c * sg)
        assert (err <= sg / 2 * (1 + qmax * 2.0 ** -23)).all()
        cr, sr = orc.quantize_row(x, dtype, orc.PER_ROW)
        err_row = np.abs(xd - orc.code_values(cr, dtype, D) * sr)
        worse += err.max() > err_row.max() * (1 + 1e-12)
        # the groups without the outlier are quantized on their own, finer step
        assert np.sort(s)[-2] < s.max() / 10
    assert worse == 0


def test_all_zero_group_has_zero_scale_and_codes(orc):
    """Reading R4 per group: an all-zero group stores scale 0 and zero codes,
    whatever the other groups hold."""
    x = np.zeros(64, np.float32)
    x[32:] = np.linspace(-3, 3, 32)
    for dtype in DTYPES:
        codes, s = orc.quantize_row(f32_to_bf16_bits(x), dtype, orc.PER_GROUP, group_size=32)
        v = orc.code_values(codes, dtype, 64)
        assert s[0] == 0.0 and not v[:32].any() and s[1] > 0 and v[32:].any()


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("k_mode,v_mode", [(4, 4), (4, 1), (2, 4)])
def test_group_cache_dequant_is_per_row_caches_of_each_group(orc, dtype, k_mode, v_mode):
    """A PER_GROUP cache (paged, shuffled blocks, several heads) dequantizes
    to the concatenation of PER_ROW caches of head_dim = group_size, each fed
    that group's channels: the scale array's [block, head, row, group] layout
    is pinned against the per-row layout."""
    rng = np.random.default_rng(dtype * 10 + k_mode + v_mode)
    NB, bs, H, D, G, L = 6, 16, 3, 64, 32, 70
    table = rng.permutation(NB).astype(np.int32)[: (L + bs - 1) // bs]
    ks = np.float32(0.05)
    c = orc.OracleCache(dtype, k_mode, v_mode, NB, bs, H, D, k_static=np.array([ks], np.float32),
                        v_static=None, group_size=G)
    k = np.stack([np.stack(rows(rng, H, D)) for _ in range(L)])
    v = np.stack([np.stack(rows(rng, H, D)) for _ in range(L)])
    t = np.arange(L)
    slots = (table[t // bs].astype(np.int64) * bs + t % bs)
    assert c.append(k, v, slots) == 0
    # the PER_GROUP side: per-row caches of head_dim G, one per group
    parts_k, parts_v = [], []
    for g in range(D // G):
        cg = orc.OracleCache(dtype, orc.PER_ROW, orc.PER_ROW, NB, bs, H, G)
        assert cg.append(np.ascontiguousarray(k[..., g * G:(g + 1) * G]),
                         np.ascontiguousarray(v[..., g * G:(g + 1) * G]), slots) == 0
        parts_k.append([cg.dequant_seq(table, h, L)[0] for h in range(H)])
        parts_v.append([cg.dequant_seq(table, h, L)[1] for h in range(H)])
    # the other side: the same mode over the full row, without group_size
    full = orc.OracleCache(dtype, k_mode if k_mode != orc.PER_GROUP else orc.PER_ROW,
                           v_mode if v_mode != orc.PER_GROUP else orc.PER_ROW, NB, bs, H, D,
                           k_static=np.array([ks], np.float32), v_static=None)
    assert full.append(k, v, slots) == 0
    for h in range(H):
        kd, vd = c.dequant_seq(table, h, L)
        kf, vf = full.dequant_seq(table, h, L)
        k_ref = np.concatenate([p[h] for p in parts_k], axis=1) if k_mode == orc.PER_GROUP else kf
        v_ref = np.concatenate([p[h] for p in parts_v], axis=1) if v_mode == orc.PER_GROUP else vf
        assert np.array_equal(kd, k_ref)
        assert np.array_equal(vd, v_ref)


def test_group_cache_attention_matches_brute_force(orc):
    """Attention over a PER_GROUP cache equals the NumPy brute force over its
    dequantized rows (the dequantization itself pinned above)."""
    rng = np.random.default_rng(5)
    NB, bs, Hkv, G_q, D, L, T = 8, 16, 2, 3, 128, 100, 2
    Hq = Hkv * G_q
    table = rng.permutation(NB).astype(np.int32)[None, : (L + bs - 1) // bs]
    c = orc.OracleCache(3, orc.PER_GROUP, orc.PER_GROUP, NB, bs, Hkv, D, group_size=32)
    k = np.stack([np.stack(rows(rng, Hkv, D)) for _ in range(L)])
    v = np.stack([np.stack(rows(rng, Hkv, D)) for _ in range(L)])
    t = np.arange(L)
    assert c.append(k, v, table[0, t // bs].astype(np.int64) * bs + t % bs) == 0
    q = np.stack([np.stack(rows(rng, Hq, D)) for _ in range(T)])[None]
    out, lse = c.attend(q, table, np.array([L], np.int32), q_tokens=T)
    kd = np.stack([c.dequant_seq(table[0], h, L)[0] for h in range(Hkv)], axis=1)
    vd = np.stack([c.dequant_seq(table[0], h, L)[1] for h in range(Hkv)], axis=1)
    ref, ref_lse = orc.brute_attention(orc.bf16_bits_to_f64(q[0]), kd, vd, L)
    assert np.allclose(out[0], ref, rtol=1e-10, atol=1e-12)
    assert np.allclose(lse[0], ref_lse, rtol=0, atol=1e-10)
