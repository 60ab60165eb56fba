"""Pins for the oracle's attention (CPU only).

The oracle dequantizes the cache and runs fp64 softmax attention.  These tests
tie it to things other than itself: torch's scaled_dot_product_attention in
float64 (a library routine), hand-worked closed forms in tests/golden, and the
invariants the pages state (replicated-head GQA, ragged lengths down to one
token, the exact head-sink rescale, the exact per-channel fold, split
invariance of the log-sum-exp merge).
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).contiguous().view(torch.int16).numpy().view(np.uint16)


def build_cache(orc, k, v, *, dtype, k_mode, v_mode, bs, k_static=None, v_static=None, shuffle_seed=None):
    """k, v: lists (one per sequence) of bf16 tensors [L_b, Hkv, D].  Returns
    (cache, block_table, seq_lens)."""
    B = len(k)
    Hkv, D = k[0].shape[1], k[0].shape[2]
    lens = [int(x.shape[0]) for x in k]
    mb = max(1, max(math.ceil(L / bs) for L in lens))
    nb = B * mb
    ids = np.arange(nb, dtype=np.int32)
    if shuffle_seed is not None:
        ids = np.random.default_rng(shuffle_seed).permutation(nb).astype(np.int32)
    table = ids.reshape(B, mb)
    cache = orc.OracleCache(dtype, k_mode, v_mode, nb, bs, Hkv, D, k_static, v_static)
    for b in range(B):
        L = lens[b]
        t = np.arange(L)
        slots = table[b, t // bs].astype(np.int64) * bs + t % bs
        assert cache.append(bf16_bits(k[b]), bf16_bits(v[b]), slots) == 0
    return cache, table, np.array(lens, np.int32)


def sdpa_reference(qd, kd, vd, L, T, *, sm_scale, window=0, sink=None):
    """torch SDPA in float64 over dequantized K/V of one sequence.
    qd [T, Hq, D]; kd, vd [L, Hkv, D].  The sink is one extra key whose logit
    is sink_i exactly and whose value row is zero."""
    Tq, Hq, D = qd.shape
    Hkv = kd.shape[1]
    G = Hq // Hkv
    q = torch.from_numpy(qd).permute(1, 0, 2)                                   # [Hq, T, D]
    k = torch.from_numpy(kd).permute(1, 0, 2).repeat_interleave(G, dim=0)       # [Hq, L, D]
    v = torch.from_numpy(vd).permute(1, 0, 2).repeat_interleave(G, dim=0)
    j = torch.arange(L)
    pos = L - T + torch.arange(T)
    mask = j[None, :] <= pos[:, None]
    if window > 0:
        mask &= j[None, :] > (pos[:, None] - window)
    mask = mask[None].expand(Hq, T, L)
    if sink is not None:
        one = torch.ones(Hq, T, 1, dtype=torch.float64)
        q = torch.cat([q, one], dim=-1)
        k = torch.cat([k, torch.zeros(Hq, L, 1, dtype=torch.float64)], dim=-1)
        ks = torch.zeros(Hq, 1, D + 1, dtype=torch.float64)
        ks[:, 0, D] = torch.tensor(sink, dtype=torch.float64) / sm_scale
        k = torch.cat([k, ks], dim=1)
        v = torch.cat([v, torch.zeros(Hq, 1, D, dtype=torch.float64)], dim=1)
        mask = torch.cat([mask, torch.ones(Hq, T, 1, dtype=torch.bool)], dim=-1)
    o = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=sm_scale)
    return o.permute(1, 0, 2).numpy()


CASES = [
    # dtype, k_mode, v_mode, Hq, Hkv, D, T, L, bs, window, sink
    (1, 1, 1, 4, 1, 64, 1, 300, 16, 0, False),
    (1, 1, 1, 24, 4, 256, 1, 97, 32, 0, True),
    (2, 2, 2, 8, 2, 128, 1, 130, 16, 0, False),
    (3, 3, 3, 12, 2, 64, 3, 77, 32, 0, False),
    (1, 3, 2, 16, 2, 64, 1, 200, 64, 50, True),
    (2, 1, 3, 8, 8, 32, 2, 45, 16, 7, True),
    (3, 1, 1, 6, 1, 16, 4, 9, 16, 0, True),
]


def _static(mode, x, qmax, rng):
    if mode == 2:
        return np.array([float(x.abs().max()) / qmax * 1.01], np.float32)
    if mode == 3:
        a = x.float().abs().amax(dim=0).numpy() / qmax * rng.uniform(1.0, 1.3, x.shape[1:])
        return np.maximum(a, 1e-3).astype(np.float32)
    return None


@pytest.mark.parametrize("case", CASES)
def test_attend_matches_library_sdpa(orc, case):
    dtype, km, vm, Hq, Hkv, D, T, L, bs, W, use_sink = case
    g = torch.Generator().manual_seed(hash(case) & 0xFFFF)
    rng = np.random.default_rng(hash(case) & 0xFFFF)
    k = torch.randn(L, Hkv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(L, Hkv, D, generator=g).to(torch.bfloat16)
    q = torch.randn(1, T, Hq, D, generator=g).to(torch.bfloat16)
    qmax = orc.QMAX[dtype]
    cache, table, lens = build_cache(orc, [k], [v], dtype=dtype, k_mode=km, v_mode=vm, bs=bs,
                                     k_static=_static(km, k, qmax, rng), v_static=_static(vm, v, qmax, rng),
                                     shuffle_seed=5)
    sink = rng.standard_normal(Hq).astype(np.float32) if use_sink else None
    sm = 1.0 / math.sqrt(D)
    out, lse = cache.attend(bf16_bits(q), table, lens, q_tokens=T, window=W, head_sink=sink)
    kd = np.zeros((L, Hkv, D))
    vd = np.zeros((L, Hkv, D))
    for h in range(Hkv):
        kd[:, h], vd[:, h] = cache.dequant_seq(table[0], h, L)
    ref = sdpa_reference(orc.bf16_bits_to_f64(bf16_bits(q))[0], kd, vd, L, T, sm_scale=sm, window=W,
                         sink=None if sink is None else sink.astype(np.float64))
    assert np.abs(out[0] - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())
    # and the independent NumPy brute force agrees, including lse
    bo, bl = orc.brute_attention(orc.bf16_bits_to_f64(bf16_bits(q))[0], kd, vd, L, window=W,
                                 head_sink=None if sink is None else sink.astype(np.float64))
    assert np.abs(out[0] - bo).max() <= 1e-12 * max(1.0, np.abs(bo).max())
    assert np.abs(lse[0] - bl).max() <= 1e-12 * max(1.0, np.abs(bl).max())


def test_dequant_matches_codes_times_scale(orc):
    """Dequantization is code x scale (row, tensor or channel scale)."""
    g = torch.Generator().manual_seed(1)
    k = torch.randn(40, 2, 64, generator=g).to(torch.bfloat16)
    ks = (k.float().abs().amax(0).numpy() / 7.0).astype(np.float32)
    cache, table, lens = build_cache(orc, [k], [k], dtype=3, k_mode=3, v_mode=1, bs=16, k_static=ks)
    kd, vd = cache.dequant_seq(table[0], 1, 40)
    for t in (0, 17, 39):
        blk, row = table[0, t // 16], t % 16
        codes = orc.code_values(cache.k_codes[blk, 1, row], 3, 64)
        assert np.array_equal(kd[t], codes * ks[1].astype(np.float64))
        vcodes = orc.code_values(cache.v_codes[blk, 1, row], 3, 64)
        assert np.array_equal(vd[t], vcodes * float(cache.v_scale[blk, 1, row]))


def _read_worked():
    cases = []
    consts = {"LN3": math.log(3.0), "LN4": math.log(4.0), "CAP": 2.0 * math.atanh(math.log(3.0) / 2.0)}

    def num(t):
        t = t.strip()
        return consts[t] if t in consts else float(t)

    def rows(s):
        return [[num(x) for x in r.split()] for r in s.split(";")]

    with open(os.path.join(GOLDEN, "attention_worked.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            p = [x.strip() for x in line.split("|")]
            cases.append(dict(name=p[0], k=rows(p[1]), v=rows(p[2]), q=rows(p[3]), sm=num(p[4]),
                              cap=num(p[5]), w=int(p[6]), sink=None if p[7] == "none" else num(p[7]),
                              out=rows(p[8]), lse=[num(x) for x in p[9].split(";")]))
    return cases


@pytest.mark.parametrize("case", _read_worked(), ids=lambda c: c["name"])
def test_worked_examples(orc, case):
    k = torch.tensor(case["k"], dtype=torch.float32)[:, None, :]
    v = torch.tensor(case["v"], dtype=torch.float32)[:, None, :]
    q = torch.tensor(case["q"], dtype=torch.float32)[None, :, None, :]
    T = q.shape[1]
    one = np.array([1.0], np.float32)
    cache, table, lens = build_cache(orc, [k], [v], dtype=1, k_mode=2, v_mode=2, bs=16, k_static=one, v_static=one)
    sink = None if case["sink"] is None else np.array([case["sink"]], np.float32)
    out, lse = cache.attend(bf16_bits(q), table, lens, q_tokens=T, sm_scale=case["sm"], softcap=case["cap"],
                            window=case["w"], head_sink=sink)
    # the sink value passes through fp32 (ln 4 rounded): allow that rounding
    tol = 1e-7 if sink is not None else 1e-12
    assert np.allclose(out[0, :, 0, :], np.array(case["out"]), atol=tol, rtol=0)
    assert np.allclose(lse[0, :, 0], np.array(case["lse"]), atol=1e-12, rtol=0)


def test_single_key_and_ragged_lengths(orc):
    """kv-quant-attn page, "Correctness": ragged lengths down to one token.
    A one-key sequence returns that key's dequantized value exactly (times the
    sink factor sigma(lse - sink) when a sink is given)."""
    g = torch.Generator().manual_seed(3)
    lens = [1, 2, 17, 33, 1]
    ks = [torch.randn(L, 2, 64, generator=g).to(torch.bfloat16) for L in lens]
    vs = [torch.randn(L, 2, 64, generator=g).to(torch.bfloat16) for L in lens]
    q = torch.randn(len(lens), 1, 4, 64, generator=g).to(torch.bfloat16)
    cache, table, sl = build_cache(orc, ks, vs, dtype=1, k_mode=1, v_mode=1, bs=16)
    sink = np.array([0.3, -1.0, 2.0, 0.0], np.float32)
    out, lse = cache.attend(bf16_bits(q), table, sl, head_sink=sink)
    for b in (0, 4):
        for i in range(4):
            h = i // 2
            _, vd = cache.dequant_seq(table[b], h, 1)
            f = 1.0 / (1.0 + math.exp(float(sink[i]) - lse[b, 0, i]))
            assert np.allclose(out[b, 0, i], vd[0] * f, rtol=0, atol=1e-14)


def test_identical_keys_give_mean_value_and_huge_scale_is_finite(orc):
    """Identical K rows (or all-zero K codes) weight every key equally: the
    output is the mean of the dequantized V rows.  With all-zero K codes and a
    K channel scale of FLT_MAX the result stays finite (INT4 PR #32515: the
    zero-code x huge-scale case must not produce inf/NaN)."""
    L, D = 50, 64
    g = torch.Generator().manual_seed(4)
    v = torch.randn(L, 1, D, generator=g).to(torch.bfloat16)
    k = torch.zeros(L, 1, D)
    ks = np.full((1, D), np.finfo(np.float32).max, np.float32)
    cache, table, lens = build_cache(orc, [k], [v], dtype=3, k_mode=3, v_mode=1, bs=16, k_static=ks)
    q = torch.randn(1, 1, 2, D, generator=g).to(torch.bfloat16) * 100
    out, lse = cache.attend(bf16_bits(q), table, lens)
    _, vd = cache.dequant_seq(table[0], 0, L)
    assert np.isfinite(out).all()
    assert np.allclose(out[0, 0, 0], vd.mean(0), atol=1e-14, rtol=0)
    assert abs(lse[0, 0, 0] - math.log(L)) < 1e-12


@pytest.mark.parametrize("G", [1, 2, 4, 6, 8])
def test_gqa_equals_replicated_heads(orc, G):
    """kv-quant-attn page, "Correctness": grouped-query ratios 1:1 through 8:1
    match a replicated-head reference (each query head given its own copy of
    its kv head's rows)."""
    Hkv, D, L = 2, 64, 70
    Hq = G * Hkv
    g = torch.Generator().manual_seed(G)
    k = torch.randn(L, Hkv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(L, Hkv, D, generator=g).to(torch.bfloat16)
    q = torch.randn(1, 2, Hq, D, generator=g).to(torch.bfloat16)
    cache, table, lens = build_cache(orc, [k], [v], dtype=1, k_mode=1, v_mode=1, bs=16)
    out, _ = cache.attend(bf16_bits(q), table, lens, q_tokens=2)
    kr = k.repeat_interleave(G, dim=1)
    vr = v.repeat_interleave(G, dim=1)
    rep, rt, rl = build_cache(orc, [kr], [vr], dtype=1, k_mode=1, v_mode=1, bs=16)
    out_r, _ = rep.attend(bf16_bits(q), rt, rl, q_tokens=2)
    assert np.array_equal(out, out_r)


def test_head_sink_closed_form(orc):
    """onnxruntime PR #29912, ApplyHeadSink: o *= 1/(1+exp(s_h - lse)), which
    equals softmax over [logits; s_h] with a zero value row for the sink; a
    sink at -1e30 reduces to no sink."""
    g = torch.Generator().manual_seed(9)
    L, D = 33, 64
    k = torch.randn(L, 1, D, generator=g).to(torch.bfloat16)
    v = torch.randn(L, 1, D, generator=g).to(torch.bfloat16)
    q = torch.randn(1, 1, 3, D, generator=g).to(torch.bfloat16)
    cache, table, lens = build_cache(orc, [k], [v], dtype=2, k_mode=1, v_mode=1, bs=16)
    sink = np.array([1.5, -2.0, -1e30], np.float32)
    out, lse = cache.attend(bf16_bits(q), table, lens, head_sink=sink)
    base, lse0 = cache.attend(bf16_bits(q), table, lens)
    kd, vd = cache.dequant_seq(table[0], 0, L)
    qd = orc.bf16_bits_to_f64(bf16_bits(q))[0, 0]
    for i in range(3):
        s = np.append(kd @ qd[i] / math.sqrt(D), float(sink[i]))
        w = np.exp(s - s.max())
        w /= w.sum()
        ref = w[:-1] @ vd
        assert np.allclose(out[0, 0, i], ref, atol=1e-14, rtol=0)
    assert np.array_equal(out[0, 0, 2], base[0, 0, 2])
    assert np.array_equal(lse, lse0)


def test_per_channel_fold_is_exact(orc):
    """INT4 PR #32515: folding the K channel scale into Q and applying the V
    channel scale to the output is exact, since dequantization is linear and
    the channel is contracted for K and free for V.  Evaluate the folded form
    from the raw codes and compare with the oracle's dequantize-first result."""
    Hkv, G, D, L = 2, 3, 64, 90
    g = torch.Generator().manual_seed(11)
    rng = np.random.default_rng(11)
    k = (torch.randn(L, Hkv, D, generator=g) * torch.exp(torch.randn(Hkv, D, generator=g))).to(torch.bfloat16)
    v = torch.randn(L, Hkv, D, generator=g).to(torch.bfloat16)
    ks = (k.float().abs().amax(0).numpy() / 7.0 * rng.uniform(1, 1.2, (Hkv, D))).astype(np.float32)
    vs = (v.float().abs().amax(0).numpy() / 7.0 * rng.uniform(1, 1.2, (Hkv, D))).astype(np.float32)
    q = torch.randn(1, 1, Hkv * G, D, generator=g).to(torch.bfloat16)
    cache, table, lens = build_cache(orc, [k], [v], dtype=3, k_mode=3, v_mode=3, bs=32, k_static=ks, v_static=vs)
    out, _ = cache.attend(bf16_bits(q), table, lens)
    qd = orc.bf16_bits_to_f64(bf16_bits(q))[0, 0]
    for i in range(Hkv * G):
        h = i // G
        t = np.arange(L)
        kc = orc.code_values(cache.k_codes[table[0, t // 32], h, t % 32], 3, D)
        vc = orc.code_values(cache.v_codes[table[0, t // 32], h, t % 32], 3, D)
        s = kc @ (qd[i] * ks[h].astype(np.float64)) / math.sqrt(D)     # fold into q
        w = np.exp(s - s.max())
        o = (w @ vc) / w.sum() * vs[h].astype(np.float64)               # scale the output
        assert np.allclose(out[0, 0, i], o, atol=1e-13, rtol=1e-13)


@pytest.mark.parametrize("nsplit", [2, 7, 64])
def test_split_and_lse_merge_is_invariant(orc, nsplit):
    """Flash-decoding split: partials merged in fixed order by the
    log-sum-exp rule equal the unsplit softmax (kv-quant-attn page, Method)."""
    g = torch.Generator().manual_seed(nsplit)
    L, D = 200, 128
    k = torch.randn(L, 2, D, generator=g).to(torch.bfloat16)
    v = torch.randn(L, 2, D, generator=g).to(torch.bfloat16)
    q = torch.randn(1, 2, 8, D, generator=g).to(torch.bfloat16)
    cache, table, lens = build_cache(orc, [k], [v], dtype=1, k_mode=1, v_mode=1, bs=16)
    sink = np.linspace(-1, 1, 8).astype(np.float32)
    a, la = cache.attend(bf16_bits(q), table, lens, q_tokens=2, head_sink=sink, window=150)
    b, lb = cache.attend(bf16_bits(q), table, lens, q_tokens=2, head_sink=sink, window=150, nsplit=nsplit)
    assert np.allclose(a, b, atol=1e-13, rtol=0) and np.allclose(la, lb, atol=1e-12, rtol=0)


def test_draft_tokens_are_causal(orc):
    """Speculative decode: draft tau of T equals a T=1 decode whose sequence
    ends at that draft (seq_len L - T + 1 + tau)."""
    g = torch.Generator().manual_seed(21)
    L, T, D = 60, 5, 64
    k = torch.randn(L, 2, D, generator=g).to(torch.bfloat16)
    v = torch.randn(L, 2, D, generator=g).to(torch.bfloat16)
    q = torch.randn(1, T, 6, D, generator=g).to(torch.bfloat16)
    cache, table, lens = build_cache(orc, [k], [v], dtype=1, k_mode=1, v_mode=1, bs=16)
    out, lse = cache.attend(bf16_bits(q), table, lens, q_tokens=T)
    for tau in range(T):
        one, l1 = cache.attend(bf16_bits(q[:, tau:tau + 1]), table, np.array([L - T + 1 + tau], np.int32))
        assert np.array_equal(out[0, tau], one[0, 0]) and np.array_equal(lse[0, tau], l1[0, 0])


def test_window_equals_truncated_sequence(orc):
    """A window of W keys equals full attention over the last W keys only."""
    g = torch.Generator().manual_seed(22)
    L, W, D = 100, 23, 64
    k = torch.randn(L, 1, D, generator=g).to(torch.bfloat16)
    v = torch.randn(L, 1, D, generator=g).to(torch.bfloat16)
    q = torch.randn(1, 1, 2, D, generator=g).to(torch.bfloat16)
    cache, table, lens = build_cache(orc, [k], [v], dtype=1, k_mode=1, v_mode=1, bs=16)
    out, _ = cache.attend(bf16_bits(q), table, lens, window=W)
    short, st, sl = build_cache(orc, [k[L - W:]], [v[L - W:]], dtype=1, k_mode=1, v_mode=1, bs=16)
    ref, _ = short.attend(bf16_bits(q), st, sl)
    assert np.allclose(out, ref, atol=1e-15, rtol=0)


def test_softcap_limits(orc):
    """Softcap c*tanh(s/c): a cap far above the logits changes nothing; a
    small cap squeezes every logit into (-c, c), so the weights flatten
    toward uniform as c -> 0."""
    g = torch.Generator().manual_seed(23)
    L, D = 40, 64
    k = torch.randn(L, 1, D, generator=g).to(torch.bfloat16)
    v = torch.randn(L, 1, D, generator=g).to(torch.bfloat16)
    q = (torch.randn(1, 1, 2, D, generator=g) * 30).to(torch.bfloat16)
    cache, table, lens = build_cache(orc, [k], [v], dtype=1, k_mode=1, v_mode=1, bs=16)
    a, _ = cache.attend(bf16_bits(q), table, lens)
    b, _ = cache.attend(bf16_bits(q), table, lens, softcap=1e9)
    assert np.allclose(a, b, atol=1e-12, rtol=0)
    c, lc = cache.attend(bf16_bits(q), table, lens, softcap=1e-9)
    _, vd = cache.dequant_seq(table[0], 0, L)
    assert np.allclose(c[0, 0, 0], vd.mean(0), atol=1e-7)
    assert abs(lc[0, 0, 0] - math.log(L)) < 1e-6


def test_append_skips_negative_and_out_of_pool_slots(orc):
    """slot_mapping (PR #29912): a negative slot is a padding token and writes
    nothing; a slot beyond the pool is reported and skipped.  Appending a row
    leaves every other row untouched (issue #29783: no re-quantization)."""
    cache = orc.OracleCache(1, 1, 1, 4, 16, 2, 64)
    g = torch.Generator().manual_seed(5)
    k = torch.randn(5, 2, 64, generator=g).to(torch.bfloat16)
    assert cache.append(bf16_bits(k[:1]), bf16_bits(k[:1]), np.array([3], np.int64)) == 0
    before = cache.k_codes.copy(), cache.k_scale.copy()
    bad = cache.append(bf16_bits(k[1:]), bf16_bits(k[1:]), np.array([-1, 64, 1000, 17], np.int64))
    assert bad == 2
    changed = np.argwhere((cache.k_codes != before[0]).any(-1))
    assert {tuple(x) for x in changed} <= {(1, 0, 1), (1, 1, 1)}
    assert np.array_equal(cache.k_codes[0, :, 3], before[0][0, :, 3])


def test_quantization_error_statistics(orc):
    """Sanity band, not a bound: the kv-quant-attn page reports the error of
    attention over the quantized cache against unquantized fp32 attention as
    1.0e-2 relative at int8 and 1.8e-1 at int4 (its data is not given).  With
    N(0,1) rows the oracle should land within a factor of ~4 of those."""
    Hq, Hkv, D, L = 24, 4, 256, 2048
    g = torch.Generator().manual_seed(31)
    k = torch.randn(L, Hkv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(L, Hkv, D, generator=g).to(torch.bfloat16)
    q = torch.randn(1, 1, Hq, D, generator=g).to(torch.bfloat16)
    qd = orc.bf16_bits_to_f64(bf16_bits(q))[0]
    ref = orc.brute_attention(qd, k.double().numpy(), v.double().numpy(), L)[0]
    errs = {}
    for dtype in (1, 3):
        cache, table, lens = build_cache(orc, [k], [v], dtype=dtype, k_mode=1, v_mode=1, bs=256)
        out, _ = cache.attend(bf16_bits(q), table, lens)
        errs[dtype] = np.linalg.norm(out[0] - ref) / np.linalg.norm(ref)
    assert 2.5e-3 < errs[1] < 4e-2, errs
    assert 4.5e-2 < errs[3] < 0.7, errs
    assert errs[3] > 5 * errs[1]


def test_latent_layout_equals_brute_force_with_v_from_k(orc):
    """Absorbed-MLA layout (onnxruntime PR #29912, kv_cache_layout LATENT,
    v_head_size): one cache, V = the leading v_head_size channels of the
    dequantized K rows.  Against the NumPy brute force fed K as V (attention
    is linear in V, so its leading channels are the latent output)."""
    D, Dv, Hkv, G, T, bs = 64, 48, 2, 2, 2, 16
    L = 37
    rng = np.random.default_rng(3)
    k = rng.standard_normal((L, Hkv, D)).astype(np.float32)
    kb = (k.view(np.uint32) >> 16).astype(np.uint16)
    oc = orc.OracleCache(orc.INT8, orc.PER_ROW, orc.PER_ROW, 4, bs, Hkv, D, latent=True, v_head_size=Dv)
    assert oc.append(kb, None, np.arange(L, dtype=np.int64)) == 0
    q = (rng.standard_normal((1, T, Hkv * G, D)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    table = np.arange(4, dtype=np.int32)[None, :]
    out, lse = oc.attend(q, table, np.array([L], np.int32), q_tokens=T)
    assert out.shape == (1, T, Hkv * G, Dv)
    kd = np.stack([oc.dequant_seq(table[0], h, L)[0] for h in range(Hkv)], axis=1)  # [L, Hkv, D]
    ref, ref_lse = orc.brute_attention(orc.bf16_bits_to_f64(q[0]), kd, kd, L)
    assert np.allclose(out[0], ref[..., :Dv], rtol=1e-12, atol=1e-12)
    assert np.allclose(lse[0], ref_lse, rtol=1e-12, atol=1e-12)
