"""The QK-RMSNorm + RoPE (+ Walsh-Hadamard) prologue on the GPU against the
oracle (QkNormRotaryTNH, onnxruntime PR #29912, Summary of Changes; the
rotation PR #32515 names as the int4 cache's follow-up).

The oracle evaluates the definitions in fp64 and rounds once to bf16.  The
kernel evaluates them in fp32 (its own fixed order), so its result differs
from the exact value by at most a bound derived here from its arithmetic;
its bf16 rows must then equal the oracle's exactly, except where the exact
value lies within that bound of a bf16 tie (there it is one of the two
neighbours).  Those near-tie elements are counted and must be rare.

The quantizer is the bit-exact contract of kvq_append_norm_rope: its codes and
scales equal the oracle quantizer's applied to the GPU's own bf16 prologue
rows (kvq_norm_rope_apply on the same K, which the fused path promises to
reproduce).  A decode over prologue-rotated queries and keys is compared with
oracle attention over the oracle's own fp64 prologue rows."""
import math

import numpy as np
import pytest
import torch

from decode_attention_quantized_gb300 import kvq, synth

from parity import bf16_bits_to_f64, bf16_neighbours

from guard import guarded

pytestmark = pytest.mark.gpu

DT = {"int8": kvq.INT8, "fp8": kvq.FP8_E4M3, "int4": kvq.INT4}
U32 = 2.0 ** -24  # unit roundoff of fp32


@pytest.fixture(scope="module")
def lib():
    from decode_attention_quantized_gb300 import build
    build.build()
    return kvq.load()


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def prologue(D, *, norm, rd, off, inter, max_pos=4096, seed=0, had=False):
    w = synth.norm_weight_bf16(D, "cpu", "gpu-normrope", seed) if norm else None
    cos, sin = synth.rope_tables(max_pos, rd) if rd else (None, None)
    dev = kvq.NormRope(norm_weight=None if w is None else w.cuda(), eps=1e-6, rotary_dim=rd, rotary_offset=off,
                       interleaved=inter,
                       cos=None if cos is None else torch.from_numpy(cos).cuda(),
                       sin=None if sin is None else torch.from_numpy(sin).cuda(), hadamard=had)
    host = dict(norm_weight=None if w is None else bits(w), eps=1e-6, rotary_dim=rd, rotary_offset=off,
                interleaved=inter, cos=cos, sin=sin, hadamard=had)
    return dev, host


def fp32_error_bound(x_bits, positions, host, ref64):
    """Per element, a bound on |kernel fp32 value - exact value| for rows x
    [N, H, D] (bf16 bits) whose exact prologue values are ref64, propagated
    through the kernel's operations (each one IEEE fp32 operation, relative
    error <= u = 2^-24).  Errors of a factor common to the whole row pass
    through the linear steps unchanged, so they are kept apart as a relative
    error c of the final value; per-element errors e are propagated with m,
    the magnitude each value is formed from:
      RMSNorm y = (x * r) * w: r, one scalar, from the sum of squares (D / 32
        terms per lane, then a 5-level butterfly), a division, an addition,
        a square root and a reciprocal: c = (D / 64 + 8) u; the two products:
        e = 2 u |y|;
      RoPE a' = y_a cos - y_b sin (two rounded products, one rounded sum):
        m = |y_a cos| + |y_b sin|, e' = e_a |cos| + e_b |sin| + 2 u m;
      Hadamard: each butterfly (a, b) -> (a + b, a - b) gives m = m_a + m_b,
        e = e_a + e_b + u m on both outputs; the scale fl(1/fl(sqrt D)) is
        exact for D = 64, 256 and within 2 u otherwise (c += 2 u), and its
        product adds u |v| per element (c += u), with e -> e / sqrt(D).
    Returns c |v| + e, times 1.05 for second-order terms."""
    x = bf16_bits_to_f64(x_bits)
    N, H, D = x.shape
    m = np.abs(x)
    e = np.zeros_like(x)
    c = 0.0
    if host["norm_weight"] is not None:
        w = bf16_bits_to_f64(host["norm_weight"])
        r = 1.0 / np.sqrt((x * x).mean(-1, keepdims=True) + float(np.float32(host["eps"])))
        m = np.abs(x * r * w)
        e = 2 * U32 * m
        c += (D / 64 + 8) * U32
    rd, off = host["rotary_dim"], host["rotary_offset"]
    if rd:
        cs = np.abs(host["cos"][positions].astype(np.float64))[:, None, :]
        sn = np.abs(host["sin"][positions].astype(np.float64))[:, None, :]
        i = np.arange(rd // 2)
        a = off + (2 * i if host["interleaved"] else i)
        b = a + (1 if host["interleaved"] else rd // 2)
        m2, e2 = m.copy(), e.copy()
        m2[..., a] = m[..., a] * cs + m[..., b] * sn
        m2[..., b] = m[..., b] * cs + m[..., a] * sn
        e2[..., a] = e[..., a] * cs + e[..., b] * sn + 2 * U32 * m2[..., a]
        e2[..., b] = e[..., b] * cs + e[..., a] * sn + 2 * U32 * m2[..., b]
        m, e = m2, e2
    if host["hadamard"]:
        span = 1
        while span < D:
            idx = np.arange(D)
            lo = idx[(idx & span) == 0]
            hi = lo + span
            ms = m[..., lo] + m[..., hi]
            es = e[..., lo] + e[..., hi] + U32 * ms
            m[..., lo], m[..., hi] = ms, ms
            e[..., lo], e[..., hi] = es, es
            span <<= 1
        e = e / math.sqrt(D)
        c += (0.0 if D in (64, 256) else 2 * U32) + U32
    return 1.05 * (c * np.abs(ref64) + e)


def check_prologue_rows(got_bits, ref_bits, ref64, bound):
    """got == oracle bf16 wherever the exact value is farther than `bound`
    from a bf16 tie; elsewhere got lies within `bound` plus half a bf16 unit
    of the exact value.  The set of near-tie elements depends only on the
    oracle and the bound; it is capped at 5% so that a bound grown loose
    cannot exempt much of a row.  Returns (near-tie elements, how many of
    them differ from the oracle)."""
    got = bf16_bits_to_f64(got_bits).reshape(-1)
    ref = bf16_bits_to_f64(ref_bits).reshape(-1)
    v = ref64.reshape(-1)
    eps = bound.reshape(-1)
    lo, hi, mid = bf16_neighbours(v)
    near = np.abs(v - mid) <= eps
    far = ~near
    bad = np.count_nonzero(got[far] != ref[far])
    assert bad == 0, f"{bad} of {far.sum()} values away from a bf16 tie differ from the oracle"
    lo2, hi2, _ = bf16_neighbours(np.abs(v) + eps)
    assert (np.abs(got[near] - v[near]) <= eps[near] + (hi2 - lo2)[near] / 2).all()
    assert near.sum() <= 0.05 * v.size, f"{near.sum()} of {v.size} values within the bound of a tie"
    return int(near.sum()), int(np.count_nonzero(got[near] != ref[near]))


CASES = [  # (D, norm, rotary_dim, rotary_offset, interleaved, hadamard)
    (64, True, 64, 0, False, False), (128, True, 128, 0, True, False), (256, True, 64, 192, False, False),
    (128, False, 32, 40, False, False), (256, True, 0, 0, False, False), (64, False, 16, 48, True, False),
    (64, True, 64, 0, False, True), (128, True, 128, 0, False, True), (256, False, 0, 0, False, True),
    (256, True, 256, 0, True, True),
]


@pytest.mark.parametrize("D,norm,rd,off,inter,had", CASES)
def test_norm_rope_apply_matches_the_fp64_oracle(lib, orc, D, norm, rd, off, inter, had):
    N, H = 37, 6  # a ragged token count
    x = synth.randn_bf16((N, H, D), "cpu", "gpu-normrope", "x", D) * 3
    pos = torch.randint(0, 4096, (N,), generator=synth.generator("cpu", "gpu-normrope", "pos", D))
    pos[0], pos[1] = 0, 4095
    dev, host = prologue(D, norm=norm, rd=rd, off=off, inter=inter, had=had)
    y = guarded(torch.zeros_like(x).cuda())
    kvq.kvq_norm_rope_apply(dev, x.cuda(), y, pos.cuda() if rd else None)
    assert kvq.kvq_get_device_error() == 0
    ref, bad, ref64 = orc.norm_rope(bits(x), positions=pos.numpy(), return_f64=True, **host)
    assert bad == 0
    bound = fp32_error_bound(bits(x), pos.numpy(), host, ref64)
    near, differ = check_prologue_rows(bits(y), ref, ref64, bound)
    print(f"near-tie elements: {near} of {ref.size}, {differ} of them on the other side of the tie")
    # in place gives the same rows
    xi = guarded(x.cuda())
    kvq.kvq_norm_rope_apply(dev, xi, xi, pos.cuda() if rd else None)
    assert torch.equal(xi, y)


def test_norm_rope_apply_flags_positions_outside_the_tables(lib, orc):
    D, N, H = 128, 8, 4
    x = synth.randn_bf16((N, H, D), "cpu", "gpu-normrope", "badpos")
    pos = torch.arange(N, dtype=torch.int64) * 60
    pos[3], pos[6] = -5, 512  # tables hold positions 0..511; the others are inside
    dev, host = prologue(D, norm=True, rd=128, off=0, inter=False, max_pos=512)
    y = guarded(torch.full((N, H, D), 7.0, dtype=torch.bfloat16, device="cuda"))
    kvq.kvq_norm_rope_apply(dev, x.cuda(), y, pos.cuda())
    assert kvq.kvq_get_device_error() == kvq.DEVERR_POSITION
    ref, bad, ref64 = orc.norm_rope(bits(x), positions=pos.numpy(), return_f64=True, **host)
    assert bad == 2
    good = [n for n in range(N) if n not in (3, 6)]
    bound = fp32_error_bound(bits(x)[good], pos.numpy()[good], host, ref64[good])
    check_prologue_rows(bits(y)[good], ref[good], ref64[good], bound)
    assert (y[[3, 6]].float() == 7.0).all().item()  # untouched


@pytest.mark.parametrize("dt", list(DT))
@pytest.mark.parametrize("km,vm", [("row", "row"), ("channel", "tensor"), ("group", "row")])
@pytest.mark.parametrize("D,norm,rd,off,inter,had", [(128, True, 128, 0, False, False), (256, True, 64, 0, True, False),
                                                     (64, False, 32, 16, False, False), (128, True, 128, 0, False, True),
                                                     (256, True, 256, 0, False, True)])
def test_append_norm_rope_codes_bit_exact(lib, orc, dt, km, vm, D, norm, rd, off, inter, had):
    """The fused prologue + quantizer writes exactly the codes (and per-row /
    per-group scales) the oracle quantizer gives for the GPU's own prologue
    rows of K (kvq_norm_rope_apply on the same rows: the fused path promises
    the same arithmetic); those rows are within the fp32 bound of the fp64
    oracle; V is quantized as given."""
    modes = {"row": kvq.PER_ROW, "tensor": kvq.PER_TENSOR, "channel": kvq.PER_CHANNEL, "group": kvq.PER_GROUP}
    dtype, kmode, vmode = DT[dt], modes[km], modes[vm]
    gs = 32 if kmode == kvq.PER_GROUP else 0
    Hkv, bs, NB, N = 2, 16, 24, 150
    g = synth.generator("cpu", "gpu-normrope-append", D, dt)
    k = synth.randn_bf16((N, Hkv, D), "cpu", "gpu-normrope-append", "k", D)
    v = synth.randn_bf16((N, Hkv, D), "cpu", "gpu-normrope-append", "v", D)
    slots = torch.randperm(NB * bs, generator=g)[:N].to(torch.int64)
    slots[4] = -1
    pos = torch.randint(0, 4096, (N,), generator=g)
    dev, host = prologue(D, norm=norm, rd=rd, off=off, inter=inter, seed=1, had=had)
    kg = guarded(torch.empty((N, Hkv, D), dtype=torch.bfloat16, device="cuda"))
    kvq.kvq_norm_rope_apply(dev, k.cuda(), kg, pos.cuda() if rd else None)
    kr = bits(kg)  # the GPU's prologue rows of K
    ref, bad, ref64 = orc.norm_rope(bits(k), positions=pos.numpy(), return_f64=True, **host)
    assert bad == 0
    check_prologue_rows(kr, ref, ref64, fp32_error_bound(bits(k), pos.numpy(), host, ref64))
    qmax = orc.QMAX[dtype]
    kf = torch.from_numpy(kr.view(np.int16)).view(torch.bfloat16).float()
    ks = None
    if kmode == kvq.PER_CHANNEL:  # calibrated on the normalized K (what the cache holds)
        ks = (kf.abs().amax(0) / qmax * 1.05).clamp_min(1e-6)
    vs = (v.float().abs().max() / qmax * 1.05).reshape(1) if vmode == kvq.PER_TENSOR else None
    cache = kvq.QuantizedPagedCache(dtype, kmode, vmode, NB, bs, Hkv, D, k_static=ks, v_static=vs, group_size=gs)
    kvq.kvq_append_norm_rope(cache, dev, k.cuda(), v.cuda(), slots.cuda(), pos.cuda() if rd else None)
    assert kvq.kvq_get_device_error() == 0
    oc = orc.OracleCache(dtype, kmode, vmode, NB, bs, Hkv, D, None if ks is None else ks.numpy(),
                         None if vs is None else vs.numpy(), group_size=gs)
    assert oc.append(kr, bits(v), slots.numpy()) == 0
    assert np.array_equal(cache.k_codes.cpu().numpy(), oc.k_codes)
    assert np.array_equal(cache.v_codes.cpu().numpy(), oc.v_codes)
    if kmode in (kvq.PER_ROW, kvq.PER_GROUP):
        assert np.array_equal(cache.k_scale.cpu().numpy().view(np.uint32), oc.k_scale.view(np.uint32))
    if vmode == kvq.PER_ROW:
        assert np.array_equal(cache.v_scale.cpu().numpy().view(np.uint32), oc.v_scale.view(np.uint32))


def test_append_norm_rope_skips_tokens_with_bad_positions(lib, orc):
    D, Hkv, bs, NB, N = 128, 2, 16, 4, 10
    k = synth.randn_bf16((N, Hkv, D), "cpu", "gpu-normrope-skip", "k")
    v = synth.randn_bf16((N, Hkv, D), "cpu", "gpu-normrope-skip", "v")
    slots = torch.arange(N, dtype=torch.int64)
    pos = torch.arange(N, dtype=torch.int64)
    pos[2] = 64  # tables hold 0..63
    dev, host = prologue(D, norm=True, rd=64, off=0, inter=False, max_pos=64)
    cache = kvq.QuantizedPagedCache(kvq.INT8, kvq.PER_ROW, kvq.PER_ROW, NB, bs, Hkv, D)
    cache.k_codes.fill_(0x5A)
    cache.v_codes.fill_(0x5A)
    kvq.kvq_append_norm_rope(cache, dev, k.cuda(), v.cuda(), slots.cuda(), pos.cuda())
    assert kvq.kvq_get_device_error() == kvq.DEVERR_POSITION
    kc = cache.k_codes.cpu().numpy()
    vc = cache.v_codes.cpu().numpy()
    assert (kc[0, :, 2] == 0x5A).all() and (vc[0, :, 2] == 0x5A).all()  # slot 2 not written
    assert not (kc[0, :, 3] == 0x5A).all()


def build_rotated_case(orc, dt, had, *, B=3, Hq=8, Hkv=2, D=128, T=2, bs=16, seed=2):
    """A cache filled through kvq_append_norm_rope, the oracle cache filled
    with the oracle's own fp64 prologue rows, and queries before the prologue."""
    L = np.array([40, 97, 2], np.int32)[:B]
    mb = 8
    NB = B * mb
    table = (np.arange(B)[:, None] * mb + np.arange(mb)[None, :]).astype(np.int32)
    dev, host = prologue(D, norm=True, rd=D, off=0, inter=False, max_pos=256, seed=seed, had=had)
    cache = kvq.QuantizedPagedCache(DT[dt], kvq.PER_ROW, kvq.PER_ROW, NB, bs, Hkv, D)
    oc = orc.OracleCache(DT[dt], kvq.PER_ROW, kvq.PER_ROW, NB, bs, Hkv, D)
    for b in range(B):
        n = int(L[b])
        k = synth.randn_bf16((n, Hkv, D), "cpu", "gpu-normrope-dec", "k", b)
        v = synth.randn_bf16((n, Hkv, D), "cpu", "gpu-normrope-dec", "v", b)
        pos = torch.arange(n, dtype=torch.int64)
        slots = torch.from_numpy(table[b, pos.numpy() // bs] * bs + pos.numpy() % bs).to(torch.int64)
        kvq.kvq_append_norm_rope(cache, dev, k.cuda(), v.cuda(), slots.cuda(), pos.cuda())
        kr, _ = orc.norm_rope(bits(k), positions=pos.numpy(), **host)
        oc.append(kr, bits(v), slots.numpy())
    q = synth.randn_bf16((B, T, Hq, D), "cpu", "gpu-normrope-dec", "q")
    qpos = torch.from_numpy(np.concatenate([np.arange(L[b] - T, L[b]) for b in range(B)])).to(torch.int64)
    qr, _ = orc.norm_rope(bits(q.reshape(B * T, Hq, D)), positions=qpos.numpy(), **host)
    ref, _ = oc.attend(qr.reshape(B, T, Hq, D), table, L, q_tokens=T)
    return dict(cache=cache, dev=dev, q=q, qpos=qpos, table=table, L=L, ref=ref, B=B, T=T, Hq=Hq, D=D, mb=mb)


@pytest.mark.parametrize("dt,had", [("int8", False), ("int4", True), ("int4", False)])
def test_decode_over_prologue_rows_matches_oracle_attention(lib, orc, dt, had):
    """q through kvq_norm_rope_apply, K through kvq_append_norm_rope (with and
    without the Hadamard rotation), then decode + combine: within 2e-3
    relative L2 of oracle attention over the oracle's own prologue rows."""
    c = build_rotated_case(orc, dt, had)
    B, T, Hq, D = c["B"], c["T"], c["Hq"], c["D"]
    qd = c["q"].reshape(B * T, Hq, D).cuda()
    kvq.kvq_norm_rope_apply(c["dev"], qd, qd, c["qpos"].cuda())
    params = kvq.make_params(B, Hq, T, c["mb"])
    bufs = kvq.alloc_decode_buffers(c["cache"], params)
    out, _ = kvq.decode_step(c["cache"], params, qd.reshape(B, T, Hq, D), torch.from_numpy(c["table"]).cuda(),
                             torch.from_numpy(c["L"]).cuda(), bufs)
    assert kvq.kvq_get_device_error() == 0
    got = out.float().cpu().numpy().astype(np.float64)
    rel = np.linalg.norm(got - c["ref"]) / np.linalg.norm(c["ref"])
    assert rel <= 2e-3, rel


def test_query_prologue_then_decode_back_to_back(lib, orc):
    """kvq_norm_rope_apply writes q and kvq_decode reads it as the very next
    kernel on the stream, with every other input staged on the device
    beforehand, so the two kernels overlap as far as programmatic dependent
    launch lets them.  With the default flags kvq_decode reads q only after
    the prologue kernel has completed: each round's output must match the
    oracle although q is poisoned (NaN) right before the prologue rewrites
    it."""
    c = build_rotated_case(orc, "int8", False)
    B, T, Hq, D = c["B"], c["T"], c["Hq"], c["D"]
    x = c["q"].reshape(B * T, Hq, D).cuda()
    qd = guarded(torch.empty_like(x))
    qpos = c["qpos"].cuda()
    table = torch.from_numpy(c["table"]).cuda()
    lens = torch.from_numpy(c["L"]).cuda()
    params = kvq.make_params(B, Hq, T, c["mb"])
    bufs = kvq.alloc_decode_buffers(c["cache"], params)
    outs = []
    torch.cuda.synchronize()
    for _ in range(20):
        qd.fill_(float("nan"))
        kvq.kvq_norm_rope_apply(c["dev"], x, qd, qpos)
        kvq.kvq_decode(c["cache"], params, qd.view(B, T, Hq, D), table, lens, bufs.workspace)
        kvq.kvq_combine(c["cache"], params, bufs.workspace, None, bufs.out, bufs.lse)
        outs.append(bufs.out.clone())
    torch.cuda.synchronize()
    assert kvq.kvq_get_device_error() == 0
    for o in outs:
        assert torch.equal(o, outs[0])
    got = outs[0].float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    rel = np.linalg.norm(got - c["ref"]) / np.linalg.norm(c["ref"])
    assert rel <= 2e-3, rel
