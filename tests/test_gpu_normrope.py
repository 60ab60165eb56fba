"""The QK-RMSNorm + RoPE prologue on the GPU against the oracle
(QkNormRotaryTNH, onnxruntime PR #29912, Summary of Changes).

kvq_norm_rope_apply's bf16 rows and kvq_append_norm_rope's codes and scales
are compared element by element with the oracle; both sides compute in fp32
in the same fixed order and round once to bf16, so the rows agree bit for
bit.  Then a decode over
prologue-rotated queries and keys is compared with oracle attention."""
import numpy as np
import pytest
import torch

from decode_attention_quantized_gb300 import kvq, synth

pytestmark = pytest.mark.gpu

DT = {"int8": kvq.INT8, "fp8": kvq.FP8_E4M3, "int4": kvq.INT4}


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


CASES = [  # (D, norm, rotary_dim, rotary_offset, interleaved, hadamard)
    (64, True, 64, 0, False, False), (128, True, 128, 0, True, False), (256, True, 64, 192, False, False),
    (128, False, 32, 40, False, False), (256, True, 0, 0, False, False), (64, False, 16, 48, True, False),
    (64, True, 64, 0, False, True), (128, True, 128, 0, False, True), (256, False, 0, 0, False, True),
]


@pytest.mark.parametrize("D,norm,rd,off,inter,had", CASES)
def test_norm_rope_apply_bit_exact(lib, orc, D, norm, rd, off, inter, had):
    N, H = 37, 6  # a ragged token count
    x = synth.randn_bf16((N, H, D), "cpu", "gpu-normrope", "x", D) * 3
    pos = torch.randint(0, 4096, (N,), generator=synth.generator("cpu", "gpu-normrope", "pos", D))
    pos[0], pos[1] = 0, 4095
    dev, host = prologue(D, norm=norm, rd=rd, off=off, inter=inter, had=had)
    y = torch.zeros_like(x).cuda()
    kvq.kvq_norm_rope_apply(dev, x.cuda(), y, pos.cuda() if rd else None)
    assert kvq.kvq_get_device_error() == 0
    ref, bad = orc.norm_rope(bits(x), positions=pos.numpy(), **host)
    assert bad == 0
    assert np.array_equal(bits(y), ref)
    # in place gives the same rows
    xi = x.cuda()
    kvq.kvq_norm_rope_apply(dev, xi, xi, pos.cuda() if rd else None)
    assert np.array_equal(bits(xi), ref)


def test_norm_rope_apply_flags_positions_outside_the_tables(lib, orc):
    D, N, H = 128, 8, 4
    x = synth.randn_bf16((N, H, D), "cpu", "gpu-normrope", "badpos")
    pos = torch.arange(N, dtype=torch.int64) * 60
    pos[3], pos[6] = -5, 512  # tables hold positions 0..511; the others are inside
    dev, host = prologue(D, norm=True, rd=128, off=0, inter=False, max_pos=512)
    y = torch.full((N, H, D), 7.0, dtype=torch.bfloat16, device="cuda")
    kvq.kvq_norm_rope_apply(dev, x.cuda(), y, pos.cuda())
    assert kvq.kvq_get_device_error() == kvq.DEVERR_POSITION
    ref, bad = orc.norm_rope(bits(x), positions=pos.numpy(), **host)
    assert bad == 2
    got = bits(y)
    good = [n for n in range(N) if n not in (3, 6)]
    assert np.array_equal(got[good], ref[good])
    assert (y[[3, 6]].float() == 7.0).all().item()  # untouched


@pytest.mark.parametrize("dt", list(DT))
@pytest.mark.parametrize("km,vm", [("row", "row"), ("channel", "tensor")])
@pytest.mark.parametrize("D,norm,rd,off,inter,had", [(128, True, 128, 0, False, False), (256, True, 64, 0, True, False),
                                                     (64, False, 32, 16, False, False), (128, True, 128, 0, False, True),
                                                     (256, True, 256, 0, False, True)])
def test_append_norm_rope_codes_bit_exact(lib, orc, dt, km, vm, D, norm, rd, off, inter, had):
    """The fused prologue + quantizer writes exactly the codes (and per-row
    scales) the oracle gets by normalizing and rotating K, rounding it to
    bf16 and quantizing that; V is quantized as given."""
    modes = {"row": kvq.PER_ROW, "tensor": kvq.PER_TENSOR, "channel": kvq.PER_CHANNEL}
    dtype, kmode, vmode = DT[dt], modes[km], modes[vm]
    Hkv, bs, NB, N = 2, 16, 24, 150
    g = synth.generator("cpu", "gpu-normrope-append", D, dt)
    k = synth.randn_bf16((N, Hkv, D), "cpu", "gpu-normrope-append", "k", D)
    v = synth.randn_bf16((N, Hkv, D), "cpu", "gpu-normrope-append", "v", D)
    slots = torch.randperm(NB * bs, generator=g)[:N].to(torch.int64)
    slots[4] = -1
    pos = torch.randint(0, 4096, (N,), generator=g)
    dev, host = prologue(D, norm=norm, rd=rd, off=off, inter=inter, seed=1, had=had)
    kr, bad = orc.norm_rope(bits(k), positions=pos.numpy(), **host)  # the oracle's own K rows
    assert bad == 0
    qmax = orc.QMAX[dtype]
    kf = torch.from_numpy(kr.view(np.int16)).view(torch.bfloat16).float()
    ks = None
    if kmode == kvq.PER_CHANNEL:  # calibrated on the normalized K (what the cache holds)
        ks = (kf.abs().amax(0) / qmax * 1.05).clamp_min(1e-6)
    vs = (v.float().abs().max() / qmax * 1.05).reshape(1) if vmode == kvq.PER_TENSOR else None
    cache = kvq.QuantizedPagedCache(dtype, kmode, vmode, NB, bs, Hkv, D, k_static=ks, v_static=vs)
    kvq.kvq_append_norm_rope(cache, dev, k.cuda(), v.cuda(), slots.cuda(), pos.cuda() if rd else None)
    assert kvq.kvq_get_device_error() == 0
    oc = orc.OracleCache(dtype, kmode, vmode, NB, bs, Hkv, D, None if ks is None else ks.numpy(),
                         None if vs is None else vs.numpy())
    assert oc.append(kr, bits(v), slots.numpy()) == 0
    assert np.array_equal(cache.k_codes.cpu().numpy(), oc.k_codes)
    assert np.array_equal(cache.v_codes.cpu().numpy(), oc.v_codes)
    if kmode == kvq.PER_ROW:
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


@pytest.mark.parametrize("dt,had", [("int8", False), ("int4", True), ("int4", False)])
def test_decode_over_prologue_rows_matches_oracle_attention(lib, orc, dt, had):
    """q through kvq_norm_rope_apply, K through kvq_append_norm_rope (with and
    without the Hadamard rotation), then decode + combine: within 2e-3
    relative L2 of oracle attention over the oracle's own prologue rows."""
    B, Hq, Hkv, D, T, bs = 3, 8, 2, 128, 2, 16
    L = np.array([40, 97, 2], np.int32)
    mb = 8
    NB = B * mb
    table = (np.arange(B)[:, None] * mb + np.arange(mb)[None, :]).astype(np.int32)
    dev, host = prologue(D, norm=True, rd=128, off=0, inter=False, max_pos=256, seed=2, had=had)
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
    qd = q.reshape(B * T, Hq, D).cuda()
    kvq.kvq_norm_rope_apply(dev, qd, qd, qpos.cuda())
    qr, _ = orc.norm_rope(bits(q.reshape(B * T, Hq, D)), positions=qpos.numpy(), **host)
    params = kvq.make_params(B, Hq, T, mb)
    bufs = kvq.alloc_decode_buffers(cache, params)
    out, _ = kvq.decode_step(cache, params, qd.reshape(B, T, Hq, D), torch.from_numpy(table).cuda(),
                             torch.from_numpy(L).cuda(), bufs)
    assert kvq.kvq_get_device_error() == 0
    ref, _ = oc.attend(qr.reshape(B, T, Hq, D), table, L, q_tokens=T)
    got = out.float().cpu().numpy().astype(np.float64)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel <= 2e-3, rel
