"""The LATENT cache layout (absorbed MLA; onnxruntime PR #29912 kv_cache_layout
and v_head_size): one cache whose rows are K, V = their leading v_head_size
channels with K's scales.  Append writes K only; decode, combine and prefill
against the oracle's latent attention (2e-3 relative L2), at head dims up to
256 and at the pages' DeepSeek-V3 shape, head_dim 576 with v_head_size 512."""
import numpy as np
import pytest
import torch

from decode_attention_quantized_gb300 import kvq, synth

from guard import guarded

pytestmark = pytest.mark.gpu

DT = {"int8": kvq.INT8, "fp8": kvq.FP8_E4M3, "int4": kvq.INT4}


@pytest.fixture(scope="module")
def lib():
    from decode_attention_quantized_gb300 import build
    build.build()
    return kvq.load()


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def build_case(orc, *, dt, kmode, D, Dv, Hq, Hkv, lens, bs=16, seed=0, group_size=0):
    B = len(lens)
    mb = max((L + bs - 1) // bs for L in lens)
    NB = B * mb + 3
    g = synth.generator("cpu", "latent", seed, "perm")
    perm = torch.randperm(NB, generator=g).numpy().astype(np.int32)
    table = perm[: B * mb].reshape(B, mb)
    qmax = orc.QMAX[DT[dt]]
    ks = None
    rows = [synth.randn_bf16((L, Hkv, D), "cpu", "latent", seed, "k", b) for b, L in enumerate(lens)]
    if kmode == kvq.PER_CHANNEL:
        ks = torch.stack([r.float().abs().amax(0) for r in rows]).amax(0) / qmax * 1.05
    elif kmode == kvq.PER_TENSOR:
        ks = (max(float(r.float().abs().max()) for r in rows) / qmax * 1.05) * torch.ones(1)
    cache = kvq.QuantizedPagedCache(DT[dt], kmode, kmode, NB, bs, Hkv, D, k_static=ks, latent=True, v_head_size=Dv,
                                    group_size=group_size)
    oc = orc.OracleCache(DT[dt], kmode, kmode, NB, bs, Hkv, D, None if ks is None else ks.numpy(), latent=True,
                         v_head_size=Dv, group_size=group_size)
    for b, (L, k) in enumerate(zip(lens, rows)):
        t = np.arange(L)
        slots = torch.from_numpy(table[b, t // bs].astype(np.int64) * bs + t % bs)
        kvq.kvq_append(cache, k.cuda(), None, slots.cuda())
        assert oc.append(bits(k), None, slots.numpy()) == 0
    assert kvq.kvq_get_device_error() == 0
    assert np.array_equal(cache.k_codes.cpu().numpy(), oc.k_codes)
    if kmode in (kvq.PER_ROW, kvq.PER_GROUP):
        assert np.array_equal(cache.k_scale.cpu().numpy().view(np.uint32), oc.k_scale.view(np.uint32))
    return cache, oc, table, np.array(lens, np.int32)


@pytest.mark.parametrize("dt", list(DT))
@pytest.mark.parametrize("kmode", [kvq.PER_ROW, kvq.PER_CHANNEL])
@pytest.mark.parametrize("D,Dv,Hq,Hkv,T", [(128, 128, 8, 2, 1), (256, 192, 16, 4, 1), (128, 64, 16, 2, 4),
                                          (256, 256, 24, 4, 8), (128, 96, 32, 4, 8)])
def test_latent_decode_matches_oracle(lib, orc, dt, kmode, D, Dv, Hq, Hkv, T):
    cache, oc, table, lens = build_case(orc, dt=dt, kmode=kmode, D=D, Dv=Dv, Hq=Hq, Hkv=Hkv, lens=[300, 41, 1000])
    B = len(lens)
    q = synth.randn_bf16((B, T, Hq, D), "cpu", "latent", "q", T)
    sink = torch.randn(Hq, generator=synth.generator("cpu", "latent", "sink"))
    params = kvq.make_params(B, Hq, T, table.shape[1])
    bufs = kvq.alloc_decode_buffers(cache, params)
    assert bufs.out.shape[-1] == Dv
    out, lse = kvq.decode_step(cache, params, q.cuda(), torch.from_numpy(table).cuda(), torch.from_numpy(lens).cuda(),
                               bufs, sink.cuda())
    assert kvq.kvq_get_device_error() == 0
    ref, ref_lse = oc.attend(bits(q), table, lens, q_tokens=T, head_sink=sink.numpy())
    got = out.float().cpu().numpy().astype(np.float64)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel <= 2e-3, rel
    assert np.allclose(lse.cpu().numpy(), ref_lse, atol=1e-3)


def test_latent_prefill_matches_oracle(lib, orc):
    cache, oc, table, lens = build_case(orc, dt="int8", kmode=kvq.PER_ROW, D=256, Dv=192, Hq=16, Hkv=4,
                                        lens=[200, 64, 700])
    B, C, Hq = len(lens), 24, 16
    q = synth.randn_bf16((B, C, Hq, 256), "cpu", "latent", "prefill-q")
    params = kvq.make_params(B, Hq, C, table.shape[1])
    ws = guarded(torch.empty((kvq.kvq_prefill_workspace_size(cache, params) + 3) // 4, dtype=torch.int32, device="cuda"))
    out = guarded(torch.empty((B, C, Hq, 192), dtype=torch.bfloat16, device="cuda"))
    kvq.kvq_prefill(cache, params, q.cuda(), torch.from_numpy(table).cuda(), torch.from_numpy(lens).cuda(), None,
                    out, None, ws)
    assert kvq.kvq_get_device_error() == 0
    ref, _ = oc.attend(bits(q), table, lens, q_tokens=C)
    rel = np.linalg.norm(out.float().cpu().numpy().astype(np.float64) - ref) / np.linalg.norm(ref)
    assert rel <= 2e-3, rel


@pytest.mark.parametrize("dt", list(DT))
@pytest.mark.parametrize("D,Dv,gsize,Hq,Hkv,T", [(128, 64, 32, 16, 2, 1), (256, 192, 64, 8, 4, 2)])
def test_latent_with_group_scales(lib, orc, dt, D, Dv, gsize, Hq, Hkv, T):
    """A LATENT cache with per-group scales: V, the leading Dv channels of the
    K row, takes K's group scales channel group by channel group."""
    cache, oc, table, lens = build_case(orc, dt=dt, kmode=kvq.PER_GROUP, D=D, Dv=Dv, Hq=Hq, Hkv=Hkv,
                                        lens=[300, 41, 1000], group_size=gsize)
    B = len(lens)
    q = synth.randn_bf16((B, T, Hq, D), "cpu", "latent", "q-group", T)
    params = kvq.make_params(B, Hq, T, table.shape[1])
    bufs = kvq.alloc_decode_buffers(cache, params)
    out, lse = kvq.decode_step(cache, params, q.cuda(), torch.from_numpy(table).cuda(), torch.from_numpy(lens).cuda(),
                               bufs)
    assert kvq.kvq_get_device_error() == 0
    ref, ref_lse = oc.attend(bits(q), table, lens, q_tokens=T)
    got = out.float().cpu().numpy().astype(np.float64)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel <= 2e-3, rel
    assert np.allclose(lse.cpu().numpy(), ref_lse, atol=1e-3)


MLA = [(8, 1, 1), (16, 2, 2), (8, 1, 4), (6, 1, 8)]  # Hq, Hkv, T: 8, 16, 32, 48 query rows per kv head


@pytest.mark.parametrize("dt", ["int8", "fp8"])
@pytest.mark.parametrize("kmode", [kvq.PER_ROW, kvq.PER_CHANNEL, kvq.PER_TENSOR])
@pytest.mark.parametrize("Hq,Hkv,T", MLA)
def test_latent_576_decode_matches_oracle(lib, orc, dt, kmode, Hq, Hkv, T):
    """head_dim 576, v_head_size 512 (the pages' DeepSeek-V3 example) on the
    mma.sync wide layout, V read from the K codes already in each stage."""
    cache, oc, table, lens = build_case(orc, dt=dt, kmode=kmode, D=576, Dv=512, Hq=Hq, Hkv=Hkv,
                                        lens=[300, 41, 1000], bs=64, seed=Hq * T + kmode)
    B = len(lens)
    q = synth.randn_bf16((B, T, Hq, 576), "cpu", "latent", "q576", T)
    sink = torch.randn(Hq, generator=synth.generator("cpu", "latent", "sink576"))
    for window, softcap in ((0, 0.0), (200, 30.0)):
        params = kvq.make_params(B, Hq, T, table.shape[1], window=window, softcap=softcap)
        bufs = kvq.alloc_decode_buffers(cache, params)
        assert bufs.out.shape[-1] == 512
        out, lse = kvq.decode_step(cache, params, q.cuda(), torch.from_numpy(table).cuda(),
                                   torch.from_numpy(lens).cuda(), bufs, sink.cuda())
        assert kvq.kvq_get_device_error() == 0
        ref, ref_lse = oc.attend(bits(q), table, lens, q_tokens=T, head_sink=sink.numpy(), window=window,
                                 softcap=softcap)
        got = out.float().cpu().numpy().astype(np.float64)
        rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert rel <= 2e-3, (window, rel)
        assert np.allclose(lse.cpu().numpy(), ref_lse, atol=1e-3)
        first = out.clone()
        kvq.decode_step(cache, params, q.cuda(), torch.from_numpy(table).cuda(), torch.from_numpy(lens).cuda(),
                        bufs, sink.cuda())
        assert torch.equal(out, first)


def test_latent_576_prefill_matches_oracle(lib, orc):
    cache, oc, table, lens = build_case(orc, dt="int8", kmode=kvq.PER_ROW, D=576, Dv=512, Hq=4, Hkv=1,
                                        lens=[200, 64, 700], bs=64, seed=5)
    B, C, Hq = len(lens), 24, 4
    q = synth.randn_bf16((B, C, Hq, 576), "cpu", "latent", "prefill-q576")
    params = kvq.make_params(B, Hq, C, table.shape[1])
    ws = guarded(torch.empty((kvq.kvq_prefill_workspace_size(cache, params) + 3) // 4, dtype=torch.int32, device="cuda"))
    out = guarded(torch.empty((B, C, Hq, 512), dtype=torch.bfloat16, device="cuda"))
    kvq.kvq_prefill(cache, params, q.cuda(), torch.from_numpy(table).cuda(), torch.from_numpy(lens).cuda(), None,
                    out, None, ws)
    assert kvq.kvq_get_device_error() == 0
    ref, _ = oc.attend(bits(q), table, lens, q_tokens=C)
    rel = np.linalg.norm(out.float().cpu().numpy().astype(np.float64) - ref) / np.linalg.norm(ref)
    assert rel <= 2e-3, rel


def test_latent_576_shapes_beyond_the_wide_layout_are_refused(lib):
    cache = kvq.QuantizedPagedCache(kvq.INT8, kvq.PER_ROW, kvq.PER_ROW, 8, 64, 1, 576, latent=True, v_head_size=512)
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_decode_workspace_size(cache, kvq.make_params(1, 8, 8, 4))  # 64 query rows per kv head
    assert e.value.status == 2


def test_latent_576_fused_prologue_on_the_rotary_suffix(lib, orc):
    """MLA rotates only the 64 positional channels after the 512 latent ones
    (rotary_offset, PR #29912): the fused append writes the codes the oracle
    quantizer gives for the GPU's own prologue rows."""
    D, Hkv, bs, NB, N = 576, 1, 64, 6, 150
    k = synth.randn_bf16((N, Hkv, D), "cpu", "latent", "mla-k")
    w = synth.norm_weight_bf16(D, "cpu", "latent", "mla-w")
    cos, sin = synth.rope_tables(4096, 64)
    pro = kvq.NormRope(norm_weight=w.cuda(), eps=1e-6, rotary_dim=64, rotary_offset=512,
                       cos=torch.from_numpy(cos).cuda(), sin=torch.from_numpy(sin).cuda())
    pos = torch.randint(0, 4096, (N,), generator=synth.generator("cpu", "latent", "mla-pos"))
    slots = torch.randperm(NB * bs, generator=synth.generator("cpu", "latent", "mla-slots"))[:N].to(torch.int64)
    kg = guarded(torch.empty((N, Hkv, D), dtype=torch.bfloat16, device="cuda"))
    kvq.kvq_norm_rope_apply(pro, k.cuda(), kg, pos.cuda())
    host = dict(norm_weight=bits(w), eps=1e-6, rotary_dim=64, rotary_offset=512, cos=cos, sin=sin)
    ref, bad, ref64 = orc.norm_rope(bits(k), positions=pos.numpy(), return_f64=True, **host)
    assert bad == 0
    # the GPU rows are the fp64 oracle's rounded to bf16, but at near-ties
    got = bits(kg)
    differ = np.count_nonzero(got != ref)
    assert differ <= 0.001 * got.size, differ
    cache = kvq.QuantizedPagedCache(kvq.INT8, kvq.PER_ROW, kvq.PER_ROW, NB, bs, Hkv, D, latent=True, v_head_size=512)
    kvq.kvq_append_norm_rope(cache, pro, k.cuda(), None, slots.cuda(), pos.cuda())
    assert kvq.kvq_get_device_error() == 0
    oc = orc.OracleCache(kvq.INT8, kvq.PER_ROW, kvq.PER_ROW, NB, bs, Hkv, D, None, latent=True, v_head_size=512)
    assert oc.append(got, None, slots.numpy()) == 0
    assert np.array_equal(cache.k_codes.cpu().numpy(), oc.k_codes)
    assert np.array_equal(cache.k_scale.cpu().numpy().view(np.uint32), oc.k_scale.view(np.uint32))
