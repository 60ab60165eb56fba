"""The LATENT cache layout (absorbed MLA; onnxruntime PR #29912 kv_cache_layout
and v_head_size): one cache whose rows are K, V = their leading v_head_size
channels with K's scales.  Append writes K only; decode, combine and prefill
against the oracle's latent attention (2e-3 relative L2)."""
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
