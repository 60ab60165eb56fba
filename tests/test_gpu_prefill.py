"""kvq_prefill (a chunk of C query tokens per sequence over the quantized
cache) against oracle attention with the same chunk: token c of sequence b
at position seq_lens[b] - C + c, causal within the chunk, sink and window as
in decode.  Within 2e-3 relative L2; lse within 1e-3; repeated calls bitwise
identical."""
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


def run_prefill(orc, *, dt, D, Hq, Hkv, C, lens, bs=16, window=0, sink=False, softcap=0.0, seed=0):
    B = len(lens)
    mb = max(1, max((L + bs - 1) // bs for L in lens))
    NB = B * mb
    table = (np.arange(B)[:, None] * mb + np.arange(mb)[None, :]).astype(np.int32)
    dtype = DT[dt]
    cache = kvq.QuantizedPagedCache(dtype, kvq.PER_ROW, kvq.PER_ROW, NB, bs, Hkv, D)
    oc = orc.OracleCache(dtype, kvq.PER_ROW, kvq.PER_ROW, NB, bs, Hkv, D)
    for b, L in enumerate(lens):
        if L == 0:
            continue
        k = synth.randn_bf16((L, Hkv, D), "cpu", "prefill", seed, "k", b)
        v = synth.randn_bf16((L, Hkv, D), "cpu", "prefill", seed, "v", b)
        t = np.arange(L)
        slots = torch.from_numpy(table[b, t // bs] * bs + t % bs).to(torch.int64)
        kvq.kvq_append(cache, k.cuda(), v.cuda(), slots.cuda())
        oc.append(bits(k), bits(v), slots.numpy())
    q = synth.randn_bf16((B, C, Hq, D), "cpu", "prefill", seed, "q")
    hs = torch.randn(Hq, generator=synth.generator("cpu", "prefill", seed, "sink")) if sink else None
    params = kvq.make_params(B, Hq, C, mb, window=window, softcap=softcap)
    ws = guarded(torch.empty((kvq.kvq_prefill_workspace_size(cache, params) + 3) // 4, dtype=torch.int32, device="cuda"))
    out = guarded(torch.empty((B, C, Hq, D), dtype=torch.bfloat16, device="cuda"))
    lse = guarded(torch.empty((B, C, Hq), dtype=torch.float32, device="cuda"))
    args = (cache, params, q.cuda(), torch.from_numpy(table).cuda(), torch.from_numpy(np.array(lens, np.int32)).cuda(),
            None if hs is None else hs.cuda(), out, lse, ws)
    kvq.kvq_prefill(*args)
    assert kvq.kvq_get_device_error() == 0
    first = out.clone()
    kvq.kvq_prefill(*args)
    assert torch.equal(first.view(torch.int16), out.view(torch.int16)), "repeated prefill differs"
    ref, ref_lse = oc.attend(bits(q), table, np.array(lens, np.int32), q_tokens=C, window=window, softcap=softcap,
                             head_sink=None if hs is None else hs.numpy())
    got = out.float().cpu().numpy().astype(np.float64)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert rel <= 2e-3, rel
    gl = lse.cpu().numpy().astype(np.float64)
    finite = np.isfinite(ref_lse)
    assert (np.isfinite(gl) == finite).all()
    assert np.allclose(gl[finite], ref_lse[finite], atol=1e-3)
    return rel


@pytest.mark.parametrize("C", [1, 5, 8, 12, 32, 64])
def test_prefill_chunk_sizes(lib, orc, C):
    run_prefill(orc, dt="int8", D=128, Hq=8, Hkv=2, C=C, lens=[C + 37, C + 200, C])


@pytest.mark.parametrize("dt,D,Hq,Hkv", [("int4", 256, 24, 4), ("fp8", 128, 32, 8), ("int8", 64, 4, 4),
                                         ("int8", 256, 48, 6)])
def test_prefill_types_and_groups(lib, orc, dt, D, Hq, Hkv):
    run_prefill(orc, dt=dt, D=D, Hq=Hq, Hkv=Hkv, C=16, lens=[300, 17, 1000])


def test_prefill_with_sink_window_and_softcap(lib, orc):
    run_prefill(orc, dt="int8", D=128, Hq=16, Hkv=4, C=24, lens=[500, 64, 2000], window=100, sink=True,
                softcap=30.0)


def test_prefill_rejects_a_virtual_batch_beyond_the_plan(lib):
    cache = kvq.QuantizedPagedCache(kvq.INT8, kvq.PER_ROW, kvq.PER_ROW, 4, 16, 1, 64)
    params = kvq.make_params(200, 4, 64, 4)  # 200 x 64 / 8 = 1600 virtual sequences > 1024
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_prefill_workspace_size(cache, params)
    assert e.value.status == 2
