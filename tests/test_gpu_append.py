"""kvq_append on the GPU against the oracle: quantized codes and per-row
scales bit-exact for every element type and scale mode."""
import numpy as np
import pytest
import torch

from decode_attention_quantized_gb300 import kvq, synth

pytestmark = pytest.mark.gpu

DT = {"int8": kvq.INT8, "fp8": kvq.FP8_E4M3, "int4": kvq.INT4}
MODES = {"row": kvq.PER_ROW, "tensor": kvq.PER_TENSOR, "channel": kvq.PER_CHANNEL}


@pytest.fixture(scope="module")
def lib():
    from decode_attention_quantized_gb300 import build
    build.build()
    return kvq.load()


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def static_scale(mode, x, qmax, g):
    if mode == kvq.PER_TENSOR:
        return (x.float().abs().max() / qmax * 1.1).reshape(1)
    if mode == kvq.PER_CHANNEL:
        f = 1.0 + 0.3 * torch.rand(x.shape[1:], generator=g)
        return (x.float().abs().amax(0) / qmax * f).clamp_min(1e-6)
    return None


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("dt", list(DT))
@pytest.mark.parametrize("km,vm", [("row", "row"), ("tensor", "tensor"), ("channel", "channel"),
                                   ("channel", "tensor"), ("row", "channel")])
def test_append_codes_and_scales_bit_exact(lib, orc, D, dt, km, vm):
    dtype, kmode, vmode = DT[dt], MODES[km], MODES[vm]
    g = torch.Generator().manual_seed(D * 7 + dtype)
    Hkv, bs, NB = 3, 16, 40
    N = 300
    k = (torch.randn(N, Hkv, D, generator=g) * torch.exp(torch.randn(Hkv, D, generator=g))).to(torch.bfloat16)
    v = torch.randn(N, Hkv, D, generator=g).to(torch.bfloat16)
    k[5] = 0  # an all-zero row (scale 0, zero codes)
    slots = torch.randperm(NB * bs, generator=g)[:N].to(torch.int64)
    slots[7] = -1   # padding token
    qmax = orc.QMAX[dtype]
    ks, vs = static_scale(kmode, k, qmax, g), static_scale(vmode, v, qmax, g)
    cache = kvq.QuantizedPagedCache(dtype, kmode, vmode, NB, bs, Hkv, D, k_static=ks, v_static=vs)
    kvq.kvq_append(cache, k.cuda(), v.cuda(), slots.cuda())
    assert kvq.kvq_get_device_error() == 0
    oc = orc.OracleCache(dtype, kmode, vmode, NB, bs, Hkv, D, None if ks is None else ks.numpy(),
                         None if vs is None else vs.numpy())
    assert oc.append(bits(k), bits(v), slots.numpy()) == 0
    assert np.array_equal(cache.k_codes.cpu().numpy(), oc.k_codes)
    assert np.array_equal(cache.v_codes.cpu().numpy(), oc.v_codes)
    if kmode == kvq.PER_ROW:
        assert np.array_equal(cache.k_scale.cpu().numpy().view(np.uint32), oc.k_scale.view(np.uint32))
    if vmode == kvq.PER_ROW:
        assert np.array_equal(cache.v_scale.cpu().numpy().view(np.uint32), oc.v_scale.view(np.uint32))


@pytest.mark.parametrize("dt", list(DT))
@pytest.mark.parametrize("scale", [1.0, 0.37, 3.1e-3, 1e-40, 7.5e5])
def test_every_bf16_value_quantizes_like_the_oracle(lib, orc, dt, scale):
    """All finite bf16 bit patterns through the GPU's conversion (e4m3 rounding
    and saturation, int8/int4 ties and clamping) against the oracle."""
    dtype = DT[dt]
    u = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = (u.astype(np.uint32) << 16).view(np.float32)
    u = u[np.isfinite(f)]
    D = 64
    n = len(u) // D
    x = torch.from_numpy(u[: n * D].view(np.int16).copy()).view(torch.bfloat16).reshape(n, 1, D)
    s = torch.tensor([scale], dtype=torch.float32)
    cache = kvq.QuantizedPagedCache(dtype, kvq.PER_TENSOR, kvq.PER_TENSOR, (n + 15) // 16, 16, 1, D,
                                    k_static=s, v_static=s)
    slots = torch.arange(n, dtype=torch.int64)
    kvq.kvq_append(cache, x.cuda(), x.cuda(), slots.cuda())
    oc = orc.OracleCache(dtype, orc.PER_TENSOR, orc.PER_TENSOR, (n + 15) // 16, 16, 1, D, s.numpy(), s.numpy())
    oc.append(bits(x), bits(x), slots.numpy())
    assert np.array_equal(cache.k_codes.cpu().numpy(), oc.k_codes)


def test_out_of_pool_slot_is_flagged_and_skipped(lib):
    kvq.kvq_get_device_error(clear=True)
    cache = kvq.QuantizedPagedCache(kvq.INT8, kvq.PER_ROW, kvq.PER_ROW, 2, 16, 1, 64)
    x = torch.ones(3, 1, 64, dtype=torch.bfloat16, device="cuda")
    slots = torch.tensor([0, 32, 5], dtype=torch.int64, device="cuda")   # 32 == capacity
    kvq.kvq_append(cache, x, x, slots)
    assert kvq.kvq_get_device_error(clear=True) == kvq.DEVERR_SLOT
    codes = cache.k_codes.cpu().numpy()
    assert (codes[0, 0, 0] == 127).all() and (codes[0, 0, 5] == 127).all()
    assert codes.reshape(-1, 64).any(axis=1).sum() == 2
