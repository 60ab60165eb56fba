"""Group-wise scales (KVQ_SCALE_PER_GROUP) on the GPU against the fp64 oracle:
kvq_append's codes and group scales byte for byte, kvq_decode + kvq_combine
within the decode tolerance, over element types, head dims, group sizes,
scale-mode pairs and query-row counts: up to 16 rows per kv head (and above
the tensor-memory bound) on the mma.sync kernel's grouped layout, 17..48 rows
at head_dim 256 and 17..64 at 128 on the tensor-memory kernel."""
import math

import numpy as np
import pytest
import torch

from decode_attention_quantized_gb300 import kvq, synth
from decode_attention_quantized_gb300.workload import GpuWorkload

from parity import OracleSide, check_lse, check_rows

from guard import guarded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from decode_attention_quantized_gb300 import build
    build.build()
    return kvq.load()


def workload(dt, km, vm, D, gsize, *, G=4, T=1, L=(150, 77, 9, 300), bs=16, seed=0, **kw):
    # no one-key sequence by default: such a row is one dequantized V row, whose
    # bf16 rounding errors share the scale's mantissa and alone can exceed the
    # 2e-3 bar (2.27e-3 for the fp64 oracle's own output on one int4 input);
    # one-token sequences are in the row-count test
    L = np.array(L, np.int32)
    mb = max(1, math.ceil(int(L.max()) / bs))
    table = np.random.default_rng(seed).permutation(len(L) * mb).astype(np.int32).reshape(len(L), mb)
    return synth.Workload("group", dt, km, vm, len(L), G * 2, 2, D, T, bs, L, table, len(L) * mb,
                          k_channel_lognormal=0.5, seed=seed, group_size=gsize, **kw)


def run(orc, w, *, window=0):
    gw = GpuWorkload(w, gen_device="cpu")
    gw.fill_history()
    k_new, v_new, slots = gw.new_tokens()
    params = gw.params(window=window)
    bufs = gw.buffers(params)
    q = w.q("cpu").to("cuda")
    out, lse = gw.step(q, k_new, v_new, slots, params, bufs)
    torch.cuda.synchronize()
    assert kvq.kvq_get_device_error(clear=True) == 0
    side = OracleSide(orc, w, range(w.batch), "cpu", gw.k_static, gw.v_static)
    side.compare_cache(gw)
    ref, ref_lse = side.attend(q, window=window, sink=gw.head_sink)
    got = out.float().cpu().numpy().astype(np.float64)
    err = check_rows(got, ref)
    check_lse(lse.cpu().numpy().astype(np.float64), ref_lse)
    return gw, params, bufs, q, err


GRID = [(64, 32), (64, 64), (128, 32), (128, 64), (128, 128), (256, 32), (256, 128)]


@pytest.mark.parametrize("dt", [kvq.INT8, kvq.FP8_E4M3, kvq.INT4])
@pytest.mark.parametrize("D,gsize", GRID)
def test_group_both_sides(lib, orc, dt, D, gsize):
    run(orc, workload(dt, kvq.PER_GROUP, kvq.PER_GROUP, D, gsize, seed=D + gsize + dt))


@pytest.mark.parametrize("dt", [kvq.INT8, kvq.FP8_E4M3, kvq.INT4])
@pytest.mark.parametrize("km,vm", [(4, 1), (1, 4), (4, 2), (3, 4), (4, 3), (2, 4)])
def test_group_with_the_other_modes(lib, orc, dt, km, vm):
    run(orc, workload(dt, km, vm, 128, 32, seed=10 * km + vm + dt))


TC_GROUP = [  # dtype, D, group size, k_mode, v_mode, G, T (17..48 rows at D 256, 17..64 at 128)
    (kvq.INT4, 256, 64, 4, 4, 6, 8), (kvq.INT8, 256, 32, 4, 4, 8, 6), (kvq.FP8_E4M3, 256, 128, 4, 4, 4, 5),
    (kvq.INT4, 128, 32, 4, 4, 8, 8), (kvq.INT8, 128, 128, 4, 1, 5, 7), (kvq.FP8_E4M3, 128, 64, 1, 4, 3, 6),
    (kvq.INT4, 256, 32, 4, 3, 6, 6), (kvq.INT8, 128, 64, 2, 4, 8, 4), (kvq.INT4, 128, 128, 3, 4, 7, 7),
]


@pytest.mark.parametrize("case", TC_GROUP, ids=lambda c: f"dt{c[0]}-D{c[1]}-g{c[2]}-km{c[3]}vm{c[4]}-rows{c[5] * c[6]}")
def test_group_on_the_tensor_memory_kernel(lib, orc, case):
    """Group scales on the tcgen05 kernel: K columns carry code x group scale
    over a per-key power of two, V^T columns the group scale under the
    running normaliser; several 128-key tiles and pieces, ragged lengths."""
    dt, D, gs, km, vm, G, T = case
    w = workload(dt, km, vm, D, gs, G=G, T=T, L=(1500, T - 1, 129, 700), bs=32, seed=D + gs + G * T)
    gw, params, bufs, q, _ = run(orc, w)
    ref = bufs.out.clone()
    kvq.decode_step(gw.cache, params, q, gw.block_table, gw.seq_lens, bufs, gw.head_sink)
    assert torch.equal(bufs.out, ref)


def test_group_on_the_tensor_memory_kernel_with_sink_softcap_window(lib, orc):
    w = workload(kvq.INT4, kvq.PER_GROUP, kvq.PER_GROUP, 256, 64, G=6, T=8, L=(900, 300, 33), bs=32,
                 use_sink=True, softcap=30.0, seed=77)
    run(orc, w)
    run(orc, w, window=200)


@pytest.mark.parametrize("G,T", [(1, 1), (8, 1), (6, 8), (8, 8), (3, 5)])
def test_group_row_counts(lib, orc, G, T):
    """1 to 64 query rows per kv head: the grouped layout up to 16 rows and
    above 48 at head_dim 256 (row groups of 8, one key warp each above 32
    rows), the tensor-memory kernel for 48."""
    run(orc, workload(kvq.INT4, kvq.PER_GROUP, kvq.PER_GROUP, 256, 64, G=G, T=T, L=(200, T, 66), seed=G + T))


def test_group_with_sink_softcap_window_and_nan_bytes(lib, orc):
    """Sink, softcap and a window together; every unwritten slot holds the e4m3
    NaN byte and every unwritten scale slot a NaN, so the keys past each
    sequence's end carry NaN codes and NaN group scales."""
    w = workload(kvq.FP8_E4M3, kvq.PER_GROUP, kvq.PER_GROUP, 128, 32, G=4, T=2, L=(37, 300, 129, 8),
                 use_sink=True, softcap=20.0, seed=3)
    gw = GpuWorkload(w, gen_device="cpu")
    gw.cache.k_codes.fill_(0x7F)
    gw.cache.v_codes.fill_(0x7F)
    gw.cache.k_scale.fill_(float("nan"))
    gw.cache.v_scale.fill_(float("nan"))
    gw.fill_history()
    k_new, v_new, slots = gw.new_tokens()
    for window in (0, 50):
        params = gw.params(window=window)
        bufs = gw.buffers(params)
        q = w.q("cpu").to("cuda")
        if window == 0:
            out, lse = gw.step(q, k_new, v_new, slots, params, bufs)
        else:
            out, lse = kvq.decode_step(gw.cache, params, q, gw.block_table, gw.seq_lens, bufs, gw.head_sink)
        torch.cuda.synchronize()
        assert kvq.kvq_get_device_error(clear=True) == 0
        got = out.float().cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all()
        side = OracleSide(orc, w, range(w.batch), "cpu", gw.k_static, gw.v_static)
        ref, ref_lse = side.attend(q, window=window, sink=gw.head_sink)
        check_rows(got, ref)
        check_lse(lse.cpu().numpy().astype(np.float64), ref_lse)


def test_group_decode_is_deterministic(lib, orc):
    gw, params, bufs, q, _ = run(orc, workload(kvq.INT8, kvq.PER_GROUP, kvq.PER_GROUP, 256, 32,
                                               L=(3000, 17, 900), seed=9))
    ref = bufs.out.clone()
    for _ in range(5):
        kvq.decode_step(gw.cache, params, q, gw.block_table, gw.seq_lens, bufs)
        assert torch.equal(bufs.out, ref)


def test_group_scales_narrow_the_int4_error_on_outlier_channels(lib):
    """The page's reason for group-wise scales: with a few outlier channels
    per kv head, int4 per-group decode is closer to unquantized attention
    than int4 per-row decode (both measured on the GPU outputs)."""
    B, Hkv, G, D, L, bs = 2, 2, 4, 128, 512, 16
    gen = torch.Generator().manual_seed(1)
    k = torch.randn(B, L, Hkv, D, generator=gen)
    v = torch.randn(B, L, Hkv, D, generator=gen)
    k[..., 5] *= 30.0
    v[..., 77] *= 30.0
    k, v = k.to(torch.bfloat16), v.to(torch.bfloat16)
    q = torch.randn(B, 1, Hkv * G, D, generator=gen).to(torch.bfloat16)
    mb = L // bs
    table = torch.arange(B * mb, dtype=torch.int32).reshape(B, mb)
    lens = torch.full((B,), L, dtype=torch.int32)
    # unquantized reference in fp64
    kd, vd = k.double(), v.double()
    ref = torch.empty(B, Hkv * G, D, dtype=torch.float64)
    for b in range(B):
        for i in range(Hkv * G):
            s = kd[b, :, i // G] @ q[b, 0, i].double() / math.sqrt(D)
            ref[b, i] = torch.softmax(s, 0) @ vd[b, :, i // G]
    errs = {}
    for mode in (kvq.PER_ROW, kvq.PER_GROUP):
        cache = kvq.QuantizedPagedCache(kvq.INT4, mode, mode, B * mb, bs, Hkv, D, group_size=32)
        slots = (table.long()[:, :, None] * bs + torch.arange(bs)).reshape(B, L)
        for b in range(B):
            kvq.kvq_append(cache, k[b].cuda(), v[b].cuda(), slots[b].cuda())
        params = kvq.make_params(B, Hkv * G, 1, mb)
        bufs = kvq.alloc_decode_buffers(cache, params)
        out, _ = kvq.decode_step(cache, params, q.cuda(), table.cuda(), lens.cuda(), bufs)
        torch.cuda.synchronize()
        got = out.float().cpu().double()[:, 0]
        errs[mode] = float((got - ref).norm() / ref.norm())
    assert errs[kvq.PER_GROUP] < 0.5 * errs[kvq.PER_ROW], errs


def test_group_prefill_matches_oracle(lib, orc):
    """kvq_prefill over a per-group cache: a 24-token chunk per sequence (three
    virtual sequences of 8), causal inside the chunk, against oracle attention."""
    w = workload(kvq.INT8, kvq.PER_GROUP, kvq.PER_GROUP, 128, 32, G=4, T=1, L=(300, 64, 700), seed=21)
    gw = GpuWorkload(w, gen_device="cpu")
    gw.fill_history()
    k_new, v_new, slots = gw.new_tokens()
    kvq.kvq_append(gw.cache, k_new, v_new, slots)
    B, C, Hq, D = w.batch, 24, w.num_q_heads, w.head_dim
    q = synth.randn_bf16((B, C, Hq, D), "cpu", "group-prefill", 0, "q")
    params = kvq.make_params(B, Hq, C, w.max_blocks)
    ws = guarded(torch.empty((kvq.kvq_prefill_workspace_size(gw.cache, params) + 3) // 4, dtype=torch.int32, device="cuda"))
    out = guarded(torch.empty((B, C, Hq, D), dtype=torch.bfloat16, device="cuda"))
    lse = guarded(torch.empty((B, C, Hq), dtype=torch.float32, device="cuda"))
    kvq.kvq_prefill(gw.cache, params, q.cuda(), gw.block_table, gw.seq_lens, None, out, lse, ws)
    torch.cuda.synchronize()
    assert kvq.kvq_get_device_error(clear=True) == 0
    side = OracleSide(orc, w, range(B), "cpu", gw.k_static, gw.v_static)
    bits = q.contiguous().view(torch.int16).numpy().view(np.uint16)
    ref, ref_lse = side.cache.attend(bits, side.table, side.lens, q_tokens=C)
    got = out.float().cpu().numpy().astype(np.float64)
    check_rows(got, ref)
    check_lse(lse.cpu().numpy().astype(np.float64), ref_lse)
