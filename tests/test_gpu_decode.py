"""kvq_decode + kvq_combine on the GPU against the fp64 oracle, at sizes the
oracle finishes in seconds that still span several 64-key tiles, several
splits and a ragged tail; plus determinism, edge cases and device-side data
checks."""
import math

import numpy as np
import pytest
import torch

from decode_attention_quantized_gb300 import kvq, synth
from decode_attention_quantized_gb300.workload import GpuWorkload

from guard import guarded
from parity import OracleSide, bits, check_lse, check_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from decode_attention_quantized_gb300 import build
    build.build()
    return kvq.load()


def run_case(orc, w, *, window=0, gen="cpu", step=0, check_cache=True, max_seq_len=None, q_scale=1.0, flags=0):
    gw = GpuWorkload(w, gen_device=gen)
    gw.fill_history()
    k_new, v_new, slots = gw.new_tokens()
    params = gw.params(window=window, max_seq_len=max_seq_len, flags=flags)
    bufs = gw.buffers(params)
    q = w.q(gen, step).to("cuda")
    if q_scale != 1.0:
        q = (q.float() * q_scale).to(q.dtype)
    out, lse = gw.step(q, k_new, v_new, slots, params, bufs)
    torch.cuda.synchronize()
    assert kvq.kvq_get_device_error(clear=True) == 0
    side = OracleSide(orc, w, range(w.batch), gen, gw.k_static, gw.v_static)
    if check_cache:
        side.compare_cache(gw)
    ref, ref_lse = side.attend(q, window=window, sink=gw.head_sink)
    got = out.float().cpu().numpy().astype(np.float64)
    err = check_rows(got, ref)
    check_lse(lse.cpu().numpy().astype(np.float64), ref_lse)
    return gw, params, bufs, q, err


SMALL = [
    ("tiny", dict()),
    ("gqa", dict(ctx=3000)),
    ("gqa", dict(ctx=1, batch=2)),
    ("paged", dict(batch=5, max_ctx=700)),
    ("spec", dict(ctx=301, batch=2)),
    ("mixed", dict(batch=6, max_ctx=5000)),
]


@pytest.mark.parametrize("name,kw", SMALL, ids=[f"{n}-{i}" for i, (n, _) in enumerate(SMALL)])
def test_workloads_small(lib, orc, name, kw):
    w = synth.make(name, **kw)
    run_case(orc, w)
    if w.window:
        run_case(orc, w, window=w.window, check_cache=False)


@pytest.mark.parametrize("dt", [kvq.INT8, kvq.FP8_E4M3, kvq.INT4])
@pytest.mark.parametrize("km,vm", [(1, 1), (2, 2), (3, 3), (1, 3), (3, 1), (2, 1)])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_type_and_scale_grid(lib, orc, dt, km, vm, D):
    L = [150, 77, 1]
    w = synth.Workload("grid", dt, km, vm, 3, 8, 2, D, 2, 32, np.array(L, np.int32),
                       np.arange(3 * 5, dtype=np.int32).reshape(3, 5)[:, ::-1].copy(), 15,
                       k_channel_lognormal=0.5, seed=dt * 100 + km * 10 + vm)
    run_case(orc, w)


@pytest.mark.parametrize("G,T", [(1, 1), (2, 3), (5, 1), (8, 1), (6, 8), (8, 8), (3, 5)])
def test_group_and_draft_shapes(lib, orc, G, T):
    Hkv = 2
    L = np.array([200, T, 66], np.int32)
    bs = 16
    mb = 14
    w = synth.Workload("shapes", kvq.INT8, kvq.PER_ROW, kvq.PER_ROW, 3, G * Hkv, Hkv, 128, T, bs, L,
                       np.random.default_rng(G * 10 + T).permutation(3 * mb).astype(np.int32).reshape(3, mb),
                       3 * mb, seed=G * 10 + T)
    run_case(orc, w)


def test_edges_empty_short_and_windows(lib, orc):
    """seq_len 0 (empty: zero rows, lse -inf), seq_len < T (early drafts see
    nothing), a window smaller than a tile and one larger than the sequence,
    block sizes below and above the 64-key tile."""
    for bs, W in ((16, 5), (512, 3000), (64, 64), (256, 1)):
        L = np.array([0, 2, 1, 700, 129], np.int32)
        mb = max(1, math.ceil(700 / bs))
        w = synth.Workload("edges", kvq.INT8, kvq.PER_ROW, kvq.PER_ROW, 5, 12, 3, 64, 4, bs, L,
                           np.arange(5 * mb, dtype=np.int32).reshape(5, mb), 5 * mb, use_sink=True, seed=bs)
        run_case(orc, w)
        run_case(orc, w, window=W, check_cache=False)


def test_softcap_and_sink_together(lib, orc):
    w = synth.make("paged", batch=3, max_ctx=500)
    w.use_sink = True
    w.softcap = 3.0      # tight enough that the cap changes the result
    run_case(orc, w)


def test_determinism_and_fresh_workspace(lib, orc):
    """kv-quant-attn "Correctness": repeated decodes are bitwise identical
    (fixed merge order, no atomics), also with a re-created workspace."""
    w = synth.make("mixed", batch=5, max_ctx=6000)
    gw, params, bufs, q, _ = run_case(orc, w)
    ref = bufs.out.clone()
    ref_lse = bufs.lse.clone()
    for i in range(10):
        kvq.decode_step(gw.cache, params, q, gw.block_table, gw.seq_lens, bufs, gw.head_sink)
        assert torch.equal(bufs.out, ref) and torch.equal(bufs.lse, ref_lse)
    fresh = gw.buffers(params)
    fresh.workspace.fill_(0x7F7F7F7F)
    kvq.decode_step(gw.cache, params, q, gw.block_table, gw.seq_lens, fresh, gw.head_sink)
    assert torch.equal(fresh.out, ref)


@pytest.mark.parametrize("name,kw", [("mixed", dict(batch=5, max_ctx=6000)), ("spec", dict(ctx=700, batch=2))])
def test_early_inputs_flag_gives_the_same_bits(lib, orc, name, kw):
    """KVQ_DECODE_EARLY_INPUTS only moves the reads of q, the block table,
    seq_lens and the static scales ahead of the wait on the preceding kernel
    (here kvq_append, which writes none of them), and KVQ_DECODE_EARLY_CACHE
    the loads of every cache tile before the one holding the appended tokens:
    the result is bitwise the default path's, on both decode kernels."""
    w = synth.make(name, **kw)
    gw, params, bufs, q, _ = run_case(orc, w)
    ref, ref_lse = bufs.out.clone(), bufs.lse.clone()
    k_new, v_new, slots = gw.new_tokens()
    for flags in (kvq.DECODE_EARLY_INPUTS, kvq.DECODE_EARLY_INPUTS | kvq.DECODE_EARLY_CACHE):
        early = gw.params(flags=flags)
        for _ in range(3):
            out, lse = gw.step(q, k_new, v_new, slots, early, bufs)
            assert torch.equal(out, ref) and torch.equal(lse, ref_lse)
    assert kvq.kvq_get_device_error() == 0


@pytest.mark.parametrize("name,kw", [("gqa", dict(ctx=3000)), ("paged", dict(batch=5, max_ctx=700)),
                                     ("spec", dict(ctx=700, batch=2)), ("mixed", dict(batch=5, max_ctx=6000))])
def test_early_flags_back_to_back_steps_with_changing_inputs(lib, orc, name, kw):
    """Steps enqueued back to back with no host synchronisation (append,
    decode, combine, append, ...) under both early flags, each step appending
    other new-token rows at the same slots and decoding another query into its
    own output: every step gives bitwise what the same step gives alone with
    the default flags.  A decode that read an appended row before its append
    finished, or wrote the shared workspace while the previous combine still
    read it, would return another step's bits."""
    w = synth.make(name, **kw)
    gw = GpuWorkload(w, gen_device="cpu")
    gw.fill_history()
    k0, v0, slots = gw.new_tokens()
    kv = [(k0, v0), (torch.roll(k0, 1, dims=-1).contiguous(), (-v0).contiguous())]
    q0 = w.q("cpu").cuda()
    qs = [q0, (-q0).contiguous(), torch.flip(q0, dims=(-1,)).contiguous()]
    base, early = gw.params(), gw.params(flags=kvq.DECODE_EARLY_INPUTS | kvq.DECODE_EARLY_CACHE)
    bufs = gw.buffers(base)
    steps = [(i % 2, i % 3) for i in range(8)]
    ref = {}
    for key in sorted(set(steps)):
        k, v = kv[key[0]]
        kvq.kvq_append(gw.cache, k, v, slots)
        kvq.decode_step(gw.cache, base, qs[key[1]], gw.block_table, gw.seq_lens, bufs, gw.head_sink)
        torch.cuda.synchronize()
        ref[key] = (bufs.out.clone(), bufs.lse.clone())
    outs = [guarded(torch.empty_like(bufs.out)) for _ in steps]
    lses = [guarded(torch.empty_like(bufs.lse)) for _ in steps]
    torch.cuda.synchronize()
    for i, (a, b) in enumerate(steps):
        k, v = kv[a]
        kvq.kvq_append(gw.cache, k, v, slots)
        kvq.kvq_decode(gw.cache, early, qs[b], gw.block_table, gw.seq_lens, bufs.workspace)
        kvq.kvq_combine(gw.cache, early, bufs.workspace, gw.head_sink, outs[i], lses[i])
    torch.cuda.synchronize()
    assert kvq.kvq_get_device_error() == 0
    for i, key in enumerate(steps):
        assert torch.equal(outs[i], ref[key][0]) and torch.equal(lses[i], ref[key][1]), f"step {i} {key}"


def test_combine_of_a_row_with_many_pieces(lib, orc):
    """A ragged batch whose rows have few pieces on average (so kvq_combine
    folds each row with one warp) but one long sequence split over about 150
    CTAs: its rows fold their pieces 32 at a time, the last group partial.
    Against the oracle, with a head sink, and bitwise repeatable."""
    B, bs = 40, 256
    L = np.array([40000] + [16] * (B - 1), np.int32)
    nb_long = -(-40000 // bs)
    table = np.zeros((B, nb_long), np.int32)
    table[0] = np.arange(nb_long)
    table[1:, 0] = nb_long + np.arange(B - 1)
    w = synth.Workload("manypieces", kvq.INT8, kvq.PER_CHANNEL, kvq.PER_TENSOR, B, 8, 2, 128, 1, bs, L, table,
                       nb_long + B - 1, use_sink=True, k_channel_lognormal=0.5, seed=17)
    gw, params, bufs, q, _ = run_case(orc, w)
    ref, ref_lse = bufs.out.clone(), bufs.lse.clone()
    kvq.decode_step(gw.cache, params, q, gw.block_table, gw.seq_lens, bufs, gw.head_sink)
    torch.cuda.synchronize()
    assert torch.equal(bufs.out, ref) and torch.equal(bufs.lse, ref_lse)


def test_large_per_channel_k_scale_with_zero_codes_is_finite(lib, orc):
    """INT4 PR #32515: q * k_scale far beyond fp16 range with every K code
    zero must not become inf * 0 = NaN; the output is the mean of V."""
    D, L = 256, 100
    w = synth.Workload("huge", kvq.INT4, kvq.PER_CHANNEL, kvq.PER_CHANNEL, 1, 6, 1, D, 1, 32,
                       np.array([L], np.int32), np.arange(4, dtype=np.int32).reshape(1, 4), 4, seed=5)
    ks = torch.full((1, D), 3.0e38)
    gw = GpuWorkload(w, gen_device="cpu", k_static=ks, v_static=None)
    gw.fill_history()
    k_new, v_new, slots = gw.new_tokens()
    kvq.kvq_append(gw.cache, torch.zeros_like(k_new), v_new, slots)
    gw.cache.k_codes.zero_()
    params = gw.params()
    bufs = gw.buffers(params)
    q = (w.q("cpu") * 100).to("cuda")
    out, lse = kvq.decode_step(gw.cache, params, q, gw.block_table, gw.seq_lens, bufs)
    torch.cuda.synchronize()
    o = out.float().cpu().numpy()
    assert np.isfinite(o).all()
    vs = gw.v_static.cpu().numpy()[0]
    vc = gw.cache.v_codes.cpu().numpy()[:, 0].reshape(-1, D // 2)[:L]
    lo = (vc & 15).astype(np.int16)
    hi = (vc >> 4).astype(np.int16)
    codes = np.stack([np.where(lo > 7, lo - 16, lo), np.where(hi > 7, hi - 16, hi)], -1).reshape(L, D)
    mean = codes.mean(0) * vs
    assert np.allclose(o[0, 0, 0], mean, rtol=1e-2, atol=2e-2 * np.abs(mean).max())
    assert np.allclose(lse.cpu().numpy(), math.log(L), atol=1e-4)


def test_bad_block_id_and_seq_len_are_flagged_not_faulted(lib):
    w = synth.make("paged", batch=3, max_ctx=300)
    gw = GpuWorkload(w, gen_device="cpu")
    gw.fill_history()
    params = gw.params()
    bufs = gw.buffers(params)
    q = w.q("cpu").to("cuda")
    kvq.kvq_get_device_error(clear=True)
    bt = gw.block_table.clone()
    bt[1, 0] = w.num_blocks + 5
    bt[2, 0] = -3
    kvq.decode_step(gw.cache, params, q, bt, gw.seq_lens, bufs)
    assert kvq.kvq_get_device_error(clear=True) & kvq.DEVERR_BLOCK_ID
    sl = gw.seq_lens.clone()
    sl[0] = w.max_blocks * w.block_size + 1
    kvq.decode_step(gw.cache, params, q, gw.block_table, sl, bufs)
    assert kvq.kvq_get_device_error(clear=True) & kvq.DEVERR_SEQ_LEN
    # the context still works afterwards
    out, _ = kvq.decode_step(gw.cache, params, q, gw.block_table, gw.seq_lens, bufs)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()


WIDE = [
    # dtype, D, G, T, k_mode, v_mode, softcap, window, sink   (rows = G*T in 17..48)
    (kvq.INT8, 128, 3, 6, kvq.PER_ROW, kvq.PER_ROW, 0.0, 0, False),
    (kvq.FP8_E4M3, 256, 4, 7, kvq.PER_TENSOR, kvq.PER_TENSOR, 20.0, 0, False),
    (kvq.INT4, 256, 5, 7, kvq.PER_ROW, kvq.PER_ROW, 0.0, 0, True),
    (kvq.INT8, 256, 8, 5, kvq.PER_CHANNEL, kvq.PER_ROW, 0.0, 100, True),
    (kvq.INT4, 256, 6, 8, kvq.PER_CHANNEL, kvq.PER_CHANNEL, 0.0, 0, False),
    (kvq.FP8_E4M3, 128, 8, 6, kvq.PER_ROW, kvq.PER_TENSOR, 0.0, 37, True),
]


@pytest.mark.parametrize("case", WIDE, ids=lambda c: f"dt{c[0]}-D{c[1]}-rows{c[2] * c[3]}")
def test_many_query_rows_layout(lib, orc, case):
    """17..48 query rows per kv head (drafts x GQA group): the tensor-memory
    kernel by default (test_gpu_wide_layout.py runs the same cases on the
    mma.sync kernel's wide layout, in which four key quarters share each
    tile's row maxima and P)."""
    dt, D, G, T, km, vm, cap, W, sink = case
    Hkv, bs = 2, 32
    L = np.array([300, T - 2, 129, 64, 1], np.int32)
    mb = 10
    w = synth.Workload("wide", dt, km, vm, len(L), G * Hkv, Hkv, D, T, bs, L,
                       np.random.default_rng(G * T).permutation(len(L) * mb).astype(np.int32).reshape(len(L), mb),
                       len(L) * mb, softcap=cap, use_sink=sink, k_channel_lognormal=0.5, seed=G * 100 + T)
    run_case(orc, w)
    if W:
        run_case(orc, w, window=W, check_cache=False)


TC = [
    # dtype, D, G, T, k_mode, v_mode, softcap, window, sink, q_scale
    # (rows = G*T in 17..48 at D 256, 17..64 at D 128: the tensor-memory layout)
    (kvq.INT4, 256, 6, 8, kvq.PER_CHANNEL, kvq.PER_CHANNEL, 0.0, 0, False, 1.0),
    (kvq.INT4, 256, 4, 5, kvq.PER_ROW, kvq.PER_ROW, 0.0, 0, True, 6.0),
    (kvq.INT8, 256, 8, 6, kvq.PER_ROW, kvq.PER_ROW, 0.0, 0, False, 1.0),
    (kvq.FP8_E4M3, 256, 6, 6, kvq.PER_TENSOR, kvq.PER_ROW, 30.0, 0, False, 6.0),
    (kvq.INT8, 128, 8, 8, kvq.PER_CHANNEL, kvq.PER_TENSOR, 0.0, 200, True, 1.0),
    (kvq.FP8_E4M3, 128, 7, 7, kvq.PER_ROW, kvq.PER_TENSOR, 0.0, 0, True, 1.0),
    (kvq.INT4, 128, 5, 8, kvq.PER_ROW, kvq.PER_CHANNEL, 0.0, 0, False, 8.0),
    (kvq.INT8, 128, 3, 6, kvq.PER_ROW, kvq.PER_ROW, 0.0, 0, False, 1.0),
    (kvq.FP8_E4M3, 256, 8, 4, kvq.PER_CHANNEL, kvq.PER_CHANNEL, 0.0, 0, False, 1.0),
]


@pytest.mark.parametrize("case", TC, ids=lambda c: f"dt{c[0]}-D{c[1]}-rows{c[2] * c[3]}-km{c[4]}vm{c[5]}")
def test_tensor_memory_layout(lib, orc, case):
    """17..64 query rows per kv head on the tcgen05 path: every code type,
    scale mode and head size it takes, ragged lengths over several 128-key
    tiles and pieces, softcap / window / sink; q_scale > 1 sharpens the
    logits so that row maxima move by more than 2^8 between tiles (the lazy
    rescale of O and l).  Repeated decodes are bitwise identical."""
    dt, D, G, T, km, vm, cap, W, sink, qs = case
    Hkv, bs = 2, 32
    L = np.array([1500, T - 1, 129, 128, 1, 700], np.int32)
    mb = 48
    w = synth.Workload("tc", dt, km, vm, len(L), G * Hkv, Hkv, D, T, bs, L,
                       np.random.default_rng(G * T + D).permutation(len(L) * mb).astype(np.int32).reshape(len(L), mb),
                       len(L) * mb, softcap=cap, use_sink=sink, k_channel_lognormal=0.5, seed=G * 100 + T + D)
    gw, params, bufs, q, _ = run_case(orc, w, q_scale=qs)
    ref = bufs.out.clone()
    kvq.decode_step(gw.cache, params, q, gw.block_table, gw.seq_lens, bufs, gw.head_sink)
    assert torch.equal(bufs.out, ref)
    if W:
        run_case(orc, w, window=W, check_cache=False, q_scale=qs)


@pytest.mark.parametrize("G,T", [(4, 1), (8, 4)], ids=["mma-sync", "tensor-memory"])
def test_fp8_nan_bytes_past_the_sequence_end(lib, orc, G, T):
    """Every slot no append wrote holds the e4m3 NaN byte 0x7F, so the keys
    past each sequence's end inside its last page are NaN codes.  Their
    weights are zero; the result must still equal the oracle's (which never
    reads them) and be finite.  Both decode layouts: 4 rows per kv head (the
    mma.sync kernel) and 32 (the tensor-memory kernel)."""
    Hkv, D, bs = 2, 128, 16
    L = np.array([37, 300, 129, 8], np.int32)
    mb = math.ceil(int(L.max()) / bs)
    table = np.random.default_rng(7).permutation(len(L) * mb).astype(np.int32).reshape(len(L), mb)
    w = synth.Workload("nan", kvq.FP8_E4M3, kvq.PER_TENSOR, kvq.PER_TENSOR, len(L), G * Hkv, Hkv, D, T, bs, L,
                       table, len(L) * mb, seed=11)
    gw = GpuWorkload(w, gen_device="cpu")
    gw.cache.k_codes.fill_(0x7F)
    gw.cache.v_codes.fill_(0x7F)
    gw.fill_history()
    k_new, v_new, slots = gw.new_tokens()
    params = gw.params()
    bufs = gw.buffers(params)
    q = w.q("cpu").to("cuda")
    out, lse = gw.step(q, k_new, v_new, slots, params, bufs)
    torch.cuda.synchronize()
    assert kvq.kvq_get_device_error(clear=True) == 0
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    side = OracleSide(orc, w, range(w.batch), "cpu", gw.k_static, gw.v_static)
    ref, ref_lse = side.attend(q, window=0, sink=gw.head_sink)
    check_rows(got, ref)
    check_lse(lse.cpu().numpy().astype(np.float64), ref_lse)


def test_bounded_wait_runs_out_and_leaves_the_context_usable(lib, orc):
    """Failure detection without a fault: a wait on a barrier nothing arrives
    on (the pipelines' bounded wait, here limited to 20 ms) gives up, the
    host reads KVQ_DEVERR_TIMEOUT, and a decode afterwards is correct."""
    import time
    kvq.kvq_get_device_error(clear=True)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    kvq.kvq_check_wait_timeout(20000)
    flags = kvq.kvq_get_device_error(clear=True)
    elapsed = time.perf_counter() - t0
    assert flags & kvq.DEVERR_TIMEOUT
    assert 0.02 <= elapsed < 1.0, elapsed
    assert kvq.kvq_get_device_error(clear=True) == 0
    run_case(orc, synth.make("tiny"))
