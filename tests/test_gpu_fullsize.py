"""The named workloads at their full sizes, in the launch configuration
bench.py times, checked on sampled output rows that the oracle computes one
by one (and the sampled sequences' cache bytes, bit for bit)."""
import numpy as np
import pytest
import torch

from decode_attention_quantized_gb300 import kvq, synth
from decode_attention_quantized_gb300.workload import GpuWorkload

from parity import OracleSide, check_lse, check_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from decode_attention_quantized_gb300 import build
    build.build()
    return kvq.load()


def sample_seqs(w, k=3):
    L = w.seq_lens
    picks = {int(np.argmax(L)), int(np.argmin(L))}
    rng = np.random.default_rng(0)
    while len(picks) < min(k, w.batch):
        picks.add(int(rng.integers(w.batch)))
    return sorted(picks)


def run_full(orc, w, windows=(0,), seqs=None):
    gw = GpuWorkload(w, gen_device="cuda")
    gw.fill_history()
    k_new, v_new, slots = gw.new_tokens()
    seqs = sample_seqs(w) if seqs is None else seqs
    side = OracleSide(orc, w, seqs, "cuda", gw.k_static, gw.v_static)
    for call, W in enumerate(windows):
        params = gw.params(window=W)
        bufs = gw.buffers(params)
        q = w.q("cuda", call)
        out, lse = gw.step(q, k_new, v_new, slots, params, bufs)
        torch.cuda.synchronize()
        assert kvq.kvq_get_device_error(clear=True) == 0
        if call == 0:
            side.compare_cache(gw)
        ref, ref_lse = side.attend(q, window=W, sink=gw.head_sink)
        got = out.float().cpu().numpy().astype(np.float64)[seqs]
        check_rows(got, ref)
        check_lse(lse.cpu().numpy().astype(np.float64)[seqs], ref_lse)


@pytest.mark.parametrize("ctx", [1024, 16384, 262144])
def test_gqa_int8_per_row_context_sweep(lib, orc, ctx):
    run_full(orc, synth.make("gqa", ctx=ctx), seqs=[0])


def test_paged_fp8_ragged_softcap(lib, orc):
    run_full(orc, synth.make("paged"))


def test_spec_int4_per_channel_eight_queries(lib, orc):
    run_full(orc, synth.make("spec"), seqs=[0, 3])


def test_mixed_sink_and_alternating_window(lib, orc):
    w = synth.make("mixed")
    run_full(orc, w, windows=(w.window_for_call(0), w.window_for_call(1)))


@pytest.mark.parametrize("name", ["gqa", "paged"])
def test_group_scales_at_full_size(lib, orc, name):
    """The workloads with group-wise scales on both sides (64-channel groups),
    as bench.py's group_scales measurement runs them."""
    import dataclasses
    base = synth.make("gqa", ctx=262144) if name == "gqa" else synth.make(name)
    w = dataclasses.replace(base, k_mode=kvq.PER_GROUP, v_mode=kvq.PER_GROUP, group_size=64)
    run_full(orc, w, seqs=[0] if name == "gqa" else None)
