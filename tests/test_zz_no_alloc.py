"""kvq_attend_noalloc: the entry point for callers that cannot allocate device
memory (a plugin inside a runtime that owns all device memory, or a loop that
must not pay cudaMalloc's implicit synchronization).  Its scratch is the
library's own fixed device array; its output must equal, bit for bit, the
regular kvq_decode + kvq_combine path with a caller workspace.

Kept in its own file, collected last, so that a run stopping at the first
failure has already run every other test; it also passes on its own in a
fresh process."""
import pytest
import torch

from decode_attention_quantized_gb300 import kvq, synth
from decode_attention_quantized_gb300.workload import GpuWorkload

from guard import guarded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from decode_attention_quantized_gb300 import build
    build.build()
    return kvq.load()


def regular_and_noalloc(w, window):
    gw = GpuWorkload(w, gen_device="cpu")
    gw.fill_history()
    k_new, v_new, slots = gw.new_tokens()
    kvq.kvq_append(gw.cache, k_new, v_new, slots)
    params = gw.params(window=window)
    q = w.q("cpu", 1).to("cuda")
    bufs = gw.buffers(params)
    kvq.decode_step(gw.cache, params, q, gw.block_table, gw.seq_lens, bufs, gw.head_sink)
    out = guarded(torch.full_like(bufs.out, float("nan")))
    lse = guarded(torch.full_like(bufs.lse, float("nan")))
    kvq.kvq_attend_noalloc(gw.cache, params, q, gw.block_table, gw.seq_lens, gw.head_sink, out, lse)
    torch.cuda.synchronize()
    assert kvq.kvq_get_device_error() == 0
    return bufs.out, bufs.lse, out, lse


def test_noalloc_matches_workspace_path_twice_in_a_row(lib):
    # two different shapes back to back: the second call reuses the scratch
    # that still holds the first call's partials
    cases = [(synth.make("gqa", ctx=5000), 0), (synth.make("mixed", batch=7, max_ctx=9000), 4096)]
    # the same kernels with the same split plan on the same inputs: bitwise
    # the workspace path's output and LSE (the merge order is fixed)
    for w, window in cases:
        ref, ref_lse, got, got_lse = regular_and_noalloc(w, window)
        assert torch.isfinite(got.float()).all()
        assert torch.equal(got, ref)
        assert torch.equal(got_lse, ref_lse)


def test_noalloc_rejects_shapes_beyond_its_scratch(lib):
    # 1024 sequences x 64 query rows x D=256 partials need far more than 16 MiB
    cache = kvq.QuantizedPagedCache(kvq.INT8, kvq.PER_ROW, kvq.PER_ROW, 64, 16, 1, 256)
    params = kvq.make_params(1024, 8, 8, 4)
    assert kvq.kvq_decode_workspace_size(cache, params) > 16 << 20
    q = torch.zeros((1024, 8, 8, 256), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((1024, 4), dtype=torch.int32, device="cuda")
    sl = torch.zeros((1024,), dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_attend_noalloc(cache, params, q, bt, sl, None, out, None)
    assert e.value.status == 3
