"""kvq_prefill on the query-tile kernel (the query rows of a chunk -- tokens x
GQA group, up to 128 per kv head -- as the MMA's M dimension; head_dim 128 or
256, no group-wise scales) against oracle attention with the same chunk: every
code type and scale mode, chunks of 24 to 512 tokens, ragged lengths, window,
softcap and head sink.  The same calls with KVQ_DECODE_NO_TCGEN05 (virtual
decode sequences on the mma.sync kernel) are checked against the oracle too.
Within 2e-3 relative L2 (8e-3 for any row); LSE within 2e-3; repeated calls
bitwise identical."""
import math

import numpy as np
import pytest
import torch

from decode_attention_quantized_gb300 import kvq, synth
from decode_attention_quantized_gb300.workload import GpuWorkload

from guard import guarded
from parity import OracleSide, check_lse, check_rows

pytestmark = pytest.mark.gpu

DT = {"int8": kvq.INT8, "fp8": kvq.FP8_E4M3, "int4": kvq.INT4}
HKV = 2

# dt, K mode, V mode, head_dim, group, chunk C, lengths (all >= C), window, softcap, sink
CASES = [
    ("int4", kvq.PER_CHANNEL, kvq.PER_CHANNEL, 256, 6, 64, (700, 64, 1500), 0, 0.0, False),  # 16 tokens x 6
    ("int8", kvq.PER_TENSOR, kvq.PER_ROW, 256, 8, 32, (300, 45, 999), 0, 0.0, False),        # 16 x 8 = 128 rows
    ("fp8", kvq.PER_ROW, kvq.PER_TENSOR, 256, 4, 128, (129, 1000, 2500), 0, 0.0, True),      # 32 x 4, sink
    ("int8", kvq.PER_CHANNEL, kvq.PER_TENSOR, 256, 2, 512, (512, 1800), 0, 0.0, False),      # 64 x 2, 8 tiles a sequence
    ("int8", kvq.PER_ROW, kvq.PER_ROW, 256, 8, 24, (400, 3000), 700, 30.0, True),            # 12 x 8, window, softcap
    ("fp8", kvq.PER_ROW, kvq.PER_ROW, 256, 1, 100, (100, 300), 0, 0.0, False),               # 100 tokens x 1
    ("int4", kvq.PER_ROW, kvq.PER_ROW, 256, 4, 48, (1000, 48), 64, 0.0, False),              # 24 x 4 (a padded warp), window 64
    ("int8", kvq.PER_TENSOR, kvq.PER_ROW, 128, 8, 32, (300, 45, 999), 0, 0.0, False),        # head_dim 128: 16 x 8
    ("fp8", kvq.PER_TENSOR, kvq.PER_TENSOR, 128, 4, 64, (70, 2000, 640), 0, 50.0, True),     # 32 x 4, softcap, sink
    ("int4", kvq.PER_CHANNEL, kvq.PER_ROW, 128, 2, 512, (512, 1300), 0, 0.0, False),         # 64 x 2
    ("int8", kvq.PER_ROW, kvq.PER_ROW, 128, 1, 100, (100, 300), 37, 0.0, False),             # 100 x 1, window 37
    ("int8", kvq.PER_ROW, kvq.PER_ROW, 128, 4, 64, (40000, 64), 0, 0.0, True),               # rows of > 32 pieces
]


@pytest.fixture(scope="module")
def lib():
    from decode_attention_quantized_gb300 import build
    build.build()
    return kvq.load()


def workload(dt, km, vm, D, G, lens, softcap, sink, seed, bs=16):
    L = np.array(lens, np.int32)
    mb = max(1, math.ceil(int(L.max()) / bs))
    table = np.random.default_rng(seed).permutation(len(L) * mb).astype(np.int32).reshape(len(L), mb)
    return synth.Workload("qtile", DT[dt], km, vm, len(L), G * HKV, HKV, D, 1, bs, L, table, len(L) * mb,
                          softcap=softcap, use_sink=sink, k_channel_lognormal=0.5, seed=seed)


def prefill(gw, w, q, C, *, window, flags):
    params = kvq.make_params(w.batch, w.num_q_heads, C, w.max_blocks, window=window, softcap=w.softcap, flags=flags)
    ws = guarded(torch.empty((kvq.kvq_prefill_workspace_size(gw.cache, params) + 3) // 4, dtype=torch.int32,
                             device="cuda"))
    out = guarded(torch.empty((w.batch, C, w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device="cuda"))
    lse = guarded(torch.empty((w.batch, C, w.num_q_heads), dtype=torch.float32, device="cuda"))
    args = (gw.cache, params, q, gw.block_table, gw.seq_lens, gw.head_sink, out, lse, ws)
    kvq.kvq_prefill(*args)
    torch.cuda.synchronize()
    assert kvq.kvq_get_device_error(clear=True) == 0
    first = out.clone()
    kvq.kvq_prefill(*args)
    torch.cuda.synchronize()
    assert torch.equal(first.view(torch.int16), out.view(torch.int16)), "repeated prefill differs"
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-km{c[1]}-vm{c[2]}-D{c[3]}-G{c[4]}-C{c[5]}")
def test_query_tile_prefill_matches_oracle(lib, orc, case):
    dt, km, vm, D, G, C, lens, window, softcap, sink = case
    w = workload(dt, km, vm, D, G, lens, softcap, sink, seed=G * 1000 + C)
    gw = GpuWorkload(w, gen_device="cpu")
    gw.fill_history()
    k_new, v_new, slots = gw.new_tokens()
    kvq.kvq_append(gw.cache, k_new, v_new, slots)
    q = synth.randn_bf16((w.batch, C, w.num_q_heads, D), "cpu", "qtile", w.seed, "q")
    side = OracleSide(orc, w, range(w.batch), "cpu", gw.k_static, gw.v_static)
    bits = q.contiguous().view(torch.int16).numpy().view(np.uint16)
    ref, ref_lse = side.cache.attend(bits, side.table, side.lens, q_tokens=C, window=window, softcap=softcap,
                                     head_sink=None if gw.head_sink is None else gw.head_sink.cpu().numpy())
    for flags in (0, kvq.DECODE_NO_TCGEN05):
        got, lse = prefill(gw, w, q.cuda(), C, window=window, flags=flags)
        check_rows(got.reshape(-1, D), ref.reshape(-1, D))
        check_lse(lse, ref_lse)


def test_query_tile_prefill_with_narrow_windows(lib, orc):
    """Windows of 1 and 5 keys (each row sees at most its own few keys, so
    nearly every key of a 64-key tile is masked for every row), and a sequence
    whose chunk starts at position 0 (its length equals the chunk)."""
    w = workload("int8", kvq.PER_ROW, kvq.PER_ROW, 256, 4, (32, 77), 0.0, False, seed=5)
    gw = GpuWorkload(w, gen_device="cpu")
    gw.fill_history()
    k_new, v_new, slots = gw.new_tokens()
    kvq.kvq_append(gw.cache, k_new, v_new, slots)
    C = 32
    q = synth.randn_bf16((w.batch, C, w.num_q_heads, 256), "cpu", "qtile-edge", 0, "q")
    side = OracleSide(orc, w, range(w.batch), "cpu", gw.k_static, gw.v_static)
    bits = q.contiguous().view(torch.int16).numpy().view(np.uint16)
    for window in (1, 5):
        ref, ref_lse = side.cache.attend(bits, side.table, side.lens, q_tokens=C, window=window)
        got, lse = prefill(gw, w, q.cuda(), C, window=window, flags=0)
        check_rows(got.reshape(-1, 256), ref.reshape(-1, 256))
        check_lse(lse, ref_lse)
