"""The algorithmic byte counts the bench's roofline figures divide by
(synth.step_bytes / decode_bytes), checked against the cache layout written
out by hand for small cases: codes of every key a query row sees, per-row or
per-group scales, q, the block-table entries of the pages read, seq_lens."""
import dataclasses

import numpy as np

from decode_attention_quantized_gb300 import synth


def small(dtype, km, vm, D=128, L=(100, 37), bs=16, T=1, group_size=0):
    L = np.array(L, np.int32)
    mb = int(np.ceil(L.max() / bs))
    table = np.arange(len(L) * mb, dtype=np.int32).reshape(len(L), mb)
    return synth.Workload("bytes", dtype, km, vm, len(L), 8, 2, D, T, bs, L, table, len(L) * mb,
                          group_size=group_size)


def test_per_row_int8_bytes_by_hand():
    w = small(synth.INT8, synth.PER_ROW, synth.PER_ROW)
    keys = 100 + 37
    kv = keys * 2 * (2 * 128 + 4 + 4)                  # K and V codes + one fp32 scale per side
    pages = int(np.ceil(100 / 16)) + int(np.ceil(37 / 16))
    q = 2 * 1 * 8 * 128 * 2
    s = synth.step_bytes(w)
    assert s["kv"] == kv and s["q"] == q and s["table"] == 4 * pages + 4 * 2
    assert synth.decode_bytes(w) == kv + q + 4 * pages + 4 * 2


def test_per_group_int4_counts_one_scale_per_group():
    for g in (32, 64, 128):
        w = small(synth.INT4, synth.PER_GROUP, synth.PER_GROUP, group_size=g)
        keys = 100 + 37
        assert synth.step_bytes(w)["kv"] == keys * 2 * (2 * 64 + 2 * 4 * (128 // g))


def test_static_scales_add_no_bytes_and_window_counts_only_visible_keys():
    w = small(synth.FP8_E4M3, synth.PER_TENSOR, synth.PER_CHANNEL)
    assert synth.step_bytes(w)["kv"] == (100 + 37) * 2 * 2 * 128
    # window 20: sequence 0 sees keys 80..99, sequence 1 keys 17..36
    assert synth.step_bytes(w, window=20)["kv"] == (20 + 20) * 2 * 2 * 128
    wg = dataclasses.replace(w, k_mode=synth.PER_GROUP, group_size=64)
    assert synth.step_bytes(wg)["kv"] == (100 + 37) * 2 * (2 * 128 + 4 * 2)
