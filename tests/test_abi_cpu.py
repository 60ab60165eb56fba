"""The C-ABI library on the host: it builds, loads, exports every symbol
include/kvq.h declares, and rejects invalid arguments before any CUDA call.
No compute call runs here (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kvq():
    from decode_attention_quantized_gb300 import build, kvq
    build.build()
    kvq.load()
    return kvq


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "kvq.h")).read()
    return sorted(set(re.findall(r"KVQ_API\s+[\w\s\*]*?\b(kvq_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    syms = declared_symbols()
    for name in ("kvq_append", "kvq_decode", "kvq_combine", "kvq_decode_workspace_size",
                 "kvq_get_device_error", "kvq_status_string"):
        assert name in syms


def test_library_exports_every_declared_symbol(kvq):
    lib = kvq.load()
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert name in kvq.SIGNATURES, f"binding lacks {name}"
    # and nothing beyond the ABI is exported as a kvq_ symbol
    out = os.popen(f"nm -D --defined-only {kvq.LIB_PATH}").read()
    exported = set(re.findall(r"\b(kvq_\w+)\b", out))
    assert exported == set(declared_symbols())


def test_status_strings(kvq):
    lib = kvq.load()
    assert lib.kvq_status_string(0) == b"ok"
    assert lib.kvq_status_string(3) == b"workspace too small"
    assert lib.kvq_status_string(99) == b"unknown status"


FAKE = 0x7F0000000000  # an aligned address that is never dereferenced on the host


def good_cache(kvq, **kw):
    d = dict(dtype=1, k_mode=1, v_mode=1, num_blocks=8, block_size=16, num_kv_heads=2, head_dim=128,
             k_codes=FAKE, v_codes=FAKE + 4096, k_scale=FAKE + 8192, v_scale=FAKE + 16384)
    d.update(kw)
    return kvq.CacheDesc(**d)


def good_params(kvq, **kw):
    d = dict(batch=2, num_q_heads=8, q_tokens=1, max_blocks_per_seq=4, max_seq_len=0, sm_scale=0.0,
             softcap=0.0, window=0)
    d.update(kw)
    return kvq.DecodeParams(**d)


@pytest.mark.parametrize("bad,status", [
    (dict(dtype=0), 1), (dict(dtype=4), 1), (dict(k_mode=0), 1), (dict(v_mode=7), 1),
    (dict(num_blocks=0), 1), (dict(block_size=24), 1), (dict(block_size=8), 1), (dict(num_kv_heads=0), 1),
    (dict(head_dim=96), 2), (dict(head_dim=32), 2), (dict(head_dim=-64), 1),
    (dict(k_codes=None), 1), (dict(v_scale=None), 1), (dict(k_codes=FAKE + 8), 1),
    (dict(k_scale=FAKE + 4), 1),
])
def test_append_rejects_bad_cache(kvq, bad, status):
    lib = kvq.load()
    c = good_cache(kvq, **bad)
    st = lib.kvq_append(ctypes.byref(c), FAKE, FAKE, FAKE, 4, None)
    assert st == status


def test_append_rejects_bad_tokens(kvq):
    lib = kvq.load()
    c = good_cache(kvq)
    assert lib.kvq_append(ctypes.byref(c), FAKE, FAKE, FAKE, -1, None) == 1
    assert lib.kvq_append(ctypes.byref(c), FAKE, FAKE, FAKE, 0, None) == 0       # no-op, no launch
    assert lib.kvq_append(ctypes.byref(c), None, FAKE, FAKE, 3, None) == 1
    assert lib.kvq_append(ctypes.byref(c), FAKE + 2, FAKE, FAKE, 3, None) == 1   # misaligned bf16 rows
    assert lib.kvq_append(None, FAKE, FAKE, FAKE, 3, None) == 1


@pytest.mark.parametrize("bad,status", [
    (dict(batch=-1), 1), (dict(num_q_heads=7), 1), (dict(num_q_heads=18), 2), (dict(q_tokens=0), 1),
    (dict(q_tokens=9), 2), (dict(max_blocks_per_seq=0), 1), (dict(max_seq_len=-5), 1), (dict(window=-1), 1),
    (dict(softcap=-1.0), 1), (dict(softcap=float("inf")), 1), (dict(sm_scale=float("nan")), 1),
    (dict(batch=1025), 2), (dict(flags=8), 1), (dict(flags=0x80000001), 1),
])
def test_decode_rejects_bad_params(kvq, bad, status):
    lib = kvq.load()
    c = good_cache(kvq)
    p = good_params(kvq, **bad)
    n = ctypes.c_size_t(0)
    assert lib.kvq_decode_workspace_size(ctypes.byref(c), ctypes.byref(p), ctypes.byref(n)) == status
    assert lib.kvq_decode(ctypes.byref(c), ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, 1 << 30, None) == status
    assert lib.kvq_combine(ctypes.byref(c), ctypes.byref(p), FAKE, 1 << 30, None, FAKE, None, None) == status


def test_decode_rejects_null_and_misaligned(kvq):
    lib = kvq.load()
    c = good_cache(kvq)
    p = good_params(kvq)
    assert lib.kvq_decode(ctypes.byref(c), ctypes.byref(p), None, FAKE, FAKE, FAKE, 1 << 30, None) == 1
    assert lib.kvq_decode(ctypes.byref(c), ctypes.byref(p), FAKE, FAKE, FAKE, FAKE + 16, 1 << 30, None) == 1
    assert lib.kvq_combine(ctypes.byref(c), ctypes.byref(p), FAKE, 1 << 30, None, None, None, None) == 1
    assert lib.kvq_combine(ctypes.byref(c), ctypes.byref(p), FAKE, 1 << 30, FAKE + 2, FAKE, None, None) == 1
    # an empty batch is a valid no-op
    p0 = good_params(kvq, batch=0)
    assert lib.kvq_decode(ctypes.byref(c), ctypes.byref(p0), None, None, None, None, 0, None) == 0
    assert lib.kvq_combine(ctypes.byref(c), ctypes.byref(p0), None, 0, None, None, None, None) == 0
    assert lib.kvq_get_device_error(None, 0, None) == 1


def test_binding_refuses_to_run_without_the_library(tmp_path):
    from decode_attention_quantized_gb300 import kvq
    saved = kvq._lib
    kvq._lib = None
    try:
        with pytest.raises(RuntimeError, match="build the CUDA library"):
            kvq.load(str(tmp_path / "missing.so"))
    finally:
        kvq._lib = saved


def good_norm_rope(kvq, **kw):
    d = dict(norm_weight=FAKE, norm_eps=1e-6, rotary_dim=64, rotary_offset=0, rotary_interleaved=0,
             cos_cache=FAKE + 4096, sin_cache=FAKE + 8192, max_position=128, hadamard=0)
    d.update(kw)
    return kvq.NormRopeDesc(**d)


@pytest.mark.parametrize("bad", [
    dict(rotary_dim=-2), dict(rotary_dim=63), dict(rotary_offset=-1), dict(rotary_offset=96),
    dict(rotary_dim=130), dict(cos_cache=None), dict(sin_cache=None), dict(max_position=0),
    dict(norm_weight=FAKE + 2), dict(cos_cache=FAKE + 2), dict(norm_eps=float("nan")), dict(hadamard=2),
])
def test_norm_rope_rejects_bad_prologue(kvq, bad):
    """Invalid prologues are refused on the host, for the Q-side call and the
    fused append alike (head_dim 128: offset + rotary_dim must fit)."""
    lib = kvq.load()
    p = good_norm_rope(kvq, **bad)
    assert lib.kvq_norm_rope_apply(ctypes.byref(p), FAKE, FAKE, FAKE, 4, 8, 128, None) == 1
    c = good_cache(kvq)
    assert lib.kvq_append_norm_rope(ctypes.byref(c), ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, 4, None) == 1


def test_norm_rope_rejects_bad_shapes_and_pointers(kvq):
    lib = kvq.load()
    p = good_norm_rope(kvq)
    assert lib.kvq_norm_rope_apply(ctypes.byref(p), FAKE, FAKE, FAKE, 4, 8, 96, None) == 2  # head_dim
    assert lib.kvq_norm_rope_apply(ctypes.byref(p), FAKE, FAKE, FAKE, -1, 8, 128, None) == 1
    assert lib.kvq_norm_rope_apply(ctypes.byref(p), FAKE, FAKE, FAKE, 4, 0, 128, None) == 1
    assert lib.kvq_norm_rope_apply(ctypes.byref(p), FAKE, FAKE, None, 4, 8, 128, None) == 1  # positions
    assert lib.kvq_norm_rope_apply(ctypes.byref(p), FAKE + 8, FAKE, FAKE, 4, 8, 128, None) == 1  # x alignment
    assert lib.kvq_norm_rope_apply(None, FAKE, FAKE, FAKE, 4, 8, 128, None) == 1
    # nothing to do: no device call is made
    assert lib.kvq_norm_rope_apply(ctypes.byref(p), FAKE, FAKE, FAKE, 0, 8, 128, None) == 0
    # RMSNorm alone needs neither tables nor positions
    q = good_norm_rope(kvq, rotary_dim=0, cos_cache=None, sin_cache=None, max_position=0)
    assert lib.kvq_norm_rope_apply(ctypes.byref(q), FAKE, FAKE, None, 0, 8, 128, None) == 0
    c = good_cache(kvq)
    assert lib.kvq_append_norm_rope(ctypes.byref(c), None, FAKE, FAKE, FAKE, FAKE, 4, None) == 1
    assert lib.kvq_append_norm_rope(ctypes.byref(c), ctypes.byref(p), FAKE, FAKE, FAKE, None, 4, None) == 1
    assert lib.kvq_append_norm_rope(ctypes.byref(c), ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, 0, None) == 0


def test_prefill_rejects_bad_arguments_on_the_host(kvq):
    lib = kvq.load()
    c = good_cache(kvq)
    n = ctypes.c_size_t(0)
    # a chunk of 0 tokens
    p = good_params(kvq, q_tokens=0)
    assert lib.kvq_prefill_workspace_size(ctypes.byref(c), ctypes.byref(p), ctypes.byref(n)) == 1
    assert lib.kvq_prefill(ctypes.byref(c), ctypes.byref(p), FAKE, FAKE, FAKE, None, FAKE, None, FAKE, 1 << 30,
                           None) == 1
    # 200 sequences x 64 tokens = 1600 virtual sequences of 8 on the decode
    # kernels: beyond the plan's 1024
    p = good_params(kvq, batch=200, q_tokens=64, flags=kvq.DECODE_NO_TCGEN05)
    assert lib.kvq_prefill_workspace_size(ctypes.byref(c), ctypes.byref(p), ctypes.byref(n)) == 2
    # on the query-tile kernel (head_dim 256, 4 query heads per kv head:
    # 32-token tiles of 128 rows) 600 x 64 tokens are 1200 virtual sequences:
    # beyond it as well
    c256 = good_cache(kvq, head_dim=256)
    p = good_params(kvq, batch=600, q_tokens=64)
    assert lib.kvq_prefill_workspace_size(ctypes.byref(c256), ctypes.byref(p), ctypes.byref(n)) == 2
    # missing or misaligned pointers
    p = good_params(kvq, q_tokens=12)
    for args in [(None, FAKE, FAKE, None, FAKE), (FAKE, FAKE, None, None, FAKE), (FAKE, FAKE, FAKE, None, None),
                 (FAKE + 8, FAKE, FAKE, None, FAKE), (FAKE, FAKE, FAKE, FAKE + 2, FAKE)]:
        q, bt, sl, hs, out = args
        assert lib.kvq_prefill(ctypes.byref(c), ctypes.byref(p), q, bt, sl, hs, out, None, FAKE, 1 << 30,
                               None) == 1
    # an empty batch is a no-op
    p = good_params(kvq, batch=0, q_tokens=12)
    assert lib.kvq_prefill(ctypes.byref(c), ctypes.byref(p), None, None, None, None, None, None, None, 0,
                           None) == 0


@pytest.mark.parametrize("bad", [dict(layout=2), dict(layout=-1), dict(layout=1, v_head_size=12),
                                 dict(layout=1, v_head_size=136), dict(layout=0, v_head_size=64),
                                 dict(layout=1, k_codes=None)])
def test_latent_layout_validation(kvq, bad):
    lib = kvq.load()
    c = good_cache(kvq, **bad)
    assert lib.kvq_append(ctypes.byref(c), FAKE, FAKE, FAKE, 4, None) == 1


def test_latent_cache_needs_no_v_arrays(kvq):
    lib = kvq.load()
    c = good_cache(kvq, layout=1, v_head_size=64, v_codes=None, v_scale=None, v_mode=0)
    # valid: nothing to append, and V arguments may be NULL
    assert lib.kvq_append(ctypes.byref(c), FAKE, None, FAKE, 0, None) == 0


@pytest.mark.parametrize("bad", [dict(k_mode=4, group_size=0), dict(v_mode=4, group_size=16),
                                 dict(k_mode=4, group_size=48), dict(k_mode=4, v_mode=4, group_size=256),
                                 dict(head_dim=64, k_mode=4, group_size=128), dict(k_mode=5, group_size=32),
                                 dict(k_mode=4, group_size=32, k_scale=FAKE + 8)])
def test_group_scale_validation(kvq, bad):
    """PER_GROUP: group_size 32, 64 or 128, at most head_dim; per-group scale
    arrays 16-byte aligned (the pipeline moves them with bulk copies)."""
    lib = kvq.load()
    c = good_cache(kvq, **bad)
    assert lib.kvq_append(ctypes.byref(c), FAKE, FAKE, FAKE, 4, None) == 1


def test_group_size_is_ignored_without_a_group_side(kvq):
    lib = kvq.load()
    c = good_cache(kvq, group_size=48)  # PER_ROW on both sides: no group size is read
    assert lib.kvq_append(ctypes.byref(c), FAKE, FAKE, FAKE, 0, None) == 0
    for g in (32, 64, 128):
        c = good_cache(kvq, k_mode=4, v_mode=4, group_size=g)
        assert lib.kvq_append(ctypes.byref(c), FAKE, FAKE, FAKE, 0, None) == 0


def test_wait_check_rejects_bad_limits_on_the_host(kvq):
    lib = kvq.load()
    assert lib.kvq_check_wait_timeout(0, None) == 1
    assert lib.kvq_check_wait_timeout(2000001, None) == 1


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=576), 2),                                                   # SEPARATE at 576
    (dict(head_dim=576, layout=1, v_head_size=512, dtype=3), 2),               # int4 codes
    (dict(head_dim=576, layout=1, v_head_size=512, k_mode=4, v_mode=4, group_size=64), 2),
    (dict(head_dim=576, layout=1, v_head_size=520), 0),
    (dict(head_dim=576, layout=1, v_head_size=512, dtype=2), 0),
    (dict(head_dim=576, layout=1, v_head_size=0, k_mode=3, v_mode=3), 0),
])
def test_head_dim_576_only_for_a_latent_cache_of_8_bit_codes(kvq, kw, status):
    """Absorbed MLA's 576 = 512 latent + 64 rotary channels: a LATENT cache with
    int8 or e4m3 codes and per-row or static scales."""
    lib = kvq.load()
    c = good_cache(kvq, **kw)
    assert lib.kvq_append(ctypes.byref(c), FAKE, FAKE, FAKE, 0, None) == status


def test_hadamard_needs_a_power_of_two_head_dim(kvq):
    lib = kvq.load()
    p = good_norm_rope(kvq, rotary_dim=0, cos_cache=None, sin_cache=None, max_position=0, hadamard=1)
    assert lib.kvq_norm_rope_apply(ctypes.byref(p), FAKE, FAKE, None, 4, 2, 576, None) == 2
    p = good_norm_rope(kvq, rotary_dim=64, rotary_offset=512)
    assert lib.kvq_norm_rope_apply(ctypes.byref(p), FAKE, FAKE, FAKE, 0, 2, 576, None) == 0
