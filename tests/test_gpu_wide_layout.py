"""The mma.sync kernel's wide layout (17..48 query rows per kv head: four key
quarters share each tile's row maxima and P), which the tensor-memory kernel
replaces for those shapes by default; kvq_decode_params.flags =
KVQ_DECODE_NO_TCGEN05 keeps them on it.  The same cases as
test_gpu_decode.py's many-row test, against the oracle."""
import numpy as np
import pytest

from decode_attention_quantized_gb300 import kvq, synth

from test_gpu_decode import WIDE, run_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from decode_attention_quantized_gb300 import build
    build.build()
    return kvq.load()


@pytest.mark.parametrize("case", WIDE, ids=lambda c: f"dt{c[0]}-D{c[1]}-rows{c[2] * c[3]}")
def test_wide_layout_with_the_tensor_memory_kernel_off(lib, orc, case):
    dt, D, G, T, km, vm, cap, W, sink = case
    L = np.array([300, T - 2, 129, 64, 1], np.int32)
    mb = 10
    w = synth.Workload("wide", dt, km, vm, len(L), G * 2, 2, D, T, 32, L,
                       np.random.default_rng(G * T).permutation(len(L) * mb).astype(np.int32).reshape(len(L), mb),
                       len(L) * mb, softcap=cap, use_sink=sink, k_channel_lognormal=0.5, seed=G * 100 + T)
    run_case(orc, w, flags=kvq.DECODE_NO_TCGEN05)
    if W:
        run_case(orc, w, window=W, check_cache=False, flags=kvq.DECODE_NO_TCGEN05)
