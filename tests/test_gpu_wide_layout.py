"""The mma.sync kernel's wide layout (17..48 query rows per kv head: four key
quarters share each tile's row maxima and P), which the tensor-memory kernel
replaces for those shapes by default; KVQ_NO_TC=1 in the environment keeps
them on it.  Each case runs in a child process started with that setting (the
launch plan is chosen once per process), against the oracle as in
test_gpu_decode.py."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

CHILD = r'''
import sys
import numpy as np
sys.path.insert(0, {root!r})
sys.path.insert(0, {here!r})
from decode_attention_quantized_gb300 import build, kvq, synth
from oracle import oracle as orc
import test_gpu_decode as t
build.build()
kvq.load()
orc.build()
case = t.WIDE[{i}]
dt, D, G, T, km, vm, cap, W, sink = case
L = np.array([300, T - 2, 129, 64, 1], np.int32)
mb = 10
w = synth.Workload("wide", dt, km, vm, len(L), G * 2, 2, D, T, 32, L,
                   np.random.default_rng(G * T).permutation(len(L) * mb).astype(np.int32).reshape(len(L), mb),
                   len(L) * mb, softcap=cap, use_sink=sink, k_channel_lognormal=0.5, seed=G * 100 + T)
t.run_case(orc, w)
if W:
    t.run_case(orc, w, window=W, check_cache=False)
print("wide case ok")
'''


def cases():
    sys.path.insert(0, HERE)
    import test_gpu_decode as t
    return list(range(len(t.WIDE)))


@pytest.mark.parametrize("i", cases())
def test_wide_layout_with_the_tensor_memory_kernel_off(i):
    env = dict(os.environ, KVQ_NO_TC="1")
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT, here=HERE, i=i)], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "wide case ok" in r.stdout
