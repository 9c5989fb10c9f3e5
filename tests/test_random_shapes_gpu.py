"""Seeded random shapes against the fp64 oracles: prefill, decode and the
backward, through the C ABI.

Each case draws from one seeded generator:
- sequence lengths;
- query / kv heads;
- r_dim, from 0 up to 64 and including multiples of 8 below 16;
- E, including 0, values below 64 and values not a multiple of 8;
- a window or none;
- a log-scale base or none;
- alpha, including negative values.

The shapes therefore land on the tcgen05 and the warp-MMA paths alike. The
tolerances are each path's own: out <= 2e-2 and lse <= 1e-3 for the
forward, and the norm-wise gradient tolerance of tests/test_backward_gpu.py.
"""
import numpy as np
import pytest

from tests.conftest import gpu_available
from tests.parity_util import compare, run_gpu
from relative_position_biased_gb300 import workloads as W

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not gpu_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import relative_position_biased_gb300 as rpb
    rpb.build()
    rpb.load_library()
    import oracle
    oracle.build()


HEADS = [(1, 1), (2, 1), (4, 1), (4, 2), (8, 2), (16, 2), (6, 3), (12, 4)]
RDIMS = [0, 8, 16, 24, 32, 48, 64]
EXTENTS = [0, 8, 40, 64, 100, 200, 1024]


def _draw(seed, decode):
    rng = np.random.default_rng(1000 + seed)
    Hq, Hkv = HEADS[rng.integers(len(HEADS))]
    r_dim = int(rng.choice(RDIMS))
    E = int(rng.choice(EXTENTS)) if r_dim else 0
    nseq = int(rng.integers(1, 5))
    if decode:
        q_lens = [int(rng.integers(1, 10)) for _ in range(nseq)]
        k_lens = [ql + int(rng.integers(0, 3000)) for ql in q_lens]
    else:
        q_lens = [int(rng.integers(1, 500)) for _ in range(nseq)]
        k_lens = [ql + (int(rng.integers(0, 200)) if rng.random() < 0.3 else 0) for ql in q_lens]
    window = int(rng.integers(1, 600)) if rng.random() < 0.4 else 0
    base = float(rng.choice([0.0, 0.0, 16.0, 300.0]))
    alpha = float(rng.choice([1 / np.sqrt(128), 0.0, -0.07, 0.3]))
    return W.custom(f"rand{'_dec' if decode else ''}{seed}", q_lens, k_lens, Hq, Hkv, r_dim, E,
                    window=window, log_scale_base=base, alpha=alpha, seed=seed)


@pytest.mark.parametrize("seed", range(30))
def test_random_prefill(seed):
    w = _draw(seed, decode=False)
    inp = W.make_inputs(w)
    compare(w, inp, run_gpu(w, inp, decode=False))


@pytest.mark.parametrize("seed", range(30))
def test_random_decode(seed):
    w = _draw(seed, decode=True)
    inp = W.make_inputs(w)
    compare(w, inp, run_gpu(w, inp, decode=True))


@pytest.mark.parametrize("seed", range(16))
def test_random_backward(seed):
    from tests.test_backward_gpu import check
    w = _draw(100 + seed, decode=False)
    check(w)                 # (every drawn r_dim is a multiple of 8)
