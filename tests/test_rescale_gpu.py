"""Rescales of the output accumulator at full steps, repeated.

The bias kernel walks key tiles from the diagonal backwards and rescales O
when a row's running max grows by more than 2^8. In its full steps (decode,
and prefills the two-head main kernel does not take, e.g. alpha <= 0) the
first half of PV(s) starts as soon as the first softmax warpgroup's P is in.
So an O rescale must not be split between the two warpgroups.

These cases make the far keys, the ones visited last, carry by far the
largest logits:
- the keys more than 600 positions back are scaled so that the row max jumps
  at a full step;
- each call runs several times, since a race shows only in some runs;
- everything is compared with the oracle.
"""
import pytest
import torch

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


def _far_keys_dominate(inp, w, back=600, scale=-6.0):
    """k rows more than `back` positions before each sequence's end, times
    `scale` (with alpha < 0, or aligned q, their logits dominate).

    v is halved. Softmax rows this peaked copy single v entries, some beyond
    4 in magnitude, where one bf16 step of the output is 2^-5. Output rounding
    alone would then use most of the absolute 2e-2 bound. A rescale race
    errs by a factor of up to 2^8, so it still fails far beyond the bound."""
    k = inp["k"].float()
    start = 0
    for lk in w.k_lens:
        k[start: start + max(0, lk - back)] *= scale
        start += lk
    inp["k"] = k.to(torch.bfloat16)
    inp["v"] = (inp["v"].float() * 0.5).to(torch.bfloat16)
    return inp


@pytest.mark.parametrize("alpha", [-0.0883883, -0.3])
def test_prefill_full_step_rescales(alpha):
    # alpha < 0: the bias kernel runs every key tile (band, then full steps)
    w = W.custom("rescale_pf", [1024, 700], [1024, 700], 8, 2, 32, 64, alpha=alpha)
    inp = _far_keys_dominate(W.make_inputs(w), w)
    for _ in range(6):
        compare(w, inp, run_gpu(w, inp, decode=False))


def test_decode_full_step_rescales():
    w = W.custom("rescale_dec", [9, 1, 4], [4000, 2500, 900], 16, 2, 64, 256, alpha=-0.0883883)
    inp = _far_keys_dominate(W.make_inputs(w), w, back=300)
    for _ in range(6):
        compare(w, inp, run_gpu(w, inp, decode=True))
