"""Failure detection without a fault: a bounded wait on a barrier phase that nothing completes
gives up (on its time limit, or at once on the CTA's abort flag), reports it, and the context
stays usable for the next attention call."""
import numpy as np
import pytest

import exact_attention_19_gb300 as fa
import oracle
import synth
from parity_util import assert_close, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_19_gb300 import build

    build.build()
    fa.load()
    oracle.build()
    yield


def test_wait_gives_up_at_its_time_limit():
    word, ns = fa.fa_selftest_wait(0)
    assert word & 1 and (word >> 8) == 1, hex(word)
    assert 1.5e9 <= ns <= 10e9, ns  # the kernels' limit is about 2 s


def test_wait_gives_up_on_the_abort_flag():
    word, ns = fa.fa_selftest_wait(1)
    assert word & 1 and (word >> 8) == 2, hex(word)
    assert ns < 0.5e9, ns  # the flag rises after about 1 ms


def test_context_usable_after_the_self_tests():
    fa.fa_selftest_wait(1)
    w = synth.Workload("after_selftest", 1, 2, 200, 200, 64, True, seed=860)
    q, k, v = w.make()
    o, lse = run_gpu(q, k, v, w.scale, True)
    o_ref, lse_ref = oracle.attention_fwd(q, k, v, w.scale, True)
    assert_close(o, lse, o_ref, lse_ref)
    st, word = fa.fa_fwd_status(None, clear=True)
    assert st == 0 and word == 0
