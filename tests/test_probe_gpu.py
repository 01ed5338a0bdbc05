"""The exp2-throughput probes (the denominator of the exponential-unit roofline)."""
import pytest

import exact_attention_19_gb300 as fa

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("method", [0, 1])
def test_probe_exp2_rate_is_plausible(method):
    import torch

    torch.cuda.init()
    rate = fa.fa_probe_exp2(method)
    # between one result per SM every 8 clocks and four per lane per clock
    assert 0.125 * 32 < rate < 128.0, rate
    again = fa.fa_probe_exp2(method)
    assert abs(again - rate) / rate < 0.1
