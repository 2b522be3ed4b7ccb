"""The FMA-ceiling instrument: the FMA count it reports, and its sink, which with mul = 1 and add = 0 holds each
CTA's sum of the chains' start values (small integers, so the fp32 sums are exact)."""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import quantized_decode_gemv_q4_gb300 as q4  # noqa: E402


def expected_cta_sum():
    t = np.arange(512)
    return float(sum(((t % 7) + j).sum() + ((t % 5) + j).sum() for j in range(8)))


@pytest.mark.parametrize("fmas", [1, 8 * 14336 * 4096, 8 * 18944 * 3584 + 12345])
def test_fma_ceiling_counts_and_sink(fmas):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    sink = torch.full((sms + 3,), -1.0, device="cuda")
    done = q4.q4_fma_ceiling(sink, fmas, mul=1.0, add=0.0)
    torch.cuda.synchronize()
    per_round = sms * 512 * 16
    assert done >= fmas and done % per_round == 0 and done - fmas < per_round
    out = sink.cpu().numpy()
    assert np.all(out[:sms] == expected_cta_sum())
    assert np.all(out[sms:] == -1.0)  # one float per SM, nothing beyond


def test_fma_ceiling_refuses_a_short_sink():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    sink = torch.zeros(sms - 1, device="cuda")
    with pytest.raises(q4.Q4Error):
        q4.q4_fma_ceiling(sink, 1000)
    with pytest.raises(q4.Q4Error):
        q4.q4_fma_ceiling(torch.zeros(sms, device="cuda"), 0)
