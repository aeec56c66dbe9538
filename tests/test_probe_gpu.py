"""The tensor-core rate probe (a measurement aid for the fused kernels'
roofline): every CTA lands on its own SM, every bounded wait completes, and
the dense kind::f16 rate it measures is a power of two in FLOP per SM clock
within the range a tensor core can have (1k to 32k)."""
import math

import pytest
import torch

import bmm_reducescatter_alltoall_gb300 as bra

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_probe_runs_one_cta_per_sm(dtype):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rec = bra.mma_rate_probe(sms, 256, dtype)
    torch.cuda.synchronize()
    r = rec.cpu().numpy()
    assert (r[:, 2] == 0).all()
    assert len(set(r[:, 3].tolist())) == sms
    per_clk = 256 * 4 * 2 * 128 * 256 * 16 / r[:, 0]
    rate = float(sorted(per_clk)[len(per_clk) // 2])
    assert 1024 <= rate <= 32768
    assert abs(math.log2(rate) - round(math.log2(rate))) < 0.15, rate


def test_probe_rejects_bad_arguments():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for ctas, iters in ((0, 1), (sms + 1, 1), (1, 0), (1, 1 << 23)):
        with pytest.raises(bra.BraError):
            bra.mma_rate_probe(ctas, iters)
