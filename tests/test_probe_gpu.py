"""The rate probes (measurement aids for the rooflines).  Tensor-core probe:
every CTA lands on its own SM, every bounded wait completes, and the dense
kind::f16 rate it measures is a power of two in FLOP per SM clock within the
range a tensor core can have (1k to 32k).  Gather probe: every CTA lands on
its own SM, the byte sums are those of random loads from the buffer, and the
rate lies between a quarter of a load and eight loads per SM clock."""
import math

import numpy as np

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


def test_gather_probe_runs_one_cta_per_sm():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    buf = torch.full((1 << 20,), 3, dtype=torch.uint8, device="cuda")
    iters = 16
    rec = bra.gather_rate_probe(buf, sms, iters)
    torch.cuda.synchronize()
    r = rec.cpu().numpy()
    assert len(set(r[:, 2].tolist())) == sms
    # every loaded byte is 3: each CTA's sum is 3 x its loads
    assert (r[:, 3] == 3 * 1024 * iters * 8).all()
    per_clk = 1024 * iters * 8 / r[:, 0]
    assert 0.25 <= float(np.median(per_clk)) <= 8.0


def test_gather_probe_rejects_bad_arguments():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ok = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    odd = torch.zeros(3 << 12, dtype=torch.uint8, device="cuda")
    small = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    for buf, ctas, iters in ((odd, 1, 1), (small, 1, 1), (ok, 0, 1), (ok, sms + 1, 1),
                             (ok, 1, 0), (ok, 1, (1 << 20) + 1)):
        with pytest.raises(bra.BraError):
            bra.gather_rate_probe(buf, ctas, iters)
