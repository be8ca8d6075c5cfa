"""FP8 path on the GPU against the float64 / exact-float32 oracle
(oracle/fp8_ref.py): the quantiser's e4m3 codes and scales bit for bit
(rotated or not, per block or per plane, row-major or transposed)."""

import numpy as np
import pytest
import torch

import exact_io_aware_order_gb300 as attn
from oracle import fp8_ref as F

pytestmark = pytest.mark.gpu


def e4m3_values(codes_u8):
    return codes_u8.cpu().view(torch.float8_e4m3fn).to(torch.float64).numpy()


def signs_for(d, seed):
    return np.where(np.random.default_rng(seed).random(d) < 0.5, -1.0, 1.0).astype(np.float32)


@pytest.mark.parametrize("planes,rows,d,rot,block,transpose", [
    (3, 300, 128, True, 128, False),
    (2, 256, 128, False, 128, True),
    (4, 1000, 128, False, 0, True),
    (2, 129, 64, True, 128, False),
    (1, 4096, 128, True, 0, False),
])
def test_quantizer_bit_exact(dev, planes, rows, d, rot, block, transpose):
    g = torch.Generator().manual_seed(rows + d)
    x = (torch.randn(planes, rows, d, generator=g) *
         torch.exp(torch.randn(planes, rows, 1, generator=g))).to(torch.bfloat16)
    x[0, :, 3] *= 30                                           # an outlier channel
    sg = signs_for(d, 5) if rot else None
    codes, scales = attn.quantize_fp8(x.to(dev), torch.from_numpy(sg).to(dev) if rot else None,
                                      block_rows=block, transpose=transpose)
    attn.check_device_status()
    x32 = x.float().numpy()
    if rot:
        x32 = F.hadamard_rotate(x32, sg)
    ref_codes, ref_scales = F.quantize_blocks(x32, block if block else rows)
    got = e4m3_values(codes)
    if transpose:
        got = got.transpose(0, 2, 1)
    assert np.array_equal(got, ref_codes)
    assert np.array_equal(scales.cpu().numpy().reshape(ref_scales.shape), ref_scales)
