"""FP8 E4M3 path: the per-head quantiser (bit-exact against the oracle's
E4M3 rounding) and attention on E4M3 inputs (oracle on the dequantised
values; output within max-abs 6e-2, lse within 1e-3, skip bits outside the
1e-3 margin bit-exact).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import _cases
import _gpu
from gen import inputs as gi
from oracle import numerics

pytestmark = pytest.mark.gpu


def gpu_quantize(bits):
    b = _gpu.bsa()
    T, H, d = bits.shape
    x = _gpu.to_dev_bf16(bits)
    codes = torch.empty((T, H, d), dtype=torch.uint8, device="cuda")
    scale = torch.empty((H,), dtype=torch.float32, device="cuda")
    b.check(b.quantize_fp8(x, T, H, d, codes, scale), "quantize")
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scale.cpu().numpy()


@pytest.mark.parametrize("key", ["gqa_ragged", "weak_sink", "tiny"])
def test_quantizer_bit_exact(key):
    p = _cases.small_problem(key)
    for x in (p.q, p.k, p.v):
        codes, scale = gpu_quantize(x)
        ref_codes, ref_scale = numerics.quantize_per_head(x)
        assert np.array_equal(scale, ref_scale)
        assert np.array_equal(codes, ref_codes)


def test_quantizer_zero_head():
    x = np.zeros((300, 3, 128), np.uint16)
    x[:, 1] = gi.bf16_bits_from_f32(np.linspace(-3, 5, 300 * 128, dtype=np.float32).reshape(300, 128))
    codes, scale = gpu_quantize(x)
    ref_codes, ref_scale = numerics.quantize_per_head(x)
    assert scale[0] == 1.0 and scale[2] == 1.0
    assert np.array_equal(scale, ref_scale) and np.array_equal(codes, ref_codes)


def quantized(p):
    out = []
    for x in (p.q, p.k, p.v):
        out.append(gpu_quantize(x))
    return (out[0][0], out[1][0], out[2][0], out[0][1], out[1][1], out[2][1])


@pytest.mark.parametrize("key,lam", [("C0", 0.01), ("gqa_ragged", 0.01), ("gqa_ragged", 0.0),
                                     ("weak_sink", 0.05), ("no_sink", 0.0), ("tiny", 0.01)])
@pytest.mark.parametrize("causal", [True, False])
def test_fp8_attention(key, lam, causal):
    p = _cases.small_problem(key)
    f8 = quantized(p)
    g = _gpu.run(p, lam=lam, causal=causal, fp8=f8)
    assert bool(torch.isfinite(g["out"]).all())
    _gpu.compare(p, g, fp8=f8)


def test_fp8_full_size_sampled():
    p = _cases.full_problem("C1")
    f8 = quantized(p)
    g = _gpu.run(p, lam=0.01, fp8=f8)
    assert bool(torch.isfinite(g["out"]).all())
    _gpu.compare(p, g, items=_gpu.sample_items(p, 12, seed=2), fp8=f8)


_C4 = {}


def _c4():
    if not _C4:
        p = _cases.full_problem("C4")
        _C4["p"], _C4["f8"] = p, quantized(p)
    return _C4["p"], _C4["f8"]


@pytest.mark.parametrize("lam", [0.01, 0.0])
def test_fp8_128k_layer_sampled(lam):
    """The FP8 variant of the 128K Llama-shaped layer, as the bench times it
    (lambda 0.01), and with skipping off (the dense FP8 kernel)."""
    p, f8 = _c4()
    g = _gpu.run(p, lam=lam, fp8=f8)
    assert bool(torch.isfinite(g["out"]).all())
    _gpu.compare(p, g, items=_gpu.sample_items(p, 32, seed=4), fp8=f8)
    if lam == 0:
        assert not g["bitmap"].any()
