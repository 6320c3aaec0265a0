"""Activation quantisation on the GPU (the device functions the layer's
permute, h-quantise and token-major GEMM epilogues use) against the oracle's
activation rule, value for value: NVFP4 (global scale 1) and MXFP8, on rows
built to sit on and next to every rounding decision."""
import numpy as np
import pytest
import torch

from sparse_moe_layer_experts_b300 import binding as B
from sparse_moe_layer_experts_b300.layer import quantize_activations

pytestmark = pytest.mark.gpu

E2M1 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)
E2M1_MIDPOINTS = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)


def e4m3_values():
    out = np.zeros(256, np.float64)
    for c in range(256):
        e, m = (c >> 3) & 15, c & 7
        mag = m / 8 * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
        out[c] = -mag if c & 0x80 else mag
    return out


def ulp_steps(x: np.ndarray, k: int) -> np.ndarray:
    """Nonzero x moved by k FP32 ulps away from zero (toward it for k < 0);
    zeros stay zero."""
    x = x.astype(np.float32)
    b = x.view(np.int32).astype(np.int64)
    out = (b + k).astype(np.int32).view(np.float32)
    return np.where(x == 0, x, out)


def nvfp4_adversarial_rows(rng) -> np.ndarray:
    e4 = e4m3_values()
    blocks = []
    for code in range(1, 127):  # every positive E4M3 block scale
        s = e4[code]
        for k in (-1, 0, 1):
            blk = np.empty(16, np.float32)
            blk[0] = 6.0 * s  # amax / 6 == s exactly
            mids = np.array(E2M1_MIDPOINTS * 2 + (4.0,), np.float64) * s
            blk[1:] = ulp_steps(mids.astype(np.float32), k)
            blk[1::2] *= -1
            blocks.append(blk)
    z = np.zeros(16, np.float32)
    blocks.append(z)
    nz = z.copy()
    nz[3] = -0.0
    blocks.append(nz)
    blocks.append(np.full(16, 1e-40, np.float32))        # subnormal block
    blocks.append(np.linspace(-1e6, 1e6, 16).astype(np.float32))  # scale saturates at 448
    while len(blocks) % 8:
        blocks.append((rng.standard_normal(16) * 10.0 ** rng.uniform(-4, 4)).astype(np.float32))
    return np.concatenate(blocks).reshape(-1, 128)


def test_nvfp4_activation_codes_match_oracle(oracle_mod):
    rng = np.random.default_rng(5)
    rows = [nvfp4_adversarial_rows(rng),
            (rng.standard_normal((300, 512)) * 10.0 ** rng.uniform(-6, 6, (300, 1))).astype(np.float32)]
    e4 = e4m3_values()
    for x in rows:
        codes, sf = quantize_activations(torch.from_numpy(x).cuda(), B.BEAM_MOE_W_NVFP4)
        torch.cuda.synchronize()
        codes, sf = codes.cpu().numpy(), sf.cpu().numpy()
        nib = np.stack([codes & 15, codes >> 4], axis=-1).reshape(x.shape[0], -1)
        val = np.where(nib & 8, -1.0, 1.0) * E2M1[nib & 7] * np.repeat(e4[sf], 16, axis=1)
        ref = oracle_mod.fake_quant_rows(x)
        assert np.array_equal(val.astype(np.float32), ref), \
            np.argwhere(val.astype(np.float32) != ref)[:5]


def mxfp8_adversarial_rows(rng) -> np.ndarray:
    e4 = e4m3_values()
    pos = np.sort(e4[1:127])
    mids = (pos[:-1] + pos[1:]) / 2  # E4M3 rounding midpoints
    blocks = []
    for scale_exp in (-20, -3, 0, 7, 40):
        s = 2.0 ** scale_exp
        for k in (-1, 0, 1):
            for start in range(0, len(mids), 31):
                blk = np.zeros(32, np.float64)
                blk[0] = 448.0 * s  # amax: shared exponent = scale_exp
                m = mids[start:start + 31] * s
                blk[1:1 + len(m)] = m
                b = ulp_steps(blk.astype(np.float32), k)
                b[0] = np.float32(448.0 * s)
                b[2::2] *= -1
                blocks.append(b)
    blocks.append(np.zeros(32, np.float32))
    blocks.append(np.full(32, -3e-39, np.float32))
    while len(blocks) % 4:
        blocks.append((rng.standard_normal(32) * 10.0 ** rng.uniform(-4, 4)).astype(np.float32))
    return np.concatenate(blocks).reshape(-1, 128)


def test_mxfp8_activation_codes_match_oracle(oracle_mod):
    rng = np.random.default_rng(6)
    rows = [mxfp8_adversarial_rows(rng),
            (rng.standard_normal((300, 512)) * 10.0 ** rng.uniform(-6, 6, (300, 1))).astype(np.float32)]
    for x in rows:
        codes, sf = quantize_activations(torch.from_numpy(x).cuda(), B.BEAM_MOE_W_MXFP8)
        torch.cuda.synchronize()
        val = oracle_mod.dequantize_mxfp8(codes.cpu().numpy(), sf.cpu().numpy()).astype(np.float32)
        ref = oracle_mod.fake_quant_mxfp8_rows(x)
        assert np.array_equal(val, ref), np.argwhere(val != ref)[:5]
