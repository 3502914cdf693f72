"""Blockwise FP8 (E4M3) weight encoding, plain reference (test infrastructure).

"Training a 1T-Params MoE on EU public infrastructure", FP8 expert weight
all-gather: the weights are split into blocks of 128 values; each block is
scaled to the FP8 E4M3 range and cast, and travels with one fp32 scale; the
receiver dequantises to bf16 before the expert computation.

Readings (the page gives no formula):
  * a block is 128 consecutive elements of the weight tensor as stored;
  * scale = amax / 448 in fp32 (448 is E4M3's largest finite value), or 1
    for an all-zero block; code = E4M3(x / scale) with the division in fp32
    and round-to-nearest-even, saturating at +-448;
  * dequantised weight = bf16(E4M3 value * scale), the product in fp32.
The precision is the page's (fp32 scale, E4M3 codes, bf16 result), so these
functions compute in fp32 where the page does.

E4M3 (as NVIDIA's e4m3 and the OCP FP8 "E4M3FN"): 1 sign bit, 4 exponent
bits with bias 7, 3 mantissa bits, subnormals below 2^-6 (step 2^-9), no
infinities, S.1111.111 is NaN, largest finite 1.75 * 2^8 = 448.
"""
from __future__ import annotations

import numpy as np
import torch

E4M3_MAX = 448.0
BLOCK = 128


def e4m3_decode(codes) -> np.ndarray:
    """float32 value of each 8-bit code (NaN for S.1111.111)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 15
    m = c & 7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    out = sign * mag
    out = np.where((e == 15) & (m == 7), np.nan, out)
    return out.astype(np.float32)


def e4m3_round(x) -> np.ndarray:
    """Round float32 values to the nearest E4M3 value, ties to even,
    saturating at +-448.  Returns float32 (exact E4M3 values, sign kept)."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    a = np.abs(x)
    _, e2 = np.frexp(a)                    # a = m * 2^e2, m in [0.5, 1)
    expo = np.maximum(e2 - 1, -6)          # normal exponent, or the subnormal floor
    quantum = np.exp2(expo - 3.0)          # 3 mantissa bits
    r = np.rint(a / quantum) * quantum     # rint: ties to even
    r = np.minimum(r, E4M3_MAX)
    return np.where(np.signbit(x), -r, r).astype(np.float32)


def e4m3_encode(v) -> np.ndarray:
    """8-bit code of exactly representable E4M3 values (sign bit from the
    float's sign, so -0.0 encodes as 0x80)."""
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    sign = np.signbit(v).astype(np.int64)
    a = np.abs(v)
    _, e2 = np.frexp(a)
    normal = a >= 2.0 ** -6
    e_field = np.where(normal, e2 - 1 + 7, 0)
    m_field = np.where(normal, (a / np.exp2(e2 - 1.0) - 1.0) * 8.0, a / 2.0 ** -9)
    if not np.all(m_field == np.round(m_field)):
        raise ValueError("value not representable in E4M3")
    code = (sign << 7) | (e_field.astype(np.int64) << 3) | m_field.astype(np.int64)
    return code.astype(np.uint8)


def quantize_blockwise(w):
    """(codes uint8, scales float32 [n/128]) of a tensor whose element count
    is a multiple of 128, blocks taken in memory order."""
    flat = torch.as_tensor(w).reshape(-1).float().numpy().astype(np.float32)
    if flat.size % BLOCK:
        raise ValueError("element count must be a multiple of 128")
    blocks = flat.reshape(-1, BLOCK)
    amax = np.abs(blocks).max(axis=1)
    scales = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    x = (blocks / scales[:, None]).astype(np.float32)   # fp32 division, round to nearest even
    codes = e4m3_encode(e4m3_round(x)).reshape(-1)
    return codes, scales


def dequantize_blockwise(codes, scales) -> torch.Tensor:
    """bf16 weights (as a torch tensor) of codes and per-block fp32 scales."""
    vals = e4m3_decode(codes).reshape(-1, BLOCK)
    prod = (vals * np.asarray(scales, dtype=np.float32)[:, None]).astype(np.float32)   # fp32 product
    return torch.from_numpy(prod.reshape(-1)).to(torch.bfloat16)
