"""CPU float64 oracle of the sparse-MLA decode over an FP8 KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
links this module: only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU baseline / reference arm use it.  It shares no code with
the CUDA path.

The pages raise an FP8 MLA KV-cache path ("feat: add XTuner TileLang sparse
MLA backend", Summary: the unsupported FP8 MLA KV-cache path is rejected;
Pull request overview: BF16 and FP8 sparse decode tests for FlashMLA) but do
not print its format.  The format read here comes from outside the pages: the
FP8 sparse-decode cache published with DeepSeek-V3.2's FlashMLA kernels.
One cache slot (one token's latent row) is 656 bytes:

    bytes [0, 512)    512 float8 e4m3 codes (the "fn" variant: no
                      infinities, codes 0x7F / 0xFF are NaN) of the latent's
                      first 512 values (the value part);
    bytes [512, 528)  4 float32 scales (little-endian); scale k applies to
                      codes 128 k .. 128 k + 127;
    bytes [528, 656)  64 bf16 values (little-endian): the latent's last 64
                      (rope) values, not quantized.

The latent row the attention uses is the dequantized row

    x[d]       = e4m3(code[d]) * scale[d // 128]      d < 512
    x[512 + i] = rope[i]                              i < 64

and the decode is the paged decode of sparse_mla_oracle over the
dequantized cache, unchanged (page mapping, masking, output and LSE).

e4m3 (OCP 8-bit floating point, E4M3): bit 7 sign s, bits 6..3 exponent e,
bits 2..0 mantissa m, bias 7:
    e = 0:        (-1)^s * 2^-6 * m / 8          (zero and subnormals)
    e = 1 .. 15:  (-1)^s * 2^(e - 7) * (1 + m / 8), except e = 15, m = 7: NaN.

Pins (tests/test_fp8_oracle_pins.py): all 256 codes against torch's
float8_e4m3fn conversion; a slot built byte by byte with its values worked
out by hand; scale homogeneity (a power-of-two factor on a scale scales its
128 values exactly); and, with power-of-two scales (dequantized values exact
in bf16), equality with the bf16 decode oracle on the dequantized cache.
"""
from __future__ import annotations

import numpy as np

from oracle import sparse_mla_oracle as orc

SLOT_BYTES = 656
CODES = 512
SCALE_OFF = 512
ROPE_OFF = 528
TILE = 128


def e4m3_value(code: int) -> float:
    """The value of one e4m3 code, from the format definition."""
    s = -1.0 if (code >> 7) & 1 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        return s * 2.0 ** -6 * (m / 8.0)
    return s * 2.0 ** (e - 7) * (1.0 + m / 8.0)


E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def dequantize_slots(cache_u8) -> np.ndarray:
    """uint8 [..., 656] -> float64 [..., 576] latent rows."""
    import torch
    b = cache_u8.cpu().numpy() if isinstance(cache_u8, torch.Tensor) else np.asarray(cache_u8)
    b = np.ascontiguousarray(b, dtype=np.uint8)
    lead = b.shape[:-1]
    flat = b.reshape(-1, SLOT_BYTES)
    vals = E4M3_TABLE[flat[:, :CODES]]                                          # [n, 512]
    scales = flat[:, SCALE_OFF:ROPE_OFF].copy().view("<f4").astype(np.float64)  # [n, 4]
    rope_bits = flat[:, ROPE_OFF:].copy().view("<u2").astype(np.uint32) << 16   # bf16 -> fp32 bits
    rope = rope_bits.astype(np.uint32).view(np.float32).astype(np.float64)      # [n, 64]
    out = np.empty((flat.shape[0], CODES + 64), dtype=np.float64)
    for k in range(CODES // TILE):
        out[:, k * TILE:(k + 1) * TILE] = vals[:, k * TILE:(k + 1) * TILE] * scales[:, k:k + 1]
    out[:, CODES:] = rope
    return out.reshape(*lead, CODES + 64)


def sparse_mla_decode_fp8(q, cache_u8, block_table, cache_seqlens, indices, sm_scale: float,
                          page_size: int = 64, d_v: int = 512, tokens=None):
    """Paged decode over an FP8 cache uint8 [num_blocks, page_size, 656]: the
    paged decode of the dequantized cache.  Arguments and results as
    sparse_mla_oracle.sparse_mla_decode."""
    kv = dequantize_slots(cache_u8)                   # [num_blocks, page, 576] float64
    return orc.sparse_mla_decode(q, kv, block_table, cache_seqlens, indices, sm_scale, page_size, d_v,
                                 tokens=tokens)
