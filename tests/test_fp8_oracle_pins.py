"""Pins of the FP8 KV-cache oracle (oracle/fp8_kv_oracle.py) against things
other than itself: torch's float8_e4m3fn conversion for every code, a cache
slot assembled byte by byte with its values worked out by hand, scale
homogeneity, and the bf16 decode oracle where the dequantized values are
exact in bf16.  Planted mistakes in the dequantization must fail a pin."""
import struct

import numpy as np
import pytest
import torch

import mla_inputs as mi
from oracle import fp8_kv_oracle as f8
from oracle import sparse_mla_oracle as orc


def test_every_e4m3_code_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = f8.E4M3_TABLE
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan) and nan.sum() == 2    # 0x7F and 0xFF
    assert np.array_equal(mine[~nan], ref[~nan])
    assert mine[0x7E] == 448.0 and mine[0x01] == 2.0 ** -9 and mine[0x38] == 1.0


def _slot(codes, scales, rope):
    b = bytes(codes) + struct.pack("<4f", *scales) + b"".join(struct.pack("<H", h) for h in rope)
    assert len(b) == 656
    return torch.tensor(list(b), dtype=torch.uint8)


def test_hand_built_slot():
    """Codes 0x38 (1.0), 0xC0 (-2.0), 0x01 (2^-9), 0x7E (448), 0x09 (2^-6 * 9/8),
    0x80 (-0); tile scales 0.5, 2, 1, 0.25; rope bf16 0x3FC0 (1.5), 0xC040 (-3)."""
    codes = [0] * 512
    codes[0], codes[1], codes[2] = 0x38, 0xC0, 0x01          # tile 0, scale 0.5
    codes[128], codes[129] = 0x7E, 0x09                       # tile 1, scale 2
    codes[300] = 0x38                                         # tile 2, scale 1
    codes[511], codes[400] = 0xC0, 0x80                       # tile 3, scale 0.25
    rope = [0] * 64
    rope[0], rope[63] = 0x3FC0, 0xC040
    x = f8.dequantize_slots(_slot(codes, (0.5, 2.0, 1.0, 0.25), rope)[None])[0]
    want = np.zeros(576)
    want[0], want[1], want[2] = 0.5, -1.0, 2.0 ** -10
    want[128], want[129] = 896.0, 2.0 ** -5 * 9 / 8
    want[300] = 1.0
    want[511] = -0.5
    want[512], want[575] = 1.5, -3.0
    assert np.array_equal(x, want)
    assert np.signbit(x[400])                                 # -0 stays -0


def test_scale_homogeneity():
    """Multiplying tile k's scale by 2^j multiplies exactly its 128 values by
    2^j and leaves the rest of the row unchanged."""
    c, u = mi.decode_case_fp8(71, batch=1, s_next=1, h_q=2, lo=40, hi=40, topk=16, page=64, spare_pages=0)
    slot = u[0, 3].clone()
    base = f8.dequantize_slots(slot[None])[0]
    for k, j in ((0, 3), (2, -5), (3, 1)):
        s2 = slot.clone()
        sc = s2[512:528].view(torch.float32).clone()
        sc[k] = sc[k] * 2.0 ** j
        s2[512:528] = sc.view(torch.uint8)
        x = f8.dequantize_slots(s2[None])[0]
        t = slice(128 * k, 128 * k + 128)
        assert np.array_equal(x[t], base[t] * 2.0 ** j)
        rest = np.ones(576, dtype=bool)
        rest[t] = False
        assert np.array_equal(x[rest], base[rest])


def test_equals_bf16_oracle_when_exact_in_bf16():
    """Power-of-two scales make every dequantized value exact in bf16: the FP8
    decode then equals the bf16 decode of that bf16 cache."""
    c, u = mi.decode_case_fp8(72, batch=3, s_next=2, h_q=4, lo=200, hi=500, topk=128, page=64, spare_pages=2,
                              pow2_scales=True)
    x = f8.dequantize_slots(u)
    finite = np.isfinite(x)
    xb = torch.from_numpy(x).to(torch.bfloat16)
    assert np.array_equal(xb.double().numpy()[finite], x[finite])      # exact in bf16
    o1, l1 = f8.sparse_mla_decode_fp8(c.q, u, c.block_table, c.cache_seqlens, c.indices, c.sm_scale, 64)
    o2, l2 = orc.sparse_mla_decode(c.q, xb, c.block_table, c.cache_seqlens, c.indices, c.sm_scale, 64)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l1, l2, rtol=1e-12, atol=1e-14)
    assert np.all(np.isfinite(o1))


def test_quantization_error_within_e4m3_step():
    """The generator's codes round each value/scale to e4m3: the dequantized
    value is within half an e4m3 step (2^-4 relative, or 2^-10 absolute in
    the subnormal range, times the scale) of the latent value."""
    c, u = mi.decode_case_fp8(73, batch=2, s_next=1, h_q=2, lo=100, hi=200, topk=32, page=64, spare_pages=1)
    lat = c.kv_cache.double().numpy().reshape(-1, 576)
    x = f8.dequantize_slots(u).reshape(-1, 576)
    ok = np.isfinite(lat).all(axis=1)
    scale = u.reshape(-1, 656)[:, 512:528].clone().view(torch.float32).double().numpy()
    for k in range(4):
        t = slice(128 * k, 128 * k + 128)
        y = lat[ok, t] / scale[ok, k:k + 1]
        step = np.maximum(np.abs(y) * 2.0 ** -4, 2.0 ** -10)
        assert np.all(np.abs(x[ok, t] / scale[ok, k:k + 1] - y) <= step * (1 + 1e-12))


MUTATIONS = {
    "mantissa_over_16": lambda code: (
        (-1.0 if code >> 7 else 1.0) * (2.0 ** (((code >> 3) & 15) - 7) * (1 + (code & 7) / 16.0)
                                        if (code >> 3) & 15 else 2.0 ** -6 * (code & 7) / 8.0)),
    "bias_8": lambda code: (
        (-1.0 if code >> 7 else 1.0) * (2.0 ** (((code >> 3) & 15) - 8) * (1 + (code & 7) / 8.0)
                                        if (code >> 3) & 15 else 2.0 ** -6 * (code & 7) / 8.0)),
    "subnormal_as_normal": lambda code: (
        (-1.0 if code >> 7 else 1.0) * 2.0 ** (((code >> 3) & 15) - 7) * (1 + (code & 7) / 8.0)),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_decode_mistake_fails_a_pin(monkeypatch, name):
    table = np.array([MUTATIONS[name](c) if c not in (0x7F, 0xFF) else np.nan for c in range(256)])
    monkeypatch.setattr(f8, "E4M3_TABLE", table)
    with pytest.raises(AssertionError):
        test_every_e4m3_code_matches_torch()
        test_hand_built_slot()


def test_planted_scale_layout_mistake_fails_a_pin(monkeypatch):
    """Scales applied to the wrong tiles (reversed order)."""
    real = f8.dequantize_slots

    def reversed_scales(b):
        b = np.array(b.cpu().numpy() if isinstance(b, torch.Tensor) else b, dtype=np.uint8, copy=True)
        flat = b.reshape(-1, 656)
        sc = flat[:, 512:528].reshape(-1, 4, 4)[:, ::-1].reshape(-1, 16).copy()
        flat[:, 512:528] = sc
        return real(flat.reshape(b.shape))
    monkeypatch.setattr(f8, "dequantize_slots", reversed_scales)
    with pytest.raises(AssertionError):
        test_hand_built_slot()
