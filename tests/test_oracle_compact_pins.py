"""Pins of the compact-page oracle to things other than itself (no GPU needed).

The pages name no compact format (the reading is stated in
``oracle/compact_pages.py``), so the format's pieces are pinned by:
  * a published constant: the CRC-32/ISO-HDLC check value (tests/golden);
  * library second opinions: zlib's crc32, torch's binary32 -> bfloat16
    conversion and binary32 product;
  * hand-worked cases: scale 1 and 2 slices whose ratios fall on halfway
    points (round half to even), a zero slice, a non-finite page, slices with
    different maxima in one row;
  * properties: every code within [-127, 127], the slice maximum coded as
    +-127, reconstruction within half a scale step plus bf16 rounding.
The mutation test at the bottom plants plausible mistakes in copies of the
oracle and requires each to fail at least one pin.
"""

import os
import types
import zlib

import numpy as np
import pytest
import torch

from oracle import compact_pages as oc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "crc32_iso_hdlc_check.txt")
HKV, D = 4, 256


def real_impl():
    return types.SimpleNamespace(crc32=oc.crc32, f32_to_bf16_bits=oc.f32_to_bf16_bits,
                                 quantize_rows=oc.quantize_rows,
                                 dequantize_rows=oc.dequantize_rows)


def bf16_bits(x):
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


def rows_from_f32(vals, n_kv=HKV, d=D):
    """bf16 bits of rows whose values are exactly representable."""
    return bf16_bits(np.asarray(vals, dtype=np.float32).reshape(-1, 2 * n_kv * d))


def golden_crc():
    fields = {}
    for line in open(GOLDEN):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    return fields["input_ascii"].encode("ascii"), int(fields["crc"], 16)


def pin_crc_check_value(impl):
    data, crc = golden_crc()
    assert impl.crc32(data) == crc


def pin_crc_zlib(impl):
    rng = np.random.default_rng(1)
    for n in (0, 1, 7, 1000, 4099):
        b = rng.integers(0, 256, n, dtype=np.uint8).tobytes()
        assert impl.crc32(b) == zlib.crc32(b)
    a, b = b"compact", b" page"
    assert impl.crc32(b, impl.crc32(a)) == zlib.crc32(a + b)


def pin_bf16_rne_torch(impl):
    rng = np.random.default_rng(2)
    x = rng.standard_normal(4096).astype(np.float32) * np.float32(37.0)
    # exact halfway cases, both parities of the last kept bit
    hi = rng.integers(0x0080, 0x7F00, 512, dtype=np.uint32)     # finite, normal
    ties = (hi << 16 | np.uint32(0x8000)).view(np.float32)
    x = np.concatenate([x, ties, -ties, np.array([0.0, -0.0, 1e-40, 3.0e38], np.float32)])
    assert np.array_equal(impl.f32_to_bf16_bits(x), bf16_bits(x))


def pin_quantize_hand(impl):
    # slice 0 (K head 0): max 127 -> s = 1; ratios on halfway points
    row = np.zeros((1, 2 * HKV * D), dtype=np.float32)
    row[0, :8] = [127.0, -127.0, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5]
    # slice 1 (K head 1): max 254 -> s = 2; x = 3 -> 1.5 -> 2, x = 5 -> 2.5 -> 2
    row[0, D:D + 4] = [254.0, 3.0, 5.0, -7.0]
    # slice 5 (V head 1): all zero; slice 7 (V head 3): a single 1.0
    row[0, 7 * D] = 1.0
    codes, scales = impl.quantize_rows(rows_from_f32(row), HKV, D)
    assert scales[0, 0] == 1.0 and scales[0, 1] == 2.0 and scales[0, 5] == 0.0
    assert scales[0, 7] == np.float32(1.0) / np.float32(127.0)
    assert list(codes[0, :8]) == [127, -127, 0, 2, 2, 0, -2, -2]
    assert list(codes[0, D:D + 4]) == [127, 2, 2, -4]          # -3.5 -> -4 (even)
    assert not codes[0, 5 * D:6 * D].any()
    assert codes[0, 7 * D] == 127 and not codes[0, 7 * D + 1:].any()


def pin_quantize_properties(impl):
    rng = np.random.default_rng(3)
    vals = rng.standard_normal((64, 2 * HKV * D)).astype(np.float32) * np.float32(3.0)
    bits = bf16_bits(vals)
    x = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    codes, scales = impl.quantize_rows(bits, HKV, D)
    assert codes.dtype == np.int8 and scales.dtype == np.float32
    assert np.abs(codes.astype(np.int64)).max() <= 127
    g = x.reshape(64, 2 * HKV, D)
    c = codes.reshape(64, 2 * HKV, D).astype(np.float64)
    s = scales.astype(np.float64)
    amax = np.abs(g).max(axis=2)
    assert np.allclose(s, amax / 127.0, rtol=2 ** -23, atol=0)
    at_max = np.abs(g) == amax[:, :, None]
    assert np.all(np.abs(c[at_max]) == 127)
    err = np.abs(c * s[:, :, None] - g)
    assert np.all(err <= 0.5 * s[:, :, None] * (1 + 1e-5))
    deq = impl.dequantize_rows(codes, scales, HKV, D)
    d = (deq.astype(np.uint32) << 16).view(np.float32).astype(np.float64).reshape(g.shape)
    assert np.all(np.abs(d - g) <= 0.5 * s[:, :, None] * (1 + 1e-5) + np.abs(d) * 2.0 ** -8)


def pin_dequantize_torch(impl):
    rng = np.random.default_rng(4)
    codes = rng.integers(-127, 128, (8, 2 * HKV * D)).astype(np.int8)
    scales = (rng.random((8, 2 * HKV)) * 0.05).astype(np.float32)
    prod = (torch.tensor(codes.astype(np.float32)).view(8, 2 * HKV, D)
            * torch.tensor(scales)[:, :, None])
    want = prod.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).reshape(8, -1)
    assert np.array_equal(impl.dequantize_rows(codes, scales, HKV, D), want)


def pin_not_convertible(impl):
    row = np.zeros((2, 2 * HKV * D), dtype=np.float32)
    bits = rows_from_f32(row)
    bits[1, 100] = 0x7FC0                                      # NaN
    assert impl.quantize_rows(bits, HKV, D) is None
    bits[1, 100] = 0x7F80                                      # +Inf
    assert impl.quantize_rows(bits, HKV, D) is None


PINS = [pin_crc_check_value, pin_crc_zlib, pin_bf16_rne_torch, pin_quantize_hand,
        pin_quantize_properties, pin_dequantize_torch, pin_not_convertible]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_compact_oracle_pin(pin):
    pin(real_impl())


def test_page_image_and_effective_rows():
    rng = np.random.default_rng(5)
    rows = bf16_bits(rng.standard_normal((150, 2 * HKV * D)).astype(np.float32))
    page = oc.convert_page(rows[64:128], HKV, D)
    assert len(page["bytes"]) == oc.compact_page_bytes_len(64, HKV, D) == 133120
    assert page["bytes"][:131072] == page["codes"].tobytes()
    assert np.array_equal(np.frombuffer(page["bytes"][131072:], "<f4").reshape(64, 8),
                          page["scales"])
    assert page["crc"] == zlib.crc32(page["bytes"])
    eff = oc.effective_rows(rows, [1], HKV, D)
    assert np.array_equal(eff[:64], rows[:64]) and np.array_equal(eff[128:], rows[128:])
    assert np.array_equal(eff[64:128], page["values"])
    with pytest.raises(ValueError):
        oc.effective_rows(rows, [2], HKV, D)                   # rows 128..149 only


# ---------------------------------------------------------------------------
# planted mistakes: each must fail at least one pin
# ---------------------------------------------------------------------------

def _crc_mut(kind):
    def crc(data, crc=0):
        init = 0 if kind == "no_init" else 0xFFFFFFFF
        c = crc ^ init
        for byte in bytes(data):
            if kind == "msb_first":
                c ^= byte << 24
                for _ in range(8):
                    c = ((c << 1) ^ 0x04C11DB7) & 0xFFFFFFFF if c & 0x80000000 else (c << 1) & 0xFFFFFFFF
            else:
                c ^= byte
                for _ in range(8):
                    c = (c >> 1) ^ 0xEDB88320 if c & 1 else c >> 1
        return c ^ (0 if kind == "no_xorout" else 0xFFFFFFFF)
    return crc


def _bf16_truncate(x):
    return (np.asarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _quant_mut(kind):
    def quantize_rows(rows_bits, n_kv_heads, head_dim):
        x = (np.asarray(rows_bits, np.uint16).astype(np.uint32) << 16).view(np.float32)
        n = x.shape[0]
        if not np.all(np.isfinite(x)):
            return None
        g = x.reshape(n, 2 * n_kv_heads, head_dim)
        if kind == "row_scale":
            amax = np.repeat(np.abs(g).max(axis=(1, 2))[:, None], 2 * n_kv_heads, axis=1)
        else:
            amax = np.abs(g).max(axis=2)
        div = np.float32(128.0 if kind == "div128" else 127.0)
        s = np.divide(amax, div, dtype=np.float32)
        codes = np.zeros(g.shape, np.int8)
        nz = s > 0
        r = np.divide(g[nz], s[nz][:, None], dtype=np.float32)
        q = np.sign(r) * np.floor(np.abs(r) + 0.5) if kind == "half_away" else np.rint(r)
        codes[nz] = np.clip(q, -127, 127).astype(np.int8)
        return codes.reshape(n, -1), s
    return quantize_rows


def _deq_mut(codes, scales, n_kv_heads, head_dim):
    c = np.asarray(codes, np.int8).reshape(codes.shape[0], 2 * n_kv_heads, head_dim)
    prod = c.astype(np.float32) * np.asarray(scales, np.float32)[:, :, None]
    return _bf16_truncate(prod).reshape(codes.shape[0], -1)


MUTANTS = {
    "crc_no_init": dict(crc32=_crc_mut("no_init")),
    "crc_no_xorout": dict(crc32=_crc_mut("no_xorout")),
    "crc_msb_first": dict(crc32=_crc_mut("msb_first")),
    "bf16_truncates": dict(f32_to_bf16_bits=_bf16_truncate),
    "round_half_away": dict(quantize_rows=_quant_mut("half_away")),
    "scale_over_128": dict(quantize_rows=_quant_mut("div128")),
    "one_scale_per_row": dict(quantize_rows=_quant_mut("row_scale")),
    "dequant_truncates": dict(dequantize_rows=_deq_mut),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_planted_mistake_is_caught(name):
    impl = real_impl()
    for k, v in MUTANTS[name].items():
        setattr(impl, k, v)
    failed = 0
    for pin in PINS:
        try:
            pin(impl)
        except AssertionError:
            failed += 1
    assert failed >= 1, f"mutant {name} passed every pin"
