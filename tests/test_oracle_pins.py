"""Pins of the CPU oracle against things other than itself (no GPU needed).

Each test checks one oracle function against a library routine (torch in
float64, torch's float8_e4m3fn / bfloat16 conversions, SDPA), a brute-force
search, an algebraic identity, a closed-form special case, or a number printed
on the source pages (tests/golden/page_figures.json).
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import codecs as C
from oracle import selection as S
from mixed_precision_paged_argus_gb300 import accounting, workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")


# ---------------------------------------------------------------- e4m3 codec

def test_e4m3_table_equals_torch_float8_e4m3fn():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    tab = C.e4m3_table()
    nan = np.isnan(ref)
    assert nan.sum() == 2 and np.array_equal(np.isnan(tab), nan)
    assert np.array_equal(tab[~nan], ref[~nan])


def test_e4m3_ocp_landmarks():
    # OCP FP8 E4M3: max normal 448, min normal 2^-6, min subnormal 2^-9, 1.0 = 0x38.
    assert C.e4m3_value(0x7E) == 448.0
    assert C.e4m3_value(0x08) == 2.0 ** -6
    assert C.e4m3_value(0x01) == 2.0 ** -9
    assert C.e4m3_value(0x38) == 1.0
    assert C.e4m3_value(0xB8) == -1.0
    assert math.isnan(C.e4m3_value(0x7F)) and math.isnan(C.e4m3_value(0xFF))


def _all_finite_fp16_as_f32():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = bits.view(np.float16).astype(np.float32)
    return x[np.isfinite(x)]


def test_e4m3_encoder_exhaustive_vs_brute_force():
    x = _all_finite_fp16_as_f32()
    got = C.e4m3_encode(x)
    vals = C.e4m3_table()[:127]                       # non-negative finite values
    a = np.minimum(np.abs(x).astype(np.float64), 448.0)
    d = np.abs(a[:, None] - vals[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    # among equally near codes take the even one (mantissa LSB 0)
    even = cand & (np.arange(127)[None, :] % 2 == 0)
    pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
    want = (pick | (np.signbit(x).astype(np.int64) << 7)).astype(np.uint8)
    assert np.array_equal(got, want)


def test_e4m3_encoder_matches_torch_inside_range():
    x = _all_finite_fp16_as_f32()
    x = x[np.abs(x) < 464.0]          # torch's conversion is not saturating beyond
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(C.e4m3_encode(x), ref)


def test_fp8_unit_against_torch_pipeline():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(4096) * 3).astype(np.float16).astype(np.float32)
    codes, scale = C.quantize_unit_fp8(x)
    tx = torch.from_numpy(x)
    tscale = tx.abs().max() / torch.tensor(448.0)
    assert np.float32(tscale.item()) == scale
    ref = (tx / tscale).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)


def test_fp8_round_trip_exact_on_representable_units():
    vals = C.e4m3_table()
    fin = vals[np.isfinite(vals)]
    scale = 2.0 ** -4
    x = np.concatenate([fin, [448.0]]) * scale
    codes, s = C.quantize_unit_fp8(x.astype(np.float32))
    assert s == np.float32(scale)
    back = C.e4m3_table()[codes.astype(int)] * np.float64(s)
    assert np.array_equal(back, x)


def test_fp8_zero_unit():
    codes, s = C.quantize_unit_fp8(np.zeros(64, np.float32))
    assert s == 0 and not codes.any()


# ---------------------------------------------------------------- INT8 codec

def test_int8_round_trip_exact():
    k = np.arange(-127, 128)
    x = (k * 2.0 ** -5).astype(np.float32)
    q, s = C.quantize_unit_int8(x)
    assert s == np.float32(2.0 ** -5)
    assert np.array_equal(q.astype(np.int64), k)
    assert np.array_equal(q.astype(np.float64) * np.float64(s), x.astype(np.float64))


def test_int8_half_even_rounding_landmarks():
    x = np.array([127.0, 2.5, 3.5, -2.5, -3.5, 0.5, -0.5], np.float32)
    q, s = C.quantize_unit_int8(x)
    assert s == 1.0
    assert q.tolist() == [127, 2, 4, -2, -4, 0, 0]


def test_int8_against_torch_pipeline():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(8192) * 2).astype(np.float16).astype(np.float32)
    q, s = C.quantize_unit_int8(x)
    tx = torch.from_numpy(x)
    ts = tx.abs().max() / torch.tensor(127.0)
    assert np.float32(ts.item()) == s
    ref = torch.round(tx / ts).clamp(-127, 127).to(torch.int8).numpy()
    assert np.array_equal(q, ref)


# ---------------------------------------------------------------- INT4 codec

def test_int4_pack_order_even_low_nibble():
    assert C.pack_int4(np.array([1, 2, 15, 0], np.uint8)).tolist() == [0x21, 0x0F]
    assert C.unpack_int4(np.array([0x21, 0x0F], np.uint8)).tolist() == [1, 2, 15, 0]


def test_int4_round_trip_exact_on_representable_groups():
    rng = np.random.default_rng(3)
    for s_exp in (-6, -3, 0, 2):
        s = 2.0 ** s_exp
        q = rng.integers(0, 16, size=(20, 32))
        q[:, 0], q[:, 1] = 0, 15
        z = rng.integers(-40, 40, size=(20, 1)) * s
        x = (q * s + z).astype(np.float32)
        codes, ss, zz = C.quantize_group_int4(x)
        assert np.all(ss.astype(np.float64) == s)
        assert np.array_equal(zz.astype(np.float64), z[:, 0])
        assert np.array_equal(codes.astype(np.int64), q)


def test_int4_error_bound_and_degenerate_group():
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((500, 32)) * rng.uniform(0.1, 10, (500, 1))).astype(np.float32)
    codes, s, z = C.quantize_group_int4(x)
    rec = codes * s.astype(np.float64)[:, None] + z.astype(np.float64)[:, None]
    lo = x.min(axis=1).astype(np.float64)
    hi = x.max(axis=1).astype(np.float64)
    s64, z64 = s.astype(np.float64), z.astype(np.float64)
    # each element is within half a step of its code, up to the fp16 rounding of z and s
    bound = 0.5 * s64 + np.abs(lo - z64) + 16 * np.abs((hi - z64) / 15 - s64) + 1e-6
    assert np.all(np.abs(rec - x) <= bound[:, None])
    assert np.all(codes.max(axis=1) >= 14)         # the maximum lands on the top code
    c, s0, z0 = C.quantize_group_int4(np.full((1, 32), 1.25, np.float32))
    assert s0[0] == 0 and z0[0] == np.float16(1.25) and not c.any()


# ---------------------------------------------------------------- INT2 codec

def test_int2_pack_order_element_4k_plus_j_in_bits_2j():
    # byte 0: 1 | 2<<2 | 3<<4 | 0<<6 = 0x39; byte 1: 3 | 3<<2 | 0<<4 | 1<<6 = 0x4F
    assert C.pack_int2(np.array([1, 2, 3, 0, 3, 3, 0, 1], np.uint8)).tolist() == [0x39, 0x4F]
    assert C.unpack_int2(np.array([0x39, 0x4F], np.uint8)).tolist() == [1, 2, 3, 0, 3, 3, 0, 1]


def test_int2_round_trip_exact_on_representable_groups():
    rng = np.random.default_rng(13)
    for s_exp in (-6, -2, 0, 3):
        s = 2.0 ** s_exp
        q = rng.integers(0, 4, size=(20, 32))
        q[:, 0], q[:, 1] = 0, 3
        z = rng.integers(-40, 40, size=(20, 1)) * s
        x = (q * s + z).astype(np.float32)
        codes, ss, zz = C.quantize_group_int2(x)
        assert np.all(ss.astype(np.float64) == s)
        assert np.array_equal(zz.astype(np.float64), z[:, 0])
        assert np.array_equal(codes.astype(np.int64), q)


def test_int2_error_bound_and_degenerate_group():
    rng = np.random.default_rng(14)
    x = (rng.standard_normal((500, 32)) * rng.uniform(0.1, 10, (500, 1))).astype(np.float32)
    codes, s, z = C.quantize_group_int2(x)
    assert codes.max() <= 3
    rec = codes * s.astype(np.float64)[:, None] + z.astype(np.float64)[:, None]
    lo = x.min(axis=1).astype(np.float64)
    hi = x.max(axis=1).astype(np.float64)
    s64, z64 = s.astype(np.float64), z.astype(np.float64)
    bound = 0.5 * s64 + np.abs(lo - z64) + 4 * np.abs((hi - z64) / 3 - s64) + 1e-6
    assert np.all(np.abs(rec - x) <= bound[:, None])
    assert np.all(codes.max(axis=1) >= 2)
    c, s0, z0 = C.quantize_group_int2(np.full((1, 32), -3.5, np.float32))
    assert s0[0] == 0 and z0[0] == np.float16(-3.5) and not c.any()


def test_int2_codes_against_a_torch_float32_pipeline():
    """torch's IEEE float32 ops (no float64 emulation) give the same codes,
    scales and zero points inside fp16's range."""
    rng = np.random.default_rng(15)
    x = (rng.standard_normal((2000, 32)) * rng.uniform(0.01, 100, (2000, 1))).astype(np.float32)
    x[::7, 5:9] = np.floor(x[::7, 5:9]) + 0.5
    codes, s, z = C.quantize_group_int2(x)
    t = torch.from_numpy(x)
    tz = t.min(dim=1).values.to(torch.float16)
    ts = ((t.max(dim=1).values - tz.float()) / 3.0).to(torch.float16)
    y = (t - tz.float()[:, None]) / torch.where(ts > 0, ts, torch.ones_like(ts)).float()[:, None]
    tq = torch.clamp(torch.round(y), 0, 3)
    tq = torch.where((ts > 0)[:, None], tq, torch.zeros_like(tq))
    assert np.array_equal(z, tz.numpy()) and np.array_equal(s, ts.numpy())
    assert np.array_equal(codes.astype(np.int64), tq.numpy().astype(np.int64))


def test_int4_codes_against_a_torch_float32_pipeline():
    """The INT4 encoder pinned on its own: torch's IEEE float32 ops (no float64
    emulation) give the same codes, scales and zero points inside fp16's
    range, including values on exact half-integer quotients."""
    rng = np.random.default_rng(16)
    x = (rng.standard_normal((3000, 32)) * rng.uniform(0.01, 300, (3000, 1))).astype(np.float32)
    x[::5, 3:11] = np.floor(x[::5, 3:11]) + 0.5
    x[::11] = np.float32(2.0 ** -3) * rng.integers(-60, 60, (len(x[::11]), 32)).astype(np.float32)
    codes, s, z = C.quantize_group_int4(x)
    t = torch.from_numpy(x)
    tz = t.min(dim=1).values.to(torch.float16)
    ts = ((t.max(dim=1).values - tz.float()) / 15.0).to(torch.float16)
    y = (t - tz.float()[:, None]) / torch.where(ts > 0, ts, torch.ones_like(ts)).float()[:, None]
    tq = torch.clamp(torch.round(y), 0, 15)
    tq = torch.where((ts > 0)[:, None], tq, torch.zeros_like(tq))
    assert np.array_equal(z, tz.numpy()) and np.array_equal(s, ts.numpy())
    assert np.array_equal(codes.astype(np.int64), tq.numpy().astype(np.int64))


def _sat_groups():
    """bf16-representable groups whose zero point or scale leaves fp16's range."""
    g = np.zeros((4, 32), np.float32)
    g[0] = np.linspace(-2.0 ** 17, 2.0 ** 20, 32)            # min and span beyond 65504
    g[0, 7] = 65504.0 * 3.5 - 65504.0                          # (x - z) / s = 3.5 when s saturates
    g[1] = np.linspace(0.0, 2.0 ** 20, 32)                     # span only: z = 0, s saturates
    g[2] = -2.0 ** 17 + np.arange(32, dtype=np.float32) * 64.0  # every value below -65504
    g[3] = np.linspace(-2.0 ** 16, 2.0 ** 16, 32)              # -65536 .. 65536
    return C.round_to_bf16(g).astype(np.float32)


@pytest.mark.parametrize("top", [15, 3, 1])
def test_affine_encoder_saturates_zero_point_and_scale_at_65504(top):
    """fp16_sat clips to +-65504 (torch's half cast would give inf there).
    Closed form per group: z = max(lo, -65504) rounded to fp16, s =
    min((hi - z) / top, 65504); codes from Python float division."""
    x = _sat_groups()
    codes, s, z = C._quantize_group_affine(x, top)
    assert np.all(np.isfinite(z.astype(np.float64))) and np.all(np.isfinite(s.astype(np.float64)))
    assert z[0] == -65504 and z[2] == -65504 and z[1] == 0 and z[3] == -65504
    assert s[0] == 65504 and s[1] == 65504
    # all values below the saturated zero point: hi - z < 0, so s < 0 and every code is 0
    assert s[2] < 0 and not codes[2].any()
    for gi in (0, 1, 3):
        zz, ss = float(z[gi]), float(s[gi])
        for e in range(32):
            xv = float(x[gi, e])
            num = float(np.float32(xv - zz))
            want = min(max(round(float(np.float32(num / ss))), 0), top)   # round(): half to even
            assert codes[gi, e] == want, (gi, e, xv)
    if top == 15:
        assert codes[0, 7] == 4                                 # 3.5 rounds to even
    # group 3: z saturates (lo = -65536); (65536 + 65504) / top is an fp16 value
    # for top 15 and 3, and saturates for top 1
    assert float(s[3]) == min((65536.0 + 65504.0) / top, 65504.0)


# ---------------------------------------------------------------- 1-bit codec

def test_int1_pack_order_element_8k_plus_j_in_bit_j():
    # byte 0: elements 0..7 = 1,0,1,1,0,0,0,1 -> 0b10001101 = 0x8D; byte 1: 0,1,0,0,0,0,1,0 -> 0x42
    codes = np.array([1, 0, 1, 1, 0, 0, 0, 1, 0, 1, 0, 0, 0, 0, 1, 0], np.uint8)
    assert C.pack_int1(codes).tolist() == [0x8D, 0x42]
    assert C.unpack_int1(np.array([0x8D, 0x42], np.uint8)).tolist() == codes.tolist()


def test_int1_round_trip_exact_on_representable_groups():
    """Groups of exactly two values z and z + s (s a power of two, z a
    multiple of s): codes are the membership bits, scale and zero exact."""
    rng = np.random.default_rng(23)
    for s_exp in (-7, -1, 0, 4):
        s = 2.0 ** s_exp
        q = rng.integers(0, 2, size=(30, 32))
        q[:, 0], q[:, 1] = 0, 1
        z = rng.integers(-50, 50, size=(30, 1)) * s
        x = (q * s + z).astype(np.float32)
        codes, ss, zz = C.quantize_group_int1(x)
        assert np.all(ss.astype(np.float64) == s)
        assert np.array_equal(zz.astype(np.float64), z[:, 0])
        assert np.array_equal(codes.astype(np.int64), q)


def test_int1_error_bound_and_degenerate_group():
    """Each value lands on the nearer of z and z + s (s = max - min up to fp16
    rounding): |x - rec| <= s / 2 plus the fp16 rounding of z and s; a group of
    equal values has s = 0, codes 0, and reconstructs to z."""
    rng = np.random.default_rng(24)
    x = (rng.standard_normal((500, 32)) * rng.uniform(0.1, 10, (500, 1))).astype(np.float32)
    codes, s, z = C.quantize_group_int1(x)
    assert codes.max() <= 1
    rec = codes * s.astype(np.float64)[:, None] + z.astype(np.float64)[:, None]
    lo = x.min(axis=1).astype(np.float64)
    hi = x.max(axis=1).astype(np.float64)
    s64, z64 = s.astype(np.float64), z.astype(np.float64)
    bound = 0.5 * s64 + np.abs(lo - z64) + 2 * np.abs((hi - z64) - s64) + 1e-6
    assert np.all(np.abs(rec - x) <= bound[:, None])
    assert np.all(codes[np.arange(500), x.argmax(axis=1)] == 1)   # the maximum takes the top code
    assert np.all(codes[np.arange(500), x.argmin(axis=1)] == 0)
    c, s0, z0 = C.quantize_group_int1(np.full((1, 32), 7.25, np.float32))
    assert s0[0] == 0 and z0[0] == np.float16(7.25) and not c.any()


def test_int1_codes_against_a_torch_float32_pipeline():
    """torch's IEEE float32 ops give the same codes, scales and zero points
    inside fp16's range, including values exactly half way between z and z+s."""
    rng = np.random.default_rng(25)
    x = (rng.standard_normal((2000, 32)) * rng.uniform(0.01, 100, (2000, 1))).astype(np.float32)
    x[::9] = np.float32(0.25) * rng.integers(-8, 8, (len(x[::9]), 32)).astype(np.float32)
    codes, s, z = C.quantize_group_int1(x)
    t = torch.from_numpy(x)
    tz = t.min(dim=1).values.to(torch.float16)
    ts = (t.max(dim=1).values - tz.float()).to(torch.float16)
    y = (t - tz.float()[:, None]) / torch.where(ts > 0, ts, torch.ones_like(ts)).float()[:, None]
    tq = torch.clamp(torch.round(y), 0, 1)
    tq = torch.where((ts > 0)[:, None], tq, torch.zeros_like(tq))
    assert np.array_equal(z, tz.numpy()) and np.array_equal(s, ts.numpy())
    assert np.array_equal(codes.astype(np.int64), tq.numpy().astype(np.int64))


# ---------------------------------------------------------------- bf16 rounding

def test_round_to_bf16_matches_torch_for_float32_inputs():
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-40, 38, 20000),
                        np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 2.0 ** -130])]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(C.f64_to_bf16_bits(x.astype(np.float64)), ref)


# ---------------------------------------------------------------- quantize_pages

def _src_pool(n, hkv, P, D, dtype, seed):
    t = W.normal((n, 2, hkv, P, D), dtype, seed)
    return W.to_bits(t)


@pytest.mark.parametrize("codec", [C.CODEC_FP8_E4M3, C.CODEC_INT8, C.CODEC_INT4_G32, C.CODEC_INT2_G32,
                                   C.CODEC_INT1_G32])
def test_quantize_pages_units_independent_and_ckey(codec):
    hkv, P, D = 2, 16, 64
    src = _src_pool(3, hkv, P, D, C.CODEC_BF16, 11)
    codes, meta = C.alloc_pool(codec, 5, hkv, P, D)
    ck = C.quantize_pages(src, C.CODEC_BF16, [2, 0], codec, codes, meta, [4, 1],
                          valid_tokens=[16, 9], want_ckey=True)
    # slot 4 <- src 2 (all tokens); slot 1 <- src 0 (9 valid tokens); others untouched
    assert not codes[0].any() and not codes[2].any() and not codes[3].any()
    x = C.bf16_bits_to_f64(src[2, 1, 1]).astype(np.float32)
    if codec == C.CODEC_FP8_E4M3:
        c, s = C.quantize_unit_fp8(x)
        assert np.array_equal(codes[4, 1, 1], c) and meta[4, 1, 1] == s
    assert not codes[1, :, :, 9:].any()
    # compressed key = bf16(mean of the stored keys), via torch in float64
    k = torch.from_numpy(C.dequant_page(codec, codes, meta, 1, 0, 1)[:9])
    want = k.mean(dim=0).to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = ck[1, 1]
    diff = np.abs(C.bf16_bits_to_f64(got) - C.bf16_bits_to_f64(want))
    ulp = np.abs(C.bf16_bits_to_f64(want)) * 2.0 ** -7 + 1e-38
    assert np.all(diff <= ulp)


def test_dequant_independent_of_oracle_helpers():
    """Dequantise FP8 / INT8 / INT4 / INT2 / INT1 with torch (library view of the codes)."""
    hkv, P, D = 1, 16, 64
    src = _src_pool(1, hkv, P, D, C.CODEC_FP16, 12)
    for codec in (C.CODEC_FP8_E4M3, C.CODEC_INT8, C.CODEC_INT4_G32, C.CODEC_INT2_G32, C.CODEC_INT1_G32):
        codes, meta = C.alloc_pool(codec, 1, hkv, P, D)
        C.quantize_pages(src, C.CODEC_FP16, [0], codec, codes, meta, [0])
        got = C.dequant_page(codec, codes, meta, 0, 1, 0)
        tc = torch.from_numpy(codes[0, 1, 0].copy())
        if codec == C.CODEC_FP8_E4M3:
            ref = tc.view(torch.float8_e4m3fn).double() * float(meta[0, 1, 0])
        elif codec == C.CODEC_INT8:
            ref = tc.view(torch.int8).double() * float(meta[0, 1, 0])
        else:
            if codec == C.CODEC_INT4_G32:
                q = torch.stack([(tc & 0xF).double(), (tc >> 4).double()], dim=-1).reshape(P, D)
            elif codec == C.CODEC_INT2_G32:   # four 2-bit codes per byte, lowest bits first
                q = torch.stack([((tc >> (2 * j)) & 3).double() for j in range(4)], dim=-1).reshape(P, D)
            else:   # eight 1-bit codes per byte, lowest bit first
                q = torch.stack([((tc >> j) & 1).double() for j in range(8)], dim=-1).reshape(P, D)
            sz = torch.from_numpy(meta[0, 1, 0].astype(np.float64))   # [P][D/32][2]
            ref = (q.reshape(P, D // 32, 32) * sz[..., :1] + sz[..., 1:]).reshape(P, D)
        assert np.array_equal(got, ref.numpy())
        x = C.f16_bits_to_f64(src[0, 1, 0])
        # INT2 keeps 4 levels per group, INT1 two: coarser (but bounded) reconstructions
        frac = {C.CODEC_INT2_G32: 0.4, C.CODEC_INT1_G32: 1.0}.get(codec, 0.1)
        assert np.max(np.abs(got - x)) <= frac * np.max(np.abs(x))


# ---------------------------------------------------------------- attention

def _torch_attention(q, K, V, scale):
    s = scale * (torch.from_numpy(K) @ torch.from_numpy(q))
    w = torch.softmax(s, dim=0)
    return (w @ torch.from_numpy(V)).numpy(), float(torch.logsumexp(s, 0)) / math.log(2)


def _fp16_paged_case(B=2, Hkv=2, G=3, D=32, P=16, lens=(37, 64), seed=21):
    Hq = Hkv * G
    q = C.f16_bits_to_f64(W.to_bits(W.normal((B, Hq, D), C.CODEC_FP16, seed)))
    maxp = max((L + P - 1) // P for L in lens)
    table, n_slots = W.paged_block_table(lens, P, maxp, seed + 1)
    pool = W.to_bits(W.normal((n_slots, 2, Hkv, P, D), C.CODEC_FP16, seed + 2))
    codecs = np.zeros((B, maxp), np.int64)
    return q, pool, table, codecs, np.array(lens), Hkv, P


def test_paged_fp16_equals_dense_softmax_via_torch():
    q, pool, table, codecs, lens, Hkv, P = _fp16_paged_case()
    o, lse2, bad = A.paged_decode(q, Hkv, P, {0: (pool, None)}, codecs, table, lens, 0.125)
    assert bad == 0
    B, Hq, D = q.shape
    G = Hq // Hkv
    for b in range(B):
        L = lens[b]
        for h in range(Hkv):
            rows = [C.f16_bits_to_f64(pool[table[b, t // P], :, h, t % P]) for t in range(L)]
            K = np.stack([r[0] for r in rows])
            V = np.stack([r[1] for r in rows])
            for g in range(G):
                ro, rl = _torch_attention(q[b, h * G + g], K, V, 0.125)
                assert np.allclose(o[b, h * G + g], ro, atol=1e-12, rtol=0)
                assert abs(lse2[b, h * G + g] - rl) < 1e-12


def test_paged_g1_equals_torch_sdpa():
    q, pool, table, codecs, lens, Hkv, P = _fp16_paged_case(G=1, lens=(48, 48))
    o, _, _ = A.paged_decode(q, Hkv, P, {0: (pool, None)}, codecs, table, lens, 0.2)
    for b in range(2):
        rows = [C.f16_bits_to_f64(pool[table[b, t // P], :, :, t % P]) for t in range(48)]
        K = torch.from_numpy(np.stack([r[0] for r in rows])).permute(1, 0, 2)  # [H][n][D]
        V = torch.from_numpy(np.stack([r[1] for r in rows])).permute(1, 0, 2)
        Q = torch.from_numpy(q[b])[:, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, scale=0.2)[:, 0]
        assert np.allclose(o[b], ref.numpy(), atol=1e-12, rtol=0)


def test_block_table_permutation_invariance_bit_identical():
    q, pool, table, codecs, lens, Hkv, P = _fp16_paged_case()
    o1, l1, _ = A.paged_decode(q, Hkv, P, {0: (pool, None)}, codecs, table, lens, 0.125)
    perm = W.permutation(pool.shape[0], 99)
    pool2 = np.empty_like(pool)
    pool2[perm] = pool
    table2 = perm[table].astype(np.int32)
    o2, l2, _ = A.paged_decode(q, Hkv, P, {0: (pool2, None)}, codecs, table2, lens, 0.125)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_special_cases_one_token_and_equal_scores():
    D = 16
    rng = np.random.default_rng(6)
    v = rng.standard_normal((1, D))
    k = rng.standard_normal((1, D))
    q = rng.standard_normal(D)
    o, l = A.softmax_attention(q, k, v, 0.3)
    assert np.array_equal(o, v[0]) and abs(l - 0.3 * (k[0] @ q) / math.log(2)) < 1e-12
    V = rng.standard_normal((7, D))
    o, l = A.softmax_attention(np.zeros(D), rng.standard_normal((7, D)), V, 0.3)
    assert np.allclose(o, V.mean(axis=0), atol=1e-14) and abs(l - math.log2(7)) < 1e-12
    # query orthogonal to every key -> uniform average
    K = np.zeros((5, D)); K[:, 0] = rng.standard_normal(5)
    qo = np.zeros(D); qo[1] = 3.0
    o, _ = A.softmax_attention(qo, K, V[:5], 1.0)
    assert np.allclose(o, V[:5].mean(axis=0), atol=1e-14)
    o, l = A.softmax_attention(q, np.zeros((0, D)), np.zeros((0, D)), 1.0)
    assert l == -math.inf and not o.any()


def test_mixed_codec_decode_equals_torch_dense_on_dequantised_pages():
    Hkv, G, D, P = 2, 4, 64, 16
    lens = [80]
    q = C.f16_bits_to_f64(W.to_bits(W.normal((1, Hkv * G, D), C.CODEC_FP16, 31)))
    pools, page_codec = {}, np.array([[6, 5, 4, 3, 2, 0, 2]])
    table = np.array([[0, 0, 0, 0, 1, 0, 0]], np.int32)
    lens = [112]
    src = W.to_bits(W.normal((7, 2, Hkv, P, D), C.CODEC_FP16, 32))
    for codec in (0, 2, 3, 4, 5, 6):
        pools[codec] = C.alloc_pool(codec, 2, Hkv, P, D)
    for p in range(7):
        c = int(page_codec[0, p])
        C.quantize_pages(src, C.CODEC_FP16, [p], c, pools[c][0], pools[c][1], [int(table[0, p])])
    o, _, bad = A.paged_decode(q, Hkv, P, pools, page_codec, table, np.array(lens), 0.125)
    assert bad == 0
    # independent dequantisation with torch views of the stored codes
    for h in range(Hkv):
        Ks, Vs = [], []
        for p in range(7):
            c, slot = int(page_codec[0, p]), int(table[0, p])
            codes, meta = pools[c]
            for kv, acc in ((0, Ks), (1, Vs)):
                t = torch.from_numpy(codes[slot, kv, h].copy())
                if c == 0:
                    acc.append(t.view(torch.float16).double())
                elif c == 2:
                    acc.append(t.view(torch.float8_e4m3fn).double() * float(meta[slot, kv, h]))
                elif c == 3:
                    acc.append(t.view(torch.int8).double() * float(meta[slot, kv, h]))
                else:
                    if c == 4:
                        qn = torch.stack([(t & 0xF).double(), (t >> 4).double()], -1).reshape(P, D)
                    elif c == 5:
                        qn = torch.stack([((t >> (2 * j)) & 3).double() for j in range(4)], -1).reshape(P, D)
                    else:
                        qn = torch.stack([((t >> j) & 1).double() for j in range(8)], -1).reshape(P, D)
                    sz = torch.from_numpy(meta[slot, kv, h].astype(np.float64))
                    acc.append((qn.reshape(P, D // 32, 32) * sz[..., :1] + sz[..., 1:]).reshape(P, D))
        K, V = torch.cat(Ks).numpy(), torch.cat(Vs).numpy()
        for g in range(G):
            ro, _ = _torch_attention(q[0, h * G + g], K, V, 0.125)
            assert np.allclose(o[0, h * G + g], ro, atol=1e-12, rtol=0)


def test_bad_slot_is_skipped_and_counted():
    q, pool, table, codecs, lens, Hkv, P = _fp16_paged_case(lens=(64, 64))
    t2 = table.copy()
    t2[0, 1] = pool.shape[0] + 5
    o, _, bad = A.paged_decode(q, Hkv, P, {0: (pool, None)}, codecs, t2, lens, 0.125)
    assert bad == Hkv
    # same as attending pages 0, 2, 3 only (selection list without page 1)
    sel = np.zeros((2, Hkv, 4), np.int32); cnt = np.zeros((2, Hkv), np.int32)
    sel[0, :, :3] = [0, 2, 3]; cnt[0] = 3
    sel[1, :, :4] = [0, 1, 2, 3]; cnt[1] = 4
    o2, _, _ = A.paged_decode(q, Hkv, P, {0: (pool, None)}, codecs, table, lens, 0.125,
                              sel_pages=sel, sel_count=cnt, sel_width=4)
    assert np.allclose(o, o2, atol=1e-13)


# ---------------------------------------------------------------- sliding window + sinks

def _window_set(L, W, S):
    """Visible positions built from plain ranges (independent of the oracle)."""
    if W <= 0:
        return set(range(L))
    return set(range(max(0, L - W), L)) | set(range(min(S, L)))


@pytest.mark.parametrize("L,W,S", [(0, 5, 2), (1, 1, 0), (37, 5, 0), (37, 5, 4), (37, 40, 4), (37, 33, 4),
                                   (37, 34, 4), (37, 1, 36), (37, 1, 37), (64, 16, 16), (64, 17, 15), (20, 3, 100)])
def test_window_positions_brute_force_and_count(L, W, S):
    vis = A.visible_positions(L, W, S)
    assert set(np.nonzero(vis)[0].tolist()) == _window_set(L, W, S)
    # closed form: the window, plus the sinks that lie before it
    assert int(vis.sum()) == min(L, W) + min(S, max(0, L - W))


def test_window_decode_equals_torch_on_gathered_positions():
    lens = (37, 64, 129)
    q, pool, table, codecs, lens, Hkv, P = _fp16_paged_case(B=3, lens=lens, seed=31)
    B, Hq, D = q.shape
    G = Hq // Hkv
    for W_, S_ in [(5, 0), (5, 4), (20, 3), (16, 16), (1, 33), (200, 4)]:
        o, lse2, bad = A.paged_decode(q, Hkv, P, {0: (pool, None)}, codecs, table, lens, 0.125,
                                      window=W_, sinks=S_)
        assert bad == 0
        for b in range(B):
            pos = sorted(_window_set(int(lens[b]), W_, S_))
            for h in range(Hkv):
                rows = [C.f16_bits_to_f64(pool[table[b, t // P], :, h, t % P]) for t in pos]
                K = np.stack([r[0] for r in rows])
                V = np.stack([r[1] for r in rows])
                for g in range(G):
                    ro, rl = _torch_attention(q[b, h * G + g], K, V, 0.125)
                    assert np.allclose(o[b, h * G + g], ro, atol=1e-12, rtol=0)
                    assert abs(lse2[b, h * G + g] - rl) < 1e-12


def test_window_zero_query_gives_log2_of_the_visible_count():
    q, pool, table, codecs, lens, Hkv, P = _fp16_paged_case(B=2, lens=(37, 64), seed=41)
    q = np.zeros_like(q)
    for W_, S_ in [(5, 4), (33, 4), (34, 4), (1, 0), (64, 3)]:
        _, lse2, _ = A.paged_decode(q, Hkv, P, {0: (pool, None)}, codecs, table, lens, 0.125,
                                    window=W_, sinks=S_)
        for b, L in enumerate(lens):
            n = min(int(L), W_) + min(S_, max(0, int(L) - W_))
            assert np.all(np.abs(lse2[b] - math.log2(n)) < 1e-12)


def test_window_wider_than_the_sequence_is_full_attention():
    q, pool, table, codecs, lens, Hkv, P = _fp16_paged_case(seed=51)
    o0, l0, _ = A.paged_decode(q, Hkv, P, {0: (pool, None)}, codecs, table, lens, 0.125)
    o1, l1, _ = A.paged_decode(q, Hkv, P, {0: (pool, None)}, codecs, table, lens, 0.125,
                               window=int(max(lens)), sinks=3)
    o2, l2, _ = A.paged_decode(q, Hkv, P, {0: (pool, None)}, codecs, table, lens, 0.125,
                               window=0, sinks=7)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)
    assert np.array_equal(o0, o2) and np.array_equal(l0, l2)


def test_window_bad_slot_counted_only_on_pages_it_reads():
    q, pool, table, codecs, lens, Hkv, P = _fp16_paged_case(lens=(64, 64), seed=61)
    t2 = table.copy()
    t2[0, 1] = pool.shape[0] + 5          # page 1 = positions 16..31
    _, _, bad = A.paged_decode(q, Hkv, P, {0: (pool, None)}, codecs, t2, lens, 0.125, window=20, sinks=4)
    assert bad == 0                       # visible: 0..3 and 44..63
    _, _, bad = A.paged_decode(q, Hkv, P, {0: (pool, None)}, codecs, t2, lens, 0.125, window=40, sinks=4)
    assert bad == Hkv                     # 24..63 reaches into page 1: one count per KV head


# ---------------------------------------------------------------- fold

def test_fold_of_any_partition_equals_single_pass():
    rng = np.random.default_rng(7)
    D, n = 8, 40
    q = rng.standard_normal(D)
    K = rng.standard_normal((n, D)) * 2
    V = rng.standard_normal((n, D))
    o_ref, l_ref = A.softmax_attention(q, K, V, 0.5)
    for trial in range(20):
        cuts = sorted(rng.choice(np.arange(0, n + 1), size=rng.integers(1, 6)))
        bounds = [0] + list(cuts) + [n]      # may contain empty and one-token parts
        order = rng.permutation(len(bounds) - 1)
        acc_o, acc_l = np.zeros((1, D)), np.full(1, -math.inf)
        for i in order:
            a, b = bounds[i], bounds[i + 1]
            po, pl = A.softmax_attention(q, K[a:b], V[a:b], 0.5)
            acc_o, acc_l = A.fold_lse(acc_o, acc_l, po[None], np.array([pl]))
        assert np.allclose(acc_o[0], o_ref, atol=1e-12) and abs(acc_l[0] - l_ref) < 1e-12


def test_fold_identity_on_empty():
    o = np.array([[1.0, 2.0]])
    r, l = A.fold_lse(o, np.array([3.0]), np.zeros((1, 2)), np.array([-math.inf]))
    assert np.array_equal(r, o) and l[0] == 3.0
    r, l = A.fold_lse(np.zeros((1, 2)), np.array([-math.inf]), o, np.array([3.0]))
    assert np.array_equal(r, o) and l[0] == 3.0


# ---------------------------------------------------------------- windows

def test_window_causality_brute_force_and_fold_of_windows():
    rng = np.random.default_rng(8)
    Hq, Hkv, D, nq, ctx = 4, 2, 8, 6, 20
    q = rng.standard_normal((Hq, nq, D))
    k = rng.standard_normal((Hkv, ctx + nq, D))
    v = rng.standard_normal((Hkv, ctx + nq, D))
    q_pos0 = ctx
    full_o, full_l = A.window_attention(q, k, v, 0, q_pos0, 0.4)
    for hq in range(Hq):
        h = hq // 2
        for i in range(nq):
            vis = [j for j in range(ctx + nq) if j <= q_pos0 + i]
            s = np.array([0.4 * q[hq, i] @ k[h, j] for j in vis])
            w = np.exp(s - s.max())
            assert np.allclose(full_o[hq, i], (w @ v[h, vis]) / w.sum(), atol=1e-12)
    acc_o = np.zeros((Hq, nq, D)); acc_l = np.full((Hq, nq), -math.inf)
    for w0, w1 in ((0, 7), (7, 20), (20, 26)):
        po, pl = A.window_attention(q, k[:, w0:w1], v[:, w0:w1], w0, q_pos0, 0.4)
        acc_o, acc_l = A.fold_lse(acc_o, acc_l, po, pl)
    assert np.allclose(acc_o, full_o, atol=1e-12) and np.allclose(acc_l, full_l, atol=1e-12)


# ---------------------------------------------------------------- paged windows (staged prefill)

def _torch_dequant(codec, codes, meta, slot, kv, h, P, D):
    """Dequantise one unit with torch views of the stored codes (independent of the oracle)."""
    t = torch.from_numpy(codes[slot, kv, h].copy())
    if codec == C.CODEC_FP16:
        return t.view(torch.float16).double()
    if codec == C.CODEC_FP8_E4M3:
        return t.view(torch.float8_e4m3fn).double() * float(meta[slot, kv, h])
    if codec == C.CODEC_INT8:
        return t.view(torch.int8).double() * float(meta[slot, kv, h])
    if codec == C.CODEC_INT4_G32:
        q = torch.stack([(t & 0xF).double(), (t >> 4).double()], -1).reshape(P, D)
    else:
        q = torch.stack([((t >> (2 * j)) & 3).double() for j in range(4)], -1).reshape(P, D)
    sz = torch.from_numpy(meta[slot, kv, h].astype(np.float64))
    return (q.reshape(P, D // 32, 32) * sz[..., :1] + sz[..., 1:]).reshape(P, D)


def _mixed_paged_cache(Hkv, D, P, n_pages, seed, codecs=(5, 4, 3, 2, 0)):
    src = W.to_bits(W.normal((n_pages, 2, Hkv, P, D), C.CODEC_FP16, seed))
    page_codec = np.array([[codecs[p % len(codecs)] for p in range(n_pages)]])
    perm = W.permutation(n_pages, seed + 1)
    table = np.zeros((1, n_pages), np.int32)
    pools = {c: C.alloc_pool(c, n_pages, Hkv, P, D) for c in set(codecs)}
    for p in range(n_pages):
        c = int(page_codec[0, p])
        table[0, p] = perm[p]
        C.quantize_pages(src, C.CODEC_FP16, [p], c, pools[c][0], pools[c][1], [int(perm[p])])
    return pools, page_codec, table


def test_gather_window_is_a_plain_gather_and_table_invariant():
    Hkv, D, P, n = 2, 32, 16, 6
    pools, pc, table = _mixed_paged_cache(Hkv, D, P, n, 70, codecs=(0,))
    codes = pools[0][0]
    K, V = A.gather_window(Hkv, P, pools, pc, table, 0, 13, 50)
    for j, p in enumerate(range(13, 63)):
        for h in range(Hkv):
            row = torch.from_numpy(codes[table[0, p // P], :, h, p % P].copy()).view(torch.float16).double()
            assert np.array_equal(K[h, j], row[0].numpy()) and np.array_equal(V[h, j], row[1].numpy())
    # the same pages under another slot permutation give the same window
    perm = W.permutation(codes.shape[0], 71)
    codes2 = np.empty_like(codes)
    codes2[perm] = codes
    K2, V2 = A.gather_window(Hkv, P, {0: (codes2, None)}, pc, perm[table].astype(np.int32), 0, 13, 50)
    assert np.array_equal(K, K2) and np.array_equal(V, V2)


def test_paged_window_attention_over_five_tiers_equals_torch_causal():
    Hkv, G, D, P, n = 2, 3, 64, 16, 10
    pools, pc, table = _mixed_paged_cache(Hkv, D, P, n, 72)
    nq, q_pos0, w0, wl = 5, 150, 21, 134            # window 21..154, crossing pages mid-page
    q = C.f16_bits_to_f64(W.to_bits(W.normal((Hkv * G, nq, D), C.CODEC_FP16, 73)))
    o, lse2 = A.paged_window_attention(q, Hkv, P, pools, pc, table, 0, w0, wl, q_pos0, 0.125)
    for h in range(Hkv):
        rows = []
        for p in range(w0, w0 + wl):
            c, slot = int(pc[0, p // P]), int(table[0, p // P])
            rows.append((_torch_dequant(c, *pools[c], slot, 0, h, P, D)[p % P],
                         _torch_dequant(c, *pools[c], slot, 1, h, P, D)[p % P]))
        K = torch.stack([r[0] for r in rows]).numpy()
        V = torch.stack([r[1] for r in rows]).numpy()
        for g in range(G):
            for i in range(nq):
                n_vis = q_pos0 + i - w0 + 1            # keys at positions <= q_pos0 + i
                ro, rl = _torch_attention(q[h * G + g, i], K[:n_vis], V[:n_vis], 0.125)
                assert np.allclose(o[h * G + g, i], ro, atol=1e-12, rtol=0)
                assert abs(lse2[h * G + g, i] - rl) < 1e-12


def test_fold_of_paged_windows_equals_one_window():
    Hkv, G, D, P, n = 2, 2, 32, 16, 8
    pools, pc, table = _mixed_paged_cache(Hkv, D, P, n, 74)
    nq, q_pos0 = 4, 124
    q = C.f16_bits_to_f64(W.to_bits(W.normal((Hkv * G, nq, D), C.CODEC_FP16, 75)))
    full_o, full_l = A.paged_window_attention(q, Hkv, P, pools, pc, table, 0, 0, 128, q_pos0, 0.2)
    acc_o = np.zeros_like(full_o)
    acc_l = np.full_like(full_l, -math.inf)
    for w0, w1 in ((0, 37), (37, 37), (37, 100), (100, 128)):
        po, pl = A.paged_window_attention(q, Hkv, P, pools, pc, table, 0, w0, w1 - w0, q_pos0, 0.2)
        acc_o, acc_l = A.fold_lse(acc_o, acc_l, po, pl)
    assert np.allclose(acc_o, full_o, atol=1e-12) and np.allclose(acc_l, full_l, atol=1e-12)


def test_staging_moves_less_with_the_pages_numbers():
    """Rows reading their selected pages in place (2,051 tokens each, the
    host-placement comment) against staging a ~985k-token cache once: the
    decision turns where the rows' reads pass the cache size."""
    g = json.load(open(GOLDEN))["selection_budget"]
    per_row = g["tokens_per_query_printed"]
    cache = 985_000
    assert A.staging_moves_less([per_row] * 1024, cache)           # 2.1 M tokens read in place
    assert not A.staging_moves_less([per_row] * 256, cache)        # 0.5 M
    n_turn = cache // per_row + 1                                   # first row count that reads more
    assert A.staging_moves_less([per_row] * n_turn, cache)
    assert not A.staging_moves_less([per_row] * (n_turn - 1), cache)
    assert not A.staging_moves_less([cache // 2, cache - cache // 2], cache)   # equal: in place


# ---------------------------------------------------------------- selection

def test_scores_equal_torch_einsum():
    rng = np.random.default_rng(9)
    B, Hkv, G, D, maxp = 2, 2, 3, 16, 9
    q = rng.standard_normal((B, Hkv * G, D))
    ck = C.f64_to_bf16_bits(rng.standard_normal((B, maxp, Hkv, D)))
    n = np.array([9, 5])
    s = S.compressed_key_scores(q, ck, n, Hkv)
    ckt = torch.from_numpy(C.bf16_bits_to_f64(ck))
    qt = torch.from_numpy(q).reshape(B, Hkv, G, D).sum(dim=2)
    ref = torch.einsum("bhd,bphd->bhp", qt, ckt).numpy()
    assert np.allclose(s[0], ref[0], atol=1e-12)
    assert np.allclose(s[1, :, :5], ref[1, :, :5], atol=1e-12) and np.all(np.isinf(s[1, :, 5:]))


def test_topk_brute_force_with_ties():
    rng = np.random.default_rng(10)
    for trial in range(30):
        n = int(rng.integers(1, 40))
        k = int(rng.integers(1, 12))
        # integer-valued keys force many exact ties
        ck = np.zeros((1, n, 1, 4))
        ck[0, :, 0, 0] = rng.integers(-3, 4, n)
        q = np.zeros((1, 1, 4)); q[0, 0, 0] = 1.0
        sel, cnt, drops = S.select_pages(q, C.f64_to_bf16_bits(ck), [n], 1, k, True, 2 * k + 8)
        score = ck[0, :, 0, 0]
        want = set()
        for p in range(n - 1):
            better = sum(1 for r in range(n - 1)
                         if score[r] > score[p] or (score[r] == score[p] and r < p))
            if better < k:
                want.add(p)
        want.add(n - 1)
        assert cnt[0, 0] == len(want) and drops == 0
        assert sel[0, 0, :cnt[0, 0]].tolist() == sorted(want)


def test_selection_width_overflow_counts_drops():
    q = np.ones((1, 1, 2))
    ck = C.f64_to_bf16_bits(np.arange(10, dtype=np.float64)[None, :, None, None] * np.ones((1, 10, 1, 2)))
    sel, cnt, drops = S.select_pages(q, ck, [10], 1, 5, True, 4)
    assert cnt[0, 0] == 4 and drops == 2
    assert sel[0, 0].tolist() == [6, 7, 8, 9]


def test_golden_selection_width_and_2051_tokens():
    g = json.load(open(GOLDEN))
    sw = g["selection_width"]
    assert 2 * sw["block_topk"] + 8 == sw["max_sel_pages"]
    bud = g["selection_budget"]
    P = bud["page_tokens"]
    top_k = bud["indexer_budget_tokens"] // P
    n_pages = 100
    seq_len = (n_pages - 1) * P + 3          # newest page holds 3 tokens
    rng = np.random.default_rng(12)
    q = rng.standard_normal((1, 1, 8))
    ck = C.f64_to_bf16_bits(rng.standard_normal((1, n_pages, 1, 8)))
    sel, cnt, _ = S.select_pages(q, ck, [n_pages], 1, top_k, True, sw["max_sel_pages"])
    toks = sum(min(P, seq_len - int(p) * P) for p in sel[0, 0, :cnt[0, 0]])
    assert toks == bud["tokens_per_query_printed"]


def test_golden_byte_accounting_of_the_32k_engine_example():
    g = json.load(open(GOLDEN))["direct_paged_engine_32k"]
    geo = g["geometry"]
    T = g["context_tokens"]
    fp16 = accounting.kv_bytes(accounting.FP16, T, geo["kv_heads"], geo["head_dim"],
                               T // geo["page_tokens"]) / 2 ** 20
    q40 = fp16 * g["q4_0_bits_per_element"] / 16.0
    # both printed figures carry the same fixed overhead above the K/V bytes
    assert abs((g["fp16_mib"] - fp16) - (g["q4_0_mib"] - q40)) < 0.01
    assert round(g["fp16_mib"] / g["q4_0_mib"], 1) == g["ratio_printed"]


def test_window_byte_accounting_matches_the_visible_positions():
    rng = np.random.default_rng(77)
    for _ in range(300):
        L = int(rng.integers(0, 3000))
        P = int(rng.choice([16, 64, 1024]))
        Wn = int(rng.integers(0, 4000))
        Sn = int(rng.integers(0, 70))
        vis = A.visible_positions(L, Wn, Sn)
        pages = {int(p) // P for p in np.nonzero(vis)[0]}
        assert accounting.window_visible(L, P, Wn, Sn) == (int(vis.sum()), len(pages))
