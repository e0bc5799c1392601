"""Codec tiers of the paged KV cache, written out step by step (oracle).

TEST INFRASTRUCTURE ONLY -- see the package docstring.

The tiers are the ones named on "ARGUS: Heterogeneous KV-cache memory
management" (summary paragraph and section "Direct paged attention": FP16,
FP8, INT8, INT4 pages) and on "feat(kvcache): host-RAM KV tier for
sparse-attention models", update 20f3b23 ("the pool stores e4m3 codes + fp32
scales; ... nothing gets re-quantized").  The pages do not spell the encoders
out; the readings taken here (all listed in the design notes) are:

* FP8 e4m3 (OCP FP8, bias 7, no infinities, S.1111.111 = NaN, max 448):
  per (page, KV head, K-or-V) unit, a = max|x|; scale = fp32(a / 448);
  code = e4m3_rne_satfinite(fp32(x / scale)); a == 0 -> scale 0, codes 0.
  Dequantised value = e4m3_value(code) * scale.
* INT8 symmetric: scale = fp32(a / 127); q = clamp(rint_even(fp32(x / scale)),
  -127, 127); a == 0 -> scale 0, codes 0.  Dequantised value = q * scale.
* INT4 with 32-element groups along head_dim ("unsigned_affine" in the
  pluggable-tier example on the ARGUS page): per token and group, lo/hi =
  min/max; z = fp16_sat(lo); s = fp16_sat(fp32(fp32(hi - z) / 15));
  q = s > 0 ? clamp(rint_even(fp32(fp32(x - z) / s)), 0, 15) : 0; two codes per
  byte, the even element in the low nibble.  Dequantised value = q * s + z.
* INT2 with 32-element groups: the same "unsigned_affine" encoder with
  bits = 2 (the pluggable-tier example registers
  NativeCodecSpec(kind="unsigned_affine", bits=2)), i.e. 3 in place of 15:
  s = fp16_sat(fp32(fp32(hi - z) / 3)), q = clamp(rint_even(...), 0, 3); four
  codes per byte, element 4k + j in bits 2j, 2j + 1 of byte k.
* 1-bit with 32-element groups (the summary's 1-bit tier): the same encoder
  with bits = 1, i.e. 1 in place of 15: s = fp16_sat(fp32(fp32(hi - z) / 1)) =
  fp16_sat(hi - z), q = clamp(rint_even(fp32(fp32(x - z) / s)), 0, 1); eight
  codes per byte, element 8k + j in bit j of byte k.

Each "fp32(...)" is one IEEE single-precision operation with
round-to-nearest-even, emulated as the float64 operation followed by a cast
to float32 (exact for one +, -, * or / of float32 operands, since
53 >= 2*24 + 2).

Layouts (shared by definition with the C ABI, not by code):
  codes  [n_slots][2 (K, V)][Hkv][P][row]  row = D halves (FP16/BF16),
         D bytes (FP8/INT8), D/2 bytes (INT4), D/4 bytes (INT2), D/8 bytes (INT1)
  meta   FP8/INT8: float32 [n_slots][2][Hkv];
         INT4 / INT2 / INT1: float16 [n_slots][2][Hkv][P][D/32][2] = (scale, zero)
"""

import math

import numpy as np

CODEC_FP16 = 0
CODEC_BF16 = 1
CODEC_FP8_E4M3 = 2
CODEC_INT8 = 3
CODEC_INT4_G32 = 4
CODEC_INT2_G32 = 5
CODEC_INT1_G32 = 6

F16_MAX = 65504.0


# --------------------------------------------------------------------------
# 16-bit float helpers (values carried as uint16 bit patterns)
# --------------------------------------------------------------------------

def f16_bits_to_f64(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def bf16_bits_to_f64(bits):
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def bits_to_f64(bits, dtype):
    if dtype == CODEC_FP16:
        return f16_bits_to_f64(bits)
    if dtype == CODEC_BF16:
        return bf16_bits_to_f64(bits)
    raise ValueError("16-bit dtype expected")


def round_to_bf16(x):
    """Round float64 values to the nearest bfloat16 value, ties to even.

    bfloat16 keeps 8 significant bits, exponent range of float32
    (normal down to 2^-126, subnormal quantum 2^-133).
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    nz = (x != 0) & np.isfinite(x)
    _, e = np.frexp(x[nz])                     # |x| = m * 2^e, 0.5 <= m < 1
    quantum_exp = np.maximum(e - 8, -133)
    y = np.rint(np.ldexp(x[nz], -quantum_exp))  # rint: half to even
    r = np.ldexp(y, quantum_exp)
    bf16_max = (2.0 - 2.0 ** -7) * 2.0 ** 127
    r = np.where(np.abs(r) > bf16_max, np.copysign(np.inf, r), r)
    out[nz] = r
    out[~np.isfinite(x)] = x[~np.isfinite(x)]
    return out


def f64_to_bf16_bits(x):
    r = round_to_bf16(x).astype(np.float32)
    return (r.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def fp16_rne_sat(x32):
    """fp32 -> fp16, round to nearest even, saturating to +-65504."""
    x32 = np.asarray(x32, dtype=np.float32)
    return np.clip(x32, np.float32(-F16_MAX), np.float32(F16_MAX)).astype(np.float16)


def _f32(x):
    return np.asarray(x, dtype=np.float64).astype(np.float32)


# --------------------------------------------------------------------------
# FP8 e4m3 (OCP 8-bit floating point, E4M3 variant)
# --------------------------------------------------------------------------

def e4m3_value(code):
    """Closed form of one e4m3 code: sign, 4 exponent bits (bias 7), 3 mantissa bits."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 0xF and man == 0x7:
        return math.nan
    if exp == 0:
        return sign * (man / 8.0) * 2.0 ** (1 - 7)
    return sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)


def e4m3_table():
    return np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


_E4M3_POS = e4m3_table()[:127]   # codes 0x00..0x7E: 0 .. 448, increasing


def e4m3_encode(x32):
    """fp32 -> e4m3 code: nearest value, ties to the even code, |x| > 448 -> 448.

    The sign bit follows the sign of the input (so -0.0 and negative values
    that round to zero give 0x80).  Inputs must be finite.
    """
    x32 = _f32(x32)
    a = np.abs(x32).astype(np.float64)
    idx = np.searchsorted(_E4M3_POS, a, side="left")   # first value >= a
    idx = np.clip(idx, 0, 126)
    lo = np.clip(idx - 1, 0, 126)
    d_hi = np.abs(_E4M3_POS[idx] - a)
    d_lo = np.abs(a - _E4M3_POS[lo])
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))
    mag = np.where(pick_lo, lo, idx)
    mag = np.where(a >= 448.0, 126, mag)
    sign = np.signbit(x32).astype(np.int64) << 7
    return (mag | sign).astype(np.uint8)


# --------------------------------------------------------------------------
# Per-unit encoders
# --------------------------------------------------------------------------

def quantize_unit_fp8(x32):
    """One (page, head, K-or-V) unit -> (uint8 codes, float32 scale)."""
    x32 = _f32(x32)
    a = np.float32(np.max(np.abs(x32))) if x32.size else np.float32(0)
    if a == 0:
        return np.zeros(x32.shape, np.uint8), np.float32(0)
    scale = _f32(np.float64(a) / 448.0)
    y = _f32(x32.astype(np.float64) / np.float64(scale))
    return e4m3_encode(y), scale


def quantize_unit_int8(x32):
    """One unit -> (int8 codes, float32 scale); symmetric, -127..127."""
    x32 = _f32(x32)
    a = np.float32(np.max(np.abs(x32))) if x32.size else np.float32(0)
    if a == 0:
        return np.zeros(x32.shape, np.int8), np.float32(0)
    scale = _f32(np.float64(a) / 127.0)
    y = _f32(x32.astype(np.float64) / np.float64(scale))
    q = np.clip(np.rint(y), -127, 127)
    return q.astype(np.int8), scale


def quantize_group_int4(x32):
    """Groups of 32 along the last axis -> (codes 0..15, fp16 scale, fp16 zero).

    x32 shape [..., 32]; returns codes [..., 32] (uint8, one per element),
    s [...] float16, z [...] float16.
    """
    return _quantize_group_affine(x32, 15)


def quantize_group_int2(x32):
    """Groups of 32 along the last axis -> (codes 0..3, fp16 scale, fp16 zero);
    the INT4 steps with 3 levels above the zero point in place of 15."""
    return _quantize_group_affine(x32, 3)


def quantize_group_int1(x32):
    """Groups of 32 along the last axis -> (codes 0..1, fp16 scale, fp16 zero);
    the INT4 steps with 1 level above the zero point in place of 15."""
    return _quantize_group_affine(x32, 1)


def _quantize_group_affine(x32, top):
    """unsigned_affine over groups of 32: codes 0..top (top = 2^bits - 1)."""
    x32 = _f32(x32)
    lo = np.min(x32, axis=-1)
    hi = np.max(x32, axis=-1)
    z = fp16_rne_sat(lo)
    span = _f32(hi.astype(np.float64) - z.astype(np.float64))
    s = fp16_rne_sat(_f32(span.astype(np.float64) / float(top)))
    num = _f32(x32.astype(np.float64) - z.astype(np.float64)[..., None])
    s64 = s.astype(np.float64)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        y = _f32(num.astype(np.float64) / np.where(s64 > 0, s64, 1.0))
    q = np.clip(np.rint(y), 0, top)
    q = np.where(s64 > 0, q, 0)
    return q.astype(np.uint8), s, z


def pack_int4(codes):
    """[..., D] codes 0..15 -> [..., D/2] bytes, even element in the low nibble."""
    c = codes.astype(np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def pack_int2(codes):
    """[..., D] codes 0..3 -> [..., D/4] bytes, element 4k + j in bits 2j of byte k."""
    c = codes.astype(np.uint8)
    return (c[..., 0::4] | (c[..., 1::4] << 2) | (c[..., 2::4] << 4) | (c[..., 3::4] << 6)).astype(np.uint8)


def pack_int1(codes):
    """[..., D] codes 0..1 -> [..., D/8] bytes, element 8k + j in bit j of byte k."""
    c = codes.astype(np.uint8)
    out = np.zeros(c.shape[:-1] + (c.shape[-1] // 8,), np.uint8)
    for j in range(8):
        out |= (c[..., j::8] << j).astype(np.uint8)
    return out


def unpack_int1(packed):
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 8,), np.uint8)
    for j in range(8):
        out[..., j::8] = (p >> j) & 1
    return out


def unpack_int2(packed):
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 4,), np.uint8)
    for j in range(4):
        out[..., j::4] = (p >> (2 * j)) & 3
    return out


def unpack_int4(packed):
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


# --------------------------------------------------------------------------
# Dequantisation of one stored unit (float64, exact)
# --------------------------------------------------------------------------

def dequant_page(codec, codes, meta, slot, kv, h):
    """Dequantise unit (slot, kv, h) of a pool -> float64 [P][D]."""
    c = codes[slot, kv, h]
    if codec in (CODEC_FP16, CODEC_BF16):
        return bits_to_f64(c, codec)
    if codec == CODEC_FP8_E4M3:
        return e4m3_table()[c.astype(np.int64)] * np.float64(meta[slot, kv, h])
    if codec == CODEC_INT8:
        return c.view(np.int8).astype(np.float64) * np.float64(meta[slot, kv, h])
    if codec in (CODEC_INT4_G32, CODEC_INT2_G32, CODEC_INT1_G32):
        unpack = {CODEC_INT4_G32: unpack_int4, CODEC_INT2_G32: unpack_int2, CODEC_INT1_G32: unpack_int1}[codec]
        q = unpack(c).astype(np.float64)                                                     # [P][D]
        P, D = q.shape
        sz = meta[slot, kv, h].astype(np.float64)          # [P][D/32][2]
        qg = q.reshape(P, D // 32, 32)
        return (qg * sz[..., 0:1] + sz[..., 1:2]).reshape(P, D)
    raise ValueError("unknown codec %r" % codec)


# --------------------------------------------------------------------------
# Page demotion over a list of pages
# --------------------------------------------------------------------------

def alloc_pool(codec, n_slots, hkv, P, D):
    """Zero-filled pool arrays (codes, meta) in the layout above."""
    if codec in (CODEC_FP16, CODEC_BF16):
        return np.zeros((n_slots, 2, hkv, P, D), np.uint16), None
    if codec in (CODEC_FP8_E4M3, CODEC_INT8):
        return (np.zeros((n_slots, 2, hkv, P, D), np.uint8),
                np.zeros((n_slots, 2, hkv), np.float32))
    if codec in (CODEC_INT4_G32, CODEC_INT2_G32, CODEC_INT1_G32):
        row = {CODEC_INT4_G32: D // 2, CODEC_INT2_G32: D // 4, CODEC_INT1_G32: D // 8}[codec]
        return (np.zeros((n_slots, 2, hkv, P, row), np.uint8),
                np.zeros((n_slots, 2, hkv, P, D // 32, 2), np.float16))
    raise ValueError("unknown codec %r" % codec)


def quantize_pages(src_bits, src_dtype, src_slots, dst_codec, dst_codes, dst_meta,
                   dst_slots, valid_tokens=None, want_ckey=False):
    """Demote pages of a 16-bit source pool into a destination pool (in place).

    src_bits   uint16 [n_src][2][Hkv][P][D] (fp16 or bf16 bit patterns)
    dst_*      arrays from alloc_pool(dst_codec, ...), updated in place
    valid_tokens  None or int [n_pages]: tokens >= valid are excluded from the
               reductions and stored as zero codes (zero metadata for INT4)
    Returns the compressed keys as bf16 bits [n_pages][Hkv][D] when
    want_ckey: the mean over the valid tokens of the *stored* (dequantised)
    keys, rounded to bfloat16 (page "feat(kvcache) ...", section "Why this
    works for sparse attention": the indexer scores a compressed slab).
    """
    n_pages = len(src_slots)
    _, _, hkv, P, D = src_bits.shape
    ckeys = np.zeros((n_pages, hkv, D), np.uint16) if want_ckey else None
    for i in range(n_pages):
        valid = P if valid_tokens is None else int(valid_tokens[i])
        valid = max(0, min(P, valid))
        si, di = int(src_slots[i]), int(dst_slots[i])
        for kv in range(2):
            for h in range(hkv):
                x = bits_to_f64(src_bits[si, kv, h], src_dtype).astype(np.float32)
                xv = x[:valid]
                if dst_codec in (CODEC_FP16, CODEC_BF16):
                    if dst_codec != src_dtype:
                        raise ValueError("16-bit destination must match the source dtype")
                    out = np.zeros((P, D), np.uint16)
                    out[:valid] = src_bits[si, kv, h, :valid]
                    dst_codes[di, kv, h] = out
                elif dst_codec == CODEC_FP8_E4M3:
                    codes, scale = quantize_unit_fp8(xv)
                    out = np.zeros((P, D), np.uint8)
                    out[:valid] = codes
                    dst_codes[di, kv, h] = out
                    dst_meta[di, kv, h] = scale
                elif dst_codec == CODEC_INT8:
                    codes, scale = quantize_unit_int8(xv)
                    out = np.zeros((P, D), np.int8)
                    out[:valid] = codes
                    dst_codes[di, kv, h] = out.view(np.uint8)
                    dst_meta[di, kv, h] = scale
                elif dst_codec in (CODEC_INT4_G32, CODEC_INT2_G32, CODEC_INT1_G32):
                    q = np.zeros((P, D), np.uint8)
                    sz = np.zeros((P, D // 32, 2), np.float16)
                    if valid:
                        enc = {CODEC_INT4_G32: quantize_group_int4, CODEC_INT2_G32: quantize_group_int2,
                               CODEC_INT1_G32: quantize_group_int1}[dst_codec]
                        qc, s, z = enc(xv.reshape(valid, D // 32, 32))
                        q[:valid] = qc.reshape(valid, D)
                        sz[:valid, :, 0] = s
                        sz[:valid, :, 1] = z
                    pack = {CODEC_INT4_G32: pack_int4, CODEC_INT2_G32: pack_int2, CODEC_INT1_G32: pack_int1}[dst_codec]
                    dst_codes[di, kv, h] = pack(q)
                    dst_meta[di, kv, h] = sz
                else:
                    raise ValueError("unknown codec %r" % dst_codec)
        if want_ckey:
            for h in range(hkv):
                k = dequant_page(dst_codec, dst_codes, dst_meta, di, 0, h)[:valid]
                mean = k.mean(axis=0) if valid else np.zeros(D)
                ckeys[i, h] = f64_to_bf16_bits(mean)
    return ckeys
