"""argus_quantize_pages on the GPU against the oracle: codes and scales bit-exact."""

import numpy as np
import pytest
import torch

import mixed_precision_paged_argus_gb300.argus as argus
from mixed_precision_paged_argus_gb300 import workloads as W
from oracle import codecs as C

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _gpu_quantize(src_t, src_dtype, codec, Hkv, P, D, src_slots, dst_slots, n_dst, valid=None, ckey=False):
    g = argus.geom(Hkv, Hkv, D, P)
    n_pages = len(src_slots)
    pool = argus.Pool.empty(codec, n_dst, Hkv, P, D, device=DEV, zero=True)
    ck = torch.zeros((n_pages, Hkv, D), dtype=torch.bfloat16, device=DEV) if ckey else None
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    argus.quantize_pages(g, src_dtype, src_t.to(DEV), src_t.shape[0],
                         torch.tensor(src_slots, dtype=torch.int32, device=DEV), pool,
                         torch.tensor(dst_slots, dtype=torch.int32, device=DEV), n_pages,
                         None if valid is None else torch.tensor(valid, dtype=torch.int32, device=DEV),
                         ck, status)
    torch.cuda.synchronize()
    return pool, ck, int(status.item())


def _codes_np(pool):
    return pool.codes.contiguous().view(torch.uint8).cpu().numpy()


def _meta_np(pool):
    if pool.meta is None:
        return None
    return pool.meta.contiguous().view(torch.uint8).cpu().numpy()


def _compare(pool, codes, meta):
    assert np.array_equal(_codes_np(pool), codes.view(np.uint8).reshape(_codes_np(pool).shape))
    if meta is not None:
        assert np.array_equal(_meta_np(pool), meta.view(np.uint8).reshape(_meta_np(pool).shape))


def test_e4m3_encoder_exhaustive_over_fp16():
    """Every finite fp16 value with |x| <= 448 encoded with scale exactly 1."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = bits.view(np.float16).astype(np.float32)
    keep = np.isfinite(x) & (np.abs(x) <= 448)
    vals = bits[keep]
    P, D = 16, 64
    per_unit = P * D - 1
    n_units = -(-len(vals) // per_unit)
    pad = np.full(n_units * per_unit, np.float16(0).view(np.uint16))
    pad[:len(vals)] = vals
    units = pad.reshape(n_units, per_unit)
    big = np.full((n_units, 1), np.float16(448).view(np.uint16))
    units = np.concatenate([units, big], axis=1).reshape(n_units, 1, 1, P, D)   # Hkv = 1, K side
    src = np.zeros((n_units, 2, 1, P, D), np.uint16)
    src[:, 0] = units[:, 0]
    src[:, 1] = units[:, 0]
    t = torch.from_numpy(src.view(np.int16)).view(torch.float16)
    pool, _, st = _gpu_quantize(t, W.FP16, W.FP8_E4M3, 1, P, D, list(range(n_units)), list(range(n_units)), n_units)
    assert st == 0
    codes, meta = C.alloc_pool(C.CODEC_FP8_E4M3, n_units, 1, P, D)
    C.quantize_pages(src, C.CODEC_FP16, list(range(n_units)), C.CODEC_FP8_E4M3, codes, meta, list(range(n_units)))
    assert np.all(meta == 1.0)
    _compare(pool, codes, meta)


def test_int8_rounding_exhaustive_over_fp16():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = bits.view(np.float16).astype(np.float32)
    vals = bits[np.isfinite(x) & (np.abs(x) <= 127)]
    P, D = 16, 128
    per_unit = P * D - 1
    n_units = -(-len(vals) // per_unit)
    pad = np.zeros(n_units * per_unit, np.uint16)
    pad[:len(vals)] = vals
    units = np.concatenate([pad.reshape(n_units, per_unit),
                            np.full((n_units, 1), np.float16(-127).view(np.uint16))], axis=1)
    src = np.zeros((n_units, 2, 1, P, D), np.uint16)
    src[:, 0, 0] = units.reshape(n_units, P, D)
    src[:, 1, 0] = units.reshape(n_units, P, D)
    t = torch.from_numpy(src.view(np.int16)).view(torch.float16)
    pool, _, _ = _gpu_quantize(t, W.FP16, W.INT8, 1, P, D, list(range(n_units)), list(range(n_units)), n_units)
    codes, meta = C.alloc_pool(C.CODEC_INT8, n_units, 1, P, D)
    C.quantize_pages(src, C.CODEC_FP16, list(range(n_units)), C.CODEC_INT8, codes, meta, list(range(n_units)))
    _compare(pool, codes, meta)


@pytest.mark.parametrize("codec", [W.FP8_E4M3, W.INT8, W.INT4_G32, W.INT2_G32, W.INT1_G32, "copy"])
@pytest.mark.parametrize("src_dtype", [W.FP16, W.BF16])
@pytest.mark.parametrize("D,P", [(64, 16), (128, 16), (128, 64), (64, 1024)])
def test_random_pages_bit_exact_with_ckeys(codec, src_dtype, D, P):
    if codec == "copy":
        codec = src_dtype
    Hkv, n_src, n_pages = 2, 7, 5
    src = W.normal((n_src, 2, Hkv, P, D), src_dtype, 100 + D + P, outlier_seed=101)
    src_slots = [6, 0, 3, 2, 5]
    dst_slots = [1, 4, 0, 6, 2]
    valid = [P, P - 3, 1, 0, P // 2]
    pool, ck, st = _gpu_quantize(src, src_dtype, codec, Hkv, P, D, src_slots, dst_slots, 8, valid, ckey=True)
    assert st == 0
    codes, meta = C.alloc_pool(codec, 8, Hkv, P, D)
    ock = C.quantize_pages(W.to_bits(src), src_dtype, src_slots, codec, codes, meta, dst_slots,
                           valid_tokens=valid, want_ckey=True)
    _compare(pool, codes, meta)
    # ckey = bf16(mean of stored keys): the GPU sums in fp32 in its own order, so
    # allow one bf16 ulp plus the fp32 summation bound n * 2^-24 * mean|k|
    got = C.bf16_bits_to_f64(W.to_bits(ck.cpu()))
    want = C.bf16_bits_to_f64(ock)
    mean_abs = np.zeros_like(want)
    for i, s_dst in enumerate(dst_slots):
        n = max(valid[i], 1)
        for h in range(Hkv):
            k = C.dequant_page(codec, codes, meta, s_dst, 0, h)[:valid[i]]
            mean_abs[i, h] = np.abs(k).sum(axis=0) / n if valid[i] else 0.0
    bound = np.abs(want) * 2.0 ** -7 + (P + 2) * 2.0 ** -24 * mean_abs + 2.0 ** -133
    assert np.all(np.abs(got - want) <= bound)


def test_bad_slots_are_counted_and_skipped():
    Hkv, P, D = 1, 16, 64
    src = W.normal((2, 2, Hkv, P, D), W.FP16, 9)
    pool, _, st = _gpu_quantize(src, W.FP16, W.FP8_E4M3, Hkv, P, D, [0, 5, 1], [0, 1, 9], 2)
    assert st == 2
    codes = _codes_np(pool)
    assert codes[0].any() and not codes[1].any()


def test_zero_unit_gives_zero_scale():
    Hkv, P, D = 1, 16, 128
    src = torch.zeros((1, 2, Hkv, P, D), dtype=torch.bfloat16)
    for codec in (W.FP8_E4M3, W.INT8, W.INT4_G32, W.INT2_G32, W.INT1_G32):
        pool, _, _ = _gpu_quantize(src, W.BF16, codec, Hkv, P, D, [0], [0], 1)
        assert not _codes_np(pool).any() and not _meta_np(pool).any()


def test_invalid_arguments_fail_closed():
    g = argus.geom(2, 2, 96, 16)
    pool = argus.Pool.empty(W.FP8_E4M3, 1, 2, 16, 64, device=DEV)
    with pytest.raises(argus.ArgusError) as e:
        argus.quantize_pages(g, W.FP16, pool.codes, 1, pool.codes, pool, pool.codes, 1)
    assert e.value.status == 2


def _near_boundary_units(boundaries, scale, P, D):
    """fp16 pages whose values x give x / scale within a few ulps of each boundary."""
    vals = []
    for m in boundaries:
        for k in range(-6, 7):
            x = np.float32(m * scale) * np.float32(1 + k * 2.0 ** -10)
            vals.append(x)
    vals = np.array(vals, np.float32).astype(np.float16)
    return vals


@pytest.mark.parametrize("codec", [W.FP8_E4M3, W.INT8])
def test_codes_near_rounding_boundaries_with_a_non_power_of_two_scale(codec):
    P, D = 16, 128
    tab = C.e4m3_table()[:127]
    if codec == W.FP8_E4M3:
        bounds = list((tab[1:] + tab[:-1]) / 2)               # e4m3 midpoints, subnormal ones included
        amax = 448.0 * 1.37
    else:
        bounds = [k + 0.5 for k in range(-127, 127)]
        amax = 127.0 * 1.37
    vals = _near_boundary_units(bounds, amax / (448.0 if codec == W.FP8_E4M3 else 127.0), P, D)
    per = P * D - 1
    n = -(-len(vals) // per)
    buf = np.zeros(n * per, np.float16)
    buf[:len(vals)] = vals
    units = np.concatenate([buf.reshape(n, per), np.full((n, 1), np.float16(amax))], axis=1).reshape(n, P, D)
    src = np.zeros((n, 2, 1, P, D), np.uint16)
    src[:, 0, 0] = units.view(np.uint16)
    src[:, 1, 0] = units.view(np.uint16)
    t = torch.from_numpy(src.view(np.int16)).view(torch.float16)
    pool, _, _ = _gpu_quantize(t, W.FP16, codec, 1, P, D, list(range(n)), list(range(n)), n)
    codes, meta = C.alloc_pool(codec, n, 1, P, D)
    C.quantize_pages(src, C.CODEC_FP16, list(range(n)), codec, codes, meta, list(range(n)))
    _compare(pool, codes, meta)


@pytest.mark.parametrize("codec", [W.INT4_G32, W.INT2_G32, W.INT1_G32])
@pytest.mark.parametrize("ckey", [False, True])
@pytest.mark.parametrize("src_dtype", [W.FP16, W.BF16])
def test_int4_groups_with_pinned_range_and_interior_values(ckey, src_dtype, codec):
    """Groups whose min and max pin z and s, interior values uniform in between
    (many land within 2^-12 of a half-integer quotient, some on exact ties when
    s is a power of two); INT4 V units use the one-lane-per-group path, K units
    the compressed-key path when ckey is set; INT2 units the cooperative path."""
    Hkv, P, D, n = 2, 16, 128, 48
    top = {W.INT4_G32: 15, W.INT2_G32: 3, W.INT1_G32: 1}[codec]
    rng = np.random.default_rng(7 + ckey + 2 * src_dtype + codec)
    groups = n * 2 * Hkv * P * (D // 32)
    z = rng.standard_normal(groups) * 4
    s = np.abs(rng.standard_normal(groups)) * 0.3 + 1e-3
    s[::5] = 2.0 ** rng.integers(-6, 0, size=len(s[::5]))          # exact ties possible
    k = rng.uniform(0, top, size=(groups, 32))
    k[:, 0], k[:, 1] = 0.0, float(top)
    k[::3, 2:] = np.floor(k[::3, 2:]) + 0.5                          # on / near the half-integers
    x = z[:, None] + k * s[:, None]
    if src_dtype == W.FP16:
        bits = x.astype(np.float16).view(np.uint16)
    else:
        bits = C.f64_to_bf16_bits(x)
    src = bits.reshape(n, 2, Hkv, P, D)
    t = torch.from_numpy(src.view(np.int16)).view(torch.float16 if src_dtype == W.FP16 else torch.bfloat16)
    pool, ck, st = _gpu_quantize(t, src_dtype, codec, Hkv, P, D, list(range(n)), list(range(n)), n,
                                 ckey=ckey)
    assert st == 0
    codes, meta = C.alloc_pool(codec, n, Hkv, P, D)
    C.quantize_pages(src, src_dtype, list(range(n)), codec, codes, meta, list(range(n)))
    _compare(pool, codes, meta)


@pytest.mark.parametrize("codec", [W.INT4_G32, W.INT2_G32, W.INT1_G32])
@pytest.mark.parametrize("ckey", [False, True])
def test_affine_zero_point_and_scale_saturate_at_65504(codec, ckey):
    """bf16 groups whose min is below -65504 or whose (max - z) / top is above
    65504: the fp16 zero point and scale saturate (never inf), the all-below
    group gets a negative scale and zero codes -- bit-exact with the oracle on
    both encode paths (one lane per group, and the compressed-key path)."""
    Hkv, P, D, n = 2, 16, 128, 6
    rng = np.random.default_rng(31 + codec + 2 * ckey)
    sat = np.zeros((4, 32), np.float32)
    sat[0] = np.linspace(-2.0 ** 17, 2.0 ** 20, 32)
    sat[0, 7] = 65504.0 * 2.5
    sat[1] = np.linspace(0.0, 2.0 ** 20, 32)
    sat[2] = -2.0 ** 17 + np.arange(32, dtype=np.float32) * 64.0
    sat[3] = np.linspace(-2.0 ** 16, 2.0 ** 16, 32)
    groups = n * 2 * Hkv * P * (D // 32)
    x = rng.standard_normal((groups, 32)) * 1e3
    pick = rng.integers(0, 4, groups)
    use = rng.random(groups) < 0.6
    x[use] = sat[pick[use]] * rng.choice([1.0, 0.5, 2.0], size=(int(use.sum()), 1))
    rng.shuffle(x, axis=1)
    bits = C.f64_to_bf16_bits(x).reshape(n, 2, Hkv, P, D)
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    pool, ck, st = _gpu_quantize(t, W.BF16, codec, Hkv, P, D, list(range(n)), list(range(n)), n, ckey=ckey)
    assert st == 0
    codes, meta = C.alloc_pool(codec, n, Hkv, P, D)
    C.quantize_pages(bits, C.CODEC_BF16, list(range(n)), codec, codes, meta, list(range(n)))
    m = meta.astype(np.float64)
    assert np.all(np.isfinite(m)) and np.any(np.abs(m) == 65504.0) and np.any(m[..., 0] < 0)
    _compare(pool, codes, meta)


@pytest.mark.slow
@pytest.mark.parametrize("codec", [W.FP8_E4M3, W.INT8, W.INT4_G32, W.INT2_G32, W.INT1_G32])
@pytest.mark.parametrize("ckey", [False, True])
def test_full_size_demotion_bit_exact_on_sampled_pages(codec, ckey):
    """The batched workload's unit shape (16 x 128 bf16) at 20,480 pages x 8 KV
    heads x K|V = 327,680 units: far more than one unit per warp of the grid, so
    the software-pipelined hand-off from unit to unit runs many times per warp.
    Pages with a partial valid-token count are mixed in.  Codes and metadata of
    sampled pages -- the first, the last, and pages whose units land on a
    warp's 2nd and later turn -- are compared bit for bit with the oracle run on
    those pages only; compressed keys within one bf16 ulp + the fp32 sum bound."""
    n_pages, Hkv, P, D = 20480, 8, 16, 128
    dev = torch.device(DEV)
    g = argus.geom(Hkv, Hkv, D, P)
    src = W.normal((n_pages, 2, Hkv, P, D), W.BF16, 4321 + codec, device=dev, outlier_seed=4322)
    rng = np.random.default_rng(77 + codec)
    valid = np.full(n_pages, P, np.int32)
    part = rng.random(n_pages) < 0.1
    valid[part] = rng.integers(0, P, int(part.sum()))
    dst_slots = rng.permutation(n_pages).astype(np.int32)
    pool = argus.Pool.empty(codec, n_pages, Hkv, P, D, device=dev)
    ck = torch.empty((n_pages, Hkv, D), dtype=torch.bfloat16, device=dev) if ckey else None
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    argus.quantize_pages(g, W.BF16, src, n_pages, torch.arange(n_pages, dtype=torch.int32, device=dev), pool,
                         torch.from_numpy(dst_slots).to(dev), n_pages, torch.from_numpy(valid).to(dev), ck, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # warps of the grid: at most 4 CTAs of 8 warps per SM, one unit per warp per turn
    n_warps = torch.cuda.get_device_properties(dev).multi_processor_count * 4 * 8
    units_per_page = 2 * Hkv
    assert n_pages * units_per_page > 20 * n_warps
    sample = sorted(set([0, 1, n_pages - 1] + [int(x) for x in rng.integers(0, n_pages, 150)] +
                        [(n_warps * t) // units_per_page + 3 for t in (1, 2, 7, 19)]))
    idx = torch.tensor(sample, dtype=torch.int64, device=dev)
    src_s = W.to_bits(src[idx])
    dsel = torch.from_numpy(dst_slots[sample].astype(np.int64)).to(dev)
    got_codes = pool.codes[dsel].contiguous().view(torch.uint8).cpu().numpy()
    got_meta = pool.meta[dsel].contiguous().view(torch.uint8).cpu().numpy()
    codes, meta = C.alloc_pool(codec, len(sample), Hkv, P, D)
    ock = C.quantize_pages(src_s, C.CODEC_BF16, list(range(len(sample))), codec, codes, meta,
                           list(range(len(sample))), valid_tokens=valid[sample], want_ckey=ckey)
    assert np.array_equal(got_codes, codes.view(np.uint8).reshape(got_codes.shape))
    assert np.array_equal(got_meta, meta.view(np.uint8).reshape(got_meta.shape))
    if ckey:
        got = C.bf16_bits_to_f64(W.to_bits(ck[idx].cpu()))
        want = C.bf16_bits_to_f64(ock)
        mean_abs = np.zeros_like(want)
        for i in range(len(sample)):
            if valid[sample[i]]:
                for h in range(Hkv):
                    kk = C.dequant_page(codec, codes, meta, i, 0, h)[:valid[sample[i]]]
                    mean_abs[i, h] = np.abs(kk).mean(axis=0)
        bound = np.abs(want) * 2.0 ** -7 + (P + 2) * 2.0 ** -24 * mean_abs + 2.0 ** -133
        assert np.all(np.abs(got - want) <= bound)
