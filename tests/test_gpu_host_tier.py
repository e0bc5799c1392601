"""Pools in page-locked host memory, read in place (the host-RAM tier).

"feat(kvcache): host-RAM KV tier for sparse-attention models", section
"Design" and the comment on "--kv-placement host": attention reads the pages of
a host-resident tier in place instead of copying them to the device.  Here a
pool with placement PLACE_HOST lives in pinned host memory; decode streams its
chunks over the host link with plain 16-byte loads.  Checked against the
double-precision oracle (which never sees where a pool lives) at the stated
tolerance, with device and host pools mixed in one call; demotion into a host
pool is compared bit for bit.
"""

import numpy as np
import pytest
import torch

import mixed_precision_paged_argus_gb300.argus as argus
from mixed_precision_paged_argus_gb300 import workloads as W
import oracle
from oracle import codecs as C
from paged_cases import DEV, build_case, run_decode, tol

pytestmark = pytest.mark.gpu


def _to_host(c, codecs):
    """Move the pools of the given codecs into page-locked host memory."""
    c.pools = [p.to_host() if p.codec in codecs else p for p in c.pools]
    return c


def _check(c, out32, lse, **kw):
    ref, ref_lse, bad = oracle.paged_decode(c.q64, c.Hkv, c.P, c.opools, c.page_codec, c.table, c.lens, c.scale, **kw)
    assert bad == 0
    got = out32.cpu().numpy()
    assert np.abs(got - ref).max() <= tol(ref)
    fin = np.isfinite(ref_lse)
    gl = lse.cpu().numpy()
    assert np.array_equal(np.isfinite(gl), fin)
    assert np.all(np.abs(gl[fin] - ref_lse[fin]) <= 1e-4 * np.maximum(1.0, np.abs(ref_lse[fin])))


@pytest.mark.parametrize("q_dtype", [W.FP16, W.BF16])
@pytest.mark.parametrize("D", [64, 128])
def test_mixed_device_and_host_pools(D, q_dtype):
    Hq, Hkv, P = 16, 2, 16
    top = W.FP16 if q_dtype == W.FP16 else W.BF16
    row = np.array([W.INT4_G32] * 5 + [W.INT8] * 5 + [W.FP8_E4M3] * 5 + [top] * 5)
    pc = np.stack([row, np.roll(row, 3), row])
    c = build_case(Hq, Hkv, D, P, [20 * P - 3, 150, 0], pc, q_dtype, seed=900 + D, outliers=True, extra_slots=2)
    _to_host(c, {W.FP8_E4M3, W.INT8, W.INT4_G32})           # older tiers in host memory
    assert sum(p.placement == argus.PLACE_HOST for p in c.pools) == 3
    for splits in (0, 1, 5):
        out, out32, lse, _ = run_decode(c, out_dtype=torch.float16 if q_dtype == W.FP16 else torch.bfloat16,
                                        num_splits=splits)
        _check(c, out32, lse)
        assert torch.equal(out.cpu(), out32.cpu().to(out.dtype))


@pytest.mark.parametrize("codec", [W.BF16, W.FP8_E4M3, W.INT4_G32])
def test_every_pool_in_host_memory(codec):
    Hq, Hkv, D, P = 32, 8, 128, 16
    lens = [300, 17, 1000]
    c = build_case(Hq, Hkv, D, P, lens, np.full((3, 64), codec), W.BF16, seed=910 + codec)
    _to_host(c, {codec})
    out, out32, lse, _ = run_decode(c, out_dtype=torch.bfloat16)
    _check(c, out32, lse)


def test_selected_pages_from_a_host_fp8_pool():
    """The sparse workload's shape in small: the indexer's selection (here drawn
    at random) read from an FP8 pool in host memory."""
    Hq, Hkv, D, P = 32, 4, 128, 64
    maxp = 40
    lens = [40 * 64 - 7, 25 * 64]
    c = build_case(Hq, Hkv, D, P, lens, np.full((2, maxp), W.FP8_E4M3), W.BF16, seed=920)
    _to_host(c, {W.FP8_E4M3})
    width = 2 * 8 + 8
    rng = np.random.default_rng(921)
    sel = np.full((2, Hkv, width), -1, np.int32)
    cnt = np.zeros((2, Hkv), np.int32)
    for b in range(2):
        n = -(-lens[b] // P)
        for h in range(Hkv):
            pages = sorted(rng.choice(n - 1, size=8, replace=False).tolist() + [n - 1])
            sel[b, h, :len(pages)] = pages
            cnt[b, h] = len(pages)
    out, out32, lse, _ = run_decode(c, out_dtype=torch.bfloat16, sel=torch.from_numpy(sel).to(DEV),
                                    sel_count=torch.from_numpy(cnt).to(DEV), sel_width=width)
    _check(c, out32, lse, sel_pages=sel, sel_count=cnt, sel_width=width)


@pytest.mark.parametrize("codec", [W.FP8_E4M3, W.INT8, W.INT4_G32])
def test_demotion_into_a_host_pool_bit_exact(codec):
    Hkv, P, D, n = 2, 16, 128, 9
    src = W.normal((n, 2, Hkv, P, D), W.BF16, 930 + codec, outlier_seed=931)
    g = argus.geom(Hkv, Hkv, D, P)
    pool = argus.Pool.empty(codec, n + 2, Hkv, P, D, device="host", zero=True)
    slots = [3, 0, 7, 1, 10, 2, 9, 4, 8]
    argus.quantize_pages(g, W.BF16, src.to(DEV), n, torch.arange(n, dtype=torch.int32, device=DEV), pool,
                         torch.tensor(slots, dtype=torch.int32, device=DEV), n)
    torch.cuda.synchronize()
    codes, meta = C.alloc_pool(codec, n + 2, Hkv, P, D)
    C.quantize_pages(W.to_bits(src), C.CODEC_BF16, list(range(n)), codec, codes, meta, slots)
    assert np.array_equal(pool.codes.view(torch.uint8).numpy().reshape(-1), codes.view(np.uint8).reshape(-1))
    assert np.array_equal(pool.meta.contiguous().view(torch.uint8).numpy().reshape(-1),
                          meta.view(np.uint8).reshape(-1))


def test_paged_prefill_staged_from_host_pools():
    Hq, Hkv, P, n_q, ctx = 8, 2, 16, 64, 300
    total = ctx + n_q
    n_pages = -(-total // P)
    pc = np.array([[W.FP8_E4M3, W.INT4_G32, W.BF16][i % 3] for i in range(n_pages)]).reshape(1, n_pages)
    c = build_case(Hq, Hkv, 128, P, [total], pc, W.BF16, seed=940, outliers=True)
    _to_host(c, {W.FP8_E4M3, W.INT4_G32})
    q = W.normal((Hq, n_q, 128), W.BF16, 941)
    g = argus.geom(Hq, Hkv, 128, P)
    acc_o = torch.empty((Hq, n_q, 128), device=DEV)
    acc_l = torch.empty((Hq, n_q), device=DEV)
    ws = torch.empty(argus.paged_window_prefill_workspace_bytes(g, n_q, total), dtype=torch.uint8, device=DEV)
    argus.paged_window_prefill_attn(g, n_q, q.to(DEV), c.pools, c.d_codec[0], c.d_table[0], n_pages, 0, total, ctx,
                                    W.softmax_scale(128), acc_o, acc_l, 0, ws)
    torch.cuda.synchronize()
    q64 = C.bf16_bits_to_f64(W.to_bits(q))
    ro, rl = oracle.paged_window_attention(q64, Hkv, P, c.opools, c.page_codec, c.table, 0, 0, total, ctx,
                                           W.softmax_scale(128))
    assert np.abs(acc_o.cpu().numpy() - ro).max() <= 1e-3 * np.abs(ro).max() + 1e-4


def test_unpinned_host_memory_and_host_pools_with_a_window_are_refused():
    Hq, Hkv, D, P = 8, 1, 64, 16
    c = build_case(Hq, Hkv, D, P, [100], np.full((1, 8), W.FP8_E4M3), W.FP16, seed=950)
    dev_pool = c.pools[0]
    c.pools = [argus.Pool(W.FP8_E4M3, dev_pool.codes.cpu(), dev_pool.meta.cpu(), dev_pool.n_slots)]   # not pinned
    with pytest.raises(argus.ArgusError) as e:
        run_decode(c)
    assert e.value.status == 1
    c.pools = [dev_pool.to_host()]
    with pytest.raises(argus.ArgusError) as e:
        run_decode(c, window=32)
    assert e.value.status == 2
