"""Windowed prefill at any shape, and over a paged, mixed-codec cache.

argus_window_prefill_attn with query counts and window lengths that are not
multiples of the 128-row tile (tiles that straddle two query heads, partial
last key blocks), in all three modes; argus_paged_window_prefill_attn, which
stages a window of the paged cache through the block table (pages of every
codec, permuted physical slots, windows starting mid-page) and attends to it
with fp16 tensor-core MMAs, against oracle.paged_window_attention.  Windows
folded by log2-sum-exp must equal single-pass attention over everything
visible.  Tolerance on the fp32 accumulator: max|err| <= 1e-3 * max|ref| + 1e-4.
"""

import numpy as np
import pytest
import torch

import mixed_precision_paged_argus_gb300.argus as argus
from mixed_precision_paged_argus_gb300 import workloads as W
import oracle
from oracle import codecs as C
from paged_cases import DEV, build_case

pytestmark = pytest.mark.gpu


def _check(go, gl, ro, rl, lse_bound=None):
    """lse_bound: per-row bound on |lse2 error| from the arithmetic (staged
    paths); else 1e-4 relative (exact bf16 operands)."""
    t = 1e-3 * np.abs(ro).max() + 1e-4
    err = np.abs(go - ro).max()
    assert err <= t, "max err %.3g > tol %.3g" % (err, t)
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(gl), fin)
    if lse_bound is None:
        assert np.abs(gl[fin] - rl[fin]).max() <= 1e-4 * np.abs(rl[fin]).max() + 1e-5
    else:
        assert np.all(np.abs(gl[fin] - rl[fin]) <= lse_bound[fin] + 1e-5 * np.abs(rl[fin]) + 1e-5)


def _staged_lse_bound(c, win_len):
    """The staged window rounds each key to fp16 (relative error <= 2^-11; the
    bf16 query is exact in fp16), so every log2-domain score moves by at most
    scale * log2(e) * 2^-11 * sum_d |q_d k_d|, and lse2 -- a softmax-weighted
    mean of the scores under perturbation -- by at most the largest of those."""
    K, _ = oracle.gather_window(c.Hkv, c.P, c.opools, c.page_codec, c.table, 0, 0, win_len)
    G = c.Hq // c.Hkv
    Kh = np.repeat(np.abs(K), G, axis=0)                                 # [Hq][W][D]
    m = np.einsum("hqd,hkd->hqk", np.abs(c.pq64), Kh).max(axis=2)         # [Hq][n_q]
    return W.softmax_scale(c.D) / np.log(2.0) * 2.0 ** -11 * m


MODES = [(1, False), (1, True), (3, True)]


@pytest.mark.parametrize("splits,use_ws", MODES)
@pytest.mark.parametrize("Hq,Hkv,n_q,ctx,cuts", [
    (2, 1, 100, 77, [77]),              # one partial tile straddling both query heads
    (16, 2, 200, 300, [130, 300]),      # 8 heads x 200 rows per KV head: tiles cross head boundaries
    (3, 3, 1, 5, [2, 5]),               # a single query row, windows of 2, 3 and 1 keys
    (4, 2, 129, 1000, [129, 640, 1000]),
])
@pytest.mark.parametrize("D", [128, 64])
def test_window_prefill_at_unaligned_shapes(Hq, Hkv, n_q, ctx, cuts, splits, use_ws, D):
    q = W.normal((Hq, n_q, D), W.BF16, 701 + n_q)
    kv_len = ctx + n_q
    k = W.normal((Hkv, kv_len, D), W.BF16, 702 + n_q)
    v = W.normal((Hkv, kv_len, D), W.BF16, 703 + n_q)
    f = lambda t: C.bf16_bits_to_f64(W.to_bits(t))
    g = argus.geom(Hq, Hkv, D, 16)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    acc_o = torch.full((Hq, n_q, D), float("nan"), dtype=torch.float32, device=DEV)
    acc_l = torch.full((Hq, n_q), float("nan"), dtype=torch.float32, device=DEV)
    bounds = [0] + cuts + [kv_len]
    for wi, (w0, w1) in enumerate(zip(bounds[:-1], bounds[1:])):
        ws = None
        if use_ws:
            n = argus.window_prefill_workspace_bytes(g, n_q, w1 - w0, splits)
            ws = torch.full((max(n, 16) // 4 + 1,), float("nan"), dtype=torch.float32, device=DEV)
        argus.window_prefill_attn(g, n_q, qd, kd[:, w0:], vd[:, w0:], kv_len * D, w1 - w0, w0, ctx,
                                  W.softmax_scale(D), acc_o, acc_l, 1 if wi else 0, num_splits=splits, ws=ws)
    torch.cuda.synchronize()
    ro, rl = oracle.window_attention(f(q), f(k), f(v), 0, ctx, W.softmax_scale(D))
    _check(acc_o.cpu().numpy(), acc_l.cpu().numpy(), ro, rl)


def _paged(Hq, Hkv, P, n_q, ctx, tiers, seed, D=128):
    """One sequence of ctx + n_q tokens in pages of the given codecs (cycled,
    oldest first), demoted by the library and by the oracle; bf16 query."""
    total = ctx + n_q
    n_pages = -(-total // P)
    pc = np.array([tiers[i % len(tiers)] for i in range(n_pages)]).reshape(1, n_pages)
    src = W.FP16 if W.FP16 in tiers else W.BF16          # a 16-bit tier stores its own source type
    c = build_case(Hq, Hkv, D, P, [total], pc, src, q_dtype=W.BF16, seed=seed, outliers=True, extra_slots=3)
    q = W.normal((Hq, n_q, D), W.BF16, seed + 50)
    c.pq = q.to(DEV)
    c.pq64 = C.bf16_bits_to_f64(W.to_bits(q))
    c.n_pages = n_pages
    return c


def _run_paged(c, n_q, ctx, cuts, splits=0, status=None):
    g = argus.geom(c.Hq, c.Hkv, c.D, c.P)
    acc_o = torch.full((c.Hq, n_q, c.D), float("nan"), dtype=torch.float32, device=DEV)
    acc_l = torch.full((c.Hq, n_q), float("nan"), dtype=torch.float32, device=DEV)
    bounds = [0] + cuts + [ctx + n_q]
    for wi, (w0, w1) in enumerate(zip(bounds[:-1], bounds[1:])):
        n = argus.paged_window_prefill_workspace_bytes(g, n_q, w1 - w0, splits)
        ws = torch.full((n,), 0xFF, dtype=torch.uint8, device=DEV)      # NaN-filled: needs no initialisation
        argus.paged_window_prefill_attn(g, n_q, c.pq, c.pools, c.d_codec[0], c.d_table[0], c.n_pages, w0, w1 - w0,
                                        ctx, W.softmax_scale(c.D), acc_o, acc_l, 1 if wi else 0, ws,
                                        num_splits=splits, status=status)
    torch.cuda.synchronize()
    return acc_o.cpu().numpy(), acc_l.cpu().numpy()


FIVE = [W.INT1_G32, W.INT2_G32, W.INT4_G32, W.INT8, W.FP8_E4M3, W.BF16]   # every tier (16-bit as BF16)


@pytest.mark.parametrize("splits", [1, 0, 3])
@pytest.mark.parametrize("P,n_q,ctx,cuts", [
    (16, 128, 37 * 16 + 5, [100, 333, 597]),      # windows start mid-page; the last one is the chunk plus a tail
    (64, 70, 900, [450]),
])
@pytest.mark.parametrize("D", [128, 64])
def test_paged_windows_five_tiers_fold_to_single_pass(P, n_q, ctx, cuts, splits, D):
    c = _paged(16, 2, P, n_q, ctx, FIVE, seed=720 + P, D=D)
    go, gl = _run_paged(c, n_q, ctx, cuts, splits=splits)
    ro, rl = oracle.paged_window_attention(c.pq64, c.Hkv, c.P, c.opools, c.page_codec, c.table, 0, 0, ctx + n_q, ctx,
                                           W.softmax_scale(D), seq_len=ctx + n_q)
    _check(go, gl, ro, rl, _staged_lse_bound(c, ctx + n_q))


@pytest.mark.parametrize("codec", [W.FP16, W.BF16, W.FP8_E4M3, W.INT8, W.INT4_G32, W.INT2_G32, W.INT1_G32])
@pytest.mark.parametrize("D", [128, 64])
def test_paged_window_single_codec(codec, D):
    c = _paged(8, 1, 16, 96, 500, [codec], seed=740 + codec, D=D)
    go, gl = _run_paged(c, 96, 500, [250])
    ro, rl = oracle.paged_window_attention(c.pq64, c.Hkv, c.P, c.opools, c.page_codec, c.table, 0, 0, 596, 500,
                                           W.softmax_scale(D), seq_len=596)
    _check(go, gl, ro, rl, _staged_lse_bound(c, 596))


def test_paged_window_bad_slot_counted_once_and_reads_as_zero():
    c = _paged(2, 1, 16, 16, 64, [W.FP8_E4M3], seed=760)
    table = c.table.copy()
    table[0, 1] = 10_000                       # page 1 (positions 16..31) points outside its pool
    c.d_table = torch.from_numpy(table).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    go, gl = _run_paged(c, 16, 64, [40], status=status)
    assert int(status.item()) == 1             # counted in the one window that holds page 1
    # the oracle on the same cache with page 1 zeroed
    codes, meta = c.opools[W.FP8_E4M3]
    codes, meta = codes.copy(), meta.copy()
    slot = sorted(set(range(codes.shape[0])) - set(int(x) for x in c.table[0]))[0]   # a slot no page uses
    codes[slot] = 0
    meta[slot] = 0
    table[0, 1] = slot
    ro, rl = oracle.paged_window_attention(c.pq64, c.Hkv, c.P, {W.FP8_E4M3: (codes, meta)}, c.page_codec, table, 0, 0,
                                           80, 64, W.softmax_scale(128))
    _check(go, gl, ro, rl, _staged_lse_bound(c, 80))


def test_paged_window_rejects_a_window_outside_the_table():
    c = _paged(2, 1, 16, 16, 64, [W.FP16], seed=770)
    g = argus.geom(2, 1, 128, 16)
    acc_o = torch.zeros((2, 16, 128), device=DEV)
    acc_l = torch.zeros((2, 16), device=DEV)
    ws = torch.zeros(argus.paged_window_prefill_workspace_bytes(g, 16, 100), dtype=torch.uint8, device=DEV)
    with pytest.raises(argus.ArgusError) as e:
        argus.paged_window_prefill_attn(g, 16, c.pq, c.pools, c.d_codec[0], c.d_table[0], c.n_pages, 0, c.n_pages * 16 + 1,
                                        64, 0.1, acc_o, acc_l, 0, ws)
    assert e.value.status == 1
