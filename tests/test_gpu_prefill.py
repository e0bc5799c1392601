"""argus_window_prefill_attn (tcgen05) on the GPU against the oracle.

Windows are slices of one cache (kv_head_stride), attended with causal
visibility by absolute position and folded by log2-sum-exp; the folded result
must equal single-pass attention over everything visible.  Tolerance on the
fp32 accumulator: max|err| <= 1e-3 * max|ref| + 1e-4.
"""

import math

import numpy as np
import pytest
import torch

import mixed_precision_paged_argus_gb300.argus as argus
from mixed_precision_paged_argus_gb300 import workloads as W
import oracle
from oracle import codecs as C

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _data(Hq, Hkv, n_q, ctx, seed, D=128):
    q = W.normal((Hq, n_q, D), W.BF16, seed)
    kv_len = ctx + n_q
    k = W.normal((Hkv, kv_len, D), W.BF16, seed + 1)
    v = W.normal((Hkv, kv_len, D), W.BF16, seed + 2)
    f = lambda t: C.bf16_bits_to_f64(W.to_bits(t))
    return q, k, v, f(q), f(k), f(v)


# (num_splits, workspace): no workspace = bf16 P.V with a hi + lo P, one CTA
# per tile; with a workspace = fp16 P.V over the scaled fp16 copy of V, with
# one or more key ranges per tile
MODES = [(1, False), (1, True), (3, True)]


def _ws(g, n_q, win_len, splits, use_ws=True):
    """A NaN-filled workspace for `splits` key ranges, or None."""
    if not use_ws:
        return None
    n = argus.window_prefill_workspace_bytes(g, n_q, win_len, splits)
    return torch.full((max(n, 16) // 4,), float("nan"), dtype=torch.float32, device=DEV)


def _run_windows(Hq, Hkv, n_q, ctx, windows, seed, scale=None, splits=1, use_ws=False, vmul=1.0, D=128):
    q, k, v, q64, k64, v64 = _data(Hq, Hkv, n_q, ctx, seed, D)
    if vmul != 1.0:
        v = (v.float() * vmul).to(torch.bfloat16)
        v64 = C.bf16_bits_to_f64(W.to_bits(v))
    scale = W.softmax_scale(D) if scale is None else scale
    g = argus.geom(Hq, Hkv, D, 16)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    kv_len = ctx + n_q
    acc_o = torch.zeros((Hq, n_q, D), dtype=torch.float32, device=DEV)
    acc_l = torch.full((Hq, n_q), float("-inf"), dtype=torch.float32, device=DEV)
    for wi, (w0, w1) in enumerate(windows):
        ws = _ws(g, n_q, w1 - w0, splits, use_ws)
        argus.window_prefill_attn(g, n_q, qd, kd[:, w0:], vd[:, w0:], kv_len * D, w1 - w0, w0, ctx, scale,
                                  acc_o, acc_l, 1 if wi > 0 else 0, num_splits=splits, ws=ws)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.window_attention(q64, k64, v64, 0, ctx, scale)
    return acc_o.cpu().numpy(), acc_l.cpu().numpy(), ref_o, ref_l


def _check(go, gl, ro, rl):
    t = 1e-3 * np.abs(ro).max() + 1e-4
    err = np.abs(go - ro).max()
    assert err <= t, "max err %.3g > tol %.3g" % (err, t)
    assert np.abs(gl - rl).max() <= 1e-4 * np.abs(rl).max() + 1e-5


@pytest.mark.parametrize("splits,use_ws", MODES + [(2, True)])
def test_single_window_full_view_small(splits, use_ws):
    go, gl, ro, rl = _run_windows(1, 1, 128, 128, [(0, 128)], seed=501, splits=splits, use_ws=use_ws)
    # the chunk itself is not part of this window: compare against the cache-only oracle
    q, k, v, q64, k64, v64 = _data(1, 1, 128, 128, 501)
    ro, rl = oracle.window_attention(q64, k64[:, :128], v64[:, :128], 0, 128, W.softmax_scale(128))
    _check(go, gl, ro, rl)


@pytest.mark.parametrize("splits,use_ws", MODES + [(2, True), (5, True)])
@pytest.mark.parametrize("D", [128, 64])
def test_causal_chunk_window_only(splits, use_ws, D):
    # a 256-row chunk attending only to itself: causal inside the chunk; with 5
    # key ranges over at most 2 visible blocks some ranges are empty
    q, k, v, q64, k64, v64 = _data(2, 1, 256, 0, 503, D)
    g = argus.geom(2, 1, D, 16)
    acc_o = torch.empty((2, 256, D), dtype=torch.float32, device=DEV)
    acc_l = torch.empty((2, 256), dtype=torch.float32, device=DEV)
    argus.window_prefill_attn(g, 256, q.to(DEV), k.to(DEV), v.to(DEV), 0, 256, 1000, 1000,
                              W.softmax_scale(D), acc_o, acc_l, 0, num_splits=splits,
                              ws=_ws(g, 256, 256, splits, use_ws))
    torch.cuda.synchronize()
    ro, rl = oracle.window_attention(q64, k64, v64, 1000, 1000, W.softmax_scale(D))
    _check(acc_o.cpu().numpy(), acc_l.cpu().numpy(), ro, rl)


@pytest.mark.parametrize("splits,use_ws", MODES)
@pytest.mark.parametrize("Hq,Hkv", [(2, 1), (16, 2)])
@pytest.mark.parametrize("D", [128, 64])
def test_windows_folded_equal_single_pass(Hq, Hkv, splits, use_ws, D):
    n_q, ctx = 256, 768
    windows = [(0, 256), (256, 768), (768, 1024)]      # two cache windows, then the chunk
    go, gl, ro, rl = _run_windows(Hq, Hkv, n_q, ctx, windows, seed=505 + Hq, splits=splits, use_ws=use_ws, D=D)
    _check(go, gl, ro, rl)


@pytest.mark.parametrize("splits,use_ws", MODES + [(4, True)])
def test_window_beyond_every_query_is_identity(splits, use_ws):
    q, k, v, q64, k64, v64 = _data(2, 1, 128, 256, 509)
    g = argus.geom(2, 1, 128, 16)
    acc_o = torch.randn((2, 128, 128), device=DEV)
    acc_l = torch.randn((2, 128), device=DEV)
    o0, l0 = acc_o.clone(), acc_l.clone()
    # keys at positions 10_000.. are after every query (positions 256..383)
    argus.window_prefill_attn(g, 128, q.to(DEV), k.to(DEV), v.to(DEV), 0, 128, 10_000, 256,
                              W.softmax_scale(128), acc_o, acc_l, 1, num_splits=splits,
                              ws=_ws(g, 128, 128, splits, use_ws))
    torch.cuda.synchronize()
    assert torch.equal(acc_o, o0) and torch.equal(acc_l, l0)


def test_rejects_unsupported_shapes():
    g = argus.geom(2, 1, 96, 16)
    t = torch.zeros((2, 128, 96), dtype=torch.bfloat16, device=DEV)
    o = torch.zeros((2, 128, 96), device=DEV)
    l = torch.zeros((2, 128), device=DEV)
    with pytest.raises(argus.ArgusError) as e:
        argus.window_prefill_attn(g, 128, t, t, t, 0, 128, 0, 0, 0.1, o, l, 0)
    assert e.value.status == 2


def test_automatic_splits_with_a_long_window():
    """4096 cached keys in one window: the automatic split count (> 1 here)
    must give the same result as one CTA per tile, within the tolerance."""
    Hq, Hkv, n_q, ctx = 16, 2, 128, 4096
    g = argus.geom(Hq, Hkv, 128, 16)
    assert argus.window_prefill_workspace_bytes(g, n_q, ctx, 0) > 0
    go, gl, ro, rl = _run_windows(Hq, Hkv, n_q, ctx, [(0, ctx), (ctx, ctx + n_q)], seed=511, splits=0,
                                  use_ws=True)
    _check(go, gl, ro, rl)


@pytest.mark.parametrize("vmul", [3.0e5, 2.0 ** -20])
@pytest.mark.parametrize("D", [128, 64])
def test_fp16_value_path_scales_v_outside_the_fp16_range(vmul, D):
    """V far above fp16's range is scaled by a power of two before the fp16
    copy (and the output scaled back); V far below keeps its accuracy."""
    go, gl, ro, rl = _run_windows(2, 1, 128, 256, [(0, 256), (256, 384)], seed=513, splits=2, use_ws=True,
                                  vmul=vmul, D=D)
    _check(go, gl, ro, rl)


def test_split_workspace_too_small_is_rejected():
    g = argus.geom(2, 1, 128, 16)
    t = torch.zeros((2, 256, 128), dtype=torch.bfloat16, device=DEV)
    o = torch.zeros((2, 256, 128), device=DEV)
    l = torch.zeros((2, 256), device=DEV)
    need = argus.window_prefill_workspace_bytes(g, 256, 256, 2)
    small = torch.zeros((need - 16) // 4, dtype=torch.float32, device=DEV)
    with pytest.raises(argus.ArgusError) as e:
        argus.window_prefill_attn(g, 256, t, t, t, 0, 256, 0, 0, 0.1, o, l, 0, num_splits=2, ws=small)
    assert e.value.status == 3


@pytest.mark.parametrize("splits,use_ws", MODES)
@pytest.mark.parametrize("ramp", ["rising", "late_key"])
@pytest.mark.parametrize("D", [128, 64])
def test_scores_growing_past_the_lazy_rescale_threshold(splits, use_ws, ramp, D):
    """Key blocks whose scores rise by more than 2^8 (8 in log2 units) over the
    running maximum, block after block: the softmax must rescale the TMEM
    accumulator of O (the lazy max moves).  "rising" scales the keys of block j
    by 1 + 1.5 j, so each softmax group (even / odd blocks) sees a jump of about
    10 at every block; "late_key" plants one key per KV head in the last cache
    block aligned with the first query rows, far above everything before it.
    The host checks on the oracle's own scores that such jumps occur."""
    Hq, Hkv, n_q, ctx = 2, 1, 128, 1024
    q, k, v, q64, k64, v64 = _data(Hq, Hkv, n_q, ctx, 521, D)
    kf = k.float()
    if ramp == "rising":
        for j in range(ctx // 128):
            kf[:, j * 128:(j + 1) * 128] *= 1.0 + 1.5 * j
    else:
        kf[:, 7 * 128 + 5] = q.float()[0, 0] * 12.0
        kf[:, 6 * 128 + 9] = q.float()[1, 3] * 9.0
    k = kf.to(torch.bfloat16)
    k64 = C.bf16_bits_to_f64(W.to_bits(k))
    scale = W.softmax_scale(D)
    # the branch is reached: some row's block maximum (log2 units) jumps by > 8
    # over the maximum of the earlier blocks its softmax group saw
    s2 = np.einsum("hqd,hkd->hqk", q64.reshape(Hq, n_q, D), np.repeat(k64[:, :ctx], Hq // Hkv, 0)) * scale / math.log(2)
    bm = s2.reshape(Hq, n_q, ctx // 128, 128).max(axis=3)           # [Hq][n_q][block]
    jumps = [np.max(bm[:, :, j] - np.maximum.accumulate(bm[:, :, g::2], axis=2)[:, :, (j - g) // 2 - 1])
             for g in (0, 1) for j in range(g + 2, ctx // 128, 2)]
    assert max(jumps) > 8.0
    g = argus.geom(Hq, Hkv, D, 16)
    kd, vd = k.to(DEV), v.to(DEV)
    kv_len = ctx + n_q
    acc_o = torch.zeros((Hq, n_q, D), dtype=torch.float32, device=DEV)
    acc_l = torch.full((Hq, n_q), float("-inf"), dtype=torch.float32, device=DEV)
    for wi, (w0, w1) in enumerate([(0, ctx), (ctx, kv_len)]):
        argus.window_prefill_attn(g, n_q, q.to(DEV), kd[:, w0:], vd[:, w0:], kv_len * D, w1 - w0, w0, ctx,
                                  scale, acc_o, acc_l, 1 if wi else 0, num_splits=splits,
                                  ws=_ws(g, n_q, w1 - w0, splits, use_ws))
    torch.cuda.synchronize()
    ro, rl = oracle.window_attention(q64, k64, v64, 0, ctx, scale)
    _check(acc_o.cpu().numpy(), acc_l.cpu().numpy(), ro, rl)
