"""argus_paged_decode_attn on the GPU against the double-precision oracle.

Tolerance (stated for attention outputs): max|err| <= 1e-3 * max|ref| + 1e-4 on
the fp32 output; the fp16 or bf16 output must equal the round-to-nearest-even
of the kernel's own fp32 output.
"""

import math

import numpy as np
import pytest
import torch

import mixed_precision_paged_argus_gb300.argus as argus
from mixed_precision_paged_argus_gb300 import workloads as W
import oracle
from oracle import codecs as C
from paged_cases import DEV, build_case, run_decode, tol

pytestmark = pytest.mark.gpu


def _check(c, out, out32, lse, sel=None, cnt=None, width=0, expect_bad=0, window=0, sinks=0):
    ref, ref_lse, bad = oracle.paged_decode(c.q64, c.Hkv, c.P, c.opools, c.page_codec, c.table, c.lens,
                                            c.scale, sel_pages=sel, sel_count=cnt, sel_width=width,
                                            window=window, sinks=sinks)
    assert bad == expect_bad
    got = out32.cpu().numpy().astype(np.float64)
    t = tol(ref)
    err = np.abs(got - ref).max()
    assert err <= t, "fp32 output max err %.3g > tol %.3g" % (err, t)
    # the 16-bit output is the round-to-nearest-even of the kernel's own fp32 output
    assert torch.equal(out.cpu(), out32.cpu().to(out.dtype))
    gl = lse.cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(gl), fin)
    assert np.all(np.abs(gl[fin] - ref_lse[fin]) <= 1e-4 * np.maximum(1.0, np.abs(ref_lse[fin])))
    return err


@pytest.mark.parametrize("codec", [W.FP16, W.FP8_E4M3, W.INT8, W.INT4_G32, W.INT2_G32, W.INT1_G32])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 7, 8])
def test_single_codec_fp16_query(codec, D, G):
    Hkv, P = 2, 16
    lens = [150, 33, 16]
    maxp = 10
    pc = np.full((3, maxp), codec)
    c = build_case(G * Hkv, Hkv, D, P, lens, pc, W.FP16, seed=11 + codec, outliers=True)
    out, out32, lse, _ = run_decode(c, num_splits=3)
    _check(c, out, out32, lse)


@pytest.mark.parametrize("codec", [W.BF16, W.FP8_E4M3, W.INT8, W.INT4_G32, W.INT2_G32, W.INT1_G32])
@pytest.mark.parametrize("G", [4, 8])
def test_single_codec_bf16_query(codec, G):
    Hkv, D, P = 2, 128, 16
    lens = [300, 17]
    pc = np.full((2, 20), codec)
    c = build_case(G * Hkv, Hkv, D, P, lens, pc, W.BF16, seed=23 + codec)
    out, out32, lse, _ = run_decode(c, out_dtype=torch.bfloat16, num_splits=0)
    _check(c, out, out32, lse)


def test_mixed_tiers_like_the_mixed_tier_workload():
    """14 q / 2 KV heads, head_dim 64, newest pages FP16, then FP8, INT8, INT4."""
    Hq, Hkv, D, P = 14, 2, 64, 64
    n = 16
    pc = W.mixed_tier_codecs(n).reshape(1, n)
    c = build_case(Hq, Hkv, D, P, [n * P - 5], pc, W.FP16, seed=31, outliers=True)
    for splits in (1, 4, 0):
        out, out32, lse, _ = run_decode(c, num_splits=splits)
        _check(c, out, out32, lse)


def test_mixed_bf16_and_quantized_pages_bf16_query():
    Hq, Hkv, D, P = 16, 2, 128, 32
    rng = np.random.default_rng(3)
    pc = rng.choice([W.BF16, W.FP8_E4M3, W.INT8, W.INT4_G32], size=(3, 12))
    c = build_case(Hq, Hkv, D, P, [384, 200, 1], pc, W.BF16, seed=41)
    out, out32, lse, _ = run_decode(c, out_dtype=torch.bfloat16, num_splits=5)
    _check(c, out, out32, lse)


def test_tiny_fp16_workload_full_size():
    """Batch 1, 14 q / 2 KV heads, head_dim 64, 4 FP16 pages of 1024 tokens."""
    Hq, Hkv, D, P = 14, 2, 64, 1024
    pc = np.zeros((1, 4), np.int64)
    c = build_case(Hq, Hkv, D, P, [4096], pc, W.FP16, seed=1000, permute=False)
    out, out32, lse, _ = run_decode(c)
    _check(c, out, out32, lse)


def test_ragged_batch_permuted_slots_and_empty_rows():
    Hq, Hkv, D, P = 32, 8, 128, 16
    lens = [0, 1, 15, 16, 17, 257, 1000]
    maxp = 64
    pc = np.full((len(lens), maxp), W.FP8_E4M3)
    c = build_case(Hq, Hkv, D, P, lens, pc, W.BF16, seed=51, extra_slots=9)
    for splits in (0, 1, 2, 9):
        out, out32, lse, _ = run_decode(c, out_dtype=torch.bfloat16, num_splits=splits)
        _check(c, out, out32, lse)
        assert torch.all(out32[0] == 0) and torch.all(torch.isinf(lse[0]))


@pytest.mark.parametrize("splits", [0, 1, 3, 50])
def test_selected_page_lists_and_invalid_entries(splits):
    """Selected entries are dealt round-robin over the splits: split counts
    that do not divide a row's count, rows with fewer entries than splits, and
    a request above the list width (clamped to it)."""
    Hq, Hkv, D, P = 32, 4, 128, 64
    maxp = 40
    lens = [40 * 64 - 10, 20 * 64 + 3]
    pc = np.full((2, maxp), W.FP8_E4M3)
    c = build_case(Hq, Hkv, D, P, lens, pc, W.BF16, seed=61)
    width = 12
    rng = np.random.default_rng(62)
    sel = np.full((2, Hkv, width), -1, np.int32)
    cnt = np.zeros((2, Hkv), np.int32)
    for b in range(2):
        n = -(-lens[b] // P)
        for h in range(Hkv):
            k = int(rng.integers(1, 9))
            pages = sorted(rng.choice(n - 1, size=k, replace=False).tolist() + [n - 1])
            sel[b, h, :len(pages)] = pages
            cnt[b, h] = len(pages)
    sel[1, 2, cnt[1, 2]] = 35           # beyond the sequence's pages -> skipped, counted
    cnt[1, 2] += 1
    cnt[0, 3] = width + 3               # more than the width -> clamped, counted
    sel[0, 3, :] = np.arange(width)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, out32, lse, _ = run_decode(c, out_dtype=torch.bfloat16,
                                    sel=torch.from_numpy(sel).to(DEV), sel_count=torch.from_numpy(cnt).to(DEV),
                                    sel_width=width, status=status, num_splits=splits)
    _check(c, out, out32, lse, sel=sel, cnt=cnt, width=width, expect_bad=2)
    assert int(status.item()) == 2


def test_bad_slot_is_skipped_and_counted():
    Hq, Hkv, D, P = 8, 1, 64, 16
    pc = np.full((1, 6), W.INT4_G32)
    c = build_case(Hq, Hkv, D, P, [96], pc, W.FP16, seed=71)
    table = c.table.copy()
    table[0, 2] = 1000
    c.table = table
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, out32, lse, _ = run_decode(c, status=status, table=torch.from_numpy(table).to(DEV))
    _check(c, out, out32, lse, expect_bad=1)
    assert int(status.item()) == 1


def test_workspace_needs_no_initialisation_and_is_repeatable():
    Hq, Hkv, D, P = 14, 2, 64, 64
    pc = W.mixed_tier_codecs(16).reshape(1, 16)
    c = build_case(Hq, Hkv, D, P, [16 * 64], pc, W.FP16, seed=81)
    out_a, o32a, lse, _ = run_decode(c, num_splits=8)
    _check(c, out_a, o32a, lse)
    args = argus.decode_args(c.g, c.B, c.q, c.pools, c.d_codec, c.d_table, c.d_lens, c.max_pages, c.scale,
                             out_f32=torch.empty_like(o32a), num_splits=8)
    ws = torch.full((argus.decode_workspace_bytes(args),), 0xFF, dtype=torch.uint8, device=DEV)  # NaN-filled
    for _ in range(2):
        argus.paged_decode_attn(args, ws)
        torch.cuda.synchronize()
        assert torch.equal(args._keep[9], o32a)


def test_unsupported_and_invalid_arguments():
    Hq, Hkv, D, P = 8, 1, 64, 16
    pc = np.full((1, 2), W.BF16)
    c = build_case(Hq, Hkv, D, P, [20], pc, W.BF16, q_dtype=W.FP16, seed=91)
    with pytest.raises(argus.ArgusError) as e:
        run_decode(c)
    assert e.value.status == 2          # BF16 pages with an FP16 query: fail closed
    c2 = build_case(Hq, Hkv, D, P, [20], np.full((1, 2), W.FP16), W.FP16, seed=92)
    args = argus.decode_args(c2.g, 1, c2.q, c2.pools, c2.d_codec, c2.d_table, c2.d_lens, 2, c2.scale,
                             out_f32=torch.empty((1, Hq, D), device=DEV), num_splits=4)
    need = argus.decode_workspace_bytes(args)
    small = torch.zeros(need - 4, dtype=torch.uint8, device=DEV)
    with pytest.raises(argus.ArgusError) as e:
        argus.paged_decode_attn(args, small)
    assert e.value.status == 3


def test_layer_chain_with_programmatic_dependent_launch():
    """Back-to-back calls with pdl=1 (each grid may start in its predecessor's
    tail) give the same bits as ordinary stream order, eagerly and replayed
    from a CUDA graph, and match the oracle."""
    Hq, Hkv, D, P = 14, 2, 64, 64
    n = 16
    pc = W.mixed_tier_codecs(n).reshape(1, n)
    cases = [build_case(Hq, Hkv, D, P, [n * P - 7 * l], pc, W.FP16, seed=300 + l, outliers=True) for l in range(4)]
    want = []
    for c in cases:
        out, out32, lse, _ = run_decode(c, num_splits=0)
        _check(c, out, out32, lse)
        want.append(out32.clone())
    outs = [torch.empty_like(w) for w in want]
    args = [argus.decode_args(c.g, c.B, c.q, c.pools, c.d_codec, c.d_table, c.d_lens, c.max_pages, c.scale,
                              out_f32=o, pdl=True) for c, o in zip(cases, outs)]
    ws = torch.empty(max(argus.decode_workspace_bytes(a) for a in args), dtype=torch.uint8, device=DEV)
    stream = torch.cuda.Stream(device=DEV)
    with torch.cuda.stream(stream):
        for _ in range(3):
            for a in args:
                argus.paged_decode_attn(a, ws, stream=stream)
        stream.synchronize()
        for o, w in zip(outs, want):
            assert torch.equal(o, w)
            o.zero_()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for a in args:
                argus.paged_decode_attn(a, ws, stream=stream)
        graph.replay()
        graph.replay()
    torch.cuda.synchronize()
    for o, w in zip(outs, want):
        assert torch.equal(o, w)


@pytest.mark.parametrize("codec", [W.FP8_E4M3, W.INT8])
@pytest.mark.parametrize("Hkv,D", [(1, 64), (3, 128), (40, 64)])
def test_scale_rows_loaded_by_the_producer(codec, Hkv, D):
    """Odd KV-head counts, or scale rows wider than the chunk's meta area,
    take the producer-side scale loads instead of the bulk-copied row."""
    P = 16
    pc = np.full((2, 8), codec)
    c = build_case(2 * Hkv, Hkv, D, P, [100, 128], pc, W.FP16, seed=400 + Hkv + codec, outliers=True)
    out, out32, lse, _ = run_decode(c, num_splits=2)
    _check(c, out, out32, lse)


@pytest.mark.parametrize("q_dtype", [W.FP16, W.BF16])
def test_narrow_ring_with_mixed_byte_and_nibble_codecs(q_dtype):
    """head_dim 128 with FP8, INT8 and INT4 pools only runs the narrow ring
    (16 chunks per stage, two per warp); chunks of different codecs share a
    warp and a stage."""
    Hq, Hkv, D, P = 16, 2, 128, 16
    rng = np.random.default_rng(77)
    pc = rng.choice([W.FP8_E4M3, W.INT8, W.INT4_G32], size=(3, 40))
    c = build_case(Hq, Hkv, D, P, [640, 333, 17], pc, q_dtype, seed=501, outliers=True)
    for splits in (0, 1, 3):
        out, out32, lse, _ = run_decode(c, out_dtype=torch.float16 if q_dtype == W.FP16 else torch.bfloat16,
                                        num_splits=splits)
        _check(c, out, out32, lse)


def test_split_count_is_capped_and_many_splits_fold():
    """An explicit split count above the cap is clamped (at most 512 splits per
    row); with hundreds of splits the combine folds several batches per thread."""
    Hq, Hkv, D, P = 8, 1, 64, 16
    n = 2000
    pc = np.full((1, n), W.FP16)
    c = build_case(Hq, Hkv, D, P, [n * P - 3], pc, W.FP16, seed=601, permute=False)
    out, out32, lse, ws = run_decode(c, num_splits=100000)
    _check(c, out, out32, lse)
    args = argus.decode_args(c.g, c.B, c.q, c.pools, c.d_codec, c.d_table, c.d_lens, c.max_pages, c.scale,
                             out_f32=torch.empty_like(out32), num_splits=100000)
    # workspace = splits * G * (D + 1) floats per row: at most 512 splits
    assert argus.decode_workspace_bytes(args) <= 512 * Hq * (D + 1) * 4


# ---------------------------------------------------------------- sliding window + sink tokens

WINDOWS = [(5, 0), (5, 4), (40, 4), (33, 16), (1, 33), (17, 15), (100000, 4), (64, 64)]


@pytest.mark.parametrize("W_,S_", WINDOWS)
@pytest.mark.parametrize("P", [16, 64])
def test_sliding_window_with_sinks_mixed_codecs(W_, S_, P):
    """Windows that start mid-chunk and mid-page, sinks that end mid-chunk or
    overlap the window, windows wider than the sequence; ragged rows."""
    Hq, Hkv, D = 14, 2, 64
    lens = [0, 1, 37, 300, 1023]
    maxp = -(-max(lens) // P)
    rng = np.random.default_rng(P + W_ + S_)
    pc = rng.choice([W.FP16, W.FP8_E4M3, W.INT8, W.INT4_G32], size=(len(lens), maxp))
    c = build_case(Hq, Hkv, D, P, lens, pc, W.FP16, seed=500 + P, outliers=True)
    for splits in (0, 1, 3):
        out, out32, lse, _ = run_decode(c, num_splits=splits, window=W_, sinks=S_)
        _check(c, out, out32, lse, window=W_, sinks=S_)


@pytest.mark.parametrize("q_dtype", [W.FP16, W.BF16])
def test_sliding_window_head_dim_128_narrow_and_wide_rings(q_dtype):
    Hq, Hkv, D, P = 32, 8, 128, 16
    lens = [2000, 513, 16]
    maxp = 125
    codecs = [W.FP8_E4M3, W.INT4_G32] if q_dtype == W.FP16 else [W.BF16, W.INT8]
    pc = np.random.default_rng(5).choice(codecs, size=(3, maxp))
    c = build_case(Hq, Hkv, D, P, lens, pc, q_dtype, seed=520)
    out_dtype = torch.float16 if q_dtype == W.FP16 else torch.bfloat16
    for W_, S_ in [(256, 4), (1000, 0), (77, 20)]:
        out, out32, lse, _ = run_decode(c, out_dtype=out_dtype, window=W_, sinks=S_)
        _check(c, out, out32, lse, window=W_, sinks=S_)


def test_sliding_window_mixed_tier_layer_full_size():
    """One layer of the mixed-tier workload (16 x 1024-token pages, 14 / 2 heads,
    head_dim 64) with a 4096-token window and 4 sink tokens."""
    Hq, Hkv, D, P = 14, 2, 64, 1024
    pc = W.mixed_tier_codecs(16).reshape(1, 16)
    c = build_case(Hq, Hkv, D, P, [16 * 1024], pc, W.FP16, seed=530, outliers=True)
    out, out32, lse, _ = run_decode(c, window=4096, sinks=4)
    _check(c, out, out32, lse, window=4096, sinks=4)
    full = run_decode(c)[1]
    assert not torch.allclose(full, out32)      # the window changes the result


def test_sliding_window_bad_slots_counted_once_per_read_page():
    Hq, Hkv, D, P = 8, 2, 64, 16
    pc = np.full((1, 8), W.INT8)
    c = build_case(Hq, Hkv, D, P, [128], pc, W.FP16, seed=540)
    table = c.table.copy()
    table[0, 1] = 1000    # positions 16..31: outside sinks 0..3 and window 58..127
    table[0, 3] = 1001    # positions 48..63: the window starts mid-page (58)
    table[0, 0] = 1002    # positions 0..15: sink tokens 0..3
    c.table = table
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, out32, lse, _ = run_decode(c, status=status, table=torch.from_numpy(table).to(DEV),
                                    window=70, sinks=4, num_splits=2)
    _check(c, out, out32, lse, expect_bad=2 * Hkv, window=70, sinks=4)
    assert int(status.item()) == 2 * Hkv
    # one page holding both sink tokens and the window's start: counted once
    c2 = build_case(Hq, Hkv, D, 64, [100], np.full((1, 2), W.INT8), W.FP16, seed=541)
    t2 = c2.table.copy()
    t2[0, 0] = 1000       # positions 0..63 hold the sinks 0..3 and the window from 40
    c2.table = t2
    status.zero_()
    out, out32, lse, _ = run_decode(c2, status=status, table=torch.from_numpy(t2).to(DEV), window=60, sinks=4)
    _check(c2, out, out32, lse, expect_bad=Hkv, window=60, sinks=4)
    assert int(status.item()) == Hkv


def test_sliding_window_argument_checks_and_smaller_workspace():
    Hq, Hkv, D, P = 8, 1, 64, 16
    c = build_case(Hq, Hkv, D, P, [200], np.full((1, 13), W.FP16), W.FP16, seed=550)
    with pytest.raises(argus.ArgusError) as e:
        run_decode(c, window=-1)
    assert e.value.status == 1
    with pytest.raises(argus.ArgusError) as e:
        run_decode(c, window=8, sinks=-2)
    assert e.value.status == 1
    sel = torch.zeros((1, Hkv, 2), dtype=torch.int32, device=DEV)
    cnt = torch.ones((1, Hkv), dtype=torch.int32, device=DEV)
    with pytest.raises(argus.ArgusError) as e:
        run_decode(c, sel=sel, sel_count=cnt, sel_width=2, window=8)
    assert e.value.status == 2
    def ws_bytes(**kw):
        a = argus.decode_args(c.g, 1, c.q, c.pools, c.d_codec, c.d_table, c.d_lens, 4096, c.scale,
                              out_f32=torch.empty((1, Hq, D), device=DEV), num_splits=0, **kw)
        return argus.decode_workspace_bytes(a)
    assert ws_bytes(window_tokens=64, sink_tokens=4) < ws_bytes()


# ---------------------------------------------------------------- INT2 tier

@pytest.mark.parametrize("q_dtype", [W.FP16, W.BF16])
@pytest.mark.parametrize("D", [64, 128])
def test_five_tiers_with_int2_oldest(q_dtype, D):
    """Newest pages FP16 (BF16 for a bf16 query), then FP8, INT8, INT4 and the
    oldest INT2; ragged rows, several split counts, with and without a window."""
    Hq, Hkv, P = 16, 2, 64
    n = 20
    top = W.FP16 if q_dtype == W.FP16 else W.BF16
    row = np.array([W.INT2_G32] * 4 + [W.INT4_G32] * 4 + [W.INT8] * 4 + [W.FP8_E4M3] * 4 + [top] * 4)
    pc = np.stack([row, np.roll(row, 7)])
    c = build_case(Hq, Hkv, D, P, [n * P - 9, 700], pc, q_dtype, seed=600 + D, outliers=True)
    out_dtype = torch.float16 if q_dtype == W.FP16 else torch.bfloat16
    for splits in (0, 1, 5):
        out, out32, lse, _ = run_decode(c, out_dtype=out_dtype, num_splits=splits)
        _check(c, out, out32, lse)
    out, out32, lse, _ = run_decode(c, out_dtype=out_dtype, window=300, sinks=4)
    _check(c, out, out32, lse, window=300, sinks=4)


def test_int2_selected_pages():
    Hq, Hkv, D, P = 32, 4, 128, 64
    maxp = 24
    lens = [24 * 64 - 3, 10 * 64 + 5]
    pc = np.full((2, maxp), W.INT2_G32)
    c = build_case(Hq, Hkv, D, P, lens, pc, W.BF16, seed=610)
    width = 8
    sel = np.full((2, Hkv, width), -1, np.int32)
    cnt = np.zeros((2, Hkv), np.int32)
    rng = np.random.default_rng(611)
    for b in range(2):
        n = -(-lens[b] // P)
        for h in range(Hkv):
            pages = sorted(rng.choice(n - 1, size=4, replace=False).tolist() + [n - 1])
            sel[b, h, :len(pages)] = pages
            cnt[b, h] = len(pages)
    out, out32, lse, _ = run_decode(c, out_dtype=torch.bfloat16, sel=torch.from_numpy(sel).to(DEV),
                                    sel_count=torch.from_numpy(cnt).to(DEV), sel_width=width)
    _check(c, out, out32, lse, sel=sel, cnt=cnt, width=width)


@pytest.mark.parametrize("q_dtype", [W.FP16, W.BF16])
@pytest.mark.parametrize("D", [64, 128])
def test_six_tiers_with_int1_oldest(q_dtype, D):
    """Every tier in one row, oldest first: 1-bit, INT2, INT4, INT8, FP8 and the
    16-bit tier; ragged rows, several split counts, with and without a window."""
    Hq, Hkv, P = 16, 2, 64
    top = W.FP16 if q_dtype == W.FP16 else W.BF16
    row = np.array([W.INT1_G32] * 3 + [W.INT2_G32] * 3 + [W.INT4_G32] * 3 + [W.INT8] * 3 + [W.FP8_E4M3] * 3 + [top] * 3)
    pc = np.stack([row, np.roll(row, 5)])
    c = build_case(Hq, Hkv, D, P, [18 * P - 11, 600], pc, q_dtype, seed=660 + D, outliers=True)
    out_dtype = torch.float16 if q_dtype == W.FP16 else torch.bfloat16
    for splits in (0, 1, 4):
        out, out32, lse, _ = run_decode(c, out_dtype=out_dtype, num_splits=splits)
        _check(c, out, out32, lse)
    out, out32, lse, _ = run_decode(c, out_dtype=out_dtype, window=250, sinks=4)
    _check(c, out, out32, lse, window=250, sinks=4)
