"""Parity at the full sizes of the benchmark workloads, in bench.py's launch
configuration (automatic splits, programmatic dependent launch, CUDA-graph
replay where the bench uses it), on outputs the oracle can afford.

Inputs come from the seeded generators on the device; the oracle receives the
generator's source pages (copied to the host) and demotes them itself.
Tolerance on attention outputs: max|err| <= 1e-3 * max|ref| + 1e-4.
"""

import math

import numpy as np
import pytest
import torch

import bench
import mixed_precision_paged_argus_gb300.argus as argus
from mixed_precision_paged_argus_gb300 import workloads as W
import oracle
from oracle import codecs as C

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = "cuda"


def _tol(ref):
    return 1e-3 * float(np.abs(ref).max()) + 1e-4


def test_mixed_tier_all_24_layers_graph_replay_layers_0_and_23():
    dev = torch.device(DEV)
    g, pools, tables, qs, codec_row, lens = bench.build_mixed_tier(dev)
    outs = [torch.empty((1, bench.HQ, bench.D), dtype=torch.float16, device=dev) for _ in range(bench.LAYERS)]
    out32 = [torch.empty((1, bench.HQ, bench.D), dtype=torch.float32, device=dev) for _ in range(bench.LAYERS)]
    args = [argus.decode_args(g, 1, qs[l], pools, codec_row, tables[l], lens, bench.NPAGES,
                              W.softmax_scale(bench.D), out=outs[l], out_f32=out32[l]) for l in range(bench.LAYERS)]
    ws = torch.empty(max(argus.decode_workspace_bytes(a) for a in args), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for a in args:
            argus.paged_decode_attn(a, ws, stream=stream)
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for a in args:
                argus.paged_decode_attn(a, ws, stream=stream)
    for o in out32:
        o.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    tiers = W.mixed_tier_codecs(bench.NPAGES)
    for layer in (0, bench.LAYERS - 1):
        src = W.to_bits(W.normal((bench.NPAGES, 2, bench.HKV, bench.P, bench.D), W.FP16,
                                 W.seed_of("mixed_tier", layer, 1), device=dev,
                                 outlier_seed=W.seed_of("mixed_tier", layer, 5)))
        q64 = C.f16_bits_to_f64(W.to_bits(qs[layer]))
        table = tables[layer].cpu().numpy()
        opools = {}
        for codec in (W.FP16, W.FP8_E4M3, W.INT8, W.INT4_G32):
            pages = [p for p in range(bench.NPAGES) if tiers[p] == codec]
            n_slots = 4 * bench.LAYERS
            codes, meta = C.alloc_pool(codec, n_slots, bench.HKV, bench.P, bench.D)
            C.quantize_pages(src, C.CODEC_FP16, pages, codec, codes, meta, [int(table[0, p]) for p in pages])
            opools[codec] = (codes, meta)
        ref, _, bad = oracle.paged_decode(q64, bench.HKV, bench.P, opools, tiers.reshape(1, -1).astype(np.uint8),
                                          table, np.array([bench.CTX]), W.softmax_scale(bench.D))
        got = out32[layer].cpu().numpy()
        assert bad == 0
        assert np.abs(got - ref).max() <= _tol(ref), "layer %d" % layer
        assert torch.equal(outs[layer].cpu(), out32[layer].cpu().to(torch.float16))


@pytest.mark.parametrize("codec", [W.BF16, W.FP8_E4M3])
def test_batched_full_batch_sampled_rows(codec):
    B, Hq, Hkv, D, P, MAXP = 32, 32, 8, 128, 16, 2048
    dev = torch.device(DEV)
    lens = W.uniform_ints(B, 8192, 32768, W.seed_of("batched", 0, 3))
    table, n_slots = W.paged_block_table(lens, P, MAXP, W.seed_of("batched", 0, 4))
    g = argus.geom(Hq, Hkv, D, P)
    src = W.normal((n_slots, 2, Hkv, P, D), W.BF16, W.seed_of("batched", 0, 1), device=dev)
    pool = argus.Pool(W.BF16, src, None, n_slots)
    if codec == W.FP8_E4M3:
        ids = torch.arange(n_slots, dtype=torch.int32, device=dev)
        pool = argus.Pool.empty(W.FP8_E4M3, n_slots, Hkv, P, D, device=dev)
        argus.quantize_pages(g, W.BF16, src, n_slots, ids, pool, ids, n_slots)
    q = W.normal((B, Hq, D), W.BF16, W.seed_of("batched", 0, 0), device=dev)
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
    out32 = torch.full((B, Hq, D), float("nan"), device=dev)
    lse = torch.empty((B, Hq), device=dev)
    a = argus.decode_args(g, B, q, [pool], torch.full((B, MAXP), codec, dtype=torch.uint8, device=dev),
                          torch.from_numpy(table).to(dev), torch.from_numpy(lens.astype(np.int32)).to(dev), MAXP,
                          W.softmax_scale(D), out=out, out_f32=out32, lse2_out=lse)
    ws = torch.empty(argus.decode_workspace_bytes(a), dtype=torch.uint8, device=dev)
    argus.paged_decode_attn(a, ws)
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), out32.cpu().to(torch.bfloat16))
    q64 = C.bf16_bits_to_f64(W.to_bits(q))
    for b in (0, int(np.argmax(lens))):
        n = (int(lens[b]) + P - 1) // P
        slots = table[b, :n]
        src_rows = W.to_bits(src[torch.from_numpy(slots.astype(np.int64)).to(dev)])   # [n][2][Hkv][P][D]
        codes, meta = C.alloc_pool(codec, n, Hkv, P, D)
        C.quantize_pages(src_rows, C.CODEC_BF16, list(range(n)), codec, codes, meta, list(range(n)))
        ref, ref_l, _ = oracle.paged_decode(q64[b:b + 1], Hkv, P, {codec: (codes, meta)},
                                            np.full((1, n), codec, np.uint8), np.arange(n, dtype=np.int32)[None],
                                            np.array([lens[b]]), W.softmax_scale(D))
        got = out32[b:b + 1].cpu().numpy()
        assert np.abs(got - ref).max() <= _tol(ref), "row %d" % b
        assert np.abs(lse[b].cpu().numpy() - ref_l[0]).max() <= 1e-4 * np.abs(ref_l).max()


def test_sparse_one_layer_full_size_sampled_sequence():
    B, Hq, Hkv, D, P, NP, K = 8, 32, 4, 128, 64, 4096, 32
    width = 2 * K + 8
    dev = torch.device(DEV)
    g = argus.geom(Hq, Hkv, D, P)
    pool = argus.Pool.empty(W.FP8_E4M3, B * NP, Hkv, P, D, device=dev)
    ck = torch.empty((B, NP, Hkv, D), dtype=torch.bfloat16, device=dev)
    ids = torch.arange(NP, dtype=torch.int32, device=dev)
    srcs = {}
    for b in range(B):
        src = W.normal((NP, 2, Hkv, P, D), W.BF16, W.seed_of("sparse", 0, 1) * 16 + b, device=dev)
        argus.quantize_pages(g, W.BF16, src, NP, ids, pool, ids + b * NP, NP, ckey_out=ck[b])
        if b == 3:
            srcs[b] = W.to_bits(src)
        del src
    q = W.normal((B, Hq, D), W.BF16, W.seed_of("sparse", 0, 0), device=dev)
    npages = torch.full((B,), NP, dtype=torch.int32, device=dev)
    sel = torch.empty((B, Hkv, width), dtype=torch.int32, device=dev)
    cnt = torch.empty((B, Hkv), dtype=torch.int32, device=dev)
    drops = torch.zeros(1, dtype=torch.int32, device=dev)
    sws = torch.empty(argus.select_workspace_bytes(g, B, NP), dtype=torch.uint8, device=dev)
    argus.select_pages(g, B, q, ck, npages, NP, K, True, sel, cnt, width, drops, sws)
    torch.cuda.synchronize()
    assert int(drops.item()) == 0 and torch.all(cnt == K + 1)
    # oracle for sequence 3: demote every page itself, compressed keys, selection, decode
    b = 3
    codes, meta = C.alloc_pool(W.FP8_E4M3, NP, Hkv, P, D)
    ock = C.quantize_pages(srcs[b], C.CODEC_BF16, list(range(NP)), W.FP8_E4M3, codes, meta, list(range(NP)),
                           want_ckey=True)
    gck = W.to_bits(ck[b].cpu())
    diff = np.abs(C.bf16_bits_to_f64(gck) - C.bf16_bits_to_f64(ock))
    assert np.all(diff <= np.abs(C.bf16_bits_to_f64(ock)) * 2.0 ** -7 + (P + 2) * 2.0 ** -24 * 8 + 1e-30)
    q64 = C.bf16_bits_to_f64(W.to_bits(q))[b:b + 1]
    osel, ocnt, _ = oracle.select_pages(q64, ock[None], [NP], Hkv, K, True, width)
    # the selection is checked on the GPU's own compressed-key slab (the slab is
    # select's input): every selected page scores within 1e-5 max|s| of the k-th
    scores = oracle.compressed_key_scores(q64, gck[None], [NP], Hkv)
    gsel = sel[b].cpu().numpy()
    for h in range(Hkv):
        s = scores[0, h, :NP - 1]
        kth = np.sort(s)[::-1][K - 1]
        slack = 1e-5 * np.abs(s).max()
        got = gsel[h, :K + 1]
        assert got[-1] == NP - 1 and list(got) == sorted(got)
        assert np.all(s[got[:-1]] >= kth - slack)
        # and every page strictly above the k-th (by more than the slack) is selected
        must = np.nonzero(s > kth + slack)[0]
        assert set(must.tolist()) <= set(got[:-1].tolist())
    # decode on the oracle's selection, full batch in the bench's configuration
    sel_o = sel.clone()
    sel_o[b] = torch.from_numpy(osel[0]).to(dev)
    out32 = torch.full((B, Hq, D), float("nan"), device=dev)
    a = argus.decode_args(g, B, q, [pool], torch.full((B, NP), W.FP8_E4M3, dtype=torch.uint8, device=dev),
                          torch.arange(B * NP, dtype=torch.int32, device=dev).reshape(B, NP),
                          torch.full((B,), NP * P, dtype=torch.int32, device=dev), NP, W.softmax_scale(D),
                          out_f32=out32, sel_pages=sel_o, sel_count=cnt, sel_width=width)
    ws = torch.empty(argus.decode_workspace_bytes(a), dtype=torch.uint8, device=dev)
    argus.paged_decode_attn(a, ws)
    torch.cuda.synchronize()
    ref, _, bad = oracle.paged_decode(q64, Hkv, P, {W.FP8_E4M3: (codes, meta)},
                                      np.full((1, NP), W.FP8_E4M3, np.uint8), np.arange(NP, dtype=np.int32)[None],
                                      np.array([NP * P]), W.softmax_scale(D), sel_pages=osel, sel_count=ocnt,
                                      sel_width=width)
    got = out32[b:b + 1].cpu().numpy()
    assert bad == 0 and np.abs(got - ref).max() <= _tol(ref)


def test_windowed_prefill_full_size_sampled_rows():
    Hq, Hkv, D, NQ, CTX, WIN = 16, 2, 128, 1024, 1 << 20, 131072
    dev = torch.device(DEV)
    kv_len = CTX + NQ
    q = W.normal((Hq, NQ, D), W.BF16, W.seed_of("prefill", 0, 0), device=dev)
    k = W.normal((Hkv, kv_len, D), W.BF16, W.seed_of("prefill", 0, 1), device=dev)
    v = W.normal((Hkv, kv_len, D), W.BF16, W.seed_of("prefill", 0, 2), device=dev)
    g = argus.geom(Hq, Hkv, D, 16)
    acc_o = torch.empty((Hq, NQ, D), dtype=torch.float32, device=dev)
    acc_l = torch.empty((Hq, NQ), dtype=torch.float32, device=dev)
    wins = [(w, w + WIN) for w in range(0, CTX, WIN)] + [(CTX, CTX + NQ)]
    # the launch configuration the benchmark times: automatic key-range splits
    ws = torch.empty(max(16, max(argus.window_prefill_workspace_bytes(g, NQ, w1 - w0) for w0, w1 in wins)),
                     dtype=torch.uint8, device=dev)
    for i, (w0, w1) in enumerate(wins):
        argus.window_prefill_attn(g, NQ, q, k[:, w0:], v[:, w0:], kv_len * D, w1 - w0, w0, CTX,
                                  W.softmax_scale(D), acc_o, acc_l, 1 if i else 0, ws=ws)
    torch.cuda.synchronize()
    rows = [0, 1, 511, NQ - 1]
    q64 = C.bf16_bits_to_f64(W.to_bits(q[:, rows]))
    got_o = acc_o[:, rows].cpu().numpy()
    got_l = acc_l[:, rows].cpu().numpy()
    for h in range(Hkv):
        k64 = C.bf16_bits_to_f64(W.to_bits(k[h]))[None]
        v64 = C.bf16_bits_to_f64(W.to_bits(v[h]))[None]
        for hq in range(h * Hq // Hkv, (h + 1) * Hq // Hkv):
            for r, i in enumerate(rows):
                qi = np.zeros((1, NQ, D))
                qi[0, i] = q64[hq, r]
                ro, rl = oracle.window_attention(qi, k64, v64, 0, CTX, W.softmax_scale(D), rows=[i])
                assert np.abs(got_o[hq, r] - ro[0, 0]).max() <= _tol(ro), (hq, i)
                assert abs(got_l[hq, r] - rl[0, 0]) <= 1e-4 * abs(rl[0, 0]) + 1e-5


def test_paged_fp8_window_prefill_full_window_sampled_rows():
    """The staged prefill at the full window size: 131,072 cached tokens in
    64-token FP8 pages (random physical slots) plus the 1,024-token chunk in
    BF16 pages, attended as two windows (the cache window, then the chunk) and
    folded; sampled query rows against the oracle's gather of the same pages."""
    Hq, Hkv, D, P, NQ, WIN = 16, 2, 128, 64, 1024, 131072
    dev = torch.device(DEV)
    n_cache, n_chunk = WIN // P, NQ // P
    n_pages = n_cache + n_chunk
    g = argus.geom(Hq, Hkv, D, P)
    src = W.normal((n_pages, 2, Hkv, P, D), W.BF16, W.seed_of("prefill", 0, 1), device=dev)
    perm = W.permutation(n_cache, W.seed_of("prefill", 0, 4))
    fp8 = argus.Pool.empty(W.FP8_E4M3, n_cache, Hkv, P, D, device=dev)
    bf = argus.Pool.empty(W.BF16, n_chunk, Hkv, P, D, device=dev)
    ids = torch.arange(n_pages, dtype=torch.int32, device=dev)
    argus.quantize_pages(g, W.BF16, src, n_pages, ids[:n_cache], fp8, torch.from_numpy(perm.astype(np.int32)).to(dev),
                         n_cache)
    argus.quantize_pages(g, W.BF16, src, n_pages, ids[n_cache:], bf, ids[:n_chunk], n_chunk)
    table = np.concatenate([perm, np.arange(n_chunk)]).astype(np.int32)
    codecs = np.array([W.FP8_E4M3] * n_cache + [W.BF16] * n_chunk, np.uint8)
    q = W.normal((Hq, NQ, D), W.BF16, W.seed_of("prefill", 0, 0), device=dev)
    acc_o = torch.empty((Hq, NQ, D), dtype=torch.float32, device=dev)
    acc_l = torch.empty((Hq, NQ), dtype=torch.float32, device=dev)
    d_codec, d_table = torch.from_numpy(codecs).to(dev), torch.from_numpy(table).to(dev)
    for i, (w0, wl) in enumerate([(0, WIN), (WIN, NQ)]):
        ws = torch.empty(argus.paged_window_prefill_workspace_bytes(g, NQ, wl), dtype=torch.uint8, device=dev)
        argus.paged_window_prefill_attn(g, NQ, q, [fp8, bf], d_codec, d_table, n_pages, w0, wl, WIN,
                                        W.softmax_scale(D), acc_o, acc_l, 1 if i else 0, ws)
        del ws
    torch.cuda.synchronize()
    # the oracle demotes the same source pages itself and gathers the window
    src_bits = W.to_bits(src)
    codes, meta = C.alloc_pool(W.FP8_E4M3, n_cache, Hkv, P, D)
    C.quantize_pages(src_bits, C.CODEC_BF16, list(range(n_cache)), W.FP8_E4M3, codes, meta, [int(x) for x in perm])
    bcodes, _ = C.alloc_pool(W.BF16, n_chunk, Hkv, P, D)
    C.quantize_pages(src_bits, C.CODEC_BF16, list(range(n_cache, n_pages)), W.BF16, bcodes, None, list(range(n_chunk)))
    pools = {W.FP8_E4M3: (codes, meta), W.BF16: (bcodes, None)}
    rows = [0, 1, 511, NQ - 1]
    q64 = C.bf16_bits_to_f64(W.to_bits(q))
    qs = np.zeros((Hq, NQ, D))
    qs[:, rows] = q64[:, rows]
    ro, rl = oracle.paged_window_attention(qs, Hkv, P, pools, codecs[None], table[None], 0, 0, WIN + NQ, WIN,
                                           W.softmax_scale(D), rows=rows, seq_len=WIN + NQ)
    got_o = acc_o[:, rows].cpu().numpy()
    got_l = acc_l[:, rows].cpu().numpy()
    assert np.abs(got_o - ro).max() <= _tol(ro)
    # lse2 within the staged window's bound: each key rounded to fp16 moves a
    # log2 score by <= scale * log2(e) * 2^-11 * sum_d |q_d k_d|; bound it with
    # Cauchy-Schwarz by |q| * max_j |k_j|
    K, _ = oracle.gather_window(Hkv, P, pools, codecs[None], table[None], 0, 0, WIN + NQ)
    kmax = np.sqrt((K ** 2).sum(axis=2)).max(axis=1)                         # [Hkv]
    qn = np.sqrt((q64[:, rows] ** 2).sum(axis=2))                           # [Hq][rows]
    bound = W.softmax_scale(D) / math.log(2) * 2.0 ** -11 * qn * np.repeat(kmax, Hq // Hkv)[:, None]
    assert np.all(np.abs(got_l - rl) <= bound + 1e-5 * np.abs(rl) + 1e-5)
