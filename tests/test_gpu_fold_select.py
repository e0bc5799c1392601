"""argus_fold_lse and argus_select_pages on the GPU against the oracle."""

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


@pytest.mark.parametrize("D", [64, 128])
def test_fold_matches_oracle_with_empty_rows(D):
    rng = np.random.default_rng(D)
    n = 1000
    ao = rng.standard_normal((n, D)).astype(np.float32)
    bo = rng.standard_normal((n, D)).astype(np.float32)
    al = (rng.standard_normal(n) * 10).astype(np.float32)
    bl = (rng.standard_normal(n) * 10).astype(np.float32)
    al[::7] = -np.inf
    bl[::11] = -np.inf
    al[::77] = -np.inf
    ro, rl = oracle.fold_lse(ao, al, bo, bl)
    acc_o, acc_l = torch.from_numpy(ao).to(DEV), torch.from_numpy(al).to(DEV)
    argus.fold_lse(acc_o, acc_l, torch.from_numpy(bo).to(DEV), torch.from_numpy(bl).to(DEV))
    torch.cuda.synchronize()
    go, gl = acc_o.cpu().numpy(), acc_l.cpu().numpy()
    assert np.abs(go - ro).max() <= 1e-3 * np.abs(ro).max() + 1e-4
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(gl), fin)
    assert np.abs(gl[fin] - rl[fin]).max() <= 1e-5 * np.abs(rl[fin]).max()


def test_fold_of_decode_splits_equals_single_pass():
    """Decode two halves of a context separately, fold them, compare to the oracle
    over the whole context (the fold identity through the GPU path)."""
    from paged_cases import build_case, run_decode
    Hq, Hkv, D, P = 8, 2, 128, 16
    pc = np.full((1, 8), W.BF16)
    c = build_case(Hq, Hkv, D, P, [128], pc, W.BF16, seed=5)
    width = 8
    outs = []
    for part in ([0, 1, 2, 3], [4, 5, 6, 7]):
        sel = np.full((1, Hkv, width), -1, np.int32)
        sel[0, :, :4] = part
        cnt = np.full((1, Hkv), 4, np.int32)
        _, o32, lse, _ = run_decode(c, out_dtype=torch.bfloat16, sel=torch.from_numpy(sel).to(DEV),
                                    sel_count=torch.from_numpy(cnt).to(DEV), sel_width=width)
        outs.append((o32.reshape(-1, D), lse.reshape(-1)))
    acc_o, acc_l = outs[0][0].clone(), outs[0][1].clone()
    argus.fold_lse(acc_o, acc_l, outs[1][0], outs[1][1])
    torch.cuda.synchronize()
    ref, ref_l, _ = oracle.paged_decode(c.q64, Hkv, P, c.opools, c.page_codec, c.table, c.lens, c.scale)
    assert np.abs(acc_o.cpu().numpy() - ref.reshape(-1, D)).max() <= 1e-3 * np.abs(ref).max() + 1e-4
    assert np.abs(acc_l.cpu().numpy() - ref_l.reshape(-1)).max() <= 1e-4 * np.abs(ref_l).max()


def _select_case(B, Hq, Hkv, D, max_pages, n_pages, seed, q_dtype=W.BF16, ties=False):
    q = W.normal((B, Hq, D), q_dtype, seed)
    if ties:
        rng = np.random.default_rng(seed)
        ck64 = np.zeros((B, max_pages, Hkv, D))
        ck64[..., 0] = rng.integers(-3, 4, size=(B, max_pages, Hkv))
        ck = C.f64_to_bf16_bits(ck64)
    else:
        ck = W.to_bits(W.normal((B, max_pages, Hkv, D), W.BF16, seed + 1))
    q64 = (C.bf16_bits_to_f64 if q_dtype == W.BF16 else C.f16_bits_to_f64)(W.to_bits(q))
    return q, q64, ck


def _run_select(q, ck, n_pages, Hq, Hkv, D, max_pages, top_k, width, keep_newest=True):
    B = q.shape[0]
    g = argus.geom(Hq, Hkv, D, 16)
    sel = torch.full((B, Hkv, width), -7, dtype=torch.int32, device=DEV)
    cnt = torch.zeros((B, Hkv), dtype=torch.int32, device=DEV)
    drops = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(argus.select_workspace_bytes(g, B, max_pages), dtype=torch.uint8, device=DEV)
    ckt = torch.from_numpy(ck.view(np.int16)).view(torch.bfloat16).to(DEV)
    argus.select_pages(g, B, q.to(DEV), ckt, torch.tensor(n_pages, dtype=torch.int32, device=DEV),
                       max_pages, top_k, keep_newest, sel, cnt, width, drops, ws)
    torch.cuda.synchronize()
    return sel.cpu().numpy(), cnt.cpu().numpy(), int(drops.item())


@pytest.mark.parametrize("D,G", [(128, 8), (64, 7)])
def test_select_matches_oracle_up_to_near_ties(D, G):
    B, Hkv, max_pages = 3, 4, 700
    Hq = G * Hkv
    n_pages = [700, 33, 2]
    q, q64, ck = _select_case(B, Hq, Hkv, D, max_pages, n_pages, 7)
    top_k, width = 32, 72
    sel, cnt, drops = _run_select(q, ck, n_pages, Hq, Hkv, D, max_pages, top_k, width)
    osel, ocnt, odrops = oracle.select_pages(q64, ck, n_pages, Hkv, top_k, True, width)
    scores = oracle.compressed_key_scores(q64, ck, n_pages, Hkv)
    assert drops == odrops == 0
    assert np.array_equal(cnt, ocnt)
    for b in range(B):
        n = n_pages[b]
        for h in range(Hkv):
            got = sel[b, h, :cnt[b, h]]
            assert np.all(sel[b, h, cnt[b, h]:] == -1)
            assert list(got) == sorted(got) and got[-1] == n - 1
            want = osel[b, h, :ocnt[b, h]]
            if n - 1 > top_k:
                s = scores[b, h, :n - 1]
                kth = np.sort(s)[::-1][top_k - 1]
                slack = 1e-5 * np.abs(s).max()
                assert np.all(s[got[:-1]] >= kth - slack)
                sure = set(np.nonzero(s > kth + slack)[0].tolist())
                assert sure <= set(got.tolist())
            else:
                assert np.array_equal(got, want)


def test_select_exact_ties_go_to_lower_page_index():
    B, Hq, Hkv, D, max_pages = 2, 4, 1, 64, 300
    n_pages = [300, 120]
    q, q64, ck = _select_case(B, Hq, Hkv, D, max_pages, n_pages, 17, ties=True)
    # make the query sum positive in dim 0 so integer keys give exact integer scores
    qn = np.zeros((B, Hq, D), np.float32)
    qn[:, :, 0] = 0.25
    q = torch.from_numpy(qn).to(torch.bfloat16)
    q64 = C.bf16_bits_to_f64(W.to_bits(q))
    for top_k in (1, 5, 40, 119, 299, 500):
        sel, cnt, drops = _run_select(q, ck, n_pages, Hq, Hkv, D, max_pages, top_k, 2 * top_k + 8)
        osel, ocnt, odrops = oracle.select_pages(q64, ck, n_pages, Hkv, top_k, True, 2 * top_k + 8)
        assert np.array_equal(cnt, ocnt) and drops == odrops
        assert np.array_equal(sel[:, :, :cnt.max()], osel[:, :, :cnt.max()])


def test_select_width_overflow_drops():
    B, Hq, Hkv, D, max_pages = 1, 8, 2, 128, 100
    q, q64, ck = _select_case(B, Hq, Hkv, D, max_pages, [100], 27)
    sel, cnt, drops = _run_select(q, ck, [100], Hq, Hkv, D, max_pages, 20, 10)
    osel, ocnt, odrops = oracle.select_pages(q64, ck, [100], Hkv, 20, True, 10)
    assert drops == odrops == 2 * 11
    assert np.array_equal(cnt, ocnt)


@pytest.mark.parametrize("max_pages,n_pages", [(4000, [4000, 3999]), (50000, [50000, 777])])
def test_select_many_ties_and_long_rows(max_pages, n_pages):
    """Scores drawn from 7 values: most pages tie, so each warp keeps far more
    than k survivors (the block-wide search takes over); rows longer than the
    shared-memory stage read their keys from memory."""
    B, Hq, Hkv, D = 2, 4, 1, 64
    q, q64, ck = _select_case(B, Hq, Hkv, D, max_pages, n_pages, 31, ties=True)
    qn = np.zeros((B, Hq, D), np.float32)
    qn[:, :, 0] = 0.25
    q = torch.from_numpy(qn).to(torch.bfloat16)
    q64 = C.bf16_bits_to_f64(W.to_bits(q))
    for top_k in (32, 200):
        sel, cnt, drops = _run_select(q, ck, n_pages, Hq, Hkv, D, max_pages, top_k, 2 * top_k + 8)
        osel, ocnt, odrops = oracle.select_pages(q64, ck, n_pages, Hkv, top_k, True, 2 * top_k + 8)
        assert np.array_equal(cnt, ocnt) and drops == odrops
        assert np.array_equal(sel[:, :, :cnt.max()], osel[:, :, :cnt.max()])


def test_select_then_decode_with_early_start():
    """argus_select_pages (its score grid starts in its predecessor's tail and
    waits for it) followed by decode with pdl=2 (starts early, reads the
    selection after the select completes), layer after layer, eagerly and from
    a CUDA graph: the same bits as stream order, and the oracle's result over
    the selected pages."""
    from paged_cases import build_case, tol
    Hq, Hkv, D, P, NP, B = 16, 2, 128, 16, 96, 2
    K, width = 8, 24
    pc = np.full((B, NP), W.FP8_E4M3)
    c = build_case(Hq, Hkv, D, P, [NP * P, NP * P - 9], pc, W.BF16, q_dtype=W.BF16, seed=900)
    g = argus.geom(Hq, Hkv, D, P)
    layers = 3
    cks = [W.normal((B, NP, Hkv, D), W.BF16, 910 + l).to(DEV) for l in range(layers)]
    npg = torch.tensor([NP, NP], dtype=torch.int32, device=DEV)
    sws = torch.empty(argus.select_workspace_bytes(g, B, NP), dtype=torch.uint8, device=DEV)

    def chain(pdl):
        sels = [torch.full((B, Hkv, width), -7, dtype=torch.int32, device=DEV) for _ in range(layers)]
        cnts = [torch.zeros((B, Hkv), dtype=torch.int32, device=DEV) for _ in range(layers)]
        outs = [torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device=DEV) for _ in range(layers)]
        lses = [torch.full((B, Hq), float("nan"), dtype=torch.float32, device=DEV) for _ in range(layers)]
        args = [argus.decode_args(c.g, c.B, c.q, c.pools, c.d_codec, c.d_table, c.d_lens, c.max_pages, c.scale,
                                  out_f32=outs[l], lse2_out=lses[l], sel_pages=sels[l], sel_count=cnts[l],
                                  sel_width=width, pdl=pdl) for l in range(layers)]
        ws = torch.empty(max(argus.decode_workspace_bytes(a) for a in args), dtype=torch.uint8, device=DEV)

        def step(stream):
            for l in range(layers):
                argus.select_pages(g, B, c.q, cks[l], npg, NP, K, True, sels[l], cnts[l], width, None, sws,
                                   stream=stream)
                argus.paged_decode_attn(args[l], ws, stream=stream)
        return sels, cnts, outs, lses, step

    ref = chain(0)
    stream = torch.cuda.Stream(device=DEV)
    with torch.cuda.stream(stream):
        ref[4](stream)
    torch.cuda.synchronize()
    got = chain(2)
    with torch.cuda.stream(stream):
        for _ in range(2):
            got[4](stream)
        stream.synchronize()
        for l in range(layers):
            for x, y in zip(got[:4], ref[:4]):
                assert torch.equal(x[l], y[l]), l
            got[2][l].fill_(float("nan"))
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            got[4](stream)
        graph.replay()
    torch.cuda.synchronize()
    for l in range(layers):
        assert torch.equal(got[2][l], ref[2][l])
    # the oracle over the pages the first layer selected
    sel0, cnt0 = ref[0][0].cpu().numpy(), ref[1][0].cpu().numpy()
    o, lse, bad = oracle.paged_decode(c.q64, c.Hkv, c.P, c.opools, c.page_codec, c.table, c.lens, c.scale,
                                      sel_pages=sel0, sel_count=cnt0, sel_width=width)
    assert bad == 0
    assert np.abs(ref[2][0].cpu().numpy() - o).max() <= tol(o)
