"""Small, self-contained cases of each kernel, sized for Nsight Compute.

  python profile_cases.py <case> [--reps N]

Every case builds its inputs with the seeded generators, runs the library
call `reps` times and synchronises.  Cases keep a few GB at most on the device
and use inputs larger than L2 where the kernel streams HBM.

  decode_mixed    one layer of the mixed-tier decode (14/2 heads, D 64, 16 pages x 1024)
  decode_bf16     batched BF16 decode, batch 8 of the batched workload's shape
  decode_fp8      the same pages demoted to FP8
  decode_int2     the same pages demoted to INT2
  decode_int1     the same pages demoted to INT1
  decode_sparse   one layer of the sparse workload: decode over the indexer's selection
  decode_host     the same decode with the FP8 pool in page-locked host memory (1024 pages per row)
  quantize_fp8    demote 128 Ki 16x128 BF16 units to FP8 (512 MB read)
  quantize_int8   the same to INT8
  quantize_int4   the same to INT4
  quantize_int2   the same to INT2
  quantize_int1   the same to INT1
  select          indexer scores + top-k for one layer of the sparse workload
  prefill         one 131072-token window of the windowed prefill
  prefill_paged   one 32768-token window of FP8 pages staged through the block table
  fold            fold a 16 x 1024 x 128 fp32 partial into an accumulator
"""

import argparse
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import mixed_precision_paged_argus_gb300.argus as argus  # noqa: E402
from mixed_precision_paged_argus_gb300 import workloads as W  # noqa: E402


def _decode_mixed(dev):
    Hq, Hkv, D, P, NP = 14, 2, 64, 1024, 16
    g = argus.geom(Hq, Hkv, D, P)
    tiers = W.mixed_tier_codecs(NP)
    src = W.normal((NP, 2, Hkv, P, D), W.FP16, W.seed_of("mixed_tier", 0, 1), device=dev,
                   outlier_seed=W.seed_of("mixed_tier", 0, 5))
    pools, table = [], np.zeros(NP, np.int32)
    for codec in (W.FP16, W.FP8_E4M3, W.INT8, W.INT4_G32):
        pages = [p for p in range(NP) if tiers[p] == codec]
        pool = argus.Pool.empty(codec, 4, Hkv, P, D, device=dev)
        argus.quantize_pages(g, W.FP16, src, NP, torch.tensor(pages, dtype=torch.int32, device=dev), pool,
                             torch.arange(4, dtype=torch.int32, device=dev), 4)
        table[pages] = np.arange(4)
        pools.append(pool)
    q = W.normal((1, Hq, D), W.FP16, W.seed_of("mixed_tier", 0, 0), device=dev)
    out = torch.empty((1, Hq, D), dtype=torch.float16, device=dev)
    a = argus.decode_args(g, 1, q, pools, torch.from_numpy(tiers.reshape(1, NP).astype(np.uint8)).to(dev),
                          torch.from_numpy(table.reshape(1, NP)).to(dev),
                          torch.tensor([NP * P], dtype=torch.int32, device=dev), NP, W.softmax_scale(D), out=out)
    ws = torch.empty(max(1, argus.decode_workspace_bytes(a)), dtype=torch.uint8, device=dev)
    return lambda: argus.paged_decode_attn(a, ws)


def _decode_batched(dev, codec):
    B, Hq, Hkv, D, P, MAXP = 8, 32, 8, 128, 16, 2048
    lens = W.uniform_ints(B, 8192, 32768, W.seed_of("batched", 0, 3))
    table, n_slots = W.paged_block_table(lens, P, MAXP, W.seed_of("batched", 0, 4))
    g = argus.geom(Hq, Hkv, D, P)
    pool = argus.Pool(W.BF16, W.normal((n_slots, 2, Hkv, P, D), W.BF16, W.seed_of("batched", 0, 1), device=dev),
                      None, n_slots)
    if codec != W.BF16:
        ids = torch.arange(n_slots, dtype=torch.int32, device=dev)
        dst = argus.Pool.empty(codec, n_slots, Hkv, P, D, device=dev)
        argus.quantize_pages(g, W.BF16, pool.codes, n_slots, ids, dst, ids, n_slots)
        pool = dst
    q = W.normal((B, Hq, D), W.BF16, W.seed_of("batched", 0, 0), device=dev)
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
    a = argus.decode_args(g, B, q, [pool], torch.full((B, MAXP), codec, dtype=torch.uint8, device=dev),
                          torch.from_numpy(table).to(dev), torch.from_numpy(lens.astype(np.int32)).to(dev), MAXP,
                          W.softmax_scale(D), out=out)
    ws = torch.empty(max(1, argus.decode_workspace_bytes(a)), dtype=torch.uint8, device=dev)
    return lambda: argus.paged_decode_attn(a, ws)


def _quantize(dev, codec):
    Hkv, P, D, n = 8, 16, 128, 8192
    g = argus.geom(Hkv, Hkv, D, P)
    src = W.normal((n, 2, Hkv, P, D), W.BF16, 77, device=dev)
    ids = torch.arange(n, dtype=torch.int32, device=dev)
    dst = argus.Pool.empty(codec, n, Hkv, P, D, device=dev)
    return lambda: argus.quantize_pages(g, W.BF16, src, n, ids, dst, ids, n)


def _decode_sparse(dev):
    B, Hq, Hkv, D, P, NP, K = 8, 32, 4, 128, 64, 4096, 32
    width = 2 * K + 8
    g = argus.geom(Hq, Hkv, D, P)
    ids = torch.arange(NP, dtype=torch.int32, device=dev)
    pool = argus.Pool.empty(W.FP8_E4M3, B * NP, Hkv, P, D, device=dev)
    ck = torch.empty((B, NP, Hkv, D), dtype=torch.bfloat16, device=dev)
    for b in range(B):
        src = W.normal((NP, 2, Hkv, P, D), W.BF16, W.seed_of("sparse", 0, 1) * 16 + b, device=dev)
        argus.quantize_pages(g, W.BF16, src, NP, ids, pool, ids + b * NP, NP, ckey_out=ck[b])
        del src
    q = W.normal((B, Hq, D), W.BF16, W.seed_of("sparse", 0, 0), device=dev)
    npg = torch.full((B,), NP, dtype=torch.int32, device=dev)
    sel = torch.empty((B, Hkv, width), dtype=torch.int32, device=dev)
    cnt = torch.empty((B, Hkv), dtype=torch.int32, device=dev)
    sws = torch.empty(argus.select_workspace_bytes(g, B, NP), dtype=torch.uint8, device=dev)
    argus.select_pages(g, B, q, ck, npg, NP, K, True, sel, cnt, width, None, sws)
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
    a = argus.decode_args(g, B, q, [pool], torch.full((B, NP), W.FP8_E4M3, dtype=torch.uint8, device=dev),
                          torch.arange(B * NP, dtype=torch.int32, device=dev).reshape(B, NP),
                          torch.full((B,), NP * P, dtype=torch.int32, device=dev), NP, W.softmax_scale(D), out=out,
                          sel_pages=sel, sel_count=cnt, sel_width=width)
    ws = torch.empty(max(1, argus.decode_workspace_bytes(a)), dtype=torch.uint8, device=dev)
    return lambda: argus.paged_decode_attn(a, ws)


def _decode_host(dev):
    """The sparse case with its FP8 pool in page-locked host memory: decode reads
    the selected pages in place over the host link."""
    B, Hq, Hkv, D, P, NP, K = 8, 32, 4, 128, 64, 1024, 32
    width = 2 * K + 8
    g = argus.geom(Hq, Hkv, D, P)
    ids = torch.arange(NP, dtype=torch.int32, device=dev)
    pool = argus.Pool.empty(W.FP8_E4M3, B * NP, Hkv, P, D, device=dev)
    ck = torch.empty((B, NP, Hkv, D), dtype=torch.bfloat16, device=dev)
    for b in range(B):
        src = W.normal((NP, 2, Hkv, P, D), W.BF16, W.seed_of("sparse", 0, 1) * 16 + b, device=dev)
        argus.quantize_pages(g, W.BF16, src, NP, ids, pool, ids + b * NP, NP, ckey_out=ck[b])
        del src
    q = W.normal((B, Hq, D), W.BF16, W.seed_of("sparse", 0, 0), device=dev)
    npg = torch.full((B,), NP, dtype=torch.int32, device=dev)
    sel = torch.empty((B, Hkv, width), dtype=torch.int32, device=dev)
    cnt = torch.empty((B, Hkv), dtype=torch.int32, device=dev)
    sws = torch.empty(argus.select_workspace_bytes(g, B, NP), dtype=torch.uint8, device=dev)
    argus.select_pages(g, B, q, ck, npg, NP, K, True, sel, cnt, width, None, sws)
    torch.cuda.synchronize()
    host = pool.to_host()
    del pool
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
    a = argus.decode_args(g, B, q, [host], torch.full((B, NP), W.FP8_E4M3, dtype=torch.uint8, device=dev),
                          torch.arange(B * NP, dtype=torch.int32, device=dev).reshape(B, NP),
                          torch.full((B,), NP * P, dtype=torch.int32, device=dev), NP, W.softmax_scale(D), out=out,
                          sel_pages=sel, sel_count=cnt, sel_width=width)
    ws = torch.empty(max(1, argus.decode_workspace_bytes(a)), dtype=torch.uint8, device=dev)
    fn = lambda: argus.paged_decode_attn(a, ws)
    fn.keep = (host, a, ws, out)
    return fn


def _select(dev):
    B, Hq, Hkv, D, NP, K = 8, 32, 4, 128, 4096, 32
    g = argus.geom(Hq, Hkv, D, 64)
    q = W.normal((B, Hq, D), W.BF16, W.seed_of("sparse", 0, 0), device=dev)
    ck = W.normal((B, NP, Hkv, D), W.BF16, W.seed_of("sparse", 0, 6), device=dev)
    npg = torch.full((B,), NP, dtype=torch.int32, device=dev)
    sel = torch.empty((B, Hkv, 2 * K + 8), dtype=torch.int32, device=dev)
    cnt = torch.empty((B, Hkv), dtype=torch.int32, device=dev)
    drops = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(argus.select_workspace_bytes(g, B, NP), dtype=torch.uint8, device=dev)
    return lambda: argus.select_pages(g, B, q, ck, npg, NP, K, True, sel, cnt, 2 * K + 8, drops, ws)


def _prefill(dev):
    Hq, Hkv, D, NQ, WIN = 16, 2, 128, 1024, 131072
    q = W.normal((Hq, NQ, D), W.BF16, W.seed_of("prefill", 0, 0), device=dev)
    k = W.normal((Hkv, WIN, D), W.BF16, W.seed_of("prefill", 0, 1), device=dev)
    v = W.normal((Hkv, WIN, D), W.BF16, W.seed_of("prefill", 0, 2), device=dev)
    g = argus.geom(Hq, Hkv, D, 16)
    acc_o = torch.zeros((Hq, NQ, D), dtype=torch.float32, device=dev)
    acc_l = torch.full((Hq, NQ), float("-inf"), device=dev)
    ws = torch.empty(max(16, argus.window_prefill_workspace_bytes(g, NQ, WIN)), dtype=torch.uint8, device=dev)
    return lambda: argus.window_prefill_attn(g, NQ, q, k, v, 0, WIN, 0, 1 << 20, W.softmax_scale(D), acc_o,
                                             acc_l, 1, ws=ws)


def _prefill_paged(dev):
    """One 32768-token window of FP8 e4m3 pages (64-token pages, random slots)
    staged through the block table and attended by a 1024-query chunk."""
    Hq, Hkv, D, P, NQ, WIN = 16, 2, 128, 64, 1024, 32768
    n_pages = WIN // P
    g = argus.geom(Hq, Hkv, D, P)
    src = W.normal((n_pages, 2, Hkv, P, D), W.BF16, W.seed_of("prefill", 0, 1), device=dev)
    slots = torch.from_numpy(W.permutation(n_pages, W.seed_of("prefill", 0, 4)).astype(np.int32)).to(dev)
    pool = argus.Pool.empty(W.FP8_E4M3, n_pages, Hkv, P, D, device=dev)
    argus.quantize_pages(g, W.BF16, src, n_pages, torch.arange(n_pages, dtype=torch.int32, device=dev), pool,
                         slots, n_pages)
    del src
    q = W.normal((Hq, NQ, D), W.BF16, W.seed_of("prefill", 0, 0), device=dev)
    codec = torch.full((n_pages,), W.FP8_E4M3, dtype=torch.uint8, device=dev)
    acc_o = torch.zeros((Hq, NQ, D), dtype=torch.float32, device=dev)
    acc_l = torch.full((Hq, NQ), float("-inf"), device=dev)
    ws = torch.empty(argus.paged_window_prefill_workspace_bytes(g, NQ, WIN), dtype=torch.uint8, device=dev)
    return lambda: argus.paged_window_prefill_attn(g, NQ, q, [pool], codec, slots, n_pages, 0, WIN, 1 << 20,
                                                   W.softmax_scale(D), acc_o, acc_l, 1, ws)


def _fold(dev):
    n, D = 16 * 1024, 128
    ao = torch.randn((n, D), device=dev)
    al = torch.randn((n,), device=dev)
    po = torch.randn((n, D), device=dev)
    pl = torch.randn((n,), device=dev)
    return lambda: argus.fold_lse(ao, al, po, pl)


CASES = {
    "decode_mixed": _decode_mixed,
    "decode_bf16": lambda d: _decode_batched(d, W.BF16),
    "decode_fp8": lambda d: _decode_batched(d, W.FP8_E4M3),
    "decode_int2": lambda d: _decode_batched(d, W.INT2_G32),
    "decode_int1": lambda d: _decode_batched(d, W.INT1_G32),
    "decode_sparse": _decode_sparse,
    "decode_host": _decode_host,
    "quantize_fp8": lambda d: _quantize(d, W.FP8_E4M3),
    "quantize_int8": lambda d: _quantize(d, W.INT8),
    "quantize_int4": lambda d: _quantize(d, W.INT4_G32),
    "quantize_int2": lambda d: _quantize(d, W.INT2_G32),
    "quantize_int1": lambda d: _quantize(d, W.INT1_G32),
    "select": _select,
    "prefill": _prefill,
    "prefill_paged": _prefill_paged,
    "fold": _fold,
}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=sorted(CASES))
    ap.add_argument("--reps", type=int, default=3)
    a = ap.parse_args(argv)
    dev = torch.device("cuda", 0)
    fn = CASES[a.case](dev)
    torch.cuda.synchronize()
    for _ in range(a.reps):
        fn()
    torch.cuda.synchronize()
    print("ok", a.case)


if __name__ == "__main__":
    sys.exit(main())
