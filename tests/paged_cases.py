"""Builders of paged decode cases shared by the GPU tests.

A case draws 16-bit source pages with the seeded generators, demotes them into
per-codec pools twice -- once on the GPU with argus_quantize_pages, once with the
oracle -- and lays out the block table.  The oracle never sees a GPU result:
both sides start from the same generator output.
"""

import numpy as np
import torch

import mixed_precision_paged_argus_gb300.argus as argus
from mixed_precision_paged_argus_gb300 import workloads as W
from oracle import codecs as C

DEV = "cuda"


def tol(ref):
    return 1e-3 * float(np.abs(ref).max()) + 1e-4


class Case:
    pass


def build_case(Hq, Hkv, D, P, lens, page_codecs, src_dtype=W.FP16, q_dtype=None, seed=7,
               outliers=False, permute=True, extra_slots=0):
    """page_codecs: int array [B][max_pages] (codec of each logical page)."""
    q_dtype = src_dtype if q_dtype is None else q_dtype
    B = len(lens)
    page_codecs = np.asarray(page_codecs)
    max_pages = page_codecs.shape[1]
    g = argus.geom(Hq, Hkv, D, P)
    # one source slot per (b, page)
    n_src = B * max_pages
    src = W.normal((n_src, 2, Hkv, P, D), src_dtype, seed + 1,
                   outlier_seed=(seed + 5) if outliers else None)
    q = W.normal((B, Hq, D), q_dtype, seed)
    src_bits = W.to_bits(src)
    src_d = src.to(DEV)
    rng = np.random.default_rng(seed + 4)
    table = np.zeros((B, max_pages), np.int32)
    pools, opools = [], {}
    used = sorted(set(int(c) for c in page_codecs.ravel()))
    for codec in used:
        bp = [(b, p) for b in range(B) for p in range(max_pages) if page_codecs[b, p] == codec]
        n_slots = len(bp) + extra_slots
        slots = rng.permutation(n_slots)[:len(bp)] if permute else np.arange(len(bp))
        srcs = [b * max_pages + p for (b, p) in bp]
        pool = argus.Pool.empty(codec, n_slots, Hkv, P, D, device=DEV, zero=True)
        if bp:
            argus.quantize_pages(g, src_dtype, src_d, n_src,
                                 torch.tensor(srcs, dtype=torch.int32, device=DEV), pool,
                                 torch.tensor(slots, dtype=torch.int32, device=DEV), len(bp))
        codes, meta = C.alloc_pool(codec, n_slots, Hkv, P, D)
        if bp:
            C.quantize_pages(src_bits, src_dtype, srcs, codec, codes, meta, list(slots))
        for (b, p), s in zip(bp, slots):
            table[b, p] = s
        pools.append(pool)
        opools[codec] = (codes, meta)
    c = Case()
    c.g, c.B, c.Hq, c.Hkv, c.D, c.P = g, B, Hq, Hkv, D, P
    c.max_pages = max_pages
    c.q = q.to(DEV)
    c.q64 = (C.f16_bits_to_f64 if q_dtype == W.FP16 else C.bf16_bits_to_f64)(W.to_bits(q))
    c.pools, c.opools = pools, opools
    c.table = table
    c.page_codec = page_codecs.astype(np.uint8)
    c.lens = np.asarray(lens, np.int64)
    c.d_table = torch.from_numpy(table).to(DEV)
    c.d_codec = torch.from_numpy(c.page_codec).to(DEV)
    c.d_lens = torch.tensor(lens, dtype=torch.int32, device=DEV)
    c.scale = W.softmax_scale(D)
    return c


def run_decode(c, out_dtype=torch.float16, num_splits=0, sel=None, sel_count=None, sel_width=0,
               status=None, table=None, window=0, sinks=0):
    out = torch.full((c.B, c.Hq, c.D), float("nan"), dtype=out_dtype, device=DEV)
    out32 = torch.full((c.B, c.Hq, c.D), float("nan"), dtype=torch.float32, device=DEV)
    lse = torch.full((c.B, c.Hq), float("nan"), dtype=torch.float32, device=DEV)
    args = argus.decode_args(c.g, c.B, c.q, c.pools, c.d_codec,
                             c.d_table if table is None else table, c.d_lens, c.max_pages, c.scale,
                             out=out, out_f32=out32, lse2_out=lse, sel_pages=sel, sel_count=sel_count,
                             sel_width=sel_width, status=status, num_splits=num_splits,
                             window_tokens=window, sink_tokens=sinks)
    ws = torch.zeros(max(1, argus.decode_workspace_bytes(args)), dtype=torch.uint8, device=DEV)
    argus.paged_decode_attn(args, ws)
    torch.cuda.synchronize()
    return out, out32, lse, ws
