"""argus_paged_decode_attn_noalloc: decode for callers that cannot allocate.

Runtimes whose memory planner owns all device memory, and host code that may
not call cudaMalloc on the decode path, cannot pass the workspace that
argus_paged_decode_attn takes.  The no-allocation entry point keeps that
scratch in a fixed device array inside the library.  These tests call it
through the C ABI and check it against the workspace entry point and against
the double-precision oracle, twice in a row (the array keeps the previous
call's contents).  This file is collected last on purpose.
"""

import numpy as np
import pytest
import torch

import mixed_precision_paged_argus_gb300.argus as argus
from mixed_precision_paged_argus_gb300 import workloads as W
import oracle
from paged_cases import DEV, build_case, run_decode, tol

pytestmark = pytest.mark.gpu


def _noalloc(c, out_dtype, num_splits):
    out = torch.full((c.B, c.Hq, c.D), float("nan"), dtype=out_dtype, device=DEV)
    out32 = torch.full((c.B, c.Hq, c.D), float("nan"), dtype=torch.float32, device=DEV)
    lse = torch.full((c.B, c.Hq), float("nan"), dtype=torch.float32, device=DEV)
    args = argus.decode_args(c.g, c.B, c.q, c.pools, c.d_codec, c.d_table, c.d_lens, c.max_pages, c.scale,
                             out=out, out_f32=out32, lse2_out=lse, num_splits=num_splits)
    argus.paged_decode_attn_noalloc(args)
    torch.cuda.synchronize()
    return out, out32, lse


@pytest.mark.parametrize("splits", [0, 5])
def test_noalloc_matches_workspace_entry_point_twice(splits):
    Hq, Hkv, D, P = 14, 2, 64, 64
    pc = W.mixed_tier_codecs(16).reshape(1, 16)
    c = build_case(Hq, Hkv, D, P, [16 * 64 - 7], pc, W.FP16, seed=301, outliers=True)
    ref_out, ref32, ref_lse, _ = run_decode(c, num_splits=splits)
    r = ref32.cpu().numpy()
    o64, _, bad = oracle.paged_decode(c.q64, c.Hkv, c.P, c.opools, c.page_codec, c.table, c.lens, c.scale)
    assert bad == 0
    for _ in range(2):
        out, out32, lse = _noalloc(c, torch.float16, splits)
        g = out32.cpu().numpy()
        assert np.all(np.isfinite(g))
        assert np.abs(g - r).max() <= tol(r)
        assert np.abs(g - o64).max() <= tol(o64)
        assert np.abs(lse.cpu().numpy() - ref_lse.cpu().numpy()).max() <= 1e-4 * np.abs(ref_lse.cpu().numpy()).max()


def test_noalloc_batched_bf16_twice():
    Hq, Hkv, D, P = 32, 8, 128, 16
    lens = [300, 17, 0, 1000]
    pc = np.full((4, 64), W.FP8_E4M3)
    c = build_case(Hq, Hkv, D, P, lens, pc, W.BF16, seed=303)
    _, ref32, _, _ = run_decode(c, out_dtype=torch.bfloat16, num_splits=7)
    r = ref32.cpu().numpy()
    o64, _, _ = oracle.paged_decode(c.q64, c.Hkv, c.P, c.opools, c.page_codec, c.table, c.lens, c.scale)
    for _ in range(2):
        out, out32, _ = _noalloc(c, torch.bfloat16, 7)
        assert np.abs(out32.cpu().numpy() - r).max() <= tol(r)
        assert np.abs(out32.cpu().numpy() - o64).max() <= tol(o64)
        assert torch.equal(out.cpu(), out32.cpu().to(torch.bfloat16))


def test_noalloc_rejects_scratch_beyond_the_fixed_size():
    Hq, Hkv, D, P = 32, 8, 128, 16
    pc = np.full((64, 2), W.FP8_E4M3)
    c = build_case(Hq, Hkv, D, P, [20] * 64, pc, W.BF16, seed=305)
    args = argus.decode_args(c.g, c.B, c.q, c.pools, c.d_codec, c.d_table, c.d_lens, 2048, c.scale,
                             out_f32=torch.empty((c.B, Hq, D), device=DEV), num_splits=512)
    assert argus.decode_workspace_bytes(args) > argus.NOALLOC_SCRATCH_BYTES
    with pytest.raises(argus.ArgusError) as e:
        argus.paged_decode_attn_noalloc(args)
    assert e.value.status == 3
