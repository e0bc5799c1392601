"""Bounded waits of the decode kernel run out without faulting the GPU.

argus_test_decode_stall limits every device wait to a few milliseconds and has
the producer warp withhold one stage's arrival, so the consumer warps' wait on
that stage runs out.  The CTA must report the timeout in bit 31 of the status
word, wait until the copies it issued have landed, end, and leave the context
usable: the next ordinary decode on the same buffers matches the oracle.
"""

import time

import numpy as np
import pytest
import torch

import mixed_precision_paged_argus_gb300.argus as argus
from mixed_precision_paged_argus_gb300 import workloads as W
import oracle
from paged_cases import DEV, build_case, run_decode, tol

pytestmark = pytest.mark.gpu


def _check_against_oracle(c, out32, lse, window=0, sinks=0):
    ref, ref_lse, bad = oracle.paged_decode(c.q64, c.Hkv, c.P, c.opools, c.page_codec, c.table, c.lens,
                                            c.scale, window=window, sinks=sinks)
    assert bad == 0
    got = out32.cpu().numpy().astype(np.float64)
    assert np.abs(got - ref).max() <= tol(ref)
    gl = lse.cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(gl), fin)
    assert np.all(np.abs(gl[fin] - ref_lse[fin]) <= 1e-4 * np.maximum(1.0, np.abs(ref_lse[fin])))


WIDE = (W.FP16, W.FP8_E4M3, W.INT8, W.INT4_G32)
NARROW = (W.FP8_E4M3, W.INT8, W.INT4_G32)          # no 16-bit pool: the narrow ring, two producer warps


@pytest.mark.parametrize("D,q_dtype,window,stall,tiers", [
    (128, W.FP16, 0, 0, WIDE),    # wide ring, the stall in the first stage
    (128, W.BF16, 0, 1, WIDE),
    (64, W.FP16, 0, 0, WIDE),
    (128, W.FP16, 96, 0, WIDE),   # the extended kernel (sliding window)
    (128, W.BF16, 0, 0, NARROW),  # narrow ring: the first producer withholds
    (128, W.FP16, 0, 2, NARROW),  # narrow ring: the second producer's first stage
    (128, W.BF16, 0, 3, NARROW + (W.INT2_G32, W.INT1_G32)),   # extended narrow kernel
])
def test_stalled_stage_times_out_and_the_context_stays_usable(D, q_dtype, window, stall, tiers):
    Hq, Hkv, P = 8, 2, 16
    # long rows (many stages: the producer meets the abort at its empty wait)
    # and short rows (one stage: the producer has issued everything when the
    # consumers give up); the empty row has no stage at all
    lens = [1024, 16, 40, 0]
    max_pages = 64
    rng = np.random.default_rng(3)
    pc = rng.choice(list(tiers), size=(len(lens), max_pages))
    if q_dtype == W.BF16:
        pc[pc == W.FP16] = W.BF16
    c = build_case(Hq, Hkv, D, P, lens, pc, q_dtype, seed=41)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out32 = torch.zeros((c.B, c.Hq, c.D), dtype=torch.float32, device=DEV)
    lse = torch.zeros((c.B, c.Hq), dtype=torch.float32, device=DEV)
    args = argus.decode_args(c.g, c.B, c.q, c.pools, c.d_codec, c.d_table, c.d_lens, c.max_pages, c.scale,
                             out_f32=out32, lse2_out=lse, status=status, num_splits=1,
                             window_tokens=window, sink_tokens=4 if window else 0)
    ws = torch.zeros(max(1, argus.decode_workspace_bytes(args)), dtype=torch.uint8, device=DEV)
    wait_us = 20000
    t0 = time.perf_counter()
    argus.test_decode_stall(args, ws, wait_us, stall)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    st = int(status.item()) & 0xFFFFFFFF
    assert st & argus.STATUS_TIMEOUT_BIT, hex(st)
    assert st & ~argus.STATUS_TIMEOUT_BIT == 0, hex(st)   # no page counted as bad
    # every CTA waited once (consumers) or a few times (producer) for 20 ms,
    # all at once: far below the default 2 s limit
    assert elapsed < 1.5, elapsed
    # the same buffers, an ordinary call: correct results, no timeout
    status.zero_()
    out32.zero_()
    argus.paged_decode_attn(args, ws)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _check_against_oracle(c, out32, lse, window=window, sinks=4 if window else 0)


def test_stall_beyond_the_last_stage_changes_nothing():
    """A CTA with fewer stages than stall_stage never withholds anything: the
    call is an ordinary decode."""
    Hq, Hkv, D, P = 8, 2, 128, 16
    lens = [64, 200]
    pc = np.full((2, 16), W.FP8_E4M3)
    c = build_case(Hq, Hkv, D, P, lens, pc, W.FP16, seed=43)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out32 = torch.zeros((c.B, c.Hq, c.D), dtype=torch.float32, device=DEV)
    lse = torch.zeros((c.B, c.Hq), dtype=torch.float32, device=DEV)
    args = argus.decode_args(c.g, c.B, c.q, c.pools, c.d_codec, c.d_table, c.d_lens, c.max_pages, c.scale,
                             out_f32=out32, lse2_out=lse, status=status, num_splits=1)
    ws = torch.zeros(max(1, argus.decode_workspace_bytes(args)), dtype=torch.uint8, device=DEV)
    argus.test_decode_stall(args, ws, 20000, 1000)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _check_against_oracle(c, out32, lse)


def test_stall_arguments_are_checked():
    Hq, Hkv, D, P = 8, 2, 64, 16
    c = build_case(Hq, Hkv, D, P, [32], np.full((1, 2), W.FP16), W.FP16, seed=44)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out32 = torch.zeros((c.B, c.Hq, c.D), dtype=torch.float32, device=DEV)
    args = argus.decode_args(c.g, c.B, c.q, c.pools, c.d_codec, c.d_table, c.d_lens, c.max_pages, c.scale,
                             out_f32=out32, status=status, num_splits=1)
    ws = torch.zeros(max(1, argus.decode_workspace_bytes(args)), dtype=torch.uint8, device=DEV)
    for bad in [(0, 0), (2000001, 0), (1000, -1)]:
        with pytest.raises(argus.ArgusError) as e:
            argus.test_decode_stall(args, ws, *bad)
        assert e.value.status == 1
    args.status = None
    with pytest.raises(argus.ArgusError):
        argus.test_decode_stall(args, ws, 1000, 0)
