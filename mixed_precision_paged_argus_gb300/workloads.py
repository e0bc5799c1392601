"""Seeded synthetic inputs for the paged mixed-codec decode-attention path.

This module only draws random numbers and lays them out; it contains none of
the method's arithmetic (no quantisation, scoring or attention).  Tests,
the smoke check and the benchmark call it, and hand the same arrays to the
CUDA library and to the CPU oracle.

Seeds follow one rule: seed = 1000 * workload_id + 10 * layer + tensor_id,
with tensor_id 0 = q, 1 = K, 2 = V, 3 = lengths, 4 = physical-slot
permutation, 5 = outlier mask for K, 6 = outlier mask for V.

Values are N(0, 1) drawn in float32 by torch's Philox-based generators (CPU or
CUDA) and rounded to fp16 or bf16 by a dtype cast; the mixed-tier workload
multiplies each element independently with probability 0.01 by 8 (the
"1% outliers x8" of its description).

The five workloads (sizes as their descriptions state):
  tiny_fp16      batch 1, 1 layer, 14 q / 2 KV heads, head_dim 64, 4 pages x 1024,
                 all FP16
  mixed_tier     batch 1, 24 layers, 14 / 2, head_dim 64, 16 pages x 1024; newest 4
                 FP16, next 4 FP8, next 4 INT8, oldest 4 INT4 (group 32)
  batched        batch 32, 1 layer, 32 / 8, head_dim 128, 16-token pages, lengths
                 uniform in [8192, 32768], slots a random permutation; BF16 or FP8
  sparse         batch 8, 12 layers, 32 / 4, head_dim 128, 262144 tokens in 64-token
                 FP8 pages, top 32 pages + the newest one per KV head
  prefill        1 layer, 16 / 2, head_dim 128, 1048576 cached BF16 tokens, a
                 1024-token causal chunk, 131072-token windows
"""

import math

import numpy as np
import torch

FP16, BF16, FP8_E4M3, INT8, INT4_G32, INT2_G32, INT1_G32 = 0, 1, 2, 3, 4, 5, 6

WORKLOAD_IDS = {"tiny_fp16": 1, "mixed_tier": 2, "batched": 3, "sparse": 4,
                "prefill": 5}

TORCH_DTYPE = {FP16: torch.float16, BF16: torch.bfloat16}


def seed_of(workload, layer, tensor_id):
    wid = WORKLOAD_IDS.get(workload, workload)
    return 1000 * int(wid) + 10 * int(layer) + int(tensor_id)


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, dtype, seed, device="cpu", outlier_seed=None, outlier_p=0.01,
           outlier_mul=8.0):
    """N(0,1) values rounded to fp16/bf16 (torch tensor of that dtype)."""
    x = torch.randn(tuple(shape), generator=_gen(seed, device), device=device,
                    dtype=torch.float32)
    if outlier_seed is not None:
        u = torch.rand(tuple(shape), generator=_gen(outlier_seed, device),
                       device=device, dtype=torch.float32)
        x = torch.where(u < outlier_p, x * outlier_mul, x)
    return x.to(TORCH_DTYPE[dtype])


def uniform_ints(n, lo, hi, seed):
    """n integers uniform in [lo, hi] (inclusive), int64 numpy."""
    g = _gen(seed, "cpu")
    return torch.randint(lo, hi + 1, (n,), generator=g).numpy().astype(np.int64)


def permutation(n, seed):
    g = _gen(seed, "cpu")
    return torch.randperm(n, generator=g).numpy().astype(np.int64)


def to_bits(t):
    """16-bit torch tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def softmax_scale(head_dim):
    """1/sqrt(head_dim) computed in double and rounded to float32."""
    return float(np.float32(1.0 / math.sqrt(head_dim)))


# --------------------------------------------------------------------------
# Paged layouts
# --------------------------------------------------------------------------

def mixed_tier_codecs(n_pages=16):
    """Codec of each logical page (page 0 = oldest) in the mixed-tier workload:
    pages 12-15 FP16, 8-11 FP8, 4-7 INT8, 0-3 INT4 (for 16 pages; the same
    quarters for other multiples of 4)."""
    q = n_pages // 4
    out = np.empty(n_pages, np.int64)
    out[:q] = INT4_G32
    out[q:2 * q] = INT8
    out[2 * q:3 * q] = FP8_E4M3
    out[3 * q:] = FP16
    return out


def paged_block_table(seq_lens, page_tokens, max_pages, seed):
    """Block table [B][max_pages] giving each used logical page a distinct
    physical slot drawn from a random permutation of all used pages; unused
    entries are 0.  Returns (table int32, n_used_slots)."""
    n_pages = [(int(L) + page_tokens - 1) // page_tokens for L in seq_lens]
    total = int(sum(n_pages))
    perm = permutation(total, seed)
    table = np.zeros((len(seq_lens), max_pages), np.int32)
    k = 0
    for b, n in enumerate(n_pages):
        table[b, :n] = perm[k:k + n]
        k += n
    return table, total
