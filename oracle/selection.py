"""Top-k page selection over a compressed-key slab (oracle).

TEST INFRASTRUCTURE ONLY -- see the package docstring.

"feat(kvcache): host-RAM KV tier for sparse-attention models", section "Why
this works for sparse attention": every attend step first runs an indexer --
top-k block selection over a compressed slab -- and then reads only the
selected pages; section "Design": the selection is compacted into a fixed
width list (2 * block_topk + 8 entries) with a drop counter instead of silent
truncation.  The comment on in-place host placement counts about 2,051 tokens
per query, i.e. a 2,048-token budget plus the partly filled newest page.

Readings taken here:
* compressed key of a page = mean of its stored keys, rounded to bfloat16
  (produced by oracle.codecs.quantize_pages);
* score(b, h, p) = sum over the G query heads of KV head h of q . ckey(b, p, h),
  in float64 on the given bfloat16 slab;
* candidates are pages 0 .. n-2; the top_k highest scores are kept, ties going
  to the lower page index; the newest page n-1 is always added;
* the list is returned in ascending page order; when it would exceed the width
  the lowest-ranked candidates are dropped and counted.
"""

import numpy as np

from .codecs import bf16_bits_to_f64


def compressed_key_scores(q_f64, ckey_bits, n_pages, Hkv):
    """Scores [B][Hkv][max_pages] (float64; pages >= n_pages[b] are -inf)."""
    B, Hq, D = q_f64.shape
    G = Hq // Hkv
    max_pages = ckey_bits.shape[1]
    ck = bf16_bits_to_f64(ckey_bits)                      # [B][maxP][Hkv][D]
    scores = np.full((B, Hkv, max_pages), -np.inf)
    for b in range(B):
        n = int(n_pages[b])
        for h in range(Hkv):
            qs = q_f64[b, h * G:(h + 1) * G]              # [G][D]
            s = ck[b, :n, h] @ qs.T                        # [n][G]
            scores[b, h, :n] = s.sum(axis=1)
    return scores


def select_pages(q_f64, ckey_bits, n_pages, Hkv, top_k, keep_newest, width):
    """Returns (sel [B][Hkv][width] int32 padded with -1, count [B][Hkv], drops)."""
    B = q_f64.shape[0]
    scores = compressed_key_scores(q_f64, ckey_bits, n_pages, Hkv)
    sel = np.full((B, Hkv, width), -1, np.int32)
    count = np.zeros((B, Hkv), np.int32)
    drops = 0
    for b in range(B):
        n = int(n_pages[b])
        for h in range(Hkv):
            if n <= 0:
                continue
            n_cand = n - 1 if keep_newest else n
            cand = sorted(range(n_cand), key=lambda p: (-scores[b, h, p], p))
            k_want = min(top_k, n_cand)
            room = width - (1 if keep_newest else 0)
            k_keep = max(0, min(k_want, room))
            drops += k_want - k_keep
            chosen = set(cand[:k_keep])
            if keep_newest and width >= 1:
                chosen.add(n - 1)
            elif keep_newest:
                drops += 1
            lst = sorted(chosen)
            count[b, h] = len(lst)
            sel[b, h, :len(lst)] = lst
    return sel, count, drops
