"""Attention over paged, mixed-codec K/V and the log2-sum-exp fold (oracle).

TEST INFRASTRUCTURE ONLY -- see the package docstring.

What is computed is the plain definition.  "ARGUS: Heterogeneous KV-cache
memory management", sections "Why decode is slow" and "Direct paged
attention", describes an *exact* online-softmax recurrence that streams one
page at a time; being exact, its result is ordinary softmax attention

    o_h = sum_j softmax_j(scale * q_h . k_j) v_j

over the visible tokens, where k_j, v_j are the dequantised stored values
(the pool is the source of truth: "feat(kvcache): host-RAM KV tier ...",
update 20f3b23).  The oracle therefore materialises the dequantised keys and
values of the visible tokens and evaluates the formula in float64 -- no
streaming, no blocking.

Each row also reports its log2-sum-exp  L = log2 sum_j 2^(scale*q.k_j*log2 e),
which is what the windowed prefill of the "--kv-placement host" comment on the
same pull request folds across windows into a float32 accumulator.
"""

import math

import numpy as np

from .codecs import bits_to_f64, dequant_page

LOG2E = 1.0 / math.log(2.0)


def softmax_attention(q, K, V, scale):
    """Dense softmax attention of one query row.

    q [D], K [n][D], V [n][D] float64; returns (o [D], lse2).  An empty key
    set gives o = 0 and lse2 = -inf.
    """
    if K.shape[0] == 0:
        return np.zeros(V.shape[1] if V.ndim == 2 else q.shape[0]), -math.inf
    s = scale * (K @ q)
    m = np.max(s)
    w = np.exp(s - m)
    l = np.sum(w)
    o = (w @ V) / l
    lse2 = (m + math.log(l)) * LOG2E
    return o, lse2


def _visible_pages(b, h, seq_len, P, max_pages, sel_pages, sel_count, sel_width):
    """Logical pages that batch row b / KV head h attends to, and the number of
    selection entries rejected as out of range."""
    n_pages = (seq_len + P - 1) // P
    if sel_pages is None:
        return list(range(min(n_pages, max_pages))), 0
    count = int(sel_count[b, h])
    bad = 0
    if count > sel_width:
        bad += 1
        count = sel_width
    pages = []
    for v in range(max(count, 0)):
        p = int(sel_pages[b, h, v])
        if p < 0 or p >= n_pages or p >= max_pages:
            bad += 1
            continue
        pages.append(p)
    return pages, bad


def visible_positions(L, window=0, sinks=0):
    """Positions 0..L-1 that the newest query of a sequence of L tokens sees.

    "ARGUS: Heterogeneous KV-cache memory management", section "v0.5:
    model-independent KV placement", lists sliding-window masks among what
    direct attention supports, and its "HuggingFace example" passes
    sink_tokens=4; neither spells the mask out.  Read plainly: a window of W
    keeps the newest W positions (L-W .. L-1) and the first `sinks` positions
    stay visible as well.  window <= 0 means no window (every position).
    Returns a boolean array of length L.
    """
    pos = np.arange(L)
    if window <= 0:
        return np.ones(L, dtype=bool)
    return (pos >= L - window) | (pos < sinks)


def paged_decode(q_f64, Hkv, P, pools, page_codec, block_table, seq_lens, scale,
                 sel_pages=None, sel_count=None, sel_width=0, window=0, sinks=0):
    """Single-token decode attention over a paged mixed-codec KV cache.

    q_f64       float64 [B][Hq][D] (the query values)
    pools       dict codec -> (codes, meta) in the layout of oracle.codecs
    page_codec  int [B][max_pages]: codec of each logical page
    block_table int [B][max_pages]: physical slot of each logical page in the
                pool of its codec (logical -> physical translation, "Design"
                section of the host-RAM KV tier pull request)
    seq_lens    int [B]: tokens in each sequence; token t of logical page p is
                position p*P + t, visible iff < seq_len
    sel_pages / sel_count / sel_width: optional selected-page lists
                [B][Hkv][width] (sparse decode over the indexer's selection)
    window / sinks: sliding window of the newest `window` positions plus the
                first `sinks` (see visible_positions); a page without a
                visible position is neither read nor checked

    Returns (o [B][Hq][D], lse2 [B][Hq], bad) where bad counts pages skipped
    because their slot is out of range plus rejected selection entries.
    """
    B, Hq, D = q_f64.shape
    G = Hq // Hkv
    max_pages = block_table.shape[1]
    o = np.zeros((B, Hq, D))
    lse2 = np.full((B, Hq), -math.inf)
    bad = 0
    for b in range(B):
        L = int(seq_lens[b])
        vis = visible_positions(L, window, sinks)
        for h in range(Hkv):
            pages, nbad = _visible_pages(b, h, L, P, max_pages, sel_pages,
                                         sel_count, sel_width)
            bad += nbad
            Ks, Vs = [], []
            for p in pages:
                n_tok = min(P, L - p * P)
                keep = vis[p * P:p * P + n_tok]
                if not keep.any():
                    continue
                codec = int(page_codec[b, p])
                slot = int(block_table[b, p])
                codes, meta = pools[codec]
                if slot < 0 or slot >= codes.shape[0]:
                    bad += 1
                    continue
                Ks.append(dequant_page(codec, codes, meta, slot, 0, h)[:n_tok][keep])
                Vs.append(dequant_page(codec, codes, meta, slot, 1, h)[:n_tok][keep])
            K = np.concatenate(Ks) if Ks else np.zeros((0, D))
            V = np.concatenate(Vs) if Vs else np.zeros((0, D))
            for g in range(G):
                o[b, h * G + g], lse2[b, h * G + g] = softmax_attention(
                    q_f64[b, h * G + g], K, V, scale)
    return o, lse2, bad


def fold_lse(acc_o, acc_lse2, part_o, part_lse2):
    """Fold one partial result into an accumulator by log2-sum-exp.

    For rows with partial (o_b, L_b) and accumulator (o_a, L_a):
        L = max + log2(2^(L_a - max) + 2^(L_b - max)),
        o = 2^(L_a - L) o_a + 2^(L_b - L) o_b,
    an empty side (L = -inf) being the identity.  Returns new (o, lse2).
    """
    acc_o = np.asarray(acc_o, np.float64)
    part_o = np.asarray(part_o, np.float64)
    La = np.asarray(acc_lse2, np.float64)
    Lb = np.asarray(part_lse2, np.float64)
    o = acc_o.copy()
    L = La.copy()
    for i in np.ndindex(La.shape):
        a, b = La[i], Lb[i]
        if b == -math.inf:
            continue
        if a == -math.inf:
            o[i] = part_o[i]
            L[i] = b
            continue
        m = max(a, b)
        Lab = m + math.log2(2.0 ** (a - m) + 2.0 ** (b - m))
        o[i] = 2.0 ** (a - Lab) * acc_o[i] + 2.0 ** (b - Lab) * part_o[i]
        L[i] = Lab
    return o, L


def window_attention(q_f64, k_f64, v_f64, win_pos0, q_pos0, scale, rows=None):
    """Attention of a query chunk against one window of cached keys.

    q_f64 [Hq][n_q][D]; k_f64, v_f64 [Hkv][W][D].  Key j of the window sits at
    absolute position win_pos0 + j, query row i at q_pos0 + i; the key is
    visible iff win_pos0 + j <= q_pos0 + i (causal inside the chunk, full view
    of earlier context).  rows: optional list of query rows to evaluate.
    Returns (o [Hq][n_rows][D], lse2 [Hq][n_rows]).
    """
    Hq, n_q, D = q_f64.shape
    Hkv, W, _ = k_f64.shape
    G = Hq // Hkv
    rows = list(range(n_q)) if rows is None else list(rows)
    o = np.zeros((Hq, len(rows), D))
    lse2 = np.full((Hq, len(rows)), -math.inf)
    for hq in range(Hq):
        h = hq // G
        for r, i in enumerate(rows):
            n_vis = int(np.clip(q_pos0 + i - win_pos0 + 1, 0, W))
            o[hq, r], lse2[hq, r] = softmax_attention(
                q_f64[hq, i], k_f64[h, :n_vis], v_f64[h, :n_vis], scale)
    return o, lse2


def gather_window(Hkv, P, pools, page_codec, block_table, b, win_pos0, win_len, seq_len=None):
    """K and V of one window of a paged, mixed-codec cache.

    The comment on "--kv-placement host" in "feat(kvcache): host-RAM KV tier
    for sparse-attention models" stages a prefill's cached pages into a
    device window before attending to it.  Here the window holds logical
    positions win_pos0 .. win_pos0 + win_len - 1 of sequence b: position p
    lies in logical page p // P at row p % P, whose codec and physical slot
    come from page_codec / block_table, and is dequantised exactly (float64).
    The window must lie inside the table's pages and, when seq_len is given,
    end at or before it.  Returns (K, V) float64 [Hkv][win_len][D]; win_len >= 1.
    """
    assert win_len >= 1
    assert 0 <= win_pos0 and win_pos0 + win_len <= block_table.shape[1] * P, "window outside the block table"
    assert seq_len is None or win_pos0 + win_len <= seq_len, "window runs past the sequence"
    Ks, Vs = [], []
    cache = {}
    for p in range(win_pos0, win_pos0 + win_len):
        page = p // P
        if page not in cache:
            codec = int(page_codec[b, page])
            slot = int(block_table[b, page])
            codes, meta = pools[codec]
            cache[page] = [(dequant_page(codec, codes, meta, slot, 0, h),
                            dequant_page(codec, codes, meta, slot, 1, h)) for h in range(Hkv)]
        kv = cache[page]
        Ks.append(np.stack([kv[h][0][p % P] for h in range(Hkv)]))
        Vs.append(np.stack([kv[h][1][p % P] for h in range(Hkv)]))
    return np.stack(Ks, axis=1), np.stack(Vs, axis=1)


def paged_window_attention(q_f64, Hkv, P, pools, page_codec, block_table, b, win_pos0, win_len,
                           q_pos0, scale, rows=None, seq_len=None):
    """window_attention over a window gathered from the paged cache
    (gather_window): the staged-prefill step, with pages in any codec tier."""
    if win_len == 0:
        K = V = np.zeros((Hkv, 0, q_f64.shape[-1]))
    else:
        K, V = gather_window(Hkv, P, pools, page_codec, block_table, b, win_pos0, win_len, seq_len)
    return window_attention(q_f64, K, V, win_pos0, q_pos0, scale, rows)


def staging_moves_less(row_read_bytes, cache_bytes):
    """The host-placement comment's staging_moves_less: a prefill stages the
    cache into device windows when the in-place reads of its rows (each row
    reading its own pages) add up to more bytes than the cache holds.  row_read_bytes:
    bytes each query row would read in place (an iterable); True means stage.
    """
    return sum(int(x) for x in row_read_bytes) > int(cache_bytes)


def to_f64(bits, dtype):
    """16-bit bit patterns (numpy uint16) -> float64 values."""
    return bits_to_f64(bits, dtype)
