"""Algorithmic byte and FLOP counts used for the roofline figures.

A decode kernel must read, at least once, every stored K/V byte of the
visible tokens plus the per-page metadata; that count divided by the kernel's
duration is its achieved bandwidth.  This is the transfer lower bound
T >= S_wire / B of "Storage contracts for hybrid KV cache offloading"
(section "Stored-byte savings are not a latency result").
"""

FP16, BF16, FP8_E4M3, INT8, INT4_G32, INT2_G32, INT1_G32 = 0, 1, 2, 3, 4, 5, 6


def code_bytes_per_row(codec, head_dim):
    """Stored code bytes of one token row of one head (K or V)."""
    if codec in (FP16, BF16):
        return 2 * head_dim
    if codec in (FP8_E4M3, INT8):
        return head_dim
    if codec == INT4_G32:
        return head_dim // 2
    if codec == INT2_G32:
        return head_dim // 4
    if codec == INT1_G32:
        return head_dim // 8
    raise ValueError(codec)


def meta_bytes_per_row(codec, head_dim):
    """Per-token metadata bytes of one head (INT4 / INT2 / INT1: one fp16 scale + zero per group)."""
    if codec in (INT4_G32, INT2_G32, INT1_G32):
        return 4 * (head_dim // 32)
    return 0


def meta_bytes_per_unit(codec):
    """Per-(page, head, K-or-V) metadata bytes (FP8 / INT8: one fp32 scale)."""
    return 4 if codec in (FP8_E4M3, INT8) else 0


def kv_bytes(codec, tokens, kv_heads, head_dim, pages):
    """Bytes of K and V for `tokens` visible tokens spread over `pages` pages."""
    per_row = code_bytes_per_row(codec, head_dim) + meta_bytes_per_row(codec, head_dim)
    return 2 * kv_heads * (tokens * per_row + pages * meta_bytes_per_unit(codec))


def bits_per_element(codec, head_dim):
    per_row = code_bytes_per_row(codec, head_dim) + meta_bytes_per_row(codec, head_dim)
    return 8.0 * per_row / head_dim


def quantize_bytes(dst_codec, src_elem_bytes, units, page_tokens, head_dim):
    """Read + write bytes of demoting `units` (page, head, K-or-V) units."""
    n = page_tokens * head_dim
    read = units * n * src_elem_bytes
    write = units * (page_tokens * (code_bytes_per_row(dst_codec, head_dim)
                                    + meta_bytes_per_row(dst_codec, head_dim))
                     + meta_bytes_per_unit(dst_codec))
    return read + write


def prefill_flops(q_heads, head_dim, n_q, visible_pairs):
    """4 * D * Hq * (number of visible (query, key) pairs): QK^T and PV."""
    return 4 * head_dim * q_heads * visible_pairs


def window_visible(seq_len, page_tokens, window, sinks):
    """(tokens, pages) a decode query reads under a sliding window of `window`
    newest tokens plus `sinks` leading ones (window <= 0: every token); pages
    counts the logical pages holding at least one visible token."""
    L, P = int(seq_len), int(page_tokens)
    if window <= 0:
        return L, (L + P - 1) // P
    lo = max(0, L - window)
    s = min(sinks, lo)                       # sinks that lie before the window
    pages = set(range((lo // P), (L + P - 1) // P)) | set(range((s + P - 1) // P))
    return (L - lo) + s, len(pages)
