"""ctypes binding of libargus.so: argument marshalling only.

Every function here forwards to the C entry point of the same name declared in
include/argus.h; tensors are passed as raw device pointers (torch is used for
device memory and streams only).  A failing status raises ArgusError with the
library's one-line reason.  There is no fallback: if the library has not been
built, lib() raises.
"""

import ctypes
import os

import torch

FP16, BF16, FP8_E4M3, INT8, INT4_G32, INT2_G32, INT1_G32 = 0, 1, 2, 3, 4, 5, 6
CODEC_NAMES = {FP16: "fp16", BF16: "bf16", FP8_E4M3: "fp8_e4m3", INT8: "int8", INT4_G32: "int4_g32",
               INT2_G32: "int2_g32", INT1_G32: "int1_g32"}
DTYPE_CODEC = {torch.float16: FP16, torch.bfloat16: BF16}

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libargus.so")
_lib = None


class ArgusError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__("argus status %d: %s" % (status, msg))
        self.status = status


class Geom(ctypes.Structure):
    _fields_ = [("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_tokens", ctypes.c_int32)]


PLACE_DEVICE, PLACE_HOST = 0, 1


class PoolDesc(ctypes.Structure):
    _fields_ = [("codec", ctypes.c_int32), ("placement", ctypes.c_int32),
                ("codes", ctypes.c_void_p), ("meta", ctypes.c_void_p),
                ("n_slots", ctypes.c_int64)]


class DecodeArgs(ctypes.Structure):
    _fields_ = [("g", Geom), ("batch", ctypes.c_int32), ("q_dtype", ctypes.c_int32),
                ("q", ctypes.c_void_p), ("pools", ctypes.POINTER(PoolDesc)),
                ("n_pools", ctypes.c_int32), ("max_pages", ctypes.c_int32),
                ("page_codec", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
                ("seq_lens", ctypes.c_void_p), ("sel_pages", ctypes.c_void_p),
                ("sel_count", ctypes.c_void_p), ("sel_width", ctypes.c_int32),
                ("softmax_scale", ctypes.c_float), ("out", ctypes.c_void_p),
                ("out_dtype", ctypes.c_int32), ("out_f32", ctypes.c_void_p),
                ("lse2_out", ctypes.c_void_p), ("status", ctypes.c_void_p),
                ("num_splits", ctypes.c_int32), ("pdl", ctypes.c_int32),
                ("window_tokens", ctypes.c_int32), ("sink_tokens", ctypes.c_int32)]


EXPORTS = ["argus_quantize_pages", "argus_decode_workspace_bytes", "argus_paged_decode_attn",
           "argus_paged_decode_attn_noalloc",
           "argus_select_workspace_bytes", "argus_select_pages", "argus_fold_lse",
           "argus_window_prefill_workspace_bytes", "argus_window_prefill_attn",
           "argus_paged_window_prefill_workspace_bytes", "argus_paged_window_prefill_attn",
           "argus_staging_moves_less", "argus_test_decode_stall",
           "argus_status_string", "argus_last_error"]


def lib_path():
    return _LIB_PATH


def lib():
    """Load libargus.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError("libargus.so is not built; run __graft_entry__.build() "
                           "(python -m mixed_precision_paged_argus_gb300.build)")
    L = ctypes.CDLL(_LIB_PATH)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    L.argus_status_string.restype = ctypes.c_char_p
    L.argus_status_string.argtypes = [ctypes.c_int]
    L.argus_last_error.restype = ctypes.c_char_p
    L.argus_last_error.argtypes = []
    L.argus_quantize_pages.restype = ctypes.c_int
    L.argus_quantize_pages.argtypes = [ctypes.POINTER(Geom), i32, vp, i64, vp, ctypes.POINTER(PoolDesc),
                                       vp, i32, vp, vp, vp, vp]
    L.argus_decode_workspace_bytes.restype = ctypes.c_int
    L.argus_decode_workspace_bytes.argtypes = [ctypes.POINTER(DecodeArgs), ctypes.POINTER(sz)]
    L.argus_paged_decode_attn.restype = ctypes.c_int
    L.argus_paged_decode_attn.argtypes = [ctypes.POINTER(DecodeArgs), vp, sz, vp]
    L.argus_test_decode_stall.restype = ctypes.c_int
    L.argus_test_decode_stall.argtypes = [ctypes.POINTER(DecodeArgs), vp, sz, ctypes.c_uint32, i32, vp]
    L.argus_paged_decode_attn_noalloc.restype = ctypes.c_int
    L.argus_paged_decode_attn_noalloc.argtypes = [ctypes.POINTER(DecodeArgs), vp]
    L.argus_select_workspace_bytes.restype = ctypes.c_int
    L.argus_select_workspace_bytes.argtypes = [ctypes.POINTER(Geom), i32, i32, ctypes.POINTER(sz)]
    L.argus_select_pages.restype = ctypes.c_int
    L.argus_select_pages.argtypes = [ctypes.POINTER(Geom), i32, vp, i32, vp, vp, i32, i32, i32,
                                     vp, vp, i32, vp, vp, sz, vp]
    L.argus_fold_lse.restype = ctypes.c_int
    L.argus_fold_lse.argtypes = [i64, i32, vp, vp, vp, vp, vp]
    L.argus_window_prefill_attn.restype = ctypes.c_int
    L.argus_window_prefill_attn.argtypes = [ctypes.POINTER(Geom), i32, vp, vp, vp, i64, i64, i64, i64,
                                            ctypes.c_float, vp, vp, i32, i32, vp, sz, vp]
    L.argus_window_prefill_workspace_bytes.restype = ctypes.c_int
    L.argus_window_prefill_workspace_bytes.argtypes = [ctypes.POINTER(Geom), i32, i64, i32, ctypes.POINTER(sz)]
    L.argus_paged_window_prefill_workspace_bytes.restype = ctypes.c_int
    L.argus_paged_window_prefill_workspace_bytes.argtypes = [ctypes.POINTER(Geom), i32, i64, i32, ctypes.POINTER(sz)]
    L.argus_paged_window_prefill_attn.restype = ctypes.c_int
    L.argus_paged_window_prefill_attn.argtypes = [ctypes.POINTER(Geom), i32, vp, ctypes.POINTER(PoolDesc), i32, vp, vp,
                                                  i32, i64, i64, i64, ctypes.c_float, vp, vp, i32, i32, vp, sz, vp, vp]
    L.argus_staging_moves_less.restype = ctypes.c_int
    L.argus_staging_moves_less.argtypes = [ctypes.POINTER(ctypes.c_int64), i64, i64, ctypes.POINTER(i32)]
    _lib = L
    return L


def _check(status):
    if status != 0:
        L = lib()
        raise ArgusError(status, L.argus_last_error().decode())


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def geom(n_q_heads, n_kv_heads, head_dim, page_tokens):
    return Geom(n_q_heads, n_kv_heads, head_dim, page_tokens)


class Pool:
    """A physical page pool of one codec: codes (and meta) tensors, on the
    device, or in page-locked host memory (placement PLACE_HOST: read in place
    by decode over the host link)."""

    def __init__(self, codec, codes, meta, n_slots, placement=None):
        self.codec, self.codes, self.meta, self.n_slots = codec, codes, meta, int(n_slots)
        if placement is None:
            placement = PLACE_HOST if (codes is not None and not codes.is_cuda) else PLACE_DEVICE
        self.placement = placement

    def desc(self):
        return PoolDesc(self.codec, self.placement, _ptr(self.codes), _ptr(self.meta), self.n_slots)

    def to_host(self):
        """A copy of this pool in page-locked host memory (PLACE_HOST)."""
        codes = self.codes.cpu().pin_memory()
        meta = None if self.meta is None else self.meta.cpu().pin_memory()
        return Pool(self.codec, codes, meta, self.n_slots, PLACE_HOST)

    @staticmethod
    def empty(codec, n_slots, n_kv_heads, page_tokens, head_dim, device="cuda", zero=False):
        """Allocate a pool in the layout of include/argus.h (device="host":
        page-locked host memory)."""
        if str(device) == "host":
            p = Pool.empty(codec, n_slots, n_kv_heads, page_tokens, head_dim, device="cpu", zero=zero)
            return Pool(codec, p.codes.pin_memory(), None if p.meta is None else p.meta.pin_memory(), n_slots,
                        PLACE_HOST)
        alloc = torch.zeros if zero else torch.empty
        shape = (n_slots, 2, n_kv_heads, page_tokens)
        if codec in (FP16, BF16):
            codes = alloc(shape + (head_dim,), dtype=torch.float16 if codec == FP16 else torch.bfloat16,
                          device=device)
            meta = None
        elif codec in (FP8_E4M3, INT8):
            codes = alloc(shape + (head_dim,), dtype=torch.uint8, device=device)
            meta = alloc((n_slots, 2, n_kv_heads), dtype=torch.float32, device=device)
        elif codec in (INT4_G32, INT2_G32, INT1_G32):
            per_byte = {INT4_G32: 2, INT2_G32: 4, INT1_G32: 8}[codec]
            codes = alloc(shape + (head_dim // per_byte,), dtype=torch.uint8, device=device)
            meta = alloc(shape + (head_dim // 32, 2), dtype=torch.float16, device=device)
        else:
            raise ValueError(codec)
        return Pool(codec, codes, meta, n_slots)


def quantize_pages(g, src_dtype, src_codes, n_src_slots, src_slots, dst, dst_slots, n_pages,
                   valid_tokens=None, ckey_out=None, status=None, stream=None):
    d = dst.desc()
    _check(lib().argus_quantize_pages(ctypes.byref(g), src_dtype, _ptr(src_codes), int(n_src_slots),
                                      _ptr(src_slots), ctypes.byref(d), _ptr(dst_slots), int(n_pages),
                                      _ptr(valid_tokens), _ptr(ckey_out), _ptr(status), _stream(stream)))


def decode_args(g, batch, q, pools, page_codec, block_table, seq_lens, max_pages, softmax_scale,
                out=None, out_f32=None, lse2_out=None, sel_pages=None, sel_count=None, sel_width=0,
                status=None, num_splits=0, pdl=False, window_tokens=0, sink_tokens=0):
    """Build an argus_decode_args struct (keeps the pool array alive on the struct)."""
    arr = (PoolDesc * max(1, len(pools)))(*[p.desc() for p in pools])
    a = DecodeArgs()
    a.g = g
    a.batch = int(batch)
    a.q_dtype = DTYPE_CODEC[q.dtype]
    a.q = _ptr(q)
    a.pools = ctypes.cast(arr, ctypes.POINTER(PoolDesc))
    a.n_pools = len(pools)
    a.max_pages = int(max_pages)
    a.page_codec = _ptr(page_codec)
    a.block_table = _ptr(block_table)
    a.seq_lens = _ptr(seq_lens)
    a.sel_pages = _ptr(sel_pages)
    a.sel_count = _ptr(sel_count)
    a.sel_width = int(sel_width)
    a.softmax_scale = float(softmax_scale)
    a.out = _ptr(out)
    a.out_dtype = DTYPE_CODEC[out.dtype] if out is not None else FP16
    a.out_f32 = _ptr(out_f32)
    a.lse2_out = _ptr(lse2_out)
    a.status = _ptr(status)
    a.num_splits = int(num_splits)
    a.pdl = int(pdl)   # False / True / 2
    a.window_tokens = int(window_tokens)
    a.sink_tokens = int(sink_tokens)
    # the struct holds raw pointers: keep every tensor it points to alive with it
    a._keep = (arr, list(pools), q, page_codec, block_table, seq_lens, sel_pages, sel_count, out,
               out_f32, lse2_out, status)
    return a


def decode_workspace_bytes(args):
    n = ctypes.c_size_t(0)
    _check(lib().argus_decode_workspace_bytes(ctypes.byref(args), ctypes.byref(n)))
    return n.value


def paged_decode_attn(args, ws, ws_bytes=None, stream=None):
    if ws_bytes is None:
        ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().argus_paged_decode_attn(ctypes.byref(args), _ptr(ws), int(ws_bytes), _stream(stream)))


STATUS_TIMEOUT_BIT = 0x80000000


def test_decode_stall(args, ws, wait_limit_us, stall_stage, stream=None):
    """Testing only: the decode with every device wait limited to wait_limit_us
    and stage stall_stage's arrival withheld, so that the waits run out."""
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().argus_test_decode_stall(ctypes.byref(args), _ptr(ws), nbytes, int(wait_limit_us),
                                         int(stall_stage), _stream(stream)))


NOALLOC_SCRATCH_BYTES = 4 << 20


def paged_decode_attn_noalloc(args, stream=None):
    """Decode with the library's fixed device scratch instead of a workspace
    (for callers that cannot allocate; calls must not overlap on the GPU)."""
    _check(lib().argus_paged_decode_attn_noalloc(ctypes.byref(args), _stream(stream)))


def select_workspace_bytes(g, batch, max_pages):
    n = ctypes.c_size_t(0)
    _check(lib().argus_select_workspace_bytes(ctypes.byref(g), int(batch), int(max_pages), ctypes.byref(n)))
    return n.value


def select_pages(g, batch, q, ckeys, n_pages, max_pages, top_k, keep_newest, sel_pages, sel_count,
                 sel_width, drop_counter, ws, stream=None):
    _check(lib().argus_select_pages(ctypes.byref(g), int(batch), _ptr(q), DTYPE_CODEC[q.dtype], _ptr(ckeys),
                                    _ptr(n_pages), int(max_pages), int(top_k), int(bool(keep_newest)),
                                    _ptr(sel_pages), _ptr(sel_count), int(sel_width), _ptr(drop_counter),
                                    _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def fold_lse(acc_o, acc_lse2, part_o, part_lse2, stream=None):
    n_rows = acc_lse2.numel()
    head_dim = acc_o.numel() // max(1, n_rows)
    _check(lib().argus_fold_lse(int(n_rows), int(head_dim), _ptr(acc_o), _ptr(acc_lse2), _ptr(part_o),
                                _ptr(part_lse2), _stream(stream)))


def window_prefill_workspace_bytes(g, n_q, win_len, num_splits=0):
    n = ctypes.c_size_t(0)
    _check(lib().argus_window_prefill_workspace_bytes(ctypes.byref(g), int(n_q), int(win_len), int(num_splits),
                                                      ctypes.byref(n)))
    return n.value


def staging_moves_less(row_read_bytes, cache_bytes):
    """Whether a prefill should stage the cache into device windows: the rows'
    in-place reads (host list of byte counts) together exceed cache_bytes."""
    vals = [int(x) for x in row_read_bytes] + [int(cache_bytes)]
    for x in vals:
        # ctypes wraps integers silently; a byte count outside int64 must not
        # turn into a small valid one
        if not (-2 ** 63 <= x < 2 ** 63):
            raise ValueError("staging_moves_less: byte count %d does not fit in int64" % x)
    rows = (ctypes.c_int64 * max(1, len(row_read_bytes)))(*vals[:-1])
    out = ctypes.c_int32(0)
    _check(lib().argus_staging_moves_less(rows, len(row_read_bytes), vals[-1], ctypes.byref(out)))
    return bool(out.value)


def window_prefill_attn(g, n_q, q, k, v, kv_head_stride, win_len, win_pos0, q_pos0, softmax_scale,
                        acc_o, acc_lse2, fold, num_splits=0, ws=None, stream=None):
    """num_splits / ws: key ranges per query tile and their partial-result
    workspace (window_prefill_workspace_bytes bytes); 0 with ws chooses the
    split count, 0 without ws is one CTA per tile."""
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().argus_window_prefill_attn(ctypes.byref(g), int(n_q), _ptr(q), _ptr(k), _ptr(v),
                                           int(kv_head_stride), int(win_len), int(win_pos0), int(q_pos0),
                                           float(softmax_scale), _ptr(acc_o), _ptr(acc_lse2), int(fold),
                                           int(num_splits), _ptr(ws), nbytes, _stream(stream)))


def paged_window_prefill_workspace_bytes(g, n_q, win_len, num_splits=0):
    n = ctypes.c_size_t(0)
    _check(lib().argus_paged_window_prefill_workspace_bytes(ctypes.byref(g), int(n_q), int(win_len), int(num_splits),
                                                            ctypes.byref(n)))
    return n.value


def paged_window_prefill_attn(g, n_q, q, pools, page_codec, block_table, max_pages, win_pos0, win_len, q_pos0,
                              softmax_scale, acc_o, acc_lse2, fold, ws, num_splits=0, status=None, stream=None):
    """Stage one window of the paged cache (block_table / page_codec rows of one
    sequence, pools of any codec) and attend the query chunk to it, folding
    into acc_o / acc_lse2; ws of paged_window_prefill_workspace_bytes bytes."""
    arr = (PoolDesc * max(1, len(pools)))(*[p.desc() for p in pools])
    _check(lib().argus_paged_window_prefill_attn(ctypes.byref(g), int(n_q), _ptr(q),
                                                 ctypes.cast(arr, ctypes.POINTER(PoolDesc)), len(pools),
                                                 _ptr(page_codec), _ptr(block_table), int(max_pages), int(win_pos0),
                                                 int(win_len), int(q_pos0), float(softmax_scale), _ptr(acc_o),
                                                 _ptr(acc_lse2), int(fold), int(num_splits), _ptr(ws),
                                                 ws.numel() * ws.element_size(), _ptr(status), _stream(stream)))
