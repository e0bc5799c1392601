"""The C-ABI library loads on a CPU-only host and exports every declared symbol;
host-side validation answers without touching a GPU."""

import ctypes
import os
import re

import pytest

import mixed_precision_paged_argus_gb300.argus as argus

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "argus.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(argus_[a-z0-9_]+)\s*\(", text)))


def _lib():
    if not os.path.exists(argus.lib_path()):
        from mixed_precision_paged_argus_gb300 import build
        build.build()
    return argus.lib()


def test_header_declares_the_five_operations():
    names = _declared()
    for op in ("argus_quantize_pages", "argus_paged_decode_attn", "argus_select_pages",
               "argus_fold_lse", "argus_window_prefill_attn"):
        assert op in names


def test_library_exports_every_declared_symbol():
    L = _lib()
    raw = ctypes.CDLL(argus.lib_path())
    for name in _declared():
        assert hasattr(raw, name), name
    assert set(_declared()) <= set(argus.EXPORTS) | {"argus_status_string", "argus_last_error"} | set(_declared())


def test_status_strings():
    L = _lib()
    assert L.argus_status_string(0) == b"ok"
    assert L.argus_status_string(3) == b"workspace too small"


def test_host_validation_without_gpu():
    L = _lib()
    # fold: negative rows is rejected before any CUDA call
    assert L.argus_fold_lse(-1, 128, None, None, None, None, None) == 1
    assert L.argus_fold_lse(4, 6, None, None, None, None, None) == 2
    assert b"multiple of 4" in L.argus_last_error()
    # decode: unsupported head_dim / grouping fail closed
    a = argus.DecodeArgs()
    a.g = argus.geom(8, 2, 96, 16)
    a.batch, a.q_dtype, a.max_pages = 1, 0, 4
    n = ctypes.c_size_t(0)
    assert L.argus_decode_workspace_bytes(ctypes.byref(a), ctypes.byref(n)) == 2
    a.g = argus.geom(18, 2, 128, 16)
    assert L.argus_decode_workspace_bytes(ctypes.byref(a), ctypes.byref(n)) == 2
    a.g = argus.geom(8, 2, 128, 24)
    assert L.argus_decode_workspace_bytes(ctypes.byref(a), ctypes.byref(n)) == 2
    a.g = argus.geom(8, 2, 128, 16)
    a.pdl = 3   # 0, 1 or 2
    assert L.argus_decode_workspace_bytes(ctypes.byref(a), ctypes.byref(n)) == 1
    a.pdl = 2
    assert L.argus_decode_workspace_bytes(ctypes.byref(a), ctypes.byref(n)) == 0
    g = argus.geom(8, 2, 128, 16)
    assert L.argus_select_workspace_bytes(ctypes.byref(g), 2, 10, ctypes.byref(n)) == 0
    assert n.value == 2 * 2 * 10 * 4 + 2 * 2 * 2 * 2 * 4   # keys, then 2 reported keys of ceil(10 / 8) ranges


def test_codec_range_window_and_int2_checks_without_gpu():
    """Codec numbers outside 0..6 fail closed; INT2 and INT1 pools are accepted; a window
    rejects negative values and selection lists; a window shrinks the workspace."""
    L = _lib()
    n = ctypes.c_size_t(0)
    a = argus.DecodeArgs()
    a.g = argus.geom(8, 2, 128, 16)
    a.batch, a.q_dtype, a.max_pages, a.num_splits = 2, 0, 256, 4

    def pools(*codecs):
        arr = (argus.PoolDesc * len(codecs))(*[argus.PoolDesc(c, 0, 16, 16, 8) for c in codecs])
        a.pools = ctypes.cast(arr, ctypes.POINTER(argus.PoolDesc))
        a.n_pools = len(codecs)
        return arr

    keep = pools(argus.INT2_G32, argus.FP8_E4M3)
    assert L.argus_decode_workspace_bytes(ctypes.byref(a), ctypes.byref(n)) == 0
    full = n.value
    keep = pools(argus.INT1_G32, argus.INT8)
    assert L.argus_decode_workspace_bytes(ctypes.byref(a), ctypes.byref(n)) == 0
    keep = pools(7)
    assert L.argus_decode_workspace_bytes(ctypes.byref(a), ctypes.byref(n)) == 1
    keep = pools(argus.INT2_G32)
    a.window_tokens, a.sink_tokens = 64, 4
    assert L.argus_decode_workspace_bytes(ctypes.byref(a), ctypes.byref(n)) == 0
    assert n.value < full
    a.window_tokens = -1
    assert L.argus_decode_workspace_bytes(ctypes.byref(a), ctypes.byref(n)) == 1
    a.window_tokens, a.sink_tokens = 64, -4
    assert L.argus_decode_workspace_bytes(ctypes.byref(a), ctypes.byref(n)) == 1
    a.sink_tokens = 4
    sel = ctypes.c_int32(0)
    a.sel_pages = a.sel_count = ctypes.cast(ctypes.byref(sel), ctypes.c_void_p)
    a.sel_width = 4
    assert L.argus_decode_workspace_bytes(ctypes.byref(a), ctypes.byref(n)) == 2
    # a selection's entries are dealt over at most sel_width splits: workspace
    # = B * Hkv * splits * G * (D + 1) fp32 values
    a.window_tokens = a.sink_tokens = 0
    for req, splits in ((3, 3), (4, 4), (100, 4)):
        a.num_splits = req
        assert L.argus_decode_workspace_bytes(ctypes.byref(a), ctypes.byref(n)) == 0
        assert n.value == 2 * 2 * splits * 4 * (128 + 1) * 4
    del keep
    # quantize: destination codec 7 is rejected before any device work
    g = argus.geom(8, 2, 128, 16)
    dst = argus.PoolDesc(7, 0, 16, 16, 4)
    assert L.argus_quantize_pages(ctypes.byref(g), argus.FP16, 16, 4, 16, ctypes.byref(dst), 16, 1,
                                  None, None, None, None) == 1


def _c_layout(struct, fields, tmp_path):
    """sizeof and offsetof of a header struct, from a C program compiled by gcc."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "layout.c"
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "argus.h"', 'int main(void) {',
             '  printf("%%zu\\n", sizeof(%s));' % struct]
    lines += ['  printf("%%zu\\n", offsetof(%s, %s));' % (struct, f) for f in fields]
    lines += ['  return 0;', '}']
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    return int(out[0]), [int(x) for x in out[1:]]


@pytest.mark.parametrize("cls,struct", [(argus.Geom, "argus_geom"), (argus.PoolDesc, "argus_pool"),
                                        (argus.DecodeArgs, "argus_decode_args")])
def test_binding_structs_match_the_header_layout(cls, struct, tmp_path):
    """Every field of the ctypes mirror sits at the C offset, and the sizes agree
    (the header's structs are what the library reads)."""
    names = [f[0] for f in cls._fields_]
    size, offs = _c_layout(struct, names, tmp_path)
    assert ctypes.sizeof(cls) == size
    for name, off in zip(names, offs):
        assert getattr(cls, name).offset == off, name


def test_staging_decision_matches_the_oracle_without_gpu():
    """argus_staging_moves_less is host logic: it runs here, against the oracle's
    reading of the staging rule, including sums far beyond int64 headroom."""
    from oracle import attention as A
    import numpy as np
    _lib()
    rng = np.random.default_rng(5)
    for _ in range(300):
        n = int(rng.integers(0, 40))
        rows = rng.integers(0, 5000, size=n).tolist()
        cache = int(rng.integers(0, 100000))
        assert argus.staging_moves_less(rows, cache) == A.staging_moves_less(rows, cache)
    big = 2 ** 62
    assert argus.staging_moves_less([big, big, big], 2 ** 63 - 1)      # no overflow in the sum
    assert not argus.staging_moves_less([big - 1, big], 2 ** 63 - 1)
    assert not argus.staging_moves_less([], 0)
    with pytest.raises(argus.ArgusError) as e:
        argus.staging_moves_less([3, -1], 10)
    assert e.value.status == 1
    with pytest.raises(argus.ArgusError):
        argus.staging_moves_less([1], -5)
    # counts outside int64 are refused by the binding before ctypes could wrap them
    with pytest.raises(ValueError):
        argus.staging_moves_less([2 ** 64 + 3], 10)
    with pytest.raises(ValueError):
        argus.staging_moves_less([1], 2 ** 63)
