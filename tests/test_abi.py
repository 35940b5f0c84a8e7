"""The C ABI library: builds, loads without a GPU, exports every declared symbol, checks host arguments."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_draft_dflash_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:[\w\s\*]+?)\b(dflash_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_calls():
    names = declared_functions()
    for n in ("dflash_ctx_project", "dflash_kv_inject", "dflash_block_attn", "dflash_cache_crop",
              "dflash_rope_table_build", "dflash_workspace_bytes", "dflash_status_get"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"libdflash.so does not export {n}"


def test_library_exports_nothing_else(lib):
    import subprocess
    from speculative_decoding_draft_dflash_gb300 import build
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True).stdout
    exported = sorted({l.split()[-1] for l in out.splitlines() if " T " in l and "dflash" in l})
    assert exported == declared_functions()


@pytest.fixture(scope="module")
def D(lib):
    from speculative_decoding_draft_dflash_gb300 import dflash
    return dflash


def _dims(D, **kw):
    base = dict(d=4096, n_h=32, n_kv=8, d_h=128, k_layers=5, block_size=16, eps=1e-6, dtype=D.DFLASH_BF16)
    base.update(kw)
    return D.dflash_dims(base["d"], base["n_h"], base["n_kv"], base["d_h"], base["k_layers"],
                         base["block_size"], base["eps"], base["dtype"])


def test_status_strings(D):
    assert D.status_string(0) == "ok"
    assert D.status_string(3) == "workspace too small"
    assert D.status_string(99) == "unknown status"


def test_workspace_bytes_host_logic(D):
    dims = _dims(D)
    small = D.dflash_workspace_bytes(dims, 1, 1056, 16)
    big = D.dflash_workspace_bytes(dims, 32, 4160, 512)
    assert 0 < small < big
    assert big % 256 == 0 and small % 256 == 0
    assert D.dflash_workspace_bytes(_dims(D, n_h=30), 1, 64, 16) == 0   # n_h % n_kv != 0
    assert D.dflash_workspace_bytes(dims, -1, 64, 16) == 0


@pytest.mark.parametrize("kw,expect", [
    (dict(n_h=30), 2), (dict(d_h=64), 2), (dict(block_size=17), 2), (dict(k_layers=9), 2),
    (dict(dtype=7), 2), (dict(d=0), 1), (dict(eps=-1.0), 1), (dict(d=4100), 2),
])
def test_unsupported_or_invalid_dims_rejected_before_launch(D, lib, kw, expect):
    dims = _dims(D, **kw)
    f = lib.dflash_ctx_project
    f.restype = ctypes.c_int
    ptrs = (ctypes.c_void_p * 8)(*([256] * 8))
    st = f(ctypes.byref(dims), ptrs, 16, ctypes.c_void_p(256), ctypes.c_void_p(256),
           ctypes.c_void_p(256), ctypes.c_void_p(256), ctypes.c_size_t(1 << 30), None)
    assert st == expect


def test_null_and_misaligned_pointers_rejected(D, lib):
    dims = _dims(D)
    f = lib.dflash_ctx_project
    f.restype = ctypes.c_int
    ptrs = (ctypes.c_void_p * 8)(*([256] * 8))
    args = [ctypes.byref(dims), ptrs, 16, ctypes.c_void_p(256), ctypes.c_void_p(256),
            ctypes.c_void_p(256), ctypes.c_void_p(256), ctypes.c_size_t(1 << 30), None]
    for i in (3, 4, 5, 6):
        a = list(args)
        a[i] = None
        assert f(*a) == 1
    a = list(args)
    a[3] = ctypes.c_void_p(258)          # W_fc not 16-byte aligned
    assert f(*a) == 1
    a = list(args)
    a[6] = ctypes.c_void_p(512 + 16)     # workspace not 256-byte aligned
    assert f(*a) == 1
    a = list(args)
    a[7] = ctypes.c_size_t(100)          # workspace too small
    assert f(*a) == 3
    a = list(args)
    a[2] = -1
    assert f(*a) == 1
    a = list(args)
    a[2] = 0                             # no rows: nothing to do
    assert f(*a) == 0


def test_cache_and_window_arguments_rejected(D, lib):
    dims = _dims(D)
    cache = D.dflash_kv_cache(256, 512, 1024, 2, 4, 64)
    f = lib.dflash_block_attn
    f.restype = ctypes.c_int
    P = ctypes.c_void_p
    base = [ctypes.byref(dims), ctypes.byref(cache), 0, P(256), P(256), P(256), P(256), P(256),
            P(256), P(256), 64, 0, ctypes.c_float(0.0), P(256), P(256), ctypes.c_size_t(100), None]
    a = list(base); a[2] = 2          # layer out of range
    assert f(*a) == 1
    a = list(base); a[11] = 8         # window smaller than the block
    assert f(*a) == 1
    a = list(base); a[11] = -1
    assert f(*a) == 1
    bad = D.dflash_kv_cache(256, 512, 1024, 2, 0, 64)   # batch 0
    a = list(base); a[1] = ctypes.byref(bad)
    assert f(*a) == 1
    a = list(base)                     # valid but workspace of 100 bytes
    assert f(*a) == 3
    crop = lib.dflash_cache_crop
    crop.restype = ctypes.c_int
    assert crop(ctypes.byref(cache), None, None) == 1
    assert crop(ctypes.byref(cache), P(1026), None) == 1


def test_accept_arguments_rejected_before_launch(lib):
    f = lib.dflash_accept
    f.restype = ctypes.c_int
    P = ctypes.c_void_p
    base = [P(256), P(512), 4, 16, P(768), P(1024), P(1280), P(1536), P(1792), None]
    a = list(base); a[2] = -1          # negative batch
    assert f(*a) == 1
    a = list(base); a[3] = 0           # empty blocks
    assert f(*a) == 1
    for i in (0, 1, 4, 5, 6, 7, 8):
        a = list(base); a[i] = None
        assert f(*a) == 1
    a = list(base); a[6] = P(1282)     # cu_rows not 4-byte aligned
    assert f(*a) == 1
    a = list(base); a[2] = 0; a[0] = None   # no sequences: only cu_rows is needed
    a[1] = a[4] = a[5] = a[7] = a[8] = None
    assert f(*a) in (0, 4)             # launches (status 0) or, without a GPU, a CUDA error


def test_layer_out_arguments_rejected_before_launch(D, lib):
    dims = _dims(D)
    ws = lib.dflash_layer_out_workspace_bytes
    ws.restype = ctypes.c_size_t
    assert ws(ctypes.byref(dims), 64, 1024) > 0
    assert ws(ctypes.byref(dims), 64, 0) == 0 and ws(ctypes.byref(dims), 64, 1002) == 0
    f = lib.dflash_layer_out
    f.restype = ctypes.c_int
    P = ctypes.c_void_p
    base = [ctypes.byref(dims), 64, P(256), P(512), P(768), P(1024), 1024, P(1280), P(1536),
            P(1792), P(2048), P(4096), ctypes.c_size_t(1 << 30), None]
    for i in (2, 3, 4, 5, 7, 8, 9, 10, 11):
        a = list(base); a[i] = None
        assert f(*a) == 1
    a = list(base); a[4] = P(770)       # W_O misaligned
    assert f(*a) == 1
    a = list(base); a[6] = 1000         # d_ff not a multiple of 64 on the bf16 path
    assert f(*a) == 2
    a = list(base); a[12] = ctypes.c_size_t(1000)
    assert f(*a) == 3
    a = list(base); a[1] = 0
    assert f(*a) == 0
    n = lib.dflash_rms_norm
    n.restype = ctypes.c_int
    assert n(ctypes.byref(dims), 4, None, P(256), P(512), None) == 1
    assert n(ctypes.byref(dims), -1, P(256), P(256), P(512), None) == 1


def test_paged_cache_arguments_rejected(D, lib):
    f = lib.dflash_kv_inject
    f.restype = ctypes.c_int
    P = ctypes.c_void_p
    dims = _dims(D)
    def call(cache, dm=dims):
        return f(ctypes.byref(dm), ctypes.byref(cache), 0, P(256), P(512), 16, P(768), P(1024),
                 P(1280), P(1536), 64, P(2048), ctypes.c_size_t(100), None)
    bad_page = D.dflash_kv_cache(256, 512, 1024, 2, 4, 256, P(4096), 64, 8)
    assert call(bad_page) == 1                      # pages must be 128 rows
    bad_cap = D.dflash_kv_cache(256, 512, 1024, 2, 4, 200, P(4096), 128, 8)
    assert call(bad_cap) == 1                       # capacity in whole pages
    no_pages = D.dflash_kv_cache(256, 512, 1024, 2, 4, 256, P(4096), 128, 0)
    assert call(no_pages) == 1
    f32 = _dims(D, dtype=D.DFLASH_F32, d=512, n_h=8, n_kv=8, d_h=64)
    paged = D.dflash_kv_cache(256, 512, 1024, 2, 4, 256, P(4096), 128, 8)
    assert call(paged, f32) == 2                    # paged layout: bf16 path only
    assert call(paged) == 3                         # valid paged cache, 100-byte workspace


def test_fp8_cache_arguments_rejected(D, lib):
    f = lib.dflash_kv_inject
    f.restype = ctypes.c_int
    P = ctypes.c_void_p
    dims = _dims(D)
    f32 = _dims(D, dtype=D.DFLASH_F32, d=512, n_h=8, n_kv=8, d_h=64)

    def call(cache, dm=dims):
        return f(ctypes.byref(dm), ctypes.byref(cache), 0, P(256), P(512), 16, P(768), P(1024),
                 P(1280), P(1536), 64, P(2048), ctypes.c_size_t(100), None)

    def cache(kv_dtype, scales=None, paged=False):
        s = None if scales is None else (ctypes.c_float * 4)(*scales)
        c = D.dflash_kv_cache(256, 512, 1024, 2, 4, 256, P(4096) if paged else None,
                              128 if paged else 0, 8 if paged else 0, kv_dtype,
                              ctypes.addressof(s) if s is not None else None)
        c._keep = s
        return c

    fp8 = D.DFLASH_FP8_E4M3
    assert call(cache(fp8, (0.5, 0.25, 1.0, 2.0))) == 3     # valid, 100-byte workspace
    assert call(cache(fp8)) == 3                            # no scales: 1 everywhere
    assert call(cache(fp8, (0.5, 0.25, 1.0, 2.0), paged=True)) == 3
    assert call(cache(D.DFLASH_BF16)) == 3                  # the dims' own type
    assert call(cache(fp8, (0.5, 0.25, 1.0, 2.0)), f32) == 2  # fp8: bf16 dims only
    assert call(cache(7)) == 2                              # unknown element type
    for bad in ((0.5, 0.0, 1.0, 2.0), (0.5, -1.0, 1.0, 2.0), (0.5, 0.25, float("nan"), 2.0),
                (0.5, 0.25, 1.0, float("inf"))):
        assert call(cache(fp8, bad)) == 1, bad


def test_binding_checks_hidden_state_tensors(D):
    """The k hidden-state pointers go through the same checks as every other tensor argument:
    a host tensor or a strided view is refused before the library is called."""
    import torch
    dims = _dims(D)
    ws = torch.zeros(256, dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA"):
        D.dflash_ctx_project(dims, [torch.zeros((4, 64))], 4, None, None, None, ws)
    strided = torch.zeros((64, 8)).t()

    class FakeCuda:                      # a strided "device" tensor, no GPU needed
        is_cuda = True

        def is_contiguous(self):
            return strided.is_contiguous()

        def data_ptr(self):
            return 4096

    with pytest.raises(ValueError, match="contiguous"):
        D.dflash_ctx_project_noalloc(dims, [FakeCuda()], 8, None, None, None)
    # raw addresses pass through unchanged
    arr = D._ptr_array([4096, 8192])
    assert [arr[0], arr[1]] == [4096, 8192]
