"""The C ABI library: builds, loads without a GPU, exports every declared symbol, checks host arguments."""
import ctypes
import glob
import os
import re

import numpy as np
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


@pytest.mark.parametrize("batch", [1, 2, 4, 8])
def test_workspace_bytes_never_shrink_with_more_rows(D, batch):
    """A workspace sized for max_rows serves every call with fewer context rows: the need
    (including the few-sequence layer launch's context partials, which grow with M until
    the launch's row tile is full) never decreases as max_rows grows."""
    dims = _dims(D)
    need = [D.dflash_workspace_bytes(dims, batch, 1088, m) for m in range(1, 400, 3)]
    assert all(b >= a for a, b in zip(need, need[1:]))
    assert need[0] >= D.dflash_workspace_bytes(dims, batch, 1088, 0)


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


class _FakeDev:
    """Stands in for a contiguous CUDA tensor of a given element type and shape (CPU only):
    the binding's checks read these attributes; nothing reaches the library when one fails."""
    is_cuda = True

    def __init__(self, shape, dtype):
        import torch
        self.shape, self.dtype = tuple(shape), dtype
        self._n = int(np.prod(shape)) if len(shape) else 1
        self._es = torch.empty((), dtype=dtype).element_size()

    def is_contiguous(self):
        return True

    def numel(self):
        return self._n

    def dim(self):
        return len(self.shape)

    def element_size(self):
        return self._es

    def data_ptr(self):
        return 1 << 20


def _serve_args(D, dt):
    """Well-formed fake arguments of the serving shape (d 4096, 32 / 8 heads of 128, k 5,
    bs 16, batch 4) in element type dt, and the cache descriptor."""
    import torch
    d, nh, nkv, dh, k, bs, B, M = 4096, 32, 8, 128, 5, 16, 4, 20
    a = dict(hidden=[_FakeDev((M, d), dt) for _ in range(k)], W_fc=_FakeDev((d, k * d), dt),
             g_h=_FakeDev((d,), dt), C=_FakeDev((M, d), dt), cu=_FakeDev((B + 1,), torch.int32),
             W_Q=_FakeDev((nh * dh, d), dt), W_K=_FakeDev((nkv * dh, d), dt),
             W_V=_FakeDev((nkv * dh, d), dt), g_q=_FakeDev((dh,), dt), g_k=_FakeDev((dh,), dt),
             rope=_FakeDev((64, dh // 2, 2), torch.float32), H=_FakeDev((B, bs, d), dt),
             out=_FakeDev((B, bs, nh * dh), dt), ws=_FakeDev((1 << 20,), torch.uint8), M=M)
    cache = D.dflash_kv_cache(4096, 8192, 12288, 1, B, 64)
    return a, cache


@pytest.mark.parametrize("field,bad", [
    ("hidden", "f32"), ("hidden", "short"), ("W_fc", "f32"), ("W_fc", "short"), ("g_h", "short"),
    ("C", "f32"), ("C", "short")])
def test_binding_refuses_ctx_project_mismatch(D, field, bad):
    """ctx_project: every tensor must be of dims.dtype and hold the elements the dims and M
    imply; an f32 or short tensor where bf16 [M][d] is needed is refused before the call."""
    import torch
    a, _ = _serve_args(D, torch.bfloat16)
    dims = _dims(D)

    def spoil(t):
        if bad == "f32":
            return _FakeDev(t.shape, torch.float32)
        return _FakeDev((t.numel() - 1,), t.dtype)

    if field == "hidden":
        a["hidden"][2] = spoil(a["hidden"][2])
    else:
        a[field] = spoil(a[field])
    for fn in (lambda: D.dflash_ctx_project(dims, a["hidden"], a["M"], a["W_fc"], a["g_h"], a["C"],
                                            a["ws"]),
               lambda: D.dflash_ctx_project_noalloc(dims, a["hidden"], a["M"], a["W_fc"], a["g_h"],
                                                    a["C"])):
        with pytest.raises(ValueError, match="element type|elements"):
            fn()


@pytest.mark.parametrize("field,bad", [
    ("C", "f32"), ("cu", "short"), ("cu", "i64"), ("W_K", "short"), ("W_V", "f32"),
    ("g_k", "short"), ("rope", "bf16"), ("rope", "short"), ("H", "short"), ("H", "f32"),
    ("W_Q", "short"), ("g_q", "f32"), ("out", "short"), ("out", "f32")])
def test_binding_refuses_layer_call_mismatch(D, field, bad):
    """kv_inject, block_attn and draft_layer refuse a tensor whose element type or size does
    not match the dims, the cache's batch, M or table_len, before the library is called."""
    import torch
    a, cache = _serve_args(D, torch.bfloat16)
    dims = _dims(D)
    t = a[field]
    a[field] = {"f32": lambda: _FakeDev(t.shape, torch.float32),
                "bf16": lambda: _FakeDev(t.shape, torch.bfloat16),
                "i64": lambda: _FakeDev(t.shape, torch.int64),
                "short": lambda: _FakeDev((t.numel() - 1,), t.dtype)}[bad]()
    calls = [lambda: D.dflash_draft_layer(dims, cache, 0, a["C"], a["cu"], a["M"], a["H"], a["W_Q"],
                                          a["W_K"], a["W_V"], a["g_q"], a["g_k"], a["rope"], 64, 0,
                                          0.0, a["out"], a["ws"])]
    if field in ("C", "cu", "W_K", "W_V", "g_k", "rope"):
        calls.append(lambda: D.dflash_kv_inject(dims, cache, 0, a["C"], a["cu"], a["M"], a["W_K"],
                                                a["W_V"], a["g_k"], a["rope"], 64, a["ws"]))
    if field not in ("C", "cu"):
        calls.append(lambda: D.dflash_block_attn(dims, cache, 0, a["H"], a["W_Q"], a["W_K"],
                                                 a["W_V"], a["g_q"], a["g_k"], a["rope"], 64, 0,
                                                 0.0, a["out"], a["ws"]))
    for fn in calls:
        with pytest.raises(ValueError, match="element type|elements"):
            fn()


def test_binding_refuses_small_calls_mismatch(D):
    """crop, accept, rms_norm, layer_out and the RoPE table builder check their tensors too."""
    import torch
    dims = _dims(D)
    cache = D.dflash_kv_cache(4096, 8192, 12288, 1, 4, 64)
    with pytest.raises(ValueError, match="elements"):
        D.dflash_cache_crop(cache, _FakeDev((3,), torch.int32))
    with pytest.raises(ValueError, match="element type"):
        D.dflash_cache_crop(cache, _FakeDev((4,), torch.int64))
    i32 = lambda *s: _FakeDev(s, torch.int32)  # noqa: E731
    ids = i32(4, 16)
    with pytest.raises(ValueError, match="elements"):
        D.dflash_accept(ids, i32(4, 15), i32(4), i32(4), i32(5), i32(4), i32(4))
    with pytest.raises(ValueError, match="elements"):
        D.dflash_accept(ids, i32(4, 16), i32(4), i32(4), i32(4), i32(4), i32(4))
    bf = lambda *s: _FakeDev(s, torch.bfloat16)  # noqa: E731
    with pytest.raises(ValueError, match="element type"):
        D.dflash_rms_norm(dims, 8, _FakeDev((8, 4096), torch.float32), bf(4096), bf(8, 4096))
    with pytest.raises(ValueError, match="elements"):
        D.dflash_rms_norm(dims, 8, bf(8, 4096), bf(4095), bf(8, 4096))
    args = [bf(8, 4096), bf(8, 4096), bf(4096, 4096), bf(4096), 12288, bf(12288, 4096),
            bf(12288, 4096), bf(4096, 12288), bf(8, 4096), _FakeDev((64,), torch.uint8)]
    for i in (0, 1, 2, 3, 5, 6, 7, 8):
        bad = list(args)
        bad[i] = _FakeDev((bad[i].numel() - 1,), torch.bfloat16)
        with pytest.raises(ValueError, match="elements"):
            D.dflash_layer_out(dims, 8, *bad)
    with pytest.raises(ValueError, match="element type"):
        D.dflash_rope_table_build(1e6, 128, 64, _FakeDev((64, 64, 2), torch.bfloat16))
    with pytest.raises(ValueError, match="elements"):
        D.dflash_rope_table_build(1e6, 128, 64, _FakeDev((63, 64, 2), torch.float32))


def test_binding_refuses_cache_of_other_dims(D):
    """A KVCache whose heads, head size or element type differ from the dims is refused."""
    import torch
    a, _ = _serve_args(D, torch.bfloat16)
    dims = _dims(D)

    class FakeCache(D.KVCache):
        def __init__(self, n_kv, d_h, dt, fp8=False):     # no device buffers are made
            self.n_kv, self.d_h, self.fp8 = n_kv, d_h, fp8
            self.k = self.v = _FakeDev((1,), dt)
            self.desc = D.dflash_kv_cache(4096, 8192, 12288, 1, 4, 64)

    for c in (FakeCache(4, 128, torch.bfloat16), FakeCache(8, 64, torch.bfloat16),
              FakeCache(8, 128, torch.float32), FakeCache(8, 128, torch.bfloat16, fp8=True)):
        with pytest.raises(ValueError, match="cache"):
            D.dflash_kv_inject(dims, c, 0, a["C"], a["cu"], a["M"], a["W_K"], a["W_V"], a["g_k"],
                               a["rope"], 64, a["ws"])
