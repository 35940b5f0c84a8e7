"""ctypes binding of libdflash.so: the C ABI of include/dflash.h, call for call.

Each function marshals torch tensors (device memory) into the C call with the
same name and raises ``DFlashError`` on a non-OK status. Nothing here
computes: every step runs in the library's CUDA kernels. There is no CPU
fallback; if libdflash.so is missing the import fails.

Streams: every call runs on ``torch.cuda.current_stream()`` unless a
``stream`` (a torch.cuda.Stream or a raw handle) is given.
"""

from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_double, c_float, c_int, c_size_t, c_uint, c_void_p

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdflash.so")

DFLASH_F32, DFLASH_BF16 = 0, 1
DEV_CAPACITY, DEV_ROPE, DEV_CROP, DEV_ROWS, DEV_TIMEOUT = 1, 2, 4, 8, 16
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_DEVICE = range(6)
KERNEL_NAMES = {1: "gemm", 2: "rmsnorm", 3: "head_epilogue", 4: "attention", 5: "combine",
                6: "lens", 7: "crop", 8: "rope_table", 9: "schedule", 10: "accept"}
KERNEL_IDS = {v: k for k, v in KERNEL_NAMES.items()}


class DFlashError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


class dflash_dims(ctypes.Structure):
    _fields_ = [("d", c_int), ("n_h", c_int), ("n_kv", c_int), ("d_h", c_int),
                ("k_layers", c_int), ("block_size", c_int), ("eps", c_float), ("dtype", c_int)]


class dflash_kv_cache(ctypes.Structure):
    _fields_ = [("k", c_void_p), ("v", c_void_p), ("lens", c_void_p), ("n_layers", c_int),
                ("batch", c_int), ("capacity", c_int), ("block_table", c_void_p),
                ("page_size", c_int), ("n_pages", c_int), ("kv_dtype", c_int),
                ("kv_scales", c_void_p)]


DFLASH_FP8_E4M3 = 2


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libdflash.so is not built ({LIB_PATH}); run "
                          "speculative_decoding_draft_dflash_gb300.build.build() first")
    lib = ctypes.CDLL(LIB_PATH)
    P = c_void_p
    sig = {
        "dflash_rope_table_build": (c_int, [c_double, c_int, c_int, P, P]),
        "dflash_workspace_bytes": (c_size_t, [P, c_int, c_int, c_int]),
        "dflash_ctx_project": (c_int, [P, P, c_int, P, P, P, P, c_size_t, P]),
        "dflash_ctx_project_noalloc": (c_int, [P, P, c_int, P, P, P, P]),
        "dflash_kv_inject": (c_int, [P, P, c_int, P, P, c_int, P, P, P, P, c_int, P, c_size_t, P]),
        "dflash_block_attn": (c_int, [P, P, c_int, P, P, P, P, P, P, P, c_int, c_int, c_float, P, P,
                                      c_size_t, P]),
        "dflash_draft_layer": (c_int, [P, P, c_int, P, P, c_int, P, P, P, P, P, P, P, c_int, c_int,
                                       c_float, P, P, c_size_t, P]),
        "dflash_cache_crop": (c_int, [P, P, P]),
        "dflash_layer_out_workspace_bytes": (c_size_t, [P, c_int, c_int]),
        "dflash_layer_out": (c_int, [P, c_int, P, P, P, P, c_int, P, P, P, P, P, c_size_t, P]),
        "dflash_rms_norm": (c_int, [P, c_int, P, P, P, P]),
        "dflash_accept": (c_int, [P, P, c_int, c_int, P, P, P, P, P, P]),
        "dflash_status_get": (c_int, [POINTER(c_uint), P]),
        "dflash_status_string": (ctypes.c_char_p, [c_int]),
        "dflash_trace_start": (c_int, [c_uint, c_int]),
        "dflash_trace_stop": (c_int, [P, P, c_int, P]),
        "dflash_launch_count": (ctypes.c_ulonglong, []),
        "dflash_test_wait_limit": (None, [ctypes.c_ulonglong]),
        "dflash_test_attn_worklist": (c_int, [P, P, c_int, P, c_int, c_int, P, c_size_t, P,
                                              c_size_t, P, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


_lib = _load()


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------

def _stream(stream):
    if stream is None:
        return c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return c_void_p(stream.cuda_stream)
    return c_void_p(int(stream))


def _ptr(t, what="tensor", dtype=None, numel=None):
    """Device address of a tensor argument after the checks the C ABI cannot make.

    The library sees bare pointers and sizes, so it cannot tell a bf16 buffer from an
    f32 one or a short buffer from a full one; a mismatch would make a kernel read or
    write past the tensor. So a torch tensor must be a contiguous CUDA tensor, of
    element type ``dtype`` when one is given, holding at least ``numel`` elements when
    that is given. ``None`` stays NULL (the library refuses it where a pointer is
    required) and an ``int`` is taken as a raw device address, unchecked: a caller who
    passes addresses vouches for their sizes."""
    if t is None:
        return None
    if isinstance(t, int):
        return c_void_p(t)
    if not t.is_cuda:
        raise ValueError(f"{what}: expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what}: expected a contiguous tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{what}: element type {t.dtype}, the call needs {dtype}")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{what}: {t.numel()} elements, the call needs at least {numel}")
    return c_void_p(t.data_ptr())


def _ptr_array(ts, what="hidden", dtype=None, numel=None):
    """C array of device pointers: tensors (checked like _ptr) or raw addresses (ints)."""
    vals = [(_ptr(t, f"{what}[{i}]", dtype, numel).value or 0) if hasattr(t, "data_ptr")
            else int(t) for i, t in enumerate(ts)]
    return (c_void_p * max(1, len(vals)))(*vals)


def _ws(workspace):
    """(pointer, size in bytes) of a workspace tensor (any element type)."""
    if workspace is None:
        return None, 0
    return _ptr(workspace, "workspace"), workspace.numel() * workspace.element_size()


def _et(dims):
    """torch element type of the activations, weights and gammas of a call."""
    return torch_dtype(dims.dtype)


def _desc(dims, cache):
    """C descriptor of a cache; a KVCache must match the call's dims and element type."""
    if not isinstance(cache, KVCache):
        return cache
    if cache.n_kv != dims.n_kv or cache.d_h != dims.d_h:
        raise ValueError(f"cache: n_kv {cache.n_kv}, d_h {cache.d_h}; the dims give "
                         f"n_kv {dims.n_kv}, d_h {dims.d_h}")
    want = torch.uint8 if cache.fp8 else _et(dims)
    if cache.k.dtype != want or cache.v.dtype != want:
        raise ValueError(f"cache: element type {cache.k.dtype}, the dims need {want}")
    return cache.desc


def _rope(dims, rope_table, table_len):
    """The RoPE table: float32 [table_len][d_h / 2][2]."""
    return _ptr(rope_table, "rope_table", torch.float32, max(0, int(table_len)) * dims.d_h)


def _check(st, where):
    if st != OK:
        raise DFlashError(st, where)


def dtype_code(dtype):
    if dtype in (torch.float32, "f32", DFLASH_F32):
        return DFLASH_F32
    if dtype in (torch.bfloat16, "bf16", DFLASH_BF16):
        return DFLASH_BF16
    raise ValueError(f"unsupported dtype {dtype}")


def torch_dtype(code):
    return torch.float32 if code == DFLASH_F32 else torch.bfloat16


def make_dims(d, n_h, n_kv, d_h, k_layers, block_size, eps=1e-6, dtype=DFLASH_BF16):
    return dflash_dims(d, n_h, n_kv, d_h, k_layers, block_size, eps, dtype_code(dtype))


class KVCache:
    """Device buffers of a draft KV cache (allocated by torch) and their C descriptor.

    Contiguous: k, v [n_layers][batch][n_kv][capacity][d_h].
    Paged (page_table given, or paged=True): k, v [n_layers][n_pages][n_kv][page_size][d_h]
    and block_table int32 [batch][capacity / page_size]; with paged=True the pages of
    the sequences are a seeded permutation of the pool (so no page is where a contiguous
    layout would put it). lens: int32 [n_layers][batch] in both layouts.
    kv="fp8": k, v hold E4M3 codes (uint8 tensors) of x / scale with kv_scales
    [n_layers][2] = (k_scale, v_scale) per layer (default 1); rows() reads them back as
    scale * value.
    """

    PAGE = 128

    def __init__(self, n_layers, batch, n_kv, capacity, d_h, dtype, device="cuda", paged=False,
                 page_table=None, n_pages=None, seed=0, kv="bf16", kv_scales=None):
        self.fp8 = kv == "fp8"
        td = torch.uint8 if self.fp8 else torch_dtype(dtype_code(dtype))
        self.scales = np.ones((n_layers, 2)) if kv_scales is None else np.asarray(kv_scales, float)
        assert self.scales.shape == (n_layers, 2)
        self.n_layers, self.batch, self.capacity, self.n_kv, self.d_h = (
            n_layers, batch, capacity, n_kv, d_h)
        self.lens = torch.zeros((n_layers, batch), dtype=torch.int32, device=device)
        self.paged = paged or page_table is not None
        if self.paged:
            P = self.PAGE
            assert capacity % P == 0
            pps = capacity // P
            if page_table is None:
                n_pages = n_pages or batch * pps
                g = torch.Generator().manual_seed(seed)
                perm = torch.randperm(n_pages, generator=g)[:batch * pps]
                page_table = perm.view(batch, pps).to(torch.int32)
            self.block_table = page_table.to(device=device, dtype=torch.int32).contiguous()
            self.n_pages = n_pages or int(self.block_table.max().item()) + 1
            shape = (n_layers, self.n_pages, n_kv, P, d_h)
            self.k = torch.zeros(shape, dtype=td, device=device)
            self.v = torch.zeros(shape, dtype=td, device=device)
            self.desc = dflash_kv_cache(self.k.data_ptr(), self.v.data_ptr(), self.lens.data_ptr(),
                                        n_layers, batch, capacity, self.block_table.data_ptr(),
                                        P, self.n_pages)
        else:
            shape = (n_layers, batch, n_kv, capacity, d_h)
            self.k = torch.zeros(shape, dtype=td, device=device)
            self.v = torch.zeros(shape, dtype=td, device=device)
            self.desc = dflash_kv_cache(self.k.data_ptr(), self.v.data_ptr(), self.lens.data_ptr(),
                                        n_layers, batch, capacity)
        if self.fp8:
            # host array the descriptor points to; kept alive with the cache
            self._scales_c = (c_float * (2 * n_layers))(*self.scales.ravel().tolist())
            self.desc.kv_dtype = DFLASH_FP8_E4M3
            self.desc.kv_scales = ctypes.addressof(self._scales_c)

    def _index(self, b, lo, hi):
        """(pages, rows) of logical slots lo .. hi-1 of sequence b (paged layout)."""
        s = torch.arange(lo, hi, device=self.block_table.device)
        return self.block_table[b, s // self.PAGE].long(), s % self.PAGE

    def rows(self, which, layer, b, lo, hi, codes=False):
        """Logical rows lo .. hi-1 of sequence b as [n_kv][hi - lo][d_h] (a copy when paged).
        fp8: float32 values, scale * value(code), or value(code) with codes=True."""
        t = self.k if which == "k" else self.v
        if not self.paged:
            x = t[layer, b, :, lo:hi]
        else:
            pages, r = self._index(b, lo, hi)
            x = t[layer, pages, :, r].permute(1, 0, 2)
        if not self.fp8:
            return x
        x = x.contiguous().view(torch.float8_e4m3fn).to(torch.float32)
        return x if codes else x * float(self.scales[layer, 0 if which == "k" else 1])

    def set_rows(self, layer, b, K, V):
        """Writes K, V [n_kv][n][d_h] to logical slots 0 .. n-1 of sequence b. The rows are
        given in stored form: the cache's element type, E4M3 codes (uint8) for fp8."""
        n = K.shape[1]
        if K.dtype != self.k.dtype or V.dtype != self.v.dtype:
            raise ValueError(f"set_rows: rows of type {K.dtype}, the cache holds {self.k.dtype}")
        if not self.paged:
            self.k[layer, b, :, :n] = K
            self.v[layer, b, :, :n] = V
            return
        pages, r = self._index(b, 0, n)
        self.k[layer, pages, :, r] = K.permute(1, 0, 2).to(self.k.dtype)
        self.v[layer, pages, :, r] = V.permute(1, 0, 2).to(self.v.dtype)


# ---------------------------------------------------------------------------
# the C calls
# ---------------------------------------------------------------------------

def status_string(st):
    return _lib.dflash_status_string(int(st)).decode()


def dflash_rope_table_build(theta, d_h, max_pos, table, stream=None):
    _check(_lib.dflash_rope_table_build(float(theta), int(d_h), int(max_pos),
                                        _ptr(table, "table", torch.float32,
                                             max(0, int(max_pos)) * int(d_h)),
                                        _stream(stream)), "dflash_rope_table_build")


def dflash_workspace_bytes(dims, batch, capacity, max_rows):
    return int(_lib.dflash_workspace_bytes(ctypes.byref(dims), int(batch), int(capacity),
                                           int(max_rows)))


def _ctx_args(dims, hidden, M, W_fc, gamma_h, C_out):
    et, d, M = _et(dims), dims.d, max(0, int(M))
    ptrs = _ptr_array(hidden, "hidden", et, M * d)
    if len(hidden) < dims.k_layers:
        raise ValueError(f"hidden: {len(hidden)} pointers, the dims give k_layers {dims.k_layers}")
    return (ptrs, _ptr(W_fc, "W_fc", et, d * dims.k_layers * d),
            _ptr(gamma_h, "gamma_h", et, d), _ptr(C_out, "C_out", et, M * d))


def dflash_ctx_project(dims, hidden, M, W_fc, gamma_h, C_out, workspace, stream=None):
    ptrs, W, g, C = _ctx_args(dims, hidden, M, W_fc, gamma_h, C_out)
    _check(_lib.dflash_ctx_project(ctypes.byref(dims), ptrs, int(M), W, g, C, *_ws(workspace),
                                   _stream(stream)), "dflash_ctx_project")


def dflash_ctx_project_noalloc(dims, hidden, M, W_fc, gamma_h, C_out, stream=None):
    """dflash_ctx_project with the library's fixed scratch array instead of a workspace."""
    ptrs, W, g, C = _ctx_args(dims, hidden, M, W_fc, gamma_h, C_out)
    _check(_lib.dflash_ctx_project_noalloc(ctypes.byref(dims), ptrs, int(M), W, g, C,
                                           _stream(stream)), "dflash_ctx_project_noalloc")


def _batch(cache):
    return int(cache.batch)


def _kv_args(dims, cache, C, cu_rows, M, W_K, W_V, gamma_k):
    et, M = _et(dims), max(0, int(M))
    nkv = dims.n_kv * dims.d_h
    return (_ptr(C, "C", et, M * dims.d), _ptr(cu_rows, "cu_rows", torch.int32, _batch(cache) + 1),
            _ptr(W_K, "W_K", et, nkv * dims.d), _ptr(W_V, "W_V", et, nkv * dims.d),
            _ptr(gamma_k, "gamma_k", et, dims.d_h))


def _block_args(dims, cache, H, W_Q, gamma_q, out):
    et, rows = _et(dims), _batch(cache) * dims.block_size
    return (_ptr(H, "H", et, rows * dims.d), _ptr(W_Q, "W_Q", et, dims.n_h * dims.d_h * dims.d),
            _ptr(gamma_q, "gamma_q", et, dims.d_h), _ptr(out, "out", et, rows * dims.n_h * dims.d_h))


def dflash_kv_inject(dims, cache, layer, C, cu_rows, M, W_K, W_V, gamma_k, rope_table, table_len,
                     workspace, stream=None):
    desc = _desc(dims, cache)
    c, cu, wk, wv, gk = _kv_args(dims, desc, C, cu_rows, M, W_K, W_V, gamma_k)
    _check(_lib.dflash_kv_inject(ctypes.byref(dims), ctypes.byref(desc), int(layer), c, cu, int(M),
                                 wk, wv, gk, _rope(dims, rope_table, table_len), int(table_len),
                                 *_ws(workspace), _stream(stream)), "dflash_kv_inject")


def dflash_block_attn(dims, cache, layer, H, W_Q, W_K, W_V, gamma_q, gamma_k, rope_table,
                      table_len, sliding_window, scaling, out, workspace, stream=None):
    desc = _desc(dims, cache)
    h, wq, gq, o = _block_args(dims, desc, H, W_Q, gamma_q, out)
    et, nkv = _et(dims), dims.n_kv * dims.d_h
    _check(_lib.dflash_block_attn(ctypes.byref(dims), ctypes.byref(desc), int(layer), h, wq,
                                  _ptr(W_K, "W_K", et, nkv * dims.d),
                                  _ptr(W_V, "W_V", et, nkv * dims.d), gq,
                                  _ptr(gamma_k, "gamma_k", et, dims.d_h),
                                  _rope(dims, rope_table, table_len), int(table_len),
                                  int(sliding_window), float(scaling), o, *_ws(workspace),
                                  _stream(stream)), "dflash_block_attn")


def dflash_draft_layer(dims, cache, layer, C, cu_rows, M, H, W_Q, W_K, W_V, gamma_q, gamma_k,
                       rope_table, table_len, sliding_window, scaling, out, workspace, stream=None):
    """dflash_kv_inject of C's rows followed by dflash_block_attn of H, as one call."""
    desc = _desc(dims, cache)
    c, cu, wk, wv, gk = _kv_args(dims, desc, C, cu_rows, M, W_K, W_V, gamma_k)
    h, wq, gq, o = _block_args(dims, desc, H, W_Q, gamma_q, out)
    _check(_lib.dflash_draft_layer(ctypes.byref(dims), ctypes.byref(desc), int(layer), c, cu,
                                   int(M), h, wq, wk, wv, gq, gk, _rope(dims, rope_table, table_len),
                                   int(table_len), int(sliding_window), float(scaling), o,
                                   *_ws(workspace), _stream(stream)), "dflash_draft_layer")


def dflash_cache_crop(cache, new_lens, stream=None):
    desc = cache.desc if isinstance(cache, KVCache) else cache
    _check(_lib.dflash_cache_crop(ctypes.byref(desc),
                                  _ptr(new_lens, "new_lens", torch.int32, int(desc.batch)),
                                  _stream(stream)), "dflash_cache_crop")


def dflash_accept(block_ids, posterior, ctx_len, accept_len, next_cu_rows, ctx_next, next_anchor,
                  stream=None):
    """Acceptance bookkeeping of a verified round; block_ids / posterior are int32 [batch][bs]."""
    batch, bs = (int(block_ids.shape[0]), int(block_ids.shape[1])) if block_ids.dim() == 2 else (0, 1)
    i32 = torch.int32
    _check(_lib.dflash_accept(_ptr(block_ids, "block_ids", i32, batch * bs),
                              _ptr(posterior, "posterior", i32, batch * bs), batch, bs,
                              _ptr(ctx_len, "ctx_len", i32, batch),
                              _ptr(accept_len, "accept_len", i32, batch),
                              _ptr(next_cu_rows, "next_cu_rows", i32, batch + 1),
                              _ptr(ctx_next, "ctx_next", i32, batch),
                              _ptr(next_anchor, "next_anchor", i32, batch), _stream(stream)),
           "dflash_accept")


def dflash_layer_out_workspace_bytes(dims, M, d_ff):
    return int(_lib.dflash_layer_out_workspace_bytes(ctypes.byref(dims), int(M), int(d_ff)))


def dflash_layer_out(dims, M, attn_out, x, W_O, gamma_post, d_ff, W_gate, W_up, W_down, x_out,
                     workspace, stream=None):
    """x_out = x1 + MLP(RMSNorm_post(x1)), x1 = x + attn_out W_O^T (rows of the blocks)."""
    et, d, M, F_ = _et(dims), dims.d, max(0, int(M)), max(0, int(d_ff))
    hd = dims.n_h * dims.d_h
    _check(_lib.dflash_layer_out(ctypes.byref(dims), int(M), _ptr(attn_out, "attn_out", et, M * hd),
                                 _ptr(x, "x", et, M * d), _ptr(W_O, "W_O", et, d * hd),
                                 _ptr(gamma_post, "gamma_post", et, d), int(d_ff),
                                 _ptr(W_gate, "W_gate", et, F_ * d), _ptr(W_up, "W_up", et, F_ * d),
                                 _ptr(W_down, "W_down", et, d * F_), _ptr(x_out, "x_out", et, M * d),
                                 *_ws(workspace), _stream(stream)), "dflash_layer_out")


def dflash_rms_norm(dims, M, x, gamma, out, stream=None):
    et, n = _et(dims), max(0, int(M)) * dims.d
    _check(_lib.dflash_rms_norm(ctypes.byref(dims), int(M), _ptr(x, "x", et, n),
                                _ptr(gamma, "gamma", et, dims.d), _ptr(out, "out", et, n),
                                _stream(stream)), "dflash_rms_norm")


def dflash_status_get(stream=None):
    """Synchronises the stream; returns the device status bits (0 = clean) and clears them."""
    v = c_uint(0)
    st = _lib.dflash_status_get(ctypes.byref(v), _stream(stream))
    if st not in (OK, ERR_DEVICE):
        raise DFlashError(st, "dflash_status_get")
    return int(v.value)


def dflash_trace_start(kinds, max_launches):
    """Records CUDA events around launches of the given kernel kinds (names or ids)."""
    mask = 0
    for k in kinds:
        mask |= 1 << (KERNEL_IDS[k] if isinstance(k, str) else int(k))
    _check(_lib.dflash_trace_start(mask, int(max_launches)), "dflash_trace_start")


def dflash_trace_stop(capacity=1 << 16):
    """Returns [(kernel name, milliseconds)] of the launches recorded since dflash_trace_start."""
    kinds = (c_int * capacity)()
    ms = (c_float * capacity)()
    n = c_int(0)
    _check(_lib.dflash_trace_stop(kinds, ms, capacity, ctypes.byref(n)), "dflash_trace_stop")
    return [(KERNEL_NAMES.get(kinds[i], str(kinds[i])), float(ms[i]))
            for i in range(min(n.value, capacity))]


def dflash_launch_count():
    return int(_lib.dflash_launch_count())


def dflash_test_wait_limit(ns):
    """Test aid: limit (ns) of the kernels' pipeline waits for later launches; 0 = 2 s."""
    _lib.dflash_test_wait_limit(int(ns))


def dflash_test_attn_worklist(dims, cache, layer, cu_rows, M, sliding_window, workspace,
                              stream=None):
    """Test aid: the tensor-core attention's work list for the cache's current lengths (plus
    the rows an inject of cu_rows / M would append), as host arrays: n_ctas, max_splits,
    item_cost, first [n_ctas + 1], items [n_ctas + n_items, 4], splits [pairs], merge_list."""
    desc = _desc(dims, cache)
    cu = _ptr(cu_rows, "cu_rows", torch.int32, _batch(desc) + 1) if M > 0 else None
    need = ctypes.c_size_t(0)
    args = (ctypes.byref(dims), ctypes.byref(desc), int(layer), cu, int(M), int(sliding_window),
            *_ws(workspace))
    st = _lib.dflash_test_attn_worklist(*args, None, 0, ctypes.byref(need), _stream(stream))
    if st != ERR_INVALID_ARG:
        _check(st, "dflash_test_attn_worklist")
    out = np.zeros(need.value, dtype=np.int32)
    _check(_lib.dflash_test_attn_worklist(*args, out.ctypes.data_as(ctypes.c_void_p), out.size,
                                          ctypes.byref(need), _stream(stream)),
           "dflash_test_attn_worklist")
    n_ctas, max_splits, item_cost, n_items, n_merge = (int(v) for v in out[:5])
    o = 5
    first = out[o:o + n_ctas + 1]
    o += n_ctas + 1
    items = out[o:o + 4 * (n_ctas + n_items)].reshape(-1, 4)
    o += 4 * (n_ctas + n_items)
    pairs = _batch(desc) * dims.n_kv
    splits = out[o:o + pairs]
    o += pairs
    return {"n_ctas": n_ctas, "max_splits": max_splits, "item_cost": item_cost, "first": first,
            "items": items, "splits": splits, "merge_list": out[o:o + n_merge]}
