"""Seeded synthetic workloads for the DFlash draft-attention step.

This module draws random inputs and nothing else: it holds none of the
method's arithmetic, so both the library's callers (tests, benchmark) and the
float64 oracle checks can take their inputs from it.

Every array comes from its own NumPy PCG64 stream keyed by
(seed, kind, index...), so any subset (one layer, one sequence) can be drawn
again on its own and gives the same values. Values for bf16 workloads are
rounded to bf16 here, once, so that the device and the oracle see the same
numbers.

Distributions (the walkthrough's example settings, used for every workload):
hidden states and block embeddings N(0, 1); weights N(0, 0.02^2); RMSNorm
gamma = 1 (or 1 + N(0, 0.1^2) when ``random_gamma``); eps = 1e-6;
rope_theta = 1e6. A pre-filled cache holds K rows N(0, 1) (the statistics of
normalised, rotated keys) and V rows N(0, (0.02 sqrt(d))^2) (those of C W_V).
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Tuple

import numpy as np

# stream tags (one per kind of array)
_T_WFC, _T_WQ, _T_WK, _T_WV, _T_GAMMA = 1, 2, 3, 4, 5
_T_HIDDEN, _T_BLOCK, _T_CACHE_K, _T_CACHE_V, _T_PREFILL_LEN, _T_ACCEPT = 6, 7, 8, 9, 10, 11
_T_WO, _T_WGATE, _T_WUP, _T_WDOWN, _T_RESID, _T_ATTN = 12, 13, 14, 15, 16, 17


@dataclass(frozen=True)
class Workload:
    """Shape and schedule of one synthetic workload.

    ``prefill_lo/hi``: cached rows per sequence before round 1, drawn uniformly
    in [lo, hi] (equal bounds = fixed length); they are synthetic cache rows
    unless ``prefill_inject`` is set, in which case they are produced by a
    context projection + inject of that many hidden-state rows.
    ``new_ctx``: context rows injected per sequence in round 1.
    ``rounds``: 1 or 2. In a two-round schedule the cache is cropped to the
    context-only length after round 1, round 2 injects a_i ~ U{1..bs} rows
    (acceptance + 1), and the cache is cropped again after round 2.
    """

    name: str
    dtype: str
    d: int
    n_h: int
    n_kv: int
    d_h: int
    k: int
    bs: int
    batch: int
    n_layers: int
    windows: Tuple[int, ...]
    prefill_lo: int
    prefill_hi: int
    new_ctx: int
    rounds: int
    prefill_inject: bool = False
    eps: float = 1e-6
    theta: float = 1e6
    seed: int = 0
    random_gamma: bool = False
    description: str = ""
    d_ff: int = 0          # MLP width of the rest of the decoder layer; 0 = 3 * d
    kv: str = "bf16"       # cache element type: the storage type, or "fp8" (E4M3 codes)

    @property
    def ffn(self):
        return self.d_ff or 3 * self.d

    @property
    def G(self):
        return self.n_h // self.n_kv

    @property
    def capacity(self):
        """Cache rows per sequence: the longest sequence's need, rounded up to 64."""
        need = self.prefill_hi + self.new_ctx + self.bs + (self.bs + self.bs if self.rounds > 1 else 0)
        return ((need + 63) // 64) * 64

    @property
    def table_len(self):
        return self.capacity

    def replace(self, **kw):
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


WORKLOADS = {
    # The walkthrough's example: d=512, 8 heads of 64, k=3 target layers, the
    # 3-token prompt at positions 0-2 and a block of 4 at positions 3-6.
    "walkthrough_f32": Workload(
        name="walkthrough_f32", dtype="f32", d=512, n_h=8, n_kv=8, d_h=64, k=3, bs=4,
        batch=1, n_layers=1, windows=(0,), prefill_lo=0, prefill_hi=0, new_ctx=3, rounds=2,
        description="walkthrough-sized single layer, fp32, batch 1, L_c=3, block 4"),
    # One Qwen3-8B-shaped draft layer, batch 1: 1024 context rows prefilled by
    # the step's own projection + inject, then 16 new context rows and a block of 16.
    "qwen3_8b_b1": Workload(
        name="qwen3_8b_b1", dtype="bf16", d=4096, n_h=32, n_kv=8, d_h=128, k=5, bs=16,
        batch=1, n_layers=1, windows=(0,), prefill_lo=1024, prefill_hi=1024, new_ctx=16,
        rounds=1, prefill_inject=True,
        description="Qwen3-8B-shaped draft layer, bf16, batch 1, 1024 cached + 16 new, block 16"),
    # Batched serving step: 32 sequences, ragged cached context in [256, 4096], two layers.
    "serve_b32": Workload(
        name="serve_b32", dtype="bf16", d=4096, n_h=32, n_kv=8, d_h=128, k=5, bs=16,
        batch=32, n_layers=2, windows=(0, 0), prefill_lo=256, prefill_hi=4096, new_ctx=16,
        rounds=2,
        description="batch 32, ragged context U[256,4096], block 16, 2 draft layers, 2 rounds with crop"),
    # Long-context step: 4 sequences of 32768 cached rows.
    "long_ctx_b4": Workload(
        name="long_ctx_b4", dtype="bf16", d=4096, n_h=32, n_kv=8, d_h=128, k=5, bs=16,
        batch=4, n_layers=1, windows=(0,), prefill_lo=32768, prefill_hi=32768, new_ctx=16,
        rounds=1,
        description="batch 4, 32768 cached rows each, inject 16, block 16, split-KV"),
    # Hybrid sliding-window draft: 64 sequences, 4 layers alternating full / window 2048.
    "hybrid_swa_b64": Workload(
        name="hybrid_swa_b64", dtype="bf16", d=4096, n_h=32, n_kv=8, d_h=128, k=5, bs=16,
        batch=64, n_layers=4, windows=(0, 2048, 0, 2048), prefill_lo=1024, prefill_hi=8192,
        new_ctx=16, rounds=2,
        description="batch 64, context U[1024,8192], 4 layers full/SWA-2048 alternating, 2 rounds"),
}


def _rng(w: Workload, *key):
    return np.random.default_rng([int(w.seed)] + [int(x) for x in key])


def to_storage(w: Workload, a: np.ndarray) -> np.ndarray:
    """Round to the workload's storage type; returns float32 holding exact values."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    if w.dtype == "f32":
        return a
    import torch
    return torch.from_numpy(a).to(torch.bfloat16).to(torch.float32).numpy()


def _normal(w, shape, std, *key):
    r = _rng(w, *key)
    a = r.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return to_storage(w, a)


# ---- weights -------------------------------------------------------------

def W_fc(w: Workload):
    """fc weight [d, k*d] (nn.Linear layout), N(0, 0.02^2)."""
    return _normal(w, (w.d, w.k * w.d), 0.02, _T_WFC)


def W_Q(w: Workload, layer: int):
    return _normal(w, (w.n_h * w.d_h, w.d), 0.02, _T_WQ, layer)


def W_K(w: Workload, layer: int):
    return _normal(w, (w.n_kv * w.d_h, w.d), 0.02, _T_WK, layer)


def W_V(w: Workload, layer: int):
    return _normal(w, (w.n_kv * w.d_h, w.d), 0.02, _T_WV, layer)


def _gamma(w, n, which, layer):
    if not w.random_gamma:
        return np.ones(n, dtype=np.float32)
    r = _rng(w, _T_GAMMA, which, layer)
    return to_storage(w, 1.0 + 0.1 * r.standard_normal(n, dtype=np.float32))


def gamma_h(w: Workload):
    """hidden_norm gamma [d]."""
    return _gamma(w, w.d, 0, 0)


def gamma_q(w: Workload, layer: int):
    """q_norm gamma [d_h]."""
    return _gamma(w, w.d_h, 1, layer)


def gamma_k(w: Workload, layer: int):
    """k_norm gamma [d_h]."""
    return _gamma(w, w.d_h, 2, layer)


def gamma_post(w: Workload, layer: int):
    """post-attention RMSNorm gamma [d]."""
    return _gamma(w, w.d, 3, layer)


# ---- the rest of the decoder layer (o_proj, MLP) ----------------------------

def W_O(w: Workload, layer: int):
    return _normal(w, (w.d, w.n_h * w.d_h), 0.02, _T_WO, layer)


def W_gate(w: Workload, layer: int):
    return _normal(w, (w.ffn, w.d), 0.02, _T_WGATE, layer)


def W_up(w: Workload, layer: int):
    return _normal(w, (w.ffn, w.d), 0.02, _T_WUP, layer)


def W_down(w: Workload, layer: int):
    return _normal(w, (w.d, w.ffn), 0.02, _T_WDOWN, layer)


def residual(w: Workload, rnd: int, layer: int):
    """The residual stream entering a layer's output part, [B * bs][d] ~ N(0, 1)."""
    return _normal(w, (w.batch * w.bs, w.d), 1.0, _T_RESID, rnd, layer)


def attn_rows(w: Workload, rnd: int, layer: int):
    """Stand-in attention output rows [B * bs][n_h * d_h] ~ N(0, 0.25) (values of V rows'
    convex combinations) for exercising the layer output alone."""
    return _normal(w, (w.batch * w.bs, w.n_h * w.d_h), 0.5, _T_ATTN, rnd, layer)


# ---- schedule ------------------------------------------------------------

def prefill_lens(w: Workload) -> np.ndarray:
    """Cached rows per sequence before round 1, U{lo..hi}."""
    if w.prefill_lo == w.prefill_hi:
        return np.full(w.batch, w.prefill_lo, dtype=np.int64)
    r = _rng(w, _T_PREFILL_LEN)
    return r.integers(w.prefill_lo, w.prefill_hi + 1, size=w.batch).astype(np.int64)


def accepted_plus_one(w: Workload, rnd: int) -> np.ndarray:
    """Context rows injected per sequence in round ``rnd`` (1-based).

    Round 1 injects ``new_ctx`` rows. Later rounds inject acceptance + 1 rows,
    drawn U{1..bs} (the walkthrough's example accepts 2 of 3 and injects 3).
    The walkthrough workload uses the example's own count, 3.
    """
    if rnd == 1:
        return np.full(w.batch, w.new_ctx, dtype=np.int64)
    if w.name.startswith("walkthrough"):
        return np.full(w.batch, 3, dtype=np.int64)
    r = _rng(w, _T_ACCEPT, rnd)
    return r.integers(1, w.bs + 1, size=w.batch).astype(np.int64)


def cu_rows(counts) -> np.ndarray:
    """Prefix offsets [B+1] of per-sequence row counts (row grouping only)."""
    out = np.zeros(len(counts) + 1, dtype=np.int64)
    out[1:] = np.cumsum(counts)
    return out


# ---- activations ---------------------------------------------------------

def hidden_states(w: Workload, rnd: int, counts=None):
    """The k target-layer hidden-state arrays [M, d] of one round, N(0, 1).

    Rows are grouped by sequence (sequence b owns counts[b] consecutive rows);
    round 0 is the prefill of a ``prefill_inject`` workload. Each sequence's
    rows come from their own stream.
    """
    if counts is None:
        counts = prefill_lens(w) if rnd == 0 else accepted_plus_one(w, rnd)
    out = []
    for j in range(w.k):
        parts = [_normal(w, (int(n), w.d), 1.0, _T_HIDDEN, rnd, j, b)
                 for b, n in enumerate(counts)]
        out.append(np.concatenate(parts, axis=0) if parts else np.zeros((0, w.d), np.float32))
    return out


def hidden_states_rows(w: Workload, rnd: int, b: int, n: int):
    """Sequence b's rows of ``hidden_states`` (same stream, drawn alone)."""
    return [_normal(w, (int(n), w.d), 1.0, _T_HIDDEN, rnd, j, b) for j in range(w.k)]


def block_embeddings(w: Workload, rnd: int, layer: int, b: int = None):
    """The block's hidden states H [B, bs, d] for one layer, N(0, 1).

    An independent draw per layer stands in for the output of the earlier
    draft layers (the decoder MLP and o_proj are outside the step).
    """
    if b is not None:
        return _normal(w, (w.bs, w.d), 1.0, _T_BLOCK, rnd, layer, b)
    return np.stack([_normal(w, (w.bs, w.d), 1.0, _T_BLOCK, rnd, layer, bb)
                     for bb in range(w.batch)], axis=0)


def kv_scales(w: Workload):
    """Per-layer (k_scales, v_scales) of an fp8 cache: fixed calibration constants that put
    the synthetic K (unit RMS) and V (RMS about 1.3) well inside the E4M3 range."""
    k = np.array([0.25 * (1 + 0.5 * l) for l in range(w.n_layers)], dtype=np.float64)
    v = np.array([0.125 * (1 + 0.25 * l) for l in range(w.n_layers)], dtype=np.float64)
    return k, v


def cache_rows(w: Workload, layer: int, b: int, n: int = None):
    """Synthetic pre-filled cache rows of one sequence: K, V as [n_kv, n, d_h]."""
    if n is None:
        n = int(prefill_lens(w)[b])
    K = _normal(w, (w.n_kv, n, w.d_h), 1.0, _T_CACHE_K, layer, b)
    V = _normal(w, (w.n_kv, n, w.d_h), 0.02 * np.sqrt(w.d), _T_CACHE_V, layer, b)
    return K, V


def to_fp8_codes(a: np.ndarray, scale: float) -> np.ndarray:
    """E4M3 codes (uint8) of a / scale by torch's float8_e4m3fn conversion: how seeded
    rows are written into an fp8 device cache before a round."""
    import torch
    x = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)) / float(scale)
    return x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def cache_rows_stored(w: Workload, layer: int, b: int, n: int = None):
    """cache_rows in the device cache's element form: storage-rounded values, or for an fp8
    cache the E4M3 codes of the rows divided by the layer's (k, v) scales."""
    K, V = cache_rows(w, layer, b, n)
    if w.kv != "fp8":
        return K, V
    ks, vs = kv_scales(w)
    return to_fp8_codes(K, ks[layer]), to_fp8_codes(V, vs[layer])
