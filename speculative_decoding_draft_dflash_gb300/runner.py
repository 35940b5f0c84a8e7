"""Drives DFlash draft rounds through the C ABI on device-resident synthetic inputs.

A round, per the walkthrough's Steps 2-4 and 7 and the source guide's part 4:
one context projection of the round's new rows (all sequences at once), then
for every draft layer a KV inject of those rows and a block attention (which
appends the block's K/V), then a crop of every layer back to the
context-only length ("crop(start)").

``DeviceWorkload`` owns the device buffers (weights, cache, RoPE table,
workspace); ``RoundInputs`` holds one round's inputs already in HBM. All
arithmetic happens in libdflash's kernels; this module only allocates (with
torch), copies inputs in and issues the calls.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import List

import numpy as np
import torch

from . import dflash as D
from . import synth


def _dev(a, dtype, device):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device=device, dtype=dtype)


@dataclass
class RoundInputs:
    rnd: int
    counts: np.ndarray           # context rows per sequence this round
    hidden: List[torch.Tensor]   # k tensors [M, d]
    cu_rows: torch.Tensor        # int32 [B+1]
    H: List[torch.Tensor]        # per layer [B, bs, d]
    crop_to: torch.Tensor        # int32 [B]: lengths after the round's crop
    M: int


class DeviceWorkload:
    def __init__(self, w: synth.Workload, device="cuda", prefill=True, capacity=None,
                 max_rows=None, paged=False):
        self.w = w
        self.device = device
        self.dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
        self.dims = D.make_dims(w.d, w.n_h, w.n_kv, w.d_h, w.k, w.bs, w.eps, w.dtype)
        dev = lambda a: _dev(a, self.dt, device)  # noqa: E731
        self.W_fc = dev(synth.W_fc(w))
        self.g_h = dev(synth.gamma_h(w))
        self.W_Q = [dev(synth.W_Q(w, l)) for l in range(w.n_layers)]
        self.W_K = [dev(synth.W_K(w, l)) for l in range(w.n_layers)]
        self.W_V = [dev(synth.W_V(w, l)) for l in range(w.n_layers)]
        self.g_q = [dev(synth.gamma_q(w, l)) for l in range(w.n_layers)]
        self.g_k = [dev(synth.gamma_k(w, l)) for l in range(w.n_layers)]
        self.capacity = capacity or w.capacity
        self.table_len = self.capacity
        if paged:  # whole pages per sequence
            self.capacity = -(-self.capacity // D.KVCache.PAGE) * D.KVCache.PAGE
            self.table_len = self.capacity
        self.cache = D.KVCache(w.n_layers, w.batch, w.n_kv, self.capacity, w.d_h, w.dtype, device,
                               paged=paged, seed=w.seed, kv=w.kv,
                               kv_scales=np.stack(synth.kv_scales(w), axis=1))
        self.rope = torch.empty((self.table_len, w.d_h // 2, 2), dtype=torch.float32, device=device)
        D.dflash_rope_table_build(w.theta, w.d_h, self.table_len, self.rope)
        self.L0 = synth.prefill_lens(w)
        rows = int(self.L0.sum()) if w.prefill_inject else 0
        self.max_rows = max_rows or max(rows, w.batch * max(w.new_ctx, w.bs), 1)
        nbytes = D.dflash_workspace_bytes(self.dims, w.batch, self.capacity, self.max_rows)
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.C = torch.empty((self.max_rows, w.d), dtype=self.dt, device=device)
        self.out = [torch.empty((w.batch, w.bs, w.n_h * w.d_h), dtype=self.dt, device=device)
                    for _ in range(w.n_layers)]
        if prefill:
            self.prefill()

    # -- set-up ---------------------------------------------------------------
    def prefill(self):
        """Fill the cache before round 1: synthetic rows, or projection + inject of real rows."""
        w = self.w
        if w.prefill_inject:
            counts = self.L0
            hid = [_dev(h, self.dt, self.device) for h in synth.hidden_states(w, 0, counts)]
            cu = torch.from_numpy(synth.cu_rows(counts).astype(np.int32)).to(self.device)
            M = int(counts.sum())
            C = torch.empty((M, w.d), dtype=self.dt, device=self.device)
            D.dflash_ctx_project(self.dims, hid, M, self.W_fc, self.g_h, C, self.ws)
            for l in range(w.n_layers):
                D.dflash_kv_inject(self.dims, self.cache, l, C, cu, M, self.W_K[l], self.W_V[l],
                                   self.g_k[l], self.rope, self.table_len, self.ws)
            self.prefill_C = C
            return
        for l in range(w.n_layers):
            for b in range(w.batch):
                n = int(self.L0[b])
                if n == 0:
                    continue
                K, V = synth.cache_rows_stored(w, l, b, n)
                et = self.cache.k.dtype
                self.cache.set_rows(l, b, _dev(K, et, self.device), _dev(V, et, self.device))
        self.cache.lens.copy_(torch.from_numpy(
            np.tile(self.L0.astype(np.int32), (w.n_layers, 1))).to(self.device))

    def round_inputs(self, rnd, lens_before, counts=None, crop_to=None) -> RoundInputs:
        """Upload round ``rnd``'s inputs. ``lens_before``: per-sequence length at the round's start."""
        w = self.w
        if counts is None:
            counts = synth.accepted_plus_one(w, rnd)
        hid = [_dev(h, self.dt, self.device) for h in synth.hidden_states(w, rnd, counts)]
        cu = torch.from_numpy(synth.cu_rows(counts).astype(np.int32)).to(self.device)
        H = [_dev(synth.block_embeddings(w, rnd, l), self.dt, self.device)
             for l in range(w.n_layers)]
        if crop_to is None:
            crop_to = np.asarray(lens_before) + counts
        crop = torch.from_numpy(np.asarray(crop_to, dtype=np.int32)).to(self.device)
        return RoundInputs(rnd, counts, hid, cu, H, crop, int(counts.sum()))

    # -- one round --------------------------------------------------------------
    def run_round(self, x: RoundInputs, crop=True, stream=None, fused_layer=True, out=None):
        """ctx_project -> for each layer (kv_inject, block_attn) -> crop. Results stay on device.

        ``fused_layer``: issue each layer's inject + block attention as one
        dflash_draft_layer call (same results) instead of two calls.
        ``out``: per-layer output buffers (default: this workload's own).
        """
        w = self.w
        out = self.out if out is None else out
        C = self.C[:x.M]
        D.dflash_ctx_project(self.dims, x.hidden, x.M, self.W_fc, self.g_h, C, self.ws, stream)
        for l in range(w.n_layers):
            if fused_layer:
                D.dflash_draft_layer(self.dims, self.cache, l, C, x.cu_rows, x.M, x.H[l],
                                     self.W_Q[l], self.W_K[l], self.W_V[l], self.g_q[l], self.g_k[l],
                                     self.rope, self.table_len, w.windows[l], 0.0, out[l],
                                     self.ws, stream)
                continue
            D.dflash_kv_inject(self.dims, self.cache, l, C, x.cu_rows, x.M, self.W_K[l],
                               self.W_V[l], self.g_k[l], self.rope, self.table_len, self.ws,
                               stream)
            D.dflash_block_attn(self.dims, self.cache, l, x.H[l], self.W_Q[l], self.W_K[l],
                                self.W_V[l], self.g_q[l], self.g_k[l], self.rope, self.table_len,
                                w.windows[l], 0.0, out[l], self.ws, stream)
        if crop:
            D.dflash_cache_crop(self.cache, x.crop_to, stream)
        return C
