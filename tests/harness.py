"""Runs a synthetic workload's rounds on the device (through the C ABI) and in the oracle.

The oracle side replays only a chosen subset of sequences: every output row
of the step depends on its own sequence alone, and the synthetic inputs of
any sequence can be drawn on their own, so a subset checks the full-size
launch exactly on the rows it covers.
"""

from __future__ import annotations

import numpy as np

from oracle import dflash_oracle as O
from speculative_decoding_draft_dflash_gb300 import synth


# ---------------------------------------------------------------------------
# tolerances (float32 path: max-abs 1e-4; bf16 storage: rel-L2 1e-2 and max-abs 3e-2)
# ---------------------------------------------------------------------------

def check_close(got, ref, dtype, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - ref)
    max_abs = float(err.max()) if err.size else 0.0
    if dtype == "f32":
        assert max_abs <= 1e-4, f"{what}: max-abs {max_abs:.3e} > 1e-4"
        return max_abs, 0.0
    nref = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(got - ref)) / nref if nref > 0 else float(np.linalg.norm(got))
    assert rel <= 1e-2, f"{what}: rel-L2 {rel:.3e} > 1e-2"
    assert max_abs <= 3e-2, f"{what}: max-abs {max_abs:.3e} > 3e-2"
    return max_abs, rel


# ---------------------------------------------------------------------------
# oracle replay of a subset of sequences
# ---------------------------------------------------------------------------

def oracle_rounds(w: synth.Workload, seqs, rounds=None):
    """Replays the workload's schedule for sequences ``seqs`` in the float64 oracle.

    Returns a list (one entry per round) of dicts with, per sequence b in seqs:
    C[b] [n_b, d], out[l][b] [bs, n_h*d_h], rows[l][b] = (K, V) rows appended this
    round (context then block), lens_block[l][b], lens_crop[b].

    fp8 cache: an E4M3 code is an integer decided by floating point, so the oracle takes
    that decision from the value the device takes it from: the context rows C as the
    device stores them (rounded to bf16) feed the inject. Everything downstream stays
    float64.
    """
    as_stored = (lambda C: synth.to_storage(w, C).astype(np.float64)) if w.kv == "fp8" else \
        (lambda C: C)
    rounds = rounds or w.rounds
    S = list(seqs)
    L0 = synth.prefill_lens(w)
    cache = O.DraftKVCache(w.n_layers, len(S), w.n_kv, w.d_h, capacity=w.capacity,
                           fp8_scales=synth.kv_scales(w) if w.kv == "fp8" else None)
    W_fc = synth.W_fc(w)
    g_h = synth.gamma_h(w)
    Wq = [synth.W_Q(w, l) for l in range(w.n_layers)]
    Wk = [synth.W_K(w, l) for l in range(w.n_layers)]
    Wv = [synth.W_V(w, l) for l in range(w.n_layers)]
    gq = [synth.gamma_q(w, l) for l in range(w.n_layers)]
    gk = [synth.gamma_k(w, l) for l in range(w.n_layers)]
    if w.prefill_inject:
        Cs = [as_stored(O.ctx_project(synth.hidden_states_rows(w, 0, b, L0[b]), W_fc, g_h, w.eps))
              for b in S]
        cu = synth.cu_rows([L0[b] for b in S])
        for l in range(w.n_layers):
            O.kv_inject(cache, l, np.concatenate(Cs), cu, Wk[l], Wv[l], gk[l], w.n_kv, w.d_h,
                        w.eps, w.theta)
    else:
        for l in range(w.n_layers):
            for i, b in enumerate(S):
                K, V = synth.cache_rows(w, l, b, int(L0[b]))
                cache.set_rows(l, i, K, V)
    results = []
    for rnd in range(1, rounds + 1):
        counts = synth.accepted_plus_one(w, rnd)
        before = cache.lens[0].copy()
        Cs = [as_stored(O.ctx_project(synth.hidden_states_rows(w, rnd, b, counts[b]), W_fc, g_h,
                                      w.eps)) for b in S]
        cu = synth.cu_rows([counts[b] for b in S])
        res = {"C": {}, "out": [], "rows": [], "lens_block": [], "before": {}}
        for i, b in enumerate(S):
            res["C"][b] = Cs[i]
            res["before"][b] = int(before[i])
        for l in range(w.n_layers):
            O.kv_inject(cache, l, np.concatenate(Cs), cu, Wk[l], Wv[l], gk[l], w.n_kv, w.d_h,
                        w.eps, w.theta)
            H = np.stack([synth.block_embeddings(w, rnd, l, b) for b in S])
            out = O.block_attn(cache, l, H, Wq[l], Wk[l], Wv[l], gq[l], gk[l], w.n_h, w.n_kv,
                               w.d_h, w.eps, w.theta, w.windows[l])
            res["out"].append({b: out[i] for i, b in enumerate(S)})
            lo = before
            res["rows"].append({b: (cache.k[l][i][:, lo[i]:], cache.v[l][i][:, lo[i]:])
                                for i, b in enumerate(S)})
            res.setdefault("rows_raw", []).append(
                {b: (cache.kraw[l][i][:, lo[i]:], cache.vraw[l][i][:, lo[i]:])
                 for i, b in enumerate(S)})
            res["lens_block"].append({b: int(cache.lens[l][i]) for i, b in enumerate(S)})
        O.cache_crop(cache, before + np.array([counts[b] for b in S]))
        res["lens_crop"] = {b: int(cache.lens[0][i]) for i, b in enumerate(S)}
        assert cache.errors == 0
        results.append(res)
    return results


# ---------------------------------------------------------------------------
# device run
# ---------------------------------------------------------------------------

def device_rounds(w: synth.Workload, seqs, rounds=None, dev=None, fused_layer=True, paged=False):
    """Runs the same schedule on the device for all sequences; returns host copies for ``seqs``."""
    import torch
    from speculative_decoding_draft_dflash_gb300 import dflash as D
    from speculative_decoding_draft_dflash_gb300.runner import DeviceWorkload

    rounds = rounds or w.rounds
    dev = dev or DeviceWorkload(w, paged=paged)
    assert D.dflash_status_get() == 0
    results = []
    lens = synth.prefill_lens(w).copy()
    assert dev.cache.lens.cpu().numpy().tolist() == [lens.tolist()] * w.n_layers
    for rnd in range(1, rounds + 1):
        x = dev.round_inputs(rnd, lens)
        res = {"C": {}, "out": [], "rows": [], "lens_block": [], "before": {}}
        C = dev.run_round(x, crop=False, fused_layer=fused_layer)
        torch.cuda.synchronize()
        lens_block = dev.cache.lens.cpu().numpy().copy()
        Ch = C.float().cpu().numpy()
        cu = synth.cu_rows(x.counts)
        for b in seqs:
            res["C"][b] = Ch[cu[b]:cu[b + 1]]
            res["before"][b] = int(lens[b])
        for l in range(w.n_layers):
            o = dev.out[l].float().cpu().numpy()
            res["out"].append({b: o[b] for b in seqs})
            res["rows"].append({b: (dev.cache.rows("k", l, b, lens[b], lens_block[l, b]).float().cpu().numpy(),
                                    dev.cache.rows("v", l, b, lens[b], lens_block[l, b]).float().cpu().numpy())
                                for b in seqs})
            if dev.cache.fp8:
                res.setdefault("codes", []).append(
                    {b: tuple(dev.cache.rows(x, l, b, lens[b], lens_block[l, b], codes=True)
                              .cpu().numpy() for x in ("k", "v")) for b in seqs})
            res["lens_block"].append({b: int(lens_block[l, b]) for b in seqs})
        res["lens_block_all"] = lens_block
        from speculative_decoding_draft_dflash_gb300 import dflash as D2
        D2.dflash_cache_crop(dev.cache, x.crop_to)
        torch.cuda.synchronize()
        lens_crop = dev.cache.lens.cpu().numpy().copy()
        res["lens_crop_all"] = lens_crop
        res["lens_crop"] = {b: int(lens_crop[0, b]) for b in seqs}
        res["status"] = D.dflash_status_get()
        expect_block = np.tile(lens + x.counts + w.bs, (w.n_layers, 1))
        assert (lens_block == expect_block).all(), "lengths after block attention"
        lens = lens + x.counts
        assert (lens_crop == np.tile(lens, (w.n_layers, 1))).all(), "lengths after crop"
        results.append(res)
    return results, dev


def compare(w, dev_res, ora_res, seqs):
    """Element-wise comparison of every recorded output; lengths bit-exact."""
    report = {}
    for r, (g, o) in enumerate(zip(dev_res, ora_res)):
        assert g["status"] == 0, f"round {r + 1}: device status {g['status']}"
        for b in seqs:
            report[f"r{r + 1}.C.{b}"] = check_close(g["C"][b], o["C"][b], w.dtype,
                                                     f"round {r + 1} C seq {b}")
            assert g["lens_crop"][b] == o["lens_crop"][b]
            for l in range(w.n_layers):
                assert g["lens_block"][l][b] == o["lens_block"][l][b]
                report[f"r{r + 1}.out.{l}.{b}"] = check_close(
                    g["out"][l][b], o["out"][l][b], w.dtype, f"round {r + 1} layer {l} out seq {b}")
                gk, gv = g["rows"][l][b]
                ok, ov = o["rows"][l][b]
                if w.kv == "fp8":
                    ks, vs = synth.kv_scales(w)
                    for name, got, raw, sc in (("K", g["codes"][l][b][0], o["rows_raw"][l][b][0], ks[l]),
                                               ("V", g["codes"][l][b][1], o["rows_raw"][l][b][1], vs[l])):
                        check_fp8_codes(got, raw / sc, f"round {r + 1} layer {l} {name} codes seq {b}")
                    continue
                check_close(gk, ok, w.dtype, f"round {r + 1} layer {l} K rows seq {b}")
                check_close(gv, ov, w.dtype, f"round {r + 1} layer {l} V rows seq {b}")
    return report


FP8_CODE_STATS = []  # (what, codes compared, codes that differ from the oracle's rounding)


def check_fp8_codes(got, y, what, max_frac=1e-2, rel_delta=2e-3):
    """Device E4M3 values ``got`` (codes read back, before the scale) against the oracle's
    unquantised rows ``y`` (already divided by the scale), [..., d_h].

    The code is an integer decided by floating point, and the two sides decide from
    values that differ slightly: the oracle takes the context rows C as stored in bf16,
    but the device rounds a float32 C and the oracle a float64 one, and the two roundings
    differ at a fraction of the elements of C; with the float32 accumulation on top, a
    cached element differs by up to about 1e-3 of its row's RMS. So: (1) every code must
    be a correct rounding of some value within ``rel_delta`` x (row RMS) of y, i.e. lie
    between the codes of y - delta and y + delta (rounding is monotone); (2) at most
    ``max_frac`` of the codes may differ from the oracle's own rounding of y (a wrong
    rounding mode or scale changes far more).
    """
    got = np.asarray(got, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    assert got.shape == y.shape, f"{what}: shape {got.shape} vs {y.shape}"
    want = O.e4m3_dequantize(O.e4m3_quantize(y))
    diff = got != want
    frac = float(diff.mean()) if diff.size else 0.0
    FP8_CODE_STATS.append((what, int(diff.size), int(diff.sum())))
    assert frac <= max_frac, f"{what}: {frac:.2e} of the codes differ from the oracle's rounding"
    if diff.any():
        delta = rel_delta * np.sqrt(np.mean(y * y, axis=-1, keepdims=True))
        lo = O.e4m3_dequantize(O.e4m3_quantize(y - delta))
        hi = O.e4m3_dequantize(O.e4m3_quantize(y + delta))
        ok = (got >= lo) & (got <= hi)
        assert ok.all(), (f"{what}: {int((~ok).sum())} codes are no rounding of a value "
                          f"within {rel_delta} x row RMS")
    return frac
