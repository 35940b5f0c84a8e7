"""Pins of the float64 oracle against facts that do not come from the oracle itself.

Each ``pin_*`` takes the oracle module and raises AssertionError when the
oracle disagrees with a closed form, a library routine, brute force on a tiny
case, or a value the source pages print. ``test_oracle_pins.py`` runs them on
the oracle as written; ``test_oracle_mutations.py`` plants plausible mistakes
in the oracle and checks that some pin catches each one.
"""

from __future__ import annotations

import json
import math
import os

import numpy as np
import torch
import torch.nn.functional as F

from speculative_decoding_draft_dflash_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _close(a, b, tol=1e-12, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} != {b.shape}"
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    scale = max(1.0, float(np.max(np.abs(b))) if b.size else 1.0)
    assert err <= tol * scale, f"{what}: max abs err {err:.3e}"


def _rand(shape, seed, std=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * std


def _walkthrough_inputs():
    w = synth.WORKLOADS["walkthrough_f32"]
    hid = synth.hidden_states(w, 1)
    return w, dict(hid=hid, W_fc=synth.W_fc(w), W_Q=synth.W_Q(w, 0), W_K=synth.W_K(w, 0),
                   W_V=synth.W_V(w, 0), g_h=synth.gamma_h(w), g_q=synth.gamma_q(w, 0),
                   g_k=synth.gamma_k(w, 0), H=synth.block_embeddings(w, 1, 0)[0])


# ---------------------------------------------------------------------------
# Shapes printed by the walkthrough
# ---------------------------------------------------------------------------

def pin_walkthrough_shapes(O):
    """Every shape the walkthrough prints for its d=512, 8-head, k=3 example."""
    g = _golden("walkthrough_shapes.json")
    w, x = _walkthrough_inputs()
    raw = O.extract_context_feature(x["hid"])
    assert list(raw.shape) == g["target_hidden_raw"]
    assert list(x["W_fc"].T.shape) == g["W_fc_page"]
    C = O.ctx_project(x["hid"], x["W_fc"], x["g_h"], w.eps)
    assert list(C.shape) == g["C"]
    assert list(x["H"].shape) == g["H"]
    out, q, k, v = O.draft_attention_forward(C, x["H"], x["W_Q"], x["W_K"], x["W_V"], x["g_q"],
                                             x["g_k"], w.n_h, w.n_kv, w.d_h, w.eps, w.theta)
    assert list(q.shape) == g["Q"] and list(k.shape) == g["K"] and list(v.shape) == g["V"]
    cos, sin = O.rope_cos_sin(np.arange(7), w.d_h, w.theta)
    assert list(cos.shape) == g["cos_sin"] and list(sin.shape) == g["cos_sin"]
    A = O.attention_weights(q, k, g["q_positions"], g["k_positions"], w.d_h ** -0.5)
    assert list(A.shape[1:]) == g["attention_per_head"]
    assert w.d_h ** -0.5 == g["scaling"]
    assert list(out.shape) == g["out"]


# ---------------------------------------------------------------------------
# RMSNorm
# ---------------------------------------------------------------------------

def pin_rmsnorm_matches_torch(O):
    """RMSNorm equals torch.nn.functional.rms_norm (float64), with gamma and a large eps."""
    x = _rand((5, 3, 16), 1, 2.0)
    g = 1.0 + _rand((16,), 2, 0.3)
    for eps in (1e-6, 0.5):
        ref = F.rms_norm(torch.from_numpy(x), (16,), torch.from_numpy(g), eps).numpy()
        _close(O.rms_norm(x, g, eps), ref, 1e-12, f"rms_norm eps={eps}")


def pin_rmsnorm_mean_square(O):
    """With gamma = 1 each output row has mean square m / (m + eps) (closed form)."""
    x = _rand((7, 64), 3, 0.1)
    eps = 1e-3
    y = O.rms_norm(x, np.ones(64), eps)
    m = np.mean(x * x, axis=-1)
    _close(np.mean(y * y, axis=-1), m / (m + eps), 1e-12, "mean square")


# ---------------------------------------------------------------------------
# RoPE
# ---------------------------------------------------------------------------

def _rot(a):
    return np.array([[math.cos(a), -math.sin(a)], [math.sin(a), math.cos(a)]])


def pin_rope_position_zero_identity(O):
    x = _rand((3, 64), 4)
    cos, sin = O.rope_cos_sin(np.zeros(3, dtype=np.int64), 64, 1e6)
    _close(O.apply_rope(x, cos, sin), x, 1e-15, "rope at position 0")


def pin_rope_2d_rotation(O):
    """d_h = 2: RoPE at position p is the plane rotation by p radians (inv_freq = 1)."""
    x = _rand((5, 2), 5)
    pos = np.array([0, 1, 2, 7, 100])
    cos, sin = O.rope_cos_sin(pos, 2, 1e4)
    y = O.apply_rope(x, cos, sin)
    ref = np.stack([_rot(float(p)) @ x[i] for i, p in enumerate(pos)])
    _close(y, ref, 1e-12, "2-D rotation")


def pin_rope_pairs_and_frequencies(O):
    """d_h = 4, theta = 100: pair (x0, x2) turns by p, pair (x1, x3) by p / 10.

    inv_freq_i = theta^(-2i/d_h) gives 1 and 100^(-1/2) = 0.1; rotate-half pairs
    coordinate i with i + d_h/2.
    """
    x = _rand((4, 4), 6)
    pos = np.array([1, 3, 5, 11])
    cos, sin = O.rope_cos_sin(pos, 4, 100.0)
    y = O.apply_rope(x, cos, sin)
    for i, p in enumerate(pos):
        a = _rot(float(p)) @ x[i, [0, 2]]
        b = _rot(float(p) * 0.1) @ x[i, [1, 3]]
        _close(y[i, [0, 2]], a, 1e-12, "pair 0")
        _close(y[i, [1, 3]], b, 1e-12, "pair 1")


def pin_rope_relative_position(O):
    """Scores depend only on j - i: shifting every position by the same amount changes nothing.

    The walkthrough's Step 4.3 alignment: Q at 3..6, K at 0..6.
    """
    q = _rand((4, 64), 7)
    k = _rand((7, 64), 8)
    qp, kp = np.arange(3, 7), np.arange(7)
    s = []
    for shift in (0, 1000, 31337):
        cq, sq = O.rope_cos_sin(qp + shift, 64, 1e6)
        ck, sk = O.rope_cos_sin(kp + shift, 64, 1e6)
        s.append(O.apply_rope(q, cq, sq) @ O.apply_rope(k, ck, sk).T)
    _close(s[1], s[0], 1e-9, "shift 1000")
    _close(s[2], s[0], 1e-9, "shift 31337")


def pin_rope_wrong_query_positions(O):
    """The walkthrough's counter-example: Q roped at [0..3] instead of [3..6].

    With the wrong positions the query of position 5 sits at 2, so its score with
    the key at position 2 equals the un-rotated dot product (angle difference 0);
    with the right positions it does not.
    """
    q = _rand((4, 64), 9)
    k = _rand((7, 64), 10)
    ck, sk = O.rope_cos_sin(np.arange(7), 64, 1e6)
    kr = O.apply_rope(k, ck, sk)
    cw, sw = O.rope_cos_sin(np.arange(0, 4), 64, 1e6)
    cr, sr = O.rope_cos_sin(np.arange(3, 7), 64, 1e6)
    wrong = O.apply_rope(q, cw, sw)[2] @ kr[2]
    right = O.apply_rope(q, cr, sr)[2] @ kr[2]
    assert abs(wrong - q[2] @ k[2]) < 1e-9
    assert abs(right - q[2] @ k[2]) > 1e-3


def pin_rope_norm_preserving(O):
    x = _rand((9, 128), 11)
    cos, sin = O.rope_cos_sin(np.arange(9) * 4001, 128, 1e6)
    _close(np.linalg.norm(O.apply_rope(x, cos, sin), axis=-1), np.linalg.norm(x, axis=-1),
           1e-12, "norm")


# ---------------------------------------------------------------------------
# Attention
# ---------------------------------------------------------------------------

def _sdpa(Q, K, V, mask, scale):
    G = Q.shape[0] // K.shape[0]
    Kr = torch.from_numpy(K).repeat_interleave(G, dim=0)
    Vr = torch.from_numpy(V).repeat_interleave(G, dim=0)
    o = F.scaled_dot_product_attention(torch.from_numpy(Q)[None], Kr[None], Vr[None],
                                       attn_mask=torch.from_numpy(mask), scale=scale)[0]
    return o.permute(1, 0, 2).reshape(Q.shape[1], -1).numpy()


def pin_attention_matches_sdpa(O):
    """Non-causal GQA attention equals torch SDPA (float64) with K/V repeat_interleaved.

    Covers MHA (G=1), GQA (G=4), the walkthrough's positions, and a sliding window.
    """
    for (n_h, n_kv, Lq, Lk, d_h, W, seed) in [(8, 8, 4, 7, 64, 0, 12), (8, 2, 5, 40, 16, 0, 13),
                                             (4, 1, 16, 300, 32, 64, 14), (6, 3, 3, 9, 8, 4, 15)]:
        Q, K, V = _rand((n_h, Lq, d_h), seed), _rand((n_kv, Lk, d_h), seed + 100), \
            _rand((n_kv, Lk, d_h), seed + 200)
        qp = np.arange(Lk - Lq, Lk)
        kp = np.arange(Lk)
        mask = np.ones((Lq, Lk), dtype=bool) if W == 0 else (qp[:, None] - kp[None, :] < W)
        s = d_h ** -0.5
        _close(O.attention(Q, K, V, qp, kp, s, W), _sdpa(Q, K, V, mask, s), 1e-12,
               f"sdpa n_h={n_h} n_kv={n_kv} W={W}")


def pin_attention_bruteforce(O):
    """Pure-Python loops on tiny cases (GQA, window, keys ahead of the query)."""
    for (n_h, n_kv, Lq, Lk, d_h, W, seed) in [(2, 1, 2, 3, 4, 0, 21), (4, 2, 3, 6, 2, 2, 22)]:
        Q, K, V = _rand((n_h, Lq, d_h), seed), _rand((n_kv, Lk, d_h), seed + 1), \
            _rand((n_kv, Lk, d_h), seed + 2)
        qp = list(range(Lk - Lq, Lk))
        s = 1.0 / math.sqrt(d_h)
        ref = np.zeros((Lq, n_h * d_h))
        G = n_h // n_kv
        for h in range(n_h):
            g = h // G
            for i in range(Lq):
                vis = [j for j in range(Lk) if W == 0 or qp[i] - j < W]
                sc = [sum(Q[h, i, t] * K[g, j, t] for t in range(d_h)) * s for j in vis]
                mx = max(sc)
                e = [math.exp(x - mx) for x in sc]
                z = sum(e)
                for t in range(d_h):
                    ref[i, h * d_h + t] = sum(e[n] / z * V[g, j, t] for n, j in enumerate(vis))
        _close(O.attention(Q, K, V, qp, list(range(Lk)), s, W), ref, 1e-12, "brute force")


def pin_softmax_rows(O):
    """Attention rows are non-negative and sum to 1 (walkthrough Step 4.4)."""
    Q, K = _rand((8, 4, 64), 30), _rand((8, 7, 64), 31)
    A = O.attention_weights(Q, K, np.arange(3, 7), np.arange(7), 0.125)
    assert np.all(A >= 0)
    _close(A.sum(-1), np.ones((8, 4)), 1e-12, "row sums")


def pin_single_and_identical_keys(O):
    """One key: out = v. Identical keys: uniform weights, out = mean of V."""
    Q = _rand((4, 3, 16), 32)
    K1, V1 = _rand((2, 1, 16), 33), _rand((2, 1, 16), 34)
    out = O.attention(Q, K1, V1, [5, 6, 7], [0], 0.25)
    ref = np.concatenate([np.repeat(V1[h // 2], 3, axis=0) for h in range(4)], axis=1)
    _close(out, ref, 1e-12, "single key")
    K = np.repeat(_rand((2, 1, 16), 35), 5, axis=1)
    V = _rand((2, 5, 16), 36)
    out = O.attention(Q, K, V, [5, 6, 7], list(range(5)), 0.25)
    ref = np.concatenate([np.repeat(V[h // 2].mean(0, keepdims=True), 3, axis=0)
                          for h in range(4)], axis=1)
    _close(out, ref, 1e-12, "identical keys")


def pin_window_reduces_to_full(O):
    Q, K, V = _rand((4, 4, 8), 40), _rand((2, 20, 8), 41), _rand((2, 20, 8), 42)
    qp, kp = np.arange(16, 20), np.arange(20)
    _close(O.attention(Q, K, V, qp, kp, 0.3, 20), O.attention(Q, K, V, qp, kp, 0.3, 0),
           1e-12, "window >= length")


# ---------------------------------------------------------------------------
# Context projection
# ---------------------------------------------------------------------------

def pin_fc_selects_layer(O):
    """W_fc = [I 0 0] gives C = RMSNorm(h^(l1)); [0 0 I] gives RMSNorm(h^(l3)).

    Pins the feature concatenation order (ascending layers, walkthrough Step 1)
    and the orientation of W_fc.
    """
    d, k = 8, 3
    hid = [_rand((5, d), 50 + j) for j in range(k)]
    g = 1.0 + _rand((d,), 53, 0.2)
    for j in range(k):
        W = np.zeros((d, k * d))
        W[:, j * d:(j + 1) * d] = np.eye(d)
        _close(O.ctx_project(hid, W, g, 1e-6), F.rms_norm(torch.from_numpy(hid[j]), (d,),
               torch.from_numpy(g), 1e-6).numpy(), 1e-12, f"select layer {j}")
    # A non-square W_fc: rows of C are the fc outputs of the concatenated features.
    W = _rand((6, k * d), 54)
    raw = np.concatenate(hid, axis=1)
    ref = F.rms_norm(torch.from_numpy(raw @ W.T), (6,), None, 1e-6).numpy()
    _close(O.ctx_project(hid, W, np.ones(6), 1e-6), ref, 1e-12, "non-square fc")


# ---------------------------------------------------------------------------
# Head layout of the projections (walkthrough Steps 4.1-4.2)
# ---------------------------------------------------------------------------

def _head_select(n_heads, d_h, d, offsets):
    """A weight [n_heads*d_h, d] whose output features h*d_h .. (h+1)*d_h-1 copy input
    features offsets[h] .. offsets[h]+d_h-1, i.e. head h of the view [n, n_heads, d_h]
    reads that slice of the input row."""
    W = np.zeros((n_heads * d_h, d))
    for h, s in enumerate(offsets):
        W[h * d_h:(h + 1) * d_h, s:s + d_h] = np.eye(d_h)
    return W


def pin_head_layout_by_selection(O):
    """Head h of a projection is output features [h*d_h, (h+1)*d_h).

    The walkthrough splits a projected row by view(bsz, q_len, -1, head_dim) (Step 4.1:
    [4, 512] -> [4, 8, 64]; Step 4.2: [7, 512] -> [7, 8, 64]): the head index is the
    slower of the two split axes. With a weight whose head-h block of rows copies one
    slice of the input, head h must hold exactly that slice (V, not normalised), its
    torch RMSNorm (Q and K at position 0, where RoPE is the identity) or that norm
    rotated at the row's position (the 2-D rotation per (i, i + d_h/2) pair); every
    other head reads zeros. Heads use distinct, overlapping slices, so a strided or
    transposed split, or a wrong head order, moves values between heads.
    """
    n_h, n_kv, d_h, d, n = 8, 2, 64, 512, 4
    H = _rand((n, d), 70)
    offs_q = [(37 * h + 5) % (d - d_h) for h in range(n_h)]
    offs_kv = [11, 300]
    WQ = _head_select(n_h, d_h, d, offs_q)
    WK = _head_select(n_kv, d_h, d, offs_kv)
    WV = _head_select(n_kv, d_h, d, offs_kv[::-1])
    ones = np.ones(d_h)
    tn = lambda x: F.rms_norm(torch.from_numpy(np.ascontiguousarray(x)), (d_h,), None,
                              1e-6).numpy()
    # position 0: RoPE is the identity, so Q = RMSNorm of the selected slice
    q = O.q_project(H, WQ, ones, n_h, d_h, 1e-6, np.zeros(n, dtype=np.int64), 1e6)
    assert q.shape == (n_h, n, d_h)
    for h in range(n_h):
        _close(q[h], tn(H[:, offs_q[h]:offs_q[h] + d_h]), 1e-12, f"Q head {h}")
    K, V = O.kv_project(H, WK, WV, ones, n_kv, d_h, 1e-6, np.zeros(n, dtype=np.int64), 1e6)
    for h in range(n_kv):
        _close(K[h], tn(H[:, offs_kv[h]:offs_kv[h] + d_h]), 1e-12, f"K head {h}")
        _close(V[h], H[:, offs_kv[::-1][h]:offs_kv[::-1][h] + d_h], 0, f"V head {h}")
    # at positions p: the normed slice rotated by p * theta^(-2i/d_h) in plane (i, i + d_h/2)
    pos = np.array([3, 4, 5, 6])
    q = O.q_project(H, WQ, ones, n_h, d_h, 1e-6, pos, 1e4)
    inv = 1e4 ** (-2.0 * np.arange(d_h // 2) / d_h)
    for h in (0, 5):
        x = tn(H[:, offs_q[h]:offs_q[h] + d_h])
        a, b = x[:, :d_h // 2], x[:, d_h // 2:]
        c, s = np.cos(pos[:, None] * inv), np.sin(pos[:, None] * inv)
        _close(q[h], np.concatenate([a * c - b * s, a * s + b * c], axis=1), 1e-12,
               f"Q head {h} roped")
    # the walkthrough's own split: [4, 512] viewed as [4, 8, 64], heads first
    x = _rand((n, d), 71)
    ref = torch.from_numpy(x).view(n, n_h, d_h).transpose(0, 1).numpy()
    _close(O.split_heads(x, n_h, d_h), ref, 0, "split_heads = view(n, n_h, d_h).transpose")


# ---------------------------------------------------------------------------
# Dual-stream K/V and the cache (walkthrough Steps 4.2-4.3, 7)
# ---------------------------------------------------------------------------

def pin_dual_stream_equals_cached_rounds(O):
    """One concatenated forward equals inject-then-block through the cache, over two rounds.

    Round 1: 3 context rows at 0-2, block at 3-6. The cache is cropped to 3, round 2
    injects 3 rows at 3-5 and runs a block at 6-9; a single forward over the 6 context
    rows gives the same output.
    """
    w, x = _walkthrough_inputs()
    C1 = O.ctx_project(x["hid"], x["W_fc"], x["g_h"], w.eps)
    H1 = x["H"]
    args = (x["W_Q"], x["W_K"], x["W_V"], x["g_q"], x["g_k"], w.n_h, w.n_kv, w.d_h, w.eps, w.theta)
    ref1, _, k1, v1 = O.draft_attention_forward(C1, H1, *args)
    cache = O.DraftKVCache(1, 1, w.n_kv, w.d_h)
    O.kv_inject(cache, 0, C1, [0, 3], x["W_K"], x["W_V"], x["g_k"], w.n_kv, w.d_h, w.eps, w.theta)
    out1 = O.block_attn(cache, 0, H1[None], *args)
    _close(out1[0], ref1, 1e-10, "round 1 output")
    _close(cache.k[0][0], k1, 1e-10, "cached K = KNorm(concat[C W_K; H W_K]) roped")
    _close(cache.v[0][0], v1, 1e-10, "cached V = concat[C W_V; H W_V]")
    O.cache_crop(cache, [3])
    C2 = _rand((3, w.d), 60)
    H2 = _rand((4, w.d), 61)
    O.kv_inject(cache, 0, C2, [0, 3], x["W_K"], x["W_V"], x["g_k"], w.n_kv, w.d_h, w.eps, w.theta)
    out2 = O.block_attn(cache, 0, H2[None], *args)
    ref2, _, _, _ = O.draft_attention_forward(np.concatenate([C1, C2]), H2, *args)
    _close(out2[0], ref2, 1e-10, "round 2 output")


def pin_cache_lengths_walkthrough(O):
    """Cache lengths 0 -> 3 -> 7 -> crop 3 -> 6 (walkthrough Step 7)."""
    g = _golden("cache_lengths_walkthrough.json")
    w, x = _walkthrough_inputs()
    cache = O.DraftKVCache(1, 1, w.n_kv, w.d_h)
    args = (x["W_Q"], x["W_K"], x["W_V"], x["g_q"], x["g_k"], w.n_h, w.n_kv, w.d_h, w.eps, w.theta)
    for st in g["steps"]:
        if st["op"] == "inject":
            C = _rand((st["rows"], w.d), 70)
            O.kv_inject(cache, 0, C, [0, st["rows"]], x["W_K"], x["W_V"], x["g_k"], w.n_kv,
                        w.d_h, w.eps, w.theta)
        elif st["op"] == "block_attn":
            O.block_attn(cache, 0, _rand((1, st["block_size"], w.d), 71), *args)
        else:
            O.cache_crop(cache, [st["to"]])
        assert int(cache.lens[0, 0]) == st["len_after"], st
    assert cache.errors == 0


def pin_crop_and_capacity_refusals(O):
    """Crop beyond the current length (or negative) and appends beyond capacity are refused."""
    cache = O.DraftKVCache(2, 2, 1, 2, capacity=5)
    K = np.zeros((1, 4, 2))
    assert cache.append(0, 0, K, K) and cache.append(1, 0, K, K)
    assert not cache.append(0, 0, K[:, :2], K[:, :2])
    assert cache.errors == 1
    cache.crop([5, 0])
    assert cache.lens.tolist() == [[4, 0], [4, 0]] and cache.errors == 3
    cache.crop([-1, 0])
    assert cache.lens.tolist() == [[4, 0], [4, 0]] and cache.errors == 5
    cache.crop([2, 0])
    assert cache.lens.tolist() == [[2, 0], [2, 0]]


def pin_acceptance(O):
    """acceptance_length: the walkthrough's example gives 2; a match after a miss does not count."""
    g = _golden("acceptance_walkthrough.json")
    assert O.acceptance_length(g["block_output_ids"], g["posterior"]) == g["acceptance_length"]
    assert g["start_before"] + g["acceptance_length"] + 1 == g["start_after"]
    assert O.acceptance_length([0, 5, 6, 7], [5, 9, 7, 0]) == 1
    assert O.acceptance_length([0, 5, 6, 7], [5, 6, 7, 0]) == 3
    assert O.acceptance_length([0, 5, 6, 7], [4, 6, 7, 0]) == 0


def pin_round_bookkeeping(O):
    """Step 6-7 state update on the walkthrough's example, plus its recurrence and edge cases."""
    g = _golden("acceptance_walkthrough.json")
    a, cu, ctx_next, anchor = O.round_bookkeeping([g["block_output_ids"]], [g["posterior"]],
                                                  [g["start_before"]])
    assert a == [g["acceptance_length"]]
    assert cu == [0, g["new_context_rows"]]
    assert ctx_next == [g["start_after"]]
    assert anchor == ["in"]                       # the target's correction becomes the anchor
    # all accepted: the bonus token after the block; none accepted: the target's first token
    a, cu, ctx_next, anchor = O.round_bookkeeping([[9, 1, 2, 3], [9, 1, 2, 3], [7]],
                                                  [[1, 2, 3, 4], [5, 2, 3, 4], [8]], [10, 20, 0])
    assert a == [3, 0, 0] and cu == [0, 4, 5, 6]
    assert ctx_next == [14, 21, 1] and anchor == [4, 5, 8]




def pin_o_proj_shapes_and_identity(O):
    """Step 4.5: [4, 8, 64] reshaped to [4, 512], projected to [4, 512]; W_O = I keeps the
    concatenated heads; head blocks of W_O select heads."""
    rng = np.random.default_rng(21)
    attn = rng.standard_normal((4, 8, 64)).reshape(4, 512)
    assert O.o_proj(attn, np.eye(512)).shape == (4, 512)
    np.testing.assert_allclose(O.o_proj(attn, np.eye(512)), attn, rtol=0, atol=0)
    W = np.zeros((64, 512))
    W[:, 3 * 64:4 * 64] = np.eye(64)                   # picks head 3
    np.testing.assert_allclose(O.o_proj(attn, W), attn[:, 192:256], rtol=0, atol=0)


def pin_silu_closed_forms(O):
    """silu(0) = 0, silu(x) -> x for large x, -> 0 for very negative x, silu(x) - silu(-x) = x."""
    x = np.linspace(-6, 6, 25)
    assert O.silu(np.zeros(3)).tolist() == [0.0, 0.0, 0.0]
    np.testing.assert_allclose(O.silu(x) - O.silu(-x), x, rtol=1e-13, atol=1e-13)
    assert abs(O.silu(40.0) - 40.0) < 1e-12 and abs(O.silu(-40.0)) < 1e-15
    np.testing.assert_allclose(O.silu(1.0), 1.0 / (1.0 + np.exp(-1.0)), rtol=1e-15)


def pin_mlp_brute_force(O):
    """SwiGLU MLP against a pure-Python triple loop, and its degenerate weights."""
    rng = np.random.default_rng(22)
    d, f, n = 6, 5, 3
    x = rng.standard_normal((n, d))
    Wg, Wu, Wd = rng.standard_normal((f, d)), rng.standard_normal((f, d)), rng.standard_normal((d, f))
    want = np.zeros((n, d))
    for r in range(n):
        h = []
        for j in range(f):
            g = sum(x[r, k] * Wg[j, k] for k in range(d))
            u = sum(x[r, k] * Wu[j, k] for k in range(d))
            h.append(g / (1.0 + np.exp(-g)) * u)
        for i in range(d):
            want[r, i] = sum(h[j] * Wd[i, j] for j in range(f))
    np.testing.assert_allclose(O.mlp(x, Wg, Wu, Wd), want, rtol=1e-12, atol=1e-12)
    assert not O.mlp(x, Wg, np.zeros_like(Wu), Wd).any()     # no up path -> nothing


def pin_layer_output_residuals(O):
    """Zero o_proj and zero MLP leave the residual stream; each path adds on top of it."""
    rng = np.random.default_rng(23)
    n, d, a, f = 3, 8, 8, 4
    x, att = rng.standard_normal((n, d)), rng.standard_normal((n, a))
    WO, Wg, Wu, Wd = (rng.standard_normal(s) for s in ((d, a), (f, d), (f, d), (d, f)))
    g = np.ones(d)
    np.testing.assert_allclose(O.layer_output(x, att, 0 * WO, g, Wg, Wu, 0 * Wd, 1e-6), x, atol=0)
    x1 = x + att @ WO.T
    np.testing.assert_allclose(O.layer_output(x, att, WO, g, Wg, Wu, 0 * Wd, 1e-6), x1, rtol=1e-13)
    nrm = x1 / np.sqrt((x1 ** 2).mean(-1, keepdims=True) + 1e-6)
    h = nrm @ Wg.T
    want = x1 + ((h / (1 + np.exp(-h))) * (nrm @ Wu.T)) @ Wd.T
    np.testing.assert_allclose(O.layer_output(x, att, WO, g, Wg, Wu, Wd, 1e-6), want, rtol=1e-12)


# ---------------------------------------------------------------------------
# fp8 (E4M3) cache storage
# ---------------------------------------------------------------------------

def _e4m3_sample():
    """float32 values inside the finite E4M3 range: every code value, every midpoint
    between neighbouring codes, and log-uniform random magnitudes, both signs."""
    pos = np.array(_E4M3_FROM_BITS, dtype=np.float64)
    mids = (pos[1:] + pos[:-1]) / 2
    rng = np.random.default_rng(41)
    rnd = np.exp2(rng.uniform(-12, np.log2(448.0), 4000))
    a = np.concatenate([pos, mids, rnd, [448.0]])
    a = np.concatenate([a, -a]).astype(np.float32)
    return a


# finite non-negative E4M3 values written out from the format (sign 0, exponent e with
# bias 7, mantissa m): subnormals m * 2^-9, normals (1 + m/8) * 2^(e-7), up to 448
_E4M3_FROM_BITS = [m * 2.0 ** -9 for m in range(8)] + \
    [(1 + m / 8) * 2.0 ** (e - 7) for e in range(1, 16) for m in range(8) if not (e == 15 and m == 7)]


def pin_e4m3_matches_torch(O):
    """Round-trip through the quantiser = torch's float8_e4m3fn conversion (in range)."""
    a = _e4m3_sample()
    want = torch.from_numpy(a).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.e4m3_dequantize(O.e4m3_quantize(a.astype(np.float64)))
    np.testing.assert_array_equal(got, want)


def pin_e4m3_codes_closed_form(O):
    """Codes fixed by the format: ones, extremes, subnormal ties, saturation, NaN."""
    cases = {1.0: 0x38, -1.0: 0xB8, 448.0: 0x7E, 500.0: 0x7E, -1e6: 0xFE, 2.0 ** -6: 0x08,
             2.0 ** -9: 0x01, 7 * 2.0 ** -9: 0x07, 1.5 * 2.0 ** -9: 0x02, 2.0 ** -10: 0x00,
             1.0625: 0x38, 1.1875: 0x3A, 0.0: 0x00, 240.0: 0x77}
    got = O.e4m3_quantize(np.array(list(cases), dtype=np.float64))
    assert got.tolist() == list(cases.values()), got.tolist()
    assert O.e4m3_quantize(np.array([np.nan]))[0] & 0x7F == 0x7F
    vals = O.e4m3_dequantize(np.arange(256))
    assert np.isnan(vals[0x7F]) and np.isnan(vals[0xFF])
    np.testing.assert_array_equal(vals[:0x7F], _E4M3_FROM_BITS)
    np.testing.assert_array_equal(vals[0x80:0xFF], -np.array(_E4M3_FROM_BITS))
    # every finite code is a fixed point of value -> code
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    np.testing.assert_array_equal(O.e4m3_quantize(O.e4m3_dequantize(codes)), codes)


def pin_e4m3_error_bound(O):
    """|x - value(code(x))| <= half the code spacing at x (2^-4 relative for normals)."""
    rng = np.random.default_rng(43)
    x = np.exp2(rng.uniform(-11, 8.8, 20000)) * rng.choice([-1, 1], 20000)
    err = np.abs(x - O.e4m3_dequantize(O.e4m3_quantize(x)))
    e = np.floor(np.log2(np.abs(x)))
    spacing = np.where(e < -6, 2.0 ** -9, 2.0 ** (np.minimum(e, 8) - 3))
    assert np.all(err <= spacing / 2 + 1e-300), float((err / spacing).max())


def pin_fp8_cache_scale(O):
    """A power-of-two scale leaves normal-range rows unchanged (exponent shift only), and
    the cache holds scale * value: scales (2, 1/2) store what scales (1, 1) store."""
    rng = np.random.default_rng(47)
    K = np.exp2(rng.uniform(-3, 5, (2, 9, 8))) * rng.choice([-1, 1], (2, 9, 8))
    V = np.exp2(rng.uniform(-3, 5, (2, 9, 8))) * rng.choice([-1, 1], (2, 9, 8))
    c1 = O.DraftKVCache(1, 1, 2, 8, fp8_scales=([1.0], [1.0]))
    c2 = O.DraftKVCache(1, 1, 2, 8, fp8_scales=([2.0], [0.5]))
    c1.append(0, 0, K, V)
    c2.append(0, 0, K, V)
    np.testing.assert_array_equal(c2.k[0][0], c1.k[0][0])
    np.testing.assert_array_equal(c2.v[0][0], c1.v[0][0])
    np.testing.assert_array_equal(c2.kraw[0][0], K)
    # relative error of a stored element is at most 2^-4 in the normal range
    assert np.all(np.abs(c1.k[0][0] - K) <= np.abs(K) * 2.0 ** -4)
    # a non-power-of-two scale: stored = s * value(code(x / s)), and crop cuts the raw rows too
    c3 = O.DraftKVCache(1, 1, 2, 8, fp8_scales=([0.3], [3.0]))
    c3.append(0, 0, K, V)
    q = O.e4m3_quantize(K / 0.3)
    np.testing.assert_allclose(c3.k[0][0], 0.3 * O.e4m3_dequantize(q), rtol=1e-15)
    c3.crop([4])
    assert c3.k[0][0].shape[1] == c3.kraw[0][0].shape[1] == c3.vraw[0][0].shape[1] == 4


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
