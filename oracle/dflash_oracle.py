"""Float64 CPU oracle for the DFlash KV-injection draft attention step.

TEST INFRASTRUCTURE. Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module. The library never
does, and this module imports nothing from the library: the two share no code.

Every function restates one passage of the source pages in plain NumPy float64,
in the order and notation the pages use:

* "DFlash KV Injection Walkthrough" (Steps 1-7), the authority on the path;
* "DFlash source guide (II): Qwen3DFlashAttention" (parts 1-5, the non-causal
  design note and the MLX comparison table);
* "KV Cache + Speculative Decoding Interview Cheat Sheet" (section 6.3 for the
  GQA head mapping, the MLA ``_rope`` helper for the inverse-frequency formula).

Weights are held in the ``nn.Linear`` layout ``[out_features, in_features]``
(the walkthrough's modules are ``nn.Linear``), so a projection is ``x @ W.T``.
The walkthrough's "W_fc in R^{1536x512}" is the transpose of that array.

Readings taken where the pages are silent or ambiguous (each is listed in the
design notes): RMSNorm without mean-centring, eps inside the square root and
gamma applied last; q/k-norm gamma of shape [d_h] shared by all heads;
rotate-half RoPE pairing (i, i + d_h/2); inverse frequency theta^(-2i/d_h);
cache slot index = absolute position; sliding window "key j is visible to a
query at position p iff p - j < W" with no upper bound.

Parity status: all functions are pinned by tests/test_oracle_pins.py against
closed forms, library routines, brute force and the integer examples the
walkthrough prints. Two readings stay "parity unpinned" by the pages: the
rotate-half pairing (the pages' invariants hold for any pairing) and the edge
keys of the sliding window. The element values of the walkthrough example are
unpinned too: the page prints shapes only. The fp8 cache format (E4M3, one scale
per layer for K and for V) is a reading of a passage that names fp8 without
fixing a format; the quantiser itself is pinned against a library conversion and
closed-form codes.
"""

from __future__ import annotations

import math

import numpy as np

F64 = np.float64


# ---------------------------------------------------------------------------
# Normalisation and rotary position embedding
# ---------------------------------------------------------------------------

def rms_norm(x, gamma, eps):
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * gamma.

    DFlash KV Injection Walkthrough, Step 2 (C = RMSNorm(...)) and Step 4.1 /
    4.2 (QNorm, KNorm); DFlash source guide (II), part 1 (Qwen3RMSNorm over
    head_dim with eps = rms_norm_eps).
    """
    x = np.asarray(x, dtype=F64)
    mean_sq = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(mean_sq + eps) * np.asarray(gamma, dtype=F64)


def rope_inv_freq(d_h, theta):
    """Inverse frequencies theta^(-2i/d_h), i = 0 .. d_h/2 - 1.

    KV Cache + Speculative Decoding Interview Cheat Sheet, section 6.3 (the
    ``_rope`` helper: base ** (-2 i / D)).
    """
    i = np.arange(d_h // 2, dtype=F64)
    return np.asarray(theta, dtype=F64) ** (-2.0 * i / d_h)


def rope_cos_sin(positions, d_h, theta):
    """cos/sin tables [n, d_h] for the given absolute positions.

    DFlash KV Injection Walkthrough, Step 4.3: cos, sin are [window, d_h]
    (7 x 64 in the example); each angle pos * inv_freq_i appears in both
    halves of the head dimension, matching ``rotate_half``.
    """
    pos = np.asarray(positions, dtype=F64)
    ang = pos[:, None] * rope_inv_freq(d_h, theta)[None, :]
    ang = np.concatenate([ang, ang], axis=-1)
    return np.cos(ang), np.sin(ang)


def rotate_half(x):
    """rotate_half([x1; x2]) = [-x2; x1] over the last axis (halves of d_h).

    DFlash KV Injection Walkthrough, Step 4.3 (``rotate_half`` in
    ``apply_rotary_pos_emb``).
    """
    x = np.asarray(x, dtype=F64)
    h = x.shape[-1] // 2
    return np.concatenate([-x[..., h:], x[..., :h]], axis=-1)


def apply_rope(x, cos, sin):
    """x * cos + rotate_half(x) * sin (rows of x align with rows of cos/sin).

    DFlash KV Injection Walkthrough, Step 4.3.
    """
    x = np.asarray(x, dtype=F64)
    return x * cos + rotate_half(x) * sin


# ---------------------------------------------------------------------------
# Context signal (Steps 1-2)
# ---------------------------------------------------------------------------

def extract_context_feature(hidden_states):
    """Concatenate the selected target layers on the feature axis.

    DFlash KV Injection Walkthrough, Step 1: target_hidden_raw[i] =
    [h^(3)_i ; h^(7)_i ; h^(11)_i], in ascending layer order.
    ``hidden_states`` is the list of k arrays [n, d].
    """
    return np.concatenate([np.asarray(h, dtype=F64) for h in hidden_states], axis=-1)


def ctx_project(hidden_states, W_fc, gamma_h, eps):
    """C = hidden_norm(fc(target_hidden_raw)), C in R^{n x d}.

    DFlash KV Injection Walkthrough, Step 2. ``W_fc`` is [d, k*d]
    (nn.Linear layout, no bias).
    """
    raw = extract_context_feature(hidden_states)
    return rms_norm(raw @ np.asarray(W_fc, dtype=F64).T, gamma_h, eps)


# ---------------------------------------------------------------------------
# Projections (Steps 4.1-4.3)
# ---------------------------------------------------------------------------

def split_heads(x, n_heads, d_h):
    """[n, n_heads*d_h] -> [n_heads, n, d_h] (view + transpose of Step 4.1)."""
    n = x.shape[0]
    return np.asarray(x, dtype=F64).reshape(n, n_heads, d_h).transpose(1, 0, 2)


def q_project(H, W_Q, gamma_q, n_h, d_h, eps, positions, theta):
    """Q = RoPE(QNorm(H W_Q)) at the block's positions -> [n_h, L_q, d_h].

    DFlash KV Injection Walkthrough, Step 4.1 (projection, per-head QNorm)
    and Step 4.3 (Q takes the last q_len rows of the window's cos/sin, i.e.
    the block's own absolute positions).
    """
    q = split_heads(np.asarray(H, dtype=F64) @ np.asarray(W_Q, dtype=F64).T, n_h, d_h)
    q = rms_norm(q, gamma_q, eps)
    cos, sin = rope_cos_sin(positions, d_h, theta)
    return apply_rope(q, cos[None], sin[None])


def kv_project(X, W_K, W_V, gamma_k, n_kv, d_h, eps, positions, theta):
    """K = RoPE(KNorm(X W_K)), V = X W_V at the rows' absolute positions.

    DFlash KV Injection Walkthrough, Step 4.2 (the same k_proj / v_proj
    weights serve context rows C and block rows H; KNorm per head; V is not
    normalised) and Step 4.3 (K uses the whole window's cos/sin, so each row
    is rotated at its true position). Returns K, V as [n_kv, n, d_h].
    """
    X = np.asarray(X, dtype=F64)
    k = split_heads(X @ np.asarray(W_K, dtype=F64).T, n_kv, d_h)
    v = split_heads(X @ np.asarray(W_V, dtype=F64).T, n_kv, d_h)
    k = rms_norm(k, gamma_k, eps)
    cos, sin = rope_cos_sin(positions, d_h, theta)
    return apply_rope(k, cos[None], sin[None]), v


# ---------------------------------------------------------------------------
# Attention (Step 4.4)
# ---------------------------------------------------------------------------

def visible_mask(q_pos, k_pos, window):
    """Boolean [L_q, L_k]: which keys each query may attend to.

    Non-causal: with no window every key is visible (DFlash KV Injection
    Walkthrough, Step 4.4: is_causal = False, a fully connected 4 x 7 matrix;
    DFlash source guide (II), non-causal design note: attention_mask None).
    With a sliding window W > 0 (DFlash source guide (II), part 5: only
    sliding_attention layers) key j is visible to a query at position p iff
    p - j < W; keys ahead of the query stay visible (the reading taken).
    """
    q_pos = np.asarray(q_pos, dtype=np.int64)
    k_pos = np.asarray(k_pos, dtype=np.int64)
    if window is None or window <= 0:
        return np.ones((q_pos.size, k_pos.size), dtype=bool)
    return (q_pos[:, None] - k_pos[None, :]) < window


def attention_weights(Q, K, q_pos, k_pos, scaling, window=0):
    """A = softmax_j(q'_i . k'_j * scaling) per query head -> [n_h, L_q, L_k].

    DFlash KV Injection Walkthrough, Step 4.4 (scaling d_h^-0.5, softmax over
    every visible key). GQA: query head h reads KV head floor(h / G) with
    G = n_h / n_kv (DFlash source guide (II), part 1: num_key_value_groups;
    Interview Cheat Sheet, section 6.3: repeat_interleave over the head axis).
    """
    Q = np.asarray(Q, dtype=F64)
    K = np.asarray(K, dtype=F64)
    n_h = Q.shape[0]
    n_kv = K.shape[0]
    G = n_h // n_kv
    vis = visible_mask(q_pos, k_pos, window)
    A = np.empty((n_h, Q.shape[1], K.shape[1]), dtype=F64)
    for h in range(n_h):
        S = (Q[h] @ K[h // G].T) * scaling
        S = np.where(vis, S, -np.inf)
        S = S - S.max(axis=-1, keepdims=True)
        E = np.exp(S)
        A[h] = E / E.sum(axis=-1, keepdims=True)
    return A


def attention(Q, K, V, q_pos, k_pos, scaling, window=0):
    """out_i = sum_j A_ij v_j, heads concatenated -> [L_q, n_h * d_h].

    DFlash KV Injection Walkthrough, Step 4.4 (out_i) and Step 4.5 (the
    reshape to [L_q, n_h * d_h] that feeds o_proj).
    """
    A = attention_weights(Q, K, q_pos, k_pos, scaling, window)
    V = np.asarray(V, dtype=F64)
    n_h, L_q, _ = A.shape
    G = n_h // V.shape[0]
    out = np.stack([A[h] @ V[h // G] for h in range(n_h)], axis=0)  # [n_h, L_q, d_h]
    return out.transpose(1, 0, 2).reshape(L_q, -1)


def draft_attention_forward(C, H, W_Q, W_K, W_V, gamma_q, gamma_k, n_h, n_kv, d_h,
                            eps, theta, ctx_start=0, scaling=None, window=0):
    """One Qwen3DFlashAttention forward without a cache, as the walkthrough writes it.

    DFlash KV Injection Walkthrough, Steps 4.1-4.4: K/V are the projections of
    concat[C; H] with KNorm applied to the concatenation, cos/sin cover the
    whole window [ctx_start, ctx_start + L_c + L_q), Q takes the last q_len
    rows of the window and K all of them. Returns (out [L_q, n_h*d_h], Q, K, V).
    """
    C = np.asarray(C, dtype=F64)
    H = np.asarray(H, dtype=F64)
    L_c, L_q = C.shape[0], H.shape[0]
    window_pos = ctx_start + np.arange(L_c + L_q)
    cos, sin = rope_cos_sin(window_pos, d_h, theta)
    W_Q, W_K, W_V = (np.asarray(w, dtype=F64) for w in (W_Q, W_K, W_V))
    q = rms_norm(split_heads(H @ W_Q.T, n_h, d_h), gamma_q, eps)
    k = split_heads(np.concatenate([C @ W_K.T, H @ W_K.T], axis=0), n_kv, d_h)
    v = split_heads(np.concatenate([C @ W_V.T, H @ W_V.T], axis=0), n_kv, d_h)
    k = rms_norm(k, gamma_k, eps)
    q = apply_rope(q, cos[None, -L_q:], sin[None, -L_q:])
    k = apply_rope(k, cos[None], sin[None])
    if scaling is None:
        scaling = d_h ** -0.5
    out = attention(q, k, v, window_pos[-L_q:], window_pos, scaling, window)
    return out, q, k, v


# ---------------------------------------------------------------------------
# Output projection and the rest of the draft layer (Steps 4.5, 5)
# ---------------------------------------------------------------------------

def o_proj(attn_out, W_O):
    """Attn_out = concat[head_1 .. head_n_h] . W_O: the heads, concatenated per row in
    head order ([rows][n_h * d_h], the layout Step 4.5 reshapes to), projected back to
    the model width d. DFlash KV Injection Walkthrough, Step 4.5 (nn.Linear, no bias)."""
    return np.asarray(attn_out, F64) @ np.asarray(W_O, F64).T


def silu(x):
    """x * sigmoid(x), the gate activation of the Qwen3 MLP (a reading: the pages name the
    decoder layers but do not print their MLP)."""
    x = np.asarray(x, F64)
    return x / (1.0 + np.exp(-x))


def mlp(x, W_gate, W_up, W_down):
    """The decoder layer's feed-forward part, read as the Qwen3 SwiGLU MLP:
    down( silu(x gate^T) * (x up^T) ). Weights [d_ff][d], [d_ff][d], [d][d_ff]."""
    x = np.asarray(x, F64)
    g = x @ np.asarray(W_gate, F64).T
    u = x @ np.asarray(W_up, F64).T
    return (silu(g) * u) @ np.asarray(W_down, F64).T


def layer_output(x, attn_out, W_O, gamma_post, W_gate, W_up, W_down, eps):
    """The rest of a draft decoder layer after its attention, read as the Qwen3 pre-norm
    residual layer (Step 5 names the two decoder layers and the final RMSNorm only):
        x1  = x + o_proj(attn_out)                       (Step 4.5, then the residual)
        out = x1 + mlp(RMSNorm_post(x1))
    x is the layer's residual input [rows][d] (the rows of the block)."""
    x1 = np.asarray(x, F64) + o_proj(attn_out, W_O)
    return x1 + mlp(rms_norm(x1, gamma_post, eps), W_gate, W_up, W_down)


# ---------------------------------------------------------------------------
# fp8 (E4M3) cache storage
# ---------------------------------------------------------------------------
# KV Cache + Speculative Decoding Interview Cheat Sheet, section 2.1 (an fp8 cache
# element takes one byte) and section 4.5 (KV quantisation, FP8 among the routes).
# The pages fix neither the fp8 format nor the scaling, so the reading taken is the
# plainest one: the E4M3 format without infinities (1 sign bit, 4 exponent bits with
# bias 7, 3 mantissa bits; exponent and mantissa all ones is NaN, so the largest
# finite value is 448), one scale per layer for K and one for V, the stored code is
# x / scale rounded to the nearest finite value (ties to the even code, magnitudes
# beyond 448 saturate to 448), and a cached element reads back as scale * value.

def e4m3_value(code):
    """Value of one E4M3 code (0..255), from its bit fields."""
    code = int(code)
    sign = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 0xF, code & 0x7
    if e == 15 and m == 7:
        return math.nan
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** (1 - 7)        # subnormal
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


# the 127 finite non-negative values, code 0 .. 126 (increasing with the code)
_E4M3_POS = np.array([e4m3_value(c) for c in range(127)], dtype=F64)


def e4m3_quantize(x):
    """Codes (uint8) of x: nearest finite E4M3 value, ties to the even code, saturating."""
    x = np.asarray(x, dtype=F64)
    a = np.abs(x).ravel()
    hi = np.clip(np.searchsorted(_E4M3_POS, a), 1, 126)   # first value >= a (clamped)
    lo = hi - 1
    d_lo, d_hi = a - _E4M3_POS[lo], _E4M3_POS[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a >= _E4M3_POS[126], 126, code)          # saturate at 448
    code = code | np.where(np.signbit(x.ravel()), 0x80, 0)
    code = np.where(np.isnan(a), 0x7F, code)
    return code.astype(np.uint8).reshape(x.shape)


def e4m3_dequantize(codes):
    """Values of E4M3 codes."""
    table = np.array([e4m3_value(c) for c in range(256)], dtype=F64)
    return table[np.asarray(codes, dtype=np.int64)]


def fp8_store(x, scale):
    """What an fp8 cache holds for x: scale * value(code(x / scale))."""
    return scale * e4m3_dequantize(e4m3_quantize(np.asarray(x, dtype=F64) / scale))


# ---------------------------------------------------------------------------
# The draft KV cache and the four calls of the step (Steps 4.2-4.4, 7)
# ---------------------------------------------------------------------------

class DraftKVCache:
    """Per-layer, per-sequence draft KV cache with lengths.

    DFlash source guide (II), part 4: ``update`` writes this round's context
    and block K/V; ``crop(start)`` keeps only the accepted prefix. DFlash KV
    Injection Walkthrough, Step 7: the cache grows round by round. Slot j of
    a sequence holds the row at absolute position j. ``capacity`` (optional)
    mirrors a fixed-size device cache: an append beyond it is refused.
    ``fp8_scales`` (optional) = (k_scales, v_scales), one per layer: the cache
    then stores rows as an E4M3 cache does (``fp8_store``); ``kraw`` / ``vraw``
    keep the rows before quantisation.
    """

    def __init__(self, n_layers, batch, n_kv, d_h, capacity=None, fp8_scales=None):
        self.n_layers, self.batch, self.n_kv, self.d_h = n_layers, batch, n_kv, d_h
        self.capacity = capacity
        self.fp8_scales = fp8_scales
        self.k = [[np.zeros((n_kv, 0, d_h)) for _ in range(batch)] for _ in range(n_layers)]
        self.v = [[np.zeros((n_kv, 0, d_h)) for _ in range(batch)] for _ in range(n_layers)]
        self.kraw = [[np.zeros((n_kv, 0, d_h)) for _ in range(batch)] for _ in range(n_layers)]
        self.vraw = [[np.zeros((n_kv, 0, d_h)) for _ in range(batch)] for _ in range(n_layers)]
        self.errors = 0

    def _stored(self, layer, K, V):
        K, V = np.asarray(K, dtype=F64), np.asarray(V, dtype=F64)
        if self.fp8_scales is None:
            return K, V
        return (fp8_store(K, self.fp8_scales[0][layer]), fp8_store(V, self.fp8_scales[1][layer]))

    def length(self, layer, b):
        return self.k[layer][b].shape[1]

    @property
    def lens(self):
        return np.array([[self.length(l, b) for b in range(self.batch)]
                         for l in range(self.n_layers)], dtype=np.int64)

    def set_rows(self, layer, b, K, V):
        """Replace the cached rows of one sequence (used to seed a pre-filled cache)."""
        self.kraw[layer][b] = np.asarray(K, dtype=F64).copy()
        self.vraw[layer][b] = np.asarray(V, dtype=F64).copy()
        self.k[layer][b], self.v[layer][b] = self._stored(layer, K, V)

    def append(self, layer, b, K, V):
        """Append rows [n_kv, n, d_h]; refused (error counted) beyond capacity."""
        n = K.shape[1]
        if self.capacity is not None and self.length(layer, b) + n > self.capacity:
            self.errors += 1
            return False
        Ks, Vs = self._stored(layer, K, V)
        self.k[layer][b] = np.concatenate([self.k[layer][b], Ks], axis=1)
        self.v[layer][b] = np.concatenate([self.v[layer][b], Vs], axis=1)
        self.kraw[layer][b] = np.concatenate([self.kraw[layer][b], K], axis=1)
        self.vraw[layer][b] = np.concatenate([self.vraw[layer][b], V], axis=1)
        return True

    def crop(self, new_lens):
        """Keep rows [0, new_lens[b]) of every layer (crop(start)).

        A target length beyond the current length, or negative, is refused
        for that layer and sequence and counted as an error (the pages are
        silent on this case; refusing is the reading taken).
        """
        for l in range(self.n_layers):
            for b in range(self.batch):
                n = int(new_lens[b])
                if n < 0 or n > self.length(l, b):
                    self.errors += 1
                    continue
                for rows in (self.k, self.v, self.kraw, self.vraw):
                    rows[l][b] = rows[l][b][:, :n]


def kv_inject(cache, layer, C, cu_rows, W_K, W_V, gamma_k, n_kv, d_h, eps, theta):
    """Append this round's context K/V for every sequence of one draft layer.

    DFlash KV Injection Walkthrough, Step 4.2 (C W_K, C W_V with KNorm),
    Step 4.3 (K at its true absolute positions) and Step 7 (the accepted
    rows' features enter the cache as incremental context). Rows
    cu_rows[b] .. cu_rows[b+1]-1 of C belong to sequence b and land at
    positions len_b .. len_b + n_b - 1.
    """
    C = np.asarray(C, dtype=F64)
    for b in range(cache.batch):
        rows = C[cu_rows[b]:cu_rows[b + 1]]
        if rows.shape[0] == 0:
            continue
        pos = cache.length(layer, b) + np.arange(rows.shape[0])
        K, V = kv_project(rows, W_K, W_V, gamma_k, n_kv, d_h, eps, pos, theta)
        cache.append(layer, b, K, V)


def block_attn(cache, layer, H, W_Q, W_K, W_V, gamma_q, gamma_k, n_h, n_kv, d_h,
               eps, theta, window=0, scaling=None):
    """Block queries over [cached context KV || block KV]; appends the block KV.

    DFlash KV Injection Walkthrough, Steps 4.1-4.4: the block occupies the
    positions right after the cache, Q and block K are roped there, and every
    block query attends (non-causally) to every cached row and every block
    row. DFlash source guide (II), part 4: the block K/V are written into the
    cache by ``update`` (and later removed by crop). Returns out
    [B, bs, n_h*d_h]; sequences whose append is refused get NaN rows.
    """
    H = np.asarray(H, dtype=F64)
    B, bs, _ = H.shape
    if scaling is None:
        scaling = d_h ** -0.5
    out = np.full((B, bs, n_h * d_h), np.nan)
    for b in range(B):
        start = cache.length(layer, b)
        pos = start + np.arange(bs)
        Q = q_project(H[b], W_Q, gamma_q, n_h, d_h, eps, pos, theta)
        Kb, Vb = kv_project(H[b], W_K, W_V, gamma_k, n_kv, d_h, eps, pos, theta)
        if not cache.append(layer, b, Kb, Vb):
            continue
        k_pos = np.arange(cache.length(layer, b))
        out[b] = attention(Q, cache.k[layer][b], cache.v[layer][b], pos, k_pos,
                           scaling, window)
    return out


def cache_crop(cache, new_lens):
    """crop(start) on every layer. DFlash source guide (II), part 4."""
    cache.crop(new_lens)


# ---------------------------------------------------------------------------
# Acceptance bookkeeping (Step 6)
# ---------------------------------------------------------------------------

def acceptance_length(block_ids, posterior):
    """Accepted-prefix length of one block.

    DFlash KV Injection Walkthrough, Step 6: match = (block[1:] ==
    posterior[:-1]); the accepted length is the number of leading matches
    (cumulative product, then sum).
    """
    match = [int(a == b) for a, b in zip(list(block_ids)[1:], list(posterior)[:-1])]
    n = 0
    for m in match:
        if not m:
            break
        n += 1
    return n


def round_bookkeeping(block_ids, posterior, ctx_len):
    """Acceptance and the next round's state for every sequence.

    DFlash KV Injection Walkthrough, Step 6 (accepted length a = leading matches of
    block[1:] against posterior[:-1]) and Step 7 (start += a + 1; the next round injects
    the a + 1 context rows of the anchor and the accepted tokens; the target's token after
    the accepted prefix becomes the next block's anchor).
      block_ids, posterior  [B][bs] token ids
      ctx_len               [B] draft cache length the round started the block at
    Returns (a [B], next_cu_rows [B + 1], ctx_next [B], next_anchor [B]).
    """
    B = len(block_ids)
    a = [acceptance_length(block_ids[b], posterior[b]) for b in range(B)]
    counts = [x + 1 for x in a]
    cu = [0]
    for c in counts:
        cu.append(cu[-1] + c)
    ctx_next = [int(ctx_len[b]) + counts[b] for b in range(B)]
    anchor = [posterior[b][a[b]] for b in range(B)]
    return a, cu, ctx_next, anchor
