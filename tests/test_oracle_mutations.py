"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins catch each one."""
import numpy as np
import pytest

import oracle_pins
from oracle import dflash_oracle as O

F64 = np.float64


def _rms_no_eps(x, gamma, eps):
    x = np.asarray(x, F64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True)) * gamma


def _rms_centred(x, gamma, eps):
    x = np.asarray(x, F64)
    x = x - x.mean(axis=-1, keepdims=True)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * gamma


def _rms_no_gamma(x, gamma, eps):
    x = np.asarray(x, F64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def _rotate_half_wrong_sign(x):
    x = np.asarray(x, F64)
    h = x.shape[-1] // 2
    return np.concatenate([x[..., h:], -x[..., :h]], axis=-1)


def _inv_freq_wrong(d_h, theta):
    return np.asarray(theta, F64) ** (-np.arange(d_h // 2, dtype=F64) / d_h)


def _cos_sin_interleaved(positions, d_h, theta):
    ang = np.asarray(positions, F64)[:, None] * O.rope_inv_freq(d_h, theta)[None, :]
    ang = np.repeat(ang, 2, axis=-1)
    return np.cos(ang), np.sin(ang)


def _attn_weights_mod_mapping(Q, K, q_pos, k_pos, scaling, window=0):
    n_kv = K.shape[0]
    Kp = np.stack([K[h % n_kv] for h in range(Q.shape[0])])
    return _ORIG["attention_weights"](Q, Kp, q_pos, k_pos, scaling, window)


def _attention_mod_mapping(Q, K, V, q_pos, k_pos, scaling, window=0):
    n_kv = K.shape[0]
    Kp = np.stack([K[h % n_kv] for h in range(Q.shape[0])])
    Vp = np.stack([V[h % n_kv] for h in range(Q.shape[0])])
    return _ORIG["attention"](Q, Kp, Vp, q_pos, k_pos, scaling, window)


def _visible_causal(q_pos, k_pos, window):
    q_pos = np.asarray(q_pos)
    k_pos = np.asarray(k_pos)
    return q_pos[:, None] >= k_pos[None, :]


def _visible_window_inclusive(q_pos, k_pos, window):
    q_pos = np.asarray(q_pos)
    k_pos = np.asarray(k_pos)
    if not window:
        return np.ones((q_pos.size, k_pos.size), bool)
    return (q_pos[:, None] - k_pos[None, :]) <= window


def _attention_no_scaling(Q, K, V, q_pos, k_pos, scaling, window=0):
    return _ORIG["attention"](Q, K, V, q_pos, k_pos, 1.0, window)


def _concat_reversed(hidden_states):
    return np.concatenate([np.asarray(h, F64) for h in hidden_states[::-1]], axis=-1)


def _q_project_untransposed(H, W_Q, gamma_q, n_h, d_h, eps, positions, theta):
    return _ORIG["q_project"](H, np.asarray(W_Q).T, gamma_q, n_h, d_h, eps, positions, theta)


def _q_project_positions_from_zero(H, W_Q, gamma_q, n_h, d_h, eps, positions, theta):
    return _ORIG["q_project"](H, W_Q, gamma_q, n_h, d_h, eps, np.arange(len(positions)), theta)


def _kv_project_norms_v(X, W_K, W_V, gamma_k, n_kv, d_h, eps, positions, theta):
    K, V = _ORIG["kv_project"](X, W_K, W_V, gamma_k, n_kv, d_h, eps, positions, theta)
    return K, O.rms_norm(V, gamma_k, eps)


def _kv_project_no_rope(X, W_K, W_V, gamma_k, n_kv, d_h, eps, positions, theta):
    return _ORIG["kv_project"](X, W_K, W_V, gamma_k, n_kv, d_h, eps, np.zeros(len(positions)),
                               theta)


def _acceptance_sum(block_ids, posterior):
    return sum(int(a == b) for a, b in zip(list(block_ids)[1:], list(posterior)[:-1]))


def _bookkeeping_no_anchor_row(block_ids, posterior, ctx_len):
    a, cu, ctx_next, anchor = _ORIG["round_bookkeeping"](block_ids, posterior, ctx_len)
    cu2 = [0]
    for x in a:                     # injects only the accepted tokens, not the anchor row
        cu2.append(cu2[-1] + x)
    return a, cu2, [c - 1 for c in ctx_next], anchor


def _bookkeeping_anchor_late(block_ids, posterior, ctx_len):
    a, cu, ctx_next, anchor = _ORIG["round_bookkeeping"](block_ids, posterior, ctx_len)
    return a, cu, ctx_next, [posterior[b][min(a[b] + 1, len(posterior[b]) - 1)]
                             for b in range(len(a))]


def _o_proj_untransposed(attn_out, W_O):
    return np.asarray(attn_out, np.float64) @ np.asarray(W_O, np.float64)


def _mlp_silu_on_up(x, W_gate, W_up, W_down):
    x = np.asarray(x, np.float64)
    return ((x @ np.asarray(W_gate).T) * O.silu(x @ np.asarray(W_up).T)) @ np.asarray(W_down).T


def _layer_norm_before_residual(x, attn_out, W_O, gamma_post, W_gate, W_up, W_down, eps):
    x1 = np.asarray(x, np.float64) + O.o_proj(attn_out, W_O)
    return x1 + O.mlp(O.rms_norm(x, gamma_post, eps), W_gate, W_up, W_down)


def _e4m3_ties_away(x):
    x = np.asarray(x, np.float64)
    codes = _ORIG["e4m3_quantize"](x)
    vals = O.e4m3_dequantize(codes)
    up = _ORIG["e4m3_quantize"](np.nextafter(np.abs(x), np.inf) * np.sign(x))
    tie = np.abs(np.abs(x) - np.abs(vals)) == np.abs(np.abs(O.e4m3_dequantize(up)) - np.abs(x))
    return np.where(tie & (up != codes), up, codes).astype(np.uint8)


def _e4m3_truncates(x):
    x = np.asarray(x, np.float64)
    codes = _ORIG["e4m3_quantize"](x)
    over = np.abs(O.e4m3_dequantize(codes)) > np.abs(x)
    return np.where(over & ((codes & 0x7F) > 0), codes - 1, codes).astype(np.uint8)


def _e4m3_no_saturation(x):
    x = np.asarray(x, np.float64)
    codes = _ORIG["e4m3_quantize"](x)
    return np.where(np.abs(x) > 448.0, 0x7F, codes).astype(np.uint8)


def _e4m3_bias_8(code):
    v = _ORIG["e4m3_value"](code)
    return v / 2.0


def _split_heads_strided(x, n_heads, d_h):
    n = x.shape[0]
    return np.asarray(x, F64).reshape(n, d_h, n_heads).transpose(2, 0, 1)


def _split_heads_reversed(x, n_heads, d_h):
    n = x.shape[0]
    return np.asarray(x, F64).reshape(n, n_heads, d_h).transpose(1, 0, 2)[::-1]


def _fp8_store_drops_scale(x, scale):
    return O.e4m3_dequantize(O.e4m3_quantize(np.asarray(x, np.float64) / scale))


_ORIG = {n: getattr(O, n) for n in ("e4m3_quantize", "e4m3_value", "attention_weights", "attention", "q_project", "kv_project",
                                    "round_bookkeeping")}

MUTATIONS = {
    "rmsnorm_drops_eps": ("rms_norm", _rms_no_eps),
    "rmsnorm_mean_centred": ("rms_norm", _rms_centred),
    "rmsnorm_drops_gamma": ("rms_norm", _rms_no_gamma),
    "rope_rotate_half_sign": ("rotate_half", _rotate_half_wrong_sign),
    "rope_inv_freq_exponent": ("rope_inv_freq", _inv_freq_wrong),
    "rope_interleaved_pairs": ("rope_cos_sin", _cos_sin_interleaved),
    "gqa_modulo_mapping_weights": ("attention_weights", _attn_weights_mod_mapping),
    "gqa_modulo_mapping": ("attention", _attention_mod_mapping),
    "causal_mask": ("visible_mask", _visible_causal),
    "window_inclusive_edge": ("visible_mask", _visible_window_inclusive),
    "attention_no_scaling": ("attention", _attention_no_scaling),
    "concat_order_reversed": ("extract_context_feature", _concat_reversed),
    "q_weight_untransposed": ("q_project", _q_project_untransposed),
    "q_positions_from_zero": ("q_project", _q_project_positions_from_zero),
    "v_normalised": ("kv_project", _kv_project_norms_v),
    "k_not_roped": ("kv_project", _kv_project_no_rope),
    "acceptance_counts_all_matches": ("acceptance_length", _acceptance_sum),
    "next_round_drops_anchor_row": ("round_bookkeeping", _bookkeeping_no_anchor_row),
    "next_anchor_one_late": ("round_bookkeeping", _bookkeeping_anchor_late),
    "o_proj_untransposed": ("o_proj", _o_proj_untransposed),
    "mlp_silu_on_up_branch": ("mlp", _mlp_silu_on_up),
    "post_norm_before_residual": ("layer_output", _layer_norm_before_residual),
    "e4m3_ties_away_from_zero": ("e4m3_quantize", _e4m3_ties_away),
    "e4m3_rounds_toward_zero": ("e4m3_quantize", _e4m3_truncates),
    "e4m3_overflow_to_nan": ("e4m3_quantize", _e4m3_no_saturation),
    "e4m3_exponent_bias_8": ("e4m3_value", _e4m3_bias_8),
    "fp8_store_drops_scale": ("fp8_store", _fp8_store_drops_scale),
    "split_heads_strided": ("split_heads", _split_heads_strided),
    "split_heads_reversed_order": ("split_heads", _split_heads_reversed),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(O, attr, fn)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(O)
        except Exception:
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name}"
