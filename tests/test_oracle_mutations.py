"""Planted mistakes in the oracle must be caught by its pins (CPU only).

Each case swaps one oracle function for a plausibly wrong variant (a
dropped term, a wrong sign, a wrong index, a wrong mask alignment) and runs
the pins of tests/test_oracle_pins.py; at least one pin has to fail.
"""

import numpy as np
import pytest

import oracle
import oracle.reference as R
import tests.test_oracle_pins as pins
from tests.conftest import read_golden


def _bad_rms_eps_outside(x_bits, w_bits, eps=R.RMS_EPS):
    x = R.bf16_to_f64(x_bits)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    n = R.f64_to_bf16(x / (np.sqrt(ms) + eps))
    return R.f64_to_bf16(R.bf16_to_f64(n) * R.bf16_to_f64(w_bits))


def _bad_rms_sum(x_bits, w_bits, eps=R.RMS_EPS):
    x = R.bf16_to_f64(x_bits)
    ms = np.sum(x * x, axis=-1, keepdims=True) / 127.0
    n = R.f64_to_bf16(x / np.sqrt(ms + eps))
    return R.f64_to_bf16(R.bf16_to_f64(n) * R.bf16_to_f64(w_bits))


def _bad_rope_sign(x_bits, cos, sin):
    x = R.bf16_to_f64(x_bits)
    x1, x2 = x[..., :64], x[..., 64:]
    c = cos.astype(np.float64)[:, None, :]
    s = sin.astype(np.float64)[:, None, :]
    return R.f64_to_bf16(np.concatenate([x1 * c - x2 * s, x2 * c - x1 * s], axis=-1))


def _bad_rope_interleaved(x_bits, cos, sin):
    x = R.bf16_to_f64(x_bits)
    x1, x2 = x[..., 0::2], x[..., 1::2]
    c = cos.astype(np.float64)[:, None, :]
    s = sin.astype(np.float64)[:, None, :]
    y = np.empty_like(x)
    y[..., 0::2] = x1 * c - x2 * s
    y[..., 1::2] = x2 * c + x1 * s
    return R.f64_to_bf16(y)


def _bad_inv_freq(theta=R.ROPE_THETA, head_dim=R.HEAD_DIM):
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(float(theta), -1.0 * i / head_dim).astype(np.float32)


def _bad_cos_sin_swapped(positions, theta=R.ROPE_THETA, head_dim=R.HEAD_DIM):
    c, s = _good["rope_cos_sin"](positions, theta, head_dim)
    return s, c


def _bad_attention_top_left(q, K, V, scale):
    Lq, Lk = q.shape[0], K.shape[0]
    K2, V2 = K, V
    out = np.empty(q.shape)
    visible = np.arange(Lk)[None, :] <= np.arange(Lq)[:, None]
    for h in range(q.shape[1]):
        g = h // (q.shape[1] // K.shape[1])
        S = np.where(visible, (q[:, h] @ K2[:, g].T) * scale, -np.inf)
        P = np.exp(S - S.max(1, keepdims=True))
        out[:, h] = (P / P.sum(1, keepdims=True)) @ V2[:, g]
    return out


def _bad_attention_gqa_modulo(q, K, V, scale):
    Lq, Lk = q.shape[0], K.shape[0]
    visible = np.arange(Lk)[None, :] <= (Lk - Lq + np.arange(Lq))[:, None]
    out = np.empty(q.shape)
    for h in range(q.shape[1]):
        g = h % K.shape[1]
        S = np.where(visible, (q[:, h] @ K[:, g].T) * scale, -np.inf)
        P = np.exp(S - S.max(1, keepdims=True))
        out[:, h] = (P / P.sum(1, keepdims=True)) @ V[:, g]
    return out


def _bad_attention_no_scale(q, K, V, scale):
    return _good["causal_gqa_attention"](q, K, V, 1.0)


def _bad_attention_pv_transposed_heads(q, K, V, scale):
    out = _good["causal_gqa_attention"](q, K, V, scale)
    return out[:, ::-1]


def _bad_gather_offset(k_cache, v_cache, block_table_row, length):
    bs = k_cache.shape[1]
    pos = np.arange(length)
    blk = np.asarray(block_table_row)[pos // bs]
    off = (pos + 1) % bs
    return R.bf16_to_f64(k_cache[blk, off]), R.bf16_to_f64(v_cache[blk, off])


def _bad_store_ignores_skip(k_bits, v_bits, slot_mapping, k_cache, v_cache):
    for t, slot in enumerate(np.asarray(slot_mapping).tolist()):
        blk, off = slot // k_cache.shape[1], slot % k_cache.shape[1]
        k_cache[blk, off] = k_bits[t]
        v_cache[blk, off] = v_bits[t]


def _bad_bf16_truncate(x):
    x = np.asarray(x, dtype=np.float64)
    return (x.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def _bad_add_norm_rounded_sum(x_bits, res_bits, w_bits, eps=R.RMS_EPS):
    # normalises the bf16-rounded residual instead of the fp32 sum
    if res_bits is None:
        return _good["add_rms_norm"](x_bits, None, w_bits, eps)
    s = R.f64_to_bf16((R.bf16_to_f64(x_bits) + R.bf16_to_f64(res_bits)).astype(np.float32).astype(np.float64))
    return R.rms_norm_rows(R.bf16_to_f64(s), w_bits, eps), s


def _bad_add_norm_keeps_old_residual(x_bits, res_bits, w_bits, eps=R.RMS_EPS):
    out, _ = _good["add_rms_norm"](x_bits, res_bits, w_bits, eps)
    return out, (np.asarray(x_bits).copy() if res_bits is None else np.asarray(res_bits).copy())


def _bad_add_norm_no_weight(x_f64, w_bits, eps=R.RMS_EPS):
    x = np.asarray(x_f64, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return R.f64_to_bf16(x / np.sqrt(ms + eps))


def _bad_traffic_reads_sum_back(hidden=R.HIDDEN, fused=True):
    return 5 * 2 * hidden


def _bad_qkv_split_kv_swapped(x_bits, w_bits):
    q, k, v = _good["qkv_projection"](x_bits, w_bits)
    return q, v, k


def _bad_qkv_transposed(x_bits, w_bits):
    # head and dimension axes of the output swapped: feature h*128 + d read as d*48 + h
    x, w = R.bf16_to_f64(x_bits), R.bf16_to_f64(w_bits)
    T = x.shape[0]
    y = R.f64_to_bf16(x @ w.T).reshape(T, 48, 128).transpose(0, 2, 1).reshape(T, 6144)
    return y[:, :4096].reshape(T, 32, 128), y[:, 4096:5120].reshape(T, 8, 128), y[:, 5120:].reshape(T, 8, 128)


def _bad_qk_weights_swapped(q_bits, k_bits, positions, q_norm_w, k_norm_w):
    return _good["qk_norm_rope"](q_bits, k_bits, positions, k_norm_w, q_norm_w)


def _bad_qk_rope_before_norm(q_bits, k_bits, positions, q_norm_w, k_norm_w):
    cos, sin = R.rope_cos_sin(positions)
    q = R.rms_norm_heads(R.apply_rope(q_bits, cos, sin), q_norm_w)
    k = R.rms_norm_heads(R.apply_rope(k_bits, cos, sin), k_norm_w)
    return q, k


def _bad_qk_position_plus_one(q_bits, k_bits, positions, q_norm_w, k_norm_w):
    return _good["qk_norm_rope"](q_bits, k_bits, np.asarray(positions) + 1, q_norm_w, k_norm_w)


def _bad_step_stores_raw_k(wl, k_cache=None, v_cache=None, seqs=None):
    saved = wl.k
    q_out, k_out = R.qk_norm_rope(wl.q, wl.k, wl.positions, wl.q_norm_w, wl.k_norm_w)
    kc, vc = (wl.materialize_cache() if k_cache is None else (k_cache.copy(), v_cache.copy()))
    R.store_kvcache(saved, wl.v, wl.slot_mapping, kc, vc)
    if wl.mode == "decode":
        out = R.paged_decode(q_out, kc, vc, wl.context_lens, wl.block_table, wl.scale)
    else:
        out = R.paged_prefill(q_out, kc, vc, R.cu_seqlens(wl.new_lens), R.cu_seqlens(wl.seq_lens_k),
                              wl.block_table, wl.scale, seqs)
    return q_out, k_out, kc, vc, out


def _bad_step_attends_raw_q(wl, k_cache=None, v_cache=None, seqs=None):
    q_out, k_out, kc, vc, _ = _good["run_step"](wl, k_cache, v_cache, seqs)
    if wl.mode == "decode":
        out = R.paged_decode(wl.q, kc, vc, wl.context_lens, wl.block_table, wl.scale)
    else:
        out = R.paged_prefill(wl.q, kc, vc, R.cu_seqlens(wl.new_lens), R.cu_seqlens(wl.seq_lens_k),
                              wl.block_table, wl.scale, seqs)
    return q_out, k_out, kc, vc, out


def _bad_qkvstore_raw_k(x_bits, w_bits, positions, slot_mapping, q_norm_w, k_norm_w, k_cache, v_cache):
    q, k, v = R.qkv_projection(x_bits, w_bits)
    q_out, _ = R.qk_norm_rope(q, k, positions, q_norm_w, k_norm_w)
    R.store_kvcache(k, v, slot_mapping, k_cache, v_cache)
    return q_out


def _bad_qkvstore_returns_projected_q(x_bits, w_bits, positions, slot_mapping, q_norm_w, k_norm_w, k_cache,
                                      v_cache):
    _good["qkv_rope_store"](x_bits, w_bits, positions, slot_mapping, q_norm_w, k_norm_w, k_cache, v_cache)
    return R.qkv_projection(x_bits, w_bits)[0]


_good = {name: getattr(R, name) for name in R.__all__ if callable(getattr(R, name))}

MUTANTS = [
    ("rms_norm_heads", _bad_rms_eps_outside),
    ("rms_norm_heads", _bad_rms_sum),
    ("apply_rope", _bad_rope_sign),
    ("apply_rope", _bad_rope_interleaved),
    ("rope_inv_freq", _bad_inv_freq),
    ("rope_cos_sin", _bad_cos_sin_swapped),
    ("causal_gqa_attention", _bad_attention_top_left),
    ("causal_gqa_attention", _bad_attention_gqa_modulo),
    ("causal_gqa_attention", _bad_attention_no_scale),
    ("causal_gqa_attention", _bad_attention_pv_transposed_heads),
    ("gather_kv", _bad_gather_offset),
    ("store_kvcache", _bad_store_ignores_skip),
    ("f64_to_bf16", _bad_bf16_truncate),
    ("add_rms_norm", _bad_add_norm_rounded_sum),
    ("add_rms_norm", _bad_add_norm_keeps_old_residual),
    ("rms_norm_rows", _bad_add_norm_no_weight),
    ("add_rmsnorm_bytes_per_token", _bad_traffic_reads_sum_back),
    ("qkv_projection", _bad_qkv_split_kv_swapped),
    ("qkv_projection", _bad_qkv_transposed),
    ("qk_norm_rope", _bad_qk_weights_swapped),
    ("qk_norm_rope", _bad_qk_rope_before_norm),
    ("qk_norm_rope", _bad_qk_position_plus_one),
    ("run_step", _bad_step_stores_raw_k),
    ("run_step", _bad_step_attends_raw_q),
    ("qkv_rope_store", _bad_qkvstore_raw_k),
    ("qkv_rope_store", _bad_qkvstore_returns_projected_q),
]


def _run_all_pins():
    failures = 0
    golden = read_golden
    for name in dir(pins):
        if not name.startswith("test_"):
            continue
        fn = getattr(pins, name)
        try:
            if "golden" in fn.__code__.co_varnames[: fn.__code__.co_argcount]:
                fn(golden)
            else:
                fn()
        except Exception:  # an AssertionError, or a crash the mutant caused
            failures += 1
    return failures


def test_pins_pass_on_the_real_oracle():
    assert _run_all_pins() == 0


@pytest.mark.parametrize("target,mutant", MUTANTS, ids=[m.__name__ for _, m in MUTANTS])
def test_planted_mistake_is_caught(monkeypatch, target, mutant):
    monkeypatch.setattr(R, target, mutant)
    monkeypatch.setattr(oracle, target, mutant)
    assert _run_all_pins() > 0
