"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test ties one oracle function to a value the pages print
(tests/golden/), a closed form, a library routine, or brute force on tiny
inputs, chosen so that a plausible slip (a dropped term, a wrong sign or
index, a transposed operand, a wrong mask alignment) fails at least one test.
"""

import math

import numpy as np
import pytest
import torch

import oracle as O
from workloads import NAN_BF16, build_workload


def f32_bf16_bits(x):
    """Independent fp32 -> bf16 conversion through torch (the library routine)."""
    t = torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def rand_bf16(rng, shape, scale=1.0):
    return f32_bf16_bits(scale * rng.standard_normal(shape).astype(np.float32))


# ---------------------------------------------------------------- golden values
def test_kv_cache_sizes_match_page(golden):
    kv, _ = golden("kv_cache_sizes.txt")
    per_tok = O.kv_bytes_per_token(int(kv["num_layers"]), int(kv["num_kv_heads"]), int(kv["head_dim"]),
                                   int(kv["dtype_bytes"]))
    assert per_tok == int(kv["bytes_per_token"])
    assert per_tok == int(kv["kib_per_token"]) * 1024
    assert per_tok * int(kv["block_tokens"]) == int(kv["mib_per_block"]) * 2 ** 20
    gb = per_tok * int(kv["full_context_tokens"]) / 1e9
    assert round(gb, 1) == float(kv["gb_per_full_context"])
    # one layer of the same geometry: 4096 bytes per token, 1 MiB per K+V block
    assert O.kv_bytes_per_token(1) == 4096
    assert O.kv_bytes_per_token(1) * O.BLOCK_SIZE == 2 ** 20


def test_varlen_mask_matches_page(golden):
    _, rows = golden("varlen_mask_T7.txt")
    assert O.flat_varlen_mask([3, 2, 2]) == rows


def test_cu_seqlens_matches_page(golden):
    kv, _ = golden("cu_seqlens_example.txt")
    lengths = [int(x) for x in kv["lengths"].split()]
    expect = [int(x) for x in kv["cu_seqlens"].split()]
    assert O.cu_seqlens(lengths).tolist() == expect


def test_rope_table_size_matches_page(golden):
    kv, _ = golden("rope_table_size.txt")
    c, s = O.rope_cos_sin(np.arange(int(kv["positions"])))
    table_bytes = c.nbytes + s.nbytes
    assert c.dtype == np.float32 and s.dtype == np.float32
    assert c.shape[1] + s.shape[1] == int(kv["values_per_position"])
    assert table_bytes == 20 * 2 ** 20
    assert round(table_bytes / 2 ** 20) == int(kv["table_mb"])


# ---------------------------------------------------------------- bf16 rounding
def test_bf16_rounding_against_torch():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-30).astype(np.float32),
        (rng.standard_normal(2000) * 1e30).astype(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0], np.float32),
    ])
    ok = np.abs(x) >= 2.0 ** -126
    ok |= x == 0
    x = x[ok]
    assert np.array_equal(O.f64_to_bf16(x.astype(np.float64)), f32_bf16_bits(x))


def test_bf16_rounding_ties_to_even():
    ulp = 2.0 ** -7  # bf16 spacing in [1, 2)
    vals = np.array([1 + ulp / 2, 1 + 1.5 * ulp, -(1 + ulp / 2), 1 + ulp / 2 + 2.0 ** -30])
    got = O.bf16_to_f64(O.f64_to_bf16(vals))
    assert got.tolist() == [1.0, 1 + 2 * ulp, -1.0, 1 + ulp]


# ---------------------------------------------------------------- RMSNorm
def test_rmsnorm_constant_row_closed_form():
    # x = c everywhere, w = 1: mean(x^2) = c^2, output = c / sqrt(c^2 + eps)
    for c in [0.5, -3.0, 1e-3, 7.25]:
        cb = O.f64_to_bf16(np.array([c]))[0]
        cv = O.bf16_to_f64(np.array([cb]))[0]
        x = np.full((1, 1, 128), cb, np.uint16)
        w = np.full(128, O.f64_to_bf16(np.array([1.0]))[0], np.uint16)
        out = O.bf16_to_f64(O.rms_norm_heads(x, w))
        expect = O.bf16_to_f64(O.f64_to_bf16(np.array([math.copysign(1.0, cv) / math.sqrt(1 + O.RMS_EPS / cv ** 2)])))
        assert np.all(out == expect[0])


def test_rmsnorm_against_torch_rms_norm():
    rng = np.random.default_rng(2)
    x = rand_bf16(rng, (64, 8, 128), scale=3.0)
    w = f32_bf16_bits(1 + 0.1 * rng.standard_normal(128).astype(np.float32))
    xt = torch.tensor(O.bf16_to_f64(x))
    normed = torch.nn.functional.rms_norm(xt, (128,), eps=O.RMS_EPS).numpy()
    expect = O.f64_to_bf16(O.bf16_to_f64(O.f64_to_bf16(normed)) * O.bf16_to_f64(w))
    got = O.rms_norm_heads(x, w)
    # fp64 rounding-order differences can only matter on an exact bf16 tie
    assert np.mean(got != expect) < 1e-4


def test_rmsnorm_weight_scaling_and_unit_rms():
    rng = np.random.default_rng(3)
    x = rand_bf16(rng, (32, 4, 128))
    one = np.full(128, O.f64_to_bf16(np.array([1.0]))[0], np.uint16)
    two = np.full(128, O.f64_to_bf16(np.array([2.0]))[0], np.uint16)
    y1 = O.bf16_to_f64(O.rms_norm_heads(x, one))
    y2 = O.bf16_to_f64(O.rms_norm_heads(x, two))
    assert np.array_equal(y2, 2 * y1)  # a power-of-two weight scales exactly
    rms = np.sqrt(np.mean(y1 ** 2, axis=-1))
    assert np.all(np.abs(rms - 1) < 4 * 2.0 ** -8)
    # per-element weight, not a per-head or per-row one
    w = np.arange(128, dtype=np.float64) / 64 + 0.5
    wb = O.f64_to_bf16(w)
    yw = O.bf16_to_f64(O.rms_norm_heads(x, wb))
    assert np.all(np.abs(yw - y1 * O.bf16_to_f64(wb)) <= np.abs(y1 * O.bf16_to_f64(wb)) * 2.0 ** -8 + 1e-30)


# ---------------------------------------------------------------- RoPE
def test_inv_freq_closed_forms():
    inv = O.rope_inv_freq().astype(np.float64)
    assert inv.shape == (64,)
    assert inv[0] == 1.0
    # theta^(-2*32/128) = theta^(-1/2) = 1e-3 for theta = 1e6
    assert inv[32] == np.float32(1e-3)
    # geometric: ratio between neighbours is theta^(-1/64)
    r = inv[1:] / inv[:-1]
    assert np.allclose(r, 1e6 ** (-1 / 64), rtol=2e-7)
    assert np.all(np.diff(inv) < 0)


def test_cos_sin_table_against_torch_construction():
    # The page builds the table as einsum("i,j->ij", t, inv_freq) then cos / sin (fp32).
    pos = np.array([0, 1, 2, 17, 255, 4095, 12345, 40959])
    c, s = O.rope_cos_sin(pos)
    inv = torch.tensor(O.rope_inv_freq())
    freqs = torch.einsum("i,j -> ij", torch.tensor(pos, dtype=torch.float32), inv)
    tc = freqs.double().cos().float().numpy()
    ts = freqs.double().sin().float().numpy()
    assert np.array_equal(c, tc) and np.array_equal(s, ts)
    assert np.all(c[0] == 1.0) and np.all(s[0] == 0.0)


def test_rope_forms_agree_and_position_zero_is_identity():
    rng = np.random.default_rng(4)
    x = rand_bf16(rng, (50, 8, 128))
    pos = rng.integers(0, 40960, 50)
    pos[0] = 0
    c, s = O.rope_cos_sin(pos)
    a = O.apply_rope(x, c, s)
    b = O.apply_rope_rotate_half(x, c, s)
    assert np.array_equal(a, b)
    assert np.array_equal(a[0], x[0])


def test_rope_preserves_pair_norms():
    rng = np.random.default_rng(5)
    x = rand_bf16(rng, (40, 4, 128))
    pos = rng.integers(0, 40960, 40)
    c, s = O.rope_cos_sin(pos)
    y = O.bf16_to_f64(O.apply_rope(x, c, s))
    xv = O.bf16_to_f64(x)
    nx = np.hypot(xv[..., :64], xv[..., 64:])
    ny = np.hypot(y[..., :64], y[..., 64:])
    assert np.all(np.abs(ny - nx) <= 2 * 2.0 ** -8 * nx + 1e-30)


def test_rope_scores_depend_on_relative_position_only():
    rng = np.random.default_rng(6)
    q = rand_bf16(rng, (1, 1, 128))
    k = rand_bf16(rng, (1, 1, 128))

    def score(m, n):
        cq, sq = O.rope_cos_sin(np.array([m]))
        ck, sk = O.rope_cos_sin(np.array([n]))
        a = O.bf16_to_f64(O.apply_rope(q, cq, sq))[0, 0]
        b = O.bf16_to_f64(O.apply_rope(k, ck, sk))[0, 0]
        return float(a @ b)

    ref = np.linalg.norm(O.bf16_to_f64(q)) * np.linalg.norm(O.bf16_to_f64(k))
    for d in [0, 1, 7, 100]:
        vals = [score(n + d, n) for n in [0, 13, 250, 999]]
        assert max(vals) - min(vals) < 2e-2 * ref
    # and it does depend on the offset
    assert abs(score(5, 0) - score(0, 5)) > 1e-3 * ref or abs(score(5, 0) - score(0, 0)) > 1e-3 * ref


# ---------------------------------------------------------------- norm, then RoPE
def _round_bf16_scalar(x):
    """Round one Python float to the nearest bf16 value, ties to even (8 significant bits)."""
    if x == 0.0:
        return 0.0
    m, e = math.frexp(x)
    return math.ldexp(round(math.ldexp(m, 8)), e - 8)  # Python's round() is half-to-even


def test_qk_norm_rope_composition_closed_form():
    # "Nano-vLLM深度解读（下）" §2 Qwen3Attention.forward: q_norm / k_norm per head, then
    # rotary_emb(positions, q, k).  A head whose only nonzero element is x[0] = c has
    # mean square c^2/128, so its norm is sign(c)*sqrt(128)/sqrt(1 + 128*eps/c^2) at
    # element 0 and exactly 0 elsewhere; after the weight, RoPE's first pair (0, 64)
    # rotates at inv_freq_0 = 1, i.e. by the angle fp32(p), so element 0 becomes
    # r*cos(p) and element 64 becomes r*sin(p), where r = bf16(bf16(norm) * w[0]).
    # The weights differ between q and k and between elements 0 and 64, so a
    # swapped weight, RoPE applied before the norm (element 64 would take w[64]) or a
    # shifted position all change the expected bits.
    positions = np.array([1, 7, 1000, 40959])
    T = len(positions)
    cq, ck = 2.0, -0.75  # bf16-exact
    q = np.zeros((T, O.NUM_Q_HEADS, 128), np.uint16)
    k = np.zeros((T, O.NUM_KV_HEADS, 128), np.uint16)
    # head h of token t carries c * 2^-(h % 3) at element 0 (all bf16-exact)
    for t in range(T):
        for h in range(O.NUM_Q_HEADS):
            q[t, h, 0] = f32_bf16_bits(np.array([cq * 2.0 ** -(h % 3)]))[0]
        for h in range(O.NUM_KV_HEADS):
            k[t, h, 0] = f32_bf16_bits(np.array([ck * 2.0 ** -(h % 3)]))[0]
    wq = np.ones(128, np.float32)
    wk = np.ones(128, np.float32)
    wq[0], wq[64] = 1.5, 0.75
    wk[0], wk[64] = 0.625, 1.25
    wq_b, wk_b = f32_bf16_bits(wq), f32_bf16_bits(wk)

    gq, gk = O.qk_norm_rope(q, k, positions, wq_b, wk_b)
    gq, gk = O.bf16_to_f64(gq), O.bf16_to_f64(gk)

    def expect(c, w0, p):
        n = math.copysign(1.0, c) * math.sqrt(128.0) / math.sqrt(1.0 + 128.0 * O.RMS_EPS / (c * c))
        r = _round_bf16_scalar(_round_bf16_scalar(n) * w0)
        ang = float(np.float32(p))  # inv_freq_0 = theta^0 = 1
        cos32 = float(np.float32(math.cos(ang)))
        sin32 = float(np.float32(math.sin(ang)))
        return _round_bf16_scalar(r * cos32), _round_bf16_scalar(r * sin32)

    for t, p in enumerate(positions.tolist()):
        for out, base, w0, H in ((gq, cq, 1.5, O.NUM_Q_HEADS), (gk, ck, 0.625, O.NUM_KV_HEADS)):
            for h in range(H):
                e0, e64 = expect(base * 2.0 ** -(h % 3), w0, p)
                assert out[t, h, 0] == e0, (t, h, p)
                assert out[t, h, 64] == e64, (t, h, p)
                rest = np.delete(out[t, h], [0, 64])
                assert np.all(rest == 0.0)
    # the norm makes the output independent of the head's input scale
    assert np.array_equal(gq[:, 0], gq[:, 1]) and np.array_equal(gk[:, 0], gk[:, 2])


def _one_hot_head_rows(T, H, c):
    x = np.zeros((T, H, 128), np.uint16)
    x[:, :, 0] = f32_bf16_bits(np.array([c]))[0]
    return x


def _rotated_pair(c, w0, p):
    """Elements 0 and 64 of a one-hot head (x[0] = c) after the norm, the weight and RoPE at position p."""
    n = math.copysign(1.0, c) * math.sqrt(128.0) / math.sqrt(1.0 + 128.0 * O.RMS_EPS / (c * c))
    r = _round_bf16_scalar(_round_bf16_scalar(n) * w0)
    ang = float(np.float32(p))
    return (_round_bf16_scalar(r * float(np.float32(math.cos(ang)))),
            _round_bf16_scalar(r * float(np.float32(math.sin(ang)))))


def _distinct_pair_weights():
    wq = np.ones(128, np.float32)
    wk = np.ones(128, np.float32)
    wq[0], wq[64] = 1.5, 0.75
    wk[0], wk[64] = 0.625, 1.25
    return f32_bf16_bits(wq), f32_bf16_bits(wk)


def test_step_decode_closed_form():
    # The whole step ("Nano-vLLM深度解读（下）" §2 then §4, "同一个 Qwen3，两种写法" §3.4 write
    # first, then read) on two sequences with one cached token each: the new token
    # (position 1) is normed, rotated, stored, then attends to keys 0 and 1.  Key 0 is a
    # zero row (score 0); key 1 is the new token's rotated k, whose score against the
    # rotated q has the closed form scale * (q0*k0 + q64*k64).  The output is then
    # (V0 + e^s V1) / (1 + e^s) with V0, V1 constant per KV head.
    wl = build_workload("closed-form step", "decode", 31, [1, 1], [1, 1], spare_blocks=1)
    assert wl.positions.tolist() == [1, 1]
    cq, ck = 2.0, -0.75
    wl.q = _one_hot_head_rows(2, O.NUM_Q_HEADS, cq)
    wl.k = _one_hot_head_rows(2, O.NUM_KV_HEADS, ck)
    wl.q_norm_w, wl.k_norm_w = _distinct_pair_weights()
    v1 = np.zeros((2, O.NUM_KV_HEADS), np.float64)
    v0 = np.zeros((2, O.NUM_KV_HEADS), np.float64)
    wl.v = np.zeros((2, O.NUM_KV_HEADS, 128), np.uint16)
    kc, vc = wl.materialize_cache()
    for b in range(2):
        blk0 = wl.block_table[b, 0]
        kc[blk0, 0] = 0
        for g in range(O.NUM_KV_HEADS):
            v1[b, g] = (g + 1) * 0.25 + b * 0.125
            v0[b, g] = -(g + 1) * 0.5
            wl.v[b, g] = f32_bf16_bits(np.full(128, v1[b, g], np.float32))
            vc[blk0, 0, g] = f32_bf16_bits(np.full(128, v0[b, g], np.float32))
    q_out, k_out, kc1, vc1, out = O.run_step(wl, kc, vc)

    q0, q64 = _rotated_pair(cq, 1.5, 1)
    k0, k64 = _rotated_pair(ck, 0.625, 1)
    s = wl.scale * (q0 * k0 + q64 * k64)
    w1 = math.exp(s) / (1.0 + math.exp(s))
    for b in range(2):
        blk, off = divmod(int(wl.slot_mapping[b]), O.BLOCK_SIZE)
        row = O.bf16_to_f64(kc1[blk, off])
        assert np.all(row[:, 0] == k0) and np.all(row[:, 64] == k64)
        assert np.all(np.delete(row, [0, 64], axis=1) == 0.0)
        assert np.array_equal(vc1[blk, off], wl.v[b])
        for h in range(O.NUM_Q_HEADS):
            expect = (1.0 - w1) * v0[b, h // 4] + w1 * v1[b, h // 4]
            np.testing.assert_allclose(out[b, h], expect, rtol=0, atol=1e-13)


def test_qkv_rope_store_closed_form():
    # "同一个 Qwen3，两种写法" §3.1 (one projection, split q | k | v) followed by the
    # norm, RoPE and the store.  Selection weights route input feature 0 to element 0
    # of every q head, feature 1 to element 0 of every k head and feature 2 to every
    # element of every v head, so q and k are one-hot heads with the closed form of the
    # composition pin above and each stored V row is x[2] everywhere.
    T = 3
    positions = np.array([0, 5, 40000])
    x = np.zeros((T, O.HIDDEN), np.uint16)
    cq, ck, cv = 2.0, -0.75, 3.5
    x[:, 0] = f32_bf16_bits(np.array([cq]))[0]
    x[:, 1] = f32_bf16_bits(np.array([ck]))[0]
    x[:, 2] = f32_bf16_bits(np.array([cv]))[0]
    x[:, 3:] = f32_bf16_bits(np.full(O.HIDDEN - 3, 9.0, np.float32))  # routed nowhere
    w = np.zeros((O.QKV_OUT, O.HIDDEN), np.float32)
    for h in range(O.NUM_Q_HEADS):
        w[h * 128, 0] = 1.0
    for g in range(O.NUM_KV_HEADS):
        w[4096 + g * 128, 1] = 1.0
        w[5120 + g * 128:5120 + (g + 1) * 128, 2] = 1.0
    wq, wk = _distinct_pair_weights()
    NB = 2
    kc = np.full((NB, O.BLOCK_SIZE, 8, 128), NAN_BF16, np.uint16)
    vc = kc.copy()
    slots = np.array([3, -1, 300], np.int32)
    q_out = O.bf16_to_f64(O.qkv_rope_store(x, f32_bf16_bits(w), positions, slots, wq, wk, kc, vc))
    for t, p in enumerate(positions.tolist()):
        q0, q64 = _rotated_pair(cq, 1.5, p)
        assert np.all(q_out[t, :, 0] == q0) and np.all(q_out[t, :, 64] == q64), t
        assert np.all(np.delete(q_out[t], [0, 64], axis=1) == 0.0)
        if slots[t] < 0:
            continue
        blk, off = divmod(int(slots[t]), O.BLOCK_SIZE)
        k0, k64 = _rotated_pair(ck, 0.625, p)
        row = O.bf16_to_f64(kc[blk, off])
        assert np.all(row[:, 0] == k0) and np.all(row[:, 64] == k64), t
        assert np.all(np.delete(row, [0, 64], axis=1) == 0.0)
        assert np.all(O.bf16_to_f64(vc[blk, off]) == cv)
    written = {3, 300}
    for s in range(NB * O.BLOCK_SIZE):
        if s not in written:
            blk, off = divmod(s, O.BLOCK_SIZE)
            assert np.all(kc[blk, off] == NAN_BF16) and np.all(vc[blk, off] == NAN_BF16)


# ---------------------------------------------------------------- store
def test_store_writes_only_mapped_slots():
    wl = build_workload("store pin", "prefill", 7, [0, 300], [5, 40], spare_blocks=3, skip_tokens=[2, 17])
    kc, vc = wl.materialize_cache()
    kc0, vc0 = kc.copy(), vc.copy()
    O.store_kvcache(wl.k, wl.v, wl.slot_mapping, kc, vc)
    written = np.zeros(kc.shape[:2], bool)
    for t, slot in enumerate(wl.slot_mapping):
        if slot < 0:
            continue
        b, o = slot // 256, slot % 256
        written[b, o] = True
        assert np.array_equal(kc[b, o], wl.k[t]) and np.array_equal(vc[b, o], wl.v[t])
    assert written.sum() == len(wl.slot_mapping) - 2
    assert np.array_equal(kc[~written], kc0[~written]) and np.array_equal(vc[~written], vc0[~written])
    # every new token can be read back through the block table at its position
    cu = O.cu_seqlens(wl.new_lens)
    for s in range(wl.num_seqs):
        K, V = O.gather_kv(kc, vc, wl.block_table[s], int(wl.seq_lens_k[s]))
        for t in range(cu[s], cu[s + 1]):
            if wl.slot_mapping[t] >= 0:
                assert np.array_equal(K[wl.positions[t]], O.bf16_to_f64(wl.k[t]))


# ---------------------------------------------------------------- attention
def repeat_kv(x, n_rep):
    """[Lk, Hkv, D] -> [Lk, Hkv*n_rep, D] by expand + reshape, as transformers materialises GQA."""
    Lk, H, D = x.shape
    return x[:, :, None, :].expand(Lk, H, n_rep, D).reshape(Lk, H * n_rep, D)


def sdpa_reference(q, K, V, scale, causal):
    qt = torch.tensor(q).permute(1, 0, 2)[None]
    kt = repeat_kv(torch.tensor(K), q.shape[1] // K.shape[1]).permute(1, 0, 2)[None]
    vt = repeat_kv(torch.tensor(V), q.shape[1] // K.shape[1]).permute(1, 0, 2)[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=causal, scale=scale)
    return o[0].permute(1, 0, 2).numpy()


def test_attention_equals_sdpa_causal_prefill():
    rng = np.random.default_rng(8)
    L = 77
    q = rng.standard_normal((L, 32, 128))
    K = rng.standard_normal((L, 8, 128))
    V = rng.standard_normal((L, 8, 128))
    got = O.causal_gqa_attention(q, K, V, 0.088)
    np.testing.assert_allclose(got, sdpa_reference(q, K, V, 0.088, True), rtol=0, atol=1e-12)


def test_attention_equals_sdpa_decode():
    rng = np.random.default_rng(9)
    q = rng.standard_normal((1, 32, 128))
    K = rng.standard_normal((300, 8, 128))
    V = rng.standard_normal((300, 8, 128))
    got = O.causal_gqa_attention(q, K, V, 1 / math.sqrt(128))
    np.testing.assert_allclose(got, sdpa_reference(q, K, V, 1 / math.sqrt(128), False), rtol=0, atol=1e-12)


def brute_force_attention(q, K, V, scale):
    Lq, H, D = q.shape
    Lk, Hk, _ = K.shape
    out = np.zeros((Lq, H, D))
    for i in range(Lq):
        pos = Lk - Lq + i
        for h in range(H):
            g = h * Hk // H
            w = [math.exp(scale * sum(q[i, h, d] * K[j, g, d] for d in range(D))) for j in range(pos + 1)]
            tot = sum(w)
            for d in range(D):
                out[i, h, d] = sum(w[j] * V[j, g, d] for j in range(pos + 1)) / tot
    return out


def test_attention_brute_force_tiny():
    rng = np.random.default_rng(10)
    for Lk in range(1, 7):
        for Lq in range(1, Lk + 1):
            q = rng.standard_normal((Lq, 8, 4))
            K = rng.standard_normal((Lk, 2, 4))
            V = rng.standard_normal((Lk, 2, 4))
            np.testing.assert_allclose(O.causal_gqa_attention(q, K, V, 0.5), brute_force_attention(q, K, V, 0.5),
                                       rtol=0, atol=1e-12)


def test_single_key_returns_v_exactly():
    wl = build_workload("single key", "decode", 11, [0, 0], [1, 1], spare_blocks=2)
    q, k, kc, vc, out = O.run_step(wl)
    for b in range(2):
        for h in range(32):
            assert np.array_equal(out[b, h], O.bf16_to_f64(wl.v[b, h // 4]))


def test_constant_keys_give_mean_of_values():
    rng = np.random.default_rng(12)
    L = 50
    q = rng.standard_normal((L, 32, 128))
    K = np.repeat(rng.standard_normal((1, 8, 128)), L, axis=0)
    V = rng.standard_normal((L, 8, 128))
    out = O.causal_gqa_attention(q, K, V, 0.1)
    for i in range(L):
        mean = V[: i + 1].mean(axis=0)  # [8, 128]
        np.testing.assert_allclose(out[i], np.repeat(mean, 4, axis=0), rtol=0, atol=1e-12)


def test_paging_invariant_under_block_permutation():
    wl = build_workload("perm", "prefill", 13, [300, 0, 600], [40, 200, 1], spare_blocks=5)
    kc, vc = wl.materialize_cache()
    _, _, kc1, vc1, out1 = O.run_step(wl, kc, vc)
    # move every physical block to a new id and rewrite the tables and slots to match
    perm = np.random.default_rng(99).permutation(wl.num_blocks)
    kc2 = np.empty_like(kc1)
    vc2 = np.empty_like(vc1)
    kc2[perm] = kc1
    vc2[perm] = vc1
    bt2 = np.where(wl.block_table >= 0, perm[np.maximum(wl.block_table, 0)], -1)
    q_out, _ = O.qk_norm_rope(wl.q, wl.k, wl.positions, wl.q_norm_w, wl.k_norm_w)
    out2 = O.paged_prefill(q_out, kc2, vc2, O.cu_seqlens(wl.new_lens), O.cu_seqlens(wl.seq_lens_k), bt2, wl.scale)
    assert np.array_equal(out1, out2)


def test_paged_equals_contiguous_attention():
    wl = build_workload("contig", "prefill", 14, [0, 0], [129, 300], spare_blocks=4)
    q_out, k_out, kc, vc, out = O.run_step(wl)
    cu = O.cu_seqlens(wl.new_lens)
    for s in range(2):
        a, b = cu[s], cu[s + 1]
        ref = sdpa_reference(O.bf16_to_f64(q_out[a:b]), O.bf16_to_f64(k_out[a:b]), O.bf16_to_f64(wl.v[a:b]),
                             wl.scale, True)
        np.testing.assert_allclose(out[a:b], ref, rtol=0, atol=1e-12)


def test_chunked_prefill_equals_one_shot():
    # prompt of 700 tokens processed whole, or as 450 cached + 250 new: same rows
    rng = np.random.default_rng(15)
    q = rng.standard_normal((700, 32, 128))
    K = rng.standard_normal((700, 8, 128))
    V = rng.standard_normal((700, 8, 128))
    whole = O.causal_gqa_attention(q, K, V, 0.09)
    tail = O.causal_gqa_attention(q[450:], K, V, 0.09)
    np.testing.assert_allclose(tail, whole[450:], rtol=0, atol=1e-12)
    # and a decode step is the last row of a prefill
    last = O.causal_gqa_attention(q[699:], K, V, 0.09)
    np.testing.assert_allclose(last, whole[699:], rtol=0, atol=1e-12)


def test_no_cross_sequence_leakage():
    wl = build_workload("leak", "decode", 16, [100, 700], [1, 1], spare_blocks=2)
    kc, vc = wl.materialize_cache()
    _, _, _, _, out1 = O.run_step(wl, kc, vc)
    kc2, vc2 = kc.copy(), vc.copy()
    for b in wl.block_table[1][wl.block_table[1] >= 0]:
        kc2[b] ^= 0x0040
        vc2[b] ^= 0x0040
    _, _, _, _, out2 = O.run_step(wl, kc2, vc2)
    assert np.array_equal(out1[0], out2[0])
    assert not np.array_equal(out1[1], out2[1])


def test_shared_prefix_blocks_equal_private_copies():
    wl = build_workload("share", "prefill", 17, [600, 530], [64, 64], spare_blocks=4, share_pairs=True)
    assert np.array_equal(wl.block_table[0, :2], wl.block_table[1, :2])
    kc, vc = wl.materialize_cache()
    q_out, k_out, kc1, vc1, out = O.run_step(wl, kc, vc)
    # give sequence 1 private copies of the shared blocks
    free = sorted(set(range(wl.num_blocks)) - set(wl.used_blocks().tolist()))
    bt = wl.block_table.copy()
    kc2, vc2 = kc1.copy(), vc1.copy()
    for j in range(2):
        nb = free[j]
        kc2[nb] = kc1[bt[1, j]]
        vc2[nb] = vc1[bt[1, j]]
        bt[1, j] = nb
    out2 = O.paged_prefill(q_out, kc2, vc2, O.cu_seqlens(wl.new_lens), O.cu_seqlens(wl.seq_lens_k), bt, wl.scale)
    assert np.array_equal(out, out2)


def test_nan_sentinels_never_reach_the_output():
    wl = build_workload("nan", "decode", 18, [16, 255, 256, 0], [1, 1, 1, 1], spare_blocks=1)
    kc, vc = wl.materialize_cache()
    assert np.any(kc == NAN_BF16)
    _, _, kc1, _, out = O.run_step(wl, kc, vc)
    assert np.all(np.isfinite(out))


# ---------------------------------------------------------------- residual add + RMSNorm ([Q3] §3.6)
def _add_norm_inputs(seed, T=12):
    rng = np.random.default_rng(seed)
    x = rand_bf16(rng, (T, O.HIDDEN))
    r = rand_bf16(rng, (T, O.HIDDEN), scale=4.0)
    w = f32_bf16_bits(1 + 0.1 * rng.standard_normal(O.HIDDEN).astype(np.float32))
    return x, r, w


def _torch_bf16(bits):
    return torch.tensor(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def test_add_rmsnorm_traffic_matches_page(golden):
    kv, _ = golden("rmsnorm_traffic.txt")
    hidden = int(kv["hidden"])
    assert hidden == O.HIDDEN
    assert 2 * hidden == int(kv["kib_per_row"]) * 1024
    assert O.add_rmsnorm_bytes_per_token(hidden, fused=False) == int(kv["unfused_kib_per_token"]) * 1024
    assert O.add_rmsnorm_bytes_per_token(hidden, fused=True) == int(kv["fused_kib_per_token"]) * 1024


def test_add_rmsnorm_residual_is_the_fp32_sum_in_bf16():
    x, r, w = _add_norm_inputs(11)
    _, res = O.add_rms_norm(x, r, w)
    expect = (_torch_bf16(x).float() + _torch_bf16(r).float()).to(torch.bfloat16)
    assert np.array_equal(res, expect.view(torch.int16).numpy().view(np.uint16))


def test_add_rmsnorm_against_torch_rms_norm():
    x, r, w = _add_norm_inputs(12)
    s32 = (_torch_bf16(x).float() + _torch_bf16(r).float()).double()  # the unrounded fp32 sum
    normed = torch.nn.functional.rms_norm(s32, (O.HIDDEN,), eps=O.RMS_EPS).numpy()
    expect = O.f64_to_bf16(O.bf16_to_f64(O.f64_to_bf16(normed)) * O.bf16_to_f64(w))
    got, _ = O.add_rms_norm(x, r, w)
    assert np.mean(got != expect) < 1e-4


def test_add_rmsnorm_first_layer_and_per_head_agreement():
    x, _, w = _add_norm_inputs(13)
    out0, res0 = O.add_rms_norm(x, None, w)
    out1, res1 = O.add_rms_norm(x, np.zeros_like(x), w)  # x + 0 is exact in fp32
    assert np.array_equal(res0, x) and np.array_equal(res1, x) and np.array_equal(out0, out1)
    # a row made of one 128-wide head repeated 32 times has the head's mean square,
    # so the row norm equals the (separately pinned) per-head norm of that head
    head = x[:, :128]
    row = np.tile(head, (1, O.HIDDEN // 128))
    wrow = np.tile(w[:128], O.HIDDEN // 128)
    got, _ = O.add_rms_norm(row, None, wrow)
    assert np.array_equal(got[:, :128], O.rms_norm_heads(head, w[:128]))


def test_add_rmsnorm_constant_row_closed_form():
    one = O.f64_to_bf16(np.array([1.0]))[0]
    w = np.full(O.HIDDEN, one, np.uint16)
    for c, d in [(0.5, 0.25), (-3.0, 1.0), (7.25, -0.25)]:
        x = np.full((1, O.HIDDEN), O.f64_to_bf16(np.array([c]))[0], np.uint16)
        r = np.full((1, O.HIDDEN), O.f64_to_bf16(np.array([d]))[0], np.uint16)
        out, res = O.add_rms_norm(x, r, w)
        s = c + d
        assert np.all(O.bf16_to_f64(res) == s)
        expect = O.f64_to_bf16(np.array([math.copysign(1.0, s) / math.sqrt(1 + O.RMS_EPS / s ** 2)]))[0]
        assert np.all(out == expect)


# ---------------------------------------------------------------- fused QKV projection ([Q3] §3.1)
def _selection_weight(offsets):
    """w [6144, 4096] whose output feature f picks input column (f + offset of its part) % 4096."""
    w = np.zeros((O.QKV_OUT, O.HIDDEN), np.uint16)
    one = O.f64_to_bf16(np.array([1.0]))[0]
    f = np.arange(O.QKV_OUT)
    part = np.where(f < 4096, 0, np.where(f < 5120, 1, 2))
    w[f, (f + np.asarray(offsets)[part]) % O.HIDDEN] = one
    return w


def test_qkv_projection_split_order_and_layout():
    rng = np.random.default_rng(31)
    x = rand_bf16(rng, (5, O.HIDDEN))
    q, k, v = O.qkv_projection(x, _selection_weight([0, 100, 2000]))
    assert q.shape == (5, 32, 128) and k.shape == (5, 8, 128) and v.shape == (5, 8, 128)
    # one nonzero product per output: the projection reproduces the chosen input bits
    assert np.array_equal(q.reshape(5, -1), x)
    assert np.array_equal(k.reshape(5, -1), np.roll(x, -100 - 4096 % O.HIDDEN, axis=1)[:, :1024])
    assert np.array_equal(v.reshape(5, -1), np.roll(x, -2000 - 5120 % O.HIDDEN, axis=1)[:, :1024])


def test_qkv_projection_brute_force_and_scaling():
    rng = np.random.default_rng(32)
    x = rand_bf16(rng, (2, O.HIDDEN))
    w = rand_bf16(rng, (O.QKV_OUT, O.HIDDEN), scale=1 / 64)
    q, k, v = O.qkv_projection(x, w)
    y = np.concatenate([q.reshape(2, -1), k.reshape(2, -1), v.reshape(2, -1)], axis=1)
    xf, wf = O.bf16_to_f64(x), O.bf16_to_f64(w)
    for t, f in [(0, 0), (1, 4095), (0, 4096), (1, 5119), (0, 5120), (1, 6143), (0, 777)]:
        exact = math.fsum(float(xf[t, i]) * float(wf[f, i]) for i in range(O.HIDDEN))
        assert y[t, f] == O.f64_to_bf16(np.array([exact]))[0]
    w2 = O.f64_to_bf16(2 * wf)  # exact: a power of two
    q2, _, _ = O.qkv_projection(x, w2)
    assert np.array_equal(O.bf16_to_f64(q2), 2 * O.bf16_to_f64(q))
