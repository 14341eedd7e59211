"""fp64 reference of the paged-KV attention step (test infrastructure only).

bf16 values travel as uint16 bit patterns.  Arithmetic is fp64; a bf16
rounding (round to nearest, ties to even) is applied exactly where the pages'
code casts back to the model dtype.  Readings of points the pages leave open
are marked "reading:".
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "NUM_Q_HEADS", "NUM_KV_HEADS", "HEAD_DIM", "BLOCK_SIZE", "ROPE_THETA", "RMS_EPS", "MAX_POSITION",
    "bf16_to_f64", "f64_to_bf16", "kv_bytes_per_token", "cu_seqlens", "flat_varlen_mask",
    "rms_norm_heads", "rope_inv_freq", "rope_cos_sin", "apply_rope", "apply_rope_rotate_half",
    "qk_norm_rope", "store_kvcache", "slot_to_row", "gather_kv", "causal_gqa_attention",
    "paged_decode", "paged_prefill", "run_step",
    "HIDDEN", "add_rms_norm", "rms_norm_rows", "add_rmsnorm_bytes_per_token",
    "QKV_OUT", "qkv_projection", "qkv_rope_store",
]

# Qwen3-8B attention geometry and constants ([Q3] §2 config table; [NV] §2
# Qwen3DecoderLayer reads rope_theta and rms_norm_eps from the config).
NUM_Q_HEADS = 32
NUM_KV_HEADS = 8
HEAD_DIM = 128
BLOCK_SIZE = 256  # nano-vllm block of 256 tokens ([Q3] §2.2 table)
ROPE_THETA = 1.0e6
RMS_EPS = 1.0e-6
MAX_POSITION = 40960
HIDDEN = 4096  # Qwen3-8B hidden size ([Q3] §2 config table, §3.6 "[T, 4096]")


# --------------------------------------------------------------------------
# bf16 <-> fp64
# --------------------------------------------------------------------------
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit pattern -> exact fp64 value (bf16 is the top half of an fp32)."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def f64_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to bf16 (8 significant bits, ties to even) -> uint16 bits.

    Written from the definition: x = m * 2**e with 0.5 <= |m| < 1, keep 8
    bits of m with round-half-even.  Inputs must be finite and either zero or
    of magnitude >= 2**-126 (the bf16 normal range), which holds for every
    value this step produces.
    """
    x = np.asarray(x, dtype=np.float64)
    if not np.all(np.isfinite(x)):
        raise ValueError("non-finite value reached a bf16 rounding point")
    nz = x != 0
    if np.any(np.abs(x[nz]) < 2.0 ** -126) or np.any(np.abs(x) >= 2.0 ** 128):
        raise ValueError("value outside the bf16 normal range")
    m, e = np.frexp(x)
    r = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)
    return (r.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# --------------------------------------------------------------------------
# Bookkeeping the pages state with numbers
# --------------------------------------------------------------------------
def kv_bytes_per_token(num_layers: int, num_kv_heads: int = NUM_KV_HEADS, head_dim: int = HEAD_DIM,
                       dtype_bytes: int = 2) -> int:
    """KV bytes one token occupies: 2 (K and V) x layers x KV heads x head_dim x bytes.

    [Q3] §2.2 "KV cache" works this out for Qwen3-8B (36 layers).
    """
    return 2 * num_layers * num_kv_heads * head_dim * dtype_bytes


def cu_seqlens(lengths) -> np.ndarray:
    """Cumulative sequence boundaries of the flat [T, ...] layout ([Q3] §3.2)."""
    out = [0]
    for n in lengths:
        out.append(out[-1] + int(n))
    return np.array(out, dtype=np.int64)


def flat_varlen_mask(lengths) -> list[str]:
    """The [T, T] visibility matrix of the flat layout, as rows of symbols.

    "✓" visible, "·" blocked by causality inside a sequence, "✗" blocked
    because the two tokens belong to different sequences ([Q3] §3.2 draws this
    matrix for three sequences of lengths 3, 2, 2).
    """
    seq_of = []
    pos_of = []
    for s, n in enumerate(lengths):
        for i in range(int(n)):
            seq_of.append(s)
            pos_of.append(i)
    rows = []
    for a in range(len(seq_of)):
        row = []
        for b in range(len(seq_of)):
            if seq_of[a] != seq_of[b]:
                row.append("✗")
            elif pos_of[b] <= pos_of[a]:
                row.append("✓")
            else:
                row.append("·")
        rows.append("".join(row))
    return rows


# --------------------------------------------------------------------------
# a1: per-head RMSNorm
# --------------------------------------------------------------------------
def rms_norm_heads(x_bits: np.ndarray, w_bits: np.ndarray, eps: float = RMS_EPS) -> np.ndarray:
    """RMSNorm over the last axis (head_dim) of every head, weight shape [head_dim].

    [NV] §2: Qwen3Attention.forward views q as [T, 32, 128] and k as
    [T, 8, 128] and applies q_norm / k_norm = RMSNorm(head_dim, eps) (they
    exist because attention_bias is false for Qwen3; [Q3] §2.1 notes that
    only head_dim is normalised).  Rounding points, reading of [Q3] §3.6
    (add_rms_forward with the residual add removed): the mean of squares and
    the scaling are done in high precision, the normalised value is cast to
    bf16, multiplied by the bf16 weight, and the product is cast to bf16.
    """
    x = bf16_to_f64(x_bits)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    normed = f64_to_bf16(x / np.sqrt(ms + eps))
    return f64_to_bf16(bf16_to_f64(normed) * bf16_to_f64(w_bits))


# --------------------------------------------------------------------------
# a2: RoPE
# --------------------------------------------------------------------------
def rope_inv_freq(theta: float = ROPE_THETA, head_dim: int = HEAD_DIM) -> np.ndarray:
    """inv_freq_i = theta^(-2i/head_dim), i < head_dim/2, rounded once to fp32.

    [Q3] §3.5 builds the table from inv_freq without printing its formula;
    reading: the standard RoPE frequencies, evaluated in fp64 and stored as
    fp32 like the rest of the table.
    """
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / head_dim).astype(np.float32)


def rope_cos_sin(positions: np.ndarray, theta: float = ROPE_THETA, head_dim: int = HEAD_DIM):
    """cos/sin rows of the precomputed table for the given positions, fp32 [T, 64].

    [Q3] §3.5: freqs = outer(t, inv_freq) (an fp32 einsum), the cache holds
    cos and sin of freqs, 64 values each, and forward indexes it by position.
    The table is fp32: 40960 positions x 128 values is the 20 MB the page
    quotes.  The angle is the fp32 product; cos and sin are evaluated in fp64
    and rounded once to fp32.
    """
    inv = rope_inv_freq(theta, head_dim)
    ang = np.asarray(positions).astype(np.float32)[:, None] * inv[None, :]  # fp32 x fp32 -> fp32
    ang64 = ang.astype(np.float64)
    return np.cos(ang64).astype(np.float32), np.sin(ang64).astype(np.float32)


def apply_rope(x_bits: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """Half-split rotation of every head, cast back to bf16 once.

    [Q3] §3.5 apply_rotary_emb: with x = [x1 | x2] (halves of head_dim),
    y1 = x1*cos - x2*sin and y2 = x2*cos + x1*sin, then cast to the input
    dtype.  x_bits [T, H, 128]; cos, sin [T, 64].
    """
    x = bf16_to_f64(x_bits)
    half = x.shape[-1] // 2
    x1, x2 = x[..., :half], x[..., half:]
    c = cos.astype(np.float64)[:, None, :]
    s = sin.astype(np.float64)[:, None, :]
    y = np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)
    return f64_to_bf16(y)


def apply_rope_rotate_half(x_bits: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """The transformers form: x*cos_full + rotate_half(x)*sin_full, cos/sin duplicated.

    [Q3] §3.5 shows this form (cos/sin concatenated with themselves to
    head_dim, rotate_half(x) = [-x2 | x1]) and states that it equals the
    half-split form.  Kept as an independent second statement for the pins.
    """
    x = bf16_to_f64(x_bits)
    half = x.shape[-1] // 2
    c = np.concatenate([cos, cos], axis=-1).astype(np.float64)[:, None, :]
    s = np.concatenate([sin, sin], axis=-1).astype(np.float64)[:, None, :]
    rot = np.concatenate([-x[..., half:], x[..., :half]], axis=-1)
    return f64_to_bf16(x * c + rot * s)


def qk_norm_rope(q_bits, k_bits, positions, q_norm_w, k_norm_w):
    """[NV] §2 Qwen3Attention.forward order: q_norm/k_norm, then rotary_emb(positions, q, k)."""
    cos, sin = rope_cos_sin(positions)
    q = apply_rope(rms_norm_heads(q_bits, q_norm_w), cos, sin)
    k = apply_rope(rms_norm_heads(k_bits, k_norm_w), cos, sin)
    return q, k


# --------------------------------------------------------------------------
# a3: slot_mapping scatter
# --------------------------------------------------------------------------
def slot_to_row(slot: int, block_size: int = BLOCK_SIZE) -> tuple[int, int]:
    """Cache row of a slot: slot = block_id * block_size + offset ([Q3] §3.3)."""
    return slot // block_size, slot % block_size


def store_kvcache(k_bits, v_bits, slot_mapping, k_cache, v_cache) -> None:
    """Write each token's K and V rows (all KV heads) into its slot, in place.

    [NV] §4 store_kvcache_kernel: one program per token reads its slot from
    slot_mapping, returns if the slot is -1, and otherwise copies the
    num_kv_heads*head_dim K and V values to row ``slot`` of k_cache / v_cache.
    Caches are uint16 [num_blocks, block_size, 8, 128].
    """
    for t, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot == -1:
            continue
        blk, off = slot_to_row(slot, k_cache.shape[1])
        k_cache[blk, off] = k_bits[t]
        v_cache[blk, off] = v_bits[t]


# --------------------------------------------------------------------------
# a4/a5: attention through the block table
# --------------------------------------------------------------------------
def gather_kv(k_cache, v_cache, block_table_row, length: int):
    """Logical positions 0..length-1 of one sequence, gathered into contiguous fp64 arrays.

    [Q3] §3.3: block_table maps logical block -> physical block; the row of
    position p is (block_table[p // block_size], p % block_size).  Only the
    first ceil(length / block_size) entries of the row are read.
    """
    bs = k_cache.shape[1]
    pos = np.arange(length)
    blk = np.asarray(block_table_row)[pos // bs]
    off = pos % bs
    return bf16_to_f64(k_cache[blk, off]), bf16_to_f64(v_cache[blk, off])


def causal_gqa_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """Textbook masked softmax attention of one sequence, fp64.

    q [Lq, 32, D]; K, V [Lk, 8, D].  Query row i sits at absolute position
    Lk - Lq + i and sees keys 0..that position (reading: causal alignment to
    the end of the key sequence, the only one under which a decode token and
    a chunk appended after a cached prefix see their whole history; [Q3]
    §3.4).  Scores are q.k * scale, positions after the query are -inf before
    the softmax ([Q3] §1.2), and Q head h reads KV head h // (32/8) (GQA 4:1,
    the grouping repeat_kv materialises in [Q3] §3.4).
    """
    Lq, Lk = q.shape[0], K.shape[0]
    group = q.shape[1] // K.shape[1]
    qpos = Lk - Lq + np.arange(Lq)
    visible = np.arange(Lk)[None, :] <= qpos[:, None]
    out = np.empty(q.shape, dtype=np.float64)
    for h in range(q.shape[1]):
        g = h // group
        S = (q[:, h, :] @ K[:, g, :].T) * scale
        S = np.where(visible, S, -np.inf)
        m = S.max(axis=1, keepdims=True)
        P = np.exp(S - m)
        P = P / P.sum(axis=1, keepdims=True)
        out[:, h, :] = P @ V[:, g, :]
    return out


def paged_decode(q_bits, k_cache, v_cache, context_lens, block_table, scale) -> np.ndarray:
    """One query token per sequence over its cached keys 0..context_len-1.

    [NV] §4 Attention.forward, decode branch: flash_attn_with_kvcache with
    q.unsqueeze(1), cache_seqlens = context_lens, the block table and
    causal=True.  context_lens counts the token stored in this step (the
    store runs before the read, [Q3] §3.4).  Returns fp64 [B, 32, 128].
    """
    q = bf16_to_f64(q_bits)
    out = np.empty(q.shape, dtype=np.float64)
    for b, L in enumerate(np.asarray(context_lens).tolist()):
        K, V = gather_kv(k_cache, v_cache, block_table[b], L)
        out[b : b + 1] = causal_gqa_attention(q[b : b + 1], K, V, scale)
    return out


def paged_prefill(q_bits, k_cache, v_cache, cu_q, cu_k, block_table, scale, seqs=None) -> np.ndarray:
    """Varlen causal prefill: sequence s owns query rows cu_q[s]..cu_q[s+1]-1 and keys 0..Lk-1.

    [NV] §4 Attention.forward, prefill branch with a block table: the keys
    are read from the paged cache (k, v = k_cache, v_cache) with cu_seqlens_q
    / cu_seqlens_k marking the sequences and causal=True; [Q3] §3.2 explains
    that the boundaries replace a [T, T] mask.  Returns fp64 [Tq, 32, 128]
    (rows of sequences not in ``seqs`` are left NaN).
    """
    q = bf16_to_f64(q_bits)
    out = np.full(q.shape, np.nan, dtype=np.float64)
    S = len(cu_q) - 1
    for s in range(S) if seqs is None else seqs:
        q0, q1 = int(cu_q[s]), int(cu_q[s + 1])
        Lk = int(cu_k[s + 1] - cu_k[s])
        if q1 == q0:
            continue
        K, V = gather_kv(k_cache, v_cache, block_table[s], Lk)
        out[q0:q1] = causal_gqa_attention(q[q0:q1], K, V, scale)
    return out


def run_step(wl, k_cache=None, v_cache=None, seqs=None):
    """The whole step for one workload: norm + RoPE, store, then attention.

    Returns (q_out_bits, k_out_bits, k_cache, v_cache, attn_out_f64).  The
    caches are copies of the initial state with this step's rows written.
    """
    if k_cache is None:
        k_cache, v_cache = wl.materialize_cache()
    else:
        k_cache, v_cache = k_cache.copy(), v_cache.copy()
    q_out, k_out = qk_norm_rope(wl.q, wl.k, wl.positions, wl.q_norm_w, wl.k_norm_w)
    store_kvcache(k_out, wl.v, wl.slot_mapping, k_cache, v_cache)
    if wl.mode == "decode":
        if seqs is None:
            out = paged_decode(q_out, k_cache, v_cache, wl.context_lens, wl.block_table, wl.scale)
        else:
            out = np.full(q_out.shape, np.nan)
            sel = np.asarray(seqs)
            out[sel] = paged_decode(q_out[sel], k_cache, v_cache, wl.context_lens[sel], wl.block_table[sel],
                                    wl.scale)
    else:
        out = paged_prefill(q_out, k_cache, v_cache, cu_seqlens(wl.new_lens), cu_seqlens(wl.seq_lens_k),
                            wl.block_table, wl.scale, seqs)
    return q_out, k_out, k_cache, v_cache, out


# --------------------------------------------------------------------------
# Next to the step: residual add fused into the decoder layer's RMSNorm
# --------------------------------------------------------------------------
def rms_norm_rows(x_f64: np.ndarray, w_bits: np.ndarray, eps: float = RMS_EPS) -> np.ndarray:
    """RMSNorm over the last axis of already-widened values -> bf16 bits.

    [Q3] §3.6 add_rms_forward, steps after the sum: the mean of squares of
    the (unrounded) values, scaling by the reciprocal square root of that
    mean plus eps, a cast to the model dtype, then a product with the bf16
    weight that is cast again.  Mean and scaling run in fp64 here.
    """
    x = np.asarray(x_f64, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    normed = f64_to_bf16(x / np.sqrt(ms + eps))
    return f64_to_bf16(bf16_to_f64(normed) * bf16_to_f64(w_bits))


def add_rms_norm(x_bits: np.ndarray, res_bits, w_bits: np.ndarray, eps: float = RMS_EPS):
    """The decoder layer's norm with the pending residual add folded in.

    [Q3] §3.6 (nano-vllm add_rms_forward): the incoming hidden state and the
    residual are widened to fp32 and added; the sum, cast back to bf16, is the
    new residual; the fp32 sum (not the rounded one) is normalised.  With no
    residual (the first layer, Qwen3DecoderLayer.forward's ``residual is
    None`` branch) the input is normalised as it is and is itself the
    residual.  Returns (out_bits, new_residual_bits).

    The sum of two bf16 values is formed exactly in fp64 and rounded once to
    fp32, which is what an fp32 addition returns.
    """
    x = bf16_to_f64(x_bits)
    if res_bits is None:
        return rms_norm_rows(x, w_bits, eps), np.asarray(x_bits, dtype=np.uint16).copy()
    s32 = (x + bf16_to_f64(res_bits)).astype(np.float32).astype(np.float64)
    return rms_norm_rows(s32, w_bits, eps), f64_to_bf16(s32)


def add_rmsnorm_bytes_per_token(hidden: int = HIDDEN, fused: bool = True) -> int:
    """HBM bytes per token of "residual add + RMSNorm" on a bf16 [T, hidden] tensor.

    [Q3] §3.6 traffic model: unfused, the add reads h and r and writes the
    sum, and the norm reads the sum back and writes its output (5 rows);
    fused, one kernel reads h and r and writes the output and the sum
    (4 rows).  The weight row is shared by all tokens and not counted.
    """
    row = 2 * hidden
    return (4 if fused else 5) * row


# --------------------------------------------------------------------------
# Next to the step: the fused QKV projection feeding norm + RoPE + store
# --------------------------------------------------------------------------
QKV_OUT = (NUM_Q_HEADS + 2 * NUM_KV_HEADS) * HEAD_DIM  # 6144


def qkv_projection(x_bits: np.ndarray, w_bits: np.ndarray):
    """One GEMM for q, k and v: [T, 4096] x [6144, 4096]^T -> bf16 q, k, v.

    [Q3] §3.1: nano-vllm's qkv_proj concatenates the q, k and v weights along
    the output dimension (q_size = 32*128, kv_size = 8*128 each, in that
    order), runs one matrix product on hidden_states and splits the result
    [q_size, kv_size, kv_size]; the weight is stored [out, in] as nn.Linear
    stores it.  The product is formed in fp64 (a library matmul) and rounded
    once to bf16, the dtype of the linear layer's output.
    """
    x = bf16_to_f64(x_bits)
    w = bf16_to_f64(w_bits)
    y = f64_to_bf16(x @ w.T)
    T = x.shape[0]
    q = y[:, :NUM_Q_HEADS * HEAD_DIM].reshape(T, NUM_Q_HEADS, HEAD_DIM)
    k = y[:, NUM_Q_HEADS * HEAD_DIM:(NUM_Q_HEADS + NUM_KV_HEADS) * HEAD_DIM].reshape(T, NUM_KV_HEADS, HEAD_DIM)
    v = y[:, (NUM_Q_HEADS + NUM_KV_HEADS) * HEAD_DIM:].reshape(T, NUM_KV_HEADS, HEAD_DIM)
    return q, k, v


def qkv_rope_store(x_bits, w_bits, positions, slot_mapping, q_norm_w, k_norm_w, k_cache, v_cache):
    """Projection, then the step's first part ([NV] §2 Qwen3Attention.forward
    order: qkv_proj, split, q_norm / k_norm, rotary_emb, then the cache store of
    [NV] §4).  Returns q after norm + RoPE; writes k and v into the caches."""
    q, k, v = qkv_projection(x_bits, w_bits)
    q_out, k_out = qk_norm_rope(q, k, positions, q_norm_w, k_norm_w)
    store_kvcache(k_out, v, slot_mapping, k_cache, v_cache)
    return q_out
