"""The attention half of a decoder layer on the GPU, stage by stage against the oracle.

hidden state + residual -> pkv_add_rmsnorm -> pkv_qkv_rope_store (projection,
q/k RMSNorm, RoPE, cache store) -> pkv_attn_prefill over a varlen batch of
three prompts; then one new token per sequence through the same two calls and
pkv_attn_decode.  Each stage is compared with the oracle run on the GPU's own
input to that stage, so rounding differences do not compound (the rules of
the per-call tests: add-norm output within 2 ulp, new residual bit-exact; the
projection's stored V within 1 ulp plus the fp32 sum bound; attention
max-abs <= 2e-2 and mean-abs <= 2e-3), and the attention outputs are also
compared with the oracle's own chain from the first input (end to end, the
attention gates).
"""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_rmsnorm_gb300 as pkv
from tests.gpu_helpers import assert_attn_close, from_dev, to_dev, ulp_bf16
from tests.test_gpu_qkv import EPS_SUM, _close
from workloads import bf16_bits_from_f32

pytestmark = pytest.mark.gpu

SCALE = 128 ** -0.5


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.build()
    pkv.init()
    yield
    torch.cuda.synchronize()


def _bf16(rng, shape, scale=1.0, shift=0.0):
    return bf16_bits_from_f32((shift + scale * rng.standard_normal(shape)).astype(np.float32))


def _check_add_norm(h_gpu, r_gpu, x, r, w):
    h_ref, r_ref = oracle.add_rms_norm(x, r, w)
    assert np.array_equal(r_gpu, r_ref), "new residual differs from the bf16 fp32 sum"
    g, e = oracle.bf16_to_f64(h_gpu), oracle.bf16_to_f64(h_ref)
    assert np.all(np.abs(g - e) <= 2 * ulp_bf16(np.abs(e))), "add + RMSNorm output beyond 2 ulp"
    assert np.mean(h_gpu != h_ref) <= 1e-3


def _check_projection_v(h_gpu, w, slots, vc_gpu, what):
    _, _, v_ref = oracle.qkv_projection(h_gpu, w)
    ok = slots >= 0
    s = slots[ok]
    S = (np.abs(oracle.bf16_to_f64(h_gpu)) @ np.abs(oracle.bf16_to_f64(w[5120:])).T).reshape(-1, 8, 128)[ok]
    _close(vc_gpu[s // 256, s % 256], v_ref[ok], np.abs(oracle.bf16_to_f64(v_ref[ok])), 1, 5e-3, what, EPS_SUM * S)


def test_add_norm_qkv_prefill_then_decode():
    rng = np.random.default_rng(4242)
    lens = [130, 300, 45]
    T = sum(lens)
    nb = 8
    perm = rng.permutation(nb).astype(np.int32)
    table = np.full((3, 2), -1, np.int32)
    table[0, 0], table[1, 0], table[1, 1], table[2, 0] = perm[:4]
    pos = np.concatenate([np.arange(L) for L in lens]).astype(np.int32)
    seq = np.repeat(np.arange(3), lens)
    slots = (table[seq, pos // 256] * 256 + pos % 256).astype(np.int32)
    cu = oracle.cu_seqlens(lens).astype(np.int32)

    x, r = _bf16(rng, (T, 4096)), _bf16(rng, (T, 4096))
    w_ln = _bf16(rng, 4096, 0.1, 1.0)
    w = _bf16(rng, (6144, 4096), 1 / 64)
    wq, wk = _bf16(rng, 128, 0.1, 1.0), _bf16(rng, 128, 0.1, 1.0)
    kc0 = np.full((nb, 256, 8, 128), 0x7FC1, np.uint16)  # rows no store writes hold NaN
    vc0 = kc0.copy()

    # ---------------- GPU: prefill of the three prompts
    kc, vc = to_dev(kc0), to_dev(vc0)
    w_d, wq_d, wk_d, wln_d = to_dev(w), to_dev(wq), to_dev(wk), to_dev(w_ln)
    r_d = to_dev(r)
    h_d = pkv.add_rmsnorm(to_dev(x), r_d, wln_d)
    q_d = pkv.qkv_rope_store(h_d, w_d, to_dev(pos), to_dev(slots), wq_d, wk_d, kc, vc)
    out_d = pkv.attn_prefill(q_d, kc, vc, to_dev(cu), to_dev(cu), to_dev(table), max(lens), max(lens), SCALE)
    torch.cuda.synchronize()
    assert pkv.check_errors() == []
    h, q, out = from_dev(h_d), from_dev(q_d), from_dev(out_d)
    kc1, vc1 = from_dev(kc), from_dev(vc)

    _check_add_norm(h, from_dev(r_d), x, r, w_ln)
    _check_projection_v(h, w, slots, vc1, "prefill: stored V")
    iso = oracle.paged_prefill(q, kc1, vc1, cu, cu, table, SCALE)
    assert_attn_close(out, iso, "prefill attention on the GPU's q and cache")

    h_ref, r_ref = oracle.add_rms_norm(x, r, w_ln)
    kc_ref, vc_ref = kc0.copy(), vc0.copy()
    q_ref = oracle.qkv_rope_store(h_ref, w, pos, slots, wq, wk, kc_ref, vc_ref)
    assert_attn_close(out, oracle.paged_prefill(q_ref, kc_ref, vc_ref, cu, cu, table, SCALE), "prefill, end to end")

    # ---------------- GPU: one decode token per sequence
    x1 = _bf16(rng, (3, 4096))
    r1 = _bf16(rng, (3, 4096))
    pos1 = np.array(lens, np.int32)
    slots1 = (table[np.arange(3), pos1 // 256] * 256 + pos1 % 256).astype(np.int32)
    ctx = pos1 + 1
    r1_d = to_dev(r1)
    h1_d = pkv.add_rmsnorm(to_dev(x1), r1_d, wln_d)
    q1_d = pkv.qkv_rope_store(h1_d, w_d, to_dev(pos1), to_dev(slots1), wq_d, wk_d, kc, vc)
    o1_d = pkv.attn_decode(q1_d, kc, vc, to_dev(ctx), to_dev(table), int(ctx.max()), SCALE)
    torch.cuda.synchronize()
    assert pkv.check_errors() == []
    h1, q1, o1 = from_dev(h1_d), from_dev(q1_d), from_dev(o1_d)
    kc2, vc2 = from_dev(kc), from_dev(vc)

    _check_add_norm(h1, from_dev(r1_d), x1, r1, w_ln)
    _check_projection_v(h1, w, slots1, vc2, "decode: stored V")
    assert np.array_equal(vc2[slots // 256, slots % 256], vc1[slots // 256, slots % 256]), "decode moved prefill rows"
    iso1 = oracle.paged_decode(q1, kc2, vc2, ctx, table, SCALE)
    assert_attn_close(o1, iso1, "decode attention on the GPU's q and cache")

    h1_ref, _ = oracle.add_rms_norm(x1, r1, w_ln)
    q1_ref = oracle.qkv_rope_store(h1_ref, w, pos1, slots1, wq, wk, kc_ref, vc_ref)
    assert_attn_close(o1, oracle.paged_decode(q1_ref, kc_ref, vc_ref, ctx, table, SCALE), "decode, end to end")
