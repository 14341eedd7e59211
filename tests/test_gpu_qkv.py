"""pkv_qkv_rope_store (QKV projection + norm + RoPE + scatter) against the oracle (GPU).

Tolerances, derived from the arithmetic: the projection sums K = 4096
products in fp32 (on the tensor core) against the oracle's fp64; the rounding
error of such a sum is at most K * 2^-24 * sum_i |x_i w_i| = 2^-12 * S (S the
sum of absolute products of that output), usually far less, so the bf16
projection can differ from the oracle's by one ulp near rounding ties (on
roughly 0.1-0.3% of elements) and, for outputs much smaller than S, by up to
2^-12 * S.  Through the norm (division by the head's rms) and the weight
multiply (two bf16 roundings) one ulp can become two of the binade below; the
rotation adds two such terms weighted by |cos| and |sin| (sum at most
sqrt(2)).  Element bounds: v within 1 ulp + 2^-12 * S; q and stored k within
3 ulp of the magnitude of the rotated inputs + 2^-12 * 2.2 * S / rms (2.2 >=
|weight| * sqrt(2) for weights near 1).  Fractions of differing elements:
at most 1% for q and k, 0.5% for v.  Every cache row not named by
slot_mapping is untouched.  With selection weights (one nonzero product per
output) the projection is exact: v bit-exact, q/k by the plain store's rule
(2 ulp, 0.1%).
"""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_rmsnorm_gb300 as pkv
from tests.gpu_helpers import from_dev, to_dev, ulp_bf16
from workloads import bf16_bits_from_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.build()
    pkv.init()
    yield
    torch.cuda.synchronize()


EPS_SUM = 2.0 ** -12  # K * 2^-24 for K = 4096


def _close(gpu_bits, ref_bits, mag, ulps, max_frac, what, abs_tol=0.0):
    g, r = oracle.bf16_to_f64(gpu_bits), oracle.bf16_to_f64(ref_bits)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    bad = np.abs(g - r) > ulps * ulp_bf16(mag) + abs_tol
    assert not bad.any(), f"{what}: {bad.sum()} elements beyond {ulps} ulp"
    frac = float(np.mean(gpu_bits != ref_bits)) if gpu_bits.size else 0.0
    assert frac <= max_frac, f"{what}: {frac:.3%} of elements differ"


def _case(seed, T, nb, weight=None, skip_every=0):
    rng = np.random.default_rng(seed)
    x = bf16_bits_from_f32(rng.standard_normal((T, oracle.HIDDEN)).astype(np.float32))
    w = weight if weight is not None else bf16_bits_from_f32(
        (rng.standard_normal((oracle.QKV_OUT, oracle.HIDDEN)) / 64).astype(np.float32))
    wq = bf16_bits_from_f32((1 + 0.1 * rng.standard_normal(128)).astype(np.float32))
    wk = bf16_bits_from_f32((1 + 0.1 * rng.standard_normal(128)).astype(np.float32))
    pos = rng.integers(0, oracle.MAX_POSITION, T).astype(np.int32)
    slots = rng.permutation(nb * 256)[:T].astype(np.int32)
    if skip_every:
        slots[3::skip_every] = -1
    kc0 = np.full((nb, 256, 8, 128), 0x7FC1, np.uint16)
    vc0 = kc0.copy()
    return x, w, wq, wk, pos, slots, kc0, vc0


def _run(x, w, wq, wk, pos, slots, kc0, vc0):
    kc, vc = to_dev(kc0), to_dev(vc0)
    q = pkv.qkv_rope_store(to_dev(x), to_dev(w), to_dev(pos), to_dev(slots), to_dev(wq), to_dev(wk), kc, vc)
    torch.cuda.synchronize()
    return from_dev(q), from_dev(kc), from_dev(vc)


def _reference(x, w, wq, wk, pos, slots, kc0, vc0):
    kc, vc = kc0.copy(), vc0.copy()
    q = oracle.qkv_rope_store(x, w, pos, slots, wq, wk, kc, vc)
    _, kpre, vpre = oracle.qkv_projection(x, w)
    return q, kc, vc, kpre, vpre


def _check(case, frac_qk, frac_v, what, ulps_qk=3):
    x, w, wq, wk, pos, slots, kc0, vc0 = case
    q, kc, vc = _run(*case)
    assert pkv.check_errors() == []
    q_ref, kc_ref, vc_ref, _, _ = _reference(*case)
    # magnitude for the q/k rule: the rotated pair's inputs (projection, normed) and the result
    qp, kp, _ = oracle.qkv_projection(x, w)
    qn = oracle.bf16_to_f64(oracle.rms_norm_heads(qp, wq))
    mag_q = np.maximum(np.abs(oracle.bf16_to_f64(q_ref)), np.maximum(np.abs(qn), np.abs(np.roll(qn, 64, axis=-1))))
    S = np.abs(oracle.bf16_to_f64(x)) @ np.abs(oracle.bf16_to_f64(w)).T  # [T, 6144]
    S_q, S_k, S_v = S[:, :4096].reshape(-1, 32, 128), S[:, 4096:5120].reshape(-1, 8, 128), S[:, 5120:].reshape(-1, 8, 128)
    rms_q = np.sqrt(np.mean(oracle.bf16_to_f64(qp) ** 2, axis=-1, keepdims=True)) + 1e-30
    exact = ulps_qk == 2
    _close(q, q_ref, mag_q, ulps_qk, frac_qk, f"{what}: q", 0.0 if exact else EPS_SUM * 2.2 * S_q / rms_q)
    written = slots >= 0
    s = slots[written]
    kn = oracle.bf16_to_f64(oracle.rms_norm_heads(kp, wk))[written]
    k_ref = kc_ref[s // 256, s % 256]
    mag_k = np.maximum(np.abs(oracle.bf16_to_f64(k_ref)), np.maximum(np.abs(kn), np.abs(np.roll(kn, 64, axis=-1))))
    rms_k = np.sqrt(np.mean(oracle.bf16_to_f64(kp[written]) ** 2, axis=-1, keepdims=True)) + 1e-30
    _close(kc[s // 256, s % 256], k_ref, mag_k, ulps_qk, frac_qk, f"{what}: k cache",
           0.0 if exact else EPS_SUM * 2.2 * S_k[written] / rms_k)
    v_ref = vc_ref[s // 256, s % 256]
    _close(vc[s // 256, s % 256], v_ref, np.abs(oracle.bf16_to_f64(v_ref)), 1, frac_v, f"{what}: v cache",
           0.0 if exact else EPS_SUM * S_v[written])
    untouched = np.ones((kc0.shape[0], 256), bool)
    untouched[s // 256, s % 256] = False
    assert np.array_equal(kc[untouched], kc0[untouched]) and np.array_equal(vc[untouched], vc0[untouched])


# tiles are 256 tokens on a CTA pair (128 per CTA): sizes around both boundaries, and a
# second CTA with no rows at all (T = 1, 128)
@pytest.mark.parametrize("T", [1, 128, 130, 256, 300, 384])
def test_qkv_rope_store_matches_oracle(T):
    _check(_case(200 + T, T, nb=4, skip_every=7), 1e-2, 5e-3, f"T={T}")


def test_qkv_rope_store_exact_projection_with_selection_weights():
    # one nonzero product per output: the projection is exact, so only the norm/RoPE rule remains
    w = np.zeros((oracle.QKV_OUT, oracle.HIDDEN), np.uint16)
    f = np.arange(oracle.QKV_OUT)
    w[f, (f * 7 + 3) % oracle.HIDDEN] = bf16_bits_from_f32(np.array([1.0], np.float32))[0]
    case = _case(9, 257, nb=2, weight=w)
    x, w_, wq, wk, pos, slots, kc0, vc0 = case
    q, kc, vc = _run(*case)
    q_ref, kc_ref, vc_ref, _, vpre = _reference(*case)
    s = slots[slots >= 0]
    assert np.array_equal(vc[s // 256, s % 256], vc_ref[s // 256, s % 256])  # v = exact selection
    _check(case, 1e-3, 0.0, "selection weights", ulps_qk=2)


def test_qkv_rope_store_at_the_prefill_batch_size():
    # the 10,780-token batch of the varlen-prefill workload; every 11th token checked
    T = 10780
    case = _case(10, T, nb=48)
    x, w, wq, wk, pos, slots, kc0, vc0 = case
    q, kc, vc = _run(*case)
    assert pkv.check_errors() == []
    rows = np.arange(0, T, 11)
    sub = (x[rows], w, wq, wk, pos[rows], slots[rows], kc0, vc0)
    q_ref, kc_ref, vc_ref, _, _ = _reference(*sub)
    qp, kp, _ = oracle.qkv_projection(x[rows], w)
    qn = oracle.bf16_to_f64(oracle.rms_norm_heads(qp, wq))
    mag_q = np.maximum(np.abs(oracle.bf16_to_f64(q_ref)), np.maximum(np.abs(qn), np.abs(np.roll(qn, 64, axis=-1))))
    S = np.abs(oracle.bf16_to_f64(x[rows])) @ np.abs(oracle.bf16_to_f64(w)).T
    rms_q = np.sqrt(np.mean(oracle.bf16_to_f64(qp) ** 2, axis=-1, keepdims=True)) + 1e-30
    _close(q[rows], q_ref, mag_q, 3, 1e-2, "T=10780 q (sampled)", EPS_SUM * 2.2 * S[:, :4096].reshape(-1, 32, 128) / rms_q)
    s = slots[rows]
    _close(vc[s // 256, s % 256], vc_ref[s // 256, s % 256], np.abs(oracle.bf16_to_f64(vc_ref[s // 256, s % 256])), 1,
           5e-3, "T=10780 v (sampled)", EPS_SUM * S[:, 5120:].reshape(-1, 8, 128))


def test_qkv_rope_store_flags_bad_positions_and_slots():
    case = list(_case(11, 40, nb=1))
    case[4] = case[4].copy()
    case[5] = case[5].copy()
    case[4][3] = oracle.MAX_POSITION  # position out of range: token 3 skipped entirely
    case[5][5] = 10 ** 6              # slot out of range: token 5's K/V not stored
    x, w, wq, wk, pos, slots, kc0, vc0 = case
    q_before = np.zeros((40, 32, 128), np.uint16)
    qd = to_dev(q_before)
    kc, vc = to_dev(kc0), to_dev(vc0)
    pkv.qkv_rope_store(to_dev(x), to_dev(w), to_dev(pos), to_dev(slots), to_dev(wq), to_dev(wk), kc, vc, q_out=qd)
    assert set(pkv.check_errors()) == {"position", "slot"}
    assert np.all(from_dev(qd)[3] == 0)
