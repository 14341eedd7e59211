"""pkv_add_rmsnorm on the GPU against the fp64 oracle (residual add folded into RMSNorm).

Tolerances: the new residual (the fp32 sum rounded to bf16) is bit-exact; the
normalised output may differ from the oracle only where the fp32 sum of
squares and rsqrt land on the other side of a bf16 rounding tie.  The
normalised value is rounded to bf16 before the weight multiply, so one ulp
there can become two ulps of a product that falls into the binade below: the
bound is 2 ulp_bf16 of the output's magnitude (the rule of the q/k norm),
on at most 0.1% of the elements.
"""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_rmsnorm_gb300 as pkv
from tests.gpu_helpers import from_dev, to_dev, ulp_bf16
from workloads import bf16_bits_from_f32

pytestmark = pytest.mark.gpu

NORM_ULPS = 2
NORM_MISMATCH_FRACTION = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.build()
    pkv.init()
    yield
    torch.cuda.synchronize()


def _inputs(seed, T, scale_r=1.0):
    rng = np.random.default_rng(seed)
    x = bf16_bits_from_f32(rng.standard_normal((T, oracle.HIDDEN)).astype(np.float32))
    r = bf16_bits_from_f32((scale_r * rng.standard_normal((T, oracle.HIDDEN))).astype(np.float32))
    w = bf16_bits_from_f32((1 + 0.1 * rng.standard_normal(oracle.HIDDEN)).astype(np.float32))
    return x, r, w


def _assert_norm_close(gpu_bits, ref_bits, what):
    g, r = oracle.bf16_to_f64(gpu_bits), oracle.bf16_to_f64(ref_bits)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    bad = np.abs(g - r) > NORM_ULPS * ulp_bf16(np.abs(r))
    assert not bad.any(), f"{what}: {bad.sum()} elements beyond {NORM_ULPS} ulp"
    frac = float(np.mean(gpu_bits != ref_bits))
    assert frac <= NORM_MISMATCH_FRACTION, f"{what}: {frac:.3%} of elements differ"


@pytest.mark.parametrize("T", [1, 3, 457, 2048])
def test_add_rmsnorm_matches_oracle(T):
    x, r, w = _inputs(100 + T, T, scale_r=3.0)
    ref_out, ref_res = oracle.add_rms_norm(x, r, w)
    xd, rd, wd = to_dev(x), to_dev(r), to_dev(w)
    out = pkv.add_rmsnorm(xd, rd, wd)
    torch.cuda.synchronize()
    assert np.array_equal(from_dev(rd), ref_res), "new residual differs from the bf16 fp32 sum"
    assert np.array_equal(from_dev(xd), x), "x was modified"
    _assert_norm_close(from_dev(out), ref_out, f"add_rmsnorm T={T}")


def test_first_layer_without_residual_and_in_place():
    x, _, w = _inputs(7, 300)
    ref_out, _ = oracle.add_rms_norm(x, None, w)
    xd, wd = to_dev(x), to_dev(w)
    out = pkv.add_rmsnorm(xd, None, wd)
    torch.cuda.synchronize()
    _assert_norm_close(from_dev(out), ref_out, "rmsnorm without residual")
    # in place (out = x) gives the same values
    pkv.add_rmsnorm(xd, None, wd, out=xd)
    torch.cuda.synchronize()
    assert np.array_equal(from_dev(xd), from_dev(out))


def test_add_rmsnorm_at_the_prefill_batch_size():
    # the 10,780-token batch of the varlen-prefill workload; every 7th row checked
    T = 10780
    x, r, w = _inputs(9, T, scale_r=2.0)
    xd, rd, wd = to_dev(x), to_dev(r), to_dev(w)
    out = pkv.add_rmsnorm(xd, rd, wd)
    torch.cuda.synchronize()
    rows = np.arange(0, T, 7)
    ref_out, ref_res = oracle.add_rms_norm(x[rows], r[rows], w)
    assert np.array_equal(from_dev(rd)[rows], ref_res)
    _assert_norm_close(from_dev(out)[rows], ref_out, "add_rmsnorm T=10780 (sampled rows)")


def test_deterministic_and_extreme_rows():
    x, r, w = _inputs(21, 64)
    # rows of very small and very large magnitude, a row of zeros plus residual, an all-zero row
    x[0] = bf16_bits_from_f32(np.full(oracle.HIDDEN, 1e-20, np.float32))
    x[1] = bf16_bits_from_f32(np.full(oracle.HIDDEN, 3e4, np.float32))
    x[2] = 0
    x[3] = 0
    r[3] = 0
    ref_out, ref_res = oracle.add_rms_norm(x, r, w)
    a = pkv.add_rmsnorm(to_dev(x), to_dev(r), to_dev(w))
    rd = to_dev(r)
    b = pkv.add_rmsnorm(to_dev(x), rd, to_dev(w))
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert np.array_equal(from_dev(rd), ref_res)
    assert np.all(from_dev(b)[3] == 0)  # 0 * rsqrt(eps) = 0
    _assert_norm_close(from_dev(b), ref_out, "extreme rows")
