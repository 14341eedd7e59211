"""Helpers for the GPU parity tests: upload a workload, run the step through
the C ABI, and compare against the oracle with the stated tolerances.

Tolerances
* cache rows written by the step: V bit-exact; K within the RoPE bound below;
  every other cache row bit-exact (index handling and NaN sentinels).
* q / k after norm + RoPE (fp32 on the GPU, fp64 in the oracle, both rounded
  to bf16 at the same points): |gpu - oracle| <= 2 ulp_bf16(M), where M is the
  largest magnitude among the result and the two rotated inputs — the error
  of a rotation scales with its inputs, not with a result that cancels — and
  at most 0.1% of the elements may differ at all.
* attention outputs (bf16) against the fp64 oracle: max-abs <= 2e-2 and
  mean-abs <= 2e-3, and no NaN.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_kv_cache_rmsnorm_gb300 as pkv

ATTN_MAX_ABS = 2e-2
ATTN_MEAN_ABS = 2e-3
ROPE_ULPS = 2
ROPE_MISMATCH_FRACTION = 1e-3


def to_dev(a: np.ndarray) -> torch.Tensor:
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def from_dev(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def upload_cache(wl, which: str) -> torch.Tensor:
    """Fill a device cache block-range by block-range (bounded host memory)."""
    dev = torch.empty((wl.num_blocks, 256, 8, 128), dtype=torch.bfloat16, device="cuda")
    step = 256
    for b0 in range(0, wl.num_blocks, step):
        b1 = min(wl.num_blocks, b0 + step)
        host = np.empty((b1 - b0, 256, 8, 128), np.uint16)
        for b in range(b0, b1):
            host[b - b0] = wl.cache_block(which, b)
        dev[b0:b1].copy_(to_dev(host))
    return dev


class GpuStep:
    """One step of a workload on the GPU, through the C ABI."""

    def __init__(self, wl, kc: np.ndarray | None = None, vc: np.ndarray | None = None):
        pkv.build()
        self.wl = wl
        self.q = to_dev(wl.q)
        self.k = to_dev(wl.k)
        self.v = to_dev(wl.v)
        self.positions = to_dev(wl.positions)
        self.slots = to_dev(wl.slot_mapping)
        self.wq = to_dev(wl.q_norm_w)
        self.wk = to_dev(wl.k_norm_w)
        self.kc = to_dev(kc) if kc is not None else upload_cache(wl, "k")
        self.vc = to_dev(vc) if vc is not None else upload_cache(wl, "v")
        self.block_table = to_dev(wl.block_table)
        self.context_lens = to_dev(wl.context_lens)
        self.cu_q = to_dev(wl.cu_seqlens_q)
        self.cu_k = to_dev(wl.cu_seqlens_k)
        self.out = None

    def store(self):
        pkv.qknorm_rope_store(self.q, self.k, self.v, self.positions, self.slots, self.wq, self.wk, self.kc, self.vc)

    def attend(self, max_context=None):
        wl = self.wl
        if wl.mode == "decode":
            self.out = pkv.attn_decode(self.q, self.kc, self.vc, self.context_lens, self.block_table,
                                       max_context or wl.max_seqlen_k, wl.scale)
        else:
            self.out = pkv.attn_prefill(self.q, self.kc, self.vc, self.cu_q, self.cu_k, self.block_table,
                                        wl.max_seqlen_q, wl.max_seqlen_k, wl.scale)
        return self.out

    def run(self, max_context=None):
        self.store()
        self.attend(max_context)
        flags = pkv.check_errors()
        assert flags == [], f"kernels flagged {flags}"
        return self


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def assert_rope_close(gpu_bits: np.ndarray, ref_bits: np.ndarray, pre_rope_bits: np.ndarray, what: str) -> None:
    g = oracle.bf16_to_f64(gpu_bits)
    r = oracle.bf16_to_f64(ref_bits)
    n = oracle.bf16_to_f64(pre_rope_bits)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    partner = np.concatenate([n[..., 64:], n[..., :64]], axis=-1)
    mag = np.maximum(np.abs(r), np.maximum(np.abs(n), np.abs(partner)))
    diff = np.abs(g - r)
    tol = ROPE_ULPS * ulp_bf16(mag)
    bad = diff > tol
    assert not bad.any(), f"{what}: {bad.sum()} elements beyond {ROPE_ULPS} ulp, worst {diff.max():.3g}"
    frac = float(np.mean(gpu_bits != ref_bits))
    assert frac <= ROPE_MISMATCH_FRACTION, f"{what}: {frac:.2%} of elements differ from the oracle"


def assert_attn_close(gpu_bits: np.ndarray, ref: np.ndarray, what: str) -> dict:
    g = oracle.bf16_to_f64(gpu_bits)
    assert np.all(np.isfinite(g)), f"{what}: non-finite outputs"
    err = np.abs(g - ref)
    stats = {"max_abs": float(err.max()) if err.size else 0.0, "mean_abs": float(err.mean()) if err.size else 0.0}
    assert stats["max_abs"] <= ATTN_MAX_ABS, f"{what}: max-abs {stats['max_abs']:.3g}"
    assert stats["mean_abs"] <= ATTN_MEAN_ABS, f"{what}: mean-abs {stats['mean_abs']:.3g}"
    return stats


def written_mask(wl) -> np.ndarray:
    m = np.zeros((wl.num_blocks, 256), bool)
    s = wl.slot_mapping[wl.slot_mapping >= 0]
    m[s // 256, s % 256] = True
    return m


def check_step(wl, gs: GpuStep, kc0: np.ndarray, vc0: np.ndarray, seqs=None, attn: bool = True) -> dict:
    """Compare one finished GPU step with the oracle's run of the same step."""
    q_ref, k_ref, kc_ref, vc_ref, out_ref = oracle.run_step(wl, kc0, vc0, seqs=seqs)
    q_pre = oracle.rms_norm_heads(wl.q, wl.q_norm_w)
    k_pre = oracle.rms_norm_heads(wl.k, wl.k_norm_w)
    assert_rope_close(from_dev(gs.q), q_ref, q_pre, "q after norm+RoPE")
    kc, vc = from_dev(gs.kc), from_dev(gs.vc)
    mask = written_mask(wl)
    assert np.array_equal(kc[~mask], kc0[~mask]), "k_cache rows outside slot_mapping changed"
    assert np.array_equal(vc[~mask], vc0[~mask]), "v_cache rows outside slot_mapping changed"
    assert np.array_equal(vc[mask], vc_ref[mask]), "stored V rows differ from the input bits"
    t_ok = wl.slot_mapping >= 0
    slots = wl.slot_mapping[t_ok]
    assert_rope_close(kc[slots // 256, slots % 256], k_ref[t_ok], k_pre[t_ok], "k stored in the cache")
    if not attn:
        return {}
    out = from_dev(gs.out)
    # isolated: the oracle's attention on the GPU's own q and cache bits, so a
    # difference here can only come from the attention kernel
    qg = from_dev(gs.q)
    if wl.mode == "decode":
        sel = np.arange(wl.num_seqs) if seqs is None else np.asarray(seqs)
        iso = oracle.paged_decode(qg[sel], kc, vc, wl.context_lens[sel], wl.block_table[sel], wl.scale)
        assert_attn_close(out[sel], iso, "attention on the GPU's q and cache")
    else:
        iso = oracle.paged_prefill(qg, kc, vc, oracle.cu_seqlens(wl.new_lens), oracle.cu_seqlens(wl.seq_lens_k),
                                   wl.block_table, wl.scale, seqs)
        rows = slice(None) if seqs is None else _rows_of(wl, seqs)
        assert_attn_close(out[rows], iso[rows], "attention on the GPU's q and cache")
    # end to end: against the oracle's own norm, RoPE and store
    if seqs is None:
        return assert_attn_close(out, out_ref, "attention")
    rows = _rows_of(wl, seqs)
    return assert_attn_close(out[rows], out_ref[rows], "attention (sampled sequences)")


def _rows_of(wl, seqs):
    cu = wl.cu_seqlens_q
    return np.concatenate([np.arange(cu[s], cu[s + 1]) for s in seqs])
