"""CUDA-graph replay of store + decode equals the eager launches, step after step (GPU)."""

import numpy as np
import pytest
import torch

import paged_kv_cache_rmsnorm_gb300 as pkv
from paged_kv_cache_rmsnorm_gb300.graphs import DecodeGraph
from tests.gpu_helpers import GpuStep, check_step, from_dev, to_dev
from workloads import bf16_bits_from_f32, config_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.build()
    pkv.init()
    yield
    torch.cuda.synchronize()


def _step_inputs(rng, wl):
    q = bf16_bits_from_f32(rng.standard_normal(wl.q.shape).astype(np.float32))
    k = bf16_bits_from_f32(rng.standard_normal(wl.k.shape).astype(np.float32))
    v = bf16_bits_from_f32(rng.standard_normal(wl.v.shape).astype(np.float32))
    return q, k, v


@pytest.mark.parametrize("cfg", [1, 3])
def test_graph_replay_matches_eager_over_steps(cfg):
    wl = config_workload(cfg)
    kc0, vc0 = wl.materialize_cache()
    eager = GpuStep(wl, kc0, vc0)  # its own buffers and cache
    # the graph's fixed buffers
    q, k, v = to_dev(wl.q), to_dev(wl.k), to_dev(wl.v)
    pos, slots = to_dev(wl.positions), to_dev(wl.slot_mapping)
    wq, wk = to_dev(wl.q_norm_w), to_dev(wl.k_norm_w)
    kc, vc = to_dev(kc0), to_dev(vc0)
    ctx, bt = to_dev(wl.context_lens), to_dev(wl.block_table)
    g = DecodeGraph(q, k, v, pos, slots, wq, wk, kc, vc, ctx, bt, wl.max_seqlen_k, wl.scale).capture()
    # the warm-up launch of capture() ran on the buffers: put the step's state back
    kc.copy_(to_dev(kc0))
    vc.copy_(to_dev(vc0))
    rng = np.random.default_rng(500 + cfg)
    for step in range(3):
        qs, ks, vs = (wl.q, wl.k, wl.v) if step == 0 else _step_inputs(rng, wl)
        q.copy_(to_dev(qs)), k.copy_(to_dev(ks)), v.copy_(to_dev(vs))
        out_g = g.replay()
        eager.q.copy_(to_dev(qs)), eager.k.copy_(to_dev(ks)), eager.v.copy_(to_dev(vs))
        eager.store()
        eager.attend()
        torch.cuda.synchronize()
        assert pkv.check_errors() == []
        assert torch.equal(out_g.view(torch.int16), eager.out.view(torch.int16)), f"step {step}: outputs differ"
        assert torch.equal(kc.view(torch.int16), eager.kc.view(torch.int16)), f"step {step}: K caches differ"
        assert torch.equal(vc.view(torch.int16), eager.vc.view(torch.int16)), f"step {step}: V caches differ"
        if step == 0:
            # and the first step is the oracle's step (same inputs as the parity tests)
            check_step(wl, eager, kc0, vc0)
