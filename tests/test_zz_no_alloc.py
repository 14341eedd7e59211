"""pkv_attn_decode_noalloc against pkv_attn_decode (GPU).

The no-allocation variant is for callers that cannot allocate device memory
(a sealed memory pool, an allocator-free embedding): instead of a caller
workspace it uses a static scratch array inside the library.  Its output must
match the workspace-based entry point's within the attention tolerance of the
other GPU tests, on two calls in a row (the second call reuses the scratch the
first one left behind).  This file is collected last on purpose.
"""

import numpy as np
import pytest
import torch

import paged_kv_cache_rmsnorm_gb300 as pkv
from tests.gpu_helpers import ATTN_MAX_ABS, ATTN_MEAN_ABS, GpuStep
from workloads import build_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.build()
    yield
    torch.cuda.synchronize()


@pytest.mark.parametrize("ctx", [[20000, 3000, 777], [40960], [1, 300, 5000, 257]])
def test_noalloc_decode_matches_workspace_decode(ctx):
    ctx = np.array(ctx)
    wl = build_workload("no-alloc decode", "decode", 41 + len(ctx), ctx - 1, np.ones(len(ctx), np.int64),
                        spare_blocks=2)
    assert pkv.decode_workspace_size(wl.num_seqs, wl.max_seqlen_k) > 0  # the split path, i.e. scratch, is used
    kc0, vc0 = wl.materialize_cache()
    gs = GpuStep(wl, kc0, vc0)
    gs.store()
    ref = pkv.attn_decode(gs.q, gs.kc, gs.vc, gs.context_lens, gs.block_table, wl.max_seqlen_k, wl.scale)
    assert pkv.check_errors() == []
    ref_f = ref.float()
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = [torch.full_like(gs.q, float("nan")) for _ in range(2)]
    torch.cuda.synchronize()
    before = torch.cuda.memory_allocated()
    for out in outs:  # two calls in a row share the static scratch
        pkv.attn_decode_noalloc(gs.q, gs.kc, gs.vc, gs.context_lens, gs.block_table, wl.max_seqlen_k, wl.scale,
                                out, error_flags=flags)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == before
    assert int(flags.item()) == 0
    for out in outs:
        err = (out.float() - ref_f).abs()
        assert torch.isfinite(out.float()).all()
        assert err.max().item() <= ATTN_MAX_ABS and err.mean().item() <= ATTN_MEAN_ABS


def test_noalloc_decode_without_split_and_default_error_word():
    wl = build_workload("no-alloc short", "decode", 49, [10, 100], [1, 1], spare_blocks=1)
    gs = GpuStep(wl)
    gs.store()
    ref = pkv.attn_decode(gs.q, gs.kc, gs.vc, gs.context_lens, gs.block_table, wl.max_seqlen_k, wl.scale)
    out = torch.empty_like(gs.q)
    pkv.attn_decode_noalloc(gs.q, gs.kc, gs.vc, gs.context_lens, gs.block_table, wl.max_seqlen_k, wl.scale, out)
    torch.cuda.synchronize()
    assert (out.float() - ref.float()).abs().max().item() <= ATTN_MAX_ABS
