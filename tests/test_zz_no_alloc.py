"""pkv_attn_decode_noalloc against pkv_attn_decode and the oracle (GPU).

The no-allocation variant serves callers that cannot allocate device memory
(code inside a sealed memory pool, an allocator-free embedding, a process that
has handed out all of its device memory up front): instead of a caller
workspace it uses a static scratch array inside the library.  It runs the same
kernel with the same split plan as pkv_attn_decode, so on two calls in a row
(the second one finds the scratch as the first left it) its output must be
bit-identical to pkv_attn_decode's, and both must match the oracle within the
attention tolerance of the other GPU tests.  Free device memory, as the driver
reports it, must not change across the two calls.  This file is collected last
on purpose, and passes alone in a fresh process as well as after the others.
"""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_rmsnorm_gb300 as pkv
from tests.gpu_helpers import GpuStep, assert_attn_close, from_dev
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
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    warm = torch.empty_like(gs.q)
    outs = [torch.full_like(gs.q, float("nan")) for _ in range(2)]
    # a first call on the device loads the kernel's module (and with it the static scratch);
    # after that, the calls must leave the driver's free-memory figure unchanged
    pkv.attn_decode_noalloc(gs.q, gs.kc, gs.vc, gs.context_lens, gs.block_table, wl.max_seqlen_k, wl.scale,
                            warm, error_flags=flags)
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for out in outs:  # two calls in a row share the static scratch
        pkv.attn_decode_noalloc(gs.q, gs.kc, gs.vc, gs.context_lens, gs.block_table, wl.max_seqlen_k, wl.scale,
                                out, error_flags=flags)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
    assert int(flags.item()) == 0
    for out in outs:
        # same kernel, same split plan: bit for bit the workspace entry point's result
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    # and the oracle's attention on the GPU's own q and cache bits
    iso = oracle.paged_decode(from_dev(gs.q), from_dev(gs.kc), from_dev(gs.vc), wl.context_lens, wl.block_table,
                              wl.scale)
    assert_attn_close(from_dev(outs[1]), iso, "no-alloc decode against the oracle")


def test_noalloc_decode_without_split_and_default_error_word():
    wl = build_workload("no-alloc short", "decode", 49, [10, 100], [1, 1], spare_blocks=1)
    gs = GpuStep(wl)
    gs.store()
    ref = pkv.attn_decode(gs.q, gs.kc, gs.vc, gs.context_lens, gs.block_table, wl.max_seqlen_k, wl.scale)
    out = torch.empty_like(gs.q)
    pkv.attn_decode_noalloc(gs.q, gs.kc, gs.vc, gs.context_lens, gs.block_table, wl.max_seqlen_k, wl.scale, out)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert pkv.check_errors() == []  # also reads (and clears) the no-alloc call's own error word


def test_noalloc_default_error_word_reaches_check_errors():
    # an out-of-pool block id is flagged in the kernel; without an error word of its own the
    # no-alloc call leaves the bit in the library's static word, which pkv_check_errors reports
    wl = build_workload("no-alloc bad block", "decode", 50, [600], [1], spare_blocks=1)
    gs = GpuStep(wl)
    gs.store()
    assert pkv.check_errors() == []
    bt = gs.block_table.clone()
    bt[0, 1] = wl.num_blocks + 5
    out = torch.empty_like(gs.q)
    pkv.attn_decode_noalloc(gs.q, gs.kc, gs.vc, gs.context_lens, bt, wl.max_seqlen_k, wl.scale, out)
    torch.cuda.synchronize()
    assert pkv.check_errors() == ["block_id"]
    assert pkv.check_errors() == []  # read once, then cleared
