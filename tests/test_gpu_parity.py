"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

All five named workloads at full size (every sequence of every batch compared
with the oracle), plus ragged and degenerate cases.
Tolerances are documented in tests/gpu_helpers.py.
"""

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_rmsnorm_gb300 as pkv
from tests.gpu_helpers import (
    GpuStep,
    assert_attn_close,
    check_step,
    from_dev,
    to_dev,
)
from workloads import build_workload, config_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.build()
    pkv.init()
    yield
    torch.cuda.synchronize()


def run_and_check(wl, seqs=None, max_context=None):
    kc0, vc0 = wl.materialize_cache()
    gs = GpuStep(wl, kc0, vc0).run(max_context)
    return gs, check_step(wl, gs, kc0, vc0, seqs)


# ---------------------------------------------------------------- the five workloads
def test_config1_tiny_decode():
    run_and_check(config_workload(1))


def test_config2_varlen_prefill():
    run_and_check(config_workload(2))


def test_config3_batched_decode():
    run_and_check(config_workload(3))


def test_config4_chunked_prefill_shared_prefix():
    wl = config_workload(4)
    gs, _ = run_and_check(wl)
    # shared prefix blocks are read by two sequences and never written
    kc = from_dev(gs.kc)
    for j in range(0, 16, 2):
        n = min(wl.hist_lens[j], wl.hist_lens[j + 1]) // 256
        for b in wl.block_table[j, :n]:
            assert np.array_equal(kc[b], wl.cache_block("k", int(b)))


_LONG_REF: dict = {}


def _long_decode_reference():
    """The oracle's output for every one of the 32 long-context sequences (fp64 [32, 32, 128]).

    The batches 1, 8 and 32 are the first sequences of one workload, so one pass serves all three.
    Each sequence runs alone, its 160 blocks regenerated into a compact pool (bounded host memory:
    about 1 GB per sequence in flight), a few sequences at a time on the host cores.
    """
    if "out" not in _LONG_REF:
        wl = config_workload(5, batch=32)

        def one(s):
            sub = wl.subset([s])
            used = sub.used_blocks()
            remap = {int(b): i for i, b in enumerate(used)}
            kc0 = np.stack([wl.cache_block("k", int(b)) for b in used])
            vc0 = np.stack([wl.cache_block("v", int(b)) for b in used])
            sub.block_table = np.where(sub.block_table >= 0,
                                       np.vectorize(lambda b: remap.get(int(b), -1))(sub.block_table), -1)
            sub.slot_mapping = np.array([remap[int(x) // 256] * 256 + int(x) % 256 for x in sub.slot_mapping],
                                        np.int32)
            sub.num_blocks = len(used)
            return oracle.run_step(sub, kc0, vc0)[4][0]

        with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
            _LONG_REF["out"] = np.stack(list(ex.map(one, range(wl.num_seqs))))
    return _LONG_REF["out"]


@pytest.mark.parametrize("batch", [1, 8, 32])
def test_config5_long_decode(batch):
    wl = config_workload(5, batch=batch)
    gs = GpuStep(wl).run()
    # every sequence of the batch against the oracle, end to end
    assert_attn_close(from_dev(gs.out), _long_decode_reference()[:batch], f"long decode B={batch}")
    # the new token's K/V rows landed in the right slots
    vc = gs.vc.view(-1, 1024)[torch.from_numpy(wl.slot_mapping.astype(np.int64)).cuda()]
    assert np.array_equal(from_dev(vc).reshape(-1, 8, 128), wl.v)


# ---------------------------------------------------------------- ragged and degenerate cases
def test_prefill_ragged_lengths():
    hist = [0, 0, 0, 0, 0, 300, 255, 1000, 5, 64, 0]
    new = [1, 63, 64, 65, 200, 1, 2, 129, 0, 192, 1000]
    run_and_check(build_workload("ragged prefill", "prefill", 31, hist, new, spare_blocks=3))


def test_prefill_at_the_maximum_prompt_length_sampled_rows():
    """One 16,384-token prompt, the longest a config-2 prompt may be (128 query tiles, up to 128 key
    tiles each), then a 300-token prompt.  The oracle's attention is exact per query row, so slices
    of rows are compared with it: the first tile, a slice across the tile boundary in the middle,
    the last tile, and the second prompt whole."""
    L = 16384
    wl = build_workload("max-length prefill", "prefill", 41, [0, 0], [L, 300], spare_blocks=2)
    kc0, vc0 = wl.materialize_cache()
    gs = GpuStep(wl, kc0, vc0).run()
    out = from_dev(gs.out)  # bf16 bits [T, 32, 128]
    q_r, k_r = oracle.qk_norm_rope(wl.q, wl.k, wl.positions, wl.q_norm_w, wl.k_norm_w)
    K, V = oracle.bf16_to_f64(k_r), oracle.bf16_to_f64(wl.v)
    # prompt 0 holds flat rows 0..L-1 at positions 0..L-1; rows a..b-1 see keys 0..b-1
    for a, b in ((0, 128), (8128, 8256), (L - 128, L)):
        ref = oracle.causal_gqa_attention(oracle.bf16_to_f64(q_r[a:b]), K[:b], V[:b], wl.scale)
        assert_attn_close(out[a:b], ref, f"max-length prompt, rows {a}..{b - 1}")
    ref = oracle.causal_gqa_attention(oracle.bf16_to_f64(q_r[L:]), K[L:], V[L:], wl.scale)
    assert_attn_close(out[L:], ref, "the 300-token prompt after it")


def test_decode_ragged_contexts():
    ctx = np.array([1, 2, 15, 16, 17, 63, 64, 65, 255, 256, 257, 511, 512, 513, 1000, 4097, 9000])
    run_and_check(build_workload("ragged decode", "decode", 32, ctx - 1, np.ones(len(ctx), np.int64), spare_blocks=2))


def test_decode_long_single_sequence_splits():
    # one long and one short sequence: the long one is split many ways, the short one is not
    ctx = np.array([20000, 300])
    run_and_check(build_workload("split decode", "decode", 33, ctx - 1, [1, 1], spare_blocks=2))


def test_decode_one_wave_plan_with_mixed_active_splits():
    # 5 sequences -> 40 (sequence, KV head) pairs -> 7 splits of 92 tiles: the sequences use
    # 7, 3, 1, 6 and 1 of them, so some merge many partials and some write bf16 directly
    ctx = np.array([40960, 12345, 777, 30001, 256])
    run_and_check(build_workload("one-wave decode", "decode", 36, ctx - 1, np.ones(len(ctx), np.int64), spare_blocks=2))


def test_decode_on_two_streams_at_once():
    # two split decodes in flight together on two streams: each stream has a workspace of its own
    # (split tickets and partials), so neither merges the other's partials
    wls = [build_workload("stream A", "decode", 37, [29999], [1], spare_blocks=1),
           build_workload("stream B", "decode", 38, [19999, 4999], [1, 1], spare_blocks=1)]
    steps = []
    for wl in wls:
        kc0, vc0 = wl.materialize_cache()
        gs = GpuStep(wl, kc0, vc0)
        gs.store()
        steps.append(gs)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [[], []]
    for _ in range(4):  # several rounds, so the two streams' kernels overlap on the GPU
        for i, (gs, st) in enumerate(zip(steps, streams)):
            with torch.cuda.stream(st):
                outs[i].append(pkv.attn_decode(gs.q, gs.kc, gs.vc, gs.context_lens, gs.block_table,
                                               gs.wl.max_seqlen_k, gs.wl.scale))
    torch.cuda.synchronize()
    assert pkv.check_errors() == []
    ws = [pkv.decode_workspace(gs.wl.num_seqs, gs.wl.max_seqlen_k, stream=st) for gs, st in zip(steps, streams)]
    assert ws[0] is not None and ws[1] is not None and ws[0].data_ptr() != ws[1].data_ptr()
    for i, gs in enumerate(steps):
        wl = gs.wl
        iso = oracle.paged_decode(from_dev(gs.q), from_dev(gs.kc), from_dev(gs.vc), wl.context_lens,
                                  wl.block_table, wl.scale)
        for out in outs[i]:
            assert_attn_close(from_dev(out), iso, f"decode on stream {i}")


def test_decode_split_plans_agree():
    ctx = np.array([3000, 700, 5000])
    wl = build_workload("plans", "decode", 34, ctx - 1, [1, 1, 1], spare_blocks=2)
    # a wider table (padded with -1) admits a larger max_context, which changes the split plan
    wl.block_table = np.concatenate([wl.block_table, np.full((3, 160 - wl.max_blocks_per_seq), -1, np.int32)], 1)
    kc0, vc0 = wl.materialize_cache()
    outs = []
    for mc in (5000, 40960):
        assert mc == 5000 or pkv.decode_workspace_size(3, mc) != pkv.decode_workspace_size(3, 5000)
        gs = GpuStep(wl, kc0, vc0).run(max_context=mc)
        check_step(wl, gs, kc0, vc0)
        outs.append(oracle.bf16_to_f64(from_dev(gs.out)))
    assert np.abs(outs[0] - outs[1]).max() <= 2e-2


def test_empty_inputs_are_no_ops():
    # zero tokens / sequences / queries through the binding: empty tensors (NULL data) are accepted,
    # nothing is written and no error bit is set
    dev = "cuda"
    kc = torch.from_numpy(np.full((2, 256, 8, 128), 0x7FC1, np.uint16).view(np.int16)).to(dev).view(torch.bfloat16)
    vc = kc.clone()
    kc0, vc0 = kc.clone(), vc.clone()
    bf = lambda *shape: torch.empty(shape, dtype=torch.bfloat16, device=dev)
    i32 = lambda *shape: torch.empty(shape, dtype=torch.int32, device=dev)
    w = torch.ones(128, dtype=torch.bfloat16, device=dev)
    pkv.qknorm_rope_store(bf(0, 32, 128), bf(0, 8, 128), bf(0, 8, 128), i32(0), i32(0), w, w, kc, vc)
    assert pkv.attn_decode(bf(0, 32, 128), kc, vc, i32(0), i32(0, 1), 0, 0.088).shape == (0, 32, 128)
    cu = torch.zeros(3, dtype=torch.int32, device=dev)
    bt = torch.full((2, 1), -1, dtype=torch.int32, device=dev)
    assert pkv.attn_prefill(bf(0, 32, 128), kc, vc, cu, cu, bt, 0, 0, 0.088).shape == (0, 32, 128)
    res = bf(0, 4096)
    assert pkv.add_rmsnorm(bf(0, 4096), res, torch.ones(4096, dtype=torch.bfloat16, device=dev)).shape == (0, 4096)
    wqkv = torch.zeros((6144, 4096), dtype=torch.bfloat16, device=dev)
    assert pkv.qkv_rope_store(bf(0, 4096), wqkv, i32(0), i32(0), w, w, kc, vc).shape == (0, 32, 128)
    torch.cuda.synchronize()
    assert pkv.check_errors() == []
    assert torch.equal(kc.view(torch.int16), kc0.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), vc0.view(torch.int16))


def test_single_key_decode_returns_v_exactly():
    wl = build_workload("single key", "decode", 35, [0, 0, 0], [1, 1, 1], spare_blocks=1)
    gs = GpuStep(wl).run()
    out = from_dev(gs.out)
    for b in range(3):
        for h in range(32):
            assert np.array_equal(out[b, h], wl.v[b, h // 4])


def test_decode_empty_context_gives_zero_row():
    wl = build_workload("empty ctx", "decode", 36, [100, 50], [1, 1], spare_blocks=1)
    gs = GpuStep(wl)
    gs.store()
    lens = gs.context_lens.clone()
    lens[1] = 0
    out = pkv.attn_decode(gs.q, gs.kc, gs.vc, lens, gs.block_table, 101, wl.scale)
    assert pkv.check_errors() == []
    o = oracle.bf16_to_f64(from_dev(out))
    assert np.all(o[1] == 0) and np.all(np.isfinite(o[0])) and np.any(o[0] != 0)


def test_store_skips_minus_one_and_accepts_fused_qkv_views():
    wl = build_workload("skip", "prefill", 37, [0, 40], [70, 9], spare_blocks=2, skip_tokens=[3, 71])
    kc0, vc0 = wl.materialize_cache()
    gs = GpuStep(wl, kc0, vc0)
    # q, k, v as column slices of one fused [T, 6144] buffer (nano-vllm's qkv.split)
    T = wl.num_tokens
    fused = torch.empty(T, 6144, dtype=torch.bfloat16, device="cuda")
    fused[:, :4096] = gs.q.view(T, 4096)
    fused[:, 4096:5120] = gs.k.view(T, 1024)
    fused[:, 5120:] = gs.v.view(T, 1024)
    q, k, v = fused.split([4096, 1024, 1024], dim=-1)
    gs.q, gs.k, gs.v = q.view(T, 32, 128), k.view(T, 8, 128), v.view(T, 8, 128)
    assert gs.q.stride(0) == 6144
    gs.store()
    assert pkv.check_errors() == []
    gs.q = gs.q.contiguous()
    # skipped tokens are not in the cache, so only the store is compared
    check_step(wl, gs, kc0, vc0, attn=False)
    assert np.array_equal(from_dev(fused[:, 4096:].contiguous()).reshape(T, 2, 8, 128)[:, 0], wl.k)


def test_out_of_range_inputs_are_flagged_not_written():
    wl = build_workload("flags", "decode", 38, [10, 20, 30], [1, 1, 1], spare_blocks=1)
    kc0, vc0 = wl.materialize_cache()
    gs = GpuStep(wl, kc0, vc0)
    gs.positions[0] = 40960        # position out of range: token 0 skipped
    gs.slots[1] = wl.num_blocks * 256  # slot out of range: token 1 not stored
    q_before = from_dev(gs.q)
    gs.store()
    flags = pkv.check_errors()
    assert set(flags) == {"position", "slot"}
    assert np.array_equal(from_dev(gs.q)[0], q_before[0])
    kc = from_dev(gs.kc)
    assert np.array_equal(kc.reshape(-1, 8, 128)[wl.slot_mapping[1]], kc0.reshape(-1, 8, 128)[wl.slot_mapping[1]])
    # a block id outside the pool: flagged, its keys treated as absent
    bt = gs.block_table.clone()
    bt[2, 0] = wl.num_blocks + 5
    pkv.attn_decode(gs.q, gs.kc, gs.vc, gs.context_lens, bt, 31, wl.scale)
    assert "block_id" in pkv.check_errors()
    # a context longer than its table row
    lens = gs.context_lens.clone()
    lens[0] = 300
    pkv.attn_decode(gs.q, gs.kc, gs.vc, lens, gs.block_table, 256, wl.scale)
    assert "context" in pkv.check_errors()
    assert pkv.check_errors() == []  # cleared


def test_prefill_more_queries_than_keys_is_flagged():
    wl = build_workload("seqlen", "prefill", 39, [0, 0], [40, 30], spare_blocks=1)
    gs = GpuStep(wl)
    gs.store()
    cu_k = gs.cu_k.clone()
    cu_k[2] = cu_k[1] + 10  # sequence 1: 30 queries over 10 keys
    out = pkv.attn_prefill(gs.q, gs.kc, gs.vc, gs.cu_q, cu_k, gs.block_table, 40, 40, wl.scale)
    assert "seqlen" in pkv.check_errors()
    o = oracle.bf16_to_f64(from_dev(out))
    assert np.all(o[40:] == 0) and np.all(np.isfinite(o[:40]))


def test_prefill_longest_first_with_an_unserved_sequence():
    # a cached prefix puts the claims in longest-first order; a sequence with more queries than
    # keys sits among the ordered units, is zeroed and flagged, and the others are unaffected
    wl = build_workload("seqlen, prefixed", "prefill", 44, [1000, 0, 300], [40, 30, 130], spare_blocks=1)
    gs = GpuStep(wl)
    gs.store()
    cu_k = gs.cu_k.clone()  # keys per sequence: 1040, 30, 430
    cu_k[2:] -= 20  # sequence 1: 30 queries over 10 keys; sequence 2 keeps its 430
    assert [int(x) for x in cu_k.diff()] == [1040, 10, 430]
    out = pkv.attn_prefill(gs.q, gs.kc, gs.vc, gs.cu_q, cu_k, gs.block_table, 130, 1040, wl.scale)
    assert "seqlen" in pkv.check_errors()
    q_ref, _, kc_ref, vc_ref, _ = oracle.run_step(wl)
    o = from_dev(out)
    assert np.all(oracle.bf16_to_f64(o[40:70]) == 0)
    q = oracle.bf16_to_f64(q_ref)
    for s, (r0, r1) in ((0, (0, 40)), (2, (70, 200))):
        K, V = oracle.gather_kv(kc_ref, vc_ref, wl.block_table[s], int(wl.seq_lens_k[s]))
        ref = oracle.causal_gqa_attention(q[r0:r1], K, V, wl.scale)
        assert_attn_close(o[r0:r1], ref, f"prefixed prefill sequence {s} next to an unserved one")


@pytest.mark.parametrize("num_seqs", [128, 150])
def test_prefill_many_sequences_with_prefixes(num_seqs):
    # 128 prefixed sequences: the most the longest-first order holds (4 per producer lane);
    # 150: more than that, so prefixed chunks go in tile-index-major order
    rng = np.random.default_rng(45 + num_seqs)
    hist = rng.integers(128, 700, size=num_seqs)
    new = rng.integers(1, 90, size=num_seqs)
    run_and_check(build_workload("many prefixed", "prefill", 45, hist, new, spare_blocks=2))


@pytest.mark.parametrize("mode", ["prefill", "decode"])
def test_no_cross_sequence_leakage(mode):
    # the flat layout and the block tables keep sequences apart ("同一个 Qwen3，两种写法" §3.2, §3.3):
    # rewriting the cache blocks of sequence 1 changes its output and leaves the others' bit for bit
    if mode == "prefill":
        wl = build_workload("leak prefill", "prefill", 52, [0, 300, 0], [700, 200, 130], spare_blocks=2)
    else:
        wl = build_workload("leak decode", "decode", 53, [4999, 299, 9999], [1, 1, 1], spare_blocks=2)
    gs = GpuStep(wl)
    gs.store()
    before = from_dev(gs.attend()).copy()
    n1 = (int(wl.seq_lens_k[1]) + 255) // 256
    own = [int(b) for b in wl.block_table[1, :n1]]
    others = {int(b) for s in (0, 2) for b in wl.block_table[s] if b >= 0}
    assert own and not others.intersection(own)
    g = torch.Generator(device="cuda").manual_seed(54)
    idx = torch.tensor(own, device="cuda", dtype=torch.int64)
    gs.kc[idx] = torch.randn(gs.kc[idx].shape, device="cuda", generator=g).to(torch.bfloat16)
    gs.vc[idx] = torch.randn(gs.vc[idx].shape, device="cuda", generator=g).to(torch.bfloat16)
    after = from_dev(gs.attend())
    assert pkv.check_errors() == []
    rows = np.concatenate([[0], np.cumsum(wl.new_lens)]).astype(np.int64)
    for s in (0, 2):
        assert np.array_equal(before[rows[s]:rows[s + 1]], after[rows[s]:rows[s + 1]]), f"sequence {s} changed"
    assert not np.array_equal(before[rows[1]:rows[2]], after[rows[1]:rows[2]])


def test_prefill_out_of_pool_block_drops_its_keys():
    # one 300-token prompt: table entry 0 holds keys 0..255, entry 1 keys 256..299
    wl = build_workload("bad block prefill", "prefill", 43, [0], [300], spare_blocks=1)
    gs = GpuStep(wl)
    gs.store()
    bt = gs.block_table.clone()
    bt[0, 1] = wl.num_blocks + 3  # entry 1 points outside the pool
    out = pkv.attn_prefill(gs.q, gs.kc, gs.vc, gs.cu_q, gs.cu_k, bt, 300, 300, wl.scale)
    assert "block_id" in pkv.check_errors()
    q_ref, _, kc_ref, vc_ref, _ = oracle.run_step(wl)
    q = oracle.bf16_to_f64(q_ref)
    K, V = oracle.gather_kv(kc_ref, vc_ref, wl.block_table[0], 256)
    # rows 0..255 never see keys past 255; rows 256.. see keys 0..255 only (one query row = all keys visible)
    ref = np.empty_like(q)
    ref[:256] = oracle.causal_gqa_attention(q[:256], K, V, wl.scale)
    for i in range(256, 300):
        ref[i:i + 1] = oracle.causal_gqa_attention(q[i:i + 1], K, V, wl.scale)
    assert_attn_close(from_dev(out), ref, "prefill with an out-of-pool block")


def test_results_are_deterministic():
    wl = config_workload(1)
    a = GpuStep(wl).run()
    b = GpuStep(wl).run()
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))
    assert torch.equal(a.kc.view(torch.int16), b.kc.view(torch.int16))
    wl2 = build_workload("det", "decode", 40, [30000], [1], spare_blocks=1)
    kc0, vc0 = wl2.materialize_cache()
    x = GpuStep(wl2, kc0, vc0).run()
    y = GpuStep(wl2, kc0, vc0).run()
    assert torch.equal(x.out.view(torch.int16), y.out.view(torch.int16))


def test_streams_are_respected():
    wl = config_workload(3)
    kc0, vc0 = wl.materialize_cache()
    gs = GpuStep(wl, kc0, vc0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        gs.store()
        gs.attend()
    s.synchronize()
    assert pkv.check_errors(s) == []
    check_step(wl, gs, kc0, vc0, seqs=[0, 100, 255])
