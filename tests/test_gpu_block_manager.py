"""The block manager drives the attention step on the GPU (shared prefix, chunked prefill, decode).

Sequence A is prefilled whole; sequence B shares A's first two full blocks,
so the manager reports 512 cached tokens and B's prefill stores and attends
only its remaining tokens, reading the prefix keys from A's blocks; then B
decodes one token into the slot the manager hands out.  Each output is
compared with the oracle's attention over the sequence's full, contiguous
K/V (tolerances of the other attention parity tests).
"""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_rmsnorm_gb300 as pkv
from paged_kv_cache_rmsnorm_gb300.block_manager import BlockManager
from tests.gpu_helpers import assert_attn_close, from_dev, to_dev
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


def _normal(rng, shape):
    return bf16_bits_from_f32(rng.standard_normal(shape).astype(np.float32))


def test_shared_prefix_chunked_prefill_and_decode_through_the_manager():
    rng = np.random.default_rng(77)
    nb = 24
    bm = BlockManager(nb)
    wq = bf16_bits_from_f32((1 + 0.1 * rng.standard_normal(128)).astype(np.float32))
    wk = bf16_bits_from_f32((1 + 0.1 * rng.standard_normal(128)).astype(np.float32))
    LA, LB = 700, 900
    ids_a = rng.integers(0, 150000, LA)
    ids_b = np.concatenate([ids_a[:600], rng.integers(0, 150000, LB - 600)])  # 512 tokens = 2 full shared blocks
    # per-position inputs; the shared prefix has the same q/k/v in both sequences
    q_a, k_a, v_a = _normal(rng, (LA, 32, 128)), _normal(rng, (LA, 8, 128)), _normal(rng, (LA, 8, 128))
    q_b, k_b, v_b = _normal(rng, (LB, 32, 128)), _normal(rng, (LB, 8, 128)), _normal(rng, (LB, 8, 128))
    k_b[:600], v_b[:600], q_b[:600] = k_a[:600], v_a[:600], q_a[:600]

    # every slot no store writes holds NaN: an output that reads one shows it
    kc = torch.full((nb, 256, 8, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = kc.clone()

    def run_prefill(seq, q, k, v):
        slots, pos, cu_q, cu_k, table = bm.prefill_batch([seq])
        sl = slice(int(pos[0]), int(pos[-1]) + 1)
        qd = to_dev(q[sl])
        pkv.qknorm_rope_store(qd, to_dev(k[sl]), to_dev(v[sl]), to_dev(pos), to_dev(slots), to_dev(wq), to_dev(wk),
                              kc, vc)
        out = pkv.attn_prefill(qd, kc, vc, to_dev(cu_q), to_dev(cu_k), to_dev(table), int(cu_q[-1]),
                               int(cu_k[-1]), SCALE)
        torch.cuda.synchronize()
        assert pkv.check_errors() == []
        return from_dev(out), int(pos[0])

    def reference(q, k, v, first_row):
        n = k.shape[0]
        qr, kr = oracle.qk_norm_rope(q, k, np.arange(n), wq, wk)
        return oracle.causal_gqa_attention(oracle.bf16_to_f64(qr[first_row:]), oracle.bf16_to_f64(kr),
                                           oracle.bf16_to_f64(v), SCALE)

    assert bm.allocate(0, ids_a) == 0
    out_a, first = run_prefill(0, q_a, k_a, v_a)
    assert first == 0
    assert_attn_close(out_a, reference(q_a, k_a, v_a, 0), "sequence A, whole prompt")

    assert bm.allocate(1, ids_b) == 512
    ta, tb = bm.block_table([0])[0], bm.block_table([1])[0]
    assert list(ta[:2]) == list(tb[:2]) and bm.ref_count(int(ta[0])) == 2
    out_b, first = run_prefill(1, q_b, k_b, v_b)
    assert first == 512
    assert_attn_close(out_b, reference(q_b, k_b, v_b, 512), "sequence B after its cached prefix")

    # one decode step of B: the new token's slot comes from the manager
    q_n, k_n, v_n = _normal(rng, (1, 32, 128)), _normal(rng, (1, 8, 128)), _normal(rng, (1, 8, 128))
    slot = bm.append(1, 12345)
    qd = to_dev(q_n)
    pkv.qknorm_rope_store(qd, to_dev(k_n), to_dev(v_n), to_dev(np.array([LB], np.int32)),
                          to_dev(np.array([slot], np.int32)), to_dev(wq), to_dev(wk), kc, vc)
    ctx = to_dev(np.array([LB + 1], np.int32))
    out = pkv.attn_decode(qd, kc, vc, ctx, to_dev(bm.block_table([1])), LB + 1, SCALE)
    torch.cuda.synchronize()
    assert pkv.check_errors() == []
    qq = np.concatenate([q_b, q_n]), np.concatenate([k_b, k_n]), np.concatenate([v_b, v_n])
    assert_attn_close(from_dev(out), reference(*qq, LB), "sequence B, decode step")
