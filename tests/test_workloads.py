"""The seeded input generators: determinism and the structure each named workload promises."""

import numpy as np

from workloads import BLOCK_SIZE, NAN_BF16, build_workload, config_workload


def test_seeded_and_deterministic():
    a = config_workload(2)
    b = config_workload(2)
    for name in ("q", "k", "v", "positions", "slot_mapping", "block_table", "q_norm_w"):
        assert np.array_equal(getattr(a, name), getattr(b, name))
    c = config_workload(2, seed=5)
    assert not np.array_equal(a.q[:10], c.q[:10])


def test_config1_layout():
    wl = config_workload(1)
    assert wl.context_lens.tolist() == [17, 64, 200, 256]
    assert wl.num_blocks == 8 and wl.positions.tolist() == [16, 63, 199, 255]
    assert len(set(wl.block_table[:, 0].tolist())) == 4


def test_config3_blocks_distinct_and_within_pool():
    wl = config_workload(3)
    lens = wl.context_lens
    assert lens.min() >= 512 and lens.max() <= 4096 and wl.num_seqs == 256
    used = [b for row, L in zip(wl.block_table, lens) for b in row[: (L + 255) // 256]]
    assert len(used) == len(set(used)) and max(used) < 4096


def test_config4_shared_prefix_pairs():
    wl = config_workload(4)
    assert wl.new_lens.tolist() == [512] * 16
    for j in range(0, 16, 2):
        n = min(wl.hist_lens[j], wl.hist_lens[j + 1]) // BLOCK_SIZE
        assert np.array_equal(wl.block_table[j, :n], wl.block_table[j + 1, :n])
        rest_a = set(wl.block_table[j, n:][wl.block_table[j, n:] >= 0].tolist())
        rest_b = set(wl.block_table[j + 1, n:][wl.block_table[j + 1, n:] >= 0].tolist())
        assert not rest_a & rest_b
    shared = set()
    for j in range(0, 16, 2):
        n = min(wl.hist_lens[j], wl.hist_lens[j + 1]) // BLOCK_SIZE
        shared |= set(wl.block_table[j, :n].tolist())
    assert not shared & set((wl.slot_mapping // BLOCK_SIZE).tolist())  # stores never touch shared blocks


def test_config5_batches_are_prefixes():
    w32 = config_workload(5, batch=32)
    w8 = config_workload(5, batch=8)
    assert np.array_equal(w8.block_table, w32.block_table[:8])
    assert np.array_equal(w8.q, w32.q[:8])
    assert w32.context_lens.tolist() == [40960] * 32 and w32.num_blocks == 5120


def test_history_and_sentinels():
    wl = build_workload("hist", "decode", 3, [300, 5], [1, 1], spare_blocks=1)
    kc, vc = wl.materialize_cache()
    b0, b1 = wl.block_table[0, :2]
    assert not np.any(kc[b0] == NAN_BF16) and np.all(kc[b1, 44:] == NAN_BF16)
    assert not np.any(kc[b1, :44] == NAN_BF16)
    assert np.array_equal(kc[b0], wl.cache_block("k", int(b0)))
    assert not np.array_equal(kc[b0], vc[b0])
