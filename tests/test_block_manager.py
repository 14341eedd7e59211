"""The host-side block manager (C++ in libpkv.so) on CPU.

Pinned three ways: the FNV-1a model to its published test vectors; the
library against the plain Python model (oracle/block_manager.py) over random
operation sequences, bit for bit; and the properties the pages state for the
paged cache (slot = block * 256 + offset, shared prefixes stored once with a
reference count, fixed-size blocks returned to the pool).
"""

import numpy as np
import pytest

from oracle.block_manager import BLOCK, BlockManagerModel, fnv1a64
from paged_kv_cache_rmsnorm_gb300 import PkvError
from paged_kv_cache_rmsnorm_gb300.block_manager import BlockManager


def test_fnv1a_published_vectors():
    assert fnv1a64(b"") == 0xCBF29CE484222325
    assert fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert fnv1a64(b"foobar") == 0x85944171F73967E8


def test_shared_prefix_is_stored_once():
    bm = BlockManager(16)
    rng = np.random.default_rng(0)
    prefix = rng.integers(0, 150000, 2 * BLOCK)
    a = np.concatenate([prefix, rng.integers(0, 150000, 100)])
    b = np.concatenate([prefix, rng.integers(0, 150000, 300)])
    assert bm.allocate(1, a) == 0
    assert bm.allocate(2, b) == 2 * BLOCK  # both full prefix blocks reused: their KV is in the cache
    ta, tb = bm.block_table([1]), bm.block_table([2])
    assert list(ta[0, :2]) == list(tb[0, :2])  # same physical blocks
    assert bm.ref_count(int(ta[0, 0])) == 2 and bm.ref_count(int(ta[0, 1])) == 2
    assert ta[0, 2] != tb[0, 2] and bm.ref_count(int(tb[0, 2])) == 1
    assert bm.num_free_blocks == 16 - 3 - 2
    # slot = physical block * 256 + offset in the block
    s = bm.slot_mapping(2, 0, 2 * BLOCK + 300)
    pos = np.arange(2 * BLOCK + 300)
    assert np.array_equal(s, tb[0, pos // BLOCK] * BLOCK + pos % BLOCK)


def test_a_partial_block_is_never_shared():
    bm = BlockManager(8)
    toks = np.arange(BLOCK + 10)
    bm.allocate(1, toks)
    assert bm.allocate(2, toks) == BLOCK  # the full block only
    t = bm.block_table([1, 2])
    assert t[0, 0] == t[1, 0] and t[0, 1] != t[1, 1]


def test_freed_prefix_stays_reusable_until_handed_out():
    bm = BlockManager(4)
    p = np.arange(2 * BLOCK)
    bm.allocate(1, p)
    blocks = list(bm.block_table([1])[0])
    bm.free(1)
    assert bm.num_free_blocks == 4 and bm.ref_count(blocks[0]) == 0
    assert bm.allocate(2, p) == 2 * BLOCK  # revived from the free list
    assert list(bm.block_table([2])[0]) == blocks
    bm.free(2)
    # a different prompt takes the other free blocks first (freed blocks go to the back) ...
    bm.allocate(3, np.arange(2 * BLOCK) + 7)
    # ... and then the cached ones, which lose their contents
    bm.allocate(4, np.arange(2 * BLOCK) + 9)
    bm.free(3)
    bm.free(4)
    assert bm.allocate(5, p) == 0


def test_decode_appends_take_a_block_at_each_boundary():
    bm = BlockManager(8)
    bm.allocate(1, np.arange(BLOCK - 1))
    assert bm.seq_info(1) == (BLOCK - 1, 1, 0)
    t0 = int(bm.block_table([1])[0, 0])
    assert bm.append(1, 5) == t0 * BLOCK + BLOCK - 1  # fills the first block
    free = bm.num_free_blocks
    s = bm.append(1, 6)  # token 257 starts a block
    assert bm.num_free_blocks == free - 1
    t1 = int(bm.block_table([1])[0, 1])
    assert s == t1 * BLOCK
    assert bm.seq_info(1) == (BLOCK + 1, 2, 0)


def test_errors_change_nothing():
    bm = BlockManager(2)
    bm.allocate(1, np.arange(BLOCK))
    with pytest.raises(PkvError):
        bm.allocate(1, np.arange(3))  # already allocated
    with pytest.raises(PkvError):
        bm.allocate(2, np.arange(2 * BLOCK))  # two blocks needed, one free
    assert bm.num_free_blocks == 1
    with pytest.raises(PkvError):
        bm.free(9)
    with pytest.raises(PkvError):
        bm.block_table([1], max_blocks=0)
    with pytest.raises(PkvError):
        bm.slot_mapping(1, 0, BLOCK + 1)


@pytest.mark.parametrize("seed", range(6))
def test_library_equals_the_model(seed):
    """Random prompts with shared prefixes, decode appends and frees: identical state throughout."""
    rng = np.random.default_rng(100 + seed)
    nb = 48
    lib, ref = BlockManager(nb), BlockManagerModel(nb)
    prefixes = [rng.integers(0, 50, rng.integers(1, 4) * BLOCK) for _ in range(3)]
    live, next_id = [], 0
    for _ in range(120):
        op = rng.random()
        if op < 0.4:
            prompt = np.concatenate([prefixes[rng.integers(3)][: rng.integers(0, 3) * BLOCK],
                                     rng.integers(0, 50, rng.integers(1, 600))])
            try:
                c_ref = ref.allocate(next_id, prompt)
            except MemoryError:
                with pytest.raises(PkvError):
                    lib.allocate(next_id, prompt)
                continue
            assert lib.allocate(next_id, prompt) == c_ref
            live.append(next_id)
            next_id += 1
        elif op < 0.8 and live:
            s = live[rng.integers(len(live))]
            for _ in range(int(rng.integers(1, 300))):
                tok = int(rng.integers(0, 50))
                try:
                    slot_ref = ref.append(s, tok)
                except MemoryError:
                    with pytest.raises(PkvError):
                        lib.append(s, tok)
                    break
                assert lib.append(s, tok) == slot_ref
        elif live:
            s = live.pop(rng.integers(len(live)))
            ref.free_seq(s)
            lib.free(s)
        assert lib.num_free_blocks == len(ref.free)
        assert [lib.ref_count(b) for b in range(nb)] == ref.ref
        for s in live:
            n = len(ref.seqs[s]["tokens"])
            assert lib.seq_info(s) == (n, len(ref.seqs[s]["table"]), ref.seqs[s]["cached"])
            mb = len(ref.seqs[s]["table"]) + 2
            assert lib.block_table([s], mb)[0].tolist() == ref.table(s, mb)
            assert lib.slot_mapping(s, 0, n).tolist() == ref.slots(s, 0, n)
