"""Seeded generators for the five workloads of the paged-KV attention step.

Every array is a plain numpy array.  bf16 tensors are held as their uint16 bit
patterns.  Randomness comes only from ``numpy.random.default_rng``:

* q, k, v of the new tokens and the cache history are N(0, 1) drawn in fp32
  and rounded to bf16 (round to nearest, ties to even);
* the q_norm / k_norm weights are 1 + 0.1 * N(0, 1), drawn in fp32, rounded
  to bf16;
* physical block ids come from ``rng.permutation(num_blocks)`` and are handed
  out in order, sequence by sequence (the pages' block manager hands out
  whole 256-token blocks from a pool allocated once, and a token's cache row
  is ``block_id * block_size + offset``: "同一个 Qwen3，两种写法" §3.3);
* the history already in the cache (tokens before the current step) is drawn
  per physical block from ``default_rng([seed, 1 or 2, block_id])`` so that
  any block can be regenerated on its own; shared-prefix blocks therefore hold
  the same content for every sequence that points at them;
* every cache row that holds no token is filled with the bf16 NaN pattern
  0x7FC1, so a kernel that reads a row it must not read (or multiplies a
  masked value by zero) shows up as NaN.
"""

from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

NUM_Q_HEADS = 32
NUM_KV_HEADS = 8
HEAD_DIM = 128
BLOCK_SIZE = 256
NAN_BF16 = 0x7FC1

CONFIG_NAMES = {
    1: "tiny decode: B=4, context {17,64,200,256}, 8-block pool",
    2: "varlen causal prefill: 8 prompts, lengths U[1,2048], empty cache",
    3: "batched decode: B=256, context U[512,4096], 4096-block pool",
    4: "chunked prefill, shared prefix: 16 seqs, prefix U[0,8192] + 512-token chunk",
    5: "long-context decode: context 40960, 5120-block pool",
}


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit pattern, round to nearest, ties to even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


def _normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    return bf16_bits_from_f32(rng.standard_normal(shape, dtype=np.float32))


@dataclass
class Workload:
    """One step of one layer: the new tokens, their cache slots and the cache state.

    Token-indexed arrays cover the new tokens of the step, flattened over
    sequences in order (the flat ``[T, ...]`` layout).
    """

    name: str
    mode: str  # "decode" or "prefill"
    seed: int
    num_blocks: int
    hist_lens: np.ndarray  # int32 [S]  tokens already in the cache before the step
    new_lens: np.ndarray  # int32 [S]   tokens added by the step (1 for decode)
    block_table: np.ndarray  # int32 [S, max_blocks], -1 past each sequence's blocks
    block_fill: np.ndarray  # int32 [num_blocks] history rows present at the top of each block
    q: np.ndarray  # uint16 [T, 32, 128]
    k: np.ndarray  # uint16 [T, 8, 128]
    v: np.ndarray  # uint16 [T, 8, 128]
    q_norm_w: np.ndarray  # uint16 [128]
    k_norm_w: np.ndarray  # uint16 [128]
    positions: np.ndarray  # int32 [T]
    slot_mapping: np.ndarray  # int32 [T], -1 = do not store
    scale: float = 1.0 / math.sqrt(HEAD_DIM)
    notes: dict = field(default_factory=dict)

    # ---- derived views (bookkeeping only) ----
    @property
    def num_seqs(self) -> int:
        return int(self.hist_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.q.shape[0])

    @property
    def seq_lens_k(self) -> np.ndarray:
        return (self.hist_lens + self.new_lens).astype(np.int32)

    @property
    def context_lens(self) -> np.ndarray:
        return self.seq_lens_k

    @property
    def cu_seqlens_q(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.new_lens)]).astype(np.int32)

    @property
    def cu_seqlens_k(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.seq_lens_k)]).astype(np.int32)

    @property
    def max_seqlen_q(self) -> int:
        return int(self.new_lens.max()) if self.num_seqs else 0

    @property
    def max_seqlen_k(self) -> int:
        return int(self.seq_lens_k.max()) if self.num_seqs else 0

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_table.shape[1])

    # ---- cache contents ----
    def cache_block(self, which: str, block_id: int) -> np.ndarray:
        """Initial content of one physical block: uint16 [256, 8, 128]."""
        out = np.full((BLOCK_SIZE, NUM_KV_HEADS, HEAD_DIM), NAN_BF16, dtype=np.uint16)
        fill = int(self.block_fill[block_id])
        if fill:
            tag = 1 if which == "k" else 2
            rng = np.random.default_rng([self.seed, tag, int(block_id)])
            out[:fill] = _normal_bf16(rng, (fill, NUM_KV_HEADS, HEAD_DIM))
        return out

    def fill_cache(self, which: str, out: np.ndarray, threads: int | None = None) -> np.ndarray:
        """Write the initial cache into ``out`` (uint16 [num_blocks, 256, 8, 128])."""
        assert out.shape == (self.num_blocks, BLOCK_SIZE, NUM_KV_HEADS, HEAD_DIM)
        assert out.dtype == np.uint16
        filled = np.nonzero(self.block_fill)[0]
        empty = np.nonzero(self.block_fill == 0)[0]
        if empty.size:
            out[empty] = NAN_BF16

        def one(b):
            out[b] = self.cache_block(which, int(b))

        if filled.size > 64:
            with ThreadPoolExecutor(max_workers=threads or min(16, os.cpu_count() or 1)) as ex:
                list(ex.map(one, filled))
        else:
            for b in filled:
                one(b)
        return out

    def materialize_cache(self) -> tuple[np.ndarray, np.ndarray]:
        shape = (self.num_blocks, BLOCK_SIZE, NUM_KV_HEADS, HEAD_DIM)
        kc = self.fill_cache("k", np.empty(shape, dtype=np.uint16))
        vc = self.fill_cache("v", np.empty(shape, dtype=np.uint16))
        return kc, vc

    def used_blocks(self) -> np.ndarray:
        bt = self.block_table
        return np.unique(bt[bt >= 0])

    def subset(self, seqs) -> "Workload":
        """The same step restricted to some sequences, on the same block pool."""
        seqs = np.asarray(seqs, dtype=np.int64)
        cu = np.concatenate([[0], np.cumsum(self.new_lens)])
        tok = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in seqs]) if seqs.size else np.zeros(0, np.int64)
        return Workload(
            name=f"{self.name} [seqs {seqs.tolist() if seqs.size <= 8 else f'{seqs.size} seqs'}]",
            mode=self.mode,
            seed=self.seed,
            num_blocks=self.num_blocks,
            hist_lens=self.hist_lens[seqs].copy(),
            new_lens=self.new_lens[seqs].copy(),
            block_table=self.block_table[seqs].copy(),
            block_fill=self.block_fill,
            q=self.q[tok],
            k=self.k[tok],
            v=self.v[tok],
            q_norm_w=self.q_norm_w,
            k_norm_w=self.k_norm_w,
            positions=self.positions[tok],
            slot_mapping=self.slot_mapping[tok],
            scale=self.scale,
            notes=dict(self.notes),
        )


def build_workload(
    name: str,
    mode: str,
    seed: int,
    hist_lens,
    new_lens,
    *,
    pool_blocks: int | None = None,
    spare_blocks: int = 16,
    share_pairs: bool = False,
    rng: np.random.Generator | None = None,
    skip_tokens=(),
) -> Workload:
    """Lay out sequences over a permuted block pool and draw the step's tensors.

    ``hist_lens[s]`` tokens of sequence s are already cached; ``new_lens[s]``
    tokens are added by this step.  With ``share_pairs`` the sequences (2j,
    2j+1) share their leading ``min(hist) // 256`` full history blocks.
    ``skip_tokens`` lists flat token indices whose slot is set to -1.
    """
    rng = rng if rng is not None else np.random.default_rng(seed)
    hist = np.asarray(hist_lens, dtype=np.int64)
    new = np.asarray(new_lens, dtype=np.int64)
    S = hist.shape[0]
    total = hist + new
    nblk = (total + BLOCK_SIZE - 1) // BLOCK_SIZE
    shared = np.zeros(S, dtype=np.int64)
    if share_pairs:
        for j in range(0, S - 1, 2):
            n = min(hist[j], hist[j + 1]) // BLOCK_SIZE
            shared[j + 1] = n  # the second sequence of the pair reuses the first one's blocks
    distinct = int(nblk.sum() - shared.sum())
    NB = int(pool_blocks) if pool_blocks is not None else distinct + spare_blocks
    if distinct > NB:
        raise ValueError(f"{distinct} blocks needed, pool has {NB}")
    perm = rng.permutation(NB).astype(np.int32)

    max_blocks = int(max(1, nblk.max() if S else 1))
    bt = np.full((S, max_blocks), -1, dtype=np.int32)
    nxt = 0
    for s in range(S):
        if shared[s]:
            bt[s, : shared[s]] = bt[s - 1, : shared[s]]
        for j in range(int(shared[s]), int(nblk[s])):
            bt[s, j] = perm[nxt]
            nxt += 1
    fill = np.zeros(NB, dtype=np.int32)
    for s in range(S):
        for j in range(int(nblk[s])):
            f = int(np.clip(hist[s] - j * BLOCK_SIZE, 0, BLOCK_SIZE))
            b = bt[s, j]
            fill[b] = max(fill[b], f)

    T = int(new.sum())
    q = _normal_bf16(rng, (T, NUM_Q_HEADS, HEAD_DIM))
    k = _normal_bf16(rng, (T, NUM_KV_HEADS, HEAD_DIM))
    v = _normal_bf16(rng, (T, NUM_KV_HEADS, HEAD_DIM))
    wq = bf16_bits_from_f32(1.0 + 0.1 * rng.standard_normal(HEAD_DIM, dtype=np.float32))
    wk = bf16_bits_from_f32(1.0 + 0.1 * rng.standard_normal(HEAD_DIM, dtype=np.float32))

    positions = np.zeros(T, dtype=np.int32)
    slots = np.zeros(T, dtype=np.int32)
    t = 0
    for s in range(S):
        for i in range(int(new[s])):
            pos = int(hist[s] + i)
            positions[t] = pos
            slots[t] = int(bt[s, pos // BLOCK_SIZE]) * BLOCK_SIZE + pos % BLOCK_SIZE
            t += 1
    for t in skip_tokens:
        slots[t] = -1

    return Workload(
        name=name,
        mode=mode,
        seed=seed,
        num_blocks=NB,
        hist_lens=hist.astype(np.int32),
        new_lens=new.astype(np.int32),
        block_table=bt,
        block_fill=fill,
        q=q,
        k=k,
        v=v,
        q_norm_w=wq,
        k_norm_w=wk,
        positions=positions,
        slot_mapping=slots,
    )


def config_workload(index: int, seed: int | None = None, batch: int | None = None) -> Workload:
    """The five named workloads, by number: 1 tiny decode (4 sequences,
    contexts 17/64/200/256), 2 varlen prefill (8 prompts of U[1, 2048]
    tokens), 3 batched decode (256 sequences, contexts U[512, 4096]),
    4 chunked prefill after a shared prefix (16 sequences, prefix U[0, 8192]
    + 512 new tokens), 5 long-context decode (contexts 40960, up to 32
    sequences).

    Integer ranges "uniform in [a, b]" are read as inclusive.  ``batch``
    selects the first ``batch`` sequences of the long-context decode (1..32).
    """
    seed = 20260 + index if seed is None else seed
    rng = np.random.default_rng(seed)
    if index == 1:
        L = np.array([17, 64, 200, 256])
        return build_workload(CONFIG_NAMES[1], "decode", seed, L - 1, np.ones(4, np.int64), pool_blocks=8, rng=rng)
    if index == 2:
        L = rng.integers(1, 2048, size=8, endpoint=True)
        return build_workload(CONFIG_NAMES[2], "prefill", seed, np.zeros(8, np.int64), L, spare_blocks=16, rng=rng)
    if index == 3:
        L = rng.integers(512, 4096, size=256, endpoint=True)
        return build_workload(CONFIG_NAMES[3], "decode", seed, L - 1, np.ones(256, np.int64), pool_blocks=4096, rng=rng)
    if index == 4:
        p = rng.integers(0, 8192, size=16, endpoint=True)
        return build_workload(
            CONFIG_NAMES[4], "prefill", seed, p, np.full(16, 512), spare_blocks=16, share_pairs=True, rng=rng
        )
    if index == 5:
        B = 32 if batch is None else int(batch)
        if not 1 <= B <= 32:
            raise ValueError("the long-context decode runs at batch 1..32")
        L = np.full(32, 40960)
        wl = build_workload(CONFIG_NAMES[5], "decode", seed, L - 1, np.ones(32, np.int64), pool_blocks=5120, rng=rng)
        if B < 32:
            wl = wl.subset(np.arange(B))
        wl.name = f"{CONFIG_NAMES[5]}, B={B}"
        return wl
    raise ValueError(f"no workload number {index}")
