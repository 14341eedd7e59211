"""Plain Python model of the host-side block manager (test infrastructure only).

The control plane of the paged cache, as the pages describe it:
  [NV] §4 — the CPU-side Block Manager manages token sequences, allocates
       blocks, keeps reference counts and reuses cached prefixes; a block
       carries {hash, ref} and its token ids;
  [Q3] §3.3 — one pool of fixed-size blocks allocated up front, one block
       table per sequence (logical -> physical block), the slot of a token is
       physical block * block_size + offset, and blocks with the same prefix
       hash are shared by sequences and stored once.
Readings of what the pages leave open (the same ones the library states):
full blocks only are hashed, the hash chains the previous block's hash with
the block's token ids (FNV-1a 64-bit, little-endian bytes), a lookup also
compares the ids, reuse runs from the first block until the first miss, a
freed block keeps its contents and goes to the back of the free list, and
decode appends take a new block at each block boundary and hash a block when
it fills.

Dictionaries and lists, one obvious step per rule; nothing from the library.
"""

from __future__ import annotations

from collections import deque

BLOCK = 256
NO_HASH = (1 << 64) - 1
FNV_OFFSET = 0xCBF29CE484222325
FNV_PRIME = 0x100000001B3


def fnv1a64(data: bytes, h: int = FNV_OFFSET) -> int:
    """FNV-1a, 64 bit: for each byte, xor it in, then multiply by the FNV prime (mod 2**64)."""
    for byte in data:
        h ^= byte
        h = (h * FNV_PRIME) & ((1 << 64) - 1)
    return h


def block_hash(prev: int, tokens) -> int:
    data = prev.to_bytes(8, "little") + b"".join(int(t).to_bytes(4, "little", signed=True) for t in tokens)
    h = fnv1a64(data)
    return h - 1 if h == NO_HASH else h


class BlockManagerModel:
    def __init__(self, num_blocks: int):
        self.ref = [0] * num_blocks
        self.hash = [NO_HASH] * num_blocks
        self.ids = [None] * num_blocks  # token ids of a full, hashed block
        self.free = deque(range(num_blocks))
        self.by_hash = {}
        self.seqs = {}  # seq id -> {"tokens": [...], "table": [...], "cached": int}

    # ---------------------------------------------------------------- blocks
    def _take_free(self):
        b = self.free.popleft()
        if self.hash[b] != NO_HASH and self.by_hash.get(self.hash[b]) == b:
            del self.by_hash[self.hash[b]]
        self.hash[b], self.ids[b], self.ref[b] = NO_HASH, None, 1
        return b

    def _set_hash(self, b, h, tokens):
        self.hash[b], self.ids[b] = h, list(tokens)
        self.by_hash[h] = b

    def _lookup(self, h, tokens):
        b = self.by_hash.get(h)
        if b is None or self.ids[b] != list(tokens):
            return None
        return b

    # ---------------------------------------------------------------- sequences
    def allocate(self, seq_id, tokens):
        tokens = [int(t) for t in tokens]
        if seq_id in self.seqs or not tokens:
            raise ValueError("bad allocation")
        need = -(-len(tokens) // BLOCK)
        if need > len(self.free):
            raise MemoryError("not enough free blocks")
        table, cached, h, miss = [], 0, NO_HASH, False
        for i in range(need):
            blk = tokens[i * BLOCK:(i + 1) * BLOCK]
            full = len(blk) == BLOCK
            h = block_hash(h, blk) if full else NO_HASH
            b = self._lookup(h, blk) if (full and not miss) else None
            if b is None:
                miss = True
            if miss:
                b = self._take_free()
            else:
                cached += BLOCK
                if self.ref[b] > 0:
                    self.ref[b] += 1
                else:
                    self.free.remove(b)
                    self.ref[b] = 1
            if full and self.hash[b] != h:
                self._set_hash(b, h, blk)
            table.append(b)
        self.seqs[seq_id] = {"tokens": tokens, "table": table, "cached": cached}
        return cached

    def append(self, seq_id, token):
        s = self.seqs[seq_id]
        n = len(s["tokens"]) + 1
        if n % BLOCK == 1:
            if not self.free:
                raise MemoryError("no free block")
            s["table"].append(self._take_free())
        s["tokens"].append(int(token))
        last = s["table"][-1]
        if n % BLOCK == 0:
            prev = self.hash[s["table"][-2]] if len(s["table"]) >= 2 else NO_HASH
            blk = s["tokens"][(len(s["table"]) - 1) * BLOCK:]
            self._set_hash(last, block_hash(prev, blk), blk)
        return last * BLOCK + (n - 1) % BLOCK

    def free_seq(self, seq_id):
        s = self.seqs.pop(seq_id)
        for b in reversed(s["table"]):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free.append(b)

    def slots(self, seq_id, start, end):
        t = self.seqs[seq_id]["table"]
        return [t[p // BLOCK] * BLOCK + p % BLOCK for p in range(start, end)]

    def table(self, seq_id, max_blocks):
        t = self.seqs[seq_id]["table"]
        return t + [-1] * (max_blocks - len(t))
