// K3: causal varlen prefill attention over the paged cache on tcgen05 tensor
// cores (sm_103a), accumulators in tensor memory; a persistent kernel.
//
// Operation ("Nano-vLLM深度解读（下）" §4 prefill branch with a block table;
// "同一个 Qwen3，两种写法" §3.2 and §3.4): sequence s owns query rows
// cu_q[s]..cu_q[s+1]-1 (Lq) and keys 0..Lk-1 read through block_table row s;
// query row i sits at position Lk - Lq + i and sees keys 0..Lk - Lq + i; query
// head h reads KV head h / 4.
//
// Work item = (pair of query heads {2p, 2p+1} of one GQA group, sequence s,
// 128-row query tile counted from the end of the sequence).  One CTA per SM
// claims items one at a time from a device counter (atomicAdd), so the SMs stay
// evenly loaded, and passes each claim to its other warps through a 4-entry
// ring in shared memory.  The two heads of an item share every K/V tile.
// Claim order: tile-index-major, so the tiles with the most keys come first;
// when some sequence has a cached prefix, longest-first over all items instead
// (see LptOrder).  The next item is claimed when the current one's last tile is
// being loaded, not when the item starts: a CTA that claimed a whole item ahead
// could still be working on it long after the others ran out of work.
// Measured on 8 prompts of U[1, 2048] / 16 chunks of 512 after prefixes of
// U[0, 8192]: 128.7 / 536 us with claims at the item start and in
// tile-index-major order, 124.6 / 508 us with late claims, 125 / 467 us with
// longest-first order for the chunks as well.
// 10 warps:
//   warp 0      claims items (the whole warp; lane 0 issues copies and waits);
//               TMA producer: both Q tiles of an item once the previous item's
//               QK^T MMAs are done (q_empty), then 128-key K and V tiles of KV
//               head p/2 into two 2-deep rings (a tile lies inside one 256-token
//               block: one block-table lookup per tile).
//   warp 1      allocates 512 TMEM columns once and issues every MMA in the
//               order PV_A(j), S_A(j+1), PV_B(j), S_B(j+1): while the softmax
//               of one head runs the tensor core works on the other.  The
//               whole warp runs the issue loop and its waits (converged, so the
//               operand descriptors stay warp-uniform) and one elected lane
//               issues each group of MMAs and commits; issuing from a lone
//               lane in divergent code cost about 80 cycles per MMA, more than
//               the 64 the tensor core needs for one.
//               S = Q K^T (M=N=128, K=128 as 8 x K16, both operands K-major in
//               128B-swizzled smem); O += P V with P read from TMEM and V
//               MN-major from smem.  The 8 MMAs of a tile issue back to back.
//   warps 2..5  softmax of head A, warps 6..9 softmax of head B: thread =
//               query row = TMEM lane.  One 128-column TMEM load per tile, row
//               max and exp2 from registers (scaling and row sums on packed
//               fp32 pairs), bf16 P written back over the S columns; the causal mask is a per-row column limit applied by
//               selection, on a separate code path taken only by warps that
//               meet the diagonal; lazy rescaling of O (only when the running
//               max grows by more than 2^8).  Warpgroup A zeroes V rows that
//               hold no token (keys >= Lk, or a block id outside the pool).  At
//               the end of an item each warpgroup reads O, releases it
//               (o_free), normalises it and stores its rows: a warp whose 32
//               rows all belong to the sequence with two bulk tensor stores
//               (64 dims x 32 rows each) from its swizzled staging buffer,
//               other warps row by row.
// Phases of every ring and barrier continue across items: each tile loads one
// K and one V and runs one S and one PV per head, so one running tile counter
// gives every stage index and parity.
// TMEM columns: S_A [0,128), S_B [128,256), O_A [256,384), O_B [384,512).
// Registers: one SM sub-partition hosts three of the ten warps, so every
// thread has at most 168 registers (a 16K register file per sub-partition).
// Launched as a programmatic dependent of the previous kernel in the stream
// (normally the store that fills the cache): barrier set-up and the TMEM
// allocation overlap that kernel's tail, and griddepcontrol.wait holds every
// read of global memory until it has completed.
// Every mbarrier wait is bounded; on timeout the CTA flags the error word and
// still releases its TMEM.
#include "tcgen05.cuh"

namespace pkv {

constexpr int kTcRows = 128;
constexpr int kTcKeys = 128;
constexpr int kTcStages = 2;
constexpr int kTcSub = 128 * 128;          // [128 rows][64 dims] bf16, 128B-swizzled: 16 KiB
constexpr int kTcTile = 2 * kTcSub;        // [128][128] bf16: 32 KiB
constexpr int kTcQOff = 0;                 // Q_A, Q_B
constexpr int kTcKOff = 2 * kTcTile;
constexpr int kTcVOff = kTcKOff + kTcStages * kTcTile;
constexpr int kTcStageOff = kTcVOff + kTcStages * kTcTile;  // 192 KiB: O staging, 4 KiB per softmax warp
constexpr int kTcStageBytes = 8 * 32 * 128;
constexpr int kTcBarOff = kTcStageOff + kTcStageBytes;   // barriers and the item ring
constexpr int kTcBarBytes = 512;
constexpr int kTcSmemBytes = kTcBarOff + kTcBarBytes + 1024;
static_assert(kTcStageOff % 1024 == 0, "the staging buffers are 128-byte-swizzled bulk-store sources");
constexpr int kTcThreads = 320;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;
constexpr int kTcClaimLead = 1;  // tiles of the current item still to load when the next is claimed

struct TcParams {
  __nv_bfloat16* out;
  const int32_t* cu_q;
  const int32_t* cu_k;
  const int32_t* block_table;
  int32_t num_seqs;
  int32_t num_ztiles;  // ceil(max_seqlen_q / 128)
  int32_t max_blocks;
  int32_t num_blocks;
  int32_t max_seqlen_q;
  int32_t max_seqlen_k;
  float scale_log2;
  int32_t prefix_hint;  // max_seqlen_k >= max_seqlen_q + 128: some sequence may have a cached prefix
  unsigned* sched;  // {next item, CTAs done}: zero on entry, returned to zero by the last CTA
  unsigned* err;
};

constexpr int kItemRing = 4;
constexpr int kItemConsumers = 9;  // the MMA thread and the 8 softmax warps

// Geometry of one work item.  Query tiles are aligned to the 128-key grid
// (each tile then meets the causal diagonal in a single key tile) unless that
// needs more tiles than cutting 128-row tiles back from the end of the
// sequence, as it can with a cached prefix.  Tile z = 0 holds the last rows,
// which see the most keys.  The producer decodes each claimed item once and
// hands the decoded item to the other roles through the shared-memory ring
// (s < 0 marks the end of the work), so they never wait on global loads of
// cu_seqlens at an item boundary.
struct Item {
  int h0, g, s, q0, rbase, Lq, off, Lk, n_tiles;
  bool invalid;  // a sequence the call cannot serve (more queries than keys, longer than its table row)
};

struct TcBars {
  uint64_t item_full[kItemRing], item_empty[kItemRing];
  Item items[kItemRing];
  uint64_t q_full, q_empty;
  uint64_t k_full[kTcStages], k_empty[kTcStages];
  uint64_t v_full[kTcStages], v_empty[kTcStages];
  uint64_t s_full[2], p_ready[2], o_ready[2], o_free[2];  // per head of the pair
  uint32_t tmem_base;
  int timeout;
};

static_assert(sizeof(TcBars) <= kTcBarBytes, "the barrier block must fit the bytes reserved after the rings");


// The query tiles of sequence s: how many there are (units) and whether they are
// aligned to the 128-key grid (each then meets the causal diagonal in a single key
// tile), which is the case unless that needs more tiles than cutting 128-row tiles
// back from the end of the sequence, as it can with a cached prefix.
struct SeqTiles {
  int q0, Lq, Lk, off, units;
  bool aligned;
};

__device__ __forceinline__ SeqTiles seq_tiles(const TcParams& p, int s) {
  SeqTiles t;
  t.q0 = __ldg(p.cu_q + s);
  t.Lq = __ldg(p.cu_q + s + 1) - t.q0;
  t.Lk = __ldg(p.cu_k + s + 1) - __ldg(p.cu_k + s);
  t.off = t.Lk - t.Lq;  // position of sequence row 0
  const int tiles_end = (t.Lq + kTcRows - 1) / kTcRows;
  const int tiles_grid = (t.Lk + kTcRows - 1) / kTcRows - (t.off > 0 ? t.off / kTcRows : 0);
  t.aligned = t.Lq > 0 && t.off >= 0 && tiles_grid <= tiles_end;
  t.units = t.aligned ? tiles_grid : tiles_end;
  return t;
}

// The work item (head pair, sequence s, query tile z) with z < the sequence's units;
// tile z = 0 holds the last rows, which see the most keys.
__device__ __forceinline__ void item_at(const TcParams& p, int pair, int s, int z, const SeqTiles& t, Item& it) {
  const int rbase = t.aligned ? ((t.Lk + kTcRows - 1) / kTcRows - 1 - z) * kTcRows - t.off  // first row of the
                              : t.Lq - (z + 1) * kTcRows;                                  // tile's position range
  it.h0 = 2 * pair;
  it.g = it.h0 / kGroup;
  it.s = s;
  it.q0 = t.q0;
  it.rbase = rbase;
  it.Lq = t.Lq;
  it.off = t.off;
  it.Lk = t.Lk;
  const int last_row = min(rbase + kTcRows, t.Lq);  // one past the tile's last row
  it.n_tiles = (t.off + last_row + kTcKeys - 1) / kTcKeys;
  it.invalid = t.Lq > t.Lk || t.Lk > p.max_blocks * kBlockSize || t.Lq > p.max_seqlen_q || t.Lk > p.max_seqlen_k;
}

// Tile-index-major order: slot w is (pair, sequence, z) with z slowest; false for
// a slot past the sequence's tiles.
__device__ __forceinline__ bool item_info(const TcParams& p, int w, Item& it) {
  const int pair = w % (kNumQHeads / 2);
  const int s = (w / (kNumQHeads / 2)) % p.num_seqs;
  const int z = w / ((kNumQHeads / 2) * p.num_seqs);
  const SeqTiles t = seq_tiles(p, s);
  if (z >= t.units) return false;
  item_at(p, pair, s, z, t, it);
  return true;
}

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ int warp_max(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Longest-first order of the work units (sequence, query tile), each unit being
// the 16 items of its head pairs.  Unit z of sequence s runs T_s - z key tiles,
// T_s = ceil(Lk / 128) (taken no smaller than the unit count, which only matters
// for sequences the call cannot serve), so the units of a sequence hold the
// distinct tile counts T_s - units_s + 1 .. T_s.  Lane l of the producer warp
// keeps (T_s, units_s) of sequences l, l + 32, ...; the u-th unit in order of
// decreasing tile count (ties by sequence) is found by a binary search on the
// count, each probe a warp sum.  Claiming the longest items first lets the
// dynamic claims end evenly when the sequences' lengths differ widely, as with
// chunks after cached prefixes of different lengths: there an item's tile count
// depends mostly on its sequence's prefix, not on its tile index.  Without a
// cached prefix the tile-index-major order is already close to longest-first
// and spreads each wave of claims over all the sequences, where longest-first
// would start every CTA on the K/V of the few longest ones (measured on 8
// prompts of U[1, 2048]: 125 us tile-index-major, 127 us longest-first; on 16
// chunks of 512 after prefixes of U[0, 8192]: 508 against 465 us).
constexpr int kLptPerLane = 4;  // up to 128 sequences; more fall back to tile-index-major order
struct LptOrder {
  int T[kLptPerLane], units[kLptPerLane];
  int total, vmax;
  bool prefixed;  // some sequence has a cached prefix of at least one key tile

  __device__ __forceinline__ void init(const TcParams& p, int lane) {
    int u = 0, vm = 0;
    bool pre = false;
#pragma unroll
    for (int k = 0; k < kLptPerLane; ++k) {
      const int s = lane + 32 * k;
      T[k] = 0;
      units[k] = 0;
      if (s < p.num_seqs) {
        const SeqTiles t = seq_tiles(p, s);
        units[k] = t.units;
        T[k] = max((t.Lk + kTcKeys - 1) / kTcKeys, t.units);
        pre = pre || (t.Lq > 0 && t.off >= kTcKeys);
      }
      u += units[k];
      vm = max(vm, T[k]);
    }
    total = warp_sum(u);
    vmax = warp_max(vm);
    prefixed = __any_sync(0xffffffffu, pre);
  }
  // units whose tile count is at least v (over the whole warp)
  __device__ __forceinline__ int count_ge(int v) const {
    int c = 0;
#pragma unroll
    for (int k = 0; k < kLptPerLane; ++k) c += max(0, min(units[k], T[k] - v + 1));
    return warp_sum(c);
  }
  // sequence s and query tile z of the u-th unit, 0 <= u < total (all lanes agree)
  __device__ __forceinline__ void unit(int u, int& s, int& z) const {
    int lo = 1, hi = vmax + 1;  // count_ge(lo) > u >= count_ge(hi)
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (count_ge(mid) > u) lo = mid;
      else hi = mid;
    }
    int r = u - count_ge(lo + 1);  // rank among the units with exactly lo tiles, by sequence
    s = 0;
    z = 0;
    bool found = false;
#pragma unroll
    for (int k = 0; k < kLptPerLane; ++k) {
      const bool has = units[k] > 0 && T[k] - units[k] + 1 <= lo && lo <= T[k];
      unsigned m = __ballot_sync(0xffffffffu, has);
      const int c = __popc(m);
      const int Tk = T[k];
      if (!found) {
        if (r < c) {
          for (int i = 0; i < r; ++i) m &= m - 1;  // drop the r lowest set lanes
          const int ln = __ffs(m) - 1;
          s = 32 * k + ln;
          z = __shfl_sync(0xffffffffu, Tk, ln) - lo;
          found = true;
        } else {
          r -= c;
        }
      }
    }
  }
};

// mbarrier wait whose result is the same for every lane of the warp, so that a
// timeout can never leave part of a warp at a warp-collective tcgen05.ld/st.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, unsigned parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

// Bulk tensor store shared -> global of a box (x, head, row) of the output, in this
// thread's bulk async-group; the group's reads of shared memory and its writes are
// waited for separately.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2), "r"(src)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
  return v;
}

// Causal mask of one S row: columns beyond `lim` become -inf, so that exp2
// gives exactly 0 for them (the scale is positive).  Chunks of 32 columns
// that every row of the warp sees whole are left alone; the others select
// column by column.
__device__ __forceinline__ void mask_row(uint32_t (&sv)[128], int lim) {
  constexpr uint32_t kNegInf = 0xff800000u;
#pragma unroll
  for (int c4 = 0; c4 < 4; ++c4) {
    if (__all_sync(0xffffffffu, lim >= c4 * 32 + 31)) continue;
#pragma unroll
    for (int c = c4 * 32; c < c4 * 32 + 32; ++c) sv[c] = c <= lim ? sv[c] : kNegInf;
  }
}

// Row max of the 128 scores of this thread's S row.
__device__ __forceinline__ float row_max(const uint32_t (&sv)[128]) {
  float m8[8];
#pragma unroll
  for (int a = 0; a < 8; ++a) m8[a] = -INFINITY;
#pragma unroll
  for (int c = 0; c < 128; c += 2)
    m8[(c >> 1) & 7] = fmax3(m8[(c >> 1) & 7], __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]));
  return fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
}

// P = exp2(s * scale_log2 - m) as bf16 pairs written over the S columns of
// this row (8 columns at a time, which keeps few values live); returns the
// fp32 row sum of P.  Scaling and summing run on packed fp32 pairs, one
// instruction per two columns.
__device__ __forceinline__ float row_exp(const uint32_t (&sv)[128], float sl2, float negm, uint32_t sbuf) {
  const uint64_t sl2x2 = f2pack(sl2, sl2), negm2 = f2pack(negm, negm);
  uint64_t sum2[2] = {0ull, 0ull};
#pragma unroll
  for (int c8 = 0; c8 < 8; ++c8) {
    uint32_t pk[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int col = c8 * 16 + 2 * c;
      const uint64_t x2 = ffma2(f2pack(__uint_as_float(sv[col]), __uint_as_float(sv[col + 1])), sl2x2, negm2);
      float x0, x1;
      f2unpack(x2, x0, x1);
      const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
      sum2[c & 1] = fadd2(sum2[c & 1], f2pack(p0, p1));
      pk[c] = pack_bf16x2(p0, p1);
    }
    tc::st8(sbuf + c8 * 8, pk);
  }
  float a0, a1, b0, b1;
  f2unpack(sum2[0], a0, a1);
  f2unpack(sum2[1], b0, b1);
  return (a0 + a1) + (b0 + b1);
}

// The TMA producer (warp 0).  The whole warp runs the loop: lane 0 issues the
// copies and waits, each wait's result is broadcast so control flow stays
// warp-uniform, and every lane takes part in finding a claimed item when the
// claims go in longest-first order.
__device__ __forceinline__ void produce(const TcParams& p, const CUtensorMap* tmQ, const CUtensorMap* tmK,
                                        const CUtensorMap* tmV, uint8_t* smem, TcBars* bars, int n_items, int lane,
                                        const LptOrder& lpt, bool longest_first) {
  const bool lane0 = lane == 0;
  if (lane0) {
    tma_prefetch_desc(tmQ);
    tma_prefetch_desc(tmK);
    tma_prefetch_desc(tmV);
  }
  uint32_t tt = 0, ic = 0, nslot = 0;  // tiles, items loaded and ring entries published by this CTA
  bool ok = true;
  // lane 0's wait, its result on every lane
  auto wait0 = [&](uint64_t* bar, unsigned parity) -> bool {
    int r = 1;
    if (lane0) r = mbar_wait(bar, parity) ? 1 : 0;
    return __shfl_sync(0xffffffffu, r, 0) != 0;
  };
  // lane 0's value on every lane
  auto from0 = [&](unsigned v) -> unsigned { return __shfl_sync(0xffffffffu, v, 0); };
  // the item at claim index w, or -1 at the end: longest-first (unit w / 16, pair
  // w % 16), else tile-index-major, where slots past a sequence's tiles are skipped
  auto claim = [&](int w, Item& it) -> int {
    if (longest_first) {
      if (w >= (kNumQHeads / 2) * lpt.total) return -1;
      int s, z;
      lpt.unit(w / (kNumQHeads / 2), s, z);
      item_at(p, w % (kNumQHeads / 2), s, z, seq_tiles(p, s), it);
      return w;
    }
    while (w < n_items && !item_info(p, w, it)) {
      unsigned v = 0;
      if (lane0) v = atomicAdd(p.sched, 1u);
      w = static_cast<int>(from0(v));
    }
    return w < n_items ? w : -1;
  };
  // the first block id of a claimed item, loaded when it is claimed so that the
  // item's first K/V loads do not wait a global-memory round trip
  auto first_block = [&](const Item& it) -> int {
    return it.invalid ? 0 : __ldg(p.block_table + static_cast<int64_t>(it.s) * p.max_blocks);
  };
  Item nxt;
  unsigned ahead = 0;  // lane 0's claim index; the other lanes see it at the claim
  if (lane0) ahead = atomicAdd(p.sched, 1u);
  int w_next = claim(static_cast<int>(from0(ahead)), nxt);
  int blk_first = w_next >= 0 ? first_block(nxt) : 0;
  while (ok) {
    const int w = w_next;
    Item it = nxt;
    if (w < 0) it.s = -1;
    const int rs = nslot % kItemRing;
    if (nslot >= kItemRing && !(ok = wait0(&bars->item_empty[rs], ((nslot / kItemRing) - 1) & 1))) break;
    if (lane0) {
      bars->items[rs] = it;
      mbar_arrive(&bars->item_full[rs]);
    }
    ++nslot;
    if (w < 0) break;
    // The next item is claimed when this item's last kTcClaimLead tiles are being
    // loaded: late enough that a CTA does not commit to more work while others are
    // about to run dry, early enough that the round trip overlaps the last loads.
    bool claimed = false;
    if (!it.invalid) {
      const int32_t* table = p.block_table + static_cast<int64_t>(it.s) * p.max_blocks;
      if (ic > 0 && !(ok = wait0(&bars->q_empty, (ic - 1) & 1))) break;
      if (lane0) {
        mbar_arrive_expect_tx(&bars->q_full, 2 * kTcTile);
        for (int t = 0; t < 2; ++t) {
          tma_load_3d(smem + kTcQOff + t * kTcTile, tmQ, &bars->q_full, 0, it.h0 + t, it.q0 + it.rbase);
          tma_load_3d(smem + kTcQOff + t * kTcTile + kTcSub, tmQ, &bars->q_full, 64, it.h0 + t,
                      it.q0 + it.rbase);
        }
      }
      int blk_cur = blk_first;
      const int claim_at = it.n_tiles > kTcClaimLead ? it.n_tiles - kTcClaimLead : 0;
      for (int j = 0; j < it.n_tiles; ++j, ++tt) {
        if (j == claim_at) {
          if (lane0) ahead = atomicAdd(p.sched, 1u);
          claimed = true;
        }
        const int st = tt % kTcStages;
        const int key0 = j * kTcKeys;
        // the next tile's block id, one tile ahead: its latency overlaps this tile's waits
        const int blk_nxt = j + 1 < it.n_tiles ? __ldg(table + (key0 + kTcKeys) / kBlockSize) : 0;
        int blk = blk_cur;
        blk_cur = blk_nxt;
        if (blk < 0 || blk >= p.num_blocks) {  // its keys are masked by the softmax; load something valid
          if (lane0) set_error(p.err, PKV_EFLAG_BLOCK_ID);
          blk = 0;
        }
        const int slot0 = blk * kBlockSize + (key0 % kBlockSize);
        if (tt >= kTcStages && !(ok = wait0(&bars->k_empty[st], ((tt / kTcStages) - 1) & 1))) break;
        uint8_t* kd = smem + kTcKOff + st * kTcTile;
        if (lane0) {
          mbar_arrive_expect_tx(&bars->k_full[st], kTcTile);
          tma_load_3d(kd, tmK, &bars->k_full[st], 0, it.g, slot0);
          tma_load_3d(kd + kTcSub, tmK, &bars->k_full[st], 64, it.g, slot0);
        }
        if (tt >= kTcStages && !(ok = wait0(&bars->v_empty[st], ((tt / kTcStages) - 1) & 1))) break;
        uint8_t* vd = smem + kTcVOff + st * kTcTile;
        if (lane0) {
          mbar_arrive_expect_tx(&bars->v_full[st], kTcTile);
          tma_load_3d(vd, tmV, &bars->v_full[st], 0, it.g, slot0);
          tma_load_3d(vd + kTcSub, tmV, &bars->v_full[st], 64, it.g, slot0);
        }
      }
      ++ic;
    }
    if (!claimed && lane0) ahead = atomicAdd(p.sched, 1u);
    w_next = claim(static_cast<int>(from0(ahead)), nxt);
    if (w_next >= 0) blk_first = first_block(nxt);
  }
  if (!ok && lane0) bars->timeout = 1;
}

__global__ void __launch_bounds__(kTcThreads, 1) prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                                                                   const __grid_constant__ CUtensorMap tmK,
                                                                   const __grid_constant__ CUtensorMap tmV,
                                                                   const __grid_constant__ CUtensorMap tmO,
                                                                   const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  TcBars* bars = reinterpret_cast<TcBars*>(smem + kTcBarOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = (kNumQHeads / 2) * p.num_seqs * p.num_ztiles;

  if (threadIdx.x == 0) {
    bars->timeout = 0;
    for (int i = 0; i < kItemRing; ++i) {
      mbar_init(&bars->item_full[i], 1);
      mbar_init(&bars->item_empty[i], kItemConsumers);
    }
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int i = 0; i < kTcStages; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_ready[i], 4);
      mbar_init(&bars->o_ready[i], 1);
      mbar_init(&bars->o_free[i], 4);
    }
    fence_barrier_init();
  }
  if (warp == 1) {
    tc::alloc(&bars->tmem_base, kTmemCols);
    tc::relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = bars->tmem_base;
  // everything above overlaps the previous kernel's tail; from here on the
  // kernel reads what that kernel wrote (q, the cache, the work counter)
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    // Longest-first claims when the host's bounds allow a cached prefix (a sequence
    // whose keys exceed its queries by a tile) and the device finds one.
    LptOrder lpt;
    bool longest_first = p.prefix_hint && p.num_seqs <= 32 * kLptPerLane;
    if (longest_first) {
      lpt.init(p, lane);
      longest_first = lpt.prefixed;
    }
    produce(p, &tmQ, &tmK, &tmV, smem, bars, n_items, lane, lpt, longest_first);
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    {
      constexpr uint32_t idS = tc::idesc_bf16_f32(kTcRows, kTcKeys, false, false);
      constexpr uint32_t idO = tc::idesc_bf16_f32(kTcRows, kHeadDim, false, true);
      const uint32_t sQ = smem_u32(smem + kTcQOff);
      // Descriptors are built once; a K-step moves the start address, which
      // sits in the low bits of the descriptor (no carry: smem addresses are
      // below 256 KiB), so stepping adds a compile-time constant.
      // The 8 MMAs of a tile are issued back to back with nothing between
      // them: any per-step arithmetic or branching here halves the tensor rate.
      // every operand descriptor, built once: Q of each head, K and V of each ring stage
      const uint64_t dq0 = tc::smem_desc_sw128(sQ, 16, 1024), dq1 = tc::smem_desc_sw128(sQ + kTcTile, 16, 1024);
      const uint64_t dk0 = tc::smem_desc_sw128(smem_u32(smem + kTcKOff), 16, 1024);
      const uint64_t dk1 = tc::smem_desc_sw128(smem_u32(smem + kTcKOff + kTcTile), 16, 1024);
      const uint64_t dv0 = tc::smem_desc_sw128(smem_u32(smem + kTcVOff), kTcSub, 1024);
      const uint64_t dv1 = tc::smem_desc_sw128(smem_u32(smem + kTcVOff + kTcTile), kTcSub, 1024);
      static_assert(kTcStages == 2, "one descriptor per ring stage");
      auto issue_s = [&](int t, uint32_t tile) {
        const uint64_t dq = t ? dq1 : dq0;
        const uint64_t dk = (tile & 1) ? dk1 : dk0;
        const uint32_t d = tmem + t * kTcKeys;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t o = static_cast<uint64_t>(((k >> 2) * kTcSub + (k & 3) * 32) >> 4);  // K16 step
          tc::mma_ss(d, dq + o, dk + o, idS, k > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int t, uint32_t tile, bool first) {
        // 16 keys = two 8-row groups (SBO 1024 B); dims 0..63 / 64..127 are the two sub-tiles (LBO)
        const uint64_t dv = (tile & 1) ? dv1 : dv0;
        const uint32_t d = tmem + 2 * kTcKeys + t * kHeadDim;
        const uint32_t a = tmem + t * kTcKeys;
        tc::mma_ts(d, a, dv, idO, first ? 0u : 1u);
#pragma unroll
        for (int k = 1; k < 8; ++k) tc::mma_ts(d, a + k * 8, dv + static_cast<uint64_t>((k * 2048) >> 4), idO, 1u);
      };
      uint32_t tt = 0, ic = 0, nslot = 0;
      bool ok = true;
      while (ok) {
        const int rs = nslot % kItemRing;
        if (!(ok = warp_wait(&bars->item_full[rs], (nslot / kItemRing) & 1))) break;
        const Item it = bars->items[rs];
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->item_empty[rs]);
        ++nslot;
        if (it.s < 0) break;
        if (it.invalid) continue;
        const int n = it.n_tiles;
        if (!(ok = warp_wait(&bars->q_full, ic & 1))) break;
        if (!(ok = warp_wait(&bars->k_full[tt % kTcStages], (tt / kTcStages) & 1))) break;
        tc::fence_after();
        if (tc::elect_one()) {
          issue_s(0, tt);
          tc::commit(&bars->s_full[0]);
          issue_s(1, tt);
          tc::commit(&bars->s_full[1]);
          tc::commit(&bars->k_empty[tt % kTcStages]);
          if (n == 1) tc::commit(&bars->q_empty);
        }
        __syncwarp();
        for (int j = 0; j < n; ++j, ++tt) {
          const int st = tt % kTcStages;
          const bool more = j + 1 < n;
          // head A: O_A += P_A(j) V_j, then S_A(j+1).  The operand waits come
          // first, so once P_A(j) is ready nothing stands between it and the MMAs.
          if (!(ok = warp_wait(&bars->v_full[st], (tt / kTcStages) & 1))) break;
          if (more && !(ok = warp_wait(&bars->k_full[(tt + 1) % kTcStages], ((tt + 1) / kTcStages) & 1))) break;
          if (j == 0 && ic > 0 && !(ok = warp_wait(&bars->o_free[0], (ic - 1) & 1))) break;
          if (!(ok = warp_wait(&bars->p_ready[0], tt & 1))) break;
          tc::fence_after();
          if (tc::elect_one()) {
            issue_pv(0, tt, j == 0);
            tc::commit(&bars->o_ready[0]);
            if (more) {
              issue_s(0, tt + 1);
              tc::commit(&bars->s_full[0]);
            }
          }
          __syncwarp();
          // head B: O_B += P_B(j) V_j, then S_B(j+1)
          if (j == 0 && ic > 0 && !(ok = warp_wait(&bars->o_free[1], (ic - 1) & 1))) break;
          if (!(ok = warp_wait(&bars->p_ready[1], tt & 1))) break;
          tc::fence_after();
          if (tc::elect_one()) {
            issue_pv(1, tt, j == 0);
            tc::commit(&bars->o_ready[1]);
            tc::commit(&bars->v_empty[st]);
            if (more) {
              issue_s(1, tt + 1);
              tc::commit(&bars->s_full[1]);
              tc::commit(&bars->k_empty[(tt + 1) % kTcStages]);
              if (j + 2 == n) tc::commit(&bars->q_empty);  // the item's last QK^T MMAs are issued
            }
          }
          __syncwarp();
        }
        ++ic;
      }
      if (!ok && lane == 0) bars->timeout = 1;
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax + epilogue (one warpgroup per head)
    const int t = (warp - 2) >> 2;      // 0: head h0, 1: head h0 + 1
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // query row of the tile = TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t sbuf = lane_base + t * kTcKeys;
    const uint32_t obuf = lane_base + 2 * kTcKeys + t * kHeadDim;
    const float sl2 = p.scale_log2;
    uint32_t tt = 0, ic = 0, nslot = 0;
    bool ok = true;
    while (ok) {
      const int rs = nslot % kItemRing;
      if (!(ok = warp_wait(&bars->item_full[rs], (nslot / kItemRing) & 1))) break;
      const Item it = bars->items[rs];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->item_empty[rs]);
      ++nslot;
      if (it.s < 0) break;
      const int i = it.rbase + r;  // row inside the sequence
      const bool valid = i >= 0 && i < it.Lq;
      if (it.invalid) {
        __nv_bfloat16* orow = p.out + (static_cast<int64_t>(it.q0 + (valid ? i : 0)) * kNumQHeads + it.h0 + t) * kHeadDim;  // a sequence the call cannot serve: zero its rows, flag it
        if (r == 0 && t == 0 && it.h0 == 0) set_error(p.err, it.Lq > it.Lk ? PKV_EFLAG_SEQLEN : PKV_EFLAG_CONTEXT);
        if (valid) {
#pragma unroll
          for (int c = 0; c < 16; ++c) reinterpret_cast<uint4*>(orow)[c] = make_uint4(0u, 0u, 0u, 0u);
        }
        continue;
      }
      const int32_t* table = p.block_table + static_cast<int64_t>(it.s) * p.max_blocks;
      const int pos = it.off + i;


      float m_used = -INFINITY, l = 0.f;
      for (int j = 0; j < it.n_tiles; ++j, ++tt) {
        if (!(ok = warp_wait(&bars->s_full[t], tt & 1))) break;
        tc::fence_after();
        const int key0 = j * kTcKeys;
        const int blk = __ldg(table + key0 / kBlockSize);
        const bool tile_ok = blk >= 0 && blk < p.num_blocks;
        // columns c <= lim of this tile are visible to the row (none of a bad block).  Padding rows
        // (outside the sequence) are never stored and rows do not mix, so they count as fully
        // visible: that keeps their warps off the masked path on every off-diagonal tile.
        const int lim = !valid ? (1 << 20) : (tile_ok ? pos - key0 : -1);
        const bool full = lim >= kTcKeys - 1;
        uint32_t sv[128];
        tc::ld128(sbuf, sv);
        // A warp takes the unmasked path only when all 32 of its rows are fully
        // visible; otherwise all lanes take the masked one.
        const bool wfull = __all_sync(0xffffffffu, full);
        // (one branch per path, each with its TMEM stores, so the two are never both evaluated)
        if (!wfull) mask_row(sv, lim);
        const float mt = row_max(sv) * sl2;
        const bool need = mt > m_used + kRescaleLog2;
        const float m_new = need ? mt : m_used;
        const float alpha = need ? fast_exp2(m_used - m_new) : 1.f;
        m_used = m_new;
        const float negm = m_used == -INFINITY ? 0.f : -m_used;
        const float rs = row_exp(sv, sl2, negm, sbuf);
        l = l * alpha + rs;
        // V rows that hold no token (keys >= Lk, or a bad block) are zeroed before P V reads them
        if (t == 0 && (key0 + kTcKeys > it.Lk || !tile_ok)) {
          const int st = tt % kTcStages;
          if (!(ok = warp_wait(&bars->v_full[st], (tt / kTcStages) & 1))) break;
          if (key0 + r >= it.Lk || !tile_ok) {
            uint4* v0 = reinterpret_cast<uint4*>(smem + kTcVOff + st * kTcTile + r * 128);
            uint4* v1 = reinterpret_cast<uint4*>(smem + kTcVOff + st * kTcTile + kTcSub + r * 128);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              v0[c] = make_uint4(0u, 0u, 0u, 0u);
              v1[c] = make_uint4(0u, 0u, 0u, 0u);
            }
          }
          tc::fence_proxy_async_smem();
        }
        // O must hold P(j-1) V(j-1) before it is rescaled (and before P(j) V(j) lands)
        if (j > 0) {
          tc::fence_after();
          if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
            for (int c4 = 0; c4 < 4; ++c4) {
              uint32_t ov[32];
              tc::ld32(obuf + c4 * 32, ov);
#pragma unroll
              for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
              tc::st32(obuf + c4 * 32, ov);
            }
          }
        }
        tc::wait_st();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_ready[t]);
      }
      if (ok) ok = warp_wait(&bars->o_ready[t], (tt - 1) & 1);
      if (!ok) break;
      // epilogue: read the whole O row in one TMEM load, hand the O columns
      // back to the MMA issuer at once, then normalise.  Each half (64 dims)
      // of the warp's 32 rows goes through a 4 KiB staging buffer (16-byte
      // chunks XOR-swizzled by row, the 128-byte swizzle of the output's tensor
      // map).  When all 32 rows belong to the item's sequence, one lane stores
      // the half with one bulk tensor store and the warp moves on; otherwise
      // the warp reads it back and stores the sequence's rows as whole 128-byte
      // lines, four rows per store instruction (a box would overwrite the
      // neighbouring sequence's rows).
      tc::fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      // which of the warp's 32 rows are stored, and where this lane stores in the
      // read-back pattern (row lane/8 + 4k, 16-byte chunk lane%8)
      const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
      const int srow = lane >> 3, schunk = lane & 7;
      __nv_bfloat16* const gdst =
          p.out + (static_cast<int64_t>(it.q0 + i - lane + srow) * kNumQHeads + it.h0 + t) * kHeadDim + schunk * 8;
      const uint32_t stg = smem_u32(smem + kTcStageOff + (warp - 2) * 4096);
      const bool whole = vmask == 0xffffffffu;
      const int row0 = it.q0 + i - lane;  // token row of the warp's first row
      uint32_t ov[128];
      tc::ld128(obuf, ov);
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->o_free[t]);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        // the half's 64 values, normalised and packed, while the previous bulk store may still read
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          float lo, hi;  // x * inv on a pair: a fused multiply-add of -0 rounds as the multiply does, zeros included
          f2unpack(ffma2(f2pack(__uint_as_float(ov[half * 64 + 2 * c]), __uint_as_float(ov[half * 64 + 2 * c + 1])),
                         f2pack(inv, inv), f2pack(-0.0f, -0.0f)), lo, hi);
          pk[c] = pack_bf16x2(lo, hi);
        }
        // the buffer may still be read by this warp's previous bulk store
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int ch = q ^ (lane & 7);
          st_shared_v4(stg + lane * 128 + ch * 16, pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
        if (whole) {
          tc::fence_proxy_async_smem();  // this thread's staging writes, before the bulk store reads them
          __syncwarp();
          if (lane == 0) tma_store_3d(&tmO, stg, half * 64, it.h0 + t, row0);
        } else {
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int row = srow + 4 * k;  // row of this warp's 32
            const uint4 v = ld_shared_v4(stg + row * 128 + ((schunk ^ (row & 7)) * 16));
            if ((vmask >> row) & 1u) *reinterpret_cast<uint4*>(gdst + k * (4 * kNumQHeads * kHeadDim) + half * 64) = v;
          }
          __syncwarp();
        }
      }
      ++ic;
    }
    if (!ok) bars->timeout = 1;
    if (lane == 0) bulk_wait_all();  // this warp's bulk stores are complete before the CTA ends
  }

  tc::fence_before();
  __syncthreads();
  if (threadIdx.x == 0) {
    if (bars->timeout) set_error(p.err, PKV_EFLAG_TIMEOUT);
    // every CTA has stopped claiming items once it gets here; the last one
    // returns the counters to zero for the next launch that uses them
    __threadfence();
    if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
      atomicExch(p.sched, 0u);
      atomicExch(p.sched + 1, 0u);
    }
  }
  if (warp == 1) {
    tc::fence_after();
    tc::dealloc(tmem, kTmemCols);
  }
}

cudaError_t prefill_tc_init_device() {
  return cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemBytes);
}

cudaError_t launch_prefill_tc(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                              const CUtensorMap& tmO, void* out,
                              const int32_t* cu_q, const int32_t* cu_k, const int32_t* block_table, int num_seqs,
                              int max_blocks, int num_blocks, int max_seqlen_q, int max_seqlen_k, float scale,
                              int num_sms, unsigned* sched, unsigned* err, cudaStream_t stream) {
  if (num_seqs == 0 || max_seqlen_q == 0) return cudaSuccess;
  TcParams prm;
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.cu_q = cu_q;
  prm.cu_k = cu_k;
  prm.block_table = block_table;
  prm.num_seqs = num_seqs;
  prm.num_ztiles = (max_seqlen_q + kTcRows - 1) / kTcRows;
  prm.max_blocks = max_blocks;
  prm.num_blocks = num_blocks;
  prm.max_seqlen_q = max_seqlen_q;
  prm.max_seqlen_k = max_seqlen_k;
  prm.scale_log2 = scale * kLog2e;
  prm.prefix_hint = max_seqlen_k >= max_seqlen_q + kTcKeys ? 1 : 0;
  prm.sched = sched;
  prm.err = err;
  const int64_t items = static_cast<int64_t>(kNumQHeads / 2) * num_seqs * prm.num_ztiles;
  const int grid = static_cast<int>(items < num_sms ? items : num_sms);
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = kTcSmemBytes;
  cfg.stream = stream;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_tc_kernel, tmQ, tmK, tmV, tmO, prm);
}

}  // namespace pkv
