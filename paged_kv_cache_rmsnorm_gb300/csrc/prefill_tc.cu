// K3: causal varlen prefill attention over the paged cache on tcgen05 tensor
// cores (sm_103a), accumulators in tensor memory.
//
// Operation ("Nano-vLLM深度解读（下）" §4 prefill branch with a block table;
// "同一个 Qwen3，两种写法" §3.2 and §3.4): sequence s owns query rows
// cu_q[s]..cu_q[s+1]-1 (Lq) and keys 0..Lk-1 read through block_table row s;
// query row i sits at position Lk - Lq + i and sees keys 0..Lk - Lq + i; query
// head h reads KV head h / 4.
//
// CTA = (pair of query heads {2p, 2p+1} of one GQA group, sequence s, 128-row
// query tile counted from the end of the sequence, so the tiles with the most
// keys launch first).  The two heads share every K/V tile.  10 warps:
//   warp 0      TMA producer: both Q tiles once, then 128-key K and V tiles of
//               KV head p/2 into two 2-deep rings (a tile lies inside one
//               256-token block: one block-table lookup per tile).
//   warp 1      allocates 512 TMEM columns; one thread issues every MMA, in
//               the order PV_A(j), S_A(j+1), PV_B(j), S_B(j+1): while the
//               softmax of one head runs, the tensor core works on the other.
//               S = Q K^T (M=N=128, K=128 as 8 x K16, both operands K-major in
//               128B-swizzled smem); O += P V with P read from TMEM and V
//               MN-major from smem.  Completion travels by tcgen05.commit.
//   warps 2..5  softmax of head A, warps 6..9 softmax of head B: thread =
//               query row = TMEM lane.  One 128-column TMEM load per tile (a
//               single wait), row max and exp2 from registers, the bf16 P
//               written back over the S columns 32 at a time; the causal mask
//               is a per-row column limit applied by selection; lazy rescaling
//               of O (only when the running max grows by more than 2^8).  Warpgroup A zeroes the V rows of keys
//               >= Lk (rows no token has written).  At the end each warpgroup
//               normalises its O, stages it in its own (now free) Q buffer and
//               stores it with TMA.
// TMEM columns: S_A [0,128), S_B [128,256), O_A [256,384), O_B [384,512).
// Registers: one SM sub-partition hosts three of the ten warps, so every
// thread has at most 168 registers (a 16K register file per sub-partition).
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
constexpr int kTcBarOff = kTcVOff + kTcStages * kTcTile;  // 192 KiB
constexpr int kTcSmemBytes = kTcBarOff + 256 + 1024;
constexpr int kTcThreads = 320;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;

struct TcParams {
  __nv_bfloat16* out;
  const int32_t* cu_q;
  const int32_t* cu_k;
  const int32_t* block_table;
  int32_t max_blocks;
  int32_t num_blocks;
  int32_t max_seqlen_q;
  int32_t max_seqlen_k;
  float scale_log2;
  unsigned* err;
};

struct TcBars {
  uint64_t q_full;
  uint64_t k_full[kTcStages], k_empty[kTcStages];
  uint64_t v_full[kTcStages], v_empty[kTcStages];
  uint64_t s_full[2], p_ready[2], o_ready[2];  // per head of the pair
  uint32_t tmem_base;
  int bad;
  int timeout;
};

__device__ __forceinline__ void zero_rows_out(const TcParams& p, int q0, int rbase, int h0) {
  for (int idx = threadIdx.x; idx < 2 * kTcRows * 16; idx += blockDim.x) {
    const int hh = idx / (kTcRows * 16);
    const int rr = rbase + (idx / 16) % kTcRows;
    if (rr < 0) continue;
    __nv_bfloat16* o = p.out + (static_cast<int64_t>(q0 + rr) * kNumQHeads + h0 + hh) * kHeadDim + (idx % 16) * 8;
    *reinterpret_cast<uint4*>(o) = make_uint4(0u, 0u, 0u, 0u);
  }
}

// mbarrier wait whose result is the same for every lane of the warp, so that a
// timeout can never leave part of a warp at a warp-collective tcgen05.ld/st.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, unsigned parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

// Row max of the 128 scores of this thread's S row; with MASKED, columns
// beyond `lim` are excluded (selected to -inf, never multiplied).
template <bool MASKED>
__device__ __forceinline__ float row_max(const uint32_t (&sv)[128], int lim) {
  float m8[8];
#pragma unroll
  for (int a = 0; a < 8; ++a) m8[a] = -INFINITY;
#pragma unroll
  for (int c = 0; c < 128; c += 2) {
    float x0 = __uint_as_float(sv[c]), x1 = __uint_as_float(sv[c + 1]);
    if (MASKED) {
      x0 = c <= lim ? x0 : -INFINITY;
      x1 = c + 1 <= lim ? x1 : -INFINITY;
    }
    m8[(c >> 1) & 7] = fmax3(m8[(c >> 1) & 7], x0, x1);
  }
  return fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
}

// P = exp2(s * scale_log2 - m) as bf16 pairs written over the S columns of
// this row (32 columns at a time); returns the fp32 row sum of P.
template <bool MASKED>
__device__ __forceinline__ float row_exp(const uint32_t (&sv)[128], int lim, float sl2, float negm, uint32_t sbuf) {
  float sum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int c4 = 0; c4 < 4; ++c4) {
    uint32_t pk[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const int col = c4 * 32 + 2 * c;
      float p0 = fast_exp2(fmaf(__uint_as_float(sv[col]), sl2, negm));
      float p1 = fast_exp2(fmaf(__uint_as_float(sv[col + 1]), sl2, negm));
      if (MASKED) {
        p0 = col <= lim ? p0 : 0.f;
        p1 = col + 1 <= lim ? p1 : 0.f;
      }
      sum[c & 3] += p0 + p1;
      pk[c] = pack_bf16x2(p0, p1);
    }
    tc::st16(sbuf + c4 * 16, pk);
  }
  return (sum[0] + sum[1]) + (sum[2] + sum[3]);
}

__global__ void __launch_bounds__(kTcThreads, 1) prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                                                                   const __grid_constant__ CUtensorMap tmK,
                                                                   const __grid_constant__ CUtensorMap tmV,
                                                                   const __grid_constant__ CUtensorMap tmO,
                                                                   const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  TcBars* bars = reinterpret_cast<TcBars*>(smem + kTcBarOff);

  const int h0 = 2 * blockIdx.x, s = blockIdx.y, zt = blockIdx.z;
  const int g = h0 / kGroup;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int q0 = __ldg(p.cu_q + s), q1 = __ldg(p.cu_q + s + 1);
  const int Lq = q1 - q0;
  const int Lk = __ldg(p.cu_k + s + 1) - __ldg(p.cu_k + s);
  const int r1 = Lq - zt * kTcRows;  // this CTA covers sequence rows [r1 - 128, r1)
  if (r1 <= 0) return;
  const int rbase = r1 - kTcRows;
  if (Lq > Lk || Lk > p.max_blocks * kBlockSize || Lq > p.max_seqlen_q || Lk > p.max_seqlen_k) {
    if (threadIdx.x == 0 && h0 == 0) set_error(p.err, Lq > Lk ? PKV_EFLAG_SEQLEN : PKV_EFLAG_CONTEXT);
    zero_rows_out(p, q0, rbase, h0);
    return;
  }
  const int off = Lk - Lq;       // position of sequence row 0
  const int key_end = off + r1;  // keys [0, key_end) are visible to some row of the tile
  const int n_tiles = (key_end + kTcKeys - 1) / kTcKeys;
  const int32_t* table = p.block_table + static_cast<int64_t>(s) * p.max_blocks;

  if (threadIdx.x == 0) {
    bars->bad = 0;
    bars->timeout = 0;
  }
  __syncthreads();
  // every block id the tile will touch must lie in the pool
  for (int i = threadIdx.x; i < (key_end + kBlockSize - 1) / kBlockSize; i += blockDim.x) {
    const int b = __ldg(table + i);
    if (b < 0 || b >= p.num_blocks) bars->bad = 1;
  }
  __syncthreads();
  if (bars->bad) {
    if (threadIdx.x == 0) set_error(p.err, PKV_EFLAG_BLOCK_ID);
    zero_rows_out(p, q0, rbase, h0);
    return;
  }

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
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

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(&bars->q_full, 2 * kTcTile);
      for (int t = 0; t < 2; ++t) {
        tma_load_3d(smem + kTcQOff + t * kTcTile, &tmQ, &bars->q_full, 0, h0 + t, q0 + rbase);
        tma_load_3d(smem + kTcQOff + t * kTcTile + kTcSub, &tmQ, &bars->q_full, 64, h0 + t, q0 + rbase);
      }
      for (int j = 0; j < n_tiles; ++j) {
        const int st = j % kTcStages;
        const int key0 = j * kTcKeys;
        const int slot0 = __ldg(table + key0 / kBlockSize) * kBlockSize + (key0 % kBlockSize);
        if (j >= kTcStages && !mbar_wait(&bars->k_empty[st], ((j / kTcStages) - 1) & 1)) {
          bars->timeout = 1;
          break;
        }
        uint8_t* kd = smem + kTcKOff + st * kTcTile;
        mbar_arrive_expect_tx(&bars->k_full[st], kTcTile);
        tma_load_3d(kd, &tmK, &bars->k_full[st], 0, g, slot0);
        tma_load_3d(kd + kTcSub, &tmK, &bars->k_full[st], 64, g, slot0);
        if (j >= kTcStages && !mbar_wait(&bars->v_empty[st], ((j / kTcStages) - 1) & 1)) {
          bars->timeout = 1;
          break;
        }
        uint8_t* vd = smem + kTcVOff + st * kTcTile;
        mbar_arrive_expect_tx(&bars->v_full[st], kTcTile);
        tma_load_3d(vd, &tmV, &bars->v_full[st], 0, g, slot0);
        tma_load_3d(vd + kTcSub, &tmV, &bars->v_full[st], 64, g, slot0);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = tc::idesc_bf16_f32(kTcRows, kTcKeys, false, false);
      constexpr uint32_t idO = tc::idesc_bf16_f32(kTcRows, kHeadDim, false, true);
      const uint32_t sQ = smem_u32(smem + kTcQOff);
      // Descriptors are built once per operand tile; a K-step moves the start
      // address, which sits in the low bits of the descriptor (no carry: smem
      // addresses are below 256 KiB), so stepping adds a compile-time constant.
      // The 8 MMAs of a tile are issued back to back with nothing between
      // them: any per-step arithmetic or branching here halves the tensor rate.
      auto issue_s = [&](int t, int j) {
        const uint64_t dq = tc::smem_desc_sw128(sQ + t * kTcTile, 16, 1024);
        const uint64_t dk = tc::smem_desc_sw128(smem_u32(smem + kTcKOff + (j % kTcStages) * kTcTile), 16, 1024);
        const uint32_t d = tmem + t * kTcKeys;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t o = static_cast<uint64_t>(((k >> 2) * kTcSub + (k & 3) * 32) >> 4);  // K16 step
          tc::mma_ss(d, dq + o, dk + o, idS, k > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int t, int j) {
        // 16 keys = two 8-row groups (SBO 1024 B); dims 0..63 / 64..127 are the two sub-tiles (LBO)
        const uint64_t dv = tc::smem_desc_sw128(smem_u32(smem + kTcVOff + (j % kTcStages) * kTcTile), kTcSub, 1024);
        const uint32_t d = tmem + 2 * kTcKeys + t * kHeadDim;
        const uint32_t a = tmem + t * kTcKeys;
        tc::mma_ts(d, a, dv, idO, j > 0 ? 1u : 0u);
#pragma unroll
        for (int k = 1; k < 8; ++k) tc::mma_ts(d, a + k * 8, dv + static_cast<uint64_t>((k * 2048) >> 4), idO, 1u);
      };
      bool ok = mbar_wait(&bars->q_full, 0) && mbar_wait(&bars->k_full[0], 0);
      if (ok) {
        tc::fence_after();
        issue_s(0, 0);
        tc::commit(&bars->s_full[0]);
        issue_s(1, 0);
        tc::commit(&bars->s_full[1]);
        tc::commit(&bars->k_empty[0]);
      }
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int st = j % kTcStages;
        const bool more = j + 1 < n_tiles;
        // head A: O_A += P_A(j) V_j, then S_A(j+1).  The operand waits come first,
        // so that once P_A(j) is ready nothing stands between it and the MMAs.
        if (!(ok = mbar_wait(&bars->v_full[st], (j / kTcStages) & 1))) break;
        if (more && !(ok = mbar_wait(&bars->k_full[(j + 1) % kTcStages], ((j + 1) / kTcStages) & 1))) break;
        if (!(ok = mbar_wait(&bars->p_ready[0], j & 1))) break;
        tc::fence_after();
        issue_pv(0, j);
        tc::commit(&bars->o_ready[0]);
        if (more) {
          issue_s(0, j + 1);
          tc::commit(&bars->s_full[0]);
        }
        // head B: O_B += P_B(j) V_j, then S_B(j+1)
        if (!(ok = mbar_wait(&bars->p_ready[1], j & 1))) break;
        tc::fence_after();
        issue_pv(1, j);
        tc::commit(&bars->o_ready[1]);
        tc::commit(&bars->v_empty[st]);
        if (more) {
          issue_s(1, j + 1);
          tc::commit(&bars->s_full[1]);
          tc::commit(&bars->k_empty[(j + 1) % kTcStages]);
        }
      }
      if (!ok) bars->timeout = 1;
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax + epilogue (one warpgroup per head)
    const int t = (warp - 2) >> 2;      // 0: head h0, 1: head h0 + 1
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // query row of the tile = TMEM lane
    const int i = rbase + r;            // row inside the sequence
    const bool valid = i >= 0;
    const int pos = off + i;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t sbuf = lane_base + t * kTcKeys;
    const uint32_t obuf = lane_base + 2 * kTcKeys + t * kHeadDim;
    const float sl2 = p.scale_log2;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      if (!(ok = warp_wait(&bars->s_full[t], j & 1))) break;
      tc::fence_after();
      const int key0 = j * kTcKeys;
      // columns c <= lim of this tile are visible to the row (none if the row is padding)
      const int lim = valid ? pos - key0 : -1;
      const bool full = lim >= kTcKeys - 1;
      // the whole S row in one TMEM load (one wait per tile), max and exp2 from registers
      uint32_t sv[128];
      tc::ld128(sbuf, sv);
      // A warp takes the unmasked path only when all 32 of its rows are fully
      // visible; otherwise all lanes take the masked one.  Two separate code
      // paths keep the per-column tests out of every off-diagonal tile.
      const bool wfull = __all_sync(0xffffffffu, full);
      const float mrow = wfull ? row_max<false>(sv, lim) : row_max<true>(sv, lim);
      const float mt = mrow * sl2;
      const bool need = mt > m_used + kRescaleLog2;
      const float m_new = need ? mt : m_used;
      const float alpha = need ? fast_exp2(m_used - m_new) : 1.f;
      m_used = m_new;
      const float negm = m_used == -INFINITY ? 0.f : -m_used;
      const float rs = wfull ? row_exp<false>(sv, lim, sl2, negm, sbuf) : row_exp<true>(sv, lim, sl2, negm, sbuf);
      l = l * alpha + rs;
      // keys >= Lk are rows no token has written: zero them in V before P V reads them
      if (t == 0 && key0 + kTcKeys > Lk) {
        const int st = j % kTcStages;
        if (!(ok = warp_wait(&bars->v_full[st], (j / kTcStages) & 1))) break;
        if (key0 + r >= Lk) {
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
        if (!(ok = warp_wait(&bars->o_ready[t], (j - 1) & 1))) break;
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
    if (ok) ok = warp_wait(&bars->o_ready[t], (n_tiles - 1) & 1);
    if (!ok) bars->timeout = 1;
    uint8_t* stg = smem + kTcQOff + t * kTcTile;  // this head's Q buffer: every MMA that read it has completed
    if (ok) {
      tc::fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      float inv_dep = inv;
      uint4* grow = reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(q0 + (valid ? i : 0)) * kNumQHeads + h0 + t) *
                                                         kHeadDim);
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {  // 32 columns = four 16-byte chunks of the output row
        uint32_t ov[32];
        tc::ld32_after(obuf + c4 * 32, ov, inv_dep);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int c = c4 * 4 + q;
          const uint4 v = make_uint4(
              pack_bf16x2(__uint_as_float(ov[8 * q]) * inv, __uint_as_float(ov[8 * q + 1]) * inv),
              pack_bf16x2(__uint_as_float(ov[8 * q + 2]) * inv, __uint_as_float(ov[8 * q + 3]) * inv),
              pack_bf16x2(__uint_as_float(ov[8 * q + 4]) * inv, __uint_as_float(ov[8 * q + 5]) * inv),
              pack_bf16x2(__uint_as_float(ov[8 * q + 6]) * inv, __uint_as_float(ov[8 * q + 7]) * inv));
          if (rbase >= 0) {
            *reinterpret_cast<uint4*>(stg + (c >> 3) * kTcSub + sw128(r, c & 7)) = v;
          } else if (valid) {
            grow[c] = v;
          }
        }
      }
    }
    if (rbase >= 0) {  // uniform over the CTA: every thread of the warpgroup reaches the barrier
      tc::fence_proxy_async_smem();
      asm volatile("bar.sync %0, 128;" ::"r"(1 + t) : "memory");
      if (quarter == 2 && lane == 0 && !bars->timeout) {  // the warpgroup's first warp
        tc::tma_store_3d(&tmO, stg, 0, h0 + t, q0 + rbase);
        tc::tma_store_3d(&tmO, stg + kTcSub, 64, h0 + t, q0 + rbase);
        tc::bulk_commit();
        tc::bulk_wait0();
      }
    }
  }

  tc::fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && bars->timeout) set_error(p.err, PKV_EFLAG_TIMEOUT);
  if (warp == 1) {
    tc::fence_after();
    tc::dealloc(tmem, kTmemCols);
  }
}

cudaError_t prefill_tc_init_device() {
  return cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemBytes);
}

cudaError_t launch_prefill_tc(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                              const CUtensorMap& tmO, void* out, const int32_t* cu_q, const int32_t* cu_k,
                              const int32_t* block_table, int num_seqs, int max_blocks, int num_blocks,
                              int max_seqlen_q, int max_seqlen_k, float scale, unsigned* err, cudaStream_t stream) {
  if (num_seqs == 0 || max_seqlen_q == 0) return cudaSuccess;
  TcParams prm;
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.cu_q = cu_q;
  prm.cu_k = cu_k;
  prm.block_table = block_table;
  prm.max_blocks = max_blocks;
  prm.num_blocks = num_blocks;
  prm.max_seqlen_q = max_seqlen_q;
  prm.max_seqlen_k = max_seqlen_k;
  prm.scale_log2 = scale * kLog2e;
  prm.err = err;
  dim3 grid(kNumQHeads / 2, num_seqs, (max_seqlen_q + kTcRows - 1) / kTcRows);
  prefill_tc_kernel<<<grid, kTcThreads, kTcSmemBytes, stream>>>(tmQ, tmK, tmV, tmO, prm);
  return cudaGetLastError();
}

}  // namespace pkv
