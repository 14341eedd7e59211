// K3: causal varlen prefill attention over the paged cache on tcgen05 tensor
// cores (sm_103a), accumulators in tensor memory.
//
// Operation ("Nano-vLLM深度解读（下）" §4 prefill branch with a block table;
// "同一个 Qwen3，两种写法" §3.2 and §3.4): sequence s owns query rows
// cu_q[s]..cu_q[s+1]-1 (Lq) and keys 0..Lk-1 read through block_table row s;
// query row i sits at position Lk - Lq + i and sees keys 0..Lk - Lq + i; query
// head h reads KV head h / 4.
//
// CTA = (query head h, sequence s, 128-row query tile counted from the end of
// the sequence, so the tiles with the most keys launch first); 6 warps:
//   warp 0      TMA producer: the Q tile once, then 128-key K and V tiles of
//               KV head h/4 into two 3-deep rings (each tile lies inside one
//               256-token block: one block-table lookup per tile).
//   warp 1      allocates 512 TMEM columns; one thread issues all MMAs:
//               S_j = Q K_j^T (M=N=128, K=128: 8 x K16, both operands K-major
//               in 128B-swizzled smem) into a double-buffered fp32 S in TMEM,
//               then O += P_{j-1} V_{j-1} with P read from TMEM and V
//               MN-major from smem.  Completion is signalled by tcgen05.commit.
//   warps 2..5  softmax: thread = query row = TMEM lane.  Loads its S row,
//               applies the causal mask by selection, keeps a running max in
//               the exp2 domain with lazy rescaling (O in TMEM is rescaled only
//               when the max grows by more than 2^8), writes P as bf16 into the
//               S columns, zeroes V rows of keys >= Lk (unwritten cache rows),
//               and at the end normalises O and writes bf16 rows to global.
// TMEM columns: S0 [0,128), S1 [128,256), O [256,384).
// Every mbarrier wait is bounded; on timeout the CTA flags the error word and
// still releases its TMEM.
#include "tcgen05.cuh"

namespace pkv {

constexpr int kTcRows = 128;
constexpr int kTcKeys = 128;
constexpr int kTcStages = 3;
constexpr int kTcSub = 128 * 128;          // [128 rows][64 dims] bf16, 128B-swizzled: 16 KiB
constexpr int kTcTile = 2 * kTcSub;        // [128][128] bf16: 32 KiB
constexpr int kTcQOff = 0;
constexpr int kTcKOff = kTcTile;
constexpr int kTcVOff = kTcKOff + kTcStages * kTcTile;
constexpr int kTcBarOff = kTcVOff + kTcStages * kTcTile;  // 224 KiB
constexpr int kTcSmemBytes = kTcBarOff + 256 + 1024;
constexpr int kTcThreads = 192;
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
  uint64_t s_full[2], p_ready[2];
  uint64_t o_ready;
  uint32_t tmem_base;
  int bad;
  int timeout;
};

__device__ __forceinline__ void zero_rows_out(const TcParams& p, int q0, int rbase, int h) {
  for (int idx = threadIdx.x; idx < kTcRows * 16; idx += blockDim.x) {
    const int rr = rbase + idx / 16;
    if (rr < 0) continue;
    __nv_bfloat16* o = p.out + (static_cast<int64_t>(q0 + rr) * kNumQHeads + h) * kHeadDim + (idx % 16) * 8;
    *reinterpret_cast<uint4*>(o) = make_uint4(0u, 0u, 0u, 0u);
  }
}

__global__ void __launch_bounds__(kTcThreads, 1) prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                                                                   const __grid_constant__ CUtensorMap tmK,
                                                                   const __grid_constant__ CUtensorMap tmV,
                                                                   const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  TcBars* bars = reinterpret_cast<TcBars*>(smem + kTcBarOff);

  const int h = blockIdx.x, s = blockIdx.y, zt = blockIdx.z;
  const int g = h / kGroup;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int q0 = __ldg(p.cu_q + s), q1 = __ldg(p.cu_q + s + 1);
  const int Lq = q1 - q0;
  const int Lk = __ldg(p.cu_k + s + 1) - __ldg(p.cu_k + s);
  const int r1 = Lq - zt * kTcRows;  // this CTA covers sequence rows [r1 - 128, r1)
  if (r1 <= 0) return;
  const int rbase = r1 - kTcRows;
  if (Lq > Lk || Lk > p.max_blocks * kBlockSize || Lq > p.max_seqlen_q || Lk > p.max_seqlen_k) {
    if (threadIdx.x == 0 && h == 0) set_error(p.err, Lq > Lk ? PKV_EFLAG_SEQLEN : PKV_EFLAG_CONTEXT);
    zero_rows_out(p, q0, rbase, h);
    return;
  }
  const int off = Lk - Lq;          // position of sequence row 0
  const int key_end = off + r1;     // keys [0, key_end) are visible to some row of the tile
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
    zero_rows_out(p, q0, rbase, h);
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
    }
    mbar_init(&bars->o_ready, 1);
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
      mbar_arrive_expect_tx(&bars->q_full, kTcTile);
      tma_load_3d(smem + kTcQOff, &tmQ, &bars->q_full, 0, h, q0 + rbase);
      tma_load_3d(smem + kTcQOff + kTcSub, &tmQ, &bars->q_full, 64, h, q0 + rbase);
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
      bool ok = mbar_wait(&bars->q_full, 0);
      for (int j = 0; ok && j <= n_tiles; ++j) {
        if (j < n_tiles) {
          const int st = j % kTcStages;
          if (!(ok = mbar_wait(&bars->k_full[st], (j / kTcStages) & 1))) break;
          tc::fence_after();
          const uint32_t sK = smem_u32(smem + kTcKOff + st * kTcTile);
          const uint32_t dS = tmem + (j & 1) * kTcKeys;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t o = (k >> 2) * kTcSub + (k & 3) * 32;  // K16 step: 32 bytes inside the swizzle row
            tc::mma_ss(dS, tc::smem_desc_sw128(sQ + o, 16, 1024), tc::smem_desc_sw128(sK + o, 16, 1024), idS,
                       k > 0);
          }
          tc::commit(&bars->s_full[j & 1]);
          tc::commit(&bars->k_empty[st]);
        }
        if (j > 0) {
          const int jj = j - 1;
          const int st = jj % kTcStages;
          if (!(ok = mbar_wait(&bars->p_ready[jj & 1], (jj >> 1) & 1))) break;
          if (!(ok = mbar_wait(&bars->v_full[st], (jj / kTcStages) & 1))) break;
          tc::fence_after();
          const uint32_t sV = smem_u32(smem + kTcVOff + st * kTcTile);
          const uint32_t aP = tmem + (jj & 1) * kTcKeys;  // P: bf16 pairs in the first 64 columns
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            // 16 keys = two 8-row groups (SBO 1024 B); d 0..63 / 64..127 are the two sub-tiles (LBO)
            tc::mma_ts(tmem + 2 * kTcKeys, aP + k * 8, tc::smem_desc_sw128(sV + k * 2048, kTcSub, 1024), idO,
                       (jj > 0 || k > 0) ? 1u : 0u);
          }
          tc::commit(&bars->v_empty[st]);
          tc::commit(&bars->o_ready);
        }
      }
      if (!ok) bars->timeout = 1;
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax + epilogue
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;       // query row of the tile = TMEM lane
    const int i = rbase + r;                 // row inside the sequence
    const bool valid = i >= 0;
    const int pos = off + i;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      if (!(ok = mbar_wait(&bars->s_full[j & 1], (j >> 1) & 1))) break;
      tc::fence_after();
      const uint32_t sbuf = lane_base + (j & 1) * kTcKeys;
      uint32_t sv[4][32];
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) tc::ld32(sbuf + c4 * 32, sv[c4]);
      const int key0 = j * kTcKeys;
      const bool unmasked = valid && key0 + kTcKeys - 1 <= pos;
      float mx = -INFINITY;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          float v = __uint_as_float(sv[c4][c]);
          if (!unmasked) v = (valid && key0 + c4 * 32 + c <= pos) ? v : -INFINITY;
          sv[c4][c] = __float_as_uint(v);
          mx = fmaxf(mx, v);
        }
      const float mt = mx * p.scale_log2;
      const bool need = mt > m_used + kRescaleLog2;
      const float m_new = need ? mt : m_used;
      const float alpha = need ? fast_exp2(m_used - m_new) : 1.f;
      m_used = m_new;
      const float mu = m_used == -INFINITY ? 0.f : m_used;
      float rs = 0.f;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int col = half * 64 + 2 * c;
          const float p0 = fast_exp2(fmaf(__uint_as_float(sv[col >> 5][col & 31]), p.scale_log2, -mu));
          const float p1 = fast_exp2(fmaf(__uint_as_float(sv[(col + 1) >> 5][(col + 1) & 31]), p.scale_log2, -mu));
          rs += p0 + p1;
          pk[c] = pack_bf16x2(p0, p1);
        }
        tc::st32(sbuf + half * 32, pk);
      }
      l = l * alpha + rs;
      // keys >= Lk are unwritten cache rows: zero their V rows before P V reads them
      if (key0 + kTcKeys > Lk) {
        const int st = j % kTcStages;
        if (!(ok = mbar_wait(&bars->v_full[st], (j / kTcStages) & 1))) break;
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
      // O must hold P_{j-1} V_{j-1} before it is rescaled (and before P_j V_j lands)
      if (j > 0) {
        if (!(ok = mbar_wait(&bars->o_ready, (j - 1) & 1))) break;
        tc::fence_after();
        if (__any_sync(0xffffffffu, need)) {
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            uint32_t ov[32];
            tc::ld32(lane_base + 2 * kTcKeys + c4 * 32, ov);
#pragma unroll
            for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
            tc::st32(lane_base + 2 * kTcKeys + c4 * 32, ov);
          }
        }
      }
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_ready[j & 1]);
    }
    if (ok) ok = mbar_wait(&bars->o_ready, (n_tiles - 1) & 1);
    if (!ok) {
      bars->timeout = 1;
    } else {
      tc::fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* orow = p.out + (static_cast<int64_t>(q0 + (valid ? i : 0)) * kNumQHeads + h) * kHeadDim;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        uint32_t ov[32];
        tc::ld32(lane_base + 2 * kTcKeys + c4 * 32, ov);
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c4 * 32);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            dst[c] = make_uint4(pack_bf16x2(__uint_as_float(ov[8 * c]) * inv, __uint_as_float(ov[8 * c + 1]) * inv),
                                pack_bf16x2(__uint_as_float(ov[8 * c + 2]) * inv, __uint_as_float(ov[8 * c + 3]) * inv),
                                pack_bf16x2(__uint_as_float(ov[8 * c + 4]) * inv, __uint_as_float(ov[8 * c + 5]) * inv),
                                pack_bf16x2(__uint_as_float(ov[8 * c + 6]) * inv, __uint_as_float(ov[8 * c + 7]) * inv));
          }
        }
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

cudaError_t launch_prefill_tc(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV, void* out,
                              const int32_t* cu_q, const int32_t* cu_k, const int32_t* block_table, int num_seqs,
                              int max_blocks, int num_blocks, int max_seqlen_q, int max_seqlen_k, float scale,
                              unsigned* err, cudaStream_t stream) {
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
  dim3 grid(kNumQHeads, num_seqs, (max_seqlen_q + kTcRows - 1) / kTcRows);
  prefill_tc_kernel<<<grid, kTcThreads, kTcSmemBytes, stream>>>(tmQ, tmK, tmV, prm);
  return cudaGetLastError();
}

}  // namespace pkv
