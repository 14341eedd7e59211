// K3 (first version): causal varlen prefill attention over the paged cache,
// mma.sync m16n8k16 tensor-core tiles, K/V streamed by TMA.
//
// Operation ("Nano-vLLM深度解读（下）" §4 prefill branch; "同一个 Qwen3，两种写法"
// §3.2, §3.4): sequence s owns query rows cu_q[s]..cu_q[s+1]-1 (Lq of them)
// and keys 0..Lk-1 through block_table row s; query row i sits at position
// Lk - Lq + i and sees keys 0..Lk - Lq + i; q head h reads KV head h / 4.
//
// CTA = (query head h, sequence s, 64-row query tile counted from the end of
// the sequence), so the tiles with the most keys are launched first.  A
// producer warp streams 64-key K/V tiles of KV head h/4 through a 3-stage TMA
// ring; 4 consumer warps own 16 query rows each and run S = Q K^T, an online
// softmax in the exp2 domain, and O += P V.  Keys past the causal diagonal are
// selected to -inf; V rows of keys >= Lk (unwritten cache rows) are zeroed in
// registers so NaN sentinels never reach the output.
#include "common.cuh"

namespace pkv {

constexpr int kPfTile = 64;      // keys per stage
constexpr int kPfRows = 64;      // query rows per CTA
constexpr int kPfStages = 3;
constexpr int kPfConsumerWarps = 4;
constexpr int kPfThreads = (kPfConsumerWarps + 1) * 32;
constexpr int kPfSubBytes = kPfTile * 64 * 2;
constexpr int kPfStageBytes = 4 * kPfSubBytes;
constexpr int kPfSmemBytes = kPfStages * kPfStageBytes + 1024 + 256;

struct PrefillParams {
  const __nv_bfloat16* q;
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

__global__ void __launch_bounds__(kPfThreads) prefill_mma_kernel(const __grid_constant__ CUtensorMap tmK,
                                                                 const __grid_constant__ CUtensorMap tmV,
                                                                 const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kPfStages * kPfStageBytes);
  uint64_t* empty = full + kPfStages;
  int* tile_bad = reinterpret_cast<int*>(empty + kPfStages);

  const int h = blockIdx.x, s = blockIdx.y, zt = blockIdx.z;
  const int g = h / kGroup;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int q0 = __ldg(p.cu_q + s), q1 = __ldg(p.cu_q + s + 1);
  const int Lq = q1 - q0;
  const int Lk = __ldg(p.cu_k + s + 1) - __ldg(p.cu_k + s);
  const int r1 = Lq - zt * kPfRows;  // this tile covers sequence rows [r1 - 64, r1)
  if (r1 <= 0) return;
  const int rbase = r1 - kPfRows;
  if (Lq > Lk || Lk > p.max_blocks * kBlockSize || Lq > p.max_seqlen_q || Lk > p.max_seqlen_k || Lq < 0) {
    // invalid sequence: zero its rows, flag it
    if (threadIdx.x == 0 && h == 0) set_error(p.err, Lq > Lk ? PKV_EFLAG_SEQLEN : PKV_EFLAG_CONTEXT);
    for (int idx = threadIdx.x; idx < kPfRows * (kHeadDim / 8); idx += blockDim.x) {
      const int rr = rbase + idx / (kHeadDim / 8);
      if (rr < 0) continue;
      __nv_bfloat16* o = p.out + (static_cast<int64_t>(q0 + rr) * kNumQHeads + h) * kHeadDim + (idx % 16) * 8;
      *reinterpret_cast<uint4*>(o) = make_uint4(0u, 0u, 0u, 0u);
    }
    return;
  }
  const int off = Lk - Lq;                     // position of sequence row 0
  const int key_end = off + r1;                // keys [0, key_end) are visible to some row
  const int n_tiles = (key_end + kPfTile - 1) / kPfTile;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kPfStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kPfConsumerWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kPfConsumerWarps) {
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const int32_t* row = p.block_table + static_cast<int64_t>(s) * p.max_blocks;
      for (int i = 0; i < n_tiles; ++i) {
        const int st = i % kPfStages;
        if (i >= kPfStages && !mbar_wait(&empty[st], ((i / kPfStages) - 1) & 1)) {
          set_error(p.err, PKV_EFLAG_TIMEOUT);
          break;
        }
        const int key0 = i * kPfTile;
        const int blk = __ldg(row + key0 / kBlockSize);
        uint8_t* dst = smem + st * kPfStageBytes;
        if (blk < 0 || blk >= p.num_blocks) {
          set_error(p.err, PKV_EFLAG_BLOCK_ID);
          tile_bad[st] = 1;
          mbar_arrive(&full[st]);
          continue;
        }
        tile_bad[st] = 0;
        const int slot0 = blk * kBlockSize + (key0 % kBlockSize);
        mbar_arrive_expect_tx(&full[st], kPfStageBytes);
        tma_load_3d(dst, &tmK, &full[st], 0, g, slot0);
        tma_load_3d(dst + kPfSubBytes, &tmK, &full[st], 64, g, slot0);
        tma_load_3d(dst + 2 * kPfSubBytes, &tmV, &full[st], 0, g, slot0);
        tma_load_3d(dst + 3 * kPfSubBytes, &tmV, &full[st], 64, g, slot0);
      }
    }
    __syncwarp();
    return;
  }

  // ---------------------------------------------------------------- consumers
  const int c = lane & 3;
  const int wrow = rbase + warp * 16;  // sequence row of this warp's fragment row 0
  const int ra = wrow + (lane >> 2), rb = ra + 8;  // the two rows this lane holds
  const bool va = ra >= 0, vb = rb >= 0;
  const int pa = off + ra, pb = off + rb;          // their positions
  uint32_t qa[8][4];
  {
    const uint32_t* qra =
        reinterpret_cast<const uint32_t*>(p.q + (static_cast<int64_t>(q0 + (va ? ra : 0)) * kNumQHeads + h) * kHeadDim);
    const uint32_t* qrb =
        reinterpret_cast<const uint32_t*>(p.q + (static_cast<int64_t>(q0 + (vb ? rb : 0)) * kNumQHeads + h) * kHeadDim);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      qa[ks][0] = va ? __ldg(qra + ks * 8 + c) : 0u;
      qa[ks][1] = vb ? __ldg(qrb + ks * 8 + c) : 0u;
      qa[ks][2] = va ? __ldg(qra + ks * 8 + 4 + c) : 0u;
      qa[ks][3] = vb ? __ldg(qrb + ks * 8 + 4 + c) : 0u;
    }
  }
  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
  const bool warp_live = wrow + 15 >= 0;
  const int warp_last_pos = off + wrow + 15;  // keys beyond this are masked for the whole warp
  const int warp_first_pos = off + wrow;

  for (int i = 0; i < n_tiles; ++i) {
    const int st = i % kPfStages;
    if (!mbar_wait(&full[st], (i / kPfStages) & 1)) {
      if (lane == 0) set_error(p.err, PKV_EFLAG_TIMEOUT);
      break;
    }
    const int key0 = i * kPfTile;
    if (warp_live && !tile_bad[st] && key0 <= warp_last_pos) {
      const uint32_t kst = smem_u32(smem + st * kPfStageBytes);
      const uint32_t vst = kst + 2 * kPfSubBytes;
      float sc[8][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
      const int mi = lane >> 3;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          const int r = np * 16 + (mi >> 1) * 8 + (lane & 7);
          const uint32_t addr = kst + (ks >> 2) * kPfSubBytes + sw128(r, (ks & 3) * 2 + (mi & 1));
          uint32_t b0, b1, b2, b3;
          ldsm_x4(addr, b0, b1, b2, b3);
          mma_bf16_16816(sc[2 * np], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
          mma_bf16_16816(sc[2 * np + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
        }
      }
      // scale + causal mask (only tiles that reach past the warp's first position need it)
      const bool need_mask = key0 + kPfTile - 1 > warp_first_pos;
      float mxa = -INFINITY, mxb = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int kk = key0 + nt * 8 + 2 * c + j;
          float ta = sc[nt][j] * p.scale_log2;
          float tb = sc[nt][2 + j] * p.scale_log2;
          if (need_mask) {
            ta = (va && kk <= pa) ? ta : -INFINITY;
            tb = (vb && kk <= pb) ? tb : -INFINITY;
          }
          sc[nt][j] = ta;
          sc[nt][2 + j] = tb;
          mxa = fmaxf(mxa, ta);
          mxb = fmaxf(mxb, tb);
        }
      }
      mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 1));
      mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 2));
      mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 1));
      mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 2));
      const float mna = fmaxf(m_a, mxa), mnb = fmaxf(m_b, mxb);
      const float mua = mna == -INFINITY ? 0.f : mna, mub = mnb == -INFINITY ? 0.f : mnb;
      const float aa = fast_exp2(m_a - mua), ab = fast_exp2(m_b - mub);
      m_a = mna;
      m_b = mnb;
      float sa = 0.f, sb = 0.f;
      uint32_t pk[8][2];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const float p0 = fast_exp2(sc[nt][0] - mua), p1 = fast_exp2(sc[nt][1] - mua);
        const float p2 = fast_exp2(sc[nt][2] - mub), p3 = fast_exp2(sc[nt][3] - mub);
        sa += p0 + p1;
        sb += p2 + p3;
        pk[nt][0] = pack_bf16x2(p0, p1);
        pk[nt][1] = pack_bf16x2(p2, p3);
      }
      l_a = l_a * aa + sa;
      l_b = l_b * ab + sb;
#pragma unroll
      for (int dt = 0; dt < 16; ++dt) {
        o[dt][0] *= aa;
        o[dt][1] *= aa;
        o[dt][2] *= ab;
        o[dt][3] *= ab;
      }
      const int nvalid = Lk - key0;  // keys >= Lk hold no token: zero their V values
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int r = kk * 16 + (mi & 1) * 8 + (lane & 7);
        const int kb = kk * 16;
        const bool tail = nvalid < kb + 16;
        const uint32_t keep_lo = (kb + 2 * c < nvalid ? 0x0000FFFFu : 0u) | (kb + 2 * c + 1 < nvalid ? 0xFFFF0000u : 0u);
        const uint32_t keep_hi =
            (kb + 8 + 2 * c < nvalid ? 0x0000FFFFu : 0u) | (kb + 9 + 2 * c < nvalid ? 0xFFFF0000u : 0u);
#pragma unroll
        for (int dp = 0; dp < 8; ++dp) {
          const int d0 = dp * 16 + (mi >> 1) * 8;
          const uint32_t addr = vst + (d0 >> 6) * kPfSubBytes + sw128(r, (d0 & 63) >> 3);
          uint32_t v0, v1, v2, v3;
          ldsm_x4_t(addr, v0, v1, v2, v3);
          if (tail) {
            v0 &= keep_lo;
            v1 &= keep_hi;
            v2 &= keep_lo;
            v3 &= keep_hi;
          }
          mma_bf16_16816(o[2 * dp], pk[2 * kk][0], pk[2 * kk][1], pk[2 * kk + 1][0], pk[2 * kk + 1][1], v0, v1);
          mma_bf16_16816(o[2 * dp + 1], pk[2 * kk][0], pk[2 * kk][1], pk[2 * kk + 1][0], pk[2 * kk + 1][1], v2, v3);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }

  l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
  const float ia = l_a > 0.f ? 1.f / l_a : 0.f, ib = l_b > 0.f ? 1.f / l_b : 0.f;
  if (va) {
    uint32_t* dst = reinterpret_cast<uint32_t*>(p.out + (static_cast<int64_t>(q0 + ra) * kNumQHeads + h) * kHeadDim);
#pragma unroll
    for (int dt = 0; dt < 16; ++dt) dst[dt * 4 + c] = pack_bf16x2(o[dt][0] * ia, o[dt][1] * ia);
  }
  if (vb) {
    uint32_t* dst = reinterpret_cast<uint32_t*>(p.out + (static_cast<int64_t>(q0 + rb) * kNumQHeads + h) * kHeadDim);
#pragma unroll
    for (int dt = 0; dt < 16; ++dt) dst[dt * 4 + c] = pack_bf16x2(o[dt][2] * ib, o[dt][3] * ib);
  }
}

cudaError_t prefill_init_device() {
  return cudaFuncSetAttribute(prefill_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPfSmemBytes);
}

cudaError_t launch_paged_prefill(const CUtensorMap& tmK, const CUtensorMap& tmV, const void* q, void* out,
                                 const int32_t* cu_q, const int32_t* cu_k, const int32_t* block_table, int num_seqs,
                                 int max_blocks, int num_blocks, int max_seqlen_q, int max_seqlen_k, float scale,
                                 unsigned* err, cudaStream_t stream) {
  if (num_seqs == 0 || max_seqlen_q == 0) return cudaSuccess;
  PrefillParams prm;
  prm.q = static_cast<const __nv_bfloat16*>(q);
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
  dim3 grid(kNumQHeads, num_seqs, (max_seqlen_q + kPfRows - 1) / kPfRows);
  prefill_mma_kernel<<<grid, kPfThreads, kPfSmemBytes, stream>>>(tmK, tmV, prm);
  return cudaGetLastError();
}

}  // namespace pkv
