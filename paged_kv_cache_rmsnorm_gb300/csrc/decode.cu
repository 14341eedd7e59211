// K2: split-K paged GQA decode attention.
//
// Operation ("Nano-vLLM深度解读（下）" §4, decode branch; "同一个 Qwen3，两种写法"
// §3.3-§3.4): for sequence b, query head h (KV head g = h / 4) and context L,
//   out[b, h] = softmax_j(scale * q[b, h] . K[j, g]) V[j, g],  j < L,
// with row j of the sequence at cache row block_table[b, j / 256] * 256 + j % 256.
//
// Design (HBM-bound: every KV byte of the batch is read once per step):
//  * CTA = (split, KV head g, sequence b).  A split is a run of `chunk` keys
//    (a multiple of 64); the host sizes `chunk` from the device's SM count so
//    that one long sequence still fills the GPU: a single resident wave of
//    CTAs while there are at most two (sequence, KV head) pairs per SM (304
//    on a GB300), otherwise about four CTAs per SM.
//  * A producer warp streams 64-key tiles of K and V for head g through a
//    3-stage TMA ring (cp.async.bulk.tensor, 128-byte swizzle, evict-first L2
//    policy; each tile lies inside one 256-token block, so one table lookup
//    per tile).  Each K/V byte is read once for all 4 query heads of the group.
//  * 4 consumer warps each take 16 keys of every tile: S = Q K^T and O += P V
//    on mma.sync m16n8k16 (the 4 query heads padded to 16 rows), with an
//    online softmax in the exp2 domain.  Keys >= L are selected away in S and
//    zeroed in the V fragments, so unwritten cache rows (NaN) never leak.
//  * Launched as a programmatic dependent of the store that precedes it:
//    the context length, the first block id and the barrier set-up overlap
//    the store's tail; griddepcontrol.wait comes before any read of q or of
//    the cache, which the store writes.
//  * The 4 warps' (m, l, O) are merged in shared memory.  With one split the
//    CTA writes bf16 output directly; otherwise it writes an fp32 partial, and
//    the last CTA of (b, g) to arrive (atomic ticket, no spin-wait) merges the
//    partials by log-sum-exp and resets the ticket to zero.  It first copies
//    them into the drained ring with two bulk copies (the plan never makes
//    more splits than fit), so the merge waits out one L2 round trip instead
//    of one per eight splits.
#include <atomic>

#include "common.cuh"

namespace pkv {

constexpr int kDecTile = 64;
constexpr int kDecStages = 3;
constexpr int kDecConsumerWarps = 4;
constexpr int kDecThreads = (kDecConsumerWarps + 1) * 32;
constexpr int kDecSubBytes = kDecTile * 64 * 2;  // 64 keys x 64 dims x bf16 = 8 KiB
constexpr int kDecStageBytes = 4 * kDecSubBytes;  // K lo, K hi, V lo, V hi
constexpr int kDecSmemBytes = kDecStages * kDecStageBytes + 1024 /* align */ + 256 /* barriers */;
// the split-K merge copies a (sequence, KV head)'s partials into the drained
// ring: 2 KiB of O, 32 B of (m, l) and 16 B of merge weights per split
constexpr int kDecMergeSmemSplits = kDecStages * kDecStageBytes / (kGroup * kHeadDim * 4 + kGroup * 2 * 4 + kGroup * 4);

struct DecodeParams {
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  const int32_t* context_lens;
  const int32_t* block_table;
  int32_t max_blocks;
  int32_t num_blocks;
  int32_t max_context;
  int32_t chunk;
  int32_t num_splits;
  float scale_log2;
  float* ws_o;        // [B*8][splits][4][128]
  float* ws_ml;       // [B*8][splits][4][2]
  unsigned* ws_cnt;   // [B*8]
  unsigned* err;
};

__global__ void __launch_bounds__(kDecThreads, 2) paged_decode_kernel(const __grid_constant__ CUtensorMap tmK,
                                                                   const __grid_constant__ CUtensorMap tmV,
                                                                   const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kDecStages * kDecStageBytes);
  uint64_t* empty = full + kDecStages;
  int* tile_bad = reinterpret_cast<int*>(empty + kDecStages);  // [kDecStages]
  int* s_flag = tile_bad + kDecStages;
  int* s_timeout = s_flag + 1;  // any wait of the CTA gave up

  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bg = b * kNumKVHeads + g;

  const int32_t* row = p.block_table + static_cast<int64_t>(b) * p.max_blocks;
  // the first tile's block id and the context length, loaded together (the
  // store writes neither; split * chunk < max_context <= max_blocks * 256
  // whenever the CTA has work, so the entry is inside the table row)
  int blk_next = warp == kDecConsumerWarps && lane == 0 && split * p.chunk < p.max_blocks * kBlockSize
                     ? __ldg(row + split * p.chunk / kBlockSize)
                     : 0;
  int L = __ldg(p.context_lens + b);
  if (L < 0 || L > p.max_blocks * kBlockSize || L > p.max_context) {
    if (threadIdx.x == 0 && split == 0 && g == 0) set_error(p.err, PKV_EFLAG_CONTEXT);
    L = 0;
  }
  if (L == 0) {  // empty context: the output row is zero
    asm volatile("griddepcontrol.wait;" ::: "memory");  // out may be read by the previous kernel
    if (split == 0 && threadIdx.x < 128) {
      const int hh = threadIdx.x >> 5, d = (threadIdx.x & 31) * 4;
      __nv_bfloat16* o = p.out + (static_cast<int64_t>(b) * kNumQHeads + g * kGroup + hh) * kHeadDim + d;
      *reinterpret_cast<uint2*>(o) = make_uint2(0u, 0u);
    }
    return;
  }
  const int k_begin = split * p.chunk;
  if (k_begin >= L) return;  // no keys for this split (uniform over the CTA)
  const int k_end = min(L, k_begin + p.chunk);
  const int n_tiles = (k_end - k_begin + kDecTile - 1) / kDecTile;
  const int active = (L + p.chunk - 1) / p.chunk;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kDecStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kDecConsumerWarps);
    }
    *s_timeout = 0;
    fence_barrier_init();
  }
  __syncthreads();
  // from here on the kernel reads what the previous kernel (the store) wrote: q and the cache
  asm volatile("griddepcontrol.wait;" ::: "memory");

  bool timed_out = false;
  int n_sent = 0;  // producer lane: tiles whose stage was filled (TMA) or marked bad
  if (warp == kDecConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const uint64_t pol = policy_evict_first();
      for (int i = 0; i < n_tiles; ++i) {
        const int st = i % kDecStages;
        const int key0 = k_begin + i * kDecTile;
        // this tile's block id was loaded one tile ahead; load the next one now
        const int blk = blk_next;
        if (i + 1 < n_tiles) blk_next = __ldg(row + (key0 + kDecTile) / kBlockSize);
        if (i >= kDecStages && !mbar_wait(&empty[st], ((i / kDecStages) - 1) & 1)) {
          timed_out = true;
          break;
        }
        uint8_t* dst = smem + st * kDecStageBytes;
        if (blk < 0 || blk >= p.num_blocks) {
          set_error(p.err, PKV_EFLAG_BLOCK_ID);
          tile_bad[st] = 1;
          mbar_arrive(&full[st]);
          n_sent = i + 1;
          continue;
        }
        tile_bad[st] = 0;
        const int slot0 = blk * kBlockSize + (key0 % kBlockSize);
        mbar_arrive_expect_tx(&full[st], kDecStageBytes);
        tma_load_3d_hint(dst, &tmK, &full[st], 0, g, slot0, pol);
        tma_load_3d_hint(dst + kDecSubBytes, &tmK, &full[st], 64, g, slot0, pol);
        tma_load_3d_hint(dst + 2 * kDecSubBytes, &tmV, &full[st], 0, g, slot0, pol);
        tma_load_3d_hint(dst + 3 * kDecSubBytes, &tmV, &full[st], 64, g, slot0, pol);
        n_sent = i + 1;
      }
    }
    __syncwarp();
  }

  // merge scratch aliases the stage ring once the pipeline has drained
  float* mrg_o = reinterpret_cast<float*>(smem);              // [4 warps][4 heads][128]
  float* mrg_ml = mrg_o + kDecConsumerWarps * kGroup * kHeadDim;  // [4 warps][4 heads][2]

  if (warp < kDecConsumerWarps) {
    // ------------------------------------------------------------ consumers
    const int hr = lane >> 2;  // fragment row: query head of the group for lanes < 16
    const int c = lane & 3;
    const bool real = lane < 16;
    // Q as the A operand (rows 0..3 real, 4..15 zero), kept in registers
    uint32_t qa[8][2];
    {
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
          p.q + (static_cast<int64_t>(b) * kNumQHeads + g * kGroup + (hr & 3)) * kHeadDim);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        qa[ks][0] = real ? __ldg(qrow + ks * 8 + c) : 0u;
        qa[ks][1] = real ? __ldg(qrow + ks * 8 + 4 + c) : 0u;
      }
    }
    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m = -INFINITY, l = 0.f;

    const int wkey = warp * 16;  // this warp's 16 keys inside each tile
    for (int i = 0; i < n_tiles; ++i) {
      const int st = i % kDecStages;
      // one verdict for the whole warp: ldmatrix, mma.sync and the shuffles below are warp-collective
      if (!warp_wait_all(&full[st], (i / kDecStages) & 1)) {
        timed_out = true;
        break;
      }
      const int base = k_begin + i * kDecTile + wkey;
      const int nvalid = tile_bad[st] ? 0 : min(16, k_end - base);
      if (nvalid > 0) {
        const uint32_t kst = smem_u32(smem + st * kDecStageBytes);
        const uint32_t vst = kst + 2 * kDecSubBytes;
        float s[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
        {
          const int mi = lane >> 3;                       // which 8x8 matrix this lane addresses
          const int r = wkey + (mi >> 1) * 8 + (lane & 7);  // key row inside the tile
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t addr = kst + (ks >> 2) * kDecSubBytes + sw128(r, (ks & 3) * 2 + (mi & 1));
            uint32_t b0, b1, b2, b3;
            ldsm_x4(addr, b0, b1, b2, b3);
            mma_bf16_16816(s[0], qa[ks][0], 0u, qa[ks][1], 0u, b0, b1);
            mma_bf16_16816(s[1], qa[ks][0], 0u, qa[ks][1], 0u, b2, b3);
          }
        }
        // scale, mask keys >= L, online softmax (row = query head hr)
        float t[2][2];
        float mx = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int kk = nt * 8 + 2 * c + j;
            t[nt][j] = kk < nvalid ? s[nt][j] * p.scale_log2 : -INFINITY;
            mx = fmaxf(mx, t[nt][j]);
          }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m, mx);
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = fast_exp2(m - m_use);
        float pr[2][2];
        float psum = 0.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            pr[nt][j] = fast_exp2(t[nt][j] - m_use);
            psum += pr[nt][j];
          }
        l = l * alpha + psum;
        m = m_new;
#pragma unroll
        for (int dt = 0; dt < 16; ++dt) {
          o[dt][0] *= alpha;
          o[dt][1] *= alpha;
        }
        const uint32_t pa0 = real ? pack_bf16x2(pr[0][0], pr[0][1]) : 0u;
        const uint32_t pa2 = real ? pack_bf16x2(pr[1][0], pr[1][1]) : 0u;
        // V fragments (transposed load); zero the values of keys >= nvalid
        const int mi = lane >> 3;
        const int r = wkey + (mi & 1) * 8 + (lane & 7);
        const bool tail = nvalid < 16;
        const uint32_t lo_keep0 = (2 * c < nvalid ? 0x0000FFFFu : 0u) | (2 * c + 1 < nvalid ? 0xFFFF0000u : 0u);
        const uint32_t hi_keep0 =
            (8 + 2 * c < nvalid ? 0x0000FFFFu : 0u) | (8 + 2 * c + 1 < nvalid ? 0xFFFF0000u : 0u);
#pragma unroll
        for (int dp = 0; dp < 8; ++dp) {
          const int d0 = dp * 16 + (mi >> 1) * 8;
          const uint32_t addr = vst + (d0 >> 6) * kDecSubBytes + sw128(r, (d0 & 63) >> 3);
          uint32_t v0, v1, v2, v3;
          ldsm_x4_t(addr, v0, v1, v2, v3);
          if (tail) {
            v0 &= lo_keep0;
            v1 &= hi_keep0;
            v2 &= lo_keep0;
            v3 &= hi_keep0;
          }
          mma_bf16_16816(o[2 * dp], pa0, 0u, pa2, 0u, v0, v1);
          mma_bf16_16816(o[2 * dp + 1], pa0, 0u, pa2, 0u, v2, v3);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    if (timed_out && lane == 0) *s_timeout = 1;  // timed_out is warp-uniform here
    // every warp is past the ring; after a timeout loads may still be in
    // flight into it, so it is then neither reused nor read
    asm volatile("bar.sync 1, 160;" ::: "memory");
    if (*s_timeout == 0 && real) {
      float* dst = mrg_o + (warp * kGroup + hr) * kHeadDim;
#pragma unroll
      for (int dt = 0; dt < 16; ++dt) {
        dst[dt * 8 + 2 * c] = o[dt][0];
        dst[dt * 8 + 2 * c + 1] = o[dt][1];
      }
      if (c == 0) {
        mrg_ml[(warp * kGroup + hr) * 2] = m;
        mrg_ml[(warp * kGroup + hr) * 2 + 1] = l;
      }
    }
  } else {
    if (timed_out && lane == 0) *s_timeout = 1;
    asm volatile("bar.sync 1, 160;" ::: "memory");
    if (*s_timeout != 0 && lane == 0) {
      // the producer waits (bounded) for the loads it issued before the CTA leaves
      set_error(p.err, PKV_EFLAG_TIMEOUT);
      // only the last kDecStages tiles sent can still be in flight
      for (int i = max(0, n_sent - kDecStages); i < n_sent; ++i) mbar_wait(&full[i % kDecStages], (i / kDecStages) & 1);
    }
  }
  __syncthreads();
  const bool bad = *s_timeout != 0;

  // ---------------------------------------------------------------- combine the 4 warps
  const int hh = (threadIdx.x >> 5) & 3, d = (threadIdx.x & 31) * 4;
  float M = -INFINITY, Lsum = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
  if (threadIdx.x < 128 && !bad) {
#pragma unroll
    for (int w = 0; w < kDecConsumerWarps; ++w) M = fmaxf(M, mrg_ml[(w * kGroup + hh) * 2]);
    const float Mu = M == -INFINITY ? 0.f : M;
#pragma unroll
    for (int w = 0; w < kDecConsumerWarps; ++w) {
      const float f = fast_exp2(mrg_ml[(w * kGroup + hh) * 2] - Mu);
      Lsum += f * mrg_ml[(w * kGroup + hh) * 2 + 1];
      const float4 ov = *reinterpret_cast<const float4*>(mrg_o + (w * kGroup + hh) * kHeadDim + d);
      acc[0] += f * ov.x;
      acc[1] += f * ov.y;
      acc[2] += f * ov.z;
      acc[3] += f * ov.w;
    }
  }
  __nv_bfloat16* out_row = p.out + (static_cast<int64_t>(b) * kNumQHeads + g * kGroup + hh) * kHeadDim + d;
  if (active == 1) {
    if (threadIdx.x < 128) {
      const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
      *reinterpret_cast<uint2*>(out_row) =
          make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv), pack_bf16x2(acc[2] * inv, acc[3] * inv));
    }
    return;
  }

  // ---------------------------------------------------------------- split-K partial + last-CTA merge
  const int64_t part = (static_cast<int64_t>(bg) * p.num_splits + split) * kGroup + hh;
  if (threadIdx.x < 128 && !bad) {
    *reinterpret_cast<float4*>(p.ws_o + part * kHeadDim + d) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    if ((threadIdx.x & 31) == 0) *reinterpret_cast<float2*>(p.ws_ml + part * 2) = make_float2(M, Lsum);
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned ticket = atomicAdd(p.ws_cnt + bg, 1u);
    *s_flag = ticket == static_cast<unsigned>(active - 1);
  }
  __syncthreads();
  if (!*s_flag) return;
  __threadfence();
  if (bad) {
    // this CTA's ring may still be receiving loads: no merge, the row is flagged
  } else if (active <= kDecMergeSmemSplits) {
    // The partials of this (sequence, KV head) are contiguous in the workspace.
    // Bulk copies bring them into the drained ring: the (m, l) pairs first, on
    // a barrier of their own, then O in two halves on two more, so the merge
    // weights are ready and the first half is being summed while the second
    // is still landing.  (Reading the partials straight from L2, eight splits
    // at a time, took 8-13 us for 72 splits.)  Warp h merges query head h in
    // split order, so the result does not depend on which CTA came last.
    uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + kDecStages * kDecStageBytes + 128);  // [3]
    float* so = reinterpret_cast<float*>(smem);                           // [active][4][128]
    float* sml = so + static_cast<int64_t>(active) * kGroup * kHeadDim;   // [active][4][2]
    float* sw = sml + active * kGroup * 2;                                // [4][active] merge weights
    const int h1 = active / 2;                                             // splits in the first O half
    if (threadIdx.x == 0) {
      for (int i = 0; i < 3; ++i) mbar_init(&mbar[i], 1);
      fence_barrier_init();
      asm volatile("fence.proxy.async.global;" ::: "memory");  // other CTAs' partials, read by the async proxy
      const float* src_o = p.ws_o + static_cast<int64_t>(bg) * p.num_splits * kGroup * kHeadDim;
      const uint32_t mb = static_cast<uint32_t>(active) * kGroup * 2 * 4;
      const uint32_t ob1 = static_cast<uint32_t>(h1) * kGroup * kHeadDim * 4;
      const uint32_t ob2 = static_cast<uint32_t>(active - h1) * kGroup * kHeadDim * 4;
      mbar_arrive_expect_tx(&mbar[0], mb);
      bulk_g2s(smem_u32(sml), p.ws_ml + static_cast<int64_t>(bg) * p.num_splits * kGroup * 2, mb, &mbar[0]);
      mbar_arrive_expect_tx(&mbar[1], ob1);
      bulk_g2s(smem_u32(so), src_o, ob1, &mbar[1]);
      mbar_arrive_expect_tx(&mbar[2], ob2);
      bulk_g2s(smem_u32(so + h1 * kGroup * kHeadDim), src_o + static_cast<int64_t>(h1) * kGroup * kHeadDim, ob2,
               &mbar[2]);
    }
    __syncthreads();
    bool landed = true;
    if (threadIdx.x < 128) {
      // the head's global max and row sum, lanes over splits; each lane keeps the weights of its splits
      landed = warp_wait_all(&mbar[0], 0);
      float Mg = -INFINITY;
      for (int sp = lane; sp < active; sp += 32) Mg = fmaxf(Mg, sml[(sp * kGroup + hh) * 2]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) Mg = fmaxf(Mg, __shfl_xor_sync(0xffffffffu, Mg, o));
      const float Mu = Mg == -INFINITY ? 0.f : Mg;
      float Lg = 0.f;
      for (int sp = lane; sp < active; sp += 32) {
        const float2 ml = *reinterpret_cast<const float2*>(sml + (sp * kGroup + hh) * 2);
        const float f = fast_exp2(ml.x - Mu);
        sw[hh * active + sp] = f;
        Lg += f * ml.y;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) Lg += __shfl_xor_sync(0xffffffffu, Lg, o);
      __syncwarp();
      float a[4] = {0.f, 0.f, 0.f, 0.f};
      landed = warp_wait_all(&mbar[1], 0) && landed;
      for (int sp = 0; sp < h1; ++sp) {
        const float f = sw[hh * active + sp];
        const float4 ov = *reinterpret_cast<const float4*>(so + (sp * kGroup + hh) * kHeadDim + d);
        a[0] += f * ov.x;
        a[1] += f * ov.y;
        a[2] += f * ov.z;
        a[3] += f * ov.w;
      }
      landed = warp_wait_all(&mbar[2], 0) && landed;
      for (int sp = h1; sp < active; ++sp) {
        const float f = sw[hh * active + sp];
        const float4 ov = *reinterpret_cast<const float4*>(so + (sp * kGroup + hh) * kHeadDim + d);
        a[0] += f * ov.x;
        a[1] += f * ov.y;
        a[2] += f * ov.z;
        a[3] += f * ov.w;
      }
      const float inv = Lg > 0.f ? 1.f / Lg : 0.f;
      if (landed)
        *reinterpret_cast<uint2*>(out_row) =
            make_uint2(pack_bf16x2(a[0] * inv, a[1] * inv), pack_bf16x2(a[2] * inv, a[3] * inv));
    }
    landed = __syncthreads_and(landed);
    if (threadIdx.x == 0 && !landed) set_error(p.err, PKV_EFLAG_TIMEOUT);
  } else if (threadIdx.x == 0) {
    set_error(p.err, PKV_EFLAG_TIMEOUT);  // unreachable: the host never plans more splits than fit (see decode_plan)
  }
  if (threadIdx.x == 0) p.ws_cnt[bg] = 0u;  // leave the ticket ready for the next call
}

// ---------------------------------------------------------------- host side
struct DecodePlan {
  int chunk;
  int splits;
};

// SM count of the current device (152 on a GB300), cached per device; 152
// when no device can be queried (host-only use of the size query).
static int plan_sms() {
  constexpr int kMaxDev = 64;
  static std::atomic<int> cache[kMaxDev];
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
    cudaGetLastError();
    return 152;
  }
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = 152;
    }
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// Keys per split, for a device of `sms` SMs (two decode CTAs fit on an SM).
// Up to 2 * sms (sequence, KV head) pairs: as many splits as fill one
// resident wave, so every CTA streams from start to end and no partial last
// wave runs at a fraction of the bandwidth (38 partials at most on 152 SMs).
// More pairs: enough CTAs to cover the SMs about four times.  Never fewer
// than 512 keys per split: each split pays for a Q load and a merge; never
// more splits than the shared-memory merge holds.
static DecodePlan decode_plan(int batch, int max_context, int sms) {
  DecodePlan pl{kDecTile, 1};
  if (max_context <= 0 || batch <= 0) return pl;
  const int64_t resident = 2 * static_cast<int64_t>(sms);
  const int64_t tiles = (max_context + kDecTile - 1) / kDecTile;
  const int64_t heads = static_cast<int64_t>(batch) * kNumKVHeads;
  int64_t per;
  if (heads <= resident) {
    int64_t splits = resident / heads;
    if (splits > kDecMergeSmemSplits) splits = kDecMergeSmemSplits;
    per = (tiles + splits - 1) / splits;
  } else {
    const int64_t target = 4 * static_cast<int64_t>(sms);
    per = (heads * tiles + target - 1) / target;
  }
  if (per < 8) per = 8;
  if (per > tiles) per = tiles;
  while ((tiles + per - 1) / per > kDecMergeSmemSplits) ++per;
  pl.chunk = static_cast<int>(per * kDecTile);
  pl.splits = static_cast<int>((tiles + per - 1) / per);
  return pl;
}

// Workspace layout: [ticket counters for 65535 x 8 (b, g) pairs | m, l partials | O partials].
// The counters sit at a fixed offset so that calls with different split plans
// never read another call's partials as counters; the last CTA of every
// (b, g) returns its counter to zero, so a zero-filled workspace stays valid.
constexpr size_t kDecCounterBytes = static_cast<size_t>(65535) * kNumKVHeads * sizeof(unsigned);
static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t decode_workspace_bytes(int batch, int max_context) {
  const DecodePlan pl = decode_plan(batch, max_context, plan_sms());
  if (pl.splits <= 1) return 0;
  const size_t bg = static_cast<size_t>(batch) * kNumKVHeads;
  const size_t ml = bg * pl.splits * kGroup * 2 * sizeof(float);
  const size_t o = bg * pl.splits * kGroup * kHeadDim * sizeof(float);
  return align256(kDecCounterBytes) + align256(ml) + align256(o);
}

int decode_num_splits(int batch, int max_context) { return decode_plan(batch, max_context, plan_sms()).splits; }

cudaError_t decode_init_device() {
  return cudaFuncSetAttribute(paged_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecSmemBytes);
}

cudaError_t launch_paged_decode(const CUtensorMap& tmK, const CUtensorMap& tmV, const void* q, void* out,
                                const int32_t* context_lens, const int32_t* block_table, int batch, int max_blocks,
                                int num_blocks, int max_context, float scale, void* workspace, unsigned* err,
                                cudaStream_t stream, bool programmatic) {
  const DecodePlan pl = decode_plan(batch, max_context, plan_sms());
  DecodeParams prm;
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.context_lens = context_lens;
  prm.block_table = block_table;
  prm.max_blocks = max_blocks;
  prm.num_blocks = num_blocks;
  prm.max_context = max_context;
  prm.chunk = pl.chunk;
  prm.num_splits = pl.splits;
  prm.scale_log2 = scale * kLog2e;
  prm.err = err;
  prm.ws_o = nullptr;
  prm.ws_ml = nullptr;
  prm.ws_cnt = nullptr;
  if (pl.splits > 1) {
    const size_t bg = static_cast<size_t>(batch) * kNumKVHeads;
    const size_t ml = bg * pl.splits * kGroup * 2 * sizeof(float);
    uint8_t* w = static_cast<uint8_t*>(workspace);
    prm.ws_cnt = reinterpret_cast<unsigned*>(w);
    prm.ws_ml = reinterpret_cast<float*>(w + align256(kDecCounterBytes));
    prm.ws_o = reinterpret_cast<float*>(w + align256(kDecCounterBytes) + align256(ml));
  }
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = programmatic ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.splits, kNumKVHeads, batch);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = kDecSmemBytes;
  cfg.stream = stream;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, paged_decode_kernel, tmK, tmV, prm);
}

}  // namespace pkv
