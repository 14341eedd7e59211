// K5: the QKV projection on tcgen05 tensor cores with the step's first part
// (per-head RMSNorm, RoPE, slot_mapping scatter) as its epilogue.
//
// Operation ("同一个 Qwen3，两种写法" §3.1 fused qkv_proj; "Nano-vLLM深度解读（下）"
// §2 Qwen3Attention.forward and §4 store_kvcache):
//   y = bf16(x W^T), x [T, 4096], W [6144, 4096] = [W_q; W_k; W_v] (out, in)
//   q[t, h]  <- rope(bf16(bf16(rms(y_q)) * w_q), pos[t])          (h < 32)
//   k_cache[slot[t], g] <- rope(bf16(bf16(rms(y_k)) * w_k), pos[t]) (g < 8)
//   v_cache[slot[t], g] <- y_v                                       (slot != -1)
// The epilogue is K1's arithmetic, so the projection's output never makes a
// round trip through HBM before it is normalised, rotated and stored.
//
// Tile = 256 tokens x 2 heads (256 output features) on a pair of CTAs (a
// cluster of two on neighbouring SMs, tcgen05 cta_group::2): every MMA is
// M=256, N=256, K=16; CTA rank r holds tokens [128 r, 128 r + 128) of the
// tile (A and the accumulator rows) and features [128 r, 128 r + 128) of W
// (half of B).  K is walked 64 at a time through a 6-stage TMA ring (A box 64 x
// 128 tokens, B box 64 x 128 features, both K-major, 128-byte swizzle: 32 KiB
// per stage per CTA).  What limits this GEMM is how fast one SM receives
// tiles from L2 (about 56 B/clk, measured): a one-CTA M=128 tile needs 96 B/clk
// at the full MMA rate, the pair's halves of W bring that to 64 B/clk.
// Persistent: each pair walks the tiles (row block major, so the pairs running
// at one time share a few row blocks of x and all of W in L2); the TMA ring
// runs on across tiles and TMEM holds two 256-column accumulators, so one
// tile's epilogue overlaps the next tile's main loop.
// Warps: 0 TMA producer (both CTAs' copies count on CTA 0's full barriers),
// 1 TMEM allocation (512 columns, both CTAs) and, in CTA 0, the MMA issuer,
// whose commits signal the barriers of both CTAs (both run their loops
// converged; one elected lane issues the copies, the MMAs and the commits),
// 2..5 epilogue: thread = token row = TMEM lane; per head one 128-column
// TMEM load, bf16 rounding of the projection, then (q and k heads) the norm
// over the row's 128 values and the half-split rotation from the fp32
// cos/sin table, all in the thread's registers; rows go to global memory
// through a swizzled per-warp staging buffer as whole 256-byte rows, two
// rows per store instruction, marked evict-first for L2.
// Every mbarrier wait is bounded; on timeout the CTA flags the error word,
// CTA 0 waits (bounded) for its MMAs in flight, and both CTAs release their
// TMEM after a cluster barrier.
#include "tcgen05.cuh"

namespace pkv {

constexpr int kQkvIn = kNumQHeads * kHeadDim;                        // 4096
constexpr int kQkvOut = (kNumQHeads + 2 * kNumKVHeads) * kHeadDim;   // 6144
constexpr int kQkvRows = 128;                                        // tokens per CTA (256 per pair tile)
constexpr int kQkvCols = 256;                                        // output features per tile (2 heads)
constexpr int kQkvKStep = 64;
constexpr int kQkvStages = 6;
constexpr int kQkvABytes = kQkvRows * kQkvKStep * 2;         // 16 KiB
constexpr int kQkvBBytes = (kQkvCols / 2) * kQkvKStep * 2;   // 16 KiB: this CTA's half of the features
constexpr int kQkvStageBytes = kQkvABytes + kQkvBBytes;
constexpr int kQkvStgOff = kQkvStages * kQkvStageBytes;  // 192 KiB: epilogue staging
constexpr int kQkvStgBytes = 4 * 32 * 256;                 // 8 KiB per epilogue warp (32 rows x 256 B)
constexpr int kQkvBarOff = kQkvStgOff + kQkvStgBytes;      // 224 KiB
constexpr int kQkvSmemBytes = kQkvBarOff + 256 + 1024;
constexpr int kQkvThreads = 192;
constexpr int kQkvPairs = kQkvOut / kQkvCols;  // 24 tiles across the output features
constexpr uint32_t kQkvTmemCols = 2 * kQkvCols;  // two accumulators

struct QkvParams {
  __nv_bfloat16* q_out;
  __nv_bfloat16* k_cache;
  __nv_bfloat16* v_cache;
  const int32_t* positions;
  const int32_t* slots;
  const __nv_bfloat16* wq;
  const __nv_bfloat16* wk;
  const float* rope;
  int64_t num_tokens;
  int64_t num_slots;
  int num_tiles;
  unsigned* err;
};

struct QkvBars {
  uint64_t full[kQkvStages], empty[kQkvStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t done;
  uint32_t tmem_base;
  int timeout;
};

__device__ __forceinline__ void qkv_st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ uint4 qkv_ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
  return v;
}

// 16-byte global store with an L2 eviction-priority policy (from createpolicy)
__device__ __forceinline__ void qkv_st_global_hint(void* ptr, uint4 v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(ptr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w), "l"(policy)
               : "memory");
}

__global__ void __launch_bounds__(kQkvThreads, 1) qkv_rope_store_kernel(const __grid_constant__ CUtensorMap tmX,
                                                                        const __grid_constant__ CUtensorMap tmW,
                                                                        const QkvParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  QkvBars* bars = reinterpret_cast<QkvBars*>(smem + kQkvBarOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kSteps = kQkvIn / kQkvKStep;  // 64
  const int num_tiles = p.num_tiles;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int pair0 = static_cast<int>(blockIdx.x >> 1), npairs = static_cast<int>(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kQkvStages; ++i) {
      mbar_init(&bars->full[i], 1);
      mbar_init(&bars->empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->acc_full[b], 1);
      mbar_init(&bars->acc_empty[b], 8);  // one arrive per epilogue warp of each CTA
    }
    mbar_init(&bars->done, 1);
    bars->timeout = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tc::pair::alloc(&bars->tmem_base, kQkvTmemCols);
    tc::pair::relinquish();
  }
  tc::fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any copy or commit reaches them
  tc::fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    {
      tma_prefetch_desc(&tmX);
      tma_prefetch_desc(&tmW);
      bool ok = true;
      uint32_t g = 0;  // k-steps issued by this CTA so far, over all its tiles
      for (int tile = pair0; tile < num_tiles && ok; tile += npairs) {
        const int row0 = (tile / kQkvPairs) * 2 * kQkvRows + static_cast<int>(rank) * kQkvRows;
        const int col0 = (tile % kQkvPairs) * kQkvCols + static_cast<int>(rank) * (kQkvCols / 2);
        for (int ks = 0; ks < kSteps; ++ks, ++g) {
          const int st = g % kQkvStages;
          if (g >= kQkvStages && !(ok = warp_wait_all(&bars->empty[st], ((g / kQkvStages) - 1) & 1))) break;
          uint8_t* a = smem + st * kQkvStageBytes;
          if (tc::elect_one()) {
            if (leader) mbar_arrive_expect_tx(&bars->full[st], 2 * kQkvStageBytes);
            const uint32_t fb = cta_addr(&bars->full[st], 0);
            tma_load_2d_pair(a, &tmX, fb, ks * kQkvKStep, row0);
            tma_load_2d_pair(a + kQkvABytes, &tmW, fb, ks * kQkvKStep, col0);
          }
          __syncwarp();
        }
      }
      // Every copy lands before the CTAs exit: CTA 0's MMAs read each stage after
      // its full barrier, and both CTAs meet at a cluster barrier once those MMAs
      // have completed.
      if (!ok && lane == 0) bars->timeout = 1;
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(2 * kQkvRows, kQkvCols, false, false);
      bool ok = true;
      uint32_t g = 0;
      int i = 0;  // tiles of this pair so far
      for (int tile = pair0; leader && tile < num_tiles && ok; tile += npairs, ++i) {
        const int b = i & 1;
        // the epilogue has read this accumulator's previous tile
        if (i >= 2 && !(ok = warp_wait_all(&bars->acc_empty[b], ((i >> 1) - 1) & 1))) break;
        tc::fence_after();
        const uint32_t d = tmem + b * kQkvCols;
        for (int ks = 0; ks < kSteps; ++ks, ++g) {
          const int st = g % kQkvStages;
          if (!(ok = warp_wait_all(&bars->full[st], (g / kQkvStages) & 1))) break;
          tc::fence_after();
          const uint64_t da = tc::smem_desc_sw128(smem_u32(smem + st * kQkvStageBytes), 16, 1024);
          const uint64_t db = tc::smem_desc_sw128(smem_u32(smem + st * kQkvStageBytes + kQkvABytes), 16, 1024);
          if (tc::elect_one()) {
#pragma unroll
            for (int k = 0; k < kQkvKStep / 16; ++k) {
              const uint64_t o = static_cast<uint64_t>((k * 32) >> 4);  // K16 step inside the 128-byte row
              tc::pair::mma_ss(d, da + o, db + o, idesc, (ks > 0 || k > 0) ? 1u : 0u);
            }
            tc::pair::commit(&bars->empty[st], 0x3);
          }
          __syncwarp();
        }
        if (ok) {
          if (tc::elect_one()) tc::pair::commit(&bars->acc_full[b], 0x3);
          __syncwarp();
        }
      }
      // every MMA issued has completed before TMEM can be released
      if (leader) {
        if (tc::elect_one()) tc::pair::commit(&bars->done, 0x1);
        __syncwarp();
        if (!warp_wait_all(&bars->done, 0)) ok = false;
      }
      if (!ok && lane == 0) bars->timeout = 1;
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // token row of the tile = TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    // 8 KiB per warp (32 rows x 256 B), 16-byte chunks XOR-swizzled by row
    const uint32_t stg = smem_u32(smem + kQkvStgOff) + (warp - 2) * 8192;
    // the outputs are not read again here: they leave L2 first, so that W and
    // the x rows still to be used by other tiles stay
    const uint64_t pol_out = policy_evict_first();
    bool ok = true;
    int i = 0;
    for (int tile = pair0; tile < num_tiles; tile += npairs, ++i) {
      const int b = i & 1;
      const int pair = tile % kQkvPairs;  // heads 2*pair, 2*pair + 1 of the 48 output heads
      const int64_t t = static_cast<int64_t>(tile / kQkvPairs) * 2 * kQkvRows + static_cast<int64_t>(rank) * kQkvRows + r;
      const bool valid = t < p.num_tokens;
      int pos = 0, slot = -1;
      if (valid) {
        pos = __ldg(p.positions + t);
        slot = __ldg(p.slots + t);
      }
      const bool pos_ok = pos >= 0 && pos < kMaxPosition;
      if (valid && !pos_ok) set_error(p.err, PKV_EFLAG_POSITION);
      bool store = slot != -1;
      if (valid && pos_ok && store && (slot < 0 || slot >= p.num_slots)) {
        set_error(p.err, PKV_EFLAG_SLOT);
        store = false;
      }
      if (!(ok = warp_wait_all(&bars->acc_full[b], (i >> 1) & 1))) break;
      tc::fence_after();
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        const int head = 2 * pair + hh;  // 0..31 q, 32..39 k, 40..47 v
        const bool is_q = head < kNumQHeads, is_v = head >= kNumQHeads + kNumKVHeads;
        uint32_t acc[128];
        tc::ld128(lane_base + b * kQkvCols + hh * kHeadDim, acc);
        if (hh == 1) {  // both heads read: the MMA thread may reuse this accumulator
          tc::fence_before();
          __syncwarp();
          if (lane == 0) {
            if (leader) mbar_arrive(&bars->acc_empty[b]);
            else mbar_arrive_remote(cta_addr(&bars->acc_empty[b], 0));
          }
        }
        // the projection's output in bf16, as the linear layer returns it
        float y[128];
#pragma unroll
        for (int c = 0; c < 128; ++c) y[c] = __bfloat162float(__float2bfloat16_rn(__uint_as_float(acc[c])));
        uint32_t outw[64];
        if (is_v) {
#pragma unroll
          for (int c = 0; c < 64; ++c) outw[c] = pack_bf16x2(y[2 * c], y[2 * c + 1]);
        } else {
          const uint4* wn = reinterpret_cast<const uint4*>(is_q ? p.wq : p.wk);
          float ss = 0.f;
#pragma unroll
          for (int c = 0; c < 128; ++c) ss = fmaf(y[c], y[c], ss);
          const float rr = rsqrtf(ss * (1.0f / kHeadDim) + PKV_RMS_EPS);
#pragma unroll
          for (int c8 = 0; c8 < 16; ++c8) {  // normalised -> bf16, times the bf16 weight -> bf16
            const uint4 w8 = __ldg(wn + c8);
            const uint32_t ww[4] = {w8.x, w8.y, w8.z, w8.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int c = c8 * 8 + 2 * j;
              y[c] = __bfloat162float(__float2bfloat16_rn(__bfloat162float(__float2bfloat16_rn(y[c] * rr)) * bf16lo(ww[j])));
              y[c + 1] = __bfloat162float(
                  __float2bfloat16_rn(__bfloat162float(__float2bfloat16_rn(y[c + 1] * rr)) * bf16hi(ww[j])));
            }
          }
          const float* cs = p.rope + static_cast<int64_t>(pos_ok ? pos : 0) * kHeadDim;  // [cos 64 | sin 64]
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            const float2 cc = __ldg(reinterpret_cast<const float2*>(cs + c));
            const float2 sn = __ldg(reinterpret_cast<const float2*>(cs + 64 + c));
            const float a0 = fmaf(y[c], cc.x, -(y[c + 64] * sn.x));
            const float a1 = fmaf(y[c + 1], cc.y, -(y[c + 65] * sn.y));
            const float b0 = fmaf(y[c + 64], cc.x, y[c] * sn.x);
            const float b1 = fmaf(y[c + 65], cc.y, y[c + 1] * sn.y);
            outw[c / 2] = pack_bf16x2(a0, a1);
            outw[32 + c / 2] = pack_bf16x2(b0, b1);
          }
        }
        // one row of 256 B per thread into the staging buffer, then out as
        // whole rows: lanes 0-15 and 16-31 each store one row per instruction
#pragma unroll
        for (int c = 0; c < 16; ++c)
          qkv_st_shared_v4(stg + lane * 256 + ((c ^ (lane & 15)) * 16), outw[4 * c], outw[4 * c + 1], outw[4 * c + 2],
                           outw[4 * c + 3]);
        __syncwarp();
        const uint32_t wmask = __ballot_sync(0xffffffffu, valid && pos_ok && (is_q || store));
        int64_t dst_row = -1;  // this lane's destination row (element offset), or -1
        if (valid && pos_ok) {
          if (is_q) dst_row = (t * kNumQHeads + head) * kHeadDim;
          else if (store) dst_row = (static_cast<int64_t>(slot) * kNumKVHeads + (head - kNumQHeads) % kNumKVHeads) * kHeadDim;
        }
        __nv_bfloat16* const base = is_q ? p.q_out : (is_v ? p.v_cache : p.k_cache);
        const int half = lane >> 4, chunk = lane & 15;
#pragma unroll 4
        for (int rr2 = 0; rr2 < 32; rr2 += 2) {
          const int row = rr2 + half;  // row of this warp's 32
          const int64_t drow = __shfl_sync(0xffffffffu, dst_row, row);
          const uint4 v = qkv_ld_shared_v4(stg + row * 256 + ((chunk ^ (row & 15)) * 16));
          if ((wmask >> row) & 1u) qkv_st_global_hint(base + drow + chunk * 8, v, pol_out);
        }
        __syncwarp();
      }
    }
    if (!ok) bars->timeout = 1;
  }

  tc::fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while CTA 0's MMAs may still use its shared memory or TMEM
  if (threadIdx.x == 0 && bars->timeout) set_error(p.err, PKV_EFLAG_TIMEOUT);
  if (warp == 1) {
    tc::fence_after();
    tc::pair::dealloc(tmem, kQkvTmemCols);
  }
}

namespace {
cudaLaunchConfig_t qkv_config(unsigned grid, cudaStream_t stream, cudaLaunchAttribute* at) {
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kQkvThreads);
  cfg.dynamicSmemBytes = kQkvSmemBytes;
  cfg.stream = stream;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cfg;
}
int g_qkv_pairs = 0;  // CTA pairs of the kernel resident at once on this device type
}  // namespace

cudaError_t qkv_init_device() {
  cudaError_t e = cudaFuncSetAttribute(qkv_rope_store_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kQkvSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute at[1];
  const cudaLaunchConfig_t cfg = qkv_config(2, nullptr, at);
  int n = 0;
  if ((e = cudaOccupancyMaxActiveClusters(&n, qkv_rope_store_kernel, &cfg)) != cudaSuccess) return e;
  if (n < 1) return cudaErrorInvalidConfiguration;  // no pair of SMs can host the kernel
  g_qkv_pairs = n;
  return cudaSuccess;
}

cudaError_t launch_qkv_rope_store(const CUtensorMap& tmX, const CUtensorMap& tmW, void* q_out, void* k_cache,
                                  void* v_cache, const int32_t* positions, const int32_t* slots, const void* wq,
                                  const void* wk, const float* rope, int64_t num_tokens, int64_t num_blocks,
                                  int num_sms, unsigned* err, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  QkvParams prm;
  prm.q_out = static_cast<__nv_bfloat16*>(q_out);
  prm.k_cache = static_cast<__nv_bfloat16*>(k_cache);
  prm.v_cache = static_cast<__nv_bfloat16*>(v_cache);
  prm.positions = positions;
  prm.slots = slots;
  prm.wq = static_cast<const __nv_bfloat16*>(wq);
  prm.wk = static_cast<const __nv_bfloat16*>(wk);
  prm.rope = rope;
  prm.num_tokens = num_tokens;
  prm.num_slots = num_blocks * kBlockSize;
  prm.err = err;
  const int64_t tiles = (num_tokens + 2 * kQkvRows - 1) / (2 * kQkvRows) * kQkvPairs;
  prm.num_tiles = static_cast<int>(tiles);
  const int64_t pairs = tiles < g_qkv_pairs ? tiles : g_qkv_pairs;
  (void)num_sms;
  cudaLaunchAttribute at[1];
  const cudaLaunchConfig_t cfg = qkv_config(static_cast<unsigned>(2 * pairs), stream, at);
  return cudaLaunchKernelEx(&cfg, qkv_rope_store_kernel, tmX, tmW, prm);
}

}  // namespace pkv
