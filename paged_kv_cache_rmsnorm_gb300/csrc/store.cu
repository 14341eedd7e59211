// K1: fused per-head q/k RMSNorm + RoPE + slot_mapping scatter.
//
// Operation ("Nano-vLLM深度解读（下）" §2 Qwen3Attention.forward and §4
// store_kvcache; rounding points per "同一个 Qwen3，两种写法" §3.5 / §3.6):
//   q[t, h]  <- rope(bf16(bf16(rms(q[t, h])) * w_q), pos[t])        (in place)
//   k_cache[slot[t], g] <- rope(bf16(bf16(rms(k[t, g])) * w_k), pos[t])
//   v_cache[slot[t], g] <- v[t, g]                                   (slot != -1)
//
// Design: HBM-bound (~24.5 KiB of traffic per token, 8 FLOP/B at most), so
// the kernel is shaped for bytes in flight, not arithmetic.  Persistent, two
// CTAs per SM; CTA c takes tokens c, c + G, c + 2G, ...  Warp 8 of a CTA is
// the producer: it reads the positions and slots of its next 32 tokens with
// one load per lane, then for each token issues bulk copies (cp.async.bulk,
// completion counted on an mbarrier) of the q row (8 KiB), the k and v rows
// (2 KiB each; skipped for slot -1) and the cos/sin row of the position
// (512 B) into a 4-stage ring in shared memory, so up to three tokens per CTA
// are in flight while one is computed.  Warps 0-7 consume: a head row is
// 128 bf16 = 256 B = 16 threads x one 16-byte vector; the 48 rows of a token
// (32 q, 8 k, 8 v) are covered in three passes of 16 rows.  The RMS reduction
// is a 4-step butterfly inside the 16-thread group, and the RoPE partner of
// element i (i + 64) lives in the thread 8 lanes away, so one xor-8 shuffle
// exchanges the halves; the arithmetic runs on fp32 pairs (f32x2 multiply /
// fma), with the sign of the rotation folded into the sin values once per
// token.  cos/sin come from a fp32 table [40960][cos 64 | sin
// 64] resident in HBM (20 MiB, L2-friendly).  q is written back in place and
// the k / v rows go to their cache slots straight from registers.  Every
// mbarrier wait is bounded; on timeout the CTA flags the error word and waits
// (bounded) for its copies in flight.
#include "common.cuh"

namespace pkv {

constexpr int kStoreCtasPerSm = 2;  // 86 registers x 288 threads; 50 KiB of shared memory each

namespace {

struct Chunk {
  uint32_t w[4];
};

__device__ __forceinline__ Chunk ld16_nc(const void* p) {
  uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
  return Chunk{{v.x, v.y, v.z, v.w}};
}
__device__ __forceinline__ void st16(void* p, const Chunk& c) {
  *reinterpret_cast<uint4*>(p) = make_uint4(c.w[0], c.w[1], c.w[2], c.w[3]);
}

__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// a bf16 pair as an fp32 pair (exact)
__device__ __forceinline__ uint64_t bf2_to_f2(uint32_t v) { return f2pack(bf16lo(v), bf16hi(v)); }
// an fp32 pair rounded to a bf16 pair
__device__ __forceinline__ uint32_t f2_to_bf2(uint64_t v) {
  float lo, hi;
  f2unpack(v, lo, hi);
  return pack_bf16x2(lo, hi);
}

// RMSNorm over the 16-thread group's 128 values, weight multiply, then the
// half-split rotation, on fp32 pairs.  w2: this thread's 8 weights as pairs;
// c2 / s2: cos and sign-folded sin of its 8 rotary indices (sin negated for
// the first half: out = x1 cos - x2 sin there, x2 cos + x1 sin in the second).
__device__ __forceinline__ Chunk norm_rope(const Chunk& x, const uint64_t (&w2)[4], const uint64_t (&c2)[4],
                                           const uint64_t (&s2)[4]) {
  uint64_t x2[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) x2[i] = bf2_to_f2(x.w[i]);
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    ss = fmaf(bf16lo(x.w[i]), bf16lo(x.w[i]), ss);
    ss = fmaf(bf16hi(x.w[i]), bf16hi(x.w[i]), ss);
  }
  ss += __shfl_xor_sync(0xffffffffu, ss, 8);
  ss += __shfl_xor_sync(0xffffffffu, ss, 4);
  ss += __shfl_xor_sync(0xffffffffu, ss, 2);
  ss += __shfl_xor_sync(0xffffffffu, ss, 1);
  const float r = rsqrtf(ss * (1.0f / kHeadDim) + PKV_RMS_EPS);
  const uint64_t r2 = f2pack(r, r);

  // normalised -> bf16, times bf16 weight -> bf16 (the product is exact in fp32)
  uint32_t y[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) y[i] = f2_to_bf2(fmul2(bf2_to_f2(f2_to_bf2(fmul2(x2[i], r2))), w2[i]));
  uint32_t other[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) other[i] = __shfl_xor_sync(0xffffffffu, y[i], 8);
  Chunk out;
#pragma unroll
  for (int i = 0; i < 4; ++i) out.w[i] = f2_to_bf2(ffma2(bf2_to_f2(y[i]), c2[i], fmul2(bf2_to_f2(other[i]), s2[i])));
  return out;
}

}  // namespace

constexpr int kStStages = 4;
constexpr int kStQ = kNumQHeads * kHeadDim * 2;    // 8 KiB: the token's q row
constexpr int kStKV = kNumKVHeads * kHeadDim * 2;  // 2 KiB: its k row, then its v row
constexpr int kStCS = kHeadDim * 4;                // 512 B: cos/sin row of its position
constexpr int kStStageBytes = kStQ + 2 * kStKV + kStCS;
constexpr int kStConsumerWarps = 8;
constexpr int kStThreads = (kStConsumerWarps + 1) * 32;
constexpr int kStBarOff = kStStages * kStStageBytes;

// ring of the per-token rows, and the position / slot of the token in each stage
struct StoreBars {
  uint64_t full[kStStages], empty[kStStages];
  int pos[kStStages], slot[kStStages];
  int timeout;
};
constexpr int kStSmemBytes = kStBarOff + 256;
static_assert(sizeof(StoreBars) <= 256, "barrier block");

__device__ __forceinline__ Chunk lds16(uint32_t a) {
  Chunk c;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(c.w[0]), "=r"(c.w[1]), "=r"(c.w[2]), "=r"(c.w[3]) : "r"(a));
  return c;
}
__device__ __forceinline__ float4 lds_f4(uint32_t a) {
  float4 f;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(f.x), "=f"(f.y), "=f"(f.z), "=f"(f.w) : "r"(a));
  return f;
}

__global__ void __launch_bounds__(kStThreads, kStoreCtasPerSm) qknorm_rope_store_kernel(
    __nv_bfloat16* __restrict__ q, int64_t q_stride, const __nv_bfloat16* __restrict__ k, int64_t k_stride,
    const __nv_bfloat16* __restrict__ v, int64_t v_stride, const int32_t* __restrict__ positions,
    const int32_t* __restrict__ slots, const __nv_bfloat16* __restrict__ wq, const __nv_bfloat16* __restrict__ wk,
    __nv_bfloat16* __restrict__ k_cache, __nv_bfloat16* __restrict__ v_cache, int64_t num_tokens,
    int64_t num_slots, const float* __restrict__ rope, unsigned* __restrict__ err) {
  extern __shared__ __align__(128) uint8_t st_smem[];
  StoreBars* bars = reinterpret_cast<StoreBars*>(st_smem + kStBarOff);
  // a kernel launched as this one's programmatic dependent (the prefill) may
  // start its set-up now; it waits for this grid before reading its output
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < kStStages; ++i) {
      mbar_init(&bars->full[i], 1);
      mbar_init(&bars->empty[i], kStConsumerWarps);
    }
    bars->timeout = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const int64_t G = gridDim.x;
  const int64_t n_mine = num_tokens > blockIdx.x ? (num_tokens - 1 - blockIdx.x) / G + 1 : 0;  // tokens blockIdx.x + i G

  if (warp == kStConsumerWarps) {
    // ---------------------------------------------------------------- producer
    bool ok = true;
    int64_t i = 0;
    for (int64_t i0 = 0; i0 < n_mine && ok; i0 += 32) {
      int pos = 0, slot = -1;
      if (i0 + lane < n_mine) {  // positions and slots of the next 32 tokens, one load each
        const int64_t t = blockIdx.x + (i0 + lane) * G;
        pos = __ldg(positions + t);
        slot = __ldg(slots + t);
      }
      const int cnt = static_cast<int>(n_mine - i0 < 32 ? n_mine - i0 : 32);
      for (int j = 0; j < cnt; ++j, ++i) {
        const int pj = __shfl_sync(0xffffffffu, pos, j), sj = __shfl_sync(0xffffffffu, slot, j);
        const int st = static_cast<int>(i % kStStages);
        if (i >= kStStages && !(ok = warp_wait_all(&bars->empty[st], ((i / kStStages) - 1) & 1))) break;
        if (lane == 0) {
          const int64_t t = blockIdx.x + (i0 + j) * G;
          bars->pos[st] = pj;
          bars->slot[st] = sj;
          const bool pos_ok = pj >= 0 && pj < kMaxPosition;
          const bool kv = pos_ok && sj >= 0 && sj < num_slots;
          const uint32_t s0 = smem_u32(st_smem + st * kStStageBytes);
          if (pos_ok) {
            mbar_arrive_expect_tx(&bars->full[st], kStQ + kStCS + (kv ? 2 * kStKV : 0));
            bulk_g2s(s0, q + t * q_stride, kStQ, &bars->full[st]);
            bulk_g2s(s0 + kStQ + 2 * kStKV, rope + static_cast<int64_t>(pj) * kHeadDim, kStCS, &bars->full[st]);
            if (kv) {
              bulk_g2s(s0 + kStQ, k + t * k_stride, kStKV, &bars->full[st]);
              bulk_g2s(s0 + kStQ + kStKV, v + t * v_stride, kStKV, &bars->full[st]);
            }
          } else {
            mbar_arrive(&bars->full[st]);  // nothing to copy: the consumers only flag the position
          }
        }
        __syncwarp();
      }
    }
    // no copy may still be landing when the CTA exits
    if (lane == 0)
      for (int64_t j = i > kStStages ? i - kStStages : 0; j < i; ++j)
        if (!mbar_wait(&bars->full[j % kStStages], (j / kStStages) & 1)) ok = false;
    if (!ok) bars->timeout = 1;
  } else {
    // ---------------------------------------------------------------- consumers
    const int sub = tid & 15;   // 16-byte chunk inside a head row
    const int row = tid >> 4;   // 0..15: head row inside a pass
    const int e0 = sub * 8;     // first element of the chunk
    const bool first = sub < 8; // chunk lies in x1 (elements 0..63)
    const int ri = e0 & 63;     // rotary index of the first element
    const Chunk wqc = ld16_nc(wq + e0);
    const Chunk wkc = ld16_nc(wk + e0);
    uint64_t wq2[4], wk2[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      wq2[j] = bf2_to_f2(wqc.w[j]);
      wk2[j] = bf2_to_f2(wkc.w[j]);
    }
    const uint64_t sgn2 = first ? f2pack(-1.0f, -1.0f) : f2pack(1.0f, 1.0f);
    bool ok = true;
    for (int64_t i = 0; i < n_mine; ++i) {
      const int st = static_cast<int>(i % kStStages);
      if (!(ok = warp_wait_all(&bars->full[st], (i / kStStages) & 1))) break;
      const int pos = bars->pos[st], slot = bars->slot[st];
      const int64_t t = blockIdx.x + i * G;
      if (!(pos >= 0 && pos < kMaxPosition)) {
        if (tid == 0) set_error(err, PKV_EFLAG_POSITION);
      } else {
        bool store = slot != -1;
        if (store && (slot < 0 || slot >= num_slots)) {
          if (tid == 0) set_error(err, PKV_EFLAG_SLOT);
          store = false;
        }
        const uint32_t s0 = smem_u32(st_smem + st * kStStageBytes);
        const Chunk x0 = lds16(s0 + row * 256 + sub * 16);
        const Chunk x1 = lds16(s0 + (16 + row) * 256 + sub * 16);
        const Chunk x2 = store ? lds16(s0 + kStQ + row * 256 + sub * 16) : Chunk{{0u, 0u, 0u, 0u}};  // k rows, then v rows
        const uint32_t ca = s0 + kStQ + 2 * kStKV + ri * 4;
        const float4 c0 = lds_f4(ca), c1 = lds_f4(ca + 16), s0v = lds_f4(ca + 256), s1v = lds_f4(ca + 272);
        const uint64_t c2[4] = {f2pack(c0.x, c0.y), f2pack(c0.z, c0.w), f2pack(c1.x, c1.y), f2pack(c1.z, c1.w)};
        const uint64_t s2[4] = {fmul2(f2pack(s0v.x, s0v.y), sgn2), fmul2(f2pack(s0v.z, s0v.w), sgn2),
                                fmul2(f2pack(s1v.x, s1v.y), sgn2), fmul2(f2pack(s1v.z, s1v.w), sgn2)};
        __nv_bfloat16* qrow = q + t * q_stride;
        st16(qrow + row * kHeadDim + e0, norm_rope(x0, wq2, c2, s2));
        st16(qrow + (16 + row) * kHeadDim + e0, norm_rope(x1, wq2, c2, s2));
        if (store) {
          const int64_t base = static_cast<int64_t>(slot) * kKVRow;
          if (row < 8) {  // warps 0-3: k heads (warp-uniform branch)
            st16(k_cache + base + row * kHeadDim + e0, norm_rope(x2, wk2, c2, s2));
          } else {  // warps 4-7: v heads, copied bit for bit
            st16(v_cache + base + (row - 8) * kHeadDim + e0, x2);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->empty[st]);
    }
    if (!ok) bars->timeout = 1;
  }
  __syncthreads();
  if (tid == 0 && bars->timeout) set_error(err, PKV_EFLAG_TIMEOUT);
}

cudaError_t store_init_device() {
  return cudaFuncSetAttribute(qknorm_rope_store_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kStSmemBytes);
}

cudaError_t launch_qknorm_rope_store(void* q, int64_t q_stride, const void* k, int64_t k_stride, const void* v,
                                     int64_t v_stride, const int32_t* positions, const int32_t* slots,
                                     const void* wq, const void* wk, void* k_cache, void* v_cache,
                                     int64_t num_tokens, int64_t num_blocks, const float* rope, int num_sms,
                                     unsigned* err, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  // persistent: two CTAs per SM, or one per token when there are fewer tokens
  const int64_t max_grid = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * kStoreCtasPerSm;
  const unsigned grid = static_cast<unsigned>(num_tokens < max_grid ? num_tokens : max_grid);
  qknorm_rope_store_kernel<<<grid, kStThreads, kStSmemBytes, stream>>>(
      static_cast<__nv_bfloat16*>(q), q_stride, static_cast<const __nv_bfloat16*>(k), k_stride,
      static_cast<const __nv_bfloat16*>(v), v_stride, positions, slots, static_cast<const __nv_bfloat16*>(wq),
      static_cast<const __nv_bfloat16*>(wk), static_cast<__nv_bfloat16*>(k_cache),
      static_cast<__nv_bfloat16*>(v_cache), num_tokens, num_blocks * kBlockSize, rope, err);
  return cudaGetLastError();
}

}  // namespace pkv
