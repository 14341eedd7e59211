// K1: fused per-head q/k RMSNorm + RoPE + slot_mapping scatter.
//
// Operation ("Nano-vLLM深度解读（下）" §2 Qwen3Attention.forward and §4
// store_kvcache; rounding points per "同一个 Qwen3，两种写法" §3.5 / §3.6):
//   q[t, h]  <- rope(bf16(bf16(rms(q[t, h])) * w_q), pos[t])        (in place)
//   k_cache[slot[t], g] <- rope(bf16(bf16(rms(k[t, g])) * w_k), pos[t])
//   v_cache[slot[t], g] <- v[t, g]                                   (slot != -1)
//
// Design: HBM-bound (~24.5 KiB of traffic per token, 8 FLOP/B at most), so
// the kernel is shaped for bytes in flight, not arithmetic.  A CTA of 256
// threads handles one token at a time and walks the tokens persistently (three
// CTAs per SM).  A head row is 128 bf16 = 256 B = 16 threads x one 16-byte
// vector; the 48 rows of a token (32 q, 8 k, 8 v) are covered in three passes
// of 16 rows.  The position and slot of the next token are loaded one
// iteration ahead, so the three 16-byte row loads and the cos/sin row of a
// token are all in flight together: one memory round trip per token.
// The RMS reduction is a 4-step butterfly inside the 16-thread group, and the
// RoPE partner of element i (i + 64) lives in the thread 8 lanes away, so one
// xor-8 shuffle exchanges the halves.  cos/sin come from a fp32 table
// [40960][cos 64 | sin 64] resident in HBM (20 MiB, L2-friendly).
#include "common.cuh"

namespace pkv {

constexpr int kStoreCtasPerSm = 3;  // 80 registers per thread: three CTAs of 256 threads per SM

namespace {

struct Chunk {
  uint32_t w[4];
};

__device__ __forceinline__ Chunk ld16(const void* p) {
  uint4 v = *reinterpret_cast<const uint4*>(p);
  return Chunk{{v.x, v.y, v.z, v.w}};
}
__device__ __forceinline__ Chunk ld16_nc(const void* p) {
  uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
  return Chunk{{v.x, v.y, v.z, v.w}};
}
__device__ __forceinline__ void st16(void* p, const Chunk& c) {
  *reinterpret_cast<uint4*>(p) = make_uint4(c.w[0], c.w[1], c.w[2], c.w[3]);
}

// RMSNorm over the 16-thread group's 128 values, weight multiply, then the
// half-split rotation.  cs[0..7] = cos, cs[8..15] = sin of this thread's 8
// rotary indices; `first` = this thread holds x1 (elements < 64).
__device__ __forceinline__ Chunk norm_rope(const Chunk& x, const Chunk& w, const float (&cs)[16], bool first) {
  float xf[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    xf[2 * i] = bf16lo(x.w[i]);
    xf[2 * i + 1] = bf16hi(x.w[i]);
  }
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) ss = fmaf(xf[i], xf[i], ss);
  ss += __shfl_xor_sync(0xffffffffu, ss, 8);
  ss += __shfl_xor_sync(0xffffffffu, ss, 4);
  ss += __shfl_xor_sync(0xffffffffu, ss, 2);
  ss += __shfl_xor_sync(0xffffffffu, ss, 1);
  const float r = rsqrtf(ss * (1.0f / kHeadDim) + PKV_RMS_EPS);

  // normalised -> bf16, times bf16 weight -> bf16 (the product is exact in fp32)
  uint32_t y[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float n0 = __bfloat162float(__float2bfloat16_rn(xf[2 * i] * r));
    const float n1 = __bfloat162float(__float2bfloat16_rn(xf[2 * i + 1] * r));
    y[i] = pack_bf16x2(n0 * bf16lo(w.w[i]), n1 * bf16hi(w.w[i]));
  }
  uint32_t other[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) other[i] = __shfl_xor_sync(0xffffffffu, y[i], 8);

  // first half:  out = x1 cos - x2 sin ; second half: out = x2 cos + x1 sin
  const float sgn = first ? -1.0f : 1.0f;
  Chunk out;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float a0 = bf16lo(y[i]), a1 = bf16hi(y[i]);
    const float b0 = bf16lo(other[i]), b1 = bf16hi(other[i]);
    const float o0 = fmaf(a0, cs[2 * i], sgn * (b0 * cs[8 + 2 * i]));
    const float o1 = fmaf(a1, cs[2 * i + 1], sgn * (b1 * cs[8 + 2 * i + 1]));
    out.w[i] = pack_bf16x2(o0, o1);
  }
  return out;
}

}  // namespace

__global__ void __launch_bounds__(256, kStoreCtasPerSm) qknorm_rope_store_kernel(
    __nv_bfloat16* __restrict__ q, int64_t q_stride, const __nv_bfloat16* __restrict__ k, int64_t k_stride,
    const __nv_bfloat16* __restrict__ v, int64_t v_stride, const int32_t* __restrict__ positions,
    const int32_t* __restrict__ slots, const __nv_bfloat16* __restrict__ wq, const __nv_bfloat16* __restrict__ wk,
    __nv_bfloat16* __restrict__ k_cache, __nv_bfloat16* __restrict__ v_cache, int64_t num_tokens,
    int64_t num_slots, const float* __restrict__ rope, unsigned* __restrict__ err) {
  const int tid = threadIdx.x;
  const int sub = tid & 15;   // 16-byte chunk inside a head row
  const int row = tid >> 4;   // 0..15: head row inside a pass
  const int e0 = sub * 8;     // first element of the chunk
  const bool first = sub < 8; // chunk lies in x1 (elements 0..63)
  const int ri = e0 & 63;     // rotary index of the first element

  const Chunk wqc = ld16_nc(wq + e0);
  const Chunk wkc = ld16_nc(wk + e0);

  // Persistent loop: the position and slot of the next token are fetched one
  // iteration ahead, so each token costs one memory round trip (rows and its
  // cos/sin row together) instead of two (index first, then the table row).
  int64_t t = blockIdx.x;
  int pos = 0, slot = -1;
  if (t < num_tokens) {
    pos = __ldg(positions + t);
    slot = __ldg(slots + t);
  }
  for (; t < num_tokens; t += gridDim.x) {
    const int64_t tn = t + gridDim.x;
    __nv_bfloat16* qrow = q + t * q_stride;
    const bool pos_ok = pos >= 0 && pos < kMaxPosition;
    bool store = slot != -1;
    Chunk x0{{0u, 0u, 0u, 0u}}, x1{{0u, 0u, 0u, 0u}}, x2{{0u, 0u, 0u, 0u}};
    float cs[16];
    if (pos_ok) {
      x0 = ld16(qrow + row * kHeadDim + e0);
      x1 = ld16(qrow + (16 + row) * kHeadDim + e0);
      if (store)  // a token with slot -1 is not cached: its k and v rows are not read
        x2 = row < 8 ? ld16_nc(k + t * k_stride + row * kHeadDim + e0)
                     : ld16_nc(v + t * v_stride + (row - 8) * kHeadDim + e0);
      const float4* tab = reinterpret_cast<const float4*>(rope + static_cast<int64_t>(pos) * kHeadDim + ri);
      const float4 c0 = __ldg(tab), c1 = __ldg(tab + 1);
      const float4 s0 = __ldg(tab + 16), s1 = __ldg(tab + 17);  // +64 floats: the sin half
      cs[0] = c0.x; cs[1] = c0.y; cs[2] = c0.z; cs[3] = c0.w;
      cs[4] = c1.x; cs[5] = c1.y; cs[6] = c1.z; cs[7] = c1.w;
      cs[8] = s0.x; cs[9] = s0.y; cs[10] = s0.z; cs[11] = s0.w;
      cs[12] = s1.x; cs[13] = s1.y; cs[14] = s1.z; cs[15] = s1.w;
    }
    int pos_n = 0, slot_n = -1;
    if (tn < num_tokens) {
      pos_n = __ldg(positions + tn);
      slot_n = __ldg(slots + tn);
    }
    if (!pos_ok) {
      if (tid == 0) set_error(err, PKV_EFLAG_POSITION);
    } else {
      if (store && (slot < 0 || slot >= num_slots)) {
        if (tid == 0) set_error(err, PKV_EFLAG_SLOT);
        store = false;
      }
      st16(qrow + row * kHeadDim + e0, norm_rope(x0, wqc, cs, first));
      st16(qrow + (16 + row) * kHeadDim + e0, norm_rope(x1, wqc, cs, first));
      if (store) {
        const int64_t base = static_cast<int64_t>(slot) * kKVRow;
        if (row < 8) {  // warps 0-3: k heads (warp-uniform branch)
          st16(k_cache + base + row * kHeadDim + e0, norm_rope(x2, wkc, cs, first));
        } else {  // warps 4-7: v heads, copied bit for bit
          st16(v_cache + base + (row - 8) * kHeadDim + e0, x2);
        }
      }
    }
    pos = pos_n;
    slot = slot_n;
  }
}

cudaError_t launch_qknorm_rope_store(void* q, int64_t q_stride, const void* k, int64_t k_stride, const void* v,
                                     int64_t v_stride, const int32_t* positions, const int32_t* slots,
                                     const void* wq, const void* wk, void* k_cache, void* v_cache,
                                     int64_t num_tokens, int64_t num_blocks, const float* rope, int num_sms,
                                     unsigned* err, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  // persistent: as many CTAs as fit on the SMs at once (three of 256 threads per SM)
  const int64_t max_grid = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * kStoreCtasPerSm;
  const unsigned grid = static_cast<unsigned>(num_tokens < max_grid ? num_tokens : max_grid);
  qknorm_rope_store_kernel<<<grid, 256, 0, stream>>>(
      static_cast<__nv_bfloat16*>(q), q_stride, static_cast<const __nv_bfloat16*>(k), k_stride,
      static_cast<const __nv_bfloat16*>(v), v_stride, positions, slots, static_cast<const __nv_bfloat16*>(wq),
      static_cast<const __nv_bfloat16*>(wk), static_cast<__nv_bfloat16*>(k_cache),
      static_cast<__nv_bfloat16*>(v_cache), num_tokens, num_blocks * kBlockSize, rope, err);
  return cudaGetLastError();
}

}  // namespace pkv
