// Residual add fused into the decoder layer's RMSNorm over the hidden size.
//
// Operation ("同一个 Qwen3，两种写法" §3.6, nano-vllm add_rms_forward):
//   s        = fp32(x[t]) + fp32(residual[t])
//   residual[t] <- bf16(s)                                   (the new residual)
//   out[t]   = bf16(bf16(s * rsqrt(mean(s^2) + eps)) * w)     (mean over the
//                                                             unrounded s)
// With no residual (the first layer) s = fp32(x[t]) and nothing is written
// back; the caller keeps x as the residual.
//
// HBM-bound: the page's traffic model is 4 rows of 8 KiB per token fused
// (read x and r, write out and the sum) against 5 unfused.  One CTA of 512
// threads holds a whole 4096-element row, 16 bytes per thread, so the sum
// never leaves registers between the add and the normalisation; the sum of
// squares is reduced across the CTA (warp shuffles, then one warp over the 16
// partials).  CTAs are persistent (three per SM) and load the next token's
// rows one iteration ahead, so the loads of one token overlap the reduction
// and stores of the previous one.
#include "common.cuh"

namespace pkv {

constexpr int kHidden = 4096;
constexpr int kArnThreads = kHidden / 8;  // one 16-byte chunk of the row per thread
constexpr int kArnCtasPerSm = 3;

namespace {

__device__ __forceinline__ uint4 ld_row16(const __nv_bfloat16* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }

__device__ __forceinline__ void widen(const uint4& v, float (&f)[8]) {
  f[0] = bf16lo(v.x); f[1] = bf16hi(v.x);
  f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
  f[4] = bf16lo(v.z); f[5] = bf16hi(v.z);
  f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
}

}  // namespace

__global__ void __launch_bounds__(kArnThreads, kArnCtasPerSm)
    add_rmsnorm_kernel(const __nv_bfloat16* __restrict__ x, __nv_bfloat16* __restrict__ residual,
                       const __nv_bfloat16* __restrict__ w, __nv_bfloat16* __restrict__ out, int64_t num_tokens,
                       float eps) {
  __shared__ float part[2][kArnThreads / 32];  // per-warp partial sums, double-buffered by iteration
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int e0 = tid * 8;
  float wf[8];
  widen(ld_row16(w + e0), wf);
  const bool add = residual != nullptr;

  int64_t t = blockIdx.x;
  uint4 xv = make_uint4(0u, 0u, 0u, 0u), rv = make_uint4(0u, 0u, 0u, 0u);
  if (t < num_tokens) {
    xv = ld_row16(x + t * kHidden + e0);
    if (add) rv = *reinterpret_cast<const uint4*>(residual + t * kHidden + e0);
  }
  for (int it = 0; t < num_tokens; t += gridDim.x, ++it) {
    const int64_t tn = t + gridDim.x;
    // the next token's rows are in flight while this one is reduced and stored
    uint4 xn = make_uint4(0u, 0u, 0u, 0u), rn = make_uint4(0u, 0u, 0u, 0u);
    if (tn < num_tokens) {
      xn = ld_row16(x + tn * kHidden + e0);
      if (add) rn = *reinterpret_cast<const uint4*>(residual + tn * kHidden + e0);
    }
    float s[8];
    widen(xv, s);
    if (add) {
      float r[8];
      widen(rv, r);
#pragma unroll
      for (int i = 0; i < 8; ++i) s[i] += r[i];
      *reinterpret_cast<uint4*>(residual + t * kHidden + e0) =
          make_uint4(pack_bf16x2(s[0], s[1]), pack_bf16x2(s[2], s[3]), pack_bf16x2(s[4], s[5]), pack_bf16x2(s[6], s[7]));
    }
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = fmaf(s[i], s[i], ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    float* pb = part[it & 1];
    if (lane == 0) pb[warp] = ss;
    __syncthreads();
    float tot = lane < kArnThreads / 32 ? pb[lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);  // every lane gets the total
    // every warp reduces the 16 partials itself: no second barrier, and the
    // other buffer of `part` is what the next iteration writes
    const float rr = rsqrtf(tot * (1.0f / kHidden) + eps);
    uint32_t y[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float n0 = __bfloat162float(__float2bfloat16_rn(s[2 * i] * rr));
      const float n1 = __bfloat162float(__float2bfloat16_rn(s[2 * i + 1] * rr));
      y[i] = pack_bf16x2(n0 * wf[2 * i], n1 * wf[2 * i + 1]);
    }
    *reinterpret_cast<uint4*>(out + t * kHidden + e0) = make_uint4(y[0], y[1], y[2], y[3]);
    xv = xn;
    rv = rn;
  }
}

cudaError_t launch_add_rmsnorm(const void* x, void* residual, const void* w, void* out, int64_t num_tokens, float eps,
                               int num_sms, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int64_t max_grid = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * kArnCtasPerSm;
  const unsigned grid = static_cast<unsigned>(num_tokens < max_grid ? num_tokens : max_grid);
  add_rmsnorm_kernel<<<grid, kArnThreads, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(residual),
      static_cast<const __nv_bfloat16*>(w), static_cast<__nv_bfloat16*>(out), num_tokens, eps);
  return cudaGetLastError();
}

}  // namespace pkv
