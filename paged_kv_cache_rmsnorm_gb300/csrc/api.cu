// Host side of the C ABI declared in include/pkv.h: argument validation,
// per-device state (RoPE table, device error word), TMA descriptor encoding
// and kernel launches.  Nothing here synchronises except pkv_check_errors.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "nvtx.cuh"

namespace pkv {
cudaError_t launch_qknorm_rope_store(void* q, int64_t q_stride, const void* k, int64_t k_stride, const void* v,
                                     int64_t v_stride, const int32_t* positions, const int32_t* slots,
                                     const void* wq, const void* wk, void* k_cache, void* v_cache,
                                     int64_t num_tokens, int64_t num_blocks, const float* rope, int num_sms,
                                     unsigned* err, cudaStream_t stream);
cudaError_t launch_add_rmsnorm(const void* x, void* residual, const void* w, void* out, int64_t num_tokens, float eps,
                               int num_sms, cudaStream_t stream);
cudaError_t decode_init_device();
cudaError_t noalloc_take_errors(unsigned* bits);
size_t decode_workspace_bytes(int batch, int max_context);
cudaError_t launch_paged_decode(const CUtensorMap& tmK, const CUtensorMap& tmV, const void* q, void* out,
                                const int32_t* context_lens, const int32_t* block_table, int batch, int max_blocks,
                                int num_blocks, int max_context, float scale, void* workspace, unsigned* err,
                                cudaStream_t stream, bool programmatic);
cudaError_t prefill_tc_init_device();
cudaError_t qkv_init_device();
cudaError_t store_init_device();
cudaError_t launch_qkv_rope_store(const CUtensorMap& tmX, const CUtensorMap& tmW, void* q_out, void* k_cache,
                                  void* v_cache, const int32_t* positions, const int32_t* slots, const void* wq,
                                  const void* wk, const float* rope, int64_t num_tokens, int64_t num_blocks,
                                  int num_sms, unsigned* err, cudaStream_t stream);
cudaError_t launch_prefill_tc(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                              const CUtensorMap& tmO, void* out,
                              const int32_t* cu_q, const int32_t* cu_k, const int32_t* block_table, int num_seqs,
                              int max_blocks, int num_blocks, int max_seqlen_q, int max_seqlen_k, float scale,
                              int num_sms, unsigned* sched, unsigned* err, cudaStream_t stream);
}  // namespace pkv

namespace {

using namespace pkv;

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(PKV_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;
// Prefill launches take their work counters from a rotation of this many
// slots, so launches in flight on different streams do not share a counter.
constexpr int kSchedSlots = 64;
constexpr size_t kStateBytes = 256 + kSchedSlots * 2 * sizeof(unsigned);
// At most 2^23 blocks, so that every slot number (block * 256 + offset) fits
// an int32 and a 32-bit TMA coordinate.
constexpr int64_t kMaxNumBlocks = (int64_t(1) << 23);

struct DeviceState {
  bool ready = false;
  float* rope = nullptr;      // [40960][cos 64 | sin 64], fp32
  unsigned* err = nullptr;    // device error word, followed by the prefill work counters
  unsigned* sched = nullptr;  // kSchedSlots pairs {next item, CTAs done}; every launch leaves its pair at zero
  std::atomic<unsigned> sched_next{0};
  int sms = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// The fp32 RoPE table, built on the host from its definition:
// inv_freq_i = theta^(-2i/128) rounded to fp32, angle = fp32(pos * inv_freq_i),
// cos / sin evaluated in double and rounded once to fp32
// ("同一个 Qwen3，两种写法" §3.5 precomputes exactly this table).
std::vector<float> build_rope_table() {
  std::vector<float> tab(static_cast<size_t>(kMaxPosition) * kHeadDim);
  float inv[kHeadDim / 2];
  for (int i = 0; i < kHeadDim / 2; ++i) inv[i] = static_cast<float>(std::pow(PKV_ROPE_THETA, -2.0 * i / kHeadDim));
  for (int p = 0; p < kMaxPosition; ++p) {
    const float fp = static_cast<float>(p);
    for (int i = 0; i < kHeadDim / 2; ++i) {
      volatile float ang = fp * inv[i];  // one fp32 rounding, no contraction
      tab[static_cast<size_t>(p) * kHeadDim + i] = static_cast<float>(std::cos(static_cast<double>(ang)));
      tab[static_cast<size_t>(p) * kHeadDim + 64 + i] = static_cast<float>(std::sin(static_cast<double>(ang)));
    }
  }
  return tab;
}

int init_device_locked(int dev, DeviceState** out) {
  if (dev < 0 || dev >= kMaxDevices) return fail(PKV_ERR_NO_DEVICE, "device %d out of range", dev);
  DeviceState& st = g_dev[dev];
  if (st.ready) {
    *out = &st;
    return PKV_OK;
  }
  cudaDeviceProp prop;
  cudaError_t e = cudaGetDeviceProperties(&prop, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
  if (prop.major != 10 || prop.minor != 3)
    return fail(PKV_ERR_NO_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a (GB300)", dev,
                prop.major, prop.minor);
  int cur = -1;
  cudaGetDevice(&cur);
  if (cur != dev && (e = cudaSetDevice(dev)) != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
  int rc = PKV_OK;
  do {
    if (!g_encode) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
        rc = fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled not available from the driver");
        break;
      }
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    std::vector<float> tab = build_rope_table();
    if ((e = cudaMalloc(&st.rope, tab.size() * sizeof(float))) != cudaSuccess) {
      rc = cuda_fail(e, "cudaMalloc(rope table)");
      break;
    }
    if ((e = cudaMemcpy(st.rope, tab.data(), tab.size() * sizeof(float), cudaMemcpyHostToDevice)) != cudaSuccess) {
      rc = cuda_fail(e, "cudaMemcpy(rope table)");
      break;
    }
    if ((e = cudaMalloc(&st.err, kStateBytes)) != cudaSuccess) {
      rc = cuda_fail(e, "cudaMalloc(error word)");
      break;
    }
    st.sched = st.err + 64;
    if ((e = cudaMemset(st.err, 0, kStateBytes)) != cudaSuccess) {
      rc = cuda_fail(e, "cudaMemset(error word)");
      break;
    }
    if ((e = decode_init_device()) != cudaSuccess) {
      rc = cuda_fail(e, "decode kernel attributes");
      break;
    }
    if ((e = prefill_tc_init_device()) != cudaSuccess) {
      rc = cuda_fail(e, "prefill kernel attributes");
      break;
    }
    if ((e = qkv_init_device()) != cudaSuccess) {
      rc = cuda_fail(e, "qkv kernel attributes");
      break;
    }
    if ((e = store_init_device()) != cudaSuccess) {
      rc = cuda_fail(e, "store kernel attributes");
      break;
    }
    st.sms = prop.multiProcessorCount;
    st.ready = true;
  } while (false);
  if (rc != PKV_OK) {
    if (st.rope) cudaFree(st.rope);
    if (st.err) cudaFree(st.err);
    st.rope = nullptr;
    st.err = nullptr;
    st.sched = nullptr;
  }
  if (cur != dev && cur >= 0) cudaSetDevice(cur);
  *out = &st;
  return rc;
}

int current_state(DeviceState** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(PKV_ERR_NO_DEVICE, "no CUDA device: %s", cudaGetErrorString(e));
  if (dev >= 0 && dev < kMaxDevices && g_dev[dev].ready) {
    *out = &g_dev[dev];
    return PKV_OK;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  return init_device_locked(dev, out);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// 3-D view of one cache [num_blocks * 256 slots][8 heads][128 dims] for TMA:
// box = `keys` slots x 1 head x 64 dims, 128-byte swizzle.
int make_cache_map(CUtensorMap* map, const void* base, int64_t num_blocks, int keys) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(kNumKVHeads),
                        static_cast<cuuint64_t>(num_blocks) * kBlockSize};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim) * 2, static_cast<cuuint64_t>(kKVRow) * 2};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(keys)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return PKV_OK;
}

// 3-D view of q [total_q tokens][32 heads][128 dims] for TMA: box = 128
// tokens x 1 head x 64 dims, 128-byte swizzle.
// 3-D view of a bf16 [total_q][32 heads][128] tensor for TMA: box = 64 dims x
// 1 head x box_rows tokens, 128-byte swizzle.
int make_q_map(CUtensorMap* map, const void* base, int64_t total_q, int box_rows) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(kNumQHeads),
                        static_cast<cuuint64_t>(total_q)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim) * 2, static_cast<cuuint64_t>(kNumQHeads) * kHeadDim * 2};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled(q / out) failed (%d)", static_cast<int>(r));
  return PKV_OK;
}

// 2-D view of a row-major bf16 matrix [rows][cols] for TMA: box = box_rows x
// 64 columns (128 bytes), 128-byte swizzle.
int make_rows_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled(rows) failed (%d)", static_cast<int>(r));
  return PKV_OK;
}

int check_cache_args(const void* k_cache, const void* v_cache, int64_t num_blocks) {
  if (!k_cache || !v_cache) return fail(PKV_ERR_NULL, "k_cache / v_cache is NULL");
  if (!aligned16(k_cache) || !aligned16(v_cache)) return fail(PKV_ERR_ALIGN, "k_cache / v_cache not 16-byte aligned");
  if (num_blocks <= 0 || num_blocks > kMaxNumBlocks)
    return fail(PKV_ERR_SHAPE, "num_blocks = %lld outside [1, %lld]", static_cast<long long>(num_blocks),
                static_cast<long long>(kMaxNumBlocks));
  return PKV_OK;
}

}  // namespace

namespace pkv {
// Record a failure for pkv_last_error() from another translation unit.
int report_error(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}
}  // namespace pkv

extern "C" {

const char* pkv_last_error(void) { return g_last_error.c_str(); }

int pkv_version(void) { return 100; }

int pkv_init(int device) {
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* st = nullptr;
  return init_device_locked(device, &st);
}

int pkv_shutdown(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  int cur = -1;
  cudaGetDevice(&cur);
  for (int d = 0; d < kMaxDevices; ++d) {
    DeviceState& st = g_dev[d];
    if (!st.ready) continue;
    cudaSetDevice(d);
    cudaFree(st.rope);
    cudaFree(st.err);
    st.ready = false;
    st.rope = nullptr;
    st.err = nullptr;
    st.sched = nullptr;
    st.sms = 0;
  }
  if (cur >= 0) cudaSetDevice(cur);
  return PKV_OK;
}

int pkv_check_errors(void* stream, uint32_t* flags) {
  DeviceState* st = nullptr;
  int rc = current_state(&st);
  if (rc != PKV_OK) return rc;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned v = 0;
  if ((e = cudaMemcpy(&v, st->err, sizeof(v), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "reading the error word");
  if (v && (e = cudaMemset(st->err, 0, sizeof(unsigned))) != cudaSuccess) return cuda_fail(e, "clearing the error word");
  unsigned nv = 0;  // bits of pkv_attn_decode_noalloc calls made without an error word of their own
  if ((e = noalloc_take_errors(&nv)) != cudaSuccess) return cuda_fail(e, "reading the no-alloc error word");
  v |= nv;
  if (flags) *flags = v;
  if (v) return fail(PKV_ERR_BOUNDS, "kernel reported out-of-range input (flags 0x%x)", v);
  return PKV_OK;
}

// After a successful launch: PKV_OK, or in debug mode the result of checking the
// stream at once (PKV_ERR_CUDA for a fault, PKV_ERR_BOUNDS for an error bit, read
// and cleared as pkv_check_errors does).  No check while the stream is captured.
static int after_launch(void* stream) {
  if (!debug_mode() || stream_capturing(static_cast<cudaStream_t>(stream))) return PKV_OK;
  return pkv_check_errors(stream, nullptr);
}

int pkv_qknorm_rope_store(void* q, int64_t q_row_stride, const void* k, int64_t k_row_stride, const void* v,
                          int64_t v_row_stride, const int32_t* positions, const int32_t* slot_mapping,
                          const void* q_norm_w, const void* k_norm_w, void* k_cache, void* v_cache,
                          int64_t num_tokens, int64_t num_blocks, void* stream) {
  PKV_NVTX_RANGE("pkv_qknorm_rope_store", num_tokens);
  if (num_tokens < 0) return fail(PKV_ERR_SHAPE, "num_tokens < 0");
  if (num_tokens == 0) return PKV_OK;  // nothing to do: no pointer is read
  if (!q || !k || !v || !positions || !slot_mapping || !q_norm_w || !k_norm_w)
    return fail(PKV_ERR_NULL, "a required pointer is NULL");
  int rc = check_cache_args(k_cache, v_cache, num_blocks);
  if (rc != PKV_OK) return rc;
  if (q_row_stride < kNumQHeads * kHeadDim || k_row_stride < kKVRow || v_row_stride < kKVRow)
    return fail(PKV_ERR_SHAPE, "row strides must be >= 4096 (q) and 1024 (k, v) elements");
  if ((q_row_stride | k_row_stride | v_row_stride) & 7)
    return fail(PKV_ERR_ALIGN, "row strides must be multiples of 8 elements");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(q_norm_w) || !aligned16(k_norm_w))
    return fail(PKV_ERR_ALIGN, "q, k, v and the norm weights must be 16-byte aligned");
  if (!aligned4(positions) || !aligned4(slot_mapping)) return fail(PKV_ERR_ALIGN, "index arrays not 4-byte aligned");
  DeviceState* st = nullptr;
  if ((rc = current_state(&st)) != PKV_OK) return rc;
  cudaError_t e = launch_qknorm_rope_store(q, q_row_stride, k, k_row_stride, v, v_row_stride, positions,
                                           slot_mapping, q_norm_w, k_norm_w, k_cache, v_cache, num_tokens,
                                           num_blocks, st->rope, st->sms, st->err, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "qknorm_rope_store launch");
  return after_launch(stream);
}

size_t pkv_attn_decode_workspace_size(int32_t batch, int32_t max_context) {
  if (batch <= 0 || max_context <= 0) return 0;
  return decode_workspace_bytes(batch, max_context);
}

int pkv_attn_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* context_lens,
                    const int32_t* block_table, int32_t batch, int32_t max_blocks_per_seq, int64_t num_blocks,
                    int32_t max_context, float scale, void* out, void* workspace, size_t workspace_bytes,
                    void* stream) {
  PKV_NVTX_RANGE("pkv_attn_decode", batch);
  if (batch < 0) return fail(PKV_ERR_SHAPE, "batch < 0");
  if (batch > 65535) return fail(PKV_ERR_UNSUPPORTED, "batch > 65535");
  if (batch == 0) return PKV_OK;  // nothing to do: no pointer is read
  if (!q || !out || !context_lens || !block_table) return fail(PKV_ERR_NULL, "a required pointer is NULL");
  int rc = check_cache_args(k_cache, v_cache, num_blocks);
  if (rc != PKV_OK) return rc;
  if (max_blocks_per_seq <= 0) return fail(PKV_ERR_SHAPE, "max_blocks_per_seq must be > 0");
  if (max_context < 0 || static_cast<int64_t>(max_context) > static_cast<int64_t>(max_blocks_per_seq) * kBlockSize)
    return fail(PKV_ERR_SHAPE, "max_context outside [0, max_blocks_per_seq * 256]");
  if (!std::isfinite(scale)) return fail(PKV_ERR_SHAPE, "scale is not finite");
  if (!aligned16(q) || !aligned16(out)) return fail(PKV_ERR_ALIGN, "q / out not 16-byte aligned");
  if (!aligned4(context_lens) || !aligned4(block_table)) return fail(PKV_ERR_ALIGN, "index arrays not 4-byte aligned");
  const size_t need = decode_workspace_bytes(batch, max_context);
  if (need > 0) {
    if (!workspace) return fail(PKV_ERR_WORKSPACE, "workspace of %zu bytes required, got NULL", need);
    if (workspace_bytes < need)
      return fail(PKV_ERR_WORKSPACE, "workspace of %zu bytes required, got %zu", need, workspace_bytes);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return fail(PKV_ERR_ALIGN, "workspace not 256-byte aligned");
  }
  DeviceState* st = nullptr;
  if ((rc = current_state(&st)) != PKV_OK) return rc;
  CUtensorMap tmK, tmV;
  if ((rc = make_cache_map(&tmK, k_cache, num_blocks, 64)) != PKV_OK) return rc;
  if ((rc = make_cache_map(&tmV, v_cache, num_blocks, 64)) != PKV_OK) return rc;
  cudaError_t e = launch_paged_decode(tmK, tmV, q, out, context_lens, block_table, batch, max_blocks_per_seq,
                                      static_cast<int>(num_blocks), max_context, scale, workspace, st->err,
                                      static_cast<cudaStream_t>(stream), true);
  if (e != cudaSuccess) return cuda_fail(e, "paged_decode launch");
  return after_launch(stream);
}

int pkv_attn_prefill(const void* q, const void* k_cache, const void* v_cache, const int32_t* cu_seqlens_q,
                     const int32_t* cu_seqlens_k, const int32_t* block_table, int32_t num_seqs,
                     int32_t max_blocks_per_seq, int64_t num_blocks, int32_t total_q, int32_t max_seqlen_q,
                     int32_t max_seqlen_k, float scale, void* out, void* stream) {
  PKV_NVTX_RANGE("pkv_attn_prefill", total_q);
  if (num_seqs < 0 || total_q < 0 || max_seqlen_q < 0 || max_seqlen_k < 0)
    return fail(PKV_ERR_SHAPE, "negative size argument");
  if (num_seqs > 65535) return fail(PKV_ERR_UNSUPPORTED, "num_seqs > 65535");
  if (num_seqs == 0 || total_q == 0) return PKV_OK;  // nothing to do: no pointer is read
  if (!q || !out || !cu_seqlens_q || !cu_seqlens_k || !block_table)
    return fail(PKV_ERR_NULL, "a required pointer is NULL");
  int rc = check_cache_args(k_cache, v_cache, num_blocks);
  if (rc != PKV_OK) return rc;
  if (max_blocks_per_seq <= 0) return fail(PKV_ERR_SHAPE, "max_blocks_per_seq must be > 0");
  if (static_cast<int64_t>(max_seqlen_k) > static_cast<int64_t>(max_blocks_per_seq) * kBlockSize)
    return fail(PKV_ERR_SHAPE, "max_seqlen_k exceeds max_blocks_per_seq * 256");
  if (max_seqlen_q > max_seqlen_k) return fail(PKV_ERR_SHAPE, "max_seqlen_q > max_seqlen_k");
  if (!std::isfinite(scale)) return fail(PKV_ERR_SHAPE, "scale is not finite");
  if (!aligned16(q) || !aligned16(out)) return fail(PKV_ERR_ALIGN, "q / out not 16-byte aligned");
  if (!aligned4(cu_seqlens_q) || !aligned4(cu_seqlens_k) || !aligned4(block_table))
    return fail(PKV_ERR_ALIGN, "index arrays not 4-byte aligned");
  DeviceState* st = nullptr;
  if ((rc = current_state(&st)) != PKV_OK) return rc;
  CUtensorMap tmQ, tmK, tmV;
  if ((rc = make_q_map(&tmQ, q, total_q, 128)) != PKV_OK) return rc;
  CUtensorMap tmO;  // the output, stored 32 rows x half a head at a time from the epilogue's staging
  if ((rc = make_q_map(&tmO, out, total_q, 32)) != PKV_OK) return rc;
  if ((rc = make_cache_map(&tmK, k_cache, num_blocks, 128)) != PKV_OK) return rc;
  if ((rc = make_cache_map(&tmV, v_cache, num_blocks, 128)) != PKV_OK) return rc;
  cudaError_t e = launch_prefill_tc(tmQ, tmK, tmV, tmO, out, cu_seqlens_q, cu_seqlens_k, block_table, num_seqs,
                                    max_blocks_per_seq, static_cast<int>(num_blocks), max_seqlen_q, max_seqlen_k,
                                    scale, st->sms, st->sched + 2 * (st->sched_next++ % kSchedSlots), st->err,
                                    static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "paged_prefill launch");
  return after_launch(stream);
}

int pkv_add_rmsnorm(const void* x, void* residual, const void* weight, void* out, int64_t num_tokens,
                    int32_t hidden, float eps, void* stream) {
  PKV_NVTX_RANGE("pkv_add_rmsnorm", num_tokens);
  if (num_tokens < 0) return fail(PKV_ERR_SHAPE, "num_tokens < 0");
  if (num_tokens == 0) return PKV_OK;  // nothing to do: no pointer is read
  if (!x || !weight || !out) return fail(PKV_ERR_NULL, "a required pointer is NULL");
  if (hidden != PKV_HIDDEN) return fail(PKV_ERR_UNSUPPORTED, "hidden must be %d", PKV_HIDDEN);
  if (!(eps >= 0.f) || !std::isfinite(eps)) return fail(PKV_ERR_SHAPE, "eps must be finite and >= 0");
  if (!aligned16(x) || !aligned16(weight) || !aligned16(out) || (residual && !aligned16(residual)))
    return fail(PKV_ERR_ALIGN, "x, residual, weight and out must be 16-byte aligned");
  if (residual && (residual == out || residual == x)) return fail(PKV_ERR_SHAPE, "residual must not alias x or out");
  DeviceState* st = nullptr;
  int rc = current_state(&st);
  if (rc != PKV_OK) return rc;
  cudaError_t e = launch_add_rmsnorm(x, residual, weight, out, num_tokens, eps, st->sms, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "add_rmsnorm launch");
  return after_launch(stream);
}

int pkv_qkv_rope_store(const void* x, const void* w_qkv, const int32_t* positions, const int32_t* slot_mapping,
                       const void* q_norm_w, const void* k_norm_w, void* q_out, void* k_cache, void* v_cache,
                       int64_t num_tokens, int64_t num_blocks, void* stream) {
  PKV_NVTX_RANGE("pkv_qkv_rope_store", num_tokens);
  if (num_tokens < 0) return fail(PKV_ERR_SHAPE, "num_tokens < 0");
  if (num_tokens > (int64_t(1) << 31) - 1) return fail(PKV_ERR_UNSUPPORTED, "num_tokens >= 2^31");
  if (num_tokens == 0) return PKV_OK;  // nothing to do: no pointer is read
  if (!x || !w_qkv || !positions || !slot_mapping || !q_norm_w || !k_norm_w || !q_out)
    return fail(PKV_ERR_NULL, "a required pointer is NULL");
  int rc = check_cache_args(k_cache, v_cache, num_blocks);
  if (rc != PKV_OK) return rc;
  if (!aligned16(x) || !aligned16(w_qkv) || !aligned16(q_out) || !aligned16(q_norm_w) || !aligned16(k_norm_w))
    return fail(PKV_ERR_ALIGN, "x, w_qkv, q_out and the norm weights must be 16-byte aligned");
  if (!aligned4(positions) || !aligned4(slot_mapping)) return fail(PKV_ERR_ALIGN, "index arrays not 4-byte aligned");
  DeviceState* st = nullptr;
  if ((rc = current_state(&st)) != PKV_OK) return rc;
  CUtensorMap tmX, tmW;
  if ((rc = make_rows_map(&tmX, x, num_tokens, PKV_HIDDEN, 128)) != PKV_OK) return rc;
  if ((rc = make_rows_map(&tmW, w_qkv, PKV_QKV_OUT, PKV_HIDDEN, 128)) != PKV_OK) return rc;  // half a tile's features per CTA
  cudaError_t e = launch_qkv_rope_store(tmX, tmW, q_out, k_cache, v_cache, positions, slot_mapping, q_norm_w, k_norm_w,
                                        st->rope, num_tokens, num_blocks, st->sms, st->err,
                                        static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "qkv_rope_store launch");
  return after_launch(stream);
}

}  // extern "C"
