// pkv_attn_decode_noalloc: the split-K paged decode of decode.cu for callers
// that cannot allocate device memory — for example code running inside a
// memory pool that has been sealed, an allocator-free embedding of the
// library, or a process whose device memory is all handed out up front and
// therefore has nowhere to put a workspace.  Such a caller has no
// cudaMalloc'd workspace to pass, so this entry point uses scratch that lives
// in this library's own static device memory instead.
//
// The scratch is one file-scope array of kNoAllocScratchBytes (8 MiB).  Every
// GPU that loads the library holds it until the process exits.  Host code
// cannot use the array's name as a device address, so the first call on each
// device, with that device current, looks up its address with
// cudaGetSymbolAddress and keeps it; that first call should therefore come
// before any stream capture.  Nothing here calls cudaMalloc, cudaFree or an
// allocating library routine.
#include <cmath>
#include <mutex>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "nvtx.cuh"

namespace pkv {
cudaError_t decode_init_device();
size_t decode_workspace_bytes(int batch, int max_context);
cudaError_t launch_paged_decode(const CUtensorMap& tmK, const CUtensorMap& tmV, const void* q, void* out,
                                const int32_t* context_lens, const int32_t* block_table, int batch, int max_blocks,
                                int num_blocks, int max_context, float scale, void* workspace, unsigned* err,
                                cudaStream_t stream, bool programmatic);
int report_error(int code, const char* fmt, ...);
}  // namespace pkv

namespace {

using namespace pkv;

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
constexpr int kMaxDevices = 64;
constexpr int64_t kMaxNumBlocks = int64_t(1) << 23;

// Shared by every call on a device; see pkv.h for the rules that follow from that.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];
// Error bits of calls that pass no error word of their own.
static __device__ __align__(256) unsigned g_noalloc_err;

struct NoAllocDevice {
  bool ready = false;
  void* scratch = nullptr;    // device address of g_noalloc_scratch on this device
  unsigned* err = nullptr;    // device address of g_noalloc_err on this device
};

std::mutex g_noalloc_mu;
NoAllocDevice g_noalloc_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_noalloc_encode = nullptr;

// One-time set-up for the current device: symbol addresses, the kernel's
// shared-memory attribute and the tensor-map encoder.  No allocation.
int noalloc_setup(NoAllocDevice** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return report_error(PKV_ERR_NO_DEVICE, "no CUDA device: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return report_error(PKV_ERR_NO_DEVICE, "device %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocDevice& st = g_noalloc_dev[dev];
  if (st.ready) {
    *out = &st;
    return PKV_OK;
  }
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3)
    return report_error(PKV_ERR_NO_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a", dev, major,
                        minor);
  void* scratch = nullptr;
  void* err = nullptr;
  if ((e = cudaGetSymbolAddress(&scratch, g_noalloc_scratch)) != cudaSuccess)
    return report_error(PKV_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
  if ((e = cudaGetSymbolAddress(&err, g_noalloc_err)) != cudaSuccess)
    return report_error(PKV_ERR_CUDA, "cudaGetSymbolAddress(error word): %s", cudaGetErrorString(e));
  if ((e = decode_init_device()) != cudaSuccess)
    return report_error(PKV_ERR_CUDA, "decode kernel attributes: %s", cudaGetErrorString(e));
  if (!g_noalloc_encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
      return report_error(PKV_ERR_CUDA, "cuTensorMapEncodeTiled not available from the driver");
    g_noalloc_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  st.scratch = scratch;
  st.err = static_cast<unsigned*>(err);
  st.ready = true;
  *out = &st;
  return PKV_OK;
}

int noalloc_cache_map(CUtensorMap* map, const void* base, int64_t num_blocks) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(kNumKVHeads),
                        static_cast<cuuint64_t>(num_blocks) * kBlockSize};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim) * 2, static_cast<cuuint64_t>(kKVRow) * 2};
  cuuint32_t box[3] = {64, 1, 64};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_noalloc_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return report_error(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return PKV_OK;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool al4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

namespace pkv {
// The error bits that no-alloc calls without an error word of their own left
// on the current device, cleared as they are read (symbol copies: no
// allocation).  Zero when this device has not made such a call.
cudaError_t noalloc_take_errors(unsigned* bits) {
  *bits = 0;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaSuccess;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_dev[dev].ready) return cudaSuccess;
  }
  unsigned v = 0;
  if ((e = cudaMemcpyFromSymbol(&v, g_noalloc_err, sizeof(v))) != cudaSuccess) return e;
  if (v) {
    const unsigned zero = 0;
    if ((e = cudaMemcpyToSymbol(g_noalloc_err, &zero, sizeof(zero))) != cudaSuccess) return e;
  }
  *bits = v;
  return cudaSuccess;
}
}  // namespace pkv

extern "C" int pkv_attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* context_lens, const int32_t* block_table, int32_t batch,
                                       int32_t max_blocks_per_seq, int64_t num_blocks, int32_t max_context,
                                       float scale, void* out, uint32_t* error_flags, void* stream) {
  PKV_NVTX_RANGE("pkv_attn_decode_noalloc", batch);
  if (batch < 0) return report_error(PKV_ERR_SHAPE, "batch < 0");
  if (batch > 65535) return report_error(PKV_ERR_UNSUPPORTED, "batch > 65535");
  if (batch == 0) return PKV_OK;  // nothing to do: no pointer is read
  if (!q || !out || !context_lens || !block_table || !k_cache || !v_cache)
    return report_error(PKV_ERR_NULL, "a required pointer is NULL");
  if (num_blocks <= 0 || num_blocks > kMaxNumBlocks)
    return report_error(PKV_ERR_SHAPE, "num_blocks outside [1, 2^23]");
  if (max_blocks_per_seq <= 0) return report_error(PKV_ERR_SHAPE, "max_blocks_per_seq must be > 0");
  if (max_context < 0 || static_cast<int64_t>(max_context) > static_cast<int64_t>(max_blocks_per_seq) * kBlockSize)
    return report_error(PKV_ERR_SHAPE, "max_context outside [0, max_blocks_per_seq * 256]");
  if (!std::isfinite(scale)) return report_error(PKV_ERR_SHAPE, "scale is not finite");
  if (!al16(q) || !al16(out) || !al16(k_cache) || !al16(v_cache))
    return report_error(PKV_ERR_ALIGN, "q, out and the caches must be 16-byte aligned");
  if (!al4(context_lens) || !al4(block_table) || (error_flags && !al4(error_flags)))
    return report_error(PKV_ERR_ALIGN, "index arrays / error word not 4-byte aligned");
  const size_t need = decode_workspace_bytes(batch, max_context);
  if (need > kNoAllocScratchBytes)
    return report_error(PKV_ERR_WORKSPACE,
                        "batch %d with max_context %d needs %zu bytes of scratch; the static scratch holds %zu",
                        batch, max_context, need, kNoAllocScratchBytes);
  NoAllocDevice* st = nullptr;
  int rc = noalloc_setup(&st);
  if (rc != PKV_OK) return rc;
  CUtensorMap tmK, tmV;
  if ((rc = noalloc_cache_map(&tmK, k_cache, num_blocks)) != PKV_OK) return rc;
  if ((rc = noalloc_cache_map(&tmV, v_cache, num_blocks)) != PKV_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (need > 0) {
    // the split tickets must start at zero; the scratch keeps whatever the last call left
    const size_t counters = static_cast<size_t>(batch) * kNumKVHeads * sizeof(unsigned);
    if ((e = cudaMemsetAsync(st->scratch, 0, counters, s)) != cudaSuccess)
      return report_error(PKV_ERR_CUDA, "clearing the scratch counters: %s", cudaGetErrorString(e));
  }
  e = launch_paged_decode(tmK, tmV, q, out, context_lens, block_table, batch, max_blocks_per_seq,
                          static_cast<int>(num_blocks), max_context, scale, need > 0 ? st->scratch : nullptr,
                          error_flags ? error_flags : st->err, s, false);
  if (e != cudaSuccess) return report_error(PKV_ERR_CUDA, "paged_decode launch: %s", cudaGetErrorString(e));
  if (!pkv::debug_mode() || pkv::stream_capturing(s)) return PKV_OK;
  // debug mode: check the call at once, still without allocating (the caller's own
  // error word, when given, is left for the caller to read)
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess)
    return report_error(PKV_ERR_CUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
  if (error_flags) return PKV_OK;
  unsigned bits = 0;
  if ((e = pkv::noalloc_take_errors(&bits)) != cudaSuccess)
    return report_error(PKV_ERR_CUDA, "reading the no-alloc error word: %s", cudaGetErrorString(e));
  if (bits) return report_error(PKV_ERR_BOUNDS, "kernel reported out-of-range input (flags 0x%x)", bits);
  return PKV_OK;
}
