// NVTX ranges around the exported calls, for timelines taken with a profiler
// (Nsight Systems / Nsight Compute's range filters).  Header-only NVTX3 from
// the CUDA toolkit: without a profiler attached every call is an early return
// through a function pointer, so a range costs a struct fill and two calls.
// Each range lives in the "pkv" domain, is named after the exported call
// (a string registered once) and carries the call's size (tokens or
// sequences) as its int64 payload, so no message is formatted per call.
#pragma once

#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

namespace pkv {

inline nvtxDomainHandle_t nvtx_domain() {
  static const nvtxDomainHandle_t d = nvtxDomainCreateA("pkv");
  return d;
}

class NvtxRange {
 public:
  NvtxRange(nvtxStringHandle_t name, int64_t size) {
    nvtxEventAttributes_t a = {};
    a.version = NVTX_VERSION;
    a.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
    a.messageType = NVTX_MESSAGE_TYPE_REGISTERED;
    a.message.registered = name;
    a.payloadType = NVTX_PAYLOAD_TYPE_INT64;
    a.payload.llValue = size;
    nvtxDomainRangePushEx(nvtx_domain(), &a);
  }
  ~NvtxRange() { nvtxDomainRangePop(nvtx_domain()); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

}  // namespace pkv

// A range named `name` (a string literal) over the rest of the enclosing scope, with payload `size`.
#define PKV_NVTX_RANGE(name, size)                                                                     \
  static const nvtxStringHandle_t pkv_nvtx_name_ = nvtxDomainRegisterStringA(pkv::nvtx_domain(), name); \
  const pkv::NvtxRange pkv_nvtx_range_(pkv_nvtx_name_, static_cast<int64_t>(size))
