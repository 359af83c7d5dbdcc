// kv_trace.cuh -- NVTX ranges around the C-ABI calls (host code).
//
// Every entry point that enqueues GPU work (or waits for it) opens a range named
// after itself in the NVTX domain "kvevict" for the duration of the host call, so
// a profiler's timeline, or `ncu --nvtx --nvtx-include "kvevict@kv_score/"`, can
// attribute each kernel to the call that launched it.  NVTX 3 is header-only: with
// no tool attached (NVTX_INJECTION64_PATH unset) a range costs one indirect call
// to an empty function.
#pragma once

#include <nvtx3/nvToolsExt.h>

namespace kvevict {

inline nvtxDomainHandle_t api_domain() {
    static const nvtxDomainHandle_t d = nvtxDomainCreateA("kvevict");
    return d;
}

class ApiRange {
  public:
    explicit ApiRange(const char *name) {
        nvtxEventAttributes_t a = {};
        a.version = NVTX_VERSION;
        a.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
        a.messageType = NVTX_MESSAGE_TYPE_ASCII;
        a.message.ascii = name;
        nvtxDomainRangePushEx(api_domain(), &a);
    }
    ~ApiRange() { nvtxDomainRangePop(api_domain()); }
    ApiRange(const ApiRange &) = delete;
    ApiRange &operator=(const ApiRange &) = delete;
};

}  // namespace kvevict

// Opens the calling entry point's range until it returns.
#define KV_API_RANGE() const ::kvevict::ApiRange kv_api_range_(__func__)
