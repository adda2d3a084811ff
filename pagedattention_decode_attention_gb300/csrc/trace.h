// NVTX ranges around the library's entry points.
//
// A profiler attached to the process (Nsight Systems, or Nsight Compute with
// --nvtx) sees every call as a range named after the entry point, in the
// "pagedattn" domain, with the kernels the call launched inside it, so a
// decode step can be split into its plan, append, attention, copy and swap
// calls.  Without a tool attached, a push or pop is a test of an unset
// function pointer.  NVTX 3 is header-only: nothing extra is linked.
#pragma once

#include <nvtx3/nvToolsExt.h>

namespace pa {

inline nvtxDomainHandle_t trace_domain() {
  static const nvtxDomainHandle_t domain = nvtxDomainCreateA("pagedattn");
  return domain;
}

class TraceRange {
 public:
  explicit TraceRange(const char* name) {
    nvtxEventAttributes_t attr = {};
    attr.version = NVTX_VERSION;
    attr.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
    attr.messageType = NVTX_MESSAGE_TYPE_ASCII;
    attr.message.ascii = name;
    nvtxDomainRangePushEx(trace_domain(), &attr);
  }
  ~TraceRange() { nvtxDomainRangePop(trace_domain()); }
  TraceRange(const TraceRange&) = delete;
  TraceRange& operator=(const TraceRange&) = delete;
};

}  // namespace pa

// One range over the rest of the enclosing scope.
#define PA_TRACE(name) ::pa::TraceRange pa_trace_range_(name)
