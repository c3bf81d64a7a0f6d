// Internal helpers shared by the library's translation units (host side).
#pragma once

#include <cstdint>
#include <string>

#include "pagedkv.h"

namespace pkv {

// Thread-local last-error text behind pkv_last_error_string().
void set_error(const std::string& msg);
void clear_error();

inline pkv_status fail(pkv_status st, const char* msg) {
    set_error(msg);
    return st;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace pkv

// An NVTX range named after the entry point around each C-ABI call, so a
// profiler (ncu --nvtx, Nsight Systems) can attribute host time per call.
// Compiled in only when the library is built with PKV_NVTX defined
// (PKV_NVTX=1 in the environment of paged_kv_cache_162_gb300/_build.py);
// otherwise the macro is empty and costs nothing.
#ifdef PKV_NVTX
#include <nvtx3/nvToolsExt.h>
namespace pkv {
struct TraceRange {
    explicit TraceRange(const char* name) { nvtxRangePushA(name); }
    ~TraceRange() { nvtxRangePop(); }
    TraceRange(const TraceRange&) = delete;
    TraceRange& operator=(const TraceRange&) = delete;
};
}  // namespace pkv
#define PKV_TRACE(name) ::pkv::TraceRange pkv_trace_range_(name)
#else
#define PKV_TRACE(name) ((void)0)
#endif
