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
