// Shared host-side helpers of the C ABI: thread-local error text and status returns.
#pragma once

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <string>

#include "paged_kv.h"

namespace pkv {

void set_error(const char* fmt, ...);
void clear_error();

// Return `code` after recording a formatted reason.
#define PKV_FAIL(code, ...)            \
  do {                                 \
    ::pkv::set_error(__VA_ARGS__);     \
    return (code);                     \
  } while (0)

#define PKV_REQUIRE(cond, code, ...)   \
  do {                                 \
    if (!(cond)) PKV_FAIL(code, __VA_ARGS__); \
  } while (0)

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace pkv
