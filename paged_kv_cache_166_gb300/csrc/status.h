// Thread-local error message plumbing shared by the library's translation units.
#pragma once

#include <cstdarg>
#include <cstdio>

#include "pkv.h"

namespace pkv {

// Sets the calling thread's last-error message and returns `code`.
int fail(int code, const char* fmt, ...);
// Clears the calling thread's last-error message and returns PKV_OK.
int ok();

}  // namespace pkv

#define PKV_REQUIRE(cond, code, ...)              \
  do {                                            \
    if (!(cond)) return ::pkv::fail((code), __VA_ARGS__); \
  } while (0)
