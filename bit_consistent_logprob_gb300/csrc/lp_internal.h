// lp_internal.h -- helpers shared by the library's translation units (not part of the ABI).
#pragma once

#include "lp.h"

// Validate a configuration against the proven set; sets the thread-local error message.
int lp_internal_validate_config(const lp_config* c);

// Record a printf-style message as lp_last_error() and return `code`.
int lp_internal_fail(int code, const char* fmt, ...);
