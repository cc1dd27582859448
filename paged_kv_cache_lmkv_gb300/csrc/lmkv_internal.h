// lmkv_internal.h -- declarations shared by the library's translation units
// (not part of the C ABI).
#pragma once

#include <cstdint>

// Adds n to the counter lmkv_launch_count() reports.
void lmkv_internal_add_launches(int64_t n);
