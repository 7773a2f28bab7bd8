// Internal host-side declarations shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>

#include "pa.h"

// Records a one-line description of the failure for pa_last_error().
void pa_set_error(const char* msg);
// pa_set_error(msg) and return `st`.
pa_status pa_fail(pa_status st, const char* msg);
