// Library-wide entry points: error string and version.
#include "host_util.h"

namespace sv {
char* error_buffer() {
    static thread_local char buf[kErrLen] = {0};
    return buf;
}
}  // namespace sv

extern "C" const char* spec_last_error(void) { return sv::error_buffer(); }

extern "C" int32_t spec_version(void) { return SPECVERIFY_VERSION; }
