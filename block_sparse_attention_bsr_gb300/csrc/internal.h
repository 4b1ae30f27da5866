// Internal host declarations shared by the library's translation units.
#pragma once

#include "bsr_attn.h"

namespace bsr {

// Records a printf-style message for bsr_last_error() on this thread and
// returns `status`.
bsr_status fail(bsr_status status, const char* fmt, ...)
#if defined(__GNUC__)
    __attribute__((format(printf, 2, 3)))
#endif
    ;

}  // namespace bsr
