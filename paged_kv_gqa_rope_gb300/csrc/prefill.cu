// Step a3 placeholder (replaced by the tcgen05 kernel).
#include "internal.h"

extern "C" int pa_prefill_varlen(const void *, const pa_cache_t *, int, const int32_t *,
                                 const int32_t *, const int32_t *, int, int, int, int, int, int,
                                 float, void *, int32_t *, pa_stream_t) {
    return PA_ERR_UNSUPPORTED;
}
