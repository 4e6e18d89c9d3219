// Step a3 entry point (the tcgen05 kernel is being brought up).
#include "internal.h"

extern "C" int pa_prefill_varlen(const void *, const pa_cache_t *, int, const int32_t *,
                                 const int32_t *, const int32_t *, int, int, int, int n_heads,
                                 int n_kv_heads, int head_dim, float, void *, int32_t *,
                                 pa_stream_t) {
    if (n_heads <= 0 || n_kv_heads <= 0 || n_heads % n_kv_heads != 0) return PA_ERR_INVALID;
    return PA_ERR_UNSUPPORTED;
}
