// prefill.cu -- placeholder until the tcgen05 prefill kernel lands.
#include "pa_internal.h"

extern "C" pa_status pa_prefill(const pa_prefill_shapes*, const void*, const void*, const void*, const void*,
                                const int32_t*, const int32_t*, const int32_t*, const int32_t*, int, float, void*,
                                float*, void*, size_t, cudaStream_t) {
    return PA_ERR_UNSUPPORTED;
}
