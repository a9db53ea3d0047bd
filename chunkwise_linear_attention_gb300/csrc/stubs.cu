// stubs.cu -- entry points whose kernels are not built yet.
#include "cla_internal.cuh"

using namespace cla;

extern "C" size_t cla_selective_scan_workspace_size(int64_t, int64_t, int64_t, int64_t) { return 256; }
extern "C" size_t cla_selective_scan_ckpt_elems(int64_t, int64_t, int64_t, int64_t) { return 0; }
extern "C" int cla_selective_scan_fwd(const uint16_t *, const float *, const float *, const uint16_t *,
                                      const uint16_t *, const float *, float *, float *, float *, int64_t,
                                      int64_t, int64_t, int64_t, void *, size_t, void *) {
    return fail(CLA_ERR_UNSUPPORTED, "cla_selective_scan_fwd: not built");
}
extern "C" int cla_selective_scan_bwd(const uint16_t *, const float *, const float *, const uint16_t *,
                                      const uint16_t *, const float *, const float *, const float *,
                                      const float *, float *, float *, float *, float *, float *, float *,
                                      int64_t, int64_t, int64_t, int64_t, void *, size_t, void *) {
    return fail(CLA_ERR_UNSUPPORTED, "cla_selective_scan_bwd: not built");
}

