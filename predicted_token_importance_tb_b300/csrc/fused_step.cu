// Fused decode step (append, score, select, attend in one cooperative launch).
#include "kernels.cuh"

namespace tb {

bool fused_step_supported(const tb_shape &sh, int64_t n_tokens, int32_t k) {
    (void)sh;
    (void)n_tokens;
    (void)k;
    return false;
}

int64_t fused_chunks(const tb_shape &sh, int64_t n_tokens) {
    (void)sh;
    (void)n_tokens;
    return 0;
}

cudaError_t launch_fused_step(const tb_shape &, const tb_step_params &, int64_t, const uint16_t *, const uint16_t *,
                              const uint16_t *, const uint16_t *, const uint16_t *, uint16_t *, uint16_t *,
                              uint16_t *, int32_t *, int32_t *, int32_t *, uint16_t *, RowCtl *, uint32_t *, float *,
                              int32_t *, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace tb
