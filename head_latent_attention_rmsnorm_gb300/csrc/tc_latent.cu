// tc_latent.cu -- latent-space (absorbed-form) attention on the tensor cores: the
// absorbed prefill and the split-KV decode.  Not yet routed to the tensor cores:
// every call of these two entry points runs the CUDA-core kernels.
#include "mla_internal.h"
#include "tc.h"
#include "tc_internal.h"

namespace mla {

bool tc_absorbed_supported(int, int, int, int) { return false; }
bool tc_decode_supported(int, int, int, int, int) { return false; }

cudaError_t tc_absorbed_prefill(const TcPrefill &, const void *, const void *, void *, float *, const void *,
                                const void *, const void *, void *, void *, void *, cudaStream_t) {
    return cudaErrorNotSupported;
}
cudaError_t tc_decode(const TcDecode &, const void *, const void *, const void *, const void *, const void *, void *,
                      float *, float *, float *, void *, void *, void *, void *, cudaStream_t) {
    return cudaErrorNotSupported;
}
cudaError_t tc_latent_read_and_clear_error(unsigned *flags, cudaStream_t) {
    (void)flags;
    return cudaSuccess;
}

cudaError_t tc_read_and_clear_error(unsigned int *flags, cudaStream_t st) {
    cudaError_t e = tc_gemm_read_and_clear_error(flags, st);
    if (e == cudaSuccess) e = tc_attn_read_and_clear_error(flags, st);
    if (e == cudaSuccess) e = tc_latent_read_and_clear_error(flags, st);
    return e;
}

}  // namespace mla
