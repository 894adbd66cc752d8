// tc_stub.cu -- placeholder until the tcgen05 kernels land: no shape is routed to
// the tensor-core path.
#include "mla_internal.h"
#include "tc.h"

namespace mla {
bool tc_explicit_supported(int, int, int, int) { return false; }
bool tc_absorbed_supported(int, int, int, int) { return false; }
bool tc_decode_supported(int, int, int, int, int) { return false; }
cudaError_t tc_explicit_prefill(const TcPrefill &, const void *, const void *, void *, float *, const void *,
                                const void *, const void *, void *, void *, cudaStream_t) {
    return cudaErrorNotSupported;
}
cudaError_t tc_absorbed_prefill(const TcPrefill &, const void *, const void *, void *, float *, const void *,
                                const void *, const void *, void *, void *, void *, cudaStream_t) {
    return cudaErrorNotSupported;
}
cudaError_t tc_decode(const TcDecode &, const void *, const void *, const void *, const void *, const void *,
                      void *, float *, float *, float *, void *, void *, void *, void *, cudaStream_t) {
    return cudaErrorNotSupported;
}
cudaError_t tc_read_and_clear_error(unsigned int *flags, cudaStream_t) {
    *flags = 0;
    return cudaSuccess;
}
}  // namespace mla
