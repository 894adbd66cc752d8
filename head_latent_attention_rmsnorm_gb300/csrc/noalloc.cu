// noalloc.cu -- mla_decode_splitkv_noalloc: the split-KV decode for callers that
// cannot allocate device memory (stream capture into a CUDA graph refuses
// cudaMalloc; some host runtimes own all device memory and hand their plugins no
// allocator).  Its scratch is one fixed file-scope device array; the call runs the
// ordinary decode entry point with that array as the workspace.
#include <mutex>

#include "mla.h"

namespace {

constexpr int MAX_DEVICES = 64;

// The scratch itself.  Every GPU that loads the library holds it until exit.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MLA_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
void *g_addr[MAX_DEVICES] = {};

// Device address of the scratch on the current device.  In host code the array's
// name is only a stand-in, so the address comes from cudaGetSymbolAddress.  It is looked
// up on every call made outside stream capture (so a context torn down and created again
// after a device reset gets the address in the new context) and remembered per device;
// a call made while `st` is capturing uses the remembered address, and looks it up only
// if it has none yet.
mla_status scratch_address(void **out, cudaStream_t st) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return MLA_ERR_CUDA;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) return MLA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (cap == cudaStreamCaptureStatusNone || !g_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MLA_ERR_CUDA;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return MLA_OK;
}

}  // namespace

extern "C" mla_status mla_decode_splitkv_noalloc(const mla_dims *dims, mla_dtype dtype, int B, int kv_len,
                                                 int n_splits, const void *q_nope, const void *q_pe,
                                                 const void *c_cache, const void *kpe_cache, const void *w_kv_b,
                                                 void *out, float *lse, void *cuda_stream) {
    if (!dims) return MLA_ERR_NULL;
    size_t need = mla_decode_workspace(dims, dtype, B, kv_len, n_splits);
    if (need == 0)   // invalid arguments or B == 0: the ordinary entry point names the outcome
        return mla_decode_splitkv(dims, dtype, B, kv_len, n_splits, q_nope, q_pe, c_cache, kpe_cache, w_kv_b,
                                  out, lse, nullptr, nullptr, nullptr, 0, cuda_stream);
    if (need > MLA_NOALLOC_SCRATCH_BYTES) return MLA_ERR_WORKSPACE;
    void *scratch = nullptr;
    mla_status st = scratch_address(&scratch, (cudaStream_t)cuda_stream);
    if (st != MLA_OK) return st;
    return mla_decode_splitkv(dims, dtype, B, kv_len, n_splits, q_nope, q_pe, c_cache, kpe_cache, w_kv_b, out,
                              lse, nullptr, nullptr, scratch, MLA_NOALLOC_SCRATCH_BYTES, cuda_stream);
}
