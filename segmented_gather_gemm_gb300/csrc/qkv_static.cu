// csgmv_qkv for callers that cannot allocate device memory at call time (see
// the declaration in csgmv.h): the h workspace of the two-kernel path is a
// fixed array in the library's own device memory instead of a caller buffer.
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "csgmv_internal.h"

namespace {

// 32 MiB of fp32 h: prefill batches up to max_tokens * c * R = 8 Mi values
// (e.g. 65536 tokens with c = 2 and R = 64).  Every GPU that loads the
// library holds this array until the process exits.
constexpr size_t kStaticScratchFloats = (size_t)8 << 20;
static __device__ __align__(256) float g_qkv_scratch[kStaticScratchFloats];

std::mutex g_mu;
void *g_addr[64];  // device address of g_qkv_scratch per device, once resolved

// The device address of the array on the current device.  Host code only
// has a stand-in symbol for it, so the address is asked from the runtime
// once per device (this can load the module; hence the first call on a
// device belongs before any stream capture).
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_qkv_scratch);
        if (e != cudaSuccess) return e;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" CSGMV_API int csgmv_qkv_static_scratch(const void *x, int64_t K, const void *A, const void *B, int64_t N,
                                                  const int32_t *slice_offsets, int num_slices, int max_slice_size,
                                                  void *base_output, const csgmv_batch_info *bi,
                                                  csgmv_stream_t stream) {
    if (!bi) return csgmv_qkv(x, K, A, B, N, slice_offsets, num_slices, max_slice_size, base_output, nullptr, 0,
                              bi, stream);  // reports the missing batch info
    const size_t need = csgmv::kWsHeader + (size_t)(bi->num_tokens > 0 ? bi->num_tokens : 0) *
                                               (size_t)(num_slices > 0 ? num_slices : 0) *
                                               (size_t)(bi->max_rank > 0 ? bi->max_rank : 0) * 4;
    if (need > kStaticScratchFloats * 4) {
        // a batch whose h does not fit may still take the one-kernel path,
        // which needs no workspace at all
        const int path = csgmv_qkv_path(bi, K, N, slice_offsets, num_slices, SIZE_MAX);
        if (path == CSGMV_PATH_FUSED || path < 0)  // (errors: csgmv_qkv reports them)
            return csgmv_qkv(x, K, A, B, N, slice_offsets, num_slices, max_slice_size, base_output, nullptr, 0, bi,
                             stream);
        char msg[160];
        snprintf(msg, sizeof msg, "csgmv_qkv_static_scratch: h needs %zu bytes, the static scratch holds %zu",
                 need, kStaticScratchFloats * 4);
        return csgmv::set_error(CSGMV_ERR_CAPACITY, msg);
    }
    void *scratch = nullptr;
    const cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) {
        char msg[160];
        snprintf(msg, sizeof msg, "csgmv_qkv_static_scratch: scratch address: %s", cudaGetErrorName(e));
        return csgmv::set_error(CSGMV_ERR_CUDA, msg);
    }
    return csgmv_qkv(x, K, A, B, N, slice_offsets, num_slices, max_slice_size, base_output, scratch,
                     kStaticScratchFloats * 4, bi, stream);
}
