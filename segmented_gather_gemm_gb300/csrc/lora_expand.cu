// Instantiations of the LoRA kernel, expand mode (token tile x buffer rank).
// Expand-only calls on 128-token tiles with R >= 16 run on the streaming
// tcgen05 expand (lora_stream.cu) instead.
#include "lora_tma.cuh"

namespace csgmv {

const void *lora_kernel_expand(int tm, int rmax, bool tc) {
#define CSGMV_K(TM_, R_) \
    if (!tc && tm == TM_ && rmax == R_) return reinterpret_cast<const void *>(lora_tma_kernel<TM_, R_, kModeExpand, false>);
    CSGMV_K(16, 16)
    CSGMV_K(16, 32)
    CSGMV_K(16, 64)
    CSGMV_K(32, 16)
    CSGMV_K(32, 32)
    CSGMV_K(32, 64)
    CSGMV_K(128, 16)
    CSGMV_K(128, 32)
    CSGMV_K(128, 64)
#undef CSGMV_K
    return nullptr;
}

}  // namespace csgmv
