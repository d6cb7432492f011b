// Instantiations of the LoRA kernel, expand mode (token tile x buffer rank).
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
    if (tc && tm == 128 && rmax == 16) return reinterpret_cast<const void *>(lora_tma_kernel<128, 16, kModeExpand, true>);
    if (tc && tm == 128 && rmax == 32) return reinterpret_cast<const void *>(lora_tma_kernel<128, 32, kModeExpand, true>);
    if (tc && tm == 128 && rmax == 64) return reinterpret_cast<const void *>(lora_tma_kernel<128, 64, kModeExpand, true>);
    return nullptr;
}

}  // namespace csgmv
