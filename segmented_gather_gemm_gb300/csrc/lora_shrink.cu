// Instantiations of the LoRA kernel, shrink mode (token tile x buffer rank).
#include "lora_tma.cuh"

namespace csgmv {

const void *lora_kernel_shrink(int tm, int rmax, bool tc) {
#define CSGMV_K(TM_, R_) \
    if (!tc && tm == TM_ && rmax == R_) return reinterpret_cast<const void *>(lora_tma_kernel<TM_, R_, kModeShrink, false>);
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
