// Instantiations of the small-tile (decode) LoRA kernel per mode, token tile
// and buffer rank.
#include "lora_small.cuh"

namespace csgmv {

const void *lora_kernel_small(int mode, int tm, int rmax) {
#define CSGMV_K(M_, TM_, R_) \
    if (mode == M_ && tm == TM_ && rmax == R_) return reinterpret_cast<const void *>(lora_small_kernel<TM_, R_, M_>);
#define CSGMV_KM(M_) \
    CSGMV_K(M_, 16, 16) CSGMV_K(M_, 16, 32) CSGMV_K(M_, 16, 64) CSGMV_K(M_, 32, 16) CSGMV_K(M_, 32, 32) CSGMV_K(M_, 32, 64)
    CSGMV_KM(kModeFused)
    CSGMV_KM(kModeShrink)
    CSGMV_KM(kModeExpand)
#undef CSGMV_KM
#undef CSGMV_K
    return nullptr;
}

}  // namespace csgmv
