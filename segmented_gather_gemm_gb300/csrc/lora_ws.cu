// Instantiations of the warp-specialized tcgen05 LoRA kernel (128-token
// tiles) per mode and buffer rank.
#include "lora_ws.cuh"

namespace csgmv {

const void *lora_kernel_ws(int mode, int rmax) {
#define CSGMV_K(M_, R_) \
    if (mode == M_ && rmax == R_) return reinterpret_cast<const void *>(lora_ws_kernel<R_, M_>);
    CSGMV_K(kModeFused, 16)
    CSGMV_K(kModeFused, 32)
    CSGMV_K(kModeFused, 64)
    CSGMV_K(kModeShrink, 16)
    CSGMV_K(kModeShrink, 32)
    CSGMV_K(kModeShrink, 64)
    CSGMV_K(kModeExpand, 16)
    CSGMV_K(kModeExpand, 32)
    CSGMV_K(kModeExpand, 64)
#undef CSGMV_K
    return nullptr;
}

}  // namespace csgmv
