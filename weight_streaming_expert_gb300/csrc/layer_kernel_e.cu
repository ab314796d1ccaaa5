// layer_kernel_e.cu -- layer kernel instances for hidden = 256 x {1,2,4,5}, fp8 expert weights
// (one of six translation units compiled in parallel).
#include "layer_kernel.cuh"

namespace wse {

LayerKernel layer_kernel_fp8_small(int kpw) {
  switch (kpw) {
    case 1: return moe_layer_kernel<1, false, true>;
    case 2: return moe_layer_kernel<2, false, true>;
    case 4: return moe_layer_kernel<4, false, true>;
    case 5: return moe_layer_kernel<5, false, true>;
    default: return nullptr;
  }
}

}  // namespace wse
