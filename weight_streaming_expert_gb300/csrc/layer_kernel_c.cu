// layer_kernel_c.cu -- layer kernel instances for hidden = 256 x {1,2,4,5}, layer variants
// (one of twelve translation units compiled in parallel).
#include "layer_kernel.cuh"

namespace wse {

LayerKernel layer_kernel_variant_small(int kpw) {
  switch (kpw) {
    case 1: return moe_layer_kernel<1, true, false, 2>;
    case 2: return moe_layer_kernel<2, true, false, 2>;
    case 4: return moe_layer_kernel<4, true, false, 2>;
    case 5: return moe_layer_kernel<5, true, false, 2>;
    default: return nullptr;
  }
}

}  // namespace wse
