// layer_kernel_c.cu -- layer kernel instances for hidden = 256 x {1,2,4,5}, layer variants
// (four translation units so that the instances compile in parallel).
#include "layer_kernel.cuh"

namespace wse {

LayerKernel layer_kernel_variant_small(int kpw) {
  switch (kpw) {
    case 1: return moe_layer_kernel<1, true>;
    case 2: return moe_layer_kernel<2, true>;
    case 4: return moe_layer_kernel<4, true>;
    case 5: return moe_layer_kernel<5, true>;
    default: return nullptr;
  }
}

}  // namespace wse
