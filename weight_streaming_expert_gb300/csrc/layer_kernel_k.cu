// layer_kernel_k.cu -- layer kernel instances for hidden = 256 x {1,2,4,5}, layer variants,
// groups of at most 8 tokens (calls with M <= 8) (one of twelve translation units compiled in parallel).
#include "layer_kernel.cuh"

namespace wse {

LayerKernel layer_kernel_variant_small_tb1(int kpw) {
  switch (kpw) {
    case 1: return moe_layer_kernel<1, true, false, 1>;
    case 2: return moe_layer_kernel<2, true, false, 1>;
    case 4: return moe_layer_kernel<4, true, false, 1>;
    case 5: return moe_layer_kernel<5, true, false, 1>;
    default: return nullptr;
  }
}

}  // namespace wse
