// layer_kernel_i.cu -- layer kernel instances for hidden = 256 x {1,2,4,5}, plain,
// groups of at most 8 tokens (calls with M <= 8) (one of twelve translation units compiled in parallel).
#include "layer_kernel.cuh"

namespace wse {

LayerKernel layer_kernel_plain_small_tb1(int kpw) {
  switch (kpw) {
    case 1: return moe_layer_kernel<1, false, false, 1>;
    case 2: return moe_layer_kernel<2, false, false, 1>;
    case 4: return moe_layer_kernel<4, false, false, 1>;
    case 5: return moe_layer_kernel<5, false, false, 1>;
    default: return nullptr;
  }
}

}  // namespace wse
