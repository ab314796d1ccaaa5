// layer_kernel_e.cu -- layer kernel instances for hidden = 256 x {1,2,4,5}, fp8 expert weights,
// groups of up to 16 tokens (one of twelve translation units compiled in parallel).
#include "layer_kernel.cuh"

namespace wse {

LayerKernel layer_kernel_fp8_small(int kpw) {
  switch (kpw) {
    case 1: return moe_layer_kernel<1, false, true, 2>;
    case 2: return moe_layer_kernel<2, false, true, 2>;
    case 4: return moe_layer_kernel<4, false, true, 2>;
    case 5: return moe_layer_kernel<5, false, true, 2>;
    default: return nullptr;
  }
}

}  // namespace wse
