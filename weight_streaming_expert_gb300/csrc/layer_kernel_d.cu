// layer_kernel_d.cu -- layer kernel instances for hidden = 256 x {8,10,12,16}, layer variants
// (one of twelve translation units compiled in parallel).
#include "layer_kernel.cuh"

namespace wse {

LayerKernel layer_kernel_variant_large(int kpw) {
  switch (kpw) {
    case 8: return moe_layer_kernel<8, true, false, 2>;
    case 10: return moe_layer_kernel<10, true, false, 2>;
    case 12: return moe_layer_kernel<12, true, false, 2>;
    case 16: return moe_layer_kernel<16, true, false, 2>;
    default: return nullptr;
  }
}

}  // namespace wse
