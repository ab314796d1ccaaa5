// layer_kernel_b.cu -- layer kernel instances for hidden = 256 x {8,10,12,16}.
#include "layer_kernel.cuh"

namespace wse {

LayerKernel layer_kernel_small(int kpw);

LayerKernel layer_kernel_for(int kpw) {
  switch (kpw) {
    case 8: return moe_layer_kernel<8>;
    case 10: return moe_layer_kernel<10>;
    case 12: return moe_layer_kernel<12>;
    case 16: return moe_layer_kernel<16>;
    default: return layer_kernel_small(kpw);
  }
}

}  // namespace wse
