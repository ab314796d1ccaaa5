// layer_kernel_f.cu -- layer kernel instances for hidden = 256 x {8,10,12,16}, fp8 expert weights
// (one of six translation units compiled in parallel).
#include "layer_kernel.cuh"

namespace wse {

LayerKernel layer_kernel_fp8_large(int kpw) {
  switch (kpw) {
    case 8: return moe_layer_kernel<8, false, true>;
    case 10: return moe_layer_kernel<10, false, true>;
    case 12: return moe_layer_kernel<12, false, true>;
    case 16: return moe_layer_kernel<16, false, true>;
    default: return nullptr;
  }
}

}  // namespace wse
