// layer_kernel_f.cu -- layer kernel instances for hidden = 256 x {8,10,12,16}, fp8 expert weights,
// groups of up to 16 tokens (one of twelve translation units compiled in parallel).
#include "layer_kernel.cuh"

namespace wse {

LayerKernel layer_kernel_fp8_large(int kpw) {
  switch (kpw) {
    case 8: return moe_layer_kernel<8, false, true, 2>;
    case 10: return moe_layer_kernel<10, false, true, 2>;
    case 12: return moe_layer_kernel<12, false, true, 2>;
    case 16: return moe_layer_kernel<16, false, true, 2>;
    default: return nullptr;
  }
}

}  // namespace wse
