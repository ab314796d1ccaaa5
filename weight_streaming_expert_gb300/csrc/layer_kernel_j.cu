// layer_kernel_j.cu -- layer kernel instances for hidden = 256 x {8,10,12,16}, plain,
// groups of at most 8 tokens (calls with M <= 8) (one of twelve translation units compiled in parallel).
#include "layer_kernel.cuh"

namespace wse {

LayerKernel layer_kernel_plain_large_tb1(int kpw) {
  switch (kpw) {
    case 8: return moe_layer_kernel<8, false, false, 1>;
    case 10: return moe_layer_kernel<10, false, false, 1>;
    case 12: return moe_layer_kernel<12, false, false, 1>;
    case 16: return moe_layer_kernel<16, false, false, 1>;
    default: return nullptr;
  }
}

}  // namespace wse
