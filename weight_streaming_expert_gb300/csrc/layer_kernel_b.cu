// layer_kernel_b.cu -- layer kernel instances for hidden = 256 x {8,10,12,16}, plain
// (four translation units so that the instances compile in parallel).
#include "layer_kernel.cuh"

namespace wse {

LayerKernel layer_kernel_plain_large(int kpw) {
  switch (kpw) {
    case 8: return moe_layer_kernel<8, false>;
    case 10: return moe_layer_kernel<10, false>;
    case 12: return moe_layer_kernel<12, false>;
    case 16: return moe_layer_kernel<16, false>;
    default: return nullptr;
  }
}

LayerKernel layer_kernel_plain_small(int kpw);
LayerKernel layer_kernel_variant_small(int kpw);
LayerKernel layer_kernel_variant_large(int kpw);

LayerKernel layer_kernel_for(int kpw, bool variant) {
  if (variant) {
    const LayerKernel k = layer_kernel_variant_large(kpw);
    return k ? k : layer_kernel_variant_small(kpw);
  }
  const LayerKernel k = layer_kernel_plain_large(kpw);
  return k ? k : layer_kernel_plain_small(kpw);
}

}  // namespace wse
