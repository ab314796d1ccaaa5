// layer_kernel_b.cu -- layer kernel instances for hidden = 256 x {8,10,12,16}, plain
// (one of twelve translation units compiled in parallel).
#include "layer_kernel.cuh"

namespace wse {

LayerKernel layer_kernel_plain_large(int kpw) {
  switch (kpw) {
    case 8: return moe_layer_kernel<8, false, false, 2>;
    case 10: return moe_layer_kernel<10, false, false, 2>;
    case 12: return moe_layer_kernel<12, false, false, 2>;
    case 16: return moe_layer_kernel<16, false, false, 2>;
    default: return nullptr;
  }
}

LayerKernel layer_kernel_plain_small(int kpw);
LayerKernel layer_kernel_variant_small(int kpw);
LayerKernel layer_kernel_variant_large(int kpw);
LayerKernel layer_kernel_fp8_small(int kpw);
LayerKernel layer_kernel_fp8_large(int kpw);
LayerKernel layer_kernel_fp8_small_tb1(int kpw);
LayerKernel layer_kernel_fp8_large_tb1(int kpw);
LayerKernel layer_kernel_plain_small_tb1(int kpw);
LayerKernel layer_kernel_plain_large_tb1(int kpw);
LayerKernel layer_kernel_variant_small_tb1(int kpw);
LayerKernel layer_kernel_variant_large_tb1(int kpw);

LayerKernel layer_kernel_for(int kpw, bool variant, bool fp8, int token_blocks) {
  if (fp8) {
    if (variant) return nullptr;  // fp8 experts: plain layers only
    if (token_blocks == 1) {
      const LayerKernel k = layer_kernel_fp8_large_tb1(kpw);
      return k ? k : layer_kernel_fp8_small_tb1(kpw);
    }
    const LayerKernel k = layer_kernel_fp8_large(kpw);
    return k ? k : layer_kernel_fp8_small(kpw);
  }
  if (variant) {
    if (token_blocks == 1) {
      const LayerKernel k = layer_kernel_variant_large_tb1(kpw);
      return k ? k : layer_kernel_variant_small_tb1(kpw);
    }
    const LayerKernel k = layer_kernel_variant_large(kpw);
    return k ? k : layer_kernel_variant_small(kpw);
  }
  if (token_blocks == 1) {
    const LayerKernel k = layer_kernel_plain_large_tb1(kpw);
    return k ? k : layer_kernel_plain_small_tb1(kpw);
  }
  const LayerKernel k = layer_kernel_plain_large(kpw);
  return k ? k : layer_kernel_plain_small(kpw);
}

}  // namespace wse
