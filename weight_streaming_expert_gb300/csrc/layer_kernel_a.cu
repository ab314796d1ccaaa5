// layer_kernel_a.cu -- layer kernel instances for hidden = 256 x {1,2,4,5}
// (split from layer_kernel_b.cu so the two compile in parallel).
#include "layer_kernel.cuh"

namespace wse {

LayerKernel layer_kernel_small(int kpw) {
  switch (kpw) {
    case 1: return moe_layer_kernel<1>;
    case 2: return moe_layer_kernel<2>;
    case 4: return moe_layer_kernel<4>;
    case 5: return moe_layer_kernel<5>;
    default: return nullptr;
  }
}

size_t layer_smem_bytes(uint32_t ring_bytes, int NP, int E) {
  return layer_detail::kRingOff + (size_t)ring_bytes + routing_smem_bytes(NP, E);
}

uint32_t layer_reduction_bytes() { return layer_detail::kRedBytes; }

}  // namespace wse
