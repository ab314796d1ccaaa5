// layer_kernel_a.cu -- layer kernel instances for hidden = 256 x {1,2,4,5}, plain
// (one of twelve translation units compiled in parallel).
#include "layer_kernel.cuh"

namespace wse {

LayerKernel layer_kernel_plain_small(int kpw) {
  switch (kpw) {
    case 1: return moe_layer_kernel<1, false, false, 2>;
    case 2: return moe_layer_kernel<2, false, false, 2>;
    case 4: return moe_layer_kernel<4, false, false, 2>;
    case 5: return moe_layer_kernel<5, false, false, 2>;
    default: return nullptr;
  }
}

size_t layer_smem_bytes(uint32_t ring_bytes, int NP, int E) {
  return layer_detail::kRingOff + (size_t)ring_bytes + routing_smem_bytes(NP, E);
}

uint32_t layer_reduction_bytes(bool fp8, int token_blocks) {
  return layer_detail::kRedBytes * (fp8 && token_blocks == 2 ? 2u : 1u);
}

}  // namespace wse
