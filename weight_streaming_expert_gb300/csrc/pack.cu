// pack.cu -- create-time re-layout of the expert weights for streaming.
//
// "Two fusions and a retune" (SwiGLU in the up-GEMM epilogue) applies a
// per-expert gate/up row interleave at weight load so gate and up land in
// adjacent output columns of one tile.  Here the same load-time pass also
// puts every weight in tensor-core fragment order, so that a warp's
// contiguous 512-byte shared-memory read hands each lane exactly its
// m16n8k16 fragment registers (conflict-free, no ldmatrix, no swizzle) and
// each tile is one contiguous block that a single bulk copy can stage.
//
// Gate/up, per expert e and tile tt (8 rows: gate r, up r for r = 4tt..4tt+3):
//   16-byte chunk (e, tt, q, lane) with g = lane/4, t = lane%4, n = g:
//     source row  = (n even) ? 4tt + n/2 : I + 4tt + n/2
//     elements    = row[32q+2t], [32q+2t+1], [32q+2t+8], [32q+2t+9],
//                   row[32q+16+2t], [+1], [+8], [+9]
//   i.e. the B fragments (k16 x n8, n = tile row) of k-steps 2q and 2q+1.
// Down, per expert e and slab sl (output rows 8sl .. 8sl+7):
//   16-byte chunk (e, sl, q, lane), row = 8sl + g:
//     row[32q+2t], [+1], [+8], [+9], row[32q+16+2t], [+1], [+8], [+9]
//   i.e. the B fragments (k16 x n8, n = output row) of k-steps 2q, 2q+1,
//   the same packing as the gate/up tiles.
#include "kernels.cuh"

namespace wse {

namespace {

__device__ __forceinline__ uint4 pack8(const uint16_t* s, int i0, int i1, int i2, int i3,
                                       const uint16_t* s2, int j0, int j1, int j2, int j3) {
  uint4 v;
  v.x = (uint32_t)s[i0] | ((uint32_t)s[i1] << 16);
  v.y = (uint32_t)s[i2] | ((uint32_t)s[i3] << 16);
  v.z = (uint32_t)s2[j0] | ((uint32_t)s2[j1] << 16);
  v.w = (uint32_t)s2[j2] | ((uint32_t)s2[j3] << 16);
  return v;
}

__global__ void pack_gate_up_kernel(const uint16_t* __restrict__ src, uint4* __restrict__ dst,
                                    int E, int I, int H) {
  const int KP = H / 32, TPG = 2 * I / 8;
  const long long total = (long long)E * TPG * KP * 32;
  for (long long c = (long long)blockIdx.x * blockDim.x + threadIdx.x; c < total;
       c += (long long)gridDim.x * blockDim.x) {
    const int lane = (int)(c & 31);
    long long r = c >> 5;
    const int q = (int)(r % KP);
    r /= KP;
    const int tt = (int)(r % TPG);
    const long long e = r / TPG;
    const int g = lane >> 2, t = lane & 3;
    const int ri = 4 * tt + (g >> 1);
    const int row = (g & 1) ? I + ri : ri;
    const uint16_t* s = src + ((size_t)e * 2 * I + row) * H;
    const int k0 = 32 * q + 2 * t, k1 = k0 + 16;
    // (b0, b1) of k-step 2q, then (b0, b1) of k-step 2q+1
    dst[c] = pack8(s, k0, k0 + 1, k0 + 8, k0 + 9, s, k1, k1 + 1, k1 + 8, k1 + 9);
  }
}

__global__ void pack_down_kernel(const uint16_t* __restrict__ src, uint4* __restrict__ dst, int E,
                                 int H, int I) {
  const int KP = I / 32, SL = H / 8;
  const long long total = (long long)E * SL * KP * 32;
  for (long long c = (long long)blockIdx.x * blockDim.x + threadIdx.x; c < total;
       c += (long long)gridDim.x * blockDim.x) {
    const int lane = (int)(c & 31);
    long long r = c >> 5;
    const int q = (int)(r % KP);
    r /= KP;
    const int sl = (int)(r % SL);
    const long long e = r / SL;
    const int g = lane >> 2, t = lane & 3;
    const uint16_t* s = src + ((size_t)e * H + 8 * sl + g) * I;  // output row 8*sl + g
    const int k0 = 32 * q + 2 * t, k1 = k0 + 16;
    // (b0, b1) of k-step 2q, then (b0, b1) of k-step 2q+1
    dst[c] = pack8(s, k0, k0 + 1, k0 + 8, k0 + 9, s, k1, k1 + 1, k1 + 8, k1 + 9);
  }
}

}  // namespace

void pack_gate_up(const __nv_bfloat16* src, __nv_bfloat16* dst, int E, int I, int H,
                  cudaStream_t s) {
  pack_gate_up_kernel<<<4096, 256, 0, s>>>(reinterpret_cast<const uint16_t*>(src),
                                           reinterpret_cast<uint4*>(dst), E, I, H);
}

void pack_down(const __nv_bfloat16* src, __nv_bfloat16* dst, int E, int H, int I, cudaStream_t s) {
  pack_down_kernel<<<4096, 256, 0, s>>>(reinterpret_cast<const uint16_t*>(src),
                                        reinterpret_cast<uint4*>(dst), E, H, I);
}

}  // namespace wse
