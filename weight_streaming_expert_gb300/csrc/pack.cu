// pack.cu -- create-time re-layout of the expert weights for streaming.
//
// "Two fusions and a retune" (SwiGLU in the up-GEMM epilogue) applies a
// per-expert gate/up row interleave at weight load so gate and up land in
// adjacent output columns of one tile.  Here the same load-time pass also
// makes every tile one contiguous block (one bulk copy) in tensor-core
// fragment order, so that a warp's contiguous 512-byte shared-memory read
// hands each lane exactly its m16n8k16 B registers (conflict-free).
//
// Fragment order.  Inside every 32-wide k chunk the MMA's logical k order is
// permuted so that lane (g, t) = (lane / 4, lane % 4) owns physical k =
// 8t .. 8t+7 of its row: logical (2t, 2t+1 | 2t+8, 2t+9) of k-step 0 are
// physical 8t + (0,1 | 2,3) and those of k-step 1 are 8t + (4,5 | 6,7).  The
// activations use the same permutation (a lane loads 16 contiguous bytes of
// a token row), which leaves every dot product unchanged.  So a lane's 16
// bytes of chunk q are simply row[32q + 8t .. 32q + 8t + 7] of the tile row
// n = g it serves:
//   gate/up tile (e, tt), 8 rows: n even -> gate row 4tt + n/2,
//                                 n odd  -> up row   4tt + n/2
//   down tile (e, sl), 8 rows: output rows 8sl .. 8sl + 7
// 16-byte chunk (tile, q, lane) sits at ((tile * H/32 + q) * 32 + lane) for
// gate/up (k = H) and ((tile * I/32 + q) * 32 + lane) for down (k = I).
//
// E4M3 codes (one byte each): tiles of 16 rows, the same bytes as 8 bf16
// rows, which are the 16 rows of the MMA's A operand (the tokens are B).
// A tile is two 8-row blocks; lane (g, t)'s 16-byte chunk q holds the codes
// of block 0's row g at k = 32q + 8t .. +7, then those of block 1's row g --
// the lane's A registers for rows g and g + 8:
//   gate/up tile (e, tt): block 0 row n = gate row 8tt + n,
//                         block 1 row n = up row   8tt + n
//     (so one lane's accumulators hold the gate and the up value of one
//     intermediate row: SwiGLU needs no exchange between lanes)
//   down slab (e, sl), block b: output rows 16sl + 8b .. 16sl + 8b + 7
#include "kernels.cuh"

namespace wse {

namespace {

__global__ void pack_gate_up_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int E,
                                    int I, int H) {
  const int KC = H / 32, TPG = 2 * I / 8, RC = H / 8;  // RC: 16-byte chunks per source row
  const long long total = (long long)E * TPG * KC * 32;
  for (long long c = (long long)blockIdx.x * blockDim.x + threadIdx.x; c < total;
       c += (long long)gridDim.x * blockDim.x) {
    const int lane = (int)(c & 31);
    long long r = c >> 5;
    const int q = (int)(r % KC);
    r /= KC;
    const int tt = (int)(r % TPG);
    const long long e = r / TPG;
    const int g = lane >> 2, t = lane & 3;
    const int ri = 4 * tt + (g >> 1);
    const int row = (g & 1) ? I + ri : ri;
    dst[c] = src[((size_t)e * 2 * I + row) * RC + 4 * q + t];
  }
}

__global__ void pack_down_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int E, int H,
                                 int I) {
  const int KC = I / 32, SL = H / 8, RC = I / 8;
  const long long total = (long long)E * SL * KC * 32;
  for (long long c = (long long)blockIdx.x * blockDim.x + threadIdx.x; c < total;
       c += (long long)gridDim.x * blockDim.x) {
    const int lane = (int)(c & 31);
    long long r = c >> 5;
    const int q = (int)(r % KC);
    r /= KC;
    const int sl = (int)(r % SL);
    const long long e = r / SL;
    const int g = lane >> 2, t = lane & 3;
    dst[c] = src[((size_t)e * H + 8 * sl + g) * RC + 4 * q + t];
  }
}

__global__ void pack_gate_up_fp8_kernel(const uint2* __restrict__ src, uint4* __restrict__ dst, int E, int I,
                                        int H) {
  const int KC = H / 32, TPG = 2 * I / 16, RC = H / 8;  // RC: 8-byte chunks per source row
  const long long total = (long long)E * TPG * KC * 32;
  for (long long c = (long long)blockIdx.x * blockDim.x + threadIdx.x; c < total;
       c += (long long)gridDim.x * blockDim.x) {
    const int lane = (int)(c & 31);
    long long r = c >> 5;
    const int q = (int)(r % KC);
    r /= KC;
    const int tt = (int)(r % TPG);
    const long long e = r / TPG;
    const int g = lane >> 2, t = lane & 3;
    uint2 v[2];
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const int row = (b ? I : 0) + 8 * tt + g;  // gate rows, then the same up rows
      v[b] = src[((size_t)e * 2 * I + row) * RC + 4 * q + t];
    }
    dst[c] = make_uint4(v[0].x, v[0].y, v[1].x, v[1].y);
  }
}

__global__ void pack_down_fp8_kernel(const uint2* __restrict__ src, uint4* __restrict__ dst, int E, int H,
                                     int I) {
  const int KC = I / 32, SL = H / 16, RC = I / 8;
  const long long total = (long long)E * SL * KC * 32;
  for (long long c = (long long)blockIdx.x * blockDim.x + threadIdx.x; c < total;
       c += (long long)gridDim.x * blockDim.x) {
    const int lane = (int)(c & 31);
    long long r = c >> 5;
    const int q = (int)(r % KC);
    r /= KC;
    const int sl = (int)(r % SL);
    const long long e = r / SL;
    const int g = lane >> 2, t = lane & 3;
    const uint2 v0 = src[((size_t)e * H + 16 * sl + g) * RC + 4 * q + t];
    const uint2 v1 = src[((size_t)e * H + 16 * sl + 8 + g) * RC + 4 * q + t];
    dst[c] = make_uint4(v0.x, v0.y, v1.x, v1.y);
  }
}

}  // namespace

void pack_gate_up(const __nv_bfloat16* src, __nv_bfloat16* dst, int E, int I, int H,
                  cudaStream_t s) {
  pack_gate_up_kernel<<<4096, 256, 0, s>>>(reinterpret_cast<const uint4*>(src),
                                           reinterpret_cast<uint4*>(dst), E, I, H);
}

void pack_down(const __nv_bfloat16* src, __nv_bfloat16* dst, int E, int H, int I, cudaStream_t s) {
  pack_down_kernel<<<4096, 256, 0, s>>>(reinterpret_cast<const uint4*>(src),
                                        reinterpret_cast<uint4*>(dst), E, H, I);
}

void pack_gate_up_fp8(const uint8_t* src, uint8_t* dst, int E, int I, int H, cudaStream_t s) {
  pack_gate_up_fp8_kernel<<<4096, 256, 0, s>>>(reinterpret_cast<const uint2*>(src), reinterpret_cast<uint4*>(dst),
                                               E, I, H);
}

void pack_down_fp8(const uint8_t* src, uint8_t* dst, int E, int H, int I, cudaStream_t s) {
  pack_down_fp8_kernel<<<4096, 256, 0, s>>>(reinterpret_cast<const uint2*>(src), reinterpret_cast<uint4*>(dst),
                                            E, H, I);
}

}  // namespace wse
