// HBM-bound kernels of the FP8 FFN backward (llmq "llama_model.cpp",
// _backward_block and the FP8 branch of backward_qmm):
//
//   transpose_u8_kernel      E4M3 matrix transpose: the page's backward_qmm
//                            transposes the weight for the input gradient and
//                            both quantised operands of the weight gradient so
//                            that every matmul is K-contiguous.  The library's
//                            backward reads those operands MN-major in the
//                            GEMM instead; the transpose stays available.
//   swiglu_backward_kernel   gradient of h = silu(g) * u w.r.t. the fused
//                            gate|up output, with its tensor abs-max.
#include "common.cuh"
#include "launch.h"

namespace qffn {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 64;          // bytes x rows of one transpose tile
constexpr int kPitch = kTile + 4;  // shared row pitch: column reads hit distinct banks

// out[Cc, R] = in[R, Cc]^T, bytes.  R and Cc are multiples of 16, so every
// 16-byte row segment a thread moves is either wholly inside or wholly
// outside the matrix.  Each thread loads 16 bytes of one input row of the
// tile, then writes 16 bytes of one output row (16 input rows of one column).
__global__ void __launch_bounds__(kThreads) transpose_u8_kernel(uint8_t* out, const uint8_t* in,
                                                                int64_t R, int64_t Cc) {
  __shared__ __align__(16) uint8_t t[kTile * kPitch];
  const int64_t r0 = int64_t(blockIdx.y) * kTile, c0 = int64_t(blockIdx.x) * kTile;
  {
    const int lr = threadIdx.x >> 2, lc = (threadIdx.x & 3) * 16;
    const int64_t gr = r0 + lr, gc = c0 + lc;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (gr < R && gc < Cc) v = ld16_ro(in + gr * Cc + gc);
    uint32_t* d = reinterpret_cast<uint32_t*>(t + lr * kPitch + lc);
    d[0] = v.x; d[1] = v.y; d[2] = v.z; d[3] = v.w;
  }
  __syncthreads();
  {
    const int oc = threadIdx.x >> 2, orr = (threadIdx.x & 3) * 16;   // output row, first column
    const int64_t gr = c0 + oc, gc = r0 + orr;
    if (gr < Cc && gc < R) {
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint8_t* s = t + (orr + 4 * q) * kPitch + oc;
        w[q] = uint32_t(s[0]) | (uint32_t(s[kPitch]) << 8) | (uint32_t(s[2 * kPitch]) << 16) |
               (uint32_t(s[3 * kPitch]) << 24);
      }
      stg16(out + gr * R + gc, make_uint4(w[0], w[1], w[2], w[3]));
    }
  }
}

QFFN_DEVI float absmax8(uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float m = 0.0f;
#pragma unroll
  for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
  return m;
}

// 8 elements of h per thread per step: 16 bytes each of dh, g and u in, 16
// bytes each of dg and du out.
__global__ void __launch_bounds__(kThreads) swiglu_backward_kernel(uint16_t* dgu, float* stats,
                                                                   const uint16_t* dh,
                                                                   const uint16_t* gu, int64_t N,
                                                                   int64_t H) {
  __shared__ float red[kThreads / 32];
  const int64_t per_row = H >> 3;
  const int64_t total = N * per_row;
  float m = 0.0f;
  for (int64_t i = int64_t(blockIdx.x) * kThreads + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * kThreads) {
    const int64_t row = i / per_row, c = i - row * per_row;
    const uint16_t* src = gu + row * 2 * H + c * 8;
    const uint4 g8 = ld16_ro_stream(src), u8 = ld16_ro_stream(src + H);
    const uint4 d8 = ld16_ro_stream(dh + row * H + c * 8);
    const uint32_t gw[4] = {g8.x, g8.y, g8.z, g8.w}, uw[4] = {u8.x, u8.y, u8.z, u8.w},
                   dw[4] = {d8.x, d8.y, d8.z, d8.w};
    uint32_t og[4], ou[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float dg0, du0, dg1, du1;
      swiglu_grad(bf16_lo(gw[j]), bf16_lo(uw[j]), bf16_lo(dw[j]), dg0, du0);
      swiglu_grad(bf16_hi(gw[j]), bf16_hi(uw[j]), bf16_hi(dw[j]), dg1, du1);
      og[j] = pack_bf16x2(dg0, dg1);
      ou[j] = pack_bf16x2(du0, du1);
    }
    const uint4 vg = make_uint4(og[0], og[1], og[2], og[3]);
    const uint4 vu = make_uint4(ou[0], ou[1], ou[2], ou[3]);
    m = fmaxf(m, fmaxf(absmax8(vg), absmax8(vu)));
    uint16_t* dst = dgu + row * 2 * H + c * 8;
    stg16(dst, vg);
    stg16(dst + H, vu);
  }
  m = warp_max(m);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = m;
  __syncthreads();
  if (warp == 0) {
    float r = lane < kThreads / 32 ? red[lane] : 0.0f;
    r = warp_max(r);
    if (lane == 0) atomic_max_nonneg(stats, r);
  }
}

}  // namespace

cudaError_t launch_transpose_u8(uint8_t* out, const uint8_t* in, int64_t R, int64_t Cc,
                                cudaStream_t s) {
  if (R == 0 || Cc == 0) return cudaSuccess;
  const dim3 grid(unsigned((Cc + kTile - 1) / kTile), unsigned((R + kTile - 1) / kTile));
  transpose_u8_kernel<<<grid, kThreads, 0, s>>>(out, in, R, Cc);
  return cudaGetLastError();
}

cudaError_t launch_swiglu_backward(uint16_t* dgu, float* stats, const uint16_t* dh,
                                   const uint16_t* gu, int64_t N, int64_t H, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(stats, 0, sizeof(float), s);
  if (e != cudaSuccess || N == 0) return e;
  int64_t blocks = (N * (H / 8) + kThreads - 1) / kThreads;
  const int64_t cap = int64_t(num_sms()) * 8;
  if (blocks > cap) blocks = cap;
  swiglu_backward_kernel<<<unsigned(blocks), kThreads, 0, s>>>(dgu, stats, dh, gu, N, H);
  return cudaGetLastError();
}

}  // namespace qffn
