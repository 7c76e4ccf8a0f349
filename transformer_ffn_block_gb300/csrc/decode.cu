// Row-scaled W8A16 GEMVs of the single-token FP8 decode FFN (metrale
// "dense_ffn_decode.rs", DenseFfnLayer::forward, FP8 arm: w8a16_gemv_dual
// for gate and up, w8a16_gemv for down).
//
// out[r] = bf16(row_scale[r] * sum_k W[r,k] * x[k]),  W E4M3, x bf16.
//
// The kernel streams the weight matrix once from HBM with 16-byte
// non-allocating loads; x sits in shared memory.  TPR threads share a row:
// each owns the 16-byte weight chunks t, t+TPR, ... and keeps up to U chunk
// loads (per matrix) in flight before using them.  The dual form reads x
// once for the gate and the up row of the same index.  The per-row
// arithmetic (chunk order, fma order, reduction tree) is the same code in the
// single and dual forms, so their results agree bit for bit.
#include "common.cuh"
#include "launch.h"

namespace qffn {
namespace {

constexpr int kThreads = 256;
constexpr int kU = 8;

// acc += sum of the 16 products of one weight chunk with its 16 x values
// (x as 16 bf16 in two uint4), in element order.
QFFN_DEVI float dot16(uint4 w, uint4 xa, uint4 xb, float acc) {
  const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
  const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float f0, f1, f2, f3;
    e4m3x4_to_f32(ww[j], f0, f1, f2, f3);
    acc = fmaf(f0, bf16_lo(xw[2 * j]), acc);
    acc = fmaf(f1, bf16_hi(xw[2 * j]), acc);
    acc = fmaf(f2, bf16_lo(xw[2 * j + 1]), acc);
    acc = fmaf(f3, bf16_hi(xw[2 * j + 1]), acc);
  }
  return acc;
}

template <bool DUAL, int TPR>
__global__ void __launch_bounds__(kThreads) gemv_kernel(uint16_t* out0, uint16_t* out1,
                                                        const uint16_t* x, const uint8_t* w0,
                                                        const float* s0, const uint8_t* w1,
                                                        const float* s1, int rows, int cols) {
  extern __shared__ uint4 xs[];
  __shared__ float red[2][kThreads / 32];
  constexpr int RPB = kThreads / TPR;   // rows per block step
  constexpr int WPR = TPR / 32;         // warps per row

  pdl_wait();       // x may come from the preceding kernel
  pdl_trigger();
  const int nvec = cols >> 3;
  for (int i = threadIdx.x; i < nvec; i += kThreads) xs[i] = ld16_once(x + size_t(i) * 8);
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = threadIdx.x / TPR, t = threadIdx.x % TPR;
  const int nchunk = cols >> 4;
  for (int base = blockIdx.x * RPB; base < rows; base += gridDim.x * RPB) {
    const int row = base + sub;
    float acc0 = 0.0f, acc1 = 0.0f;
    if (row < rows) {
      const uint8_t* r0 = w0 + size_t(row) * size_t(cols);
      const uint8_t* r1 = DUAL ? w1 + size_t(row) * size_t(cols) : nullptr;
      for (int c = t; c < nchunk; c += TPR * kU) {
        uint4 a[kU], b[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int cc = c + TPR * u;
          if (cc < nchunk) {
            a[u] = ld16_ro_stream(r0 + size_t(cc) * 16);
            if (DUAL) b[u] = ld16_ro_stream(r1 + size_t(cc) * 16);
          }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int cc = c + TPR * u;
          if (cc < nchunk) {
            const uint4 xa = xs[2 * cc], xb = xs[2 * cc + 1];
            acc0 = dot16(a[u], xa, xb, acc0);
            if (DUAL) acc1 = dot16(b[u], xa, xb, acc1);
          }
        }
      }
    }
    acc0 = warp_sum(acc0);
    if (DUAL) acc1 = warp_sum(acc1);
    if (WPR > 1) {
      if (lane == 0) {
        red[0][warp] = acc0;
        red[1][warp] = acc1;
      }
      __syncthreads();
      if (t == 0) {
        float s = 0.0f, s1v = 0.0f;
        for (int w = 0; w < WPR; ++w) {
          s += red[0][warp + w];
          s1v += red[1][warp + w];
        }
        acc0 = s;
        acc1 = s1v;
      }
      __syncthreads();
    }
    if (t == 0 && row < rows) {
      out0[row] = f32_to_bf16(s0[row] * acc0);
      if (DUAL) out1[row] = f32_to_bf16(s1[row] * acc1);
    }
  }
}

template <bool DUAL, int TPR>
cudaError_t launch_t(uint16_t* out0, uint16_t* out1, const uint16_t* x, const uint8_t* w0,
                     const float* s0, const uint8_t* w1, const float* s1, int rows, int cols,
                     bool pdl, cudaStream_t s) {
  const size_t smem = size_t(cols) * 2;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(gemv_kernel<DUAL, TPR>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
  }
  constexpr int RPB = kThreads / TPR;
  const int blocks_needed = (rows + RPB - 1) / RPB;
  const int cap = num_sms() * 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks_needed < cap ? blocks_needed : cap);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemv_kernel<DUAL, TPR>, out0, out1, x, w0, s0, w1, s1, rows,
                            cols);
}

template <bool DUAL>
cudaError_t launch_d(uint16_t* out0, uint16_t* out1, const uint16_t* x, const uint8_t* w0,
                     const float* s0, const uint8_t* w1, const float* s1, int rows, int cols,
                     bool pdl, cudaStream_t s) {
  const int nchunk = cols / 16;
  if (nchunk <= 32 * kU) return launch_t<DUAL, 32>(out0, out1, x, w0, s0, w1, s1, rows, cols, pdl, s);
  if (nchunk <= 64 * kU) return launch_t<DUAL, 64>(out0, out1, x, w0, s0, w1, s1, rows, cols, pdl, s);
  if (nchunk <= 128 * kU) return launch_t<DUAL, 128>(out0, out1, x, w0, s0, w1, s1, rows, cols, pdl, s);
  return launch_t<DUAL, 256>(out0, out1, x, w0, s0, w1, s1, rows, cols, pdl, s);
}

}  // namespace

cudaError_t launch_gemv(uint16_t* out0, uint16_t* out1, const uint16_t* x, const uint8_t* w0,
                        const float* s0, const uint8_t* w1, const float* s1, int64_t rows,
                        int64_t cols, bool pdl, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  if (w1 != nullptr)
    return launch_d<true>(out0, out1, x, w0, s0, w1, s1, int(rows), int(cols), pdl, s);
  return launch_d<false>(out0, nullptr, x, w0, s0, nullptr, nullptr, int(rows), int(cols), pdl, s);
}

}  // namespace qffn
