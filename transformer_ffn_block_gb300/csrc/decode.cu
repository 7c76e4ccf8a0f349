// Row-scaled W8A16 GEMVs of the single-token FP8 decode FFN (metrale
// "dense_ffn_decode.rs", DenseFfnLayer::forward, FP8 arm: w8a16_gemv_dual
// for gate and up, silu_mul, w8a16_gemv for down).
//
//   out[r] = bf16(row_scale[r] * sum_k W[r,k] * x[k]),  W E4M3, x bf16.
//
// Each warp streams its weight rows from HBM into a private shared-memory
// ring with 16-byte asynchronous copies (cp.async, no registers held while the
// data is in flight), several stages ahead of the stage it multiplies, so an
// SM keeps about 150 KB of loads in flight.  x sits in shared memory as fp32.
// A lane owns the 16-byte pieces lane, lane+32, ... of the warp's columns and
// accumulates them with packed fp32x2 fmas (even and odd elements in the two
// halves).  Rows longer than 4096 columns are split over a team of 2, 4 or 8
// warps (K parts), whose sums the team leader adds in part order.
//
// Per row the arithmetic depends only on the row length (team size, K parts,
// piece order, packed fma order, warp butterfly, parts in order), so the
// single and dual GEMVs give the same bits row for row, and so does the down
// GEMV whose input h = bf16(silu(g) * u) it forms itself from g and u (the
// decode's silu_mul folded into the down projection's prologue).
#include <cuda_fp16.h>

#include "common.cuh"
#include "launch.h"
#include "pipeline.cuh"

namespace qffn {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kChunk = 4096;               // columns per ring stage (a multiple of 512)
constexpr int kSmemBudget = 220 * 1024;

struct Gemv {
  const uint8_t* w[2];
  const float* s[2];
  uint16_t* out[2];
  const uint16_t* x;        // input (bf16), or with SILU: g
  const uint16_t* u;        // SILU: up values
  int rows, cols, nmat;
  int team;                 // warps per row (power of two)
  int kpart;                // columns per warp of a team (multiple of 16)
  int nstage;               // ring stages per warp
  int stage_bytes;          // kChunk * nmat
};

QFFN_DEVI void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
QFFN_DEVI void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
QFFN_DEVI void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
QFFN_DEVI void cp_async_wait_dyn(int n) {
  // wait until at most n groups of this thread are pending
  switch (n) {
    case 0: cp_async_wait<0>(); break;
    case 1: cp_async_wait<1>(); break;
    case 2: cp_async_wait<2>(); break;
    case 3: cp_async_wait<3>(); break;
    case 4: cp_async_wait<4>(); break;
    case 5: cp_async_wait<5>(); break;
    default: cp_async_wait<6>(); break;
  }
}
QFFN_DEVI uint4 ld_shared128(uint32_t addr) {
  uint4 r;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(addr));
  return r;
}
QFFN_DEVI float4 ld_shared_f4(uint32_t addr) {
  float4 r;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
               : "r"(addr));
  return r;
}

// acc += the 16 products of one 16-byte weight piece with its 16 x values
// (fp32 in shared memory at xa), element pairs in order, even elements in the
// low half of acc and odd elements in the high half.
QFFN_DEVI void dot16_packed(uint4 w, uint32_t xa, uint64_t& acc) {
  const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t h01, h23;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h01) : "h"(uint16_t(ww[j] & 0xFFFF)));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h23) : "h"(uint16_t(ww[j] >> 16)));
    const float2 fa = __half22float2(*reinterpret_cast<__half2*>(&h01));
    const float2 fb = __half22float2(*reinterpret_cast<__half2*>(&h23));
    const float4 xv = ld_shared_f4(xa + 16u * j);
    acc = f2_fma(f2_pack(fa.x, fa.y), f2_pack(xv.x, xv.y), acc);
    acc = f2_fma(f2_pack(fb.x, fb.y), f2_pack(xv.z, xv.w), acc);
  }
}

// x (or h = bf16(silu(g) * u)) into shared memory as fp32, whole CTA.
template <bool SILU>
QFFN_DEVI void stage_x(float* xs, const Gemv& G) {
  for (int c = threadIdx.x; c < (G.cols >> 3); c += kThreads) {
    uint4 v;
    if (SILU) v = swiglu8(ld16_once(G.x + size_t(c) * 8), ld16_once(G.u + size_t(c) * 8));
    else v = ld16_once(G.x + size_t(c) * 8);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float4* dst = reinterpret_cast<float4*>(xs + size_t(c) * 8);
    dst[0] = make_float4(bf16_lo(w[0]), bf16_hi(w[0]), bf16_lo(w[1]), bf16_hi(w[1]));
    dst[1] = make_float4(bf16_lo(w[2]), bf16_hi(w[2]), bf16_lo(w[3]), bf16_hi(w[3]));
  }
}

// SILU: the input is h = bf16(silu(g) * u) (g in G.x, u in G.u), formed after
// the programmatic-launch dependency wait; the first weight stages are
// already in flight by then.
template <int NMAT, bool SILU>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(const Gemv G) {
  extern __shared__ __align__(16) uint8_t smem[];
  float* xs = reinterpret_cast<float*>(smem);
  uint8_t* rings = smem + size_t(G.cols) * 4;
  __shared__ float red[2][kWarps][2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nteams = kWarps / G.team;
  const int team = warp / G.team, part = warp % G.team;
  const int k0 = part * G.kpart;
  const int k1 = min(G.cols, k0 + G.kpart);
  const int nchunks = k1 > k0 ? (k1 - k0 + kChunk - 1) / kChunk : 0;
  // rows of this CTA, then of this team
  const int r0 = int((int64_t(G.rows) * blockIdx.x) / gridDim.x);
  const int r1 = int((int64_t(G.rows) * (blockIdx.x + 1)) / gridDim.x);
  const int my_rows = r1 - r0 > team ? (r1 - r0 - team + nteams - 1) / nteams : 0;
  const int nstages = my_rows * nchunks;
  uint8_t* ring = rings + size_t(warp) * G.nstage * G.stage_bytes;
  const uint32_t ring0 = uint32_t(__cvta_generic_to_shared(ring));

  // stage i of this warp: row r0 + team + (i / nchunks) * nteams, chunk i % nchunks
  auto issue = [&](int i) {
    if (i < nstages) {
      const int row = r0 + team + (i / nchunks) * nteams;
      const int c0 = k0 + (i % nchunks) * kChunk;
      const int nbytes = min(kChunk, k1 - c0);
      const uint32_t dst = ring0 + uint32_t((i % G.nstage) * G.stage_bytes);
#pragma unroll
      for (int m = 0; m < NMAT; ++m) {
        const uint8_t* src = G.w[m] + size_t(row) * G.cols + c0;
        for (int p = lane; p < (nbytes >> 4); p += 32) cp_async16(dst + uint32_t(m * kChunk + 16 * p), src + 16 * p);
      }
    }
    cp_async_commit();               // (empty groups keep the counting uniform)
  };
  for (int i = 0; i < G.nstage - 1; ++i) issue(i);
  if (SILU) pdl_wait();              // g, u come from the preceding kernel
  pdl_trigger();
  if (SILU) stage_x<true>(xs, G);
  else stage_x<false>(xs, G);
  __syncthreads();
  const uint32_t xs0 = uint32_t(__cvta_generic_to_shared(xs));

  uint64_t acc[2] = {0ull, 0ull};
  int rowi = 0;
  for (int i = 0; i < nstages; ++i) {
    issue(i + G.nstage - 1);
    cp_async_wait_dyn(G.nstage - 1);
    __syncwarp();
    const int chunk = i % nchunks;
    const int c0 = k0 + chunk * kChunk;
    const int nbytes = min(kChunk, k1 - c0);
    const uint32_t src = ring0 + uint32_t((i % G.nstage) * G.stage_bytes);
    for (int p = lane; p < (nbytes >> 4); p += 32) {
      const uint32_t xa = xs0 + 4u * uint32_t(c0 + 16 * p);
#pragma unroll
      for (int m = 0; m < NMAT; ++m) dot16_packed(ld_shared128(src + uint32_t(m * kChunk + 16 * p)), xa, acc[m]);
    }
    __syncwarp();                    // every lane is done with this ring slot
    if (chunk == nchunks - 1) {
      const int row = r0 + team + (i / nchunks) * nteams;
      float tot[2];
#pragma unroll
      for (int m = 0; m < NMAT; ++m) {
        float lo, hi;
        f2_unpack(acc[m], lo, hi);
        tot[m] = warp_sum(lo + hi);
        acc[m] = 0ull;
      }
      if (G.team == 1) {
        if (lane == 0)
          for (int m = 0; m < NMAT; ++m) G.out[m][row] = f32_to_bf16(G.s[m][row] * tot[m]);
      } else {
        if (lane == 0)
          for (int m = 0; m < NMAT; ++m) red[rowi & 1][warp][m] = tot[m];
        named_sync(1 + team, G.team * 32);
        if (part == 0 && lane == 0) {
          for (int m = 0; m < NMAT; ++m) {
            float t = 0.0f;
            for (int q = 0; q < G.team; ++q) t += red[rowi & 1][warp + q][m];
            G.out[m][row] = f32_to_bf16(G.s[m][row] * t);
          }
        }
      }
      ++rowi;
    }
  }
  cp_async_wait<0>();
}

}  // namespace

cudaError_t launch_gemv_ex(uint16_t* out0, uint16_t* out1, const uint16_t* x, const uint16_t* u_silu,
                           const uint8_t* w0, const float* s0, const uint8_t* w1, const float* s1,
                           int64_t rows, int64_t cols, bool silu, bool pdl, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  Gemv G{};
  G.w[0] = w0;
  G.s[0] = s0;
  G.out[0] = out0;
  G.w[1] = w1;
  G.s[1] = s1;
  G.out[1] = out1;
  G.x = x;
  G.u = u_silu;
  G.rows = int(rows);
  G.cols = int(cols);
  G.nmat = w1 != nullptr ? 2 : 1;
  int parts = int((cols + kChunk - 1) / kChunk);
  G.team = 1;
  while (G.team < parts && G.team < kWarps) G.team <<= 1;
  G.kpart = int(((cols + G.team - 1) / G.team + 15) / 16 * 16);
  G.stage_bytes = kChunk * G.nmat;
  const size_t xbytes = size_t(cols) * 4;
  int ns = int((kSmemBudget - int64_t(xbytes)) / (int64_t(kWarps) * G.stage_bytes));
  if (ns > 6) ns = 6;
  if (ns < 2) return cudaErrorInvalidValue;
  G.nstage = ns;
  const size_t smem = xbytes + size_t(kWarps) * ns * G.stage_bytes;
  cudaError_t e;
  const void* fn = G.nmat == 2 ? (silu ? reinterpret_cast<const void*>(gemv_kernel<2, true>)
                                       : reinterpret_cast<const void*>(gemv_kernel<2, false>))
                               : (silu ? reinterpret_cast<const void*>(gemv_kernel<1, true>)
                                       : reinterpret_cast<const void*>(gemv_kernel<1, false>));
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms());
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  void* args[] = {&G};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t launch_gemv(uint16_t* out0, uint16_t* out1, const uint16_t* x, const uint8_t* w0,
                        const float* s0, const uint8_t* w1, const float* s1, int64_t rows,
                        int64_t cols, bool pdl, cudaStream_t s) {
  return launch_gemv_ex(out0, out1, x, nullptr, w0, s0, w1, s1, rows, cols, false, pdl, s);
}

cudaError_t launch_decode(uint16_t* out, const uint16_t* x, const uint8_t* w_gate,
                          const float* s_gate, const uint8_t* w_up, const float* s_up,
                          const uint8_t* w_down, const float* s_down, int64_t C, int64_t H,
                          uint16_t* g, uint16_t* u, cudaStream_t s) {
  cudaError_t e = launch_gemv_ex(g, u, x, nullptr, w_gate, s_gate, w_up, s_up, H, C, false, false, s);
  if (e != cudaSuccess) return e;
  return launch_gemv_ex(out, nullptr, g, u, w_down, s_down, nullptr, nullptr, C, H, true, true, s);
}

cudaError_t decode_take_status(unsigned int* status) {
  *status = 0;      // the decode kernels have no bounded waits
  return cudaSuccess;
}

}  // namespace qffn
