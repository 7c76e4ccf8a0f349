// Row-scaled W8A16 GEMVs of the single-token FP8 decode FFN (metrale
// "dense_ffn_decode.rs", DenseFfnLayer::forward, FP8 arm: w8a16_gemv_dual
// for gate and up, silu_mul, w8a16_gemv for down).
//
//   out[r] = bf16(row_scale[r] * sum_k W[r,k] * x[k]),  W E4M3, x bf16.
//
// A warp owns 8-row blocks.  It streams them through a private shared-memory
// ring with 16-byte asynchronous copies (cp.async: row-contiguous 512-byte
// spans per copy instruction, nothing held in registers while in flight),
// several 256-column stages ahead, and multiplies each stage with warp-level
// tensor-core MMAs (m16n8k16, f16 inputs, fp32 accumulation): the 8 rows are
// the 8 columns of the B operand (E4M3 -> f16 is exact; a 16-byte row pitch
// pad makes the fragment reads conflict-free), x is row 0 of the A operand.
// x enters as f16 after an exact power-of-two scaling 2^k chosen from max|x|
// (every x with |x| >= max|x| 2^-29 is exact in f16, nothing overflows);
// 2^-k is applied to the finished sum.  Rows longer than 4096 columns are
// split over a team of 2, 4 or 8 warps (K parts) whose sums the team leader
// adds in part order.
//
// Per row the arithmetic depends only on the row length, so the single and
// dual GEMVs agree bit for bit, and so does the down GEMV that forms its own
// input h = bf16(silu(g) * u) (the decode's silu_mul folded into its
// prologue).  That kernel is a programmatic dependent launch: its first weight
// stages are in flight before it waits for the dual GEMV's g and u.
#include <cuda_fp16.h>

#include "common.cuh"
#include "launch.h"
#include "pipeline.cuh"

namespace qffn {
namespace {

constexpr int kWarps = 12;
constexpr int kThreads = kWarps * 32;
constexpr int kBlockRows = 8;              // rows per MMA (the n8 of m16n8k16)
constexpr int kSeg = 256;                  // columns per ring stage
constexpr int kPitch = kSeg + 16;          // bytes per row in a stage (bank-conflict pad)
constexpr int kMatStage = kBlockRows * kPitch;
constexpr int kPartMax = 4096;             // columns per K part at most
constexpr int kSmemBudget = 226 * 1024;

struct Gemv {
  uint16_t* out[2];
  const uint16_t* x;         // input bf16 [cols], or with SILU: g
  const uint16_t* u;         // SILU: up values
  const uint8_t* w[2];
  const float* s[2];
  int rows, cols;
  int team, kpart;           // warps per block and columns per warp (multiple of 16)
  int nstage;                // ring stages per warp
};

QFFN_DEVI void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
QFFN_DEVI void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
QFFN_DEVI void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
QFFN_DEVI void cp_async_wait_dyn(int n) {   // at most n of this thread's groups still pending
  switch (n) {
    case 0: cp_async_wait<0>(); break;
    case 1: cp_async_wait<1>(); break;
    case 2: cp_async_wait<2>(); break;
    case 3: cp_async_wait<3>(); break;
    case 4: cp_async_wait<4>(); break;
    case 5: cp_async_wait<5>(); break;
    case 6: cp_async_wait<6>(); break;
    default: cp_async_wait<7>(); break;
  }
}
QFFN_DEVI uint32_t ld_shared32(uint32_t addr) {
  uint32_t r;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(r) : "r"(addr));
  return r;
}
QFFN_DEVI uint2 ld_shared64(uint32_t addr) {
  uint2 r;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(addr));
  return r;
}
QFFN_DEVI uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(uint16_t(two_codes)));
  return r;
}
// D += A(16x16, f16, row) * B(16x8, f16, col), fp32 accumulate
QFFN_DEVI void mma_16816(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9},"
      " {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

// x (or h = bf16(silu(g) * u)) into shared memory as f16 scaled by 2^k, by
// the whole CTA; returns 2^-k.
template <bool SILU>
QFFN_DEVI float stage_x(uint16_t* xs, const Gemv& G, float* xmax) {
  const int tid = threadIdx.x;
  float m = 0.0f;
  for (int c = tid; c < (G.cols >> 3); c += kThreads) {
    uint4 v;
    if (SILU) v = swiglu8(ld16_once(G.x + size_t(c) * 8), ld16_once(G.u + size_t(c) * 8));
    else v = ld16_once(G.x + size_t(c) * 8);
    *reinterpret_cast<uint4*>(xs + size_t(c) * 8) = v;
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
  }
  m = warp_max(m);
  if ((tid & 31) == 0) xmax[tid >> 5] = m;
  __syncthreads();
  float amax = 0.0f;
  for (int w = 0; w < kWarps; ++w) amax = fmaxf(amax, xmax[w]);
  int e = 0;
  frexpf(amax, &e);                                   // amax = f * 2^e, f in [0.5, 1)
  const int k = amax > 0.0f ? 15 - e : 0;             // amax * 2^k in [2^14, 2^15)
  const float up = ldexpf(1.0f, k);
  for (int c = tid; c < (G.cols >> 3); c += kThreads) {
    const uint4 v = *reinterpret_cast<uint4*>(xs + size_t(c) * 8);
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __half2 h = __floats2half2_rn(bf16_lo(w[j]) * up, bf16_hi(w[j]) * up);
      w[j] = *reinterpret_cast<const uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(xs + size_t(c) * 8) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  __syncthreads();
  return ldexpf(1.0f, -k);
}

template <int NMAT, bool SILU>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(const Gemv G) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);
  uint8_t* rings = smem + ((size_t(G.cols) * 2 + 127) / 128) * 128;
  __shared__ float xmax[kWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g8 = lane >> 2, t4 = lane & 3;
  const int nteams = kWarps / G.team;
  const int team = warp / G.team, part = warp % G.team;
  const int k0 = part * G.kpart;
  const int k1 = min(G.cols, k0 + G.kpart);
  const int nseg = k1 > k0 ? (k1 - k0 + kSeg - 1) / kSeg : 0;
  const int nblocks = (G.rows + kBlockRows - 1) / kBlockRows;
  const int gteam = blockIdx.x * nteams + team, nteam_all = gridDim.x * nteams;
  const bool active = team < nteams;            // warps left over when team does not divide 12
  const int my_blocks = active && nblocks > gteam ? (nblocks - gteam + nteam_all - 1) / nteam_all : 0;
  const int nstages = my_blocks * nseg;
  const int stage_bytes = NMAT * kMatStage;
  const uint32_t ring0 = uint32_t(__cvta_generic_to_shared(rings)) + uint32_t(warp * G.nstage * stage_bytes);

  // stage i of this warp: block gteam + (i / nseg) * nteam_all, segment i % nseg
  auto issue = [&](int i) {
    if (i < nstages) {
      const int b = gteam + (i / nseg) * nteam_all;
      const int c0 = k0 + (i % nseg) * kSeg;
      const int npiece = min(kSeg, k1 - c0) >> 4;
      const int nr = min(kBlockRows, G.rows - b * kBlockRows);
      const uint32_t dst = ring0 + uint32_t((i % G.nstage) * stage_bytes);
#pragma unroll
      for (int m = 0; m < NMAT; ++m)
        for (int q = lane; q < kBlockRows * (kSeg / 16); q += 32) {
          const int r = q / (kSeg / 16), p = q % (kSeg / 16);
          if (r < nr && p < npiece)
            cp_async16(dst + uint32_t(m * kMatStage + r * kPitch + 16 * p),
                       G.w[m] + size_t(b * kBlockRows + r) * G.cols + c0 + 16 * p);
        }
    }
    cp_async_commit();               // (empty groups keep the counting uniform)
  };
  for (int i = 0; i < G.nstage - 1; ++i) issue(i);
  if (SILU) pdl_wait();              // g and u come from the preceding kernel
  pdl_trigger();
  const float down = stage_x<SILU>(xs, G, xmax);
  const uint32_t xs0 = uint32_t(__cvta_generic_to_shared(xs));

  float d[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
  int blk = 0;
  for (int i = 0; i < nstages; ++i) {
    issue(i + G.nstage - 1);
    cp_async_wait_dyn(G.nstage - 1);
    __syncwarp();
    const int seg = i % nseg;
    const int c0 = k0 + seg * kSeg;
    const int nstep = min(kSeg, k1 - c0) >> 4;
    const uint32_t src = ring0 + uint32_t((i % G.nstage) * stage_bytes);
    for (int st = 0; st < nstep; ++st) {
      uint32_t a0 = 0u, a2 = 0u;
      if (lane < 4) {
        const uint2 xv = ld_shared64(xs0 + 2u * uint32_t(c0 + 16 * st + 4 * t4));
        a0 = xv.x;
        a2 = xv.y;
      }
#pragma unroll
      for (int m = 0; m < NMAT; ++m) {
        const uint32_t wv = ld_shared32(src + uint32_t(m * kMatStage + g8 * kPitch + 16 * st + 4 * t4));
        mma_16816(d[m], a0, a2, e4m3x2_to_f16x2(wv & 0xFFFFu), e4m3x2_to_f16x2(wv >> 16));
      }
    }
    __syncwarp();                    // every lane is done with this ring slot
    if (seg == nseg - 1) {
      const int b = gteam + (i / nseg) * nteam_all;
      // lanes 0..3 hold rows 8b + 2*lane (d[m][0]) and 8b + 2*lane + 1 (d[m][1])
      float v[2][2];
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        v[m][0] = d[m][0];
        v[m][1] = d[m][1];
        d[m][0] = d[m][1] = d[m][2] = d[m][3] = 0.0f;
      }
      if (G.team == 1) {
        if (lane < 4)
#pragma unroll
          for (int m = 0; m < NMAT; ++m)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int row = b * kBlockRows + 2 * lane + e;
              if (row < G.rows) G.out[m][row] = f32_to_bf16(G.s[m][row] * (v[m][e] * down));
            }
      } else {
        // team: every warp leaves its 8 row sums (per matrix) in shared memory
        __shared__ float tred[2][kWarps][2][kBlockRows];
        if (lane < 4)
#pragma unroll
          for (int m = 0; m < NMAT; ++m) {
            tred[blk & 1][warp][m][2 * lane] = v[m][0];
            tred[blk & 1][warp][m][2 * lane + 1] = v[m][1];
          }
        named_sync(1 + team, G.team * 32);
        if (part == 0 && lane < kBlockRows * NMAT) {
          const int m = lane / kBlockRows, r = lane % kBlockRows;
          const int row = b * kBlockRows + r;
          float t = 0.0f;
          for (int q = 0; q < G.team; ++q) t += tred[blk & 1][warp + q][m][r];
          if (row < G.rows) G.out[m][row] = f32_to_bf16(G.s[m][row] * (t * down));
        }
      }
      ++blk;
    }
  }
  cp_async_wait<0>();
}

template <int NMAT, bool SILU>
cudaError_t launch_t(Gemv G, bool pdl, cudaStream_t s) {
  int parts = (G.cols + kPartMax - 1) / kPartMax;
  G.team = 1;
  while (G.team < parts) G.team <<= 1;
  if (G.team > 8) return cudaErrorInvalidValue;         // cols > 32768
  G.kpart = ((G.cols + G.team - 1) / G.team + 15) / 16 * 16;
  const size_t xbytes = (size_t(G.cols) * 2 + 127) / 128 * 128;
  const int stage_bytes = NMAT * kMatStage;
  int ns = int((kSmemBudget - int64_t(xbytes) - 1024) / (int64_t(kWarps) * stage_bytes));
  if (ns > 8) ns = 8;
  if (ns < 2) return cudaErrorInvalidValue;
  G.nstage = ns;
  const size_t smem = xbytes + size_t(kWarps) * ns * stage_bytes;
  auto fn = gemv_kernel<NMAT, SILU>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  const int nblocks = (G.rows + kBlockRows - 1) / kBlockRows;
  const int nteams = kWarps / G.team;
  const int needed = (nblocks + nteams - 1) / nteams;
  const int grid = needed < num_sms() ? needed : num_sms();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, fn, G);
}

}  // namespace

cudaError_t launch_gemv(uint16_t* out0, uint16_t* out1, const uint16_t* x, const uint8_t* w0,
                        const float* s0, const uint8_t* w1, const float* s1, int64_t rows,
                        int64_t cols, bool pdl, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  Gemv G{};
  G.out[0] = out0;
  G.out[1] = out1;
  G.x = x;
  G.w[0] = w0;
  G.s[0] = s0;
  G.w[1] = w1;
  G.s[1] = s1;
  G.rows = int(rows);
  G.cols = int(cols);
  return w1 != nullptr ? launch_t<2, false>(G, pdl, s) : launch_t<1, false>(G, pdl, s);
}

cudaError_t launch_decode(uint16_t* out, const uint16_t* x, const uint8_t* w_gate,
                          const float* s_gate, const uint8_t* w_up, const float* s_up,
                          const uint8_t* w_down, const float* s_down, int64_t C, int64_t H,
                          uint16_t* g, uint16_t* u, cudaStream_t s) {
  cudaError_t e = launch_gemv(g, u, x, w_gate, s_gate, w_up, s_up, H, C, false, s);
  if (e != cudaSuccess) return e;
  Gemv G{};
  G.out[0] = out;
  G.x = g;
  G.u = u;
  G.w[0] = w_down;
  G.s[0] = s_down;
  G.rows = int(C);
  G.cols = int(H);
  return launch_t<1, true>(G, true, s);
}

cudaError_t decode_take_status(unsigned int* status) {
  *status = 0;      // the decode kernels have no bounded waits
  return cudaSuccess;
}

}  // namespace qffn
