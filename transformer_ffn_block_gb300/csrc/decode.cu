// Row-scaled W8A16 GEMVs of the single-token FP8 decode FFN (metrale
// "dense_ffn_decode.rs", DenseFfnLayer::forward, FP8 arm: w8a16_gemv_dual
// for gate and up, silu_mul, w8a16_gemv for down).
//
//   out[r] = bf16(row_scale[r] * sum_k W[r,k] * x[k]),  W E4M3, x bf16.
//
// The weights are streamed once from HBM by every warp of the grid with
// 16-byte loads straight into registers; the products run on warp-level
// tensor-core MMAs (m16n8k16, f16 inputs, fp32 accumulation): 8 weight rows
// are the 8 columns of the B operand (E4M3 -> f16 is exact) and x is row 0 of
// the A operand, so a warp spends about one load, two converts and one MMA
// per 128 weight bytes.  x enters as f16 from shared memory after an exact
// power-of-two scaling 2^k chosen from max|x| (every x with |x| >= max|x|
// 2^-29 is exact in f16 and nothing overflows); 2^-k is applied to the
// finished sum.
//
// Work unit: an 8-row block times a 512-column piece of K.  Per row the
// arithmetic is fixed by the row length alone: in a piece, 64-column steps in
// order, each lane's 16 bytes feeding four MMAs in order; a fresh accumulator
// per piece; the pieces' partial sums added in piece order.  The standalone
// GEMVs give each warp whole blocks (pieces summed in registers); the fused
// decode spreads units over all warps, keeps piece partials in the workspace
// and lets the warp that completes a block's last piece add them up.  Both
// give the same bits for the same row, and so do the single and dual forms.
//
// The fused decode runs the whole FFN in one cooperative launch: phase 0 is
// the dual gate/up GEMV (g, u to the workspace), a grid-wide barrier, then
// phase 1 is the down GEMV on h = bf16(silu(g) * u), which every CTA forms for
// the whole vector.  The barrier wait is bounded (about 2 s); on expiry the
// kernel raises its device status word and finishes without waiting.
#include <cuda_fp16.h>

#include "common.cuh"
#include "launch.h"
#include "pipeline.cuh"

namespace qffn {
namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kBlockRows = 8;              // weight rows per MMA (the n8 of m16n8k16)
constexpr int kPieceMax = 4096;            // columns of K per work unit at most
constexpr int kStep = 64;                  // columns per load step (16 bytes per lane, 4 MMAs)
constexpr int kSteps = 4;                  // load steps per warp per unit (cw <= 256)
constexpr int kMaxCols = 32768;
constexpr unsigned long long kWaitNs = 2000000000ull;

__device__ unsigned int g_decode_status;

struct Phase {
  const uint8_t* w[2];
  const float* s[2];
  uint16_t* out[2];
  int rows, cols, nmat;
  int pieces, piece;      // K pieces per row and their width (ceil(cols / pieces) rounded to 64)
  int cw;                 // columns of a piece per warp: piece / 16 rounded up to 64
  int nblocks;            // ceil(rows / 8)
  unsigned int* done;     // fused: pieces finished per block (zeroed before launch)
  float* partial;         // fused: [nmat][pieces][rows] piece partial sums
};

struct Params {
  Phase ph[2];
  const uint16_t* x;         // phase-0 input
  const uint16_t* g;         // fused: phase-1 input is silu(g) * u
  const uint16_t* u;
  unsigned int* barrier;     // fused: grid barrier counter (zeroed before launch)
};

QFFN_DEVI uint4 ld_shared128(uint32_t addr) {
  uint4 r;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(addr));
  return r;
}
// L2-coherent loads (data written by other CTAs of the same kernel)
QFFN_DEVI uint4 ld_cg16(const void* p) {
  uint4 r;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p) : "memory");
  return r;
}
QFFN_DEVI float ld_cg_f32(const float* p) {
  float r;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(r) : "l"(p) : "memory");
  return r;
}
QFFN_DEVI unsigned int atomic_add_acq_rel(unsigned int* p, unsigned int v) {
  unsigned int old;
  asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
QFFN_DEVI uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(uint16_t(two_codes)));
  return r;
}
// D += A(16x16, f16, row) * B(16x8, f16, col), fp32 accumulate
QFFN_DEVI void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9},"
      " {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}


// x for a phase into shared memory as f16 scaled by 2^k (k from max|x|), by
// the whole CTA; returns 2^-k.  FROM_GU forms x = bf16(silu(g) * u) first.
template <bool FROM_GU>
QFFN_DEVI float stage_x(uint16_t* xs, const uint16_t* x, const uint16_t* g, const uint16_t* u,
                        int cols, float* xmax) {
  const int tid = threadIdx.x;
  float m = 0.0f;
  for (int c = tid; c < (cols >> 3); c += kThreads) {
    uint4 v;
    if (FROM_GU) v = swiglu8(ld_cg16(g + size_t(c) * 8), ld_cg16(u + size_t(c) * 8));
    else v = ld16_once(x + size_t(c) * 8);
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
  for (int c = tid; c < (cols >> 3); c += kThreads) {
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

// Work unit of a CTA: rows [8b, 8b+8) times piece j of the columns.  Warp w
// covers columns [w*cw, w*cw + cw) of the piece (cw = the piece width / 16
// rounded up to 64), in 64-column steps; lane (g, t) loads 16 bytes of row
// 8b + g at column 16t of each step, which feed four MMAs in order.
struct Unit {
  int b, j;
};

QFFN_DEVI Unit unit_of(const Phase& P, int u) { return Unit{u / P.pieces, u % P.pieces}; }

template <int NMAT>
QFFN_DEVI void load_unit(const Phase& P, Unit un, int warp, int lane, uint4 (&wv)[kSteps][NMAT]) {
  const int g = lane >> 2, t = lane & 3;
  const int row = un.b * kBlockRows + g;
  const int cbase = un.j * P.piece + warp * P.cw;
  const int cend = min(P.cols, (un.j + 1) * P.piece);
#pragma unroll
  for (int q = 0; q < kSteps; ++q) {
    const int col = cbase + q * kStep + 16 * t;
    const bool ok = row < P.rows && q * kStep < P.cw && col < cend;
#pragma unroll
    for (int m = 0; m < NMAT; ++m)
      wv[q][m] = ok ? ld16_ro_stream(P.w[m] + size_t(row) * P.cols + col) : make_uint4(0, 0, 0, 0);
  }
}

// MMAs of one unit; lanes 0..3 end with the warp's partial sums of rows
// 8b + 2*lane (d[m][0]) and 8b + 2*lane + 1 (d[m][1]).
template <int NMAT>
QFFN_DEVI void mma_unit(const Phase& P, Unit un, int warp, int lane, uint32_t xs0,
                        const uint4 (&wv)[kSteps][NMAT], float (&d)[2][4]) {
  const int t = lane & 3;
  const int cbase = un.j * P.piece + warp * P.cw;
  const int cend = min(P.cols, (un.j + 1) * P.piece);
#pragma unroll
  for (int m = 0; m < 2; ++m) d[m][0] = d[m][1] = d[m][2] = d[m][3] = 0.0f;
#pragma unroll
  for (int q = 0; q < kSteps; ++q) {
    const int c0 = cbase + q * kStep;
    if (q * kStep >= P.cw || c0 >= cend) break;
    uint4 xa = make_uint4(0, 0, 0, 0), xb = xa;
    if (lane < 4 && c0 + 16 * t < cend) {
      const uint32_t a = xs0 + 2u * uint32_t(c0 + 16 * t);
      xa = ld_shared128(a);
      xb = ld_shared128(a + 16u);
    }
    const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int m = 0; m < NMAT; ++m) {
        const uint32_t word = i == 0 ? wv[q][m].x : i == 1 ? wv[q][m].y : i == 2 ? wv[q][m].z : wv[q][m].w;
        mma_16816(d[m], xw[2 * i], 0u, xw[2 * i + 1], 0u, e4m3x2_to_f16x2(word & 0xFFFFu),
                  e4m3x2_to_f16x2(word >> 16));
      }
    }
  }
}

// The units [u0, u1) of one phase for this CTA.  Loads of unit u+1 are in
// flight while unit u is multiplied and reduced.  SPLIT: units are (block,
// piece) pairs whose piece sums go to P.partial and the CTA adding a block's
// last piece finishes the block; otherwise this CTA owns whole blocks and
// sums their pieces in order itself.
template <int NMAT, bool SPLIT>
QFFN_DEVI void run_units(const Phase& P, int u0, int u1, uint32_t xs0, float down, float* red) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t = lane & 3;
  uint4 wa[kSteps][NMAT], wb[kSteps][NMAT];
  float acc = 0.0f;                      // finishing threads: running sum over pieces
  if (u0 < u1) load_unit<NMAT>(P, unit_of(P, u0), warp, lane, wa);
  auto finish = [&](int u, const uint4 (&cur)[kSteps][NMAT]) {
    const Unit un = unit_of(P, u);
    float d[2][4];
    mma_unit<NMAT>(P, un, warp, lane, xs0, cur, d);
    float* rb = red + (u & 1) * (2 * kWarps * kBlockRows);
    if (lane < 4) {
#pragma unroll
      for (int m = 0; m < NMAT; ++m) {
        rb[(m * kWarps + warp) * kBlockRows + 2 * t] = d[m][0];
        rb[(m * kWarps + warp) * kBlockRows + 2 * t + 1] = d[m][1];
      }
    }
    __syncthreads();
    if (tid < kBlockRows * NMAT) {
      const int m = tid / kBlockRows, r = tid % kBlockRows;
      const int row = un.b * kBlockRows + r;
      float pj = 0.0f;
      for (int w = 0; w < kWarps; ++w) pj += rb[(m * kWarps + w) * kBlockRows + r];
      if (SPLIT) {
        if (row < P.rows) P.partial[(size_t(m) * P.pieces + un.j) * P.rows + row] = pj;
      } else {
        acc = un.j == 0 ? pj : acc + pj;
        if (un.j == P.pieces - 1 && row < P.rows)
          P.out[m][row] = f32_to_bf16(P.s[m][row] * (acc * down));
      }
    }
    if (SPLIT && warp == 0) {
      // publish this piece (release) and learn whether it was the block's last
      // (acquire); the warp barrier orders lanes 1..7's writes before lane 0's
      __syncwarp();
      unsigned int done = 0;
      if (lane == 0) done = atomic_add_acq_rel(P.done + un.b, 1u);
      done = __shfl_sync(0xffffffffu, done, 0);
      if (done == unsigned(P.pieces - 1) && lane < kBlockRows * NMAT) {
        const int m = lane / kBlockRows, row = un.b * kBlockRows + lane % kBlockRows;
        if (row < P.rows) {
          float s = 0.0f;
          for (int jj = 0; jj < P.pieces; ++jj) {
            const float v = ld_cg_f32(P.partial + (size_t(m) * P.pieces + jj) * P.rows + row);
            s = jj == 0 ? v : s + v;
          }
          P.out[m][row] = f32_to_bf16(P.s[m][row] * (s * down));
        }
      }
    }
  };
  for (int u = u0; u < u1; u += 2) {
    if (u + 1 < u1) load_unit<NMAT>(P, unit_of(P, u + 1), warp, lane, wb);
    finish(u, wa);
    if (u + 1 < u1) {
      if (u + 2 < u1) load_unit<NMAT>(P, unit_of(P, u + 2), warp, lane, wa);
      finish(u + 1, wb);
    }
  }
}

// contiguous share [u0, u1) of `n` units for this CTA
QFFN_DEVI void cta_range(int n, int& u0, int& u1) {
  u0 = int((int64_t(n) * blockIdx.x) / gridDim.x);
  u1 = int((int64_t(n) * (blockIdx.x + 1)) / gridDim.x);
}

// Standalone single / dual GEMV: each CTA owns whole 8-row blocks.
template <int NMAT>
__global__ void __launch_bounds__(kThreads) gemv_kernel(const Phase P, const uint16_t* x) {
  extern __shared__ uint16_t xs[];
  __shared__ float xmax[kWarps];
  __shared__ float red[2 * 2 * kWarps * kBlockRows];
  const float down = stage_x<false>(xs, x, nullptr, nullptr, P.cols, xmax);
  const uint32_t xs0 = uint32_t(__cvta_generic_to_shared(xs));
  int b0, b1;
  cta_range(P.nblocks, b0, b1);
  run_units<NMAT, false>(P, b0 * P.pieces, b1 * P.pieces, xs0, down, red);
}

__global__ void __launch_bounds__(kThreads) decode_fused_kernel(const Params p) {
  extern __shared__ uint16_t xs[];
  __shared__ float xmax[kWarps];
  __shared__ float red[2 * 2 * kWarps * kBlockRows];
  __shared__ int s_abort;
  const uint32_t xs0 = uint32_t(__cvta_generic_to_shared(xs));
  // phase 0: g, u = dual GEMV of x (whole blocks per CTA)
  float down = stage_x<false>(xs, p.x, nullptr, nullptr, p.ph[0].cols, xmax);
  int u0, u1;
  cta_range(p.ph[0].nblocks, u0, u1);
  run_units<2, false>(p.ph[0], u0 * p.ph[0].pieces, u1 * p.ph[0].pieces, xs0, down, red);
  // grid-wide barrier: every CTA has written its g and u rows
  __syncthreads();
  if (threadIdx.x == 0) {
    s_abort = 0;
    __threadfence();
    atomicAdd(p.barrier, 1u);
    const unsigned long long t0 = globaltimer();
    while (*reinterpret_cast<volatile unsigned int*>(p.barrier) < gridDim.x) {
      __nanosleep(64);
      if (globaltimer() - t0 > kWaitNs) {
        s_abort = 1;
        atomicOr(&g_decode_status, 2u);
        break;
      }
    }
    __threadfence();
  }
  __syncthreads();
  if (s_abort) return;            // uniform across the CTA
  // phase 1: out = down GEMV of h = bf16(silu(g) * u), (block, piece) units over CTAs
  down = stage_x<true>(xs, nullptr, p.g, p.u, p.ph[1].cols, xmax);
  cta_range(p.ph[1].nblocks * p.ph[1].pieces, u0, u1);
  run_units<1, true>(p.ph[1], u0, u1, xs0, down, red);
}

void set_phase(Phase& P, int rows, int cols, int nmat) {
  P.rows = rows;
  P.cols = cols;
  P.nmat = nmat;
  P.pieces = (cols + kPieceMax - 1) / kPieceMax;
  P.piece = ((cols + P.pieces - 1) / P.pieces + kStep - 1) / kStep * kStep;
  P.cw = ((P.piece + kWarps - 1) / kWarps + kStep - 1) / kStep * kStep;
  P.nblocks = (rows + kBlockRows - 1) / kBlockRows;
}

cudaError_t set_smem_attr(const void* fn, size_t smem) {
  if (smem <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
}

}  // namespace

size_t decode_counter_bytes(int64_t C, int64_t /*H*/) {
  // grid barrier, then pieces done per 8-row block of out
  return (size_t(1) + size_t((C + kBlockRows - 1) / kBlockRows)) * sizeof(unsigned int);
}

size_t decode_partial_bytes(int64_t C, int64_t H) {
  // piece sums of the down projection: one per K piece of h per output row
  return size_t((H + kPieceMax - 1) / kPieceMax) * size_t(C) * sizeof(float);
}

cudaError_t launch_gemv(uint16_t* out0, uint16_t* out1, const uint16_t* x, const uint8_t* w0,
                        const float* s0, const uint8_t* w1, const float* s1, int64_t rows,
                        int64_t cols, bool /*pdl*/, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  Phase P{};
  P.w[0] = w0;
  P.s[0] = s0;
  P.out[0] = out0;
  P.w[1] = w1;
  P.s[1] = s1;
  P.out[1] = out1;
  set_phase(P, int(rows), int(cols), w1 != nullptr ? 2 : 1);
  const size_t smem = size_t(cols) * 2;
  const int blocks_needed = (P.nblocks + kWarps - 1) / kWarps;
  const int cap = num_sms() * 2;
  const int grid = blocks_needed < cap ? blocks_needed : cap;
  cudaError_t e;
  if (P.nmat == 2) {
    e = set_smem_attr(reinterpret_cast<const void*>(gemv_kernel<2>), smem);
    if (e != cudaSuccess) return e;
    gemv_kernel<2><<<grid, kThreads, smem, s>>>(P, x);
  } else {
    e = set_smem_attr(reinterpret_cast<const void*>(gemv_kernel<1>), smem);
    if (e != cudaSuccess) return e;
    gemv_kernel<1><<<grid, kThreads, smem, s>>>(P, x);
  }
  return cudaGetLastError();
}

cudaError_t launch_decode_fused(uint16_t* out, const uint16_t* x, const uint8_t* w_gate,
                                const float* s_gate, const uint8_t* w_up, const float* s_up,
                                const uint8_t* w_down, const float* s_down, int64_t C, int64_t H,
                                uint16_t* g, uint16_t* u, unsigned int* counter, float* partial,
                                cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(counter, 0, decode_counter_bytes(C, H), s);
  if (e != cudaSuccess) return e;
  Params p{};
  Phase& A = p.ph[0];
  A.w[0] = w_gate;
  A.s[0] = s_gate;
  A.out[0] = g;
  A.w[1] = w_up;
  A.s[1] = s_up;
  A.out[1] = u;
  set_phase(A, int(H), int(C), 2);
  Phase& D = p.ph[1];
  D.w[0] = w_down;
  D.s[0] = s_down;
  D.out[0] = out;
  set_phase(D, int(C), int(H), 1);
  D.done = counter + 1;
  D.partial = partial;
  p.x = x;
  p.g = g;
  p.u = u;
  p.barrier = counter;
  const size_t smem = size_t(C > H ? C : H) * 2;
  e = set_smem_attr(reinterpret_cast<const void*>(decode_fused_kernel), smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_fused_kernel, kThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  if (per_sm > 2) per_sm = 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms() * per_sm);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_fused_kernel, p);
}

cudaError_t decode_take_status(unsigned int* status) {
  unsigned int v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_decode_status, sizeof(v));
  if (e != cudaSuccess) return e;
  if (v != 0) e = cudaMemcpyToSymbol(g_decode_status, &zero, sizeof(zero));
  *status = v;
  return e;
}

}  // namespace qffn
