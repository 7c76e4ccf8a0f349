// Row-scaled W8A16 GEMVs of the single-token FP8 decode FFN (metrale
// "dense_ffn_decode.rs", DenseFfnLayer::forward, FP8 arm: w8a16_gemv_dual
// for gate and up, silu_mul, w8a16_gemv for down).
//
//   out[r] = bf16(row_scale[r] * sum_k W[r,k] * x[k]),  W E4M3, x bf16.
//
// Streaming: one persistent CTA per SM.  A producer thread moves 8-row blocks
// of the weight matrices (split along K into pieces of at most 2048 bytes)
// from HBM into a shared-memory ring with bulk copies; 16 consumer warps
// reduce each piece with warp-level tensor-core MMAs (m16n8k16, f16 inputs,
// fp32 accumulation): the 8 weight rows are the 8 columns of the B operand
// (E4M3 -> f16 is exact), x is row 0 of the A operand, so one MMA does 8 rows
// x 16 columns and a warp needs 1 shared load, 2 converts and 1 MMA per 128
// weight bytes.  x enters as f16 after an exact power-of-two scaling 2^k
// chosen from max|x| (so every x with |x| >= max|x| 2^-29 is exact in f16 and
// nothing overflows); 2^-k is applied to the finished sum.
//
// Per row the arithmetic depends only on the row length: the K split, the
// columns each warp covers, the MMA order, the warp sums added in warp order
// and the split partials added in split order.  So the single, dual and fused
// forms give the same bits for the same row.
//
// The fused decode runs the whole FFN in one cooperative launch: phase 0 is
// the dual gate/up GEMV (g, u to the workspace), then a grid-wide barrier,
// then phase 1 is the down GEMV on h = bf16(silu(g) * u), which every CTA
// forms for the whole vector.  The producer keeps streaming down weights into
// the ring during the barrier.  Phase 1 hands out (8-row block, K piece) units
// so the work splits evenly over the SMs; the CTA finishing the last piece of
// a block adds the pieces' partial sums in piece order.
//
// Every wait is bounded (about 2 s); on expiry the kernel raises its device
// status word and runs to the end without further waiting.
#include <cuda_fp16.h>

#include "common.cuh"
#include "launch.h"
#include "pipeline.cuh"

namespace qffn {
namespace {

constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kBlockRows = 8;              // weight rows per MMA (the n8 of m16n8k16)
constexpr int kPieceMax = 2048;            // bytes of K per piece
constexpr int kSmemBudget = 226 * 1024;
constexpr unsigned long long kWaitNs = 2000000000ull;
constexpr unsigned long long kDrainNs = 200000000ull;
constexpr int kAllConsumers = 15;          // named barrier of the 16 consumer warps

__device__ unsigned int g_decode_status;

struct Phase {
  const uint8_t* w[2];
  const float* s[2];
  uint16_t* out[2];
  int rows, cols, nmat;
  int pieces, piece;      // K pieces per row and their width (bytes, multiple of 256 but the last)
  int nblocks;            // ceil(rows / 8)
  int split;              // 1: units are (block, piece) spread over CTAs; 0: units are blocks
};

struct Params {
  Phase ph[2];
  const uint16_t* x;         // phase-0 input
  const uint16_t* g;         // fused: phase-1 input is silu(g) * u
  const uint16_t* u;
  unsigned int* counter;     // fused: [0] grid barrier, [1 + b] pieces done of block b (zeroed)
  float* partial;            // fused: [pieces][rows] split partial sums of phase 1
  int slot_bytes, nslots, xcap;
};

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

// contiguous share [u0, u1) of `n` units for this CTA
QFFN_DEVI void unit_range(int n, int& u0, int& u1) {
  u0 = int((int64_t(n) * blockIdx.x) / gridDim.x);
  u1 = int((int64_t(n) * (blockIdx.x + 1)) / gridDim.x);
}

// The stages of a phase for this CTA, in order: (block, piece) pairs.
struct StageIter {
  int u, u1, pieces, split;
  QFFN_DEVI StageIter(const Phase& P) : pieces(P.pieces), split(P.split) {
    int a, b;
    unit_range(P.split ? P.nblocks * P.pieces : P.nblocks, a, b);
    u = P.split ? a : a * P.pieces;
    u1 = P.split ? b : b * P.pieces;
  }
  QFFN_DEVI bool more() const { return u < u1; }
  QFFN_DEVI int block() const { return u / pieces; }
  QFFN_DEVI int piece() const { return u % pieces; }
  QFFN_DEVI void next() { ++u; }
};


// x for a phase into shared memory as f16 scaled by 2^k (k from max|x|);
// returns 2^-k.  Phase 1 of the fused decode forms x = bf16(silu(g) * u).
template <bool FROM_GU>
QFFN_DEVI float stage_x(uint16_t* xs, const uint16_t* x, const uint16_t* g, const uint16_t* u,
                        int cols, float* xmax) {
  const int tid = threadIdx.x;
  float m = 0.0f;
  for (int c = tid; c < (cols >> 3); c += kConsumers) {
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
  named_sync(kAllConsumers, kConsumers);
  float amax = 0.0f;
  for (int w = 0; w < kConsumerWarps; ++w) amax = fmaxf(amax, xmax[w]);
  int e = 0;
  frexpf(amax, &e);                                   // amax = f * 2^e, f in [0.5, 1)
  const int k = amax > 0.0f ? 15 - e : 0;             // amax * 2^k in [2^14, 2^15)
  const float up = ldexpf(1.0f, k);
  for (int c = tid; c < (cols >> 3); c += kConsumers) {
    uint4 v = *reinterpret_cast<uint4*>(xs + size_t(c) * 8);
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __half2 h = __floats2half2_rn(bf16_lo(w[j]) * up, bf16_hi(w[j]) * up);
      w[j] = *reinterpret_cast<const uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(xs + size_t(c) * 8) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  named_sync(kAllConsumers, kConsumers);
  return ldexpf(1.0f, -k);
}

template <bool FUSED>
__global__ void __launch_bounds__(kThreads, 1) gemv_stream_kernel(const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~uintptr_t(127));
  uint16_t* xs = reinterpret_cast<uint16_t*>(ring + size_t(p.nslots) * p.slot_bytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(xs + p.xcap);
  float* red = reinterpret_cast<float*>(bars + 2 * p.nslots);     // [2 bufs][2 mats][16 warps][8 rows]
  float* xmax = red + 2 * 2 * kConsumerWarps * kBlockRows;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(xmax + kConsumerWarps);
  const uint32_t bar0 = smem_u32(bars);
  const uint32_t ring0 = smem_u32(ring);
  const uint32_t xs0 = smem_u32(xs);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int nphases = FUSED ? 2 : 1;

  if (tid == 0) {
    for (int s = 0; s < p.nslots; ++s) {
      mbar_init(bar0 + 8u * s, 1);                              // full: the producer's expect_tx
      mbar_init(bar0 + 8u * (p.nslots + s), kConsumerWarps);    // empty: every consumer warp
    }
    *abort_flag = 0;
    mbar_init_fence();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t issued = 0, issued_par = 0;
      int it = 0;
      bool ok = true;
      for (int ph = 0; ok && ph < nphases; ++ph) {
        const Phase& P = p.ph[ph];
        for (StageIter si(P); si.more(); si.next(), ++it) {
          const int b = si.block(), j = si.piece();
          const int nr = min(kBlockRows, P.rows - b * kBlockRows);
          const int width = min(P.piece, P.cols - j * P.piece);
          const int s = it % p.nslots;
          const uint32_t par = uint32_t(it / p.nslots) & 1u;
          if (!mbar_wait_bounded(bar0 + 8u * (p.nslots + s), par ^ 1u, abort_flag,
                                 &g_decode_status, true, kWaitNs)) {
            ok = false;
            break;
          }
          const uint32_t full = bar0 + 8u * s;
          mbar_expect_tx(full, uint32_t(nr * width * P.nmat));
          const uint32_t dst = ring0 + uint32_t(s) * uint32_t(p.slot_bytes);
          for (int m = 0; m < P.nmat; ++m)
            for (int r = 0; r < nr; ++r)
              bulk_load(dst + uint32_t((m * kBlockRows + r) * P.piece),
                        P.w[m] + size_t(b * kBlockRows + r) * size_t(P.cols) + size_t(j) * P.piece,
                        uint32_t(width), full);
          issued |= 1u << s;
          issued_par = (issued_par & ~(1u << s)) | (par << s);
        }
      }
      for (int s = 0; s < p.nslots; ++s)
        if (issued & (1u << s))
          mbar_wait_bounded(bar0 + 8u * s, (issued_par >> s) & 1u, abort_flag, &g_decode_status,
                            false, kDrainNs);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g8 = lane >> 2, t4 = lane & 3;
  int it = 0;
  float acc[2] = {0.0f, 0.0f};           // finishing threads: running sum over pieces
  for (int ph = 0; ph < nphases; ++ph) {
    const Phase& P = p.ph[ph];
    float down = 1.0f;
    if (FUSED && ph == 1) {
      // grid-wide barrier: every CTA has written its g and u rows
      named_sync(kAllConsumers, kConsumers);
      if (tid == 0 && !*abort_flag) {
        __threadfence();
        atomicAdd(p.counter, 1u);
        const unsigned long long t0 = globaltimer();
        while (*reinterpret_cast<volatile unsigned int*>(p.counter) < gridDim.x) {
          __nanosleep(64);
          if (globaltimer() - t0 > kWaitNs) {
            *abort_flag = 1;
            atomicOr(&g_decode_status, 2u);
            break;
          }
        }
        __threadfence();
      }
      named_sync(kAllConsumers, kConsumers);
      down = stage_x<true>(xs, nullptr, p.g, p.u, P.cols, xmax);
    } else {
      down = stage_x<false>(xs, p.x, nullptr, nullptr, P.cols, xmax);
    }
    // columns of each piece a warp covers (a multiple of 16: whole MMA steps)
    const int cw = ((P.piece / 16 + kConsumerWarps - 1) / kConsumerWarps) * 16;
    for (StageIter si(P); si.more(); si.next(), ++it) {
      const int b = si.block(), j = si.piece();
      const int width = min(P.piece, P.cols - j * P.piece);
      const int s = it % p.nslots;
      const uint32_t par = uint32_t(it / p.nslots) & 1u;
      mbar_wait_bounded(bar0 + 8u * s, par, abort_flag, &g_decode_status, true, kWaitNs);
      const uint32_t slot = ring0 + uint32_t(s) * uint32_t(p.slot_bytes);
      float d[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
      for (int c = warp * cw; c < min(warp * cw + cw, width); c += 16) {
        uint32_t a0 = 0u, a2 = 0u;
        if (lane < 4) {
          const uint2 xv = ld_shared64(xs0 + 2u * uint32_t(j * P.piece + c + 4 * t4));
          a0 = xv.x;
          a2 = xv.y;
        }
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          if (m < P.nmat) {
            const uint32_t wv = ld_shared32(slot + uint32_t((m * kBlockRows + g8) * P.piece + c + 4 * t4));
            mma_16816(d[m], a0, 0u, a2, 0u, e4m3x2_to_f16x2(wv & 0xFFFFu), e4m3x2_to_f16x2(wv >> 16));
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar0 + 8u * (p.nslots + s));   // this warp is done with the slot
      float* rb = red + (it & 1) * (2 * kConsumerWarps * kBlockRows);
      if (lane < 4) {
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          rb[(m * kConsumerWarps + warp) * kBlockRows + 2 * t4] = d[m][0];
          rb[(m * kConsumerWarps + warp) * kBlockRows + 2 * t4 + 1] = d[m][1];
        }
      }
      named_sync(kAllConsumers, kConsumers);
      if (tid < kBlockRows * P.nmat) {
        const int m = tid / kBlockRows, r = tid % kBlockRows;
        const int row = b * kBlockRows + r;
        float pj = 0.0f;
        for (int w = 0; w < kConsumerWarps; ++w) pj += rb[(m * kConsumerWarps + w) * kBlockRows + r];
        if (FUSED && P.split) {
          if (row < P.rows) p.partial[size_t(j) * P.rows + row] = pj;
        } else {
          acc[m] = (j == 0) ? pj : acc[m] + pj;
          if (j == P.pieces - 1 && row < P.rows)
            P.out[m][row] = f32_to_bf16(P.s[m][row] * (acc[m] * down));
        }
      }
      if (FUSED && P.split && warp == 0) {
        // the CTA that adds the last piece of block b finishes it, adding the
        // pieces' partial sums in piece order
        __threadfence();
        __syncwarp();
        unsigned int done = 0;
        if (lane == 0) done = atomicAdd(p.counter + 1 + b, 1u);
        done = __shfl_sync(0xffffffffu, done, 0);
        if (done == unsigned(P.pieces - 1)) {
          __threadfence();
          const int row = b * kBlockRows + lane;
          if (lane < kBlockRows && row < P.rows) {
            float t = 0.0f;
            for (int jj = 0; jj < P.pieces; ++jj) {
              const float v = ld_cg_f32(p.partial + size_t(jj) * P.rows + row);
              t = (jj == 0) ? v : t + v;
            }
            P.out[0][row] = f32_to_bf16(P.s[0][row] * (t * down));
          }
        }
      }
    }
  }
}

void set_phase(Phase& P, int rows, int cols, int nmat, int split) {
  P.rows = rows;
  P.cols = cols;
  P.nmat = nmat;
  P.pieces = (cols + kPieceMax - 1) / kPieceMax;
  P.piece = ((cols + P.pieces - 1) / P.pieces + 255) / 256 * 256;
  P.nblocks = (rows + kBlockRows - 1) / kBlockRows;
  P.split = split;
}

template <bool FUSED>
cudaError_t launch_stream(Params& p, int nphases, cudaStream_t s) {
  p.slot_bytes = 0;
  p.xcap = 0;
  for (int i = 0; i < nphases; ++i) {
    const int b = kBlockRows * p.ph[i].piece * p.ph[i].nmat;
    if (b > p.slot_bytes) p.slot_bytes = b;
    if (p.ph[i].cols > p.xcap) p.xcap = p.ph[i].cols;
  }
  const int fixed = 128 + p.xcap * 2 + 2 * 2 * kConsumerWarps * kBlockRows * 4 + kConsumerWarps * 4 + 16;
  p.nslots = (kSmemBudget - fixed - 16 * 32) / p.slot_bytes;
  if (p.nslots > 32) p.nslots = 32;
  if (p.nslots < 2) return cudaErrorInvalidValue;
  const size_t smem = size_t(p.nslots) * p.slot_bytes + fixed + 16 * p.nslots;
  static int attr_done[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    e = cudaFuncSetAttribute(gemv_stream_kernel<FUSED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBudget);
    if (e != cudaSuccess) return e;
    attr_done[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms());
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = FUSED ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemv_stream_kernel<FUSED>, p);
}

}  // namespace

size_t decode_counter_bytes(int64_t C) {
  return (size_t(1) + size_t((C + kBlockRows - 1) / kBlockRows)) * sizeof(unsigned int);
}

size_t decode_partial_bytes(int64_t C, int64_t H) {
  return size_t((H + kPieceMax - 1) / kPieceMax) * size_t(C) * sizeof(float);
}

cudaError_t launch_gemv(uint16_t* out0, uint16_t* out1, const uint16_t* x, const uint8_t* w0,
                        const float* s0, const uint8_t* w1, const float* s1, int64_t rows,
                        int64_t cols, bool /*pdl*/, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  Params p{};
  Phase& P = p.ph[0];
  P.w[0] = w0;
  P.s[0] = s0;
  P.out[0] = out0;
  P.w[1] = w1;
  P.s[1] = s1;
  P.out[1] = out1;
  set_phase(P, int(rows), int(cols), w1 != nullptr ? 2 : 1, 0);
  p.x = x;
  return launch_stream<false>(p, 1, s);
}

cudaError_t launch_decode_fused(uint16_t* out, const uint16_t* x, const uint8_t* w_gate,
                                const float* s_gate, const uint8_t* w_up, const float* s_up,
                                const uint8_t* w_down, const float* s_down, int64_t C, int64_t H,
                                uint16_t* g, uint16_t* u, unsigned int* counter, float* partial,
                                cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(counter, 0, decode_counter_bytes(C), s);
  if (e != cudaSuccess) return e;
  Params p{};
  Phase& A = p.ph[0];
  A.w[0] = w_gate;
  A.s[0] = s_gate;
  A.out[0] = g;
  A.w[1] = w_up;
  A.s[1] = s_up;
  A.out[1] = u;
  set_phase(A, int(H), int(C), 2, 0);
  Phase& D = p.ph[1];
  D.w[0] = w_down;
  D.s[0] = s_down;
  D.out[0] = out;
  set_phase(D, int(C), int(H), 1, 1);
  p.x = x;
  p.g = g;
  p.u = u;
  p.counter = counter;
  p.partial = partial;
  return launch_stream<true>(p, 2, s);
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
