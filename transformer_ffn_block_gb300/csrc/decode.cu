// Row-scaled W8A16 GEMVs of the single-token FP8 decode FFN (metrale
// "dense_ffn_decode.rs", DenseFfnLayer::forward, FP8 arm: w8a16_gemv_dual
// for gate and up, silu_mul, w8a16_gemv for down).
//
//   out[r] = bf16(row_scale[r] * sum_k W[r,k] * x[k]),  W E4M3, x bf16.
//
// One persistent CTA per SM streams a contiguous range of weight rows from
// HBM into a shared-memory ring with bulk copies (one producer thread), while
// eight consumer warps reduce the rows from shared memory: consumer thread t
// owns the 16-byte chunks t, t+256, ... of every row and keeps the matching
// x values in registers for the whole pass.  Per row the arithmetic is fixed
// (chunks in order, one fma chain per thread, a warp butterfly, then the
// eight warp sums in order), so the single, dual and fused forms below give
// the same bits for the same row.
//
// The fused decode form runs both halves of the FFN in one cooperative
// launch: phase 0 is the dual gate/up GEMV (g, u to the workspace), then a
// grid-wide barrier, then phase 1 is the down GEMV whose input h =
// bf16(silu(g) * u) each thread forms for its own chunks.  The producer does
// not wait at the barrier: it keeps streaming the down weights (which do not
// depend on h) into the ring, so HBM stays busy across the phase boundary.
//
// Every wait is bounded (about 2 s); on expiry the kernel raises its device
// status word, all consumers leave together after their next barrier, and the
// producer drains its copies before returning.
#include "common.cuh"
#include "launch.h"
#include "pipeline.cuh"

namespace qffn {
namespace {

constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kRingBytes = 192 * 1024;
constexpr int kSlotTarget = 16 * 1024;
constexpr int kMaxRowsPerStage = 16;
constexpr int kMaxSlots = 32;
constexpr int kMaxK = 4;                   // chunks per lane per row (x kept in registers)
constexpr unsigned long long kWaitNs = 2000000000ull;
constexpr unsigned long long kDrainNs = 200000000ull;
constexpr int kAllConsumersBarrier = 15;

__device__ unsigned int g_decode_status;

struct Phase {
  const uint8_t* w[2];
  const float* s[2];
  uint16_t* out[2];
  int rows, cols, nmat, rps;
};

struct Params {
  Phase ph[2];
  const uint16_t* x;         // phase-0 input
  const uint16_t* g;         // fused: phase-1 input is silu(g) * u
  const uint16_t* u;
  unsigned int* counter;     // fused: grid barrier counter (zeroed before launch)
  int slot_bytes, nslots;
};

QFFN_DEVI uint4 ld_shared16(uint32_t addr) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(addr));
  return r;
}
// L2-coherent load (data written by other CTAs of the same kernel)
QFFN_DEVI uint4 ld_cg16(const void* p) {
  uint4 r;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p) : "memory");
  return r;
}

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

QFFN_DEVI void row_range(int rows, int& r0, int& r1) {
  r0 = int((int64_t(rows) * blockIdx.x) / gridDim.x);
  r1 = int((int64_t(rows) * (blockIdx.x + 1)) / gridDim.x);
}

// warps per row for a row of `cols` bytes: enough that a lane holds at most
// kMaxK 16-byte chunks, rounded up to a power of two
QFFN_DEVI_HOST int team_warps(int cols) {
  const int nchunk = cols >> 4;
  int s = 1;
  while (s * 32 * kMaxK < nchunk) s <<= 1;
  return s;
}

template <bool FUSED>
__global__ void __launch_bounds__(kThreads, 1) gemv_stream_kernel(const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~uintptr_t(127));
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + size_t(p.nslots) * p.slot_bytes);
  unsigned int* slot_cnt = reinterpret_cast<unsigned int*>(bars + 2 * p.nslots);
  float* red = reinterpret_cast<float*>(slot_cnt + kMaxSlots);   // [warp][2 bufs][2 mats]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(red + kConsumerWarps * 4);
  const uint32_t bar0 = smem_u32(bars);
  const uint32_t ring0 = smem_u32(ring);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int nphases = FUSED ? 2 : 1;

  if (tid == 0) {
    for (int s = 0; s < p.nslots; ++s) {
      mbar_init(bar0 + 8u * s, 1);                 // full: the producer's expect_tx
      mbar_init(bar0 + 8u * (p.nslots + s), 1);    // empty: the last row of the slot
      slot_cnt[s] = 0;
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
        int r0, r1;
        row_range(P.rows, r0, r1);
        for (int row = r0; row < r1; row += P.rps, ++it) {
          const int n = min(P.rps, r1 - row);
          const int s = it % p.nslots;
          const uint32_t par = uint32_t(it / p.nslots) & 1u;
          if (!mbar_wait_bounded(bar0 + 8u * (p.nslots + s), par ^ 1u, abort_flag, &g_decode_status,
                                 true, kWaitNs)) {
            ok = false;
            break;
          }
          const uint32_t bytes = uint32_t(n) * uint32_t(P.cols);
          const uint32_t full = bar0 + 8u * s;
          mbar_expect_tx(full, bytes * uint32_t(P.nmat));
          const uint32_t dst = ring0 + uint32_t(s) * uint32_t(p.slot_bytes);
          for (int m = 0; m < P.nmat; ++m)
            bulk_load(dst + uint32_t(m) * uint32_t(P.rps) * uint32_t(P.cols),
                      P.w[m] + size_t(row) * size_t(P.cols), bytes, full);
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
  // Teams of S warps own whole rows: row i of this CTA's range goes to team
  // i % NT.  A team finishes its row on its own (warp sums, then the team's
  // leader adds its S warp sums in order) and the last row of a slot to finish
  // hands the slot back to the producer.  Consumers never leave early: after a
  // timed-out wait every later wait returns at once and the kernel runs out.
  int stage_base = 0;
  for (int ph = 0; ph < nphases; ++ph) {
    const Phase& P = p.ph[ph];
    const int S = team_warps(P.cols);
    const int NT = kConsumerWarps / S;
    const int team = warp / S, wt = warp % S;
    const int tt = wt * 32 + lane;                  // thread index within the team
    const int stride = S * 32;                      // chunk stride of a lane
    const int nchunk = P.cols >> 4;
    if (FUSED && ph == 1) {
      // grid-wide barrier: every CTA has written its g and u rows
      named_sync(kAllConsumersBarrier, kConsumers);
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
      named_sync(kAllConsumersBarrier, kConsumers);
    }
    // this lane's x chunks for the whole phase
    uint4 xr[kMaxK][2];
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {
      const int c = tt + stride * k;
      if (c < nchunk) {
        if (FUSED && ph == 1) {
          const uint16_t* gp = p.g + size_t(c) * 16;
          const uint16_t* up = p.u + size_t(c) * 16;
          xr[k][0] = swiglu8(ld_cg16(gp), ld_cg16(up));
          xr[k][1] = swiglu8(ld_cg16(gp + 8), ld_cg16(up + 8));
        } else {
          xr[k][0] = ld16_once(p.x + size_t(c) * 16);
          xr[k][1] = ld16_once(p.x + size_t(c) * 16 + 8);
        }
      } else {
        xr[k][0] = xr[k][1] = make_uint4(0, 0, 0, 0);
      }
    }
    int r0, r1;
    row_range(P.rows, r0, r1);
    const int nrows = r1 - r0;
    int nrow_team = 0;
    for (int i = team; i < nrows; i += NT, ++nrow_team) {
      const int st = stage_base + i / P.rps;
      const int s = st % p.nslots;
      const uint32_t par = uint32_t(st / p.nslots) & 1u;
      const int ri = i % P.rps;
      mbar_wait_bounded(bar0 + 8u * s, par, abort_flag, &g_decode_status, true, kWaitNs);
      const uint32_t slot = ring0 + uint32_t(s) * uint32_t(p.slot_bytes);
      float part[2];
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        part[m] = 0.0f;
        if (m < P.nmat) {
          const uint32_t wrow = slot + uint32_t(m * P.rps + ri) * uint32_t(P.cols);
          float a0 = 0.0f, a1 = 0.0f;
#pragma unroll
          for (int k = 0; k < kMaxK; k += 2) {
            const int c0 = tt + stride * k, c1 = c0 + stride;
            if (c0 < nchunk) a0 = dot16(ld_shared16(wrow + uint32_t(c0) * 16u), xr[k][0], xr[k][1], a0);
            if (c1 < nchunk) a1 = dot16(ld_shared16(wrow + uint32_t(c1) * 16u), xr[k + 1][0], xr[k + 1][1], a1);
          }
          part[m] = warp_sum(a0 + a1);
        }
      }
      float tot[2] = {part[0], part[1]};
      if (S > 1) {
        float* rb = red + 4 * team * S;                   // this team's [S warps][2 bufs][2]
        if (lane == 0) {
          rb[wt * 4 + (nrow_team & 1) * 2 + 0] = part[0];
          rb[wt * 4 + (nrow_team & 1) * 2 + 1] = part[1];
        }
        named_sync(1 + team, S * 32);
        if (tt == 0) {
          tot[0] = tot[1] = 0.0f;
          for (int w = 0; w < S; ++w) {
            tot[0] += rb[w * 4 + (nrow_team & 1) * 2 + 0];
            tot[1] += rb[w * 4 + (nrow_team & 1) * 2 + 1];
          }
        }
      }
      if (tt == 0) {
        const int row = r0 + i;
        for (int m = 0; m < P.nmat; ++m) P.out[m][row] = f32_to_bf16(P.s[m][row] * tot[m]);
        // this row's slot data has been read by the whole team (it fed the sums)
        const int n_in_slot = min(P.rps, nrows - (i / P.rps) * P.rps);
        if (atomicAdd(&slot_cnt[s], 1u) == unsigned(n_in_slot - 1)) {
          slot_cnt[s] = 0;
          mbar_arrive(bar0 + 8u * (p.nslots + s));
        }
      }
    }
    stage_base += (nrows + P.rps - 1) / P.rps;
  }
}

int phase_rps(int cols, int nmat) {
  int rps = kSlotTarget / (cols * nmat);
  if (rps < 1) rps = 1;
  if (rps > kMaxRowsPerStage) rps = kMaxRowsPerStage;
  return rps;
}

template <bool FUSED>
cudaError_t launch_stream(Params& p, int nphases, cudaStream_t s) {
  p.slot_bytes = 0;
  for (int i = 0; i < nphases; ++i) {
    p.ph[i].rps = phase_rps(p.ph[i].cols, p.ph[i].nmat);
    const int b = p.ph[i].rps * p.ph[i].cols * p.ph[i].nmat;
    if (b > p.slot_bytes) p.slot_bytes = b;
  }
  p.nslots = kRingBytes / p.slot_bytes;
  if (p.nslots > kMaxSlots) p.nslots = kMaxSlots;
  const size_t smem = size_t(p.nslots) * p.slot_bytes + 128 + 16 * p.nslots + 4 * kMaxSlots +
                      4 * kConsumerWarps * 4 + 16;
  static int attr_done[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && !(attr_done[dev] & 1)) {
    e = cudaFuncSetAttribute(gemv_stream_kernel<FUSED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kRingBytes + 4096));
    if (e != cudaSuccess) return e;
    attr_done[dev] |= 1;
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

cudaError_t launch_gemv(uint16_t* out0, uint16_t* out1, const uint16_t* x, const uint8_t* w0,
                        const float* s0, const uint8_t* w1, const float* s1, int64_t rows,
                        int64_t cols, bool /*pdl*/, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  Params p{};
  p.ph[0].w[0] = w0;
  p.ph[0].s[0] = s0;
  p.ph[0].out[0] = out0;
  p.ph[0].w[1] = w1;
  p.ph[0].s[1] = s1;
  p.ph[0].out[1] = out1;
  p.ph[0].rows = int(rows);
  p.ph[0].cols = int(cols);
  p.ph[0].nmat = w1 != nullptr ? 2 : 1;
  p.x = x;
  return launch_stream<false>(p, 1, s);
}

cudaError_t launch_decode_fused(uint16_t* out, const uint16_t* x, const uint8_t* w_gate,
                                const float* s_gate, const uint8_t* w_up, const float* s_up,
                                const uint8_t* w_down, const float* s_down, int64_t C, int64_t H,
                                uint16_t* g, uint16_t* u, unsigned int* counter, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(counter, 0, sizeof(unsigned int), s);
  if (e != cudaSuccess) return e;
  Params p{};
  p.ph[0].w[0] = w_gate;
  p.ph[0].s[0] = s_gate;
  p.ph[0].out[0] = g;
  p.ph[0].w[1] = w_up;
  p.ph[0].s[1] = s_up;
  p.ph[0].out[1] = u;
  p.ph[0].rows = int(H);
  p.ph[0].cols = int(C);
  p.ph[0].nmat = 2;
  p.ph[1].w[0] = w_down;
  p.ph[1].s[0] = s_down;
  p.ph[1].out[0] = out;
  p.ph[1].rows = int(C);
  p.ph[1].cols = int(H);
  p.ph[1].nmat = 1;
  p.x = x;
  p.g = g;
  p.u = u;
  p.counter = counter;
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
