// HBM-bound kernels of the FFN block: fused residual + RMSNorm + abs-max,
// tensor abs-max, per-tensor and per-row E4M3 quantisation, SwiGLU with
// abs-max, SwiGLU requantisation and the decode silu_mul.
//
// All of them move 16-byte vectors per thread, reduce in registers, then by
// warp shuffles and one shared-memory step per block, and record a tensor
// abs-max with one atomicMax per block on the bits of a non-negative float.
#include "common.cuh"
#include "launch.h"

namespace qffn {

namespace {

constexpr int kThreads = 256;

int g_sm_count[64] = {0};

__device__ __forceinline__ float block_reduce_max(float v, float* red) {
  v = warp_max(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = 0.0f;
  if (warp == 0) {
    r = lane < (int)(blockDim.x >> 5) ? red[lane] : 0.0f;
    r = warp_max(r);
  }
  return r;  // valid in warp 0
}

// ------------------------------------------------------------------ A1
// One block of 128 threads per row; thread t owns the 16-byte chunks
// t, t+128, ... of the row and keeps its residual sums in registers between
// the sum-of-squares pass and the normalisation pass.
//
// y is rounded once from an almost exact value, so it agrees with the
// correctly rounded r * rstd * g: each r^2 is exact in fp32 and is summed as
// a double-float (about 48 bits); mean, eps and 1/sqrt are formed once per
// row as a double-float (rstd = hi + lo, about 43 bits); r * g is exact in
// fp32 and (r * g) * (hi + lo) is formed as a double-float with two fmas
// before the single rounding to bf16.
template <int V>
__global__ void __launch_bounds__(128) rmsnorm_kernel(uint16_t* res_out, uint16_t* y, float* rstd,
                                                      float* stats, const uint16_t* res_in,
                                                      const uint16_t* x, const uint16_t* gain,
                                                      float eps, int C) {
  __shared__ float red[8];
  __shared__ float s_rstd[2];
  pdl_trigger();                     // lets the next kernel of a chain be scheduled
  const int64_t row = blockIdx.x;
  const int nchunk = C >> 3;
  const int tid = threadIdx.x;
  const size_t base = size_t(row) * size_t(C);
  uint4 rv[V];
  // two packed double-float accumulators: four independent (hi, lo) lanes
  uint64_t acc_hi[2] = {0ull, 0ull}, acc_lo[2] = {0ull, 0ull};
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int c = tid + i * 128;
    if (c < nchunk) {
      uint4 xv = ld16_once(x + base + size_t(c) * 8);
      uint4 r = xv;
      if (res_in != nullptr) {
        uint4 a = ld16_once(res_in + base + size_t(c) * 8);
        // bf16 + bf16 in fp32, one rounding to bf16 (equals rounding the exact sum)
        r.x = pack_bf16x2(bf16_lo(a.x) + bf16_lo(xv.x), bf16_hi(a.x) + bf16_hi(xv.x));
        r.y = pack_bf16x2(bf16_lo(a.y) + bf16_lo(xv.y), bf16_hi(a.y) + bf16_hi(xv.y));
        r.z = pack_bf16x2(bf16_lo(a.z) + bf16_lo(xv.z), bf16_hi(a.z) + bf16_hi(xv.z));
        r.w = pack_bf16x2(bf16_lo(a.w) + bf16_lo(xv.w), bf16_hi(a.w) + bf16_hi(xv.w));
        stg16(res_out + base + size_t(c) * 8, r);
      }
      rv[i] = r;
      const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint64_t v = bf16x2_to_f2(w[j]);
        f2_df_add(acc_hi[j & 1], acc_lo[j & 1], f2_mul(v, v));   // squares of bf16 are exact
      }
    }
  }
  float ss_hi, ss_lo;
  {
    float h[4], l[4];
    f2_unpack(acc_hi[0], h[0], h[1]);
    f2_unpack(acc_hi[1], h[2], h[3]);
    f2_unpack(acc_lo[0], l[0], l[1]);
    f2_unpack(acc_lo[1], l[2], l[3]);
    ss_hi = h[0];
    ss_lo = l[0];
    for (int k = 1; k < 4; ++k) df_add_df(ss_hi, ss_lo, h[k], l[k]);
  }
  // block sum of squares (double-float), then rstd in fp64 by one thread
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float oh = __shfl_xor_sync(0xffffffffu, ss_hi, o);
    const float ol = __shfl_xor_sync(0xffffffffu, ss_lo, o);
    df_add_df(ss_hi, ss_lo, oh, ol);
  }
  if ((tid & 31) == 0) {
    red[2 * (tid >> 5)] = ss_hi;
    red[2 * (tid >> 5) + 1] = ss_lo;
  }
  __syncthreads();
  if (tid == 0) {
    float h = red[0], l = red[1];
    for (int w = 1; w < 4; ++w) df_add_df(h, l, red[2 * w], red[2 * w + 1]);
    // ms = (h + l) / C as a double-float: q1 + q2
    const float fc = float(C);
    const float q1 = h / fc;
    const float q2 = (fmaf(-q1, fc, h) + l) / fc;   // the fma residual h - q1*C is exact
    // m = ms + eps
    float mh, ml;
    two_sum(q1, eps, mh, ml);
    ml += q2;
    fast_two_sum(mh, ml);
    // rstd = 1/sqrt(m): approximate reciprocal square root, then one Newton
    // step r0 + r0 * (1 - m r0^2) / 2 with the residual formed from exact
    // products (fma), good to about 2^-43 relative
    const float r0 = rsqrtf(mh);
    const float p = r0 * r0, pl = fmaf(r0, r0, -p);          // r0^2 = p + pl exactly
    const float t = mh * p, tl = fmaf(mh, p, -t);            // mh * p = t + tl exactly
    const float e = ((1.0f - t) - tl) - fmaf(mh, pl, ml * p);
    float rs_hi = r0, rs_lo = 0.5f * r0 * e;
    fast_two_sum(rs_hi, rs_lo);
    s_rstd[0] = rs_hi;
    s_rstd[1] = rs_lo;
    rstd[row] = rs_hi;
  }
  __syncthreads();
  const float rs_hi = s_rstd[0], rs_lo = s_rstd[1];
  const uint64_t rs_hi2 = f2_pack(rs_hi, rs_hi);

  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int c = tid + i * 128;
    if (c < nchunk) {
      const uint4 g = ld16_ro(gain + size_t(c) * 8);
      const uint32_t rw[4] = {rv[i].x, rv[i].y, rv[i].z, rv[i].w};
      const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        // t = (r * g) * rstd: r * g is exact; th = fl((r * g) * rs_hi) is within two
        // float ulps of t, so its bf16 rounding is t's unless th lies within three
        // ulps of a bf16 halfway point (low 16 bits near 0x8000); those rare
        // elements are finished with the exact double-float product
        const uint64_t rg = f2_mul(bf16x2_to_f2(rw[j]), bf16x2_to_f2(gw[j]));
        float th0, th1;
        f2_unpack(f2_mul(rg, rs_hi2), th0, th1);
        o[j] = pack_bf16x2(th0, th1);
        const uint32_t b0 = __float_as_uint(th0), b1 = __float_as_uint(th1);
        if (((b0 + 0x8003u) & 0xFFFFu) <= 6u || ((b1 + 0x8003u) & 0xFFFFu) <= 6u) {
          float rg0, rg1;
          f2_unpack(rg, rg0, rg1);
          const uint32_t lo = bf16_round_df(th0, fmaf(rg0, rs_lo, fmaf(rg0, rs_hi, -th0)));
          const uint32_t hi = bf16_round_df(th1, fmaf(rg1, rs_lo, fmaf(rg1, rs_hi, -th1)));
          o[j] = lo | (hi << 16);
        }
        amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(o[j])), fabsf(bf16_hi(o[j]))));
      }
      stg16(y + base + size_t(c) * 8, make_uint4(o[0], o[1], o[2], o[3]));
    }
  }
  if (stats != nullptr) {
    __syncthreads();  // red[] reuse
    const float m = block_reduce_max(amax, red);
    if (tid == 0) atomic_max_nonneg(stats, m);
  }
}

// ------------------------------------------------------------------ abs-max
__global__ void __launch_bounds__(kThreads) absmax_kernel(float* stats, const uint16_t* in,
                                                          int64_t n) {
  __shared__ float red[kThreads / 32];
  float m = 0.0f;
  const int64_t nchunk = n >> 3;
  for (int64_t c = int64_t(blockIdx.x) * kThreads + threadIdx.x; c < nchunk;
       c += int64_t(gridDim.x) * kThreads) {
    const uint4 v = ld16_ro_stream(in + c * 8);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
  }
  if (blockIdx.x == 0) {
    for (int64_t i = nchunk * 8 + threadIdx.x; i < n; i += kThreads) m = fmaxf(m, fabsf(bf16_to_f32(in[i])));
  }
  m = block_reduce_max(m, red);
  if (threadIdx.x == 0) atomic_max_nonneg(stats, m);
}

// ------------------------------------------------------------------ A2
// 16 elements per thread per step: two 16-byte loads, one 16-byte store.
__global__ void __launch_bounds__(kThreads) quantize_kernel(uint8_t* q, float* stats,
                                                            const uint16_t* in, int64_t n,
                                                            float* zero_stat) {
  pdl_wait();                        // in a chain: the preceding kernel has completed
  pdl_trigger();
  if (zero_stat != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *zero_stat = 0.0f;
  const float amax = stats[0];
  const bool zero = !(amax > 0.0f);
  const float inv = zero ? 0.0f : 448.0f / amax;
  if (blockIdx.x == 0 && threadIdx.x == 0) stats[1] = zero ? 1.0f : amax / 448.0f;
  const int64_t nchunk = n >> 4;
  for (int64_t c = int64_t(blockIdx.x) * kThreads + threadIdx.x; c < nchunk;
       c += int64_t(gridDim.x) * kThreads) {
    uint4 o = make_uint4(0, 0, 0, 0);
    if (!zero) {
      const uint4 a = ld16_once(in + c * 16);
      const uint4 b = ld16_once(in + c * 16 + 8);
      const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      uint32_t p[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint16_t lo = f32x2_to_e4m3x2(bf16_lo(w[2 * j]) * inv, bf16_hi(w[2 * j]) * inv);
        const uint16_t hi = f32x2_to_e4m3x2(bf16_lo(w[2 * j + 1]) * inv, bf16_hi(w[2 * j + 1]) * inv);
        p[j] = uint32_t(lo) | (uint32_t(hi) << 16);
      }
      o = make_uint4(p[0], p[1], p[2], p[3]);
    }
    stg16(q + c * 16, o);
  }
  if (blockIdx.x == 0) {
    for (int64_t i = nchunk * 16 + threadIdx.x; i < n; i += kThreads) {
      const uint16_t v = zero ? 0 : f32x2_to_e4m3x2(bf16_to_f32(in[i]) * inv, 0.0f);
      q[i] = uint8_t(v & 0xFF);
    }
  }
}

// ------------------------------------------------------------------ per-row records
// One block per row: the row abs-max, then the row quantised with it.
__global__ void __launch_bounds__(kThreads) quantize_rows_kernel(uint8_t* q, float* row_scale,
                                                                 const uint16_t* w, int cols) {
  __shared__ float red[kThreads / 32];
  __shared__ float s_amax;
  const int64_t row = blockIdx.x;
  const uint16_t* src = w + size_t(row) * cols;
  uint8_t* dst = q + size_t(row) * cols;
  const int nchunk = cols >> 4;
  float m = 0.0f;
  for (int c = threadIdx.x; c < nchunk; c += kThreads) {
    const uint4 a = ld16_ro(src + c * 16), b = ld16_ro(src + c * 16 + 8);
    const uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) m = fmaxf(m, fmaxf(fabsf(bf16_lo(v[j])), fabsf(bf16_hi(v[j]))));
  }
  m = block_reduce_max(m, red);
  if (threadIdx.x == 0) s_amax = m;
  __syncthreads();
  const float amax = s_amax;
  const bool zero = !(amax > 0.0f);
  const float inv = zero ? 0.0f : 448.0f / amax;
  if (threadIdx.x == 0) row_scale[row] = zero ? 1.0f : amax / 448.0f;
  for (int c = threadIdx.x; c < nchunk; c += kThreads) {
    uint4 o = make_uint4(0, 0, 0, 0);
    if (!zero) {
      const uint4 a = ld16_ro(src + c * 16), b = ld16_ro(src + c * 16 + 8);
      const uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      uint32_t p[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint16_t lo = f32x2_to_e4m3x2(bf16_lo(v[2 * j]) * inv, bf16_hi(v[2 * j]) * inv);
        const uint16_t hi = f32x2_to_e4m3x2(bf16_lo(v[2 * j + 1]) * inv, bf16_hi(v[2 * j + 1]) * inv);
        p[j] = uint32_t(lo) | (uint32_t(hi) << 16);
      }
      o = make_uint4(p[0], p[1], p[2], p[3]);
    }
    stg16(dst + c * 16, o);
  }
}

// ------------------------------------------------------------------ A4 (standalone)
// 8 outputs per thread per step: 16 bytes of gate, 16 bytes of up (swiglu8 in common.cuh).
__device__ __forceinline__ float absmax8(uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float m = 0.0f;
#pragma unroll
  for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
  return m;
}

__global__ void __launch_bounds__(kThreads) swiglu_absmax_kernel(uint16_t* h, float* stats,
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
    const uint4 hv = swiglu8(ld16_ro_stream(src), ld16_ro_stream(src + H));
    m = fmaxf(m, absmax8(hv));
    if (h != nullptr) stg16(h + row * H + c * 8, hv);
  }
  m = block_reduce_max(m, red);
  if (threadIdx.x == 0) atomic_max_nonneg(stats, m);
}

__global__ void __launch_bounds__(kThreads) swiglu_requant_kernel(uint8_t* hq, float* stats,
                                                                  const uint16_t* gu, int64_t N,
                                                                  int64_t H) {
  const float amax = stats[0];
  const bool zero = !(amax > 0.0f);
  const float inv = zero ? 0.0f : 448.0f / amax;
  if (blockIdx.x == 0 && threadIdx.x == 0) stats[1] = zero ? 1.0f : amax / 448.0f;
  const int64_t per_row = H >> 3;
  const int64_t total = N * per_row;
  for (int64_t i = int64_t(blockIdx.x) * kThreads + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * kThreads) {
    const int64_t row = i / per_row, c = i - row * per_row;
    const uint16_t* src = gu + row * 2 * H + c * 8;
    uint2 o = make_uint2(0, 0);
    if (!zero) {
      const uint4 hv = swiglu8(ld16_ro_stream(src), ld16_ro_stream(src + H));
      const uint32_t w[4] = {hv.x, hv.y, hv.z, hv.w};
      uint32_t p[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint16_t lo = f32x2_to_e4m3x2(bf16_lo(w[2 * j]) * inv, bf16_hi(w[2 * j]) * inv);
        const uint16_t hi = f32x2_to_e4m3x2(bf16_lo(w[2 * j + 1]) * inv, bf16_hi(w[2 * j + 1]) * inv);
        p[j] = uint32_t(lo) | (uint32_t(hi) << 16);
      }
      o = make_uint2(p[0], p[1]);
    }
    *reinterpret_cast<uint2*>(hq + row * H + c * 8) = o;
  }
}

// ------------------------------------------------------------------ A7
__global__ void __launch_bounds__(kThreads) silu_mul_kernel(uint16_t* g, const uint16_t* u,
                                                            int64_t n) {
  pdl_wait();
  pdl_trigger();
  const int64_t nchunk = n >> 3;
  for (int64_t c = int64_t(blockIdx.x) * kThreads + threadIdx.x; c < nchunk;
       c += int64_t(gridDim.x) * kThreads) {
    const uint4 hv = swiglu8(ld16_once(g + c * 8), ld16_once(u + c * 8));
    stg16(g + c * 8, hv);
  }
}

int grid_for(int64_t work_items, int blocks_per_sm) {
  const int64_t cap = int64_t(num_sms()) * blocks_per_sm;
  int64_t need = (work_items + kThreads - 1) / kThreads;
  if (need < 1) need = 1;
  return int(need < cap ? need : cap);
}

}  // namespace

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return kNumSMsHint;
  if (g_sm_count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = kNumSMsHint;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

cudaError_t launch_rmsnorm(uint16_t* res_out, uint16_t* y, float* rstd, float* stats,
                           const uint16_t* res_in, const uint16_t* x, const uint16_t* gain,
                           float eps, int64_t N, int C, cudaStream_t s) {
  if (stats != nullptr) {
    cudaError_t e = cudaMemsetAsync(stats, 0, sizeof(float), s);
    if (e != cudaSuccess) return e;
  }
  if (N == 0) return cudaSuccess;
  const int per_thread = (C / 8 + 127) / 128;
  const dim3 grid(static_cast<unsigned>(N));
  if (per_thread <= 1)
    rmsnorm_kernel<1><<<grid, 128, 0, s>>>(res_out, y, rstd, stats, res_in, x, gain, eps, C);
  else if (per_thread <= 2)
    rmsnorm_kernel<2><<<grid, 128, 0, s>>>(res_out, y, rstd, stats, res_in, x, gain, eps, C);
  else if (per_thread <= 4)
    rmsnorm_kernel<4><<<grid, 128, 0, s>>>(res_out, y, rstd, stats, res_in, x, gain, eps, C);
  else if (per_thread <= 8)
    rmsnorm_kernel<8><<<grid, 128, 0, s>>>(res_out, y, rstd, stats, res_in, x, gain, eps, C);
  else
    rmsnorm_kernel<16><<<grid, 128, 0, s>>>(res_out, y, rstd, stats, res_in, x, gain, eps, C);
  return cudaGetLastError();
}

cudaError_t launch_absmax(float* stats, const uint16_t* in, int64_t n, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(stats, 0, sizeof(float), s);
  if (e != cudaSuccess) return e;
  if (n == 0) return cudaSuccess;
  absmax_kernel<<<grid_for(n / 8 + 1, 8), kThreads, 0, s>>>(stats, in, n);
  return cudaGetLastError();
}

cudaError_t launch_quantize(uint8_t* q, float* stats, const uint16_t* in, int64_t n,
                            cudaStream_t s, bool pdl, float* zero_stat) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid_for(n / 16 + 1, 8));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, quantize_kernel, q, stats, in, n, zero_stat);
}

cudaError_t launch_quantize_rows(uint8_t* q, float* row_scale, const uint16_t* w, int64_t rows,
                                 int cols, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  quantize_rows_kernel<<<unsigned(rows), kThreads, 0, s>>>(q, row_scale, w, cols);
  return cudaGetLastError();
}

cudaError_t launch_swiglu_absmax(uint16_t* h, float* stats, const uint16_t* gate_up, int64_t N,
                                 int64_t H, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(stats, 0, sizeof(float), s);
  if (e != cudaSuccess) return e;
  if (N == 0) return cudaSuccess;
  swiglu_absmax_kernel<<<grid_for(N * (H / 8), 8), kThreads, 0, s>>>(h, stats, gate_up, N, H);
  return cudaGetLastError();
}

cudaError_t launch_swiglu_requant(uint8_t* hq, float* stats, const uint16_t* gate_up, int64_t N,
                                  int64_t H, cudaStream_t s) {
  swiglu_requant_kernel<<<grid_for(N * (H / 8) + 1, 8), kThreads, 0, s>>>(hq, stats, gate_up, N, H);
  return cudaGetLastError();
}

cudaError_t launch_silu_mul(uint16_t* g, const uint16_t* u, int64_t n, bool pdl, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid_for(n / 8, 4));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, silu_mul_kernel, g, u, n);
}

}  // namespace qffn
