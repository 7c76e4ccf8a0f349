// Internal launchers of the qffn kernels.  Each enqueues work on `s` and
// returns the CUDA error of the launch; argument checking is done by the
// C-ABI layer (api.cu) before any of these is called.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace qffn {

// Number of SMs of the current device (cached per device).
int num_sms();

// ---- elementwise / reduction kernels (elementwise.cu)
cudaError_t launch_rmsnorm(uint16_t* res_out, uint16_t* y, float* rstd, float* stats,
                           const uint16_t* res_in, const uint16_t* x, const uint16_t* gain,
                           float eps, int64_t N, int C, cudaStream_t s);
cudaError_t launch_absmax(float* stats, const uint16_t* in, int64_t n, cudaStream_t s);
// Chained launches (pdl): the kernel is a programmatic dependent launch; it
// waits for the preceding kernel on `s` before touching global memory.
// zero_stat (optional): set to 0 by the kernel once that wait is over, so a
// later kernel of the same chain can record an abs-max there without a
// memset (which would break the chain).
cudaError_t launch_quantize(uint8_t* q, float* stats, const uint16_t* in, int64_t n,
                            cudaStream_t s, bool pdl = false, float* zero_stat = nullptr);
cudaError_t launch_quantize_rows(uint8_t* q, float* row_scale, const uint16_t* w, int64_t rows,
                                 int cols, cudaStream_t s);
// SwiGLU over gate_up [N, 2H]: writes h (if non-NULL) and max|h| into stats[0]
// (zeroed first).
cudaError_t launch_swiglu_absmax(uint16_t* h, float* stats, const uint16_t* gate_up, int64_t N,
                                 int64_t H, cudaStream_t s);
// Recomputes h from gate_up and quantises it with stats[0]; writes stats[1].
cudaError_t launch_swiglu_requant(uint8_t* hq, float* stats, const uint16_t* gate_up, int64_t N,
                                  int64_t H, cudaStream_t s);
cudaError_t launch_silu_mul(uint16_t* g, const uint16_t* u, int64_t n, bool pdl, cudaStream_t s);

// ---- tcgen05 FP8 GEMMs (gemm_fp8.cu)
// out[M,N] = bf16(a_scale*w_scale * A[M,K] . W[N,K]^T + bias[N] (+ out[M,N])):
// bias (bf16, optional) and, with `accumulate`, the previous contents of out
// are added to the scaled fp32 accumulator before the rounding.  With a_mn
// (w_mn) the operand is given MN-major, i.e. A as [K, M] (W as [K, N]) with
// the M (N) index contiguous; M (N) must then be a multiple of 16.
cudaError_t launch_gemm_bf16(uint16_t* out, const uint8_t* A, const float* a_scale,
                             const uint8_t* W, const float* w_scale, int64_t M, int64_t N,
                             int64_t K, cudaStream_t s, const uint16_t* bias = nullptr,
                             bool accumulate = false, bool a_mn = false, bool w_mn = false,
                             bool pdl = false);
// h[M,H] = bf16(silu(g)*u) with g, u the bf16-rounded gate / up products of
// W1 = [2H, K]; records max|h| into stats_h[0] (zeroed first by a memset,
// or, with `chained`, already zeroed by an earlier kernel of the chain: the
// GEMM is then a programmatic dependent launch).
cudaError_t launch_gemm_swiglu(uint16_t* h, float* stats_h, const uint8_t* A, const float* a_scale,
                               const uint8_t* W1, const float* w_scale, int64_t M, int64_t H,
                               int64_t K, cudaStream_t s, bool chained = false);
// hq[M,H] = e4m3(h * 448 / stats_h[0]) for the h of launch_gemm_swiglu, with
// the abs-max given (not recorded); writes stats_h[1] = scale.
cudaError_t launch_gemm_swiglu_quant(uint8_t* hq, float* stats_h, const uint8_t* A,
                                     const float* a_scale, const uint8_t* W1, const float* w_scale,
                                     int64_t M, int64_t H, int64_t K, cudaStream_t s,
                                     bool pdl = false);
// d_gu[M,2H] = SwiGLU gradient for dh [M,H] and the gate|up product of A and
// W1 = [2H, K] (the recompute of gate_up fused with swiglu_backward); records
// max|d_gu| into stats[0] (zeroed first).
cudaError_t launch_gemm_swiglu_bwd(uint16_t* d_gu, float* stats, const uint16_t* dh,
                                   const uint8_t* A, const float* a_scale, const uint8_t* W1,
                                   const float* w_scale, int64_t M, int64_t H, int64_t K,
                                   cudaStream_t s);
// Reads and clears the GEMM kernels' device status word of the current device.
cudaError_t gemm_take_status(unsigned int* status);
// SM clock cycles and nanoseconds that the first CTA of the most recent GEMM
// launch on the current device spent from its start to its end.
cudaError_t gemm_clock_sample(unsigned long long out[2]);
// Failure-path self-test of the GEMMs' bounded barrier wait (one CTA, two
// waits; out[4] as qffn_selftest_bounded_wait documents).
cudaError_t launch_wait_selftest(unsigned long long* out, int arrive, unsigned long long limit_ns,
                                 cudaStream_t s);

// ---- FP8 backward (backward.cu)
// out[Cc, R] = in[R, Cc]^T for E4M3 codes; R and Cc multiples of 16.
cudaError_t launch_transpose_u8(uint8_t* out, const uint8_t* in, int64_t R, int64_t Cc,
                                cudaStream_t s);
// dgu[N, 2H] = (dh * u * silu'(g) | dh * silu(g)) from gu = [N, 2H] (gate
// first) and dh [N, H]; records max|dgu| into stats[0] (zeroed first).
cudaError_t launch_swiglu_backward(uint16_t* dgu, float* stats, const uint16_t* dh,
                                   const uint16_t* gu, int64_t N, int64_t H, cudaStream_t s);

// ---- decode GEMVs (decode.cu)
// out0[r] = bf16(s0[r] * W0[r,:] . x); with W1 != NULL also out1 from W1, s1.
// With `pdl` the launch is a programmatic dependent launch that issues its
// first weight loads before waiting for the preceding kernel.
cudaError_t launch_gemv(uint16_t* out0, uint16_t* out1, const uint16_t* x, const uint8_t* w0,
                        const float* s0, const uint8_t* w1, const float* s1, int64_t rows,
                        int64_t cols, bool pdl, cudaStream_t s);
// out[r] = bf16(s[r] * W[r,:] . h) with h = bf16(silu(g) * u) formed while the
// input vector is staged (the fused-SiLU-input arm's down GEMV).
cudaError_t launch_gemv_silu_input(uint16_t* out, const uint16_t* g, const uint16_t* u,
                                   const uint8_t* w, const float* row_scale, int64_t rows,
                                   int64_t cols, cudaStream_t s);
// The whole decode FFN: the dual GEMV (g, u), then the down GEMV on
// h = bf16(silu(g) * u) formed in its prologue, launched as a programmatic
// dependent launch so its first weight loads overlap the dual GEMV's tail.
// `early`: the dual GEMV may read w_gate and w_up before the preceding kernel
// on the stream has finished.  Same bits as launch_gemv + launch_silu_mul +
// launch_gemv.
cudaError_t launch_decode(uint16_t* out, const uint16_t* x, const uint8_t* w_gate,
                          const float* s_gate, const uint8_t* w_up, const float* s_up,
                          const uint8_t* w_down, const float* s_down, int64_t C, int64_t H,
                          uint16_t* g, uint16_t* u, bool early, cudaStream_t s);
// Reads and clears the decode kernels' device status word of the current device.
cudaError_t decode_take_status(unsigned int* status);

}  // namespace qffn
