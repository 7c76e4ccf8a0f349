// C ABI of libqffn: argument checking and the orchestration of the kernels.
// The contract of every entry point is stated in include/qffn.h.
#include <math.h>
#include <stdint.h>

#include <nvtx3/nvToolsExt.h>

#include "../../include/qffn.h"
#include "launch.h"

namespace {

using qffn::num_sms;

constexpr int kAbiVersion = 1;

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }
inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline qffn_status from_cuda(cudaError_t e) { return e == cudaSuccess ? QFFN_OK : QFFN_ERR_CUDA; }

// An NVTX range named after the entry point around everything it enqueues, so
// a timeline (Nsight Systems, ncu's NVTX filters) shows which call launched
// which kernels.  Header-only NVTX: without an attached tool a push / pop is
// a check of a function pointer.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
#define QFFN_RANGE() NvtxRange qffn_nvtx_range_(__func__)

#define QFFN_REQUIRE(cond, err) \
  do {                          \
    if (!(cond)) return (err);  \
  } while (0)
#define QFFN_PTR(p) QFFN_REQUIRE((p) != nullptr, QFFN_ERR_INVALID_ARG)
#define QFFN_ALIGNED(p) QFFN_REQUIRE((p) == nullptr || aligned16(p), QFFN_ERR_MISALIGNED)
// fp32 scalars and vectors (stats pairs, scales, rstd, row scales): natural alignment
#define QFFN_ALIGNED4(p) QFFN_REQUIRE((reinterpret_cast<uintptr_t>(p) & 3u) == 0, QFFN_ERR_MISALIGNED)
#define QFFN_CUDA(expr)                              \
  do {                                               \
    cudaError_t e_ = (expr);                         \
    if (e_ != cudaSuccess) return QFFN_ERR_CUDA;     \
  } while (0)

constexpr int64_t kMaxDim = int64_t(1) << 20;
constexpr int64_t kMaxRows = (int64_t(1) << 31) - 1;

// workspace layout of qffn_forward: y [N,C] bf16 | yq [N,C] e4m3 | h [N,H] bf16 | hq [N,H] e4m3
void forward_offsets(int64_t N, int64_t C, int64_t H, size_t off[5]) {
  off[0] = 0;
  off[1] = round_up(off[0] + size_t(N) * size_t(C) * 2, 256);
  off[2] = round_up(off[1] + size_t(N) * size_t(C), 256);
  off[3] = round_up(off[2] + size_t(N) * size_t(H) * 2, 256);
  off[4] = round_up(off[3] + size_t(N) * size_t(H), 256);
}

// backward_qmm workspace: dout_q [N,OC] E4M3
void bqmm_offsets(int64_t N, int64_t IC, int64_t OC, size_t off[2]) {
  (void)IC;
  off[0] = 0;
  off[1] = round_up(size_t(N) * size_t(OC), 256);
}

// FFN backward workspace: dh [N,H] bf16 | d_gu [N,2H] bf16 | the larger of the
// two backward_qmm workspaces
void ffn_bwd_offsets(int64_t N, int64_t C, int64_t H, size_t off[4]) {
  size_t down[2], up[2];
  bqmm_offsets(N, H, C, down);
  bqmm_offsets(N, C, 2 * H, up);
  off[0] = 0;
  off[1] = round_up(size_t(N) * size_t(H) * 2, 256);
  off[2] = round_up(off[1] + size_t(N) * size_t(2 * H) * 2, 256);
  off[3] = off[2] + (down[1] > up[1] ? down[1] : up[1]);
}

qffn_status check_bqmm_shape(int64_t N, int64_t IC, int64_t OC) {
  QFFN_REQUIRE(N >= 0 && IC >= 0 && OC >= 0, QFFN_ERR_INVALID_ARG);
  QFFN_REQUIRE(N % 16 == 0 && N <= kMaxRows, QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_REQUIRE(IC % 32 == 0 && IC >= 32 && IC <= kMaxDim, QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_REQUIRE(OC % 32 == 0 && OC >= 32 && OC <= kMaxDim, QFFN_ERR_UNSUPPORTED_SHAPE);
  return QFFN_OK;
}

// The FP8 branch of backward_qmm on pointers already checked; ws holds dout_q.
// The page transposes W, dout_q and inp_q so that both matmuls are
// K-contiguous; here the tensor cores read them MN-major where they lie.
cudaError_t run_backward_qmm(uint16_t* dinp, uint16_t* dw, float* stats_dout, const uint16_t* dout,
                             const uint8_t* inp_q, const float* inp_scale, const uint8_t* w,
                             const float* w_scale, int64_t N, int64_t IC, int64_t OC,
                             bool accumulate, uint8_t* ws, cudaStream_t s) {
  uint8_t* dq = ws;
  cudaError_t e;
  // quantize_with_abs_max(dout.Quant, scale, dout.Value, dout.Quant.abs_max())
  if ((e = qffn::launch_quantize(dq, stats_dout, dout, N * OC, s)) != cudaSuccess) return e;
  if (dinp != nullptr) {
    // dinp[N,IC] = dout_q[N,OC] . W[OC,IC], scales W.scale * dout.scale (W read MN-major)
    if ((e = qffn::launch_gemm_bf16(dinp, dq, stats_dout + 1, w, w_scale, N, IC, OC, s, nullptr,
                                    false, false, true)) != cudaSuccess)
      return e;
  }
  // no tokens: the weight gradient is a sum over nothing (0, or unchanged when accumulating)
  if (N == 0) return accumulate ? cudaSuccess : cudaMemsetAsync(dw, 0, size_t(OC) * size_t(IC) * 2, s);
  // dW[OC,IC] (+)= dout_q[N,OC]^T . inp_q[N,IC], scales inp.scale * dout.scale (both MN-major)
  return qffn::launch_gemm_bf16(dw, dq, stats_dout + 1, inp_q, inp_scale, OC, IC, N, s, nullptr,
                                accumulate, true, true);
}

// decode workspace: g [H] bf16 (holds h after the call) | u [H] bf16, each
// 256-byte aligned
void decode_offsets(int64_t H, size_t off[3]) {
  const size_t vec = round_up(size_t(H) * 2, 256);
  off[0] = 0;                                  // g, then h
  off[1] = vec;                                // u
  off[2] = 2 * vec;                            // end
}

qffn_status check_forward_shape(int64_t B, int64_t T, int64_t C, int64_t H) {
  QFFN_REQUIRE(B >= 0 && T >= 0 && C >= 0 && H >= 0, QFFN_ERR_INVALID_ARG);
  QFFN_REQUIRE(B == 0 || T <= kMaxRows / B, QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_REQUIRE(C % 128 == 0 && C >= 128 && C <= 16384, QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_REQUIRE(H % 128 == 0 && H >= 128 && H <= kMaxDim, QFFN_ERR_UNSUPPORTED_SHAPE);
  return QFFN_OK;
}

}  // namespace

extern "C" {

const char* qffn_status_string(qffn_status s) {
  switch (s) {
    case QFFN_OK: return "ok";
    case QFFN_ERR_INVALID_ARG: return "invalid argument";
    case QFFN_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case QFFN_ERR_MISALIGNED: return "misaligned pointer";
    case QFFN_ERR_CUDA: return "CUDA error";
    case QFFN_ERR_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

int qffn_abi_version(void) { return kAbiVersion; }

qffn_status qffn_check_status(qffn_stream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return QFFN_ERR_CUDA;
  unsigned int st = 0, sd = 0;
  if (qffn::gemm_take_status(&st) != cudaSuccess) return QFFN_ERR_CUDA;
  if (qffn::decode_take_status(&sd) != cudaSuccess) return QFFN_ERR_CUDA;
  return (st | sd) != 0 ? QFFN_ERR_TIMEOUT : QFFN_OK;
}

qffn_status qffn_gemm_clock_sample(uint64_t* out, qffn_stream_t stream) {
  QFFN_PTR(out);
  if (cudaStreamSynchronize(stream) != cudaSuccess) return QFFN_ERR_CUDA;
  unsigned long long v[2] = {0ull, 0ull};
  if (qffn::gemm_clock_sample(v) != cudaSuccess) return QFFN_ERR_CUDA;
  out[0] = v[0];
  out[1] = v[1];
  return QFFN_OK;
}

qffn_status qffn_selftest_bounded_wait(uint64_t* out, int arrive, int64_t limit_ns,
                                       qffn_stream_t stream) {
  QFFN_RANGE();
  QFFN_PTR(out);
  QFFN_REQUIRE(limit_ns >= 100000 && limit_ns <= 2000000000, QFFN_ERR_INVALID_ARG);
  QFFN_REQUIRE(reinterpret_cast<uintptr_t>(out) % 8 == 0, QFFN_ERR_MISALIGNED);
  return from_cuda(qffn::launch_wait_selftest(reinterpret_cast<unsigned long long*>(out),
                                              arrive != 0, (unsigned long long)limit_ns, stream));
}

qffn_status qffn_rmsnorm_absmax(uint16_t* res_out, uint16_t* y, float* rstd, float* stats,
                                const uint16_t* res_in, const uint16_t* x, const uint16_t* gain,
                                float eps, int64_t N, int64_t C, qffn_stream_t stream) {
  QFFN_RANGE();
  QFFN_PTR(y); QFFN_PTR(rstd); QFFN_PTR(x); QFFN_PTR(gain);
  if (res_in != nullptr) QFFN_PTR(res_out);
  QFFN_REQUIRE(N >= 0 && C >= 0, QFFN_ERR_INVALID_ARG);
  QFFN_REQUIRE(isfinite(eps) && eps >= 0.0f, QFFN_ERR_INVALID_ARG);
  QFFN_REQUIRE(N <= kMaxRows, QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_REQUIRE(C % 8 == 0 && C >= 8 && C <= 16384, QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_ALIGNED(y); QFFN_ALIGNED(x); QFFN_ALIGNED(gain); QFFN_ALIGNED4(rstd);
  if (res_in != nullptr) { QFFN_ALIGNED(res_in); QFFN_ALIGNED(res_out); }
  QFFN_ALIGNED4(stats);
  return from_cuda(qffn::launch_rmsnorm(res_out, y, rstd, stats, res_in, x, gain, eps, N, int(C),
                                        stream));
}

qffn_status qffn_absmax(float* stats, const uint16_t* in, int64_t n, qffn_stream_t stream) {
  QFFN_RANGE();
  QFFN_PTR(stats); QFFN_PTR(in);
  QFFN_REQUIRE(n >= 0, QFFN_ERR_INVALID_ARG);
  QFFN_ALIGNED4(stats); QFFN_ALIGNED(in);
  return from_cuda(qffn::launch_absmax(stats, in, n, stream));
}

qffn_status qffn_quantize(uint8_t* q, float* stats, const uint16_t* in, int64_t n,
                          qffn_stream_t stream) {
  QFFN_RANGE();
  QFFN_PTR(q); QFFN_PTR(stats); QFFN_PTR(in);
  QFFN_REQUIRE(n >= 0, QFFN_ERR_INVALID_ARG);
  QFFN_ALIGNED(q); QFFN_ALIGNED4(stats); QFFN_ALIGNED(in);
  return from_cuda(qffn::launch_quantize(q, stats, in, n, stream));
}

qffn_status qffn_quantize_rows(uint8_t* q, float* row_scale, const uint16_t* w, int64_t rows,
                               int64_t cols, qffn_stream_t stream) {
  QFFN_RANGE();
  QFFN_PTR(q); QFFN_PTR(row_scale); QFFN_PTR(w);
  QFFN_REQUIRE(rows >= 0 && cols >= 0, QFFN_ERR_INVALID_ARG);
  QFFN_REQUIRE(rows <= kMaxRows, QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_REQUIRE(cols % 16 == 0 && cols >= 16 && cols <= 65536, QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_ALIGNED(q); QFFN_ALIGNED4(row_scale); QFFN_ALIGNED(w);
  return from_cuda(qffn::launch_quantize_rows(q, row_scale, w, rows, int(cols), stream));
}

qffn_status qffn_fp8_gemm_scaled(uint16_t* out, const uint8_t* A, const float* a_scale,
                                 const uint8_t* W, const float* w_scale, int64_t M, int64_t N,
                                 int64_t K, qffn_stream_t stream) {
  QFFN_RANGE();
  QFFN_PTR(out); QFFN_PTR(A); QFFN_PTR(a_scale); QFFN_PTR(W); QFFN_PTR(w_scale);
  QFFN_REQUIRE(M >= 0 && N >= 0 && K >= 0, QFFN_ERR_INVALID_ARG);
  QFFN_REQUIRE(M <= kMaxRows, QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_REQUIRE(N % 32 == 0 && N >= 32 && N <= kMaxDim, QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_REQUIRE(K % 16 == 0 && K >= 16 && K <= kMaxDim, QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_REQUIRE((M + 127) / 128 * ((N + 255) / 256) < (int64_t(1) << 31), QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_ALIGNED(out); QFFN_ALIGNED(A); QFFN_ALIGNED(W); QFFN_ALIGNED4(a_scale); QFFN_ALIGNED4(w_scale);
  return from_cuda(qffn::launch_gemm_bf16(out, A, a_scale, W, w_scale, M, N, K, stream));
}

qffn_status qffn_qmm(uint16_t* out, uint8_t* q, float* stats, const uint16_t* in,
                     const uint16_t* bias, const uint8_t* W, const float* w_scale, int64_t M,
                     int64_t N, int64_t K, qffn_stream_t stream) {
  QFFN_RANGE();
  QFFN_PTR(out); QFFN_PTR(q); QFFN_PTR(stats); QFFN_PTR(in); QFFN_PTR(W); QFFN_PTR(w_scale);
  QFFN_REQUIRE(M >= 0 && N >= 0 && K >= 0, QFFN_ERR_INVALID_ARG);
  QFFN_REQUIRE(M <= kMaxRows, QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_REQUIRE(N % 32 == 0 && N >= 32 && N <= kMaxDim, QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_REQUIRE(K % 16 == 0 && K >= 16 && K <= kMaxDim, QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_REQUIRE((M + 127) / 128 * ((N + 255) / 256) < (int64_t(1) << 31), QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_ALIGNED(out); QFFN_ALIGNED(q); QFFN_ALIGNED4(stats); QFFN_ALIGNED(in); QFFN_ALIGNED(bias);
  QFFN_ALIGNED(W); QFFN_ALIGNED4(w_scale);
  // quantize_with_abs_max: q, stats[1]; then the scaled matmul with the bias
  QFFN_CUDA(qffn::launch_quantize(q, stats, in, M * K, stream));
  return from_cuda(qffn::launch_gemm_bf16(out, q, stats + 1, W, w_scale, M, N, K, stream, bias));
}

qffn_status qffn_gate_up_swiglu(uint16_t* h, float* stats_h, const uint8_t* yq,
                                const float* y_scale, const uint8_t* w1, const float* w1_scale,
                                int64_t N, int64_t C, int64_t H, qffn_stream_t stream) {
  QFFN_RANGE();
  QFFN_PTR(h); QFFN_PTR(stats_h); QFFN_PTR(yq); QFFN_PTR(y_scale); QFFN_PTR(w1); QFFN_PTR(w1_scale);
  QFFN_REQUIRE(N >= 0 && C >= 0 && H >= 0, QFFN_ERR_INVALID_ARG);
  QFFN_REQUIRE(N <= kMaxRows, QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_REQUIRE(C % 16 == 0 && C >= 16 && C <= kMaxDim, QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_REQUIRE(H % 128 == 0 && H >= 128 && H <= kMaxDim, QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_REQUIRE((N + 127) / 128 * (H / 128) < (int64_t(1) << 31), QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_ALIGNED(h); QFFN_ALIGNED4(stats_h); QFFN_ALIGNED(yq); QFFN_ALIGNED(w1);
  QFFN_ALIGNED4(y_scale); QFFN_ALIGNED4(w1_scale);
  return from_cuda(qffn::launch_gemm_swiglu(h, stats_h, yq, y_scale, w1, w1_scale, N, H, C, stream));
}

qffn_status qffn_swiglu_quant(uint16_t* h, uint8_t* hq, float* stats, const uint16_t* gate_up,
                              int64_t N, int64_t H, qffn_stream_t stream) {
  QFFN_RANGE();
  QFFN_PTR(hq); QFFN_PTR(stats); QFFN_PTR(gate_up);
  QFFN_REQUIRE(N >= 0 && H >= 0, QFFN_ERR_INVALID_ARG);
  QFFN_REQUIRE(H % 8 == 0 && H >= 8 && H <= kMaxDim && N <= kMaxRows, QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_ALIGNED(h); QFFN_ALIGNED(hq); QFFN_ALIGNED4(stats); QFFN_ALIGNED(gate_up);
  QFFN_CUDA(qffn::launch_swiglu_absmax(h, stats, gate_up, N, H, stream));
  if (h != nullptr) return from_cuda(qffn::launch_quantize(hq, stats, h, N * H, stream));
  return from_cuda(qffn::launch_swiglu_requant(hq, stats, gate_up, N, H, stream));
}

qffn_status qffn_swiglu_forward_quant(uint8_t* hq, float* stats, const uint16_t* gate_up,
                                      int64_t N, int64_t H, qffn_stream_t stream) {
  QFFN_RANGE();
  QFFN_PTR(hq); QFFN_PTR(stats); QFFN_PTR(gate_up);
  QFFN_REQUIRE(N >= 0 && H >= 0, QFFN_ERR_INVALID_ARG);
  QFFN_REQUIRE(H % 8 == 0 && H >= 8 && H <= kMaxDim && N <= kMaxRows, QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_ALIGNED(hq); QFFN_ALIGNED4(stats); QFFN_ALIGNED(gate_up);
  return from_cuda(qffn::launch_swiglu_requant(hq, stats, gate_up, N, H, stream));
}

qffn_status qffn_gate_up_swiglu_quant(uint8_t* hq, float* stats_h, const uint8_t* yq,
                                      const float* y_scale, const uint8_t* w1,
                                      const float* w1_scale, int64_t N, int64_t C, int64_t H,
                                      qffn_stream_t stream) {
  QFFN_RANGE();
  QFFN_PTR(hq); QFFN_PTR(stats_h); QFFN_PTR(yq); QFFN_PTR(y_scale); QFFN_PTR(w1); QFFN_PTR(w1_scale);
  QFFN_REQUIRE(N >= 0 && C >= 0 && H >= 0, QFFN_ERR_INVALID_ARG);
  QFFN_REQUIRE(N <= kMaxRows, QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_REQUIRE(C % 16 == 0 && C >= 16 && C <= kMaxDim, QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_REQUIRE(H % 128 == 0 && H >= 128 && H <= kMaxDim, QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_REQUIRE((N + 127) / 128 * (H / 128) < (int64_t(1) << 31), QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_ALIGNED(hq); QFFN_ALIGNED4(stats_h); QFFN_ALIGNED(yq); QFFN_ALIGNED(w1);
  QFFN_ALIGNED4(y_scale); QFFN_ALIGNED4(w1_scale);
  return from_cuda(
      qffn::launch_gemm_swiglu_quant(hq, stats_h, yq, y_scale, w1, w1_scale, N, H, C, stream));
}

size_t qffn_forward_workspace_size(int64_t B, int64_t T, int64_t C, int64_t H) {
  if (check_forward_shape(B, T, C, H) != QFFN_OK) return 0;
  size_t off[5];
  forward_offsets(B * T, C, H, off);
  return off[4] > 0 ? off[4] : 256;
}

qffn_status qffn_forward_workspace_offsets(int64_t B, int64_t T, int64_t C, int64_t H,
                                           size_t offsets[4]) {
  QFFN_PTR(offsets);
  const qffn_status st = check_forward_shape(B, T, C, H);
  if (st != QFFN_OK) return st;
  size_t off[5];
  forward_offsets(B * T, C, H, off);
  for (int i = 0; i < 4; ++i) offsets[i] = off[i];
  return QFFN_OK;
}

qffn_status qffn_forward(uint16_t* res_out, uint16_t* out, float* rstd, float* stats_y,
                         float* stats_h, const uint16_t* res_in, const uint16_t* x,
                         const uint16_t* gain, float eps, const uint8_t* w1,
                         const float* w1_scale, const uint8_t* w2, const float* w2_scale,
                         int64_t B, int64_t T, int64_t C, int64_t H, void* workspace,
                         size_t workspace_bytes, qffn_stream_t stream) {
  QFFN_RANGE();
  QFFN_PTR(out); QFFN_PTR(rstd); QFFN_PTR(stats_y); QFFN_PTR(stats_h); QFFN_PTR(x);
  QFFN_PTR(gain); QFFN_PTR(w1); QFFN_PTR(w1_scale); QFFN_PTR(w2); QFFN_PTR(w2_scale);
  QFFN_PTR(workspace);
  if (res_in != nullptr) QFFN_PTR(res_out);
  QFFN_REQUIRE(isfinite(eps) && eps >= 0.0f, QFFN_ERR_INVALID_ARG);
  const qffn_status st = check_forward_shape(B, T, C, H);
  if (st != QFFN_OK) return st;
  const int64_t N = B * T;
  size_t off[5];
  forward_offsets(N, C, H, off);
  QFFN_REQUIRE(workspace_bytes >= off[4], QFFN_ERR_INVALID_ARG);
  QFFN_REQUIRE(aligned256(workspace), QFFN_ERR_MISALIGNED);
  QFFN_ALIGNED(out); QFFN_ALIGNED4(rstd); QFFN_ALIGNED4(stats_y); QFFN_ALIGNED4(stats_h);
  QFFN_ALIGNED(x); QFFN_ALIGNED(gain); QFFN_ALIGNED(w1); QFFN_ALIGNED(w2);
  QFFN_ALIGNED4(w1_scale); QFFN_ALIGNED4(w2_scale);
  if (res_in != nullptr) { QFFN_ALIGNED(res_in); QFFN_ALIGNED(res_out); }

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint16_t* y = reinterpret_cast<uint16_t*>(ws + off[0]);
  uint8_t* yq = ws + off[1];
  uint16_t* h = reinterpret_cast<uint16_t*>(ws + off[2]);
  uint8_t* hq = ws + off[3];

  // The launches after A1 form a chain of programmatic dependent launches:
  // each kernel is scheduled while its predecessor drains and waits for it
  // to complete before touching global memory.  The stats_h[0] word is
  // zeroed by A2's kernel instead of a memset, which would break the chain.
  // A1: r, y, rstd, stats_y[0]
  QFFN_CUDA(qffn::launch_rmsnorm(res_out, y, rstd, stats_y, res_in, x, gain, eps, N, int(C), stream));
  // A2: yq, stats_y[1]; stats_h[0] = 0
  QFFN_CUDA(qffn::launch_quantize(yq, stats_y, y, N * C, stream, true, stats_h));
  // A3 + A4: h, stats_h[0]
  QFFN_CUDA(qffn::launch_gemm_swiglu(h, stats_h, yq, stats_y + 1, w1, w1_scale, N, H, C, stream,
                                     true));
  // A4 requantisation: hq, stats_h[1]
  QFFN_CUDA(qffn::launch_quantize(hq, stats_h, h, N * H, stream, true));
  // A5: out
  return from_cuda(qffn::launch_gemm_bf16(out, hq, stats_h + 1, w2, w2_scale, N, C, H, stream,
                                          nullptr, false, false, false, true));
}

qffn_status qffn_forward_recompute(uint16_t* res_out, uint16_t* out, float* rstd, float* stats_y,
                                  float* stats_h, const uint16_t* res_in, const uint16_t* x,
                                  const uint16_t* gain, float eps, const uint8_t* w1,
                                  const float* w1_scale, const uint8_t* w2, const float* w2_scale,
                                  int64_t B, int64_t T, int64_t C, int64_t H, void* workspace,
                                  size_t workspace_bytes, qffn_stream_t stream) {
  QFFN_RANGE();
  QFFN_PTR(out); QFFN_PTR(rstd); QFFN_PTR(stats_y); QFFN_PTR(stats_h); QFFN_PTR(x);
  QFFN_PTR(gain); QFFN_PTR(w1); QFFN_PTR(w1_scale); QFFN_PTR(w2); QFFN_PTR(w2_scale);
  QFFN_PTR(workspace);
  if (res_in != nullptr) QFFN_PTR(res_out);
  QFFN_REQUIRE(isfinite(eps) && eps >= 0.0f, QFFN_ERR_INVALID_ARG);
  const qffn_status st = check_forward_shape(B, T, C, H);
  if (st != QFFN_OK) return st;
  const int64_t N = B * T;
  size_t off[5];
  forward_offsets(N, C, H, off);
  QFFN_REQUIRE(workspace_bytes >= off[4], QFFN_ERR_INVALID_ARG);
  QFFN_REQUIRE(aligned256(workspace), QFFN_ERR_MISALIGNED);
  QFFN_ALIGNED(out); QFFN_ALIGNED4(rstd); QFFN_ALIGNED4(stats_y); QFFN_ALIGNED4(stats_h);
  QFFN_ALIGNED(x); QFFN_ALIGNED(gain); QFFN_ALIGNED(w1); QFFN_ALIGNED(w2);
  QFFN_ALIGNED4(w1_scale); QFFN_ALIGNED4(w2_scale);
  if (res_in != nullptr) { QFFN_ALIGNED(res_in); QFFN_ALIGNED(res_out); }

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint16_t* y = reinterpret_cast<uint16_t*>(ws + off[0]);
  uint8_t* yq = ws + off[1];
  uint8_t* hq = ws + off[3];

  // A1 without recording an abs-max: r, y, rstd
  QFFN_CUDA(qffn::launch_rmsnorm(res_out, y, rstd, nullptr, res_in, x, gain, eps, N, int(C), stream));
  // (the launches after A1 are chained as in qffn_forward)
  // A2 with the given abs-max of y: yq, stats_y[1]
  QFFN_CUDA(qffn::launch_quantize(yq, stats_y, y, N * C, stream, true));
  // A3 + A4 with the given abs-max of h: hq, stats_h[1] (bf16 h is never written)
  QFFN_CUDA(qffn::launch_gemm_swiglu_quant(hq, stats_h, yq, stats_y + 1, w1, w1_scale, N, H, C,
                                           stream, true));
  // A5: out
  return from_cuda(qffn::launch_gemm_bf16(out, hq, stats_h + 1, w2, w2_scale, N, C, H, stream,
                                          nullptr, false, false, false, true));
}

qffn_status qffn_transpose_e4m3(uint8_t* out, const uint8_t* in, int64_t rows, int64_t cols,
                                qffn_stream_t stream) {
  QFFN_RANGE();
  QFFN_PTR(out); QFFN_PTR(in);
  QFFN_REQUIRE(rows >= 0 && cols >= 0, QFFN_ERR_INVALID_ARG);
  QFFN_REQUIRE(rows % 16 == 0 && cols % 16 == 0 && rows <= kMaxRows && cols <= kMaxRows,
               QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_REQUIRE(rows / 64 < 65535, QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_ALIGNED(out); QFFN_ALIGNED(in);
  return from_cuda(qffn::launch_transpose_u8(out, in, rows, cols, stream));
}

qffn_status qffn_swiglu_backward(uint16_t* d_gate_up, float* stats, const uint16_t* dh,
                                 const uint16_t* gate_up, int64_t N, int64_t H,
                                 qffn_stream_t stream) {
  QFFN_RANGE();
  QFFN_PTR(d_gate_up); QFFN_PTR(stats); QFFN_PTR(dh); QFFN_PTR(gate_up);
  QFFN_REQUIRE(N >= 0 && H >= 0, QFFN_ERR_INVALID_ARG);
  QFFN_REQUIRE(H % 8 == 0 && H >= 8 && H <= kMaxDim && N <= kMaxRows, QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_ALIGNED(d_gate_up); QFFN_ALIGNED4(stats); QFFN_ALIGNED(dh); QFFN_ALIGNED(gate_up);
  return from_cuda(qffn::launch_swiglu_backward(d_gate_up, stats, dh, gate_up, N, H, stream));
}

size_t qffn_backward_qmm_workspace_size(int64_t N, int64_t IC, int64_t OC) {
  if (check_bqmm_shape(N, IC, OC) != QFFN_OK) return 0;
  size_t off[2];
  bqmm_offsets(N, IC, OC, off);
  return off[1] > 0 ? off[1] : 256;
}

qffn_status qffn_backward_qmm(uint16_t* dinp, uint16_t* dw, float* stats_dout,
                              const uint16_t* dout, const uint8_t* inp_q, const float* inp_scale,
                              const uint8_t* w, const float* w_scale, int64_t N, int64_t IC,
                              int64_t OC, int accumulate, void* workspace, size_t workspace_bytes,
                              qffn_stream_t stream) {
  QFFN_RANGE();
  QFFN_PTR(dw); QFFN_PTR(stats_dout); QFFN_PTR(dout); QFFN_PTR(inp_q); QFFN_PTR(inp_scale);
  QFFN_PTR(w); QFFN_PTR(w_scale); QFFN_PTR(workspace);
  const qffn_status st = check_bqmm_shape(N, IC, OC);
  if (st != QFFN_OK) return st;
  QFFN_REQUIRE(workspace_bytes >= qffn_backward_qmm_workspace_size(N, IC, OC), QFFN_ERR_INVALID_ARG);
  QFFN_REQUIRE(aligned256(workspace), QFFN_ERR_MISALIGNED);
  QFFN_ALIGNED(dinp); QFFN_ALIGNED(dw); QFFN_ALIGNED4(stats_dout); QFFN_ALIGNED(dout);
  QFFN_ALIGNED(inp_q); QFFN_ALIGNED4(inp_scale); QFFN_ALIGNED(w); QFFN_ALIGNED4(w_scale);
  return from_cuda(run_backward_qmm(dinp, dw, stats_dout, dout, inp_q, inp_scale, w, w_scale, N, IC,
                                    OC, accumulate != 0, static_cast<uint8_t*>(workspace), stream));
}

size_t qffn_ffn_backward_workspace_size(int64_t N, int64_t C, int64_t H) {
  if (check_bqmm_shape(N, H, C) != QFFN_OK || check_bqmm_shape(N, C, 2 * H) != QFFN_OK) return 0;
  if (H % 128 != 0) return 0;
  size_t off[4];
  ffn_bwd_offsets(N, C, H, off);
  return off[3];
}

qffn_status qffn_ffn_backward_workspace_offsets(int64_t N, int64_t C, int64_t H,
                                                size_t offsets[2]) {
  QFFN_PTR(offsets);
  if (qffn_ffn_backward_workspace_size(N, C, H) == 0) return QFFN_ERR_UNSUPPORTED_SHAPE;
  size_t off[4];
  ffn_bwd_offsets(N, C, H, off);
  for (int i = 0; i < 2; ++i) offsets[i] = off[i];
  return QFFN_OK;
}

qffn_status qffn_gate_up_swiglu_backward(uint16_t* d_gate_up, float* stats, const uint16_t* dh,
                                         const uint8_t* yq, const float* y_scale,
                                         const uint8_t* w1, const float* w1_scale, int64_t N,
                                         int64_t C, int64_t H, qffn_stream_t stream) {
  QFFN_RANGE();
  QFFN_PTR(d_gate_up); QFFN_PTR(stats); QFFN_PTR(dh); QFFN_PTR(yq); QFFN_PTR(y_scale);
  QFFN_PTR(w1); QFFN_PTR(w1_scale);
  QFFN_REQUIRE(N >= 0 && C >= 0 && H >= 0, QFFN_ERR_INVALID_ARG);
  QFFN_REQUIRE(N <= kMaxRows, QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_REQUIRE(C % 16 == 0 && C >= 16 && C <= kMaxDim, QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_REQUIRE(H % 128 == 0 && H >= 128 && H <= kMaxDim, QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_REQUIRE((N + 127) / 128 * (H / 128) < (int64_t(1) << 31), QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_ALIGNED(d_gate_up); QFFN_ALIGNED4(stats); QFFN_ALIGNED(dh); QFFN_ALIGNED(yq);
  QFFN_ALIGNED4(y_scale); QFFN_ALIGNED(w1); QFFN_ALIGNED4(w1_scale);
  return from_cuda(qffn::launch_gemm_swiglu_bwd(d_gate_up, stats, dh, yq, y_scale, w1, w1_scale, N,
                                                H, C, stream));
}

qffn_status qffn_ffn_backward(uint16_t* d_ln2, uint16_t* dw1, uint16_t* dw2, float* stats_dout,
                              float* stats_dgu, const uint16_t* dout, const uint8_t* yq,
                              const float* y_scale, const uint8_t* hq, const float* h_scale,
                              const uint8_t* w1, const float* w1_scale, const uint8_t* w2,
                              const float* w2_scale, int64_t N, int64_t C, int64_t H, int accumulate,
                              void* workspace, size_t workspace_bytes, qffn_stream_t stream) {
  QFFN_RANGE();
  QFFN_PTR(d_ln2); QFFN_PTR(dw1); QFFN_PTR(dw2); QFFN_PTR(stats_dout); QFFN_PTR(stats_dgu);
  QFFN_PTR(dout); QFFN_PTR(yq); QFFN_PTR(y_scale); QFFN_PTR(hq); QFFN_PTR(h_scale);
  QFFN_PTR(w1); QFFN_PTR(w1_scale); QFFN_PTR(w2); QFFN_PTR(w2_scale); QFFN_PTR(workspace);
  QFFN_REQUIRE(N >= 0 && C >= 0 && H >= 0, QFFN_ERR_INVALID_ARG);
  const size_t need = qffn_ffn_backward_workspace_size(N, C, H);
  QFFN_REQUIRE(need > 0, QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_REQUIRE(workspace_bytes >= need, QFFN_ERR_INVALID_ARG);
  QFFN_REQUIRE(aligned256(workspace), QFFN_ERR_MISALIGNED);
  QFFN_ALIGNED(d_ln2); QFFN_ALIGNED(dw1); QFFN_ALIGNED(dw2); QFFN_ALIGNED4(stats_dout);
  QFFN_ALIGNED4(stats_dgu); QFFN_ALIGNED(dout); QFFN_ALIGNED(yq); QFFN_ALIGNED4(y_scale);
  QFFN_ALIGNED(hq); QFFN_ALIGNED4(h_scale); QFFN_ALIGNED(w1); QFFN_ALIGNED4(w1_scale);
  QFFN_ALIGNED(w2); QFFN_ALIGNED4(w2_scale);
  size_t off[4];
  ffn_bwd_offsets(N, C, H, off);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint16_t* dh = reinterpret_cast<uint16_t*>(ws + off[0]);
  uint16_t* dgu = reinterpret_cast<uint16_t*>(ws + off[1]);
  uint8_t* bq = ws + off[2];
  const bool acc = accumulate != 0;
  // down projection: dh = d(SwiGLU output), dW2
  QFFN_CUDA(run_backward_qmm(dh, dw2, stats_dout, dout, hq, h_scale, w2, w2_scale, N, H, C, acc, bq,
                             stream));
  // the up projection's output recomputed (forward_qmm of _recompute_block) and
  // swiglu_backward with the abs-max of d(gate|up), in one GEMM epilogue
  QFFN_CUDA(qffn::launch_gemm_swiglu_bwd(dgu, stats_dgu, dh, yq, y_scale, w1, w1_scale, N, H, C,
                                         stream));
  // up projection: d_ln2, dW1
  return from_cuda(run_backward_qmm(d_ln2, dw1, stats_dgu, dgu, yq, y_scale, w1, w1_scale, N, C,
                                    2 * H, acc, bq, stream));
}

qffn_status qffn_gemv_dual(uint16_t* g, uint16_t* u, const uint16_t* x, const uint8_t* w_gate,
                           const float* s_gate, const uint8_t* w_up, const float* s_up,
                           int64_t H, int64_t C, qffn_stream_t stream) {
  QFFN_RANGE();
  QFFN_PTR(g); QFFN_PTR(u); QFFN_PTR(x); QFFN_PTR(w_gate); QFFN_PTR(s_gate); QFFN_PTR(w_up); QFFN_PTR(s_up);
  QFFN_REQUIRE(H >= 1 && C >= 0, QFFN_ERR_INVALID_ARG);
  QFFN_REQUIRE(C % 16 == 0 && C >= 16 && C <= 32768 && H <= kMaxRows, QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_ALIGNED(x); QFFN_ALIGNED(w_gate); QFFN_ALIGNED(w_up); QFFN_ALIGNED4(s_gate); QFFN_ALIGNED4(s_up);
  return from_cuda(qffn::launch_gemv(g, u, x, w_gate, s_gate, w_up, s_up, H, C, false, stream));
}

qffn_status qffn_gemv(uint16_t* out, const uint16_t* x, const uint8_t* w, const float* row_scale,
                      int64_t rows, int64_t cols, qffn_stream_t stream) {
  QFFN_RANGE();
  QFFN_PTR(out); QFFN_PTR(x); QFFN_PTR(w); QFFN_PTR(row_scale);
  QFFN_REQUIRE(rows >= 1 && cols >= 0, QFFN_ERR_INVALID_ARG);
  QFFN_REQUIRE(cols % 16 == 0 && cols >= 16 && cols <= 32768 && rows <= kMaxRows,
               QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_ALIGNED(x); QFFN_ALIGNED(w); QFFN_ALIGNED4(row_scale);
  return from_cuda(qffn::launch_gemv(out, nullptr, x, w, row_scale, nullptr, nullptr, rows, cols,
                                     false, stream));
}

qffn_status qffn_gemv_silu_input(uint16_t* out, const uint16_t* g, const uint16_t* u,
                                 const uint8_t* w, const float* row_scale, int64_t rows,
                                 int64_t cols, qffn_stream_t stream) {
  QFFN_RANGE();
  QFFN_PTR(out); QFFN_PTR(g); QFFN_PTR(u); QFFN_PTR(w); QFFN_PTR(row_scale);
  QFFN_REQUIRE(rows >= 1 && cols >= 0, QFFN_ERR_INVALID_ARG);
  QFFN_REQUIRE(cols % 16 == 0 && cols >= 16 && cols <= 32768 && rows <= kMaxRows,
               QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_ALIGNED(g); QFFN_ALIGNED(u); QFFN_ALIGNED(w); QFFN_ALIGNED4(row_scale);
  return from_cuda(qffn::launch_gemv_silu_input(out, g, u, w, row_scale, rows, cols, stream));
}

qffn_status qffn_silu_mul(uint16_t* g, const uint16_t* u, int64_t n, qffn_stream_t stream) {
  QFFN_RANGE();
  QFFN_PTR(g); QFFN_PTR(u);
  QFFN_REQUIRE(n >= 0, QFFN_ERR_INVALID_ARG);
  QFFN_REQUIRE(n % 8 == 0, QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_ALIGNED(g); QFFN_ALIGNED(u);
  return from_cuda(qffn::launch_silu_mul(g, u, n, false, stream));
}

size_t qffn_decode_workspace_size(int64_t C, int64_t H) {
  if (C < 16 || H < 16 || C > 32768 || H > 32768) return 0;
  size_t off[3];
  decode_offsets(H, off);
  return off[2];
}

qffn_status qffn_decode_workspace_offsets(int64_t C, int64_t H, size_t offsets[2]) {
  QFFN_PTR(offsets);
  QFFN_REQUIRE(C >= 16 && H >= 16 && C <= 32768 && H <= 32768, QFFN_ERR_UNSUPPORTED_SHAPE);
  size_t off[3];
  decode_offsets(H, off);
  offsets[0] = off[0];
  offsets[1] = off[1];
  return QFFN_OK;
}

qffn_status qffn_decode_forward_ex(uint16_t* out, const uint16_t* x, const uint8_t* w_gate,
                                   const float* s_gate, const uint8_t* w_up, const float* s_up,
                                   const uint8_t* w_down, const float* s_down, int64_t C, int64_t H,
                                   void* workspace, size_t workspace_bytes, unsigned int flags,
                                   qffn_stream_t stream) {
  QFFN_RANGE();
  QFFN_PTR(out); QFFN_PTR(x); QFFN_PTR(w_gate); QFFN_PTR(s_gate); QFFN_PTR(w_up); QFFN_PTR(s_up);
  QFFN_PTR(w_down); QFFN_PTR(s_down); QFFN_PTR(workspace);
  QFFN_REQUIRE((flags & ~QFFN_DECODE_WEIGHTS_STABLE) == 0u, QFFN_ERR_INVALID_ARG);
  QFFN_REQUIRE(C % 16 == 0 && H % 16 == 0 && C >= 16 && H >= 16 && C <= 32768 && H <= 32768,
               QFFN_ERR_UNSUPPORTED_SHAPE);
  QFFN_REQUIRE(workspace_bytes >= qffn_decode_workspace_size(C, H), QFFN_ERR_INVALID_ARG);
  QFFN_ALIGNED(out); QFFN_ALIGNED(x); QFFN_ALIGNED(w_gate); QFFN_ALIGNED(w_up); QFFN_ALIGNED(w_down);
  QFFN_ALIGNED4(s_gate); QFFN_ALIGNED4(s_up); QFFN_ALIGNED4(s_down);
  QFFN_ALIGNED(workspace);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  size_t off[3];
  decode_offsets(H, off);
  // A6 with A7 folded into its output, then A8 (see decode.cu)
  return from_cuda(qffn::launch_decode(out, x, w_gate, s_gate, w_up, s_up, w_down, s_down, C, H,
                                       reinterpret_cast<uint16_t*>(ws + off[0]),
                                       reinterpret_cast<uint16_t*>(ws + off[1]),
                                       (flags & QFFN_DECODE_WEIGHTS_STABLE) != 0u, stream));
}

qffn_status qffn_decode_forward(uint16_t* out, const uint16_t* x, const uint8_t* w_gate,
                                const float* s_gate, const uint8_t* w_up, const float* s_up,
                                const uint8_t* w_down, const float* s_down, int64_t C, int64_t H,
                                void* workspace, size_t workspace_bytes, qffn_stream_t stream) {
  return qffn_decode_forward_ex(out, x, w_gate, s_gate, w_up, s_up, w_down, s_down, C, H, workspace,
                                workspace_bytes, 0u, stream);
}

qffn_status qffn_decode_forward_gu(uint16_t* out, const uint16_t* x, const uint8_t* w_gu,
                                   const float* gu_row_scale, const uint8_t* w_down,
                                   const float* s_down, int64_t C, int64_t H, void* workspace,
                                   size_t workspace_bytes, qffn_stream_t stream) {
  QFFN_PTR(w_gu); QFFN_PTR(gu_row_scale);
  QFFN_REQUIRE(C >= 0 && H >= 0 && C <= 32768 && H <= 32768, QFFN_ERR_UNSUPPORTED_SHAPE);
  return qffn_decode_forward_ex(out, x, w_gu, gu_row_scale, w_gu + size_t(H) * size_t(C),
                                gu_row_scale + H, w_down, s_down, C, H, workspace, workspace_bytes,
                                0u, stream);
}

}  // extern "C"
