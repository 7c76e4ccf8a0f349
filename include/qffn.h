/*
 * qffn -- FP8-quantised SwiGLU feed-forward block for one NVIDIA GB300 (sm_103a).
 *
 * C ABI.  Every entry point takes plain pointers and sizes and returns a
 * qffn_status; nothing here allocates device memory, and every buffer is
 * owned by the caller.
 *
 * Sources of the operations (page title, function):
 *   [llmq-model]  IST-DASLab/llmq "src/models/llama_model.cpp":
 *                 LLamaModel::_forward_block (FFN half), forward_qmm,
 *                 _recompute_block (swiglu_forward_quant), fill_block_shapes,
 *                 LLamaModel::forward (fill_zero of the abs-max block).
 *   [llmq-state]  IST-DASLab/llmq "src/models/llama_run_state.cpp":
 *                 activation shapes and dtypes, the stats block (two floats per
 *                 quantised tensor: abs-max, then scale).
 *   [metrale]     metrale "layers/dense_ffn_decode.rs", DenseFfnLayer::forward,
 *                 FP8 arm: w8a16_gemv_dual, silu_mul, w8a16_gemv.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Tensors are row-major and contiguous.  uint16_t* holds bf16 bit patterns,
 *    uint8_t* holds OCP FP8 E4M3 ("fn") codes, float* is IEEE binary32.
 *  - "stats" points at two device floats {abs_max, scale} [llmq-state].  A
 *    call that records an abs-max first zeroes stats[0] on the stream (the
 *    trainer's fill_zero before the forward) and then max-accumulates into it.
 *  - scale = abs_max / 448 is the dequantisation multiplier (448 = largest
 *    finite E4M3); codes are e4m3(x * (448 / abs_max)) with the product in
 *    fp32, rounded to nearest even and saturated to +-448.  abs_max == 0 gives
 *    scale 1 and all-zero codes.
 *  - bf16 and E4M3 tensors must start on a 16-byte boundary, fp32 pointers
 *    (stats pairs, scales, rstd, row scales) on a 4-byte boundary
 *    (QFFN_ERR_MISALIGNED otherwise); required pointers must be non-NULL
 *    (QFFN_ERR_INVALID_ARG).
 *  - Arguments are checked on the host before anything is enqueued; on any
 *    error nothing is enqueued.  Work is enqueued asynchronously on `stream`
 *    (NULL = the legacy default stream) and the call returns without waiting.
 *    Launch failures are reported as QFFN_ERR_CUDA.
 *  - The GEMM kernels bound every wait on their internal pipeline barriers.
 *    A wait that runs out (about 2 s) makes the kernel stop, set a device
 *    status word and return; qffn_check_status() reports it.
 *  - Output buffers must not overlap inputs unless a call says otherwise.
 */
#ifndef QFFN_H_
#define QFFN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* qffn_stream_t;

typedef enum qffn_status {
  QFFN_OK = 0,
  QFFN_ERR_INVALID_ARG = 1,       /* NULL pointer, negative size, bad eps, small workspace */
  QFFN_ERR_UNSUPPORTED_SHAPE = 2, /* a size outside the rules stated per call */
  QFFN_ERR_MISALIGNED = 3,        /* a pointer below its required alignment */
  QFFN_ERR_CUDA = 4,              /* a CUDA runtime call or launch failed */
  QFFN_ERR_TIMEOUT = 5            /* a device-side bounded wait ran out */
} qffn_status;

/* Static description of a status code. */
const char* qffn_status_string(qffn_status status);

/* Version of this ABI (bumped on any signature change). */
int qffn_abi_version(void);

/* Synchronises `stream`, then reports (and clears) the device status word:
 * QFFN_ERR_TIMEOUT if a GEMM kernel gave up on a pipeline wait since the last
 * check, QFFN_ERR_CUDA if the synchronisation failed, else QFFN_OK. */
qffn_status qffn_check_status(qffn_stream_t stream);

/* Measurement aid (no counterpart on the pages).  Synchronises `stream`, then
 * writes, for the most recent GEMM launch on the current device, the SM clock
 * cycles (%clock64) and the nanoseconds (%globaltimer) that its first CTA
 * spent from its start to its end: out[0] / out[1] is the mean SM clock of
 * that launch in GHz.  With the tensor cores' dense FP8 rate of 16384 FLOP
 * per clock per SM it gives the peak the launch could reach at the clock it
 * ran at.  Both are 0 before the first GEMM launch of the process.
 *   out: host, 2 x uint64.  QFFN_ERR_CUDA if the synchronisation or the read
 *   fails. */
qffn_status qffn_gemm_clock_sample(uint64_t* out, qffn_stream_t stream);

/* Self-test of the failure path (no counterpart on the pages, which stop on
 * any CUDA error; this library bounds its device-side waits instead).  One
 * CTA runs the GEMMs' bounded barrier wait on two barriers of arrival count 1:
 * lane 0 of warp 0 waits up to `limit_ns` on barrier 0; lane 0 of warp 1 waits
 * up to 4 x limit_ns on barrier 1 and leaves early if the CTA abort flag is
 * raised.  With `arrive` != 0 both barriers get their arrival first and both
 * waits succeed at once.  With arrive == 0 nothing arrives: warp 0 runs out,
 * raises the abort flag and sets the device status word (the next
 * qffn_check_status returns QFFN_ERR_TIMEOUT and clears it), and warp 1
 * returns on the abort flag after about limit_ns.  Nothing faults or hangs and
 * the context stays usable.
 *   out: device, 4 x uint64, written by the kernel: out[0], out[1] = 1 if the
 *        wait of warp 0 / warp 1 succeeded else 0; out[2], out[3] = the
 *        nanoseconds (%globaltimer) each wait took.  8-byte aligned.
 *   limit_ns: 100000 .. 2000000000 (QFFN_ERR_INVALID_ARG otherwise). */
qffn_status qffn_selftest_bounded_wait(uint64_t* out, int arrive, int64_t limit_ns,
                                       qffn_stream_t stream);

/* ---- Step A1: fused residual add + RMSNorm + abs-max -----------------------
 * [llmq-model] fused_residual_rmsnorm_forward (and rmsnorm_forward when
 * res_in == NULL), called in _forward_block before the up projection.
 *   res_out[N,C] = bf16(res_in + x)                        (skipped if res_in == NULL)
 *   rstd[N]      = 1 / sqrt(mean_C(r^2) + eps),  r = res_out (or x)
 *   y[N,C]       = bf16(r * rstd * gain)
 *   stats[0]     = max |y|   (zeroed first; stats == NULL records nothing)
 * res_out may alias res_in or x (in place).  N >= 0, C % 8 == 0,
 * 8 <= C <= 16384; eps >= 0 and finite. */
qffn_status qffn_rmsnorm_absmax(uint16_t* res_out, uint16_t* y, float* rstd, float* stats,
                                const uint16_t* res_in, const uint16_t* x, const uint16_t* gain,
                                float eps, int64_t N, int64_t C, qffn_stream_t stream);

/* ---- Tensor abs-max -------------------------------------------------------
 * [llmq-model] abs_max: stats[0] = max |in[i]| over n bf16 values (zeroed
 * first).  Used to build per-tensor FP8 weight records.  n >= 0. */
qffn_status qffn_absmax(float* stats, const uint16_t* in, int64_t n, qffn_stream_t stream);

/* ---- Step A2: quantise with a recorded abs-max -----------------------------
 * [llmq-model] forward_qmm -> quantize_with_abs_max.  Reads stats[0]
 * (abs_max, produced earlier on the stream), writes stats[1] = scale and
 * q[i] = e4m3(in[i] * 448 / abs_max).  n >= 0. */
qffn_status qffn_quantize(uint8_t* q, float* stats, const uint16_t* in, int64_t n,
                          qffn_stream_t stream);

/* ---- Per-row FP8 weight record (decode weights) ---------------------------
 * [metrale] fp8 weights carry a per-output-row fp32 row_scale.  For each row:
 * row_scale[r] = max_k |w[r,k]| / 448, q[r,k] = e4m3(w[r,k] * 448 / rowmax)
 * (a zero row gives scale 1, codes 0).  rows >= 0, cols % 16 == 0,
 * 16 <= cols <= 65536. */
qffn_status qffn_quantize_rows(uint8_t* q, float* row_scale, const uint16_t* w, int64_t rows,
                               int64_t cols, qffn_stream_t stream);

/* ---- Steps A3 / A5: scaled FP8 GEMM ---------------------------------------
 * [llmq-model] forward_qmm -> matmul(out, W, X, bias=none, scale_W, scale_X,
 * OC, B*T, C, TN): both operands FP8 with K contiguous, bf16 output.
 *   out[M,N] = bf16(a_scale[0] * w_scale[0] * sum_k A[m,k] * W[n,k])
 * fp32 accumulation on the tensor cores.  a_scale / w_scale are device
 * pointers to one float each.  M >= 0, N % 32 == 0, K % 16 == 0, K >= 16,
 * N, K <= 2^20. */
qffn_status qffn_fp8_gemm_scaled(uint16_t* out, const uint8_t* A, const float* a_scale,
                                 const uint8_t* W, const float* w_scale, int64_t M, int64_t N,
                                 int64_t K, qffn_stream_t stream);

/* ---- forward_qmm: quantise with the recorded abs-max, then the matmul -----
 * [llmq-model] forward_qmm(out, inp, weight, bias, ...): quantize_with_abs_max
 * of inp, then matmul with weight.scale() and inp.Quant.scale().
 * _forward_block uses it for the attention projections: the QKV projection of
 * LN1 (after qffn_rmsnorm_absmax), with the optional Attn_QKV_b bias, and the
 * output projection of the attention result (after qffn_absmax).
 *   q[M,K]   = e4m3(in * 448 / stats[0]);  stats[1] = scale
 *   out[M,N] = bf16(stats[1] * w_scale[0] * sum_k q[m,k] * W[n,k] + bias[n])
 * The bias (bf16 [N], may be NULL) is added to the scaled fp32 accumulator
 * before the one rounding.  q is caller scratch of M*K bytes, readable after
 * the call.  Shape rules of qffn_fp8_gemm_scaled. */
qffn_status qffn_qmm(uint16_t* out, uint8_t* q, float* stats, const uint16_t* in,
                     const uint16_t* bias, const uint8_t* W, const float* w_scale, int64_t M,
                     int64_t N, int64_t K, qffn_stream_t stream);

/* ---- Steps A3 + A4 fused: gate|up GEMM with the SwiGLU epilogue -----------
 * [llmq-model] forward_qmm on MLP_Up_w (W1 = [2H, C], gate rows [0,H) then up
 * rows [H,2H)) followed by swiglu_forward with its abs-max.  The gate and up
 * products are each rounded to bf16 (the mlp_up buffer dtype) before
 *   h[N,H]      = bf16(silu(g) * u),  silu(z) = z / (1 + exp(-z))
 *   stats_h[0]  = max |h|   (zeroed first)
 * The [N, 2H] up-projection output is never written.  N >= 0,
 * C % 16 == 0, C >= 16, H % 128 == 0, H >= 128, C, H <= 2^20. */
qffn_status qffn_gate_up_swiglu(uint16_t* h, float* stats_h, const uint8_t* yq,
                                const float* y_scale, const uint8_t* w1, const float* w1_scale,
                                int64_t N, int64_t C, int64_t H, qffn_stream_t stream);

/* ---- Step A4 standalone: SwiGLU + abs-max + requantisation ----------------
 * [llmq-model] swiglu_forward then quantize_with_abs_max; the h == NULL form
 * is swiglu_forward_quant of _recompute_block (h recomputed for the second
 * pass, bit-identical).  gate_up is [N, 2H] bf16 (gate = cols [0,H)).
 *   h[N,H] = bf16(silu(g) * u); stats[0] = max|h|; stats[1] = scale;
 *   hq[N,H] = e4m3(h * 448 / max|h|).   N >= 0, H % 8 == 0. */
qffn_status qffn_swiglu_quant(uint16_t* h, uint8_t* hq, float* stats, const uint16_t* gate_up,
                              int64_t N, int64_t H, qffn_stream_t stream);

/* ---- Step A4, recompute form: SwiGLU quantised with a given abs-max -------
 * [llmq-model] _recompute_block: swiglu_forward_quant(SwiGLu.Quant, scale,
 * MlpUp, SwiGLu.Quant.abs_max(), B, T, D) -- the abs-max the forward
 * recorded is read, not recomputed.  gate_up is [N, 2H] bf16 (gate = cols
 * [0,H)).  Reads stats[0] (abs_max, >= 0), writes stats[1] = scale and
 *   hq[N,H] = e4m3(bf16(silu(g) * u) * 448 / abs_max)
 * Values beyond the given abs-max saturate at +-448.  With the abs-max that
 * qffn_swiglu_quant recorded, hq is bit-identical to that call's hq.
 * N >= 0, H % 8 == 0. */
qffn_status qffn_swiglu_forward_quant(uint8_t* hq, float* stats, const uint16_t* gate_up,
                                      int64_t N, int64_t H, qffn_stream_t stream);

/* ---- Steps A3 + A4 fused, recompute form: E4M3 h straight from the GEMM ---
 * [llmq-model] _recompute_block: forward_qmm on MLP_Up_w followed by
 * swiglu_forward_quant with the recorded abs-max.  The epilogue of the
 * gate|up GEMM forms h exactly as qffn_gate_up_swiglu does and quantises it
 * with the abs-max read from stats_h[0]:
 *   hq[N,H] = e4m3(h * 448 / stats_h[0]),  stats_h[1] = scale
 * Neither the [N, 2H] up-projection output nor bf16 h is written.  Given
 * the abs-max qffn_gate_up_swiglu recorded, hq equals qffn_quantize of that
 * call's h bit for bit.  Shape rules of qffn_gate_up_swiglu. */
qffn_status qffn_gate_up_swiglu_quant(uint8_t* hq, float* stats_h, const uint8_t* yq,
                                      const float* y_scale, const uint8_t* w1,
                                      const float* w1_scale, int64_t N, int64_t C, int64_t H,
                                      qffn_stream_t stream);

/* ---- Whole prefill FFN: A1 -> A2 -> A3+A4 -> A2 -> A5 ---------------------
 * [llmq-model] _forward_block, FFN half, for B*T tokens:
 *   r = bf16(res_in + x); y = rmsnorm(r) * gain; yq = quant(y);
 *   h = swiglu(yq @ W1^T); hq = quant(h); out = bf16(hq @ W2^T * scales)
 * Outputs: res_out [N,C] (the residual the next layer adds `out` to), out
 * [N,C] bf16, rstd [N] fp32, stats_y[2], stats_h[2].  w1 = [2H, C] E4M3 with
 * per-tensor scale w1_scale[1]; w2 = [C, H] E4M3 with w2_scale[1] (device).
 * res_in == NULL runs the plain RMSNorm (res_out unused, may be NULL).
 * workspace: device scratch of at least qffn_forward_workspace_size() bytes,
 * 256-byte aligned, holding y, yq, h, hq at the offsets that
 * qffn_forward_workspace_offsets() returns (readable after the call).
 * N = B*T >= 0, C % 128 == 0, H % 128 == 0, 128 <= C <= 16384,
 * 128 <= H <= 2^20.
 * Five kernels (and one 4-byte memset) on `stream`; the four after the norm
 * are programmatic dependent launches, scheduled while their predecessor
 * drains and waiting for it before touching memory (no effect on results;
 * stream capture keeps the edges). */
size_t qffn_forward_workspace_size(int64_t B, int64_t T, int64_t C, int64_t H);
qffn_status qffn_forward_workspace_offsets(int64_t B, int64_t T, int64_t C, int64_t H,
                                           size_t offsets[4] /* y, yq, h, hq */);
qffn_status qffn_forward(uint16_t* res_out, uint16_t* out, float* rstd, float* stats_y,
                         float* stats_h, const uint16_t* res_in, const uint16_t* x,
                         const uint16_t* gain, float eps, const uint8_t* w1,
                         const float* w1_scale, const uint8_t* w2, const float* w2_scale,
                         int64_t B, int64_t T, int64_t C, int64_t H, void* workspace,
                         size_t workspace_bytes, qffn_stream_t stream);

/* ---- Whole prefill FFN with the activation abs-maxes given ---------------
 * [llmq-model] _recompute_block, FFN half:
 *   - the norm re-runs without recording an abs-max;
 *   - LN2 is quantised with the abs-max its stats slot holds;
 *   - swiglu_forward_quant uses the recorded SwiGLU abs-max.
 * The down projection then runs as in the forward, so the call yields the
 * block output.  Arguments, workspace and shape rules are those of
 * qffn_forward, except that stats_y[0] and stats_h[0] are inputs (abs-maxes,
 * >= 0) and only stats_y[1] and stats_h[1] (the scales) are written.  Four
 * launches: A1 (no abs-max), A2, the gate|up GEMM with the E4M3 SwiGLU
 * epilogue (qffn_gate_up_swiglu_quant), A5.  The h slot of the workspace is
 * not written.  Given the stats a qffn_forward call left, every output (res_out,
 * out, rstd, and yq and hq in the workspace) equals that call's bit for bit.
 * Elements beyond a given abs-max saturate at +-448. */
qffn_status qffn_forward_recompute(uint16_t* res_out, uint16_t* out, float* rstd, float* stats_y,
                                  float* stats_h, const uint16_t* res_in, const uint16_t* x,
                                  const uint16_t* gain, float eps, const uint8_t* w1,
                                  const float* w1_scale, const uint8_t* w2, const float* w2_scale,
                                  int64_t B, int64_t T, int64_t C, int64_t H, void* workspace,
                                  size_t workspace_bytes, qffn_stream_t stream);

/* ---- FP8 backward of the FFN -----------------------------------------------
 * [llmq-model] _backward_block (FFN half) and the FP8 branch of backward_qmm.
 * Gradients are bf16; their FP8 copies are E4M3 quantised with a recorded
 * abs-max, exactly as activations are (qffn_quantize). */

/* E4M3 transpose: out[cols, rows] = in[rows, cols]^T, the transpose the
 * page's backward_qmm applies to the weight and to the quantised operands
 * (qffn_backward_qmm itself reads them MN-major instead).  rows and cols are
 * multiples of 16; rows < 64 * 65535. */
qffn_status qffn_transpose_e4m3(uint8_t* out, const uint8_t* in, int64_t rows, int64_t cols,
                                qffn_stream_t stream);

/* [llmq-model] swiglu_backward(DMlpUp.Value, DSwiGLU, MlpUp,
 * DMlpUp.Quant.abs_max(), B, T, D).  With g, u the bf16 gate / up halves of
 * gate_up [N, 2H] and dh [N, H] the gradient of h = silu(g) * u:
 *   d_gate_up[:, j]     = bf16(dh * u * s * (1 + g * (1 - s))),  s = sigmoid(g)
 *   d_gate_up[:, H + j] = bf16(dh * silu(g))
 *   stats[0] = max |d_gate_up|   (zeroed first)
 * fp32 arithmetic, one rounding per output.  N >= 0, H % 8 == 0. */
qffn_status qffn_swiglu_backward(uint16_t* d_gate_up, float* stats, const uint16_t* dh,
                                 const uint16_t* gate_up, int64_t N, int64_t H,
                                 qffn_stream_t stream);

/* [llmq-model] backward_qmm, FP8 weights, for one projection out = inp @ W^T
 * with dout [N, OC] bf16, the forward's quantised input inp_q [N, IC] E4M3 with
 * inp_scale[1], W [OC, IC] E4M3 with w_scale[1]:
 *   dq = e4m3(dout * 448 / stats_dout[0]);  stats_dout[1] = scale
 *   dinp[N, IC] = bf16(stats_dout[1] * w_scale * sum_oc dq[n, oc] * W[oc, ic])
 *   dw[OC, IC]  = bf16(stats_dout[1] * inp_scale * sum_n dq[n, oc] * inp_q[n, ic]
 *                      (+ dw[OC, IC] when accumulate != 0))
 * stats_dout[0] is the recorded abs-max of dout (an input).  dinp may be NULL
 * (weight gradient only).  The page transposes the weight and both operands
 * of the weight gradient so that each matmul is K-contiguous; here the tensor
 * cores read W, dq and inp_q MN-major where they lie, and the workspace holds
 * only dq.  workspace: >= qffn_backward_qmm_workspace_size() bytes, 256-byte
 * aligned; dq [N, OC] is at offset 0 after the call.  N % 16 == 0, IC % 32 == 0, OC % 32 == 0 (all >= 32
 * except N >= 0), IC, OC <= 2^20. */
size_t qffn_backward_qmm_workspace_size(int64_t N, int64_t IC, int64_t OC);
qffn_status qffn_backward_qmm(uint16_t* dinp, uint16_t* dw, float* stats_dout,
                              const uint16_t* dout, const uint8_t* inp_q, const float* inp_scale,
                              const uint8_t* w, const float* w_scale, int64_t N, int64_t IC,
                              int64_t OC, int accumulate, void* workspace, size_t workspace_bytes,
                              qffn_stream_t stream);

/* Recompute of the up projection fused with swiglu_backward: the gate|up
 * GEMM of qffn_gate_up_swiglu, whose epilogue rounds g and u to bf16 (the
 * recomputed mlp_up buffer of _recompute_block), reads dh [N, H] and writes
 * d_gate_up [N, 2H] and stats[0] = max |d_gate_up| (zeroed first) exactly as
 * qffn_fp8_gemm_scaled into [N, 2H] followed by qffn_swiglu_backward would.
 * The [N, 2H] gate|up product is never written.  Shape rules of
 * qffn_gate_up_swiglu. */
qffn_status qffn_gate_up_swiglu_backward(uint16_t* d_gate_up, float* stats, const uint16_t* dh,
                                         const uint8_t* yq, const float* y_scale,
                                         const uint8_t* w1, const float* w1_scale, int64_t N,
                                         int64_t C, int64_t H, qffn_stream_t stream);

/* The FFN half of _backward_block after the norm, for the block output
 * gradient dout [N, C] (bf16, stats_dout[0] = its recorded abs-max):
 *   1. backward_qmm of the down projection (inp = hq [N, H] of the forward,
 *      W2 [C, H]) -> dh [N, H], dw2 [C, H];
 *   2. the up projection's output recomputed from yq and W1 (forward_qmm of
 *      _recompute_block) and swiglu_backward on it, fused
 *      (qffn_gate_up_swiglu_backward) -> d_gate_up [N, 2H], stats_dgu[0];
 *   3. backward_qmm of the up projection (inp = yq [N, C], W1 [2H, C])
 *      -> d_ln2 [N, C], dw1 [2H, C].
 * stats_dout[1] and stats_dgu[1] receive the two gradient scales.  With
 * accumulate != 0 the weight gradients add to dw1 and dw2.  workspace: >=
 * qffn_ffn_backward_workspace_size() bytes, 256-byte aligned; after the call
 * it holds dh and d_gate_up (bf16) at the offsets that
 * qffn_ffn_backward_workspace_offsets() returns.  Seven kernels.
 * N % 16 == 0, C % 32 == 0, H % 128 == 0, C, H >= 128. */
size_t qffn_ffn_backward_workspace_size(int64_t N, int64_t C, int64_t H);
qffn_status qffn_ffn_backward_workspace_offsets(int64_t N, int64_t C, int64_t H,
                                                size_t offsets[2] /* dh, d_gate_up */);
qffn_status qffn_ffn_backward(uint16_t* d_ln2, uint16_t* dw1, uint16_t* dw2, float* stats_dout,
                              float* stats_dgu, const uint16_t* dout, const uint8_t* yq,
                              const float* y_scale, const uint8_t* hq, const float* h_scale,
                              const uint8_t* w1, const float* w1_scale, const uint8_t* w2,
                              const float* w2_scale, int64_t N, int64_t C, int64_t H, int accumulate,
                              void* workspace, size_t workspace_bytes, qffn_stream_t stream);

/* ---- Step A6: dual row-scaled FP8 GEMV ------------------------------------
 * [metrale] w8a16_gemv_dual: one pass over x for two weight matrices.
 *   g[r] = bf16(s_gate[r] * sum_k Wg[r,k] * x[k]),  u likewise with Wu, s_up.
 * Wg, Wu are [H, C] E4M3; s_gate, s_up [H] fp32; x [C] bf16; g, u [H] bf16.
 * C % 16 == 0, 16 <= C <= 32768, H >= 1. */
qffn_status qffn_gemv_dual(uint16_t* g, uint16_t* u, const uint16_t* x, const uint8_t* w_gate,
                           const float* s_gate, const uint8_t* w_up, const float* s_up,
                           int64_t H, int64_t C, qffn_stream_t stream);

/* ---- Row-scaled FP8 GEMV (steps A6 per projection, A8) --------------------
 * [metrale] w8a16_gemv: out[r] = bf16(row_scale[r] * sum_k W[r,k] * x[k]).
 * W [rows, cols] E4M3, x [cols] bf16.  Bit-identical, row for row, to the
 * corresponding output of qffn_gemv_dual.  cols % 16 == 0,
 * 16 <= cols <= 32768, rows >= 1. */
qffn_status qffn_gemv(uint16_t* out, const uint16_t* x, const uint8_t* w, const float* row_scale,
                      int64_t rows, int64_t cols, qffn_stream_t stream);

/* ---- Step A8, fused-SiLU-input arm ---------------------------------------
 * [metrale] w8a16_gemv_silu_input(gate_out, up_out, down weights, row_scale,
 * output): the down GEMV forms its input h = bf16(silu(g) * u) itself.
 *   out[r] = bf16(row_scale[r] * sum_k W[r,k] * h[k])
 * h is formed once per CTA while the input vector is staged in shared
 * memory.  The result is bit-identical to qffn_silu_mul(g, u) followed by
 * qffn_gemv, and g and u are not modified.  W [rows, cols] E4M3; g, u [cols]
 * bf16.  cols % 16 == 0, 16 <= cols <= 32768, rows >= 1. */
qffn_status qffn_gemv_silu_input(uint16_t* out, const uint16_t* g, const uint16_t* u,
                                 const uint8_t* w, const float* row_scale, int64_t rows,
                                 int64_t cols, qffn_stream_t stream);

/* ---- Step A7: silu_mul, in place ------------------------------------------
 * [metrale] silu_mul(gate_out, up_out -> gate_out): g[i] = bf16(silu(g[i]) * u[i]).
 * n >= 0, n % 8 == 0. */
qffn_status qffn_silu_mul(uint16_t* g, const uint16_t* u, int64_t n, qffn_stream_t stream);

/* ---- Whole single-token decode FFN: A6 -> A7 -> A8 ------------------------
 * [metrale] DenseFfnLayer::forward, FP8 split-SiLU arm.  x [C] bf16 (already
 * normalised), Wg, Wu [H, C] E4M3 with s_gate, s_up [H]; Wd [C, H] E4M3 with
 * s_down [C]; out [C] bf16.  C % 16 == 0, H % 16 == 0, 16 <= C, H <= 32768.
 * workspace >= qffn_decode_workspace_size() bytes, 16-byte aligned, any
 * content.  After the call it holds, as the split-SiLU arm leaves its
 * buffers, h = bf16(silu(g) * u) [H] bf16 (the gate buffer) and u [H] bf16
 * at the byte offsets qffn_decode_workspace_offsets() returns (0 and
 * round_up(2H, 256)).  Two launches: the dual gate/up GEMV with silu_mul
 * applied as g and u are produced, then the down GEMV as a programmatic
 * dependent launch; bit-identical to qffn_gemv_dual, qffn_silu_mul,
 * qffn_gemv.
 *
 * Ordering: both launches are programmatic dependent launches.  The down
 * GEMV starts streaming w_down before the dual GEMV has finished (it waits
 * only for h), which is always safe: it cannot start before the work that
 * preceded the call has finished.  Without QFFN_DECODE_WEIGHTS_STABLE the
 * dual GEMV reads nothing before the preceding work on the stream has
 * finished. */
size_t qffn_decode_workspace_size(int64_t C, int64_t H);
qffn_status qffn_decode_workspace_offsets(int64_t C, int64_t H, size_t offsets[2] /* h, u */);
qffn_status qffn_decode_forward(uint16_t* out, const uint16_t* x, const uint8_t* w_gate,
                                const float* s_gate, const uint8_t* w_up, const float* s_up,
                                const uint8_t* w_down, const float* s_down, int64_t C, int64_t H,
                                void* workspace, size_t workspace_bytes, qffn_stream_t stream);

/* qffn_decode_forward with flags.
 * QFFN_DECODE_WEIGHTS_STABLE: the dual GEMV starts streaming w_gate and w_up
 * (not x, the row scales or the workspace) before the kernel enqueued just
 * before this call on the stream has finished, so the weight stream of a
 * decode step overlaps the end of the previous one.  Set it only when no
 * work that can still be running at that point writes those weights: not
 * the kernel just before this call (for example qffn_quantize_rows building
 * them), nor, when that kernel is itself a programmatic dependent launch,
 * the kernels it may overlap.  Weights written before a stream or event
 * synchronisation, or before an ordinary (non-programmatic) launch that
 * precedes this call on the stream, are safe.  Unknown flag bits give
 * QFFN_ERR_INVALID_ARG. */
#define QFFN_DECODE_WEIGHTS_STABLE 1u
qffn_status qffn_decode_forward_ex(uint16_t* out, const uint16_t* x, const uint8_t* w_gate,
                                   const float* s_gate, const uint8_t* w_up, const float* s_up,
                                   const uint8_t* w_down, const float* s_down, int64_t C, int64_t H,
                                   void* workspace, size_t workspace_bytes, unsigned int flags,
                                   qffn_stream_t stream);

/* The decode with the gate and up weights as one fused record, the layout
 * of the fused up projection (R1: gate rows first): w_gu [2H, C] E4M3 (rows
 * [0, H) gate, [H, 2H) up) with gu_row_scale [2H] fp32.  Forwards to
 * qffn_decode_forward with w_gate = w_gu, w_up = w_gu + H*C,
 * s_gate = gu_row_scale, s_up = gu_row_scale + H; the same rules apply. */
qffn_status qffn_decode_forward_gu(uint16_t* out, const uint16_t* x, const uint8_t* w_gu,
                                   const float* gu_row_scale, const uint8_t* w_down,
                                   const float* s_down, int64_t C, int64_t H, void* workspace,
                                   size_t workspace_bytes, qffn_stream_t stream);

/* ---- Decode FFN without a caller workspace ---------------------------------
 * The pages have no counterpart of this call; it exists for callers that
 * cannot allocate device memory (for example code running where cudaMalloc is
 * not permitted, such as a plugin's enqueue step or a host callback, or a
 * process whose device memory is all owned by another allocator) and so
 * cannot supply the workspace of qffn_decode_forward.
 * Computes exactly what qffn_decode_forward computes (same kernels, same
 * bits), with its scratch (the g and u vectors) in a fixed array inside the
 * library: 2 x 32768 bf16 (128 KiB) per GPU that loads the library, held
 * until the process exits.  H > 32768 (and C > 32768) is rejected with
 * QFFN_ERR_UNSUPPORTED_SHAPE; the other size and alignment rules are those of
 * qffn_decode_forward.  Nothing is allocated by this call.
 * The first call with a given current CUDA context looks up the array's
 * device address in that context (after cudaDeviceReset, or under another
 * context, it is looked up again); make that first call before any stream
 * capture.  All calls on a device share the array and it keeps the last
 * call's contents (g and u are written before they are read, so nothing
 * needs clearing).  Calls that overlap in time on the GPU race on the
 * array: order them on one stream or with events. */
qffn_status qffn_decode_forward_noalloc(uint16_t* out, const uint16_t* x, const uint8_t* w_gate,
                                        const float* s_gate, const uint8_t* w_up,
                                        const float* s_up, const uint8_t* w_down,
                                        const float* s_down, int64_t C, int64_t H,
                                        qffn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QFFN_H_ */
