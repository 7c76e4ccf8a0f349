// Scaled FP8 (E4M3) GEMMs on the 5th-generation tensor cores (tcgen05, sm_103a).
//
//   gemm_bf16   : out[M,N]  = bf16(sA*sW * A[M,K] . W[N,K]^T (+ bias[N]) (+ out[M,N]))
//   gemm_swiglu : h[M,H]    = bf16(silu(g)*u), g / u the bf16-rounded gate and
//                 up products of W1 = [2H, K] (gate rows [0,H), up rows
//                 [H,2H)); the tensor abs-max of h is recorded on the way.
//   gemm_swiglu_quant : hq[M,H] = e4m3(h * 448 / amax_h) with amax_h given
//                 (read from stats_h[0], not recorded); stats_h[1] = scale.
//   gemm_swiglu_bwd : d_gu[M,2H] = (dh * u * silu'(g) | dh * silu(g)) for the
//                 recomputed bf16 g, u and dh [M,H] read in the epilogue; the
//                 abs-max of d_gu is recorded (recompute + swiglu_backward).
//
// These are the two matmuls of the FFN half of llmq "llama_model.cpp",
// LLamaModel::_forward_block (forward_qmm -> matmul with weight and
// activation scales; the up projection followed by swiglu_forward), and the
// up projection of _recompute_block followed by swiglu_forward_quant, which
// quantises h with the abs-max the forward recorded.
//
// Design: SM pairs.  The grid is a set of 2-CTA clusters, one CTA per SM,
// persistent over 256 x 256 output tiles.  Each tile is one chain of
// tcgen05.mma.cta_group::2 (M=256, N=256, K=32) issued by the pair's leader:
// CTA rank r stages rows [128r, 128r+128) of the tile's A slice and rows
// [128r, 128r+128) of its B slice, so per 128 of K an SM loads 16 KB of A and
// 16 KB of B instead of the 16 + 32 KB a one-SM 128 x 256 tile needs, and
// accumulates its own 128 rows x 256 columns in its own TMEM.
//   warp 0      TMA producer (both CTAs): 128x128-byte boxes, 128-byte
//               swizzle, two boxes of K per stage into a 3-stage ring of
//               256 K; the loads of both CTAs complete on the leader's
//               stage barrier.
//   warp 1      allocates 512 TMEM columns (pair-wide allocation); in the
//               leader one thread issues the MMAs and commits stage /
//               accumulator barriers to both CTAs at once (multicast).
//   warps 2..5  epilogue (both CTAs): tcgen05.ld of the fp32 accumulator
//               (one TMEM lane quarter per warp, one output row per thread,
//               8 columns per step in a rolled loop; the SwiGLU forward
//               forms at K <= 2048 take 16 per step, the next load in
//               flight), scaling, bf16 rounding, SwiGLU, abs-max; outputs
//               leave by TMA stores of 32 x 64 boxes from a swizzled
//               staging buffer, two per warp in flight (the E4M3 form
//               stores its codes directly); the accumulator is handed back
//               to the leader's MMA thread by a remote mbarrier arrive.
// The first CTA records its SM cycles and nanoseconds from start to end
// (gemm_clock_sample), from which the launch's mean SM clock follows.
// Operands are K-major (K contiguous, "TN") by default.  The bf16 form also
// reads A and / or W MN-major (the M or N index contiguous, i.e. the
// transposed matrix as it lies in memory): the TMA box is then 128 bytes of
// M (N) by 128 rows of K, which in the 128-byte swizzle is the canonical
// MN-major layout with one swizzle atom along M (N) per CTA, and the MMA
// reads it with the operand's major-ness bit set.  The FP8 backward uses it
// for W^T in the input gradient and for both operands of the weight gradient.
// Two 256-column accumulators in TMEM let the epilogue of tile i overlap the
// MMAs of tile i+1.  In the SwiGLU form CTA 0 stages 128 gate rows and CTA 1
// the matching 128 up rows, so the accumulator holds gate in columns
// [0,128) and up in [128,256) for each row.
//
// Every mbarrier wait is bounded (about 2 s on %globaltimer); a wait that
// runs out raises the CTA's abort flag and the device status word, all roles
// leave their loops, in-flight MMAs are drained (again bounded), both CTAs
// meet at a final cluster barrier, TMEM is freed and the kernel returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"
#include "pipeline.cuh"

namespace qffn {
namespace {

constexpr int BM = 128;        // rows of A per CTA (256 per pair)
constexpr int BN = 256;        // accumulator columns (N of one MMA)
constexpr int BK = 128;        // bytes (= E4M3 elements) of K per TMA box: one swizzle atom row
constexpr int KBOX = 2;        // boxes of K per stage (256 K per stage, 8 MMAs)
constexpr int BOX_BYTES = 128 * BK;        // one 128-row box of A or of this CTA's B half
constexpr int UMMA_K = 32;     // K of one kind::f8f6f4 MMA
// Three stages of 256 K rather than six of 128: the same shared memory, but
// each barrier round trip (full wait, fence, commit) now carries 8 MMAs
// instead of 4.  Measured with ncu on the gate|up GEMM: tensor pipe active
// 82.5% -> 92.2% of cycles (down GEMM 84% -> 89%).
constexpr int STAGES = 3;
constexpr int A_BYTES = KBOX * BOX_BYTES;  // this CTA's A rows of a stage
constexpr int B_BYTES = KBOX * BOX_BYTES;  // this CTA's half of the B rows of a stage
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NUM_THREADS = 192;
constexpr int TMEM_COLS = 2 * BN;
// + two per epilogue warp: its staging boxes' TMA loads (dh of the SwiGLU
// backward, the previous output of the accumulating bf16 form)
constexpr int NUM_BARS = 2 * STAGES + 5 + 8;
// SwiGLU h staging for the TMA stores: 4 epilogue warps x 2 buffers of a
// 32-row x 64-column bf16 box (4 KB, 128-byte swizzle)
constexpr int STAGE_BOX_BYTES = 32 * 64 * 2;
constexpr int STAGING_BYTES = 4 * 2 * STAGE_BOX_BYTES;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + STAGING_BYTES + 1024 + NUM_BARS * 8 + 16;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory of one CTA");
constexpr int GROUP_M = 8;     // tile raster: 8 pair M-blocks (2048 rows) sweep a band of N-blocks together
                                // (16, 32 and 64 measured: more DRAM reads or slower; one, N-fastest: the
                                // down GEMM's 58.7 MB weight matrix is not kept in L2 either)
constexpr uint16_t kBothCtas = 0x3;
constexpr uint16_t kLeaderOnly = 0x1;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;
constexpr unsigned long long kDrainLimitNs = 200000000ull;

// Instruction descriptor of tcgen05.mma.kind::f8f6f4: D f32 (bits 4-5 = 1),
// A and B E4M3 (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0),
// N >> 3 at bits 17-22, M >> 4 at bits 24-28 (M = 256 over the CTA pair).
constexpr uint32_t kIdesc = (1u << 4) | (uint32_t(BN >> 3) << 17) | (uint32_t((2 * BM) >> 4) << 24);
// Bits 15 / 16: A / B read MN-major.
constexpr uint32_t idesc_for(bool a_mn, bool b_mn) {
  return kIdesc | (a_mn ? (1u << 15) : 0u) | (b_mn ? (1u << 16) : 0u);
}
// The same descriptor with another N (bits 17-22 hold N >> 3).
constexpr uint32_t idesc_n(uint32_t idesc, int n) {
  return (idesc & ~(0x3Fu << 17)) | (uint32_t(n >> 3) << 17);
}
// Byte step of one UMMA_K slice inside a stage: along the 128-byte row for a
// K-major operand, UMMA_K rows of 128 bytes for an MN-major one.
constexpr uint32_t kStepK = UMMA_K;
constexpr uint32_t kStepMN = UMMA_K * 128;

__device__ unsigned int g_status;
// SM clock cycles and nanoseconds from start to end of the first CTA of the
// most recent launch (read by gemm_clock_sample).
__device__ unsigned long long g_clock_sample[2];

// Epilogue forms
constexpr int EPI_BF16 = 0;          // out = bf16(scaled accumulator)
constexpr int EPI_SWIGLU = 1;        // h = bf16(silu(g) * u), abs-max recorded
constexpr int EPI_SWIGLU_E4M3 = 2;   // hq = e4m3(h * 448 / given abs-max)
constexpr int EPI_SWIGLU_BWD = 3;    // d_gu = swiglu gradient from dh, abs-max recorded

struct GemmArgs {
  void* out;
  const float* a_scale;
  const float* w_scale;
  float* amax;   // SwiGLU: stats_h {abs_max, scale}
  const uint16_t* bias;   // bf16 output: optional bf16 bias per output column
  const uint16_t* dh;     // SwiGLU backward: gradient of h [M, H]
  int accumulate;         // bf16 output: add the previous contents of out (weight gradients)
  int M, N, K;   // N: output columns (SwiGLU: H)
  int H;         // SwiGLU: first up row of W1
  int tiles_m, tiles_n, num_tiles, num_kb;
  int band_n;    // N-blocks per raster band (tile_coords)
  // Work units below split_from are 256-column tiles; each unit from there on
  // is one 128-column half of the tiles split_from, split_from + 1, ...:
  // a last partial wave of R tiles runs as 2R half tiles in half the time
  // (the bf16 form with K-major operands that does not accumulate, and the
  // SwiGLU forward forms; split_from = num_tiles otherwise).
  int split_from;
};

// Bounded wait on a pipeline barrier of this kernel (status word g_status).
QFFN_DEVI bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                         bool honour_abort = true, unsigned long long limit = kWaitLimitNs) {
  return mbar_wait_bounded(bar, parity, abort_flag, &g_status, honour_abort, limit);
}

// Same, with cluster-scope acquire: for a barrier that the peer CTA arrives on.
QFFN_DEVI bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
QFFN_DEVI bool mbar_wait_cluster(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((i & 31u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        atomicOr(&g_status, 1u);
        return false;
      }
    }
  }
}

QFFN_DEVI uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
QFFN_DEVI uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
QFFN_DEVI uint32_t num_clusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// shared::cluster address of the same shared-memory offset in CTA `rank`
QFFN_DEVI uint32_t map_to_rank(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
QFFN_DEVI void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
QFFN_DEVI void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// 2-D tile load whose completion is signalled on a barrier of either CTA of
// the pair (`bar` is a shared::cluster address).
QFFN_DEVI void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// 2-D tile load into this CTA's shared memory, completing on its barrier `bar`;
// elements outside the tensor are filled with zeros.
QFFN_DEVI void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// 2-D tile store from shared memory (bulk-group completion); rows or columns
// beyond the tensor's extent are not written.
QFFN_DEVI void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(src)
               : "memory");
}
QFFN_DEVI void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most one committed store group still reads shared memory.
QFFN_DEVI void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// Wait until no committed store group still reads shared memory.
QFFN_DEVI void bulk_wait_read_0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Wait until every committed store group has completed.
QFFN_DEVI void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Order this thread's generic shared-memory writes before later async-proxy reads.
QFFN_DEVI void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

QFFN_DEVI void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

QFFN_DEVI void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
QFFN_DEVI void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor for a K-major operand in the 128-byte
// swizzle layout written by TMA: rows of 128 B, 8-row groups 1024 B apart
// (stride byte offset), leading byte offset unused for this layout (16 B),
// descriptor version 1 (bit 46), swizzle mode 2 = 128 B (bits 61-63).
QFFN_DEVI uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = uint64_t((saddr >> 4) & 0x3FFFu);
  d |= uint64_t(16 >> 4) << 16;
  d |= uint64_t(1024 >> 4) << 32;
  d |= uint64_t(1) << 46;
  d |= uint64_t(2) << 61;
  return d;
}

// D(tmem, both CTAs) (+)= A(smem, both CTAs) . B(smem, both CTAs)^T
QFFN_DEVI void mma_f8_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                            uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on the barrier at offset `bar` of every CTA in `mask` when all
// previously issued MMAs of this thread have completed.
QFFN_DEVI void mma_commit_mc(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

// Eight 32-bit TMEM columns of this warp's lane quarter.
QFFN_DEVI void tmem_ld8(uint32_t taddr, uint32_t (&v)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
               "tcgen05.wait::ld.sync.aligned;\n"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]) : "r"(taddr) : "memory");
}
// Eight 32-bit TMEM columns at each of two addresses (this warp's lane
// quarter), one wait for both.
QFFN_DEVI void tmem_ld8x2(uint32_t ta, uint32_t tb, uint32_t (&a)[8], uint32_t (&b)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%16];\n"
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8,%9,%10,%11,%12,%13,%14,%15}, [%17];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]),
        "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7])
      : "r"(ta), "r"(tb)
      : "memory");
}

// Issue the loads of sixteen 32-bit TMEM columns at each of two addresses
// (this warp's lane quarter) without waiting; tmem_wait_ld16 makes them usable.
QFFN_DEVI void tmem_ld16x2_issue(uint32_t ta, uint32_t tb, uint32_t (&a)[16], uint32_t (&b)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33];\n"
      : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]), "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]), "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]), "=r"(b[8]), "=r"(b[9]), "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15])
      : "r"(ta), "r"(tb)
      : "memory");
}
// Wait for this thread's TMEM loads.  The registers of the load being waited
// for pass through the wait, so that no use of them is placed before it.
QFFN_DEVI void tmem_wait_ld16(uint32_t (&a)[16], uint32_t (&b)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]), "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]), "+r"(a[15]), "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]), "+r"(b[6]), "+r"(b[7]), "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]), "+r"(b[12]), "+r"(b[13]), "+r"(b[14]), "+r"(b[15])
               :
               : "memory");
}
// Thirty-two 32-bit TMEM columns of this warp's lane quarter.
QFFN_DEVI void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
               "tcgen05.wait::ld.sync.aligned;\n"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
               : "r"(taddr)
               : "memory");
}
// Running max of |v| over bf16 pairs: lane-wise max of m and the absolute
// values of the two bf16 in v (exact, no rounding).
QFFN_DEVI uint32_t bf16x2_absmax(uint32_t m, uint32_t v) {
  uint32_t a, r;
  asm("abs.bf16x2 %0, %1;" : "=r"(a) : "r"(v));
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(m), "r"(a));
  return r;
}

// h for two adjacent accumulator columns: the packed bf16 pair
// (silu(g0) * u0, silu(g1) * u1) with g, u the scaled accumulators rounded to
// bf16 -- silu_mul_f32 on each, the multiplications done pairwise by f32x2
// instructions (each lane rounds as the scalar instruction does, so the
// result is the same bits).
QFFN_DEVI uint32_t swiglu_pair(uint32_t ga, uint32_t gb, uint32_t ua, uint32_t ub, uint64_t scale2) {
  float g0, g1, u0, u1;
  f2_unpack(f2_mul(f2_pack(__uint_as_float(ga), __uint_as_float(gb)), scale2), g0, g1);
  f2_unpack(f2_mul(f2_pack(__uint_as_float(ua), __uint_as_float(ub)), scale2), u0, u1);
  const uint32_t gr = pack_bf16x2(g0, g1), ur = pack_bf16x2(u0, u1);
  const uint64_t G = f2_pack(bf16_lo(gr), bf16_hi(gr));
  const uint64_t U = f2_pack(bf16_lo(ur), bf16_hi(ur));
  const float e0 = __expf(-fabsf(bf16_lo(gr))), e1 = __expf(-fabsf(bf16_hi(gr)));
  const uint64_t E = f2_pack(e0, e1);
  float d0, d1;
  f2_unpack(f2_add(f2_pack(1.0f, 1.0f), E), d0, d1);
  const float r0 = __fdividef(1.0f, d0), r1 = __fdividef(1.0f, d1);
  float er0, er1;
  f2_unpack(f2_mul(E, f2_pack(r0, r1)), er0, er1);
  const uint64_t S = f2_pack(bf16_lo(gr) >= 0.0f ? r0 : er0, bf16_hi(gr) >= 0.0f ? r1 : er1);
  float h0, h1;
  f2_unpack(f2_mul(f2_mul(G, S), U), h0, h1);
  return pack_bf16x2(h0, h1);
}

// Pair tile -> (pair M-block of 256 rows, N-block)
QFFN_DEVI void tile_coords(int tile, const GemmArgs& a, int& mb, int& nb);
// Work unit -> (pair M-block, N-block, half): half = -1 for a whole tile,
// 0 / 1 for the first / second 128 columns of a split one.
QFFN_DEVI void unit_coords(int u, const GemmArgs& a, int& mb, int& nb, int& half) {
  if (u < a.split_from) {
    tile_coords(u, a, mb, nb);
    half = -1;
  } else {
    const int h = u - a.split_from;
    tile_coords(a.split_from + (h >> 1), a, mb, nb);
    half = h & 1;
  }
}
// The raster: the N-blocks are cut into bands of band_n blocks; within a band,
// groups of GROUP_M pair M-blocks sweep the band's N-blocks with the M-block
// varying fastest (concurrent tiles share weight slices in L2), and odd groups
// sweep backwards (serpentine), so a group starts on the weight slices the
// previous group read last.  A band small enough to stay in L2 is read once
// while the activation groups cycle through it.
QFFN_DEVI void tile_coords(int tile, const GemmArgs& a, int& mb, int& nb) {
  const int band_tiles = a.tiles_m * a.band_n;
  const int band = tile / band_tiles;
  const int n0 = band * a.band_n;
  const int wb = min(a.band_n, a.tiles_n - n0);          // N-blocks of this band (the last may be short)
  const int t = tile - band * band_tiles;
  const int per_group = GROUP_M * wb;
  const int group = t / per_group;
  const int first_m = group * GROUP_M;
  const int gsize = min(a.tiles_m - first_m, GROUP_M);
  const int r = t - group * per_group;
  mb = first_m + r % gsize;
  nb = n0 + ((group & 1) ? wb - 1 - r / gsize : r / gsize);
}

template <int EPI, bool A_MN = false, bool B_MN = false, bool WIDE = false>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_fp8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC,
                    const __grid_constant__ CUtensorMap tmD,
                    const GemmArgs args) {
  const bool clock_cta = blockIdx.x == 0 && threadIdx.x == 0;
  const long long clk_start = clock_cta ? clock64() : 0;
  const unsigned long long ns_start = clock_cta ? globaltimer() : 0ull;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint8_t* sStaging = smem + STAGES * STAGE_BYTES;       // 1024-byte aligned
  uint64_t* bars = reinterpret_cast<uint64_t*>(sStaging + STAGING_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  // Barriers (same offsets in both CTAs):
  //   full[s]    leader: both CTAs' loads of stage s landed (1 arrival + tx)
  //   empty[s]   each CTA: the MMAs reading stage s are done (leader's commit)
  //   tfull[a]   each CTA: accumulator a holds a finished tile (leader's commit)
  //   tempty[a]  leader: both CTAs' epilogues have read accumulator a (8 warps)
  //   drain      leader: all MMAs issued have completed
  auto full_bar = [&](int s) { return bar0 + 8u * uint32_t(s); };
  auto empty_bar = [&](int s) { return bar0 + 8u * uint32_t(STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * uint32_t(2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * uint32_t(2 * STAGES + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * uint32_t(2 * STAGES + 4);
  //   ld[q][b]   epilogue warp of lane quarter q: the TMA load into its
  //              staging box b has landed
  auto ld_bar = [&](int q, int b) { return bar0 + 8u * uint32_t(2 * STAGES + 5 + 2 * q + b); };
  auto dh_bar = [&](int q) { return ld_bar(q, 0); };

  constexpr bool SWIGLU = EPI != EPI_BF16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair = int(cluster_id_x()), num_pairs = int(num_clusters_x());

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 8);
    }
    mbar_init(drain_bar, 1);
    for (int q = 0; q < 4; ++q) {
      mbar_init(ld_bar(q, 0), 1);
      mbar_init(ld_bar(q, 1), 1);
    }
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (EPI == EPI_SWIGLU || EPI == EPI_SWIGLU_BWD || EPI == EPI_BF16) tma_prefetch_desc(&tmC);
    if (EPI == EPI_SWIGLU_BWD) tma_prefetch_desc(&tmD);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  // both CTAs' barriers are initialised before either CTA signals the other's
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Launched as a programmatic dependent launch in the forward chains: the
  // set-up above overlaps the preceding kernel's tail; nothing in global
  // memory is read or written before the preceding kernel has completed.
  // (Both are no-ops in a plain launch.)
  pdl_wait();
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      uint32_t issued = 0, issued_parity = 0;
      int it = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < args.num_tiles; tile += num_pairs) {
        int mb, nb, half;
        unit_coords(tile, args, mb, nb, half);
        const int rowA = mb * (2 * BM) + int(rank) * BM;
        // a half tile's B rows: 64 per CTA, from the tensor map with 64-row boxes
        // SwiGLU: CTA 0 stages gate rows, CTA 1 the matching up rows (64 of
        // each in a half tile)
        const int rowB = SWIGLU ? (half < 0 ? (rank == 0 ? nb * 128 : args.H + nb * 128)
                                            : (rank == 0 ? 0 : args.H) + nb * 128 + half * 64)
                         : half < 0 ? nb * BN + int(rank) * 128
                                    : nb * BN + half * 128 + int(rank) * 64;
        const CUtensorMap* mapB = half < 0 ? &tmB : &tmD;
        const uint32_t stage_tx = half < 0 ? 2 * STAGE_BYTES : 2 * (A_BYTES + B_BYTES / 2);
        for (int kb = 0; kb < args.num_kb; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = uint32_t(it / STAGES) & 1u;
          if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag)) { ok = false; break; }
          if (rank == 0) mbar_expect_tx(full_bar(s), stage_tx);
          const uint32_t fb = map_to_rank(full_bar(s), 0);
          // K-major: x = K offset, y = row; MN-major: x = M (N) offset, y = K row
#pragma unroll
          for (int bx = 0; bx < KBOX; ++bx) {
            const int kx = (kb * KBOX + bx) * BK;
            const uint32_t da = smem_u32(sA + s * A_BYTES + bx * BOX_BYTES);
            const uint32_t db = smem_u32(sB + s * B_BYTES + bx * BOX_BYTES);
            if (A_MN) tma_load_2d_pair(da, &tmA, fb, rowA, kx);
            else tma_load_2d_pair(da, &tmA, fb, kx, rowA);
            if (B_MN) tma_load_2d_pair(db, &tmB, fb, rowB, kx);
            else tma_load_2d_pair(db, mapB, fb, kx, rowB);
          }
          issued |= 1u << s;
          issued_parity = (issued_parity & ~(1u << s)) | (ph << s);
        }
      }
      // drain (leader): every phase it armed has completed, so both CTAs'
      // loads into those stages have landed before shared memory is released
      if (rank == 0)
        for (int s = 0; s < STAGES; ++s)
          if (issued & (1u << s))
            mbar_wait(full_bar(s), (issued_parity >> s) & 1u, abort_flag, false, kDrainLimitNs);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ------------------------------------------------------------ MMA issuer (leader)
      int it = 0, local = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < args.num_tiles; tile += num_pairs, ++local) {
        const int acc = local & 1;
        const uint32_t aph = uint32_t(local >> 1) & 1u;
        if (!mbar_wait_cluster(tempty_bar(acc), aph ^ 1u, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + uint32_t(acc * BN);
        // a half tile is N = 128 (64 B rows per CTA)
        const uint32_t idesc = tile < args.split_from ? idesc_for(A_MN, B_MN)
                                                      : idesc_n(idesc_for(A_MN, B_MN), BN / 2);
        for (int kb = 0; kb < args.num_kb; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = uint32_t(it / STAGES) & 1u;
          if (!mbar_wait(full_bar(s), ph, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + s * A_BYTES);
          const uint32_t b0 = smem_u32(sB + s * B_BYTES);
#pragma unroll
          for (int bx = 0; bx < KBOX; ++bx)
#pragma unroll
            for (int kk = 0; kk < BK / UMMA_K; ++kk)
              mma_f8_pair(d_tmem, sdesc_sw128(a0 + bx * BOX_BYTES + kk * (A_MN ? kStepMN : kStepK)),
                          sdesc_sw128(b0 + bx * BOX_BYTES + kk * (B_MN ? kStepMN : kStepK)),
                          idesc, uint32_t(kb | bx | kk));
          mma_commit_mc(empty_bar(s), kBothCtas);
        }
        if (!ok) break;
        mma_commit_mc(tfull_bar(acc), kBothCtas);
      }
      // drain: all MMAs issued by this thread have completed
      mma_commit_mc(drain_bar, kLeaderOnly);
      mbar_wait(drain_bar, 0, abort_flag, false, kDrainLimitNs);
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;                  // TMEM lane quarter of this warp
    const int row_in_tile = int(rank) * BM + q * 32 + lane;
    const float scale = args.a_scale[0] * args.w_scale[0];
    float amax = 0.0f;
    uint32_t amax2 = 0u;     // WIDE EPI_SWIGLU: running max of |h| on bf16 pairs (exact)
    const uint64_t scale2 = f2_pack(scale, scale);
    int sbuf = 0;            // TMA-store forms: which of this warp's two staging boxes is next
    // EPI_SWIGLU_E4M3: quantise h with the given abs-max, as quantize_with_abs_max
    // does (fp32 product with 448 / abs_max, nearest even, saturating)
    float qinv = 0.0f;
    bool qzero = true;
    if (EPI == EPI_SWIGLU_E4M3) {
      const float given = args.amax[0];
      qzero = !(given > 0.0f);
      qinv = qzero ? 0.0f : 448.0f / given;
      if (blockIdx.x == 0 && threadIdx.x == 64) args.amax[1] = qzero ? 1.0f : given / 448.0f;
    }
    // (The two forms below that prefetch by TMA run whole tiles only -- the
    // host does not split their last wave -- so their work units map to
    // tiles one to one.)
    // EPI_SWIGLU_BWD: dh comes in by TMA, one 32-row x 64-column box per warp
    // and half tile, into staging box A of the warp; dg is written back over
    // it and du into box B, and both go out by TMA stores.  The first half's
    // box of the next tile is requested as soon as this tile's stores have
    // read the boxes, so it lands while the next accumulator is computed.
    uint8_t* boxA = sStaging + (q * 2) * STAGE_BOX_BYTES;
    uint8_t* boxB = boxA + STAGE_BOX_BYTES;
    uint32_t dh_par = 0;
    bool dh_pending = false;   // lane 0: a dh load has been issued and not waited for
    auto load_dh = [&](int t, int half) {    // lane 0
      int pmb, pnb;
      tile_coords(t, args, pmb, pnb);
      const int prow0 = pmb * (2 * BM) + int(rank) * BM + q * 32;
      mbar_expect_tx(dh_bar(q), STAGE_BOX_BYTES);
      tma_load_2d(smem_u32(boxA), &tmD, dh_bar(q), pnb * 128 + half * 64, prow0);
      dh_pending = true;
    };
    if (EPI == EPI_SWIGLU_BWD && lane == 0 && pair < args.num_tiles) load_dh(pair, 0);
    // accumulating bf16 form: the previous output comes in by TMA, one 32-row
    // x 64-column box (group g of the tile's 256 columns) into staging box
    // g & 1, the next group's load in flight while a group is summed
    uint32_t old_par[2] = {0u, 0u};
    bool old_pending[2] = {false, false};   // lane 0
    auto load_old = [&](int t, int g) {     // lane 0
      int pmb, pnb;
      tile_coords(t, args, pmb, pnb);
      const int prow0 = pmb * (2 * BM) + int(rank) * BM + q * 32;
      const int b = g & 1;
      mbar_expect_tx(ld_bar(q, b), STAGE_BOX_BYTES);
      tma_load_2d(smem_u32(sStaging + (q * 2 + b) * STAGE_BOX_BYTES), &tmC, ld_bar(q, b),
                  pnb * BN + g * 64, prow0);
      old_pending[b] = true;
    };
    if (EPI == EPI_BF16 && args.accumulate && lane == 0 && pair < args.num_tiles) load_old(pair, 0);
    int local = 0;
    for (int tile = pair; tile < args.num_tiles; tile += num_pairs, ++local) {
      const int acc = local & 1;
      const uint32_t aph = uint32_t(local >> 1) & 1u;
      if (!mbar_wait(tfull_bar(acc), aph, abort_flag)) break;
      tc_fence_after();
      int mb, nb, half;
      unit_coords(tile, args, mb, nb, half);
      const int row = mb * (2 * BM) + row_in_tile;
      const bool row_ok = row < args.M;
      const uint32_t tbase = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(acc * BN);
      if (!SWIGLU && !args.accumulate) {
        // bf16 out staged in shared memory and stored with TMA, one 32-row x
        // 64-column box per warp at a time (two buffers), as h in the SwiGLU
        // form: a warp's per-row 16-byte global stores would touch 32 rows
        // per instruction and load the L1 data pipe that the tensor core's
        // shared-memory operand reads also use.  The tensor map clips rows
        // beyond M and columns beyond N.
        const int row0 = mb * (2 * BM) + int(rank) * BM + q * 32;
        // a half tile holds 128 accumulator columns, starting at column 128 * half
        const int cbase = nb * BN + (half < 0 ? 0 : half * (BN / 2));
        const int ncols = half < 0 ? BN : BN / 2;
        // 32 columns per step, one tcgen05.ld x32: each TMEM load has a fixed
        // cost, which the last tile's epilogue (not hidden behind any main
        // loop) pays in full: 4.5 -> 3.2 us for one 256-column tile with 8
        // columns per load, about 1 us off every launch of this form.
#pragma unroll 1
        for (int c0 = 0; c0 < ncols; c0 += 32) {
          uint32_t v[32];
          tmem_ld32(tbase + uint32_t(c0), v);
          const int col = cbase + c0;
          uint8_t* sbox = sStaging + (q * 2 + sbuf) * STAGE_BOX_BYTES;
          if ((c0 & 63) == 0) {
            if (lane == 0) bulk_wait_read_1();   // the store that last read this box is done
            __syncwarp();
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int chunk = ((c0 & 63) >> 3) + k;
            uint32_t p[4];
            if (args.bias != nullptr) {
              const uint4 b4 = col + 8 * k < args.N ? ld16_ro(args.bias + col + 8 * k) : make_uint4(0, 0, 0, 0);
              const uint32_t bw[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
              for (int j = 0; j < 4; ++j)
                p[j] = pack_bf16x2(__uint_as_float(v[8 * k + 2 * j]) * scale + bf16_lo(bw[j]),
                                   __uint_as_float(v[8 * k + 2 * j + 1]) * scale + bf16_hi(bw[j]));
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                p[j] = pack_bf16x2(__uint_as_float(v[8 * k + 2 * j]) * scale,
                                   __uint_as_float(v[8 * k + 2 * j + 1]) * scale);
            }
            *reinterpret_cast<uint4*>(sbox + lane * 128 + ((chunk ^ (lane & 7)) << 4)) =
                make_uint4(p[0], p[1], p[2], p[3]);
          }
          if ((c0 & 63) == 32) {
            fence_proxy_async_smem();
            __syncwarp();
            const int x = cbase + (c0 & ~63);
            if (lane == 0) {
              if (row0 < args.M && x < args.N) tma_store_2d(&tmC, smem_u32(sbox), x, row0);
              bulk_commit();
            }
            sbuf ^= 1;
          }
        }
      } else if (!SWIGLU) {
        // accumulating form (weight gradients): out = bf16((acc + bias) + old),
        // old from the staging box the TMA load filled, written back in place
        // and stored by TMA
        const int row0 = mb * (2 * BM) + int(rank) * BM + q * 32;
        bool ok = true;
        for (int g = 0; g < BN / 64; ++g) {
          const int b = g & 1;
          uint8_t* box = sStaging + (q * 2 + b) * STAGE_BOX_BYTES;
          if (g + 1 < BN / 64) {
            if (lane == 0) {
              bulk_wait_read_0();              // the store that last read box (g+1)&1 is done
              load_old(tile, g + 1);
            }
            __syncwarp();
          }
          if (!mbar_wait(ld_bar(q, b), old_par[b], abort_flag)) { ok = false; break; }
          old_par[b] ^= 1u;
          if (lane == 0) old_pending[b] = false;
#pragma unroll 1
          for (int c8 = 0; c8 < 8; ++c8) {
            const int c0 = g * 64 + c8 * 8;
            const int col = nb * BN + c0;
            uint32_t v[8];
            tmem_ld8(tbase + uint32_t(c0), v);
            const uint32_t off = uint32_t(lane) * 128u + (uint32_t(c8 ^ (lane & 7)) << 4);
            const uint4 o4 = *reinterpret_cast<const uint4*>(box + off);
            const uint4 b4 = (args.bias != nullptr && col < args.N) ? ld16_ro(args.bias + col)
                                                                     : make_uint4(0, 0, 0, 0);
            const uint32_t bw[4] = {b4.x, b4.y, b4.z, b4.w}, ow[4] = {o4.x, o4.y, o4.z, o4.w};
            uint32_t p[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
              p[j] = pack_bf16x2(
                  (__uint_as_float(v[2 * j]) * scale + bf16_lo(bw[j])) + bf16_lo(ow[j]),
                  (__uint_as_float(v[2 * j + 1]) * scale + bf16_hi(bw[j])) + bf16_hi(ow[j]));
            *reinterpret_cast<uint4*>(box + off) = make_uint4(p[0], p[1], p[2], p[3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          const int x = nb * BN + g * 64;
          if (lane == 0) {
            if (row0 < args.M && x < args.N) tma_store_2d(&tmC, smem_u32(box), x, row0);
            bulk_commit();
          }
        }
        if (!ok) break;
        if (lane == 0) {
          bulk_wait_read_0();                  // this tile's stores have read both boxes
          if (tile + num_pairs < args.num_tiles) load_old(tile + num_pairs, 0);
        }
        __syncwarp();
      } else if (EPI == EPI_SWIGLU_BWD) {
        const int row0 = mb * (2 * BM) + int(rank) * BM + q * 32;
        bool ok = true;
        for (int half = 0; half < 2; ++half) {
          if (half == 1) {
            if (lane == 0) {
              bulk_wait_read_0();              // half 0's stores have read both boxes
              load_dh(tile, 1);
            }
            __syncwarp();
          }
          if (!mbar_wait(dh_bar(q), dh_par, abort_flag)) { ok = false; break; }
          dh_par ^= 1u;
          if (lane == 0) dh_pending = false;
#pragma unroll 1
          for (int c8 = 0; c8 < 8; ++c8) {
            const int c0 = half * 64 + c8 * 8;
            uint32_t g[8], u[8];
            tmem_ld8x2(tbase + uint32_t(c0), tbase + uint32_t(128 + c0), g, u);
            // this lane's row, 16-byte chunk c8 of the 128-byte-swizzled boxes
            const uint32_t off = uint32_t(lane) * 128u + (uint32_t(c8 ^ (lane & 7)) << 4);
            const uint4 d4 = *reinterpret_cast<const uint4*>(boxA + off);
            const uint32_t dw[4] = {d4.x, d4.y, d4.z, d4.w};
            uint32_t pg[4], pu[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              // g, u rounded to bf16 as the recomputed gate|up buffer holds them,
              // then the SwiGLU gradient with dh of the same row and columns
              float dg0, du0, dg1, du1;
              swiglu_grad(round_bf16(__uint_as_float(g[2 * j]) * scale),
                          round_bf16(__uint_as_float(u[2 * j]) * scale), bf16_lo(dw[j]), dg0, du0);
              swiglu_grad(round_bf16(__uint_as_float(g[2 * j + 1]) * scale),
                          round_bf16(__uint_as_float(u[2 * j + 1]) * scale), bf16_hi(dw[j]), dg1, du1);
              pg[j] = pack_bf16x2(dg0, dg1);
              pu[j] = pack_bf16x2(du0, du1);
              if (row_ok)
                amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16_lo(pg[j])), fabsf(bf16_hi(pg[j]))),
                                         fmaxf(fabsf(bf16_lo(pu[j])), fabsf(bf16_hi(pu[j])))));
            }
            *reinterpret_cast<uint4*>(boxA + off) = make_uint4(pg[0], pg[1], pg[2], pg[3]);
            *reinterpret_cast<uint4*>(boxB + off) = make_uint4(pu[0], pu[1], pu[2], pu[3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            // rows beyond M are clipped by the tensor map
            if (row0 < args.M) {
              tma_store_2d(&tmC, smem_u32(boxA), nb * 128 + half * 64, row0);
              tma_store_2d(&tmC, smem_u32(boxB), args.N + nb * 128 + half * 64, row0);
            }
            bulk_commit();
          }
        }
        if (!ok) break;
        if (lane == 0) {
          bulk_wait_read_0();                  // the stores have read box A
          if (tile + num_pairs < args.num_tiles) load_dh(tile + num_pairs, 0);
        }
        __syncwarp();
      } else {
        // a half tile holds 64 gate columns then the 64 matching up columns
        const int hbase = half < 0 ? 0 : half * 64;          // first h column of the unit
        const int hcols = half < 0 ? 128 : 64;
        const int up_off = half < 0 ? 128 : 64;               // accumulator column of u
        const size_t hoff = size_t(row) * size_t(args.N) + size_t(nb) * 128 + size_t(hbase);
        uint8_t* qrow = static_cast<uint8_t*>(args.out) + hoff;
        if constexpr (WIDE) {
          // Sixteen columns of g and u per step, two steps per turn of a rolled
          // loop (the launcher picks this form for K <= 2048, where the
          // epilogue and not the MMAs sets the tile rate; at longer K the
          // eight-column loop below measured faster).  One warp per
          // sub-partition runs this loop, so its rate is set by the
          // instruction-level parallelism of a step: sixteen columns give
          // sixteen independent SwiGLU chains, their multiplications paired in
          // f32x2 instructions.  The TMEM load of the next step is issued
          // before this step's arithmetic.
          uint32_t gq[2][16], uq[2][16];
          tmem_ld16x2_issue(tbase, tbase + uint32_t(up_off), gq[0], uq[0]);
#pragma unroll 1
          for (int c00 = 0; c00 < hcols; c00 += 32) {
#pragma unroll
            for (int st = 0; st < 2; ++st) {
              const int c0 = c00 + 16 * st;
              tmem_wait_ld16(gq[st], uq[st]);          // this step's columns have landed
              if (c0 + 16 < hcols) {
                __syncwarp();
                tmem_ld16x2_issue(tbase + uint32_t(c0 + 16), tbase + uint32_t(up_off + c0 + 16),
                                  gq[st ^ 1], uq[st ^ 1]);
              }
              // EPI_SWIGLU stages h in shared memory and stores it with TMA, one
              // 32-row x 64-column box per warp and half tile: each lane writes
              // its row's 16-byte chunks into the 128-byte-swizzled box (4
              // wavefronts per warp store), where per-thread 16-byte global
              // stores would touch 32 rows per instruction.
              uint8_t* sbox = sStaging + (q * 2 + sbuf) * STAGE_BOX_BYTES;
              if (EPI == EPI_SWIGLU && (c0 & 63) == 0) {
                if (lane == 0) bulk_wait_read_1();   // the store that last read this box is done
                __syncwarp();
              }
              uint32_t p[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                p[j] = swiglu_pair(gq[st][2 * j], gq[st][2 * j + 1], uq[st][2 * j], uq[st][2 * j + 1], scale2);
                if (EPI == EPI_SWIGLU && row_ok) amax2 = bf16x2_absmax(amax2, p[j]);
              }
              if (EPI == EPI_SWIGLU) {
                const int chunk = (c0 & 63) >> 3;      // even: this step fills chunks chunk, chunk + 1
#pragma unroll
                for (int k = 0; k < 2; ++k)
                  *reinterpret_cast<uint4*>(sbox + lane * 128 + (((chunk + k) ^ (lane & 7)) << 4)) =
                      make_uint4(p[4 * k], p[4 * k + 1], p[4 * k + 2], p[4 * k + 3]);
                if (chunk == 6) {
                  fence_proxy_async_smem();
                  __syncwarp();
                  const int row0 = mb * (2 * BM) + int(rank) * BM + q * 32;
                  if (lane == 0) {
                    if (row0 < args.M)
                      tma_store_2d(&tmC, smem_u32(sbox), nb * 128 + hbase + (c0 & ~63), row0);
                    bulk_commit();
                  }
                  sbuf ^= 1;
                }
              }
              if (EPI == EPI_SWIGLU_E4M3 && row_ok) {
                uint32_t c[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  const uint16_t lo = qzero ? uint16_t(0)
                                            : f32x2_to_e4m3x2(bf16_lo(p[2 * j]) * qinv, bf16_hi(p[2 * j]) * qinv);
                  const uint16_t hi = qzero ? uint16_t(0)
                                            : f32x2_to_e4m3x2(bf16_lo(p[2 * j + 1]) * qinv,
                                                              bf16_hi(p[2 * j + 1]) * qinv);
                  c[j] = uint32_t(lo) | (uint32_t(hi) << 16);
                }
                *reinterpret_cast<uint4*>(qrow + c0) = make_uint4(c[0], c[1], c[2], c[3]);
              }
            }
          }
        } else {
          // Eight columns of g and u per step in a rolled loop: the epilogue's
          // code stays small, so it does not crowd the producer's and the MMA
          // issuer's loops out of the instruction cache of the SM sub-partitions
          // it shares with them (measured: 2.4% fewer cycles per GEMM than a
          // fully unrolled 32-column step).
  #pragma unroll 1
          for (int c0 = 0; c0 < hcols; c0 += 8) {
            uint32_t g[8], u[8];
            tmem_ld8x2(tbase + uint32_t(c0), tbase + uint32_t(up_off + c0), g, u);
            {
              // EPI_SWIGLU stages h in shared memory and stores it with TMA, one
              // 32-row x 64-column box per warp and half tile: each lane writes
              // its row's 16 bytes into the 128-byte-swizzled box (4 wavefronts
              // per warp store), where per-thread 16-byte global stores would
              // touch 32 rows per instruction.
              uint8_t* sbox = sStaging + (q * 2 + sbuf) * STAGE_BOX_BYTES;
              if (EPI == EPI_SWIGLU && (c0 & 63) == 0) {
                if (lane == 0) bulk_wait_read_1();   // the store that last read this box is done
                __syncwarp();
              }
              uint32_t p[4];
  #pragma unroll
              for (int j = 0; j < 4; ++j) {
                const float g0 = round_bf16(__uint_as_float(g[2 * j]) * scale);
                const float g1 = round_bf16(__uint_as_float(g[2 * j + 1]) * scale);
                const float u0 = round_bf16(__uint_as_float(u[2 * j]) * scale);
                const float u1 = round_bf16(__uint_as_float(u[2 * j + 1]) * scale);
                p[j] = pack_bf16x2(silu_mul_f32(g0, u0), silu_mul_f32(g1, u1));
                if (EPI == EPI_SWIGLU && row_ok)
                  amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(p[j])), fabsf(bf16_hi(p[j]))));
              }
              if (EPI == EPI_SWIGLU) {
                const int chunk = (c0 & 63) >> 3;
                *reinterpret_cast<uint4*>(sbox + lane * 128 + ((chunk ^ (lane & 7)) << 4)) =
                    make_uint4(p[0], p[1], p[2], p[3]);
                if (chunk == 7) {
                  fence_proxy_async_smem();
                  __syncwarp();
                  const int row0 = mb * (2 * BM) + int(rank) * BM + q * 32;
                  if (lane == 0) {
                    if (row0 < args.M)
                      tma_store_2d(&tmC, smem_u32(sbox), nb * 128 + hbase + (c0 & ~63), row0);
                    bulk_commit();
                  }
                  sbuf ^= 1;
                }
              }
              if (EPI == EPI_SWIGLU_E4M3 && row_ok) {
                uint32_t c[2];
  #pragma unroll
                for (int j = 0; j < 2; ++j) {
                  const uint16_t lo = qzero ? uint16_t(0)
                                            : f32x2_to_e4m3x2(bf16_lo(p[2 * j]) * qinv, bf16_hi(p[2 * j]) * qinv);
                  const uint16_t hi = qzero ? uint16_t(0)
                                            : f32x2_to_e4m3x2(bf16_lo(p[2 * j + 1]) * qinv,
                                                              bf16_hi(p[2 * j + 1]) * qinv);
                  c[j] = uint32_t(lo) | (uint32_t(hi) << 16);
                }
                *reinterpret_cast<uint2*>(qrow + c0) = make_uint2(c[0], c[1]);
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(map_to_rank(tempty_bar(acc), 0));
    }
    // the TMA stores complete (shared memory read, global memory written) and
    // no TMA load into shared memory is in flight before exit
    if ((EPI == EPI_SWIGLU || EPI == EPI_SWIGLU_BWD || EPI == EPI_BF16) && lane == 0) bulk_wait_all();
    if (EPI == EPI_BF16 && args.accumulate && lane == 0)
      for (int b = 0; b < 2; ++b)
        if (old_pending[b]) mbar_wait(ld_bar(q, b), old_par[b], abort_flag, false, kDrainLimitNs);
    if (EPI == EPI_SWIGLU_BWD && lane == 0 && dh_pending)
      mbar_wait(dh_bar(q), dh_par, abort_flag, false, kDrainLimitNs);
    if (EPI == EPI_SWIGLU || EPI == EPI_SWIGLU_BWD) {
      if (EPI == EPI_SWIGLU && WIDE) amax = fmaxf(amax, fmaxf(bf16_lo(amax2), bf16_hi(amax2)));
      amax = warp_max(amax);
      if (lane == 0) atomic_max_nonneg(args.amax, amax);
    }
  }

  // Both CTAs finish together: the leader's MMAs write the peer's TMEM and
  // both CTAs signal barriers of the other, so neither frees TMEM or exits
  // while the other may still touch it.
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS)
                 : "memory");
  }
  if (clock_cta) {
    g_clock_sample[0] = static_cast<unsigned long long>(clock64() - clk_start);
    g_clock_sample[1] = globaltimer() - ns_start;
  }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D E4M3 tensor [rows, k] (k contiguous), boxes of box_rows rows x 128 bytes.
bool make_map(CUtensorMap* map, const uint8_t* ptr, int64_t rows, int64_t k,
              uint32_t box_rows = 128) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {cuuint64_t(k), cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(k)};
  cuuint32_t box[2] = {cuuint32_t(BK), box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D bf16 tensor [rows, cols] (cols contiguous) for the epilogue's TMA
// stores (and the SwiGLU backward's dh loads): boxes of 32 rows x 64
// columns, 128-byte swizzle.
bool make_store_map_bf16(CUtensorMap* map, uint16_t* ptr, int64_t rows, int64_t cols) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(cols) * 2};
  cuuint32_t box[2] = {64u, 32u};
  cuuint32_t estr[2] = {1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Number of 2-CTA clusters of this kernel that fit on the device at once
// (cached per device and form).
template <int EPI, bool A_MN = false, bool B_MN = false, bool WIDE = false>
cudaError_t max_pairs(int* pairs) {
  static int cached[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && cached[dev] > 0) {
    *pairs = cached[dev];
    return cudaSuccess;
  }
  e = cudaFuncSetAttribute(gemm_fp8_kernel<EPI, A_MN, B_MN, WIDE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (num_sms() / 2));
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, gemm_fp8_kernel<EPI, A_MN, B_MN, WIDE>, &cfg);
  if (e != cudaSuccess) return e;
  if (n < 1) return cudaErrorInvalidConfiguration;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  *pairs = n;
  return cudaSuccess;
}

template <int EPI, bool A_MN = false, bool B_MN = false, bool WIDE = false>
cudaError_t launch(const CUtensorMap& ma, const CUtensorMap& mb, GemmArgs a, cudaStream_t s,
                   const CUtensorMap* mc = nullptr, bool pdl = false,
                   const CUtensorMap* md = nullptr) {
  int pairs = 0;
  cudaError_t e = max_pairs<EPI, A_MN, B_MN, WIDE>(&pairs);
  if (e != cudaSuccess) return e;
  if (a.num_tiles < pairs) pairs = a.num_tiles;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, gemm_fp8_kernel<EPI, A_MN, B_MN, WIDE>, ma, mb, mc != nullptr ? *mc : ma,
                            md != nullptr ? *md : ma, a);
}

// A last partial wave of R <= pairs / 2 tiles runs as 2R half tiles (N = 128)
// in half a tile's time: sets split_from and num_tiles, and the weight tensor
// map with 64-row boxes that the half tiles' B loads use.  Leaves the
// arguments unchanged otherwise.
template <int EPI, bool WIDE = false>
cudaError_t split_last_wave(GemmArgs* a, CUtensorMap* mb_half, const uint8_t* W, int64_t wrows,
                            int64_t K) {
  int pairs = 0;
  cudaError_t e = max_pairs<EPI, false, false, WIDE>(&pairs);
  if (e != cudaSuccess) return e;
  const int r = a->num_tiles % pairs;
  if (a->num_tiles > pairs && r > 0 && 2 * r <= pairs) {
    if (!make_map(mb_half, W, wrows, K, 64)) return cudaErrorInvalidValue;
    a->split_from = a->num_tiles - r;
    a->num_tiles += r;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_gemm_bf16(uint16_t* out, const uint8_t* A, const float* a_scale,
                             const uint8_t* W, const float* w_scale, int64_t M, int64_t N,
                             int64_t K, cudaStream_t s, const uint16_t* bias, bool accumulate,
                             bool a_mn, bool w_mn, bool pdl) {
  if (M == 0) return cudaSuccess;
  CUtensorMap ma, mb;
  // an MN-major operand lies in memory as [K rows, M (N) contiguous]
  const bool ok = (a_mn ? make_map(&ma, A, K, M) : make_map(&ma, A, M, K)) &&
                  (w_mn ? make_map(&mb, W, K, N) : make_map(&mb, W, N, K));
  if (!ok) return cudaErrorInvalidValue;
  GemmArgs a{};
  a.out = out;
  a.a_scale = a_scale;
  a.w_scale = w_scale;
  a.amax = nullptr;
  a.bias = bias;
  a.accumulate = accumulate ? 1 : 0;
  a.M = int(M);
  a.N = int(N);
  a.K = int(K);
  a.H = 0;
  a.tiles_m = int((M + 2 * BM - 1) / (2 * BM));
  a.tiles_n = int((N + BN - 1) / BN);
  a.num_tiles = a.tiles_m * a.tiles_n;
  // one band: the bf16-output GEMMs' activation operand is the larger one
  // (down: 235 MB against 59 MB of weights), and cutting the weights into
  // bands re-reads it per band (measured: 1.1-1.45 GB read instead of 0.92)
  a.band_n = a.tiles_n;
  a.num_kb = int((K + KBOX * BK - 1) / (KBOX * BK));
  a.split_from = a.num_tiles;
  // the output tensor map of the epilogue's TMA stores (and, when
  // accumulating, of its loads of the previous output)
  CUtensorMap mc;
  if (!make_store_map_bf16(&mc, out, M, N)) return cudaErrorInvalidValue;
  const CUtensorMap* pmc = &mc;
  if (a_mn && w_mn) return launch<EPI_BF16, true, true>(ma, mb, a, s, pmc, pdl);
  if (a_mn) return launch<EPI_BF16, true, false>(ma, mb, a, s, pmc, pdl);
  if (w_mn) return launch<EPI_BF16, false, true>(ma, mb, a, s, pmc, pdl);
  // K-major, not accumulating: a short last wave runs as half tiles
  CUtensorMap mb_half;
  if (!accumulate) {
    cudaError_t e = split_last_wave<EPI_BF16>(&a, &mb_half, W, N, K);
    if (e != cudaSuccess) return e;
  }
  return launch<EPI_BF16>(ma, mb, a, s, pmc, pdl, a.split_from < a.num_tiles ? &mb_half : nullptr);
}

namespace {
// N-blocks per raster band of the SwiGLU forms: about 32 MB of W1 (an N-block
// is 128 gate and 128 up rows of K bytes).  Measured at the 8B shape (ncu DRAM
// bytes per launch of the gate|up GEMM): one band 817 MB read, bands of 16 MB
// 595, 32 MB 544, 64 MB 694; time within 2%.
int band_blocks(int tiles_n, int64_t K) {
  const int64_t per = int64_t(256) * K;
  int64_t b = (int64_t(32) << 20) / (per > 0 ? per : 1);
  if (b < 1) b = 1;
  return b > tiles_n ? tiles_n : int(b);
}

// The SwiGLU forward forms' epilogue: sixteen columns per step (WIDE) when a
// tile's main loop is at most 8 stages (K <= 2048), where the epilogue and
// not the MMAs sets the tile rate; eight otherwise.  Per-tile clock stamps at
// K = 2048 (Llama-3.2-1B gate|up): main loop 4.07 us, epilogue 5.0 us with
// eight columns per step.  Measured, gate|up alone, interleaved: K = 2048
// 0.091 -> 0.082 ms with the wide step; K = 3584 and 4096 0.541 -> 0.558 and
// 0.924 -> 0.948 ms, so the long-K forms keep the narrow step.
bool wide_epilogue(int64_t K) { return K <= 2048; }

// Tensor maps and arguments shared by the two SwiGLU forms.
bool swiglu_args(GemmArgs* a, CUtensorMap* ma, CUtensorMap* mb, void* out, float* stats_h,
                 const uint8_t* A, const float* a_scale, const uint8_t* W1, const float* w_scale,
                 int64_t M, int64_t H, int64_t K) {
  if (!make_map(ma, A, M, K) || !make_map(mb, W1, 2 * H, K)) return false;
  *a = GemmArgs{};
  a->out = out;
  a->a_scale = a_scale;
  a->w_scale = w_scale;
  a->amax = stats_h;
  a->M = int(M);
  a->N = int(H);
  a->K = int(K);
  a->H = int(H);
  a->tiles_m = int((M + 2 * BM - 1) / (2 * BM));
  a->tiles_n = int(H / 128);
  a->num_tiles = a->tiles_m * a->tiles_n;
  a->band_n = band_blocks(a->tiles_n, K);
  a->num_kb = int((K + KBOX * BK - 1) / (KBOX * BK));
  a->split_from = a->num_tiles;
  return true;
}
}  // namespace

cudaError_t launch_gemm_swiglu(uint16_t* h, float* stats_h, const uint8_t* A, const float* a_scale,
                               const uint8_t* W1, const float* w_scale, int64_t M, int64_t H,
                               int64_t K, cudaStream_t s, bool chained) {
  if (!chained) {
    cudaError_t e = cudaMemsetAsync(stats_h, 0, sizeof(float), s);
    if (e != cudaSuccess) return e;
  }
  if (M == 0) return cudaSuccess;
  CUtensorMap ma, mb;
  GemmArgs a;
  if (!swiglu_args(&a, &ma, &mb, h, stats_h, A, a_scale, W1, w_scale, M, H, K))
    return cudaErrorInvalidValue;
  CUtensorMap mc;
  if (!make_store_map_bf16(&mc, h, M, H)) return cudaErrorInvalidValue;
  CUtensorMap mb_half;
  if (wide_epilogue(K)) {
    cudaError_t e = split_last_wave<EPI_SWIGLU, true>(&a, &mb_half, W1, 2 * H, K);
    if (e != cudaSuccess) return e;
    return launch<EPI_SWIGLU, false, false, true>(ma, mb, a, s, &mc, chained,
                                                  a.split_from < a.num_tiles ? &mb_half : nullptr);
  }
  cudaError_t e = split_last_wave<EPI_SWIGLU>(&a, &mb_half, W1, 2 * H, K);
  if (e != cudaSuccess) return e;
  return launch<EPI_SWIGLU>(ma, mb, a, s, &mc, chained,
                            a.split_from < a.num_tiles ? &mb_half : nullptr);
}

cudaError_t launch_gemm_swiglu_quant(uint8_t* hq, float* stats_h, const uint8_t* A,
                                     const float* a_scale, const uint8_t* W1, const float* w_scale,
                                     int64_t M, int64_t H, int64_t K, cudaStream_t s,
                                     bool pdl) {
  // no rows: only the scale word is written (the elementwise form with N = 0)
  if (M == 0) return launch_swiglu_requant(hq, stats_h, nullptr, 0, H, s);
  CUtensorMap ma, mb;
  GemmArgs a;
  if (!swiglu_args(&a, &ma, &mb, hq, stats_h, A, a_scale, W1, w_scale, M, H, K))
    return cudaErrorInvalidValue;
  CUtensorMap mb_half;
  if (wide_epilogue(K)) {
    cudaError_t e = split_last_wave<EPI_SWIGLU_E4M3, true>(&a, &mb_half, W1, 2 * H, K);
    if (e != cudaSuccess) return e;
    return launch<EPI_SWIGLU_E4M3, false, false, true>(ma, mb, a, s, nullptr, pdl,
                                                       a.split_from < a.num_tiles ? &mb_half : nullptr);
  }
  cudaError_t e = split_last_wave<EPI_SWIGLU_E4M3>(&a, &mb_half, W1, 2 * H, K);
  if (e != cudaSuccess) return e;
  return launch<EPI_SWIGLU_E4M3>(ma, mb, a, s, nullptr, pdl,
                                 a.split_from < a.num_tiles ? &mb_half : nullptr);
}

cudaError_t launch_gemm_swiglu_bwd(uint16_t* d_gu, float* stats, const uint16_t* dh,
                                   const uint8_t* A, const float* a_scale, const uint8_t* W1,
                                   const float* w_scale, int64_t M, int64_t H, int64_t K,
                                   cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(stats, 0, sizeof(float), s);
  if (e != cudaSuccess || M == 0) return e;
  CUtensorMap ma, mb;
  GemmArgs a;
  if (!swiglu_args(&a, &ma, &mb, d_gu, stats, A, a_scale, W1, w_scale, M, H, K))
    return cudaErrorInvalidValue;
  a.dh = dh;
  // d_gu [M, 2H] written and dh [M, H] read by TMA in 32 x 64 boxes
  CUtensorMap mc, md;
  if (!make_store_map_bf16(&mc, d_gu, M, 2 * H) ||
      !make_store_map_bf16(&md, const_cast<uint16_t*>(dh), M, H))
    return cudaErrorInvalidValue;
  return launch<EPI_SWIGLU_BWD>(ma, mb, a, s, &mc, false, &md);
}

// Self-test of the failure path: the bounded pipeline wait every GEMM role
// uses, on two barriers of arrival count 1 in one CTA.  Lane 0 of warp 0
// waits on barrier 0 for `limit` ns; lane 0 of warp 1 waits on barrier 1 for
// 4 x limit and honours the CTA abort flag.  With `arrive` each barrier gets
// its arrival first and both waits succeed at once.  Without it nothing
// arrives: warp 0 runs out (abort flag up, g_status bit 0) and warp 1 leaves
// on the abort flag, after about `limit` rather than its own 4 x limit.
// out[0..1] = 1 if the wait of warp 0 / 1 succeeded, out[2..3] = its ns.
__global__ void __launch_bounds__(64) wait_selftest_kernel(unsigned long long* out, int arrive,
                                                           unsigned long long limit) {
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ int abort_word;
  volatile int* abort_flag = &abort_word;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(smem_u32(&bars[0]), 1);
    mbar_init(smem_u32(&bars[1]), 1);
    mbar_init_fence();
    if (arrive) {
      mbar_arrive(smem_u32(&bars[0]));
      mbar_arrive(smem_u32(&bars[1]));
    }
  }
  __syncthreads();
  if (lane == 0) {
    const unsigned long long t0 = globaltimer();
    const bool ok = mbar_wait(smem_u32(&bars[warp]), 0, abort_flag, true,
                              warp == 0 ? limit : 4 * limit);
    out[warp] = ok ? 1ull : 0ull;
    out[2 + warp] = globaltimer() - t0;
  }
}

cudaError_t launch_wait_selftest(unsigned long long* out, int arrive, unsigned long long limit_ns,
                                 cudaStream_t s) {
  wait_selftest_kernel<<<1, 64, 0, s>>>(out, arrive, limit_ns);
  return cudaGetLastError();
}

cudaError_t gemm_clock_sample(unsigned long long out[2]) {
  return cudaMemcpyFromSymbol(out, g_clock_sample, 2 * sizeof(unsigned long long));
}

cudaError_t gemm_take_status(unsigned int* status) {
  unsigned int v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_status, sizeof(v));
  if (e != cudaSuccess) return e;
  if (v != 0) e = cudaMemcpyToSymbol(g_status, &zero, sizeof(zero));
  *status = v;
  return e;
}

}  // namespace qffn
