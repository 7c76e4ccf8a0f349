// mbarrier / bulk-copy helpers shared by the pipelined kernels (inline PTX, sm_103a).
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace qffn {

QFFN_DEVI uint32_t smem_u32(const void* p) { return uint32_t(__cvta_generic_to_shared(p)); }

QFFN_DEVI void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
QFFN_DEVI void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
QFFN_DEVI void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
QFFN_DEVI bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
QFFN_DEVI unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Make the barrier initialisations visible to the async proxy (TMA / bulk copies).
QFFN_DEVI void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Waits for the phase of `bar` with the given parity to complete.  Returns
// false if the CTA abort flag is up (when honoured) or `limit` ns pass; running
// out raises the abort flag and sets bit 0 of *status.
QFFN_DEVI bool mbar_wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                 unsigned int* status, bool honour_abort,
                                 unsigned long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 31u) == 0) {
      if (honour_abort && *abort_flag) return false;
      if (globaltimer() - t0 > limit) {
        *abort_flag = 1;
        atomicOr(status, 1u);
        return false;
      }
    }
  }
}

// Contiguous global -> shared bulk copy (16-byte aligned addresses, size a
// multiple of 16) completing on `bar` with `bytes` transaction bytes.
QFFN_DEVI void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Barrier over the first `count` threads of the CTA (named barrier `id`).
QFFN_DEVI void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

}  // namespace qffn
