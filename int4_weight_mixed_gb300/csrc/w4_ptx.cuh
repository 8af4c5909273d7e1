// w4_ptx.cuh — thin inline-PTX wrappers for sm_103a: mbarriers, bulk and
// tensor TMA copies, and the tcgen05 (5th-generation tensor core / tensor
// memory) instructions used by the GEMM mainloop.  Every wait here is
// bounded: it gives up after W4_WAIT_TIMEOUT_NS of wall time, records a
// timeout in the kernel's status word and returns false.
#pragma once
#include <cstdint>
#include <cuda.h>

#ifndef W4_WAIT_TIMEOUT_NS
#define W4_WAIT_TIMEOUT_NS 2000000000ull  // 2 s
#endif

namespace w4 {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// a / b for non-negative 64-bit values, in 32-bit arithmetic when both fit:
// division by a runtime value is a long dependent instruction sequence, and
// the 64-bit one several times longer (it delays a CTA's first copy).
__device__ __forceinline__ int64_t div_nn(int64_t a, int64_t b) {
  if (((a | b) >> 32) == 0)
    return static_cast<int64_t>(static_cast<uint32_t>(a) / static_cast<uint32_t>(b));
  return a / b;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
// With SLEEP, a waiting thread is suspended in hardware until the phase
// completes or W4_WAIT_HINT_NS has passed (then the caller checks its abort
// flag and the time limit and waits again) instead of returning to a polling
// loop: in the tensor-core kernel the idle converter warps otherwise spend a
// large share of an SM's issue slots polling, next to the warps doing the
// work (all its waits sleep: measured 3% faster).  The decode and
// quantization kernels poll (measured 0.5% slower with the hint).
#ifndef W4_WAIT_HINT_NS
#define W4_WAIT_HINT_NS 100000u  // 100 us
#endif
template <bool SLEEP = false>
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  if (SLEEP && W4_WAIT_HINT_NS != 0u)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(static_cast<uint32_t>(W4_WAIT_HINT_NS))
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
  return ok != 0;
}

// Non-blocking test of the same condition.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase with the given parity has completed.  Gives up when
// *abort is set by another thread of the CTA, or after the time limit (then
// it sets *abort and the status word).  Returns true on success.
template <bool SLEEP = false>
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          int* status) {
  if (mbar_test_wait(bar, parity)) return true;
  uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait<SLEEP>(bar, parity)) return true;
    if ((SLEEP && W4_WAIT_HINT_NS != 0u) || (it & 63u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > W4_WAIT_TIMEOUT_NS) {
        *abort = 1;
        if (status) atomicExch(status, 5 /* W4_ERR_TIMEOUT */);
        return false;
      }
    }
  }
}

// Wait until the high half of a global counter (bits 16..31) reaches
// `target`, reading it with acquire semantics at device scope; bounded like
// mbar_wait.
__device__ __forceinline__ bool wait_count_hi(const int* ctr, int target, volatile int* abort,
                                              int* status) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    if ((v >> 16) >= target) return true;
    if (it == 0) {
      t0 = global_timer_ns();
    } else if ((it & 15u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > W4_WAIT_TIMEOUT_NS) {
        *abort = 1;
        if (status) atomicExch(status, 5 /* W4_ERR_TIMEOUT */);
        return false;
      }
    }
    __nanosleep(64);
  }
}

// ------------------------------------------------------- global accesses
// 32 contiguous bytes (16-byte aligned) loaded at L2 (bypassing L1, which
// does not see other SMs' writes) or stored.
__device__ __forceinline__ void ld_cg_v8(const void* p, uint32_t (&v)[8]) {
  const uint4* q = static_cast<const uint4*>(p);
  const uint4 a = __ldcg(q), b = __ldcg(q + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void st_v8(void* p, const uint32_t* v) {
  uint4* q = static_cast<uint4*>(p);
  q[0] = make_uint4(v[0], v[1], v[2], v[3]);
  q[1] = make_uint4(v[4], v[5], v[6], v[7]);
}
// 8 words as two 16-byte halves `half` words apart (a warp's lanes 16 bytes
// apart: each load or store instruction covers 512 contiguous bytes).
__device__ __forceinline__ void ld_cg_halves(const uint32_t* p, int half, uint32_t (&v)[8]) {
  const uint4 a = __ldcg(reinterpret_cast<const uint4*>(p));
  const uint4 b = __ldcg(reinterpret_cast<const uint4*>(p + half));
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void st_halves(uint32_t* p, int half, const uint32_t* v) {
  *reinterpret_cast<uint4*>(p) = make_uint4(v[0], v[1], v[2], v[3]);
  *reinterpret_cast<uint4*>(p + half) = make_uint4(v[4], v[5], v[6], v[7]);
}
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// ------------------------------------------------------------- bulk copies
// 1-D bulk copy global -> shared, completion counted on `bar` (bytes must be
// a multiple of 16, both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// 2-D tiled tensor copy global -> shared (x = innermost coordinate).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// The same two copies with shared-memory destinations given as 32-bit
// shared addresses.
__device__ __forceinline__ void bulk_g2s_a(uint32_t dst, const void* src, uint32_t bytes,
                                           uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d_a(uint32_t dst, const CUtensorMap* map, int32_t x,
                                              int32_t y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx_a(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ----------------------------------------------------------------- tcgen05
// Tensor memory allocation (whole warp).  The base address is written to
// shared memory at `slot`.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(slot)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[128 x N] (+)= A[128 x 16] * B[16 x N]; A read from tensor memory, B from
// shared memory through a matrix descriptor; kind::f16 (f16 or bf16 inputs,
// fp32 accumulator).
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Four MMAs covering one K block (64 K of f16 / bf16, or 128 K of E4M3):
// A columns a0 + 8*kk, B descriptors desc + 2*kk (32 bytes further along the
// 128-byte swizzled rows each).  Operands are formed before the asm block;
// the first MMA overwrites D when `accumulate` is 0.  F8: kind::f8f6f4
// (E4M3 x E4M3, 32 K per MMA) instead of kind::f16 (16 K per MMA).
#define W4_MMA4_STR(KIND)                                  \
  "{\n\t.reg .pred p, t;\n\t"                              \
  "setp.ne.b32 p, %4, 0;\n\t"                              \
  "setp.eq.b32 t, %4, %4;\n\t"                             \
  "tcgen05.mma.cta_group::1.kind::" KIND " [%0], [%1], %2, %3, p;\n\t"  \
  "tcgen05.mma.cta_group::1.kind::" KIND " [%0], [%5], %6, %3, t;\n\t"  \
  "tcgen05.mma.cta_group::1.kind::" KIND " [%0], [%7], %8, %3, t;\n\t"  \
  "tcgen05.mma.cta_group::1.kind::" KIND " [%0], [%9], %10, %3, t;\n\t}"
template <bool F8 = false>
__device__ __forceinline__ void mma_ts_stage(uint32_t d_tmem, uint32_t a0, uint64_t desc,
                                             uint32_t idesc, uint32_t accumulate) {
  const uint32_t a1 = a0 + 8, a2 = a0 + 16, a3 = a0 + 24;
  const uint64_t d1 = desc + 2, d2 = desc + 4, d3 = desc + 6;
  if constexpr (F8)
    asm volatile(W4_MMA4_STR("f8f6f4")::"r"(d_tmem), "r"(a0), "l"(desc), "r"(idesc),
                 "r"(accumulate), "r"(a1), "l"(d1), "r"(a2), "l"(d2), "r"(a3), "l"(d3)
                 : "memory");
  else
    asm volatile(W4_MMA4_STR("f16")::"r"(d_tmem), "r"(a0), "l"(desc), "r"(idesc),
                 "r"(accumulate), "r"(a1), "l"(d1), "r"(a2), "l"(d2), "r"(a3), "l"(d3)
                 : "memory");
}

// Sixteen MMAs covering a stage made of four K blocks: A columns a0 + 8*i
// (i = 0..15); B descriptors desc + j*sub + 2*kk for block j and step kk.
// All 32 operands are formed first (independent adds from three
// registers), then the 16 MMAs issue back to back: an add between two MMAs
// that depends on the previous operand stalls the issue.
#define W4_MMA16_LINE(KIND, A, B, P) \
  "tcgen05.mma.cta_group::1.kind::" KIND " [%0], [%" #A "], %" #B ", %1, " P ";\n\t"
#define W4_MMA16_STR(KIND)                                                              \
  "{\n\t.reg .pred p, t;\n\t"                                                           \
  "setp.ne.b32 p, %2, 0;\n\t"                                                           \
  "setp.eq.b32 t, %2, %2;\n\t" W4_MMA16_LINE(KIND, 3, 19, "p")                          \
      W4_MMA16_LINE(KIND, 4, 20, "t") W4_MMA16_LINE(KIND, 5, 21, "t")                   \
      W4_MMA16_LINE(KIND, 6, 22, "t") W4_MMA16_LINE(KIND, 7, 23, "t")                   \
      W4_MMA16_LINE(KIND, 8, 24, "t") W4_MMA16_LINE(KIND, 9, 25, "t")                   \
      W4_MMA16_LINE(KIND, 10, 26, "t") W4_MMA16_LINE(KIND, 11, 27, "t")                 \
      W4_MMA16_LINE(KIND, 12, 28, "t") W4_MMA16_LINE(KIND, 13, 29, "t")                 \
      W4_MMA16_LINE(KIND, 14, 30, "t") W4_MMA16_LINE(KIND, 15, 31, "t")                 \
      W4_MMA16_LINE(KIND, 16, 32, "t") W4_MMA16_LINE(KIND, 17, 33, "t")                 \
      W4_MMA16_LINE(KIND, 18, 34, "t") "}"
#define W4_MMA16_OPS                                                                     \
  "r"(d_tmem), "r"(idesc), "r"(accumulate), "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]),  \
      "r"(a[4]), "r"(a[5]), "r"(a[6]), "r"(a[7]), "r"(a[8]), "r"(a[9]), "r"(a[10]),     \
      "r"(a[11]), "r"(a[12]), "r"(a[13]), "r"(a[14]), "r"(a[15]), "l"(b[0]), "l"(b[1]),  \
      "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]), "l"(b[7]), "l"(b[8]),       \
      "l"(b[9]), "l"(b[10]), "l"(b[11]), "l"(b[12]), "l"(b[13]), "l"(b[14]), "l"(b[15])
template <bool F8 = false>
__device__ __forceinline__ void mma_ts_stage16(uint32_t d_tmem, uint32_t a0, uint64_t desc,
                                               uint64_t sub, uint32_t idesc,
                                               uint32_t accumulate) {
  uint32_t a[16];
  uint64_t b[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    a[i] = a0 + 8 * i;
    b[i] = desc + static_cast<uint64_t>(i >> 2) * sub + 2 * (i & 3);
  }
  if constexpr (F8)
    asm volatile(W4_MMA16_STR("f8f6f4")::W4_MMA16_OPS : "memory");
  else
    asm volatile(W4_MMA16_STR("f16")::W4_MMA16_OPS : "memory");
}

// Four / eight MMAs from explicit operands (A tensor-memory columns a[i], B
// descriptors b[i]), all formed before the first one issues, into one
// accumulator; the first accumulates only when `accumulate` is non-zero.
// The issuing thread is held inside each MMA for about its execution time,
// so the work it does between MMA groups leaves the tensor pipe idle: the
// more MMAs per group, the less that costs.
#define W4_MMA_N_LINE(KIND, A, B, P) \
  "tcgen05.mma.cta_group::1.kind::" KIND " [%0], [%" #A "], %" #B ", %1, " P ";\n\t"
#define W4_MMA_X4_STR(KIND)                                                         \
  "{\n\t.reg .pred p, t;\n\t"                                                      \
  "setp.ne.b32 p, %2, 0;\n\t"                                                      \
  "setp.eq.b32 t, %2, %2;\n\t" W4_MMA_N_LINE(KIND, 3, 7, "p")                      \
      W4_MMA_N_LINE(KIND, 4, 8, "t") W4_MMA_N_LINE(KIND, 5, 9, "t")                \
      W4_MMA_N_LINE(KIND, 6, 10, "t") "}"
#define W4_MMA_X4_OPS                                                               \
  "r"(d_tmem), "r"(idesc), "r"(accumulate), "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), \
      "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3])
template <bool F8 = false>
__device__ __forceinline__ void mma_ts_4(uint32_t d_tmem, const uint32_t* a, const uint64_t* b,
                                         uint32_t idesc, uint32_t accumulate) {
  if constexpr (F8)
    asm volatile(W4_MMA_X4_STR("f8f6f4")::W4_MMA_X4_OPS : "memory");
  else
    asm volatile(W4_MMA_X4_STR("f16")::W4_MMA_X4_OPS : "memory");
}

#define W4_MMA_X8_STR(KIND)                                                         \
  "{\n\t.reg .pred p, t;\n\t"                                                      \
  "setp.ne.b32 p, %2, 0;\n\t"                                                      \
  "setp.eq.b32 t, %2, %2;\n\t" W4_MMA_N_LINE(KIND, 3, 11, "p")                     \
      W4_MMA_N_LINE(KIND, 4, 12, "t") W4_MMA_N_LINE(KIND, 5, 13, "t")              \
      W4_MMA_N_LINE(KIND, 6, 14, "t") W4_MMA_N_LINE(KIND, 7, 15, "t")              \
      W4_MMA_N_LINE(KIND, 8, 16, "t") W4_MMA_N_LINE(KIND, 9, 17, "t")              \
      W4_MMA_N_LINE(KIND, 10, 18, "t") "}"
#define W4_MMA_X8_OPS                                                               \
  "r"(d_tmem), "r"(idesc), "r"(accumulate), "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), \
      "r"(a[4]), "r"(a[5]), "r"(a[6]), "r"(a[7]), "l"(b[0]), "l"(b[1]), "l"(b[2]),    \
      "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]), "l"(b[7])
template <bool F8 = false>
__device__ __forceinline__ void mma_ts_8(uint32_t d_tmem, const uint32_t (&a)[8],
                                         const uint64_t (&b)[8], uint32_t idesc,
                                         uint32_t accumulate) {
  if constexpr (F8)
    asm volatile(W4_MMA_X8_STR("f8f6f4")::W4_MMA_X8_OPS : "memory");
  else
    asm volatile(W4_MMA_X8_STR("f16")::W4_MMA_X8_OPS : "memory");
}

// 3-D tiled tensor copy global -> shared.
__device__ __forceinline__ void tma_load_3d_a(uint32_t dst, const CUtensorMap* map, int32_t x,
                                              int32_t y, int32_t z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// Arrive once on `bar` when all previously issued tcgen05 async operations
// of this thread have completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns, one lane per thread of the warp.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
      "%29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
      "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
      "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
      : "memory");
}
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&v)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand stored in the
// 128-byte-swizzled canonical layout (rows of 128 bytes, 8-row atoms of 1024
// bytes): start address, leading-dimension offset (unused for this layout,
// encoded as 1), stride-dimension offset 1024 bytes, descriptor version 1,
// swizzle mode 2 (128B).
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1u) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, A and B of the same
// 16-bit type (0 = f16, 1 = bf16), both K-major, M = 128, N = n.  The same
// fields serve kind::f8f6f4, where type code 0 is E4M3.
__host__ __device__ __forceinline__ uint32_t idesc_f16(uint32_t ab_format, uint32_t n) {
  return (1u << 4) | (ab_format << 7) | (ab_format << 10) | ((n >> 3) << 17) |
         ((128u >> 4) << 24);
}

// --------------------------------------------- CTA pairs (cta_group::2)
// A cluster of two CTAs on two SMs shares each tcgen05.mma: rank 0 issues
// it, each CTA holds its half of the A rows (tensor memory) and of the B
// columns (shared memory), and each CTA's tensor memory receives its half of
// D.  Every tcgen05 instruction of such a kernel takes cta_group::2.
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster; orders shared-memory writes
// (barrier initialisation included) before the other CTAs' later accesses.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                   "memory");
}
// Shared::cluster address of the same object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// Arrive on an mbarrier given by its shared::cluster address, which may lie
// in the other CTA of the pair.  What the arrival publishes there is tensor
// memory written with tcgen05.st (completed by tcgen05.wait::st and ordered by
// tcgen05.fence::before_thread_sync before the arrival) and shared memory
// filled by TMA (complete once the arriving thread observed its barrier), both
// read by the other CTA's MMAs after tcgen05.fence::after_thread_sync; the
// default (CTA-scope) release suffices for that, and the cluster-scope form
// made the pair kernel 18-26% slower.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t caddr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(caddr) : "memory");
}
// Tensor memory of a CTA pair: one warp of each of the two CTAs issues these.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(slot)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// Arrive once on the barrier at the same shared-memory offset in both CTAs of
// the pair when every MMA this thread issued before has completed.
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], %1;" ::"r"(smem_addr(bar)),
      "h"(static_cast<uint16_t>(3))
      : "memory");
}
// Four / eight pair MMAs (M = 256 across the two CTAs), operands as mma_ts_4
// / mma_ts_8.
#define W4_MMA2_LINE(KIND, A, B, P) \
  "tcgen05.mma.cta_group::2.kind::" KIND " [%0], [%" #A "], %" #B ", %1, " P ";\n\t"
#define W4_MMA2_X4_STR(KIND)                                                        \
  "{\n\t.reg .pred p, t;\n\t"                                                      \
  "setp.ne.b32 p, %2, 0;\n\t"                                                      \
  "setp.eq.b32 t, %2, %2;\n\t" W4_MMA2_LINE(KIND, 3, 7, "p")                       \
      W4_MMA2_LINE(KIND, 4, 8, "t") W4_MMA2_LINE(KIND, 5, 9, "t")                  \
      W4_MMA2_LINE(KIND, 6, 10, "t") "}"
template <bool F8 = false>
__device__ __forceinline__ void mma_pair_4(uint32_t d_tmem, const uint32_t* a, const uint64_t* b,
                                           uint32_t idesc, uint32_t accumulate) {
  if constexpr (F8)
    asm volatile(W4_MMA2_X4_STR("f8f6f4")::W4_MMA_X4_OPS : "memory");
  else
    asm volatile(W4_MMA2_X4_STR("f16")::W4_MMA_X4_OPS : "memory");
}
#define W4_MMA2_X8_STR(KIND)                                                        \
  "{\n\t.reg .pred p, t;\n\t"                                                      \
  "setp.ne.b32 p, %2, 0;\n\t"                                                      \
  "setp.eq.b32 t, %2, %2;\n\t" W4_MMA2_LINE(KIND, 3, 11, "p")                      \
      W4_MMA2_LINE(KIND, 4, 12, "t") W4_MMA2_LINE(KIND, 5, 13, "t")                \
      W4_MMA2_LINE(KIND, 6, 14, "t") W4_MMA2_LINE(KIND, 7, 15, "t")                \
      W4_MMA2_LINE(KIND, 8, 16, "t") W4_MMA2_LINE(KIND, 9, 17, "t")                \
      W4_MMA2_LINE(KIND, 10, 18, "t") "}"
template <bool F8 = false>
__device__ __forceinline__ void mma_pair_8(uint32_t d_tmem, const uint32_t (&a)[8],
                                           const uint64_t (&b)[8], uint32_t idesc,
                                           uint32_t accumulate) {
  if constexpr (F8)
    asm volatile(W4_MMA2_X8_STR("f8f6f4")::W4_MMA_X8_OPS : "memory");
  else
    asm volatile(W4_MMA2_X8_STR("f16")::W4_MMA_X8_OPS : "memory");
}
// Instruction descriptor with an explicit M (128, or 256 for a CTA pair).
__host__ __device__ __forceinline__ uint32_t idesc_f16_m(uint32_t ab_format, uint32_t n,
                                                        uint32_t m) {
  return (1u << 4) | (ab_format << 7) | (ab_format << 10) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace w4
