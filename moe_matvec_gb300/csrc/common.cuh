// Device-side building blocks shared by the qmv kernels: format constants,
// mbarrier / TMA wrappers (inline PTX for sm_103a), bounded waits, the device
// error word and the per-32 activation quantizer.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/qmv.h"

namespace qmv {

// ---------------------------------------------------------------------------
// Format geometry.  A "chunk" is the K-slice one pipeline stage carries:
// 1024 weights = 32 sub-blocks of 32, one sub-block per lane (F32 rows: 512).
// ---------------------------------------------------------------------------
constexpr int KCHUNK = 1024;
constexpr int BLK = 32;

template <int F>
struct Fmt;
template <>
struct Fmt<QMV_Q8_0> {
  static constexpr int GW = 256, GB = 272;  // weights / bytes per group
};
template <>
struct Fmt<QMV_Q4_K> {
  static constexpr int GW = 256, GB = 144;
};
template <>
struct Fmt<QMV_IQ4_XS> {
  static constexpr int GW = 512, GB = 272;
};
template <>
struct Fmt<QMV_Q5_K> {
  static constexpr int GW = 256, GB = 176;
};
template <>
struct Fmt<QMV_Q6_K> {
  static constexpr int GW = 256, GB = 208;
};
template <>
struct Fmt<QMV_Q8_G64> {
  static constexpr int GW = 512, GB = 528;
};
template <>
struct Fmt<QMV_Q8_G128> {
  static constexpr int GW = 1024, GB = 1040;
};
// unquantized rows: a "group" is one 32-weight block of plain values
template <>
struct Fmt<QMV_F16> {
  static constexpr int GW = 32, GB = 64;
};
template <>
struct Fmt<QMV_F32> {
  static constexpr int GW = 32, GB = 128;
};
__host__ __device__ constexpr bool is_float(int F) { return F == QMV_F16 || F == QMV_F32; }
// Weights per chunk: 1024, except F32 rows, whose chunk of 512 weights keeps
// a row chunk at 2048 bytes (the size of an F16 one).
__host__ __device__ constexpr int kchunk_of(int F) { return F == QMV_F32 ? 512 : KCHUNK; }
// int8 codes used as they are (one fp16 scale per 32, 64 or 128 weights)
__host__ __device__ constexpr bool is_q8(int F) { return F == QMV_Q8_0 || F == QMV_Q8_G64 || F == QMV_Q8_G128; }
// Formats with a per-sub-block minimum (w = d sc q - dmin m): their min term
// needs each activation block's code sum.
__host__ __device__ constexpr bool has_min(int F) { return F == QMV_Q4_K || F == QMV_Q5_K; }
template <int F>
constexpr int chunk_bytes() {
  return (kchunk_of(F) / Fmt<F>::GW) * Fmt<F>::GB;
}

// ---------------------------------------------------------------------------
// Device error word (QMV_DEVERR_* bits).
// ---------------------------------------------------------------------------
// The word lives in the dispatcher's unit; kernels receive its address.
__device__ __forceinline__ void set_error(unsigned* err, unsigned bits) {
  if (err) atomicOr(err, bits);
}

// ---------------------------------------------------------------------------
// Software range checks (builds with QMV_DEBUG defined).
// ---------------------------------------------------------------------------
// A checked access tests its index against a bound that does not come from
// the kernel's own tiling: a global buffer against the extent the host
// derived from the call's arguments, a dynamic shared-memory address against
// the CTA's allocation (%dynamic_smem_size), a static shared array against
// its declared length.  A failed check sets QMV_DEVERR_RANGE and the access
// is skipped; nothing traps.
// Every check is written QMV_CHECK(in_range(...)) (or smem_in_range,
// in_array), and the extents and the parameters that carry them are written
// QMV_DEBUG_ONLY(...).  In release builds QMV_CHECK is the literal true and
// QMV_DEBUG_ONLY drops its argument, so not even the checks' arguments reach
// the compiler: the release kernels' parameter blocks and code are those of
// a library without checks.
#ifdef QMV_DEBUG
#define QMV_DEBUG_ONLY(...) __VA_ARGS__
#define QMV_CHECK(...) (__VA_ARGS__)
#else
#define QMV_DEBUG_ONLY(...)
#define QMV_CHECK(...) true
#endif

// elements [i, i + n) of a buffer of len elements
__device__ __forceinline__ bool in_range(long long i, long long n, long long len, unsigned* err) {
  if (i >= 0 && n >= 0 && i <= len - n) return true;
  set_error(err, QMV_DEVERR_RANGE);
  return false;
}

// index i of a static (shared-memory) array of N elements
template <class T, int N>
__device__ __forceinline__ bool in_array(const T (&)[N], long long i, unsigned* err) {
  return in_range(i, 1, N, err);
}

__device__ __forceinline__ uint32_t dynamic_smem_size() {
  uint32_t r;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(r));
  return r;
}

// shared-window address of the CTA's dynamic shared memory
__device__ __forceinline__ uint32_t dynamic_smem_base() {
  extern __shared__ __align__(16) uint8_t qmv_dynamic_smem[];
  return static_cast<uint32_t>(__cvta_generic_to_shared(qmv_dynamic_smem));
}

// bytes [addr, addr + n) (a shared-window address) inside the CTA's dynamic
// shared memory
__device__ __forceinline__ bool smem_in_range(uint32_t addr, uint32_t n, unsigned* err) {
  return in_range((long long)addr - (long long)dynamic_smem_base(), n, dynamic_smem_size(), err);
}
__device__ __forceinline__ bool smem_in_range(const void* p, uint32_t n, unsigned* err) {
  return smem_in_range(static_cast<uint32_t>(__cvta_generic_to_shared(p)), n, err);
}

// ---------------------------------------------------------------------------
// Shared-memory address helpers and mbarriers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Completes `bytes` of the current phase's expected transaction count without
// a copy: a copy skipped by a failed range check still lets the phase end.
__device__ __forceinline__ void mbar_complete_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait that may suspend the thread (up to `ns` nanoseconds) until the
// phase completes, instead of returning at once: a waiting warp then takes
// no issue slots from the warps that compute.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint64_t* bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// Bounded wait: gives up after `limit` SM cycles, sets the timeout bit and
// returns false.  No wait in this library is unbounded: the kernels use
// mbar_wait below (about a second, a compile-time constant, so that their hot
// loops carry no other code); the wait probe (qmv_wait_probe) runs the same
// loop with a caller's limit on a barrier that never completes.
constexpr long long WAIT_CYCLES = 1ll << 31;
constexpr uint32_t WAIT_SUSPEND_NS = 1u << 20;
__device__ __forceinline__ bool mbar_wait_until(uint64_t* bar, uint32_t parity, unsigned* err, long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  long long t0 = clock64();
  while (!mbar_try_wait_suspend(bar, parity, WAIT_SUSPEND_NS)) {
    if (clock64() - t0 > limit) {
      set_error(err, QMV_DEVERR_TIMEOUT);
      return false;
    }
  }
  return true;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned* err) {
  return mbar_wait_until(bar, parity, err, WAIT_CYCLES);
}

// L2 policy for streamed weights: evict first, so activations and outputs
// stay resident.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 2-D tiled TMA load (global -> shared, completion on an mbarrier).  x is the
// innermost coordinate in elements of the map (8-byte elements here), which
// keeps every x * 8 a multiple of 16 bytes because group sizes are.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

// 2-D tiled TMA prefetch of a box into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

// Bulk (non-tensor) copy global -> shared of `bytes` (a multiple of 16;
// both addresses 16-byte aligned), completion on an mbarrier.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// The same with an L2 cache policy (createpolicy) for the source.
__device__ __forceinline__ void bulk_copy_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                                   uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Named barrier over `nthreads` threads (the consumer warps).
__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Register re-split between warpgroups (all four warps of a warpgroup run
// the same instruction): dec gives registers back to the CTA's pool, inc
// takes them (waiting until the pool holds them; the launcher checks that
// the CTA was launched with enough registers for every warpgroup's share).
template <int N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// Programmatic dependent launch: wait for the preceding grid's results
// (no-op when launched without the attribute).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Branch-free correctly rounded a / 127 and 1 / d for the activation rule.
// The IEEE division / reciprocal of the toolkit carry a branch to a slow path
// for special operands, which keeps independent quantizations from being
// interleaved.  Both functions below use the FMA-based correction of a
// quotient or reciprocal (Newton-Raphson with an exact FMA residual, as in
// P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990) and are equal to the
// IEEE round-to-nearest results on their stated ranges; tests compare them
// exhaustively against __fdiv_rn / __frcp_rn (qmv_check_rounding).
// ---------------------------------------------------------------------------
// RN(a / 127) for 0 <= a <= FLT_MAX with a / 127 >= 2^-126 or a == 0.
__device__ __forceinline__ float div127_rn(float a) {
  const float c = 0.007874015718698502f;  // RN(1 / 127)
  const float q0 = __fmul_rn(a, c);
  const float r = __fmaf_rn(-q0, 127.0f, a);  // exact residual
  return __fmaf_rn(r, c, q0);
}
// RN(1 / d) for 2^-126 <= d <= 2^126.
__device__ __forceinline__ float rcp_rn(float d) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(d));
  float e = __fmaf_rn(-d, y, 1.0f);
  y = __fmaf_rn(y, e, y);
  e = __fmaf_rn(-d, y, 1.0f);
  return __fmaf_rn(y, e, y);
}

// ---------------------------------------------------------------------------
// Loads that bypass L1 for data read once.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ldg_stream(const float* p) {
  float v;
  asm volatile("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

}  // namespace qmv
