// Building blocks of the 5th-generation tensor cores (tcgen05) for sm_103a,
// as inline PTX: tensor-memory (TMEM) allocation, shared-memory matrix and
// instruction descriptors, MMA issue by one thread, completion tracked by an
// mbarrier, and loads of accumulators from TMEM into registers.
//
// Operand layout used throughout ("K-major, no swizzle"): an operand tile of
// R rows x KB bytes of K is a grid of core matrices, each 8 rows x 16 bytes
// stored as 128 contiguous bytes (row i of the core matrix at byte 16 i).
// Core matrix (g, c) -- rows 8g .. 8g+7, K bytes 16c .. 16c+15 -- sits at
// byte (g * KB / 16 + c) * 128 of the tile, so core matrices adjacent along
// K are LBO = 128 bytes apart and 8-row groups SBO = 8 KB bytes apart.
#pragma once
#include "common.cuh"

namespace qmv {
namespace tc {

// Byte offset of element byte kb (0 .. KB-1) of row r in a K-major tile
// with KB bytes of K per row.
__host__ __device__ constexpr uint32_t kmajor_offset(int r, int kb, int KB) {
  return (uint32_t)(((r >> 3) * (KB >> 4) + (kb >> 4)) * 128 + (r & 7) * 16 + (kb & 15));
}

// Allocate ncols columns (a power of two, 32 .. 512) of tensor memory for
// this CTA; one whole warp executes it and the TMEM address (lane 0, first
// column) lands in *slot in shared memory.  Every allocation is released
// with tmem_dealloc by the same warp before the CTA exits.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Ordering of tcgen05 operations across a thread barrier.
__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Generic-proxy writes to shared memory made visible to the tensor core's
// (async-proxy) reads; each writing thread executes it before the barrier
// that precedes the MMA.
__device__ __forceinline__ void fence_smem_to_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major tile without swizzle starting
// at shared address saddr (16-byte aligned): start address, leading-dimension
// byte offset (between core matrices along K), stride-dimension byte offset
// (between 8-row groups), the descriptor version bit of this architecture
// (bit 46), base offset 0, layout "no swizzle" (bits 61-63 = 0).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  return d;
}

// Instruction descriptor (both operands K-major, no negation, dense):
// bits 4-5 accumulator type (1: f32), 7-9 / 10-12 operand types (0: f16),
// 17-22 N / 8, 24-28 M / 16.  (sm_103a's tcgen05 MMA has no int8 kind:
// int8 codes enter as f16, which holds every integer up to 2048 exactly.)
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {  // f16 x f16 -> f32
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D (TMEM) = A x B^T (+ D if acc), issued by one thread; asynchronous.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"((uint32_t)acc)
      : "memory");
}
// The mbarrier receives one arrival when every MMA this thread issued so
// far has completed (and its TMEM results are visible).
__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Loads of 32 lanes x 32-bit columns: lane i of the warp receives TMEM lane
// (lane field of taddr) + i, columns (column field) .. + 7 (x8), + 15 (x16)
// or + 31 (x32).  A warp may only address the 32-lane quarter of its warp
// index modulo 4.  Each load waits for its own completion inside the same
// asm statement, so the compiler never reads the registers early.
__device__ __forceinline__ void tmem_ld_x8(uint32_t taddr, uint32_t (&v)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n"
      "tcgen05.wait::ld.sync.aligned;"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; i++) v[i] = __uint_as_float(r[i]);
}

// Per-thread asynchronous copies global -> shared (16, 8 or 4 bytes, both
// addresses aligned to the size), grouped with commit and waited for by the
// issuing thread: after wait<N>, all but the N most recent groups have landed.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Two loads of 32 columns (32 lanes x 32 bits each) waited for together.
__device__ __forceinline__ void tmem_ld2_x32(uint32_t ta, uint32_t tb, float (&a)[32], float (&b)[32]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%64];\n"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, "
      "%45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%65];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(ta), "r"(tb));
#pragma unroll
  for (int i = 0; i < 32; i++) {
    a[i] = __uint_as_float(r[i]);
    b[i] = __uint_as_float(r[32 + i]);
  }
}

// Two int8 codes (bytes 0 and 1 of w) as an f16 pair, exactly: for
// |c| <= 128 the binary16 value 1024 + 128 + c has the integer c + 1152
// in its mantissa (the exponent of 1024 spans 1024 .. 2047), so building
// 0x6400 | (c + 128) and subtracting 1152 gives c exactly.
__device__ __forceinline__ uint32_t s8x2_to_f16x2(uint32_t w) {
  const uint32_t b = (w ^ 0x8080u) & 0xFFFFu;                      // c + 128, bytes 0 and 1
  const uint32_t h = __byte_perm(b, 0x64646464u, 0x5140) ;         // 0x64 | byte, per half
  __half2 v = *reinterpret_cast<const __half2*>(&h);
  v = __hsub2(v, __half2half2(__ushort_as_half(0x6480u)));        // - 1152
  return *reinterpret_cast<const uint32_t*>(&v);
}

}  // namespace tc
}  // namespace qmv
