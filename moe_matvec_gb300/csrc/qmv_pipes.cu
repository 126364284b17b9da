// Diagnostics of the arithmetic pipes the matvecs rely on:
//   qmv_tc_probe: one 128-row tile times an N-row tile of int8 codes over one
//     32-element block, through the 5th-generation tensor cores with the
//     codes held exactly as f16 and an fp32 accumulator (the form a quantized
//     contraction takes on sm_103a, whose tcgen05 MMA has no int8 kind: ptxas
//     rejects .kind::i8 for this target), read back from tensor memory;
//     tests compare it with exact integer sums.
//   qmv_measure_pipes: per-SM issue rates (per clock) of the instructions of
//     the decode path (dp4a, byte permute, fp32 FMA, packed fp32x2 FMA,
//     int-to-float conversion), of the legacy warp-level MMA and of tcgen05
//     MMAs, each measured on every SM with clock64 around a fixed amount of
//     work.  These are the denominators of the path's ALU roofline.
//   qmv_wait_probe: the kernels' bounded mbarrier wait, run with a
//     caller's cycle limit on a barrier that never completes.
// Every wait is bounded; tensor memory is always released before exit.
#include <algorithm>
#include <vector>

#include "launch.h"
#include "tc_core.cuh"

namespace qmv {

// --------------------------------------------------------------------------
// Tensor-core probe
// --------------------------------------------------------------------------

constexpr int PROBE_M = 128;

// A [128][32] and B [N][32] int8 (row-major); Df [128][N] f32: Df = A B^T
// through kind::f16 (two K = 16 steps, the second accumulating).
__global__ void __launch_bounds__(128) tc_probe_kernel(const int8_t* __restrict__ A, const int8_t* __restrict__ B,
                                                       int N, float* __restrict__ Df, unsigned* err) {
  extern __shared__ __align__(1024) uint8_t smem[];
  // f16 tiles: 64 bytes of K per row
  uint8_t* a16 = smem;                    // 128 x 64
  uint8_t* b16 = a16 + PROBE_M * 64;      // N x 64
  __shared__ uint64_t bar;
  __shared__ uint32_t tslot;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {
    tc::tmem_alloc(&tslot, 256);
    tc::tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  // operands into the core-matrix layout, converted by element pairs
  for (int i = threadIdx.x; i < (PROBE_M + N) * 16; i += blockDim.x) {
    const int r = i >> 4, k2 = (i & 15) * 2;  // rows of A then B; element pair k2, k2 + 1
    const int8_t* src = r < PROBE_M ? A + r * 32 : B + (r - PROBE_M) * 32;
    const uint32_t w = (uint32_t)(uint8_t)src[k2] | ((uint32_t)(uint8_t)src[k2 + 1] << 8);
    const int rr = r < PROBE_M ? r : r - PROBE_M;
    uint8_t* t16 = r < PROBE_M ? a16 : b16;
    *reinterpret_cast<uint32_t*>(t16 + tc::kmajor_offset(rr, 2 * k2, 64)) = tc::s8x2_to_f16x2(w);
  }
  tc::fence_smem_to_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tslot;
  if (threadIdx.x == 0) {
    const uint32_t sa16 = smem_u32(a16), sb16 = smem_u32(b16);
    const uint32_t i16 = tc::idesc_f16_f32(PROBE_M, N);
    // K = 16 f16 elements (32 bytes, two core matrices) per MMA
    tc::mma_f16(tmem, tc::smem_desc(sa16, 128, 512), tc::smem_desc(sb16, 128, 512), i16, false);
    tc::mma_f16(tmem, tc::smem_desc(sa16 + 256, 128, 512), tc::smem_desc(sb16 + 256, 128, 512), i16, true);
    tc::commit(&bar);
  }
  const bool ok = mbar_wait(&bar, 0, err);
  tc::fence_after_sync();
  __syncwarp();  // the TMEM loads below are warp-aligned instructions
  if (ok) {
    const int row = warp * 32 + lane;
    const uint32_t lanes = (uint32_t)(warp * 32) << 16;
    for (int c = 0; c < N; c += 8) {
      uint32_t vf[8];
      tc::tmem_ld_x8(tmem + lanes + c, vf);
#pragma unroll
      for (int j = 0; j < 8; j++) Df[row * N + c + j] = __uint_as_float(vf[j]);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

// --------------------------------------------------------------------------
// Pipe rates
// --------------------------------------------------------------------------

constexpr int PIPE_ITERS = 2048;

// Each kernel: one CTA per SM, every thread runs PIPE_ITERS steps of 8
// independent chains; thread 0 records the clock64 span between two CTA
// barriers around the loop.  The chains' results are written out so the
// work is kept.
__global__ void __launch_bounds__(1024) pipe_dp4a(int* out, long long* cyc, int seed) {
  int a0 = threadIdx.x ^ seed, b = seed * 3 + 1, acc[8];
#pragma unroll
  for (int i = 0; i < 8; i++) acc[i] = i;
  __syncthreads();
  const long long t0 = clock64();
  for (int it = 0; it < PIPE_ITERS; it++) {
#pragma unroll
    for (int i = 0; i < 8; i++) acc[i] = __dp4a(a0 + i, b, acc[i]);
    b += 0x01010101;
  }
  __syncthreads();
  const long long t1 = clock64();
  int s = 0;
#pragma unroll
  for (int i = 0; i < 8; i++) s += acc[i];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}

__global__ void __launch_bounds__(1024) pipe_prmt(int* out, long long* cyc, int seed) {
  unsigned a = threadIdx.x ^ seed, b = seed * 7u, acc[8];
#pragma unroll
  for (int i = 0; i < 8; i++) acc[i] = i * 0x1111u;
  __syncthreads();
  const long long t0 = clock64();
  for (int it = 0; it < PIPE_ITERS; it++) {
#pragma unroll
    for (int i = 0; i < 8; i++) acc[i] = __byte_perm(a + i, b, acc[i]);
    b += 1;
  }
  __syncthreads();
  const long long t1 = clock64();
  unsigned s = 0;
#pragma unroll
  for (int i = 0; i < 8; i++) s += acc[i];
  out[blockIdx.x * blockDim.x + threadIdx.x] = (int)s;
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}

__global__ void __launch_bounds__(1024) pipe_ffma(int* out, long long* cyc, int seed) {
  const float a = threadIdx.x * 1e-3f, b = 0.999f + seed * 1e-9f;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; i++) acc[i] = (float)i;
  __syncthreads();
  const long long t0 = clock64();
  for (int it = 0; it < PIPE_ITERS; it++) {
#pragma unroll
    for (int i = 0; i < 8; i++) acc[i] = fmaf(acc[i], b, a);
  }
  __syncthreads();
  const long long t1 = clock64();
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 8; i++) s += acc[i];
  out[blockIdx.x * blockDim.x + threadIdx.x] = (int)s;
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}

__global__ void __launch_bounds__(1024) pipe_ffma2(int* out, long long* cyc, int seed) {
  const float2 a = make_float2(threadIdx.x * 1e-3f, threadIdx.x * 2e-3f);
  const float2 b = make_float2(0.999f + seed * 1e-9f, 0.998f);
  float2 acc[8];
#pragma unroll
  for (int i = 0; i < 8; i++) acc[i] = make_float2((float)i, (float)(i + 1));
  __syncthreads();
  const long long t0 = clock64();
  for (int it = 0; it < PIPE_ITERS; it++) {
#pragma unroll
    for (int i = 0; i < 8; i++) acc[i] = __ffma2_rn(acc[i], b, a);
  }
  __syncthreads();
  const long long t1 = clock64();
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 8; i++) s += acc[i].x + acc[i].y;
  out[blockIdx.x * blockDim.x + threadIdx.x] = (int)s;
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}

__global__ void __launch_bounds__(1024) pipe_i2f(int* out, long long* cyc, int seed) {
  const int a = threadIdx.x ^ seed;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; i++) acc[i] = 0.f;
  __syncthreads();
  const long long t0 = clock64();
  for (int it = 0; it < PIPE_ITERS; it++) {
#pragma unroll
    for (int i = 0; i < 8; i++) acc[i] += __int2float_rn(a + i + it);
  }
  __syncthreads();
  const long long t1 = clock64();
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 8; i++) s += acc[i];
  out[blockIdx.x * blockDim.x + threadIdx.x] = (int)s;
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}

// warp-level m16n8k32 s8 MMA: 4096 multiply-adds per warp instruction
__global__ void __launch_bounds__(1024) pipe_mma_sync_s8(int* out, long long* cyc, int seed) {
  const unsigned a0 = threadIdx.x ^ seed, a1 = a0 + 1, a2 = a0 + 2, a3 = a0 + 3, b0 = seed, b1 = seed + 5;
  int c[4][4] = {};
  __syncthreads();
  const long long t0 = clock64();
  for (int it = 0; it < PIPE_ITERS / 4; it++) {
#pragma unroll
    for (int j = 0; j < 4; j++)
      asm volatile(
          "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
          : "+r"(c[j][0]), "+r"(c[j][1]), "+r"(c[j][2]), "+r"(c[j][3])
          : "r"(a0 + j), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
  __syncthreads();
  const long long t1 = clock64();
  int s = 0;
#pragma unroll
  for (int j = 0; j < 4; j++)
#pragma unroll
    for (int i = 0; i < 4; i++) s += c[j][i];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}

// warp-level m16n8k16 f16 MMA, f32 accumulator: 2048 multiply-adds per warp instruction
__global__ void __launch_bounds__(1024) pipe_mma_sync_f16(int* out, long long* cyc, int seed) {
  const unsigned a0 = 0x3c003c00u ^ (threadIdx.x & 1), b0 = 0x3c003c00u + seed;
  float c[4][4] = {};
  __syncthreads();
  const long long t0 = clock64();
  for (int it = 0; it < PIPE_ITERS / 4; it++) {
#pragma unroll
    for (int j = 0; j < 4; j++)
      asm volatile(
          "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
          : "+f"(c[j][0]), "+f"(c[j][1]), "+f"(c[j][2]), "+f"(c[j][3])
          : "r"(a0 + j), "r"(a0), "r"(a0), "r"(a0), "r"(b0), "r"(b0));
  }
  __syncthreads();
  const long long t1 = clock64();
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < 4; j++)
#pragma unroll
    for (int i = 0; i < 4; i++) s += c[j][i];
  out[blockIdx.x * blockDim.x + threadIdx.x] = (int)s;
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}

// tcgen05 MMA rate: thread 0 issues `iters` f16 MMAs of 128 x N x 16
// accumulating into one TMEM tile, then waits for their completion; the span
// runs from the first issue to the completion.  Operands: zeroed 16 KB areas
// (every address the descriptors reach lies inside them).
__global__ void __launch_bounds__(128) pipe_tc(int N, int iters, long long* cyc, unsigned* err) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tslot;
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < 32768 / 16; i += blockDim.x) reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  if (warp == 0) {
    tc::tmem_alloc(&tslot, 256);
    tc::tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  tc::fence_smem_to_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tslot;
  if (threadIdx.x == 0) {
    const uint64_t a = tc::smem_desc(smem_u32(smem), 128, 256), b = tc::smem_desc(smem_u32(smem + 16384), 128, 256);
    const uint32_t id = tc::idesc_f16_f32(128, N);
    const long long t0 = clock64();
    for (int i = 0; i < iters; i++) tc::mma_f16(tmem, a, b, id, i > 0);
    tc::commit(&bar);
    mbar_wait(&bar, 0, err);
    cyc[blockIdx.x] = clock64() - t0;
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

typedef void (*pipe_fn)(int*, long long*, int);

// Median over the SMs of (operations per thread x threads / cycles).
static double median_rate(const std::vector<long long>& cyc, double ops) {
  std::vector<long long> c = cyc;
  std::sort(c.begin(), c.end());
  const double med = (double)c[c.size() / 2];
  return med > 0 ? ops / med : 0.0;
}

// One warp waits on an mbarrier that nothing ever completes, with the
// library's bounded wait loop and the caller's limit (qmv_wait_probe).
__global__ void wait_probe_kernel(long long limit, unsigned* err, unsigned long long* cycles) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const long long t0 = clock64();
  const bool ok = mbar_wait_until(&bar, 0, err, limit);  // phase 0 never completes
  const long long t1 = clock64();
  if (threadIdx.x == 0 && cycles) *cycles = ok ? 0ull : (unsigned long long)(t1 - t0);
}

}  // namespace qmv

using namespace qmv;

extern "C" int qmv_wait_probe(long long limit_cycles, unsigned long long* cycles, cudaStream_t stream) {
  if (limit_cycles < 1 || limit_cycles > WAIT_CYCLES) return QMV_ERR_SHAPE;
  if (cycles && (reinterpret_cast<uintptr_t>(cycles) & 7u)) return QMV_ERR_ALIGN;
  unsigned* err = device_error_word();
  if (!err) return QMV_ERR_CUDA;
  wait_probe_kernel<<<1, 32, 0, stream>>>(limit_cycles, err, cycles);
  return cudaGetLastError() == cudaSuccess ? QMV_OK : QMV_ERR_CUDA;
}

extern "C" int qmv_tc_probe(const int8_t* A, const int8_t* B, int N, float* Df, cudaStream_t stream) {
  if (!A || !B || !Df) return QMV_ERR_NULL;
  if (N < 16 || N > 256 || N % 16) return QMV_ERR_SHAPE;
  if (device_sm_count() < 1) return QMV_ERR_CUDA;
  const size_t smem = (size_t)PROBE_M * 64 + 256 * 64;
  if (cudaFuncSetAttribute(tc_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return QMV_ERR_CUDA;
  tc_probe_kernel<<<1, 128, smem, stream>>>(A, B, N, Df, device_error_word());
  return cudaGetLastError() == cudaSuccess ? QMV_OK : QMV_ERR_CUDA;
}

extern "C" size_t qmv_measure_pipes_scratch_bytes(void) {
  const size_t sms = (size_t)device_sm_count();
  return sms * 1024 * sizeof(int) + sms * sizeof(long long);
}

extern "C" int qmv_measure_pipes(double* rates, int count, void* scratch, size_t scratch_bytes,
                                 cudaStream_t stream) {
  if (!rates || !scratch) return QMV_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(scratch) & 15u) != 0) return QMV_ERR_ALIGN;
  const int sms = device_sm_count();
  if (scratch_bytes < qmv_measure_pipes_scratch_bytes()) return QMV_ERR_WORKSPACE;
  int* d_out = static_cast<int*>(scratch);
  long long* d_cyc = reinterpret_cast<long long*>(d_out + (size_t)sms * 1024);
  std::vector<long long> cyc(sms);
  std::vector<double> r;
  bool ok = true;
  auto collect = [&](double ops) {
    ok = ok && cudaStreamSynchronize(stream) == cudaSuccess &&
         cudaMemcpy(cyc.data(), d_cyc, sizeof(long long) * sms, cudaMemcpyDeviceToHost) == cudaSuccess;
    r.push_back(ok ? median_rate(cyc, ops) : 0.0);
  };
  // thread instructions per clock per SM (1024 threads x 8 chains x PIPE_ITERS)
  const double thread_ops = 1024.0 * 8 * PIPE_ITERS;
  const pipe_fn alu[5] = {pipe_dp4a, pipe_prmt, pipe_ffma, pipe_ffma2, pipe_i2f};
  for (int i = 0; i < 5; i++) {
    alu[i]<<<sms, 1024, 0, stream>>>(d_out, d_cyc, 1);  // warm
    alu[i]<<<sms, 1024, 0, stream>>>(d_out, d_cyc, 3);
    collect(thread_ops);
  }
  // legacy warp MMAs: multiply-adds per clock per SM (32 warps x PIPE_ITERS instructions)
  pipe_mma_sync_s8<<<sms, 1024, 0, stream>>>(d_out, d_cyc, 1);
  pipe_mma_sync_s8<<<sms, 1024, 0, stream>>>(d_out, d_cyc, 3);
  collect(32.0 * PIPE_ITERS * 4096);
  pipe_mma_sync_f16<<<sms, 1024, 0, stream>>>(d_out, d_cyc, 1);
  pipe_mma_sync_f16<<<sms, 1024, 0, stream>>>(d_out, d_cyc, 3);
  collect(32.0 * PIPE_ITERS * 2048);
  // tcgen05: multiply-adds per clock per SM; one CTA per SM (its 64 KB of
  // shared memory, of which 32 KB are used, keeps a second one off the SM)
  const int tc_iters = 2048;
  const size_t tc_smem = 64 * 1024;
  ok = ok && cudaFuncSetAttribute(pipe_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc_smem) == cudaSuccess;
  const int tc_n[3] = {256, 64, 32};
  for (int j = 0; j < 3 && ok; j++) {
    const int N = tc_n[j];
    pipe_tc<<<sms, 128, tc_smem, stream>>>(N, tc_iters, d_cyc, device_error_word());
    pipe_tc<<<sms, 128, tc_smem, stream>>>(N, tc_iters, d_cyc, device_error_word());
    collect((double)tc_iters * 128 * N * 16);
  }
  if (!ok) return QMV_ERR_CUDA;
  const int n = count < (int)r.size() ? count : (int)r.size();
  for (int i = 0; i < n; i++) rates[i] = r[i];
  return n;
}
