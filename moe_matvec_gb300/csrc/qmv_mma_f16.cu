// Tensor-core matvec for F16 weight rows and 5 to 16 tokens, and its launcher.
//
// The operation is the F16 row path's ("Castagna Veloce", section "Kernels
// for the MI50": the small-batch matvecs also serve F16 rows): Xhat = x (fp32,
// unquantized), y = sum_k w_k x_k in fp32, within 1e-5 * sum_k |w_k x_k|.  The
// CUDA-core path issues one fp32 FMA per weight per token, which bounds it
// from 8 tokens on; here the warps' tensor-core MMA (mma.sync m16n8k16, f16
// operands, fp32 accumulation) forms the products of 16 rows x 8 token slots:
//   - A operand: the weights, f16 as stored (no decode: ldmatrix straight from
//     the stage);
//   - B operand: the activations of 8 token slots, each scaled by a power of
//     two s_t (exact) so that its largest magnitude in the split range lies in
//     [2^14, 2^15), and split into two f16 parts, x s = hi + lo + r with
//     |r| <= 2^-22 |x s| (hi = f16(x s), lo = f16(x s - hi); the difference is
//     exact in fp32).  Two MMAs per step, one on each part; every product of
//     two f16 values is exact in the fp32 accumulator;
//   - the accumulators run over the whole split range and are multiplied by
//     1 / s_t (exact) at the store.
// Structure as the Q4_K tensor-core kernel (qmv_mma.cuh): persistent CTAs over
// tiles of 64 rows, one producer lane streaming 256-weight chunks by 2-D TMA
// into a ring of stages whose rows are 528 bytes apart (the box takes 16 bytes
// more of every row: an odd number of 16-byte units, so the 8 rows of an
// ldmatrix phase fall in 8 bank groups), eight consumer warps taking two
// 16-weight steps of each chunk for all 64 rows, partial sums added across the
// warps in a fixed order through shared memory.  The activations of a split
// range are staged once per CTA (the caller's split keeps the range small).
#include <atomic>

#include "launch.h"
#include "qmv_mma.cuh"

namespace qmv {

constexpr int MF_CW = 8;                        // consumer warps
constexpr int MF_THREADS = (MF_CW + 1) * 32;    // + producer warp
constexpr int MF_KC = 256;                      // weights per stage chunk
constexpr int MF_PITCH = MF_KC * 2 + 16;        // 528 = 33 x 16 bytes per staged row
constexpr int MF_STAGE = MK_ROWS * MF_PITCH;    // 33,792 bytes
static_assert(MF_CW * 32 == MF_KC, "each warp takes two 16-weight steps of a chunk");
static_assert(MMA_F16_BOX_BYTES == MF_PITCH, "tensor maps match the stage layout");

// Shared memory: [stages][64 rows][528] weights; xh, xl [NT][xpitch] f16 (the
// two parts of the scaled activations of the split range, 16 bytes of padding
// per token); inv [16] f32 (1 / s_t); red [8 warps][NT][72] f32; mbarriers.
struct MfLayout {
  size_t xh, xl, inv, red, bars, total;
  int xpitch;
  __host__ __device__ MfLayout(int nt, int stages, int kmax) {
    xpitch = kmax * 2 + 16;
    xh = (size_t)stages * MF_STAGE;
    xl = xh + (size_t)nt * xpitch;
    inv = xl + (size_t)nt * xpitch;
    red = inv + 16 * sizeof(float);
    bars = red + (size_t)MF_CW * nt * MK_RED_LD * 4;
    total = bars + (2 * MAX_STAGES) * 8;
  }
};

// The shared-memory ranges of a warp's step at weight kc of a chunk: the
// weight stage and the NT token rows of both activation parts over the
// step's 32 weights.
template <int NT>
__device__ __forceinline__ bool mf_step_in_range(uint32_t sbase, uint32_t xh_base, uint32_t xl_base, int xpitch,
                                                 int kc, unsigned* err) {
  const uint32_t n = (uint32_t)((NT - 1) * xpitch + 64);
  return smem_in_range(sbase, MF_STAGE, err) && smem_in_range(xh_base + 2 * kc, n, err) &&
         smem_in_range(xl_base + 2 * kc, n, err);
}

template <int NT>
__global__ void __launch_bounds__(MF_THREADS, 1)
    qmv_mma_f16_kernel(const __grid_constant__ CUtensorMap map_tile, const __grid_constant__ CUtensorMap map_unit,
                       const DenseParams p) {
  static_assert(NT == 8 || NT == 16, "8 or 16 token slots");
  constexpr int TG = NT / 8;     // token tiles
  constexpr int RP = MK_UNITS / 2;  // row pairs of a tile
  extern __shared__ __align__(128) uint8_t smem[];
  const MfLayout L(NT, p.stages, p.nbmax * BLK);
  uint8_t* stages = smem;
  uint8_t* xh = smem + L.xh;
  uint8_t* xl = smem + L.xl;
  float* inv = reinterpret_cast<float*>(smem + L.inv);
  float* red = reinterpret_cast<float*>(smem + L.red);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + MAX_STAGES;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  init_pipeline(full, empty, p.stages, MF_CW);
  pdl_launch_dependents();

  if (warp == MF_CW) {
    // ---------------- producer: one elected lane, 2-D TMA ----------------
    if (lane == 0) {
      prefetch_tensormap(&map_tile);
      prefetch_tensormap(&map_unit);
      const uint64_t pol = policy_evict_first();
      TileWalk<MK_UNITS> walk(p);
      int s, u, nu;
      Ring ring;
      bool alive = true;
      while (alive && walk.next(s, u, nu)) {
        int g0, g1;
        split_range(p, s, g0, g1);
        const int klen = (g1 - g0) * BLK, nck = (klen + MF_KC - 1) / MF_KC;
        for (int c = 0; c < nck; c++, ring.advance(p.stages)) {
          if (!producer_acquire(empty, ring, p.stages, p.err)) {
            alive = false;
            break;
          }
          const int st = ring.st;
          uint8_t* dst = stages + st * MF_STAGE;
          const int x = (g0 * BLK + c * MF_KC) / 4;  // 8-byte elements (4 weights); x * 8 = 2 * first weight
          if (!QMV_CHECK(smem_in_range(dst, nu * UNIT_ROWS * MF_PITCH, p.err))) {
            mbar_arrive(&full[st]);  // skipped: the stage completes without data
          } else if (nu == MK_UNITS) {
            mbar_arrive_expect_tx(&full[st], MF_STAGE);
            tma_load_2d(dst, &map_tile, &full[st], x, u * UNIT_ROWS, pol);
          } else {
            mbar_arrive_expect_tx(&full[st], nu * UNIT_ROWS * MF_PITCH);
            for (int i = 0; i < nu; i++)
              tma_load_2d(dst + i * UNIT_ROWS * MF_PITCH, &map_unit, &full[st], x, (u + i) * UNIT_ROWS, pol);
          }
        }
      }
      producer_drain(full, ring.n, p.stages, p.err);
    }
    return;
  }

  // ---------------- consumers ----------------
  const int cw = warp, g = lane >> 2, t4 = lane & 3;
  const int t0 = p.t0 + blockIdx.y * NT, ntk = p.nt;
  const int xpitch = L.xpitch;
  const uint32_t stage_base = smem_u32(stages), xh_base = smem_u32(xh), xl_base = smem_u32(xl);
  // ldmatrix source rows of this lane: weights (A: rows 0-7 / 8-15 of a row
  // pair, k 0-7 / 8-15 of a step) and activations (B: token row lane % 8 of a
  // tile; k 0-7 / 8-15; hi part for lanes 0-15, lo for 16-31)
  const int m4 = lane >> 3;
  const uint32_t a_off = (uint32_t)(((lane & 7) + 8 * (m4 & 1)) * MF_PITCH + 16 * (m4 >> 1));
  const uint32_t b_off = (uint32_t)((lane & 7) * xpitch + 16 * (m4 & 1)) + ((m4 >> 1) ? xl_base : xh_base);
  bool alive = true;
  TileWalk<MK_UNITS> walk(p);
  int s, u, nu;
  Ring ring;
  int staged_split = -1;

  // the activations may come from the preceding kernel: wait for it only
  // now, so that the set-up above (parameters only) runs while it finishes
  pdl_wait();
  while (walk.next(s, u, nu)) {
    int g0, g1;
    split_range(p, s, g0, g1);
    const int klen = (g1 - g0) * BLK, nck = (klen + MF_KC - 1) / MF_KC;
    if (s != staged_split) {
      if (staged_split >= 0) named_sync(1, MF_CW * 32);  // nobody still reads the previous range
      // the split range's activations: per token the power of two s_t that
      // puts its largest magnitude in [2^14, 2^15) (2^127 at most, for a zero
      // or tiny range), then the two f16 parts of x s_t
      for (int tt = cw; tt < NT; tt += MF_CW) {
        const bool real = tt < ntk;
        const float* xr = p.x + (long long)(t0 + (real ? tt : 0)) * p.K + (long long)g0 * BLK;
        float m = 0.0f;
        if (real)
          for (int k = 4 * lane; k < klen; k += 128) {
            if (!QMV_CHECK(in_range(xr - p.x + k, 4, p.x_len, p.err))) continue;
            const float4 v = __ldg(reinterpret_cast<const float4*>(xr + k));
            m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
          }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
        int e = (int)((__float_as_uint(m) >> 23) & 0xFF) - 127;  // floor(log2 m) for a normal m
        e = max(e, -113);
        const float sc = __uint_as_float((uint32_t)(127 + 14 - e) << 23);  // 2^(14 - e)
        uint8_t* hrow = xh + (size_t)tt * xpitch;
        uint8_t* lrow = xl + (size_t)tt * xpitch;
        for (int k = 2 * lane; k < klen; k += 64) {
          float2 v = make_float2(0.0f, 0.0f);
          if (real && QMV_CHECK(in_range(xr - p.x + k, 2, p.x_len, p.err))) v = __ldg(reinterpret_cast<const float2*>(xr + k));
          const float a = v.x * sc, b = v.y * sc;  // exact: a power of two
          const __half2 hi = __floats2half2_rn(a, b);
          const float2 hf = __half22float2(hi);
          const __half2 lo = __floats2half2_rn(a - hf.x, b - hf.y);  // the differences are exact
          if (QMV_CHECK(smem_in_range(hrow + 2 * k, 4, p.err))) *reinterpret_cast<__half2*>(hrow + 2 * k) = hi;
          if (QMV_CHECK(smem_in_range(lrow + 2 * k, 4, p.err))) *reinterpret_cast<__half2*>(lrow + 2 * k) = lo;
        }
        if (lane == 0 && QMV_CHECK(smem_in_range(inv + tt, 4, p.err))) inv[tt] = 1.0f / sc;  // exact
      }
      named_sync(1, MF_CW * 32);
      staged_split = s;
    }
    const long long row0 = (long long)u * UNIT_ROWS;
    const int nrows = (int)min((long long)nu * UNIT_ROWS, p.M - row0);
    float acc[RP][TG][4];
#pragma unroll
    for (int r = 0; r < RP; r++)
#pragma unroll
      for (int h = 0; h < TG; h++) acc[r][h][0] = acc[r][h][1] = acc[r][h][2] = acc[r][h][3] = 0.0f;

    for (int c = 0; c < nck && alive; c++, ring.advance(p.stages)) {
      const int st = ring.st;
      // the stage's work is warp-wide (ldmatrix, mma.sync): the lanes vote
      if (!__all_sync(FULL, mbar_wait(&full[st], ring.parity(), p.err))) {
        alive = false;
        break;
      }
      const int kc = c * MF_KC + 32 * cw;  // this warp's first weight of the chunk, relative to the range
      // (klen is a multiple of 32: both steps are in range)
      if (kc < klen && QMV_CHECK(mf_step_in_range<NT>(stage_base + st * MF_STAGE, xh_base, xl_base, xpitch, kc, p.err))) {
        const uint32_t sbase = stage_base + st * MF_STAGE + 64 * cw;
#pragma unroll
        for (int ss = 0; ss < 2; ss++) {
          uint32_t A[RP][4];
#pragma unroll
          for (int r = 0; r < RP; r++) ldsm_x4(sbase + 32 * ss + 16 * r * MF_PITCH + a_off, A[r]);
          uint32_t B[TG][4];  // hi b0, b1, lo b0, b1
#pragma unroll
          for (int h = 0; h < TG; h++) ldsm_x4(b_off + (uint32_t)(8 * h * xpitch + 2 * (kc + 16 * ss)), B[h]);
#pragma unroll
          for (int r = 0; r < RP; r++)
#pragma unroll
            for (int h = 0; h < TG; h++) {
              mma_16816(acc[r][h], A[r], B[h][0], B[h][1]);
              mma_16816(acc[r][h], A[r], B[h][2], B[h][3]);
            }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }

    // ---- the eight warps' partial sums, added in warp order, scaled, stored ----
    named_sync(2, MF_CW * 32);  // the previous tile's sums have been read
#pragma unroll
    for (int r = 0; r < RP; r++)
#pragma unroll
      for (int h = 0; h < TG; h++)
#pragma unroll
        for (int i = 0; i < 2; i++) {
          float* q = red + (cw * NT + 8 * h + 2 * t4) * MK_RED_LD + 16 * r + 8 * i + g;
          if (!QMV_CHECK(smem_in_range(q, MK_RED_LD * 4 + 4, p.err))) continue;
          q[0] = acc[r][h][2 * i];
          q[MK_RED_LD] = acc[r][h][2 * i + 1];
        }
    named_sync(2, MF_CW * 32);
    float* out = p.out + (long long)s * p.ntot * p.M;
    for (int o = threadIdx.x; o < NT * MK_ROWS; o += MF_CW * 32) {
      const int tok = o / MK_ROWS, r = o - tok * MK_ROWS;
      float v = QMV_CHECK(smem_in_range(red + tok * MK_RED_LD + r, 4, p.err)) ? red[tok * MK_RED_LD + r] : 0.f;
#pragma unroll
      for (int w = 1; w < MF_CW; w++)
        if (QMV_CHECK(smem_in_range(red + (w * NT + tok) * MK_RED_LD + r, 4, p.err))) v += red[(w * NT + tok) * MK_RED_LD + r];
      if (tok < ntk && r < nrows) {
        const long long oi = (long long)(t0 + tok) * p.M + row0 + r;
        if (!QMV_CHECK(in_range((long long)s * p.ntot * p.M + oi, 1, p.out_len, p.err)) || !QMV_CHECK(smem_in_range(inv + tok, 4, p.err)))
          continue;
        v *= inv[tok];
        out[oi] = p.add ? v + (QMV_CHECK(in_range(oi, 1, p.add_len, p.err)) ? p.add[oi] : 0.f) : v;
      }
    }
  }
}

template <int NT>
static cudaError_t launch_mma_f16_nt(const DenseLaunch& L) {
  auto kern = qmv_mma_f16_kernel<NT>;
  // bit per device ordinal; host threads racing on a first launch both set
  // the same attribute, which is harmless
  static std::atomic<unsigned long long> configured{0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !((configured.load(std::memory_order_acquire) >> dev) & 1ull)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, device_smem_optin());
    if (e != cudaSuccess) return e;
    configured.fetch_or(1ull << dev, std::memory_order_acq_rel);
  }
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  make_config(cfg, attr, dim3(L.grid, L.passes), dim3(MF_THREADS), L.smem, L.stream, L.pdl);
  return cudaLaunchKernelEx(&cfg, kern, L.map_tile, L.map_unit, *L.p);
}

cudaError_t launch_mma_f16(const DenseLaunch& L) {
  switch (L.nt_tmpl) {
    case 8: return launch_mma_f16_nt<8>(L);
    case 16: return launch_mma_f16_nt<16>(L);
  }
  return cudaErrorInvalidValue;
}

size_t mma_f16_smem_bytes(int nt, int stages, int kmax) { return MfLayout(nt, stages, kmax).total; }

}  // namespace qmv
