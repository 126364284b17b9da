// Tensor-core small-batch matvec for Q4_K weights and 5 to 16 tokens.
//
// The operation and its arithmetic are those of the dense kernel
// (qmv_dense.cuh, "Castagna Veloce", section "Kernels for the MI50":
// small-batch matvecs over K-quants): per row m, token t and 32-weight block
// j, the exact integer dot product I = sum_i q_i * xq_i of the block, then
//   y += (d * sc_j * d_x) * I - (dmin * m_j) * (d_x * s)     (fp32 FMAs)
// in the same formula and rounding as the dp4a path.  What differs is who
// forms I.  From eight tokens on the dp4a path is bound by its issue rate
// (one dp4a per four weights per token, half the FMA rate); here the warps'
// tensor-core MMA (mma.sync m16n8k16, f16 operands, fp32 accumulation) forms
// the block sums of 16 rows x 8 token slots at once:
//   - A operand: 16 weight rows, each nibble entering as the f16 1024 + q
//     (the nibble as the mantissa of 1024; one lop3 per two weights);
//   - B operand: the activation codes of 8 token slots (exact f16 integers,
//     converted in registers from the staged int8 codes);
//   - C operand: -1024 * s of each token, so that the MMA yields I itself,
//     exactly (every partial sum is an integer below 2^23);
//   - the logical k order inside a block is a permutation of the physical
//     one that lets each lane's operand pairs come from one 32-bit word of
//     the payload (q_4c, q_4c+2 | q_4c+1, q_4c+3 | their high nibbles), with
//     the activations read in the same permuted order.
// The accumulator pairs are (token 2c, 2c + 1) of one row, so the token
// scales are read as pairs and the row scales are kept duplicated: each
// fold is one packed multiply and two packed FMAs.
// Structure: persistent CTAs over tiles of 64 rows (8 units of 8), the
// (split, unit) space cut as in the dense kernel.  One producer lane streams
// each tile's 768-weight chunks (3 superblocks, 432 bytes per row: an odd
// number of 16-byte units, so the 8 rows read by one ldmatrix phase fall in
// 8 different bank groups) by 2-D TMA into a ring of stages.  Twelve
// consumer warps (three per scheduler; the producer warpgroup hands them its
// registers) split each chunk by blocks (warp w: blocks 2w, 2w + 1) and
// cover all 64 rows: the activation operand of a block is converted once per
// warp and used for all 4 row pairs; each warp first turns its rows' block
// scales into fp32 (d * sc, -dmin * m) in a small shared-memory area.  At
// the end of a tile the twelve warps' partial sums are added in a fixed
// order through shared memory (deterministic) and stored.
#pragma once
#include "qmv_dense.cuh"

namespace qmv {

constexpr int MK_CW = 12;                          // consumer warps (one per block pair of a chunk)
constexpr int MK_PW = 4;                           // producer warpgroup
constexpr int MK_THREADS = (MK_CW + MK_PW) * 32;   // 512
constexpr int MK_REG_PRODUCER = 32, MK_REG_CONSUMER = 160;
static_assert(MK_PW * 32 * MK_REG_PRODUCER + MK_CW * 32 * MK_REG_CONSUMER <= 65536,
              "register re-split exceeds the launch's registers");
constexpr int MK_UNITS = 8;                        // 8-row units per tile
constexpr int MK_ROWS = MK_UNITS * UNIT_ROWS;      // 64
constexpr int MK_GROUPS = 3;                       // Q4_K superblocks per chunk
constexpr int MK_BLOCKS = MK_GROUPS * 8;           // 32-weight blocks per chunk
constexpr int MK_CB = MK_GROUPS * 144;             // bytes of a row's chunk
constexpr int MK_PITCH = MK_CB;                    // 432 = 27 x 16: odd, so 8 rows hit 8 bank groups
constexpr int MK_STAGE = MK_ROWS * MK_PITCH;       // 27,648 bytes
constexpr int MK_RED_LD = 72;                      // floats per (warp, token) row of the partial sums
constexpr int MK_RW = MK_CW / 2;                   // warps whose sums one reduction round holds

// Shared-memory layout of the kernel (host and device compute the same):
//   [stages][64 rows][432]        weight ring
//   codes [NT][apitch]            staged activation codes of the split range
//                                 (the library's Q8 order, 16 bytes of padding
//                                 per token so that 8 tokens hit 8 bank groups)
//   dx [NT][dpitch] f32, xs [NT][dpitch] i32   block scales and code sums
//   scl [12 warps][2 blocks][64 rows] float4  (a_r, a_r, -c_r, -c_r)
//   red [6 warps][NT][72] f32     partial sums of a tile (two rounds)
//   mbarriers: full[8], empty[8], activation copies, first staging done
struct MmaLayout {
  size_t codes, dx, xs, scl, red, bars, total;
  int apitch, dpitch;
  __host__ __device__ MmaLayout(int nt, int stages, int nbmax) {
    apitch = nbmax * 32 + 16;
    dpitch = nbmax + 4;
    codes = (size_t)stages * MK_STAGE;
    dx = codes + (size_t)nt * apitch;
    xs = dx + (size_t)nt * dpitch * 4;
    scl = xs + (size_t)nt * dpitch * 4;
    red = scl + (size_t)MK_CW * 2 * MK_ROWS * 16;
    bars = red + (size_t)MK_RW * nt * MK_RED_LD * 4;
    total = bars + (2 * MAX_STAGES + 2) * 8;
  }
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// d += A B for one m16n8k16 tile (f16 operands, fp32 accumulators).
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// d = A B + c for one m16n8k16 tile.
__device__ __forceinline__ void mma_16816c(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                           const float (&c)[4]) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%10, %11, %12, %13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

// Bytes 0 and 2 of w (int8 codes) as an exact f16 pair: with the sign bit
// flipped a byte is x + 128, the mantissa of the f16 1024 + (x + 128); the
// f16 subtraction of 1152 leaves x (exact).
__device__ __forceinline__ uint32_t s8x2_f16(uint32_t w) {
  uint32_t h, r;
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(h) : "r"(w), "r"(0x00FF00FFu), "r"(0x64806480u));  // (a & b) ^ c
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(0x64806480u));
  return r;
}

// Nibbles at bits 0-3 and 16-19 of w as the f16 pair 1024 + q (one lop3).
__device__ __forceinline__ uint32_t u4x2_f16(uint32_t w) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(w), "r"(0x000F000Fu), "r"(0x64006400u));  // (a & b) | c
  return r;
}

// Token slots [nt, NT) of the block scales and sums: zero (their sums are
// never stored; zeros keep them finite).
template <int NT>
__device__ __forceinline__ void mk_zero_slots(float* dxa, int32_t* xsa, int dpitch, int nt, int nblk, int tid,
                                              unsigned* err) {
  const int rest = NT - nt;
  for (int i = tid; i < rest * nblk; i += MK_CW * 32) {
    const int t = nt + i / nblk, b = i - (t - nt) * nblk;
    if (QMV_CHECK(smem_in_range(dxa + t * dpitch + b, 4, err))) dxa[t * dpitch + b] = 0.0f;
    if (QMV_CHECK(smem_in_range(xsa + t * dpitch + b, 4, err))) xsa[t * dpitch + b] = 0;
  }
}

// The shared-memory ranges of a warp's step over blocks kbase, kbase + 1 of
// a chunk: the weight stage, the NT token slots' codes (the 256-byte group
// that holds both blocks), scales and sums of those blocks, and the warp's
// scale area.
template <int NT>
__device__ __forceinline__ bool mk_step_in_range(uint32_t sbase, uint32_t codes_base, const float* dxa,
                                                 const int32_t* xsa, const float4* wscl, int apitch, int dpitch,
                                                 int kbase, unsigned* err) {
  const uint32_t g = (uint32_t)(kbase >> 3) * 256;
  return smem_in_range(sbase, MK_STAGE, err) && smem_in_range(codes_base + g, (NT - 1) * apitch + 256, err) &&
         smem_in_range(dxa + kbase, ((NT - 1) * dpitch + 2) * 4, err) &&
         smem_in_range(xsa + kbase, ((NT - 1) * dpitch + 2) * 4, err) &&
         smem_in_range(wscl, 2 * MK_ROWS * 16, err);
}

// Activation staging of tokens [0, nt) of the pass (rows t0 + t of x),
// blocks [kb0, kb0 + nblk): fp32 rows quantized by the activation rule
// (quant_units, the dense path's code); codes in the library's Q8 order.
template <int NT>
__device__ __forceinline__ void mk_stage_fp32(const DenseParams& p, int t0, int nt, int kb0, int nblk,
                                              uint8_t* codes, float* dxa, int32_t* xsa, int apitch, int dpitch,
                                              int cw, int lane) {
  constexpr int SU = 4;
  const int sub = lane >> 2, li = lane & 3;
  const int total = nt * nblk;
  for (int base = cw * 8 * SU; base < total; base += MK_CW * 8 * SU) {  // warp-uniform trip count
    float4 v[SU][2];
    uint32_t w0[SU], w1[SU];
    float dd[SU];
    int ss[SU], tt[SU], bb[SU];
    bool real[SU];
#pragma unroll
    for (int u = 0; u < SU; u++) {
      const int idx = base + 8 * u + sub;
      real[u] = idx < total;
      tt[u] = real[u] ? idx / nblk : 0;
      bb[u] = idx - tt[u] * nblk;
      if (real[u] && !QMV_CHECK(in_range((long long)(t0 + tt[u]) * p.K + (long long)(kb0 + bb[u]) * BLK, BLK, p.x_len, p.err)))
        real[u] = false;
      v[u][0] = v[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (real[u]) {
        const float4* src = reinterpret_cast<const float4*>(p.x + (long long)(t0 + tt[u]) * p.K +
                                                            (long long)(kb0 + bb[u]) * BLK) + 2 * li;
        v[u][0] = __ldg(src);
        v[u][1] = __ldg(src + 1);
      }
    }
    quant_units<SU>(v, w0, w1, dd, ss);
#pragma unroll
    for (int u = 0; u < SU; u++) {
      if (real[u]) {
        uint8_t* q = codes + (size_t)tt[u] * apitch + act_pos(bb[u], 8 * li);
        if (QMV_CHECK(smem_in_range(q, 8, p.err))) *reinterpret_cast<uint2*>(q) = make_uint2(w0[u], w1[u]);
        if (li == 0 && QMV_CHECK(smem_in_range(dxa + tt[u] * dpitch + bb[u], 4, p.err)) &&
            QMV_CHECK(smem_in_range(xsa + tt[u] * dpitch + bb[u], 4, p.err))) {
          dxa[tt[u] * dpitch + bb[u]] = dd[u];
          xsa[tt[u] * dpitch + bb[u]] = ss[u];
        }
      }
    }
  }
  mk_zero_slots<NT>(dxa, xsa, dpitch, nt, nblk, cw * 32 + lane, p.err);
}

// The same from pre-quantized rows (the library's Q8 layout): three bulk
// copies per token (codes, scales, sums).  Warp 0 lane 0 posts the byte
// count first.  Returns false (timeout bit set) if the copies never land.
template <int NT>
__device__ __forceinline__ bool mk_stage_q8(const DenseParams& p, int t0, int nt, int kb0, int nblk, uint8_t* codes,
                                            float* ldx, int32_t* lxs, int apitch, int dpitch, uint64_t* bar,
                                            uint32_t parity, int cw, int lane) {
  if (cw == 0 && lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(nt * nblk * (BLK + 8)));
  // the previous range's scales and sums were read (and its unused token
  // slots written) by the generic proxy: order that before the copies
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  named_sync(1, MK_CW * 32);  // the byte count is posted before any copy completes
  const long long nbr = p.K / BLK;
  for (int i = cw * 32 + lane; i < 3 * nt; i += MK_CW * 32) {
    const int t = i / 3, k = i - 3 * t;
    const long long row = t0 + t;
    const uint32_t bytes = (uint32_t)nblk * (k == 0 ? BLK : 4);
    void* dst = k == 0 ? (void*)(codes + (size_t)t * apitch) : k == 1 ? (void*)(ldx + t * dpitch) : (void*)(lxs + t * dpitch);
    if (!QMV_CHECK(in_range(row * p.K + (long long)kb0 * BLK, (long long)nblk * BLK, p.x_len, p.err)) ||
        !QMV_CHECK(smem_in_range(dst, bytes, p.err))) {
      mbar_complete_tx(bar, bytes);  // skipped: the phase still completes
      continue;
    }
    if (k == 0)
      bulk_copy_g2s(dst, p.xq + row * p.K + (long long)kb0 * BLK, bytes, bar);
    else if (k == 1)
      bulk_copy_g2s(dst, p.xd + row * nbr + kb0, bytes, bar);
    else
      bulk_copy_g2s(dst, p.xs + row * nbr + kb0, bytes, bar);
  }
  mk_zero_slots<NT>(ldx, lxs, dpitch, nt, nblk, cw * 32 + lane, p.err);
  return mbar_wait(bar, parity, p.err);
}

// Fields sc_j, m_j, sc_j+1, m_j+1 (6 bits each, from bit 0) of the sub-block
// pair k (j = 2k) of a Q4_K header: bits [24k, 24k + 24) of the 96-bit string
// in header words 1-3.
__device__ __forceinline__ uint32_t q4k_pair_fields(const uint4& h, int k) {
  return k == 0 ? h.y : (k == 1 ? __funnelshift_r(h.y, h.z, 24) : (k == 2 ? __funnelshift_r(h.z, h.w, 16) : h.w >> 8));
}

template <int NT>
__global__ void __launch_bounds__(MK_THREADS, 1)
    qmv_mma_q4k_kernel(const __grid_constant__ CUtensorMap map_tile, const __grid_constant__ CUtensorMap map_unit,
                       const DenseParams p) {
  static_assert(NT == 8 || NT == 16, "8 or 16 token slots");
  constexpr int TG = NT / 8;  // token groups of a lane: slots g and g + 8
  extern __shared__ __align__(128) uint8_t smem[];
  const MmaLayout L(NT, p.stages, p.nbmax);
  uint8_t* stages = smem;
  uint8_t* codes = smem + L.codes;
  float* dxa = reinterpret_cast<float*>(smem + L.dx);
  int32_t* xsa = reinterpret_cast<int32_t*>(smem + L.xs);
  float4* scl = reinterpret_cast<float4*>(smem + L.scl);
  float* red = reinterpret_cast<float*>(smem + L.red);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + MAX_STAGES;
  uint64_t* abar = full + 2 * MAX_STAGES;  // [0] activation copies, [1] first staging done

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(abar, 1);
    mbar_init(abar + 1, 1);
  }
  init_pipeline(full, empty, p.stages, MK_CW);
  pdl_launch_dependents();
  const bool q8in = p.x == nullptr;

  if (warp >= MK_CW) {
    // ---------------- producer: one elected lane, 2-D TMA ----------------
    // The producer warpgroup hands all but MK_REG_PRODUCER registers each to
    // the consumers.  With pre-quantized activations (whose copies are the
    // critical path at the start) only two stages are requested before the
    // consumers have staged them, as in the dense kernel.  (A box past the
    // row's end reads zeros.)
    regs_dec<MK_REG_PRODUCER>();
    if (warp == MK_CW && lane == 0) {
      prefetch_tensormap(&map_tile);
      prefetch_tensormap(&map_unit);
      const uint64_t pol = policy_evict_first();
      const long long gate = q8in ? 2 : -1;
      TileWalk<MK_UNITS> walk(p);
      int s, u, nu;
      Ring ring;
      bool alive = true;
      while (alive && walk.next(s, u, nu)) {
        int g0, g1;
        split_range(p, s, g0, g1);
        const int nck = (g1 - g0 + MK_GROUPS - 1) / MK_GROUPS;
        for (int c = 0; c < nck; c++, ring.advance(p.stages)) {
          if (ring.n == gate && !mbar_wait(abar + 1, 0, p.err)) {
            alive = false;
            break;
          }
          if (!producer_acquire(empty, ring, p.stages, p.err)) {
            alive = false;
            break;
          }
          const int st = ring.st;
          uint8_t* dst = stages + st * MK_STAGE;
          const int x = (g0 + c * MK_GROUPS) * (144 / 8);  // 8-byte elements; x * 8 = 144 * group
          if (!QMV_CHECK(smem_in_range(dst, nu * UNIT_ROWS * MK_PITCH, p.err))) {
            mbar_arrive(&full[st]);  // skipped: the stage completes without data
          } else if (nu == MK_UNITS) {
            mbar_arrive_expect_tx(&full[st], MK_STAGE);
            tma_load_2d(dst, &map_tile, &full[st], x, u * UNIT_ROWS, pol);
          } else {
            mbar_arrive_expect_tx(&full[st], nu * UNIT_ROWS * MK_PITCH);
            for (int i = 0; i < nu; i++)
              tma_load_2d(dst + i * UNIT_ROWS * MK_PITCH, &map_unit, &full[st], x, (u + i) * UNIT_ROWS, pol);
          }
        }
      }
      producer_drain(full, ring.n, p.stages, p.err);
    }
    return;
  }

  // ---------------- consumers ----------------
  // A warp that gives up on a wait keeps walking the tiles (without waiting
  // or computing) so that the named barriers of the others still complete;
  // the timeout bit is already set.
  constexpr int RP = MK_UNITS / 2;  // row pairs (16 rows: the MMA's M) of a tile
  regs_inc<MK_REG_CONSUMER>();
  const int cw = warp, g = lane >> 2, t4 = lane & 3;
  const int t0 = p.t0 + blockIdx.y * NT, ntk = p.nt;
  const int apitch = L.apitch, dpitch = L.dpitch;
  const uint32_t stage_base = smem_u32(stages), codes_base = smem_u32(codes);
  // this warp's blocks of a chunk: 2 cw, 2 cw + 1 = sub-blocks j0, j0 + 1 of superblock sb
  const int sb = cw >> 2, kp = cw & 3, j0 = 2 * kp;
  // ldmatrix source row of this lane: unit lane / 8 of a quad of units, row lane % 8
  const uint32_t lm_off = (uint32_t)(((lane >> 3) * UNIT_ROWS + (lane & 7)) * MK_PITCH + sb * 144 + 16 + 16 * j0);
  static_assert(MK_CW * 2 == MK_BLOCKS, "each warp takes two blocks of a chunk");
  float4* wscl = scl + cw * 2 * MK_ROWS;  // [block of the pair][row]
  bool alive = true;
  TileWalk<MK_UNITS> walk(p);
  int s, u, nu;
  Ring ring;
  int staged_split = -1;
  uint32_t aphase = 0;

  // the activations may come from the preceding kernel: wait for it only
  // now, so that the set-up above (parameters only) runs while it finishes
  pdl_wait();
  while (walk.next(s, u, nu)) {
    int g0, g1;
    split_range(p, s, g0, g1);
    const int kb0 = g0 * 8, nblk = (g1 - g0) * 8;
    if (s != staged_split) {
      if (staged_split >= 0) named_sync(1, MK_CW * 32);  // nobody still reads the previous range (or the partial sums)
      if (!q8in) {
        mk_stage_fp32<NT>(p, t0, ntk, kb0, nblk, codes, dxa, xsa, apitch, dpitch, cw, lane);
      } else {
        alive = __all_sync(FULL, mk_stage_q8<NT>(p, t0, ntk, kb0, nblk, codes, dxa, xsa, apitch, dpitch, abar,
                                                 aphase, cw, lane)) &&
                alive;
        aphase ^= 1;
      }
      named_sync(1, MK_CW * 32);
      if (threadIdx.x == 0 && staged_split < 0) mbar_arrive(abar + 1);  // the producer may go on
      staged_split = s;
    }
    const long long row0 = (long long)u * UNIT_ROWS;
    const int nrows = (int)min((long long)nu * UNIT_ROWS, p.M - row0);
    const int nck = (g1 - g0 + MK_GROUPS - 1) / MK_GROUPS;
    float2 acc[RP][TG][2];  // [row pair][token tile][row g, g + 8]: tokens 2 t4, 2 t4 + 1
#pragma unroll
    for (int i = 0; i < RP; i++)
#pragma unroll
      for (int k = 0; k < TG; k++) acc[i][k][0] = acc[i][k][1] = make_float2(0.f, 0.f);

    for (int c = 0; c < nck && alive; c++, ring.advance(p.stages)) {
      const int st = ring.st;
      // the stage's work is warp-wide (ldmatrix, mma.sync): the lanes vote
      if (!__all_sync(FULL, mbar_wait(&full[st], ring.parity(), p.err))) {
        alive = false;
        break;
      }
      const int kbase = c * MK_BLOCKS + 2 * cw;  // this warp's first block, relative to kb0
      // (a last chunk of one or two superblocks leaves warps 4-11 or 8-11 idle)
      if (kbase < nblk && QMV_CHECK(mk_step_in_range<NT>(stage_base + st * MK_STAGE, codes_base, dxa, xsa, wscl, apitch,
                                               dpitch, kbase, p.err))) {
        const uint32_t sbase = stage_base + st * MK_STAGE;
        {
          // (a, a, -c, -c) of rows 2 lane, 2 lane + 1 for both blocks
          const uint8_t* hrow = stages + st * MK_STAGE + (2 * lane) * MK_PITCH + sb * 144;
          const uint4 ha = *reinterpret_cast<const uint4*>(hrow);
          const uint4 hb = *reinterpret_cast<const uint4*>(hrow + MK_PITCH);
          const float2 da = __half22float2(*reinterpret_cast<const __half2*>(&ha.x));  // d | dmin
          const float2 db = __half22float2(*reinterpret_cast<const __half2*>(&hb.x));
          const uint32_t fa = q4k_pair_fields(ha, kp), fb = q4k_pair_fields(hb, kp);
#pragma unroll
          for (int jj = 0; jj < 2; jj++) {
            const int sh = 12 * jj;
            const float aa = da.x * (float)((fa >> sh) & 63u), ca = da.y * (float)((fa >> (sh + 6)) & 63u);
            const float ab = db.x * (float)((fb >> sh) & 63u), cb = db.y * (float)((fb >> (sh + 6)) & 63u);
            wscl[jj * MK_ROWS + 2 * lane] = make_float4(aa, aa, -ca, -ca);
            wscl[jj * MK_ROWS + 2 * lane + 1] = make_float4(ab, ab, -cb, -cb);
          }
        }
        __syncwarp();
#pragma unroll
        for (int jj = 0; jj < 2; jj++) {
          const int kb = kbase + jj;
          // the B operand of block kb for token tiles h: token slot 8 h + g
          const uint32_t ra = codes_base + g * apitch + (kb >> 3) * 256 + (kb & 7) * 16 + 4 * t4;
          uint32_t B[TG][4];
          float2 DX[TG], DS[TG];
          float C[TG][4];  // the MMA's C operand: -1024 s of tokens 2 t4, 2 t4 + 1 (rows g and g + 8)
#pragma unroll
          for (int h = 0; h < TG; h++) {
            const uint32_t x0 = lds32(ra + h * 8 * apitch), x1 = lds32(ra + h * 8 * apitch + 128);
            B[h][0] = s8x2_f16(x0);
            B[h][1] = s8x2_f16(x0 >> 8);
            B[h][2] = s8x2_f16(x1);
            B[h][3] = s8x2_f16(x1 >> 8);
            // block scales and code sums of tokens 2 t4, 2 t4 + 1 of the tile:
            // d_x, d_x * s (the min term's multiplier, the product the dp4a path
            // forms) and -1024 * s (the MMA's C operand, exact)
            const int tk = (8 * h + 2 * t4) * dpitch + kb;
            DX[h] = make_float2(dxa[tk], dxa[tk + dpitch]);
            const float2 sf = make_float2((float)xsa[tk], (float)xsa[tk + dpitch]);
            DS[h] = __fmul2_rn(DX[h], sf);
            const float2 ns = __fmul2_rn(sf, make_float2(-1024.0f, -1024.0f));
            C[h][0] = C[h][2] = ns.x;
            C[h][1] = C[h][3] = ns.y;
          }
          // the 64 rows' words (ldmatrix: units 0-3, then 4-7), all branch-free
          // (units past the tile's rows compute on stale rows and are never
          // stored), so that the MMAs and folds of the row pairs interleave
          uint32_t wq[MK_UNITS];
          ldsm_x4(sbase + lm_off + 16 * jj, *reinterpret_cast<uint32_t(*)[4]>(wq));
          ldsm_x4(sbase + lm_off + 16 * jj + 4 * UNIT_ROWS * MK_PITCH, *reinterpret_cast<uint32_t(*)[4]>(wq + 4));
          // operands of the 4 row pairs, then the first MMA of every (row
          // pair, token tile), then the second (each 8 MMAs after its
          // first, so its latency is covered), then the folds
          uint32_t A1[RP][4], A2[RP][4];
#pragma unroll
          for (int r = 0; r < RP; r++) {
            const uint32_t wa = wq[2 * r], wb = wq[2 * r + 1];  // rows 16 r + g, 16 r + 8 + g
            A1[r][0] = u4x2_f16(wa);
            A1[r][1] = u4x2_f16(wb);
            A1[r][2] = u4x2_f16(wa >> 8);
            A1[r][3] = u4x2_f16(wb >> 8);
            A2[r][0] = u4x2_f16(wa >> 4);
            A2[r][1] = u4x2_f16(wb >> 4);
            A2[r][2] = u4x2_f16(wa >> 12);
            A2[r][3] = u4x2_f16(wb >> 12);
          }
          float d[RP][TG][4];
#pragma unroll
          for (int r = 0; r < RP; r++)
#pragma unroll
            for (int h = 0; h < TG; h++) mma_16816c(d[r][h], A1[r], B[h][0], B[h][1], C[h]);
#pragma unroll
          for (int r = 0; r < RP; r++)
#pragma unroll
            for (int h = 0; h < TG; h++) mma_16816(d[r][h], A2[r], B[h][2], B[h][3]);
#pragma unroll
          for (int r = 0; r < RP; r++) {
            const float4 sa = wscl[jj * MK_ROWS + 16 * r + g], sb8 = wscl[jj * MK_ROWS + 16 * r + 8 + g];
#pragma unroll
            for (int h = 0; h < TG; h++) {
              const float2 p0 = __fmul2_rn(make_float2(sa.x, sa.y), DX[h]);
              const float2 p1 = __fmul2_rn(make_float2(sb8.x, sb8.y), DX[h]);
              acc[r][h][0] = __ffma2_rn(make_float2(sa.z, sa.w), DS[h],
                                        __ffma2_rn(p0, make_float2(d[r][h][0], d[r][h][1]), acc[r][h][0]));
              acc[r][h][1] = __ffma2_rn(make_float2(sb8.z, sb8.w), DS[h],
                                        __ffma2_rn(p1, make_float2(d[r][h][2], d[r][h][3]), acc[r][h][1]));
            }
          }
        }
        __syncwarp();  // the scale area is rewritten for the next chunk
      }
      if (lane == 0) mbar_arrive(&empty[st]);
    }

    // ---- the twelve warps' partial sums, added in a fixed order, stored ----
    // Two rounds through a 6-warp area: warps 6-11 write, warps 0-5 add them
    // to their own, then warps 0-5 write and every thread sums the six.
    auto put = [&]() {
#pragma unroll
      for (int r = 0; r < RP; r++)
#pragma unroll
        for (int h = 0; h < TG; h++)
#pragma unroll
          for (int i = 0; i < 2; i++) {
            float* q = red + ((cw % MK_RW) * NT + 8 * h + 2 * t4) * MK_RED_LD + 16 * r + 8 * i + g;
            if (!QMV_CHECK(smem_in_range(q, MK_RED_LD * 4 + 4, p.err))) continue;
            q[0] = acc[r][h][i].x;
            q[MK_RED_LD] = acc[r][h][i].y;
          }
    };
    named_sync(2, MK_CW * 32);  // the previous tile's sums have been read
    if (cw >= MK_RW) put();
    named_sync(2, MK_CW * 32);
    if (cw < MK_RW) {
#pragma unroll
      for (int r = 0; r < RP; r++)
#pragma unroll
        for (int h = 0; h < TG; h++)
#pragma unroll
          for (int i = 0; i < 2; i++) {
            const float* q = red + (cw * NT + 8 * h + 2 * t4) * MK_RED_LD + 16 * r + 8 * i + g;
            if (!QMV_CHECK(smem_in_range(q, MK_RED_LD * 4 + 4, p.err))) continue;
            acc[r][h][i].x += q[0];
            acc[r][h][i].y += q[MK_RED_LD];
          }
    }
    named_sync(2, MK_CW * 32);
    if (cw < MK_RW) put();
    named_sync(2, MK_CW * 32);
    float* out = p.out + (long long)s * p.ntot * p.M;
    for (int o = threadIdx.x; o < NT * MK_ROWS; o += MK_CW * 32) {
      const int tok = o / MK_ROWS, r = o - tok * MK_ROWS;
      float v = QMV_CHECK(smem_in_range(red + tok * MK_RED_LD + r, 4, p.err)) ? red[tok * MK_RED_LD + r] : 0.f;
#pragma unroll
      for (int w = 1; w < MK_RW; w++)
        if (QMV_CHECK(smem_in_range(red + (w * NT + tok) * MK_RED_LD + r, 4, p.err))) v += red[(w * NT + tok) * MK_RED_LD + r];
      if (tok < ntk && r < nrows) {
        const long long oi = (long long)(t0 + tok) * p.M + row0 + r;
        if (!QMV_CHECK(in_range((long long)s * p.ntot * p.M + oi, 1, p.out_len, p.err))) continue;
        out[oi] = p.add ? v + (QMV_CHECK(in_range(oi, 1, p.add_len, p.err)) ? p.add[oi] : 0.f) : v;
      }
    }
  }
}

}  // namespace qmv
