// Dense small-batch quantized matvec (and its split-K first pass).
//
// Y[t][m] = sum_k What[m][k] * Xhat[t][k] for a few tokens t: the decode-time
// matrix-vector product over block-quantized weights ("Castagna Veloce",
// section "Kernels for the MI50": small-batch matvecs for K-quants, IQ4_XS and
// Q8_0 with a split-K variant; "Running GLM-5.3 on Two 8-GPU AMD W7900D
// Machines", section "A single decode row is not a large matrix
// multiplication": weight reads dominate).
//
// Structure (one persistent CTA per SM):
//   - warp 8 (producer): one elected lane streams the CTA's weight tiles,
//     TILE_ROWS rows x 1024 weights, with 2-D TMA loads into a ring of
//     shared-memory stages guarded by full/empty mbarriers;
//   - warps 0..7 (consumers): quantize the activations of the K-range into
//     shared memory (per-32 int8, the activation rule), then for every stage
//     decode RW = 4 rows each in registers (one 32-weight block per lane),
//     form exact int32 block dot products with dp4a, apply the block scales in
//     fp32 and, at the end of a tile, reduce across lanes and store.
// Work split: the (split, 8-row unit) space is cut into contiguous,
// equal-sized ranges, one per CTA; a tile never crosses a split.
#pragma once
#include "common.cuh"

namespace qmv {

constexpr int CONSUMER_WARPS = 8;
constexpr int RW = 4;                                 // rows per consumer warp
constexpr int TILE_ROWS = CONSUMER_WARPS * RW;        // 32
constexpr int UNIT_ROWS = 8;                          // partition / tail-box granularity
constexpr int THREADS = (CONSUMER_WARPS + 1) * 32;    // + producer warp
constexpr int CONSUMER_THREADS = CONSUMER_WARPS * 32;
constexpr int MAX_STAGES = 8;
constexpr unsigned FULL = 0xffffffffu;

struct DenseParams {
  const float* x;      // fp32 activations [ntot][K], or nullptr when pre-quantized
  const int8_t* xq;    // pre-quantized activations [ntot][K] (natural order)
  const float* xd;     // [ntot][K/32]
  const int32_t* xs;   // [ntot][K/32]
  float* out;          // y [ntot][M] (n_split == 1) or partial [n_split][ntot][M]
  long long M;
  int K;               // weights per row
  int ntot;            // tokens held by x / out
  int t0;              // first token of this pass
  int nt;              // tokens of this pass (<= NT)
  int n_split;
  int groups;          // K / group weights
  int units;           // ceil(M / UNIT_ROWS)
  int stages;
  int act_stride;      // bytes per token row of the activation area
  int act_blk;         // blocks per token row of the scale areas (act_stride / 32)
  unsigned* err;       // device error word
};

// Shared-memory position of byte p (0..31) of activation block b of a token
// row: within every 256-weight group, the first 16 bytes of the 8 blocks come
// first, then the last 16, so that the 8 lanes of a quarter-warp read 128
// contiguous bytes.
__device__ __forceinline__ int act_pos(int b, int p) {
  return (b >> 3) * 256 + (p >> 4) * 128 + (b & 7) * 16 + (p & 15);
}

// Quantize four consecutive elements of a 32-block spread over 8 lanes
// (lanes 8g..8g+7 hold block g of the warp); returns the packed int8 codes of
// this lane, the block scale d and the block sum s (identical in the 8 lanes).
struct Quad {
  uint32_t q;
  float d;
  int s;
};
__device__ __forceinline__ Quad quant_quad(float4 v) {
  float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
  m = fmaxf(m, __shfl_xor_sync(FULL, m, 1));
  m = fmaxf(m, __shfl_xor_sync(FULL, m, 2));
  m = fmaxf(m, __shfl_xor_sync(FULL, m, 4));
  float d = __fdiv_rn(m, 127.0f);
  float id = d > 0.0f ? __fdiv_rn(1.0f, d) : 0.0f;
  int q0 = max(-127, min(127, __float2int_rn(__fmul_rn(v.x, id))));
  int q1 = max(-127, min(127, __float2int_rn(__fmul_rn(v.y, id))));
  int q2 = max(-127, min(127, __float2int_rn(__fmul_rn(v.z, id))));
  int q3 = max(-127, min(127, __float2int_rn(__fmul_rn(v.w, id))));
  int s = q0 + q1 + q2 + q3;
  s += __shfl_xor_sync(FULL, s, 1);
  s += __shfl_xor_sync(FULL, s, 2);
  s += __shfl_xor_sync(FULL, s, 4);
  uint32_t packed = (uint32_t)(q0 & 0xFF) | ((uint32_t)(q1 & 0xFF) << 8) | ((uint32_t)(q2 & 0xFF) << 16) |
                    ((uint32_t)(q3 & 0xFF) << 24);
  return {packed, d, s};
}

// Store the packed codes of elements 4*li..4*li+3 of block b (li = lane & 7)
// into the activation area in the byte order format F consumes.  For IQ4_XS
// a block is stored interleaved (byte 2i = x_i, byte 2i+1 = x_{i+16}), the
// order in which its codebook lookups come out; the other formats use the
// natural order.  Must be called by all 32 lanes (it shuffles).
template <int F>
__device__ __forceinline__ void store_act_quad(uint8_t* row, int b, int li, uint32_t packed, bool ok) {
  if constexpr (F == QMV_IQ4_XS) {
    uint32_t hi = __shfl_xor_sync(FULL, packed, 4);  // elements 16 + 4*li ..
    if (ok && li < 4) {
      uint2 w;
      w.x = __byte_perm(packed, hi, 0x5140);
      w.y = __byte_perm(packed, hi, 0x7362);
      *reinterpret_cast<uint2*>(row + act_pos(b, 8 * li)) = w;
    }
  } else {
    if (ok) *reinterpret_cast<uint32_t*>(row + act_pos(b, 4 * li)) = packed;
  }
}

// Stage the activations of tokens [t0, t0 + nt) and blocks [kb0, kb0 + nblk)
// into shared memory: codes, scales d and (Q4_K) d * s.
template <int F>
__device__ void stage_activations(const DenseParams& p, int kb0, int nblk, uint8_t* act_q, float* act_d,
                                  float* act_ds, int cw, int lane) {
  const int sub = lane >> 3, li = lane & 7;
  const int total = p.nt * nblk;
  for (int base = cw * 4; base < total; base += CONSUMER_WARPS * 4) {
    const int idx = base + sub;
    const bool ok = idx < total;
    const int t = ok ? idx / nblk : 0;
    const int b = ok ? idx - t * nblk : 0;
    const long long tok = p.t0 + t;
    uint32_t packed;
    float d;
    int s;
    if (p.x != nullptr) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (ok) v = __ldg(reinterpret_cast<const float4*>(p.x + tok * p.K + (long long)(kb0 + b) * 32) + li);
      Quad qd = quant_quad(v);
      packed = qd.q;
      d = qd.d;
      s = qd.s;
    } else {
      packed = 0;
      d = 0.f;
      s = 0;
      if (ok) {
        packed = __ldg(reinterpret_cast<const uint32_t*>(p.xq + tok * p.K + (long long)(kb0 + b) * 32) + li);
        d = __ldg(p.xd + tok * (p.K / 32) + kb0 + b);
        s = __ldg(p.xs + tok * (p.K / 32) + kb0 + b);
      }
    }
    store_act_quad<F>(act_q + t * p.act_stride, b, li, packed, ok);
    if (ok && li == 0) {
      act_d[t * p.act_blk + b] = d;
      if constexpr (F == QMV_Q4_K) act_ds[t * p.act_blk + b] = d * (float)s;
    }
  }
}

// Codebook lookup of four 4-bit codes held as the nibbles of the low 16 bits
// of `sel` (nibble k -> byte k of the result).  pl = sel & 0x7777 (low three
// bits of each code) picks from the lower and the upper half of the codebook
// with two byte permutes; the fourth bit of each code becomes a byte mask
// through the sign-replicating mode of a third permute (msb of the selected
// byte copied to all 8 bits), fed with sel and sel << 4 so that the fourth bits
// of the four codes sit at byte msbs.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
__device__ __forceinline__ uint32_t iq4_lookup4(uint32_t pl, uint32_t p, uint32_t p4, uint32_t mask_sel) {
  constexpr uint32_t T0 = 0xBFAD9881u, T1 = 0xF6EADDCFu;  // codes 0..7
  constexpr uint32_t T2 = 0x26190D01u, T3 = 0x71594535u;  // codes 8..15
  uint32_t lo = prmt(T0, T1, pl);
  uint32_t hi = prmt(T2, T3, pl);
  uint32_t m = prmt(p4, p, mask_sel);
  return (hi & m) | (lo & ~m);
}

template <int F, int NT>
struct Consumer {
  // Accumulate one chunk: rows r < nrows of this warp (tile rows wr0 .. wr0+RW),
  // the lane's block l of the chunk (global block index kb within the K-range).
  static __device__ __forceinline__ void chunk(const uint8_t* stage, int wr0, int nrows, int lane, int kb,
                                               const uint8_t* act_q, const float* act_d, const float* act_ds,
                                               const DenseParams& p, float (&acc)[RW][NT]) {
    constexpr int CB = chunk_bytes<F>();
    uint32_t w[RW][8];   // decoded int8 operands, paired with act words 0..7
    float sA[RW];        // per-row multiplier of d_x * isum
    float sB[RW];        // Q4_K: dmin * m (multiplier of d_x * s)
#pragma unroll
    for (int r = 0; r < RW; r++) {
      sA[r] = 0.f;
      sB[r] = 0.f;
#pragma unroll
      for (int i = 0; i < 8; i++) w[r][i] = 0;
      if (wr0 + r < nrows) {
        const uint8_t* row = stage + (wr0 + r) * CB;
        if constexpr (F == QMV_Q8_0) {
          const int g = lane >> 3, b8 = lane & 7;
          const uint8_t* grp = row + g * 272;
          uint4 a = *reinterpret_cast<const uint4*>(grp + 16 + 16 * b8);
          uint4 c = *reinterpret_cast<const uint4*>(grp + 16 + 128 + 16 * b8);
          w[r][0] = a.x; w[r][1] = a.y; w[r][2] = a.z; w[r][3] = a.w;
          w[r][4] = c.x; w[r][5] = c.y; w[r][6] = c.z; w[r][7] = c.w;
          sA[r] = __half2float(*reinterpret_cast<const __half*>(grp + 2 * b8));
        } else if constexpr (F == QMV_Q4_K) {
          const int g = lane >> 3, j = lane & 7;
          const uint8_t* grp = row + g * 144;
          uint4 h = *reinterpret_cast<const uint4*>(grp);
          uint4 q = *reinterpret_cast<const uint4*>(grp + 16 + 16 * j);
          const uint32_t qq[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
          for (int i = 0; i < 4; i++) {
            w[r][i] = qq[i] & 0x0F0F0F0Fu;
            w[r][4 + i] = (qq[i] >> 4) & 0x0F0F0F0Fu;
          }
          // 12-bit field j (sc | m << 6) of the 96-bit string in h.y..h.w
          const int bit = 12 * j;
          const uint32_t wa = bit < 32 ? h.y : (bit < 64 ? h.z : h.w);
          const uint32_t wb = bit < 32 ? h.z : (bit < 64 ? h.w : 0u);
          const uint32_t f = __funnelshift_r(wa, wb, bit & 31) & 0xFFFu;
          const float d = __half2float(__ushort_as_half((unsigned short)(h.x & 0xFFFF)));
          const float dmin = __half2float(__ushort_as_half((unsigned short)(h.x >> 16)));
          sA[r] = d * (float)(f & 63u);
          sB[r] = dmin * (float)(f >> 6);
        } else {
          const int g = lane >> 4, sb = (lane >> 3) & 1, j = lane & 7;
          const uint8_t* grp = row + g * 272;
          const uint2 meta = *reinterpret_cast<const uint2*>(grp + 8 * sb);
          const uint4 q = *reinterpret_cast<const uint4*>(grp + 16 + 128 * sb + 16 * j);
          const uint64_t m64 = ((uint64_t)meta.y << 32) | meta.x;
          const int ls = (int)((m64 >> (16 + 6 * j)) & 63u);
          const float d = __half2float(__ushort_as_half((unsigned short)(meta.x & 0xFFFF)));
          sA[r] = d * (float)(ls - 32);
          const uint32_t qq[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
          for (int i = 0; i < 4; i++) {
            const uint32_t pw = qq[i];
            const uint32_t pl = pw & 0x77777777u;
            const uint32_t p4 = pw << 4;
            w[r][2 * i] = iq4_lookup4(pl, pw, p4, 0xD9C8u);
            w[r][2 * i + 1] = iq4_lookup4(pl >> 16, pw, p4, 0xFBEAu);
          }
        }
      }
    }
    const int pos = act_pos(kb, 0);
#pragma unroll
    for (int t = 0; t < NT; t++) {
      if (t < p.nt) {
        const uint8_t* arow = act_q + t * p.act_stride;
        const uint4 xa = *reinterpret_cast<const uint4*>(arow + pos);
        const uint4 xb = *reinterpret_cast<const uint4*>(arow + pos + 128);
        const float dx = act_d[t * p.act_blk + kb];
        float dxs = 0.f;
        if constexpr (F == QMV_Q4_K) dxs = act_ds[t * p.act_blk + kb];
#pragma unroll
        for (int r = 0; r < RW; r++) {
          int is = __dp4a((int)w[r][0], (int)xa.x, 0);
          is = __dp4a((int)w[r][1], (int)xa.y, is);
          is = __dp4a((int)w[r][2], (int)xa.z, is);
          is = __dp4a((int)w[r][3], (int)xa.w, is);
          is = __dp4a((int)w[r][4], (int)xb.x, is);
          is = __dp4a((int)w[r][5], (int)xb.y, is);
          is = __dp4a((int)w[r][6], (int)xb.z, is);
          is = __dp4a((int)w[r][7], (int)xb.w, is);
          float v = acc[r][t] + (sA[r] * dx) * (float)is;
          if constexpr (F == QMV_Q4_K) v -= sB[r] * dxs;
          acc[r][t] = v;
        }
      }
    }
  }
};

// Per-CTA walk over its tiles: a contiguous range of the flattened
// (split, 8-row unit) space, cut into tiles of up to 4 units that stay inside
// one split.
struct TileWalk {
  long long f, f_end;
  int units;
  __device__ TileWalk(const DenseParams& p) {
    const long long total = (long long)p.n_split * p.units;
    f = total * blockIdx.x / gridDim.x;
    f_end = total * (blockIdx.x + 1) / gridDim.x;
    units = p.units;
  }
  // Next tile: split s, first unit u, number of units nu.
  __device__ bool next(int& s, int& u, int& nu) {
    if (f >= f_end) return false;
    s = (int)(f / units);
    u = (int)(f - (long long)s * units);
    long long lim = f_end - f;
    int rest = units - u;
    nu = (int)min((long long)min(TILE_ROWS / UNIT_ROWS, rest), lim);
    f += nu;
    return true;
  }
};

__device__ __forceinline__ void split_range(const DenseParams& p, int s, int& g0, int& g1) {
  g0 = (int)((long long)p.groups * s / p.n_split);
  g1 = (int)((long long)p.groups * (s + 1) / p.n_split);
}

template <int F, int NT>
__global__ void __launch_bounds__(THREADS, 1)
    qmv_dense_kernel(const __grid_constant__ CUtensorMap map_tile, const __grid_constant__ CUtensorMap map_unit,
                     const DenseParams p) {
  constexpr int CB = chunk_bytes<F>();
  constexpr int GW = Fmt<F>::GW, GB = Fmt<F>::GB;
  constexpr int STAGE_BYTES = TILE_ROWS * CB;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* stages = smem;
  uint8_t* act_q = stages + p.stages * STAGE_BYTES;
  float* act_d = reinterpret_cast<float*>(act_q + NT * p.act_stride);
  float* act_ds = act_d + NT * p.act_blk;
  uint64_t* full = reinterpret_cast<uint64_t*>(act_ds + NT * p.act_blk);
  uint64_t* empty = full + MAX_STAGES;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; s++) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], CONSUMER_WARPS);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == CONSUMER_WARPS) {
    // ---------------- producer ----------------
    if (lane == 0) {
      prefetch_tensormap(&map_tile);
      prefetch_tensormap(&map_unit);
      const uint64_t pol = policy_evict_first();
      pdl_wait();  // the weights may have been written by the preceding kernel
      TileWalk walk(p);
      int s, u, nu;
      long long it = 0;
      bool alive = true;
      while (alive && walk.next(s, u, nu)) {
        int g0, g1;
        split_range(p, s, g0, g1);
        const int nck = ((g1 - g0) * GW + KCHUNK - 1) / KCHUNK;
        for (int c = 0; c < nck; c++, it++) {
          const int st = (int)(it % p.stages);
          if (it >= p.stages && !mbar_wait(&empty[st], (uint32_t)(((it / p.stages) - 1) & 1), p.err)) {
            alive = false;
            break;
          }
          uint8_t* dst = stages + st * STAGE_BYTES;
          const int x = (g0 * GB + c * CB) / 8;
          if (nu == TILE_ROWS / UNIT_ROWS) {
            mbar_arrive_expect_tx(&full[st], STAGE_BYTES);
            tma_load_2d(dst, &map_tile, &full[st], x, u * UNIT_ROWS, pol);
          } else {
            mbar_arrive_expect_tx(&full[st], nu * UNIT_ROWS * CB);
            for (int i = 0; i < nu; i++)
              tma_load_2d(dst + i * UNIT_ROWS * CB, &map_unit, &full[st], x, (u + i) * UNIT_ROWS, pol);
          }
        }
      }
      // Do not leave while copies may still be landing in shared memory.
      const long long first = it > p.stages ? it - p.stages : 0;
      for (long long j = first; j < it; j++) mbar_wait(&full[j % p.stages], (uint32_t)((j / p.stages) & 1), p.err);
    }
    return;
  }

  // ---------------- consumers ----------------
  // A consumer that gives up on a wait keeps walking the tiles (without
  // waiting or computing) so that the named barriers of the others still
  // complete; the timeout bit is already set.
  pdl_wait();  // activations may come from the preceding kernel
  const int cw = warp;
  bool alive = true;
  TileWalk walk(p);
  int s, u, nu;
  long long it = 0;
  int staged_split = -1;
  float acc[RW][NT];
#pragma unroll
  for (int r = 0; r < RW; r++)
#pragma unroll
    for (int t = 0; t < NT; t++) acc[r][t] = 0.f;

  while (walk.next(s, u, nu)) {
    int g0, g1;
    split_range(p, s, g0, g1);
    const int kb0 = g0 * (GW / BLK), nblk = (g1 - g0) * (GW / BLK);
    if (s != staged_split) {
      named_sync(1, CONSUMER_THREADS);  // nobody still reads the previous range
      stage_activations<F>(p, kb0, nblk, act_q, act_d, act_ds, cw, lane);
      named_sync(1, CONSUMER_THREADS);
      staged_split = s;
    }
    const long long row0 = (long long)u * UNIT_ROWS;
    const int nrows = (int)min((long long)nu * UNIT_ROWS, p.M - row0);
    const int nck = (nblk * BLK + KCHUNK - 1) / KCHUNK;
    for (int c = 0; c < nck && alive; c++, it++) {
      const int st = (int)(it % p.stages);
      if (!mbar_wait(&full[st], (uint32_t)((it / p.stages) & 1), p.err)) {
        alive = false;
        break;
      }
      const int kb = c * (KCHUNK / BLK) + lane;
      if (cw * RW < nrows && kb < nblk)
        Consumer<F, NT>::chunk(stages + st * STAGE_BYTES, cw * RW, nrows, lane, kb, act_q, act_d, act_ds, p, acc);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    alive = __all_sync(FULL, alive);
    if (!alive) continue;
    // reduce across lanes and store rows row0 + cw*RW + r
    float* out = p.out + (long long)s * p.ntot * p.M;
#pragma unroll
    for (int r = 0; r < RW; r++) {
#pragma unroll
      for (int t = 0; t < NT; t++) {
        float v = acc[r][t];
        v += __shfl_xor_sync(FULL, v, 16);
        v += __shfl_xor_sync(FULL, v, 8);
        v += __shfl_xor_sync(FULL, v, 4);
        v += __shfl_xor_sync(FULL, v, 2);
        v += __shfl_xor_sync(FULL, v, 1);
        const int row = cw * RW + r;
        if (lane == ((r * NT + t) & 31) && t < p.nt && row < nrows)
          out[(long long)(p.t0 + t) * p.M + row0 + row] = v;
        acc[r][t] = 0.f;
      }
    }
  }
}

}  // namespace qmv
