// Dense small-batch quantized matvec (and its split-K first pass).
//
// Y[t][m] = sum_k What[m][k] * Xhat[t][k] for a few tokens t: the decode-time
// matrix-vector product over block-quantized weights ("Castagna Veloce",
// section "Kernels for the MI50": small-batch matvecs for K-quants, IQ4_XS and
// Q8_0 with a split-K variant; "Running GLM-5.3 on Two 8-GPU AMD W7900D
// Machines", section "A single decode row is not a large matrix
// multiplication": weight reads dominate).
//
// Structure (persistent CTAs; 8 consumer warps and a producer warp, or from
// 8 tokens on 12 consumer warps and a producer warpgroup that hands its
// registers to them):
//   - the producer: one elected lane streams the CTA's weight
//     tiles, TILE_ROWS rows x 1024 weights, with 2-D TMA loads into a ring of
//     shared-memory stages guarded by full/empty mbarriers.  The weights are
//     read-only inputs, so streaming starts at once, before the preceding
//     grid in the stream has finished (programmatic dependent launch);
//   - the consumer warps: wait for the preceding grid, quantize the
//     activations of the K-range into shared memory (per-32 int8, the
//     activation rule), then for every stage decode RW rows each in registers
//     (one 32-weight block per lane), form exact int32 block dot products with
//     dp4a, apply the block scales in fp32 and, at the end of a tile, reduce
//     across lanes and store.
// Work split: the (split, 8-row unit) space is cut into contiguous,
// equal-sized ranges, one per CTA; a tile never crosses a split.
#pragma once
#include "qmv_core.cuh"

namespace qmv {

struct DenseParams {
  const float* x;      // fp32 activations [ntot][K], or nullptr when pre-quantized
  const int8_t* xq;    // pre-quantized activations [ntot][K] (natural order)
  const float* xd;     // [ntot][K/32]
  const int32_t* xs;   // [ntot][K/32]
  float* out;          // y [ntot][M] (n_split == 1) or partial [n_split][ntot][M]
  const float* add;    // n_split == 1: added to y after the dot product ([ntot][M], may be out), or nullptr
  long long M;
  int K;               // weights per row
  int ntot;            // tokens held by x / out
  int t0;              // first token of this launch's first pass (blockIdx.y: pass of NT tokens)
  int nt;              // tokens of every pass of this launch (<= NT)
  int n_split;
  int groups;          // K / group weights
  int units;           // ceil(M / UNIT_ROWS)
  int stages;
  int act_nck;         // chunks of the activation area
  int prefetch;        // L2 lookahead of the producer past the ring (iterations; 0: none)
  unsigned* err;       // device error word
  // used by the tensor-core kernel (qmv_mma.cuh), which copies rows itself
  const uint8_t* w;    // the weight rows
  long long rb;        // bytes per row
  int nbmax;           // blocks of the longest split range
  // QMV_DEBUG builds: extents of the caller's buffers (elements), derived on
  // the host from the call's arguments, for the range checks
  QMV_DEBUG_ONLY(long long x_len;    // x or xq: ntot * K
                 long long out_len;  // out: ntot * M, or n_split * ntot * M
                 long long add_len;) // add: ntot * M (0 without add)
};

// Per-CTA walk over its tiles: a contiguous range of the flattened
// (split, 8-row unit) space, cut into tiles of up to TU units that stay
// inside one split.
template <int TU>
struct TileWalk {
  long long f, f_end;
  int units, s, u;  // split and unit at f
  __device__ TileWalk(const DenseParams& p) {
    const long long total = (long long)p.n_split * p.units;
    f = total * blockIdx.x / gridDim.x;
    f_end = total * (blockIdx.x + 1) / gridDim.x;
    units = p.units;
    s = (int)(f / units);
    u = (int)(f - (long long)s * units);
  }
  // Next tile: split ts, first unit tu, number of units nu.
  __device__ bool next(int& ts, int& tu, int& nu) {
    if (f >= f_end) return false;
    ts = s;
    tu = u;
    const long long lim = f_end - f;
    const int rest = units - u;
    nu = (int)min((long long)min(TU, rest), lim);
    f += nu;
    u += nu;
    if (u == units) {
      u = 0;
      s++;
    }
    return true;
  }
};

// Groups [g0, g1) of split s (groups * n_split <= 2^20: K <= 2^20, n_split <= 256).
__device__ __forceinline__ void split_range(const DenseParams& p, int s, int& g0, int& g1) {
  if (p.n_split == 1) {
    g0 = 0;
    g1 = p.groups;
  } else {
    g0 = p.groups * s / p.n_split;
    g1 = p.groups * (s + 1) / p.n_split;
  }
}

// Consumer warps of the dense kernel (CW): from 8 tokens on the warps are
// register-bound (the accumulators of 4 rows x NT tokens), and twelve of
// them (three per scheduler) hide more latency than eight, where their
// larger tiles leave room for a ring of weight stages.

// Q8IN: the activations come pre-quantized (bulk copies) instead of as fp32
// rows quantized while staging; separate instantiations, so each kernel
// carries only its own staging code.
// ADD: the residual of p.add is added at the store (separate instantiations,
// so the plain matvec carries none of its code).
template <int F, int NT, bool Q8IN, int CW, bool ADD>
__global__ void __launch_bounds__(Shape<CW>::THREADS, is_float(F) ? 1 : dense_min_blocks<NT, CW>())
    qmv_dense_kernel(const __grid_constant__ CUtensorMap map_tile, const __grid_constant__ CUtensorMap map_unit,
                     const DenseParams p) {
  using SH = Shape<CW>;
  constexpr int TILE_ROWS = SH::TILE_ROWS, TU = TILE_ROWS / UNIT_ROWS, CONSUMER_THREADS = SH::CONSUMER_THREADS;
  constexpr int CB = chunk_bytes<F>(), KC = kchunk_of(F), ACTB = act_chunk_bytes(F);
  constexpr int GW = Fmt<F>::GW, GB = Fmt<F>::GB;
  constexpr int STAGE_BYTES = TILE_ROWS * CB;
  static_assert(!is_float(F) || !Q8IN, "F16 / F32 rows take fp32 activations");
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* stages = smem;
  ActArea a;
  a.carve(stages + p.stages * STAGE_BYTES, F, NT, p.act_nck);
  uint64_t* full = reinterpret_cast<uint64_t*>(stages + p.stages * STAGE_BYTES + act_area_bytes(F, NT, p.act_nck));
  uint64_t* empty = full + MAX_STAGES;
  uint64_t* abar = full + 2 * MAX_STAGES;  // [0] bulk copies of pre-quantized activations, [1] first staging done
  float* red = reinterpret_cast<float*>(abar + 2);  // [CW][RW * NT]: cross-warp sums of thin tiles

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(abar, 1);
    mbar_init(abar + 1, 1);
  }
  init_pipeline(full, empty, p.stages, CW);
  pdl_launch_dependents();

  if (warp >= CW) {
    // ---------------- producer ----------------
    if constexpr (SH::RESPLIT) regs_dec<SH::REG_PRODUCER>();
    if (warp == CW && lane == 0) {
      prefetch_tensormap(&map_tile);
      prefetch_tensormap(&map_unit);
      const uint64_t pol = policy_evict_first();
      // The ring alone keeps enough bytes in flight: a deeper L2 lookahead
      // only queues weight reads ahead of the activation reads at the start
      // of the call, which sit on the critical path.  For the same reason,
      // with pre-quantized activations (whose bulk copies are then the
      // critical path) only GATE stages are requested before the consumers
      // have staged them.  Only small matrices (p.prefetch > 0: a few
      // microseconds of HBM time in all) have their tiles past the ring
      // requested into L2 at once, so that the last ones do not wait for a
      // free stage at the end of a short call.
      constexpr long long GATE = Q8IN ? 2 : -1;
      struct Cursor {
        TileWalk<TU> w;
        int s, u, nu, g0, g1, nck, c;
        bool valid;
        __device__ Cursor(const DenseParams& p) : w(p), c(0) { load(p); }
        __device__ void load(const DenseParams& p) {
          valid = w.next(s, u, nu);
          if (valid) {
            split_range(p, s, g0, g1);
            nck = ((g1 - g0) * GW + KC - 1) / KC;
          }
          c = 0;
        }
        __device__ void advance(const DenseParams& p) {
          if (++c == nck) load(p);
        }
      } pf(p);
      long long pf_n = 0;
      auto prefetch_to = [&](long long target) {
        for (; pf.valid && pf_n < target; pf_n++, pf.advance(p)) {
          if (pf_n < p.stages) continue;  // these go straight to shared memory
          const int x = (pf.g0 * GB + pf.c * CB) / 8;
          if (pf.nu == TU)
            tma_prefetch_2d(&map_tile, x, pf.u * UNIT_ROWS);
          else
            for (int i = 0; i < pf.nu; i++) tma_prefetch_2d(&map_unit, x, (pf.u + i) * UNIT_ROWS);
        }
      };
      TileWalk<TU> walk(p);
      int s, u, nu;
      Ring ring;
      bool alive = true;
      while (alive && walk.next(s, u, nu)) {
        int g0, g1;
        split_range(p, s, g0, g1);
        const int nck = ((g1 - g0) * GW + KC - 1) / KC;
        for (int c = 0; c < nck; c++, ring.advance(p.stages)) {
          if (p.prefetch > 0 && ring.n >= p.stages) prefetch_to(ring.n + p.prefetch);
          if (ring.n == GATE && !mbar_wait(abar + 1, 0, p.err)) {
            alive = false;
            break;
          }
          if (!producer_acquire(empty, ring, p.stages, p.err)) {
            alive = false;
            break;
          }
          const int st = ring.st;
          uint8_t* dst = stages + st * STAGE_BYTES;
          const int x = (g0 * GB + c * CB) / 8;
          if (!QMV_CHECK(smem_in_range(dst, nu * UNIT_ROWS * CB, p.err))) {
            mbar_arrive(&full[st]);  // skipped: the stage completes without data
          } else if (nu == TU) {
            mbar_arrive_expect_tx(&full[st], STAGE_BYTES);
            tma_load_2d(dst, &map_tile, &full[st], x, u * UNIT_ROWS, pol);
          } else {
            mbar_arrive_expect_tx(&full[st], nu * UNIT_ROWS * CB);
            for (int i = 0; i < nu; i++)
              tma_load_2d(dst + i * UNIT_ROWS * CB, &map_unit, &full[st], x, (u + i) * UNIT_ROWS, pol);
          }
        }
      }
      producer_drain(full, ring.n, p.stages, p.err);
    }
    return;
  }

  // ---------------- consumers ----------------
  // A consumer that gives up on a wait keeps walking the tiles (without
  // waiting or computing) so that the named barriers of the others still
  // complete; the timeout bit is already set.
  if constexpr (SH::RESPLIT) regs_inc<SH::REG_CONSUMER>();
  const int cw = warp;
  bool alive = true;
  TileWalk<TU> walk(p);
  int s, u, nu;
  Ring ring;
  int staged_split = -1;
  const ConsumerOf<F, NT> cons(lane);
  const uint32_t stage_base = smem_u32(stages), aq_base = smem_u32(a.q), ad_base = smem_u32(a.d),
                 as_base = smem_u32(a.s);
  // token pass blockIdx.y: tokens t0 .. t0 + ntk - 1 of the call
  const int t0 = p.t0 + blockIdx.y * NT, ntk = p.nt;
  const ActSource src{p.x, p.xq, p.xd, p.xs, p.K, nullptr, t0, nullptr, nullptr, nullptr
                          QMV_DEBUG_ONLY(, p.x_len, 0, p.err)};
  uint32_t aphase = 0;
  // the activations may come from the preceding kernel: wait for it only
  // now, so that the set-up above (which reads parameters only) runs while
  // it finishes
  pdl_wait();

  while (walk.next(s, u, nu)) {
    int g0, g1;
    split_range(p, s, g0, g1);
    const int kb0 = g0 * (GW / BLK), nblk = (g1 - g0) * (GW / BLK);
    if (s != staged_split) {
      if (staged_split >= 0) named_sync(1, CONSUMER_THREADS);  // nobody still reads the previous range
      if constexpr (is_float(F)) {
        stage_float<F, NT, CW>(src, (long long)kb0 * BLK, nblk * BLK, ntk, a, cw, lane);
      } else if constexpr (!Q8IN) {
        // one token: two units of 8 blocks per warp step, so that its row
        // spreads over more warps (IQ4_XS 6144 x 2048: 4.58 -> 4.18 us)
        stage_activations<F, NT, (NT >= 8 ? 8 : NT == 1 ? 2 : 4), CW>(src, kb0, nblk, ntk, a, cw, lane);
      } else {
        alive = __all_sync(FULL, stage_q8_bulk<F, NT, CW>(src, kb0, nblk, ntk, a, abar, aphase, p.err, cw, lane)) &&
                alive;
        aphase ^= 1;
      }
      named_sync(1, CONSUMER_THREADS);
      if (threadIdx.x == 0 && staged_split < 0) mbar_arrive(abar + 1);  // the producer may go on
      staged_split = s;
    }
    const long long row0 = (long long)u * UNIT_ROWS;
    const int nrows = (int)min((long long)nu * UNIT_ROWS, p.M - row0);
    const int nck = (nblk * BLK + KC - 1) / KC;
    AccTile<NT> acc;  // zeroed per tile: no accumulator is live while staging
    acc.zero();
    // Thin tiles (a few units) would leave most warps without rows: there
    // the tile's 2 * nu row groups of RW rows are each taken by ks warps
    // (the most of 4, 2, 1 that the warps cover), warp part k working on the
    // chunks c with c mod ks == k, and the parts are added across warps (in
    // part order) before the store.
    const int ks = 8 * nu <= CW ? 4 : (4 * nu <= CW ? 2 : 1);
    const int rg = CW / ks;  // warps per part (row groups with rows: 2 * nu <= rg)
    const int grp = cw % rg, part = cw / rg;
    // residual add: the values this warp adds at the store are requested
    // into L1 now, so the store does not wait for them
    if constexpr (ADD)
      if (part == 0 && lane < ntk && grp * RW < nrows &&
          QMV_CHECK(in_range((long long)(t0 + lane) * p.M + row0 + grp * RW, 1, p.add_len, p.err)))
        asm volatile("prefetch.global.L1 [%0];" ::"l"(p.add + (long long)(t0 + lane) * p.M + row0 + grp * RW));
    for (int c = 0; c < nck && alive; c++, ring.advance(p.stages)) {
      const int st = ring.st;
      if (!mbar_wait(&full[st], ring.parity(), p.err)) {
        alive = false;
        break;
      }
      if (grp * RW < nrows && (c & (ks - 1)) == part &&  // ks is 1, 2 or 4
          QMV_CHECK(chunk_reads_in_range<F, NT>(stage_base + st * STAGE_BYTES + grp * RW * CB, RW * CB,
                                      aq_base + c * NT * ACTB, ad_base + c * NT * 128, as_base + c * NT * 128,
                                      p.err)))
        cons.chunk(stage_base + st * STAGE_BYTES + grp * RW * CB, aq_base + c * NT * ACTB,
                   ad_base + c * NT * 128, as_base + c * NT * 128, ntk, acc);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    alive = __all_sync(FULL, alive);
    if (!alive) {
      // a warp that gave up on a wait stores nothing, but still takes part
      // in the cross-warp barriers of a thin tile
      if (ks > 1) {
        named_sync(2, CONSUMER_THREADS);
        named_sync(2, CONSUMER_THREADS);
      }
      continue;
    }
    // reduce across lanes and store rows row0 + grp * RW + r
    float* out = p.out + (long long)s * p.ntot * p.M;
    constexpr int V = RW * NT, HELD = V >= 32 ? V / 32 : 1;
    float v[V];
    int idx = 0;
    bool lead;  // this lane holds sums idx .. idx + HELD - 1 (V >= 32: all lanes)
    if constexpr (NT <= 2) {
      // few values per lane: one shuffle tree each; lane o keeps sum o
#pragma unroll
      for (int r = 0; r < RW; r++)
#pragma unroll
        for (int t = 0; t < NT; t++) {
          const float w = warp_sum(acc.get(r, t));
          if (lane == r * NT + t) v[0] = w;
        }
      idx = lane;
      lead = lane < V;
    } else {
#pragma unroll
      for (int r = 0; r < RW; r++)
#pragma unroll
        for (int t = 0; t < NT; t++) v[r * NT + t] = acc.get(r, t);
      LaneButterfly<V, 0>::run(v, lane, idx);
      lead = V >= 32 || (lane & (32 / V - 1)) == 0;
    }
    acc.zero();
    if (ks > 1) {
      if (lead)
#pragma unroll
        for (int i = 0; i < HELD; i++)
          if (QMV_CHECK(smem_in_range(red + cw * V + idx + i, 4, p.err))) red[cw * V + idx + i] = v[i];
      named_sync(2, CONSUMER_THREADS);
      if (part == 0 && lead)
#pragma unroll
        for (int i = 0; i < HELD; i++) {
          float w = QMV_CHECK(smem_in_range(red + grp * V + idx + i, 4, p.err)) ? red[grp * V + idx + i] : 0.f;
          for (int k = 1; k < ks; k++)
            if (QMV_CHECK(smem_in_range(red + (k * rg + grp) * V + idx + i, 4, p.err))) w += red[(k * rg + grp) * V + idx + i];
          v[i] = w;
        }
      named_sync(2, CONSUMER_THREADS);  // red is free for the next tile
    }
    if (part == 0 && lead) {
#pragma unroll
      for (int i = 0; i < HELD; i++) {
        const int o = idx + i, r = o / NT, t = o - r * NT, row = grp * RW + r;
        if (t < ntk && row < nrows) {
          const long long o = (long long)(t0 + t) * p.M + row0 + row;
          if (!QMV_CHECK(in_range((long long)s * p.ntot * p.M + o, 1, p.out_len, p.err))) continue;
          if constexpr (ADD)
            out[o] = v[i] + (QMV_CHECK(in_range(o, 1, p.add_len, p.err)) ? p.add[o] : 0.f);
          else
            out[o] = v[i];
        }
      }
    }
  }
}

}  // namespace qmv
