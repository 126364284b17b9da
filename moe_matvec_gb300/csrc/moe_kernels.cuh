// Expert-grouped MoE decode kernels.
//
// One MoE FFN layer for a batch of up to 64 tokens, each routed to top_k
// experts ("Castagna Veloce", section "Kernels for the MI50": i-quant MoE
// decode kernels for batches of up to 64 tokens and the expert-grouped
// quantized MoE scheme; section "Fused operations": gate/up + SwiGLU):
//   kernel GATE_UP: for every routed expert, stream its gate and up rows once
//     and, for all tokens routed to it, g = Wgate x, u = Wup x,
//     h = silu(g) * u  (SwiGLU in the epilogue, fp32);
//   kernel DOWN:   for every routed expert, quantize its tokens' h by the
//     activation rule while staging (writing q8(h) back to the workspace) and
//     stream its down rows once: o = Wdown h;
//   kernel COMBINE: y[t] = sum_k gates[t][k] * o[t, k], added in k order.
// Expert grouping: every CTA rebuilds the groups from ids in its prologue
// (at most 512 slots): a 64-bit mask of the tokens routed to each expert
// gives each slot its rank within the expert, so the slot lists come out in
// token order without sorting, identically in every CTA.  Work is the
// flattened (expert group, 8-row unit) space, split evenly over persistent
// CTAs; a tile stays inside one expert group, whose activations are staged
// once per CTA.
#pragma once
#include "qmv_core.cuh"

namespace qmv {

constexpr int MOE_MAX_EXPERTS = 512;
constexpr int MOE_MAX_SLOTS = QMV_MAX_TOKENS * QMV_MAX_TOPK;  // 512
constexpr int MOE_GATE_UP = 0, MOE_DOWN = 1;

struct MoeParams {
  const int32_t* ids;   // [n_tok][top_k]
  const float* src;     // GATE_UP: x [n_tok][K]; DOWN: h [S][K]
  float* dst;           // GATE_UP: h [S][R];     DOWN: o [S][R]
  int8_t* hq;           // DOWN: write-back of the quantized h [S][K]
  float* hd;            // [S][K/32]
  int32_t* hs;          // [S][K/32]
  int n_tok, top_k, n_experts;
  int K;                // reduction length (hidden for GATE_UP, ffn for DOWN)
  int R;                // outputs per expert (ffn for GATE_UP, hidden for DOWN)
  int pool_rows;        // rows per expert in the weight pool (2*ffn or hidden)
  int groups;           // K / group weights
  int stages, act_nck;
  unsigned* err;
  // QMV_DEBUG builds: extents of the buffers (elements), derived on the host
  // from the call's arguments, for the range checks
  QMV_DEBUG_ONLY(long long ids_len;  // ids: n_tok * top_k
                 long long src_len;  // GATE_UP x: n_tok * K; DOWN h: S * K
                 long long dst_len;  // S * R
                 long long hq_len;)  // DOWN: S * K (0 for GATE_UP)
};

// Expert groups of one launch, in shared memory.
struct MoeRouting {
  int ids[MOE_MAX_SLOTS];                    // copy of the launch's ids
  unsigned long long mask[MOE_MAX_EXPERTS];  // tokens routed to each expert
  int off[MOE_MAX_EXPERTS];                  // first slot-list index of each expert
  int slots[MOE_MAX_SLOTS];                  // slots (t * top_k + k), grouped by expert, in token order
  int pair_expert[MOE_MAX_SLOTS];            // per (expert, token group)
  int pair_first[MOE_MAX_SLOTS];
  int pair_count[MOE_MAX_SLOTS];
  int pair_cost[MOE_MAX_SLOTS + 1];          // prefix sums of the groups' work weights
                                             // (< 512 x 2^17 units x 22 < 2^31)
  int wsum[32][3];                           // per-warp totals of the expert scan
  int n_pairs;
};

// A slot routes when its id lies in [0, E) and does not repeat an earlier id
// of the same token.
__device__ __forceinline__ int slot_status(const int32_t* ids, int top_k, int E, int p) {
  const int t = p / top_k, k = p - t * top_k;
  const int e = ids[p];
  if (e < 0 || e >= E) return QMV_DEVERR_EXPERT_RANGE;
  for (int kk = 0; kk < k; kk++)
    if (ids[t * top_k + kk] == e) return QMV_DEVERR_EXPERT_DUP;
  return 0;
}

// Work weight of a group of c token slots per 8-row unit: its decode
// (unit_base) plus one per token slot it computes (slots go in pairs from
// two on).
__device__ __forceinline__ int group_weight(int c, int nt_group, int unit_base) {
  return unit_base + (nt_group >= 2 ? (c + 1) & ~1 : c);
}

// The expert groups of a launch with at most 32 slots, built by warp 0 alone
// in registers while the other warps wait at the closing barrier: lane s
// holds slot s as a key (expert, token, slot), a bitonic sort across the
// lanes puts the routed slots in (expert, token) order, which is the slot
// list, and ballots, bit scans and one warp scan give every group (expert,
// first slot, slot count) and its work prefix.  The tables are the general
// build's, with a short chain of shuffles in place of its shared-memory
// atomics and barriers, which cost about a microsecond per step beside a
// decoding CTA on the same SM.
__device__ __forceinline__ void build_routing_small(MoeRouting& rt, const MoeParams& p, int nt_group, bool report,
                                                    int unit_base, int units_per_pair) {
  const int S = p.n_tok * p.top_k, E = p.n_experts;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int t = lane / p.top_k, k = lane - t * p.top_k;
    int e = -1;
    if (lane < S && QMV_CHECK(in_range(lane, 1, p.ids_len, p.err))) e = p.ids[lane];
    // the slot does not route when its id is out of range or repeats an
    // earlier id of the same token (lanes t top_k .. lane - 1)
    bool dup = false;
#pragma unroll
    for (int kk = 1; kk < QMV_MAX_TOPK; kk++) {
      const int o = __shfl_up_sync(FULL, e, kk);
      dup = dup || (kk <= k && o == e);
    }
    const int st = lane >= S ? 0 : (e < 0 || e >= E ? QMV_DEVERR_EXPERT_RANGE : (dup ? QMV_DEVERR_EXPERT_DUP : 0));
    if (report && st) set_error(p.err, (unsigned)st);
    // key: expert (9 bits), token (6 bits), slot (9 bits); slots that do
    // not route sort last
    unsigned key = lane < S && st == 0 ? ((unsigned)e << 15) | ((unsigned)t << 9) | (unsigned)lane : 0xFFFFFFFFu;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        const unsigned other = __shfl_xor_sync(FULL, key, stride);
        const bool up = (lane & size) == 0, lower = (lane & stride) == 0;
        key = up == lower ? min(key, other) : max(key, other);
      }
    const int V = __popc(__ballot_sync(FULL, key != 0xFFFFFFFFu));  // routed slots: lanes 0 .. V - 1
    const bool have = lane < V;
    const int se = (int)(key >> 15);
    if (have && QMV_CHECK(in_array(rt.slots, lane, p.err))) rt.slots[lane] = (int)(key & 511u);
    // runs of equal experts, cut into groups of up to nt_group slots
    const int prev = __shfl_up_sync(FULL, se, 1);
    const unsigned starts = __ballot_sync(FULL, have && (lane == 0 || prev != se));
    const unsigned upto = 0xFFFFFFFFu >> (31 - lane);  // bits 0 .. lane
    const int rs = 31 - __clz(starts & upto);          // the run's first lane
    const unsigned later = starts & ~upto;
    const int re = later ? __ffs(later) - 1 : V;       // the lane past the run
    const bool begins = have && ((lane - rs) & (nt_group - 1)) == 0;
    const int cnt = min(nt_group, re - lane);
    const unsigned bmask = __ballot_sync(FULL, begins);
    const int w = begins ? group_weight(cnt, nt_group, unit_base) * units_per_pair : 0;
    int incl = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(FULL, incl, o);
      if (lane >= o) incl += a;
    }
    const int pi = __popc(bmask & ((1u << lane) - 1u));
    if (begins && QMV_CHECK(in_array(rt.pair_expert, pi, p.err))) {
      rt.pair_expert[pi] = se;
      rt.pair_first[pi] = lane;
      rt.pair_count[pi] = cnt;
      rt.pair_cost[pi] = incl - w;
    }
    const int total = __shfl_sync(FULL, incl, 31);
    if (lane == 0) {
      rt.n_pairs = __popc(bmask);
      rt.pair_cost[__popc(bmask)] = total;
    }
  }
  __syncthreads();
}

// Build the expert groups (called by all threads of the CTA).  The experts
// are scanned in rounds of (warps x 32): each warp scans its 32 experts'
// slot, group and work counts with shuffles, the warps' totals go through
// shared memory, and every expert then writes its slot offset and its
// groups (expert, first slot, slot count, work prefix).
__device__ __forceinline__ void build_routing(MoeRouting& rt, const MoeParams& p, int nt_group, bool report,
                                              int unit_base, int units_per_pair) {
  const int S = p.n_tok * p.top_k;
  if (S <= 32) {
    build_routing_small(rt, p, nt_group, report, unit_base, units_per_pair);
    return;
  }
  const int E = p.n_experts;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  // one coalesced read of ids; every later look-up is in shared memory
  for (int s = threadIdx.x; s < S; s += blockDim.x)
    rt.ids[s] = QMV_CHECK(in_array(rt.ids, s, p.err)) && QMV_CHECK(in_range(s, 1, p.ids_len, p.err)) ? p.ids[s] : -1;
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    if (QMV_CHECK(in_array(rt.mask, e, p.err))) rt.mask[e] = 0ull;
  __syncthreads();
  for (int s = threadIdx.x; s < S; s += blockDim.x) {
    const int st = slot_status(rt.ids, p.top_k, E, s);
    if (st == 0) {
      if (QMV_CHECK(in_array(rt.mask, rt.ids[s], p.err))) atomicOr(&rt.mask[rt.ids[s]], 1ull << (s / p.top_k));
    } else if (report) {
      set_error(p.err, (unsigned)st);
    }
  }
  __syncthreads();
  int carry_s = 0, carry_p = 0, carry_w = 0;  // the same in every thread
  for (int base = 0; base < E; base += nwarps * 32) {
    const int e = base + warp * 32 + lane;
    const int c = e < E && QMV_CHECK(in_array(rt.mask, e, p.err)) ? __popcll(rt.mask[e]) : 0;
    const int ng = (c + nt_group - 1) / nt_group;
    // work of the expert's groups: ng - 1 full ones and the rest
    const int w = ng == 0 ? 0
                          : ((ng - 1) * group_weight(nt_group, nt_group, unit_base) +
                             group_weight(c - (ng - 1) * nt_group, nt_group, unit_base)) *
                                units_per_pair;
    int cs = c, cp = ng, cw = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(FULL, cs, o), b = __shfl_up_sync(FULL, cp, o), d = __shfl_up_sync(FULL, cw, o);
      if (lane >= o) {
        cs += a;
        cp += b;
        cw += d;
      }
    }
    if (lane == 31 && QMV_CHECK(in_array(rt.wsum, warp, p.err))) {
      rt.wsum[warp][0] = cs;
      rt.wsum[warp][1] = cp;
      rt.wsum[warp][2] = cw;
    }
    __syncthreads();
    int ps = carry_s, pp = carry_p, pw = carry_w;  // before this warp's experts
    for (int v = 0; v < nwarps; v++) {
      const int ts = rt.wsum[v][0], tp = rt.wsum[v][1], tw = rt.wsum[v][2];
      if (v < warp) {
        ps += ts;
        pp += tp;
        pw += tw;
      }
      carry_s += ts;
      carry_p += tp;
      carry_w += tw;
    }
    if (e < E && QMV_CHECK(in_array(rt.off, e, p.err))) {
      const int off = ps + cs - c, poff = pp + cp - ng;
      int wacc = pw + cw - w;
      rt.off[e] = off;
      for (int g = 0; g < ng; g++) {
        const int cg = min(nt_group, c - g * nt_group);
        if (!QMV_CHECK(in_array(rt.pair_expert, poff + g, p.err))) continue;
        rt.pair_expert[poff + g] = e;
        rt.pair_first[poff + g] = off + g * nt_group;
        rt.pair_count[poff + g] = cg;
        rt.pair_cost[poff + g] = wacc;
        wacc += group_weight(cg, nt_group, unit_base) * units_per_pair;
      }
    }
    __syncthreads();  // wsum is read before the next round writes it
  }
  if (threadIdx.x == 0) {
    // every index the walk reads (pair_cost[0 .. n_pairs]) is at most n_pairs
    rt.n_pairs = QMV_CHECK(in_array(rt.pair_cost, carry_p, p.err)) ? carry_p : 0;
    if (QMV_CHECK(in_array(rt.pair_cost, carry_p, p.err))) rt.pair_cost[carry_p] = carry_w;
  }
  for (int s = threadIdx.x; s < S; s += blockDim.x) {
    if (slot_status(rt.ids, p.top_k, E, s) == 0) {
      const int e = rt.ids[s], t = s / p.top_k;
      const int rank = __popcll(rt.mask[e] & ((1ull << t) - 1ull));
      if (QMV_CHECK(in_array(rt.slots, rt.off[e] + rank, p.err))) rt.slots[rt.off[e] + rank] = s;
    }
  }
  __syncthreads();
}

// Walk over this CTA's part of the flattened (pair, unit) space.  The parts
// are cut by work, not by units: a unit of a group that computes more token
// slots weighs more (pair_cost), so CTAs end together.  A cut at work
// position P falls on the first unit that starts at or after P; every CTA
// computes the same cuts.
struct MoeWalk {
  long long f, f_end;
  int units, tile_units, q, u;  // pair and unit at f
  __device__ static long long locate(const MoeRouting& rt, int units, long long P) {
    int lo = 0, hi = rt.n_pairs;  // pair lo with pair_cost[lo] <= P < pair_cost[lo + 1]
    if (P >= rt.pair_cost[hi]) return (long long)hi * units;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (rt.pair_cost[mid] <= P)
        lo = mid;
      else
        hi = mid;
    }
    const long long d = P - rt.pair_cost[lo];
    const long long w = (rt.pair_cost[lo + 1] - rt.pair_cost[lo]) / units;  // weight of one unit
    const long long uu = w < (1ll << 31) && d < (1ll << 31) ? (long long)(((unsigned)d + (unsigned)w - 1u) / (unsigned)w)
                                                           : (d + w - 1) / w;
    return (long long)lo * units + uu;
  }
  __device__ MoeWalk(const MoeRouting& rt, int units_per_pair, int tile_units_) {
    const unsigned C = (unsigned)rt.pair_cost[rt.n_pairs];  // < 2^31
    units = units_per_pair;
    tile_units = tile_units_;
    const unsigned G = gridDim.x, b = blockIdx.x;
    // C * b / G exactly in 32-bit arithmetic: C = cq G + cr, so C b / G =
    // cq b + (cr b) / G with cr b < G^2
    const unsigned cq = C / G, cr = C - cq * G;
    const long long P0 = (long long)(cq * b + (cr * b) / G);
    const long long P1 = (long long)(cq * (b + 1) + (cr * (b + 1)) / G);
    f = locate(rt, units, P0);
    f_end = locate(rt, units, P1);
    q = (int)(f / units);
    u = (int)(f - (long long)q * units);
  }
  __device__ bool next(int& tq, int& tu, int& nu) {
    if (f >= f_end) return false;
    tq = q;
    tu = u;
    const long long lim = f_end - f;
    nu = (int)min((long long)min(tile_units, units - u), lim);
    f += nu;
    u += nu;
    if (u == units) {
      u = 0;
      q++;
    }
    return true;
  }
};

template <int F, int NT, int MODE, int CW>
__global__ void __launch_bounds__(Shape<CW>::THREADS, NT <= 4 && CW == CONSUMER_WARPS ? 2 : 1)
    moe_qmv_kernel(const __grid_constant__ CUtensorMap map_tile, const __grid_constant__ CUtensorMap map_unit,
                   const MoeParams p) {
  using SH = Shape<CW>;
  constexpr int CB = chunk_bytes<F>();
  constexpr int STAGE_BYTES = SH::TILE_ROWS * CB, CONSUMER_THREADS = SH::CONSUMER_THREADS;
  // GATE_UP: a tile is up to CW / 4 units of 8 outputs j: gate rows j in
  // stage rows 0 .. HALF - 1, up rows j in stage rows HALF .. 2 HALF - 1
  // (HALF = 2 CW); warp w takes outputs j0 + 2w and j0 + 2w + 1 (stage rows
  // 2w, 2w+1 and HALF+2w, HALF+2w+1).
  // DOWN: a tile is up to CW / 2 units of 8 rows; warp w takes rows 4w .. 4w+3.
  constexpr int TILE_UNITS = MODE == MOE_GATE_UP ? CW / 4 : CW / 2;
  constexpr int HALF = 2 * CW;
  __shared__ MoeRouting rt;
  __shared__ int s_rows[16];
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* stages = smem;
  ActArea a;
  a.carve(stages + p.stages * STAGE_BYTES, F, NT, p.act_nck);
  uint64_t* full = reinterpret_cast<uint64_t*>(stages + p.stages * STAGE_BYTES + act_area_bytes(F, NT, p.act_nck));
  uint64_t* empty = full + MAX_STAGES;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  init_pipeline(full, empty, p.stages, CW);
  // GATE_UP reads ids, which the preceding kernel may produce, so it waits
  // before routing and only then lets the next kernel launch; DOWN launches
  // after every GATE_UP CTA passed that wait, so its ids are complete.
  if (MODE == MOE_GATE_UP) pdl_wait();
  pdl_launch_dependents();
  const int units_per_pair = p.R / UNIT_ROWS;
  // decode work of one unit relative to one token slot of it
  constexpr int UNIT_BASE = F == QMV_IQ4_XS ? 6 : (F == QMV_Q4_K ? 2 : 1);
  build_routing(rt, p, NT, MODE == MOE_GATE_UP && blockIdx.x == 0, UNIT_BASE, units_per_pair);
  const int nck = (p.K + KCHUNK - 1) / KCHUNK;

  if (warp >= CW) {
    // ---------------- producer ----------------
    if constexpr (SH::RESPLIT) regs_dec<SH::REG_PRODUCER>();
    if (warp == CW && lane == 0) {
      prefetch_tensormap(&map_tile);
      prefetch_tensormap(&map_unit);
      const uint64_t pol = policy_evict_first();
      // No L2 lookahead past the ring: it would queue expert rows ahead of
      // the activation reads on the critical path (see the dense kernel).
      MoeWalk walk(rt, units_per_pair, TILE_UNITS);
      int q, u, nu;
      Ring ring;
      bool alive = true;
      while (alive && walk.next(q, u, nu)) {
        const int base = (QMV_CHECK(in_array(rt.pair_expert, q, p.err)) ? rt.pair_expert[q] : 0) * p.pool_rows;
        for (int c = 0; c < nck; c++, ring.advance(p.stages)) {
          if (!producer_acquire(empty, ring, p.stages, p.err)) {
            alive = false;
            break;
          }
          const int st = ring.st;
          uint8_t* dst = stages + st * STAGE_BYTES;
          const int x = c * CB / 8;
          if (!QMV_CHECK(smem_in_range(dst, MODE == MOE_GATE_UP ? (HALF + nu * UNIT_ROWS) * CB : nu * UNIT_ROWS * CB, p.err))) {
            mbar_arrive(&full[st]);  // skipped: the stage completes without data
          } else if constexpr (MODE == MOE_GATE_UP) {
            mbar_arrive_expect_tx(&full[st], 2 * nu * UNIT_ROWS * CB);
            for (int i = 0; i < nu; i++) {
              const int j = (u + i) * UNIT_ROWS;
              tma_load_2d(dst + i * UNIT_ROWS * CB, &map_unit, &full[st], x, base + j, pol);
              tma_load_2d(dst + (HALF + i * UNIT_ROWS) * CB, &map_unit, &full[st], x, base + p.R + j, pol);
            }
          } else {
            if (nu == TILE_UNITS) {
              mbar_arrive_expect_tx(&full[st], STAGE_BYTES);
              tma_load_2d(dst, &map_tile, &full[st], x, base + u * UNIT_ROWS, pol);
            } else {
              mbar_arrive_expect_tx(&full[st], nu * UNIT_ROWS * CB);
              for (int i = 0; i < nu; i++)
                tma_load_2d(dst + i * UNIT_ROWS * CB, &map_unit, &full[st], x, base + (u + i) * UNIT_ROWS, pol);
            }
          }
        }
      }
      producer_drain(full, ring.n, p.stages, p.err);
    }
    return;
  }

  // ---------------- consumers ----------------
  if constexpr (SH::RESPLIT) regs_inc<SH::REG_CONSUMER>();
  const int cw = warp;
  bool alive = true;
  MoeWalk walk(rt, units_per_pair, TILE_UNITS);
  int q, u, nu;
  Ring ring;
  int staged_pair = -1, nt = 0, first = 0;
  const Consumer<F, NT> cons(lane);
  AccTile<NT> acc;
  acc.zero();
  const uint32_t stage_base = smem_u32(stages), aq_base = smem_u32(a.q), ad_base = smem_u32(a.d),
                 as_base = smem_u32(a.s);
  int roff[RW];  // stage row of each of the warp's rows
  if constexpr (MODE == MOE_GATE_UP) {
    roff[0] = 2 * cw;
    roff[1] = 2 * cw + 1;
    roff[2] = HALF + 2 * cw;
    roff[3] = HALF + 1 + 2 * cw;
  } else {
#pragma unroll
    for (int r = 0; r < RW; r++) roff[r] = cw * RW + r;
  }
  const int nblk = p.K / BLK;
  // rows whose length is 512 past a multiple of 1024 (the down projection of
  // an FFN of 1536) end in a half chunk; the tiles of 8 and 16 tokens split it
  // between lane pairs (at fewer tokens the extra code spills registers and
  // costs more than the zero fill it saves)
  const bool half_last = NT >= 8 && p.K % KCHUNK == KCHUNK / 2;
  // DOWN: h comes from the preceding kernel; waited for only now, so that
  // the set-up above runs while that kernel finishes
  if (MODE == MOE_DOWN) pdl_wait();

  while (walk.next(q, u, nu)) {
    if (q != staged_pair) {
      first = QMV_CHECK(in_array(rt.pair_first, q, p.err)) ? rt.pair_first[q] : 0;
      nt = QMV_CHECK(in_array(rt.pair_count, q, p.err)) ? rt.pair_count[q] : 0;
      if (staged_pair >= 0) named_sync(1, CONSUMER_THREADS);  // nobody still reads the previous group's rows
      if (threadIdx.x < nt && QMV_CHECK(in_array(rt.slots, first + threadIdx.x, p.err)) &&
          QMV_CHECK(in_array(s_rows, threadIdx.x, p.err))) {
        const int slot = rt.slots[first + threadIdx.x];
        s_rows[threadIdx.x] = MODE == MOE_GATE_UP ? slot / p.top_k : slot;
      }
      named_sync(1, CONSUMER_THREADS);
      ActSource src{p.src, nullptr, nullptr, nullptr, p.K, s_rows, 0, nullptr, nullptr, nullptr
                    QMV_DEBUG_ONLY(, p.src_len, p.hq_len, p.err)};
      if (MODE == MOE_DOWN && u == 0) {  // the CTA that owns the group's first unit publishes q8(h)
        src.wq = p.hq;
        src.wd = p.hd;
        src.ws = p.hs;
      }
      // 1-2 slots: two units of 8 blocks per warp step, so that a single
      // token's row spreads over more warps (and fewer registers are live)
      stage_activations<F, NT, (NT <= 2 ? 2 : 4), CW>(src, 0, nblk, nt, a, cw, lane);
      named_sync(1, CONSUMER_THREADS);
      staged_pair = q;
    }
    // valid outputs of this tile: GATE_UP nu * 8 columns j, DOWN nu * 8 rows
    const int nvalid = nu * UNIT_ROWS;
    const bool active = MODE == MOE_GATE_UP ? 2 * cw < nvalid : cw * RW < nvalid;
    for (int c = 0; c < nck && alive; c++, ring.advance(p.stages)) {
      const int st = ring.st;
      if (!mbar_wait(&full[st], ring.parity(), p.err)) {
        alive = false;
        break;
      }
      if (active) {
        // GATE_UP: rows (2cw, 2cw + 1) of the gate half and the same of the
        // up half, 16 rows apart; DOWN: 4 consecutive rows
        constexpr int PS = (MODE == MOE_GATE_UP ? HALF : 2) * CB;
        const uint32_t rows = stage_base + st * STAGE_BYTES + roff[0] * CB;
        if (!QMV_CHECK(chunk_reads_in_range<F, NT>(rows, PS + 2 * CB, aq_base + c * NT * ACT_BYTES,
                                                   ad_base + c * NT * 128, as_base + c * NT * 128, p.err))) {
          // skipped (QMV_DEBUG builds only)
        } else if (MODE == MOE_DOWN && NT >= 8 && half_last && c == nck - 1) {
          // the last 512 weights of the rows: a half chunk, each block split
          // between two lanes (no lane works on zero fill)
          const Consumer<F, NT> ch(lane & 15);
          ch.template chunk_half<PS>(lane >> 4, rows, aq_base + c * NT * ACT_BYTES, ad_base + c * NT * 128,
                                     as_base + c * NT * 128, nt, acc);
        } else {
          cons.template chunk<PS>(rows, aq_base + c * NT * ACT_BYTES, ad_base + c * NT * 128,
                                  as_base + c * NT * 128, nt, acc);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    alive = __all_sync(FULL, alive);  // warp-uniform from here on
    if (!alive) continue;
    const int row0 = u * UNIT_ROWS;
    // (QMV_DEBUG builds) element i of the output row of group slot si lies in dst
    QMV_DEBUG_ONLY(auto dst_ok = [&](int si, long long i) {
      return in_array(rt.slots, si, p.err) && in_range((long long)rt.slots[si] * p.R + i, 1, p.dst_len, p.err);
    };)
    if constexpr (NT <= 2) {
      // few values per lane: one shuffle tree each
#pragma unroll
      for (int t = 0; t < NT; t++) {
        if (t >= nt) break;  // slots of this group without a token
        if constexpr (MODE == MOE_GATE_UP) {
#pragma unroll
          for (int i = 0; i < 2; i++) {
            const float g = warp_sum(acc.get(i, t));
            const float v = warp_sum(acc.get(2 + i, t));
            const int j = 2 * cw + i;
            if (lane == ((2 * t + i) & 31) && j < nvalid) {
              const float h = g / (1.0f + expf(-g)) * v;
              if (QMV_CHECK(dst_ok(first + t, row0 + j))) p.dst[(long long)rt.slots[first + t] * p.R + row0 + j] = h;
            }
          }
        } else {
#pragma unroll
          for (int r = 0; r < RW; r++) {
            const float v = warp_sum(acc.get(r, t));
            if (lane == ((r * NT + t) & 31) && roff[r] < nvalid && QMV_CHECK(dst_ok(first + t, row0 + roff[r])))
              p.dst[(long long)rt.slots[first + t] * p.R + row0 + roff[r]] = v;
          }
        }
      }
    } else {
      // butterfly over all RW x NT values; value r * NT + t ends in lane
      // group idx.  GATE_UP: rows 0, 1 are gate, rows 2, 3 the matching up
      // rows, so each up sum lies 16 lanes above its gate sum.
      constexpr int V = RW * NT, HELD = V >= 32 ? V / 32 : 1;
      float v[V];
#pragma unroll
      for (int r = 0; r < RW; r++)
#pragma unroll
        for (int t = 0; t < NT; t++) v[r * NT + t] = acc.get(r, t);
      int idx = 0;
      LaneButterfly<V, 0>::run(v, lane, idx);
      const bool lead = V >= 32 || (lane & (32 / V - 1)) == 0;
#pragma unroll
      for (int i = 0; i < HELD; i++) {
        const int o = idx + i, r = o / NT, t = o - r * NT;
        if constexpr (MODE == MOE_GATE_UP) {
          const float up = __shfl_down_sync(FULL, v[i], 16);
          const int j = 2 * cw + r;
          if (lead && lane < 16 && t < nt && j < nvalid) {
            const float g = v[i];
            if (QMV_CHECK(dst_ok(first + t, row0 + j)))
              p.dst[(long long)rt.slots[first + t] * p.R + row0 + j] = g / (1.0f + expf(-g)) * up;
          }
        } else {
          if (lead && t < nt && roff[r] < nvalid && QMV_CHECK(dst_ok(first + t, row0 + roff[r])))
            p.dst[(long long)rt.slots[first + t] * p.R + row0 + roff[r]] = v[i];
        }
      }
    }
    acc.zero();
  }
}

}  // namespace qmv
