// Expert-grouped MoE layer for large batches (prefill) on the tcgen05 tensor
// cores.
//
// The same layer as moe_qmv_run -- gate/up projections with SwiGLU, the
// activation rule applied to h, the down projection and the gate-weighted
// combine in k order -- for batches of hundreds to thousands of tokens, where
// each routed expert receives enough tokens for its weights to form a dense
// contraction ("Castagna Veloce", section "Kernels for the MI50", second
// bullet: the expert-grouped quantized MoE GEMM for prompt processing).
//
// Steps (one stream, five launches):
//   route   : per expert, the list of its valid slots (t * top_k + k) in
//             token order, its count and the list's offset (one CTA per
//             expert scanning all slots, so the lists are stable);
//   quantize: x by the activation rule (the library's standalone quantizer);
//   gate/up : per work item (expert, 128 outputs j, up to 64 of its slots):
//             for every 32-weight block of the hidden dimension, the CUDA
//             cores decode the 128 gate rows and 128 up rows into f16 tiles
//             (the int8 / 4-bit codes are exact in f16), the tensor core
//             forms the exact integer block dot products with the 64 slots'
//             int8 activation codes (also exact in f16, accumulated in fp32:
//             every partial sum is an integer below 2^24), and the epilogue
//             applies the fp32 block scales (d_w (x sub-scale) x d_x, and the
//             Q4_K minimum term) exactly as the decode kernels do; at the end
//             h = silu(g) u, quantized by the activation rule (one warp per
//             32-wide block of j);
//   down    : the same over the quantized h, o[slot] = Wdown_e Hhat;
//   combine : y[t] = sum_k gates[t][k] o[t, k] in k order (the decode
//             path's combine kernel).
// The block scales are applied per 32-weight block because they are
// arbitrary fp32 / fp16 values (no block-scaled MMA kind can carry them
// exactly); the integer part of every block is exact, as on the dp4a path.
// PF_LAG + 1 shared-memory tile buffers and TMEM accumulators let the tensor
// core work on block k while the threads decode block k + 1 and scale block
// k - PF_LAG (the MMA's completion latency stays off the critical path).
// Reuse conditions, with the iteration order decode(k), barrier, MMA(k),
// epilogue(k - LAG): a tile buffer is rewritten by decode(k) after this
// thread waited for MMA(k - NBUF) in epilogue(k - NBUF) (NBUF >= LAG + 1);
// a TMEM accumulator is rewritten by MMA(k) after every thread read it in
// epilogue(k - NBUF), before barrier k (NBUF >= LAG + 1); a scale-ring slot
// is rewritten by decode(k + RING) after barrier k + RING - 1, which every
// thread passes only after epilogue(k) (RING >= LAG + 2).
#include "launch.h"
#include "qmv_core.cuh"
#include "tc_core.cuh"

namespace qmv {

constexpr int PF_M = 128;        // weight rows per tile (the MMA's M)
constexpr int PF_N = 64;         // token slots per tile (the MMA's N at most)
constexpr int PF_THREADS = 256;  // 8 warps
constexpr int PF_LAG = 1;        // steps between a block's MMA and its epilogue
constexpr int PF_NBUF = PF_LAG + 1;  // smem tile buffers and TMEM accumulators
constexpr int PF_RING = 2 * PF_NBUF;  // slots of the per-block scale ring
constexpr int PF_MAX_E = 512;
constexpr int PF_GATE_UP = 0, PF_DOWN = 1;
constexpr int PF_A_TILE = PF_M * 64;  // bytes: 128 rows x 32 f16
constexpr int PF_B_TILE = PF_N * 64;  // bytes: 64 rows x 32 f16

struct PrefillParams {
  const uint8_t* W;   // expert pool [E][pool_rows][rb]
  long long rb;       // bytes per row
  int pool_rows;      // rows per expert (2F for gate/up, H for down)
  int K;              // reduction length
  int R;              // outputs per expert (F for gate/up, H for down)
  int E, top_k, n_tok;
  const int* cnt;     // [E] valid slots per expert
  const int* off;     // [E] first entry of the expert's list
  const int* list;    // [S] slots grouped by expert, token order within
  const int8_t* bq;   // activation codes: gate/up x (library layout, row t), down hq (natural, row slot)
  const float* bd;    // [rows][K/32]
  const int32_t* bs;  // [rows][K/32]
  float* h;           // gate/up outputs: h [S][F] and its quantization
  int8_t* hq;
  float* hd;
  int32_t* hs;
  float* o;           // down output [S][H]
  unsigned* err;
  // QMV_DEBUG builds: extents of the buffers (elements), derived on the host
  // from the call's arguments, for the range checks
  QMV_DEBUG_ONLY(long long bq_len;     // codes: gate/up n_tok * H, down S * F (bd, bs: bq_len / 32)
                 long long out_len;    // gate/up h, hq: S * F (hd, hs: out_len / 32); down o: S * H
                 long long list_len;)  // list: S (cnt, off: E)
};

// ---------------------------------------------------------------------------
// Routing: CTA e counts the valid slots routed to expert e and those routed
// to lower experts (its list's offset), then writes its slots in order.  A
// slot is valid when its id lies in [0, E) and does not repeat an earlier id
// of the same token (the error word records the others, CTA 0 only).
// ---------------------------------------------------------------------------
__device__ __forceinline__ int pf_slot_state(const int32_t* ids, int top_k, int E, int s, int& id) {
  const int t = s / top_k, k = s - t * top_k;
  id = ids[s];
  if (id < 0 || id >= E) return QMV_DEVERR_EXPERT_RANGE;
  for (int kk = 0; kk < k; kk++)
    if (ids[t * top_k + kk] == id) return QMV_DEVERR_EXPERT_DUP;
  return 0;
}

__global__ void __launch_bounds__(256) prefill_route_kernel(const int32_t* __restrict__ ids, int n_tok, int top_k,
                                                            int E, int* __restrict__ cnt, int* __restrict__ off,
                                                            int* __restrict__ list, unsigned* err
                                                                QMV_DEBUG_ONLY(, long long ids_len, long long cnt_len,
                                                                               long long list_len)) {
  const int e = blockIdx.x, S = n_tok * top_k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ int wc[8][2];
  int n_eq = 0, n_lt = 0;  // running totals (the same in every thread)
  // pass 1: counts
  for (int s0 = 0; s0 < S; s0 += 256) {
    const int s = s0 + threadIdx.x;
    bool eq = false, lt = false;
    if (s < S && QMV_CHECK(in_range(s, 1, ids_len, err))) {  // (the reads are ids[t top_k .. s])
      int id;
      const int st = pf_slot_state(ids, top_k, E, s, id);
      if (st && e == 0) set_error(err, (unsigned)st);
      eq = st == 0 && id == e;
      lt = st == 0 && id < e;
    }
    const unsigned beq = __ballot_sync(FULL, eq), blt = __ballot_sync(FULL, lt);
    if (lane == 0 && QMV_CHECK(in_array(wc, warp, err))) {
      wc[warp][0] = __popc(beq);
      wc[warp][1] = __popc(blt);
    }
    __syncthreads();
    for (int w = 0; w < 8; w++) {
      n_eq += wc[w][0];
      n_lt += wc[w][1];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0 && QMV_CHECK(in_range(e, 1, cnt_len, err))) {
    cnt[e] = n_eq;
    off[e] = n_lt;
  }
  // pass 2: the expert's slots in order
  int base = n_lt;
  for (int s0 = 0; s0 < S && base < n_lt + n_eq; s0 += 256) {
    const int s = s0 + threadIdx.x;
    bool eq = false;
    if (s < S && QMV_CHECK(in_range(s, 1, ids_len, err))) {
      int id;
      eq = pf_slot_state(ids, top_k, E, s, id) == 0 && id == e;
    }
    const unsigned beq = __ballot_sync(FULL, eq);
    if (lane == 0 && QMV_CHECK(in_array(wc, warp, err))) wc[warp][0] = __popc(beq);
    __syncthreads();
    int pre = 0, tot = 0;
    for (int w = 0; w < 8; w++) {
      pre += w < warp ? wc[w][0] : 0;
      tot += wc[w][0];
    }
    if (eq && QMV_CHECK(in_range(base + pre + __popc(beq & ((1u << lane) - 1u)), 1, list_len, err)))
      list[base + pre + __popc(beq & ((1u << lane) - 1u))] = s;
    base += tot;
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// Decoding one 32-weight block of a row into f16 pairs, in the K order the
// activation tile uses for that format (Q8_0 / Q4_K: natural; IQ4_XS:
// interleaved, K position 2i = element i, 2i + 1 = element i + 16, the order
// its codebook decode yields), with the block's scales: the block adds
// d_x (sA isum - sB s_x) to an output (sB, Q4_K's minimum term, else 0).
// ---------------------------------------------------------------------------
template <int F>
struct PfFmt;
template <>
struct PfFmt<QMV_Q8_0> {
  static constexpr int GW = 256, GB = 272, BPG = 8;  // weights, bytes, blocks per group
  static constexpr bool INTERLEAVED = false, MIN = false;
};
template <>
struct PfFmt<QMV_Q4_K> {
  static constexpr int GW = 256, GB = 144, BPG = 8;
  static constexpr bool INTERLEAVED = false, MIN = true;
};
template <>
struct PfFmt<QMV_IQ4_XS> {
  static constexpr int GW = 512, GB = 272, BPG = 16;
  static constexpr bool INTERLEAVED = true, MIN = false;
};

// Bytes 0-1 / 2-3 of w (values 0..255 below 1024) as an f16 pair.
__device__ __forceinline__ uint32_t u8x2_to_f16x2(uint32_t w, uint32_t sel) {
  const uint32_t h = __byte_perm(w, 0x64646464u, sel);  // 0x64 | byte: 1024 + byte
  __half2 v = *reinterpret_cast<const __half2*>(&h);
  v = __hsub2(v, __half2half2(__ushort_as_half(0x6400u)));  // - 1024
  return *reinterpret_cast<const uint32_t*>(&v);
}

// The payload bytes of block jj of a group: where they start in the group.
template <int F>
__device__ __forceinline__ int pf_payload(int jj, int half) {
  if constexpr (F == QMV_Q8_0) return 16 + 128 * half + 16 * jj;  // codes 16 half .. 16 half + 15
  if constexpr (F == QMV_Q4_K) return 16 + 16 * jj;
  return 16 + 128 * (jj >> 3) + 16 * (jj & 7);  // IQ4_XS
}

// Scales of block jj from the group's 16-byte header.
template <int F>
__device__ __forceinline__ void pf_scales(const uint4 hdr, int jj, float& sA, float& sB) {
  if constexpr (F == QMV_Q8_0) {
    const int wi = jj >> 1;
    const uint32_t w = wi == 0 ? hdr.x : (wi == 1 ? hdr.y : (wi == 2 ? hdr.z : hdr.w));
    sA = __half2float(__ushort_as_half((unsigned short)((jj & 1) ? w >> 16 : w & 0xFFFFu)));
    sB = 0.f;
  } else if constexpr (F == QMV_Q4_K) {
    // d | dmin in the first word; field jj at bits [12 jj, 12 jj + 12) of the
    // 96-bit string in words 1..3
    const int b = 12 * jj, wi = b >> 5, sh = b & 31;
    const uint32_t lo = wi == 0 ? hdr.y : (wi == 1 ? hdr.z : hdr.w);
    const uint32_t hi = wi == 0 ? hdr.z : (wi == 1 ? hdr.w : 0u);
    const uint32_t f = __funnelshift_r(lo, hi, sh);
    const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&hdr.x));
    sA = dd.x * (float)(f & 63u);
    sB = dd.y * (float)((f >> 6) & 63u);
  } else {
    // superblock sb = jj / 8: d in bytes [8 sb, 8 sb + 2), ls_j at bits
    // [16 + 6 j, 22 + 6 j) of the superblock's 8-byte header
    const int sb = jj >> 3, j = jj & 7;
    const uint32_t w0 = sb ? hdr.z : hdr.x, w1 = sb ? hdr.w : hdr.y;
    const int b = 16 + 6 * j;
    const uint32_t f = b < 32 ? __funnelshift_r(w0, w1, b) : w1 >> (b - 32);
    sA = __half2float(__ushort_as_half((unsigned short)(w0 & 0xFFFFu))) * (float)((int)(f & 63u) - 32);
    sB = 0.f;
  }
}

// 16 K positions (the half `half` of the block) as 8 f16 pairs out[0..7],
// from the block's payload word group p (Q8_0: the 16 codes of that half;
// Q4_K / IQ4_XS: the block's 16 payload bytes).
template <int F>
__device__ __forceinline__ void pf_decode_half(const uint4 p, int half, const uint32_t (&cb)[4], uint32_t (&out)[8]) {
  const uint32_t w[4] = {p.x, p.y, p.z, p.w};
  if constexpr (F == QMV_Q8_0) {
#pragma unroll
    for (int i = 0; i < 4; i++) {
      out[2 * i] = tc::s8x2_to_f16x2(w[i]);
      out[2 * i + 1] = tc::s8x2_to_f16x2(w[i] >> 16);
    }
  } else if constexpr (F == QMV_Q4_K) {
    // half 0: low nibbles (elements 0..15), half 1: high nibbles (16..31)
#pragma unroll
    for (int i = 0; i < 4; i++) {
      const uint32_t n = (half ? w[i] >> 4 : w[i]) & 0x0F0F0F0Fu;
      out[2 * i] = u8x2_to_f16x2(n, 0x5140u);
      out[2 * i + 1] = u8x2_to_f16x2(n, 0x7362u);
    }
  } else {
    // half 0: payload bytes 0..7 (K positions 0..15), half 1: bytes 8..15;
    // each 32-bit word holds 8 nibbles = K positions in order
#pragma unroll
    for (int i = 0; i < 2; i++) {
      const uint32_t pw = w[2 * half + i];
      const uint32_t pl = pw & 0x77777777u, p4 = pw << 4;
      const uint32_t c0 = iq4_lookup4(pl, pw, p4, 0xD9C8u, cb);        // K positions 8i .. 8i+3
      const uint32_t c1 = iq4_lookup4(pl >> 16, pw, p4, 0xFBEAu, cb);  // 8i+4 .. 8i+7
      out[4 * i] = tc::s8x2_to_f16x2(c0);
      out[4 * i + 1] = tc::s8x2_to_f16x2(c0 >> 16);
      out[4 * i + 2] = tc::s8x2_to_f16x2(c1);
      out[4 * i + 3] = tc::s8x2_to_f16x2(c1 >> 16);
    }
  }
}

// ---------------------------------------------------------------------------
// The projection kernel: 8 decode / epilogue warps and one issue warp,
// synchronised by mbarriers only (no CTA barrier inside a work item).
//
// Data movement per unit of 4 blocks (128 weights of K): the issue warp posts
// the stage's byte count on its full mbarrier and issues 2-D TMA loads of the
// tiles' rows (a 16-byte box of the group header and 64-byte boxes of the
// block payloads, 128 rows each); the slots' 128 activation codes and 4
// block scales (and code sums) are bulk-copied by the decode threads, one copy
// each.  Stages form a ring of NST units.
// Per block k the decode warps wait for the block's unit and for the tile
// buffer (MMA k - NBUF done), decode their rows into the f16 A tile and the
// slots' codes into the B tile, and arrive on tile_full; the issue warp waits
// for tile_full and for the TMEM accumulator (epilogue k - NBUF done), issues
// the MMAs and commits them to mma_done; the decode warps then run the
// epilogue of block k - LAG (wait mma_done, TMEM loads, scales) and arrive on
// acc_free.  A unit's stage is released (stage_empty) after its last block's
// decode.  Reuse chains: a scale-ring slot written at decode(k) is read by
// epilogue(k) and rewritten at decode(k + RING), which follows
// mma_done(k + RING - NBUF), which follows acc_free(k + RING - 2 NBUF): so
// RING >= 2 NBUF; every parity wait is at most one phase behind its barrier.
// Epilogue: gate/up -- warps 0-3 scale the gate sums, warps 4-7 the up sums,
// each for all slots of the item (rows = TMEM lanes of the warp's quarter);
// down -- the two warp halves share the slots.
// ---------------------------------------------------------------------------
constexpr int PF_UB = 4;           // K blocks per unit (128 weights)
constexpr int PF_DEC = 256;        // decode / epilogue threads (8 warps)
constexpr int PF_ALL = PF_DEC + 32;  // + the issue warp

template <int F, int MODE>
struct PfStage {
  static constexpr int NA = MODE == PF_GATE_UP ? 2 : 1;
  static constexpr int NPIECE = F == QMV_Q8_0 ? 2 : 1;   // 64-byte payload boxes per row
  static constexpr int HDR = PF_M * 16;                  // per tile
  static constexpr int PAY = PF_M * 64;                  // per tile and piece
  static constexpr int CODES = PF_N * 128;               // 128 codes per slot
  static constexpr int SC = PF_N * 16;                   // 4 scales (or sums) per slot
  static constexpr int W_BYTES = NA * (HDR + NPIECE * PAY);
  static constexpr int BYTES = W_BYTES + CODES + 2 * SC;
  static constexpr int NST = NA * NPIECE > 2 ? 3 : 4;    // units in flight
  __device__ static int hdr(int a) { return a * HDR; }
  __device__ static int pay(int a, int piece) { return NA * HDR + (a * NPIECE + piece) * PAY; }
};

// Payload box (64 bytes: blocks jj0 .. jj0 + 3) of a unit starting at block
// jj0 of its group, piece 0 or 1 (Q8_0: codes 0-15 / 16-31 of the blocks).
template <int F>
__device__ __forceinline__ int pf_unit_payload(int jj0, int piece) {
  if constexpr (F == QMV_Q8_0) return 16 + 128 * piece + 16 * jj0;
  if constexpr (F == QMV_Q4_K) return 16 + 16 * jj0;
  return 16 + 128 * (jj0 >> 3) + 16 * (jj0 & 7);  // IQ4_XS
}

template <int F, int MODE>
__global__ void __launch_bounds__(PF_ALL, 1)
    moe_prefill_kernel(const __grid_constant__ CUtensorMap map_hdr, const __grid_constant__ CUtensorMap map_pay,
                       const PrefillParams p) {
  using FM = PfFmt<F>;
  using SG = PfStage<F, MODE>;
  constexpr int NA = SG::NA;
  constexpr int TB = NA * PF_N;                    // TMEM columns per buffer
  constexpr int TCOLS = MODE == PF_GATE_UP ? 256 : 128;
  static_assert(PF_NBUF * TB <= TCOLS, "TMEM accumulators");
  static_assert(PF_RING >= 2 * PF_NBUF && PF_LAG < PF_NBUF, "reuse chains");
  constexpr bool HALF = MODE == PF_DOWN;           // two threads per weight row
  constexpr int NST = SG::NST;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stg = smem;                                            // [NST][stage]
  uint8_t* a_buf = stg + NST * SG::BYTES;                         // [NBUF][NA][A tile]; item end: up sums
  uint8_t* b_buf = a_buf + PF_NBUF * NA * PF_A_TILE;              // [NBUF][B tile]
  float* ring_sa = reinterpret_cast<float*>(b_buf + PF_NBUF * PF_B_TILE);  // [RING][NA * 128]
  float* ring_sb = ring_sa + PF_RING * NA * PF_M;                          // [RING][NA * 128]
  float* ring_dx = ring_sb + PF_RING * NA * PF_M;                          // [RING][64]
  float* ring_dxs = ring_dx + PF_RING * PF_N;                              // [RING][64]
  __shared__ uint64_t tile_full[PF_NBUF], mma_done[PF_NBUF], acc_free[PF_NBUF];
  __shared__ uint64_t full[4], stage_empty[4];
  __shared__ uint32_t tslot;
  __shared__ int prefix[PF_MAX_E + 1];  // work items before each expert
  __shared__ int s_slot[PF_N];
  __shared__ int s_part[PF_ALL / 32];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool issuer = warp == PF_DEC / 32;
  if (warp == 0) {
    tc::tmem_alloc(&tslot, TCOLS);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int b = 0; b < PF_NBUF; b++) {
      mbar_init(&tile_full[b], PF_DEC);
      mbar_init(&mma_done[b], 1);
      mbar_init(&acc_free[b], PF_DEC);
    }
    for (int b = 0; b < NST; b++) {
      mbar_init(&full[b], 1);
      mbar_init(&stage_empty[b], PF_DEC);
    }
    fence_mbar_init();
  }
  if (issuer && lane == 0) {
    prefetch_tensormap(&map_hdr);
    prefetch_tensormap(&map_pay);
  }
  // work items of each expert: (R / 128) row tiles x ceil(cnt / 64) slot tiles;
  // block scan of the counts (two experts per decode thread)
  const int mtiles = p.R / PF_M;
  {
    int c0 = 0, c1 = 0;
    const int e0 = 2 * tid, e1 = 2 * tid + 1;
    if (!issuer && e0 < p.E && QMV_CHECK(in_range(e0, 1, p.E, p.err))) c0 = mtiles * ((p.cnt[e0] + PF_N - 1) / PF_N);
    if (!issuer && e1 < p.E && QMV_CHECK(in_range(e1, 1, p.E, p.err))) c1 = mtiles * ((p.cnt[e1] + PF_N - 1) / PF_N);
    int v = c0 + c1, incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(FULL, incl, o);
      if (lane >= o) incl += a;
    }
    if (lane == 31 && QMV_CHECK(in_array(s_part, warp, p.err))) s_part[warp] = incl;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < warp; w++) before += s_part[w];
    const int excl = before + incl - v;
    if (!issuer) {
      if (e0 <= p.E && QMV_CHECK(in_array(prefix, e0, p.err))) prefix[e0] = excl;
      if (e1 <= p.E && QMV_CHECK(in_array(prefix, e1, p.err))) prefix[e1] = excl + c0;
      if (tid == PF_DEC - 1 && 2 * PF_DEC <= p.E && QMV_CHECK(in_array(prefix, p.E, p.err)))
        prefix[p.E] = before + incl;  // E = 512
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tslot;
  const int total = QMV_CHECK(in_array(prefix, p.E, p.err)) ? prefix[p.E] : 0;
  const long long i0 = (long long)total * blockIdx.x / gridDim.x, i1 = (long long)total * (blockIdx.x + 1) / gridDim.x;

  // a decode thread's weight row and epilogue place
  const int arow = tid & (PF_M - 1);
  const int atile = HALF ? 0 : (tid >> 7) & 1;  // gate / up
  const int ahalf = HALF ? (tid >> 7) & 1 : 0;
  const int q4 = warp & 3, wh = (warp >> 2) & 1;  // TMEM lane quarter; gate / up (gate/up) or slot half (down)
  const int erow = 32 * q4 + lane;                // epilogue row within the tile
  uint32_t cb[4];
  cb[0] = __shfl_sync(FULL, IQ4_T0, 0);
  cb[1] = __shfl_sync(FULL, IQ4_T1, 0);
  cb[2] = __shfl_sync(FULL, IQ4_T2, 0);
  cb[3] = __shfl_sync(FULL, IQ4_T3, 0);
  const uint64_t pol = policy_evict_first();
  const int nK = p.K / 32, nU = nK / PF_UB;
  // bounded waits; after its first timeout (error bit set) a thread stops
  // waiting, so a stalled pipeline costs one limit per thread, not one per wait
  bool dead = false;
  auto pw = [&](uint64_t* b, uint32_t parity) {
    if (!dead && !mbar_wait(b, parity, p.err)) dead = true;
  };
  long long it = 0;  // K steps of this CTA (buffer / ring / phase position)
  long long ut = 0;  // units of this CTA (stage / phase position)

  for (long long item = i0; item < i1; item++) {
    // locate (expert, row tile, slot tile)
    int lo = 0, hi = p.E;  // prefix[lo] <= item < prefix[lo + 1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] <= item)
        lo = mid;
      else
        hi = mid;
    }
    // (the search reads prefix[1 .. E - 1], the item's expert prefix[e] and p.cnt[e], e < E)
    const int e = lo, cnt_e = QMV_CHECK(in_range(e, 1, p.E, p.err)) ? p.cnt[e] : 0;
    const int ntl = (cnt_e + PF_N - 1) / PF_N;
    const int idx = (int)(item - prefix[e]), mt = idx / ntl, nt = idx - mt * ntl;
    const int count = min(PF_N, cnt_e - nt * PF_N);
    const int nmma = (count + 15) & ~15;
    __syncthreads();  // the previous item's readers of s_slot, the stages and the up sums are done
    if (tid < PF_N) {
      const long long li = tid < count && QMV_CHECK(in_range(e, 1, p.E, p.err)) ? (long long)p.off[e] + nt * PF_N + tid : -1;
      s_slot[tid] = li >= 0 && QMV_CHECK(in_range(li, 1, p.list_len, p.err)) ? p.list[li] : -1;
    }
    __syncthreads();
    const int j0 = mt * PF_M;
    const long long base = it, ubase = ut;  // this item's first K step and unit

    if (issuer) {
      // ---- the issue warp: weight boxes of each unit, and the MMAs ----
      if (lane == 0) {
        auto issue_w = [&](int u, int st) {
          uint8_t* sp = stg + st * SG::BYTES;
          mbar_arrive_expect_tx(&full[st], (uint32_t)(SG::W_BYTES + count * (128 + 16 + (FM::MIN ? 16 : 0))));
          if (!QMV_CHECK(smem_in_range(sp, SG::W_BYTES, p.err))) {
            mbar_complete_tx(&full[st], SG::W_BYTES);  // skipped: the phase still completes
            return;
          }
          const int g = (PF_UB * u) / FM::BPG, jj0 = (PF_UB * u) % FM::BPG;
#pragma unroll
          for (int a = 0; a < NA; a++) {
            const int row0 = e * p.pool_rows + (MODE == PF_GATE_UP ? a * p.R : 0) + j0;
            tma_load_2d(sp + SG::hdr(a), &map_hdr, &full[st], g * FM::GB / 8, row0, pol);
#pragma unroll
            for (int pc = 0; pc < SG::NPIECE; pc++)
              tma_load_2d(sp + SG::pay(a, pc), &map_pay, &full[st], (g * FM::GB + pf_unit_payload<F>(jj0, pc)) / 8,
                          row0, pol);
          }
        };
        for (int u = 0; u < NST - 1 && u < nU; u++) issue_w(u, (int)((ubase + u) % NST));
        for (int k = 0; k < nK; k++) {
          const long long cur = base + k;
          const int u = k / PF_UB, l = k - u * PF_UB;
          if (l == 0 && u + NST - 1 < nU) {
            const long long U = ubase + u + NST - 1;  // its stage held unit U - NST
            if (u >= 1) pw(&stage_empty[U % NST], (uint32_t)(((U - NST) / NST) & 1));
            issue_w(u + NST - 1, (int)(U % NST));
          }
          const int buf = (int)(cur % PF_NBUF);
          pw(&tile_full[buf], (uint32_t)((cur / PF_NBUF) & 1));
          if (cur >= PF_NBUF) pw(&acc_free[buf], (uint32_t)(((cur - PF_NBUF) / PF_NBUF) & 1));
          tc::fence_after_sync();
          const uint32_t idesc = tc::idesc_f16_f32(PF_M, nmma);
          const uint32_t sb = smem_u32(b_buf + buf * PF_B_TILE);
#pragma unroll
          for (int a = 0; a < NA; a++) {
            const uint32_t sa = smem_u32(a_buf + (buf * NA + a) * PF_A_TILE);
            const uint32_t d = tmem + (uint32_t)(buf * TB + a * PF_N);
            tc::mma_f16(d, tc::smem_desc(sa, 128, 512), tc::smem_desc(sb, 128, 512), idesc, false);
            tc::mma_f16(d, tc::smem_desc(sa + 256, 128, 512), tc::smem_desc(sb + 256, 128, 512), idesc, true);
          }
          tc::commit(&mma_done[buf]);
        }
      }
      __syncwarp();
    } else {
      // ---- the decode / epilogue warps ----
      // their copies of a unit's slot data: kind [codes lo, (codes hi), d, (s)] x slot
      constexpr int CPS = (MODE == PF_GATE_UP ? 2 : 1) + 1 + (FM::MIN ? 1 : 0);
      const int ckind = tid / PF_N, cslot = tid - ckind * PF_N;
      const bool cact = ckind < CPS && cslot < count;
      const long long crow = cact ? (MODE == PF_GATE_UP ? s_slot[cslot] / p.top_k : s_slot[cslot]) : -1;
      auto issue_c = [&](int u, int st) {
        if (!cact) return;
        uint8_t* sp = stg + st * SG::BYTES;
        const int kd = MODE == PF_GATE_UP ? ckind : (ckind == 0 ? 0 : ckind + 1);  // 0 lo, 1 hi, 2 d, 3 s
        // one copy: global element gi of codes (kd <= 1) or of scales / sums, to dst
        long long gi;
        uint8_t* dst;
        uint32_t bytes;
        if (kd <= 1) {
          // gate/up: the library layout, elements 0-15 of the unit's blocks, then 16-31 (128 further)
          gi = crow * (long long)p.K + (MODE == PF_GATE_UP ? (u >> 1) * 256 + (u & 1) * 64 + 128 * kd : u * 128);
          dst = sp + SG::W_BYTES + cslot * 128 + (MODE == PF_GATE_UP ? 64 * kd : 0);
          bytes = MODE == PF_GATE_UP ? 64 : 128;
        } else {
          gi = crow * (p.K / 32) + PF_UB * u;
          dst = sp + SG::W_BYTES + SG::CODES + (kd == 3 ? SG::SC : 0) + cslot * 16;
          bytes = 16;
        }
        if (!QMV_CHECK(in_range(gi, kd <= 1 ? bytes : bytes / 4, kd <= 1 ? p.bq_len : p.bq_len / 32, p.err)) || !QMV_CHECK(smem_in_range(dst, bytes, p.err))) {
          mbar_complete_tx(&full[st], bytes);  // skipped: the phase still completes
          return;
        }
        if (kd <= 1)
          bulk_copy_g2s(dst, p.bq + gi, bytes, &full[st]);
        else if (kd == 2)
          bulk_copy_g2s(dst, p.bd + gi, bytes, &full[st]);
        else
          bulk_copy_g2s(dst, p.bs + gi, bytes, &full[st]);
      };
      for (int u = 0; u < NST - 1 && u < nU; u++) issue_c(u, (int)((ubase + u) % NST));
      // B staging: slot tile row n, core matrix q (K positions 8q .. 8q + 7)
      const int bn = tid >> 2, bqq = tid & 3;
      const bool bval = bn < count;
      // epilogue: slots [en0, en0 + ecnt) of the warp
      const int ecnt = MODE == PF_GATE_UP ? count : (count > 32 ? min(32, count - 32 * wh) : min(16, count - 16 * wh));
      const int en0 = MODE == PF_GATE_UP ? 0 : (count > 32 ? 32 * wh : 16 * wh);
      float acc[MODE == PF_GATE_UP ? 64 : 32];
#pragma unroll
      for (int i = 0; i < (MODE == PF_GATE_UP ? 64 : 32); i++) acc[i] = 0.f;

      for (int k = 0; k < nK + PF_LAG; k++) {
        const long long cur = base + k;
        if (k < nK) {
          const int buf = (int)(cur % PF_NBUF), slot = (int)(cur % PF_RING);
          const int u = k / PF_UB, l = k - u * PF_UB;
          const int st = (int)((ubase + u) % NST);
          const uint8_t* sp = stg + st * SG::BYTES;
          if (l == 0) {
            if (u + NST - 1 < nU) {
              const long long U = ubase + u + NST - 1;  // its stage held unit U - NST
              if (u >= 1) pw(&stage_empty[U % NST], (uint32_t)(((U - NST) / NST) & 1));
              issue_c(u + NST - 1, (int)(U % NST));
            }
            pw(&full[st], (uint32_t)(((ubase + u) / NST) & 1));  // the unit has landed
          }
          if (cur >= PF_NBUF) pw(&mma_done[buf], (uint32_t)(((cur - PF_NBUF) / PF_NBUF) & 1));
          // ---- decode the weights of block k into the A tile ----
          const uint8_t* hp = sp + SG::hdr(atile) + arow * 16;
          const uint4 hdr = QMV_CHECK(smem_in_range(hp, 16, p.err)) ? *reinterpret_cast<const uint4*>(hp) : make_uint4(0, 0, 0, 0);
          const int jj = k % FM::BPG;
          float sA, sB;
          pf_scales<F>(hdr, jj, sA, sB);
          uint8_t* at = a_buf + (buf * NA + atile) * PF_A_TILE;
          // a 16-byte load from the stage and a 16-byte store into the A tile
          auto ld16 = [&](const uint8_t* q) {
            return QMV_CHECK(smem_in_range(q, 16, p.err)) ? *reinterpret_cast<const uint4*>(q) : make_uint4(0, 0, 0, 0);
          };
          auto st16 = [&](uint8_t* q, uint4 v) {
            if (QMV_CHECK(smem_in_range(q, 16, p.err))) *reinterpret_cast<uint4*>(q) = v;
          };
          if (HALF) {
            const uint4 pay = ld16(sp + SG::pay(0, SG::NPIECE == 2 ? ahalf : 0) + arow * 64 + 16 * l);
            uint32_t o[8];
            pf_decode_half<F>(pay, ahalf, cb, o);
            st16(at + tc::kmajor_offset(arow, 32 * ahalf, 64), make_uint4(o[0], o[1], o[2], o[3]));
            st16(at + tc::kmajor_offset(arow, 32 * ahalf + 16, 64), make_uint4(o[4], o[5], o[6], o[7]));
          } else {
#pragma unroll
            for (int hv = 0; hv < 2; hv++) {
              const uint4 pay = ld16(sp + SG::pay(atile, SG::NPIECE == 2 ? hv : 0) + arow * 64 + 16 * l);
              uint32_t o[8];
              pf_decode_half<F>(pay, hv, cb, o);
              st16(at + tc::kmajor_offset(arow, 32 * hv, 64), make_uint4(o[0], o[1], o[2], o[3]));
              st16(at + tc::kmajor_offset(arow, 32 * hv + 16, 64), make_uint4(o[4], o[5], o[6], o[7]));
            }
          }
          if (!HALF || ahalf == 0) {
            const int ri = slot * NA * PF_M + atile * PF_M + arow;
            if (QMV_CHECK(smem_in_range(ring_sa + ri, 4, p.err))) ring_sa[ri] = sA;
            if constexpr (FM::MIN)
              if (QMV_CHECK(smem_in_range(ring_sb + ri, 4, p.err))) ring_sb[ri] = sB;
          }
          // ---- the activation codes of block k into the B tile ----
          uint4 v = make_uint4(0, 0, 0, 0);
          if (bval && QMV_CHECK(smem_in_range(sp + SG::W_BYTES + bn * 128, 128, p.err))) {  // the slot's codes
            const uint8_t* cr = sp + SG::W_BYTES + bn * 128;
            uint32_t x0, x1;
            if (FM::INTERLEAVED) {  // elements 4q .. 4q+3 and 16+4q .. 16+4q+3
              const int o0 = MODE == PF_GATE_UP ? l * 16 + 4 * bqq : l * 32 + 4 * bqq;
              const int o1 = MODE == PF_GATE_UP ? 64 + l * 16 + 4 * bqq : l * 32 + 16 + 4 * bqq;
              const uint32_t lo2 = *reinterpret_cast<const uint32_t*>(cr + o0),
                             hi2 = *reinterpret_cast<const uint32_t*>(cr + o1);
              x0 = __byte_perm(lo2, hi2, 0x5140u);
              x1 = __byte_perm(lo2, hi2, 0x7362u);
            } else {  // elements 8q .. 8q+7
              const int o0 = MODE == PF_GATE_UP ? (bqq >> 1) * 64 + l * 16 + 8 * (bqq & 1) : l * 32 + 8 * bqq;
              const uint2 w = *reinterpret_cast<const uint2*>(cr + o0);
              x0 = w.x;
              x1 = w.y;
            }
            v = make_uint4(tc::s8x2_to_f16x2(x0), tc::s8x2_to_f16x2(x0 >> 16), tc::s8x2_to_f16x2(x1),
                           tc::s8x2_to_f16x2(x1 >> 16));
          }
          st16(b_buf + buf * PF_B_TILE + tc::kmajor_offset(bn, 16 * bqq, 64), v);
          if (tid < PF_N) {
            float dx = 0.f, dxs = 0.f;
            const float* dp = reinterpret_cast<const float*>(sp + SG::W_BYTES + SG::CODES) + tid * 4 + l;
            const int* sq = reinterpret_cast<const int*>(sp + SG::W_BYTES + SG::CODES + SG::SC) + tid * 4 + l;
            if (tid < count && QMV_CHECK(smem_in_range(dp, 4, p.err))) {
              dx = *dp;
              if constexpr (FM::MIN)
                if (QMV_CHECK(smem_in_range(sq, 4, p.err))) dxs = dx * (float)*sq;
            }
            if (QMV_CHECK(smem_in_range(ring_dx + slot * PF_N + tid, 4, p.err))) ring_dx[slot * PF_N + tid] = dx;
            if (QMV_CHECK(smem_in_range(ring_dxs + slot * PF_N + tid, 4, p.err))) ring_dxs[slot * PF_N + tid] = dxs;
          }
          tc::fence_smem_to_async();
          mbar_arrive(&tile_full[buf]);
          if (l == PF_UB - 1) mbar_arrive(&stage_empty[st]);  // this thread is done with the unit's stage
        }
        if (k >= PF_LAG) {
          // ---- epilogue of block k - LAG: scale its integer sums into acc ----
          const long long prev = cur - PF_LAG;
          const int pbuf = (int)(prev % PF_NBUF), pslot = (int)(prev % PF_RING);
          pw(&mma_done[pbuf], (uint32_t)((prev / PF_NBUF) & 1));
          tc::fence_after_sync();
          __syncwarp();  // the TMEM loads below are warp-aligned instructions
          const int a_ep = MODE == PF_GATE_UP ? wh : 0;
          const uint32_t tcol = tmem + ((uint32_t)(32 * q4) << 16) + (uint32_t)(pbuf * TB + a_ep * PF_N + en0);
          const int ri = pslot * NA * PF_M + a_ep * PF_M + erow;
          const float sa = QMV_CHECK(smem_in_range(ring_sa + ri, 4, p.err)) ? ring_sa[ri] : 0.f;
          const float2 sa2 = make_float2(sa, sa);
          float2 nsb2 = make_float2(0.f, 0.f);
          if constexpr (FM::MIN) {
            const float sb = QMV_CHECK(smem_in_range(ring_sb + ri, 4, p.err)) ? ring_sb[ri] : 0.f;
            nsb2 = make_float2(-sb, -sb);
          }
          const float* dxp = ring_dx + pslot * PF_N + en0;
          const float* dxsp = ring_dxs + pslot * PF_N + en0;
          auto scale_into = [&](const float (&D)[32], int a0, int nv) {
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              if (i < nv && QMV_CHECK(smem_in_range(dxp + a0 + i, 8, p.err)) && QMV_CHECK(smem_in_range(dxsp + a0 + i, 8, p.err))) {
                const float2 dx = *reinterpret_cast<const float2*>(dxp + a0 + i);
                float2 r = __ffma2_rn(__fmul2_rn(sa2, dx), make_float2(D[i], D[i + 1]),
                                      make_float2(acc[a0 + i], acc[a0 + i + 1]));
                if constexpr (FM::MIN) r = __ffma2_rn(nsb2, *reinterpret_cast<const float2*>(dxsp + a0 + i), r);
                acc[a0 + i] = r.x;
                acc[a0 + i + 1] = r.y;
              }
            }
          };
          if (MODE == PF_GATE_UP) {
            if (count > 32) {
              float D0[32], D1[32];
              tc::tmem_ld2_x32(tcol, tcol + 32, D0, D1);
              scale_into(D0, 0, 32);
              if constexpr (MODE == PF_GATE_UP) scale_into(D1, 32, 32);
            } else {
              float D0[32];
              tc::tmem_ld_x32(tcol, D0);
              scale_into(D0, 0, 32);
            }
          } else if (ecnt > 0) {
            if (count > 32) {
              float D0[32];
              tc::tmem_ld_x32(tcol, D0);
              scale_into(D0, 0, 32);
            } else {
              uint32_t r16[16];
              tc::tmem_ld_x16(tcol, r16);
              float D0[32];
#pragma unroll
              for (int i = 0; i < 16; i++) D0[i] = __uint_as_float(r16[i]);
#pragma unroll
              for (int i = 16; i < 32; i++) D0[i] = 0.f;
              scale_into(D0, 0, 16);
            }
          }
          tc::fence_before_sync();
          mbar_arrive(&acc_free[pbuf]);  // this thread's reads of the accumulator are complete
        }
      }
      // ---- outputs of the down projection ----
      if constexpr (MODE == PF_DOWN) {
        const int j = j0 + erow;
#pragma unroll
        for (int i = 0; i < 32; i++) {
          if (i >= ecnt) break;  // warp-uniform
          if (!QMV_CHECK(in_array(s_slot, en0 + i, p.err))) continue;
          const long long oi = (long long)s_slot[en0 + i] * p.R + j;
          if (QMV_CHECK(in_range(oi, 1, p.out_len, p.err))) p.o[oi] = acc[i];
        }
      } else {
        // gate/up: the up sums to the gate warps through shared memory (the
        // A tiles are free: the last MMA has completed), [slot][row]
        float* up = reinterpret_cast<float*>(a_buf);
        if (wh == 1) {
#pragma unroll
          for (int i = 0; i < 64; i++) {
            if (i >= count) break;  // warp-uniform
            if (QMV_CHECK(smem_in_range(up + i * PF_M + erow, 4, p.err))) up[i * PF_M + erow] = acc[i];
          }
        }
        named_sync(1, PF_DEC);
        if (wh == 0) {
          const int F_ = p.R, j = j0 + erow;
#pragma unroll
          for (int i = 0; i < 64; i++) {
            if (i >= count) break;  // warp-uniform
            const long long sl = QMV_CHECK(in_array(s_slot, i, p.err)) ? s_slot[i] : 0;
            const float g = acc[i], uu = QMV_CHECK(smem_in_range(up + i * PF_M + erow, 4, p.err)) ? up[i * PF_M + erow] : 0.f;
            const bool put_ok = QMV_CHECK(in_range(sl * F_ + j, 1, p.out_len, p.err));
            const float hv = g / (1.0f + expf(-g)) * uu;
            if (put_ok) p.h[sl * F_ + j] = hv;
            // the activation rule over the warp's 32 consecutive j (one block)
            const unsigned ab = __float_as_uint(fabsf(hv));
            const float amax = __uint_as_float(__reduce_max_sync(FULL, ab));
            const float d = __fdiv_rn(amax, 127.0f);
            const float id = d > 0.0f ? __frcp_rn(d) : 0.0f;
            float pq = __fmul_rn(hv, id);
            pq = pq != pq ? 0.0f : fminf(fmaxf(pq, -127.0f), 127.0f);
            const int q = __float2int_rn(pq);
            const int s = __reduce_add_sync(FULL, q);
            if (put_ok) p.hq[sl * F_ + j] = (int8_t)q;
            if (lane == 0 && QMV_CHECK(in_range(sl * (F_ / 32) + j / 32, 1, p.out_len / 32, p.err))) {
              p.hd[sl * (F_ / 32) + j / 32] = d;
              p.hs[sl * (F_ / 32) + j / 32] = s;
            }
          }
        }
      }
    }
    it += nK;
    ut += nU;
  }
  if (dead) {  // let copies this thread may not have waited for land before the CTA exits
    for (int i = 0; i < 1000; i++) __nanosleep(10000);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, TCOLS);
}

template <int F, int MODE>
static cudaError_t launch_prefill(const PrefillParams& p, int grid, cudaStream_t stream) {
  using SG = PfStage<F, MODE>;
  constexpr int NA = SG::NA;
  const size_t smem = (size_t)SG::NST * SG::BYTES + (size_t)PF_NBUF * NA * PF_A_TILE + PF_NBUF * PF_B_TILE +
                      (size_t)PF_RING * NA * PF_M * 2 * sizeof(float) + (size_t)PF_RING * PF_N * 2 * sizeof(float);
  // the pool's rows as 8-byte elements; boxes of 128 rows x 16 bytes (group
  // header) and x 64 bytes (4 blocks of payload)
  const long long rows = (long long)p.E * p.pool_rows;
  CUtensorMap map_hdr, map_pay;
  if (!encode_rows(&map_hdr, p.W, rows, p.rb, 16, PF_M) || !encode_rows(&map_pay, p.W, rows, p.rb, 64, PF_M))
    return cudaErrorInvalidValue;
  auto kern = moe_prefill_kernel<F, MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, PF_ALL, smem, stream>>>(map_hdr, map_pay, p);
  return cudaGetLastError();
}

template <int MODE>
static cudaError_t launch_prefill_fmt(int fmt, const PrefillParams& p, int grid, cudaStream_t stream) {
  switch (fmt) {
    case QMV_Q8_0: return launch_prefill<QMV_Q8_0, MODE>(p, grid, stream);
    case QMV_Q4_K: return launch_prefill<QMV_Q4_K, MODE>(p, grid, stream);
    default: return launch_prefill<QMV_IQ4_XS, MODE>(p, grid, stream);
  }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
namespace {
constexpr int PF_NOFF = 11;

size_t al256(size_t v) { return (v + 255) & ~(size_t)255; }

int pf_group_weights(int fmt) { return fmt == QMV_IQ4_XS ? 512 : 256; }

// [0] h f32 [S][F], [1] hq i8 [S][F], [2] hd f32 [S][F/32], [3] hs i32
// [S][F/32], [4] o f32 [S][H], [5] xq i8 [n][H], [6] xd f32 [n][H/32],
// [7] xs i32 [n][H/32], [8] cnt i32 [E], [9] off i32 [E], [10] list i32 [S]
size_t pf_layout(const moe_experts* e, int n_tok, int top_k, size_t off[PF_NOFF]) {
  const size_t S = (size_t)n_tok * top_k, F = (size_t)e->ffn, H = (size_t)e->hidden, n = (size_t)n_tok;
  const size_t sizes[PF_NOFF] = {S * F * 4, S * F, S * (F / 32) * 4, S * (F / 32) * 4, S * H * 4,
                                 n * H,     n * (H / 32) * 4,        n * (H / 32) * 4, (size_t)e->n_experts * 4,
                                 (size_t)e->n_experts * 4, S * 4};
  size_t cur = 0;
  for (int i = 0; i < PF_NOFF; i++) {
    off[i] = cur;
    cur = al256(cur + sizes[i]);
  }
  return cur;
}

int pf_check(const moe_experts* e, int n_tok, int top_k) {
  if (!e) return QMV_ERR_NULL;
  const int fg = e->fmt_gate_up, fd = e->fmt_down;
  const bool ok_fmt = (fg == QMV_Q8_0 || fg == QMV_Q4_K || fg == QMV_IQ4_XS) &&
                      (fd == QMV_Q8_0 || fd == QMV_Q4_K || fd == QMV_IQ4_XS);
  if (!ok_fmt) return QMV_ERR_FORMAT;
  if (e->n_experts < 1 || e->n_experts > PF_MAX_E || e->hidden <= 0 || e->ffn <= 0 || e->hidden > (1 << 20) ||
      e->ffn > (1 << 20) || e->hidden % PF_M || e->ffn % PF_M || e->hidden % pf_group_weights(fg) ||
      e->ffn % pf_group_weights(fd))
    return QMV_ERR_SHAPE;
  if (n_tok < 1 || n_tok > QMV_MAX_PREFILL_TOKENS || top_k < 1 || top_k > QMV_MAX_TOPK || top_k > e->n_experts)
    return QMV_ERR_NTOK;
  return QMV_OK;
}
}  // namespace

}  // namespace qmv

using namespace qmv;

extern "C" size_t moe_qmv_prefill_workspace_bytes(const moe_experts* e, int n_tok, int top_k) {
  if (pf_check(e, n_tok, top_k)) return 0;
  size_t off[PF_NOFF];
  return pf_layout(e, n_tok, top_k, off);
}

extern "C" int moe_qmv_prefill_workspace_offsets(const moe_experts* e, int n_tok, int top_k, size_t offsets[5]) {
  int rc = pf_check(e, n_tok, top_k);
  if (rc) return rc;
  if (!offsets) return QMV_ERR_NULL;
  size_t off[PF_NOFF];
  pf_layout(e, n_tok, top_k, off);
  for (int i = 0; i < 5; i++) offsets[i] = off[i];
  return QMV_OK;
}

extern "C" int moe_qmv_prefill_run(const moe_experts* e, const int32_t* ids, const float* gates, const float* x,
                                   float* y, int n_tok, int top_k, void* ws, size_t ws_bytes, cudaStream_t stream) {
  int rc = pf_check(e, n_tok, top_k);
  if (rc) return rc;
  if (!ids || !gates || !x || !y || !ws || !e->w_gate_up || !e->w_down) return QMV_ERR_NULL;
  auto a16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
  if (!a16(ids) || !a16(gates) || !a16(x) || !a16(y) || !a16(ws) || !a16(e->w_gate_up) || !a16(e->w_down))
    return QMV_ERR_ALIGN;
  size_t off[PF_NOFF];
  if (ws_bytes < pf_layout(e, n_tok, top_k, off)) return QMV_ERR_WORKSPACE;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return QMV_ERR_CUDA;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) return QMV_ERR_DEVICE;
  uint8_t* w = static_cast<uint8_t*>(ws);
  float* h = reinterpret_cast<float*>(w + off[0]);
  int8_t* hq = reinterpret_cast<int8_t*>(w + off[1]);
  float* hd = reinterpret_cast<float*>(w + off[2]);
  int32_t* hs = reinterpret_cast<int32_t*>(w + off[3]);
  float* o = reinterpret_cast<float*>(w + off[4]);
  int8_t* xq = reinterpret_cast<int8_t*>(w + off[5]);
  float* xd = reinterpret_cast<float*>(w + off[6]);
  int32_t* xs = reinterpret_cast<int32_t*>(w + off[7]);
  int* cnt = reinterpret_cast<int*>(w + off[8]);
  int* offs = reinterpret_cast<int*>(w + off[9]);
  int* list = reinterpret_cast<int*>(w + off[10]);
  const int E = e->n_experts, H = e->hidden, F = e->ffn;
  unsigned* err = device_error_word();

  const long long S = (long long)n_tok * top_k;
  prefill_route_kernel<<<E, 256, 0, stream>>>(ids, n_tok, top_k, E, cnt, offs, list, err QMV_DEBUG_ONLY(, S, E, S));
  if (cudaGetLastError() != cudaSuccess) return QMV_ERR_CUDA;
  if (launch_act_quant(x, H, n_tok, xq, xd, xs, (long long)n_tok * H, stream, false) != cudaSuccess)
    return QMV_ERR_CUDA;

  const int grid = device_sm_count();
  PrefillParams p{};
  p.E = E;
  p.top_k = top_k;
  p.n_tok = n_tok;
  p.cnt = cnt;
  p.off = offs;
  p.list = list;
  p.err = err;
  QMV_DEBUG_ONLY(p.list_len = S;)
  // gate / up + SwiGLU + the activation rule on h
  p.W = static_cast<const uint8_t*>(e->w_gate_up);
  p.rb = qmv_row_bytes(e->fmt_gate_up, H);
  p.pool_rows = 2 * F;
  p.K = H;
  p.R = F;
  p.bq = xq;
  p.bd = xd;
  p.bs = xs;
  p.h = h;
  p.hq = hq;
  p.hd = hd;
  p.hs = hs;
  QMV_DEBUG_ONLY(p.bq_len = (long long)n_tok * H; p.out_len = S * F;)
  if (launch_prefill_fmt<PF_GATE_UP>(e->fmt_gate_up, p, grid, stream) != cudaSuccess) return QMV_ERR_CUDA;
  // down
  PrefillParams pd = p;
  pd.W = static_cast<const uint8_t*>(e->w_down);
  pd.rb = qmv_row_bytes(e->fmt_down, F);
  pd.pool_rows = H;
  pd.K = F;
  pd.R = H;
  pd.bq = hq;
  pd.bd = hd;
  pd.bs = hs;
  pd.o = o;
  QMV_DEBUG_ONLY(pd.bq_len = S * F; pd.out_len = S * H;)
  if (launch_prefill_fmt<PF_DOWN>(e->fmt_down, pd, grid, stream) != cudaSuccess) return QMV_ERR_CUDA;
  return launch_moe_combine(ids, gates, o, y, n_tok, top_k, E, H, stream, false) == cudaSuccess ? QMV_OK
                                                                                                 : QMV_ERR_CUDA;
}
