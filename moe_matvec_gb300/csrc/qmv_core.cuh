// Core of every quantized matvec kernel in the library: the activation
// staging (per-32 int8 quantization into shared memory, in the byte order each
// weight format consumes) and the consumer step that decodes one 1024-weight
// chunk of RW weight rows in registers and accumulates exact int32 block dot
// products (dp4a) scaled in fp32.
//
// Shared by the dense matvec / split-K kernel and the expert-grouped MoE
// kernels ("Castagna Veloce", section "Kernels for the MI50": small-batch
// matvecs and MoE decode kernels; section "Fused operations": Q8 activations
// reused across weight types).
//
// Shared-memory activation area (NT token slots, nck chunks of 1024 weights):
//   q  [nck][NT][1024] int8   codes, blocks of one chunk interleaved (act_pos)
//   d  [nck][NT][32]   f32    block scales
//   ds [nck][NT][32]   f32    block scale x block code sum (Q4_K only)
// Token slots past the staged tokens and blocks past the K-range are zero, so
// the consumer needs no per-token or per-block predicates: a zero code and a
// zero scale add exactly nothing.
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
constexpr int PREFETCH_STAGES = 16;                   // L2 lookahead of the producer (iterations, at most)
constexpr long long PREFETCH_ALL_BYTES = 40ll << 20;  // matrices up to this size: all tiles requested at once
constexpr int ACT_BYTES = KCHUNK;                     // codes per token per chunk
constexpr unsigned FULL = 0xffffffffu;

// CTA shape with CW consumer warps.  Eight consumers run beside one producer
// warp.  Twelve consumers (three per scheduler, for kernels whose warps are
// register-bound) run beside a producer warpgroup whose four warps hand all
// but REG_PRODUCER registers each to the consumers (REG_CONSUMER each):
// 128 x REG_PRODUCER + 384 x REG_CONSUMER = 65,536, the registers of a
// 512-thread CTA launched at 128 per thread.
template <int CW>
struct Shape {
  static_assert(CW == 8 || CW == 12, "8 or 12 consumer warps");
  static constexpr int TILE_ROWS = CW * RW;
  static constexpr int CONSUMER_THREADS = CW * 32;
  static constexpr int PRODUCER_WARPS = CW == 8 ? 1 : 4;
  static constexpr int THREADS = (CW + PRODUCER_WARPS) * 32;
  static constexpr bool RESPLIT = CW != 8;
  static constexpr int REG_LAUNCH = 65536 / THREADS;  // 128 when re-split
  static constexpr int REG_PRODUCER = 32, REG_CONSUMER = 160;
  static_assert(!RESPLIT || PRODUCER_WARPS * 32 * REG_PRODUCER + CW * 32 * REG_CONSUMER <= THREADS * REG_LAUNCH,
                "register re-split exceeds the launch's registers");
};

// Byte p (0..31) of block l (0..31) of a token's 1024-byte chunk of codes:
// within every 8 blocks the first 16 bytes come first, then the last 16, so
// that the 8 lanes of a quarter-warp read 128 contiguous bytes.
__device__ __forceinline__ int act_pos(int l, int p) {
  return (l >> 3) * 256 + (p >> 4) * 128 + (l & 7) * 16 + (p & 15);
}

// Activation area of nt_slots token slots over nck chunks, chunk-major:
//   codes  [chunk][slot] 1024 bytes (each 256-element group in act_pos order),
//   scales [chunk][slot] 32 fp32 d (block order),
//   sums   [chunk][slot] 32 int32 s (Q4_K only: its min term needs them),
// so that within a chunk every slot sits at a fixed offset.  A slot's chunk
// of codes, scales or sums is one contiguous piece of the library's
// pre-quantized activation rows, so those arrive by bulk copies.
// (F16 / F32 weights take fp32 activations: [chunk][slot] kchunk_of(F)
// floats, no scales or sums.)
__host__ __device__ constexpr size_t act_area_bytes(int F, int nt_slots, int nck) {
  return is_float(F) ? (size_t)nck * nt_slots * kchunk_of(F) * sizeof(float)
                     : (size_t)nck * nt_slots * (ACT_BYTES + 32 * sizeof(float) * (has_min(F) ? 2 : 1));
}
// Bytes of one token slot's activations in a chunk.
__host__ __device__ constexpr int act_chunk_bytes(int F) {
  return is_float(F) ? kchunk_of(F) * (int)sizeof(float) : ACT_BYTES;
}

struct ActArea {
  uint8_t* q;  // [nck][ns][1024]
  float* d;    // [nck][ns][32]
  int32_t* s;  // [nck][ns][32]
  int ns;      // slots per chunk
  __device__ void carve(uint8_t* base, int F, int nt_slots, int nck) {
    ns = nt_slots;
    q = base;
    d = reinterpret_cast<float*>(base + (size_t)nck * nt_slots * ACT_BYTES);
    s = reinterpret_cast<int32_t*>(d + (size_t)nck * nt_slots * 32);
    (void)F;
  }
  __device__ __forceinline__ uint8_t* codes(int c, int t) const { return q + ((size_t)c * ns + t) * ACT_BYTES; }
  __device__ __forceinline__ int scale(int c, int t) const { return (c * ns + t) * 32; }
};

// The shared-memory ranges one consumer step reads: rows_bytes of weight
// rows from `rows`, and one chunk's activations of NT token slots (codes or
// fp32 values at aq, scales at ad, Q4_K / Q5_K sums at as).
template <int F, int NT>
__device__ __forceinline__ bool chunk_reads_in_range(uint32_t rows, uint32_t rows_bytes, uint32_t aq, uint32_t ad,
                                                     uint32_t as, unsigned* err) {
  bool ok = smem_in_range(rows, rows_bytes, err) && smem_in_range(aq, NT * act_chunk_bytes(F), err);
  if constexpr (!is_float(F)) ok = ok && smem_in_range(ad, NT * 128, err);
  if constexpr (has_min(F)) ok = ok && smem_in_range(as, NT * 128, err);
  return ok;
}

// Where the activation rows come from: fp32 rows (quantized while staging)
// or pre-quantized rows in the library's Q8 activation layout (codes of each
// 256-element group in act_pos order, one scale and one sum per block); token
// slot t reads source row rows[t] (a shared-memory list) or row0 + t.  When
// wq is set, the quantized codes, scales and sums are also written back to
// global memory (natural order), which is how the MoE path exposes the
// quantized h.
struct ActSource {
  const float* x;
  const int8_t* xq;
  const float* xd;
  const int32_t* xs;
  long long ld;      // elements per source row
  const int* rows;   // nullptr: rows row0 .. row0 + nt - 1
  long long row0;
  int8_t* wq;
  float* wd;
  int32_t* ws;
  // QMV_DEBUG builds: extents for the range checks and the error word
  QMV_DEBUG_ONLY(long long x_len;  // elements of x (or of xq; xd and xs hold x_len / 32)
                 long long w_len;  // elements of wq (wd and ws hold w_len / 32)
                 unsigned* err;)
  __device__ __forceinline__ long long row(int t) const { return rows ? (long long)rows[t] : row0 + t; }
};

// The activation rule for SU units of 8 blocks, four lanes per block (lane
// group sub = lane / 4 holds block sub of each unit, lane li = lane % 4 its
// elements 8 li .. 8 li + 7 in v[u][0..1]); called by full warps.  Returns the
// lane's 8 codes packed in w0 / w1 (natural order) and the block's d and s
// in every lane of the block.  Four lanes share a block: a load instruction
// of the warp touches 8 blocks; two shuffle steps combine maximum and sum.
template <int SU>
__device__ __forceinline__ void quant_units(const float4 (&v)[SU][2], uint32_t (&w0)[SU], uint32_t (&w1)[SU],
                                            float (&dd)[SU], int (&ss)[SU]) {
  float m[SU];
#pragma unroll
  for (int u = 0; u < SU; u++) {
    m[u] = fmaxf(fmaxf(fmaxf(fabsf(v[u][0].x), fabsf(v[u][0].y)), fmaxf(fabsf(v[u][0].z), fabsf(v[u][0].w))),
                 fmaxf(fmaxf(fabsf(v[u][1].x), fabsf(v[u][1].y)), fmaxf(fabsf(v[u][1].z), fabsf(v[u][1].w))));
    m[u] = fmaxf(m[u], __shfl_xor_sync(FULL, m[u], 1));
    m[u] = fmaxf(m[u], __shfl_xor_sync(FULL, m[u], 2));
  }
  // Fast path: every block has amax == 0 or amax >= 2^-100, where the
  // branch-free sequences are exact and no code needs clamping
  // (|x * id| <= amax * id < 127.5).  Otherwise the whole warp takes the IEEE
  // operations with the clamp.
  bool slow = false;
#pragma unroll
  for (int u = 0; u < SU; u++) slow |= m[u] > 0.0f && m[u] < 0x1p-100f;
  slow = __any_sync(FULL, slow);
  float id[SU];
  if (!slow) {
#pragma unroll
    for (int u = 0; u < SU; u++) {
      dd[u] = div127_rn(m[u]);
      id[u] = m[u] > 0.0f ? rcp_rn(fmaxf(dd[u], 0x1p-126f)) : 0.0f;
    }
  } else {
#pragma unroll
    for (int u = 0; u < SU; u++) {
      dd[u] = __fdiv_rn(m[u], 127.0f);
      id[u] = dd[u] > 0.0f ? __frcp_rn(dd[u]) : 0.0f;
    }
  }
#pragma unroll
  for (int u = 0; u < SU; u++) {
    float f[8] = {v[u][0].x, v[u][0].y, v[u][0].z, v[u][0].w, v[u][1].x, v[u][1].y, v[u][1].z, v[u][1].w};
    int q[8];
    // The slow path clamps the integer: the conversion takes +-inf (1 / d
    // overflows to infinity for blocks whose amax is below about 3.7e-37) to
    // the ends of the int range and a not-a-number (0 * inf, a zero element of
    // such a block) to 0, the codes the rule gives them.
#pragma unroll
    for (int k = 0; k < 8; k++) {
      q[k] = __float2int_rn(__fmul_rn(f[k], id[u]));
      if (slow) q[k] = min(max(q[k], -127), 127);
    }
    w0[u] = (uint32_t)(q[0] & 0xFF) | ((uint32_t)(q[1] & 0xFF) << 8) | ((uint32_t)(q[2] & 0xFF) << 16) |
            ((uint32_t)q[3] << 24);
    w1[u] = (uint32_t)(q[4] & 0xFF) | ((uint32_t)(q[5] & 0xFF) << 8) | ((uint32_t)(q[6] & 0xFF) << 16) |
            ((uint32_t)q[7] << 24);
    int sm = __dp4a((int)w1[u], 0x01010101, __dp4a((int)w0[u], 0x01010101, 0));
    sm += __shfl_xor_sync(FULL, sm, 1);
    sm += __shfl_xor_sync(FULL, sm, 2);
    ss[u] = sm;
  }
}

// Store a lane's 8 codes of block l (lane li of the block's four) into a
// slot's chunk of codes.  IQ4_XS reads its activations interleaved (byte
// 2i = x_i, byte 2i + 1 = x_{i+16}, the order its codebook decode yields):
// lanes 0, 1 of the block take the elements 16.. of lanes 2, 3.  Called by
// full warps.
template <int F>
__device__ __forceinline__ void store_codes(uint8_t* chunk, int l, int li, uint32_t w0,
                                            uint32_t w1 QMV_DEBUG_ONLY(, unsigned* err)) {
  if constexpr (F == QMV_IQ4_XS) {
    const uint32_t h0 = __shfl_xor_sync(FULL, w0, 2), h1 = __shfl_xor_sync(FULL, w1, 2);
    if (li < 2 && QMV_CHECK(smem_in_range(chunk + act_pos(l, 16 * li), 16, err)))
      *reinterpret_cast<uint4*>(chunk + act_pos(l, 16 * li)) =
          make_uint4(__byte_perm(w0, h0, 0x5140), __byte_perm(w0, h0, 0x7362), __byte_perm(w1, h1, 0x5140),
                     __byte_perm(w1, h1, 0x7362));
  } else {
    if (QMV_CHECK(smem_in_range(chunk + act_pos(l, 8 * li), 8, err)))
      *reinterpret_cast<uint2*>(chunk + act_pos(l, 8 * li)) = make_uint2(w0, w1);
  }
}

// Stage blocks [kb0, kb0 + nblk) of tokens [0, nt) of `src` into the area,
// zero-filling the blocks past nblk of the last chunk (and the slots up to
// the next power of two, which the consumers read in pairs).  Called by all
// consumer warps; a warp step covers SU units of 8 blocks with all of its
// loads issued first and no branch inside a unit, so the units overlap.
template <int F, int NT, int SU = 4, int CW = CONSUMER_WARPS>
__device__ __forceinline__ void stage_activations(const ActSource& src, int kb0, int nblk, int nt, const ActArea& a,
                                                  int cw, int lane) {
  const int sub = lane >> 2, li = lane & 3;
  const int nck = (nblk + 31) / 32;
  int sh = 0;
  while ((1 << sh) < nt) sh++;
  if (NT >= 2 && sh == 0) sh = 1;
  const int total = nck * 32 << sh;  // a multiple of 32 = blocks of one warp step
  for (int base = cw * 8 * SU; base < total; base += CW * 8 * SU) {
    int tt[SU], cc[SU], l[SU];
    long long gblk[SU];
    bool real[SU];
    uint32_t w0[SU], w1[SU];
    float dd[SU];
    int ss[SU];
    float4 v[SU][2];
#pragma unroll
    for (int u = 0; u < SU; u++) {
      const int idx = base + 8 * u + sub;
      l[u] = idx & 31;
      tt[u] = (idx >> 5) & ((1 << sh) - 1);
      cc[u] = idx >> (5 + sh);
      const int b = cc[u] * 32 + l[u];
      real[u] = tt[u] < nt && b < nblk;
      gblk[u] = real[u] ? src.row(tt[u]) * (src.ld / 32) + kb0 + b : 0;
      if (real[u] && !QMV_CHECK(in_range(gblk[u] * 32, 32, src.x_len, src.err))) real[u] = false;
      v[u][0] = v[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
      w0[u] = w1[u] = 0u;
      dd[u] = 0.f;
      ss[u] = 0;
      if (real[u]) {
        if (src.x != nullptr) {
          const float4* p = reinterpret_cast<const float4*>(src.x + gblk[u] * 32) + 2 * li;
          v[u][0] = __ldg(p);
          v[u][1] = __ldg(p + 1);
        } else {
          // pre-quantized rows: codes in act_pos order within each group
          const int gb = (int)(gblk[u] & 7);
          const uint2 q = __ldg(reinterpret_cast<const uint2*>(src.xq + (gblk[u] - gb) * 32 +
                                                               act_pos(gb, 8 * li)));
          w0[u] = q.x;
          w1[u] = q.y;
          dd[u] = __ldg(src.xd + gblk[u]);
          ss[u] = __ldg(src.xs + gblk[u]);
        }
      }
    }
    if (src.x != nullptr) {
      quant_units<SU>(v, w0, w1, dd, ss);
      if (src.wq != nullptr) {
#pragma unroll
        for (int u = 0; u < SU; u++) {
          if (real[u] && QMV_CHECK(in_range(gblk[u] * 32, 32, src.w_len, src.err))) {
            reinterpret_cast<uint2*>(src.wq + gblk[u] * 32)[li] = make_uint2(w0[u], w1[u]);
            if (li == 0) {
              src.wd[gblk[u]] = dd[u];
              src.ws[gblk[u]] = ss[u];
            }
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < SU; u++) {
      store_codes<F>(a.codes(cc[u], tt[u]), l[u], li, w0[u], w1[u] QMV_DEBUG_ONLY(, src.err));
      if (li == 0) {
        const int di = a.scale(cc[u], tt[u]) + l[u];
        if (QMV_CHECK(smem_in_range(a.d + di, 4, src.err))) a.d[di] = dd[u];
        if constexpr (has_min(F))
          if (QMV_CHECK(smem_in_range(a.s + di, 4, src.err))) a.s[di] = ss[u];
      }
    }
  }
}

// Pre-quantized activations (the library's layout) of blocks [kb0, kb0 +
// nblk) of tokens [0, nt), brought into the area by bulk copies, one per
// (token, chunk) and kind (codes, scales, Q4_K sums): each is one contiguous
// piece in global memory and in the area.  Lane 0 of warp 0 first posts the
// byte count on `bar`; then every consumer thread issues its share of the
// copies, zeroes the scales past nblk of the last chunk, waits for `bar`
// (phase `parity`) and, for IQ4_XS, reorders each block's codes into the
// interleaved order its decode reads.  Returns false (timeout bit set) if
// the copies never land.
template <int F, int NT, int CW = CONSUMER_WARPS>
__device__ __forceinline__ bool stage_q8_bulk(const ActSource& src, int kb0, int nblk, int nt, const ActArea& a,
                                              uint64_t* bar, uint32_t parity, unsigned* err, int cw, int lane) {
  constexpr int NCOPY = has_min(F) ? 3 : 2;
  const int nck = (nblk + 31) / 32;
  if (cw == 0 && lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(nt * nblk * (32 + 4 * (NCOPY - 1))));
  named_sync(1, CW * 32);  // the byte count is posted before any copy completes
  {
    // one copy per (token, chunk, kind): codes, scales, sums; spread over all consumer threads
    for (int i = cw * 32 + lane; i < nt * nck * NCOPY; i += CW * 32) {
      const int t = i / (nck * NCOPY), r = i - t * nck * NCOPY, c = r / NCOPY, k = r - c * NCOPY;
      const int nb = min(32, nblk - c * 32);
      const long long row = src.row(t), b0 = (long long)kb0 + c * 32;  // first block of the piece
      const uint32_t bytes = (uint32_t)nb * (k == 0 ? 32 : 4);
      void* dst = k == 0 ? (void*)a.codes(c, t) : k == 1 ? (void*)(a.d + a.scale(c, t)) : (void*)(a.s + a.scale(c, t));
      if (!QMV_CHECK(in_range((row * (src.ld / 32) + b0) * 32, nb * 32, src.x_len, err)) || !QMV_CHECK(smem_in_range(dst, bytes, err))) {
        mbar_complete_tx(bar, bytes);  // skipped: the phase still completes
        continue;
      }
      if (k == 0)
        bulk_copy_g2s(dst, src.xq + row * src.ld + b0 * 32, bytes, bar);
      else if (k == 1)
        bulk_copy_g2s(dst, src.xd + row * (src.ld / 32) + b0, bytes, bar);
      else
        bulk_copy_g2s(dst, src.xs + row * (src.ld / 32) + b0, bytes, bar);
    }
  }
  // scales (and sums) of the blocks past nblk in the last chunk: zero
  const int nb_last = nblk - (nck - 1) * 32, tail = 32 - nb_last;
  for (int i = cw * 32 + lane; i < nt * tail; i += CW * 32) {
    const int t = i / tail, b = nb_last + (i - t * tail);
    if (QMV_CHECK(smem_in_range(a.d + a.scale(nck - 1, t) + b, 4, err))) a.d[a.scale(nck - 1, t) + b] = 0.f;
    if constexpr (has_min(F))
      if (QMV_CHECK(smem_in_range(a.s + a.scale(nck - 1, t) + b, 4, err))) a.s[a.scale(nck - 1, t) + b] = 0;
  }
  const bool ok = mbar_wait(bar, parity, err);
  if constexpr (F == QMV_IQ4_XS) {
    // x_0..15 and x_16..31 of a block sit in two 16-byte pieces; interleave
    for (int i = cw * 32 + lane; i < nt * nck * 32; i += CW * 32) {
      const int t = i / (nck * 32), r = i - t * nck * 32, c = r >> 5, l = r & 31;
      uint8_t* chunk = a.codes(c, t);
      uint4* p0 = reinterpret_cast<uint4*>(chunk + act_pos(l, 0));
      uint4* p1 = reinterpret_cast<uint4*>(chunk + act_pos(l, 16));
      if (!QMV_CHECK(smem_in_range(p0, 16, err)) || !QMV_CHECK(smem_in_range(p1, 16, err))) continue;
      const uint4 lo = *p0, hi = *p1;
      *p0 = make_uint4(__byte_perm(lo.x, hi.x, 0x5140), __byte_perm(lo.x, hi.x, 0x7362),
                       __byte_perm(lo.y, hi.y, 0x5140), __byte_perm(lo.y, hi.y, 0x7362));
      *p1 = make_uint4(__byte_perm(lo.z, hi.z, 0x5140), __byte_perm(lo.z, hi.z, 0x7362),
                       __byte_perm(lo.w, hi.w, 0x5140), __byte_perm(lo.w, hi.w, 0x7362));
    }
  }
  return ok;
}

// dp4a with unsigned bytes in a and signed bytes in b.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// Codebook lookup of four 4-bit codes held as the nibbles of the low 16 bits
// of a word (nibble k -> byte k of the result).  pl (the word & 0x7777...)
// picks from the lower and the upper half of the codebook with two byte
// permutes; the fourth bit of each code becomes a byte mask through the
// sign-replicating mode of a third permute (msb of the selected byte copied
// to all 8 bits), fed with the word and the word << 4 so that the fourth bits
// of the four codes sit at byte msbs.
// The codebook as four words (codes 0..7, then 8..15), the data operands
// of the two table permutes.
constexpr uint32_t IQ4_T0 = 0xBFAD9881u, IQ4_T1 = 0xF6EADDCFu;
constexpr uint32_t IQ4_T2 = 0x26190D01u, IQ4_T3 = 0x71594535u;
__device__ __forceinline__ uint32_t iq4_lookup4(uint32_t pl, uint32_t p, uint32_t p4, uint32_t mask_sel,
                                                const uint32_t (&t)[4]) {
  uint32_t lo = prmt(t[0], t[1], pl);
  uint32_t hi = prmt(t[2], t[3], pl);
  uint32_t m = prmt(p4, p, mask_sel);
  return (hi & m) | (lo & ~m);
}

// Shared-memory loads by 32-bit shared address.
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ float2 lds_f2(uint32_t a) {
  const uint2 v = lds64(a);
  return make_float2(__uint_as_float(v.x), __uint_as_float(v.y));
}

// The accumulators of a warp's RW rows x NT token slots, kept as fp32 pairs
// of consecutive slots (a register pair each, operand of the packed fp32x2
// instructions); with one slot only .x is used.
template <int NT>
struct AccTile {
  static constexpr int NP = NT >= 2 ? NT / 2 : 1;
  float2 v[RW][NP];
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int r = 0; r < RW; r++)
#pragma unroll
      for (int q = 0; q < NP; q++) v[r][q] = make_float2(0.f, 0.f);
  }
  __device__ __forceinline__ float get(int r, int t) const { return (t & 1) ? v[r][t >> 1].y : v[r][t >> 1].x; }
};

// The consumer step.  Each lane owns one 32-weight block of every chunk; its
// byte offsets inside a staged row chunk and inside the activation chunk are
// fixed for the whole kernel.
template <int F, int NT>
struct Consumer {
  uint32_t w_off;  // payload of the lane's block in a row chunk
  uint32_t h_off;  // first header word the lane reads in a row chunk
  uint32_t f_off;  // Q4_K / IQ4_XS: word holding (the start of) the lane's 6/12-bit scale field
  uint32_t fsh;    // bit offset of that field in the word pair at f_off
  uint32_t a_off;  // the lane's block in a token's activation chunk
  uint32_t d_off;  // the lane's scale in a chunk's scales (token slot 0)
  uint32_t x_off;  // Q5_K: the word of fifth bits of the lane's block in a row chunk
  uint32_t cb[4];  // IQ4_XS: the codebook words, held in registers for the whole kernel (a
                   // shuffle hides their values, so they are not re-created before every use)

  __device__ explicit Consumer(int lane) {
    const int j = lane & 7;
    if constexpr (F == QMV_Q8_0) {
      const int g = lane >> 3;
      w_off = g * 272 + 16 + 16 * j;
      h_off = g * 272 + 2 * j;
      f_off = fsh = 0;
    } else if constexpr (F == QMV_Q8_G64) {
      // two 512-weight groups per chunk; 16 blocks each, a scale per 2 blocks
      const int g = lane >> 4, h = (lane >> 3) & 1;
      w_off = g * 528 + 16 + 256 * h + 16 * j;
      h_off = g * 528 + 2 * ((lane & 15) >> 1);
      f_off = fsh = 0;
    } else if constexpr (F == QMV_Q8_G128) {
      // one 1024-weight group per chunk; a scale per 4 blocks
      const int h = lane >> 3;
      w_off = 16 + 256 * h + 16 * j;
      h_off = 2 * (lane >> 2);
      f_off = fsh = 0;
    } else if constexpr (F == QMV_Q4_K) {
      const int g = lane >> 3;
      w_off = g * 144 + 16 + 16 * j;
      h_off = g * 144;
      // bits [12j, 12j + 12) of the 96-bit string at header byte 4 (for the
      // last fields the second word is the first payload word, unused bits)
      f_off = h_off + 4 + 4 * ((12 * j) >> 5);
      fsh = (12 * j) & 31;
    } else if constexpr (F == QMV_Q5_K) {
      const int g = lane >> 3;
      w_off = g * 176 + 48 + 16 * j;
      h_off = g * 176;
      f_off = h_off + 4 + 4 * ((12 * j) >> 5);  // the sc / m string as in Q4_K
      fsh = (12 * j) & 31;
      x_off = g * 176 + 16 + 4 * j;
    } else if constexpr (F == QMV_Q6_K) {
      const int g = lane >> 3;
      w_off = g * 208 + 80 + 16 * j;
      h_off = g * 208;
      // sc_{2j}, sc_{2j+1}: bits [14j, 14j + 14) of the 112-bit string at byte 2
      f_off = h_off + 4 * ((16 + 14 * j) >> 5);
      fsh = (16 + 14 * j) & 31;
      x_off = g * 208 + 16 + 8 * j;
    } else {
      const int g = lane >> 4, sb = (lane >> 3) & 1;
      w_off = g * 272 + 16 + 128 * sb + 16 * j;
      h_off = g * 272 + 8 * sb;
      // ls_j: bits [16 + 6j, 22 + 6j) of the superblock's 8-byte header
      f_off = h_off + 4 * ((16 + 6 * j) >> 5);
      fsh = (16 + 6 * j) & 31;
    }
    a_off = act_pos(lane, 0);
    d_off = 4 * lane;
    if constexpr (F == QMV_IQ4_XS) {
      cb[0] = __shfl_sync(FULL, IQ4_T0, 0);
      cb[1] = __shfl_sync(FULL, IQ4_T1, 0);
      cb[2] = __shfl_sync(FULL, IQ4_T2, 0);
      cb[3] = __shfl_sync(FULL, IQ4_T3, 0);
    }
  }

  // Q4_K with 4 or more tokens: both nibble halves as 16 x code, one chain.
  static constexpr bool Q4K_LO16 = NT >= 4;

  // row0: shared address of the warp's first row chunk in the stage; row r
  // starts at row0 + (r & 1) * chunk_bytes + (r >> 1) * PAIR_STRIDE (rows in
  // pairs: consecutive rows use PAIR_STRIDE = 2 * chunk_bytes).  aq / ad /
  // as: shared addresses of this chunk's activation codes / scales / sums in
  // token slot 0; slot t is t * 1024 (codes) or t * 128 (scales, sums) bytes
  // further.
  // nt: slots holding tokens (the accumulators of the others are left as
  // they are).
  template <int PAIR_STRIDE = 2 * chunk_bytes<F>()>
  __device__ __forceinline__ void chunk(uint32_t row0, uint32_t aq, uint32_t ad, uint32_t as, int nt,
                                        AccTile<NT>& acc) const {
    constexpr uint32_t sq = ACT_BYTES, sd = 32 * 4;
    constexpr int CB = chunk_bytes<F>();
    uint32_t w[RW][8];  // decoded operands, paired with activation words 0..7
    float sA[RW];       // multiplier of d_x * isum
    int scl[RW] = {}, sch[RW] = {};  // Q6_K: the integer sub-scales of weights 0..15 and 16..31
    float sB[RW];       // Q4_K: dmin * m, multiplier of d_x * s
#pragma unroll
    for (int r = 0; r < RW; r++) {
      const uint32_t row = row0 + (r & 1) * CB + (r >> 1) * PAIR_STRIDE;
      if constexpr (is_q8(F)) {
        const uint4 x0 = lds128(row + w_off);
        const uint4 x1 = lds128(row + w_off + 128);
        w[r][0] = x0.x; w[r][1] = x0.y; w[r][2] = x0.z; w[r][3] = x0.w;
        w[r][4] = x1.x; w[r][5] = x1.y; w[r][6] = x1.z; w[r][7] = x1.w;
        // the lane's fp16 d is the low or high half of an aligned word
        const uint32_t hw = lds32(row + (h_off & ~3u));
        sA[r] = __half2float(__ushort_as_half((unsigned short)((h_off & 2) ? hw >> 16 : hw & 0xFFFF)));
        sB[r] = 0.f;
      } else if constexpr (F == QMV_Q4_K) {
        const uint32_t dh = lds32(row + h_off);  // d | dmin
        const uint32_t f0 = lds32(row + f_off);
        const uint32_t f1 = lds32(row + f_off + 4);
        const uint4 q = lds128(row + w_off);
        const uint32_t qq[4] = {q.x, q.y, q.z, q.w};
        // high nibbles left in place (16 x code) for an unsigned-byte dp4a;
        // low nibbles as bytes (the dot product scales their sum by 16) or,
        // for one dp4a chain, shifted up to 16 x code as well.  sA carries
        // the 1/16 (exact: a power of two).
#pragma unroll
        for (int i = 0; i < 4; i++) {
          w[r][i] = Q4K_LO16 ? (qq[i] << 4) & 0xF0F0F0F0u : qq[i] & 0x0F0F0F0Fu;
          w[r][4 + i] = qq[i] & 0xF0F0F0F0u;
        }
        const uint32_t f = __funnelshift_r(f0, f1, fsh);
        const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&dh));
        sA[r] = dd.x * (float)(f & 63u) * 0.0625f;  // the dot product is 16 x the block sum
        sB[r] = dd.y * (float)((f >> 6) & 63u);
      } else if constexpr (F == QMV_Q5_K) {
        const uint32_t dh = lds32(row + h_off);  // d | dmin
        const uint32_t f0 = lds32(row + f_off);
        const uint32_t f1 = lds32(row + f_off + 4);
        const uint32_t hb = lds32(row + x_off);  // bit i: fifth bit of weight i
        const uint4 q = lds128(row + w_off);
        const uint32_t qq[4] = {q.x, q.y, q.z, q.w};
        // codes as unsigned bytes: the low four bits from the nibbles, the
        // fifth from hb, its four bits for a word spread to the bytes by a
        // multiply (the shifted copies do not overlap) and moved to bit 4
#pragma unroll
        for (int i = 0; i < 4; i++) {
          const uint32_t lo = (((hb >> (4 * i)) & 0xFu) * 0x00204081u) & 0x01010101u;
          const uint32_t hi = (((hb >> (16 + 4 * i)) & 0xFu) * 0x00204081u) & 0x01010101u;
          w[r][i] = (qq[i] & 0x0F0F0F0Fu) | (lo << 4);
          w[r][4 + i] = ((qq[i] >> 4) & 0x0F0F0F0Fu) | (hi << 4);
        }
        const uint32_t f = __funnelshift_r(f0, f1, fsh);
        const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&dh));
        sA[r] = dd.x * (float)(f & 63u);
        sB[r] = dd.y * (float)((f >> 6) & 63u);
      } else if constexpr (F == QMV_Q6_K) {
        const uint32_t dw = lds32(row + h_off);
        const uint32_t f0 = lds32(row + f_off);
        const uint32_t f1 = lds32(row + f_off + 4);
        const uint2 hb = lds64(row + x_off);  // top two bits: weights 0..15, 16..31
        const uint4 q = lds128(row + w_off);
        const uint32_t qq[4] = {q.x, q.y, q.z, q.w};
        // each code byte is v << 2 = 4 (q - 32) as int8: the low four bits
        // from the nibbles at bits 2-5, the top two at bits 6-7 (word k of
        // a half keeps them at bits 8b + 2k of its bit word)
#pragma unroll
        for (int i = 0; i < 4; i++) {
          w[r][i] = ((qq[i] << 2) & 0x3C3C3C3Cu) | ((hb.x << (6 - 2 * i)) & 0xC0C0C0C0u);
          w[r][4 + i] = ((qq[i] >> 2) & 0x3C3C3C3Cu) | ((hb.y << (6 - 2 * i)) & 0xC0C0C0C0u);
        }
        const uint32_t f = __funnelshift_r(f0, f1, fsh);
        scl[r] = (int)(f & 127u);
        sch[r] = (int)((f >> 7) & 127u);
        sA[r] = __half2float(__ushort_as_half((unsigned short)(dw & 0xFFFF))) * 0.25f;  // the dots are 4 x
        sB[r] = 0.f;
      } else {
        const uint32_t dw = lds32(row + h_off);
        const uint32_t f0 = lds32(row + f_off);
        const uint32_t f1 = lds32(row + f_off + 4);
        const uint4 q = lds128(row + w_off);
        const int ls = (int)(__funnelshift_r(f0, f1, fsh) & 63u);
        sA[r] = __half2float(__ushort_as_half((unsigned short)(dw & 0xFFFF))) * (float)(ls - 32);
        sB[r] = 0.f;
        const uint32_t qq[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; i++) {
          const uint32_t pw = qq[i];
          const uint32_t pl = pw & 0x77777777u;
          const uint32_t p4 = pw << 4;
          w[r][2 * i] = iq4_lookup4(pl, pw, p4, 0xD9C8u, cb);
          w[r][2 * i + 1] = iq4_lookup4(pl >> 16, pw, p4, 0xFBEAu, cb);
        }
      }
    }
    const uint32_t ap = aq + a_off, dp = ad + d_off, sp = as + d_off;
    if constexpr (NT == 1) {
      const uint4 xa = lds128(ap);
      const uint4 xb = lds128(ap + 128);
      const float dx = __uint_as_float(lds32(dp));
      float dxs = 0.f;
      if constexpr (has_min(F)) dxs = dx * (float)(int)lds32(sp);
#pragma unroll
      for (int r = 0; r < RW; r++) {
        float v = fmaf(sA[r] * dx, (float)dotr(w[r], xa, xb, scl[r], sch[r]), acc.v[r][0].x);
        if constexpr (has_min(F)) v = fmaf(-sB[r], dxs, v);
        acc.v[r][0].x = v;
      }
    } else {
      // token pairs: the scale products and accumulations of two tokens go
      // through packed fp32x2 multiply / fma (each lane of the pair rounds
      // like the scalar operation)
      float2 sA2[RW], nsB2[RW];
#pragma unroll
      for (int r = 0; r < RW; r++) {
        sA2[r] = make_float2(sA[r], sA[r]);
        nsB2[r] = make_float2(-sB[r], -sB[r]);
      }
#pragma unroll
      for (int t = 0; t < NT; t += 2) {
        if (t >= nt) break;  // slots without a token (a short MoE group, a last pass)
        const uint4 xa0 = lds128(ap + t * sq);
        const uint4 xb0 = lds128(ap + t * sq + 128);
        const uint4 xa1 = lds128(ap + (t + 1) * sq);
        const uint4 xb1 = lds128(ap + (t + 1) * sq + 128);
        const float2 dx = make_float2(__uint_as_float(lds32(dp + t * sd)), __uint_as_float(lds32(dp + (t + 1) * sd)));
        float2 dxs = make_float2(0.f, 0.f);
        if constexpr (has_min(F))
          dxs = __fmul2_rn(dx, make_float2((float)(int)lds32(sp + t * sd), (float)(int)lds32(sp + (t + 1) * sd)));
#pragma unroll
        for (int r = 0; r < RW; r++) {
          const float2 is = make_float2((float)dotr(w[r], xa0, xb0, scl[r], sch[r]), (float)dotr(w[r], xa1, xb1, scl[r], sch[r]));
          float2 v = __ffma2_rn(__fmul2_rn(sA2[r], dx), is, acc.v[r][t >> 1]);
          if constexpr (has_min(F)) v = __ffma2_rn(nsB2[r], dxs, v);
          acc.v[r][t >> 1] = v;
        }
      }
    }
  }

  // The same step over a half chunk: the last 16 blocks of a row whose
  // length is 512 past a multiple of 1024 (the MoE down projection's 1536),
  // where a whole-chunk step would leave half of the lanes decoding and
  // multiplying zero fill.  Here every block is split between two lanes:
  // lane l < 16 takes weights 0..15 of block l (operand words 0..3 with
  // activation group xa), lane l + 16 weights 16..31 (words 4..7 with xb).
  // The consumer must have been built for block lane % 16; h = lane / 16.
  // Each half's integer sum is exact and scaled by the block's scales as in
  // chunk(); the block's min term is added by its h = 0 lane only.  The
  // lanes' sums meet in the caller's cross-lane reduction as before.
  template <int PAIR_STRIDE = 2 * chunk_bytes<F>()>
  __device__ __forceinline__ void chunk_half(int h, uint32_t row0, uint32_t aq, uint32_t ad, uint32_t as, int nt,
                                             AccTile<NT>& acc) const {
    static_assert(F == QMV_Q8_0 || F == QMV_Q4_K || F == QMV_IQ4_XS, "the expert formats");
    constexpr uint32_t sq = ACT_BYTES, sd = 32 * 4;
    constexpr int CB = chunk_bytes<F>();
    uint32_t w[RW][4];  // decoded operands of the lane's half, paired with activation words 4h..4h+3
    float sA[RW], sB[RW];
#pragma unroll
    for (int r = 0; r < RW; r++) {
      const uint32_t row = row0 + (r & 1) * CB + (r >> 1) * PAIR_STRIDE;
      if constexpr (F == QMV_Q8_0) {
        const uint4 x = lds128(row + w_off + 128 * h);
        w[r][0] = x.x; w[r][1] = x.y; w[r][2] = x.z; w[r][3] = x.w;
        const uint32_t hw = lds32(row + (h_off & ~3u));
        sA[r] = __half2float(__ushort_as_half((unsigned short)((h_off & 2) ? hw >> 16 : hw & 0xFFFF)));
        sB[r] = 0.f;
      } else if constexpr (F == QMV_Q4_K) {
        const uint32_t dh = lds32(row + h_off);  // d | dmin
        const uint32_t f0 = lds32(row + f_off);
        const uint32_t f1 = lds32(row + f_off + 4);
        const uint4 q = lds128(row + w_off);
        const uint32_t qq[4] = {q.x, q.y, q.z, q.w};
        // both halves as 16 x code (h = 0: the low nibbles shifted up); sA
        // carries the 1/16 as in chunk()
#pragma unroll
        for (int i = 0; i < 4; i++) w[r][i] = (h == 0 ? qq[i] << 4 : qq[i]) & 0xF0F0F0F0u;
        const uint32_t f = __funnelshift_r(f0, f1, fsh);
        const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&dh));
        sA[r] = dd.x * (float)(f & 63u) * 0.0625f;
        sB[r] = h == 0 ? dd.y * (float)((f >> 6) & 63u) : 0.f;
      } else {
        const uint32_t dw = lds32(row + h_off);
        const uint32_t f0 = lds32(row + f_off);
        const uint32_t f1 = lds32(row + f_off + 4);
        const uint2 q = lds64(row + w_off + 8 * h);  // payload words 2h, 2h + 1
        const int ls = (int)(__funnelshift_r(f0, f1, fsh) & 63u);
        sA[r] = __half2float(__ushort_as_half((unsigned short)(dw & 0xFFFF))) * (float)(ls - 32);
        sB[r] = 0.f;
        const uint32_t qq[2] = {q.x, q.y};
#pragma unroll
        for (int i = 0; i < 2; i++) {
          const uint32_t pw = qq[i];
          const uint32_t pl = pw & 0x77777777u;
          const uint32_t p4 = pw << 4;
          w[r][2 * i] = iq4_lookup4(pl, pw, p4, 0xD9C8u, cb);
          w[r][2 * i + 1] = iq4_lookup4(pl >> 16, pw, p4, 0xFBEAu, cb);
        }
      }
    }
    const uint32_t ap = aq + a_off + 128 * h, dp = ad + d_off, sp = as + d_off;
    if constexpr (NT == 1) {
      const uint4 x = lds128(ap);
      const float dx = __uint_as_float(lds32(dp));
      float dxs = 0.f;
      if constexpr (has_min(F)) dxs = dx * (float)(int)lds32(sp);
#pragma unroll
      for (int r = 0; r < RW; r++) {
        float v = fmaf(sA[r] * dx, (float)dot_half(w[r], x), acc.v[r][0].x);
        if constexpr (has_min(F)) v = fmaf(-sB[r], dxs, v);
        acc.v[r][0].x = v;
      }
    } else {
      float2 sA2[RW], nsB2[RW];
#pragma unroll
      for (int r = 0; r < RW; r++) {
        sA2[r] = make_float2(sA[r], sA[r]);
        nsB2[r] = make_float2(-sB[r], -sB[r]);
      }
#pragma unroll
      for (int t = 0; t < NT; t += 2) {
        if (t >= nt) break;
        const uint4 x0 = lds128(ap + t * sq);
        const uint4 x1 = lds128(ap + (t + 1) * sq);
        const float2 dx = make_float2(__uint_as_float(lds32(dp + t * sd)), __uint_as_float(lds32(dp + (t + 1) * sd)));
        float2 dxs = make_float2(0.f, 0.f);
        if constexpr (has_min(F))
          dxs = __fmul2_rn(dx, make_float2((float)(int)lds32(sp + t * sd), (float)(int)lds32(sp + (t + 1) * sd)));
#pragma unroll
        for (int r = 0; r < RW; r++) {
          const float2 is = make_float2((float)dot_half(w[r], x0), (float)dot_half(w[r], x1));
          float2 v = __ffma2_rn(__fmul2_rn(sA2[r], dx), is, acc.v[r][t >> 1]);
          if constexpr (has_min(F)) v = __ffma2_rn(nsB2[r], dxs, v);
          acc.v[r][t >> 1] = v;
        }
      }
    }
  }

  // Exact int32 dot product of one half block (four operand words) with its
  // four activation words (Q4_K: 16 x the sum, unsigned codes).
  __device__ __forceinline__ int dot_half(const uint32_t (&w)[4], uint4 x) const {
    if constexpr (F == QMV_Q4_K) {
      int s = dp4a_us(w[0], x.x, 0);
      s = dp4a_us(w[1], x.y, s);
      s = dp4a_us(w[2], x.z, s);
      return dp4a_us(w[3], x.w, s);
    } else {
      int s = __dp4a((int)w[0], (int)x.x, 0);
      s = __dp4a((int)w[1], (int)x.y, s);
      s = __dp4a((int)w[2], (int)x.z, s);
      return __dp4a((int)w[3], (int)x.w, s);
    }
  }

  // The block's integer dot product with its sub-scales applied (Q6_K: two
  // halves of 16 weights, each with its own integer scale; other formats
  // have one scale per block, carried in sA, and ignore lo / hi).
  __device__ __forceinline__ int dotr(const uint32_t (&w)[8], uint4 xa, uint4 xb, int lo, int hi) const {
    if constexpr (F == QMV_Q6_K) {
      int ia = __dp4a((int)w[0], (int)xa.x, 0);
      int ib = __dp4a((int)w[4], (int)xb.x, 0);
      ia = __dp4a((int)w[1], (int)xa.y, ia);
      ib = __dp4a((int)w[5], (int)xb.y, ib);
      ia = __dp4a((int)w[2], (int)xa.z, ia);
      ib = __dp4a((int)w[6], (int)xb.z, ib);
      ia = __dp4a((int)w[3], (int)xa.w, ia);
      ib = __dp4a((int)w[7], (int)xb.w, ib);
      return ia * lo + ib * hi;  // |4 x 16 x 128 x 127| x 127 x 2 < 2^31
    } else {
      (void)lo;
      (void)hi;
      return dot(w, xa, xb);
    }
  }

  // Exact int32 dot product of one 32-weight block with the activation words
  // xa (elements 0..15 of the block) and xb (16..31) (Q4_K and Q5_K: unsigned
  // codes, the min term is added by the caller).  Q4_K: 16 x the sum
  // (both nibble halves weigh 16; sA carries the 1/16).  With one token the
  // two halves run as independent chains.
  __device__ __forceinline__ int dot(const uint32_t (&w)[8], uint4 xa, uint4 xb) const {
    if constexpr (F == QMV_Q4_K) {
      if constexpr (Q4K_LO16) {
        int s = dp4a_us(w[0], xa.x, 0);
        s = dp4a_us(w[1], xa.y, s);
        s = dp4a_us(w[2], xa.z, s);
        s = dp4a_us(w[3], xa.w, s);
        s = dp4a_us(w[4], xb.x, s);
        s = dp4a_us(w[5], xb.y, s);
        s = dp4a_us(w[6], xb.z, s);
        return dp4a_us(w[7], xb.w, s);
      } else {
        int ia = dp4a_us(w[0], xa.x, 0);
        int ib = dp4a_us(w[4], xb.x, 0);
        ia = dp4a_us(w[1], xa.y, ia);
        ib = dp4a_us(w[5], xb.y, ib);
        ia = dp4a_us(w[2], xa.z, ia);
        ib = dp4a_us(w[6], xb.z, ib);
        ia = dp4a_us(w[3], xa.w, ia);
        ib = dp4a_us(w[7], xb.w, ib);
        return ia * 16 + ib;
      }
    } else if constexpr (F == QMV_Q5_K) {
      // unsigned codes in [0, 31]; with one token the halves as two chains
      if constexpr (NT == 1) {
        int ia = dp4a_us(w[0], xa.x, 0);
        int ib = dp4a_us(w[4], xb.x, 0);
        ia = dp4a_us(w[1], xa.y, ia);
        ib = dp4a_us(w[5], xb.y, ib);
        ia = dp4a_us(w[2], xa.z, ia);
        ib = dp4a_us(w[6], xb.z, ib);
        ia = dp4a_us(w[3], xa.w, ia);
        ib = dp4a_us(w[7], xb.w, ib);
        return ia + ib;
      } else {
        int s = dp4a_us(w[0], xa.x, 0);
        s = dp4a_us(w[1], xa.y, s);
        s = dp4a_us(w[2], xa.z, s);
        s = dp4a_us(w[3], xa.w, s);
        s = dp4a_us(w[4], xb.x, s);
        s = dp4a_us(w[5], xb.y, s);
        s = dp4a_us(w[6], xb.z, s);
        return dp4a_us(w[7], xb.w, s);
      }
    } else if constexpr (NT == 1) {
      int ia = __dp4a((int)w[0], (int)xa.x, 0);
      int ib = __dp4a((int)w[4], (int)xb.x, 0);
      ia = __dp4a((int)w[1], (int)xa.y, ia);
      ib = __dp4a((int)w[5], (int)xb.y, ib);
      ia = __dp4a((int)w[2], (int)xa.z, ia);
      ib = __dp4a((int)w[6], (int)xb.z, ib);
      ia = __dp4a((int)w[3], (int)xa.w, ia);
      ib = __dp4a((int)w[7], (int)xb.w, ib);
      return ia + ib;
    } else {
      int s = __dp4a((int)w[0], (int)xa.x, 0);
      s = __dp4a((int)w[1], (int)xa.y, s);
      s = __dp4a((int)w[2], (int)xa.z, s);
      s = __dp4a((int)w[3], (int)xa.w, s);
      s = __dp4a((int)w[4], (int)xb.x, s);
      s = __dp4a((int)w[5], (int)xb.y, s);
      s = __dp4a((int)w[6], (int)xb.z, s);
      return __dp4a((int)w[7], (int)xb.w, s);
    }
  }
};

// Two CTAs fit on an SM for small token counts (so that consecutive calls
// overlap under programmatic dependent launch); larger token counts keep more
// accumulators in registers.
// F16 / F32 weights ("Castagna Veloce", section "Kernels for the MI50": the
// small-batch matvec over F16 and F32 weights as well): the activations are
// staged as they are, fp32, and every product and sum is an fp32 FMA.
//
// Stage weights [k0, k0 + nw) of tokens [0, nt) of `src` (k0 and nw
// multiples of 32) into the area, [chunk][slot][kchunk_of(F)] floats, zero
// past nw in the last chunk; slots from nt on are left as they are (the
// consumer never stores their sums).  F16: within each 256-element piece,
// elements 8l .. 8l+3 sit at 4l and 8l+4 .. 8l+7 at 128 + 4l, so that the
// lanes' two 16-byte loads of a piece are each 512 contiguous bytes.  Called
// by all consumer warps.
template <int F, int NT, int CW = CONSUMER_WARPS>
__device__ __forceinline__ void stage_float(const ActSource& src, long long k0, int nw, int nt, const ActArea& a,
                                            int cw, int lane) {
  constexpr int KC = kchunk_of(F), Q = KC / 4;  // float4 per slot chunk
  constexpr int B = 8;                           // loads in flight per thread
  const int nck = (nw + KC - 1) / KC;
  const int per_tok = nck * Q, total = nt * per_tok;
  float4* dst = reinterpret_cast<float4*>(a.q);
  for (int base = cw * 32 + lane; base < total; base += B * CW * 32) {
    float4 v[B];
#pragma unroll
    for (int j = 0; j < B; j++) {  // all loads first
      const int i = base + j * CW * 32;
      v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i < total) {
        const int t = i / per_tok, e4 = i - t * per_tok;  // float4 e4 of the token's range
        if (4 * e4 < nw && QMV_CHECK(in_range(src.row(t) * src.ld + k0 + 4 * e4, 4, src.x_len, src.err)))
          v[j] = __ldg(reinterpret_cast<const float4*>(src.x + src.row(t) * src.ld + k0) + e4);
      }
    }
#pragma unroll
    for (int j = 0; j < B; j++) {
      const int i = base + j * CW * 32;
      if (i < total) {
        const int t = i / per_tok, e4 = i - t * per_tok, c = e4 / Q;
        int o = e4 - c * Q;  // float4 within the chunk
        if constexpr (F == QMV_F16) o = (o & ~63) | ((o & 1) << 5) | ((o >> 1) & 31);
        if (QMV_CHECK(smem_in_range(dst + ((size_t)c * NT + t) * Q + o, 16, src.err))) dst[((size_t)c * NT + t) * Q + o] = v[j];
      }
    }
  }
}

// Consumer step for F16 / F32 rows: a row chunk (2048 bytes) is four
// 512-byte pieces; in piece s lane l takes the 16 bytes at 512 s + 16 l, that
// is 8 F16 or 4 F32 weights at element E s + (E / 32) l (E: weights per
// piece), paired with the same elements of every token's activations.
template <int F, int NT>
struct FloatConsumer {
  uint32_t w_off, x_off;  // the lane's bytes in a row chunk / a token's chunk of activations
  __device__ explicit FloatConsumer(int lane) {
    w_off = 16 * lane;
    x_off = 16 * lane;  // F16: and 512 bytes further (the staging's order)
  }
  template <int PAIR_STRIDE = 2 * chunk_bytes<F>()>
  __device__ __forceinline__ void chunk(uint32_t row0, uint32_t aq, uint32_t ad, uint32_t as, int nt,
                                        AccTile<NT>& acc) const {
    (void)ad;
    (void)as;
    constexpr int CB = chunk_bytes<F>();
    constexpr int EL = F == QMV_F16 ? 8 : 4;     // weights per lane per piece
    constexpr uint32_t sq = kchunk_of(F) * 4;   // bytes of a token slot's chunk
    // the pieces stay a loop: unrolled, the step's code (up to 2048 FMAs
    // for 16 tokens) outgrows the instruction cache
#pragma unroll 1
    for (int s = 0; s < 4; s++) {
      float w[RW][EL];
#pragma unroll
      for (int r = 0; r < RW; r++) {
        const uint4 q = lds128(row0 + (r & 1) * CB + (r >> 1) * PAIR_STRIDE + 512 * s + w_off);
        if constexpr (F == QMV_F16) {
          const uint32_t qq[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
          for (int i = 0; i < 4; i++) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&qq[i]));
            w[r][2 * i] = f.x;
            w[r][2 * i + 1] = f.y;
          }
        } else {
          w[r][0] = __uint_as_float(q.x);
          w[r][1] = __uint_as_float(q.y);
          w[r][2] = __uint_as_float(q.z);
          w[r][3] = __uint_as_float(q.w);
        }
      }
      const uint32_t xp = aq + 4 * EL * 32 * s + x_off;  // piece s of the token's chunk
      // tokens in pairs (slot t + 1 past nt holds stale values: its sums are
      // never stored), 2 RW independent chains
#pragma unroll
      for (int t = 0; t < NT; t += 2) {
        if (t >= nt) break;
        float xa[EL], xb[EL];
        load_x(xp + t * sq, xa);
        if constexpr (NT > 1) load_x(xp + (t + 1) * sq, xb);
#pragma unroll
        for (int i = 0; i < EL; i++)
#pragma unroll
          for (int r = 0; r < RW; r++) {
            acc.v[r][t >> 1].x = fmaf(w[r][i], xa[i], acc.v[r][t >> 1].x);
            if constexpr (NT > 1) acc.v[r][t >> 1].y = fmaf(w[r][i], xb[i], acc.v[r][t >> 1].y);
          }
      }
    }
  }

  template <int EL>
  static __device__ __forceinline__ void load_x(uint32_t a, float (&xv)[EL]) {
    const uint4 x0 = lds128(a);
    xv[0] = __uint_as_float(x0.x);
    xv[1] = __uint_as_float(x0.y);
    xv[2] = __uint_as_float(x0.z);
    xv[3] = __uint_as_float(x0.w);
    if constexpr (EL == 8) {
      const uint4 x1 = lds128(a + 512);
      xv[4] = __uint_as_float(x1.x);
      xv[5] = __uint_as_float(x1.y);
      xv[6] = __uint_as_float(x1.z);
      xv[7] = __uint_as_float(x1.w);
    }
  }
};

// The consumer of format F.
template <int F, int NT>
struct ConsumerSel {
  using type = Consumer<F, NT>;
};
template <int NT>
struct ConsumerSel<QMV_F16, NT> {
  using type = FloatConsumer<QMV_F16, NT>;
};
template <int NT>
struct ConsumerSel<QMV_F32, NT> {
  using type = FloatConsumer<QMV_F32, NT>;
};
template <int F, int NT>
using ConsumerOf = typename ConsumerSel<F, NT>::type;

template <int NT, int CW = CONSUMER_WARPS>
constexpr int dense_min_blocks() {
  return NT <= 4 && CW == CONSUMER_WARPS ? 2 : 1;
}

// Sums over the 32 lanes of V per-lane values v[0 .. V) (V a power of two),
// as a butterfly: each of the first log2(V) steps (at most 5) exchanges half
// of the values with the partner lane and keeps the other half, so the
// values are spread over the lanes instead of each being reduced on its
// own.  Afterwards v[0 .. max(V / 32, 1)) hold the sums of values idx, idx +
// 1, ... (idx returned); for V < 32 the 32 / V lanes of a group hold the same
// sums.  Unrolled by template, so every index is a constant.
template <int V, int STEP>
struct LaneButterfly {
  static __device__ __forceinline__ void run(float (&v)[V], int lane, int& idx) {
    constexpr int OFF = 16 >> STEP;
    constexpr int CNT = (V >> STEP) > 1 ? (V >> STEP) : 1;  // values still held before this step
    if constexpr (CNT > 1) {
      constexpr int H = CNT / 2;
      const bool up = (lane & OFF) != 0;
#pragma unroll
      for (int i = 0; i < H; i++) {
        const float keep = up ? v[i + H] : v[i];
        const float send = up ? v[i] : v[i + H];
        v[i] = keep + __shfl_xor_sync(FULL, send, OFF);
      }
      if (up) idx += H;
    } else {
      v[0] += __shfl_xor_sync(FULL, v[0], OFF);
    }
    if constexpr (STEP < 4) LaneButterfly<V, STEP + 1>::run(v, lane, idx);
  }
};

// Sum of v over the 32 lanes, returned in every lane.
__device__ __forceinline__ float warp_sum(float v) {
  v += __shfl_xor_sync(FULL, v, 16);
  v += __shfl_xor_sync(FULL, v, 8);
  v += __shfl_xor_sync(FULL, v, 4);
  v += __shfl_xor_sync(FULL, v, 2);
  v += __shfl_xor_sync(FULL, v, 1);
  return v;
}

// Pipeline barriers of a CTA: init by thread 0, then __syncthreads.
__device__ __forceinline__ void init_pipeline(uint64_t* full, uint64_t* empty, int stages,
                                              int consumers = CONSUMER_WARPS) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; s++) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], consumers);
    }
    fence_mbar_init();
  }
  __syncthreads();
}

// Position in the stage ring: iteration n uses stage st = n % stages in round
// n / stages (tracked incrementally; the full barrier of round r completes
// phase r, i.e. parity r & 1).
struct Ring {
  int st = 0, round = 0;
  long long n = 0;
  __device__ __forceinline__ void advance(int stages) {
    n++;
    if (++st == stages) {
      st = 0;
      round++;
    }
  }
  __device__ __forceinline__ uint32_t parity() const { return (uint32_t)(round & 1); }
};

// Producer side: wait until the ring's current stage is free.
__device__ __forceinline__ bool producer_acquire(uint64_t* empty, const Ring& r, int stages, unsigned* err) {
  if (r.n < stages) return true;
  return mbar_wait(&empty[r.st], (uint32_t)((r.round - 1) & 1), err);
}

// Producer side, before leaving: wait (bounded) for the copies of the last
// `stages` iterations, so no copy lands in shared memory after exit.
__device__ __forceinline__ void producer_drain(uint64_t* full, long long issued, int stages, unsigned* err) {
  const long long first = issued > stages ? issued - stages : 0;
  for (long long j = first; j < issued; j++) mbar_wait(&full[j % stages], (uint32_t)((j / stages) & 1), err);
}

}  // namespace qmv
