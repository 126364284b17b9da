// C ABI of the library (declared in include/qmv.h): argument checking, launch
// geometry, TMA descriptors and kernel dispatch.  Nothing here allocates.
#include <cudaTypedefs.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include <cmath>

#include "launch.h"
#include "moe_kernels.cuh"
#include "qmv_dense.cuh"

namespace qmv {

static __device__ unsigned int g_qmv_error = 0;


// ---------------------------------------------------------------------------
// Device facts (cached per device ordinal).
// ---------------------------------------------------------------------------
struct DevInfo {
  int sms = 0, smem_optin = 0, major = 0, minor = 0;
  unsigned* err = nullptr;
  bool ok = false;
};
static DevInfo g_dev[64];
static std::mutex g_dev_mu;

static const DevInfo* dev_info() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (!d.ok) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return nullptr;
    if (cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return nullptr;
    cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev);
    void* ep = nullptr;
    if (cudaGetSymbolAddress(&ep, g_qmv_error) == cudaSuccess) d.err = static_cast<unsigned*>(ep);
    d.ok = true;
  }
  return &d;
}

int device_smem_optin() {
  const DevInfo* d = dev_info();
  return d ? d->smem_optin : 0;
}
unsigned* device_error_word() {
  const DevInfo* d = dev_info();
  return d ? d->err : nullptr;
}
int device_sm_count() {
  const DevInfo* d = dev_info();
  return d ? d->sms : 1;
}

static std::atomic<long long> g_output_shrink{0};
long long output_extent(long long n) {
  const long long v = n - g_output_shrink.load(std::memory_order_relaxed);
  return v > 0 ? v : 0;
}

// ---------------------------------------------------------------------------
// Tensor-map encoder from the driver, reached through the runtime (no link
// against libcuda).
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::once_flag g_encode_once;

static PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

// 2-D map over a weight matrix seen as rows x (row_bytes / 8) 8-byte
// elements; box = box_rows x (box_bytes / 8).
bool encode_rows(CUtensorMap* map, const void* W, long long rows, long long row_bytes, int box_bytes,
                 int box_rows) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)(row_bytes / 8), (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  cuuint32_t box[2] = {(cuuint32_t)(box_bytes / 8), (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void*>(W), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ---------------------------------------------------------------------------
// Validation helpers.
// ---------------------------------------------------------------------------
static int group_weights(int fmt) {
  if (is_float(fmt)) return 32;
  return fmt == QMV_IQ4_XS || fmt == QMV_Q8_G64 ? 512 : (fmt == QMV_Q8_G128 ? 1024 : 256);
}
static int group_bytes(int fmt) {
  switch (fmt) {
    case QMV_F16: return 64;
    case QMV_F32: return 128;
    case QMV_Q4_K: return 144;
    case QMV_Q5_K: return 176;
    case QMV_Q6_K: return 208;
    case QMV_Q8_G64: return 528;
    case QMV_Q8_G128: return 1040;
  }
  return 272;  // Q8_0, IQ4_XS
}
static int chunk_bytes_of(int fmt) { return (kchunk_of(fmt) / group_weights(fmt)) * group_bytes(fmt); }
static bool fmt_ok(int fmt) {
  return fmt >= QMV_Q8_0 && fmt <= QMV_F32;
}
// formats the MoE kernels are instantiated for
static bool moe_fmt_ok(int fmt) { return fmt == QMV_Q8_0 || fmt == QMV_Q4_K || fmt == QMV_IQ4_XS; }
static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
constexpr long long MAX_K = 1ll << 20;
// fp32 activations of a split range that split-K choices give F16 / F32
// rows (for one pass of up to 16 tokens): they fit beside two weight stages
constexpr long long FLOAT_ACT_BYTES = 96 * 1024;
constexpr long long MAX_M = 1ll << 30;

static int check_device() {
  const DevInfo* d = dev_info();
  if (!d) return QMV_ERR_CUDA;
  if (d->major != 10 || d->minor != 3) return QMV_ERR_DEVICE;
  return QMV_OK;
}

// ---------------------------------------------------------------------------
// Dense / split-K launch planning.
// ---------------------------------------------------------------------------
struct Plan {
  int nt_tmpl, stages, grid;
  int cw, tile_rows;
  int act_nck;
  size_t smem;
};

// Shared memory a CTA may take so that two fit on one SM (each CTA also
// carries 1 KB reserved by the system).
constexpr size_t TWO_PER_SM_BYTES = 112 * 1024;
constexpr int TWO_PER_SM_STAGES = 4;

// Stage count and shared-memory size for an activation area of `act` bytes:
// small token counts aim for two CTAs per SM (so that consecutive calls
// overlap under programmatic dependent launch) with a short ring; otherwise
// one CTA per SM with a deeper ring.
static bool plan_stages(int nt, int cw, size_t act, int stage_bytes, size_t budget, int& stages, size_t& smem) {
  // mbarriers (full, empty, 2 more) and the cross-warp sums of thin tiles
  const size_t fixed = act + 2 * MAX_STAGES * sizeof(uint64_t) + 128 + (size_t)cw * RW * 16 * sizeof(float);
  if (nt <= 4 && cw == 8 && fixed + 2 * (size_t)stage_bytes <= TWO_PER_SM_BYTES) {  // two CTAs per SM
    int st = (int)((TWO_PER_SM_BYTES - fixed) / stage_bytes);
    stages = st > TWO_PER_SM_STAGES ? TWO_PER_SM_STAGES : st;
  } else if (fixed + 2 * (size_t)stage_bytes <= budget) {
    // one CTA per SM; twelve warps with up to 4 token slots still take at
    // most 4 stages (deeper rings only queue weight reads ahead of the
    // activation staging)
    const int cap = nt <= 4 && cw == 12 ? TWO_PER_SM_STAGES : MAX_STAGES;
    int st = (int)((budget - fixed) / stage_bytes);
    stages = st > cap ? cap : st;
  } else {
    return false;
  }
  smem = (size_t)stages * stage_bytes + fixed;
  return true;
}

// Choose the compiled token count and the number of stages so that the
// activation area plus at least two weight stages fit in shared memory.
static bool plan_dense(int fmt, long long M, long long K, int n_tok, int n_split, bool q8in, Plan& pl) {
  const int gw = group_weights(fmt);
  const long long groups = K / gw;
  const long long max_range = ((groups + n_split - 1) / n_split) * gw;  // weights
  pl.act_nck = (int)((max_range + kchunk_of(fmt) - 1) / kchunk_of(fmt));
  const size_t budget = (size_t)device_smem_optin();
  int nt = 16;
  while (nt > n_tok && nt > 1) nt >>= 1;
  if (nt < n_tok && nt < 16) nt <<= 1;  // smallest power of two >= n_tok (<= 16)
  // Twelve consumer warps where their tiles fit, else eight (F16 / F32 rows:
  // eight), from 8 tokens on and at 4 tokens; at 4 tokens with pre-quantized
  // activations on a tall matrix (8+ units of rows per SM) two CTAs of eight
  // per SM instead.  Measured on GB300 at 4 tokens, pre-quantized: Q4_K 17408
  // x 5120 17.0 us with two CTAs of eight against 17.8 with twelve, Q4_K 5120
  // x 5120 10.3 against 9.7, IQ4_XS 6144 x 2048 7.9 against 6.8; at 3 tokens
  // (staged from fp32, where the eight-warp kernel spills) twelve always:
  // Q4_K 17408 x 5120 18.4 -> 16.4, Q6_K 21.3 -> 18.4, Q4_K 5120 x 5120 11.5
  // -> 8.5, IQ4_XS 2048 x 6144 10.5 -> 7.7.
  const long long work_units = (M + UNIT_ROWS - 1) / UNIT_ROWS * n_split;
  const bool twelve_at_4 = !(q8in && work_units >= 8ll * device_sm_count());
  for (;; nt >>= 1) {
    bool ok = false;
    for (int cw = !is_float(fmt) && (nt >= 8 || (nt == 4 && twelve_at_4)) ? 12 : 8; cw >= 8 && !ok; cw -= 4) {
      pl.cw = cw;
      pl.tile_rows = cw * RW;
      ok = plan_stages(nt, cw, act_area_bytes(fmt, nt, pl.act_nck), pl.tile_rows * chunk_bytes_of(fmt), budget,
                       pl.stages, pl.smem);
    }
    if (ok) break;
    if (nt == 1) return false;
  }
  pl.nt_tmpl = nt;
  const long long units = (M + UNIT_ROWS - 1) / UNIT_ROWS;
  const long long work = units * n_split;
  // two CTAs per SM when they fit (more warps to hide latency), else one
  const int ctas = device_sm_count() * (pl.smem <= TWO_PER_SM_BYTES && nt <= 4 && pl.cw == 8 ? 2 : 1);
  pl.grid = (int)(work < ctas ? work : ctas);
  return true;
}

static cudaError_t launch_dense_any(int fmt, const DenseLaunch& L) {
  switch (fmt) {
    case QMV_Q8_0: return launch_dense_q8_0(L);
    case QMV_Q4_K: return launch_dense_q4_k(L);
    case QMV_Q5_K: return launch_dense_q5_k(L);
    case QMV_Q6_K: return launch_dense_q6_k(L);
    case QMV_Q8_G64: return launch_dense_q8_g64(L);
    case QMV_Q8_G128: return launch_dense_q8_g128(L);
    case QMV_F16: return launch_dense_f16(L);
    case QMV_F32: return launch_dense_f32(L);
    default: return launch_dense_iq4_xs(L);
  }
}

// Runs pass 1 (all token passes) writing `out` (y, or the split partials).
static int run_dense(int fmt, const void* W, const float* x, const int8_t* xq, const float* xd, const int32_t* xs,
                     float* out, long long M, long long K, int n_tok, int n_split, cudaStream_t stream,
                     const float* add = nullptr) {
  Plan pl;
  if (!plan_dense(fmt, M, K, n_tok, n_split, xq != nullptr, pl)) return QMV_ERR_SHAPE;
  const long long rb = qmv_row_bytes(fmt, K);
  DenseLaunch L;
  if (!encode_rows(&L.map_tile, W, M, rb, chunk_bytes_of(fmt), pl.tile_rows)) return QMV_ERR_CUDA;
  if (!encode_rows(&L.map_unit, W, M, rb, chunk_bytes_of(fmt), UNIT_ROWS)) return QMV_ERR_CUDA;
  DenseParams p;
  p.x = x;
  p.xq = xq;
  p.xd = xd;
  p.xs = xs;
  p.out = out;
  p.add = n_split == 1 ? add : nullptr;
  p.M = M;
  p.K = (int)K;
  p.ntot = n_tok;
  p.n_split = n_split;
  p.groups = (int)(K / group_weights(fmt));
  p.units = (int)((M + UNIT_ROWS - 1) / UNIT_ROWS);
  p.stages = pl.stages;
  p.act_nck = pl.act_nck;
  // L2 lookahead only for small matrices (a few microseconds of HBM time):
  // there the CTAs' tiles past the ring are requested at the start of the call
  p.prefetch = M * rb <= PREFETCH_ALL_BYTES ? PREFETCH_STAGES : 0;
  p.err = device_error_word();
  p.w = static_cast<const uint8_t*>(W);
  p.rb = rb;
  p.nbmax = 0;
  // y is the caller's result; split partials live in the workspace
  QMV_DEBUG_ONLY(p.x_len = (long long)n_tok * K;
                 p.out_len = n_split == 1 ? output_extent((long long)n_tok * M) : (long long)n_split * n_tok * M;
                 p.add_len = p.add ? (long long)n_tok * M : 0;)
  L.p = &p;
  L.nt_tmpl = pl.nt_tmpl;
  L.cw = pl.cw;
  L.grid = pl.grid;
  L.smem = pl.smem;
  L.stream = stream;
  L.pdl = true;
  // Q4_K passes of 8 or 16 token slots: the tensor-core kernel, whenever its
  // shared memory (activation area, partial sums and at least two weight
  // stages) fits and the matrix is tall enough to repay its larger fixed cost
  // per call (measured on K = 5120: it overtakes the dp4a kernel from about
  // 7000 rows at 8 tokens and 5800 rows at 16); it takes one CTA per SM.
  bool mma = false;
  const long long mma_min_rows = pl.nt_tmpl == 8 ? 7168 : 6144;
  if (fmt == QMV_Q4_K && pl.nt_tmpl >= 8 && rb >= MMA_BOX_BYTES && M >= mma_min_rows) {
    const int nbmax = (int)(((p.groups + n_split - 1) / n_split) * 8);
    int st = MAX_STAGES;
    while (st >= 2 && mma_smem_bytes(pl.nt_tmpl, st, nbmax) > (size_t)device_smem_optin()) st--;
    CUtensorMap mt, mu;
    if (st >= 2 && encode_rows(&mt, W, M, rb, MMA_BOX_BYTES, MMA_TILE_ROWS) &&
        encode_rows(&mu, W, M, rb, MMA_BOX_BYTES, UNIT_ROWS)) {
      mma = true;
      L.map_tile = mt;
      L.map_unit = mu;
      p.nbmax = nbmax;
      p.stages = st;
      L.smem = mma_smem_bytes(pl.nt_tmpl, st, nbmax);
      const long long work = (long long)p.units * n_split;
      L.grid = (int)(work < device_sm_count() ? work : device_sm_count());
    }
  }
  // F16 rows, passes of 8 or 16 token slots: the tensor-core F16 kernel when
  // the split range's two f16 parts of the activations fit beside at least
  // two weight stages, and the matrix is tall enough for its fixed cost
  bool mma_f16 = false;
  if (fmt == QMV_F16 && pl.nt_tmpl >= 8 && rb >= MMA_F16_BOX_BYTES && M >= 4096) {
    const int kmax = (int)(((p.groups + n_split - 1) / n_split) * 32);
    int st = MAX_STAGES;
    while (st >= 2 && mma_f16_smem_bytes(pl.nt_tmpl, st, kmax) > (size_t)device_smem_optin()) st--;
    CUtensorMap mt, mu;
    if (st >= 2 && encode_rows(&mt, W, M, rb, MMA_F16_BOX_BYTES, MMA_TILE_ROWS) &&
        encode_rows(&mu, W, M, rb, MMA_F16_BOX_BYTES, UNIT_ROWS)) {
      mma_f16 = true;
      L.map_tile = mt;
      L.map_unit = mu;
      p.nbmax = kmax / 32;
      p.stages = st;
      L.smem = mma_f16_smem_bytes(pl.nt_tmpl, st, kmax);
      const long long work = (long long)p.units * n_split;
      L.grid = (int)(work < device_sm_count() ? work : device_sm_count());
    }
  }
  auto launch = [&]() {
    return mma ? launch_mma_q4_k(L) : (mma_f16 ? launch_mma_f16(L) : launch_dense_any(fmt, L));
  };
  // the full token passes in one launch (grid y), so that they run side by
  // side, and a last partial pass in a second one
  const int full = n_tok / pl.nt_tmpl, rem = n_tok - full * pl.nt_tmpl;
  if (full > 0) {
    p.t0 = 0;
    p.nt = pl.nt_tmpl;
    L.passes = full;
    if (launch() != cudaSuccess) return QMV_ERR_CUDA;
  }
  if (rem > 0) {
    p.t0 = full * pl.nt_tmpl;
    p.nt = rem;
    L.passes = 1;
    if (launch() != cudaSuccess) return QMV_ERR_CUDA;
  }
  return QMV_OK;
}

static int check_dense_args(int fmt, const void* W, const void* x, const float* y, long long M, long long K,
                            int n_tok) {
  if (!fmt_ok(fmt)) return QMV_ERR_FORMAT;
  if (M <= 0 || M > MAX_M || K <= 0 || K > MAX_K || K % group_weights(fmt)) return QMV_ERR_SHAPE;
  if (n_tok < 1 || n_tok > QMV_MAX_TOKENS) return QMV_ERR_NTOK;
  if (!W || !x || !y) return QMV_ERR_NULL;
  if (!aligned16(W) || !aligned16(x) || !aligned16(y)) return QMV_ERR_ALIGN;
  return QMV_OK;
}

// ---------------------------------------------------------------------------
// MoE planning.
// ---------------------------------------------------------------------------
constexpr int MOE_NOFF = 5;

static size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// Workspace: [0] h f32 [S][F], [1] hq i8 [S][F], [2] hd f32 [S][F/32],
// [3] hs i32 [S][F/32], [4] o f32 [S][H]; S = n_tok * top_k.
static size_t moe_layout(const moe_experts* e, int n_tok, int top_k, size_t off[MOE_NOFF]) {
  const size_t S = (size_t)n_tok * top_k, F = (size_t)e->ffn, H = (size_t)e->hidden;
  const size_t sizes[MOE_NOFF] = {S * F * 4, S * F, S * (F / 32) * 4, S * (F / 32) * 4, S * H * 4};
  size_t cur = 0;
  for (int i = 0; i < MOE_NOFF; i++) {
    off[i] = cur;
    cur = align256(cur + sizes[i]);
  }
  return cur;
}

static int check_moe_shape(const moe_experts* e, int n_tok, int top_k) {
  if (!e) return QMV_ERR_NULL;
  if (!moe_fmt_ok(e->fmt_gate_up) || !moe_fmt_ok(e->fmt_down)) return QMV_ERR_FORMAT;
  if (e->n_experts < 1 || e->n_experts > MOE_MAX_EXPERTS || e->hidden <= 0 || e->ffn <= 0 ||
      e->hidden > MAX_K || e->ffn > MAX_K || e->hidden % group_weights(e->fmt_gate_up) ||
      e->ffn % group_weights(e->fmt_down) || e->hidden % UNIT_ROWS || e->ffn % UNIT_ROWS)
    return QMV_ERR_SHAPE;
  if ((long long)e->n_experts * 2 * e->ffn > MAX_M || (long long)e->n_experts * e->hidden > MAX_M)
    return QMV_ERR_SHAPE;
  if (n_tok < 1 || n_tok > QMV_MAX_TOKENS || top_k < 1 || top_k > QMV_MAX_TOPK || top_k > e->n_experts)
    return QMV_ERR_NTOK;
  return QMV_OK;
}

static cudaError_t launch_moe_any(int mode, int fmt, const MoeLaunch& L) {
  if (mode == MOE_GATE_UP) {
    switch (fmt) {
      case QMV_Q8_0: return launch_moe_gate_up_q8_0(L);
      case QMV_Q4_K: return launch_moe_gate_up_q4_k(L);
      default: return launch_moe_gate_up_iq4_xs(L);
    }
  }
  switch (fmt) {
    case QMV_Q8_0: return launch_moe_down_q8_0(L);
    case QMV_Q4_K: return launch_moe_down_q4_k(L);
    default: return launch_moe_down_iq4_xs(L);
  }
}

// One expert-grouped projection: weights `pool` (E experts x pool_rows rows
// of K weights in format fmt).
static int run_moe_proj(int mode, int fmt, const void* pool, MoeParams& p, int nt, cudaStream_t stream) {
  const long long rb = qmv_row_bytes(fmt, p.K);
  const long long rows = (long long)p.n_experts * p.pool_rows;
  MoeLaunch L;
  p.act_nck = (p.K + KCHUNK - 1) / KCHUNK;
  p.groups = p.K / group_weights(fmt);
  // the routing tables are static shared memory: count them with the
  // activation area when sizing, and leave them out of the dynamic size
  const size_t static_bytes = sizeof(MoeRouting) + 16 * sizeof(int) + 256;
  size_t smem = 0;
  // from 8 token slots on twelve consumer warps (beside a producer warpgroup
  // that hands its registers to them) where their tiles fit, else eight
  bool ok = false;
  for (int cw = nt >= 8 ? 12 : 8; cw >= 8 && !ok; cw -= 4) {
    L.cw = cw;
    ok = plan_stages(nt, cw, act_area_bytes(fmt, nt, p.act_nck) + static_bytes, cw * RW * chunk_bytes_of(fmt),
                     (size_t)device_smem_optin(), p.stages, smem);
  }
  if (!ok) return QMV_ERR_SHAPE;
  if (!encode_rows(&L.map_tile, pool, rows, rb, chunk_bytes_of(fmt), L.cw * RW)) return QMV_ERR_CUDA;
  if (!encode_rows(&L.map_unit, pool, rows, rb, chunk_bytes_of(fmt), UNIT_ROWS)) return QMV_ERR_CUDA;
  L.p = &p;
  L.nt_tmpl = nt;
  L.grid = device_sm_count() * (nt <= 4 && smem <= TWO_PER_SM_BYTES ? 2 : 1);
  L.smem = smem - static_bytes;
  L.stream = stream;
  L.pdl = true;
  return launch_moe_any(mode, fmt, L) == cudaSuccess ? QMV_OK : QMV_ERR_CUDA;
}

}  // namespace qmv

using namespace qmv;

extern "C" {

int64_t qmv_row_bytes(int fmt, int64_t K) {
  if (!fmt_ok(fmt)) return QMV_ERR_FORMAT;
  if (K <= 0 || K > MAX_K || K % group_weights(fmt)) return QMV_ERR_SHAPE;
  return (K / group_weights(fmt)) * group_bytes(fmt);
}

int qmv_quantize_weights(int fmt, const float* w, int64_t M, int64_t K, void* W, cudaStream_t stream) {
  if (!fmt_ok(fmt)) return QMV_ERR_FORMAT;
  if (M <= 0 || M > MAX_M || K <= 0 || K > MAX_K || K % group_weights(fmt)) return QMV_ERR_SHAPE;
  if (!w || !W) return QMV_ERR_NULL;
  if (!aligned16(w) || !aligned16(W)) return QMV_ERR_ALIGN;
  int rc = check_device();
  if (rc) return rc;
  return launch_quantize_weights(fmt, w, M, (int)K, W, stream) == cudaSuccess ? QMV_OK : QMV_ERR_CUDA;
}

int qmv_quantize_act(const float* x, int64_t K, int n_tok, int8_t* q, float* d, int32_t* sum,
                     cudaStream_t stream) {
  if (K <= 0 || K > MAX_K || K % 256) return QMV_ERR_SHAPE;
  if (n_tok < 1 || n_tok > QMV_MAX_TOKENS) return QMV_ERR_NTOK;
  if (!x || !q || !d || !sum) return QMV_ERR_NULL;
  if (!aligned16(x) || !aligned16(q) || !aligned16(d) || !aligned16(sum)) return QMV_ERR_ALIGN;
  int rc = check_device();
  if (rc) return rc;
  return launch_act_quant(x, (int)K, n_tok, q, d, sum, output_extent((long long)n_tok * K), stream, true) ==
                 cudaSuccess
             ? QMV_OK
             : QMV_ERR_CUDA;
}

int qmv_run(int fmt, const void* W, const float* x, float* y, int64_t M, int64_t K, int n_tok,
            cudaStream_t stream) {
  int rc = check_dense_args(fmt, W, x, y, M, K, n_tok);
  if (rc) return rc;
  if ((rc = check_device())) return rc;
  return run_dense(fmt, W, x, nullptr, nullptr, nullptr, y, M, K, n_tok, 1, stream);
}

int qmv_run_q8(int fmt, const void* W, const int8_t* xq, const float* xd, const int32_t* xs, float* y, int64_t M,
               int64_t K, int n_tok, cudaStream_t stream) {
  int rc = check_dense_args(fmt, W, xq, y, M, K, n_tok);
  if (rc) return rc;
  if (is_float(fmt)) return QMV_ERR_FORMAT;  // F16 / F32 rows take fp32 activations
  if (!xd || !xs) return QMV_ERR_NULL;
  if (!aligned16(xd) || !aligned16(xs)) return QMV_ERR_ALIGN;
  if ((rc = check_device())) return rc;
  return run_dense(fmt, W, nullptr, xq, xd, xs, y, M, K, n_tok, 1, stream);
}

int qmv_splitk_choose(int fmt, int64_t M, int64_t K, int n_tok) {
  if (!fmt_ok(fmt)) return QMV_ERR_FORMAT;
  if (M <= 0 || K <= 0 || K % group_weights(fmt)) return QMV_ERR_SHAPE;
  const long long units = (M + UNIT_ROWS - 1) / UNIT_ROWS;
  const long long want = 2ll * device_sm_count();  // >= 2 row units per SM
  // F16 / F32 rows stage a split's fp32 activations whole: enough splits for
  // one pass of the tokens (up to 16) to fit in FLOAT_ACT_BYTES
  const long long kc = kchunk_of(fmt), chunks = (K + kc - 1) / kc;
  long long fmin = 1;
  if (is_float(fmt)) {
    long long nt = 1;
    while (nt < n_tok && nt < 16) nt <<= 1;
    fmin = (K * nt * 4 + FLOAT_ACT_BYTES - 1) / FLOAT_ACT_BYTES;
  }
  if (units >= want && fmin <= 1) return 1;
  long long target = units >= want ? 1 : (want + units - 1) / units;
  if (target < fmin) target = fmin;
  if (target > 64) target = 64;
  // smallest divisor of the chunk count that reaches the target, so that
  // every split covers whole chunks
  for (long long s = target; s <= 64 && s <= chunks; s++)
    if (chunks % s == 0) return (int)s;
  return (int)(target < chunks ? target : chunks);
}

size_t qmv_splitk_workspace_bytes(int64_t M, int n_tok, int n_split) {
  if (M <= 0 || n_tok <= 0 || n_split <= 0) return 0;
  return (size_t)n_split * n_tok * M * sizeof(float);
}

size_t qmv_act_q8_bytes(int64_t K, int n_tok) {
  if (K <= 0 || K > MAX_K || K % 256 || n_tok < 1 || n_tok > QMV_MAX_TOKENS) return 0;
  const size_t nb = (size_t)n_tok * (size_t)(K / 32);
  return align256((size_t)n_tok * (size_t)K) + 2 * align256(nb * 4);
}

// Split-K matvec (n_split 0: chosen from the shape), y = What Xhat (+ add).
static int splitk_impl(int fmt, const void* W, const float* x, const float* add, float* y, int64_t M, int64_t K,
                       int n_tok, int n_split, void* ws, size_t ws_bytes, cudaStream_t stream) {
  int rc = check_dense_args(fmt, W, x, y, M, K, n_tok);
  if (rc) return rc;
  if (n_split < 0 || n_split > 256 || n_split > K / group_weights(fmt)) return QMV_ERR_SHAPE;
  if (n_split > 1) {
    if (!ws) return QMV_ERR_NULL;
    if (!aligned16(ws)) return QMV_ERR_ALIGN;
    if (ws_bytes < qmv_splitk_workspace_bytes(M, n_tok, n_split)) return QMV_ERR_WORKSPACE;
  }
  if ((rc = check_device())) return rc;
  if (n_split == 0) {
    n_split = qmv_splitk_choose(fmt, M, K, n_tok);
    if (n_split > 1) {
      if (!ws) return QMV_ERR_NULL;
      if (!aligned16(ws)) return QMV_ERR_ALIGN;
      if (ws_bytes < qmv_splitk_workspace_bytes(M, n_tok, n_split)) return QMV_ERR_WORKSPACE;
    }
  }
  // With room after the partial sums and more than 4 tokens, the activations
  // are quantized once into the workspace (one more launch) and every CTA
  // brings its range in by bulk copies; otherwise each CTA quantizes its
  // range while staging.  Same arithmetic, bitwise equal results.  Measured
  // on GB300 (graph replay): up to 4 tokens staging from fp32 is faster on
  // every shape (Q4_K 17408 x 5120 16.2 against 16.5 us, IQ4_XS 6144 x 2048
  // 5.2 against 6.5); at 5-8 tokens it is faster for one split of K <= 4096
  // below the 8-slot tensor-core kernel's height (IQ4_XS 6144 x 2048 7.6
  // against 8.4, Q8_0 4096 x 4096 9.4 against 9.8) and slower above (Q4_K
  // 5120 x 5120 12.9 against 12.6); at 16 tokens quantizing once wins.
  const size_t part = n_split > 1 ? align256(qmv_splitk_workspace_bytes(M, n_tok, n_split)) : 0;
  const size_t q8 = qmv_act_q8_bytes(K, n_tok);
  const int8_t* xq = nullptr;
  const float* xd = nullptr;
  const int32_t* xs = nullptr;
  const bool stage_fp32 = n_tok <= 4 || (n_tok <= 8 && n_split == 1 && K <= 4096 && M < 7168);
  if (!stage_fp32 && !is_float(fmt) && ws && aligned16(ws) && q8 && ws_bytes >= part + q8) {
    uint8_t* base = static_cast<uint8_t*>(ws) + part;
    const size_t nb = (size_t)n_tok * (size_t)(K / 32);
    int8_t* q = reinterpret_cast<int8_t*>(base);
    float* d = reinterpret_cast<float*>(base + align256((size_t)n_tok * (size_t)K));
    int32_t* sm = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(d) + align256(nb * 4));
    if (launch_act_quant(x, (int)K, n_tok, q, d, sm, (long long)n_tok * K, stream, true) != cudaSuccess)
      return QMV_ERR_CUDA;
    xq = q;
    xd = d;
    xs = sm;
  }
  const float* xf = xq ? nullptr : x;
  if (n_split == 1) return run_dense(fmt, W, xf, xq, xd, xs, y, M, K, n_tok, 1, stream, add);
  float* partial = static_cast<float*>(ws);
  rc = run_dense(fmt, W, xf, xq, xd, xs, partial, M, K, n_tok, n_split, stream);
  if (rc) return rc;
  return launch_splitk_reduce(partial, y, add, M, n_tok, n_split, stream, true) == cudaSuccess ? QMV_OK
                                                                                                : QMV_ERR_CUDA;
}

int qmv_splitk_run(int fmt, const void* W, const float* x, float* y, int64_t M, int64_t K, int n_tok, int n_split,
                   void* ws, size_t ws_bytes, cudaStream_t stream) {
  return splitk_impl(fmt, W, x, nullptr, y, M, K, n_tok, n_split, ws, ws_bytes, stream);
}

int qmv_run_residual(int fmt, const void* W, const float* x, const float* r, float* y, int64_t M, int64_t K,
                     int n_tok, int n_split, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!r) return QMV_ERR_NULL;
  if (!aligned16(r)) return QMV_ERR_ALIGN;
  return splitk_impl(fmt, W, x, r, y, M, K, n_tok, n_split, ws, ws_bytes, stream);
}

int qmv_run_siblings(int count, const int* fmts, const void* const* W, const int64_t* M, float* const* y,
                     const float* x, int64_t K, int n_tok, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (count < 1 || count > QMV_MAX_SIBLINGS) return QMV_ERR_SHAPE;
  if (!fmts || !W || !M || !y) return QMV_ERR_NULL;
  int rc;
  for (int i = 0; i < count; i++)
    if ((rc = check_dense_args(fmts[i], W[i], x, y[i], M[i], K, n_tok))) return rc;
  // F16 / F32 siblings take x as it is; the others share one quantization
  bool quant = false;
  for (int i = 0; i < count; i++) quant = quant || !is_float(fmts[i]);
  const size_t q8 = qmv_act_q8_bytes(K, n_tok);
  if (n_tok >= 4 && quant) {
    if (!ws) return QMV_ERR_NULL;
    if (!aligned16(ws)) return QMV_ERR_ALIGN;
    if (ws_bytes < q8) return QMV_ERR_WORKSPACE;
  }
  if ((rc = check_device())) return rc;
  if (n_tok < 4 || !quant) {
    // few tokens: every matvec quantizes the activations while staging
    for (int i = 0; i < count; i++)
      if ((rc = run_dense(fmts[i], W[i], x, nullptr, nullptr, nullptr, y[i], M[i], K, n_tok, 1, stream))) return rc;
    return QMV_OK;
  }
  // the activations quantized once, every matvec copies them in
  uint8_t* base = static_cast<uint8_t*>(ws);
  const size_t nb = (size_t)n_tok * (size_t)(K / 32);
  int8_t* q = reinterpret_cast<int8_t*>(base);
  float* d = reinterpret_cast<float*>(base + align256((size_t)n_tok * (size_t)K));
  int32_t* sm = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(d) + align256(nb * 4));
  if (launch_act_quant(x, (int)K, n_tok, q, d, sm, (long long)n_tok * K, stream, true) != cudaSuccess)
    return QMV_ERR_CUDA;
  for (int i = 0; i < count; i++) {
    rc = is_float(fmts[i]) ? run_dense(fmts[i], W[i], x, nullptr, nullptr, nullptr, y[i], M[i], K, n_tok, 1, stream)
                           : run_dense(fmts[i], W[i], nullptr, q, d, sm, y[i], M[i], K, n_tok, 1, stream);
    if (rc) return rc;
  }
  return QMV_OK;
}

size_t moe_qmv_workspace_bytes(const moe_experts* e, int n_tok, int top_k) {
  if (check_moe_shape(e, n_tok, top_k)) return 0;
  size_t off[MOE_NOFF];
  return moe_layout(e, n_tok, top_k, off);
}

int moe_qmv_workspace_offsets(const moe_experts* e, int n_tok, int top_k, size_t offsets[5]) {
  int rc = check_moe_shape(e, n_tok, top_k);
  if (rc) return rc;
  if (!offsets) return QMV_ERR_NULL;
  moe_layout(e, n_tok, top_k, offsets);
  return QMV_OK;
}

int moe_qmv_run(const moe_experts* e, const int32_t* ids, const float* gates, const float* x, float* y, int n_tok,
                int top_k, void* ws, size_t ws_bytes, cudaStream_t stream) {
  int rc = check_moe_shape(e, n_tok, top_k);
  if (rc) return rc;
  if (!ids || !gates || !x || !y || !ws || !e->w_gate_up || !e->w_down) return QMV_ERR_NULL;
  if (!aligned16(ids) || !aligned16(gates) || !aligned16(x) || !aligned16(y) || !aligned16(ws) ||
      !aligned16(e->w_gate_up) || !aligned16(e->w_down))
    return QMV_ERR_ALIGN;
  size_t off[MOE_NOFF];
  if (ws_bytes < moe_layout(e, n_tok, top_k, off)) return QMV_ERR_WORKSPACE;
  if ((rc = check_device())) return rc;
  uint8_t* w = static_cast<uint8_t*>(ws);
  float* h = reinterpret_cast<float*>(w + off[0]);
  float* o = reinterpret_cast<float*>(w + off[4]);
  // Token slots per expert group: a power of two covering the typical group
  // (tokens per expert ~ lambda = n_tok * top_k / E, plus two standard
  // deviations); larger groups are split into several groups, each reading the
  // expert's weights again.  From 4 tokens on at least 8 slots: their kernels'
  // twelve consumer warps (beside a producer warpgroup) run faster than the
  // smaller slot counts' two CTAs of eight per SM, even for groups of one or
  // two tokens (empty slots cost no arithmetic).  Below that the single-token
  // kernels win.
  const double lam = (double)n_tok * top_k / e->n_experts;
  const double want = lam + 2.0 * sqrt(lam);
  int nt = 1;
  while (nt < want && nt < 16) nt <<= 1;
  while (nt > n_tok && nt > 1) nt >>= 1;
  if (n_tok >= 4 && nt < 8) nt = 8;

  MoeParams p{};
  const long long S = (long long)n_tok * top_k;
  p.ids = ids;
  p.n_tok = n_tok;
  p.top_k = top_k;
  p.n_experts = e->n_experts;
  p.err = device_error_word();
  QMV_DEBUG_ONLY(p.ids_len = S;)
  // gate / up + SwiGLU: h [S][F]
  p.src = x;
  p.dst = h;
  p.K = e->hidden;
  p.R = e->ffn;
  p.pool_rows = 2 * e->ffn;
  QMV_DEBUG_ONLY(p.src_len = (long long)n_tok * e->hidden; p.dst_len = S * e->ffn; p.hq_len = 0;)
  if ((rc = run_moe_proj(MOE_GATE_UP, e->fmt_gate_up, e->w_gate_up, p, nt, stream))) return rc;
  // down (h quantized while staging, published to the workspace): o [S][H]
  MoeParams pd = p;
  pd.src = h;
  pd.dst = o;
  pd.hq = reinterpret_cast<int8_t*>(w + off[1]);
  pd.hd = reinterpret_cast<float*>(w + off[2]);
  pd.hs = reinterpret_cast<int32_t*>(w + off[3]);
  pd.K = e->ffn;
  pd.R = e->hidden;
  pd.pool_rows = e->hidden;
  QMV_DEBUG_ONLY(pd.src_len = S * e->ffn; pd.dst_len = S * e->hidden; pd.hq_len = S * e->ffn;)
  if ((rc = run_moe_proj(MOE_DOWN, e->fmt_down, e->w_down, pd, nt, stream))) return rc;
  return launch_moe_combine(ids, gates, o, y, n_tok, top_k, e->n_experts, e->hidden, stream, true) == cudaSuccess
             ? QMV_OK
             : QMV_ERR_CUDA;
}

int moe_route_run(int fmt, const void* Wr, const float* x, int n_experts, int64_t hidden, int n_tok, int top_k,
                  int gating, float* logits, int32_t* ids, float* gates, cudaStream_t stream) {
  int rc = check_dense_args(fmt, Wr, x, logits, n_experts, hidden, n_tok);
  if (rc) return rc;
  if (n_experts > MOE_MAX_EXPERTS || (gating != QMV_GATING_SOFTMAX && gating != QMV_GATING_SIGMOID))
    return QMV_ERR_SHAPE;
  if (top_k < 1 || top_k > QMV_MAX_TOPK || top_k > n_experts) return QMV_ERR_NTOK;
  if (!ids || !gates) return QMV_ERR_NULL;
  if (!aligned16(ids) || !aligned16(gates)) return QMV_ERR_ALIGN;
  if ((rc = check_device())) return rc;
  if ((rc = run_dense(fmt, Wr, x, nullptr, nullptr, nullptr, logits, n_experts, hidden, n_tok, 1, stream)))
    return rc;
  return launch_route_topk(logits, n_tok, n_experts, top_k, gating, ids, gates, stream, true) == cudaSuccess
             ? QMV_OK
             : QMV_ERR_CUDA;
}

int qmv_check_rounding(unsigned long long* mismatches, cudaStream_t stream) {
  if (!mismatches) return QMV_ERR_NULL;
  if (!aligned16(mismatches)) return QMV_ERR_ALIGN;
  int rc = check_device();
  if (rc) return rc;
  return launch_check_rounding(mismatches, stream) == cudaSuccess ? QMV_OK : QMV_ERR_CUDA;
}


int qmv_debug_shrink_outputs(int64_t n) {
#ifdef QMV_DEBUG
  if (n < 0) return QMV_ERR_SHAPE;
  g_output_shrink.store(n, std::memory_order_relaxed);
  return QMV_OK;
#else
  (void)n;
  return QMV_ERR_UNAVAILABLE;
#endif
}

int qmv_get_device_error(cudaStream_t stream, int* err) {
  if (!err) return QMV_ERR_NULL;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return QMV_ERR_CUDA;
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_qmv_error, sizeof(v)) != cudaSuccess) return QMV_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_qmv_error, &zero, sizeof(zero)) != cudaSuccess) return QMV_ERR_CUDA;
  *err = (int)v;
  return QMV_OK;
}

const char* qmv_strerror(int code) {
  switch (code) {
    case QMV_OK: return "success";
    case QMV_ERR_FORMAT: return "unknown weight format";
    case QMV_ERR_SHAPE: return "invalid shape (M, K, ffn, hidden or split count)";
    case QMV_ERR_NTOK: return "n_tok outside [1, 64] or top_k outside [1, 8]";
    case QMV_ERR_NULL: return "a required pointer is NULL";
    case QMV_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case QMV_ERR_WORKSPACE: return "workspace too small";
    case QMV_ERR_CUDA: return "CUDA runtime error";
    case QMV_ERR_DEVICE: return "no usable sm_103 device";
    case QMV_ERR_UNAVAILABLE: return "not available in this build";
  }
  return "unknown status";
}

}  // extern "C"
