// Host side of the C ABI declared in include/moe_gb300.h: argument checks,
// workspace carve-up, TMA descriptor encoding and the launch sequence of
// each entry point. Nothing here allocates device memory or synchronises
// with the device.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "moe_internal.h"

using namespace moe;

namespace {

// ---------------------------------------------------------------- checks ----

constexpr int64_t kMaxDim = 65536;

moe_status check_shape(const moe_shape* s) {
  if (s == nullptr) return MOE_ERR_NULL;
  if (s->T < 0 || s->H <= 0 || s->E <= 0 || s->top_k <= 0 || s->h <= 0) return MOE_ERR_SHAPE;
  if (!isfinite(s->capacity_factor) || !(s->capacity_factor > 0.0)) return MOE_ERR_SHAPE;
  if (s->E > kMaxExperts || s->top_k > kMaxTopK || s->top_k > s->E) return MOE_ERR_UNSUPPORTED;
  if (s->H % 64 != 0 || s->h % 64 != 0 || s->H > kMaxDim || s->h > kMaxDim)
    return MOE_ERR_UNSUPPORTED;
  if (s->T > (int64_t(1) << 31) || s->T * s->top_k >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define MOE_REQUIRE(p) \
  do {                 \
    if ((p) == nullptr) return MOE_ERR_NULL; \
    if (!aligned16(p)) return MOE_ERR_ALIGN; \
  } while (0)

#define MOE_OPTIONAL(p) \
  do {                  \
    if ((p) != nullptr && !aligned16(p)) return MOE_ERR_ALIGN; \
  } while (0)

#define MOE_CUDA(x)                                \
  do {                                             \
    if ((x) != cudaSuccess) return MOE_ERR_CUDA;   \
  } while (0)

#define MOE_TRY(x)                         \
  do {                                     \
    const moe_status _s = (x);             \
    if (_s != MOE_OK) return _s;           \
  } while (0)

// ------------------------------------------------------------- workspace ----

struct Ws {
  uint16_t* gateT;
  int32_t* tile_cnt;
  int32_t* tile_base;
  uint8_t* rank8;
  float* ppart;
  int32_t* routed;
  float* P;
  float* aux;
  int32_t* kept;
  int32_t* offsets;
  int32_t* cap;  // expert parallelism: this rank's capacity per expert
  uint32_t* status;
  uint32_t* ticket;
  int32_t* topk_idx;
  float* topk_w;
  int32_t* dest_row;
  int32_t* src_token;
  uint16_t* x_perm;
  uint16_t* act;
  uint16_t* y_perm;
  // FP8 path only (moe_workspace_size_fp8); the e4m3 dispatched rows live in
  // the x_perm bytes
  float* x_scale;
  uint8_t* act_q;
  float* act_scale;
  uint32_t* act_amax;
  float* y_scale;  // block scales of the e4m3 expert outputs (which live in the y_perm bytes)
};

struct Dims {
  int T, H, E, k, h, E_pad, n_tiles;
  int64_t A, C;
};

Dims dims_of(const moe_shape* s) {
  Dims d;
  d.T = static_cast<int>(s->T);
  d.H = static_cast<int>(s->H);
  d.E = static_cast<int>(s->E);
  d.k = static_cast<int>(s->top_k);
  d.h = static_cast<int>(s->h);
  d.E_pad = (d.E + 15) & ~15;
  d.n_tiles = (d.T + kTileTokens - 1) / kTileTokens;
  d.A = s->T * s->top_k;
  d.C = moe_capacity(s->T, s->E, s->top_k, s->capacity_factor);
  return d;
}

// Lays the scratch arrays out from `base` (256-byte aligned pieces); with
// base == nullptr only the size is computed.
size_t layout(const Dims& d, uint8_t* base, Ws* w, bool fp8 = false) {
  size_t off = 0;
  auto take = [&](size_t bytes) -> void* {
    void* p = base ? base + off : nullptr;
    off += (bytes + 255) & ~size_t(255);
    return p;
  };
  const size_t A = static_cast<size_t>(d.A);
  const size_t ET = static_cast<size_t>(d.E) * d.n_tiles;
  Ws v;
  v.gateT = static_cast<uint16_t*>(take(static_cast<size_t>(d.E_pad) * d.H * 2));
  v.tile_cnt = static_cast<int32_t*>(take(ET * 4));
  v.tile_base = static_cast<int32_t*>(take(ET * 4));
  v.rank8 = static_cast<uint8_t*>(take(A));
  v.ppart = static_cast<float*>(take(ET * 4));
  v.routed = static_cast<int32_t*>(take(static_cast<size_t>(d.E) * 4));
  v.P = static_cast<float*>(take(static_cast<size_t>(d.E) * 4));
  v.aux = static_cast<float*>(take(4));
  v.kept = static_cast<int32_t*>(take(static_cast<size_t>(d.E) * 4));
  v.offsets = static_cast<int32_t*>(take(static_cast<size_t>(d.E + 1) * 4));
  v.cap = static_cast<int32_t*>(take(static_cast<size_t>(d.E) * 4));
  v.status = static_cast<uint32_t*>(take(4));
  v.ticket = static_cast<uint32_t*>(take(4));
  v.topk_idx = static_cast<int32_t*>(take(A * 4));
  v.topk_w = static_cast<float*>(take(A * 4));
  v.dest_row = static_cast<int32_t*>(take(A * 4));
  v.src_token = static_cast<int32_t*>(take(A * 4));
  v.x_perm = static_cast<uint16_t*>(take(A * d.H * 2));
  v.act = static_cast<uint16_t*>(take(A * d.h * 2));
  v.y_perm = static_cast<uint16_t*>(take(A * d.H * 2));
  v.x_scale = nullptr;
  v.act_q = nullptr;
  v.act_scale = nullptr;
  v.act_amax = nullptr;
  v.y_scale = nullptr;
  if (fp8) {
    v.x_scale = static_cast<float*>(take(A * 4));
    v.act_q = static_cast<uint8_t*>(take(A * d.h));
    v.act_scale = static_cast<float*>(take(A * 4));
    v.act_amax = static_cast<uint32_t*>(take(A * 4));
    v.y_scale = static_cast<float*>(take(A * static_cast<size_t>((d.H + 127) / 128) * 4));
  }
  if (w) *w = v;
  return off;
}

moe_status carve(const moe_shape* s, const Dims& d, void* ws, size_t ws_bytes, Ws* w,
                 bool fp8 = false) {
  const size_t need = layout(d, nullptr, nullptr, fp8);
  if (ws == nullptr) return MOE_ERR_NULL;
  if (!aligned16(ws)) return MOE_ERR_ALIGN;
  if (ws_bytes < need) return MOE_ERR_WORKSPACE;
  layout(d, static_cast<uint8_t*>(ws), w, fp8);
  (void)s;
  return MOE_OK;
}

// ------------------------------------------------------ device queries ----

int num_sms() {
  // per-device cache; atomics so that concurrent callers on several host
  // threads read and fill it without a data race
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

uint64_t wait_timeout_ns() {
  static uint64_t v = [] {
    const char* e = getenv("MOE_GB300_WAIT_TIMEOUT_NS");
    if (e != nullptr) {
      const unsigned long long x = strtoull(e, nullptr, 10);
      if (x > 0) return static_cast<uint64_t>(x);
    }
    return kDefaultTimeoutNs;
  }();
  return v;
}

// The CTA-pair grouped GEMM moves a third less shared-memory traffic per FLOP
// and wins from a few thousand rows up; below that the single-CTA kernel's
// finer 128-row tiles waste less on ragged segments.
constexpr int64_t kPairGemmMinRows = 4096;

// ------------------------------------------------------------ TMA maps ----

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// A bf16 row-major matrix [outer, inner] read in boxes of box_outer rows x
// box_inner (= 64, one 128-byte swizzle row) columns.
bool tmap_bf16_2d(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer,
                  uint32_t box_inner, uint32_t box_outer,
                  CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t gdim[2] = {inner, outer};
  const cuuint64_t gstride[1] = {inner * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estride[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), gdim, gstride, box,
            estride, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A bf16 row-major matrix [rows, K] (K % 64 == 0) seen as 64-element
// k-blocks: 3-D {64, rows, K/64}, the k-block dimension 128 bytes apart, read
// in boxes of box_rows rows x kbps consecutive k-blocks. A box lands in shared
// memory k-block by k-block, each the box_rows x 128-byte swizzled tile that
// a 2-D {64, box_rows} box would give.
bool tmap_bf16_kblocks(CUtensorMap* m, const void* ptr, uint64_t K, uint64_t rows,
                       uint32_t box_rows, int kbps) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t gdim[3] = {64, rows, K / 64};
  const cuuint64_t gstride[2] = {K * 2, 128};
  const cuuint32_t box[3] = {64, box_rows, static_cast<cuuint32_t>(kbps)};
  const cuuint32_t estride[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), gdim, gstride, box,
            estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Per-expert bf16 matrices W [E][K][N] (row-major, N % 64 == 0) seen as
// 4-D {64 columns, K, N/64 column blocks, E}, the column-block dimension
// 128 bytes apart, read in boxes of box_k rows x 2 column blocks of one
// expert: one copy fills a CTA's 128-column B slice, block by block (each
// block the box_k x 128-byte swizzled tile a 2-D {64, box_k} box gives).
// Rows past K and blocks past N read as zeros.
bool tmap_bf16_experts(CUtensorMap* m, const void* ptr, uint64_t N, uint64_t K, uint64_t E,
                       uint32_t box_k) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t gdim[4] = {64, K, N / 64, E};
  const cuuint64_t gstride[3] = {N * 2, 128, N * K * 2};
  const cuuint32_t box[4] = {64, box_k, 2, 1};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), gdim, gstride, box,
            estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A byte (e4m3) row-major matrix [outer, inner] in 128 x 128 boxes (one
// 128-byte swizzle row of K per box row); inner must be a multiple of 16.
bool tmap_u8_2d(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t gdim[2] = {inner, outer};
  const cuuint64_t gstride[1] = {inner};
  const cuuint32_t box[2] = {128, 128};
  const cuuint32_t estride[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), gdim, gstride, box,
            estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------- stages ----

struct RouteOut {
  int32_t* topk_idx;
  float* topk_w;
  int32_t* routed;
  float* P;
  float* aux;
  float* logits_out;
};

struct Noise {
  const float* u;     // [T,E] uniforms or nullptr
  float temperature;  // used with u
};

moe_status run_route(const Dims& d, const moe_bf16* x, const moe_bf16* gate, const float* bias,
                     const float* logits_in, const RouteOut& o, uint32_t* status, const Ws& w,
                     cudaStream_t st, Noise noise = Noise{nullptr, 1.0f}) {
  if (d.T == 0) {
    MOE_CUDA(cudaMemsetAsync(o.routed, 0, sizeof(int32_t) * d.E, st));
    MOE_CUDA(cudaMemsetAsync(o.P, 0, sizeof(float) * d.E, st));
    if (o.aux) MOE_CUDA(cudaMemsetAsync(o.aux, 0, sizeof(float), st));
    return MOE_OK;
  }
  RouteArgs a;
  a.T = d.T;
  a.H = d.H;
  a.E = d.E;
  a.E_pad = d.E_pad;
  a.k = d.k;
  a.n_tiles = d.n_tiles;
  a.gate_mode = kGateTransposed;
  a.stages = 0;
  a.bias = bias;
  a.noise_u = noise.u;
  a.temperature = noise.temperature;
  a.logits_in = logits_in;
  a.topk_idx = o.topk_idx;
  a.topk_w = o.topk_w;
  a.logits_out = o.logits_out;
  a.tile_cnt = w.tile_cnt;
  a.rank8 = w.rank8;
  a.ppart = w.ppart;
  a.ticket = w.ticket;
  a.dev_status = status;
  a.timeout_ns = wait_timeout_ns();
  if (logits_in != nullptr) {
    MOE_CUDA(launch_route_logits(a, st));
  } else {
    CUtensorMap tm_x, tm_g;
    // The gate [H,E] is the UMMA's B operand as given (MN-major TMA boxes of
    // 64 experts) when E >= 64 and its rows are 16-byte multiples; otherwise
    // a transposed, padded copy [E_pad,H] is made in the workspace first.
    const int sms = num_sms();
    a.gate_mode = (d.E >= 64 && d.E % 8 == 0) ? kGateMnMajor : kGateTransposed;
    route_plan(a, sms);
    if (a.gate_mode == kGateMnMajor &&
        !tmap_bf16_2d(&tm_g, gate, d.E, d.H, 64, static_cast<uint32_t>(kBlockK * a.kbps))) {
      a.gate_mode = kGateTransposed;
      route_plan(a, sms);
    }
    if (a.gate_mode == kGateTransposed) {
      MOE_CUDA(launch_gate_transpose(gate, w.gateT, d.H, d.E, d.E_pad, st));
      if (!tmap_bf16_kblocks(&tm_g, w.gateT, d.H, d.E_pad, d.E_pad, a.kbps)) return MOE_ERR_CUDA;
    }
    if (!tmap_bf16_kblocks(&tm_x, x, d.H, d.T, kTileTokens, a.kbps)) return MOE_ERR_CUDA;
    MOE_CUDA(launch_route_gemm(tm_x, tm_g, a, st, sms));
  }
  return MOE_OK;
}

moe_status run_scan(const Dims& d, bool with_stats, int32_t* routed, float* P, float* aux,
                    int32_t* kept, int32_t* offsets, const Ws& w, cudaStream_t st) {
  ScanArgs s;
  s.T = d.T;
  s.E = d.E;
  s.k = d.k;
  s.n_tiles = d.n_tiles;
  s.C = d.C;
  s.tile_cnt = w.tile_cnt;
  s.tile_base = w.tile_base;
  s.ppart = with_stats ? w.ppart : nullptr;
  s.routed = routed;
  s.P = P;
  s.aux = with_stats ? aux : nullptr;
  s.kept = kept;
  s.offsets = offsets;
  s.ticket = w.ticket;
  MOE_CUDA(launch_scan(s, st));
  return MOE_OK;
}

moe_status run_gather(const Dims& d, const moe_bf16* x, const int32_t* idx, const int32_t* offsets,
                      int32_t* dest_row, int32_t* src_token, moe_bf16* x_perm, uint32_t* status,
                      const Ws& w, cudaStream_t st) {
  GatherArgs g;
  g.T = d.T;
  g.H = d.H;
  g.E = d.E;
  g.k = d.k;
  g.n_tiles = d.n_tiles;
  g.C = d.C;
  g.x = x;
  g.topk_idx = idx;
  g.rank8 = w.rank8;
  g.tile_base = w.tile_base;
  g.offsets = offsets;
  g.dest_row = dest_row;
  g.src_token = src_token;
  g.x_perm = x_perm;
  g.dev_status = status;
  MOE_CUDA(launch_gather(g, num_sms(), st));
  return MOE_OK;
}

moe_status run_gather_fp8(const Dims& d, const moe_bf16* x, const int32_t* idx,
                          const int32_t* offsets, int32_t* dest_row, int32_t* src_token,
                          uint8_t* xq, float* xs, uint32_t* status, const Ws& w, cudaStream_t st) {
  GatherArgs g;
  g.T = d.T;
  g.H = d.H;
  g.E = d.E;
  g.k = d.k;
  g.n_tiles = d.n_tiles;
  g.C = d.C;
  g.x = x;
  g.topk_idx = idx;
  g.rank8 = w.rank8;
  g.tile_base = w.tile_base;
  g.offsets = offsets;
  g.dest_row = dest_row;
  g.src_token = src_token;
  g.x_perm = nullptr;
  g.dev_status = status;
  MOE_CUDA(launch_gather_fp8(g, xq, xs, num_sms(), st));
  return MOE_OK;
}

// With a_rows, A row r is row a_rows[r] of A (a tensor of a_src_rows rows),
// gathered by the CTA-pair kernel's TMA (box one row high).
moe_status run_gemm(const Dims& d, const moe_bf16* A, const moe_bf16* W, const int32_t* offsets,
                    int K, int N, moe_bf16* D, int gelu, uint32_t* status, cudaStream_t st,
                    const int32_t* a_rows = nullptr, int a_src_rows = 0) {
  if (d.A == 0) return MOE_OK;
  CUtensorMap tm_a, tm_b;
  const bool pair = d.A >= kPairGemmMinRows || a_rows != nullptr;
  if (a_rows != nullptr) {
    if (!tmap_bf16_2d(&tm_a, A, K, a_src_rows, kBlockK, 1)) return MOE_ERR_CUDA;
  } else if (pair) {
    // the CTA-pair kernel's stages hold two k-blocks of its 128 rows
    if (!tmap_bf16_kblocks(&tm_a, A, K, d.A, 128, 2)) return MOE_ERR_CUDA;
  } else if (!tmap_bf16_2d(&tm_a, A, K, d.A, kBlockK, 128)) {
    return MOE_ERR_CUDA;
  }
  if (pair) {
    // W [E][K][N] in boxes of 128 columns x 64 (gathered A) or 128 k-rows of
    // one expert: rows past K read as zeros
    if (!tmap_bf16_experts(&tm_b, W, N, K, d.E, a_rows != nullptr ? kBlockK : 2 * kBlockK))
      return MOE_ERR_CUDA;
  } else if (!tmap_bf16_2d(&tm_b, W, N, static_cast<uint64_t>(d.E) * K, 64, kBlockK)) {
    return MOE_ERR_CUDA;
  }
  GemmArgs g;
  g.offsets = offsets;
  g.E = d.E;
  g.K = K;
  g.N = N;
  g.rows = static_cast<int>(d.A);
  g.D = D;
  g.gelu = gelu;
  g.a_scale = nullptr;
  g.b_scale = nullptr;
  g.row_amax = nullptr;
  g.Dq = nullptr;
  g.d_scale = nullptr;
  g.a_rows = a_rows;
  g.a_src_rows = a_src_rows;
  g.stages = 0;
  g.dev_status = status;
  g.timeout_ns = wait_timeout_ns();
  if (pair)
    MOE_CUDA(launch_grouped_gemm_pair(tm_a, tm_b, g, num_sms(), st));
  else
    MOE_CUDA(launch_grouped_gemm(tm_a, tm_b, g, num_sms(), st));
  return MOE_OK;
}

// The FP8 grouped GEMM (CTA-pair kernel at every size): A e4m3 [A, K] with
// row scales, B^T e4m3 [E*N, K] with column scales; with row_amax the
// epilogue also records each output row's largest magnitude.
moe_status run_gemm_fp8(const Dims& d, const uint8_t* Aq, const float* a_scale,
                        const uint8_t* Wq, const float* w_scale, const int32_t* offsets, int K,
                        int N, moe_bf16* D, int gelu, uint32_t* row_amax, uint32_t* status,
                        cudaStream_t st, uint8_t* Dq = nullptr, float* d_scale = nullptr) {
  if (d.A == 0) return MOE_OK;
  CUtensorMap tm_a, tm_b;
  if (!tmap_u8_2d(&tm_a, Aq, K, d.A)) return MOE_ERR_CUDA;
  if (!tmap_u8_2d(&tm_b, Wq, K, static_cast<uint64_t>(d.E) * N)) return MOE_ERR_CUDA;
  GemmArgs g;
  g.offsets = offsets;
  g.E = d.E;
  g.K = K;
  g.N = N;
  g.rows = static_cast<int>(d.A);
  g.D = D;
  g.gelu = gelu;
  g.a_scale = a_scale;
  g.b_scale = w_scale;
  g.row_amax = row_amax;
  g.Dq = Dq;
  g.d_scale = d_scale;
  g.a_rows = nullptr;
  g.a_src_rows = 0;
  g.stages = 0;
  g.dev_status = status;
  g.timeout_ns = wait_timeout_ns();
  MOE_CUDA(launch_grouped_gemm_pair_fp8(tm_a, tm_b, g, num_sms(), st));
  return MOE_OK;
}

// FP8 expert FFN on dispatched e4m3 rows: GEMM1 (+GELU, row maxima of act),
// act quantised per row, GEMM2 into bf16 y_perm or, with y_q, into e4m3
// with 128-column block scales.
moe_status run_ffn_fp8(const Dims& d, const uint8_t* xq, const float* xs, const int32_t* offsets,
                       const uint8_t* W1q, const float* w1s, const uint8_t* W2q,
                       const float* w2s, moe_bf16* act, moe_bf16* y_perm, uint32_t* status,
                       const Ws& w, cudaStream_t st, void* const* events,
                       uint8_t* y_q = nullptr, float* y_scale = nullptr) {
  if (d.A == 0) return MOE_OK;
  MOE_CUDA(cudaMemsetAsync(w.act_amax, 0, sizeof(uint32_t) * static_cast<size_t>(d.A), st));
  MOE_TRY(run_gemm_fp8(d, xq, xs, W1q, w1s, offsets, d.H, d.h, act, 1, w.act_amax, status, st));
  MOE_CUDA(launch_row_quant(act, w.act_amax, w.act_q, w.act_scale, offsets, d.E,
                            static_cast<int>(d.A), d.h, num_sms(), st));
  if (events && cudaEventRecord(static_cast<cudaEvent_t>(events[0]), st) != cudaSuccess)
    return MOE_ERR_CUDA;
  MOE_TRY(run_gemm_fp8(d, w.act_q, w.act_scale, W2q, w2s, offsets, d.h, d.H, y_perm, 0, nullptr,
                       status, st, y_q, y_scale));
  return MOE_OK;
}

moe_status run_combine_fp8(const Dims& d, const uint8_t* y_q, const float* y_scale,
                           const int32_t* dest_row, const float* topk_w, moe_bf16* y,
                           cudaStream_t st) {
  CombineArgs c;
  c.T = d.T;
  c.H = d.H;
  c.k = d.k;
  c.y_perm = nullptr;
  c.dest_row = dest_row;
  c.topk_w = topk_w;
  c.y = y;
  MOE_CUDA(launch_combine_fp8(c, y_q, y_scale, num_sms(), st));
  return MOE_OK;
}

moe_status run_combine(const Dims& d, const moe_bf16* y_perm, const int32_t* dest_row,
                       const float* topk_w, moe_bf16* y, cudaStream_t st) {
  CombineArgs c;
  c.T = d.T;
  c.H = d.H;
  c.k = d.k;
  c.y_perm = y_perm;
  c.dest_row = dest_row;
  c.topk_w = topk_w;
  c.y = y;
  MOE_CUDA(launch_combine(c, num_sms(), st));
  return MOE_OK;
}

}  // namespace

// ================================================================ ABI ====

extern "C" {

int moe_abi_version(void) { return MOE_GB300_ABI_VERSION; }

int64_t moe_capacity(int64_t T, int64_t E, int64_t top_k, double capacity_factor) {
  if (T < 0 || E < 1 || top_k < 1 || !isfinite(capacity_factor) || !(capacity_factor > 0.0))
    return -1;
  const double c = ceil(capacity_factor * static_cast<double>(T * top_k) / static_cast<double>(E));
  const int64_t ci = static_cast<int64_t>(c);
  return ci < 1 ? 1 : ci;
}

const char* moe_status_str(moe_status st) {
  switch (st) {
    case MOE_OK: return "ok";
    case MOE_ERR_NULL: return "a required pointer is NULL";
    case MOE_ERR_SHAPE: return "invalid shape or capacity factor";
    case MOE_ERR_UNSUPPORTED: return "shape outside the supported ranges";
    case MOE_ERR_WORKSPACE: return "workspace smaller than moe_workspace_size";
    case MOE_ERR_ALIGN: return "pointer not 16-byte aligned";
    case MOE_ERR_CUDA: return "CUDA call or kernel launch failed";
  }
  return "unknown status";
}

moe_status moe_workspace_size(const moe_shape* s, size_t* bytes) {
  if (bytes == nullptr) return MOE_ERR_NULL;
  MOE_TRY(check_shape(s));
  *bytes = layout(dims_of(s), nullptr, nullptr);
  return MOE_OK;
}

moe_status moe_route(const moe_shape* s, const moe_bf16* x, const moe_bf16* gate,
                     const float* gate_bias, int32_t* topk_idx, float* topk_w,
                     int32_t* routed_counts, float* P, float* aux, float* logits_out,
                     uint32_t* dev_status, void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(check_shape(s));
  MOE_REQUIRE(x);
  MOE_REQUIRE(gate);
  MOE_REQUIRE(topk_idx);
  MOE_REQUIRE(topk_w);
  MOE_OPTIONAL(gate_bias);
  MOE_OPTIONAL(routed_counts);
  MOE_OPTIONAL(P);
  MOE_OPTIONAL(aux);
  MOE_OPTIONAL(logits_out);
  MOE_OPTIONAL(dev_status);
  const Dims d = dims_of(s);
  Ws w;
  MOE_TRY(carve(s, d, ws, ws_bytes, &w));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  RouteOut o{topk_idx, topk_w, routed_counts ? routed_counts : w.routed, P ? P : w.P, aux,
             logits_out};
  uint32_t* status = dev_status ? dev_status : w.status;
  MOE_TRY(run_route(d, x, gate, gate_bias, nullptr, o, status, w, st));
  if (d.T > 0) MOE_TRY(run_scan(d, true, o.routed, o.P, aux, nullptr, nullptr, w, st));
  return MOE_OK;
}

moe_status moe_route_logits(const moe_shape* s, const float* logits, int32_t* topk_idx,
                            float* topk_w, int32_t* routed_counts, float* P, float* aux,
                            uint32_t* dev_status, void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(check_shape(s));
  MOE_REQUIRE(logits);
  MOE_REQUIRE(topk_idx);
  MOE_REQUIRE(topk_w);
  MOE_OPTIONAL(routed_counts);
  MOE_OPTIONAL(P);
  MOE_OPTIONAL(aux);
  MOE_OPTIONAL(dev_status);
  const Dims d = dims_of(s);
  Ws w;
  MOE_TRY(carve(s, d, ws, ws_bytes, &w));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  RouteOut o{topk_idx, topk_w, routed_counts ? routed_counts : w.routed, P ? P : w.P, aux,
             nullptr};
  uint32_t* status = dev_status ? dev_status : w.status;
  MOE_TRY(run_route(d, nullptr, nullptr, nullptr, logits, o, status, w, st));
  if (d.T > 0) MOE_TRY(run_scan(d, true, o.routed, o.P, aux, nullptr, nullptr, w, st));
  return MOE_OK;
}

moe_status moe_permute(const moe_shape* s, const moe_bf16* x, const int32_t* topk_idx,
                       int32_t* kept_counts, int32_t* offsets, int32_t* dest_row,
                       int32_t* src_token, moe_bf16* x_perm, uint32_t* dev_status, void* ws,
                       size_t ws_bytes, void* stream) {
  MOE_TRY(check_shape(s));
  MOE_REQUIRE(x);
  MOE_REQUIRE(topk_idx);
  MOE_REQUIRE(offsets);
  MOE_REQUIRE(dest_row);
  MOE_OPTIONAL(x_perm);  // NULL: the permutation only (for moe_expert_ffn_gathered)
  MOE_OPTIONAL(kept_counts);
  MOE_OPTIONAL(src_token);
  MOE_OPTIONAL(dev_status);
  if (x_perm == nullptr && src_token == nullptr) return MOE_ERR_NULL;
  const Dims d = dims_of(s);
  Ws w;
  MOE_TRY(carve(s, d, ws, ws_bytes, &w));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* status = dev_status ? dev_status : w.status;
  if (d.T == 0) {
    MOE_CUDA(cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (d.E + 1), st));
    if (kept_counts) MOE_CUDA(cudaMemsetAsync(kept_counts, 0, sizeof(int32_t) * d.E, st));
    return MOE_OK;
  }
  RankArgs r;
  r.T = d.T;
  r.E = d.E;
  r.k = d.k;
  r.n_tiles = d.n_tiles;
  r.topk_idx = topk_idx;
  r.tile_cnt = w.tile_cnt;
  r.rank8 = w.rank8;
  r.ticket = w.ticket;
  r.dev_status = status;
  MOE_CUDA(launch_rank(r, st));
  MOE_TRY(run_scan(d, false, w.routed, w.P, nullptr, kept_counts, offsets, w, st));
  MOE_TRY(run_gather(d, x, topk_idx, offsets, dest_row, src_token, x_perm, status, w, st));
  return MOE_OK;
}

moe_status moe_expert_ffn(const moe_shape* s, const moe_bf16* x_perm, const int32_t* offsets,
                          const moe_bf16* W1, const moe_bf16* W2, moe_bf16* act,
                          moe_bf16* y_perm, uint32_t* dev_status, void* ws, size_t ws_bytes,
                          void* stream) {
  MOE_TRY(check_shape(s));
  MOE_REQUIRE(x_perm);
  MOE_REQUIRE(offsets);
  MOE_REQUIRE(W1);
  MOE_REQUIRE(W2);
  MOE_REQUIRE(act);
  MOE_REQUIRE(y_perm);
  MOE_OPTIONAL(dev_status);
  const Dims d = dims_of(s);
  uint32_t* status = dev_status;
  if (status == nullptr) {
    Ws w;
    MOE_TRY(carve(s, d, ws, ws_bytes, &w));
    status = w.status;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MOE_TRY(run_gemm(d, x_perm, W1, offsets, d.H, d.h, act, 1, status, st));
  MOE_TRY(run_gemm(d, act, W2, offsets, d.h, d.H, y_perm, 0, status, st));
  return MOE_OK;
}

moe_status moe_expert_ffn_gathered(const moe_shape* s, const moe_bf16* x,
                                   const int32_t* src_token, const int32_t* offsets,
                                   const moe_bf16* W1, const moe_bf16* W2, moe_bf16* act,
                                   moe_bf16* y_perm, uint32_t* dev_status, void* ws,
                                   size_t ws_bytes, void* stream) {
  MOE_TRY(check_shape(s));
  MOE_REQUIRE(x);
  MOE_REQUIRE(src_token);
  MOE_REQUIRE(offsets);
  MOE_REQUIRE(W1);
  MOE_REQUIRE(W2);
  MOE_REQUIRE(act);
  MOE_REQUIRE(y_perm);
  MOE_OPTIONAL(dev_status);
  const Dims d = dims_of(s);
  uint32_t* status = dev_status;
  if (status == nullptr) {
    Ws w;
    MOE_TRY(carve(s, d, ws, ws_bytes, &w));
    status = w.status;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MOE_TRY(run_gemm(d, x, W1, offsets, d.H, d.h, act, 1, status, st, src_token, d.T));
  MOE_TRY(run_gemm(d, act, W2, offsets, d.h, d.H, y_perm, 0, status, st));
  return MOE_OK;
}

moe_status moe_combine(const moe_shape* s, const moe_bf16* y_perm, const int32_t* dest_row,
                       const float* topk_w, moe_bf16* y, void* stream) {
  MOE_TRY(check_shape(s));
  MOE_REQUIRE(y_perm);
  MOE_REQUIRE(dest_row);
  MOE_REQUIRE(topk_w);
  MOE_REQUIRE(y);
  const Dims d = dims_of(s);
  return run_combine(d, y_perm, dest_row, topk_w, y, static_cast<cudaStream_t>(stream));
}

// Quantised expert weights of the FP8 layer: W1q [E,h,H], W2q [E,H,h] e4m3
// (transposed), w1s [E,h], w2s [E,H] column scales.
struct Fp8Weights {
  const uint8_t* W1q;
  const float* w1s;
  const uint8_t* W2q;
  const float* w2s;
};

static moe_status layer_fwd(const moe_shape* s, const moe_bf16* x, const moe_bf16* gate,
                     const float* gate_bias, const moe_bf16* W1, const moe_bf16* W2, moe_bf16* y,
                     float* aux, int32_t* topk_idx, float* topk_w, int32_t* routed_counts,
                     float* P, int32_t* kept_counts, int32_t* offsets, int32_t* dest_row,
                     uint32_t* dev_status, void* ws, size_t ws_bytes, void* stream,
                     void* const* events, Noise noise, const Fp8Weights* q = nullptr) {
  MOE_TRY(check_shape(s));
  MOE_REQUIRE(x);
  MOE_REQUIRE(gate);
  if (q == nullptr) {
    MOE_REQUIRE(W1);
    MOE_REQUIRE(W2);
  } else {
    MOE_REQUIRE(q->W1q);
    MOE_REQUIRE(q->w1s);
    MOE_REQUIRE(q->W2q);
    MOE_REQUIRE(q->w2s);
  }
  MOE_REQUIRE(y);
  MOE_OPTIONAL(gate_bias);
  MOE_OPTIONAL(aux);
  MOE_OPTIONAL(topk_idx);
  MOE_OPTIONAL(topk_w);
  MOE_OPTIONAL(routed_counts);
  MOE_OPTIONAL(P);
  MOE_OPTIONAL(kept_counts);
  MOE_OPTIONAL(offsets);
  MOE_OPTIONAL(dest_row);
  MOE_OPTIONAL(dev_status);
  const Dims d = dims_of(s);
  Ws w;
  MOE_TRY(carve(s, d, ws, ws_bytes, &w, q != nullptr));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* status = dev_status ? dev_status : w.status;
  int32_t* idx = topk_idx ? topk_idx : w.topk_idx;
  float* wts = topk_w ? topk_w : w.topk_w;
  int32_t* routed = routed_counts ? routed_counts : w.routed;
  float* Pp = P ? P : w.P;
  int32_t* kept = kept_counts ? kept_counts : w.kept;
  int32_t* off = offsets ? offsets : w.offsets;
  int32_t* dest = dest_row ? dest_row : w.dest_row;
  auto mark = [&](int i) -> bool {
    return events == nullptr ||
           cudaEventRecord(static_cast<cudaEvent_t>(events[i]), st) == cudaSuccess;
  };
  if (!mark(0)) return MOE_ERR_CUDA;
  if (d.T == 0) {
    MOE_CUDA(cudaMemsetAsync(routed, 0, sizeof(int32_t) * d.E, st));
    MOE_CUDA(cudaMemsetAsync(Pp, 0, sizeof(float) * d.E, st));
    MOE_CUDA(cudaMemsetAsync(kept, 0, sizeof(int32_t) * d.E, st));
    MOE_CUDA(cudaMemsetAsync(off, 0, sizeof(int32_t) * (d.E + 1), st));
    if (aux) MOE_CUDA(cudaMemsetAsync(aux, 0, sizeof(float), st));
    for (int i = 1; i < MOE_LAYER_NUM_EVENTS; ++i)
      if (!mark(i)) return MOE_ERR_CUDA;
    return MOE_OK;
  }
  RouteOut o{idx, wts, routed, Pp, aux, nullptr};
  MOE_TRY(run_route(d, x, gate, gate_bias, nullptr, o, status, w, st, noise));
  if (!mark(1)) return MOE_ERR_CUDA;
  MOE_TRY(run_scan(d, true, routed, Pp, aux, kept, off, w, st));
  if (!mark(2)) return MOE_ERR_CUDA;
  if (q == nullptr) {
    MOE_TRY(run_gather(d, x, idx, off, dest, w.src_token, w.x_perm, status, w, st));
    if (!mark(3)) return MOE_ERR_CUDA;
    MOE_TRY(run_gemm(d, w.x_perm, W1, off, d.H, d.h, w.act, 1, status, st));
    if (!mark(4)) return MOE_ERR_CUDA;
    MOE_TRY(run_gemm(d, w.act, W2, off, d.h, d.H, w.y_perm, 0, status, st));
  } else {
    uint8_t* xq = reinterpret_cast<uint8_t*>(w.x_perm);
    MOE_TRY(run_gather_fp8(d, x, idx, off, dest, w.src_token, xq, w.x_scale, status, w, st));
    if (!mark(3)) return MOE_ERR_CUDA;
    MOE_TRY(run_ffn_fp8(d, xq, w.x_scale, off, q->W1q, q->w1s, q->W2q, q->w2s, w.act, nullptr,
                        status, w, st, events ? events + 4 : nullptr,
                        reinterpret_cast<uint8_t*>(w.y_perm), w.y_scale));
  }
  if (!mark(5)) return MOE_ERR_CUDA;
  if (q == nullptr)
    MOE_TRY(run_combine(d, w.y_perm, dest, wts, y, st));
  else
    MOE_TRY(run_combine_fp8(d, reinterpret_cast<const uint8_t*>(w.y_perm), w.y_scale, dest, wts,
                            y, st));
  if (!mark(6)) return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_layer_fwd(const moe_shape* s, const moe_bf16* x, const moe_bf16* gate,
                         const float* gate_bias, const moe_bf16* W1, const moe_bf16* W2,
                         moe_bf16* y, float* aux, int32_t* topk_idx, float* topk_w,
                         int32_t* routed_counts, float* P, int32_t* kept_counts,
                         int32_t* offsets, int32_t* dest_row, uint32_t* dev_status, void* ws,
                         size_t ws_bytes, void* stream, void* const* events) {
  return layer_fwd(s, x, gate, gate_bias, W1, W2, y, aux, topk_idx, topk_w, routed_counts, P,
                   kept_counts, offsets, dest_row, dev_status, ws, ws_bytes, stream, events,
                   Noise{nullptr, 1.0f});
}

static moe_status check_noise(const float* noise_u, float temperature) {
  if (noise_u == nullptr) return MOE_ERR_NULL;
  if (!aligned16(noise_u)) return MOE_ERR_ALIGN;
  if (!isfinite(temperature) || !(temperature > 0.0f)) return MOE_ERR_SHAPE;
  return MOE_OK;
}

moe_status moe_route_gumbel(const moe_shape* s, const moe_bf16* x, const moe_bf16* gate,
                            const float* gate_bias, const float* noise_u, float temperature,
                            int32_t* topk_idx, float* topk_w, int32_t* routed_counts, float* P,
                            float* aux, float* scores_out, uint32_t* dev_status, void* ws,
                            size_t ws_bytes, void* stream) {
  MOE_TRY(check_shape(s));
  MOE_TRY(check_noise(noise_u, temperature));
  MOE_REQUIRE(x);
  MOE_REQUIRE(gate);
  MOE_REQUIRE(topk_idx);
  MOE_REQUIRE(topk_w);
  MOE_OPTIONAL(gate_bias);
  MOE_OPTIONAL(routed_counts);
  MOE_OPTIONAL(P);
  MOE_OPTIONAL(aux);
  MOE_OPTIONAL(scores_out);
  MOE_OPTIONAL(dev_status);
  const Dims d = dims_of(s);
  Ws w;
  MOE_TRY(carve(s, d, ws, ws_bytes, &w));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  RouteOut o{topk_idx, topk_w, routed_counts ? routed_counts : w.routed, P ? P : w.P, aux,
             scores_out};
  uint32_t* status = dev_status ? dev_status : w.status;
  MOE_TRY(run_route(d, x, gate, gate_bias, nullptr, o, status, w, st, Noise{noise_u, temperature}));
  if (d.T > 0) MOE_TRY(run_scan(d, true, o.routed, o.P, aux, nullptr, nullptr, w, st));
  return MOE_OK;
}

moe_status moe_layer_fwd_gumbel(const moe_shape* s, const moe_bf16* x, const moe_bf16* gate,
                                const float* gate_bias, const float* noise_u, float temperature,
                                const moe_bf16* W1, const moe_bf16* W2, moe_bf16* y, float* aux,
                                int32_t* topk_idx, float* topk_w, int32_t* routed_counts, float* P,
                                int32_t* kept_counts, int32_t* offsets, int32_t* dest_row,
                                uint32_t* dev_status, void* ws, size_t ws_bytes, void* stream,
                                void* const* events) {
  MOE_TRY(check_noise(noise_u, temperature));
  return layer_fwd(s, x, gate, gate_bias, W1, W2, y, aux, topk_idx, topk_w, routed_counts, P,
                   kept_counts, offsets, dest_row, dev_status, ws, ws_bytes, stream, events,
                   Noise{noise_u, temperature});
}

moe_status moe_workspace_size_fp8(const moe_shape* s, size_t* bytes) {
  if (bytes == nullptr) return MOE_ERR_NULL;
  MOE_TRY(check_shape(s));
  *bytes = layout(dims_of(s), nullptr, nullptr, true);
  return MOE_OK;
}

moe_status moe_quantize_weights_fp8(int64_t E, int64_t K, int64_t N, const moe_bf16* W,
                                    uint8_t* Wq, float* w_scale, void* stream) {
  if (E <= 0 || K <= 0 || N <= 0) return MOE_ERR_SHAPE;
  if (E > kMaxExperts || K % 64 != 0 || N % 64 != 0 || K > kMaxDim || N > kMaxDim)
    return MOE_ERR_UNSUPPORTED;
  MOE_REQUIRE(W);
  MOE_REQUIRE(Wq);
  MOE_REQUIRE(w_scale);
  MOE_CUDA(launch_quantize_weights(W, Wq, w_scale, static_cast<int>(E), static_cast<int>(K),
                                   static_cast<int>(N), static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

moe_status moe_permute_fp8(const moe_shape* s, const moe_bf16* x, const int32_t* topk_idx,
                           int32_t* kept_counts, int32_t* offsets, int32_t* dest_row,
                           int32_t* src_token, uint8_t* x_q, float* x_scale,
                           uint32_t* dev_status, void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(check_shape(s));
  MOE_REQUIRE(x);
  MOE_REQUIRE(topk_idx);
  MOE_REQUIRE(offsets);
  MOE_REQUIRE(dest_row);
  MOE_REQUIRE(x_q);
  MOE_REQUIRE(x_scale);
  MOE_OPTIONAL(kept_counts);
  MOE_OPTIONAL(src_token);
  MOE_OPTIONAL(dev_status);
  const Dims d = dims_of(s);
  Ws w;
  MOE_TRY(carve(s, d, ws, ws_bytes, &w));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* status = dev_status ? dev_status : w.status;
  if (d.T == 0) {
    MOE_CUDA(cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (d.E + 1), st));
    if (kept_counts) MOE_CUDA(cudaMemsetAsync(kept_counts, 0, sizeof(int32_t) * d.E, st));
    return MOE_OK;
  }
  RankArgs r;
  r.T = d.T;
  r.E = d.E;
  r.k = d.k;
  r.n_tiles = d.n_tiles;
  r.topk_idx = topk_idx;
  r.tile_cnt = w.tile_cnt;
  r.rank8 = w.rank8;
  r.ticket = w.ticket;
  r.dev_status = status;
  MOE_CUDA(launch_rank(r, st));
  MOE_TRY(run_scan(d, false, w.routed, w.P, nullptr, kept_counts, offsets, w, st));
  MOE_TRY(run_gather_fp8(d, x, topk_idx, offsets, dest_row, src_token, x_q, x_scale, status, w,
                         st));
  return MOE_OK;
}

moe_status moe_expert_ffn_fp8(const moe_shape* s, const uint8_t* x_q, const float* x_scale,
                              const int32_t* offsets, const uint8_t* W1q, const float* w1_scale,
                              const uint8_t* W2q, const float* w2_scale, moe_bf16* act,
                              moe_bf16* y_perm, uint8_t* y_q, float* y_scale,
                              uint32_t* dev_status, void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(check_shape(s));
  MOE_REQUIRE(x_q);
  MOE_REQUIRE(x_scale);
  MOE_REQUIRE(offsets);
  MOE_REQUIRE(W1q);
  MOE_REQUIRE(w1_scale);
  MOE_REQUIRE(W2q);
  MOE_REQUIRE(w2_scale);
  MOE_REQUIRE(act);
  // the expert outputs: bf16 y_perm, or e4m3 y_q with its block scales
  if (y_perm != nullptr && y_q != nullptr) return MOE_ERR_UNSUPPORTED;
  if (y_q != nullptr) {
    MOE_REQUIRE(y_q);
    MOE_REQUIRE(y_scale);
  } else {
    MOE_REQUIRE(y_perm);
  }
  MOE_OPTIONAL(dev_status);
  const Dims d = dims_of(s);
  Ws w;
  MOE_TRY(carve(s, d, ws, ws_bytes, &w, true));
  uint32_t* status = dev_status ? dev_status : w.status;
  return run_ffn_fp8(d, x_q, x_scale, offsets, W1q, w1_scale, W2q, w2_scale, act, y_perm, status,
                     w, static_cast<cudaStream_t>(stream), nullptr, y_q, y_scale);
}

moe_status moe_combine_fp8(const moe_shape* s, const uint8_t* y_q, const float* y_scale,
                           const int32_t* dest_row, const float* topk_w, moe_bf16* y,
                           void* stream) {
  MOE_TRY(check_shape(s));
  MOE_REQUIRE(y_q);
  MOE_REQUIRE(y_scale);
  MOE_REQUIRE(dest_row);
  MOE_REQUIRE(topk_w);
  MOE_REQUIRE(y);
  const Dims d = dims_of(s);
  return run_combine_fp8(d, y_q, y_scale, dest_row, topk_w, y, static_cast<cudaStream_t>(stream));
}

moe_status moe_layer_fwd_fp8(const moe_shape* s, const moe_bf16* x, const moe_bf16* gate,
                             const float* gate_bias, const uint8_t* W1q, const float* w1_scale,
                             const uint8_t* W2q, const float* w2_scale, moe_bf16* y, float* aux,
                             int32_t* topk_idx, float* topk_w, int32_t* routed_counts, float* P,
                             int32_t* kept_counts, int32_t* offsets, int32_t* dest_row,
                             uint32_t* dev_status, void* ws, size_t ws_bytes, void* stream,
                             void* const* events) {
  const Fp8Weights q{W1q, w1_scale, W2q, w2_scale};
  return layer_fwd(s, x, gate, gate_bias, nullptr, nullptr, y, aux, topk_idx, topk_w,
                   routed_counts, P, kept_counts, offsets, dest_row, dev_status, ws, ws_bytes,
                   stream, events, Noise{nullptr, 1.0f}, &q);
}

static size_t host_ws_bytes(const Dims& d, bool fp8) {
  const size_t io = (static_cast<size_t>(d.T) * d.H * 2 + 255) & ~size_t(255);
  return layout(d, nullptr, nullptr, fp8) + 4 * io + 512;
}

moe_status moe_host_workspace_size(const moe_shape* s, size_t* bytes) {
  if (bytes == nullptr) return MOE_ERR_NULL;
  MOE_TRY(check_shape(s));
  *bytes = host_ws_bytes(dims_of(s), false);
  return MOE_OK;
}

moe_status moe_host_workspace_size_fp8(const moe_shape* s, size_t* bytes) {
  if (bytes == nullptr) return MOE_ERR_NULL;
  MOE_TRY(check_shape(s));
  *bytes = host_ws_bytes(dims_of(s), true);
  return MOE_OK;
}

// The three-stream micro-batch pipeline around one device layer call (bf16
// weights, or FP8 weights when q is set).
static moe_status layer_fwd_host(const moe_shape* s, int64_t n_micro,
                                 const moe_bf16* const* x_host, moe_bf16* const* y_host,
                                 float* aux_host, const moe_bf16* gate, const float* gate_bias,
                                 const moe_bf16* W1, const moe_bf16* W2, const Fp8Weights* q,
                                 uint32_t* dev_status, void* ws, size_t ws_bytes,
                                 void* const* streams, void* const* events) {
  MOE_TRY(check_shape(s));
  if (n_micro < 0) return MOE_ERR_SHAPE;
  if (x_host == nullptr || y_host == nullptr || streams == nullptr || events == nullptr)
    return MOE_ERR_NULL;
  MOE_REQUIRE(gate);
  if (q == nullptr) {
    MOE_REQUIRE(W1);
    MOE_REQUIRE(W2);
  } else {
    MOE_REQUIRE(q->W1q);
    MOE_REQUIRE(q->w1s);
    MOE_REQUIRE(q->W2q);
    MOE_REQUIRE(q->w2s);
  }
  MOE_OPTIONAL(gate_bias);
  MOE_OPTIONAL(dev_status);
  if (ws == nullptr) return MOE_ERR_NULL;
  if (!aligned16(ws)) return MOE_ERR_ALIGN;
  if (ws_bytes < host_ws_bytes(dims_of(s), q != nullptr)) return MOE_ERR_WORKSPACE;
  for (int i = 0; i < 3; ++i)
    if (streams[i] == nullptr) return MOE_ERR_NULL;
  for (int i = 0; i < 6; ++i)
    if (events[i] == nullptr) return MOE_ERR_NULL;
  for (int64_t i = 0; i < n_micro; ++i)
    if (x_host[i] == nullptr || y_host[i] == nullptr) return MOE_ERR_NULL;

  const Dims d = dims_of(s);
  const size_t layer_bytes = layout(d, nullptr, nullptr, q != nullptr);
  const size_t tok_bytes = static_cast<size_t>(d.T) * d.H * 2;
  const size_t io = (tok_bytes + 255) & ~size_t(255);
  uint8_t* base = static_cast<uint8_t*>(ws);
  moe_bf16* xbuf[2] = {reinterpret_cast<moe_bf16*>(base + layer_bytes),
                       reinterpret_cast<moe_bf16*>(base + layer_bytes + io)};
  moe_bf16* ybuf[2] = {reinterpret_cast<moe_bf16*>(base + layer_bytes + 2 * io),
                       reinterpret_cast<moe_bf16*>(base + layer_bytes + 3 * io)};
  float* auxbuf[2] = {reinterpret_cast<float*>(base + layer_bytes + 4 * io),
                      reinterpret_cast<float*>(base + layer_bytes + 4 * io + 256)};
  cudaStream_t sc = static_cast<cudaStream_t>(streams[0]);
  cudaStream_t sin = static_cast<cudaStream_t>(streams[1]);
  cudaStream_t sout = static_cast<cudaStream_t>(streams[2]);
  cudaEvent_t ev_in[2] = {static_cast<cudaEvent_t>(events[0]), static_cast<cudaEvent_t>(events[1])};
  cudaEvent_t ev_layer[2] = {static_cast<cudaEvent_t>(events[2]),
                             static_cast<cudaEvent_t>(events[3])};
  cudaEvent_t ev_out[2] = {static_cast<cudaEvent_t>(events[4]), static_cast<cudaEvent_t>(events[5])};

  for (int64_t i = 0; i < n_micro; ++i) {
    const int b = static_cast<int>(i & 1);
    // tokens in: buffer b is free once the layer of micro-batch i-2 is done
    if (i >= 2) MOE_CUDA(cudaStreamWaitEvent(sin, ev_layer[b], 0));
    if (tok_bytes)
      MOE_CUDA(cudaMemcpyAsync(xbuf[b], x_host[i], tok_bytes, cudaMemcpyHostToDevice, sin));
    MOE_CUDA(cudaEventRecord(ev_in[b], sin));
    // the layer: needs its tokens, and output buffer b drained (i-2 copied out)
    MOE_CUDA(cudaStreamWaitEvent(sc, ev_in[b], 0));
    if (i >= 2) MOE_CUDA(cudaStreamWaitEvent(sc, ev_out[b], 0));
    MOE_TRY(layer_fwd(s, xbuf[b], gate, gate_bias, W1, W2, ybuf[b], auxbuf[b], nullptr, nullptr,
                      nullptr, nullptr, nullptr, nullptr, nullptr, dev_status, ws, layer_bytes, sc,
                      nullptr, Noise{nullptr, 1.0f}, q));
    MOE_CUDA(cudaEventRecord(ev_layer[b], sc));
    // outputs out
    MOE_CUDA(cudaStreamWaitEvent(sout, ev_layer[b], 0));
    if (tok_bytes)
      MOE_CUDA(cudaMemcpyAsync(y_host[i], ybuf[b], tok_bytes, cudaMemcpyDeviceToHost, sout));
    if (aux_host)
      MOE_CUDA(cudaMemcpyAsync(aux_host + i, auxbuf[b], sizeof(float), cudaMemcpyDeviceToHost, sout));
    MOE_CUDA(cudaEventRecord(ev_out[b], sout));
  }
  return MOE_OK;
}

moe_status moe_layer_fwd_host(const moe_shape* s, int64_t n_micro, const moe_bf16* const* x_host,
                              moe_bf16* const* y_host, float* aux_host, const moe_bf16* gate,
                              const float* gate_bias, const moe_bf16* W1, const moe_bf16* W2,
                              uint32_t* dev_status, void* ws, size_t ws_bytes,
                              void* const* streams, void* const* events) {
  return layer_fwd_host(s, n_micro, x_host, y_host, aux_host, gate, gate_bias, W1, W2, nullptr,
                        dev_status, ws, ws_bytes, streams, events);
}

moe_status moe_pipelined_workspace_size(const moe_shape* s, size_t* bytes) {
  if (bytes == nullptr) return MOE_ERR_NULL;
  MOE_TRY(check_shape(s));
  *bytes = 2 * layout(dims_of(s), nullptr, nullptr);
  return MOE_OK;
}

// Micro-batch i uses layer workspace i % 2. Dispatch stream: route, scan and
// permute of micro-batch i, then (once its GEMMs are done) the combine of
// micro-batch i-1; expert stream: the two GEMMs of micro-batch i once its
// permute is done. The permute of i+1 and the combine of i-1 thus run while
// the GEMMs of i do, on the SM resources the GEMM leaves free. A workspace
// is reused only after the combine that last read it, which precedes the
// next route on the dispatch stream.
moe_status moe_layer_fwd_pipelined(const moe_shape* s, int64_t n_micro, const moe_bf16* x,
                                   const moe_bf16* gate, const float* gate_bias,
                                   const moe_bf16* W1, const moe_bf16* W2, moe_bf16* y,
                                   float* aux, uint32_t* dev_status, void* ws, size_t ws_bytes,
                                   void* const* streams, void* const* events) {
  MOE_TRY(check_shape(s));
  if (n_micro < 0 || s->T * n_micro >= (int64_t(1) << 31)) return MOE_ERR_SHAPE;
  if (streams == nullptr || events == nullptr) return MOE_ERR_NULL;
  for (int i = 0; i < 2; ++i)
    if (streams[i] == nullptr) return MOE_ERR_NULL;
  for (int i = 0; i < 4; ++i)
    if (events[i] == nullptr) return MOE_ERR_NULL;
  if (n_micro > 0) {
    MOE_REQUIRE(x);
    MOE_REQUIRE(y);
  }
  MOE_REQUIRE(gate);
  MOE_REQUIRE(W1);
  MOE_REQUIRE(W2);
  MOE_OPTIONAL(gate_bias);
  MOE_OPTIONAL(aux);
  MOE_OPTIONAL(dev_status);
  const Dims d = dims_of(s);
  const size_t one = layout(d, nullptr, nullptr);
  if (ws == nullptr) return MOE_ERR_NULL;
  if (!aligned16(ws)) return MOE_ERR_ALIGN;
  if (ws_bytes < 2 * one) return MOE_ERR_WORKSPACE;
  Ws w[2];
  layout(d, static_cast<uint8_t*>(ws), &w[0]);
  layout(d, static_cast<uint8_t*>(ws) + one, &w[1]);
  cudaStream_t sd = static_cast<cudaStream_t>(streams[0]);
  cudaStream_t se = static_cast<cudaStream_t>(streams[1]);
  cudaEvent_t ev_disp[2] = {static_cast<cudaEvent_t>(events[0]),
                            static_cast<cudaEvent_t>(events[1])};
  cudaEvent_t ev_ffn[2] = {static_cast<cudaEvent_t>(events[2]), static_cast<cudaEvent_t>(events[3])};
  const size_t rows = static_cast<size_t>(d.T) * d.H;
  auto combine_of = [&](int64_t i) -> moe_status {
    const Ws& wb = w[i & 1];
    MOE_CUDA(cudaStreamWaitEvent(sd, ev_ffn[i & 1], 0));
    return run_combine(d, wb.y_perm, wb.dest_row, wb.topk_w, y + static_cast<size_t>(i) * rows, sd);
  };
  for (int64_t i = 0; i < n_micro; ++i) {
    const Ws& wb = w[i & 1];
    uint32_t* status = dev_status ? dev_status : wb.status;
    const moe_bf16* xi = x + static_cast<size_t>(i) * rows;
    if (d.T == 0) break;
    RouteOut o{wb.topk_idx, wb.topk_w, wb.routed, wb.P, aux ? aux + i : nullptr, nullptr};
    MOE_TRY(run_route(d, xi, gate, gate_bias, nullptr, o, status, wb, sd));
    MOE_TRY(run_scan(d, true, wb.routed, wb.P, o.aux, wb.kept, wb.offsets, wb, sd));
    MOE_TRY(run_gather(d, xi, wb.topk_idx, wb.offsets, wb.dest_row, wb.src_token, wb.x_perm,
                       status, wb, sd));
    MOE_CUDA(cudaEventRecord(ev_disp[i & 1], sd));
    MOE_CUDA(cudaStreamWaitEvent(se, ev_disp[i & 1], 0));
    MOE_TRY(run_gemm(d, wb.x_perm, W1, wb.offsets, d.H, d.h, wb.act, 1, status, se));
    MOE_TRY(run_gemm(d, wb.act, W2, wb.offsets, d.h, d.H, wb.y_perm, 0, status, se));
    MOE_CUDA(cudaEventRecord(ev_ffn[i & 1], se));
    if (i >= 1) MOE_TRY(combine_of(i - 1));
  }
  if (n_micro > 0 && d.T > 0) MOE_TRY(combine_of(n_micro - 1));
  if (d.T == 0 && aux != nullptr && n_micro > 0)
    MOE_CUDA(cudaMemsetAsync(aux, 0, sizeof(float) * n_micro, sd));
  return MOE_OK;
}

moe_status moe_ep_permute(const moe_shape* s, int64_t world, int64_t rank,
                          const int32_t* routed_all, int64_t T_global, const moe_bf16* x,
                          const int32_t* topk_idx, int32_t* kept_counts, int32_t* offsets,
                          int32_t* dest_row, int32_t* src_token, moe_bf16* x_perm,
                          int32_t* send_counts, uint32_t* dev_status, void* ws, size_t ws_bytes,
                          void* stream) {
  MOE_TRY(check_shape(s));
  if (world < 1 || rank < 0 || rank >= world || s->E % world != 0) return MOE_ERR_SHAPE;
  MOE_REQUIRE(x);
  MOE_REQUIRE(topk_idx);
  MOE_REQUIRE(offsets);
  MOE_REQUIRE(dest_row);
  MOE_REQUIRE(x_perm);
  MOE_REQUIRE(send_counts);
  MOE_OPTIONAL(routed_all);
  MOE_OPTIONAL(kept_counts);
  MOE_OPTIONAL(src_token);
  MOE_OPTIONAL(dev_status);
  Dims d = dims_of(s);
  if (routed_all != nullptr) {
    // the capacity of the group's batch, served in global token order
    if (T_global < s->T || T_global * s->top_k >= (int64_t(1) << 31)) return MOE_ERR_SHAPE;
    d.C = moe_capacity(T_global, s->E, s->top_k, s->capacity_factor);
  }
  Ws w;
  MOE_TRY(carve(s, d, ws, ws_bytes, &w));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* status = dev_status ? dev_status : w.status;
  if (d.T == 0) {
    MOE_CUDA(cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (d.E + 1), st));
    MOE_CUDA(cudaMemsetAsync(send_counts, 0, sizeof(int32_t) * world, st));
    if (kept_counts) MOE_CUDA(cudaMemsetAsync(kept_counts, 0, sizeof(int32_t) * d.E, st));
    return MOE_OK;
  }
  RankArgs r;
  r.T = d.T;
  r.E = d.E;
  r.k = d.k;
  r.n_tiles = d.n_tiles;
  r.topk_idx = topk_idx;
  r.tile_cnt = w.tile_cnt;
  r.rank8 = w.rank8;
  r.ticket = w.ticket;
  r.dev_status = status;
  MOE_CUDA(launch_rank(r, st));
  ScanArgs sc;
  sc.T = d.T;
  sc.E = d.E;
  sc.k = d.k;
  sc.n_tiles = d.n_tiles;
  sc.C = d.C;
  sc.tile_cnt = w.tile_cnt;
  sc.tile_base = w.tile_base;
  sc.ppart = nullptr;
  sc.routed = w.routed;
  sc.P = w.P;
  sc.aux = nullptr;
  sc.kept = kept_counts;
  sc.offsets = offsets;
  sc.ticket = w.ticket;
  sc.routed_all = routed_all;
  sc.world = static_cast<int>(world);
  sc.rank = static_cast<int>(rank);
  sc.cap = w.cap;
  sc.send_counts = send_counts;
  MOE_CUDA(launch_scan(sc, st));
  GatherArgs g;
  g.T = d.T;
  g.H = d.H;
  g.E = d.E;
  g.k = d.k;
  g.n_tiles = d.n_tiles;
  g.C = d.C;
  g.cap = routed_all != nullptr ? w.cap : nullptr;
  g.x = x;
  g.topk_idx = topk_idx;
  g.rank8 = w.rank8;
  g.tile_base = w.tile_base;
  g.offsets = offsets;
  g.dest_row = dest_row;
  g.src_token = src_token;
  g.x_perm = x_perm;
  g.dev_status = status;
  MOE_CUDA(launch_gather(g, num_sms(), st));
  return MOE_OK;
}

moe_status moe_ep_regroup(int64_t world, int64_t E_local, int64_t H, int64_t rows,
                          int to_expert_major, const int32_t* counts, const moe_bf16* src,
                          moe_bf16* dst, int32_t* local_offsets, void* stream) {
  if (world < 1 || E_local < 1 || H <= 0 || rows < 0) return MOE_ERR_SHAPE;
  if (world * E_local > kMaxExperts || H % 64 != 0 || H > kMaxDim ||
      rows >= (int64_t(1) << 31))
    return MOE_ERR_UNSUPPORTED;
  MOE_REQUIRE(counts);
  MOE_OPTIONAL(local_offsets);
  if (rows > 0) {
    MOE_REQUIRE(src);
    MOE_REQUIRE(dst);
  }
  MOE_CUDA(launch_ep_regroup(static_cast<int>(world), static_cast<int>(E_local),
                             static_cast<int>(H), static_cast<int>(rows), to_expert_major ? 1 : 0,
                             counts, src, dst, local_offsets, num_sms(),
                             static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

moe_status moe_layer_fwd_host_fp8(const moe_shape* s, int64_t n_micro,
                                  const moe_bf16* const* x_host, moe_bf16* const* y_host,
                                  float* aux_host, const moe_bf16* gate, const float* gate_bias,
                                  const uint8_t* W1q, const float* w1_scale, const uint8_t* W2q,
                                  const float* w2_scale, uint32_t* dev_status, void* ws,
                                  size_t ws_bytes, void* const* streams, void* const* events) {
  const Fp8Weights q{W1q, w1_scale, W2q, w2_scale};
  return layer_fwd_host(s, n_micro, x_host, y_host, aux_host, gate, gate_bias, nullptr, nullptr,
                        &q, dev_status, ws, ws_bytes, streams, events);
}

}  // extern "C"
