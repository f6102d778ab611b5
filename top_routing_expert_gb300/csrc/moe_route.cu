// Router: logits GEMM on the tensor cores (tcgen05, accumulator in TMEM)
// fused with the routing epilogue - softmax over E, top-k with renormalised
// weights, per-tile partial sums of the probabilities, per-tile expert
// histograms and in-tile arrival ranks (MoE module notes, section 3.1 router
// listing; MoE comm bottleneck, section 3.2 auxiliary-loss statistics).
//
// One CTA = one tile of 128 tokens = one UMMA M. Thread r of the CTA owns
// token row r, which is TMEM lane r, so softmax and top-k need no
// cross-thread exchange.
#include <math.h>

#include "moe_internal.h"
#include "moe_ptx.cuh"

namespace moe {

namespace {


// ----------------------------------------------------------- top-k list ----

// A list of the KMAX best (logit, expert) pairs in registers, ordered by
// descending logit and, among equal logits, ascending expert index; its
// first k entries are the top-k for any k <= KMAX. An inserted pair sinks
// past every entry that precedes it in that order; a displaced entry carries
// on down the list the same way. The comparison is written without
// short-circuit operators: as `a || (b && c)` it compiled to divergent
// branches and the fine-grained router's epilogue (64 experts, top-6) spent
// 6.1 us in its first pass instead of 3.8.
template <int KMAX>
struct TopK {
  float v[KMAX];
  int i[KMAX];
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      v[j] = -INFINITY;
      i[j] = -1;
    }
  }
  __device__ __forceinline__ void insert(float cv, int ce) {
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      const bool gt = (cv > v[j]) | ((cv == v[j]) & (ce < i[j]));
      const float ov = v[j];
      const int oi = i[j];
      v[j] = gt ? cv : ov;
      i[j] = gt ? ce : oi;
      cv = gt ? ov : cv;
      ce = gt ? oi : ce;
    }
  }
};

// ---------------------------------------------------- tile ranks / counts --

// Called by all 128 threads of a routing tile. `e[j]` (j < k) is the
// thread's expert for slot j or -1 for an unusable slot. Produces for every
// slot the number of earlier tokens of the tile that chose the same expert
// (warp bit masks in shared memory, OR-ed, so the result does not depend on
// thread timing) and writes the tile's per-expert counts.
template <int KMAX>
__device__ __forceinline__ void tile_ranks(uint32_t* masks, int E_stride, int E, int k,
                                           const int (&e)[KMAX], bool row_valid,
                                           int (&rank)[KMAX], int32_t* tile_cnt,
                                           int n_tiles, int tile) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (row_valid) {
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (j < k && e[j] >= 0) atomicOr(&masks[warp * E_stride + e[j]], 1u << lane);
  }
  __syncthreads();
  const uint32_t below = (1u << lane) - 1u;
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    rank[j] = 0;
    if (j < k && row_valid && e[j] >= 0) {
      int r = __popc(masks[warp * E_stride + e[j]] & below);
      for (int w = 0; w < warp; ++w) r += __popc(masks[w * E_stride + e[j]]);
      rank[j] = r;
    }
  }
  for (int x = tid; x < E; x += kTileTokens) {
    int c = 0;
#pragma unroll
    for (int w = 0; w < kTileTokens / 32; ++w) c += __popc(masks[w * E_stride + x]);
    tile_cnt[static_cast<size_t>(x) * n_tiles + tile] = c;
  }
}

// --------------------------------------------------------------- sources ----

// Each epilogue thread owns one token row (TMEM lane) and one part of `cpt`
// expert columns of it: a CTA runs kTileTokens * npart threads, warp w
// reading lane quadrant w % 4 and part w / 4. Columns are handled 8 at a
// time in loops that are not unrolled, which keeps the code small.
constexpr int kChunk = 8;

// Router scores of the thread's row from TMEM (GEMM path): the logits plus
// the bias, and for the training router (module notes, section 3.1) plus
// Gumbel noise g = -log(-log(u + 1e-9) + 1e-9) from caller-drawn uniforms,
// divided by the temperature. The epilogue reads the scores in three passes:
// load_first serves the first and, with noise, writes the finished scores
// back over the accumulator (the uniforms are read and the logs taken once);
// load_next serves the others. `noisy` is the same for every thread.
struct TmemSource {
  uint32_t taddr;       // TMEM address of (this warp's lane quadrant, column 0)
  const float* bias_s;  // shared, zero past E
  const float* u_row;   // this token's uniforms [E], or nullptr (no noise / no token)
  float temperature;
  int E;
  bool noisy;           // the training router: scores are written back in pass 1
  __device__ __forceinline__ void load_first(int c, float (&v)[kChunk]) const {
    uint32_t r[kChunk];
    tmem_ld_32x32b_x8(taddr + static_cast<uint32_t>(c), r);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < kChunk; ++i) v[i] = __uint_as_float(r[i]) + bias_s[c + i];
    if (noisy) {
      if (u_row != nullptr) {
#pragma unroll
        for (int i = 0; i < kChunk; ++i) {
          if (c + i < E) {
            const float g = -logf(-logf(u_row[c + i] + 1e-9f) + 1e-9f);
            v[i] = (v[i] + g) / temperature;
          }
        }
      }
#pragma unroll
      for (int i = 0; i < kChunk; ++i) r[i] = __float_as_uint(v[i]);
      tmem_st_32x32b_x8(taddr + static_cast<uint32_t>(c), r);
    }
  }
  // after pass 1: the written-back scores are visible to this thread's loads
  __device__ __forceinline__ void first_done() const {
    if (noisy) tmem_st_wait();
  }
  __device__ __forceinline__ void load_next(int c, float (&v)[kChunk]) const {
    uint32_t r[kChunk];
    tmem_ld_32x32b_x8(taddr + static_cast<uint32_t>(c), r);
    tmem_ld_wait();
    if (noisy) {
#pragma unroll
      for (int i = 0; i < kChunk; ++i) v[i] = __uint_as_float(r[i]);
    } else {
#pragma unroll
      for (int i = 0; i < kChunk; ++i) v[i] = __uint_as_float(r[i]) + bias_s[c + i];
    }
  }
};

__device__ __forceinline__ const float* noise_row(const RouteArgs& a, int t) {
  return (a.noise_u != nullptr && t < a.T) ? a.noise_u + static_cast<size_t>(t) * a.E : nullptr;
}

// Logits of the thread's row from global memory (logits entry point).
struct GlobalSource {
  const float* row;
  int E;
  bool valid;
  __device__ __forceinline__ void load_first(int c, float (&v)[kChunk]) const { load_next(c, v); }
  __device__ __forceinline__ void first_done() const {}
  __device__ __forceinline__ void load_next(int c, float (&v)[kChunk]) const {
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      const int e = c + i;
      v[i] = (valid && e < E) ? row[e] : 0.f;
    }
  }
};

// Parts per token row (epilogue warps per TMEM lane quadrant) and columns
// per part: a multiple of 8, npart * cpt >= E.
__host__ __device__ inline int route_parts_of(int E) {
  return E <= 16 ? 1 : (E <= 32 ? 2 : (E <= 128 ? 4 : 8));
}
__host__ __device__ inline int route_cpt_of(int E) {
  const int n = route_parts_of(E);
  return ((E + n - 1) / n + kChunk - 1) / kChunk * kChunk;
}

// Shared scratch of the routing epilogue, laid out for `npart` parts.
struct EpiScratch {
  float* cand_v;  // [kTileTokens][npart][KMAX] per-part top-k; part 0 ends merged
  int* cand_i;
  float* psum;    // [kTileTokens][npart] per-part softmax partial sums
  float* rowmax;  // [kTileTokens]
  float* rowsum;  // [kTileTokens]
};

__host__ __device__ inline size_t epi_scratch_bytes(int npart, int kmax) {
  return static_cast<size_t>(kTileTokens) * npart * kmax * 8 + static_cast<size_t>(kTileTokens) * npart * 4 +
         2 * kTileTokens * 4;
}

__device__ __forceinline__ EpiScratch carve_epi(uint8_t* p, int npart, int kmax) {
  EpiScratch e;
  e.cand_v = reinterpret_cast<float*>(p);
  e.cand_i = reinterpret_cast<int*>(e.cand_v + kTileTokens * npart * kmax);
  e.psum = reinterpret_cast<float*>(e.cand_i + kTileTokens * npart * kmax);
  e.rowmax = e.psum + kTileTokens * npart;
  e.rowsum = e.rowmax + kTileTokens;
  return e;
}

// The routing epilogue shared by both paths; identical arithmetic, so equal
// logits give bit-identical results. All threads of the CTA call it.
//   1. each thread: top-k of its columns (ascending expert order);
//   2. part 0 merges the parts' lists in part order -> the token's top-k and
//      its max m (the order-defined comparator makes the merge exact);
//   3. softmax denominator: per-part sums of exp(l - m), added in part order;
//   4. weights exp(l_j - m) / sum_j exp(l_j - m) over the chosen k;
//   5. in-tile arrival ranks and per-tile expert counts from warp bit masks;
//   6. per-expert sums of p over the tile's tokens (fixed butterfly per warp,
//      then quadrants in order).
// The epilogue's thread group: the whole CTA (synchronised by
// __syncthreads) or, in the persistent router, the epilogue warps only
// (named barrier 1), numbered from `first_thread`.
struct CtaGroup {
  __device__ __forceinline__ int tid() const { return threadIdx.x; }
  __device__ __forceinline__ int size() const { return blockDim.x; }
  __device__ __forceinline__ void sync() const { __syncthreads(); }
};

struct WarpGroup {
  int first_thread, nthreads;
  __device__ __forceinline__ int tid() const { return threadIdx.x - first_thread; }
  __device__ __forceinline__ int size() const { return nthreads; }
  __device__ __forceinline__ void sync() const {
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
  }
};

template <int KMAX, class Src, class Group>
__device__ __forceinline__ void route_epilogue(const Src& src, const RouteArgs& a, int tile,
                                               EpiScratch es, uint32_t* masks, float* red,
                                               int E_stride, int npart, int cpt,
                                               const Group& grp) {
  const int tid = grp.tid(), lane = tid & 31, warp = tid >> 5;
  const int q = warp & 3, part = warp >> 2;
  const int r = 32 * q + lane;
  const int E = a.E, k = a.k;
  const int t = tile * kTileTokens + r;
  const bool valid = t < a.T;
  const int c0 = cpt * part;
  const int cend = c0 + cpt;

  TopK<KMAX> tk;
  tk.init();
  bool bad = false;
  float* lrow = (a.logits_out && valid) ? a.logits_out + static_cast<size_t>(t) * E : nullptr;
#pragma unroll 1
  for (int c = c0; c < cend; c += kChunk) {
    float v[kChunk];
    src.load_first(c, v);
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      const int e = c + i;
      if (e < E) {
        bad |= !isfinite(v[i]);
        tk.insert(v[i], e);
        if (lrow) lrow[e] = v[i];
      }
    }
  }
  src.first_done();
  const int cbase = (r * npart + part) * KMAX;
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    es.cand_v[cbase + j] = tk.v[j];
    es.cand_i[cbase + j] = tk.i[j];
  }
  grp.sync();
  if (part == 0) {
#pragma unroll 1
    for (int pp = 1; pp < npart; ++pp) {
      const int b = (r * npart + pp) * KMAX;
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (j < k) tk.insert(es.cand_v[b + j], es.cand_i[b + j]);
    }
    es.rowmax[r] = tk.v[0];
  }
  grp.sync();
  const float m = es.rowmax[r];
  float s_loc = 0.f;
#pragma unroll 1
  for (int c = c0; c < cend; c += kChunk) {
    float v[kChunk];
    src.load_next(c, v);
#pragma unroll
    for (int i = 0; i < kChunk; ++i)
      if (c + i < E) s_loc += expf(v[i] - m);
  }
  es.psum[r * npart + part] = s_loc;
  grp.sync();

  int eid[KMAX];
  float ex[KMAX];
  float den = 0.f;
  if (part == 0) {
    float s = es.psum[r * npart];
#pragma unroll 1
    for (int pp = 1; pp < npart; ++pp) s += es.psum[r * npart + pp];
    es.rowsum[r] = s;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      eid[j] = (j < k) ? tk.i[j] : -1;
      ex[j] = (j < k && tk.i[j] >= 0) ? expf(tk.v[j] - m) : 0.f;
      den += ex[j];
      if (valid && eid[j] >= 0) atomicOr(&masks[q * E_stride + eid[j]], 1u << lane);
    }
  }
  grp.sync();

  // per-expert probability sums over the warp's 32 tokens, 8 columns at a
  // time: three halving rounds (partners 4, 2, 1 apart; a lane keeps the
  // half of its columns its lane bit selects and adds the partner's copy of
  // that half) leave lane l the sum over its 8-lane group of column l & 7,
  // and two butterfly rounds (8, 16) add the four groups: 9 shuffles per 8
  // columns instead of 40, in a fixed order
  const float inv_s = 1.0f / es.rowsum[r];
#pragma unroll 1
  for (int c = c0; c < cend; c += kChunk) {
    float v[kChunk];
    src.load_next(c, v);
    float pv[kChunk];
#pragma unroll
    for (int i = 0; i < kChunk; ++i) pv[i] = (valid && c + i < E) ? expf(v[i] - m) * inv_s : 0.f;
#pragma unroll
    for (int h = kChunk / 2; h > 0; h >>= 1) {
      const bool up = (lane & h) != 0;
#pragma unroll
      for (int i = 0; i < h; ++i) {
        const float send = up ? pv[i] : pv[i + h];
        const float keep = up ? pv[i + h] : pv[i];
        pv[i] = keep + __shfl_xor_sync(0xffffffffu, send, h);
      }
    }
    float tot = pv[0];
    tot += __shfl_xor_sync(0xffffffffu, tot, 8);
    tot += __shfl_xor_sync(0xffffffffu, tot, 16);
    if (lane < kChunk && c + lane < E) red[q * E_stride + c + lane] = tot;
  }

  if (part == 0 && valid) {
    const uint32_t below = (1u << lane) - 1u;
    const size_t base = static_cast<size_t>(t) * k;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (j < k) {
        int rk = 0;
        if (eid[j] >= 0) {
          rk = __popc(masks[q * E_stride + eid[j]] & below);
          for (int w = 0; w < q; ++w) rk += __popc(masks[w * E_stride + eid[j]]);
        }
        a.topk_idx[base + j] = eid[j];
        a.topk_w[base + j] = ex[j] / den;
        a.rank8[base + j] = static_cast<uint8_t>(rk);
      }
    }
  }
  if (bad && valid) atomicOr(a.dev_status, MOE_DEV_NONFINITE);
  for (int x = tid; x < E; x += grp.size()) {
    int c = 0;
#pragma unroll
    for (int w = 0; w < kTileTokens / 32; ++w) c += __popc(masks[w * E_stride + x]);
    a.tile_cnt[static_cast<size_t>(x) * a.n_tiles + tile] = c;
  }
  grp.sync();
  for (int x = tid; x < E; x += grp.size()) {
    float sum = red[x];
#pragma unroll
    for (int w = 1; w < kTileTokens / 32; ++w) sum += red[w * E_stride + x];
    a.ppart[static_cast<size_t>(x) * a.n_tiles + tile] = sum;
  }
}

// ---------------------------------------------------------------- kernels ---

__global__ void gate_transpose_kernel(const uint16_t* __restrict__ gate,
                                      uint16_t* __restrict__ gateT, int H, int E, int E_pad) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t n = static_cast<int64_t>(E_pad) * H;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int e = static_cast<int>(i / H);
    const int hh = static_cast<int>(i - static_cast<int64_t>(e) * H);
    gateT[i] = e < E ? gate[static_cast<int64_t>(hh) * E + e] : uint16_t(0);
  }
}

// A pipeline stage holds a.kbps consecutive 64-deep k-blocks (kb0 ..
// kb0+kbps-1): first x, one 3-D TMA box of 128 rows x 64 k x kbps k-blocks
// (k-block r at r * 16 KB, the K-major 128-byte-swizzled layout per
// k-block), then the gate. Fewer, larger copies keep more of x in flight
// per instruction: streaming 512 MB through 152 SMs with 64 KB copies ran
// 25 % faster than with 16 KB ones on GB300.
//
// The gate's part: one 3-D box of the transposed gate [E_pad, H] (k-block
// r's E_pad rows at r * E_pad * 128 bytes), or ceil(E_pad/64) boxes of 64
// expert columns x 64*kbps k rows of the gate [H, E] as given (column block
// cb at cb * kbps * 8 KB, k-block r at r * 8 KB inside it; the inner
// coordinate is a multiple of 64 elements, so every box starts on a
// 128-byte boundary).
__device__ __forceinline__ void load_route_stage(uint8_t* dst, const CUtensorMap* tm_x,
                                                 const CUtensorMap* tm_gate, uint64_t* bar,
                                                 int tile, int kb0, const RouteArgs& a) {
  tma_load_3d(dst, tm_x, bar, 0, tile * kTileTokens, kb0);
  uint8_t* g = dst + static_cast<size_t>(a.kbps) * kTileTokens * kBlockK * 2;
  if (a.gate_mode == kGateMnMajor) {
    for (int cb = 0; cb < (a.E_pad + 63) / 64; ++cb)
      tma_load_2d(g + 8192 * a.kbps * cb, tm_gate, bar, 64 * cb, kb0 * kBlockK);
  } else {
    tma_load_3d(g, tm_gate, bar, 0, 0, kb0);
  }
}

// The UMMAs of one stage: D[128 x E_pad] (+)= X[128 x 64] * gate^T[64 x
// E_pad] for each of its k-blocks, 16-deep K steps. Gate descriptors:
// K-major 128-byte rows (32 bytes per step), or MN-major 128-byte rows of 64
// experts, one per k (16 rows = 2 KB per step, column blocks kbps * 8 KB
// apart).
__device__ __forceinline__ void route_stage_mma(uint32_t d_tmem, uint32_t stage_addr,
                                                uint32_t idesc, bool first, const RouteArgs& a) {
  const uint32_t b_addr = stage_addr + static_cast<uint32_t>(a.kbps) * kTileTokens * kBlockK * 2;
  for (int r = 0; r < a.kbps; ++r) {
#pragma unroll
    for (int kk = 0; kk < kBlockK / 16; ++kk) {
      const uint64_t ad = smem_desc_sw128(stage_addr + 16384u * r + 32u * kk, 16u, 1024u);
      const uint64_t bd =
          a.gate_mode == kGateMnMajor
              ? smem_desc_sw128(b_addr + 8192u * r + 2048u * kk, 8192u * a.kbps, 1024u)
              : smem_desc_sw128(b_addr + static_cast<uint32_t>(a.E_pad) * 128u * r + 32u * kk,
                                16u, 1024u);
      umma_bf16(d_tmem, ad, bd, idesc, (first && (r | kk) == 0) ? 0u : 1u);
    }
  }
}

__device__ __forceinline__ uint32_t route_idesc(const RouteArgs& a) {
  return idesc_bf16_f32(kTileTokens, static_cast<uint32_t>(a.E_pad), false,
                        a.gate_mode == kGateMnMajor);
}

// Shared-memory carve-up of the router kernel after the 1024-aligned
// pipeline stages (the stages are reused as epilogue scratch once the
// accumulator is complete).
struct RouteSmem {
  uint64_t* full;
  uint64_t* empty;
  uint64_t* done;
  uint32_t* tmem_slot;
  uint32_t* abort_flag;
  float* bias_s;
  uint32_t* masks;
  float* red;
};

__device__ __forceinline__ RouteSmem carve_route_smem(uint8_t* p, int stages, int E32) {
  RouteSmem s;
  s.full = reinterpret_cast<uint64_t*>(p);
  s.empty = s.full + stages;
  s.done = s.empty + stages;
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.done + 1);
  s.abort_flag = s.tmem_slot + 1;
  s.bias_s = reinterpret_cast<float*>(s.abort_flag + 2);
  s.masks = reinterpret_cast<uint32_t*>(s.bias_s + E32);
  s.red = reinterpret_cast<float*>(s.masks + 4 * E32);
  return s;
}

// One CTA per 128-token tile; the launcher picks this kernel when there are
// no more tiles than SMs (the persistent kernel takes larger batches), so
// one CTA per SM and a stage ring of up to ~200 KB.
template <int KMAX>
__global__ void __launch_bounds__(kTileTokens * 8, 1)
    route_gemm_kernel(const __grid_constant__ CUtensorMap tm_x,
                      const __grid_constant__ CUtensorMap tm_gate, RouteArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_up_1024(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tile = blockIdx.x;
  const int S = a.stages;
  const int npart = route_parts_of(a.E), cpt = route_cpt_of(a.E);
  const int ecols = npart * cpt;                // columns the epilogue reads (>= E)
  const int E32 = ((ecols > a.E_pad ? ecols : a.E_pad) + 31) & ~31;
  const uint32_t stage_bytes = route_stage_bytes(a.E_pad, a.gate_mode, a.kbps);
  RouteSmem sm = carve_route_smem(smem + static_cast<size_t>(S) * stage_bytes, S, E32);
  const uint32_t ncols = static_cast<uint32_t>(route_tmem_cols(E32));

  if (warp == 0) {
    tmem_alloc(sm.tmem_slot, ncols);
    tmem_relinquish();
  }
  if (warp == 1 && lane == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    mbar_init(sm.done, 1);
    *sm.abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp == 2 && lane == 0) {
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_gate);
  }
  // the prologue above touches no global memory; everything below may
  // depend on the previous kernel on the stream
  grid_dependency_wait();
  grid_launch_dependents();
  if (tile == 0 && tid == 0) *a.ticket = 0u;
  for (int i = tid; i < E32; i += blockDim.x)
    sm.bias_s[i] = (a.bias != nullptr && i < a.E) ? a.bias[i] : 0.f;
  for (int i = tid; i < 4 * E32; i += blockDim.x) sm.masks[i] = 0u;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_slot;
  const WaitCtl wc{sm.abort_flag, a.dev_status, a.timeout_ns};
  const int ns = a.H / (kBlockK * a.kbps);  // stages per tile

  if (warp == 0 && lane == 0) {
    // TMA producer (an L2 prefetch of whole 512-byte row pieces ahead of
    // these loads measured 2-8 % slower and was dropped)
    int i = 0;
    for (; i < ns; ++i) {
      const int s = i % S;
      if (i >= S && !mbar_wait(&sm.empty[s], ((i / S) - 1) & 1, wc)) break;
      mbar_arrive_expect_tx(&sm.full[s], stage_bytes);
      load_route_stage(smem + static_cast<size_t>(s) * stage_bytes, &tm_x, &tm_gate, &sm.full[s],
                       tile, i * a.kbps, a);
    }
    if (i < ns) {
      // aborted: let the loads already issued land before the CTA exits
      for (int d = (i > S ? i - S : 0); d < i; ++d)
        mbar_wait_drain(&sm.full[d % S], (d / S) & 1, kDrainLimitNs);
    }
  } else if (warp == 1 && lane == 0) {
    // UMMA issuer
    const uint32_t idesc = route_idesc(a);
    for (int i = 0; i < ns; ++i) {
      const int s = i % S;
      if (!mbar_wait(&sm.full[s], (i / S) & 1, wc)) break;
      tc_fence_after();
      route_stage_mma(tmem, smem_u32(smem + static_cast<size_t>(s) * stage_bytes), idesc, i == 0,
                      a);
      umma_commit(&sm.empty[s]);
    }
    umma_commit(sm.done);
  }
  __syncwarp();

  // all threads: wait for the accumulator, then the routing epilogue (the
  // decision is made CTA-uniform because the epilogue synchronises)
  // `done` is committed even on abort and fires once the issued UMMAs are
  // finished, which TMEM release must wait for: a fixed drain limit, not
  // the (caller-settable) pipeline timeout.
  const bool done_ok = mbar_wait_drain(sm.done, 0, kDrainLimitNs);
  const int go = __syncthreads_and(done_ok && *sm.abort_flag == 0u);
  tc_fence_after();
  if (go) {
    const int t_row = tile * kTileTokens + 32 * (warp & 3) + lane;
    TmemSource src{tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16), sm.bias_s,
                   noise_row(a, t_row), a.temperature, a.E, a.noise_u != nullptr};
    // the pipeline stages are free now: they hold the epilogue scratch
    route_epilogue<KMAX>(src, a, tile, carve_epi(smem, npart, KMAX), sm.masks, sm.red, E32,
                         npart, cpt, CtaGroup{});
  } else if (tid == 0) {
    atomicOr(a.dev_status, MOE_DEV_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, ncols);
}

// Persistent router (used when there are more tiles than SMs): one CTA per
// SM takes tiles blockIdx.x, +gridDim.x, ...
// Warp 0 streams x and the gate through the stage ring across tile
// boundaries, warp 1 issues the UMMAs into one of two TMEM accumulators,
// and 4 * npart epilogue warps (warps 4..) route the previous tile from the
// other accumulator meanwhile, synchronising among themselves only.
constexpr int kPersistParts = 4;

__host__ __device__ inline int persist_parts_of(int E) {
  const int n = route_parts_of(E);
  return n > kPersistParts ? kPersistParts : n;
}
__host__ __device__ inline int persist_cpt_of(int E) {
  const int n = persist_parts_of(E);
  return ((E + n - 1) / n + kChunk - 1) / kChunk * kChunk;
}

struct PersistLayout {
  int S, npart, cpt, E32;
  uint32_t stage_bytes, ncols;
  size_t off_bar, off_bias, off_masks, off_red, off_epi, total;
};

__host__ __device__ inline PersistLayout persist_layout(int E, int E_pad, int kmax, int gate_mode,
                                                        int kbps) {
  PersistLayout L;
  L.npart = persist_parts_of(E);
  L.cpt = persist_cpt_of(E);
  const int ecols = L.npart * L.cpt;
  L.E32 = ((ecols > E_pad ? ecols : E_pad) + 31) & ~31;
  L.stage_bytes = route_stage_bytes(E_pad, gate_mode, kbps);
  int c = 32;
  while (c < 2 * L.E32) c <<= 1;
  L.ncols = static_cast<uint32_t>(c);
  const size_t fixed = 8 * 24 + 16 + static_cast<size_t>(L.E32) * 4 * 9 + epi_scratch_bytes(L.npart, kmax);
  int S = static_cast<int>((225 * 1024 - 1024 - fixed) / L.stage_bytes);
  L.S = S > 8 ? 8 : S;
  L.off_bar = static_cast<size_t>(L.S) * L.stage_bytes;
  L.off_bias = L.off_bar + 8 * (2 * L.S + 5) + 16;
  L.off_masks = L.off_bias + 4 * L.E32;
  L.off_red = L.off_masks + 16 * L.E32;
  L.off_epi = L.off_red + 16 * L.E32;
  L.total = 1024 + L.off_epi + epi_scratch_bytes(L.npart, kmax);
  return L;
}

template <int KMAX>
__global__ void __launch_bounds__(kTileTokens + kTileTokens * kPersistParts, 1)
    route_persistent_kernel(const __grid_constant__ CUtensorMap tm_x,
                            const __grid_constant__ CUtensorMap tm_gate, RouteArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_up_1024(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const PersistLayout L = persist_layout(a.E, a.E_pad, KMAX, a.gate_mode, a.kbps);
  const int S = L.S, E32 = L.E32;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.off_bar);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  uint32_t* abort_flag = tmem_slot + 1;
  float* bias_s = reinterpret_cast<float*>(smem + L.off_bias);
  uint32_t* masks = reinterpret_cast<uint32_t*>(smem + L.off_masks);
  float* red = reinterpret_cast<float*>(smem + L.off_red);
  const EpiScratch es = carve_epi(smem + L.off_epi, L.npart, KMAX);
  const int n_epi = kTileTokens * L.npart;

  if (warp == 0) {
    tmem_alloc(tmem_slot, L.ncols);
    tmem_relinquish();
  }
  if (warp == 1 && lane == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], n_epi);
    }
    mbar_init(drain, 1);
    *abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp == 2 && lane == 0) {
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_gate);
  }
  // the prologue above touches no global memory; everything below may
  // depend on the previous kernel on the stream
  grid_dependency_wait();
  grid_launch_dependents();
  if (blockIdx.x == 0 && tid == 0) *a.ticket = 0u;
  for (int i = tid; i < E32; i += blockDim.x)
    bias_s[i] = (a.bias != nullptr && i < a.E) ? a.bias[i] : 0.f;
  for (int i = tid; i < 4 * E32; i += blockDim.x) masks[i] = 0u;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{abort_flag, a.dev_status, a.timeout_ns};
  const int ns = a.H / (kBlockK * a.kbps);  // stages per tile

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer ----
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool aborted = false;
      for (int tile = blockIdx.x; tile < a.n_tiles && !aborted; tile += gridDim.x) {
        for (int i = 0; i < ns; ++i) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, wc)) {
            aborted = true;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], L.stage_bytes);
          load_route_stage(smem + static_cast<size_t>(stage) * L.stage_bytes, &tm_x, &tm_gate,
                           &full[stage], tile, i * a.kbps, a);
          ++issued;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (aborted) {
        int s = stage;
        uint32_t ph = phase;
        for (int d = 0; d < S && d < issued; ++d) {
          if (--s < 0) {
            s = S - 1;
            ph ^= 1u;
          }
          mbar_wait_drain(&full[s], ph, kDrainLimitNs);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------- UMMA issuer ----
      const uint32_t idesc = route_idesc(a);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool aborted = false;
      for (int tile = blockIdx.x; tile < a.n_tiles && !aborted; tile += gridDim.x) {
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, wc)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * E32);
        for (int i = 0; i < ns; ++i) {
          if (!mbar_wait(&full[stage], phase, wc)) {
            aborted = true;
            break;
          }
          tc_fence_after();
          route_stage_mma(d_tmem, smem_u32(smem + static_cast<size_t>(stage) * L.stage_bytes),
                          idesc, i == 0, a);
          umma_commit(&empty[stage]);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (aborted) break;
        umma_commit(&tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // TMEM is released only after every issued UMMA is done
      umma_commit(drain);
      mbar_wait_drain(drain, 0, kDrainLimitNs);
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------- epilogue ----
    const WarpGroup grp{kTileTokens, n_epi};
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < a.n_tiles; tile += gridDim.x) {
      if (!mbar_wait(&tfull[acc], acc_phase, wc)) break;
      tc_fence_after();
      TmemSource src{tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(acc * E32),
                     bias_s, noise_row(a, tile * kTileTokens + 32 * q + lane), a.temperature, a.E,
                     a.noise_u != nullptr};
      route_epilogue<KMAX>(src, a, tile, es, masks, red, E32, L.npart, L.cpt, grp);
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      // clear the bit masks for the next tile (ordered before its use by the
      // next tile's first group barrier)
      for (int i = grp.tid(); i < 4 * E32; i += n_epi) masks[i] = 0u;
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, L.ncols);
}

template <int KMAX>
__global__ void __launch_bounds__(kTileTokens * 8, 1) route_logits_kernel(RouteArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tile = blockIdx.x;
  const int npart = route_parts_of(a.E), cpt = route_cpt_of(a.E);
  const int E32 = (npart * cpt + 31) & ~31;
  EpiScratch es = carve_epi(smem_raw, npart, KMAX);
  uint32_t* masks = reinterpret_cast<uint32_t*>(smem_raw + epi_scratch_bytes(npart, KMAX));
  float* red = reinterpret_cast<float*>(masks + 4 * E32);
  grid_dependency_wait();
  grid_launch_dependents();
  if (tile == 0 && tid == 0) *a.ticket = 0u;
  for (int i = tid; i < 4 * E32; i += blockDim.x) masks[i] = 0u;
  __syncthreads();
  const int t = tile * kTileTokens + 32 * (warp & 3) + lane;
  GlobalSource src{a.logits_in + static_cast<size_t>(t < a.T ? t : 0) * a.E, a.E, t < a.T};
  route_epilogue<KMAX>(src, a, tile, es, masks, red, E32, npart, cpt, CtaGroup{});
}

// Tile counts and ranks from caller-given indices. A slot is unusable if its
// expert is outside [0,E) or repeats an earlier slot of the same token; the
// gather kernel applies the same rule and drops it.
__global__ void __launch_bounds__(kTileTokens) rank_kernel(RankArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const int tid = threadIdx.x;
  const int tile = blockIdx.x;
  const int E32 = (a.E + 31) & ~31;
  uint32_t* masks = reinterpret_cast<uint32_t*>(smem_raw);
  grid_dependency_wait();
  grid_launch_dependents();
  if (tile == 0 && tid == 0) *a.ticket = 0u;
  for (int i = tid; i < 4 * E32; i += kTileTokens) masks[i] = 0u;
  __syncthreads();
  const int t = tile * kTileTokens + tid;
  const bool valid = t < a.T;
  int e[kMaxTopK];
  uint32_t bits = 0;
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    e[j] = -1;
    if (valid && j < a.k) {
      const int v = a.topk_idx[static_cast<size_t>(t) * a.k + j];
      bool ok = v >= 0 && v < a.E;
      if (!ok) bits |= MOE_DEV_BAD_INDEX;
#pragma unroll
      for (int jj = 0; jj < j; ++jj)
        if (ok && e[jj] == v) {
          ok = false;
          bits |= MOE_DEV_DUP_INDEX;
        }
      e[j] = ok ? v : -1;
    }
  }
  if (bits) atomicOr(a.dev_status, bits);
  int rank[kMaxTopK];
  tile_ranks<kMaxTopK>(masks, E32, a.E, a.k, e, valid, rank, a.tile_cnt, a.n_tiles, tile);
  if (valid) {
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      if (j < a.k) a.rank8[static_cast<size_t>(t) * a.k + j] = static_cast<uint8_t>(rank[j]);
  }
}

}  // namespace

// ------------------------------------------------------------------ host ----

size_t route_smem_bytes(int E_pad, int stages, int gate_mode, int kbps) {
  const int E = E_pad;  // upper bound for the epilogue's column span
  const int ecols = route_parts_of(E) * route_cpt_of(E);
  const int E32 = ((ecols > E_pad ? ecols : E_pad) + 31) & ~31;
  const size_t stage = route_stage_bytes(E_pad, gate_mode, kbps);
  return 1024 + stage * stages + 8 * (2 * stages + 1) + 16 + 4 * E32 + 2 * 4 * 4 * E32;
}

cudaError_t launch_gate_transpose(const uint16_t* gate, uint16_t* gateT, int H, int E, int E_pad,
                                  cudaStream_t st) {
  const int64_t n = static_cast<int64_t>(H) * E_pad;
  int blocks = static_cast<int>((n + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  return launch_pdl(gate_transpose_kernel, dim3(blocks), dim3(256), 0, st, gate, gateT, H, E, E_pad);
}

template <int KMAX>
cudaError_t launch_route_gemm_k(const CUtensorMap& tm_x, const CUtensorMap& tm_gate,
                                const RouteArgs& a, cudaStream_t st) {
  const int npart = route_parts_of(a.E);
  // the epilogue scratch lives in the pipeline stages once they are free
  const size_t stage_area =
      static_cast<size_t>(a.stages) * route_stage_bytes(a.E_pad, a.gate_mode, a.kbps);
  if (epi_scratch_bytes(npart, KMAX) > stage_area) return cudaErrorInvalidConfiguration;
  const size_t smem = route_smem_bytes(a.E_pad, a.stages, a.gate_mode, a.kbps);
  cudaError_t err = cudaFuncSetAttribute(route_gemm_kernel<KMAX>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  return launch_pdl(route_gemm_kernel<KMAX>, dim3(a.n_tiles), dim3(kTileTokens * npart), smem, st,
                    tm_x, tm_gate, a);
}

template <int KMAX>
cudaError_t launch_route_persistent_k(const CUtensorMap& tm_x, const CUtensorMap& tm_gate,
                                      const RouteArgs& a, int num_sms, cudaStream_t st) {
  const PersistLayout L = persist_layout(a.E, a.E_pad, KMAX, a.gate_mode, a.kbps);
  if (L.S < 2) return cudaErrorInvalidConfiguration;
  cudaError_t err = cudaFuncSetAttribute(route_persistent_kernel<KMAX>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(L.total));
  if (err != cudaSuccess) return err;
  const int grid = a.n_tiles < num_sms ? a.n_tiles : num_sms;
  return launch_pdl(route_persistent_kernel<KMAX>, dim3(grid),
                    dim3(kTileTokens + kTileTokens * L.npart), L.total, st, tm_x, tm_gate, a);
}

bool route_use_persistent(const RouteArgs& a, int num_sms) {
  return a.n_tiles > num_sms;
}

// k-blocks per stage: 4, 2 or 1, the largest that divides H/64 and leaves at
// least two stages in the kernel's ring; the per-tile kernel then takes as
// many stages as fit in ~200 KB (at most 10).
void route_plan(RouteArgs& a, int num_sms) {
  const int nk = a.H / kBlockK;
  const int kmax = a.k <= 2 ? 2 : a.k <= 4 ? 4 : a.k <= 6 ? 6 : 8;
  const bool persistent = route_use_persistent(a, num_sms);
  constexpr int kRing = 200 * 1024;
  for (int r = 4; r >= 1; r >>= 1) {
    if (nk % r != 0) continue;
    a.kbps = r;
    const bool fits =
        persistent ? persist_layout(a.E, a.E_pad, kmax, a.gate_mode, r).S >= 2
                   : kRing / static_cast<int>(route_stage_bytes(a.E_pad, a.gate_mode, r)) >= 2;
    if (fits) break;
  }
  a.stages = 0;
  if (!persistent) {
    const int s = kRing / static_cast<int>(route_stage_bytes(a.E_pad, a.gate_mode, a.kbps));
    a.stages = s < 2 ? 2 : (s > 10 ? 10 : s);
  }
}

cudaError_t launch_route_gemm(const CUtensorMap& tm_x, const CUtensorMap& tm_gate,
                              const RouteArgs& a, cudaStream_t st, int num_sms) {
  if (route_use_persistent(a, num_sms)) {
    if (a.k <= 2) return launch_route_persistent_k<2>(tm_x, tm_gate, a, num_sms, st);
    if (a.k <= 4) return launch_route_persistent_k<4>(tm_x, tm_gate, a, num_sms, st);
    if (a.k <= 6) return launch_route_persistent_k<6>(tm_x, tm_gate, a, num_sms, st);
    return launch_route_persistent_k<8>(tm_x, tm_gate, a, num_sms, st);
  }
  if (a.k <= 2) return launch_route_gemm_k<2>(tm_x, tm_gate, a, st);
  if (a.k <= 4) return launch_route_gemm_k<4>(tm_x, tm_gate, a, st);
  if (a.k <= 6) return launch_route_gemm_k<6>(tm_x, tm_gate, a, st);
  return launch_route_gemm_k<8>(tm_x, tm_gate, a, st);
}

template <int KMAX>
cudaError_t launch_route_logits_k(const RouteArgs& a, cudaStream_t st) {
  const int npart = route_parts_of(a.E);
  const int E32 = (npart * route_cpt_of(a.E) + 31) & ~31;
  const size_t smem = epi_scratch_bytes(npart, KMAX) + 2 * 4 * 4 * static_cast<size_t>(E32);
  cudaError_t err = cudaFuncSetAttribute(route_logits_kernel<KMAX>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  return launch_pdl(route_logits_kernel<KMAX>, dim3(a.n_tiles), dim3(kTileTokens * npart), smem, st,
                    a);
}

cudaError_t launch_route_logits(const RouteArgs& a, cudaStream_t st) {
  if (a.k <= 2) return launch_route_logits_k<2>(a, st);
  if (a.k <= 4) return launch_route_logits_k<4>(a, st);
  if (a.k <= 6) return launch_route_logits_k<6>(a, st);
  return launch_route_logits_k<8>(a, st);
}

cudaError_t launch_rank(const RankArgs& a, cudaStream_t st) {
  const int E32 = (a.E + 31) & ~31;
  return launch_pdl(rank_kernel, dim3(a.n_tiles), dim3(kTileTokens), 4 * 4 * E32, st, a);
}

}  // namespace moe
