// Internal interface between the host entry points (moe_api.cu) and the
// kernel files. Not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "moe_gb300.h"

namespace moe {

constexpr int kTileTokens = 128;  // tokens per routing tile = router GEMM M
constexpr int kMaxTopK = 8;
constexpr int kMaxExperts = 256;
constexpr int kBlockK = 64;       // K per pipeline stage (one 128-byte swizzle row of bf16)
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // 2 s per pipeline wait
constexpr uint64_t kDrainLimitNs = 200000000ull;      // waits for in-flight copies/MMAs on abort

// Router epilogue arguments (GEMM and logits entry points).
struct RouteArgs {
  int T, H, E, E_pad, k, n_tiles, stages;
  int kbps;                // 64-deep k-blocks per pipeline stage (1, 2 or 4; divides H/64)
  int gate_mode;           // how the gate reaches shared memory (kGate* below)
  const float* bias;       // [E] or nullptr (GEMM path only)
  const float* noise_u;    // [T,E] uniforms in [0,1) for Gumbel noise, or nullptr
  float temperature;       // scores = (logits + gumbel(u)) / temperature when noise_u
  const float* logits_in;  // [T,E] (logits path only)
  int32_t* topk_idx;       // [T,k]
  float* topk_w;           // [T,k]
  float* logits_out;       // [T,E] or nullptr
  int32_t* tile_cnt;       // [E][n_tiles] assignments per routing tile
  uint8_t* rank8;          // [T*k] rank of the token among its tile's tokens of that expert
  float* ppart;            // [E][n_tiles] sum of p over the tile's tokens
  uint32_t* ticket;        // reset to 0 by block 0 (used by the scan)
  uint32_t* dev_status;
  uint64_t timeout_ns;
};

// Tile counts and ranks from caller-given indices (dispatch without route).
struct RankArgs {
  int T, E, k, n_tiles;
  const int32_t* topk_idx;
  int32_t* tile_cnt;
  uint8_t* rank8;
  uint32_t* ticket;
  uint32_t* dev_status;
};

struct ScanArgs {
  int T, E, k, n_tiles;
  int64_t C;
  const int32_t* tile_cnt;  // [E][n_tiles]
  int32_t* tile_base;       // [E][n_tiles] exclusive prefix over tiles
  const float* ppart;       // [E][n_tiles] or nullptr (no P / aux)
  int32_t* routed;          // [E]
  float* P;                 // [E]
  float* aux;               // [1] or nullptr
  int32_t* kept;            // [E] or nullptr
  int32_t* offsets;         // [E+1] or nullptr
  uint32_t* ticket;
  // expert parallelism (all nullptr / 0 otherwise): the experts are spread
  // over `world` ranks (E/world consecutive experts each) and every expert
  // serves the group's tokens in global order, rank after rank
  const int32_t* routed_all = nullptr;  // [world][E] assignments of every rank, before drops
  int world = 1, rank = 0;
  int32_t* cap = nullptr;               // [E] out: this rank's capacity left per expert
  int32_t* send_counts = nullptr;       // [world] out: kept rows for each rank's experts
};

struct GatherArgs {
  int T, H, E, k, n_tiles;
  int64_t C;
  const int32_t* cap = nullptr;  // [E] per-expert capacity (expert parallelism), else C
  const uint16_t* x;
  const int32_t* topk_idx;
  const uint8_t* rank8;
  const int32_t* tile_base;
  const int32_t* offsets;
  int32_t* dest_row;
  int32_t* src_token;  // or nullptr
  uint16_t* x_perm;
  uint32_t* dev_status;
};

struct CombineArgs {
  int T, H, k;
  const uint16_t* y_perm;
  const int32_t* dest_row;
  const float* topk_w;
  uint16_t* y;
};

// TMEM columns the router allocates: a power of two >= 32 covering E_pad.
__host__ __device__ inline int route_tmem_cols(int E_pad) {
  int c = 32;
  while (c < E_pad) c <<= 1;
  return c;
}

struct GemmArgs {
  const int32_t* offsets;  // [E+1] row segments of the expert-major buffer
  int E, K, N;             // reduction size, output columns
  int rows;                // rows of the A and D buffers (T*k)
  uint16_t* D;             // [rows, N] bf16
  int gelu;                // 1: act = gelu_tanh(acc), 0: plain
  const float* a_scale;    // FP8 mode: per-row scales of A [rows]
  const float* b_scale;    // FP8 mode: per-column scales of B [E, N]
  uint32_t* row_amax;      // FP8 mode, optional: max |bf16 output| per row, fp32 bits,
                           // combined with atomicMax (zeroed by the caller)
  uint8_t* Dq;             // FP8 mode, optional: e4m3 output [rows, N] instead of D, with
  float* d_scale;          //   one scale per (row, 128-column block): [rows, ceil(N/128)]
  const int32_t* a_rows;   // optional: A row r is row a_rows[r] of the A tensor (a gather,
  int a_src_rows;          //   by TMA, from a tensor of a_src_rows rows); CTA-pair kernel
  int stages;              // CTA-pair kernel: pipeline depth (set by its launcher)
  uint32_t* dev_status;
  uint64_t timeout_ns;
};

// How the router's B operand (the gate, N = E_pad experts x K = H) reaches
// each pipeline stage:
//   kGateTransposed - TMA from a transposed, zero-padded copy [E_pad, H] made
//                     in the workspace by a separate kernel (K-major rows:
//                     E_pad TMA rows of 128 bytes per stage);
//   kGateMnMajor    - TMA from the gate [H, E] as given, MN-major, in boxes of
//                     64 experts x 64 k (E % 8 == 0, so rows are 16-byte
//                     multiples). Used for E >= 64, where the boxes are full;
//                     for fewer experts most of each box is zero fill, and 64
//                     TMA rows per stage instead of E_pad slow the router
//                     (large-expert router 76 -> 93 us on GB300).
enum { kGateTransposed = 0, kGateMnMajor = 1 };

// Shared-memory bytes of the gate per 64-deep k-block.
__host__ __device__ inline uint32_t route_gate_stage_bytes(int E_pad, int gate_mode) {
  return gate_mode == kGateMnMajor ? static_cast<uint32_t>((E_pad + 63) / 64) * 8192u
                                   : static_cast<uint32_t>(E_pad) * kBlockK * 2;
}

// Shared-memory bytes of one router pipeline stage of `kbps` k-blocks: the
// tile's 128 rows of x and the gate's rows for those k-blocks.
__host__ __device__ inline uint32_t route_stage_bytes(int E_pad, int gate_mode, int kbps) {
  return static_cast<uint32_t>(kbps) *
         (static_cast<uint32_t>(kTileTokens * kBlockK * 2) + route_gate_stage_bytes(E_pad, gate_mode));
}

size_t gemm_smem_bytes(int E);

cudaError_t launch_gate_transpose(const uint16_t* gate, uint16_t* gateT, int H, int E, int E_pad,
                                  cudaStream_t st);
// Launches `kernel` on `st` with programmatic stream serialisation: its
// CTAs may start, and run the prologue that touches no global memory, while
// the previous kernel on the stream finishes (that kernel's
// grid_launch_dependents()). Every kernel launched this way calls
// grid_dependency_wait() before its first global access.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Sets a.kbps and a.stages for the router kernel launch_route_gemm will run
// (a.E, a.E_pad, a.H, a.k, a.n_tiles and a.gate_mode set).
void route_plan(RouteArgs& a, int num_sms);
size_t route_smem_bytes(int E_pad, int stages, int gate_mode, int kbps);
cudaError_t launch_route_gemm(const CUtensorMap& tm_x, const CUtensorMap& tm_gate,
                              const RouteArgs& a, cudaStream_t st, int num_sms);
cudaError_t launch_route_logits(const RouteArgs& a, cudaStream_t st);
cudaError_t launch_rank(const RankArgs& a, cudaStream_t st);
cudaError_t launch_scan(const ScanArgs& a, cudaStream_t st);
cudaError_t launch_gather(const GatherArgs& a, int num_sms, cudaStream_t st);
cudaError_t launch_combine(const CombineArgs& a, int num_sms, cudaStream_t st);
cudaError_t launch_grouped_gemm(const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                                const GemmArgs& a, int num_sms, cudaStream_t st);
cudaError_t launch_grouped_gemm_pair(const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                                     const GemmArgs& a, int num_sms, cudaStream_t st);
size_t gemm_pair_smem_bytes(int E, int stages, bool fp8, int kb_per_stage);
// FP8 operands; writes D (bf16), or Dq + d_scale when a.Dq is set
cudaError_t launch_grouped_gemm_pair_fp8(const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                                         const GemmArgs& a, int num_sms, cudaStream_t st);
cudaError_t launch_combine_fp8(const CombineArgs& a, const uint8_t* y_q, const float* y_scale,
                               int num_sms, cudaStream_t st);
cudaError_t launch_quantize_weights(const uint16_t* W, uint8_t* Wq, float* Ws, int E, int K,
                                    int N, cudaStream_t st);
cudaError_t launch_row_quant(const uint16_t* src, const uint32_t* amax, uint8_t* dst,
                             float* scale, const int32_t* offsets, int E, int rows, int K,
                             int num_sms, cudaStream_t st);
cudaError_t launch_gather_fp8(const GatherArgs& a, uint8_t* xq, float* xs, int num_sms,
                              cudaStream_t st);
// Rows between the source-major order a rank receives them in and the
// expert-major order of its experts (expert parallelism).
cudaError_t launch_ep_regroup(int world, int E_loc, int H, int rows, int to_expert_major,
                              const int32_t* counts, const uint16_t* src, uint16_t* dst,
                              int32_t* local_offsets, int num_sms, cudaStream_t st);

}  // namespace moe
