// Expert parallelism: the experts are spread over `world` ranks, E/world
// consecutive experts each, and each token's rows travel to the rank that
// holds its expert and back (the dispatch and combine all-to-alls of the MoE
// comm bottleneck page, section 1.1). A rank's dispatch buffer is already
// ordered by destination rank (it is expert-major); what a rank receives
// comes source by source, each source's rows of this rank's experts in
// expert order. The grouped GEMM wants them expert by expert, so
// regroup_kernel moves rows between the two orders:
//
//   source-major : block (r, e) for r = 0..world-1, then e = 0..E_loc-1
//   expert-major : block (r, e) for e = 0..E_loc-1, then r = 0..world-1
//
// With sources in rank order inside an expert, the expert-major rows of an
// expert are its rows in global token order, rank after rank.
#include "moe_internal.h"
#include "moe_ptx.cuh"

namespace moe {

namespace {

constexpr int kRegroupThreads = 256;  // >= world * E_loc (at most 256 experts)

// Inclusive Hillis-Steele scan of one value per thread over the block.
__device__ __forceinline__ int block_inclusive_scan(int v, int* sh) {
  sh[threadIdx.x] = v;
  __syncthreads();
  for (int o = 1; o < kRegroupThreads; o <<= 1) {
    const int add = threadIdx.x >= o ? sh[threadIdx.x - o] : 0;
    __syncthreads();
    sh[threadIdx.x] += add;
    __syncthreads();
  }
  const int r = sh[threadIdx.x];
  __syncthreads();
  return r;
}

// counts[r * E_loc + e]: rows source r sends for local expert e (negative
// counts are read as 0). Each block forms both prefix tables, then warps copy
// rows; rows at or past `rows` (the buffers' size) are never touched.
__global__ void __launch_bounds__(kRegroupThreads)
    regroup_kernel(int world, int E_loc, int H, int rows, int to_expert_major,
                   const int32_t* __restrict__ counts, const uint4* __restrict__ src,
                   uint4* __restrict__ dst, int32_t* __restrict__ local_offsets) {
  __shared__ int scan_sh[kRegroupThreads];
  __shared__ int src_off[kRegroupThreads + 1];  // rows before block b, source-major
  __shared__ int exp_off[kRegroupThreads + 1];  // rows before block j, expert-major
  grid_dependency_wait();
  grid_launch_dependents();
  const int n = world * E_loc;
  const int tid = threadIdx.x;
  // source-major block b = r * E_loc + e; expert-major block j = e * world + r
  int c_src = 0, c_exp = 0;
  if (tid < n) {
    c_src = max(counts[tid], 0);
    const int e = tid / world, r = tid - e * world;
    c_exp = max(counts[r * E_loc + e], 0);
  }
  const int inc_src = block_inclusive_scan(c_src, scan_sh);
  const int inc_exp = block_inclusive_scan(c_exp, scan_sh);
  if (tid < n) {
    src_off[tid + 1] = inc_src;
    exp_off[tid + 1] = inc_exp;
  }
  if (tid == 0) src_off[0] = exp_off[0] = 0;
  __syncthreads();
  const int total = src_off[n];
  const int live = total < rows ? total : rows;
  if (blockIdx.x == 0 && to_expert_major && local_offsets != nullptr) {
    if (tid < E_loc) local_offsets[tid] = min(exp_off[tid * world], rows);
    if (tid == 0) local_offsets[E_loc] = live;
  }

  const int lane = tid & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int nvec = H >> 3;  // 16-byte vectors per row
  for (int i = (blockIdx.x * blockDim.x + tid) >> 5; i < live; i += warps) {
    // the source-major block holding row i: the last b with src_off[b] <= i
    // (an empty block shares its start with the next one, so the last such b
    // is never empty)
    int lo = 0, hi = n - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (src_off[mid] <= i) lo = mid; else hi = mid - 1;
    }
    const int r = lo / E_loc, e = lo - r * E_loc;
    const int j = exp_off[e * world + r] + (i - src_off[lo]);
    if (j >= rows) continue;
    const uint4* from = src + static_cast<size_t>(to_expert_major ? i : j) * nvec;
    uint4* to = dst + static_cast<size_t>(to_expert_major ? j : i) * nvec;
    for (int v = lane; v < nvec; v += 32) to[v] = from[v];
  }
}

}  // namespace

cudaError_t launch_ep_regroup(int world, int E_loc, int H, int rows, int to_expert_major,
                              const int32_t* counts, const uint16_t* src, uint16_t* dst,
                              int32_t* local_offsets, int num_sms, cudaStream_t st) {
  int blocks = (rows + 7) / 8;  // 8 warps (rows) per block
  const int cap = num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_pdl(regroup_kernel, dim3(blocks), dim3(kRegroupThreads), 0, st, world, E_loc, H,
                    rows, to_expert_major, counts, reinterpret_cast<const uint4*>(src),
                    reinterpret_cast<uint4*>(dst), local_offsets);
}

}  // namespace moe
