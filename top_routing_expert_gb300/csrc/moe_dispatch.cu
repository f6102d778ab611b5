// Dispatch and combine without a collective: the single-GPU form of the two
// all-to-alls of an MoE layer (MoE comm bottleneck, section 1.1).
//
//  scan    - per expert, an exclusive scan of the routing tiles' counts gives
//            each tile's first arrival position; the last block to finish
//            applies the capacity (section 3.1: C = ceil(cf*T*k/E), later
//            tokens dropped), scans the kept counts into segment offsets and
//            forms the balance statistics (section 3.2).
//  gather  - one warp per token: position = tile base + in-tile rank; kept
//            rows are copied to the expert-major buffer with 16-byte loads.
//  combine - one warp per token: fp32 weighted sum of its kept expert rows.
//
// Integer work only decides who goes where, so routing, drops and the
// permutation are exact and independent of thread timing.
#include "moe_internal.h"
#include "moe_ptx.cuh"

namespace moe {

namespace {

constexpr int kScanThreads = 256;

// Exclusive scan over a 256-thread block; `total` gets the block sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int* sh, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) sh[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int s = lane < kScanThreads / 32 ? sh[lane] : 0;
    int si = s;
#pragma unroll
    for (int o = 1; o < kScanThreads / 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, si, o);
      if (lane >= o) si += n;
    }
    if (lane < kScanThreads / 32) sh[lane] = si - s;
    if (lane == kScanThreads / 32 - 1) sh[kScanThreads / 32] = si;
  }
  __syncthreads();
  const int r = sh[warp] + incl - v;
  total = sh[kScanThreads / 32];
  __syncthreads();
  return r;
}

// Sum over a 256-thread block in a fixed tree order (deterministic). fp32:
// the sums are of at most a few thousand per-tile partials, and fp64 is
// slow on this part (the scan took 10.2 us with fp64 sums, 7.6 with fp32).
__device__ __forceinline__ float block_sum(float v, float* sh) {
  sh[threadIdx.x] = v;
  __syncthreads();
#pragma unroll
  for (int s = kScanThreads / 2; s > 0; s >>= 1) {
    if (threadIdx.x < s) sh[threadIdx.x] += sh[threadIdx.x + s];
    __syncthreads();
  }
  const float r = sh[0];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kScanThreads) scan_kernel(ScanArgs a) {
  __shared__ int shi[kScanThreads / 32 + 1];
  __shared__ float shf[kScanThreads];
  __shared__ int last;
  grid_dependency_wait();
  grid_launch_dependents();
  const int e = blockIdx.x, tid = threadIdx.x;
  const int n = a.n_tiles;
  const int per = (n + kScanThreads - 1) / kScanThreads;
  const int i0 = min(tid * per, n), i1 = min(i0 + per, n);
  const int32_t* cnt = a.tile_cnt + static_cast<size_t>(e) * n;
  int32_t* base = a.tile_base + static_cast<size_t>(e) * n;

  int local = 0;
  for (int i = i0; i < i1; ++i) local += cnt[i];
  int total;
  int run = block_exclusive_scan(local, shi, total);
  for (int i = i0; i < i1; ++i) {
    base[i] = run;
    run += cnt[i];
  }
  if (tid == 0) a.routed[e] = total;
  if (a.ppart != nullptr) {
    const float* pp = a.ppart + static_cast<size_t>(e) * n;
    float ps = 0.f;
    for (int i = i0; i < i1; ++i) ps += pp[i];
    const float tot = block_sum(ps, shf);
    if (tid == 0) a.P[e] = a.T > 0 ? tot / static_cast<float>(a.T) : 0.f;
  }

  // the last block to arrive sees every expert's totals
  __threadfence();
  __syncthreads();
  if (tid == 0) last = (atomicAdd(a.ticket, 1u) == gridDim.x - 1) ? 1 : 0;
  __syncthreads();
  if (!last) return;
  __threadfence();

  const int r = tid < a.E ? __ldcg(&a.routed[tid]) : 0;
  int64_t cap = a.C;
  if (a.routed_all != nullptr && tid < a.E) {
    // expert parallelism: the ranks before this one claim their assignments
    // to the expert first (global token order), this rank gets what is left
    int64_t before = 0;
    for (int q = 0; q < a.rank; ++q) before += a.routed_all[static_cast<size_t>(q) * a.E + tid];
    cap = a.C - before < 0 ? 0 : a.C - before;
    if (a.cap) a.cap[tid] = static_cast<int32_t>(cap);
  }
  const int kept = static_cast<int>(r < cap ? r : cap);
  int all;
  const int off = block_exclusive_scan(tid < a.E ? kept : 0, shi, all);
  if (tid < a.E) {
    if (a.kept) a.kept[tid] = kept;
    if (a.offsets) a.offsets[tid] = off;
  }
  if (tid == 0 && a.offsets) a.offsets[a.E] = all;
  if (a.send_counts != nullptr) {
    // rank g holds experts g*E/world .. (g+1)*E/world - 1: its rows are
    // the offsets between those two expert boundaries
    __shared__ int off_sh[kMaxExperts + 1];
    if (tid < a.E) off_sh[tid] = off;
    if (tid == 0) off_sh[a.E] = all;
    __syncthreads();
    const int per = a.E / a.world;
    if (tid < a.world) a.send_counts[tid] = off_sh[(tid + 1) * per] - off_sh[tid * per];
  }
  if (a.aux != nullptr) {
    float term = 0.f;
    if (tid < a.E && a.T > 0)
      term = (static_cast<float>(r) / (static_cast<float>(a.T) * static_cast<float>(a.k))) *
             __ldcg(&a.P[tid]);
    const float s = block_sum(term, shf);
    if (tid == 0) *a.aux = a.T > 0 ? static_cast<float>(a.E) * s : 0.f;
  }
  if (tid == 0) *a.ticket = 0u;
}

// One warp per token. Lane j < k owns slot j.
template <int U>
__global__ void __launch_bounds__(256) gather_kernel(GatherArgs a) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int nvec = a.H >> 3;  // 16-byte vectors per row
  const uint4* __restrict__ xv = reinterpret_cast<const uint4*>(a.x);
  uint4* __restrict__ pv = reinterpret_cast<uint4*>(a.x_perm);
  const int64_t rows = static_cast<int64_t>(a.T) * a.k;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < a.T; t += warps) {
    int e = -1;
    if (lane < a.k) e = a.topk_idx[static_cast<size_t>(t) * a.k + lane];
    bool ok = lane < a.k && e >= 0 && e < a.E;
    uint32_t bits = (lane < a.k && !ok) ? MOE_DEV_BAD_INDEX : 0u;
    for (int jj = 0; jj < a.k; ++jj) {
      const int other = __shfl_sync(0xffffffffu, e, jj);
      if (jj < lane && ok && other == e) {
        ok = false;
        bits |= MOE_DEV_DUP_INDEX;
      }
    }
    int dest = -1;
    if (ok) {
      const int64_t pos = static_cast<int64_t>(a.tile_base[static_cast<size_t>(e) * a.n_tiles + t / kTileTokens]) +
                          a.rank8[static_cast<size_t>(t) * a.k + lane];
      const int64_t row = static_cast<int64_t>(a.offsets[e]) + pos;
      // rows outside the buffer can only come from routing state left
      // incomplete by an aborted kernel (MOE_DEV_TIMEOUT): never written
      const int64_t cap = a.cap != nullptr ? a.cap[e] : a.C;
      if (pos >= 0 && pos < cap && row >= 0 && row < rows) dest = static_cast<int>(row);
    }
    if (lane < a.k) {
      a.dest_row[static_cast<size_t>(t) * a.k + lane] = dest;
      if (dest >= 0 && a.src_token) a.src_token[dest] = t;
      if (bits) atomicOr(a.dev_status, bits);
    }
    int d[kMaxTopK];
    bool any = false;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      d[j] = __shfl_sync(0xffffffffu, dest, j);
      any |= j < a.k && d[j] >= 0;
    }
    // index-only dispatch (GEMM1 gathers the rows itself), or a token whose
    // every slot was dropped: its row is not read at all
    if (pv == nullptr || !any) continue;

    const uint4* src = xv + static_cast<size_t>(t) * nvec;
    for (int b = 0; b < nvec; b += 32 * U) {
      uint4 buf[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = b + 32 * u + lane;
        if (i < nvec) buf[u] = __ldg(src + i);
      }
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j) {
        if (j < a.k && d[j] >= 0) {
          uint4* dst = pv + static_cast<size_t>(d[j]) * nvec;
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int i = b + 32 * u + lane;
            if (i < nvec) dst[i] = buf[u];
          }
        }
      }
    }
  }
}

// One warp per token; slots accumulate in ascending j, fp32. Every kept
// slot's vectors are loaded before any is used, so a token's k row reads are
// in flight together.
template <int KMAX, int U>
__global__ void __launch_bounds__(256, (KMAX * U > 8) ? 2 : 3) combine_kernel(CombineArgs a) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int nvec = a.H >> 3;
  const uint4* __restrict__ yv = reinterpret_cast<const uint4*>(a.y_perm);
  uint4* __restrict__ ov = reinterpret_cast<uint4*>(a.y);
  const int rows = a.T * a.k;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < a.T; t += warps) {
    int dl = -1;
    float wl = 0.f;
    if (lane < a.k) {
      dl = a.dest_row[static_cast<size_t>(t) * a.k + lane];
      wl = a.topk_w[static_cast<size_t>(t) * a.k + lane];
      if (dl < 0 || dl >= rows) dl = -1;  // only rows of the buffer are read
    }
    int d[KMAX];
    float w[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      d[j] = __shfl_sync(0xffffffffu, dl, j);
      w[j] = __shfl_sync(0xffffffffu, wl, j);
      if (j >= a.k) d[j] = -1;
    }
    for (int b = 0; b < nvec; b += 32 * U) {
      uint4 v[KMAX][U];
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int i = b + 32 * u + lane;
          v[j][u] = (d[j] >= 0 && i < nvec) ? __ldg(yv + static_cast<size_t>(d[j]) * nvec + i)
                                           : make_uint4(0, 0, 0, 0);
        }
      float acc[U][8];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[u][q] = 0.f;
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (d[j] >= 0) {
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const uint32_t wd[4] = {v[j][u].x, v[j][u].y, v[j][u].z, v[j][u].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              acc[u][2 * q] = fmaf(w[j], bf16_lo(wd[q]), acc[u][2 * q]);
              acc[u][2 * q + 1] = fmaf(w[j], bf16_hi(wd[q]), acc[u][2 * q + 1]);
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = b + 32 * u + lane;
        if (i < nvec) {
          uint4 o;
          o.x = pack_bf16x2(acc[u][0], acc[u][1]);
          o.y = pack_bf16x2(acc[u][2], acc[u][3]);
          o.z = pack_bf16x2(acc[u][4], acc[u][5]);
          o.w = pack_bf16x2(acc[u][6], acc[u][7]);
          ov[static_cast<size_t>(t) * nvec + i] = o;
        }
      }
    }
  }
}

int warp_grid(int T, int num_sms) {
  const int need = (T + 7) / 8;  // 8 warps per 256-thread block
  const int cap = num_sms * 8;
  return need < cap ? need : cap;
}

}  // namespace

cudaError_t launch_scan(const ScanArgs& a, cudaStream_t st) {
  return launch_pdl(scan_kernel, dim3(a.E), dim3(kScanThreads), 0, st, a);
}

cudaError_t launch_gather(const GatherArgs& a, int num_sms, cudaStream_t st) {
  if (a.T == 0) return cudaSuccess;
  const int grid = warp_grid(a.T, num_sms);
  return launch_pdl(gather_kernel<8>, dim3(grid), dim3(256), 0, st, a);
}

cudaError_t launch_combine(const CombineArgs& a, int num_sms, cudaStream_t st) {
  if (a.T == 0) return cudaSuccess;
  const int grid = warp_grid(a.T, num_sms);
  if (a.k <= 2) return launch_pdl(combine_kernel<2, 4>, dim3(grid), dim3(256), 0, st, a);
  if (a.k <= 4) return launch_pdl(combine_kernel<4, 2>, dim3(grid), dim3(256), 0, st, a);
  if (a.k <= 6) return launch_pdl(combine_kernel<6, 2>, dim3(grid), dim3(256), 0, st, a);
  return launch_pdl(combine_kernel<8, 1>, dim3(grid), dim3(256), 0, st, a);
}

}  // namespace moe
