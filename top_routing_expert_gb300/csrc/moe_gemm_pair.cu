// Grouped GEMM over ragged expert segments, CTA-pair version: the same
// product as grouped_gemm_kernel (D[r,:] = A[r,:] . B[e(r)], optional GELU)
// with a 2-CTA UMMA (cta_group::2, M=256, N=256). Each CTA of a cluster pair
// holds its own 128 rows of A and its own 128 columns of B per 64-deep
// k-block, 32 KB instead of 48 KB, so shared memory moves a third less data
// per FLOP than the single-CTA kernel. In the bf16 kernel that loads A by
// tile, a pipeline stage holds two k-blocks (64 KB, three stages): A as one
// 3-D TMA box of 128 rows x 2 k-blocks, B as two boxes of 64 columns x 128
// k-rows. On the power-capped large-expert layer this took GEMM1 from 0.81
// to 0.89 and GEMM2 from 0.87 to 0.92 of the measured burst peak on GB300
// against one k-block per 32 KB stage (seven stages): half as many stage
// hand-offs and barrier waits for the same bytes. The FP8 kernel's stages
// hold two 128-deep k-blocks as one 2-D box each of A and B; the
// gathered-A kernel keeps one k-block per stage.
//
// A pair tile is (expert e, pair index pm, n-tile): CTA rank r computes the
// expert's local m-tile 2*pm + r (128 rows) against all 256 columns. An
// expert with an odd m-tile count leaves the last pair's second half past
// the segment end; its rows are computed and never stored.
//
// Roles per CTA (320 threads): warp 0 = TMA producer (both CTAs, own halves,
// transaction bytes counted on the leader's barrier); warp 1 = UMMA issuer
// (leader only) and TMEM allocation (both, collectively); warps 2-9 =
// epilogue of the CTA's own 128 rows, two warps per TMEM lane quadrant, each
// taking half of the 256 columns. Stage and accumulator barriers are
// released to both CTAs by multicast commits; the leader waits for both
// epilogues before reusing an accumulator.
#include <cuda_fp8.h>

#include "moe_internal.h"
#include "moe_ptx.cuh"

namespace moe {

namespace {

constexpr int kBM = 128;           // rows per CTA; the pair computes 256
constexpr int kBN = 256;           // columns per pair tile (128 held by each CTA)
constexpr int kMaxStages = 7;  // bf16 with E <= 234; FP8 (scale area) and larger E: 6
constexpr int kEpiWarps = 8;                             // 2 per TMEM lane quadrant
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr uint32_t kABytes = kBM * kBlockK * 2;          // 16 KB
constexpr uint32_t kBBytes = (kBN / 2) * kBlockK * 2;    // 16 KB
constexpr uint32_t kStageBytes = kABytes + kBBytes;      // 32 KB per k-block
constexpr int kWideKB = 2;  // k-blocks per stage of the bf16 tile-loaded kernel
constexpr uint32_t kTmemCols = 2 * kBN;                  // two accumulators
// Pair m-tiles per raster group: 16 when the experts average at least 16
// pair m-tiles (4096 rows) and A's rows are short, so that a group stays
// within one expert's weights (1.7 % faster on the power-capped large-expert
// layer, whose DRAM traffic it lowers); 8 for smaller or ragged experts
// (0.5-0.8 % faster there) and for A rows of 16 KB or more, where a group's
// A panels are 8 x 256 such rows (the large-expert bf16 GEMM2, K = 14336,
// read 9.7 instead of 10.9 GB per launch, in the same time).
__device__ __forceinline__ int raster_group(int total_pm, int E, int a_row_bytes) {
  return (total_pm >= 16 * E && a_row_bytes < 16384) ? 16 : 8;
}

struct PairTile {
  int e, row0, row_end, n0;
};

// n-tile index of pair tile L (the raster arithmetic of decode_pair).
__device__ __forceinline__ int pair_tile_nt(int L, int E, int total_pm, int n_tiles_n,
                                            int a_row_bytes) {
  const int group = raster_group(total_pm, E, a_row_bytes);
  const int per_group = group * n_tiles_n;
  const int g = L / per_group;
  const int gsz = min(group, total_pm - g * group);
  return (L - g * per_group) / gsz;
}

__device__ __forceinline__ PairTile decode_pair(int L, const int* pm_prefix, const int* offs,
                                                int E, int total_pm, int n_tiles_n, int rank,
                                                int a_row_bytes) {
  const int group = raster_group(total_pm, E, a_row_bytes);
  const int per_group = group * n_tiles_n;
  const int g = L / per_group;
  const int first = g * group;
  const int gsz = min(group, total_pm - first);
  const int r = L - g * per_group;
  const int pm = first + r % gsz;
  const int nt = r / gsz;
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pm_prefix[mid] <= pm) lo = mid; else hi = mid - 1;
  }
  PairTile t;
  t.e = lo;
  t.row0 = offs[lo] + (2 * (pm - pm_prefix[lo]) + rank) * kBM;
  t.row_end = offs[lo + 1];
  t.n0 = nt * kBN;
  return t;
}

__device__ __forceinline__ float gelu_tanh_f(float u) {
  // 0.5 u (1 + tanh(z)) = u / (1 + exp(-2 z)),  z = sqrt(2/pi) (u + 0.044715 u^3)
  const float z2 = 1.5957691216057308f * fmaf(0.044715f * u, u * u, u);
  return __fdividef(u, 1.0f + __expf(-z2));
}

// kFp8: A and B are e4m3 (both K-major, 128 elements = 128 bytes per
// stage row), the UMMA is kind::f8f6f4 and the epilogue multiplies by the
// row scale of A and the column scale of B. Otherwise bf16 A (K-major) and
// bf16 B (MN-major), 64 elements per stage row.
// kGather (bf16): A row r is row a_rows[r] of the token matrix, fetched by
// TMA tile::gather4 - the dispatch's permutation fused into the A load, so
// no permuted copy of the tokens is written or read. The whole producer warp
// issues: lane l gathers rows 4l..4l+3 of the CTA's 128-row tile.
// kQOut (with kFp8): the output is e4m3 with one scale per 128-column block
// of a row - exactly the columns one epilogue warp holds - formed from the
// bf16-rounded values: a first pass over the warp's TMEM chunks finds the
// block maximum, a second one converts and stores.
template <bool kFp8, bool kQOut, bool kGather>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tm_a,
                             const __grid_constant__ CUtensorMap tm_b, GemmArgs p) {
  constexpr int kKE = kFp8 ? 128 : kBlockK;  // K elements per k-block
  constexpr int kKBS = kGather ? 1 : kWideKB;  // k-blocks per stage
  constexpr uint32_t kSB = kKBS * kStageBytes;             // bytes per stage
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_up_1024(smem_raw);
  const int nst = p.stages;  // pipeline depth, chosen by the launcher to fit shared memory
  // FP8 column scales of the current tile, 128 per epilogue warp
  float* col_scale = reinterpret_cast<float*>(smem + nst * kSB);
  uint64_t* full = reinterpret_cast<uint64_t*>(col_scale + (kFp8 ? kEpiWarps * (kBN / 2) : 0));
  uint64_t* empty = full + nst;
  uint64_t* tfull = empty + nst;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* xbar = drain + 1;  // leader: the peer's count of loaded stages has arrived
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xbar + 1);
  uint32_t* abort_flag = tmem_slot + 1;
  uint32_t* peer_issued = abort_flag + 1;              // leader: stages the peer loaded
  int* offs = reinterpret_cast<int*>(peer_issued + 1);  // [E+1]
  int* pm_prefix = offs + (p.E + 1);                    // [E+1]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = p.E;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;

  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == 2 && lane == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 2 * kEpiWarps * 32);  // both CTAs' epilogue threads
    }
    mbar_init(drain, 1);
    mbar_init(xbar, 1);
    *abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp == 3 && lane == 0) {
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
  }
  // the prologue above touches no global memory; the segment offsets and
  // everything after may come from the previous kernel on the stream
  grid_dependency_wait();
  grid_launch_dependents();
  for (int i = tid; i <= E; i += kThreads) {
    const int v = p.offsets[i];
    offs[i] = v < 0 ? 0 : (v > p.rows ? p.rows : v);  // rows outside the buffer are never written
  }
  __syncthreads();
  if (tid == 0)
    for (int i = 1; i <= E; ++i) offs[i] = offs[i] < offs[i - 1] ? offs[i - 1] : offs[i];
  __syncthreads();
  if (warp == 0) {
    // pair m-tiles per expert (ceil of half its 128-row m-tiles), prefix
    int carry = 0;
    for (int b = 0; b < E; b += 32) {
      const int e = b + lane;
      const int mt = e < E ? (offs[e + 1] - offs[e] + kBM - 1) / kBM : 0;
      const int pm = (mt + 1) >> 1;
      int incl = pm;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      if (e < E) pm_prefix[e] = carry + incl - pm;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) pm_prefix[E] = carry;
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // barrier initialisation visible to the peer before any remote use
  tc_fence_after();

  const uint32_t tmem_base = *tmem_slot;
  const int total_pm = pm_prefix[E];
  const int n_tiles_n = (p.N + kBN - 1) / kBN;
  const int a_row_bytes = p.K * (kFp8 ? 1 : 2);
  const int total = total_pm * n_tiles_n;
  // stages per tile; a partial last stage reads zeros past K (A and B are
  // bounded by K in their tensor maps)
  const int nk = (p.K + kKE * kKBS - 1) / (kKE * kKBS);
  const WaitCtl wc{abort_flag, p.dev_status, p.timeout_ns};
  // A wait that gives up stops the peer CTA too: its waits see the raised
  // flag within a few polls, so the pair aborts together.
  const uint32_t peer_abort = mapa_shared(smem_u32(abort_flag), rank ^ 1u);
  auto pair_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (mbar_wait(bar, parity, wc)) return true;
    st_u32_cluster(peer_abort, 1u);
    return false;
  };

  if (warp == 0) {
    // lanes 1-31 leave at once unless they gather (they must not fall
    // through to the epilogue branch below)
    if (kGather || lane == 0) {
      // ------------------------------------------------------ TMA producer ----
      // lane 0 waits, arms the barrier and loads B (and A when not gathered);
      // with kGather every lane of the warp also gathers four A rows
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool aborted = false;
      const uint64_t pol_a = l2_policy_evict_last();
      for (int L = cluster; L < total && !aborted; L += n_clusters) {
        const PairTile c = decode_pair(L, pm_prefix, offs, E, total_pm, n_tiles_n, rank, a_row_bytes);
        // A last n-tile of at most 128 columns runs as an N = 128 UMMA, each
        // CTA holding 64 of its columns (the loads stay the same size: the
        // extra columns are read and never used).
        const bool half_n = p.N - c.n0 <= kBN / 2;
        const int b_col = c.n0 + static_cast<int>(rank) * (half_n ? kBN / 4 : kBN / 2);
        int gr[4] = {0, 0, 0, 0};
        if constexpr (kGather) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int r = c.row0 + 4 * lane + q;
            int t = r < c.row_end ? p.a_rows[r] : 0;  // rows past the segment: any valid row
            gr[q] = t < 0 ? 0 : (t >= p.a_src_rows ? p.a_src_rows - 1 : t);
          }
        }
        for (int kb = 0; kb < nk; ++kb) {
          bool ok = true;
          if (lane == 0) ok = pair_wait(&empty[stage], phase ^ 1u);
          if constexpr (kGather) ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          if (!ok) {
            aborted = true;
            break;
          }
          const uint32_t bar = mapa_shared(smem_u32(&full[stage]), 0);
          uint8_t* sa = smem + stage * kSB;
          uint8_t* sb = sa + kKBS * kABytes;
          if (lane == 0) {
            if (leader) mbar_arrive_expect_tx(&full[stage], 2 * kSB);
            // A rows are reused by every n-tile of the group: keep them in L2
            if constexpr (kFp8) {
              // A e4m3 [rows, K] and B^T [E*N, K] (this CTA's 128 output
              // columns as K-major rows): one box per k-block, a k-block
              // past K read as zeros
              for (int r = 0; r < kKBS; ++r) {
                const int k0 = (kb * kKBS + r) * kKE;
                tma_load_2d_pair_hint(sa + r * kABytes, &tm_a, bar, k0, c.row0, pol_a);
                tma_load_2d_pair(sb + r * kBBytes, &tm_b, bar, k0, c.e * p.N + b_col);
              }
            } else if constexpr (!kGather) {
              // A: {64 k, 128 rows, kKBS k-blocks}
              tma_load_3d_pair_hint(sa, &tm_a, bar, 0, c.row0, kb * kKBS, pol_a);
            }
            if constexpr (!kFp8) {
              // B [E][K][N]: this CTA's two 64-column blocks x 64*kKBS k-rows
              // of expert e in one copy (a copy's cost is mostly per
              // instruction: three per stage held the shared-memory fill
              // rate to ~55 B per SM clock)
              tma_load_4d_pair(sb, &tm_b, bar, 0, kb * kKBS * kBlockK, b_col / 64, c.e);
            }
          }
          if constexpr (kGather)
            tma_gather4_pair(sa + 512 * lane, &tm_a, bar, kb * kKE, gr[0], gr[1], gr[2], gr[3]);
          ++issued;
          if (++stage == nst) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Every load either CTA issued lands before either CTA can exit (the
      // kernel ends with a cluster barrier, which the leader reaches only
      // after this drain). Both CTAs' loads count their bytes on the
      // leader's barriers, and after an abort the leader may not have armed
      // a stage the peer loaded into, or armed one the peer never loaded:
      // so the peer reports how many stages it loaded, and the leader makes
      // the accounting of each stage still in flight whole before waiting
      // for it. Stages more than a ring behind the last one issued were
      // consumed by the UMMA, so they have landed.
      if constexpr (kGather) __syncwarp();
      if (lane == 0) {
        if (!leader) {
          st_async_u32_cluster(mapa_shared(smem_u32(peer_issued), 0),
                               static_cast<uint32_t>(issued), mapa_shared(smem_u32(xbar), 0));
        } else {
          mbar_arrive_expect_tx(xbar, 4);
          int theirs = issued;
          if (mbar_wait_drain(xbar, 0, p.timeout_ns + kDrainLimitNs)) {
            // the peer cannot load more than a ring ahead of what this CTA armed
            theirs = min(static_cast<int>(*reinterpret_cast<volatile uint32_t*>(peer_issued)),
                         issued + nst);
          } else {
            atomicOr(p.dev_status, MOE_DEV_TIMEOUT);
          }
          const int hi = max(issued, theirs);
          for (int i = max(0, hi - nst); i < hi; ++i) {
            uint64_t* b = &full[i % nst];
            if (i >= issued)
              mbar_arrive_expect_tx(b, kSB);  // armed here for the peer's half alone
            else if (i >= theirs)
              mbar_complete_tx(b, kSB);       // the peer's half will never come
            mbar_wait_drain(b, static_cast<uint32_t>(i / nst) & 1u, kDrainLimitNs);
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------- UMMA issuer (leader) ----
      const uint32_t idesc_full =
          kFp8 ? idesc_e4m3_f32(2 * kBM, kBN) : idesc_bf16_f32(2 * kBM, kBN, false, true);
      const uint32_t idesc_half = kFp8 ? idesc_e4m3_f32(2 * kBM, kBN / 2)
                                       : idesc_bf16_f32(2 * kBM, kBN / 2, false, true);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool aborted = false;
      for (int L = cluster; L < total && !aborted; L += n_clusters) {
        if (!pair_wait(&tempty[acc], acc_phase ^ 1u)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
        const int nt = pair_tile_nt(L, E, total_pm, n_tiles_n, a_row_bytes);
        const uint32_t idesc = p.N - nt * kBN <= kBN / 2 ? idesc_half : idesc_full;
        for (int kb = 0; kb < nk; ++kb) {
          if (!pair_wait(&full[stage], phase)) {
            aborted = true;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * kSB);
          const uint32_t b_addr = a_addr + kKBS * kABytes;
#pragma unroll
          for (int r = 0; r < kKBS; ++r) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              // A: K-major 128-byte rows, k-block r at r * 16 KB; one UMMA K
              // step (16 bf16 or 32 e4m3) is 32 bytes.
              const uint64_t ad = smem_desc_sw128(a_addr + kABytes * r + 32u * kk, 16u, 1024u);
              const uint32_t acc_in = (kb | r | kk) != 0 ? 1u : 0u;
              if constexpr (kFp8) {
                // B: K-major like A
                const uint64_t bd = smem_desc_sw128(b_addr + kBBytes * r + 32u * kk, 16u, 1024u);
                umma_f8_pair(d_tmem, ad, bd, idesc, acc_in);
              } else {
                // B: MN-major, one 128-byte row per k (16-row K step = 2 KB,
                // k-block r at r * 8 KB), this CTA's two 64-column blocks
                // kKBS * 8 KB apart.
                const uint64_t bd = smem_desc_sw128(b_addr + 8192u * r + 2048u * kk,
                                                    kKBS * 64u * kBlockK * 2, 1024u);
                umma_bf16_pair(d_tmem, ad, bd, idesc, acc_in);
              }
            }
          }
          umma_commit_pair_multicast(&empty[stage], 0x3);
          if (++stage == nst) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (aborted) break;
        umma_commit_pair_multicast(&tfull[acc], 0x3);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // every UMMA issued must finish before TMEM is released
      umma_commit_pair(drain);
      mbar_wait_drain(drain, 0, kDrainLimitNs);
    }
  } else {
    // ------------------------------------------------------ epilogue ----
    // warp w reads TMEM lane quadrant w % 4 (the only one it may access) and
    // columns [128*half, 128*half + 128) of the accumulator
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    float* wscale = col_scale + (warp - 2) * (kBN / 2);
    const uint32_t tempty_leader[2] = {mapa_shared(smem_u32(&tempty[0]), 0),
                                       mapa_shared(smem_u32(&tempty[1]), 0)};
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int L = cluster; L < total; L += n_clusters) {
      const PairTile c = decode_pair(L, pm_prefix, offs, E, total_pm, n_tiles_n, rank, a_row_bytes);
      const int row = c.row0 + 32 * q + lane;
      const bool valid = row < c.row_end;
      const int col0 = c.n0 + half * (kBN / 2);
      // whole 32-column chunks: N is a multiple of 64
      const int n_chunks = col0 >= p.N ? 0 : min(4, (p.N - col0) / 32);
      float rs = 1.f;
      if constexpr (kFp8) {
        // scales are fetched before the accumulator wait, hiding their latency
        __syncwarp();  // the previous tile's reads of wscale are done
        const int col = col0 + 4 * lane;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (col < p.N)
          v = *reinterpret_cast<const float4*>(p.b_scale + static_cast<size_t>(c.e) * p.N + col);
        reinterpret_cast<float4*>(wscale)[lane] = v;
        if (valid) rs = p.a_scale[row];
        __syncwarp();
      }
      if (!pair_wait(&tfull[acc], acc_phase)) break;
      tc_fence_after();
      uint16_t* drow = p.D + static_cast<size_t>(valid ? row : 0) * p.N;
      float row_max = 0.f;  // FP8 mode: max |output| of this row in these columns
      const uint32_t t_base = tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                              static_cast<uint32_t>(acc * kBN + half * (kBN / 2));
      // two register sets: the next chunk's TMEM load overlaps this chunk's math
      uint32_t ra[32], rb[32];
      if constexpr (kQOut) {
        const int n_it = 2 * n_chunks;  // pass 1: block maximum; pass 2: convert
        float bmax = 0.f, inv = 0.f;
        if (n_it > 0) {
          tmem_ld_32x32b_x32(t_base, ra);
          tmem_ld_wait();
        }
#pragma unroll
        for (int it = 0; it < 8; ++it) {
          if (it < n_it) {
            uint32_t(&r)[32] = (it & 1) ? rb : ra;
            uint32_t(&nx)[32] = (it & 1) ? ra : rb;
            const int cc = it < n_chunks ? it : it - n_chunks;
            if (it + 1 < n_it) {
              const int nc = it + 1 < n_chunks ? it + 1 : it + 1 - n_chunks;
              tmem_ld_32x32b_x32(t_base + 32u * nc, nx);
            }
            if (it == n_chunks) inv = bmax > 0.f ? 448.0f / bmax : 0.f;
            if (valid) {
              uint32_t q4[8];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                float v0 = __uint_as_float(r[2 * i]) * rs * wscale[32 * cc + 2 * i];
                float v1 = __uint_as_float(r[2 * i + 1]) * rs * wscale[32 * cc + 2 * i + 1];
                if (p.gelu) {
                  v0 = gelu_tanh_f(v0);
                  v1 = gelu_tanh_f(v1);
                }
                const uint32_t b2 = pack_bf16x2(v0, v1);  // the bf16 outputs
                if (it < n_chunks) {
                  bmax = fmaxf(bmax, fmaxf(fabsf(bf16_lo(b2)), fabsf(bf16_hi(b2))));
                } else {
                  const uint32_t h = __nv_cvt_float2_to_fp8x2(
                      make_float2(bf16_lo(b2) * inv, bf16_hi(b2) * inv), __NV_SATFINITE, __NV_E4M3);
                  if (i & 1) q4[i >> 1] |= h << 16;
                  else q4[i >> 1] = h;
                }
              }
              if (it >= n_chunks) {
                uint4* dst = reinterpret_cast<uint4*>(p.Dq + static_cast<size_t>(row) * p.N + col0 +
                                                      32 * cc);
                st_global_cs_v4(dst, make_uint4(q4[0], q4[1], q4[2], q4[3]));
                st_global_cs_v4(dst + 1, make_uint4(q4[4], q4[5], q4[6], q4[7]));
              }
            }
            if (it + 1 < n_it) tmem_ld_wait();
          }
        }
        if (valid && n_chunks > 0)
          p.d_scale[static_cast<size_t>(row) * ((p.N + 127) / 128) + col0 / 128] = bmax / 448.0f;
      } else {
        if (n_chunks > 0) {
          tmem_ld_32x32b_x32(t_base, ra);
          tmem_ld_wait();
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          if (cc < n_chunks) {
            uint32_t(&r)[32] = (cc & 1) ? rb : ra;
            uint32_t(&nx)[32] = (cc & 1) ? ra : rb;
            if (cc + 1 < n_chunks) tmem_ld_32x32b_x32(t_base + 32u * (cc + 1), nx);
            if (valid) {
              uint32_t packed[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                float v0 = __uint_as_float(r[2 * i]);
                float v1 = __uint_as_float(r[2 * i + 1]);
                if constexpr (kFp8) {
                  v0 = v0 * rs * wscale[32 * cc + 2 * i];
                  v1 = v1 * rs * wscale[32 * cc + 2 * i + 1];
                }
                if (p.gelu) {
                  v0 = gelu_tanh_f(v0);
                  v1 = gelu_tanh_f(v1);
                }
                if constexpr (kFp8) row_max = fmaxf(row_max, fmaxf(fabsf(v0), fabsf(v1)));
                packed[i] = pack_bf16x2(v0, v1);
              }
              // outputs are read once, by the next kernel: stream them past L2
              uint4* dst = reinterpret_cast<uint4*>(drow + col0 + 32 * cc);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                st_global_cs_v4(dst + i, make_uint4(packed[4 * i], packed[4 * i + 1],
                                                    packed[4 * i + 2], packed[4 * i + 3]));
            }
            if (cc + 1 < n_chunks) tmem_ld_wait();
          }
        }
      }
      if constexpr (kFp8 && !kQOut) {
        // bf16 rounding is monotonic, so the rounded maximum is the maximum
        // of the rounded (stored) values
        if (p.row_amax != nullptr && valid && n_chunks > 0)
          atomicMax(p.row_amax + row, __float_as_uint(bf16_lo(pack_bf16x2(row_max, 0.f))));
      }
      tc_fence_before();
      mbar_arrive_cluster(tempty_leader[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the peer may still signal it
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, kTmemCols);
}

}  // namespace

size_t gemm_pair_smem_bytes(int E, int stages, bool fp8, int kb_per_stage) {
  return 1024 + static_cast<size_t>(stages) * kStageBytes * kb_per_stage +
         (fp8 ? 4 * kEpiWarps * (kBN / 2) : 0) +
         8 * (2 * stages + 6) + 16 + 8 * static_cast<size_t>(E + 1);
}

template <bool kFp8, bool kQOut, bool kGather>
cudaError_t launch_pair(const CUtensorMap& tm_a, const CUtensorMap& tm_b, const GemmArgs& a,
                        int num_sms, cudaStream_t st) {
  // the deepest ring that fits: every stage in flight hides TMA latency
  int dev = 0, optin = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (err != cudaSuccess) return err;
  GemmArgs args = a;
  constexpr int kbs = kGather ? 1 : kWideKB;
  args.stages = kMaxStages;
  while (args.stages > 2 &&
         gemm_pair_smem_bytes(a.E, args.stages, kFp8, kbs) > static_cast<size_t>(optin))
    --args.stages;
  const size_t smem = gemm_pair_smem_bytes(a.E, args.stages, kFp8, kbs);
  err = cudaFuncSetAttribute(grouped_gemm_pair_kernel<kFp8, kQOut, kGather>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * (num_sms / 2)), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // may start while the previous kernel on the stream finishes (the kernel
  // waits for it before its first global access)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  err = cudaLaunchKernelEx(&cfg, grouped_gemm_pair_kernel<kFp8, kQOut, kGather>, tm_a, tm_b,
                           args);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

cudaError_t launch_grouped_gemm_pair(const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                                     const GemmArgs& a, int num_sms, cudaStream_t st) {
  if (a.a_rows != nullptr) return launch_pair<false, false, true>(tm_a, tm_b, a, num_sms, st);
  return launch_pair<false, false, false>(tm_a, tm_b, a, num_sms, st);
}

cudaError_t launch_grouped_gemm_pair_fp8(const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                                         const GemmArgs& a, int num_sms, cudaStream_t st) {
  if (a.Dq != nullptr) return launch_pair<true, true, false>(tm_a, tm_b, a, num_sms, st);
  return launch_pair<true, false, false>(tm_a, tm_b, a, num_sms, st);
}

}  // namespace moe
