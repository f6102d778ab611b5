// Grouped GEMM over ragged expert segments on the 5th-generation tensor
// cores: D[r, :] = A[r, :] . B[e(r)] for the rows r of expert e's segment
// [offsets[e], offsets[e+1]), with an optional GELU (tanh form) epilogue.
// This is the expert FFN of the MoE comm bottleneck page, section 5.1 (many
// experts' small GEMMs in one kernel instead of one launch per expert).
//
// Persistent, warp-specialised, one CTA per SM:
//   warp 0      TMA producer: A tile 128 x 64 (K-major, 128-byte swizzle) and
//               B tile 64 x BN (MN-major: weights are [E, K, N] with N
//               contiguous) into a STAGES-deep shared-memory ring;
//   warp 1      one thread issues tcgen05.mma (M=128, N=BN, K=16) into one of
//               two TMEM accumulators and commits stage/accumulator barriers;
//   warps 2-5   epilogue: tcgen05.ld of their TMEM lane quadrant, optional
//               GELU, bf16 rounding, masked stores (rows past the segment
//               end belong to the next expert and are not written).
// Tiles are the (expert m-tile, n-tile) pairs; the m-tile list is rebuilt on
// the device from `offsets`, so no host synchronisation is needed. Every
// tile costs the same (same K), so a static round-robin over CTAs balances
// skewed routing as well as even routing.
#include "moe_internal.h"
#include "moe_ptx.cuh"

namespace moe {

namespace {

constexpr int kBM = 128;
constexpr int kGroupM = 16;  // m-tiles per rasterisation group (L2 reuse)
constexpr int kGemmThreads = 192;

template <int BN>
struct GemmCfg {
  static constexpr uint32_t kABytes = kBM * kBlockK * 2;   // 16 KB
  static constexpr uint32_t kBBytes = BN * kBlockK * 2;    // 32 KB at BN = 256
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = (200 * 1024) / kStageBytes > 6 ? 6 : (200 * 1024) / kStageBytes;
  static constexpr uint32_t kTmemCols = 2 * BN;            // two accumulators
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN");
  static_assert(kTmemCols <= 512, "TMEM");
};

struct TileCoord {
  int e, row0, row_end, n0;
};

__device__ __forceinline__ TileCoord decode_tile(int L, const int* mt_prefix, const int* offs,
                                                 int E, int total_mt, int n_tiles_n, int BN) {
  const int per_group = kGroupM * n_tiles_n;
  const int g = L / per_group;
  const int first_m = g * kGroupM;
  const int gsz = min(kGroupM, total_mt - first_m);
  const int r = L - g * per_group;
  const int m = first_m + r % gsz;
  const int nt = r / gsz;
  // expert owning global m-tile m: largest e with mt_prefix[e] <= m
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (mt_prefix[mid] <= m) lo = mid; else hi = mid - 1;
  }
  TileCoord c;
  c.e = lo;
  c.row0 = offs[lo] + (m - mt_prefix[lo]) * kBM;
  c.row_end = offs[lo + 1];
  c.n0 = nt * BN;
  return c;
}

__device__ __forceinline__ float gelu_tanh_f(float u) {
  // 0.5 u (1 + tanh(z)) = u / (1 + exp(-2 z)),  z = sqrt(2/pi) (u + 0.044715 u^3)
  const float z2 = 1.5957691216057308f * fmaf(0.044715f * u, u * u, u);
  return __fdividef(u, 1.0f + __expf(-z2));
}

template <int BN>
__global__ void __launch_bounds__(kGemmThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tm_a,
                        const __grid_constant__ CUtensorMap tm_b, GemmArgs p) {
  using Cfg = GemmCfg<BN>;
  constexpr int S = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_up_1024(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * Cfg::kStageBytes);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  uint32_t* abort_flag = tmem_slot + 1;
  int* offs = reinterpret_cast<int*>(abort_flag + 2);  // [E+1]
  int* mt_prefix = offs + (p.E + 1);                    // [E+1]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = p.E;

  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 2 && lane == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4 * 32);
    }
    mbar_init(drain, 1);
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
  for (int i = tid; i <= E; i += kGemmThreads) {
    const int v = p.offsets[i];
    offs[i] = v < 0 ? 0 : (v > p.rows ? p.rows : v);  // rows outside the buffer are never written
  }
  __syncthreads();
  if (tid == 0)
    for (int i = 1; i <= E; ++i) offs[i] = offs[i] < offs[i - 1] ? offs[i - 1] : offs[i];
  __syncthreads();
  if (warp == 0) {
    // m-tiles per expert and their exclusive prefix (E <= 256)
    int carry = 0;
    for (int b = 0; b < E; b += 32) {
      const int e = b + lane;
      const int mt = e < E ? (offs[e + 1] - offs[e] + kBM - 1) / kBM : 0;
      int incl = mt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      if (e < E) mt_prefix[e] = carry + incl - mt;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) mt_prefix[E] = carry;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem_base = *tmem_slot;
  const int total_mt = mt_prefix[E];
  const int n_tiles_n = (p.N + BN - 1) / BN;
  const int total = total_mt * n_tiles_n;
  const int nk = p.K / kBlockK;
  const WaitCtl wc{abort_flag, p.dev_status, p.timeout_ns};

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer ----
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool aborted = false;
      for (int L = blockIdx.x; L < total && !aborted; L += gridDim.x) {
        const TileCoord c = decode_tile(L, mt_prefix, offs, E, total_mt, n_tiles_n, BN);
        const int b_row = c.e * p.K;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, wc)) {
            aborted = true;
            break;
          }
          uint8_t* sa = smem + stage * Cfg::kStageBytes;
          uint8_t* sb = sa + Cfg::kABytes;
          mbar_arrive_expect_tx(&full[stage], Cfg::kStageBytes);
          tma_load_2d(sa, &tm_a, &full[stage], kb * kBlockK, c.row0);
#pragma unroll
          for (int cb = 0; cb < BN / 64; ++cb)
            tma_load_2d(sb + cb * (64 * kBlockK * 2), &tm_b, &full[stage], c.n0 + 64 * cb,
                        b_row + kb * kBlockK);
          ++issued;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (aborted) {
        // let the last loads issued land before the CTA exits
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
      const uint32_t idesc = idesc_bf16_f32(kBM, BN, false, true);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool aborted = false;
      for (int L = blockIdx.x; L < total && !aborted; L += gridDim.x) {
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, wc)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&full[stage], phase, wc)) {
            aborted = true;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * Cfg::kStageBytes);
          const uint32_t b_addr = a_addr + Cfg::kABytes;
#pragma unroll
          for (int kk = 0; kk < kBlockK / 16; ++kk) {
            // A: K-major rows of 128 B; a 16-element K step is 32 bytes.
            const uint64_t ad = smem_desc_sw128(a_addr + 32u * kk, 16u, 1024u);
            // B: MN-major, one 128-byte row per k; a 16-row K step is 2 KB;
            // 64-column blocks are 64 rows x 128 B = 8 KB apart.
            const uint64_t bd = smem_desc_sw128(b_addr + 2048u * kk, 64u * kBlockK * 2, 1024u);
            umma_bf16(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
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
      // every UMMA issued must finish before TMEM is released
      umma_commit(drain);
      mbar_wait_drain(drain, 0, kDrainLimitNs);
    }
  } else {
    // ------------------------------------------------------ epilogue ----
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int L = blockIdx.x; L < total; L += gridDim.x) {
      const TileCoord c = decode_tile(L, mt_prefix, offs, E, total_mt, n_tiles_n, BN);
      if (!mbar_wait(&tfull[acc], acc_phase, wc)) break;
      tc_fence_after();
      const int row = c.row0 + 32 * q + lane;
      const bool valid = row < c.row_end;
      uint16_t* drow = p.D + static_cast<size_t>(valid ? row : 0) * p.N;
      const uint32_t t_base =
          tmem_base + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(acc * BN);
#pragma unroll 1
      for (int cc = 0; cc < BN / 32; ++cc) {
        const int col = c.n0 + 32 * cc;
        if (col >= p.N) break;  // N is a multiple of 64: whole chunks
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_base + 32u * cc, r);
        tmem_ld_wait();
        if (valid) {
          uint32_t packed[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float v0 = __uint_as_float(r[2 * i]);
            float v1 = __uint_as_float(r[2 * i + 1]);
            if (p.gelu) {
              v0 = gelu_tanh_f(v0);
              v1 = gelu_tanh_f(v1);
            }
            packed[i] = pack_bf16x2(v0, v1);
          }
          uint4* dst = reinterpret_cast<uint4*>(drow + col);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
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
  if (warp == 1) tmem_dealloc(tmem_base, Cfg::kTmemCols);
}

constexpr int kBN = 256;

}  // namespace

size_t gemm_smem_bytes(int E) {
  using Cfg = GemmCfg<kBN>;
  return 1024 + static_cast<size_t>(Cfg::kStages) * Cfg::kStageBytes + 8 * (2 * Cfg::kStages + 5) + 16 +
         8 * static_cast<size_t>(E + 1);
}

cudaError_t launch_grouped_gemm(const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                                const GemmArgs& a, int num_sms, cudaStream_t st) {
  const size_t smem = gemm_smem_bytes(a.E);
  cudaError_t err = cudaFuncSetAttribute(grouped_gemm_kernel<kBN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  return launch_pdl(grouped_gemm_kernel<kBN>, dim3(num_sms), dim3(kGemmThreads), smem, st, tm_a,
                    tm_b, a);
}

}  // namespace moe
