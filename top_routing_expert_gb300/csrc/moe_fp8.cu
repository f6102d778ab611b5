// FP8 (e4m3) support for the dispatch and the expert FFN (MoE comm
// bottleneck, section 5.3: FP8 hidden states halve the dispatch bytes; the
// expert GEMM then runs on the FP8 tensor-core path).
//
// Scaling: one fp32 scale per token row for activations and per output
// column for weights. For a row (or column) with largest magnitude amax,
//   inv = 448 / amax, q = e4m3_rn_satfinite(v * inv), scale = amax / 448,
// every operation in fp32; a zero row has q = 0 and scale = 0. A value is
// then q * scale, and a GEMM of two quantised operands is the fp32
// accumulation of q products times the row scale times the column scale.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "moe_internal.h"
#include "moe_ptx.cuh"

namespace moe {

namespace {

constexpr float kE4M3Max = 448.0f;

__device__ __forceinline__ uint32_t fp8x4(float a, float b, float c, float d) {
  const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// 8 bf16 (one uint4) scaled and converted to 8 e4m3 bytes (one uint2).
__device__ __forceinline__ uint2 quant8(const uint4 v, float inv) {
  uint2 o;
  o.x = fp8x4(bf16_lo(v.x) * inv, bf16_hi(v.x) * inv, bf16_lo(v.y) * inv, bf16_hi(v.y) * inv);
  o.y = fp8x4(bf16_lo(v.z) * inv, bf16_hi(v.z) * inv, bf16_lo(v.w) * inv, bf16_hi(v.w) * inv);
  return o;
}

__device__ __forceinline__ float amax8(const uint4 v) {
  float m = fabsf(bf16_lo(v.x));
  m = fmaxf(m, fabsf(bf16_hi(v.x)));
  m = fmaxf(m, fabsf(bf16_lo(v.y)));
  m = fmaxf(m, fabsf(bf16_hi(v.y)));
  m = fmaxf(m, fabsf(bf16_lo(v.z)));
  m = fmaxf(m, fabsf(bf16_hi(v.z)));
  m = fmaxf(m, fabsf(bf16_lo(v.w)));
  m = fmaxf(m, fabsf(bf16_hi(v.w)));
  return m;
}

// A read-once load that does not displace L2 lines others reuse.
__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.cs.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ---------------------------------------------------------- weights ----

// Pass 1: per-column magnitude maxima of W [E, K, N] (N contiguous) as fp32
// bits in amax [E, N] (zeroed by the caller); blocks cover (expert, 256
// columns, a K range) and combine with atomicMax on the non-negative bits.
__global__ void weight_amax_kernel(const uint16_t* __restrict__ W, uint32_t* __restrict__ amax,
                                   int K, int N, int k_chunk) {
  const int e = blockIdx.z;
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  const int k0 = blockIdx.y * k_chunk;
  const int k1 = min(K, k0 + k_chunk);
  if (n >= N) return;
  const uint16_t* w = W + (static_cast<size_t>(e) * K) * N + n;
  float m = 0.f;
  for (int k = k0; k < k1; ++k) m = fmaxf(m, fabsf(__uint_as_float(static_cast<uint32_t>(w[static_cast<size_t>(k) * N]) << 16)));
  atomicMax(&amax[static_cast<size_t>(e) * N + n], __float_as_uint(m));
}

// Pass 2: quantise and transpose through a 64 x 64 shared tile: Wq [E, N, K]
// (each output column a row, contiguous over K). Reads are 128-byte rows of
// W; each thread then converts 16 consecutive k of one column and writes
// them as one 16-byte vector.
__global__ void __launch_bounds__(256) weight_quant_kernel(const uint16_t* __restrict__ W,
                                                           const uint32_t* __restrict__ amax,
                                                           uint8_t* __restrict__ Wq, int K,
                                                           int N) {
  __shared__ float tile[64][65];
  const int e = blockIdx.z;
  const int n0 = blockIdx.x * 64, k0 = blockIdx.y * 64;
  const int tid = threadIdx.x;
  // load: 64 rows (k) x 64 columns (n); thread = (row tid / 4, 16 columns as
  // two 16-byte vectors). K and N are multiples of 64 (checked by the host).
  {
    const int r = tid >> 2, cq = (tid & 3) * 16;
    const uint4* src = reinterpret_cast<const uint4*>(
        W + (static_cast<size_t>(e) * K + k0 + r) * N + n0 + cq);
    const uint4 a = __ldg(src), b = __ldg(src + 1);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      tile[r][cq + 2 * i] = bf16_lo(w[i]);
      tile[r][cq + 2 * i + 1] = bf16_hi(w[i]);
    }
  }
  __syncthreads();
  // store: column n = tid / 4, k range (tid % 4) * 16 .. +16
  const int c = tid >> 2, kq = (tid & 3) * 16;
  const int n = n0 + c;
  const float am = __uint_as_float(amax[static_cast<size_t>(e) * N + n]);
  const float inv = am > 0.f ? kE4M3Max / am : 0.f;
  uint32_t w4[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    w4[j] = fp8x4(tile[kq + 4 * j][c] * inv, tile[kq + 4 * j + 1][c] * inv,
                  tile[kq + 4 * j + 2][c] * inv, tile[kq + 4 * j + 3][c] * inv);
  *reinterpret_cast<uint4*>(Wq + (static_cast<size_t>(e) * N + n) * K + k0 + kq) =
      make_uint4(w4[0], w4[1], w4[2], w4[3]);
}

// Pass 3: the maxima become the dequantisation scales, in place.
__global__ void weight_scale_kernel(float* __restrict__ s, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) s[i] = s[i] / kE4M3Max;
}

// ------------------------------------------------------------- rows ----

// One warp per row r < offsets[E] (the kept rows, known on the device):
// bf16 [rows, K] -> e4m3 [rows, K] and a scale per row, the row maxima
// given (fp32 bits, from the producing GEMM's epilogue).
__global__ void __launch_bounds__(256) row_quant_kernel(const uint16_t* __restrict__ src,
                                                        const uint32_t* __restrict__ amax,
                                                        uint8_t* __restrict__ dst,
                                                        float* __restrict__ scale,
                                                        const int32_t* __restrict__ offsets,
                                                        int E, int rows, int K) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  int n = offsets[E];
  n = n < 0 ? 0 : (n > rows ? rows : n);
  const int nvec = K >> 3;
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < n; r += warps) {
    const uint4* s = reinterpret_cast<const uint4*>(src + static_cast<size_t>(r) * K);
    const float m = __uint_as_float(amax[r]);
    const float inv = m > 0.f ? kE4M3Max / m : 0.f;
    uint2* d = reinterpret_cast<uint2*>(dst + static_cast<size_t>(r) * K);
    for (int i = lane; i < nvec; i += 32) d[i] = quant8(ldg_stream(s + i), inv);
    if (lane == 0) scale[r] = m / kE4M3Max;
  }
}

// ---------------------------------------------------------- dispatch ----

// The FP8 dispatch: one warp per token; the token row is quantised once
// (scale from its own maximum) and the e4m3 row is written to each kept
// destination, with the scale. Destinations as in the bf16 gather.
__global__ void __launch_bounds__(256) gather_fp8_kernel(GatherArgs a, uint8_t* __restrict__ xq,
                                                         float* __restrict__ xs) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int nvec = a.H >> 3;
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
      if (j >= a.k) d[j] = -1;
      any |= d[j] >= 0;
    }
    if (!any) continue;
    const uint4* src = reinterpret_cast<const uint4*>(a.x) + static_cast<size_t>(t) * nvec;
    // both passes keep kGatherU 16-byte loads per lane in flight (the second
    // pass re-reads the row from cache)
    constexpr int kGatherU = 4;
    float m = 0.f;
    for (int b = 0; b < nvec; b += 32 * kGatherU) {
      uint4 v[kGatherU];
#pragma unroll
      for (int u = 0; u < kGatherU; ++u) {
        const int i = b + 32 * u + lane;
        v[u] = i < nvec ? __ldg(src + i) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kGatherU; ++u) m = fmaxf(m, amax8(v[u]));
    }
    m = warp_max(m);
    const float inv = m > 0.f ? kE4M3Max / m : 0.f;
    for (int b = 0; b < nvec; b += 32 * kGatherU) {
      uint4 v[kGatherU];
#pragma unroll
      for (int u = 0; u < kGatherU; ++u) {
        const int i = b + 32 * u + lane;
        if (i < nvec) v[u] = __ldg(src + i);
      }
#pragma unroll
      for (int u = 0; u < kGatherU; ++u) {
        const int i = b + 32 * u + lane;
        if (i < nvec) {
          const uint2 q = quant8(v[u], inv);
#pragma unroll
          for (int j = 0; j < kMaxTopK; ++j)
            if (d[j] >= 0) reinterpret_cast<uint2*>(xq + static_cast<size_t>(d[j]) * a.H)[i] = q;
        }
      }
    }
    if (lane < a.k && dest >= 0) xs[dest] = m / kE4M3Max;
  }
}

// ----------------------------------------------------------- combine ----

// 16 e4m3 values (one uint4) -> fp32, through the exact e4m3 -> f16 convert.
__device__ __forceinline__ void e4m3x16_to_f32(const uint4 v, float (&f)[16]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(
          static_cast<__nv_fp8x2_storage_t>((w[q] >> (16 * h)) & 0xFFFFu), __NV_E4M3);
      const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&r));
      f[4 * q + 2 * h] = t.x;
      f[4 * q + 2 * h + 1] = t.y;
    }
  }
}

// The FP8 combine: y[t] = bf16(sum over kept slots, ascending j, of w[t,j] *
// q[dest, c] * scale[dest, c / 128]); one warp per token, 16 columns per
// lane and vector, every slot's loads issued before any is used.
template <int KMAX, int U>
__global__ void __launch_bounds__(256, 2) combine_fp8_kernel(CombineArgs a,
                                                             const uint8_t* __restrict__ y_q,
                                                             const float* __restrict__ y_scale) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int nvec = a.H >> 4;
  const int nblk = (a.H + 127) >> 7;
  const uint4* __restrict__ yv = reinterpret_cast<const uint4*>(y_q);
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
      float sc[KMAX][U];
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int i = b + 32 * u + lane;
          const bool ok = d[j] >= 0 && i < nvec;
          v[j][u] = ok ? __ldg(yv + static_cast<size_t>(d[j]) * nvec + i) : make_uint4(0, 0, 0, 0);
          sc[j][u] = ok ? __ldg(y_scale + static_cast<size_t>(d[j]) * nblk + (i >> 3)) : 0.f;
        }
      float acc[U][16];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int q = 0; q < 16; ++q) acc[u][q] = 0.f;
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (d[j] >= 0) {
#pragma unroll
          for (int u = 0; u < U; ++u) {
            float f[16];
            e4m3x16_to_f32(v[j][u], f);
#pragma unroll
            for (int q = 0; q < 16; ++q) acc[u][q] = fmaf(w[j], f[q] * sc[j][u], acc[u][q]);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = b + 32 * u + lane;
        if (i < nvec) {
          uint4 o0, o1;
          o0.x = pack_bf16x2(acc[u][0], acc[u][1]);
          o0.y = pack_bf16x2(acc[u][2], acc[u][3]);
          o0.z = pack_bf16x2(acc[u][4], acc[u][5]);
          o0.w = pack_bf16x2(acc[u][6], acc[u][7]);
          o1.x = pack_bf16x2(acc[u][8], acc[u][9]);
          o1.y = pack_bf16x2(acc[u][10], acc[u][11]);
          o1.z = pack_bf16x2(acc[u][12], acc[u][13]);
          o1.w = pack_bf16x2(acc[u][14], acc[u][15]);
          uint4* dst = ov + static_cast<size_t>(t) * (a.H >> 3) + 2 * i;
          dst[0] = o0;
          dst[1] = o1;
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_combine_fp8(const CombineArgs& a, const uint8_t* y_q, const float* y_scale,
                               int num_sms, cudaStream_t st) {
  if (a.T == 0) return cudaSuccess;
  int grid = (a.T + 7) / 8;
  if (grid > num_sms * 8) grid = num_sms * 8;
  if (a.k <= 2) return launch_pdl(combine_fp8_kernel<2, 3>, dim3(grid), dim3(256), 0, st, a, y_q, y_scale);
  if (a.k <= 4) return launch_pdl(combine_fp8_kernel<4, 1>, dim3(grid), dim3(256), 0, st, a, y_q, y_scale);
  if (a.k <= 6) return launch_pdl(combine_fp8_kernel<6, 1>, dim3(grid), dim3(256), 0, st, a, y_q, y_scale);
  return launch_pdl(combine_fp8_kernel<8, 1>, dim3(grid), dim3(256), 0, st, a, y_q, y_scale);
}

cudaError_t launch_quantize_weights(const uint16_t* W, uint8_t* Wq, float* Ws, int E, int K,
                                    int N, cudaStream_t st) {
  uint32_t* amax = reinterpret_cast<uint32_t*>(Ws);
  cudaError_t err = cudaMemsetAsync(amax, 0, sizeof(uint32_t) * static_cast<size_t>(E) * N, st);
  if (err != cudaSuccess) return err;
  const int k_chunk = 256;
  dim3 g1((N + 255) / 256, (K + k_chunk - 1) / k_chunk, E);
  weight_amax_kernel<<<g1, 256, 0, st>>>(W, amax, K, N, k_chunk);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  dim3 g2((N + 63) / 64, (K + 63) / 64, E);
  weight_quant_kernel<<<g2, 256, 0, st>>>(W, amax, Wq, K, N);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  const int n = E * N;
  weight_scale_kernel<<<(n + 255) / 256, 256, 0, st>>>(Ws, n);
  return cudaGetLastError();
}

cudaError_t launch_row_quant(const uint16_t* src, const uint32_t* amax, uint8_t* dst,
                             float* scale, const int32_t* offsets, int E, int rows, int K,
                             int num_sms, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  int grid = (rows + 7) / 8;
  if (grid > num_sms * 8) grid = num_sms * 8;
  return launch_pdl(row_quant_kernel, dim3(grid), dim3(256), 0, st, src, amax, dst, scale, offsets,
                    E, rows, K);
}

cudaError_t launch_gather_fp8(const GatherArgs& a, uint8_t* xq, float* xs, int num_sms,
                              cudaStream_t st) {
  if (a.T == 0) return cudaSuccess;
  int grid = (a.T + 7) / 8;
  if (grid > num_sms * 8) grid = num_sms * 8;
  return launch_pdl(gather_fp8_kernel, dim3(grid), dim3(256), 0, st, a, xq, xs);
}

}  // namespace moe
