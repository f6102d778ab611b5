// moe_permute_noalloc: the dispatch permutation without a caller workspace.
//
// Some callers cannot hand this library a device buffer: a plugin run by an
// inference runtime that owns every byte of device memory and offers no
// allocation hook, or code that must not allocate because it runs while a
// CUDA stream is being captured into a graph or from a real-time path where
// a cudaMalloc could block. For them this variant keeps its scratch (tile
// histograms, tile bases, in-tile ranks, a ticket and a status word) in one
// fixed device array that the library itself defines, so the caller passes
// only inputs and outputs.
//
// Costs and rules of that choice:
//   - The array is kStaticScratchBytes (1 MiB) per GPU that loads the
//     library, held until the process exits.
//   - Shapes whose scratch does not fit are rejected with
//     MOE_ERR_UNSUPPORTED before anything is launched.
//   - The first call in a CUDA context looks up the array's device address
//     (once per device and context: a context torn down and made again, as
//     by cudaDeviceReset, reloads the library's module and moves the array,
//     so the address is looked up again); make that first call before any
//     stream capture.
//   - Every call on a device shares the one array and leaves its contents
//     behind. What must start at zero (the scan ticket) is cleared by the
//     call's own first kernel; calls that overlap on the GPU (two streams,
//     or two host threads without ordering) race on the array and must be
//     serialised by the caller.
#include <mutex>

#include "moe_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(1) << 20;

// The static scratch. In host code this name is a host-side stand-in, not a
// device address: host code must use the address from
// cudaGetSymbolAddress (see scratch_for_current_device) and never pass the
// name itself to a kernel.
static __device__ __align__(256) unsigned char g_dispatch_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Process-unique id of the current CUDA context (0 if there is none yet),
// through the driver entry points the runtime hands out. false if the
// driver offers no context ids.
bool current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (get_current == nullptr || get_id == nullptr) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return false;
  *id = 0;
  return ctx == nullptr || get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_dispatch_scratch in the current device's current
// context, looked up with that device current the first time a context is
// seen and again whenever the device's context has changed (a reset context
// holds a new copy of the array). nullptr on failure.
unsigned char* scratch_for_current_device() {
  static std::mutex mu;
  static unsigned char* addr[kMaxDevices] = {nullptr};
  static unsigned long long ctx_of[kMaxDevices] = {0};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  unsigned long long id = 0;
  if (!current_context_id(&id)) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr || id == 0 || ctx_of[dev] != id) {
    void* p = nullptr;
    // makes the device's primary context current if nothing has yet
    if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess) return nullptr;
    if (!current_context_id(&id) || id == 0) return nullptr;
    addr[dev] = static_cast<unsigned char*>(p);
    ctx_of[dev] = id;
  }
  return addr[dev];
}

size_t round256(size_t b) { return (b + 255) & ~size_t(255); }

}  // namespace

extern "C" moe_status moe_permute_noalloc(const moe_shape* s, const moe_bf16* x,
                                          const int32_t* topk_idx, int32_t* kept_counts,
                                          int32_t* offsets, int32_t* dest_row,
                                          int32_t* src_token, moe_bf16* x_perm,
                                          uint32_t* dev_status, void* stream) {
  using namespace moe;
  if (s == nullptr) return MOE_ERR_NULL;
  size_t unused = 0;
  const moe_status shape_ok = moe_workspace_size(s, &unused);  // the same shape checks
  if (shape_ok != MOE_OK) return shape_ok;
  // as moe_permute: x_perm may be NULL when src_token is given (the
  // permutation only)
  if (x == nullptr || topk_idx == nullptr || offsets == nullptr || dest_row == nullptr ||
      (x_perm == nullptr && src_token == nullptr))
    return MOE_ERR_NULL;
  const void* ptrs[] = {x, topk_idx, kept_counts, offsets, dest_row, src_token, x_perm, dev_status};
  for (const void* p : ptrs)
    if ((reinterpret_cast<uintptr_t>(p) & 15u) != 0) return MOE_ERR_ALIGN;

  const int T = static_cast<int>(s->T), H = static_cast<int>(s->H), E = static_cast<int>(s->E),
            k = static_cast<int>(s->top_k);
  const int n_tiles = (T + kTileTokens - 1) / kTileTokens;
  const size_t tiles_bytes = round256(static_cast<size_t>(E) * n_tiles * 4);
  // tile counts and tile bases, in-tile ranks, routed counts and P, the
  // scan ticket and a status word (the same pieces `take` carves below)
  const size_t need = 2 * tiles_bytes + round256(static_cast<size_t>(T) * k) +
                      2 * round256(static_cast<size_t>(E) * 4) + 2 * 256;
  if (need > kStaticScratchBytes) return MOE_ERR_UNSUPPORTED;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (T == 0) {
    if (cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), st) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (kept_counts && cudaMemsetAsync(kept_counts, 0, sizeof(int32_t) * E, st) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  }
  unsigned char* base = scratch_for_current_device();
  if (base == nullptr) return MOE_ERR_CUDA;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    unsigned char* p = base + off;
    off += round256(bytes);
    return p;
  };
  int32_t* tile_cnt = reinterpret_cast<int32_t*>(take(static_cast<size_t>(E) * n_tiles * 4));
  int32_t* tile_base = reinterpret_cast<int32_t*>(take(static_cast<size_t>(E) * n_tiles * 4));
  uint8_t* rank8 = take(static_cast<size_t>(T) * k);
  int32_t* routed = reinterpret_cast<int32_t*>(take(static_cast<size_t>(E) * 4));
  float* P = reinterpret_cast<float*>(take(static_cast<size_t>(E) * 4));
  uint32_t* ticket = reinterpret_cast<uint32_t*>(take(4));
  uint32_t* status_slot = reinterpret_cast<uint32_t*>(take(4));
  uint32_t* status = dev_status ? dev_status : status_slot;

  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MOE_ERR_CUDA;

  RankArgs r;
  r.T = T;
  r.E = E;
  r.k = k;
  r.n_tiles = n_tiles;
  r.topk_idx = topk_idx;
  r.tile_cnt = tile_cnt;
  r.rank8 = rank8;
  r.ticket = ticket;  // the rank kernel's block 0 clears it for the scan
  r.dev_status = status;
  if (launch_rank(r, st) != cudaSuccess) return MOE_ERR_CUDA;

  ScanArgs sc;
  sc.T = T;
  sc.E = E;
  sc.k = k;
  sc.n_tiles = n_tiles;
  sc.C = moe_capacity(s->T, s->E, s->top_k, s->capacity_factor);
  sc.tile_cnt = tile_cnt;
  sc.tile_base = tile_base;
  sc.ppart = nullptr;
  sc.routed = routed;
  sc.P = P;
  sc.aux = nullptr;
  sc.kept = kept_counts;
  sc.offsets = offsets;
  sc.ticket = ticket;
  if (launch_scan(sc, st) != cudaSuccess) return MOE_ERR_CUDA;

  GatherArgs g;
  g.T = T;
  g.H = H;
  g.E = E;
  g.k = k;
  g.n_tiles = n_tiles;
  g.C = sc.C;
  g.x = x;
  g.topk_idx = topk_idx;
  g.rank8 = rank8;
  g.tile_base = tile_base;
  g.offsets = offsets;
  g.dest_row = dest_row;
  g.src_token = src_token;
  g.x_perm = x_perm;
  g.dev_status = status;
  if (launch_gather(g, sms, st) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}
