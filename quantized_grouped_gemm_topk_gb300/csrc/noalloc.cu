// Router logits without a caller workspace.
//
// moe_router_logits needs scratch memory for the per-slice partial sums of
// its split reduction over H, and takes it from the workspace the caller
// allocated. Some callers cannot allocate device memory at the point where
// they need logits: code that runs inside an allocator-free region (a
// custom memory pool that must not grow, a plugin host that hands out no
// device buffers, a real-time path where cudaMalloc's implicit device
// synchronisation is not allowed). For them this file keeps the partials in
// one static device array that exists from library load to process exit on
// every GPU that loads the library.
//
// Rules of the shared array:
//   * it holds kNoAllocScratchFloats floats (4 MiB); a call whose partials
//     would not fit returns MOE_ERR_WORKSPACE and enqueues nothing;
//   * every call on a device uses the same array and leaves its partials in
//     it; each call overwrites every partial it later reads, so nothing has
//     to be zeroed between calls;
//   * two calls whose kernels may overlap on the GPU (different streams with
//     no ordering between them, or several host threads) race on the array:
//     serialise them;
//   * the array's device address is looked up (cudaGetSymbolAddress) the
//     first time a call is made in a given CUDA context and cached under
//     that context's unique id (cuCtxGetId): the device's primary context,
//     a context the caller created, or one converted from a green context
//     each hold their own copy of the array and get their own lookup, and
//     the context that replaces a primary context after cudaDeviceReset has
//     a new id, so a stale address is never reused. Make the first call in
//     each context before any stream capture in it.
// The result is bit-identical to moe_router_logits: the same kernels, the
// same split count and the same summation order.
#include <mutex>

#include "internal.cuh"

namespace moe {

constexpr size_t kNoAllocScratchFloats = size_t(1) << 20;   // 4 MiB
constexpr int kNoAllocCacheSlots = 64;

static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchFloats];

// Driver entry points, resolved through the runtime so the library needs no
// link against the driver library.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

struct CtxFns {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};

static const CtxFns& ctx_fns() {
  static const CtxFns f = [] {
    CtxFns r;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      r.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      r.get_id = reinterpret_cast<CtxGetIdFn>(p);
    return r;
  }();
  return f;
}

// Unique id of the calling thread's current context; false when there is
// none yet (the runtime has not made its primary context current) or the
// driver cannot say.
static bool current_ctx_id(unsigned long long* id) {
  const CtxFns& f = ctx_fns();
  if (!f.get_current || !f.get_id) return false;
  CUcontext c = nullptr;
  if (f.get_current(&c) != CUDA_SUCCESS || !c) return false;
  return f.get_id(c, id) == CUDA_SUCCESS;
}

static std::mutex g_noalloc_mu;
static unsigned long long g_noalloc_ctx[kNoAllocCacheSlots] = {};
static float* g_noalloc_ptr[kNoAllocCacheSlots] = {};
static int g_noalloc_next = 0;

// Device address of g_noalloc_scratch in the current context; nullptr on
// failure.
static float* noalloc_scratch() {
  unsigned long long id = 0;
  bool have = current_ctx_id(&id);
  if (have) {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    for (int i = 0; i < kNoAllocCacheSlots; ++i)
      if (g_noalloc_ptr[i] && g_noalloc_ctx[i] == id) return g_noalloc_ptr[i];
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
  // the lookup makes the runtime's context current if none was
  if (!have) have = current_ctx_id(&id);
  if (have) {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    const int i = g_noalloc_next;
    g_noalloc_next = (g_noalloc_next + 1) % kNoAllocCacheSlots;
    g_noalloc_ctx[i] = id;
    g_noalloc_ptr[i] = reinterpret_cast<float*>(p);
  }
  return reinterpret_cast<float*>(p);
}

__global__ void k_sum_partials_noalloc(const float* __restrict__ part, int KS, int64_t n, float* __restrict__ out) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    float v = part[i];
    for (int ks = 1; ks < KS; ++ks) v += part[(int64_t)ks * n + i];
    out[i] = v;
  }
}

}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_router_logits_noalloc(const moe_config_t* cfg, const uint16_t* x, const float* W_r,
                                                  int T, float* logits, void* stream) {
  moe_status_t s = moe_config_validate(cfg);
  if (s != MOE_OK) return s;
  if (T < 0 || T > cfg->T_max) return MOE_ERR_INVALID_ARG;
  if (!W_r || ((uintptr_t)W_r & 15u)) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!x || !logits || ((uintptr_t)x & 15u) || ((uintptr_t)logits & 15u))) return MOE_ERR_INVALID_ARG;
  reset_launch_count();
  if (T == 0) return MOE_OK;
  const int KS = router_splits(T, cfg->H, cfg->E);
  cudaStream_t st = (cudaStream_t)stream;
  if (KS == 1) {
    // one slice: the router kernel writes the logits directly, no scratch
    return launch_router(x, W_r, T, cfg->H, cfg->E, 1, logits, st) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
  const int64_t n = (int64_t)T * cfg->E;
  if ((size_t)KS * (size_t)n > kNoAllocScratchFloats) return MOE_ERR_WORKSPACE;
  float* part = noalloc_scratch();
  if (!part) return MOE_ERR_CUDA;
  if (launch_router(x, W_r, T, cfg->H, cfg->E, KS, part, st) != cudaSuccess) return MOE_ERR_CUDA;
  const int blocks = (int)std::min<int64_t>((n + 255) / 256, 4096);
  k_sum_partials_noalloc<<<blocks, 256, 0, st>>>(part, KS, n, logits);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
