// Host-side status reporting shared by every entry point of the C ABI.
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include <cuda.h>

#include "common.cuh"

namespace argus {

static thread_local char g_last_error[512] = "";

argus_status fail(argus_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return s;
}

argus_status launch_status(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    return fail(ARGUS_E_LAUNCH, "%s: launch failed: %s", what, cudaGetErrorString(e));
  }
  return ARGUS_OK;
}

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
  return n > 0 ? n : 1;
}

argus_status pool_device_ptrs(const argus_pool& pool, const void** codes, const void** meta) {
  *codes = pool.codes;
  *meta = pool.meta;
  if (pool.placement == ARGUS_PLACE_DEVICE) return ARGUS_OK;
  if (pool.placement != ARGUS_PLACE_HOST) return fail(ARGUS_E_INVALID, "pool placement %d unknown", pool.placement);
  if (pool.n_slots == 0) return ARGUS_OK;
  // page-locked (allocated or registered with CUDA) host memory only: pageable
  // memory is refused even where the platform could reach it
  auto pinned = [](const void* ptr) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, ptr) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    return at.type == cudaMemoryTypeHost;
  };
  void* dc = nullptr;
  void* dm = nullptr;
  if (!pool.codes || !pinned(pool.codes) || (pool.meta && !pinned(pool.meta)) ||
      cudaHostGetDevicePointer(&dc, pool.codes, 0) != cudaSuccess ||
      (pool.meta && cudaHostGetDevicePointer(&dm, pool.meta, 0) != cudaSuccess)) {
    cudaGetLastError();   // clear the (non-sticky) error of a failed query
    return fail(ARGUS_E_INVALID, "host pool (codec %d) is not page-locked memory the device can map", pool.codec);
  }
  *codes = dc;
  *meta = dm;
  return ARGUS_OK;
}

// The driver's cuCtxGetCurrent / cuCtxGetId, reached through the runtime's
// entry-point query so that the library links against the runtime only.
unsigned long long context_id() {
  typedef CUresult (*GetCurrentFn)(CUcontext*);
  typedef CUresult (*GetIdFn)(CUcontext, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* a = nullptr;
    void* b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 4000, cudaEnableDefault, &qa) == cudaSuccess &&
        qa == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) == cudaSuccess &&
        qb == cudaDriverEntryPointSuccess) {
      get_current = reinterpret_cast<GetCurrentFn>(a);
      get_id = reinterpret_cast<GetIdFn>(b);
    }
  });
  if (!get_current || !get_id) return 0ull;
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (get_current(&c) != CUDA_SUCCESS || c == nullptr) return 0ull;
  if (get_id(c, &id) != CUDA_SUCCESS) return 0ull;
  return id;
}

}  // namespace argus

extern "C" const char* argus_status_string(argus_status s) {
  switch (s) {
    case ARGUS_OK: return "ok";
    case ARGUS_E_INVALID: return "invalid argument";
    case ARGUS_E_UNSUPPORTED: return "unsupported shape or codec";
    case ARGUS_E_WORKSPACE: return "workspace too small";
    case ARGUS_E_LAUNCH: return "kernel launch failed";
  }
  return "unknown status";
}

extern "C" const char* argus_last_error(void) { return argus::g_last_error; }

// Host-only decision of the staged prefill: stage when the rows' in-place
// reads together exceed the cache ("--kv-placement host" comment of the
// host-RAM KV tier pull request).  Each row is compared with the headroom
// left under cache_bytes, so no sum can overflow.
extern "C" argus_status argus_staging_moves_less(const int64_t* row_read_bytes, int64_t n_rows,
                                                 int64_t cache_bytes, int32_t* stage) {
  using argus::fail;
  if (!stage) return fail(ARGUS_E_INVALID, "staging: stage is NULL");
  if (n_rows < 0 || cache_bytes < 0) return fail(ARGUS_E_INVALID, "staging: negative n_rows or cache_bytes");
  if (n_rows > 0 && !row_read_bytes) return fail(ARGUS_E_INVALID, "staging: row_read_bytes is NULL");
  int64_t sum = 0;
  int32_t more = 0;
  for (int64_t i = 0; i < n_rows; ++i) {
    const int64_t b = row_read_bytes[i];
    if (b < 0) return fail(ARGUS_E_INVALID, "staging: row %lld reads a negative byte count", (long long)i);
    if (!more) {
      if (b > cache_bytes - sum) more = 1;   // sum <= cache_bytes: the difference is >= 0
      else sum += b;
    }
  }
  *stage = more;
  return ARGUS_OK;
}
