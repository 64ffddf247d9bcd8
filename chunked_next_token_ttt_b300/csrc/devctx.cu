// Per-context host state of libttt: state a CUDA context owns (function
// attributes, symbol addresses, SM counts) is cached under the context's
// process-unique id, so it is never reused on another device or after a
// device reset; and the per-thread PDL switch of the current API call.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"

namespace ttt {

namespace {

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_ctx_once;

void load_ctx_entry_points() {
  std::call_once(g_ctx_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    else
      cudaGetLastError();
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
    else
      cudaGetLastError();
  });
}

std::mutex g_mu;
std::map<std::pair<const void*, unsigned long long>, size_t> g_smem;   // (kernel, context) -> bytes opted in
std::map<std::pair<const void*, unsigned long long>, void*> g_sym;     // (symbol, context) -> device address
std::map<unsigned long long, int> g_sms;                               // context -> SM count

thread_local bool t_pdl = true;

}  // namespace

unsigned long long current_context_id() {
  load_ctx_entry_points();
  if (!g_ctx_current || !g_ctx_id) return 0;
  CUcontext c = nullptr;
  if (g_ctx_current(&c) != CUDA_SUCCESS || !c) {
    // no context bound to this thread yet: bind the current device's primary
    // context (cudaSetDevice initialises it)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    if (g_ctx_current(&c) != CUDA_SUCCESS || !c) return 0;
  }
  unsigned long long id = 0;
  if (g_ctx_id(c, &id) != CUDA_SUCCESS) return 0;
  return id + 1;   // 0 stays "unknown"
}

cudaError_t ensure_dyn_smem(const void* func, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_mu);
  auto key = std::make_pair(func, ctx);
  auto it = g_smem.find(key);
  if (ctx != 0 && it != g_smem.end() && it->second >= bytes) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess && ctx != 0) g_smem[key] = bytes;
  return e;
}

cudaError_t symbol_address(const void* symbol, void** out) {
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_mu);
  auto key = std::make_pair(symbol, ctx);
  auto it = g_sym.find(key);
  if (ctx != 0 && it != g_sym.end()) {
    *out = it->second;
    return cudaSuccess;
  }
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, symbol);
  if (e != cudaSuccess) return e;
  if (ctx != 0) g_sym[key] = p;
  *out = p;
  return cudaSuccess;
}

int current_sm_count() {
  const unsigned long long ctx = current_context_id();
  {
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = g_sms.find(ctx);
    if (ctx != 0 && it != g_sms.end()) return it->second;
  }
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = 148;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (ctx != 0) g_sms[ctx] = n;
  return n;
}

bool pdl_enabled() { return t_pdl; }

PdlScope::PdlScope(bool on) : saved_(t_pdl) { t_pdl = on; }
PdlScope::~PdlScope() { t_pdl = saved_; }

}  // namespace ttt
