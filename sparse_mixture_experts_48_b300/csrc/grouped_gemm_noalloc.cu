// moe_grouped_gemm_noalloc: the grouped expert GEMM for callers that cannot
// allocate device memory.
//
// moe_grouped_gemm takes its scratch (the status word and the per-group tile
// table, a few KB) from a workspace the caller allocates.  Some callers have no
// way to do that at call time: a host program whose device memory is planned
// and handed out once at start-up, a plugin that runs inside a framework which
// owns every allocation, or a latency-bound loop that must not call cudaMalloc
// (it can synchronise the whole device).  This entry point takes the same
// inputs and outputs but no workspace: its scratch is the file-scope device
// array below, of a fixed size, which every GPU that loads this library keeps
// until the process exits.
//
// Set-up: the first call in each CUDA context (normally a device's primary
// context), with that device current, looks up the array's device address with
// cudaGetSymbolAddress and keeps it, keyed by the context's ID; make that first
// call before any stream capture.  Later calls in the same context reuse the
// address.  If the context is destroyed and made again (cudaDeviceReset, or a
// context recreated after an error), the library's module is loaded again and
// the array can move: the new context has a new ID, so the next call looks the
// address up again and is a first call once more.  (In host code the array's
// name is only a host-side stand-in, never a device address, so kernels are
// always given the looked-up address.)
//
// Sharing: every call on a device uses the same array, and it keeps the last
// call's contents.  Each call clears the status word before its kernels run and
// rewrites the whole tile table, so nothing of an earlier call leaks into a
// later one.  Calls that may overlap on the GPU (different streams without an
// ordering between them) race on the array: order them, or use
// moe_grouped_gemm with one workspace per stream.
//
// Device-side failures (a bounded wait that ran out, offsets outside [0, M])
// are recorded in the array's status word but are not reported by this entry
// point: with bad offsets no group gets rows and C is left untouched.  A caller
// that needs to detect them uses moe_grouped_gemm and moe_check_device_errors.
//
// Nothing here allocates: no cudaMalloc, cudaFree or allocating library call.
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

using namespace moe;

namespace {

constexpr size_t kHeaderBytes = 256;           // status word region (sizeof(WsHeader))
constexpr size_t kTableBytes = (6 * kGroupedGemmMaxGroups + 1) * 4;
constexpr size_t kNoAllocScratchBytes = kHeaderBytes + (kTableBytes + 255) / 256 * 256;   // 6656 bytes
static_assert(sizeof(WsHeader) == kHeaderBytes, "status word region");

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// The current context's ID, through the driver entry points (this library does
// not link libcuda).  False if there is no current context or no entry point.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

bool current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = (CtxGetCurrentFn)p;
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = (CtxGetIdFn)p;
  });
  if (!get_current || !get_id) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

constexpr int kMaxDevices = 64;
struct CachedAddress {
  bool valid;
  unsigned long long ctx_id;
  void* addr;                                  // device address of g_noalloc_scratch in that context
};
std::mutex g_mu;
CachedAddress g_cache[kMaxDevices];

moe_status scratch_of_current_context(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  unsigned long long id = 0;
  bool have_id = current_context_id(&id);
  std::lock_guard<std::mutex> lock(g_mu);
  CachedAddress& c = g_cache[dev];
  if (have_id && c.valid && c.ctx_id == id) {
    *out = c.addr;
    return MOE_OK;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
  // The lookup makes the device's primary context current if none was.
  if (!have_id) have_id = current_context_id(&id);
  c.valid = have_id;                           // without a context ID, look up again on every call
  c.ctx_id = id;
  c.addr = p;
  *out = p;
  return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_grouped_gemm_noalloc(int32_t dtype, int32_t act, int32_t G, const int32_t* seg_offsets,
                                               int64_t M, int32_t K, int32_t N, const void* A, const void* B,
                                               const void* B3, const void* bias, void* C, moe_stream stream,
                                               const moe_launch_opts* opts) {
  // The fixed scratch holds the tile table of at most kGroupedGemmMaxGroups
  // groups; larger G is rejected (MOE_ERR_UNSUPPORTED) by the shared checks.
  static_assert(kNoAllocScratchBytes >= 256 + (6 * kGroupedGemmMaxGroups + 1) * 4, "scratch holds the table");
  const moe_status st = check_grouped_gemm_args(dtype, act, G, seg_offsets, M, K, N, A, B, B3, bias, C);
  if (st != MOE_OK) return st;
  void* scratch = nullptr;
  const moe_status sst = scratch_of_current_context(&scratch);
  if (sst != MOE_OK) return sst;
  return launch_grouped_gemm_on_scratch(dtype, act, G, seg_offsets, M, K, N, A, B, B3, bias, C, (uint8_t*)scratch,
                                        stream, opts);
}
