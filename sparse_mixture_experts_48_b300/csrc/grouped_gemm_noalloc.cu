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
// Set-up: the first call on each device, with that device current, looks up the
// array's device address with cudaGetSymbolAddress and keeps it; make that first
// call before any stream capture.  Later calls reuse the address.  (In host code
// the array's name is only a host-side stand-in, never a device address, so
// kernels are always given the looked-up address.)
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
// point: with bad offsets no group gets rows and C is left untouched.
//
// Nothing here allocates: no cudaMalloc, cudaFree or allocating library call.
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

using namespace moe;

namespace {

constexpr int kNoAllocMaxGroups = 264;        // the grouped GEMM's own limit on G
constexpr size_t kHeaderBytes = 256;           // status word region (sizeof(WsHeader))
constexpr size_t kTableBytes = (6 * kNoAllocMaxGroups + 1) * 4;
constexpr size_t kNoAllocScratchBytes = kHeaderBytes + (kTableBytes + 255) / 256 * 256;   // 6656 bytes
static_assert(sizeof(WsHeader) == kHeaderBytes, "status word region");

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices];             // device address of g_noalloc_scratch, per device

moe_status scratch_of_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

extern "C" moe_status moe_grouped_gemm_noalloc(int32_t dtype, int32_t act, int32_t G, const int32_t* seg_offsets,
                                               int64_t M, int32_t K, int32_t N, const void* A, const void* B,
                                               const void* B3, const void* bias, void* C, moe_stream stream,
                                               const moe_launch_opts* opts) {
  if (dtype != MOE_DT_F32 && dtype != MOE_DT_BF16) return MOE_ERR_INVALID_ARG;
  if (act != MOE_ACT_NONE && act != MOE_ACT_RELU && act != MOE_ACT_GELU && act != MOE_ACT_SWIGLU)
    return MOE_ERR_INVALID_ARG;
  if (G <= 0 || M < 0 || K <= 0 || N <= 0 || !seg_offsets || !A || !B || !C) return MOE_ERR_INVALID_ARG;
  if ((act == MOE_ACT_SWIGLU) != (B3 != nullptr)) return MOE_ERR_INVALID_ARG;
  if (G > kNoAllocMaxGroups) return MOE_ERR_UNSUPPORTED;   // the fixed scratch holds at most this many groups
  if (dtype == MOE_DT_BF16 && (K % 64 != 0 || N % 64 != 0)) return MOE_ERR_UNSUPPORTED;
  if (M >= ((int64_t)1 << 31) - 2 * kGemmBM) return MOE_ERR_UNSUPPORTED;
  const void* all[] = {seg_offsets, A, B, B3, bias, C};
  for (const void* p : all)
    if (p && !aligned16(p)) return MOE_ERR_INVALID_ARG;

  void* scratch = nullptr;
  moe_status st = scratch_of_current_device(&scratch);
  if (st != MOE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* ws = (uint8_t*)scratch;
  WsHeader* hdr = (WsHeader*)ws;
  SegTable seg;
  int* tab = (int*)(ws + kHeaderBytes);
  seg.rows = tab;
  seg.w = tab + G;
  seg.out_row = tab + 2 * G;
  seg.a_row = tab + 3 * G;
  seg.a_src = tab + 4 * G;
  seg.mtile_start = tab + 5 * G;
  if (cudaMemsetAsync(hdr, 0, sizeof(WsHeader), s) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_segments_from_offsets(seg_offsets, G, M, seg, &hdr->err, s) != cudaSuccess) return MOE_ERR_CUDA;
  GemmArgs g;
  memset(&g, 0, sizeof(g));
  g.dtype = dtype; g.act = act; g.G = G; g.K = K; g.N = N; g.a_from_out_rows = true; g.seg = seg;
  g.A0 = A; g.rows_A0 = M > 0 ? M : 1; g.A1 = nullptr; g.B = B; g.B3 = B3; g.Gw = G; g.bias = bias; g.C = C;
  g.max_mtiles = M > 0 ? (M + kGemmBM - 1) / kGemmBM + G : 0;
  g.err = &hdr->err;
  g.timeout_ns = (opts && opts->wait_timeout_ns > 0) ? opts->wait_timeout_ns : 2000000000LL;
  if (opts && opts->stage_events && cudaEventRecord((cudaEvent_t)opts->stage_events[0], s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (launch_grouped_gemm(g, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (opts && opts->stage_events && cudaEventRecord((cudaEvent_t)opts->stage_events[1], s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
