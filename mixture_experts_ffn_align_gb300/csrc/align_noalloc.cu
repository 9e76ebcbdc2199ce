// moe_align_permute_noalloc: the routing + permute stage for callers that must
// not allocate device memory.
//
// Some programs that embed this library cannot hand it a workspace: a serving
// engine that reserves all device memory for its own pool at start-up and
// forbids its plug-ins from calling cudaMalloc, or a latency-critical loop
// where cudaMalloc's implicit device synchronisation is not acceptable.  This
// entry point does the same work as moe_align_permute, but the only scratch it
// needs -- the per-segment expert histograms -- lives in a fixed array that is
// part of the library's device image, so nothing is allocated at call time.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it (kNoAllocScratchBytes) until the process exits.  Host code
// may not use its name as a pointer (that names a host-side stand-in), so the
// device address is looked up with cudaGetSymbolAddress once per device, with
// that device current, on the first call made on that device.
#include <mutex>

#include "../../include/moe_ffn.h"
#include "moe_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = MOE_NOALLOC_SCRATCH_BYTES;
static_assert(kNoAllocScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");

// Per-segment histograms of the routing kernels.  Every call overwrites the
// part it uses before reading it (k_route_hist writes all E counters of each
// segment), so nothing has to be cleared between calls.
static __device__ __align__(256) int32_t g_align_scratch[kNoAllocScratchBytes / sizeof(int32_t)];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of g_align_scratch on the current device (looked up once).
moe_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_align_scratch);
    if (e != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_align_permute_noalloc(const moe_problem* p, const void* x,
                                                const int32_t* topk_ids, const float* topk_weights,
                                                int32_t* sorted_ids, int32_t* block_expert_ids,
                                                int32_t* expert_offsets, int32_t* num_post_padded,
                                                int32_t* inv_perm, void* x_perm,
                                                float* x_perm_scale, void* stream) {
  const size_t need = moe_align_workspace_bytes(p);
  if (need == 0) return MOE_ERR_INVALID_ARG;                     // invalid problem
  if (need > kNoAllocScratchBytes) return MOE_ERR_WORKSPACE_TOO_SMALL;  // beyond the fixed array
  void* scratch = nullptr;
  const moe_status st = scratch_address(&scratch);
  if (st != MOE_OK) return st;
  return moe_align_permute(p, x, topk_ids, topk_weights, sorted_ids, block_expert_ids,
                           expert_offsets, num_post_padded, inv_perm, x_perm, x_perm_scale,
                           scratch, kNoAllocScratchBytes, stream);
}
