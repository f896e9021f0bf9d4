// mgq_moe_permute_noalloc: the permute + quantise call for callers that
// cannot allocate device memory.
//
// Some callers have no way to obtain device scratch: for example a plugin
// whose host framework owns every device allocation and hands it only its
// inputs and outputs, or a runtime that forbids allocation once it is
// running (an allocation can block on the device and has no bounded cost).
// This entry point takes the routing scratch from a fixed device array that
// is part of the library image instead of a caller-provided workspace; it
// makes no call that allocates (no cudaMalloc, cudaFree, or allocating
// library routine).
#include <mutex>

#include "mgq_internal.h"

namespace {

// Routing scratch of mgq_moe_permute_noalloc: one int32 per (chunk of 1024
// routed entries, expert). 1 MiB; every GPU that loads the library holds it
// until the process exits.
constexpr size_t kScratchInts = 262144;
static __device__ __align__(256) int32_t g_permute_scratch[kScratchInts];

constexpr int kMaxDevices = 64;
int32_t* g_scratch_dev[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device. Resolved once
// per device (with that device current) and cached. In host code the array's
// name only denotes a host-side stand-in, so kernels must get this address.
int32_t* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_dev[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || p == nullptr) return nullptr;
    g_scratch_dev[dev] = static_cast<int32_t*>(p);
  }
  return g_scratch_dev[dev];
}

}  // namespace

extern "C" {

int mgq_moe_permute_noalloc(const void* x_bf16, int T, int H, const int32_t* topk_idx, int k, int E, int align,
                            const mgq_qdesc* q, void* out_bf16, int64_t R_cap, int32_t* row_id_map,
                            int32_t* src_row, int32_t* offsets, int32_t* counts, void* stream) {
  const size_t need = mgq_permute_workspace_size(T, k, E);
  if (need > sizeof(g_permute_scratch)) return MGQ_ERR_INVALID_ARG;   // beyond the fixed scratch
  int32_t* scratch = scratch_address();
  if (!scratch) return MGQ_ERR_CUDA;
  // The routing kernels write every scratch entry they later read, so the
  // array needs no clearing between calls.
  return mgq_moe_permute(x_bf16, T, H, topk_idx, k, E, align, q, out_bf16, R_cap, row_id_map, src_row, offsets,
                         counts, scratch, sizeof(g_permute_scratch), stream);
}

}  // extern "C"
