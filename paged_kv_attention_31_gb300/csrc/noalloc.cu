// noalloc.cu -- pkv_paged_attention_noalloc: decode attention with the split
// scratch space taken from a fixed, library-owned device array instead of a
// caller-provided workspace.
//
// Who needs it: callers that are handed only their input and output buffers
// and have no way to obtain device scratch -- for example a plugin invoked by
// a host engine that owns every device allocation and offers no workspace
// hook, or a latency-critical step that must not call cudaMalloc (which can
// synchronise the device and may fail at run time).  This entry point
// allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
//
// The scratch array below lives in this file for as long as the library is
// loaded: every GPU that loads the library holds kNoAllocScratchBytes of it
// until the process exits.
#include "pkv_common.cuh"
#include "pkv_launch.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB

// Device-side scratch shared by every call of pkv_paged_attention_noalloc.
// In host code this name is only a stand-in for the device symbol; its device
// address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {nullptr};
std::atomic<bool> g_scratch_ready[kMaxDevices];

// Per-device set-up: resolve the device address of the scratch array with
// that device current.  Done once per device, on its first call.
pkv_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ERR_CUDA;
  const cudaError_t e = pkv::once_per_device(g_scratch_ready, dev, [&]() -> cudaError_t {
    void* ptr = nullptr;
    const cudaError_t r = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (r != cudaSuccess) return r;
    if (!ptr) return cudaErrorInvalidSymbol;
    g_scratch_addr[dev] = ptr;
    return cudaSuccess;
  });
  if (e != cudaSuccess) return PKV_ERR_CUDA;
  *out = g_scratch_addr[dev];
  return PKV_OK;
}

}  // namespace

extern "C" {

size_t pkv_paged_attention_noalloc_max_scratch(void) { return kNoAllocScratchBytes; }

pkv_status pkv_paged_attention_noalloc(const void* q, const void* k_pool, const void* v_pool,
                                       const pkv_pool_desc* pool, const int32_t* block_tables,
                                       int32_t max_blocks_per_seq, const int32_t* context_lens,
                                       int32_t num_seqs, int32_t num_q_heads,
                                       int32_t max_context_len, float scale,
                                       int32_t partition_tokens, void* out, void* stream) {
  // the argument checks of pkv_paged_attention, so that both report the
  // same status for the same arguments
  pkv_status st = pkv::decode_args_status(q, k_pool, v_pool, pool, block_tables,
                                          max_blocks_per_seq, context_lens, num_seqs,
                                          num_q_heads, max_context_len, scale, partition_tokens,
                                          out);
  if (st != PKV_OK || num_seqs == 0) return st;
  const size_t need = pkv_paged_attention_workspace_size(num_seqs, num_q_heads, max_context_len,
                                                         partition_tokens, pool);
  if (need == 0) return PKV_ERR_INVALID_ARG;
  if (need > kNoAllocScratchBytes) return PKV_ERR_WORKSPACE;  // beyond the fixed maximum
  void* scratch = nullptr;
  if ((st = scratch_address(&scratch)) != PKV_OK) return st;
  // The decode path needs no zeroed scratch: its planner kernel rewrites the
  // work counters and item list before the decode kernel reads them, and every
  // partial result is written before the merge reads it.
  return pkv_paged_attention(q, k_pool, v_pool, pool, block_tables, max_blocks_per_seq,
                             context_lens, num_seqs, num_q_heads, max_context_len, scale,
                             partition_tokens, scratch, kNoAllocScratchBytes, out, stream);
}

}  // extern "C"
