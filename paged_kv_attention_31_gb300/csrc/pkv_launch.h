// pkv_launch.h -- kernel parameter blocks and launchers (internal; host and
// device code of the library include it, the public ABI is include/pkv.h).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>
#include <mutex>
#include <utility>

#include "../../include/pkv.h"

namespace pkv {

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel of the stream finishes (it must call pdl_wait() before
// touching memory that kernel uses), hiding launch latency between the
// kernels of one step.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Per-device one-time host set-up (kernel attributes, cached lookups) that
// concurrent host threads may reach together: `setup` runs under one lock
// until it first succeeds for the device; `done[dev]` then publishes its
// results (release / acquire) and later calls skip the lock.
inline std::mutex& setup_mutex() {
  static std::mutex m;
  return m;
}
template <typename F>
cudaError_t once_per_device(std::atomic<bool>* done, int dev, F&& setup) {
  if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  std::lock_guard<std::mutex> lock(setup_mutex());
  if (done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
  const cudaError_t e = setup();
  if (e == cudaSuccess) done[dev].store(true, std::memory_order_release);
  return e;
}

struct AppendParams {
  const void* k_new;            // bf16 [T][Hkv][D]
  const void* v_new;
  const int64_t* slot_mapping;  // [T]
  void* k_pool;
  void* v_pool;
  int64_t num_slots;            // num_blocks * block_size
  int32_t num_tokens, num_kv_heads, block_size, head_dim;
  float k_scale, v_scale;
  const float* k_scales;        // optional per-kv-head scales (override the scalars)
  const float* v_scales;
  int32_t fp8;
  int32_t* err;
};

// Work item of the split-K decode: (sequence, partition index).
struct DecodeParams {
  const void* q;                // bf16 [B][Hq][D]
  const uint8_t* k_pool;
  const uint8_t* v_pool;
  const int32_t* block_tables;  // [B][max_blocks]
  const int32_t* context_lens;  // [B]
  void* out;                    // bf16 [B][Hq][D]
  float* ws_acc;                // [B][Hq][max_splits][D], unnormalised
  float* ws_ml;                 // [B][Hq][max_splits][2]: running max (log2), sum
  int2* items;                  // [B * max_splits] from the planner
  int32_t* counters;            // [0] item count, [1] work-fetch counter
  int32_t* err;
  int32_t num_seqs, num_q_heads, num_kv_heads, head_dim, block_size;
  int32_t max_blocks, num_blocks;
  int32_t max_len;              // effective cap on context lengths
  int32_t partition;            // tokens per split partition (multiple of block_size)
  int32_t max_splits;
  float q_mult;                 // scale * k_scale * log2(e) (k_scale 1 with per-head scales)
  float v_mult;                 // v_scale (FP8, per tensor) or 1
  const float* k_scales;        // optional per-kv-head FP8 scales, multiplied in per head
  const float* v_scales;
  // pkv_paged_attention_append: this step's appends, done by the planning
  // launch (every CTA scatters rows; CTA 0 also plans)
  int32_t fuse_append;
  AppendParams append;
};

struct PrefillParams {
  const void* q;                // bf16 [Tq][Hq][D]
  const int32_t* cu_seqlens_q;  // [n + 1]
  const int32_t* block_tables;  // [n][max_blocks]
  const int32_t* context_lens;  // [n]
  void* out;                    // bf16 [Tq][Hq][D]
  int32_t* err;
  int32_t num_seqs, num_q_heads, num_kv_heads, head_dim, block_size;
  int32_t max_blocks, num_blocks, num_q_tokens;
  int32_t tiles_per_seq;        // ceil(max_q_len * G / 128)
  float q_mult;                 // scale * k_scale * log2(e) (k_scale: FP8 per tensor, else 1)
  float v_mult;                 // v_scale (FP8 per tensor) or 1
  const float* k_scales;        // optional per-kv-head FP8 scales, multiplied in per head
  const float* v_scales;
  int32_t fp8;                  // the pools hold E4M3 codes
};

// Split plan shared by the host (workspace sizing) and the kernels.
__host__ __device__ inline int decode_num_splits(int len, int partition) {
  return len <= partition ? 1 : (len + partition - 1) / partition;
}

// Workspace layout of pkv_paged_attention (byte offsets, 256-aligned).
struct DecodeWorkspace {
  size_t counters, items, ml, acc, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline DecodeWorkspace decode_workspace_layout(int num_seqs, int num_q_heads, int head_dim,
                                               int max_splits) {
  DecodeWorkspace w;
  const size_t rows = size_t(num_seqs) * num_q_heads * max_splits;
  w.counters = 0;
  w.items = align256(w.counters + 4 * sizeof(int32_t));
  w.ml = align256(w.items + size_t(num_seqs) * max_splits * 8);
  w.acc = align256(w.ml + rows * 2 * sizeof(float));
  w.total = align256(w.acc + rows * head_dim * sizeof(float));
  return w;
}

cudaError_t launch_kv_append(const AppendParams& p, int num_sms, cudaStream_t stream);

// Whole-block copies (all kv heads of K and of V) for copy-on-write.
struct CopyParams {
  const int32_t* pairs;   // [num_pairs][2]: (source block, destination block)
  int32_t num_pairs;
  int32_t num_blocks;
  int64_t block_bytes;    // Hkv * P * D * element size: one block of one pool
  void* k_pool;
  void* v_pool;
  int32_t* err;
};
cudaError_t launch_copy_blocks(const CopyParams& p, int num_sms, cudaStream_t stream);
// split planner and partial merge of the decode (decode.cu)
cudaError_t launch_decode_plan(const DecodeParams& p, int num_sms, cudaStream_t stream);
cudaError_t launch_decode_merge(const DecodeParams& p, cudaStream_t stream);
// head_dim 128, 4 or 8 q heads per kv head, bf16 or FP8 KV (decode_mma.cu)
cudaError_t launch_decode_mma(const DecodeParams& p, bool fp8, int num_sms, cudaStream_t stream);
// Returns cudaErrorNotSupported for shapes without a kernel instance.
cudaError_t launch_decode(const DecodeParams& p, bool fp8, int num_sms, cudaStream_t stream);
cudaError_t launch_prefill(const PrefillParams& p, const void* k_pool, const void* v_pool,
                           int num_sms, cudaStream_t stream);

// Host validation shared by the decode entry points (pkv_api.cu): the status
// a decode call reports for these arguments before its workspace is looked at.
pkv_status decode_args_status(const void* q, const void* k_pool, const void* v_pool,
                              const pkv_pool_desc* pool, const int32_t* block_tables,
                              int32_t max_blocks_per_seq, const int32_t* context_lens,
                              int32_t num_seqs, int32_t num_q_heads, int32_t max_context_len,
                              float scale, int32_t partition_tokens, const void* out);

}  // namespace pkv
