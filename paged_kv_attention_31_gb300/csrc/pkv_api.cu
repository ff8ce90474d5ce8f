// pkv_api.cu -- the C ABI of include/pkv.h: host-side validation, split
// planning and kernel dispatch.  No allocation happens here; every kernel is
// enqueued on the caller's stream.
#include <math.h>
#include <string.h>

#include "pkv_common.cuh"
#include "pkv_launch.h"

// Sticky per-device error word written by the kernels (first error wins).
__device__ int32_t g_pkv_device_error = 0;
// Where pkv_get_device_error's exchange kernel leaves the word it took.
__device__ int32_t g_pkv_device_error_taken = 0;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  int num_sms = 0;
  int32_t* err = nullptr;
  int32_t* taken = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::atomic<bool> g_dev_ready[kMaxDevices];

pkv_status device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ERR_CUDA;
  DeviceInfo& d = g_dev[dev];
  const cudaError_t e = pkv::once_per_device(g_dev_ready, dev, [&]() -> cudaError_t {
    int sms = 0;
    void* addr = nullptr;
    cudaError_t r = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (r != cudaSuccess) return r;
    r = cudaGetSymbolAddress(&addr, g_pkv_device_error);
    if (r != cudaSuccess) return r;
    void* taken = nullptr;
    r = cudaGetSymbolAddress(&taken, g_pkv_device_error_taken);
    if (r != cudaSuccess) return r;
    d.num_sms = sms;
    d.err = static_cast<int32_t*>(addr);
    d.taken = static_cast<int32_t*>(taken);
    return cudaSuccess;
  });
  if (e != cudaSuccess) return PKV_ERR_CUDA;
  *out = &d;
  return PKV_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

pkv_status check_pool(const pkv_pool_desc* pool) {
  if (!pool) return PKV_ERR_INVALID_ARG;
  if (pool->num_blocks <= 0 || pool->num_kv_heads <= 0) return PKV_ERR_INVALID_ARG;
  if (pool->kv_dtype != PKV_KV_BF16 && pool->kv_dtype != PKV_KV_FP8_E4M3)
    return PKV_ERR_INVALID_ARG;
  if (pool->head_dim != 64 && pool->head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (pool->block_size != 16 && pool->block_size != 32 && pool->block_size != 64 &&
      pool->block_size != 128)
    return PKV_ERR_UNSUPPORTED;
  if (pool->kv_dtype == PKV_KV_FP8_E4M3) {
    if (!pool->k_scales && (!(pool->k_scale > 0.f) || !isfinite(pool->k_scale)))
      return PKV_ERR_INVALID_ARG;
    if (!pool->v_scales && (!(pool->v_scale > 0.f) || !isfinite(pool->v_scale)))
      return PKV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(pool->k_scales) & 3) ||
        (reinterpret_cast<uintptr_t>(pool->v_scales) & 3))
      return PKV_ERR_INVALID_ARG;
  }
  return PKV_OK;
}

thread_local cudaError_t g_last_cuda_error = cudaSuccess;

pkv_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return PKV_OK;
  g_last_cuda_error = e;
  if (e == cudaErrorNotSupported) return PKV_ERR_UNSUPPORTED;
  return PKV_ERR_CUDA;
}

// Split-K partition length: explicit (validated) or automatic.  The automatic
// choice keeps the largest work unit (one kv head of one partition) at about
// 1/8 of one CTA's share of an estimated total (half the maximum context per
// sequence), so the longest-first dynamic schedule stays balanced; never below
// 512 tokens, and no split when every sequence fits in one unit anyway.
int choose_partition(int32_t requested, int num_seqs, int num_kv_heads, int max_len,
                     int block_size, int elem_bytes, int head_dim, int num_sms) {
  if (requested > 0) return requested;
  const double per_tok = 2.0 * head_dim * elem_bytes;  // K+V bytes per token per kv head
  const double total = double(num_seqs) * num_kv_heads * (max_len / 2.0 + 1) * per_tok;
  const double per_cta = total / (double(num_sms) * 2.0);
  double tok = per_cta / 8.0 / per_tok;
  int part = 512;
  while (part * 2 <= tok && part < 8192) part *= 2;
  if (part >= max_len) part = ((max_len + block_size - 1) / block_size) * block_size;
  if (part < block_size) part = block_size;
  part = (part / block_size) * block_size;
  return part;
}

pkv_status validate_partition(int32_t partition, int block_size) {
  if (partition < 0) return PKV_ERR_INVALID_ARG;
  if (partition > 0 && (partition % block_size != 0 || partition > 16368))
    return PKV_ERR_INVALID_ARG;
  return PKV_OK;
}

// Self-test of the failure path: a wait on a barrier that nothing arrives at
// must give up after `limit` cycles, record PKV_ERR_DEVICE_TIMEOUT and raise
// the abort flag, after which a second wait returns at once.  out[0..4]:
// first wait's result (0), second wait's result (0), abort flag (1), first
// wait took >= limit cycles (1), second took < limit / 4 cycles (1).
__global__ void self_test_wait_kernel(int32_t* err, long long limit, int32_t* out) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    pkv::mbar_init(&bar, 1);
    abort_flag = 0;
    pkv::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  volatile int* flag = &abort_flag;
  const long long t0 = clock64();
  const bool first = pkv::mbar_wait_bounded(&bar, 0, err, flag, limit);
  const long long t1 = clock64();
  const bool second = pkv::mbar_wait_bounded(&bar, 0, err, flag, limit);
  const long long t2 = clock64();
  out[0] = first ? 1 : 0;
  out[1] = second ? 1 : 0;
  out[2] = *flag;
  out[3] = (t1 - t0) >= limit ? 1 : 0;
  out[4] = (t2 - t1) < limit / 4 ? 1 : 0;
}

// Read and clear the error word in one atomic step, so an error a kernel on
// another stream records meanwhile is either returned now or kept for the
// next read, never lost.
__global__ void take_error_kernel(int32_t* err, int32_t* taken) { *taken = atomicExch(err, 0); }

}  // namespace

extern "C" {

int32_t pkv_version(void) { return 101; }

const char* pkv_last_cuda_error(void) { return cudaGetErrorString(g_last_cuda_error); }

const char* pkv_status_string(int32_t s) {
  switch (s) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case PKV_ERR_WORKSPACE: return "workspace too small or misaligned";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_DEVICE_BOUNDS: return "device data out of range (page id, slot or length)";
    case PKV_ERR_DEVICE_TIMEOUT: return "bounded wait in a kernel ran out";
    case PKV_ERR_OUT_OF_BLOCKS: return "not enough free KV-cache blocks";
    default: return "unknown status";
  }
}

// Validated append parameters (status before anything is enqueued).
static pkv_status make_append(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                              int32_t num_tokens, void* k_pool, void* v_pool,
                              const pkv_pool_desc* pool, pkv::AppendParams* p, int32_t* err) {
  if (num_tokens < 0) return PKV_ERR_INVALID_ARG;
  if (!k_new || !v_new || !slot_mapping || !k_pool || !v_pool) return PKV_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7))
    return PKV_ERR_INVALID_ARG;
  p->k_new = k_new;
  p->v_new = v_new;
  p->slot_mapping = slot_mapping;
  p->k_pool = k_pool;
  p->v_pool = v_pool;
  p->num_slots = int64_t(pool->num_blocks) * pool->block_size;
  p->num_tokens = num_tokens;
  p->num_kv_heads = pool->num_kv_heads;
  p->block_size = pool->block_size;
  p->head_dim = pool->head_dim;
  p->k_scale = pool->k_scale;
  p->v_scale = pool->v_scale;
  const bool fp8_pool = pool->kv_dtype == PKV_KV_FP8_E4M3;
  p->k_scales = fp8_pool ? pool->k_scales : nullptr;
  p->v_scales = fp8_pool ? pool->v_scales : nullptr;
  p->fp8 = fp8_pool;
  p->err = err;
  return PKV_OK;
}

pkv_status pkv_kv_append(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                         int32_t num_tokens, void* k_pool, void* v_pool,
                         const pkv_pool_desc* pool, void* stream) {
  pkv_status st = check_pool(pool);
  if (st != PKV_OK) return st;
  if (num_tokens < 0) return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return PKV_OK;
  pkv::AppendParams p;
  if ((st = make_append(k_new, v_new, slot_mapping, num_tokens, k_pool, v_pool, pool, &p,
                        nullptr)) != PKV_OK)
    return st;
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != PKV_OK) return st;
  p.err = dev->err;
  return from_cuda(pkv::launch_kv_append(p, dev->num_sms, static_cast<cudaStream_t>(stream)));
}

pkv_status pkv_copy_blocks(void* k_pool, void* v_pool, const pkv_pool_desc* pool,
                           const int32_t* pairs, int32_t num_pairs, void* stream) {
  pkv_status st = check_pool(pool);
  if (st != PKV_OK) return st;
  if (num_pairs < 0) return PKV_ERR_INVALID_ARG;
  if (num_pairs == 0) return PKV_OK;
  if (!k_pool || !v_pool || !pairs || !aligned16(k_pool) || !aligned16(v_pool) ||
      (reinterpret_cast<uintptr_t>(pairs) & 3))
    return PKV_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != PKV_OK) return st;
  pkv::CopyParams p;
  p.pairs = pairs;
  p.num_pairs = num_pairs;
  p.num_blocks = pool->num_blocks;
  p.block_bytes = int64_t(pool->num_kv_heads) * pool->block_size * pool->head_dim *
                  (pool->kv_dtype == PKV_KV_FP8_E4M3 ? 1 : 2);
  p.k_pool = k_pool;
  p.v_pool = v_pool;
  p.err = dev->err;
  return from_cuda(pkv::launch_copy_blocks(p, dev->num_sms, static_cast<cudaStream_t>(stream)));
}

size_t pkv_paged_attention_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                          int32_t max_context_len, int32_t partition_tokens,
                                          const pkv_pool_desc* pool) {
  if (check_pool(pool) != PKV_OK || num_seqs < 0 || num_q_heads <= 0 || max_context_len < 0)
    return 0;
  if (validate_partition(partition_tokens, pool->block_size) != PKV_OK) return 0;
  DeviceInfo* dev = nullptr;
  int sms = 152;
  if (device_info(&dev) == PKV_OK) sms = dev->num_sms;
  const int eb = pool->kv_dtype == PKV_KV_FP8_E4M3 ? 1 : 2;
  const int part = choose_partition(partition_tokens, num_seqs, pool->num_kv_heads,
                                    max_context_len, pool->block_size, eb, pool->head_dim, sms);
  const int splits = pkv::decode_num_splits(max_context_len, part);
  return pkv::decode_workspace_layout(num_seqs, num_q_heads, pool->head_dim, splits).total;
}

pkv_status pkv_paged_attention_plan(int32_t num_seqs, int32_t num_q_heads,
                                   int32_t max_context_len, int32_t partition_tokens,
                                   const pkv_pool_desc* pool, int32_t* partition_out,
                                   int32_t* max_splits_out) {
  pkv_status st = check_pool(pool);
  if (st != PKV_OK) return st;
  if (!partition_out || !max_splits_out || num_seqs < 0 || num_q_heads <= 0 ||
      max_context_len < 0)
    return PKV_ERR_INVALID_ARG;
  if ((st = validate_partition(partition_tokens, pool->block_size)) != PKV_OK) return st;
  DeviceInfo* dev = nullptr;
  int sms = 152;
  if (device_info(&dev) == PKV_OK) sms = dev->num_sms;
  const int eb = pool->kv_dtype == PKV_KV_FP8_E4M3 ? 1 : 2;
  const int part = choose_partition(partition_tokens, num_seqs, pool->num_kv_heads,
                                    max_context_len, pool->block_size, eb, pool->head_dim, sms);
  *partition_out = part;
  *max_splits_out = pkv::decode_num_splits(max_context_len, part);
  return PKV_OK;
}

}  // extern "C"

namespace pkv {

// Host validation of a decode call's arguments other than its workspace, in
// the order the status codes are reported; PKV_OK for num_seqs == 0 once the
// sizes are valid (the pointers are then not looked at).
pkv_status decode_args_status(const void* q, const void* k_pool, const void* v_pool,
                              const pkv_pool_desc* pool, const int32_t* block_tables,
                              int32_t max_blocks_per_seq, const int32_t* context_lens,
                              int32_t num_seqs, int32_t num_q_heads, int32_t max_context_len,
                              float scale, int32_t partition_tokens, const void* out) {
  pkv_status st = check_pool(pool);
  if (st != PKV_OK) return st;
  if (num_seqs < 0 || num_q_heads <= 0 || max_context_len < 0 || max_blocks_per_seq <= 0)
    return PKV_ERR_INVALID_ARG;
  if (num_q_heads % pool->num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  const int G = num_q_heads / pool->num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return PKV_ERR_UNSUPPORTED;
  if (!isfinite(scale)) return PKV_ERR_INVALID_ARG;
  if ((st = validate_partition(partition_tokens, pool->block_size)) != PKV_OK) return st;
  if (num_seqs == 0) return PKV_OK;
  if (!q || !k_pool || !v_pool || !block_tables || !context_lens || !out)
    return PKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(block_tables) & 3) ||
      (reinterpret_cast<uintptr_t>(context_lens) & 3))
    return PKV_ERR_INVALID_ARG;
  return PKV_OK;
}

}  // namespace pkv

extern "C" {

// Decode attention; with `app`, the step's appends run in the planning launch.
static pkv_status paged_attention_impl(const void* q, const void* k_pool, const void* v_pool,
                                       const pkv_pool_desc* pool, const int32_t* block_tables,
                                       int32_t max_blocks_per_seq, const int32_t* context_lens,
                                       int32_t num_seqs, int32_t num_q_heads,
                                       int32_t max_context_len, float scale,
                                       int32_t partition_tokens, void* workspace,
                                       size_t workspace_bytes, void* out, void* stream,
                                       const pkv::AppendParams* app) {
  pkv_status st = pkv::decode_args_status(q, k_pool, v_pool, pool, block_tables,
                                          max_blocks_per_seq, context_lens, num_seqs,
                                          num_q_heads, max_context_len, scale, partition_tokens,
                                          out);
  if (st != PKV_OK || num_seqs == 0) return st;
  if (!workspace) return PKV_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return PKV_ERR_WORKSPACE;
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != PKV_OK) return st;

  const bool fp8 = pool->kv_dtype == PKV_KV_FP8_E4M3;
  const int eb = fp8 ? 1 : 2;
  const int64_t cap64 = int64_t(max_blocks_per_seq) * pool->block_size;
  const int max_len = int(cap64 < max_context_len ? cap64 : max_context_len);
  // the plan is chosen from the caller's max_context_len exactly as the
  // workspace query does; the clamped max_len can only lower the split count
  const int part = choose_partition(partition_tokens, num_seqs, pool->num_kv_heads,
                                    max_context_len, pool->block_size, eb, pool->head_dim,
                                    dev->num_sms);
  const int splits = pkv::decode_num_splits(max_len, part);
  const pkv::DecodeWorkspace ws =
      pkv::decode_workspace_layout(num_seqs, num_q_heads, pool->head_dim, splits);
  if (workspace_bytes < ws.total) return PKV_ERR_WORKSPACE;

  uint8_t* w = static_cast<uint8_t*>(workspace);
  pkv::DecodeParams p;
  p.q = q;
  p.k_pool = static_cast<const uint8_t*>(k_pool);
  p.v_pool = static_cast<const uint8_t*>(v_pool);
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.out = out;
  p.counters = reinterpret_cast<int32_t*>(w + ws.counters);
  p.items = reinterpret_cast<int2*>(w + ws.items);
  p.ws_ml = reinterpret_cast<float*>(w + ws.ml);
  p.ws_acc = reinterpret_cast<float*>(w + ws.acc);
  p.err = dev->err;
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = pool->num_kv_heads;
  p.head_dim = pool->head_dim;
  p.block_size = pool->block_size;
  p.max_blocks = max_blocks_per_seq;
  p.num_blocks = pool->num_blocks;
  p.max_len = max_len;
  p.partition = part;
  p.max_splits = splits;
  // per-head scales multiply in inside the kernels, per kv head
  p.k_scales = fp8 ? pool->k_scales : nullptr;
  p.v_scales = fp8 ? pool->v_scales : nullptr;
  p.q_mult = scale * (fp8 && !p.k_scales ? pool->k_scale : 1.0f) * 1.4426950408889634f;
  p.v_mult = fp8 && !p.v_scales ? pool->v_scale : 1.0f;
  p.fuse_append = app != nullptr;
  if (app) {
    p.append = *app;
    p.append.err = dev->err;
  }
  return from_cuda(pkv::launch_decode(p, fp8, dev->num_sms, static_cast<cudaStream_t>(stream)));
}

pkv_status pkv_paged_attention(const void* q, const void* k_pool, const void* v_pool,
                               const pkv_pool_desc* pool, const int32_t* block_tables,
                               int32_t max_blocks_per_seq, const int32_t* context_lens,
                               int32_t num_seqs, int32_t num_q_heads, int32_t max_context_len,
                               float scale, int32_t partition_tokens, void* workspace,
                               size_t workspace_bytes, void* out, void* stream) {
  return paged_attention_impl(q, k_pool, v_pool, pool, block_tables, max_blocks_per_seq,
                              context_lens, num_seqs, num_q_heads, max_context_len, scale,
                              partition_tokens, workspace, workspace_bytes, out, stream, nullptr);
}

pkv_status pkv_paged_attention_append(const void* q, const void* k_new, const void* v_new,
                                      const int64_t* slot_mapping, int32_t num_new_tokens,
                                      void* k_pool, void* v_pool, const pkv_pool_desc* pool,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      const int32_t* context_lens, int32_t num_seqs,
                                      int32_t num_q_heads, int32_t max_context_len, float scale,
                                      int32_t partition_tokens, void* workspace,
                                      size_t workspace_bytes, void* out, void* stream) {
  pkv_status st = check_pool(pool);
  if (st != PKV_OK) return st;
  if (num_new_tokens < 0) return PKV_ERR_INVALID_ARG;
  pkv::AppendParams app;
  if (num_new_tokens > 0 &&
      (st = make_append(k_new, v_new, slot_mapping, num_new_tokens, k_pool, v_pool, pool, &app,
                        nullptr)) != PKV_OK)
    return st;
  if (num_seqs == 0)  // nothing to attend: the append alone
    return pkv_kv_append(k_new, v_new, slot_mapping, num_new_tokens, k_pool, v_pool, pool,
                         stream);
  return paged_attention_impl(q, k_pool, v_pool, pool, block_tables, max_blocks_per_seq,
                              context_lens, num_seqs, num_q_heads, max_context_len, scale,
                              partition_tokens, workspace, workspace_bytes, out, stream,
                              num_new_tokens > 0 ? &app : nullptr);
}

pkv_status pkv_paged_prefill(const void* q, const int32_t* cu_seqlens_q, const void* k_pool,
                             const void* v_pool, const pkv_pool_desc* pool,
                             const int32_t* block_tables, int32_t max_blocks_per_seq,
                             const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                             int32_t max_q_len, int32_t num_q_tokens, float scale, void* out,
                             void* stream) {
  pkv_status st = check_pool(pool);
  if (st != PKV_OK) return st;
  if (num_seqs < 0 || num_q_heads <= 0 || max_q_len < 0 || num_q_tokens < 0 ||
      max_blocks_per_seq <= 0)
    return PKV_ERR_INVALID_ARG;
  if (num_q_heads % pool->num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  const int G = num_q_heads / pool->num_kv_heads;
  if (G > 128 || 128 % G != 0) return PKV_ERR_UNSUPPORTED;
  if (!isfinite(scale) || !(scale > 0.f)) return PKV_ERR_INVALID_ARG;
  if (num_seqs == 0 || num_q_tokens == 0 || max_q_len == 0) return PKV_OK;
  if (!q || !cu_seqlens_q || !k_pool || !v_pool || !block_tables || !context_lens || !out)
    return PKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(block_tables) & 3) ||
      (reinterpret_cast<uintptr_t>(context_lens) & 3) ||
      (reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3))
    return PKV_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != PKV_OK) return st;
  pkv::PrefillParams p;
  p.q = q;
  p.cu_seqlens_q = cu_seqlens_q;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.out = out;
  p.err = dev->err;
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = pool->num_kv_heads;
  p.head_dim = pool->head_dim;
  p.block_size = pool->block_size;
  p.max_blocks = max_blocks_per_seq;
  p.num_blocks = pool->num_blocks;
  p.num_q_tokens = num_q_tokens;
  p.tiles_per_seq = (int)((int64_t(max_q_len) * G + 127) / 128);
  const bool fp8 = pool->kv_dtype == PKV_KV_FP8_E4M3;
  p.fp8 = fp8;
  // per-head scales multiply in inside the kernel, per kv head
  p.k_scales = fp8 ? pool->k_scales : nullptr;
  p.v_scales = fp8 ? pool->v_scales : nullptr;
  p.q_mult = scale * (fp8 && !p.k_scales ? pool->k_scale : 1.0f) * 1.4426950408889634f;
  p.v_mult = fp8 && !p.v_scales ? pool->v_scale : 1.0f;
  return from_cuda(
      pkv::launch_prefill(p, k_pool, v_pool, dev->num_sms, static_cast<cudaStream_t>(stream)));
}

pkv_status pkv_self_test_bounded_wait(int64_t limit_cycles, int32_t* out, void* stream) {
  if (!out || (reinterpret_cast<uintptr_t>(out) & 3) || limit_cycles <= 0 ||
      limit_cycles > pkv::kWaitLimitCycles)
    return PKV_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  pkv_status st = device_info(&dev);
  if (st != PKV_OK) return st;
  self_test_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev->err, limit_cycles,
                                                                        out);
  return from_cuda(cudaGetLastError());
}

pkv_status pkv_get_device_error(int32_t* code, void* stream) {
  if (!code) return PKV_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  pkv_status st = device_info(&dev);
  if (st != PKV_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the landing slot is shared by the host threads that read the word
  static std::mutex m;
  std::lock_guard<std::mutex> lock(m);
  int32_t v = 0;
  take_error_kernel<<<1, 1, 0, s>>>(dev->err, dev->taken);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaMemcpyAsync(&v, dev->taken, sizeof(v), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    g_last_cuda_error = e;
    return PKV_ERR_CUDA;
  }
  *code = v;
  return PKV_OK;
}

}  // extern "C"
