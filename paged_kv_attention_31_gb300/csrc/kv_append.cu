// kv_append.cu -- scatter this step's new K/V rows into their pool slots
// (the row loop itself is in pkv_append.cuh), and copy whole blocks for
// copy-on-write of shared pages.
//
// "TensorRT-LLM框架解析与高性能推理优化实践" §4.2 (KV缓存管理细节): a growing
// sequence's tokens live in non-contiguous pages; the caller's page allocator
// gives each new token a slot = page * block_size + offset.
#include "pkv_append.cuh"

namespace pkv {

template <bool FP8>
__global__ void __launch_bounds__(256) kv_append_kernel(const AppendParams p) {
  pdl_launch_dependents();  // the next kernel may start its prologue now
  append_rows<FP8>(p, int64_t(blockIdx.x) * blockDim.x + threadIdx.x,
                   int64_t(gridDim.x) * blockDim.x);
}

cudaError_t launch_kv_append(const AppendParams& p, int num_sms, cudaStream_t stream) {
  const int64_t total = int64_t(p.num_tokens) * p.num_kv_heads * (p.head_dim / 8);
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = int64_t(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (p.fp8)
    kv_append_kernel<true><<<int(blocks), threads, 0, stream>>>(p);
  else
    kv_append_kernel<false><<<int(blocks), threads, 0, stream>>>(p);
  return cudaGetLastError();
}

// Copy-on-write of shared blocks: pair i copies block pairs[2i] to block
// pairs[2i + 1] in both pools.  One (page, kv head) run is contiguous, so a
// block of one pool is one contiguous Hkv * P * D * elem run: the copy is a
// straight 16-byte-vector stream, CTAs of one pair splitting it along x.
// An out-of-range block id is recorded and its pair skipped.
__global__ void __launch_bounds__(256) copy_blocks_kernel(const CopyParams p) {
  const int64_t nvec = p.block_bytes / 16;
  for (int pair = blockIdx.y; pair < p.num_pairs; pair += gridDim.y) {
    const int32_t src = __ldg(p.pairs + 2 * pair);
    const int32_t dst = __ldg(p.pairs + 2 * pair + 1);
    if (src < 0 || src >= p.num_blocks || dst < 0 || dst >= p.num_blocks) {
      if (blockIdx.x == 0 && threadIdx.x == 0) record_error(p.err, kDevBadPage);
      continue;
    }
    const uint4* ks = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.k_pool) +
                                                     src * p.block_bytes);
    const uint4* vs = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.v_pool) +
                                                     src * p.block_bytes);
    uint4* kd = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.k_pool) + dst * p.block_bytes);
    uint4* vd = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.v_pool) + dst * p.block_bytes);
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec;
         i += int64_t(gridDim.x) * blockDim.x) {
      kd[i] = ks[i];
      vd[i] = vs[i];
    }
  }
}

cudaError_t launch_copy_blocks(const CopyParams& p, int num_sms, cudaStream_t stream) {
  if (p.num_pairs == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t nvec = p.block_bytes / 16;
  int64_t bx = (nvec + threads - 1) / threads;
  if (bx > 16) bx = 16;
  int64_t by = p.num_pairs;
  const int64_t cap = int64_t(num_sms) * 16;   // enough CTAs to fill the GPU
  if (by * bx > cap) by = cap / bx > 0 ? cap / bx : 1;
  if (by > 65535) by = 65535;
  copy_blocks_kernel<<<dim3(unsigned(bx), unsigned(by)), threads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace pkv
