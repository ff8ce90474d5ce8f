// kv_append.cu -- scatter this step's new K/V rows into their pool slots.
//
// "TensorRT-LLM框架解析与高性能推理优化实践" §4.2 (KV缓存管理细节): a growing
// sequence's tokens live in non-contiguous pages; the caller's page allocator
// gives each new token a slot = page * block_size + offset.  FP8 pools store
// the token quantised with a per-tensor scale (§7.2 KV Cache量化).
//
// One thread moves one 16-byte chunk (8 bf16) of one (token, kv head) row of K
// and of V: reads are fully coalesced, writes are 16 B (bf16) or 8 B (FP8)
// per thread into a contiguous head_dim run of the pool.
#include "pkv_common.cuh"
#include "pkv_launch.h"

namespace pkv {

template <bool FP8>
__device__ __forceinline__ void store_row_chunk(uint8_t* pool, int64_t elem, uint4 x, float scale);

template <>
__device__ __forceinline__ void store_row_chunk<false>(uint8_t* pool, int64_t elem, uint4 x, float) {
  *reinterpret_cast<uint4*>(pool + elem * 2) = x;
}

// code = e4m3_rn_satfinite(x / scale); the quotient is an IEEE binary32
// division (round to nearest), so the code matches a host encoder exactly.
__device__ __forceinline__ uint16_t encode_pair(uint32_t w, float scale) {
  const float2 f = bf16x2_to_float2(w);
  const float2 y = make_float2(__fdiv_rn(f.x, scale), __fdiv_rn(f.y, scale));
  return static_cast<uint16_t>(__nv_cvt_float2_to_fp8x2(y, __NV_SATFINITE, __NV_E4M3));
}

template <>
__device__ __forceinline__ void store_row_chunk<true>(uint8_t* pool, int64_t elem, uint4 x,
                                                      float scale) {
  uint2 o;
  o.x = uint32_t(encode_pair(x.x, scale)) | (uint32_t(encode_pair(x.y, scale)) << 16);
  o.y = uint32_t(encode_pair(x.z, scale)) | (uint32_t(encode_pair(x.w, scale)) << 16);
  *reinterpret_cast<uint2*>(pool + elem) = o;
}

template <bool FP8>
__global__ void __launch_bounds__(256) kv_append_kernel(const AppendParams p) {
  pdl_launch_dependents();  // the next kernel may start its prologue now
  const int chunks = p.head_dim / 8;  // 16-byte chunks per (token, head) row
  const int64_t per_tok = int64_t(p.num_kv_heads) * chunks;
  const int64_t total = int64_t(p.num_tokens) * per_tok;
  const uint4* kn = static_cast<const uint4*>(p.k_new);
  const uint4* vn = static_cast<const uint4*>(p.v_new);
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t t = i / per_tok;
    const int64_t slot = __ldg(p.slot_mapping + t);
    if (slot < 0) continue;  // padding token
    const int64_t r = i - t * per_tok;
    if (slot >= p.num_slots) {
      if (r == 0) record_error(p.err, kDevBadPage);
      continue;
    }
    const int h = int(r / chunks);
    const int c = int(r - int64_t(h) * chunks);
    const int64_t page = slot / p.block_size;
    const int64_t off = slot - page * p.block_size;
    const int64_t elem = ((page * p.num_kv_heads + h) * p.block_size + off) * p.head_dim + c * 8;
    const uint4 kx = __ldg(kn + i);
    const uint4 vx = __ldg(vn + i);
    const float ks = (FP8 && p.k_scales) ? __ldg(p.k_scales + h) : p.k_scale;
    const float vs = (FP8 && p.v_scales) ? __ldg(p.v_scales + h) : p.v_scale;
    store_row_chunk<FP8>(static_cast<uint8_t*>(p.k_pool), elem, kx, ks);
    store_row_chunk<FP8>(static_cast<uint8_t*>(p.v_pool), elem, vx, vs);
  }
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
