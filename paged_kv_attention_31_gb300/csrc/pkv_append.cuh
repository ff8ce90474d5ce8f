// pkv_append.cuh -- the scatter of new K/V rows into their pool slots, as a
// grid-stride device loop shared by kv_append_kernel and the fused
// plan-and-append launch of the decode step.
//
// "TensorRT-LLM框架解析与高性能推理优化实践" §4.2 (KV缓存管理细节): a growing
// sequence's tokens live in non-contiguous pages; the caller's page allocator
// gives each new token a slot = page * block_size + offset.  FP8 pools store
// the token quantised with a per-tensor or per-kv-head scale (§7.2 KV Cache量化).
//
// Thread i of the loop moves one 16-byte chunk (8 bf16) of one (token, kv
// head) row of K and of V: reads are fully coalesced, writes are 16 B (bf16)
// or 8 B (FP8) per thread into a contiguous head_dim run of the pool.
#pragma once

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

// Chunks first, first + stride, ... of the append; a slot < 0 is a padding
// token (skipped), a slot past the pool is recorded and skipped.
template <bool FP8>
__device__ __forceinline__ void append_rows(const AppendParams& p, int64_t first, int64_t stride) {
  const int chunks = p.head_dim / 8;  // 16-byte chunks per (token, head) row
  const int64_t per_tok = int64_t(p.num_kv_heads) * chunks;
  const int64_t total = int64_t(p.num_tokens) * per_tok;
  const uint4* kn = static_cast<const uint4*>(p.k_new);
  const uint4* vn = static_cast<const uint4*>(p.v_new);
  for (int64_t i = first; i < total; i += stride) {
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

}  // namespace pkv
