// prefill.cu -- chunked-prefill attention over a paged KV cache with the
// 5th-generation tensor cores (tcgen05 + TMEM) and TMA (sm_103a).
//
// "TensorRT-LLM框架解析与高性能推理优化实践" §5.3 (分块上下文处理): a long prompt
// is processed as chunks interleaved with decode steps; each chunk's queries
// attend causally to everything before them in the sequence, whose K/V sit
// in pages (§4.2, §6.2).  §6.1 (Flash Attention实现): 64-128-token key tiles,
// running max / sum, partial results kept on chip.
//
// One CTA computes one 128-row query tile of one (sequence, kv head).  The
// 128 rows pack TQ = 128/G chunk tokens x the G q heads that share the kv
// head (row r = token (r / G), head g = r % G), so every K/V page is read
// once per kv head and the tile is a dense M = 128 contraction.
//
// Per key block of NK = 64 keys (NK / block_size pages):
//   TMA     each page (block_size rows x 128 B, one box per d-half) lands in a
//           128-byte-swizzled shared-memory tile; page ids come from the block
//           table; pages past the sequence use an out-of-range coordinate, so
//           TMA fills zeros.
//   S       tcgen05.mma kind::f16 (bf16 x bf16 -> fp32), M=128 N=64 K=128,
//           Q and K both K-major in shared memory, S accumulates in TMEM.
//   softmax each of the 128 threads owns one row (TMEM lane): tcgen05.ld the
//           64 scores, causal mask, running max kept with a lag of up to 2^8
//           (the O accumulator is rescaled only when the max grows by more
//           than that; the normalisation at the end uses the same max, so the
//           result is exact), P = 2^(s - m) rounded to bf16 into shared memory.
//   PV      tcgen05.mma M=128 N=128 K=64, P K-major, V MN-major (d contiguous),
//           O accumulates in TMEM.
// K/V use a two-stage ring with separate K and V barriers so the next K block
// loads while the current block's softmax and PV run.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "pkv_common.cuh"
#include "pkv_launch.h"

namespace pkv {
namespace {

constexpr int kD = 128;          // head_dim
constexpr int kM = 128;          // query rows per tile
constexpr int kNK = 64;          // keys per block
constexpr int kThreads = 128;
constexpr uint32_t kTmemCols = 256;  // S: cols [0, 64), O: cols [128, 256)
constexpr uint32_t kColS = 0, kColO = 128;

// shared memory layout (offsets from a 1024-aligned base)
constexpr int kQBytes = 2 * kM * 128;        // 32 KB: two d-halves of [128 rows][128 B]
constexpr int kKVStageBytes = 2 * kNK * 128; // 16 KB: two d-halves of [64 keys][128 B]
constexpr int kPBytes = kM * 128;            // 16 KB: [128 rows][64 keys bf16]
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQBytes;
constexpr int kOffV = kOffK + 2 * kKVStageBytes;
constexpr int kOffP = kOffV + 2 * kKVStageBytes;
constexpr int kOffBar = kOffP + kPBytes;     // barriers: q, k[2], v[2], s, o
constexpr int kOffMisc = kOffBar + 8 * 8;
// The 128-byte-swizzled tiles need a 1024-aligned base.  Dynamic shared memory
// starts at least 128-aligned, so at most 896 bytes of padding are needed;
// with that slack two CTAs fit in one SM's 228 KB.
constexpr int kMaxPad = 1024 - 128;
constexpr int kSmemBytes = kOffMisc + 16 + kMaxPad;

// ---- tcgen05 / TMA wrappers ------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, one elected thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` once all previously issued MMAs of this thread complete.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
  uint32_t r[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(v[i]);
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, int c3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (sm_100 family format:
// start >> 4 in bits 0-13, leading byte offset >> 4 in 16-29, stride byte
// offset >> 4 in 32-45, version 1 in 46-47, swizzle mode 2 = 128B in 61-63).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= uint64_t((saddr >> 4) & 0x3FFF);
  d |= uint64_t((lbo >> 4) & 0x3FFF) << 16;
  d |= uint64_t((sbo >> 4) & 0x3FFF) << 32;
  d |= uint64_t(1) << 46;
  d |= uint64_t(2) << 61;
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulate, bf16 A and B.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn_major ? (1u << 16) : 0u) |
         (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

__global__ void __launch_bounds__(kThreads, 2)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
  const int mt = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
  const int G = p.num_q_heads / p.num_kv_heads;
  const int TQ = kM / G;
  const int q0 = __ldg(p.cu_seqlens_q + s);
  const int C = __ldg(p.cu_seqlens_q + s + 1) - q0;
  if (C <= 0 || mt * TQ >= C) return;
  const int L = __ldg(p.context_lens + s);
  const int P = p.block_size;
  if (L < C || L > p.max_blocks * P) {
    if (threadIdx.x == 0) record_error(p.err, kDevBadPage);
    return;
  }

  extern __shared__ __align__(128) uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  if (pad > uint32_t(kMaxPad)) {  // cannot happen with a 128-aligned base; never index past the end
    if (threadIdx.x == 0) record_error(p.err, kDevBadPage);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sK = smem + kOffK;
  uint8_t* sV = smem + kOffV;
  uint8_t* sP = smem + kOffP;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* bar_q = bar + 0;
  uint64_t* bar_k = bar + 1;  // [2]
  uint64_t* bar_v = bar + 3;  // [2]
  uint64_t* bar_s = bar + 5;
  uint64_t* bar_o = bar + 6;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int tok0 = mt * TQ;                      // first chunk token of the tile
  const int ntok = min(TQ, C - tok0);
  const int minpos = L - C + tok0;               // position of the tile's first token
  const int maxpos = L - C + tok0 + ntok - 1;    // position of its last token
  const int nblk = maxpos / kNK + 1;             // key blocks 0 .. nblk-1
  const int npages = (L + P - 1) / P;
  const int pages_per_blk = kNK / P;

  if (tid == 0) {
    mbar_init(bar_q, 1);
    mbar_init(&bar_k[0], 1);
    mbar_init(&bar_k[1], 1);
    mbar_init(&bar_v[0], 1);
    mbar_init(&bar_v[1], 1);
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = uint32_t(warp * 32) << 16;

  // page id of logical page j, or an out-of-range id (TMA fills zeros)
  auto page_of = [&](int j) -> int {
    if (j >= npages) return p.num_blocks;
    int pid = __ldg(p.block_tables + size_t(s) * p.max_blocks + j);
    if (pid < 0 || pid >= p.num_blocks) {
      record_error(p.err, kDevBadPage);
      pid = p.num_blocks;
    }
    return pid;
  };
  auto load_kv = [&](const CUtensorMap* map, uint8_t* base, uint64_t* b, int blk) {
    mbar_arrive_expect_tx(b, kKVStageBytes);
    for (int i = 0; i < pages_per_blk; ++i) {
      const int pid = page_of(blk * pages_per_blk + i);
#pragma unroll
      for (int dh = 0; dh < 2; ++dh)
        tma_load_4d(base + dh * (kNK * 128) + i * P * 128, map, dh * 64, 0, h, pid, b);
    }
  };

  if (tid == 0) {
    mbar_arrive_expect_tx(bar_q, kQBytes);
#pragma unroll
    for (int dh = 0; dh < 2; ++dh) tma_load_4d(sQ + dh * (kM * 128), &tm_q, dh * 64, 0, h, q0 + tok0, bar_q);
    load_kv(&tm_k, sK, &bar_k[0], 0);
    load_kv(&tm_v, sV, &bar_v[0], 0);
    if (nblk > 1) {
      load_kv(&tm_k, sK + kKVStageBytes, &bar_k[1], 1);
      load_kv(&tm_v, sV + kKVStageBytes, &bar_v[1], 1);
    }
  }

  // this thread's query row
  const int row = tid;
  const int tok = tok0 + row / G;
  const bool row_valid = (row / G) < ntok;
  const int pos = row_valid ? L - C + tok : -1;  // keys 0 .. pos are visible
  float m_used = -INFINITY, l_sum = 0.f;
  const float qm = p.q_mult;
  constexpr uint32_t kIdescS = idesc_bf16(kM, kNK, false);
  constexpr uint32_t kIdescO = idesc_bf16(kM, kD, true);

  for (int j = 0; j < nblk; ++j) {
    const int st = j & 1;
    const uint32_t use_par = uint32_t(j >> 1) & 1;
    // ---- S = Q K^T ---------------------------------------------------------------
    if (tid == 0) {
      if (j == 0) mbar_wait_bounded(bar_q, 0, p.err);
      mbar_wait_bounded(&bar_k[st], use_par, p.err);
      tc_fence_after();
      const uint32_t qa = smem_u32(sQ), ka = smem_u32(sK + st * kKVStageBytes);
#pragma unroll
      for (int ks = 0; ks < kD / 16; ++ks) {
        const int dh = ks >> 2, w = ks & 3;
        const uint64_t ad = sw128_desc(qa + dh * (kM * 128) + w * 32, 16, 1024);
        const uint64_t bd = sw128_desc(ka + dh * (kNK * 128) + w * 32, 16, 1024);
        mma_bf16(tmem + kColS, ad, bd, kIdescS, ks > 0);
      }
      mma_commit(bar_s);
      // K of block j-1 was consumed by S_{j-1} (complete): refill its stage
      if (j >= 1 && j + 1 < nblk) load_kv(&tm_k, sK + ((j + 1) & 1) * kKVStageBytes, &bar_k[(j + 1) & 1], j + 1);
    }
    mbar_wait_bounded(bar_s, uint32_t(j) & 1, p.err);
    tc_fence_after();

    // ---- scores of this row --------------------------------------------------------
    float sv[kNK];
    tmem_ld32(tmem + lane_base + kColS, sv);
    tmem_ld32(tmem + lane_base + kColS + 32, sv + 32);
    const int kbase = j * kNK;
    float mx = -INFINITY;
    if (kbase + kNK - 1 <= minpos) {       // block fully visible to every valid row
#pragma unroll
      for (int c = 0; c < kNK; ++c) {
        sv[c] = row_valid ? sv[c] * qm : -INFINITY;
        mx = fmaxf(mx, sv[c]);
      }
    } else {
#pragma unroll
      for (int c = 0; c < kNK; ++c) {
        sv[c] = (kbase + c <= pos) ? sv[c] * qm : -INFINITY;
        mx = fmaxf(mx, sv[c]);
      }
    }
    // lagged running max: move it only when the block max exceeds it by > 8
    float alpha = 1.f;
    if (mx > m_used + 8.f || (m_used == -INFINITY && mx != -INFINITY)) {
      alpha = fast_exp2(m_used - mx);    // 0 when m_used = -inf
      m_used = mx;
      l_sum *= alpha;
    }

    // PV_{j-1} must be done before P is overwritten and O is rescaled
    if (j > 0) {
      mbar_wait_bounded(bar_o, uint32_t(j - 1) & 1, p.err);
      tc_fence_after();
      if (tid == 0 && j + 1 < nblk)
        load_kv(&tm_v, sV + ((j + 1) & 1) * kKVStageBytes, &bar_v[(j + 1) & 1], j + 1);
      // tcgen05.ld/st are warp-collective: rescale if any row of the warp needs
      // it (rows that do not have alpha == 1)
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int cc = 0; cc < kD; cc += 32) {
          float o[32];
          tmem_ld32(tmem + lane_base + kColO + cc, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(tmem + lane_base + kColO + cc, o);
        }
      }
    }

    // ---- P = 2^(s - m) in bf16, swizzled K-major rows of 128 B ----------------------
    float psum = 0.f;
    uint8_t* prow = sP + row * 128;
#pragma unroll
    for (int c8 = 0; c8 < kNK / 8; ++c8) {
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float a = m_used == -INFINITY ? 0.f : fast_exp2(sv[c8 * 8 + 2 * i] - m_used);
        const float b = m_used == -INFINITY ? 0.f : fast_exp2(sv[c8 * 8 + 2 * i + 1] - m_used);
        const __nv_bfloat162 pb = __floats2bfloat162_rn(a, b);
        const float2 back = __bfloat1622float2(pb);
        psum += back.x + back.y;
        w[i] = *reinterpret_cast<const uint32_t*>(&pb);
      }
      *reinterpret_cast<uint4*>(prow + ((c8 ^ (row & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    l_sum += psum;

    // V rows past the sequence end may hold anything (never-written slots):
    // zero them so 0 * V stays 0 in the PV product
    if (kbase + kNK > L) {
      mbar_wait_bounded(&bar_v[st], use_par, p.err);
      const int first = max(0, L - kbase);
      for (int i = tid; i < (kNK - first) * 2 * 8; i += kThreads) {
        const int r = first + (i >> 4), rest = i & 15;
        const int dh = rest >> 3, chunk = rest & 7;
        *reinterpret_cast<uint4*>(sV + st * kKVStageBytes + dh * (kNK * 128) + r * 128 + chunk * 16) =
            make_uint4(0, 0, 0, 0);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- O += P V ---------------------------------------------------------------------
    if (tid == 0) {
      mbar_wait_bounded(&bar_v[st], use_par, p.err);
      tc_fence_after();
      const uint32_t pa = smem_u32(sP), va = smem_u32(sV + st * kKVStageBytes);
#pragma unroll
      for (int ks = 0; ks < kNK / 16; ++ks) {
        const uint64_t ad = sw128_desc(pa + ks * 32, 16, 1024);
        const uint64_t bd = sw128_desc(va + ks * 2048, kNK * 128, 1024);
        mma_bf16(tmem + kColO, ad, bd, kIdescO, (j > 0 || ks > 0) ? 1u : 0u);
      }
      mma_commit(bar_o);
    }
  }

  // ---- epilogue: O / l -> bf16 -------------------------------------------------------
  mbar_wait_bounded(bar_o, uint32_t(nblk - 1) & 1, p.err);
  tc_fence_after();
  const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
  __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) +
                       (size_t(q0 + tok) * p.num_q_heads + size_t(h) * G + (row % G)) * kD;
#pragma unroll
  for (int cc = 0; cc < kD; cc += 32) {
    float o[32];
    tmem_ld32(tmem + lane_base + kColO + cc, o);
    if (row_valid) {
#pragma unroll
      for (int i = 0; i < 32; i += 8) {
        uint4 u;
        __nv_bfloat162 b0 = __floats2bfloat162_rn(o[i] * inv, o[i + 1] * inv);
        __nv_bfloat162 b1 = __floats2bfloat162_rn(o[i + 2] * inv, o[i + 3] * inv);
        __nv_bfloat162 b2 = __floats2bfloat162_rn(o[i + 4] * inv, o[i + 5] * inv);
        __nv_bfloat162 b3 = __floats2bfloat162_rn(o[i + 6] * inv, o[i + 7] * inv);
        u.x = *reinterpret_cast<uint32_t*>(&b0);
        u.y = *reinterpret_cast<uint32_t*>(&b1);
        u.z = *reinterpret_cast<uint32_t*>(&b2);
        u.w = *reinterpret_cast<uint32_t*>(&b3);
        *reinterpret_cast<uint4*>(dst + cc + i) = u;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ---- host: tensor maps ------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 4-D bf16 map: dims (inner first) d0..d3, row strides in bytes for d1..d3.
bool make_map(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
              uint64_t d3, uint64_t s1, uint64_t s2, uint64_t s3, uint32_t b0, uint32_t b1,
              uint32_t b2, uint32_t b3) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {d0, d1, d2, d3};
  const cuuint64_t strides[3] = {s1, s2, s3};
  const cuuint32_t box[4] = {b0, b1, b2, b3};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams& p, const void* k_pool, const void* v_pool,
                           int num_sms, cudaStream_t stream) {
  (void)num_sms;
  if (p.head_dim != kD) return cudaErrorNotSupported;
  const int G = p.num_q_heads / p.num_kv_heads;
  if (G < 1 || kM % G != 0 || kNK % p.block_size != 0) return cudaErrorNotSupported;
  if (p.num_blocks >= (1 << 30)) return cudaErrorInvalidValue;
  const uint64_t D = kD, P = p.block_size, Hkv = p.num_kv_heads, E = 2;
  CUtensorMap tq, tk, tv;
  // q [T][Hkv][G][D] with box (64, G, 1, 128/G): rows ordered token-major, head-minor
  if (!make_map(&tq, p.q, D, G, Hkv, uint64_t(p.num_q_tokens), D * E, G * D * E, Hkv * G * D * E,
                64, uint32_t(G), 1, uint32_t(kM / G)))
    return cudaErrorInvalidValue;
  // pools [nb][Hkv][P][D] with box (64, P, 1, 1): one page of one kv head
  if (!make_map(&tk, k_pool, D, P, Hkv, uint64_t(p.num_blocks), D * E, P * D * E, Hkv * P * D * E,
                64, uint32_t(P), 1, 1))
    return cudaErrorInvalidValue;
  if (!make_map(&tv, v_pool, D, P, Hkv, uint64_t(p.num_blocks), D * E, P * D * E, Hkv * P * D * E,
                64, uint32_t(P), 1, 1))
    return cudaErrorInvalidValue;
  static bool configured[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  dim3 grid(p.tiles_per_seq, p.num_kv_heads, p.num_seqs);
  if (grid.z > 65535) return cudaErrorInvalidValue;
  prefill_kernel<<<grid, kThreads, kSmemBytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace pkv
