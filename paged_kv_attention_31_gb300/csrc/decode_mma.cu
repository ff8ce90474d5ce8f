// decode_mma.cu -- paged decode attention with 4 or 8 q heads per kv head
// (head_dim 128, bf16 or FP8 E4M3 KV) on warp-level tensor-core MMAs
// (sm_103a).
//
// Same computation, work decomposition, split plan and merge as decode.cu
// ("TensorRT-LLM框架解析与高性能推理优化实践" §6.2 paged attention, §6.1 running
// max / sum, §7.2 KV quantised and dequantised inside the kernel).  With G
// packed q heads a kv head's token costs 2G multiply-adds per element (QK and
// PV), which the CUDA cores cannot sustain at HBM speed for G >= 4 (and for
// FP8 not at all); here each warp does the per-tile contractions with
// mma.sync m16n8k16 with fp32 accumulation: bf16 x bf16 for bf16 KV, and
// f16 x f16 for FP8 KV with the E4M3 codes converted to f16 (exactly) in
// registers and each head's q scaled by a power of two into f16's range
// (exact; the scores are scaled back).
//
// Per 16-token tile (one warp, lane = 4 r + c):
//   QK  S^T[16 tokens x 8 heads] = K[16 x 128] q^T: M = tokens, N = heads
//       (padded to 8), K = head_dim in 8 steps of 16.  The reduction index is
//       permuted consistently in A (K) and B (q): step s of lane c covers 4
//       head_dim values of a fixed per-lane set (FP8: 32c .. 32c + 31; bf16:
//       16c .. 16c + 15 and 64 + 16c .. 64 + 16c + 15), so each lane reads
//       its share of rows r and r + 8 with 16-byte loads.
//   softmax per head over the 16 tokens: the scores of head 2c + {0,1} sit in
//       the 8 lanes with the same c (xor-4/8/16 butterflies); running max and
//       sum in the log2 domain; P rounded to the MMA's type (bf16 for bf16
//       KV, f16 for FP8 KV; the running max is exact, so P <= 1), the row
//       sum taken over the unrounded fp32 values.
//   PV  O^T[128 x 8] += V^T[128 x 16 tokens] P^T: M = head_dim (8 tiles of
//       16), N = heads, K = tokens.  The M index is permuted so that lane r
//       owns 16 head_dim values (FP8: 16r .. 16r + 15; bf16: two 8-value
//       chunks of one half row); its V elements of tokens 2c, 2c+1, 2c+8,
//       2c+9 come from 16-byte loads and are interleaved pairwise with byte
//       permutes (FP8: then converted two at a time).  P's B fragment is the
//       S accumulator transposed 8x8 at a time with movmatrix.
// K/V tiles (16 rows, 128-byte boxes) arrive by 2-D TMA with 128-byte swizzle
// into a per-warp 2-stage ring; the swizzle makes both the row reads (QK) and
// the column reads (PV) free of shared-memory bank conflicts.
#include "pkv_common.cuh"
#include "pkv_launch.h"
#include "pkv_tmap.h"

namespace pkv {
namespace {

constexpr int kD = 128;        // head_dim
constexpr int kTT = 16;        // tokens per tile
constexpr int kNW = 4;         // warps per CTA
#ifndef PKV_MMA_STAGES
#define PKV_MMA_STAGES 2
#endif
constexpr int kST = PKV_MMA_STAGES;  // ring stages per warp
constexpr int kN = 8;          // MMA N: packed q heads (padded)
constexpr int kBox = kTT * 128;  // one TMA box: 16 rows x 128 B

// shared memory layout (offsets from a 1024-aligned base)
template <bool FP8>
struct MmaCfg {
  static constexpr int TB = kTT * kD * (FP8 ? 1 : 2);        // bytes of a K (or V) tile
  static constexpr int BOXES = TB / kBox;                    // 1 (FP8) or 2 (bf16 halves)
  static constexpr int OFF_K = 0;                            // [NW][ST] K tiles
  static constexpr int OFF_V = OFF_K + kNW * kST * TB;       // [NW][ST] V tiles
  static constexpr int OFF_CM = OFF_V + kNW * kST * TB;      // float2 [NW][8] (m, l)
  static constexpr int OFF_BAR = OFF_CM + kNW * kN * 8;      // u64 [NW][ST]
  static constexpr int OFF_MISC = OFF_BAR + kNW * kST * 8;   // int [4]
  static constexpr int OFF_PG = OFF_MISC + 16;               // int [pages of a unit]
  // the warp-combine buffer float [NW][8][128] reuses the K ring, which is
  // idle between units
  static_assert(kNW * kST * TB >= kNW * kN * kD * 4, "combine buffer must fit the K ring");
};

template <bool FP8>
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (FP8) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

// Transpose of an 8x8 b16 matrix held one row pair per lane.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// Four E4M3 codes (bytes 0..3 of w) -> f16x2 (b0, b1) and (b2, b3), exact;
// the lower byte of each pair lands in the lower half.  One cvt per pair, no
// repacking.
__device__ __forceinline__ void e4m3x4_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\t"
      "mov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// Two floats -> the MMA's 16-bit pair type (f16 for FP8 KV, bf16 otherwise).
template <bool FP8>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (FP8) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  } else {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
}

__device__ __forceinline__ uint4 lds128(const uint8_t* p) {
  return *reinterpret_cast<const uint4*>(p);
}

// 16-byte chunk `chunk` of row `row` in a 128-byte-swizzled 16 x 128 B box
__device__ __forceinline__ const uint8_t* swz(const uint8_t* box, int row, int chunk) {
  return box + row * 128 + ((chunk ^ (row & 7)) << 4);
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

__device__ __forceinline__ int unit_len(int L, int cap, int32_t* err) {
  if (L < 0 || L > cap) {
    record_error(err, kDevBadPage);
    return L < 0 ? 0 : cap;
  }
  return L;
}

template <int G, bool FP8>
__global__ void __launch_bounds__(kNW * 32)
    decode_mma_kernel(const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
  static_assert(G == 4 || G == 8, "4 or 8 q heads per kv head");
  using C = MmaCfg<FP8>;
  constexpr int TB = C::TB;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, c = lane & 3;
  uint8_t* const kbuf = smem + C::OFF_K + warp * kST * TB;
  uint8_t* const vbuf = smem + C::OFF_V + warp * kST * TB;
  float2* const cm = reinterpret_cast<float2*>(smem + C::OFF_CM);
  float* const ca = reinterpret_cast<float*>(smem + C::OFF_K);
  uint64_t* const bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR) + warp * kST;
  int* const misc = reinterpret_cast<int*>(smem + C::OFF_MISC);
  int* const pages = reinterpret_cast<int*>(smem + C::OFF_PG);
  volatile int* const abort_flag = misc + 2;

  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < kST; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  pdl_wait();  // planner output and this step's appends are visible
  if (threadIdx.x == 0) {
    misc[0] = atomicAdd(p.counters + 1, 1);
    misc[2] = 0;
  }
  __syncthreads();

  const int Hkv = p.num_kv_heads, P = p.block_size;
  const int n_units = p.counters[0] * Hkv;
  uint32_t jt = 0;            // tiles this warp has consumed
  int unit = misc[0];
  // bf16 PV: lane r owns chunks (r & 3) and (r & 3) + 4 of half (r >> 2)
  const int pv_half = r >> 2, pv_chunk = r & 3;

  while (unit < n_units) {
    int next = 0;
    if (threadIdx.x == 0) next = atomicAdd(p.counters + 1, 1);
    const int2 item = p.items[unit / Hkv];
    const int h = unit - (unit / Hkv) * Hkv;
    const int s = item.x, k = item.y;
    const int L = unit_len(__ldg(p.context_lens + s), p.max_len, p.err);
    const int ns = decode_num_splits(L, p.partition);
    const int t0 = ns == 1 ? 0 : k * p.partition;
    const int t1 = ns == 1 ? L : min(L, t0 + p.partition);
    const int pg0 = t0 / P;
    const int npg = (t1 - t0 + P - 1) / P;
    // score multiplier scale * k_scale * log2(e) and output multiplier v_scale,
    // with the kv head's scales when per-head scales are given
    const float qm = p.k_scales ? p.q_mult * __ldg(p.k_scales + h) : p.q_mult;
    const float vm = p.v_scales ? p.v_mult * __ldg(p.v_scales + h) : p.v_mult;
    for (int i = threadIdx.x; i < npg; i += kNW * 32) {
      int pid = __ldg(p.block_tables + size_t(s) * p.max_blocks + pg0 + i);
      if (pid < 0 || pid >= p.num_blocks) {
        record_error(p.err, kDevBadPage);
        pid = -1;
      }
      pages[i] = pid;
    }
    // B fragments of q for the 8 reduction steps (head g = r, zero past G):
    // qb[2s] holds the first, qb[2s+1] the second pair of step s
    uint32_t qb[16];
    // FP8: the unscale factors 2^-k of heads 2c and 2c + 1 (see below)
    float q_unscale[2] = {1.f, 1.f};
    {
      const int g = r;
      if constexpr (FP8) {
        // head_dim 32c .. 32c + 31 of head g, as f16.  f16 holds every bf16
        // value of magnitude 2^-14 .. 65280 exactly but not the rest of
        // bf16's range, so each head's q is first multiplied by an exact
        // power of two 2^k that puts its largest |q| in [2^15, 2^16); the
        // scores of that head are multiplied by 2^-k afterwards.  Elements
        // more than 2^29 below the head's largest stay within f16's normal
        // range; smaller ones round to f16 subnormals, far below the fp32
        // accumulation error of the dot product.
        uint4 u[4] = {};
        float amax = 0.f;
        if (g < G) {
          const uint4* src = reinterpret_cast<const uint4*>(
              static_cast<const __nv_bfloat16*>(p.q) +
              (size_t(s) * p.num_q_heads + size_t(h) * G + g) * kD + 32 * c);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            u[i] = __ldg(src + i);
            const uint32_t w[4] = {u[i].x, u[i].y, u[i].z, u[i].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float2 f = bf16x2_to_float2(w[j]);
              amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
          }
        }
        // the 4 lanes of head g (lane = 4g + c) hold its 128 elements
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        // k = 15 - floor(log2 amax), clamped to [-126, 126] so that 2^k and
        // 2^-k are normal floats (a head whose largest |q| is an fp32
        // subnormal ends up below 2^15, still inside f16's range); an
        // all-zero head keeps k = 0
        const int e = int((__float_as_uint(amax) >> 23) & 0xFF) - 127;  // -127 if subnormal
        const int k = amax > 0.f ? max(-126, min(126, 15 - e)) : 0;
        const float up = __uint_as_float(uint32_t(127 + k) << 23);
        const float down = __uint_as_float(uint32_t(127 - k) << 23);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t w[4] = {u[i].x, u[i].y, u[i].z, u[i].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 f = bf16x2_to_float2(w[j]);
            qb[4 * i + j] = pack2<true>(f.x * up, f.y * up);  // exact products
          }
        }
        // heads 2c and 2c + 1 own this lane's score columns
        q_unscale[0] = __shfl_sync(0xffffffffu, down, 4 * (2 * c));
        q_unscale[1] = __shfl_sync(0xffffffffu, down, 4 * (2 * c + 1));
      } else if (g < G) {
        const __nv_bfloat16* qrow =
            static_cast<const __nv_bfloat16*>(p.q) + (size_t(s) * p.num_q_heads + size_t(h) * G + g) * kD;
        {  // head_dim 16c .. 16c + 15 and 64 + 16c .. 64 + 16c + 15, as is
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const uint4* src = reinterpret_cast<const uint4*>(qrow + 64 * hf + 16 * c);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const uint4 u = __ldg(src + i);
              qb[8 * hf + 4 * i] = u.x;
              qb[8 * hf + 4 * i + 1] = u.y;
              qb[8 * hf + 4 * i + 2] = u.z;
              qb[8 * hf + 4 * i + 3] = u.w;
            }
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) qb[i] = 0u;
      }
    }
    __syncthreads();  // pages[] visible; the combine buffer (K ring) is free

    const int ntile = (t1 - t0 + kTT - 1) / kTT;
    const int my_n = warp < ntile ? (ntile - warp + kNW - 1) / kNW : 0;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};  // heads 2c, 2c+1
    float o[8][4];  // O^T m-tile i: rows (this lane's head_dim) x heads 2c, 2c+1
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[i][e] = 0.f;

    auto issue = [&](int j) {  // lane 0: TMA of this warp's j-th tile of the unit
      const int stage = int((jt + j) % kST);
      const int ts = t0 + (warp + j * kNW) * kTT;
      int pid = pages[ts / P - pg0];
      if (pid < 0) pid = p.num_blocks;  // out of range: zero fill, tile masked
      mbar_arrive_expect_tx(&bars[stage], 2 * TB);
#pragma unroll
      for (int b = 0; b < C::BOXES; ++b) {
        tma_load_4d(kbuf + stage * TB + b * kBox, &tm_k, 64 * b, ts % P, h, pid, &bars[stage]);
        tma_load_4d(vbuf + stage * TB + b * kBox, &tm_v, 64 * b, ts % P, h, pid, &bars[stage]);
      }
    };
    if (lane == 0) {
      fence_proxy_async_smem();  // the K ring was just read as the combine buffer
      for (int j = 0; j < min(kST, my_n); ++j) issue(j);
    }

    for (int j = 0; j < my_n; ++j) {
      const int stage = int((jt + j) % kST);
      const uint32_t parity = ((jt + j) / kST) & 1;
      const int ts = t0 + (warp + j * kNW) * kTT;
      const int ntok = pages[ts / P - pg0] < 0 ? 0 : min(kTT, t1 - ts);
      if (!warp_wait_bounded(&bars[stage], parity, p.err, abort_flag)) {
        // a wait gave up: compute nothing more; let this warp's copies in
        // flight (tiles j .. j + kST - 1) land before the CTA leaves
        if (lane == 0)
          for (int jj = j; jj < min(j + kST, my_n); ++jj)
            mbar_drain_wait(&bars[(jt + jj) % kST], ((jt + jj) / kST) & 1, p.err);
        __syncwarp();
        break;
      }
      const uint8_t* kt = kbuf + stage * TB;
      const uint8_t* vt = vbuf + stage * TB;

      // ---- S^T = K q^T (two independent accumulator chains) ------------------------
      float sacc[4] = {0.f, 0.f, 0.f, 0.f}, sacc2[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (FP8) {
        const uint4 ka = lds128(swz(kt, r, 2 * c)), kb = lds128(swz(kt, r, 2 * c + 1));
        const uint4 la = lds128(swz(kt, r + 8, 2 * c)), lb = lds128(swz(kt, r + 8, 2 * c + 1));
        const uint32_t wr[8] = {ka.x, ka.y, ka.z, ka.w, kb.x, kb.y, kb.z, kb.w};
        const uint32_t w8[8] = {la.x, la.y, la.z, la.w, lb.x, lb.y, lb.z, lb.w};
#pragma unroll
        for (int st = 0; st < 8; ++st) {
          uint32_t a0, a1, a2, a3;  // rows r / r+8, head_dim 32c + 4st + {0,1} / {2,3}
          e4m3x4_f16x2(wr[st], a0, a2);
          e4m3x4_f16x2(w8[st], a1, a3);
          mma_16816<true>((st & 1) ? sacc2 : sacc, a0, a1, a2, a3, qb[2 * st], qb[2 * st + 1]);
        }
      } else {
        uint32_t wr[16], w8[16];  // rows r / r+8: chunks 2c, 2c+1 of both halves
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const uint4 u = lds128(swz(kt + hf * kBox, r, 2 * c + q));
            const uint4 v = lds128(swz(kt + hf * kBox, r + 8, 2 * c + q));
            const int o4 = 8 * hf + 4 * q;
            wr[o4] = u.x; wr[o4 + 1] = u.y; wr[o4 + 2] = u.z; wr[o4 + 3] = u.w;
            w8[o4] = v.x; w8[o4 + 1] = v.y; w8[o4 + 2] = v.z; w8[o4 + 3] = v.w;
          }
#pragma unroll
        for (int st = 0; st < 8; ++st)
          mma_16816<false>((st & 1) ? sacc2 : sacc, wr[2 * st], w8[2 * st], wr[2 * st + 1],
                           w8[2 * st + 1], qb[2 * st], qb[2 * st + 1]);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[e] += sacc2[e];
      // sacc: [0] token r head 2c, [1] token r head 2c+1, [2] token r+8 head 2c,
      // [3] token r+8 head 2c+1
      const bool v0 = r < ntok, v1 = r + 8 < ntok;
      if constexpr (FP8) {  // back from each head's 2^k-scaled q
        sacc[0] *= q_unscale[0];
        sacc[1] *= q_unscale[1];
        sacc[2] *= q_unscale[0];
        sacc[3] *= q_unscale[1];
      }
      float sv[4] = {v0 ? sacc[0] * qm : -INFINITY, v0 ? sacc[1] * qm : -INFINITY,
                     v1 ? sacc[2] * qm : -INFINITY, v1 ? sacc[3] * qm : -INFINITY};

      // ---- online softmax per head over the tile's 16 tokens ----------------------
      float pv[4];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float mx = fmaxf(sv[hh], sv[hh + 2]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float m_new = fmaxf(m_run[hh], mx);
        float alpha = 1.f, p0 = 0.f, p1 = 0.f;
        if (m_new != -INFINITY) {
          alpha = fast_exp2(m_run[hh] - m_new);
          p0 = fast_exp2(sv[hh] - m_new);
          p1 = fast_exp2(sv[hh + 2] - m_new);
        }
        float sum = p0 + p1;
        sum += __shfl_xor_sync(0xffffffffu, sum, 4);
        sum += __shfl_xor_sync(0xffffffffu, sum, 8);
        sum += __shfl_xor_sync(0xffffffffu, sum, 16);
        l_run[hh] = l_run[hh] * alpha + sum;
        m_run[hh] = m_new;
        pv[hh] = p0;
        pv[hh + 2] = p1;
        if (alpha != 1.f) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            o[i][hh] *= alpha;
            o[i][hh + 2] *= alpha;
          }
        }
      }
      // B fragments of P^T: the accumulator rows (tokens) r / r+8 transposed
      const uint32_t pb0 = movmatrix_trans(pack2<FP8>(pv[0], pv[1]));
      const uint32_t pb1 = movmatrix_trans(pack2<FP8>(pv[2], pv[3]));

      // ---- O^T += V^T P^T -----------------------------------------------------------
      if constexpr (FP8) {
        uint4 x0 = lds128(swz(vt, 2 * c, r)), x1 = lds128(swz(vt, 2 * c + 1, r));
        uint4 y0 = lds128(swz(vt, 2 * c + 8, r)), y1 = lds128(swz(vt, 2 * c + 9, r));
        if (ntok < kTT) {  // rows past the tile end: zero (never-written slots may hold NaN)
          const uint4 z = make_uint4(0, 0, 0, 0);
          if (2 * c >= ntok) x0 = z;
          if (2 * c + 1 >= ntok) x1 = z;
          if (2 * c + 8 >= ntok) y0 = z;
          if (2 * c + 9 >= ntok) y1 = z;
        }
        const uint32_t X0[4] = {x0.x, x0.y, x0.z, x0.w}, X1[4] = {x1.x, x1.y, x1.z, x1.w};
        const uint32_t Y0[4] = {y0.x, y0.y, y0.z, y0.w}, Y1[4] = {y1.x, y1.y, y1.z, y1.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          // bytes 4q..4q+3 of each row = head_dim 16r + 4q .. + 3 = m-tiles 2q, 2q+1
          const uint32_t e = __byte_perm(X0[q], X1[q], 0x5140);
          const uint32_t f = __byte_perm(X0[q], X1[q], 0x7362);
          const uint32_t ey = __byte_perm(Y0[q], Y1[q], 0x5140);
          const uint32_t fy = __byte_perm(Y0[q], Y1[q], 0x7362);
          uint32_t a0, a1, a2, a3;
          e4m3x4_f16x2(e, a0, a1);
          e4m3x4_f16x2(ey, a2, a3);
          mma_16816<true>(o[2 * q], a0, a1, a2, a3, pb0, pb1);
          e4m3x4_f16x2(f, a0, a1);
          e4m3x4_f16x2(fy, a2, a3);
          mma_16816<true>(o[2 * q + 1], a0, a1, a2, a3, pb0, pb1);
        }
      } else {
        // tokens 2c, 2c+1, 2c+8, 2c+9: chunks pv_chunk and pv_chunk + 4 of half pv_half
        uint32_t X0[8], X1[8], Y0[8], Y1[8];
        const uint8_t* vh = vt + pv_half * kBox;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const uint4 a = lds128(swz(vh, 2 * c, pv_chunk + 4 * q));
          const uint4 b = lds128(swz(vh, 2 * c + 1, pv_chunk + 4 * q));
          const uint4 cc = lds128(swz(vh, 2 * c + 8, pv_chunk + 4 * q));
          const uint4 dd = lds128(swz(vh, 2 * c + 9, pv_chunk + 4 * q));
          X0[4 * q] = a.x; X0[4 * q + 1] = a.y; X0[4 * q + 2] = a.z; X0[4 * q + 3] = a.w;
          X1[4 * q] = b.x; X1[4 * q + 1] = b.y; X1[4 * q + 2] = b.z; X1[4 * q + 3] = b.w;
          Y0[4 * q] = cc.x; Y0[4 * q + 1] = cc.y; Y0[4 * q + 2] = cc.z; Y0[4 * q + 3] = cc.w;
          Y1[4 * q] = dd.x; Y1[4 * q + 1] = dd.y; Y1[4 * q + 2] = dd.z; Y1[4 * q + 3] = dd.w;
        }
        if (ntok < kTT) {  // rows past the tile end: zero (never-written slots may hold NaN)
          const bool zx0 = 2 * c >= ntok, zx1 = 2 * c + 1 >= ntok;
          const bool zy0 = 2 * c + 8 >= ntok, zy1 = 2 * c + 9 >= ntok;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (zx0) X0[i] = 0u;
            if (zx1) X1[i] = 0u;
            if (zy0) Y0[i] = 0u;
            if (zy1) Y1[i] = 0u;
          }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)  // word i = head_dim pair (d, d+1) = m-tile i rows r / r+8
          mma_16816<false>(o[i], __byte_perm(X0[i], X1[i], 0x5410), __byte_perm(X0[i], X1[i], 0x7632),
                           __byte_perm(Y0[i], Y1[i], 0x5410), __byte_perm(Y0[i], Y1[i], 0x7632),
                           pb0, pb1);
      }
      __syncwarp();
      if (lane == 0 && j + kST < my_n) {
        fence_proxy_async_smem();
        issue(j + kST);
      }
    }
    jt += uint32_t(my_n);

    // ---- combine the warps ---------------------------------------------------------
    __syncthreads();  // every warp is done with its tiles: the K ring becomes `ca`
    if (r == 0) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
        if (2 * c + hh < G) cm[warp * G + 2 * c + hh] = make_float2(m_run[hh], l_run[hh]);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int g = 2 * c + (e & 1);
        // head_dim of m-tile i, row r (+8 for e >= 2)
        const int d = FP8 ? 16 * r + 2 * i + (e >> 1)
                          : 64 * pv_half + 8 * pv_chunk + 32 * (i >> 2) + 2 * (i & 3) + (e >> 1);
        if (g < G) ca[(warp * G + g) * kD + d] = o[i][e];
      }
    if (threadIdx.x == 0) misc[1] = next;
    __syncthreads();
    const int next_unit = misc[1];
    // The abort flag changes only inside the tile loops: between the
    // barrier above and the next unit's first barrier every thread reads the
    // same value.  After an abort the unit's results are not written and the
    // CTA takes no further work.
    const bool aborted = *abort_flag != 0;
    for (int idx = threadIdx.x; idx < G * kD && !aborted; idx += kNW * 32) {
      const int g = idx / kD, d = idx - g * kD;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kNW; ++w) M = fmaxf(M, cm[w * G + g].x);
      float lsum = 0.f, a = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kNW; ++w) {
          const float2 ml = cm[w * G + g];
          const float sw = fast_exp2(ml.x - M);
          lsum = fmaf(sw, ml.y, lsum);
          a = fmaf(sw, ca[(w * G + g) * kD + d], a);
        }
      }
      const size_t row = size_t(s) * p.num_q_heads + size_t(h) * G + g;
      if (ns == 1) {
        const float out = lsum > 0.f ? a / lsum * vm : 0.f;
        static_cast<__nv_bfloat16*>(p.out)[row * kD + d] = __float2bfloat16_rn(out);
      } else {
        const size_t prow = row * p.max_splits + k;
        p.ws_acc[prow * kD + d] = a;
        if (d == 0) reinterpret_cast<float2*>(p.ws_ml)[prow] = make_float2(M, lsum);
      }
    }
    fence_proxy_async_smem();  // the combine buffer is refilled by TMA next
    __syncthreads();           // shared state is reused by the next unit
    if (aborted) break;
    unit = next_unit;
  }
  pdl_launch_dependents();  // out of work: the merge may launch
}

template <int G, bool FP8>
cudaError_t launch_g(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                     int num_sms, cudaStream_t stream) {
  using C = MmaCfg<FP8>;
  auto kern = decode_mma_kernel<G, FP8>;
  const int max_pages = (p.partition + p.block_size - 1) / p.block_size + 1;
  const int smem = C::OFF_PG + 4 * max_pages + 16 + 1024;  // + alignment slack
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  static std::atomic<bool> configured[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  e = once_per_device(configured, dev, [&] {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  });
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kNW * 32, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  if ((e = launch_decode_plan(p, num_sms, stream)) != cudaSuccess) return e;
  e = launch_pdl(kern, dim3(num_sms * per_sm), dim3(kNW * 32), smem, stream, tk, tv, p);
  if (e != cudaSuccess) return e;
  if (p.max_splits > 1 && (e = launch_decode_merge(p, stream)) != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_mma(const DecodeParams& p, bool fp8, int num_sms, cudaStream_t stream) {
  const int G = p.num_q_heads / p.num_kv_heads;
  if (p.head_dim != kD || (G != 4 && G != 8) || kTT > p.block_size) return cudaErrorNotSupported;
  if (p.num_blocks >= (1 << 30)) return cudaErrorInvalidValue;
  // pools [num_blocks][Hkv][P][128]; one box = 16 rows x 128 B of one page
  // (bf16: two boxes per tile, the halves of head_dim)
  const uint64_t P = p.block_size, Hkv = p.num_kv_heads, E = fp8 ? 1 : 2;
  const auto type = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint32_t box0 = uint32_t(128 / E);
  CUtensorMap tk, tv;
  if (!make_map_4d(&tk, type, p.k_pool, kD, P, Hkv, uint64_t(p.num_blocks), kD * E, P * kD * E,
                   Hkv * P * kD * E, box0, kTT, 1, 1))
    return cudaErrorInvalidValue;
  if (!make_map_4d(&tv, type, p.v_pool, kD, P, Hkv, uint64_t(p.num_blocks), kD * E, P * kD * E,
                   Hkv * P * kD * E, box0, kTT, 1, 1))
    return cudaErrorInvalidValue;
  if (fp8) return G == 8 ? launch_g<8, true>(p, tk, tv, num_sms, stream)
                         : launch_g<4, true>(p, tk, tv, num_sms, stream);
  return G == 8 ? launch_g<8, false>(p, tk, tv, num_sms, stream)
                : launch_g<4, false>(p, tk, tv, num_sms, stream);
}

}  // namespace pkv
