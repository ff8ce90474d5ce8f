// decode.cu -- paged decode attention on CUDA cores (sm_103a).
//
// Follows "TensorRT-LLM框架解析与高性能推理优化实践" §6.2 (Paged Attention优化):
// for each (sequence, head) walk the block table, dot q with every key of
// every page and accumulate the softmax-weighted values; §6.1 (Flash Attention
// 实现): tiles of keys, running max / running sum, partial results kept in
// registers.  Split-K over long contexts with a separate merge kernel is this
// library's own addition for load balance on 152 SMs.
//
// Work decomposition
//   * planner (CTA 0 of the planning launch): for every sequence, nsplit = 1
//     if L <= partition else ceil(L / partition); emits the (sequence,
//     partition) items sorted by size, longest first, and resets the
//     work-fetch counter.  For pkv_paged_attention_append every CTA of that
//     launch also scatters its share of the step's new K/V rows.
//   * decode (persistent, #SM x occupancy CTAs of NW warps): a CTA takes work
//     units (item, kv head) from an atomic counter.  All G = Hq/Hkv q heads of
//     a kv head are packed in the unit, so each K/V page is read from HBM once
//     per kv head.  The unit's tiles of TT tokens are dealt round-robin to the
//     warps; each warp streams its tiles through a private ST-stage
//     shared-memory ring filled by 1-D bulk copies (cp.async.bulk, the TMA
//     engine) and keeps its own running max / sum / accumulators.  The NW
//     warp states are combined in shared memory at the end of the unit and
//     written either as the final bf16 output (one partition) or as an
//     unnormalised partial (m, l, acc[D]) to the workspace.
//   * merge (separate kernel, one warp per split row):
//     out = sum_k 2^(m_k - M) acc_k / sum_k 2^(m_k - M) l_k.
// The planning launch, the decode and the merge are chained with
// programmatic dependent launch: each waits (griddepcontrol.wait) for the
// previous grid before touching its output.
//
// Inner tile (per warp, TT tokens):
//   QK   TPT lanes per token, E head_dim elements per lane, G q heads packed;
//        partial dots are reduced with a reduce-scatter butterfly (G-1 +
//        log2(TPT/G) shuffles per token group instead of G*log2(TPT)).
//   soft 32/G lanes per q head; running max / sum in the log2 domain
//        (q is pre-multiplied by scale*log2(e)), p = 2^(s - m).
//   PV   each lane owns D/32 output columns of all G heads; p is broadcast
//        from shared memory.
#include "pkv_append.cuh"
#include "pkv_common.cuh"
#include "pkv_launch.h"

namespace pkv {

// Per-warp bulk-copy ring depth and warps per CTA.  Two stages beat three or
// four on GB300: the smaller ring lets three CTAs share an SM, and the extra
// resident warps hide the tile compute's latency better than deeper
// prefetch (measured on the Llama-2-13B and Llama-3-8B decode shapes).
#ifndef PKV_DECODE_STAGES
#define PKV_DECODE_STAGES 2
#endif
#ifndef PKV_DECODE_WARPS
#define PKV_DECODE_WARPS 4
#endif

constexpr int kTT = 16;  // tokens per tile (divides every supported block size)
constexpr int kNW = PKV_DECODE_WARPS;  // warps per CTA
constexpr int kMaxBuckets = 1024;

__host__ __device__ constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

template <int D, int G, bool FP8, int ST>
struct DecodeCfg {
  static constexpr int TT = kTT, NW = kNW, NTHR = kNW * 32;
  static constexpr int EB = FP8 ? 1 : 2;
  static constexpr int RB = D * EB;               // bytes of one token row
  static constexpr int TB = TT * RB;              // bytes of one K (or V) tile
  static constexpr int E = (G <= 4) ? 16 : 8;     // head_dim elements per lane (QK)
  static constexpr int TPT = D / E;               // lanes per token (QK)
  static constexpr int NT = 32 / TPT;             // tokens per pass
  static constexpr int PASSES = TT / NT;
  static constexpr int EC = FP8 ? E : 8;          // elements per shared-memory load
  static constexpr int NCH = E / EC;
  static constexpr int CB = EC * EB;              // bytes per load (16 or 8)
  static constexpr int DV = D / 32;               // output columns per lane (PV)
  static constexpr int LPG = 32 / G;              // lanes per q head (softmax)
  static constexpr int TPL = (TT + LPG - 1) / LPG;
  static_assert(TPT >= G && TPT <= 32 && PASSES >= 1, "bad QK mapping");
  // shared memory layout, bytes
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + NW * ST * TB;
  static constexpr int OFF_SC = OFF_V + NW * ST * TB;         // float [NW][TT*G]
  static constexpr int OFF_AL = OFF_SC + NW * TT * G * 4;     // float [NW][G]
  static constexpr int OFF_CM = align_up(OFF_AL + NW * G * 4, 16);   // float2 [NW][G]
  static constexpr int OFF_CA = align_up(OFF_CM + NW * G * 8, 16);   // float [NW][G][D]
  static constexpr int OFF_BAR = align_up(OFF_CA + NW * G * D * 4, 16);  // u64 [NW][ST]
  static constexpr int OFF_MISC = OFF_BAR + NW * ST * 8;      // int [4]
  static constexpr int OFF_PG = OFF_MISC + 16;                // int [pages of a unit]
};

// ---- element loads from shared memory ----------------------------------------
template <bool FP8, int N>
__device__ __forceinline__ void load_cvt(const uint8_t* p, float* f) {
  if constexpr (!FP8) {
    if constexpr (N == 8) {
      const uint4 u = *reinterpret_cast<const uint4*>(p);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 v = bf16x2_to_float2(w[i]);
        f[2 * i] = v.x;
        f[2 * i + 1] = v.y;
      }
    } else if constexpr (N == 4) {
      const uint2 u = *reinterpret_cast<const uint2*>(p);
      const float2 a = bf16x2_to_float2(u.x), b = bf16x2_to_float2(u.y);
      f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    } else {
      static_assert(N == 2, "unsupported");
      const float2 a = bf16x2_to_float2(*reinterpret_cast<const uint32_t*>(p));
      f[0] = a.x; f[1] = a.y;
    }
  } else {
    if constexpr (N == 16) {
      const uint4 u = *reinterpret_cast<const uint4*>(p);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 a = e4m3x2_to_float2(uint16_t(w[i] & 0xFFFFu));
        const float2 b = e4m3x2_to_float2(uint16_t(w[i] >> 16));
        f[4 * i] = a.x; f[4 * i + 1] = a.y; f[4 * i + 2] = b.x; f[4 * i + 3] = b.y;
      }
    } else if constexpr (N == 8) {
      const uint2 u = *reinterpret_cast<const uint2*>(p);
      const uint32_t w[2] = {u.x, u.y};
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float2 a = e4m3x2_to_float2(uint16_t(w[i] & 0xFFFFu));
        const float2 b = e4m3x2_to_float2(uint16_t(w[i] >> 16));
        f[4 * i] = a.x; f[4 * i + 1] = a.y; f[4 * i + 2] = b.x; f[4 * i + 3] = b.y;
      }
    } else if constexpr (N == 4) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
      const float2 a = e4m3x2_to_float2(uint16_t(w & 0xFFFFu));
      const float2 b = e4m3x2_to_float2(uint16_t(w >> 16));
      f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    } else {
      static_assert(N == 2, "unsupported");
      const float2 a = e4m3x2_to_float2(*reinterpret_cast<const uint16_t*>(p));
      f[0] = a.x; f[1] = a.y;
    }
  }
}

// bf16 q elements -> fp32 registers (N multiple of 8, 16-byte aligned source).
template <int N>
__device__ __forceinline__ void load_q(const __nv_bfloat16* src, float mult, float* f) {
#pragma unroll
  for (int i = 0; i < N / 8; ++i) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(src) + i);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 v = bf16x2_to_float2(w[j]);
      f[8 * i + 2 * j] = v.x * mult;
      f[8 * i + 2 * j + 1] = v.y * mult;
    }
  }
}

// Sum v[0..G) over the TPT lanes of a token group, leaving in every lane the
// full sum for head g = c / (TPT / G) (c = lane index within the group).
template <int G, int TPT>
__device__ __forceinline__ float reduce_scatter(float* v, int c) {
  int o = TPT / 2;
#pragma unroll
  for (int n = G; n > 1; n >>= 1) {
    const bool upper = (c & o) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? v[i] : v[i + n / 2];
      const float keep = upper ? v[i + n / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
    o >>= 1;
  }
  float r = v[0];
#pragma unroll
  for (int k = TPT / G / 2; k >= 1; k >>= 1) r += __shfl_xor_sync(0xffffffffu, r, k);
  return r;
}

// Effective context length: clamped to what the block table and workspace
// plan can hold; a length outside [0, cap] is recorded as a bounds error.
__device__ __forceinline__ int effective_len(int L, int cap, int32_t* err) {
  if (L < 0 || L > cap) {
    record_error(err, kDevBadPage);
    return L < 0 ? 0 : cap;
  }
  return L;
}

// ---- planner --------------------------------------------------------------------
// Counting sort of the (sequence, partition) items by length, longest first,
// and reset of the work counter; one CTA of 512 threads.
__device__ void plan_items(const DecodeParams& p) {
  __shared__ int hist[kMaxBuckets];
  __shared__ int offs[kMaxBuckets];
  const int nb = p.partition / kTT + 1;  // bucket = tiles in the item (0 .. partition/TT)
  for (int i = threadIdx.x; i < nb; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  for (int s = threadIdx.x; s < p.num_seqs; s += blockDim.x) {
    const int L = effective_len(__ldg(p.context_lens + s), p.max_len, nullptr);
    const int ns = decode_num_splits(L, p.partition);
    for (int k = 0; k < ns; ++k) {
      const int len = ns == 1 ? L : min(p.partition, L - k * p.partition);
      atomicAdd(&hist[(len + kTT - 1) / kTT], 1);
    }
  }
  __syncthreads();
  // offs[b] = items in the buckets above b (longest items first): an
  // exclusive scan over the buckets in decreasing order, two buckets per
  // thread (nb <= 2 * blockDim.x)
  {
    __shared__ int warp_sum[32];
    const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
    const int r0 = 2 * t, r1 = 2 * t + 1;  // positions in decreasing bucket order
    const int v0 = r0 < nb ? hist[nb - 1 - r0] : 0;
    const int v1 = r1 < nb ? hist[nb - 1 - r1] : 0;
    int incl = v0 + v1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_sum[wid] = incl;
    __syncthreads();
    if (wid == 0) {
      const int nw = (blockDim.x + 31) >> 5;
      int w = lane < nw ? warp_sum[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      if (lane < nw) warp_sum[lane] = w;  // inclusive totals of warps 0 .. lane
      if (lane == nw - 1) {
        p.counters[0] = w;
        p.counters[1] = 0;
      }
    }
    __syncthreads();
    const int before = (wid > 0 ? warp_sum[wid - 1] : 0) + incl - (v0 + v1);
    if (r0 < nb) offs[nb - 1 - r0] = before;
    if (r1 < nb) offs[nb - 1 - r1] = before + v0;
  }
  __syncthreads();
  for (int s = threadIdx.x; s < p.num_seqs; s += blockDim.x) {
    const int L = effective_len(__ldg(p.context_lens + s), p.max_len, nullptr);
    const int ns = decode_num_splits(L, p.partition);
    for (int k = 0; k < ns; ++k) {
      const int len = ns == 1 ? L : min(p.partition, L - k * p.partition);
      const int idx = atomicAdd(&offs[(len + kTT - 1) / kTT], 1);
      p.items[idx] = make_int2(s, k);
    }
  }
}

__global__ void __launch_bounds__(512) decode_plan_kernel(const DecodeParams p) {
  pdl_launch_dependents();
  pdl_wait();  // the step's kv_append (and anything before it) is done
  plan_items(p);
}

// The decode step's append fused into the planning launch: CTA 0 plans and
// every CTA scatters its share of the new rows.  The planner reads only the
// context lengths, which the append does not write; the decode kernels wait
// for this whole grid (griddepcontrol.wait), so they see every appended row.
template <bool FP8>
__global__ void __launch_bounds__(512) decode_plan_append_kernel(const DecodeParams p) {
  pdl_launch_dependents();
  pdl_wait();  // earlier kernels of the stream (readers of the pool) are done
  if (blockIdx.x == 0) plan_items(p);
  append_rows<FP8>(p.append, int64_t(blockIdx.x) * blockDim.x + threadIdx.x,
                   int64_t(gridDim.x) * blockDim.x);
}

// ---- decode -----------------------------------------------------------------------
template <int D, int G, bool FP8, int ST>
__global__ void __launch_bounds__(kNW * 32) decode_kernel(const DecodeParams p) {
  using C = DecodeCfg<D, G, FP8, ST>;
  constexpr int TT = C::TT, NW = C::NW, RB = C::RB, TB = C::TB;
  constexpr int TPT = C::TPT, NT = C::NT, E = C::E, EC = C::EC, CB = C::CB, DV = C::DV;
  constexpr int LPG = C::LPG, TPL = C::TPL, EB = C::EB;
  extern __shared__ __align__(128) uint8_t smem[];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* const kbuf = smem + C::OFF_K + warp * ST * TB;
  uint8_t* const vbuf = smem + C::OFF_V + warp * ST * TB;
  float* const sc = reinterpret_cast<float*>(smem + C::OFF_SC) + warp * TT * G;
  float* const al = reinterpret_cast<float*>(smem + C::OFF_AL) + warp * G;
  float2* const cm = reinterpret_cast<float2*>(smem + C::OFF_CM);
  float* const ca = reinterpret_cast<float*>(smem + C::OFF_CA);
  uint64_t* const bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR) + warp * ST;
  int* const misc = reinterpret_cast<int*>(smem + C::OFF_MISC);
  int* const pages = reinterpret_cast<int*>(smem + C::OFF_PG);

  volatile int* const abort_flag = misc + 2;  // raised by a timed-out wait
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < ST; ++s) mbar_init(&bars[s], 1);
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
  const uint64_t pol = policy_evict_first();
  const int tk = lane / TPT, c = lane % TPT;   // QK mapping
  const int gs = lane / LPG, li = lane % LPG;  // softmax mapping
  uint32_t jt = 0;                             // tiles this warp has consumed
  int unit = misc[0];

  while (unit < n_units) {
    int next = 0;
    if (threadIdx.x == 0) next = atomicAdd(p.counters + 1, 1);
    const int2 item = p.items[unit / Hkv];
    const int h = unit - (unit / Hkv) * Hkv;
    const int s = item.x, k = item.y;
    const int L = effective_len(__ldg(p.context_lens + s), p.max_len, p.err);
    const int ns = decode_num_splits(L, p.partition);
    const int t0 = ns == 1 ? 0 : k * p.partition;
    const int t1 = ns == 1 ? L : min(L, t0 + p.partition);
    const int pg0 = t0 / P;
    const int npg = (t1 - t0 + P - 1) / P;
    for (int i = threadIdx.x; i < npg; i += C::NTHR) {
      int pid = __ldg(p.block_tables + size_t(s) * p.max_blocks + pg0 + i);
      if (pid < 0 || pid >= p.num_blocks) {
        record_error(p.err, kDevBadPage);
        pid = -1;
      }
      pages[i] = pid;
    }
    // per-kv-head FP8 scales fold into the score and output multipliers
    const float qm_h = p.k_scales ? p.q_mult * __ldg(p.k_scales + h) : p.q_mult;
    const float vm_h = p.v_scales ? p.v_mult * __ldg(p.v_scales + h) : p.v_mult;
    // q of the G packed heads, pre-scaled into the log2 domain
    float2 q2[G][E / 2];  // (d, d+1) pairs for packed fp32 FMA
    {
      const __nv_bfloat16* qrow =
          static_cast<const __nv_bfloat16*>(p.q) + (size_t(s) * p.num_q_heads + size_t(h) * G) * D;
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int j = 0; j < C::NCH; ++j)
          load_q<EC>(qrow + g * D + (c + j * TPT) * EC, qm_h,
                     reinterpret_cast<float*>(&q2[g][j * EC / 2]));
    }
    __syncthreads();  // pages[] visible

    const int ntile = (t1 - t0 + TT - 1) / TT;
    const int my_n = warp < ntile ? (ntile - warp + NW - 1) / NW : 0;
    float m_run = -INFINITY, l_run = 0.f;
    float2 acc[G][DV / 2];  // (column, column+1) pairs
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < DV / 2; ++e) acc[g][e] = make_float2(0.f, 0.f);

    // lane 0 issues the copies of this warp's j-th tile of the unit
    auto issue = [&](int j) {
      const int stage = int((jt + j) % ST);
      const int ts = t0 + (warp + j * NW) * TT;
      const int ntok = min(TT, t1 - ts);
      const int pid = pages[ts / P - pg0];
      if (pid < 0) {
        mbar_arrive(&bars[stage]);  // nothing to copy; tile is masked
      } else {
        const size_t elem = ((size_t(pid) * Hkv + h) * P + (ts % P)) * size_t(D);
        const uint32_t bytes = uint32_t(ntok * RB);
        mbar_arrive_expect_tx(&bars[stage], 2 * bytes);
        bulk_g2s(kbuf + stage * TB, p.k_pool + elem * EB, bytes, &bars[stage], pol);
        bulk_g2s(vbuf + stage * TB, p.v_pool + elem * EB, bytes, &bars[stage], pol);
      }
    };
    if (lane == 0)
      for (int j = 0; j < min(ST, my_n); ++j) issue(j);

    for (int j = 0; j < my_n; ++j) {
      const int stage = int((jt + j) % ST);
      const uint32_t parity = ((jt + j) / ST) & 1;
      const int ts = t0 + (warp + j * NW) * TT;
      const int ntok = pages[ts / P - pg0] < 0 ? 0 : min(TT, t1 - ts);
      if (!warp_wait_bounded(&bars[stage], parity, p.err, abort_flag)) {
        // a wait gave up: compute nothing more; let this warp's copies in
        // flight (tiles j .. j + ST - 1) land before the CTA leaves
        if (lane == 0)
          for (int jj = j; jj < min(j + ST, my_n); ++jj)
            mbar_drain_wait(&bars[(jt + jj) % ST], ((jt + jj) / ST) & 1, p.err);
        __syncwarp();
        break;
      }
      const uint8_t* kb = kbuf + stage * TB;
      const uint8_t* vb = vbuf + stage * TB;

      // ---- scores ------------------------------------------------------------
#pragma unroll
      for (int ps = 0; ps < C::PASSES; ++ps) {
        const int t = ps * NT + tk;
        const uint8_t* row = kb + t * RB;
        // packed fp32 FMAs: even and odd head_dim elements accumulate in the
        // two halves of part2 and are added at the end
        float2 part2[G];
#pragma unroll
        for (int g = 0; g < G; ++g) part2[g] = make_float2(0.f, 0.f);
#pragma unroll
        for (int jc = 0; jc < C::NCH; ++jc) {
          float2 k2[EC / 2];
          load_cvt<FP8, EC>(row + (c + jc * TPT) * CB, reinterpret_cast<float*>(k2));
#pragma unroll
          for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < EC / 2; ++e)
              part2[g] = __ffma2_rn(q2[g][jc * EC / 2 + e], k2[e], part2[g]);
        }
        float part[G];
#pragma unroll
        for (int g = 0; g < G; ++g) part[g] = part2[g].x + part2[g].y;
        const float r = reduce_scatter<G, TPT>(part, c);
        if ((c & (TPT / G - 1)) == 0) sc[t * G + c / (TPT / G)] = t < ntok ? r : -INFINITY;
      }
      __syncwarp();

      // ---- online softmax (log2 domain) --------------------------------------
      {
        float sv[TPL];
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < TPL; ++i) {
          const int t = li + i * LPG;
          sv[i] = t < TT ? sc[t * G + gs] : -INFINITY;
          mx = fmaxf(mx, sv[i]);
        }
#pragma unroll
        for (int o = LPG / 2; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float m_new = fmaxf(m_run, mx);
        float alpha = 1.f, sum = 0.f;
        if (m_new != -INFINITY) {
          alpha = fast_exp2(m_run - m_new);
#pragma unroll
          for (int i = 0; i < TPL; ++i) {
            sv[i] = fast_exp2(sv[i] - m_new);
            sum += sv[i];
          }
        } else {
#pragma unroll
          for (int i = 0; i < TPL; ++i) sv[i] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < TPL; ++i) {
          const int t = li + i * LPG;
          if (t < TT) sc[t * G + gs] = sv[i];
        }
#pragma unroll
        for (int o = LPG / 2; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        l_run = l_run * alpha + sum;
        m_run = m_new;
        if (li == 0) al[gs] = alpha;
      }
      __syncwarp();

      // ---- P V ------------------------------------------------------------------
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float2 a = make_float2(al[g], al[g]);
#pragma unroll
        for (int e = 0; e < DV / 2; ++e) acc[g][e] = __fmul2_rn(a, acc[g][e]);
      }
      auto pv = [&](int t) {
        float2 v2[DV / 2];
        load_cvt<FP8, DV>(vb + t * RB + lane * DV * EB, reinterpret_cast<float*>(v2));
        float pg[G];
        if constexpr (G % 4 == 0) {
#pragma unroll
          for (int g4 = 0; g4 < G / 4; ++g4) {
            const float4 x = *reinterpret_cast<const float4*>(sc + t * G + 4 * g4);
            pg[4 * g4] = x.x; pg[4 * g4 + 1] = x.y; pg[4 * g4 + 2] = x.z; pg[4 * g4 + 3] = x.w;
          }
        } else if constexpr (G == 2) {
          const float2 x = *reinterpret_cast<const float2*>(sc + t * 2);
          pg[0] = x.x; pg[1] = x.y;
        } else {
          pg[0] = sc[t];
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float2 pp = make_float2(pg[g], pg[g]);
#pragma unroll
          for (int e = 0; e < DV / 2; ++e) acc[g][e] = __ffma2_rn(pp, v2[e], acc[g][e]);
        }
      };
      if (ntok == TT) {
#pragma unroll
        for (int t = 0; t < TT; ++t) pv(t);
      } else {
#pragma unroll 4
        for (int t = 0; t < ntok; ++t) pv(t);
      }
      __syncwarp();
      if (lane == 0 && j + ST < my_n) {
        fence_proxy_async_smem();
        issue(j + ST);
      }
    }
    jt += uint32_t(my_n);

    // ---- combine the NW warps ------------------------------------------------------
    if (li == 0) cm[warp * G + gs] = make_float2(m_run, l_run);
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < DV / 2; ++e)
        *reinterpret_cast<float2*>(&ca[(warp * G + g) * D + lane * DV + 2 * e]) = acc[g][e];
    if (threadIdx.x == 0) misc[1] = next;
    __syncthreads();
    const int next_unit = misc[1];
    // The abort flag changes only inside the tile loops: between the
    // barrier above and the next unit's first barrier every thread reads the
    // same value.  After an abort the unit's results are not written and the
    // CTA takes no further work.
    const bool aborted = *abort_flag != 0;
    for (int idx = threadIdx.x; idx < G * D && !aborted; idx += C::NTHR) {
      const int g = idx / D, d = idx - g * D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NW; ++w) M = fmaxf(M, cm[w * G + g].x);
      float lsum = 0.f, a = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          const float2 ml = cm[w * G + g];
          const float sw = fast_exp2(ml.x - M);
          lsum = fmaf(sw, ml.y, lsum);
          a = fmaf(sw, ca[(w * G + g) * D + d], a);
        }
      }
      const size_t row = size_t(s) * p.num_q_heads + size_t(h) * G + g;
      if (ns == 1) {
        const float o = lsum > 0.f ? a / lsum * vm_h : 0.f;
        static_cast<__nv_bfloat16*>(p.out)[row * D + d] = __float2bfloat16_rn(o);
      } else {
        const size_t prow = row * p.max_splits + k;
        p.ws_acc[prow * D + d] = a;
        if (d == 0) reinterpret_cast<float2*>(p.ws_ml)[prow] = make_float2(M, lsum);
      }
    }
    __syncthreads();  // shared state is reused by the next unit
    if (aborted) break;
    unit = next_unit;
  }
  pdl_launch_dependents();  // out of work: the merge may launch
}

// ---- merge -------------------------------------------------------------------------
// One warp per (sequence, q head) with more than one partition.  Lane k holds
// partition k's (m, l): the warp takes M = max m and L = sum 2^(m - M) l with
// shuffles, then every lane accumulates its D/32 output columns over the
// partitions, four partial rows in flight at a time.
template <int D>
__device__ __forceinline__ void load_cols(const float* src, float (&v)[D / 32]) {
  if constexpr (D == 128) {
    const float4 x = *reinterpret_cast<const float4*>(src);
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  } else {
    const float2 x = *reinterpret_cast<const float2*>(src);
    v[0] = x.x; v[1] = x.y;
  }
}

template <int D>
__global__ void __launch_bounds__(256) decode_merge_kernel(const DecodeParams p) {
  constexpr int DV = D / 32;
  pdl_wait();  // every partial of the decode grid is written
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= p.num_seqs * p.num_q_heads) return;
  const int s = gw / p.num_q_heads;
  const int L = effective_len(__ldg(p.context_lens + s), p.max_len, nullptr);
  const int ns = decode_num_splits(L, p.partition);
  if (ns <= 1) return;
  const size_t prow = size_t(gw) * p.max_splits;
  const float2* ml = reinterpret_cast<const float2*>(p.ws_ml) + prow;
  float M = -INFINITY;
  for (int k = lane; k < ns; k += 32) M = fmaxf(M, ml[k].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float lsum = 0.f, a[DV];
#pragma unroll
  for (int e = 0; e < DV; ++e) a[e] = 0.f;
  if (M != -INFINITY) {
    for (int k0 = 0; k0 < ns; k0 += 32) {
      float sw = 0.f;
      if (k0 + lane < ns) {
        const float2 v = ml[k0 + lane];
        sw = fast_exp2(v.x - M);
        lsum = fmaf(sw, v.y, lsum);
      }
      const int nk = min(32, ns - k0);
      const float* base = p.ws_acc + (prow + k0) * D + lane * DV;
      int i = 0;
      for (; i + 4 <= nk; i += 4) {
        float v0[DV], v1[DV], v2[DV], v3[DV];
        load_cols<D>(base + (i + 0) * D, v0);
        load_cols<D>(base + (i + 1) * D, v1);
        load_cols<D>(base + (i + 2) * D, v2);
        load_cols<D>(base + (i + 3) * D, v3);
        const float w0 = __shfl_sync(0xffffffffu, sw, i);
        const float w1 = __shfl_sync(0xffffffffu, sw, i + 1);
        const float w2 = __shfl_sync(0xffffffffu, sw, i + 2);
        const float w3 = __shfl_sync(0xffffffffu, sw, i + 3);
#pragma unroll
        for (int e = 0; e < DV; ++e)
          a[e] = fmaf(w3, v3[e], fmaf(w2, v2[e], fmaf(w1, v1[e], fmaf(w0, v0[e], a[e]))));
      }
      for (; i < nk; ++i) {
        float v0[DV];
        load_cols<D>(base + i * D, v0);
        const float w0 = __shfl_sync(0xffffffffu, sw, i);
#pragma unroll
        for (int e = 0; e < DV; ++e) a[e] = fmaf(w0, v0[e], a[e]);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
  }
  __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + size_t(gw) * D + lane * DV;
  const int kvh = (gw - s * p.num_q_heads) / (p.num_q_heads / p.num_kv_heads);
  const float vm = p.v_scales ? p.v_mult * __ldg(p.v_scales + kvh) : p.v_mult;
  const float inv = lsum > 0.f ? vm / lsum : 0.f;
#pragma unroll
  for (int e = 0; e < DV; ++e) dst[e] = __float2bfloat16_rn(a[e] * inv);
}

// ---- host launch ----------------------------------------------------------------
namespace {

template <int D, int G, bool FP8>
cudaError_t launch_one(const DecodeParams& p, int num_sms, cudaStream_t stream) {
  // 4-8 packed q heads: the per-token work (G multiply-adds per element for
  // QK and again for PV) outruns the CUDA cores; it runs on warp-level
  // tensor-core MMAs instead (decode_mma.cu)
  if constexpr (D == 128 && (G == 4 || G == 8)) {
    if (p.block_size >= 16) return launch_decode_mma(p, FP8, num_sms, stream);
  }
  constexpr int ST = PKV_DECODE_STAGES;
  using C = DecodeCfg<D, G, FP8, ST>;
  auto kern = decode_kernel<D, G, FP8, ST>;
  const int max_pages = (p.partition + p.block_size - 1) / p.block_size + 1;
  const int smem = align_up(C::OFF_PG + 4 * max_pages, 16);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  // the shared-memory ceiling is raised once per device; smem varies with
  // the partition, so occupancy is queried for the size at hand
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
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, C::NTHR, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  if ((e = launch_decode_plan(p, num_sms, stream)) != cudaSuccess) return e;
  if ((e = launch_pdl(kern, dim3(num_sms * per_sm), dim3(C::NTHR), smem, stream, p)) !=
      cudaSuccess)
    return e;
  if (p.max_splits > 1) {
    const int warps = p.num_seqs * p.num_q_heads;
    e = launch_pdl(decode_merge_kernel<D>, dim3((warps + 7) / 8), dim3(256), 0, stream, p);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

template <int D, bool FP8>
cudaError_t launch_g(const DecodeParams& p, int num_sms, cudaStream_t stream) {
  switch (p.num_q_heads / p.num_kv_heads) {
    case 1: return launch_one<D, 1, FP8>(p, num_sms, stream);
    case 2: return launch_one<D, 2, FP8>(p, num_sms, stream);
    case 4: return launch_one<D, 4, FP8>(p, num_sms, stream);
    case 8: return launch_one<D, 8, FP8>(p, num_sms, stream);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace

cudaError_t launch_decode_plan(const DecodeParams& p, int num_sms, cudaStream_t stream) {
  if (!p.fuse_append) return launch_pdl(decode_plan_kernel, dim3(1), dim3(512), 0, stream, p);
  const int64_t chunks = int64_t(p.append.num_tokens) * p.append.num_kv_heads * (p.head_dim / 8);
  int64_t blocks = (chunks + 511) / 512;
  if (blocks > int64_t(num_sms) * 4) blocks = int64_t(num_sms) * 4;
  if (blocks < 1) blocks = 1;
  return p.append.fp8
             ? launch_pdl(decode_plan_append_kernel<true>, dim3(unsigned(blocks)), dim3(512), 0,
                          stream, p)
             : launch_pdl(decode_plan_append_kernel<false>, dim3(unsigned(blocks)), dim3(512), 0,
                          stream, p);
}

cudaError_t launch_decode_merge(const DecodeParams& p, cudaStream_t stream) {
  const int warps = p.num_seqs * p.num_q_heads;
  const dim3 grid((warps + 7) / 8), block(256);
  return p.head_dim == 128 ? launch_pdl(decode_merge_kernel<128>, grid, block, 0, stream, p)
                           : launch_pdl(decode_merge_kernel<64>, grid, block, 0, stream, p);
}

cudaError_t launch_decode(const DecodeParams& p, bool fp8, int num_sms, cudaStream_t stream) {
  if (p.partition / kTT + 1 > kMaxBuckets) return cudaErrorInvalidValue;
  if (p.head_dim == 128) return fp8 ? launch_g<128, true>(p, num_sms, stream)
                                    : launch_g<128, false>(p, num_sms, stream);
  if (p.head_dim == 64) return fp8 ? launch_g<64, true>(p, num_sms, stream)
                                   : launch_g<64, false>(p, num_sms, stream);
  return cudaErrorNotSupported;
}

}  // namespace pkv
