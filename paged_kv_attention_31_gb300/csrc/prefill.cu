// prefill.cu -- chunked-prefill attention over a paged KV cache with the
// 5th-generation tensor cores (tcgen05 + TMEM) and TMA (sm_103a).
//
// "TensorRT-LLM框架解析与高性能推理优化实践" §5.3 (分块上下文处理): a long prompt
// is processed as chunks interleaved with decode steps; each chunk's queries
// attend causally to everything before them in the sequence, whose K/V sit
// in pages (§4.2, §6.2).  §6.1 (Flash Attention实现): key tiles, double
// buffering, running max / sum, partial results kept on chip.
//
// A query tile is 128 rows: TQ = 128/G chunk tokens x the G q heads that
// share one kv head (row r = token r / G, head r % G), so every K/V page is
// read once per kv head and the tile is a dense M = 128 contraction.  One CTA
// (one per SM) takes two consecutive tiles of one (sequence, kv head) and
// specialises its warps:
//   warps 9, 10 loaders: TMA of Q and the K pages (warp 9) and of the V
//               pages (warp 10) into 2-stage rings of 128-key blocks shared
//               by both tiles; page ids from the block table, read a few
//               blocks ahead; pages past the sequence use an out-of-range
//               coordinate so TMA fills zeros; the V loader zeroes the last
//               block's rows past the sequence end before handing it over.
//   warp 8      lane 0 alone issues every tcgen05.mma and waits on every
//               barrier of its loop, with descriptors made once per CTA:
//                 S_t = Q_t K_j^T  (M=128, N=128, K=128; A, B in shared memory)
//                 O_t += P_t V_j   (M=128, N=128, K=128; A = P in TMEM, B = V)
//   warps 0-3   softmax of tile 0, warps 4-7 softmax of tile 1: one thread
//   warps 4-7   per row (TMEM lane).  One tcgen05.ld brings a block's 128
//               scores into registers (causal mask on diagonal blocks); the
//               running max is lagged: it moves only when it grows by more
//               than 2^8 (O is then rescaled in TMEM; the final
//               normalisation uses the same max, so the result is exact),
//               and the block-max pass runs only where that can happen; P =
//               2^(s - m) goes as bf16 pairs over the first half of S's own
//               TMEM columns.
// TMEM (512 columns): S_t at 128 t, O_t at 256 + 128 t.  P never leaves
// TMEM: the PV product reads its A operand there, so shared memory holds
// only Q, K and V and feeds one operand per PV MMA.  Per tile the chain is
// S_j -> softmax_j -> (PV_j, S_{j+1}); the MMA issuer alternates the tiles, so
// while one tile's softmax runs the tensor core works on the other tile.
// Every hand-off is an mbarrier: tcgen05.commit signals "S ready", "last PV
// done" and "K / V stage free"; the softmax warps signal "P ready".  The
// commit behind "S_{j+1} ready" also covers PV_j, so the softmax of block
// j + 1 may rescale O without another wait.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "pkv_common.cuh"
#include "pkv_launch.h"
#include "pkv_tmap.h"

namespace pkv {
namespace {

constexpr int kM = 128;          // query rows per tile
constexpr int kNK = 128;         // keys per block
constexpr int kTiles = 2;        // query tiles per CTA
constexpr int kSoftmaxThreads = 128 * kTiles;
constexpr int kMmaWarp = kSoftmaxThreads / 32;   // warp 8: issues every tcgen05.mma
constexpr int kKLoadWarp = kMmaWarp + 1;         // warp 9: TMA of Q and of the K ring
constexpr int kVLoadWarp = kMmaWarp + 2;         // warp 10: TMA of the V ring
constexpr int kThreads = kSoftmaxThreads + 3 * 32;
constexpr uint32_t kTmemCols = 512;
// TMEM columns: S (then P) of tile t at 128 t, O of tile t at 256 + D t
constexpr uint32_t kColS = 0, kColO = 256;
// CTA order: end positions of up to kMaxRankGroups (sequence, tile pair) groups
constexpr int kMaxRankGroups = 256;
// The 128-byte-swizzled tiles need a 1024-aligned base; dynamic shared memory
// starts at least 128-aligned, so at most 896 bytes of padding are needed.
constexpr int kMaxPad = 1024 - 128;

// 1: the softmax skips its max pass where the block's P sum shows that the
// lagged running max need not move (0: a max pass on every block).
#ifndef PKV_PF_SKIP_MAX
#define PKV_PF_SKIP_MAX 1
#endif

// FP8 pools: operand stages of f16 K (and V) blocks, 1 or 2; the code ring
// of each then has 3 - that many stages (shared memory holds no more).  Two
// operand stages let a converter work a block ahead of the MMAs (87 against
// 105 us on the FP8 mixed step's prefill, one code stage against two).
#ifndef PKV_PF_FP8_OPSTAGES
#define PKV_PF_FP8_OPSTAGES 2
#endif

// Shared memory layout for head_dim D (offsets from a 1024-aligned base).
// Rows of Q, K and V are split into D/64 halves of 64 16-bit values (128
// bytes, one swizzle atom): a tile is [half][rows][128 B].  bf16 pools: K and
// V stream by TMA straight into 2-stage rings of such blocks.  FP8 pools: the
// TMA lands each key block's E4M3 codes, row-major [key][D], in a raw ring;
// a converter warp turns them into f16 K (V) blocks of the same swizzled
// layout.
template <int D, bool FP8>
struct PfLayout {
  static constexpr int kHalves = D / 64;
  static constexpr int kStagesK = FP8 ? PKV_PF_FP8_OPSTAGES : 2;  // K operand stages (key blocks)
  static constexpr int kStagesV = FP8 ? PKV_PF_FP8_OPSTAGES : 2;  // V operand stages
  static constexpr int kRawStages = FP8 ? 3 - PKV_PF_FP8_OPSTAGES : 0;  // code stages, K and V each
  static constexpr int kQBytes = kHalves * kM * 128;         // per tile
  static constexpr int kKVStageBytes = kHalves * kNK * 128;  // one key block of K or V
  static constexpr int kRawBytes = kNK * D;                  // one key block of FP8 codes
  // barriers: q, k[SK], kfree[SK], v[SV], vfree[SV], s[tiles], p[tiles],
  // o[tiles], drain (the MMA thread's last commit after an abort), vz (the
  // last V block's rows past the sequence zeroed); FP8 also qc (Q
  // converted), kraw[R], vraw[R] (code blocks landed)
  static constexpr int kNumBars =
      1 + 2 * kStagesK + 2 * kStagesV + 3 * kTiles + 2 + (FP8 ? 1 + 2 * kRawStages : 0);
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kTiles * kQBytes;
  static constexpr int kOffV = kOffK + kStagesK * kKVStageBytes;
  static constexpr int kOffRawK = kOffV + kStagesV * kKVStageBytes;
  static constexpr int kOffRawV = kOffRawK + kRawStages * kRawBytes;
  static constexpr int kOffBar = kOffRawV + kRawStages * kRawBytes;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kOffRank = kOffMisc + 16;
  static constexpr int kSmemBytes = kOffRank + 4 * kMaxRankGroups + kMaxPad;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert(kColO + kTiles * D <= kTmemCols, "TMEM budget");
};

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

// 32 consecutive fp32 columns of this thread's TMEM lane (load and wait).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// 128 consecutive fp32 columns of this thread's TMEM lane (one load, one wait).
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, float* v) {
  uint32_t r[128];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%128];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 128; ++i) v[i] = __uint_as_float(r[i]);
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

// max(a, b, c) in one instruction (3-input max.f32, sm_100 family).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// D[tmem] (+)= A[tmem] * B[smem]: A is 128 lanes x K with two bf16 per
// 32-bit column (K-major), one elected thread.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// 16 consecutive 32-bit columns of this thread's TMEM lane; completion is
// awaited separately with tmem_wait_st().
__device__ __forceinline__ void tmem_st16_async(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
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

// Instruction descriptor, kind::f16: fp32 accumulate (bits 4-5 = 1), A and B
// both bf16 (bits 7-9 and 10-12 = 1) or both f16 (= 0), B K-major or
// MN-major (bit 16), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_f16_kind(int M, int N, bool b_mn_major, bool f16) {
  return (1u << 4) | (f16 ? 0u : (1u << 7) | (1u << 10)) | (b_mn_major ? (1u << 16) : 0u) |
         (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// Four E4M3 codes (bytes 0..3 of w) -> f16x2 (b0, b1) and (b2, b3), exact
// (every E4M3 value is a normal f16); the lower byte lands in the lower half.
__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\t"
      "mov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// The register file is handed out per group of four warps, so the 11-warp
// CTA is budgeted as 12 warps: at most 168 registers per thread.
//
// FP8 pools (FP8 = true): tm_k / tm_v map the E4M3 pools (unswizzled page
// boxes); each loader warp converts its blocks to f16 (exact) and both
// products run as kind::f16 MMAs on f16 operands: Q is converted in place to
// f16 by the softmax threads, each row first multiplied by an exact power of
// two 2^k that puts its largest |q| in [2^15, 2^16) (the row's scores are
// multiplied by 2^-k), and P is written to TMEM as f16.  k_scale multiplies
// the scores, v_scale the output (per tensor, or per kv head).
template <int D, bool FP8>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
  constexpr int kD = D;
  using Lay = PfLayout<D, FP8>;
  constexpr int kHalves = Lay::kHalves, kQBytes = Lay::kQBytes;
  constexpr int kKVStageBytes = Lay::kKVStageBytes, kRawBytes = Lay::kRawBytes;
  constexpr int kRawRing = FP8 ? Lay::kRawStages : 1;  // (the bf16 kernel has no code ring)
  constexpr int kStagesK = Lay::kStagesK, kStagesV = Lay::kStagesV;
  constexpr int kOffQ = Lay::kOffQ, kOffK = Lay::kOffK, kOffV = Lay::kOffV;
  constexpr int kOffBar = Lay::kOffBar, kOffMisc = Lay::kOffMisc, kOffRank = Lay::kOffRank;
  if (threadIdx.x == 32 * kKLoadWarp) {  // the loaders' tensor maps, fetched ahead of their first copies
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_q)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_k)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_v)) : "memory");
  }
  pdl_wait();  // inputs written by earlier kernels of the stream are visible
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  if (pad > uint32_t(kMaxPad)) {  // cannot happen with a 128-aligned base; never index past the end
    if (threadIdx.x == 0) record_error(p.err, kDevBadPage);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  const int G = p.num_q_heads / p.num_kv_heads;
  const int TQ = kM / G;

  // Longest work first: CTA k takes kv head k % Hkv of the (sequence, tile
  // pair) group of rank k / Hkv, ranked by the position of the group's last
  // query (its key count), ties by group index.  The block scheduler starts
  // CTAs in index order, so this is the longest-processing-time-first list
  // schedule; groups past a sequence's chunk rank last and exit at once.
  const int max_pairs = (p.tiles_per_seq + kTiles - 1) / kTiles;
  const int n_groups = p.num_seqs * max_pairs;
  const int h = int(blockIdx.x) % p.num_kv_heads;
  int group = int(blockIdx.x) / p.num_kv_heads;
  if (n_groups > kMaxRankGroups) {  // too many to rank here: later tile pairs first
    group = (group / max_pairs) * max_pairs + (max_pairs - 1 - group % max_pairs);
  } else {
    int* const gend = reinterpret_cast<int*>(smem + kOffRank);
    int* const gsel = reinterpret_cast<int*>(smem + kOffMisc + 8);
    for (int g = threadIdx.x; g < n_groups; g += blockDim.x) {
      const int gs = g / max_pairs, ta = (g - gs * max_pairs) * kTiles * TQ;
      const int c0 = __ldg(p.cu_seqlens_q + gs), cg = __ldg(p.cu_seqlens_q + gs + 1) - c0;
      gend[g] = (cg > 0 && ta < cg) ? max(0, __ldg(p.context_lens + gs) - cg + min(cg, ta + kTiles * TQ))
                                    : -1;
    }
    __syncthreads();
    const int want = group;
    for (int g = threadIdx.x; g < n_groups; g += blockDim.x) {
      const int e = gend[g];
      int r = 0;
      for (int o = 0; o < n_groups; ++o) {
        const int eo = gend[o];
        r += (eo > e || (eo == e && o < g)) ? 1 : 0;
      }
      if (r == want) *gsel = g;
    }
    __syncthreads();
    group = *gsel;
    __syncthreads();  // the rank area is reused below only through other offsets
  }
  const int s = group / max_pairs, pair = group - s * max_pairs;
  const int q0 = __ldg(p.cu_seqlens_q + s);
  const int q1 = __ldg(p.cu_seqlens_q + s + 1);
  // the chunk's rows must lie inside q / out and inside the grid's tiles
  // (max_q_len): otherwise the sequence is recorded and skipped
  if (q0 < 0 || q1 < q0 || q1 > p.num_q_tokens ||
      int64_t(q1 - q0) * G > int64_t(p.tiles_per_seq) * kM) {
    if (threadIdx.x == 0 && pair == 0) record_error(p.err, kDevBadPage);
    return;
  }
  const int C = q1 - q0;
  const int tokA = pair * kTiles * TQ;            // first chunk token of tile 0
  if (C <= 0 || tokA >= C) return;
  const int L = __ldg(p.context_lens + s);
  const int P = p.block_size;
  if (L < C || L > p.max_blocks * P) {
    if (threadIdx.x == 0) record_error(p.err, kDevBadPage);
    return;
  }
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sK = smem + kOffK;
  uint8_t* sV = smem + kOffV;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* bar_q = bar;
  uint64_t* bar_k = bar + 1;                      // [kStagesK] K block landed
  uint64_t* bar_kfree = bar_k + kStagesK;         // [kStagesK] S MMAs done with the K stage
  uint64_t* bar_v = bar_kfree + kStagesK;         // [kStagesV] V block landed
  uint64_t* bar_vfree = bar_v + kStagesV;         // [kStagesV] PV MMAs done with the V stage
  // per tile, one phase per key block (each side waits every phase in order)
  uint64_t* bar_s = bar_vfree + kStagesV;         // [kTiles] S_t of the next block ready
  uint64_t* bar_p = bar_s + kTiles;               // [kTiles] P_t written (4 warps)
  uint64_t* bar_o = bar_p + kTiles;               // [kTiles] last PV of tile t done (one phase)
  uint64_t* bar_drain = bar_o + kTiles;           // every issued MMA done (after an abort)
  uint64_t* bar_vz = bar_drain + 1;               // bf16: last V block's tail rows zeroed
  // FP8 only: Q converted to f16 (8 softmax warps), code blocks landed
  uint64_t* bar_qc = bar_vz + 1;
  uint64_t* bar_kraw = bar_qc + 1;                // [kRawStages]
  uint64_t* bar_vraw = bar_kraw + Lay::kRawStages;  // [kRawStages]
  uint8_t* sRawK = smem + Lay::kOffRawK;
  uint8_t* sRawV = smem + Lay::kOffRawV;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // per-tile extent: valid tokens, first position, key blocks to visit
  static_assert(kTiles == 2, "two query tiles per CTA");
  const int ntok0 = max(0, min(TQ, C - tokA));
  const int ntok1 = max(0, min(TQ, C - (tokA + TQ)));
  const int nb0 = ntok0 > 0 ? (L - C + tokA + ntok0 - 1) / kNK + 1 : 0;
  const int nb1 = ntok1 > 0 ? (L - C + tokA + TQ + ntok1 - 1) / kNK + 1 : 0;
  const int nblk = max(nb0, nb1);                 // key blocks loaded for the CTA
  const int npages = (L + P - 1) / P;
  const int pages_per_blk = kNK / P;              // 2 .. 8

  if (tid == 0) {
    mbar_init(bar_q, 1);
    for (int i = 0; i < kStagesK; ++i) {
      mbar_init(&bar_k[i], 1);
      mbar_init(&bar_kfree[i], 1);
    }
    for (int i = 0; i < kStagesV; ++i) {
      mbar_init(&bar_v[i], 1);
      mbar_init(&bar_vfree[i], 1);
    }
    for (int t = 0; t < kTiles; ++t) {
      mbar_init(&bar_s[t], 1);
      mbar_init(&bar_p[t], 4);
      mbar_init(&bar_o[t], 1);
    }
    mbar_init(bar_drain, 1);
    mbar_init(bar_vz, 1);
    if constexpr (FP8) {
      mbar_init(bar_qc, 8);
      for (int i = 0; i < Lay::kRawStages; ++i) {
        mbar_init(&bar_kraw[i], 1);
        mbar_init(&bar_vraw[i], 1);
      }
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // ============================ loaders and MMA issuer ============================
  auto page_of = [&](int j) -> int {
    if (j >= npages) return p.num_blocks;  // past the sequence: TMA zero fill
    int pid = __ldg(p.block_tables + size_t(s) * p.max_blocks + j);
    if (pid < 0 || pid >= p.num_blocks) {
      record_error(p.err, kDevBadPage);
      pid = p.num_blocks;
    }
    return pid;
  };
  // loader warps: lane i holds the id of page i of key block `blk`
  auto fetch_ids = [&](int blk) -> int {
    return (lane < pages_per_blk && blk < nblk) ? page_of(blk * pages_per_blk + lane) : 0;
  };
  // TMA of one key block's pages into its ring stage (whole loader warp)
  auto load_blk = [&](const CUtensorMap* map, uint8_t* ring, uint64_t* bars, int stages, int blk,
                      int ids) {
    const int st = blk % stages;
    if (lane == 0) mbar_arrive_expect_tx(&bars[st], kKVStageBytes);
#pragma unroll
    for (int i = 0; i < kNK / 16; ++i) {  // at most 8 pages per block (block_size >= 16)
      const int pid = __shfl_sync(0xffffffffu, ids, i);
      if (lane == 0 && i < pages_per_blk) {
#pragma unroll
        for (int dh = 0; dh < kHalves; ++dh)
          tma_load_4d(ring + st * kKVStageBytes + dh * (kNK * 128) + i * P * 128, map, dh * 64,
                      0, h, pid, &bars[st]);
      }
    }
  };
  // a loader streams blocks 0 .. nblk-1 into its ring; block b reuses the
  // stage of block b - stages once `freed` says the MMAs reading it are done.
  // With `tail_bar` (the V ring) and a last block that reaches past the
  // sequence, the loader waits for that block to land, zeroes its rows from
  // the sequence end on (never-written slots may hold NaN, and 0 * V must
  // stay 0 in the PV product) and then arrives on `tail_bar`, which the MMA
  // thread waits instead of the block's own barrier.
  // If a wait gives up it stops issuing; either way it returns only after
  // the copies it issued into the ring have landed (on the normal path the
  // MMA thread has already seen them all, so this returns at once).
  auto run_loader = [&](const CUtensorMap* map, uint8_t* ring, uint64_t* full, uint64_t* freed,
                        int stages, uint64_t* tail_bar) {
    constexpr int kLead = 3;  // page ids are read kLead blocks ahead
    int ids[kLead];
#pragma unroll
    for (int k = 0; k < kLead; ++k) ids[k] = fetch_ids(k);
    int issued = 0;
    for (int b = 0; b < nblk; ++b) {
      if (b >= stages && !warp_wait_bounded(&freed[b % stages],
                                            uint32_t((b - stages) / stages) & 1, p.err,
                                            abort_flag))
        break;
      load_blk(map, ring, full, stages, b, ids[0]);
      issued = b + 1;
#pragma unroll
      for (int k = 0; k + 1 < kLead; ++k) ids[k] = ids[k + 1];
      ids[kLead - 1] = fetch_ids(b + kLead);
      if (tail_bar != nullptr && b == nblk - 1 && b * kNK + kNK > L) {
        if (!warp_wait_bounded(&full[b % stages], uint32_t(b / stages) & 1, p.err, abort_flag))
          break;
        uint8_t* const st = ring + (b % stages) * kKVStageBytes;
        const int first = max(0, L - b * kNK);
        for (int i = lane; i < (kNK - first) * 8 * kHalves; i += 32) {
          const int r = first + i / (8 * kHalves), dh = (i / 8) % kHalves, chunk = i % 8;
          *reinterpret_cast<uint4*>(st + dh * (kNK * 128) + r * 128 + chunk * 16) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();  // the PV MMAs (async proxy) read the block next
        __syncwarp();
        if (lane == 0) mbar_arrive(tail_bar);
      }
    }
    if (lane == 0)
      for (int b = max(0, issued - stages); b < issued; ++b)
        mbar_drain_wait(&full[b % stages], uint32_t(b / stages) & 1, p.err);
    __syncwarp();
  };

  // ---- FP8 pools: code blocks by TMA, converted to f16 operand blocks ----
  // TMA of one key block's code pages (row-major [key][D]) into raw stage
  // blk % kRawStages (whole loader warp)
  auto load_raw = [&](const CUtensorMap* map, uint8_t* raw, uint64_t* bars, int blk, int ids) {
    const int st = blk % kRawRing;
    if (lane == 0) mbar_arrive_expect_tx(&bars[st], kRawBytes);
#pragma unroll
    for (int i = 0; i < kNK / 16; ++i) {  // at most 8 pages per block (block_size >= 16)
      const int pid = __shfl_sync(0xffffffffu, ids, i);
      if (lane == 0 && i < pages_per_blk)
        tma_load_4d(raw + st * kRawBytes + i * P * kD, map, 0, 0, h, pid, &bars[st]);
    }
  };
  // the codes of one key block -> f16 in the swizzled operand layout (the
  // one a 128-byte-swizzled TMA box of 16-bit values gives); key rows from
  // zero_from on are written as zeros: slots past the sequence may hold NaN
  // codes, and 0 * V must stay 0 in the PV product.
  // A lane turns 16 codes (one quarter of a row half) into two 16-byte
  // chunks.  Each group of 8 lanes (one shared-memory phase of 16-byte
  // accesses) takes the quarters of two adjacent rows, r in one half and
  // r + 1 in the other for D = 128 (both in the one half for D = 64), so its
  // loads cover 128 distinct bytes of banks and its stores, whose swizzle
  // (chunk ^ (row & 7)) differs in parity between the two rows, land in 8
  // distinct chunk positions.  The loads of four tasks are issued before
  // their conversions.
  auto convert_blk = [&](const uint8_t* raw, uint8_t* dst, int zero_from) {
    constexpr int kTasks = kNK * kHalves * 4;  // 16-code tasks per block
    constexpr int kBatch = 4;                  // tasks in flight per lane
    static_assert(kTasks % (32 * kBatch) == 0, "whole batches");
    for (int i0 = 0; i0 < kTasks; i0 += 32 * kBatch) {
      uint4 u[kBatch];
      int row[kBatch], hf[kBatch], qt[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int i = i0 + b * 32 + lane;
        const int g = i >> 3, w = i & 7;       // phase group, lane in it
        const int pr = w >> 2;                 // which row of the pair
        qt[b] = w & 3;                         // quarter of the half row
        if constexpr (kHalves == 2) {          // groups alternate the half pairing
          row[b] = 2 * (g >> 1) + pr;
          hf[b] = pr ^ (g & 1);
        } else {
          row[b] = 2 * g + pr;
          hf[b] = 0;
        }
        u[b] = *reinterpret_cast<const uint4*>(raw + row[b] * kD + hf[b] * 64 + qt[b] * 16);
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const uint4 v = row[b] >= zero_from ? make_uint4(0u, 0u, 0u, 0u) : u[b];
        uint32_t f[8];
        e4m3x4_to_f16x2(v.x, f[0], f[1]);
        e4m3x4_to_f16x2(v.y, f[2], f[3]);
        e4m3x4_to_f16x2(v.z, f[4], f[5]);
        e4m3x4_to_f16x2(v.w, f[6], f[7]);
        uint8_t* const d = dst + hf[b] * (kNK * 128) + row[b] * 128;
        const int c = 2 * qt[b], x = row[b] & 7;
        *reinterpret_cast<uint4*>(d + ((c ^ x) << 4)) = make_uint4(f[0], f[1], f[2], f[3]);
        *reinterpret_cast<uint4*>(d + (((c + 1) ^ x) << 4)) = make_uint4(f[4], f[5], f[6], f[7]);
      }
    }
  };

  // a converter warp keeps kRawStages code blocks in flight; block b is
  // converted into operand stage b % stages once `freed` says the MMAs that
  // read its previous block are done, and `ready` then signals the MMA warp.
  // If a wait gives up it stops; either way it returns only after its code
  // copies in flight have landed.
  auto run_converter = [&](const CUtensorMap* map, uint8_t* raw, uint64_t* raw_full,
                           uint8_t* ops, uint64_t* ready, uint64_t* freed, int stages) {
    constexpr int R = kRawRing;
    constexpr int kLead = 3;  // page ids are read kLead blocks ahead
    int ids[kLead];
#pragma unroll
    for (int k = 0; k < kLead; ++k) ids[k] = fetch_ids(k);
    int issued = 0;  // code blocks whose copies were issued
    auto issue_next = [&]() {
      load_raw(map, raw, raw_full, issued, ids[0]);
#pragma unroll
      for (int k = 0; k + 1 < kLead; ++k) ids[k] = ids[k + 1];
      ids[kLead - 1] = fetch_ids(issued + kLead);
      ++issued;
    };
    while (issued < R && issued < nblk) issue_next();
    for (int b = 0; b < nblk; ++b) {
      if (!warp_wait_bounded(&raw_full[b % R], uint32_t(b / R) & 1, p.err, abort_flag)) break;
      if (b >= stages && !warp_wait_bounded(&freed[b % stages],
                                            uint32_t((b - stages) / stages) & 1, p.err,
                                            abort_flag))
        break;
      convert_blk(raw + (b % R) * kRawBytes, ops + (b % stages) * kKVStageBytes, L - b * kNK);
      // the MMAs (async proxy) read the block next, and the next code copy
      // (async proxy) rewrites the raw stage just read
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ready[b % stages]);
      if (issued < nblk) issue_next();
    }
    if (lane == 0)
      for (int b = max(0, issued - R); b < issued; ++b)
        mbar_drain_wait(&raw_full[b % R], uint32_t(b / R) & 1, p.err);
    __syncwarp();
  };

  if (warp == kKLoadWarp) {
    if (lane == 0) {
      mbar_arrive_expect_tx(bar_q, kTiles * kQBytes);
      for (int t = 0; t < kTiles; ++t)
#pragma unroll
        for (int dh = 0; dh < kHalves; ++dh)
          tma_load_4d(sQ + t * kQBytes + dh * (kM * 128), &tm_q, dh * 64, 0, h,
                      q0 + tokA + t * TQ, bar_q);
    }
    if constexpr (FP8)
      run_converter(&tm_k, sRawK, bar_kraw, sK, bar_k, bar_kfree, kStagesK);
    else
      run_loader(&tm_k, sK, bar_k, bar_kfree, kStagesK, nullptr);
    if (lane == 0) mbar_drain_wait(bar_q, 0, p.err);  // Q landed (normally seen long ago)
    __syncwarp();
  } else if (warp == kVLoadWarp) {
    if constexpr (FP8)
      run_converter(&tm_v, sRawV, bar_vraw, sV, bar_v, bar_vfree, kStagesV);
    else
      run_loader(&tm_v, sV, bar_v, bar_vfree, kStagesV, bar_vz);
  } else if (warp == kMmaWarp) {
    // One thread issues every MMA and waits on every barrier of this loop.  A
    // tcgen05.mma issue proceeds at about the tensor core's own pace (only a
    // few products queue ahead), so the thread's path from one tile's last
    // product to the other tile's first must stay short, or the tensor core
    // idles: no warp-wide votes or syncs inside the loop.
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_f16_kind(kM, kNK, false, FP8);
      constexpr uint32_t kIdescO = idesc_f16_kind(kM, kD, true, FP8);
      const uint32_t q_base = smem_u32(sQ), k_base = smem_u32(sK), v_base = smem_u32(sV);
      // shared-memory descriptors of every operand step, made once: the
      // issuing thread's path per MMA is then the instruction itself
      static_assert(kStagesK <= 2 && kStagesV <= 2, "one or two operand stages");
      uint64_t dq[kTiles][kD / 16], dk[kStagesK][kD / 16], dv[kStagesV][kNK / 16];
#pragma unroll
      for (int ks = 0; ks < kD / 16; ++ks) {
        const int dh = ks >> 2, w = ks & 3;
#pragma unroll
        for (int t = 0; t < kTiles; ++t)
          dq[t][ks] = sw128_desc(q_base + t * kQBytes + dh * (kM * 128) + w * 32, 16, 1024);
#pragma unroll
        for (int st = 0; st < kStagesK; ++st)
          dk[st][ks] =
              sw128_desc(k_base + st * kKVStageBytes + dh * (kNK * 128) + w * 32, 16, 1024);
      }
#pragma unroll
      for (int ks = 0; ks < kNK / 16; ++ks)
#pragma unroll
        for (int st = 0; st < kStagesV; ++st)
          dv[st][ks] = sw128_desc(v_base + st * kKVStageBytes + ks * 2048, kNK * 128, 1024);
      auto issue_s = [&](int t, int blk) {  // S_t of block blk
        const bool st = kStagesK == 2 && (blk & 1) != 0;
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks)
          mma_bf16(tmem + kColS + t * kNK, dq[t][ks], st ? dk[kStagesK - 1][ks] : dk[0][ks],
                   kIdescS, ks > 0);
        mma_commit(&bar_s[t]);
      };
      auto issue_pv = [&](int t, int blk, bool last) {  // O_t += P_t V_blk
        const bool st = kStagesV == 2 && (blk & 1) != 0;
#pragma unroll
        for (int ks = 0; ks < kNK / 16; ++ks) {
          mma_bf16_ts(tmem + kColO + t * kD, tmem + kColS + t * kNK + ks * 8,
                      st ? dv[kStagesV - 1][ks] : dv[0][ks], kIdescO,
                      (blk > 0 || ks > 0) ? 1u : 0u);
        }
        if (last) mma_commit(&bar_o[t]);
      };
      auto wait_k = [&](int b) {
        return mbar_wait_bounded(&bar_k[b % kStagesK], uint32_t(b / kStagesK) & 1, p.err,
                                 abort_flag);
      };
      // bf16: a last V block reaching past the sequence is handed over by
      // the V loader once it has zeroed the rows there (FP8: the converter
      // writes those rows as zeros)
      const bool vtail = !FP8 && nblk * kNK > L;

      // `alive` turns false when a wait gives up: no further MMA is issued.
      // FP8: Q is read once the softmax warps have converted it to f16.
      bool alive = mbar_wait_bounded(FP8 ? bar_qc : bar_q, 0, p.err, abort_flag);
      if (alive && nblk > 0) {
        alive = wait_k(0);
        if (alive) {
          tc_fence_after();
          if (nb0 > 0) issue_s(0, 0);
          if (nb1 > 0) issue_s(1, 0);
          mma_commit(&bar_kfree[0]);
        }
      }
      for (int j = 0; alive && j < nblk; ++j) {
        const int sv = j % kStagesV;
        const bool z = vtail && j == nblk - 1;
        if (!mbar_wait_bounded(z ? bar_vz : &bar_v[sv], z ? 0u : uint32_t(j / kStagesV) & 1,
                               p.err, abort_flag)) {
          alive = false;
          break;
        }
        // per tile: O_t += P_t V_j once the softmax warps have written P_t,
        // then S_t of block j + 1 into the same TMEM columns (the tensor core
        // runs MMAs in issue order, so the PV has read P before S overwrites it)
        bool k_ready = false;
#pragma unroll
        for (int t = 0; t < kTiles; ++t) {
          const int nbt = t == 0 ? nb0 : nb1;
          if (j >= nbt) continue;
          if (!mbar_wait_bounded(&bar_p[t], uint32_t(j) & 1, p.err, abort_flag)) {
            alive = false;
            break;
          }
          tc_fence_after();
          issue_pv(t, j, j == nbt - 1);
          if (j + 1 < nbt) {
            if (!k_ready) {
              if (!wait_k(j + 1)) {
                alive = false;
                break;
              }
              k_ready = true;
            }
            issue_s(t, j + 1);
          }
        }
        if (!alive) break;
        // stage release: V_j after both tiles' PV, K_{j+1} after both tiles' S
        mma_commit(&bar_vfree[sv]);
        if (j + 1 < nblk) mma_commit(&bar_kfree[(j + 1) % kStagesK]);
      }
      if (!alive) {
        // every MMA this thread issued completes before TMEM is released (a
        // commit arrives once all of the thread's earlier MMAs are done)
        mma_commit(bar_drain);
        mbar_drain_wait(bar_drain, 0, p.err);
      }
    }
    __syncwarp();
  } else if (warp < kMmaWarp) {
    // ================================ softmax ====================================
    const int t = warp >> 2;                        // tile of this warpgroup
    const int row = tid & 127;
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    const uint32_t colS = kColS + t * kNK, colO = kColO + t * kD;
    const int tok = tokA + t * TQ + row / G;
    const bool row_valid = (row / G) < (t == 0 ? ntok0 : ntok1);
    const int pos = row_valid ? L - C + tok : -1;  // keys 0 .. pos are visible
    const int minpos = L - C + tokA + t * TQ;      // first token of the tile
    float qm = p.q_mult;                           // scale * k_scale * log2(e) > 0
    float m_used = -INFINITY, l_sum = 0.f;
    const int nb = t == 0 ? nb0 : nb1;

    bool alive = true;  // false once a wait gives up: no more TMEM work, no stores
    if constexpr (FP8) {
      if (p.k_scales) qm *= __ldg(p.k_scales + h);
      // This thread's row of Q to f16 in place, times 2^k with k = 15 -
      // floor(log2 max|q|) (clamped to [-126, 64], so that 2^k and the row's
      // score multiplier qm * 2^-k stay normal floats): f16 then holds every
      // value of the row within 2^29 of its largest exactly.
      alive = warp_wait_bounded(bar_q, 0, p.err, abort_flag);
      if (alive) {
        uint8_t* const qrow = sQ + t * kQBytes + row * 128;
        float amax = 0.f;
#pragma unroll
        for (int dh = 0; dh < kHalves; ++dh)
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 u =
                *reinterpret_cast<const uint4*>(qrow + dh * (kM * 128) + ((c ^ (row & 7)) << 4));
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 f = bf16x2_to_float2(w[i]);
              amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
          }
        const int e = int((__float_as_uint(amax) >> 23) & 0xFF) - 127;  // -127 if subnormal
        const int k = amax > 0.f ? max(-126, min(64, 15 - e)) : 0;
        const float up = __uint_as_float(uint32_t(127 + k) << 23);
        qm *= __uint_as_float(uint32_t(127 - k) << 23);
#pragma unroll
        for (int dh = 0; dh < kHalves; ++dh)
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint4* at =
                reinterpret_cast<uint4*>(qrow + dh * (kM * 128) + ((c ^ (row & 7)) << 4));
            const uint4 u = *at;
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 f = bf16x2_to_float2(w[i]);
              const __half2 hv = __floats2half2_rn(f.x * up, f.y * up);  // exact products
              o[i] = *reinterpret_cast<const uint32_t*>(&hv);
            }
            *at = make_uint4(o[0], o[1], o[2], o[3]);
          }
        fence_proxy_async_smem();  // the S MMAs (async proxy) read Q next
      }
      __syncwarp();
      if (alive && lane == 0) mbar_arrive(bar_qc);
    }
    for (int j = 0; alive && j < nb; ++j) {
      // lanes leave the polling loop separately; the TMEM loads are
      // collective, and the warp takes one branch on the result
      if (!warp_wait_bounded(&bar_s[t], uint32_t(j) & 1, p.err, abort_flag)) {
        alive = false;
        break;
      }
      tc_fence_after();
      const int kbase = j * kNK;
      const bool diag = kbase + kNK - 1 > minpos;   // causal mask inside this block
      // Per score the softmax spends half a packed FMA, one ex2, half a
      // packed add and half a 16-bit-pair conversion (the P pass), and half
      // a 3-input max in the blocks that need a max pass; masks cost extra
      // only in diagonal blocks.  One warp's pass is a chain of dependent
      // steps per pair of scores and takes about 2.7 times its ex2 issue time
      // (ex2.approx.f32: 4 cycles per warp instruction per sub-partition).
      // tcgen05.ld / st are warp-collective: every lane runs them, whatever
      // its row (rows past the chunk compute unused values).
      // The block's 128 scores in one tcgen05.ld, kept in registers for both
      // passes: the max (four independent chains of 3-input max) and P.
      float sv[kNK];
      tmem_ld128(tmem + lane_base + colS, sv);
      if (diag) {
#pragma unroll
        for (int i = 0; i < kNK; ++i) sv[i] = (kbase + i <= pos) ? sv[i] : -INFINITY;
      }
      // Block max and lagged running max: the max moves only when the block
      // max exceeds it by more than 8 (log2 domain), so P <= 2^8.  The max
      // pass runs where a row has no running max yet (its first block);
      // elsewhere P is computed with the running max first and the block's
      // P sum decides: a sum above 2^15 = 128 x 2^8 means some P exceeds 2^8
      // (the running max must move), and the block is redone after a max
      // pass.  Otherwise every P <= 2^15 fits the 16-bit operand type and the
      // max pass is skipped.  Rows past the chunk take no part in either test.
      float alpha = 1.f, blk_sum = 0.f;
      bool do_max = PKV_PF_SKIP_MAX == 0 ||
                    __any_sync(0xffffffffu, row_valid && m_used == -INFINITY);
#pragma unroll 1
      for (;;) {
        if (do_max) {
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int i = 0; i < kNK; i += 8) {
            m4[0] = fmax3(m4[0], sv[i], sv[i + 1]);
            m4[1] = fmax3(m4[1], sv[i + 2], sv[i + 3]);
            m4[2] = fmax3(m4[2], sv[i + 4], sv[i + 5]);
            m4[3] = fmax3(m4[3], sv[i + 6], sv[i + 7]);
          }
          const float mx = row_valid ? fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * qm
                                     : -INFINITY;  // log2 domain (qm > 0)
          if (mx > m_used + 8.f) {
            const float a = fast_exp2(m_used - mx);  // 0 when m_used = -inf
            alpha *= a;
            m_used = mx;
            l_sum *= a;
          }
        }
        // P = 2^(s * qm - m) as 16-bit pairs over the first half of S's
        // columns (chunk c's pairs land in columns c/2 .. c/2 + 15; S is
        // already in registers); masked scores are -inf and give 0
        const float negm = m_used != -INFINITY ? -m_used : 0.f;
        const float2 qm2 = make_float2(qm, qm), nm2 = make_float2(negm, negm);
        float2 acc2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < kNK; c += 32) {
          uint32_t pw[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 x2 = __ffma2_rn(make_float2(sv[c + i], sv[c + i + 1]), qm2, nm2);
            const float2 e2 = make_float2(fast_exp2(x2.x), fast_exp2(x2.y));
            acc2[(i >> 1) & 1] = __fadd2_rn(acc2[(i >> 1) & 1], e2);
            if constexpr (FP8) {  // the PV product's operands are f16
              const __half2 ph = __floats2half2_rn(e2.x, e2.y);
              pw[i / 2] = *reinterpret_cast<const uint32_t*>(&ph);
            } else {
              const __nv_bfloat162 pb = __floats2bfloat162_rn(e2.x, e2.y);
              pw[i / 2] = *reinterpret_cast<const uint32_t*>(&pb);
            }
          }
          tmem_st16_async(tmem + lane_base + colS + c / 2, pw);
        }
        const float2 a2 = __fadd2_rn(acc2[0], acc2[1]);
        blk_sum = a2.x + a2.y;
        if (do_max || !__any_sync(0xffffffffu, row_valid && blk_sum > 32768.f)) break;
        do_max = true;   // (rare) redo the block after the max pass
        tmem_wait_st();  // the stores above land before the ones that replace them
      }
      l_sum += blk_sum;

      // O rescale (rare: the running max moves by > 2^8 only early in a row).
      // PV_{j-1} is complete: the commit behind "S_j ready" covers it.
      // tcgen05.ld/st are warp-collective: the whole warp rescales (rows that
      // do not need it multiply by 1).
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
        for (int cc = 0; cc < kD; cc += 32) {  // 32 columns at a time: bounded registers
          float o[32];
          tmem_ld32(tmem + lane_base + colO + cc, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(tmem + lane_base + colO + cc, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_p[t]);
    }

    // ---- epilogue: O / l -> bf16 ----------------------------------------------------
    // the last PV's commit also covers every earlier MMA of the producer
    if (nb > 0 && alive && warp_wait_bounded(&bar_o[t], 0, p.err, abort_flag)) {
      tc_fence_after();
      // v_scale (FP8 pools; 1 otherwise) applied once, with the normalisation
      const float vm = p.v_scales ? p.v_mult * __ldg(p.v_scales + h) : p.v_mult;
      const float inv = l_sum > 0.f ? vm / l_sum : 0.f;
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) +
                           (size_t(q0 + tok) * p.num_q_heads + size_t(h) * G + (row % G)) * kD;
#pragma unroll 1
      for (int cc = 0; cc < kD; cc += 32) {
        float o[32];
        tmem_ld32(tmem + lane_base + colO + cc, o);
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
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

namespace {

template <int D, bool FP8>
cudaError_t launch_prefill_d(const PrefillParams& p, const void* k_pool, const void* v_pool,
                             cudaStream_t stream) {
  using Lay = PfLayout<D, FP8>;
  const int G = p.num_q_heads / p.num_kv_heads;
  if (G < 1 || kM % G != 0 || kNK % p.block_size != 0) return cudaErrorNotSupported;
  if (p.num_blocks >= (1 << 30)) return cudaErrorInvalidValue;
  const uint64_t P = p.block_size, Hkv = p.num_kv_heads, E = 2;
  CUtensorMap tq, tk, tv;
  // q [T][Hkv][G][D] with box (64, G, 1, 128/G): rows ordered token-major, head-minor
  const auto kBf16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!make_map_4d(&tq, kBf16, p.q, D, G, Hkv, uint64_t(p.num_q_tokens), D * E, G * D * E,
                   Hkv * G * D * E, 64, uint32_t(G), 1, uint32_t(kM / G)))
    return cudaErrorInvalidValue;
  if constexpr (FP8) {
    // E4M3 pools [nb][Hkv][P][D] bytes with box (D, P, 1, 1): one page of
    // one kv head, unswizzled (row-major [key][D] in shared memory)
    const auto kU8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    if (!make_map_4d(&tk, kU8, k_pool, D, P, Hkv, uint64_t(p.num_blocks), D, P * D, Hkv * P * D,
                     uint32_t(D), uint32_t(P), 1, 1, CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
    if (!make_map_4d(&tv, kU8, v_pool, D, P, Hkv, uint64_t(p.num_blocks), D, P * D, Hkv * P * D,
                     uint32_t(D), uint32_t(P), 1, 1, CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  } else {
    // pools [nb][Hkv][P][D] with box (64, P, 1, 1): one page of one kv head
    if (!make_map_4d(&tk, kBf16, k_pool, D, P, Hkv, uint64_t(p.num_blocks), D * E, P * D * E,
                     Hkv * P * D * E, 64, uint32_t(P), 1, 1))
      return cudaErrorInvalidValue;
    if (!make_map_4d(&tv, kBf16, v_pool, D, P, Hkv, uint64_t(p.num_blocks), D * E, P * D * E,
                     Hkv * P * D * E, 64, uint32_t(P), 1, 1))
      return cudaErrorInvalidValue;
  }
  auto kern = prefill_kernel<D, FP8>;
  static std::atomic<bool> configured[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  e = once_per_device(configured, dev, [&] {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Lay::kSmemBytes);
  });
  if (e != cudaSuccess) return e;
  // one CTA per pair of 128-row query tiles of one kv head
  const int64_t ctas =
      int64_t((p.tiles_per_seq + kTiles - 1) / kTiles) * p.num_kv_heads * p.num_seqs;
  if (ctas > (int64_t(1) << 31) - 1) return cudaErrorInvalidValue;
  const dim3 grid{static_cast<unsigned>(ctas)};
  e = launch_pdl(kern, grid, dim3(kThreads), Lay::kSmemBytes, stream, tq, tk, tv, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams& p, const void* k_pool, const void* v_pool,
                           int num_sms, cudaStream_t stream) {
  (void)num_sms;
  if (p.head_dim == 128)
    return p.fp8 ? launch_prefill_d<128, true>(p, k_pool, v_pool, stream)
                 : launch_prefill_d<128, false>(p, k_pool, v_pool, stream);
  if (p.head_dim == 64)
    return p.fp8 ? launch_prefill_d<64, true>(p, k_pool, v_pool, stream)
                 : launch_prefill_d<64, false>(p, k_pool, v_pool, stream);
  return cudaErrorNotSupported;
}

}  // namespace pkv
