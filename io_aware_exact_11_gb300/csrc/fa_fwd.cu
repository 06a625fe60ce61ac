// fa_fwd.cu — forward attention on tcgen05 tensor cores (bf16 or E4M3 in,
// fp32 accumulate).
//
// One CTA owns two 128-row query tiles Q_0, Q_1 (256 consecutive rows) of one
// (b, h) and streams every key/value tile K_j, V_j (128 keys) past both, as in
// the two-loop structure of "FlashAttention：IO-aware 的注意力 kernel" §2 / §3.3
// (outer loop over query tiles, inner loop over key/value tiles).  Per key tile
// and per query tile i:
//   S_i = Q_i K_jᵀ                        tcgen05.mma into TMEM (fp32)
//   m_new = max(m, rowmax(σ S_i))         softmax warps, one thread per row
//   P̃ = e^(σS_i − m_new), ℓ = e^(m−m_new)ℓ + rowsum(P̃)      (§3.2)
//   O_i = e^(m−m_new) O_i + P̃ V_j         rescale in TMEM, then tcgen05.mma
// and after the last tile O_i/ℓ and LSE = m + ln ℓ are written once.
// Exponentials run in base 2 with σ·log2(e) folded into the scores.
//
// P̃ never leaves the SM's tensor memory: the softmax warps write it (bf16
// pairs, or four E4M3 codes, per 32-bit column) over the columns of S_i, and
// O_i += P̃_i V_j takes it from there as its A operand (V from shared memory).
// An M = N = 128 MMA with both operands in shared memory already uses the tensor
// cores' whole shared-memory read path, so a P̃ round trip through shared
// memory would cost tensor throughput.  Because S_i(j+1) overwrites P̃_i(j), the
// MMA warp issues it right after P̃_i(j)V_j (a thread's tcgen05 MMAs execute in
// order), and the two query tiles alternate:
//   … P̃_0(j)V_j, S_0(j+1), P̃_1(j)V_j, S_1(j+1), P̃_0(j+1)V_{j+1} …
// so each softmax warpgroup's exponentials overlap the other tile's MMAs.
// One tcgen05.commit per query tile and key tile: s_full[i] says S_i(j) is in
// TMEM and, because it follows P̃_i(j−1)V_{j−1}, that O_i is stable for a
// rescale; once S_1(j) is complete both tiles have read K_j and V_{j−1}, so a
// softmax thread of tile 1 hands those ring slots back to the producer.
//
// Warp roles (bf16: 320 threads, s0 = 2; E4M3: 384 threads, s0 = 4, warps 2, 3
// idle, and the softmax warpgroups take the registers the others give up):
//   warp 0       TMA producer: Q_0, Q_1 once, then K_0, V_0, K_1, V_1, … through
//                a shared-memory ring (5 slots at d = 128 bf16)
//   warp 1       TMEM owner and MMA issuer (the converged warp, one elected lane
//                issuing)
//   warps s0..s0+3    softmax / rescale / epilogue of Q_0 (warp w reads TMEM
//                     lanes 32·(w%4)…)
//   warps s0+4..s0+7  the same for Q_1
// TMEM: S_0 / P̃_0 (columns 0..127), S_1 / P̃_1 (128..255), O_0 (256..), O_1 (384..).
// Epilogue: each softmax thread writes its row of O/ℓ (bf16) into 128-byte-
// swizzled blocks in ring slots that no MMA still reads, and one thread per
// query tile stores the blocks with TMA, so O leaves in full lines instead of
// one 16-byte piece of 32 different rows per warp store (d = 64 keeps the
// direct stores, which measured faster there).
// Shared memory holds Q, K, V in the 128-byte-swizzled layout TMA writes:
// blocks of [128 rows][128 bytes].
//
// Causal mask (the lesson's §5 lab uses is_causal=True), bottom-right aligned:
// row i sees keys j <= i + (N_kv − N_q).  A CTA streams only the key tiles its
// last row can see; rows mask the rest of their diagonal tile with −∞.  The
// causal grid is (heads of a group, query-block rank, head group): heads are
// taken in groups small enough that a group's K and V stay in L2, and within a
// group the heaviest query blocks of every head go out first, so the short
// blocks fill each group's tail and the last group's fill the grid's.
//
// FP8 (E4M3) variant, FlashAttention-3's addition noted in the lesson (§3.3) and
// the interview notes (§四.5): Q, K, V arrive as E4M3 with per-tensor descale
// factors, the MMAs run as kind::f8f6f4 (32 elements per instruction, still 32
// bytes per k-step), P̃ is stored as E4M3 (lazy rescaling keeps it <= 256, inside
// E4M3's ±448) and ℓ sums the unrounded fp32 values; O leaves as bf16.
//
// P̃ goes over in two halves: a softmax warp whose rows keep their reference
// max signals p_half once P̃ of the first 64 keys is in TMEM, and the MMA warp
// issues that half of P̃_iV_j while the second half's exponentials are still
// running (a warp that rescales O signals both halves after the rescale, so no
// P̃V MMA reads O before it).  The MMAs and their order are unchanged, so the
// results are identical.  Measured on GB300 with the converged MMA warp: E4M3
// +10 %, bf16 +2 % at the prefill shape and +3 % causal (with a single
// issuing thread the same split had cost bf16 3–16 %).
//
// Lazy rescaling: a row keeps its reference max m until a tile's max exceeds
// it by more than kRescaleLog2 (base-2 units).  Until then P̃ = 2^(σ'S − m) is
// at most 2^kRescaleLog2 and O, ℓ keep accumulating against the same m, so the
// final O/ℓ and LSE = m + ln ℓ are the same numbers in exact arithmetic; only
// when the max really moves is O rescaled in TMEM by e^(m_old − m_new).
#include <cuda_fp8.h>

#include <algorithm>

#include "fa_kernels.h"
#include "sm103.cuh"

namespace fa {
namespace {

constexpr int kBM = 128;          // rows per query tile
constexpr int kQT = 2;            // query tiles per CTA
constexpr int kBN = 128;          // keys per key/value tile
constexpr int kTileBytes = 128 * 128;  // one [128 rows][128 bytes] swizzled block
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;
constexpr float kRescaleLog2 = 8.0f;
// E4M3 instances run 384 threads: warps 0-3 hand registers to the two softmax
// warpgroups (setmaxnreg).  setmaxnreg.inc waits until the block's pool can
// supply the registers, so the launcher checks the launch count first.
constexpr int kRegsLaunch = 168;
constexpr int kRegsControl = 56;
constexpr int kRegsSoftmax = 224;
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= (128 + kQT * 128) * kRegsLaunch, "register split");

template <int D, bool FP8>
struct FwdLayout {
  static constexpr int kEB = FP8 ? 1 : 2;            // bytes per element
  static constexpr int kNKB = D * kEB / 128;         // 128-byte blocks along the head dim
  static constexpr int kSlot = kNKB * kTileBytes;    // one Q, K or V tile
  static constexpr int kStepK = 32 / kEB;            // elements per MMA k-step (32 bytes)
  static constexpr int kRing = kSlot >= 32768 ? 5 : 8;
  // First softmax warp: bf16 instances 2 (warps 0, 1 are the producer and the
  // MMA issuer); E4M3 instances 4, so the softmax warps form whole warpgroups
  // for the register split (measured on GB300: E4M3 +4 %, bf16 unchanged to −2 %).
  static constexpr int kSoft0 = FP8 ? 4 : 2;
  static constexpr int kThreads = 32 * kSoft0 + kQT * 128;
  static constexpr int kQ = 0;
  static constexpr int kR = kQ + kQT * kSlot;
  static constexpr int kBar = kR + kRing * kSlot;
  static constexpr int kUsed = kBar + 512;
  // +1 KB so the base can be rounded up to 1024; at least 120 KB so only one
  // CTA (which owns all 512 TMEM columns) is resident per SM.
  static constexpr int kSmem = (kUsed + 1024) < 120 * 1024 ? 120 * 1024 : (kUsed + 1024);
};

struct FwdBars {
  uint64_t q_full;
  uint64_t r_full[8], r_empty[8];
  uint64_t s_full[kQT];  // S_i(j) in TMEM; after the last key tile: O_i complete
  uint64_t p_full[kQT];  // P̃_i(j) in TMEM (and O_i rescaled if needed)
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  uint64_t p_half[kQT];  // P̃_i(j) of the first 64 keys in TMEM, O_i rescaled
};

__device__ __forceinline__ unsigned int site(unsigned int s) { return (kKernFwd << 8) | s; }

// True on one lane of a converged warp (elect.sync).
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(pred));
  return pred != 0;
}

// Four fp32 values -> four E4M3 bytes (round to nearest even, saturating), the
// first value in the lowest byte.
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// GROUPED: the causal launch's head-grouped grid (see the launcher); the
// unmasked launches use the (query blocks, H, B) grid and GROUPED = false.
// The launcher pairs the two one to one, so the mask is a compile-time choice
// here (measured on GB300: +2.3 % at the unmasked prefill shape, +1.5 % causal
// over reading p.causal).
template <int D, bool FP8, bool GROUPED>
__global__ void __launch_bounds__(FwdLayout<D, FP8>::kThreads, 1) fwd_kernel(const __grid_constant__ FwdParams p) {
  using L = FwdLayout<D, FP8>;
  constexpr bool kCausal = GROUPED;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  FwdBars* bars = reinterpret_cast<FwdBars*>(smem + L::kBar);
  volatile int* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Grids are (query blocks, H, B); grouped (causal) grids are (heads of a
  // group, query-block rank, head group), heaviest blocks first within each
  // group, and the last group may be partly empty.
  int mt = kCausal ? static_cast<int>(gridDim.z - 1 - blockIdx.z) : static_cast<int>(blockIdx.x);
  int h = kCausal ? blockIdx.x : blockIdx.y;
  int b = kCausal ? blockIdx.y : blockIdx.z;
  if constexpr (GROUPED) {
    const int fh = static_cast<int>(blockIdx.z * gridDim.x + blockIdx.x);
    if (fh >= p.B * p.H) return;
    mt = static_cast<int>(gridDim.y - 1 - blockIdx.y);
    h = fh % p.H;
    b = fh / p.H;
  }
  const int m0 = mt * (kQT * kBM);
  const int off = p.Nkv - p.Nq;  // >= 0 whenever causal
  const int kv_end = kCausal ? min(p.Nkv, m0 + kQT * kBM + off) : p.Nkv;
  const int T = (kv_end + kBN - 1) / kBN;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < L::kRing; ++s) {
      mbar_init(&bars->r_full[s], 1);
      mbar_init(&bars->r_empty[s], 1);
    }
    for (int i = 0; i < kQT; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], 128);
      mbar_init(&bars->p_half[i], 128);
    }
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if constexpr (FP8) reg_dealloc<kRegsControl>();
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      mbar_arrive_expect_tx(&bars->q_full, kQT * L::kSlot);
      for (int i = 0; i < kQT; ++i)
        for (int kb = 0; kb < L::kNKB; ++kb)
          tma_load_4d(smem + L::kQ + i * L::kSlot + kb * kTileBytes, &p.tm_q, &bars->q_full, kb * (128 / L::kEB),
                      m0 + i * kBM, h, b);
      // Load t is K_{t/2} (t even) or V_{t/2} (t odd), into slot t % kRing.
      int issued = 0;
      for (int t = 0; t < 2 * T; ++t) {
        const int slot = t % L::kRing;
        const uint32_t u = t / L::kRing;
        if (!mbar_wait_inl(&bars->r_empty[slot], (u & 1) ^ 1, abort_flag, p.err, site(1))) break;
        mbar_arrive_expect_tx(&bars->r_full[slot], L::kSlot);
        const CUtensorMap* tm = (t & 1) ? &p.tm_v : &p.tm_k;
        for (int kb = 0; kb < L::kNKB; ++kb)
          tma_load_4d(smem + L::kR + slot * L::kSlot + kb * kTileBytes, tm, &bars->r_full[slot],
                      kb * (128 / L::kEB), (t >> 1) * kBN, h, b);
        ++issued;
      }
      if (*abort_flag) {
        mbar_wait_drain_inl(&bars->q_full, 0, 200000000ull);
        for (int t = (issued > L::kRing ? issued - L::kRing : 0); t < issued; ++t)
          mbar_wait_drain_inl(&bars->r_full[t % L::kRing], (t / L::kRing) & 1, 200000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if constexpr (FP8) reg_dealloc<kRegsControl>();
    // The whole warp runs the loop, so shared-memory descriptors are warp-
    // uniform values, and one elected lane issues; a single issuing thread
    // loses issue slots to the softmax warps of its sub-partition.  Every lane
    // takes the same wait results.  (Measured on GB300, together with the
    // inlined barrier waits: +4 % at the prefill shape, +7 % at d = 64, +6 %
    // for E4M3 and the causal mask; either change alone cost the unmasked bf16
    // d = 128 instance 3–5 %.)
    const bool leader = elect_one();
    auto agree = [](bool v) { return static_cast<bool>(__all_sync(0xffffffffu, v)); };
    {
      constexpr uint32_t kIdescS = FP8 ? idesc_e4m3_f32(kBM, kBN, false, false) : idesc_bf16_f32(kBM, kBN, false, false);
      constexpr uint32_t kIdescO = FP8 ? idesc_e4m3_f32(kBM, D, false, true) : idesc_bf16_f32(kBM, D, false, true);
      const uint32_t sQ = smem_u32(smem + L::kQ);
      const uint32_t sR = smem_u32(smem + L::kR);
      auto ring_wait = [&](int t, unsigned int where) -> bool {
        return agree(mbar_wait_inl(&bars->r_full[t % L::kRing], (t / L::kRing) & 1, abort_flag, p.err, site(where)));
      };
      auto issue_s = [&](int i, uint32_t kb) {  // S_i = Q_i K_jᵀ
        const uint32_t qb = sQ + i * L::kSlot;
#pragma unroll
        for (int kk = 0; kk < D / L::kStepK; ++kk) {
          const uint32_t o = (kk >> 2) * kTileBytes + (kk & 3) * 32;
          const uint64_t ad = sdesc_sw128(qb + o, 16, 1024), bd = sdesc_sw128(kb + o, 16, 1024);
          if (leader) {
            if (FP8)
              mma_e4m3_ss(tmem + i * kBN, ad, bd, kIdescS, kk > 0 ? 1u : 0u);
            else
              mma_bf16_ss(tmem + i * kBN, ad, bd, kIdescS, kk > 0 ? 1u : 0u);
          }
        }
      };
      bool ok = agree(mbar_wait_inl(&bars->q_full, 0, abort_flag, p.err, site(5))) && ring_wait(0, 6);
      if (ok) {
        tc_fence_after();
        for (int i = 0; i < kQT; ++i) {
          issue_s(i, sR);
          if (leader) mma_commit(&bars->s_full[i]);
        }
      }
      for (int j = 0; ok && j < T; ++j) {
        const int tv = 2 * j + 1;
        if (!(ok = ring_wait(tv, 3))) break;
        const uint32_t vb = sR + (tv % L::kRing) * L::kSlot;
        const bool next = j + 1 < T;
        const uint32_t kb = sR + ((tv + 1) % L::kRing) * L::kSlot;
        for (int i = 0; i < kQT && ok; ++i) {
          if (!(ok = agree(mbar_wait_inl(&bars->p_half[i], j & 1, abort_flag, p.err, site(4)))))
            break;
          if (i == 0 && next && !(ok = ring_wait(tv + 1, 6))) break;
          tc_fence_after();
          // O_i += P̃_i V_j: A = P̃_i from S_i's TMEM columns (32 bytes of keys = 8
          // columns per k-step), B = V_j read MN-major (head dim contiguous).
          constexpr int kHalf = kBN / L::kStepK / 2;
#pragma unroll
          for (int kk = 0; kk < kBN / L::kStepK; ++kk) {
            if (kk == kHalf) {  // the second half of P̃_i
              if (!(ok = agree(mbar_wait_inl(&bars->p_full[i], j & 1, abort_flag, p.err, site(4))))) break;
              tc_fence_after();
            }
            const uint64_t bd = sdesc_sw128(vb + kk * L::kStepK * 128, kTileBytes, 1024);
            const uint32_t acc = (j > 0 || kk > 0) ? 1u : 0u;
            if (leader) {
              if (FP8)
                mma_e4m3_ts(tmem + kColO + i * 128, tmem + i * kBN + kk * 8, bd, kIdescO, acc);
              else
                mma_bf16_ts(tmem + kColO + i * 128, tmem + i * kBN + kk * 8, bd, kIdescO, acc);
            }
          }
          if (!ok) break;
          if (next) issue_s(i, kb);
          if (leader) mma_commit(&bars->s_full[i]);
        }
      }
      if (*abort_flag) {
        if (leader) mma_commit(&bars->drain);
        mbar_wait_drain_inl(&bars->drain, 0, 200000000ull);
      }
    }
  } else if (FP8 && warp < L::kSoft0) {
    reg_dealloc<kRegsControl>();  // idle until the end
  } else {
    // ------------------------------------------------- softmax / epilogue
    if constexpr (FP8) reg_alloc<kRegsSoftmax>();
    const int qt = (warp - L::kSoft0) >> 2;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t s_col = qt * kBN;
    const uint32_t o_col = kColO + qt * 128;
    const float sl2 = p.scale_log2;
    const bool releaser = qt == kQT - 1 && wq == 0 && lane == 0;
    float m_run = -INFINITY;
    float l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < T; ++j) {
      ok = mbar_wait_inl(&bars->s_full[qt], j & 1, abort_flag, p.err, site(8));
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      // S_1(j) is complete, so K_j and V_{j−1} have been read by both tiles.
      if (releaser) {
        mbar_arrive(&bars->r_empty[(2 * j) % L::kRing]);
        if (j >= 1) mbar_arrive(&bars->r_empty[(2 * j - 1) % L::kRing]);
      }
      tc_fence_after();
      float s[128];
      {
        uint32_t r0[32], r1[32], r2[32], r3[32];
        const uint32_t sa = tmem + lane_base + s_col;
        tmem_ld32(sa + 0, r0);
        tmem_ld32(sa + 32, r1);
        tmem_ld32(sa + 64, r2);
        tmem_ld32(sa + 96, r3);
        tmem_wait_ld();
        reg_fence(r0);
        reg_fence(r1);
        reg_fence(r2);
        reg_fence(r3);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          s[c] = __uint_as_float(r0[c]);
          s[32 + c] = __uint_as_float(r1[c]);
          s[64 + c] = __uint_as_float(r2[c]);
          s[96 + c] = __uint_as_float(r3[c]);
        }
      }
      int kv_valid = p.Nkv - j * kBN;
      if (kCausal) kv_valid = min(kv_valid, m0 + qt * kBM + row + off + 1 - j * kBN);
      if (kv_valid < kBN) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c >= kv_valid) s[c] = -INFINITY;
      }
      // Row max: four independent chains of three-input maxima.
      float mx4[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) mx4[i] = fmax3(s[i], s[4 + i], s[8 + i]);
#pragma unroll
      for (int c = 12; c < 124; c += 8) {
#pragma unroll
        for (int i = 0; i < 4; ++i) mx4[i] = fmax3(mx4[i], s[c + i], s[c + 4 + i]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) mx4[i] = fmaxf(mx4[i], s[124 + i]);
      const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      const float m_cand = fmaxf(m_run, mx * sl2);
      const bool need = m_cand > m_run + kRescaleLog2;  // always true while m_run = −∞
      const float m_new = need ? m_cand : m_run;
      const float corr = need ? ex2_approx(m_run - m_new) : 1.f;
      const bool resc = j >= 1 && __any_sync(0xffffffffu, need);  // this warp rescales O
      float rs[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) rs[i] = 0.f;
      const float nm = -m_new;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        // P̃ for keys 64·hf … 64·hf+63 into TMEM: 32 columns of bf16 pairs, or
        // 16 columns of four E4M3 codes (first key in the lowest bits).
        uint32_t w[32];
#pragma unroll
        for (int c = 64 * hf; c < 64 * hf + 64; c += 8) {
          float x[8];
#pragma unroll
          for (int i = 0; i < 8; i += 2) {
            ffma2(x[i], x[i + 1], s[c + i], s[c + i + 1], sl2, sl2, nm, nm);
            x[i] = ex2_approx(x[i]);
            x[i + 1] = ex2_approx(x[i + 1]);
            fadd2(rs[i], rs[i + 1], rs[i], rs[i + 1], x[i], x[i + 1]);
          }
          const int wc = (c - 64 * hf) >> (FP8 ? 2 : 1);
          if (FP8) {
            w[wc] = pack_e4m3x4(x[0], x[1], x[2], x[3]);
            w[wc + 1] = pack_e4m3x4(x[4], x[5], x[6], x[7]);
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) w[wc + i] = pack_bf16x2(x[2 * i], x[2 * i + 1]);
          }
        }
        if (FP8)
          tmem_st16(tmem + lane_base + s_col + 16 * hf, reinterpret_cast<uint32_t(&)[16]>(w));
        else
          tmem_st32(tmem + lane_base + s_col + 32 * hf, w);
        if (hf == 0 && !resc) {  // the first half goes early
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&bars->p_half[qt]);
        }
      }
      const float rsum = ((rs[0] + rs[1]) + (rs[2] + rs[3])) + ((rs[4] + rs[5]) + (rs[6] + rs[7]));
      l_run = l_run * corr + rsum;
      // O_i is stable here (its last update came before S_i(j)); rescale it in
      // TMEM only when some row of this warp moved its reference max.
      if (resc) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          const uint32_t oa = tmem + lane_base + o_col + c * 32;
          tmem_ld32(oa, r);
          tmem_wait_ld();
          reg_fence(r);
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * corr);
          tmem_st32(oa, r);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      if (resc) mbar_arrive(&bars->p_half[qt]);
      mbar_arrive(&bars->p_full[qt]);
      m_run = m_new;
    }
    if constexpr (D == 64) {
      // Head dim 64: each thread writes its 128-byte row directly (measured
      // faster here than staging through shared memory).
      if (ok) {
        ok = mbar_wait_inl(&bars->s_full[qt], T & 1, abort_flag, p.err, site(10));
        if (__all_sync(0xffffffffu, ok)) {
          tc_fence_after();
          const float inv = p.o_scale / l_run;
          const int grow = m0 + qt * kBM + row;
          __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.o) + b * p.o_sb + h * p.o_sh +
                                static_cast<int64_t>(grow) * p.o_sn;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(tmem + lane_base + o_col + c * 32, r);
            tmem_wait_ld();
            reg_fence(r);
            if (grow < p.Nq) {
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4) {
                uint4 v;
                v.x = pack_bf16x2(__uint_as_float(r[8 * q4 + 0]) * inv, __uint_as_float(r[8 * q4 + 1]) * inv);
                v.y = pack_bf16x2(__uint_as_float(r[8 * q4 + 2]) * inv, __uint_as_float(r[8 * q4 + 3]) * inv);
                v.z = pack_bf16x2(__uint_as_float(r[8 * q4 + 4]) * inv, __uint_as_float(r[8 * q4 + 5]) * inv);
                v.w = pack_bf16x2(__uint_as_float(r[8 * q4 + 6]) * inv, __uint_as_float(r[8 * q4 + 7]) * inv);
                *reinterpret_cast<uint4*>(orow + c * 32 + q4 * 8) = v;
              }
            }
          }
          if (p.lse != nullptr && grow < p.Nq)
            p.lse[(static_cast<int64_t>(b) * p.H + h) * p.Nq + grow] = (m_run + __log2f(l_run)) * 0.69314718055994531f;
        }
      }
    } else {
      // O goes out through shared memory and TMA: the ring slots are idle once
      // O is complete.  Each thread writes its row into 128-byte-swizzled
      // [128 rows][64 columns] blocks, then one thread stores the blocks.  Every
      // warp of the warpgroup reaches the barrier once, even after an abort (the
      // store is then skipped), so none waits for a warp that left.
      bool eok = false;
      if (ok) {
        ok = mbar_wait_inl(&bars->s_full[qt], T & 1, abort_flag, p.err, site(10));
        eok = __all_sync(0xffffffffu, ok);
      }
      const int grow = m0 + qt * kBM + row;
      // Staging blocks go to the ring slots the next loads would have used,
      // (2T + n) mod kRing: those last held K/V tiles of key tile T−3 or earlier,
      // which every issued MMA has finished with, and at most 4 < kRing slots are
      // taken, so they never reach slot (2T−1) mod kRing, whose V tile the other
      // query tile's last P̃V may still be reading.
      constexpr int kBps = L::kSlot / kTileBytes;  // 16 KB blocks per ring slot
      auto stage_block = [&](int n) -> uint8_t* {    // n = qt·(D/64) + kb
        return smem + L::kR + ((2 * T + n / kBps) % L::kRing) * L::kSlot + (n % kBps) * kTileBytes;
      };
      static_assert(kQT * (D / 64) / (L::kSlot / kTileBytes) + 1 <= L::kRing, "staging slots");
      if (eok) {
        tc_fence_after();
        const float inv = p.o_scale / l_run;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_base + o_col + c * 32, r);
          tmem_wait_ld();
          reg_fence(r);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(r[8 * q4 + 0]) * inv, __uint_as_float(r[8 * q4 + 1]) * inv);
            v.y = pack_bf16x2(__uint_as_float(r[8 * q4 + 2]) * inv, __uint_as_float(r[8 * q4 + 3]) * inv);
            v.z = pack_bf16x2(__uint_as_float(r[8 * q4 + 4]) * inv, __uint_as_float(r[8 * q4 + 5]) * inv);
            v.w = pack_bf16x2(__uint_as_float(r[8 * q4 + 6]) * inv, __uint_as_float(r[8 * q4 + 7]) * inv);
            const int ch = c * 4 + q4;  // 16-byte chunk of the row
            *reinterpret_cast<uint4*>(stage_block(qt * (D / 64) + (ch >> 3)) + row * 128 + (((ch & 7) ^ (row & 7)) << 4)) =
                v;
          }
        }
        if (p.lse != nullptr && grow < p.Nq)
          p.lse[(static_cast<int64_t>(b) * p.H + h) * p.Nq + grow] = (m_run + __log2f(l_run)) * 0.69314718055994531f;
      }
      fence_proxy_async_smem();
      named_sync(1 + qt, 128);
      if (wq == 0 && lane == 0 && !*abort_flag && m0 + qt * kBM < p.Nq) {  // rows past N_q are clipped
        for (int kb = 0; kb < D / 64; ++kb)
          tma_store_4d(&p.tm_o, stage_block(qt * (D / 64) + kb), kb * 64, m0 + qt * kBM, h, b);
        bulk_commit();
        bulk_wait_read();  // the source must stay until read; the writes complete with the grid
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool FP8, bool GROUPED>
cudaError_t check_regs() {
  if (!FP8) return cudaSuccess;
  cudaFuncAttributes a;
  const cudaError_t e = cudaFuncGetAttributes(&a, fwd_kernel<D, FP8, GROUPED>);
  if (e != cudaSuccess) return e;
  return a.numRegs < kRegsLaunch ? cudaErrorInvalidConfiguration : cudaSuccess;
}

template <int D, bool FP8>
cudaError_t launch_impl(const FwdParams& p, cudaStream_t stream) {
  using L = FwdLayout<D, FP8>;
  const unsigned n_mt = (p.Nq + kQT * kBM - 1) / (kQT * kBM);
  if (!p.causal) {
    cudaError_t e =
        cudaFuncSetAttribute(fwd_kernel<D, FP8, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmem);
    if (e != cudaSuccess) return e;
    if ((e = check_regs<D, FP8, false>()) != cudaSuccess) return e;
    fwd_kernel<D, FP8, false><<<dim3(n_mt, p.H, p.B), L::kThreads, L::kSmem, stream>>>(p);
    return cudaGetLastError();
  }
  cudaError_t e =
      cudaFuncSetAttribute(fwd_kernel<D, FP8, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmem);
  if (e != cudaSuccess) return e;
  if ((e = check_regs<D, FP8, true>()) != cudaSuccess) return e;
  dim3 grid;
  {
    // Heads per group: their K and V together about 32 MiB, a quarter of L2.
    const int64_t bh = static_cast<int64_t>(p.B) * p.H;
    const int64_t per_head = 2ll * p.Nkv * D * (FP8 ? 1 : 2);
    int64_t g = std::max<int64_t>(1, (int64_t{32} << 20) / per_head);
    g = std::min(g, bh);
    g = std::max(g, (bh + 65534) / 65535);  // the group count must fit the z axis
    grid = dim3(static_cast<unsigned>(g), n_mt, static_cast<unsigned>((bh + g - 1) / g));
  }
  fwd_kernel<D, FP8, true><<<grid, L::kThreads, L::kSmem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_bf16(int d, const FwdParams& p, cudaStream_t stream) {
  if (d == 128) return launch_impl<128, false>(p, stream);
  if (d == 64) return launch_impl<64, false>(p, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_fwd_fp8(int d, const FwdParams& p, cudaStream_t stream) {
  if (d == 128) return launch_impl<128, true>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
