// fa_fwd_d64.cu — unmasked bf16 forward at head dim 64 on tcgen05 tensor cores.
//
// Same method as fa_fwd.cu (exact softmax attention with the online-softmax
// recurrence of "FlashAttention：IO-aware 的注意力 kernel", inference-learning-path
// .pages.dev, §3.2; lazy rescaling of O in TMEM), laid out for d = 64.  At d = 64
// an MMA over a 128-key tile is half as long as at d = 128 while the softmax of
// the tile is not, so two query tiles cannot keep the tensor pipe busy.  Here a
// CTA owns QT query tiles of 128 rows and streams 64-key tiles: each tile's
// softmax (64 exponentials per row) runs while the other QT − 1 tiles' MMAs run.
// TMEM holds every tile's S (64 fp32 columns, later P̃ as bf16 pairs over its
// first 32) and O (64 columns): QT · 128 ≤ 512 columns.
//
// Warp roles (64 + 128·QT threads): warp 0 TMA producer (Q_0 … Q_{QT−1} once,
// then K_0, V_0, K_1, V_1, … into a ring of 8 KB slots); warp 1 TMEM owner and
// MMA issuer (the converged warp with one elected lane issuing, so descriptors
// are warp-uniform and issue does not lose slots to the softmax warps of its
// sub-partition); QT softmax warpgroups, one per query tile, thread = row.  Per
// key tile j the MMA warp issues, for i = 0 … QT−1, P̃_i(j)V_j then
// S_i(j+1) = Q_i K_{j+1}ᵀ (S_i(j+1) overwrites P̃_i(j), which the in-order tensor
// pipe has read first), and commits s_full[i], which says both "S_i(j+1)
// ready" and "O_i stable".  Once S of the last tile for key tile j is
// complete, K_j and V_{j−1} are free.  The epilogue divides by ℓ and stores each
// row of O (128 bytes) directly, with LSE = (m + log2 ℓ)·ln 2.
#include <type_traits>

#include "fa_kernels.h"
#include "sm103.cuh"

namespace fa {
namespace {

constexpr int kBM = 128;                // rows per query tile
constexpr int kBN = 64;                 // keys per key/value tile
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;
constexpr int kQBytes = kBM * 128;      // one Q tile: [128 rows][64 bf16], 128-byte swizzle
constexpr int kSlot = kBN * 128;        // one K or V tile: [64 rows][64 bf16]

template <int QT>
struct D64Cfg {
  static constexpr int kThreads = 64 + QT * 128;
  static constexpr uint32_t kColO = QT * kBN;  // O_i at kColO + 64·i
  static constexpr int kRing = 12;
  static constexpr int kOffQ = 0;
  static constexpr int kOffR = kOffQ + QT * kQBytes;
  static constexpr int kOffBar = kOffR + kRing * kSlot;
  static constexpr int kSmem = kOffBar + 512 + 1024;
  static_assert(QT * 2 * kBN <= static_cast<int>(kTmemCols), "TMEM columns");
};

template <int QT>
struct D64Bars {
  uint64_t q_full;
  uint64_t r_full[D64Cfg<QT>::kRing], r_empty[D64Cfg<QT>::kRing];
  uint64_t s_full[QT];  // S_i(j) in TMEM; after the last key tile: O_i complete
  uint64_t p_full[QT];  // P̃_i(j) in TMEM (and O_i rescaled if needed)
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ unsigned int site(unsigned int s) { return (kKernFwd << 8) | (0x40u | s); }

// True on one lane of a converged warp (elect.sync).
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(pred));
  return pred != 0;
}

template <int QT>
__global__ void __launch_bounds__(D64Cfg<QT>::kThreads, 1) fwd_d64_kernel(const __grid_constant__ FwdParams p) {
  using C = D64Cfg<QT>;
  using Bars = D64Bars<QT>;
  static_assert(sizeof(Bars) <= 512, "barrier block");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kOffBar);
  volatile int* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int mt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int m0 = mt * (QT * kBM);
  const int T = (p.Nkv + kBN - 1) / kBN;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < C::kRing; ++s) {
      mbar_init(&bars->r_full[s], 1);
      mbar_init(&bars->r_empty[s], 1);
    }
    for (int i = 0; i < QT; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], 128);
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
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      mbar_arrive_expect_tx(&bars->q_full, QT * kQBytes);
      for (int i = 0; i < QT; ++i)
        tma_load_4d(smem + C::kOffQ + i * kQBytes, &p.tm_q, &bars->q_full, 0, m0 + i * kBM, h, b);
      // Load t is K_{t/2} (t even) or V_{t/2} (t odd), into slot t % kRing.
      int issued = 0;
      for (int t = 0; t < 2 * T; ++t) {
        const int slot = t % C::kRing;
        const uint32_t u = t / C::kRing;
        if (!mbar_wait_inl(&bars->r_empty[slot], (u & 1) ^ 1, abort_flag, p.err, site(1))) break;
        mbar_arrive_expect_tx(&bars->r_full[slot], kSlot);
        tma_load_4d(smem + C::kOffR + slot * kSlot, (t & 1) ? &p.tm_v : &p.tm_k, &bars->r_full[slot], 0,
                    (t >> 1) * kBN, h, b);
        ++issued;
      }
      if (*abort_flag) {
        mbar_wait_drain_inl(&bars->q_full, 0, 200000000ull);
        for (int t = (issued > C::kRing ? issued - C::kRing : 0); t < issued; ++t)
          mbar_wait_drain_inl(&bars->r_full[t % C::kRing], (t / C::kRing) & 1, 200000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const bool leader = elect_one();
    auto agree = [](bool v) { return static_cast<bool>(__all_sync(0xffffffffu, v)); };
    constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, false, false);
    constexpr uint32_t kIdescO = idesc_bf16_f32(kBM, 64, false, true);
    const uint32_t sQ = smem_u32(smem + C::kOffQ);
    const uint32_t sR = smem_u32(smem + C::kOffR);
    auto ring_wait = [&](int t, unsigned int where) -> bool {
      return agree(mbar_wait_inl(&bars->r_full[t % C::kRing], (t / C::kRing) & 1, abort_flag, p.err, site(where)));
    };
    auto issue_s = [&](int i, uint32_t kb) {  // S_i = Q_i K_jᵀ: 64 head dims in 4 k-steps of 16
      const uint32_t qb = sQ + i * kQBytes;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t ad = sdesc_sw128(qb + kk * 32, 16, 1024), bd = sdesc_sw128(kb + kk * 32, 16, 1024);
        if (leader) mma_bf16_ss(tmem + i * kBN, ad, bd, kIdescS, kk > 0 ? 1u : 0u);
      }
    };
    bool ok = agree(mbar_wait_inl(&bars->q_full, 0, abort_flag, p.err, site(5))) && ring_wait(0, 6);
    if (ok) {
      tc_fence_after();
      for (int i = 0; i < QT; ++i) {
        issue_s(i, sR);
        if (leader) mma_commit(&bars->s_full[i]);
      }
    }
    for (int j = 0; ok && j < T; ++j) {
      const int tv = 2 * j + 1;
      if (!(ok = ring_wait(tv, 3))) break;
      const uint32_t vb = sR + (tv % C::kRing) * kSlot;
      const bool next = j + 1 < T;
      const uint32_t kb = sR + ((tv + 1) % C::kRing) * kSlot;
      for (int i = 0; i < QT && ok; ++i) {
        if (!(ok = agree(mbar_wait_inl(&bars->p_full[i], j & 1, abort_flag, p.err, site(4))))) break;
        if (i == 0 && next && !(ok = ring_wait(tv + 1, 6))) break;
        tc_fence_after();
        // O_i += P̃_i V_j: A = P̃_i from S_i's TMEM columns (16 keys = 8 columns
        // per k-step), B = V_j read MN-major (the 64 head dims contiguous).
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint64_t bd = sdesc_sw128(vb + kk * 2048, kSlot, 1024);
          if (leader)
            mma_bf16_ts(tmem + C::kColO + i * 64, tmem + i * kBN + kk * 8, bd, kIdescO, (j > 0 || kk > 0) ? 1u : 0u);
        }
        if (next) issue_s(i, kb);
        if (leader) mma_commit(&bars->s_full[i]);
      }
    }
    if (*abort_flag) {
      if (leader) mma_commit(&bars->drain);
      mbar_wait_drain_inl(&bars->drain, 0, 200000000ull);
    }
  } else {
    // ------------------------------------------------- softmax / epilogue
    const int qt = (warp - 2) >> 2;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t s_col = qt * kBN;
    const uint32_t o_col = C::kColO + qt * 64;
    const float sl2 = p.scale_log2;
    const bool releaser = qt == QT - 1 && wq == 0 && lane == 0;
    float m_run = -INFINITY;
    float l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < T; ++j) {
      ok = mbar_wait_inl(&bars->s_full[qt], j & 1, abort_flag, p.err, site(8));
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      // S of the last query tile for key tile j is complete: every tile has read
      // K_j, and every P̃·V_{j−1} (issued before it) is done.
      if (releaser) {
        mbar_arrive(&bars->r_empty[(2 * j) % C::kRing]);
        if (j >= 1) mbar_arrive(&bars->r_empty[(2 * j - 1) % C::kRing]);
      }
      tc_fence_after();
      float s[64];
      {
        uint32_t r0[32], r1[32];
        tmem_ld32(tmem + lane_base + s_col, r0);
        tmem_ld32(tmem + lane_base + s_col + 32, r1);
        tmem_wait_ld();
        reg_fence(r0);
        reg_fence(r1);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          s[c] = __uint_as_float(r0[c]);
          s[32 + c] = __uint_as_float(r1[c]);
        }
      }
      const int kv_valid = p.Nkv - j * kBN;
      if (kv_valid < kBN) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c >= kv_valid) s[c] = -INFINITY;
      }
      // Row max: four chains of three-input maxima.
      float mx4[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) mx4[i] = fmax3(s[i], s[4 + i], s[8 + i]);
#pragma unroll
      for (int c = 12; c < 60; c += 8) {
#pragma unroll
        for (int i = 0; i < 4; ++i) mx4[i] = fmax3(mx4[i], s[c + i], s[c + 4 + i]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) mx4[i] = fmaxf(mx4[i], s[60 + i]);
      const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      const float m_cand = fmaxf(m_run, mx * sl2);
      const bool need = m_cand > m_run + kRescaleLog2;  // always true while m_run = −∞
      const float m_new = need ? m_cand : m_run;
      const float corr = need ? ex2_approx(m_run - m_new) : 1.f;
      float rs[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) rs[i] = 0.f;
      const float nm = -m_new;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        // P̃ for keys 32·hf … 32·hf+31 into TMEM: 16 columns of bf16 pairs.
        uint32_t w[16];
#pragma unroll
        for (int c = 32 * hf; c < 32 * hf + 32; c += 8) {
          float x[8];
#pragma unroll
          for (int i = 0; i < 8; i += 2) {
            ffma2(x[i], x[i + 1], s[c + i], s[c + i + 1], sl2, sl2, nm, nm);
            x[i] = ex2_approx(x[i]);
            x[i + 1] = ex2_approx(x[i + 1]);
            fadd2(rs[i], rs[i + 1], rs[i], rs[i + 1], x[i], x[i + 1]);
          }
          const int wc = (c - 32 * hf) >> 1;
#pragma unroll
          for (int i = 0; i < 4; ++i) w[wc + i] = pack_bf16x2(x[2 * i], x[2 * i + 1]);
        }
        tmem_st16(tmem + lane_base + s_col + 16 * hf, w);
      }
      const float rsum = ((rs[0] + rs[1]) + (rs[2] + rs[3])) + ((rs[4] + rs[5]) + (rs[6] + rs[7]));
      l_run = l_run * corr + rsum;
      // O_i is stable here (its last update came before S_i(j)); rescale it in
      // TMEM only when some row of this warp moved its reference max.
      if (j >= 1 && __any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
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
      mbar_arrive(&bars->p_full[qt]);
      m_run = m_new;
    }
    // Epilogue: O_i is complete once the commit after the last P̃·V arrives.
    if (ok) {
      ok = mbar_wait_inl(&bars->s_full[qt], T & 1, abort_flag, p.err, site(10));
      if (__all_sync(0xffffffffu, ok)) {
        tc_fence_after();
        const float inv = p.o_scale / l_run;
        const int grow = m0 + qt * kBM + row;
        __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.o) + b * p.o_sb + h * p.o_sh +
                              static_cast<int64_t>(grow) * p.o_sn;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
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
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_fwd_d64_tiles(int query_tiles, const FwdParams& p, cudaStream_t stream) {
  auto go = [&](auto qt_tag) -> cudaError_t {
    constexpr int QT = decltype(qt_tag)::value;
    using C = D64Cfg<QT>;
    cudaError_t e = cudaFuncSetAttribute(fwd_d64_kernel<QT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    const unsigned n_mt = (p.Nq + QT * kBM - 1) / (QT * kBM);
    fwd_d64_kernel<QT><<<dim3(n_mt, p.H, p.B), C::kThreads, C::kSmem, stream>>>(p);
    return cudaGetLastError();
  };
  if (p.causal) return cudaErrorInvalidValue;  // the causal mask stays on fa_fwd.cu's kernel
  if (query_tiles == 4) return go(std::integral_constant<int, 4>{});
  if (query_tiles == 3) return go(std::integral_constant<int, 3>{});
  return cudaErrorInvalidValue;
}

}  // namespace fa
