// fa_fwd.cu — forward attention on tcgen05 tensor cores (bf16 in, fp32 accumulate).
//
// One CTA owns a 128-row tile Q_i of one (b, h) and streams all key/value tiles
// K_j, V_j (128 keys each) past it, as in the two-loop structure of
// "FlashAttention：IO-aware 的注意力 kernel" §2 / §3.3 (outer loop over query
// tiles, inner loop over key/value tiles).  Per key tile:
//   S_j = Q_i K_jᵀ                       tcgen05.mma into TMEM (fp32)
//   m_new = max(m, rowmax(σ S_j))        softmax warps, one thread per row
//   P̃ = e^(σS_j − m_new), ℓ = e^(m−m_new)ℓ + rowsum(P̃)      (§3.2)
//   O = e^(m−m_new) O + P̃ V_j            rescale in TMEM, then tcgen05.mma
// and after the last tile O/ℓ and LSE = m + ln ℓ are written once.
// Exponentials run in base 2 with σ·log2(e) folded into the scores.
//
// Warp roles (192 threads):
//   warp 0      TMA producer: Q once, then K_j / V_j into a 2-stage ring
//   warp 1      TMEM owner and MMA issuer (one thread)
//   warps 2..5  softmax / rescale / epilogue; warp w reads TMEM lanes 32·(w%4)+…
// TMEM: two S buffers (columns 0..255) so S_{j+1} is computed while the
// softmax of tile j runs, and the O accumulator at column 256.
// Shared memory holds every operand in the 128-byte-swizzled layout TMA writes:
// blocks of [128 rows][64 bf16].
#include "fa_kernels.h"
#include "sm103.cuh"

namespace fa {
namespace {

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kTileBytes = 128 * 128;  // one [128 rows][64 bf16] swizzled block
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;

template <int D>
struct FwdLayout {
  static constexpr int kNKB = D / 64;  // 128-byte blocks along the head dim
  static constexpr int kStages = 2;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kNKB * kTileBytes;
  static constexpr int kV = kK + kStages * kNKB * kTileBytes;
  static constexpr int kP = kV + kStages * kNKB * kTileBytes;
  static constexpr int kBar = kP + 2 * kTileBytes;
  static constexpr int kUsed = kBar + 512;
  // +1 KB so the base can be rounded up to 1024; at least 120 KB so only one
  // CTA (which owns all 512 TMEM columns) is resident per SM.
  static constexpr int kSmem = (kUsed + 1024) < 120 * 1024 ? 120 * 1024 : (kUsed + 1024);
};

struct FwdBars {
  uint64_t q_full;
  uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full, o_done, drain;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ unsigned int site(unsigned int s) { return (kKernFwd << 8) | s; }

template <int D>
__global__ void __launch_bounds__(kThreads, 1) fwd_bf16_kernel(const __grid_constant__ FwdParams p) {
  using L = FwdLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  FwdBars* bars = reinterpret_cast<FwdBars*>(smem + L::kBar);
  volatile int* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * kBM;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int T = (p.Nkv + kBN - 1) / kBN;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->s_free[s], 128);
    }
    mbar_init(&bars->p_full, 128);
    mbar_init(&bars->o_done, 1);
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
      mbar_arrive_expect_tx(&bars->q_full, L::kNKB * kTileBytes);
      for (int kb = 0; kb < L::kNKB; ++kb)
        tma_load_4d(smem + L::kQ + kb * kTileBytes, &p.tm_q, &bars->q_full, kb * 64, m0, h, b);
      int nk = 0, nv = 0;
      for (int j = 0; j < T; ++j) {
        const int s = j % L::kStages;
        const uint32_t ph = (j / L::kStages) & 1;
        if (!mbar_wait(&bars->k_empty[s], ph ^ 1, abort_flag, p.err, site(1))) break;
        mbar_arrive_expect_tx(&bars->k_full[s], L::kNKB * kTileBytes);
        for (int kb = 0; kb < L::kNKB; ++kb)
          tma_load_4d(smem + L::kK + (s * L::kNKB + kb) * kTileBytes, &p.tm_k, &bars->k_full[s], kb * 64,
                      j * kBN, h, b);
        ++nk;
        if (!mbar_wait(&bars->v_empty[s], ph ^ 1, abort_flag, p.err, site(2))) break;
        mbar_arrive_expect_tx(&bars->v_full[s], L::kNKB * kTileBytes);
        for (int kb = 0; kb < L::kNKB; ++kb)
          tma_load_4d(smem + L::kV + (s * L::kNKB + kb) * kTileBytes, &p.tm_v, &bars->v_full[s], kb * 64,
                      j * kBN, h, b);
        ++nv;
      }
      if (*abort_flag) {
        // Let every copy this thread started land before the CTA exits.
        mbar_wait_drain(&bars->q_full, 0, 200000000ull);
        for (int t = (nk > L::kStages ? nk - L::kStages : 0); t < nk; ++t)
          mbar_wait_drain(&bars->k_full[t % L::kStages], (t / L::kStages) & 1, 200000000ull);
        for (int t = (nv > L::kStages ? nv - L::kStages : 0); t < nv; ++t)
          mbar_wait_drain(&bars->v_full[t % L::kStages], (t / L::kStages) & 1, 200000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, false, false);
      constexpr uint32_t kIdescO = idesc_bf16_f32(kBM, D, false, true);
      const uint32_t sQ = smem_u32(smem + L::kQ);
      const uint32_t sK = smem_u32(smem + L::kK);
      const uint32_t sV = smem_u32(smem + L::kV);
      const uint32_t sP = smem_u32(smem + L::kP);
      auto issue_pv = [&](int i) -> bool {
        const int s = i % L::kStages;
        const uint32_t ph = (i / L::kStages) & 1;
        if (!mbar_wait(&bars->p_full, i & 1, abort_flag, p.err, site(3))) return false;
        if (!mbar_wait(&bars->v_full[s], ph, abort_flag, p.err, site(4))) return false;
        tc_fence_after();
        const uint32_t vb = sV + s * L::kNKB * kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          // A = P̃ (K-major, keys along K); B = V_j (MN-major: head dim contiguous).
          const uint64_t ad = sdesc_sw128(sP + (kk >> 2) * kTileBytes + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(vb + kk * 2048, kTileBytes, 1024);
          mma_bf16_ss(tmem + kColO, ad, bd, kIdescO, (i > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&bars->o_done);
        mma_commit(&bars->v_empty[s]);
        return true;
      };
      bool ok = mbar_wait(&bars->q_full, 0, abort_flag, p.err, site(5));
      for (int j = 0; ok && j < T; ++j) {
        const int s = j % L::kStages;
        const uint32_t ph = (j / L::kStages) & 1;
        const int sb = j & 1;
        ok = mbar_wait(&bars->k_full[s], ph, abort_flag, p.err, site(6)) &&
             mbar_wait(&bars->s_free[sb], ((j >> 1) & 1) ^ 1, abort_flag, p.err, site(7));
        if (!ok) break;
        tc_fence_after();
        const uint32_t kb = sK + s * L::kNKB * kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kTileBytes + (kk & 3) * 32;
          mma_bf16_ss(tmem + sb * kBN, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(kb + off, 16, 1024),
                      kIdescS, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars->s_full[sb]);
        mma_commit(&bars->k_empty[s]);
        if (j >= 1) ok = issue_pv(j - 1);
      }
      if (ok) issue_pv(T - 1);
      if (*abort_flag) {
        mma_commit(&bars->drain);
        mbar_wait_drain(&bars->drain, 0, 200000000ull);
      }
    }
  } else {
    // ------------------------------------------------- softmax / epilogue
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const float sl2 = p.scale_log2;
    uint8_t* sP = smem + L::kP;
    float m_run = -INFINITY;
    float l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < T; ++j) {
      const int sb = j & 1;
      ok = mbar_wait(&bars->s_full[sb], (j >> 1) & 1, abort_flag, p.err, site(8));
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t r0[32], r1[32], r2[32], r3[32];
      const uint32_t sa = tmem + lane_base + sb * kBN;
      tmem_ld32(sa + 0, r0);
      tmem_ld32(sa + 32, r1);
      tmem_ld32(sa + 64, r2);
      tmem_ld32(sa + 96, r3);
      tmem_wait_ld();
      reg_fence(r0);
      reg_fence(r1);
      reg_fence(r2);
      reg_fence(r3);
      tc_fence_before();
      mbar_arrive(&bars->s_free[sb]);

      float s[128];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        s[c] = __uint_as_float(r0[c]);
        s[32 + c] = __uint_as_float(r1[c]);
        s[64 + c] = __uint_as_float(r2[c]);
        s[96 + c] = __uint_as_float(r3[c]);
      }
      const int kv_valid = p.Nkv - j * kBN;
      if (kv_valid < kBN) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c >= kv_valid) s[c] = -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int c = 1; c < 128; ++c) mx = fmaxf(mx, s[c]);
      const float m_new = fmaxf(m_run, mx * sl2);
      const float corr = ex2_approx(m_run - m_new);
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < 128; ++c) {
        s[c] = ex2_approx(fmaf(s[c], sl2, -m_new));
        rs += s[c];
      }
      l_run = l_run * corr + rs;

      if (j >= 1) {
        ok = mbar_wait(&bars->o_done, (j - 1) & 1, abort_flag, p.err, site(9));
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      }
      // P̃ → shared memory, bf16, 128-byte-swizzled K-major rows.
#pragma unroll
      for (int c8 = 0; c8 < 16; ++c8) {
        uint4 v;
        v.x = pack_bf16x2(s[8 * c8 + 0], s[8 * c8 + 1]);
        v.y = pack_bf16x2(s[8 * c8 + 2], s[8 * c8 + 3]);
        v.z = pack_bf16x2(s[8 * c8 + 4], s[8 * c8 + 5]);
        v.w = pack_bf16x2(s[8 * c8 + 6], s[8 * c8 + 7]);
        const int kb = c8 >> 3;
        const int cc = c8 & 7;
        *reinterpret_cast<uint4*>(sP + kb * kTileBytes + row * 128 + ((cc ^ (row & 7)) << 4)) = v;
      }
      // Rescale the running output when any row of this warp saw a new max.
      if (j >= 1 && __any_sync(0xffffffffu, corr < 1.f)) {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          const uint32_t oa = tmem + lane_base + kColO + c * 32;
          tmem_ld32(oa, r);
          tmem_wait_ld();
          reg_fence(r);
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * corr);
          tmem_st32(oa, r);
        }
        tmem_wait_st();
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->p_full);
      m_run = m_new;
    }
    if (ok) {
      ok = mbar_wait(&bars->o_done, (T - 1) & 1, abort_flag, p.err, site(10));
      if (__all_sync(0xffffffffu, ok)) {
        tc_fence_after();
        const float inv = 1.f / l_run;
        const int grow = m0 + row;
        __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.o) + b * p.o_sb + h * p.o_sh +
                              static_cast<int64_t>(grow) * p.o_sn;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_base + kColO + c * 32, r);
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

template <int D>
cudaError_t launch_impl(const FwdParams& p, cudaStream_t stream) {
  using L = FwdLayout<D>;
  cudaError_t e = cudaFuncSetAttribute(fwd_bf16_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmem);
  if (e != cudaSuccess) return e;
  dim3 grid((p.Nq + kBM - 1) / kBM, p.H, p.B);
  fwd_bf16_kernel<D><<<grid, kThreads, L::kSmem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_bf16(int d, const FwdParams& p, cudaStream_t stream) {
  if (d == 128) return launch_impl<128>(p, stream);
  if (d == 64) return launch_impl<64>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
