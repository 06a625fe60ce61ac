// fa_bwd.cu — attention backward by recomputation on tcgen05 tensor cores.
//
// The forward kept only O and LSE.  As the FlashAttention walkthrough
// (kyonqi.github.io, "Flash Attention Backward") and the interview notes
// (omica.com.cn news 1422242, §二.5) describe, S and P are rebuilt tile by tile
// from Q, K and the saved statistics instead of being stored.  The gradient
// formulas are the textbook ones for O = softmax(σQKᵀ)V (the pages give none):
//   D_i = Σ_t dO_it O_it          (kernel 1, with LSE rescaled to base 2)
//   P   = e^(σ S − LSE)           S = Q Kᵀ recomputed
//   dV  = Pᵀ dO,  dP = dO Vᵀ,  dS = P ∘ (dP − D),  dK = σ dSᵀ Q,  dQ = σ dS K
//
// Kernel 2: one CTA per 128-key tile K_j, V_j of one (b, h); it loops over all
// 128-row query tiles i and accumulates dK_j, dV_j in TMEM.  Per tile, five MMAs
// run on the tensor cores, all transposed so the key tile is the M side:
//   Sᵀ = K_j Q_iᵀ, dPᵀ = V_j dO_iᵀ, dV += Pᵀ dO_i, dK += dSᵀ Q_i, dQ_i = dS K_j.
// dQ_i is added into an fp32 accumulator in global memory (kernel 3 scales it
// by σ and converts it to bf16).
//
// Warp roles (320 threads): warp 0 TMA producer; warp 1 TMEM owner + MMA issuer;
// warps 2..5 compute Pᵀ and dSᵀ (thread = key row) and write dK/dV at the end;
// warps 6..9 drain dQ_i from TMEM (thread = query row) into the accumulator.
// TMEM columns: Sᵀ 0..127, dPᵀ (then dQ_i) 128..255, dV 256..383, dK 384..511.
#include "fa_kernels.h"
#include "sm103.cuh"

namespace fa {
namespace {

constexpr int kD = 128;
constexpr int kTile = 128;
constexpr int kTileBytes = 128 * 128;   // [128 rows][64 bf16], 128-byte swizzle
constexpr int kOpBytes = 2 * kTileBytes;  // one 128 × 128 bf16 operand
constexpr int kThreads = 320;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 384;

constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kOpBytes;
constexpr int kOffQ = kOffV + kOpBytes;
constexpr int kOffDO = kOffQ + kOpBytes;
constexpr int kOffPT = kOffDO + kOpBytes;
constexpr int kOffDST = kOffPT + kOpBytes;
constexpr int kOffStats = kOffDST + kOpBytes;      // lse2[2][128], delta[2][128]
constexpr int kOffBar = kOffStats + 4 * 128 * 4;
constexpr int kSmem = kOffBar + 512 + 1024;

struct BwdBars {
  uint64_t kv_full, qdo_full, qdo_empty;
  uint64_t s_full, s_free, dp_full, dq_full, dq_free;
  uint64_t p_ready, ds_ready, ps_free, acc_done, drain;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ unsigned int site(unsigned int s) { return (kKernBwd << 8) | s; }

__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// ---------------------------------------------------------------- kernel 1
// D_i = Σ_t dO_it O_it and LSE·log2(e), one half-warp per row.
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const BwdParams p) {
  const int64_t rows = static_cast<int64_t>(p.B) * p.H * p.N;
  const int half = (threadIdx.x & 31) >> 4;
  const int l16 = threadIdx.x & 15;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t r = gw * 2 + half; r < rows; r += nw * 2) {
    const uint4 a = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(p.o) + r * kD * 2 + l16 * 16);
    const uint4 g = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(p.dout) + r * kD * 2 + l16 * 16);
    const uint32_t wa[4] = {a.x, a.y, a.z, a.w};
    const uint32_t wg[4] = {g.x, g.y, g.z, g.w};
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc = fmaf(__uint_as_float(wa[i] << 16), __uint_as_float(wg[i] << 16), acc);
      acc = fmaf(__uint_as_float(wa[i] & 0xFFFF0000u), __uint_as_float(wg[i] & 0xFFFF0000u), acc);
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (l16 == 0) {
      p.delta[r] = acc;
      p.lse_log2[r] = p.lse[r] * 1.4426950408889634f;
    }
  }
}

// ---------------------------------------------------------------- kernel 3
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const BwdParams p) {
  const int64_t n4 = static_cast<int64_t>(p.B) * p.H * p.N * kD / 4;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(p.dq_acc)[i];
    uint2 w;
    w.x = pack_bf16x2(a.x * p.scale, a.y * p.scale);
    w.y = pack_bf16x2(a.z * p.scale, a.w * p.scale);
    reinterpret_cast<uint2*>(p.dq)[i] = w;
  }
}

// Writes one 128-value bf16 row segment of 32 values (4 × 16 bytes) from fp32.
__device__ __forceinline__ void store_row32(__nv_bfloat16* dst, const uint32_t (&r)[32], float mul) {
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
    uint4 v;
    v.x = pack_bf16x2(__uint_as_float(r[8 * q4 + 0]) * mul, __uint_as_float(r[8 * q4 + 1]) * mul);
    v.y = pack_bf16x2(__uint_as_float(r[8 * q4 + 2]) * mul, __uint_as_float(r[8 * q4 + 3]) * mul);
    v.z = pack_bf16x2(__uint_as_float(r[8 * q4 + 4]) * mul, __uint_as_float(r[8 * q4 + 5]) * mul);
    v.w = pack_bf16x2(__uint_as_float(r[8 * q4 + 6]) * mul, __uint_as_float(r[8 * q4 + 7]) * mul);
    *reinterpret_cast<uint4*>(dst + q4 * 8) = v;
  }
}

// ---------------------------------------------------------------- kernel 2
__global__ void __launch_bounds__(kThreads, 1) bwd_main_kernel(const __grid_constant__ BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  BwdBars* bars = reinterpret_cast<BwdBars*>(smem + kOffBar);
  float* s_lse = reinterpret_cast<float*>(smem + kOffStats);   // [2][128]
  float* s_del = s_lse + 2 * 128;                              // [2][128]
  volatile int* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int j = blockIdx.x;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int64_t bh = static_cast<int64_t>(b) * p.H + h;
  const int T = p.N / kTile;

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    mbar_init(&bars->qdo_full, 1);
    mbar_init(&bars->qdo_empty, 1);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, 128);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_free, 128);
    mbar_init(&bars->p_ready, 128);
    mbar_init(&bars->ds_ready, 128);
    mbar_init(&bars->ps_free, 1);
    mbar_init(&bars->acc_done, 1);
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
      tma_prefetch_desc(&p.tm_do);
      mbar_arrive_expect_tx(&bars->kv_full, 2 * kOpBytes);
      for (int kb = 0; kb < 2; ++kb) {
        tma_load_4d(smem + kOffK + kb * kTileBytes, &p.tm_k, &bars->kv_full, kb * 64, j * kTile, h, b);
        tma_load_4d(smem + kOffV + kb * kTileBytes, &p.tm_v, &bars->kv_full, kb * 64, j * kTile, h, b);
      }
      int issued = 0;
      for (int i = 0; i < T; ++i) {
        if (!mbar_wait(&bars->qdo_empty, (i & 1) ^ 1, abort_flag, p.err, site(1))) break;
        mbar_arrive_expect_tx(&bars->qdo_full, 2 * kOpBytes);
        for (int kb = 0; kb < 2; ++kb) {
          tma_load_4d(smem + kOffQ + kb * kTileBytes, &p.tm_q, &bars->qdo_full, kb * 64, i * kTile, h, b);
          tma_load_4d(smem + kOffDO + kb * kTileBytes, &p.tm_do, &bars->qdo_full, kb * 64, i * kTile, h, b);
        }
        ++issued;
      }
      if (*abort_flag) {
        mbar_wait_drain(&bars->kv_full, 0, 200000000ull);
        if (issued > 0) mbar_wait_drain(&bars->qdo_full, (issued - 1) & 1, 200000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescKK = idesc_bf16_f32(128, 128, false, false);  // Sᵀ, dPᵀ
      constexpr uint32_t kIdescKM = idesc_bf16_f32(128, kD, false, true);    // dV, dK
      constexpr uint32_t kIdescMM = idesc_bf16_f32(128, kD, true, true);     // dQ
      const uint32_t sK = smem_u32(smem + kOffK), sV = smem_u32(smem + kOffV);
      const uint32_t sQ = smem_u32(smem + kOffQ), sDO = smem_u32(smem + kOffDO);
      const uint32_t sPT = smem_u32(smem + kOffPT), sDST = smem_u32(smem + kOffDST);
      bool ok = mbar_wait(&bars->kv_full, 0, abort_flag, p.err, site(2));
      for (int i = 0; ok && i < T; ++i) {
        const uint32_t ph = i & 1;
        ok = mbar_wait(&bars->qdo_full, ph, abort_flag, p.err, site(3)) &&
             mbar_wait(&bars->s_free, ph ^ 1, abort_flag, p.err, site(4));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {  // Sᵀ = K_j Q_iᵀ
          const uint32_t off = (kk >> 2) * kTileBytes + (kk & 3) * 32;
          mma_bf16_ss(tmem + kColS, sdesc_sw128(sK + off, 16, 1024), sdesc_sw128(sQ + off, 16, 1024), kIdescKK,
                      kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars->s_full);
        if (!(ok = mbar_wait(&bars->dq_free, ph ^ 1, abort_flag, p.err, site(5)))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {  // dPᵀ = V_j dO_iᵀ
          const uint32_t off = (kk >> 2) * kTileBytes + (kk & 3) * 32;
          mma_bf16_ss(tmem + kColDP, sdesc_sw128(sV + off, 16, 1024), sdesc_sw128(sDO + off, 16, 1024), kIdescKK,
                      kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars->dp_full);
        if (!(ok = mbar_wait(&bars->p_ready, ph, abort_flag, p.err, site(6)))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {  // dV += Pᵀ dO_i
          mma_bf16_ss(tmem + kColDV, sdesc_sw128(sPT + (kk >> 2) * kTileBytes + (kk & 3) * 32, 16, 1024),
                      sdesc_sw128(sDO + kk * 2048, kTileBytes, 1024), kIdescKM, (i > 0 || kk > 0) ? 1u : 0u);
        }
        if (!(ok = mbar_wait(&bars->ds_ready, ph, abort_flag, p.err, site(7)))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {  // dK += dSᵀ Q_i
          mma_bf16_ss(tmem + kColDK, sdesc_sw128(sDST + (kk >> 2) * kTileBytes + (kk & 3) * 32, 16, 1024),
                      sdesc_sw128(sQ + kk * 2048, kTileBytes, 1024), kIdescKM, (i > 0 || kk > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {  // dQ_i = dS K_j (dS read MN-major from dSᵀ)
          mma_bf16_ss(tmem + kColDP, sdesc_sw128(sDST + kk * 2048, kTileBytes, 1024),
                      sdesc_sw128(sK + kk * 2048, kTileBytes, 1024), kIdescMM, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars->dq_full);
        mma_commit(&bars->qdo_empty);
        mma_commit(&bars->ps_free);
      }
      mma_commit(&bars->acc_done);
      if (*abort_flag) {
        mma_commit(&bars->drain);
        mbar_wait_drain(&bars->drain, 0, 200000000ull);
      }
    }
  } else if (warp < 6) {
    // -------------------------------------------- Pᵀ / dSᵀ, then dK / dV out
    const int wq = warp & 3;
    const int r = wq * 32 + lane;             // key row within the tile
    const int tr = threadIdx.x - 64;          // 0..127, for staging row stats
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const float sl2 = p.scale_log2;
    uint8_t* sPT = smem + kOffPT;
    uint8_t* sDST = smem + kOffDST;
    bool ok = true;
    for (int i = 0; i < T; ++i) {
      const uint32_t ph = i & 1;
      float* lse_t = s_lse + ph * 128;
      float* del_t = s_del + ph * 128;
      lse_t[tr] = p.lse_log2[bh * p.N + i * kTile + tr];
      del_t[tr] = p.delta[bh * p.N + i * kTile + tr];
      named_sync(1, 128);

      ok = mbar_wait(&bars->s_full, ph, abort_flag, p.err, site(8));
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t r0[32], r1[32], r2[32], r3[32];
      tmem_ld32(tmem + lane_base + kColS + 0, r0);
      tmem_ld32(tmem + lane_base + kColS + 32, r1);
      tmem_ld32(tmem + lane_base + kColS + 64, r2);
      tmem_ld32(tmem + lane_base + kColS + 96, r3);
      tmem_wait_ld();
      reg_fence(r0);
      reg_fence(r1);
      reg_fence(r2);
      reg_fence(r3);
      tc_fence_before();
      mbar_arrive(&bars->s_free);
      float pv[128];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        pv[c] = ex2_approx(fmaf(__uint_as_float(r0[c]), sl2, -lse_t[c]));
        pv[32 + c] = ex2_approx(fmaf(__uint_as_float(r1[c]), sl2, -lse_t[32 + c]));
        pv[64 + c] = ex2_approx(fmaf(__uint_as_float(r2[c]), sl2, -lse_t[64 + c]));
        pv[96 + c] = ex2_approx(fmaf(__uint_as_float(r3[c]), sl2, -lse_t[96 + c]));
      }
      ok = mbar_wait(&bars->ps_free, ph ^ 1, abort_flag, p.err, site(9));
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
#pragma unroll
      for (int c8 = 0; c8 < 16; ++c8) {
        uint4 v;
        v.x = pack_bf16x2(pv[8 * c8 + 0], pv[8 * c8 + 1]);
        v.y = pack_bf16x2(pv[8 * c8 + 2], pv[8 * c8 + 3]);
        v.z = pack_bf16x2(pv[8 * c8 + 4], pv[8 * c8 + 5]);
        v.w = pack_bf16x2(pv[8 * c8 + 6], pv[8 * c8 + 7]);
        *reinterpret_cast<uint4*>(sPT + (c8 >> 3) * kTileBytes + r * 128 + (((c8 & 7) ^ (r & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars->p_ready);

      ok = mbar_wait(&bars->dp_full, ph, abort_flag, p.err, site(10));
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t rd[32];
        tmem_ld32(tmem + lane_base + kColDP + cc * 32, rd);
        tmem_wait_ld();
        reg_fence(rd);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          float ds[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int c = cc * 32 + q4 * 8 + e;
            ds[e] = pv[c] * (__uint_as_float(rd[q4 * 8 + e]) - del_t[c]);
          }
          uint4 v;
          v.x = pack_bf16x2(ds[0], ds[1]);
          v.y = pack_bf16x2(ds[2], ds[3]);
          v.z = pack_bf16x2(ds[4], ds[5]);
          v.w = pack_bf16x2(ds[6], ds[7]);
          const int c8 = cc * 4 + q4;
          *reinterpret_cast<uint4*>(sDST + (c8 >> 3) * kTileBytes + r * 128 + (((c8 & 7) ^ (r & 7)) << 4)) = v;
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->ds_ready);
    }
    if (ok) {
      ok = mbar_wait(&bars->acc_done, 0, abort_flag, p.err, site(11));
      if (__all_sync(0xffffffffu, ok)) {
        tc_fence_after();
        const int64_t grow = bh * p.N + static_cast<int64_t>(j) * kTile + r;
        __nv_bfloat16* dv_row = reinterpret_cast<__nv_bfloat16*>(p.dv) + grow * kD;
        __nv_bfloat16* dk_row = reinterpret_cast<__nv_bfloat16*>(p.dk) + grow * kD;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t rr[32];
          tmem_ld32(tmem + lane_base + kColDV + cc * 32, rr);
          tmem_wait_ld();
          reg_fence(rr);
          store_row32(dv_row + cc * 32, rr, 1.f);
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t rr[32];
          tmem_ld32(tmem + lane_base + kColDK + cc * 32, rr);
          tmem_wait_ld();
          reg_fence(rr);
          store_row32(dk_row + cc * 32, rr, p.scale);
        }
      }
    }
  } else {
    // ------------------------------------------------------ dQ_i drain
    const int wq = warp & 3;
    const int r = wq * 32 + lane;  // query row within the tile
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    for (int i = 0; i < T; ++i) {
      const bool ok = mbar_wait(&bars->dq_full, i & 1, abort_flag, p.err, site(12));
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      uint32_t r0[32], r1[32], r2[32], r3[32];
      tmem_ld32(tmem + lane_base + kColDP + 0, r0);
      tmem_ld32(tmem + lane_base + kColDP + 32, r1);
      tmem_ld32(tmem + lane_base + kColDP + 64, r2);
      tmem_ld32(tmem + lane_base + kColDP + 96, r3);
      tmem_wait_ld();
      reg_fence(r0);
      reg_fence(r1);
      reg_fence(r2);
      reg_fence(r3);
      tc_fence_before();
      mbar_arrive(&bars->dq_free);
      float4* dst = reinterpret_cast<float4*>(p.dq_acc + (bh * p.N + static_cast<int64_t>(i) * kTile + r) * kD);
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        atomicAdd(dst + c4, make_float4(__uint_as_float(r0[4 * c4]), __uint_as_float(r0[4 * c4 + 1]),
                                        __uint_as_float(r0[4 * c4 + 2]), __uint_as_float(r0[4 * c4 + 3])));
        atomicAdd(dst + 8 + c4, make_float4(__uint_as_float(r1[4 * c4]), __uint_as_float(r1[4 * c4 + 1]),
                                            __uint_as_float(r1[4 * c4 + 2]), __uint_as_float(r1[4 * c4 + 3])));
        atomicAdd(dst + 16 + c4, make_float4(__uint_as_float(r2[4 * c4]), __uint_as_float(r2[4 * c4 + 1]),
                                             __uint_as_float(r2[4 * c4 + 2]), __uint_as_float(r2[4 * c4 + 3])));
        atomicAdd(dst + 24 + c4, make_float4(__uint_as_float(r3[4 * c4]), __uint_as_float(r3[4 * c4 + 1]),
                                             __uint_as_float(r3[4 * c4 + 2]), __uint_as_float(r3[4 * c4 + 3])));
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

cudaError_t launch_bwd_bf16(int d, const BwdParams& p, cudaStream_t stream, int* launches) {
  *launches = 0;
  if (d != kD) return cudaErrorInvalidValue;
  const int64_t rows = static_cast<int64_t>(p.B) * p.H * p.N;
  cudaError_t e = cudaMemsetAsync(p.dq_acc, 0, static_cast<size_t>(rows) * kD * sizeof(float), stream);
  if (e != cudaSuccess) return e;
  const int pre_blocks = static_cast<int>(std::min<int64_t>((rows + 15) / 16, 152 * 16));
  bwd_preprocess_kernel<<<pre_blocks, 256, 0, stream>>>(p);
  ++*launches;
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(bwd_main_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem)) != cudaSuccess)
    return e;
  bwd_main_kernel<<<dim3(p.N / kTile, p.H, p.B), kThreads, kSmem, stream>>>(p);
  ++*launches;
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t n4 = rows * kD / 4;
  const int cv_blocks = static_cast<int>(std::min<int64_t>((n4 + 255) / 256, 152 * 8));
  bwd_dq_convert_kernel<<<cv_blocks, 256, 0, stream>>>(p);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace fa
