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
//   Sᵀ = K_j Q_iᵀ, dPᵀ = V_j dO_iᵀ, dV += Pᵀ dO_i, dK += dSᵀ Q_i, dQ_iᵀ = K_jᵀ dSᵀ.
// Pᵀ is written back into TMEM over Sᵀ (bf16 pairs) and feeds dV with A read
// from TMEM; dSᵀ goes to shared memory, where it is the K-major A of dK and,
// read MN-major, the A of dQ.  Q_i and dO_i are double-buffered, and the MMA
// warp issues Sᵀ_{i+1} before dK_i and dQ_i, so the compute warps start the
// next tile's exponentials while the tensor cores finish the current one:
//   tensor order: Sᵀ_0 dPᵀ_0 dV_0 Sᵀ_1 dK_0 dQ_0 dPᵀ_1 dV_1 Sᵀ_2 dK_1 dQ_1 …
// dQ_i is added into an fp32 accumulator in global memory (kernel 3 scales it
// by σ and converts it to bf16).  It is computed transposed (both operands read
// MN-major from the K_j and dSᵀ tiles) so that TMEM lane = head-dim index; a
// 4 × 4 exchange among neighbouring lanes then gives each lane four consecutive
// head dims of one query row, and every 16-byte-per-lane reduction covers four
// full 128-byte lines.  Those reductions (as many bytes as the whole fp32 dQ
// once per key tile) are what the L2 has to absorb, and it absorbs them faster
// the more warps issue them, so two warpgroups do, each for half of the query
// columns.
//
// Causal mask (query i sees key j when j <= i): key tile j only meets query
// tiles i >= j, so the loop starts at its diagonal tile, where Pᵀ entries with
// key > query are zeroed (and with them dSᵀ).
//
// Warp roles (640 threads, five warpgroups, registers rebalanced with
// setmaxnreg): warp 0 TMA producer and warp 1 TMEM owner + MMA issuer (warps 2,
// 3 idle); warps 4..7 and 8..11 compute Pᵀ and dSᵀ (thread = key row) for query
// columns 0..63 and 64..127 and write dV and dK at the end; warps 12..15 and
// 16..19 drain dQ_iᵀ columns 0..63 and 64..127 from TMEM (thread = head-dim
// index) into the accumulator.
// TMEM columns: Sᵀ 0..127 (then Pᵀ in 0..31 and 64..95), dPᵀ (then dQ_iᵀ) 128..255,
// dV 256..383, dK 384..511.
#include <algorithm>

#include "fa_kernels.h"
#include "sm103.cuh"

namespace fa {
namespace {

constexpr int kD = 128;  // layout width: shared-memory tiles and TMEM columns are sized for d = 128
constexpr int kTile = 128;
constexpr int kTileBytes = 128 * 128;   // [128 rows][64 bf16], 128-byte swizzle
constexpr int kOpBytes = 2 * kTileBytes;  // one 128 × 128 bf16 operand
constexpr int kThreads = 640;  // five warpgroups: control, two compute, two dQ drains
// Register split (setmaxnreg): the kernel launches with kRegsLaunch per thread
// (all ptxas allows for 640 threads, five warps per sub-partition); the control
// and drain warpgroups give registers to the compute warpgroups.  Each
// sub-partition holds one warp of every warpgroup, so the split must fit
// 640 × kRegsLaunch; the launcher refuses to run if ptxas assigned fewer
// registers than that.
constexpr int kRegsLaunch = 96;
constexpr int kRegsControl = 56;
constexpr int kRegsCompute = 120;
constexpr int kRegsDrain = 88;
static_assert(128 * (kRegsControl + 2 * kRegsCompute + 2 * kRegsDrain) <= kThreads * kRegsLaunch, "register split");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 384;

constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kOpBytes;
constexpr int kOffQ = kOffV + kOpBytes;       // two buffers
constexpr int kOffDO = kOffQ + 2 * kOpBytes;  // two buffers
constexpr int kOffDST = kOffDO + 2 * kOpBytes;
constexpr int kOffStats = kOffDST + kOpBytes;  // lse2[128], delta[128]
constexpr int kOffBar = kOffStats + 2 * 128 * 4;
constexpr int kSmem = kOffBar + 256 + 1024;
static_assert(kSmem <= 232448, "shared memory budget");

struct BwdBars {
  uint64_t kv_full;
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full, dp_full, dq_full, dq_free;
  uint64_t p_ready, ds_ready, ds_free, acc_done, drain;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(BwdBars) <= 256, "barrier block");

__device__ __forceinline__ unsigned int site(unsigned int s) { return (kKernBwd << 8) | s; }

// True on one lane of a converged warp (elect.sync).
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(pred));
  return pred != 0;
}

// Adds 32 columns of dQᵀ (this lane's head dim, columns cbase … cbase+31) into
// the fp32 accumulator rows: per block of four columns, a 4 × 4 exchange among
// lanes 4g … 4g+3 gives lane 4g + r4 column c0 + r4 for head dims 4g … 4g+3,
// added with one 16-byte reduction (rows >= rows_valid, past N, are skipped).
// dst points at head dim 4g of row 0; rows are D floats apart.
template <int D>
__device__ __forceinline__ void reduce_cols(const uint32_t (&v)[32], float* dst, int cbase, int r4, int rows_valid) {
#pragma unroll
  for (int c0 = 0; c0 < 32; c0 += 4) {
    float a0 = __uint_as_float(v[c0]), a1 = __uint_as_float(v[c0 + 1]);
    float a2 = __uint_as_float(v[c0 + 2]), a3 = __uint_as_float(v[c0 + 3]);
    {
      const bool o = r4 & 1;  // swap the odd/even halves of each lane pair
      const float y0 = __shfl_xor_sync(0xffffffffu, o ? a0 : a1, 1);
      const float y1 = __shfl_xor_sync(0xffffffffu, o ? a2 : a3, 1);
      if (o) { a0 = y0; a2 = y1; } else { a1 = y0; a3 = y1; }
    }
    {
      const bool o = r4 & 2;  // then the 2 × 2 blocks of each lane quad
      const float y0 = __shfl_xor_sync(0xffffffffu, o ? a0 : a2, 2);
      const float y1 = __shfl_xor_sync(0xffffffffu, o ? a1 : a3, 2);
      if (o) { a0 = y0; a1 = y1; } else { a2 = y0; a3 = y1; }
    }
    float* q = dst + static_cast<int64_t>(cbase + c0 + r4) * D;
    if (cbase + c0 + r4 < rows_valid)
      asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(q), "f"(a0), "f"(a1), "f"(a2), "f"(a3)
                   : "memory");
  }
}

// ---------------------------------------------------------------- kernel 1
// D_i = Σ_t dO_it O_it and LSE·log2(e), D/8 lanes per row (8 bf16 each).
template <int D>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const BwdParams p) {
  constexpr int kLanes = D / 8;           // lanes per row
  constexpr int kRowsPerWarp = 32 / kLanes;
  const int64_t rows = static_cast<int64_t>(p.B) * p.H * p.N;
  const int sub = (threadIdx.x & 31) / kLanes;
  const int l16 = threadIdx.x % kLanes;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t r = gw * kRowsPerWarp + sub; r < rows; r += nw * kRowsPerWarp) {
    const uint4 a = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(p.o) + r * D * 2 + l16 * 16);
    const uint4 g = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(p.dout) + r * D * 2 + l16 * 16);
    const uint32_t wa[4] = {a.x, a.y, a.z, a.w};
    const uint32_t wg[4] = {g.x, g.y, g.z, g.w};
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc = fmaf(__uint_as_float(wa[i] << 16), __uint_as_float(wg[i] << 16), acc);
      acc = fmaf(__uint_as_float(wa[i] & 0xFFFF0000u), __uint_as_float(wg[i] & 0xFFFF0000u), acc);
    }
#pragma unroll
    for (int o = kLanes / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (l16 == 0) {
      p.delta[r] = acc;
      p.lse_log2[r] = p.lse[r] * 1.4426950408889634f;
    }
  }
}

// ---------------------------------------------------------------- kernel 3
template <int D>
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const BwdParams p) {
  const int64_t n4 = static_cast<int64_t>(p.B) * p.H * p.N * D / 4;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(p.dq_acc)[i];
    uint2 w;
    w.x = pack_bf16x2(a.x * p.scale, a.y * p.scale);
    w.y = pack_bf16x2(a.z * p.scale, a.w * p.scale);
    reinterpret_cast<uint2*>(p.dq)[i] = w;
  }
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ---------------------------------------------------------------- kernel 2
// CAUSAL: the mask and the head-grouped causal grid are compile-time properties
// of the instance (the launcher picks the instance from p.causal); measured on
// GB300 +3.3 % unmasked and +1 % causal over reading the flag at run time.
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1) bwd_main_kernel(const __grid_constant__ BwdParams p) {
  constexpr int kNKB = D / 64;  // 64-column blocks a Q, K, V or dO tile fills
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  BwdBars* bars = reinterpret_cast<BwdBars*>(smem + kOffBar);
  float* s_lse = reinterpret_cast<float*>(smem + kOffStats);   // [128]
  float* s_del = s_lse + 128;                                  // [128]
  volatile int* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Causal grids are (heads of a group, key tile, head group): key tile j meets
  // T − j query tiles, so within a group of heads (small enough that their Q, dO
  // and dQ stay in L2) every head's longest tiles (small j) launch first; the
  // last group may be partly empty.
  int j = static_cast<int>(blockIdx.x), h = static_cast<int>(blockIdx.y), b = static_cast<int>(blockIdx.z);
  if (CAUSAL) {
    const int fh = static_cast<int>(blockIdx.z * gridDim.x + blockIdx.x);
    if (fh >= p.B * p.H) return;
    j = static_cast<int>(blockIdx.y);
    h = fh % p.H;
    b = fh / p.H;
  }
  const int64_t bh = static_cast<int64_t>(b) * p.H + h;
  const int T = (p.N + kTile - 1) / kTile;  // the last tile may be ragged
  const int i0 = CAUSAL ? j : 0;  // first query tile this key tile meets
  const int nT = T - i0;            // query tiles visited; "it" counts them from 0

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    for (int q = 0; q < 2; ++q) {
      mbar_init(&bars->q_full[q], 1);
      mbar_init(&bars->q_empty[q], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_free, 2 * D);  // the drain threads that own head dims < D
    mbar_init(&bars->p_ready, 256);
    mbar_init(&bars->ds_ready, 256);
    mbar_init(&bars->ds_free, 1);
    mbar_init(&bars->acc_done, 1);
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if constexpr (D < kD) {
    // K's head dims D..127 are never loaded; the dQᵀ MMA reads them as rows of
    // its M = 128 operand, so they must be zeros.
    for (int o = threadIdx.x * 16; o < (kD - D) / 64 * kTileBytes; o += kThreads * 16)
      *reinterpret_cast<uint4*>(smem + kOffK + kNKB * kTileBytes + o) = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp < 4) {
    // Control warpgroup (producer, MMA issuer, two idle warps) gives registers
    // to the compute warpgroup; every role ends at the same named barrier,
    // after which the MMA warp frees TMEM.
    reg_dealloc<kRegsControl>();
    if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      tma_prefetch_desc(&p.tm_do);
      mbar_arrive_expect_tx(&bars->kv_full, 2 * kNKB * kTileBytes);
      for (int kb = 0; kb < kNKB; ++kb) {
        tma_load_4d(smem + kOffK + kb * kTileBytes, &p.tm_k, &bars->kv_full, kb * 64, j * kTile, h, b);
        tma_load_4d(smem + kOffV + kb * kTileBytes, &p.tm_v, &bars->kv_full, kb * 64, j * kTile, h, b);
      }
      int issued = 0;
      for (int it = 0; it < nT; ++it) {
        const int i = i0 + it;
        const int qb = it & 1;
        if (!mbar_wait_inl(&bars->q_empty[qb], ((it >> 1) & 1) ^ 1, abort_flag, p.err, site(1))) break;
        mbar_arrive_expect_tx(&bars->q_full[qb], 2 * kNKB * kTileBytes);
        for (int kb = 0; kb < kNKB; ++kb) {
          tma_load_4d(smem + kOffQ + qb * kOpBytes + kb * kTileBytes, &p.tm_q, &bars->q_full[qb], kb * 64,
                      i * kTile, h, b);
          tma_load_4d(smem + kOffDO + qb * kOpBytes + kb * kTileBytes, &p.tm_do, &bars->q_full[qb], kb * 64,
                      i * kTile, h, b);
        }
        ++issued;
      }
      if (*abort_flag) {
        mbar_wait_drain_inl(&bars->kv_full, 0, 200000000ull);
        for (int t = (issued > 2 ? issued - 2 : 0); t < issued; ++t)
          mbar_wait_drain_inl(&bars->q_full[t & 1], (t >> 1) & 1, 200000000ull);
      }
    }
    } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop, so shared-memory descriptors are warp-
    // uniform values, and one elected lane issues: a single issuing thread
    // loses issue slots to the compute and drain warps of its sub-partition
    // (+1.8 % measured on GB300).  Every lane takes the same wait results.
    {
      const bool leader = elect_one();
      auto agree = [](bool v) { return static_cast<bool>(__all_sync(0xffffffffu, v)); };
      constexpr uint32_t kIdescKK = idesc_bf16_f32(128, 128, false, false);  // Sᵀ, dPᵀ
      constexpr uint32_t kIdescKM = idesc_bf16_f32(128, D, false, true);     // dV (A in TMEM), dK
      // dQᵀ keeps M = 128 for every D: with D = 64 its A operand (K read MN-major)
      // covers a zeroed second 64-column block, so TMEM lanes 64..127 hold zeros.
      constexpr uint32_t kIdescMM = idesc_bf16_f32(128, kTile, true, true);  // dQᵀ
      const uint32_t sK = smem_u32(smem + kOffK), sV = smem_u32(smem + kOffV);
      const uint32_t sQ = smem_u32(smem + kOffQ), sDO = smem_u32(smem + kOffDO);
      const uint32_t sDST = smem_u32(smem + kOffDST);
      auto issue_st = [&](int it) {  // Sᵀ = K_j Q_iᵀ for the it-th visited query tile
        const uint32_t q = sQ + (it & 1) * kOpBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kTileBytes + (kk & 3) * 32;
          if (leader)
            mma_bf16_ss(tmem + kColS, sdesc_sw128(sK + off, 16, 1024), sdesc_sw128(q + off, 16, 1024), kIdescKK,
                        kk > 0 ? 1u : 0u);
        }
        if (leader) mma_commit(&bars->s_full);
      };
      bool ok = agree(mbar_wait_inl(&bars->kv_full, 0, abort_flag, p.err, site(2))) &&
                agree(mbar_wait_inl(&bars->q_full[0], 0, abort_flag, p.err, site(3)));
      if (ok) {
        tc_fence_after();
        issue_st(0);
      }
      for (int it = 0; ok && it < nT; ++it) {
        const uint32_t ph = it & 1;
        const uint32_t dob = sDO + (it & 1) * kOpBytes;
        const uint32_t qb = sQ + (it & 1) * kOpBytes;
        // dPᵀ_i = V_j dO_iᵀ into columns that held dQ_{i−1}: wait until it is drained.
        if (!(ok = agree(mbar_wait_inl(&bars->dq_free, ph ^ 1, abort_flag, p.err, site(4))))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kTileBytes + (kk & 3) * 32;
          if (leader)
            mma_bf16_ss(tmem + kColDP, sdesc_sw128(sV + off, 16, 1024), sdesc_sw128(dob + off, 16, 1024), kIdescKK,
                        kk > 0 ? 1u : 0u);
        }
        if (leader) mma_commit(&bars->dp_full);
        // dV += Pᵀ dO_i with Pᵀ (bf16 pairs) read from TMEM columns 0..63.
        if (!(ok = agree(mbar_wait_inl(&bars->p_ready, ph, abort_flag, p.err, site(5))))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          if (leader)
            mma_bf16_ts(tmem + kColDV, tmem + kColS + (kk >> 2) * 64 + (kk & 3) * 8,
                        sdesc_sw128(dob + kk * 2048, kTileBytes, 1024), kIdescKM, (it > 0 || kk > 0) ? 1u : 0u);
        // Sᵀ_{i+1} overwrites Pᵀ_i, which the dV MMAs above read first (in order).
        if (it + 1 < nT) {
          if (!(ok = agree(mbar_wait_inl(&bars->q_full[(it + 1) & 1], ((it + 1) >> 1) & 1, abort_flag, p.err,
                                         site(6)))))
            break;
          tc_fence_after();
          issue_st(it + 1);
        }
        if (!(ok = agree(mbar_wait_inl(&bars->ds_ready, ph, abort_flag, p.err, site(7))))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {  // dK += dSᵀ Q_i
          if (leader)
            mma_bf16_ss(tmem + kColDK, sdesc_sw128(sDST + (kk >> 2) * kTileBytes + (kk & 3) * 32, 16, 1024),
                        sdesc_sw128(qb + kk * 2048, kTileBytes, 1024), kIdescKM, (it > 0 || kk > 0) ? 1u : 0u);
        }
        // dK is the last reader of Q_i (dQ reads K_j and dSᵀ) and dV, long done, the
        // last of dO_i: the producer may refill the buffer while dQ runs (measured
        // on GB300: causal +3 %, unmasked +0.3 %).
        if (leader) mma_commit(&bars->q_empty[it & 1]);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {  // dQ_iᵀ = K_jᵀ dSᵀ (A = K_j and B = dSᵀ, both MN-major)
          if (leader)
            mma_bf16_ss(tmem + kColDP, sdesc_sw128(sK + kk * 2048, kTileBytes, 1024),
                        sdesc_sw128(sDST + kk * 2048, kTileBytes, 1024), kIdescMM, kk > 0 ? 1u : 0u);
        }
        if (leader) mma_commit(&bars->dq_full);
        if (leader) mma_commit(&bars->ds_free);
      }
      if (leader) mma_commit(&bars->acc_done);
      if (*abort_flag) {
        if (leader) mma_commit(&bars->drain);
        mbar_wait_drain_inl(&bars->drain, 0, 200000000ull);
      }
    }
    }
    tc_fence_before();
    named_sync(2, kThreads);
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tmem, kTmemCols);
    }
  } else if (warp < 12) {
    reg_alloc<kRegsCompute>();
    // ----------------------- Pᵀ / dSᵀ for 64 query columns, then dV or dK out
    // Two warpgroups; warpgroup cw owns query columns 64·cw … 64·cw+63 of every
    // tile (P and dS are elementwise per query column, so the halves never
    // meet); thread = key row.  Each writes its Pᵀ over its own Sᵀ columns
    // (64·cw …, 32 columns of bf16 pairs) and its dSᵀ into its own 64-column
    // block of shared memory.
    const int cw = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;               // key row within the tile
    const bool key_pad = j * kTile + r >= p.N;  // past N in a ragged last key tile
    const int ct = threadIdx.x - 128 * (1 + cw);  // 0..127 within the warpgroup
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const float sl2 = p.scale_log2;
    uint8_t* sDST = smem + kOffDST;
    float* lse_h = s_lse + cw * 64;  // this warpgroup's query columns
    float* del_h = s_del + cw * 64;
    const int bar_id = 1 + 2 * cw;   // named barriers 1 and 3 (2 ends the kernel)
    // The named barriers below are reached on every iteration by all four
    // warps; after an abort a warp keeps iterating without doing work, so no
    // warp is ever left waiting at a barrier another warp has abandoned.
    bool ok = true;
    for (int it = 0; it < nT; ++it) {
      const int i = i0 + it;
      const uint32_t ph = it & 1;
      const bool diag = CAUSAL && i == j;  // mask query columns c < r (key r > query c)
      named_sync(bar_id, 128);  // every thread is done reading the previous tile's stats
      // Query rows past N (a ragged last tile) get LSE = +∞, so their P is 0.
      if (ct < 64) {
        const int qrow = i * kTile + cw * 64 + ct;
        lse_h[ct] = qrow < p.N ? p.lse_log2[bh * p.N + qrow] : INFINITY;
        del_h[ct] = qrow < p.N ? p.delta[bh * p.N + qrow] : 0.f;
      }
      named_sync(bar_id, 128);
      if (!ok) continue;

      ok = mbar_wait(&bars->s_full, ph, abort_flag, p.err, site(8));
      if (!__all_sync(0xffffffffu, ok)) { ok = false; continue; }
      tc_fence_after();
      // Pᵀ row = e^(σ Sᵀ row − LSE) as bf16 pairs: pk[w] holds local query
      // columns 2w, 2w + 1.
      uint32_t pk[32];
      {
        uint32_t ra[32], rb[32];
        tmem_ld32(tmem + lane_base + kColS + cw * 64, ra);
        tmem_ld32(tmem + lane_base + kColS + cw * 64 + 32, rb);
        tmem_wait_ld();
        reg_fence(ra);
        reg_fence(rb);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int c = 2 * e;
          float a0 = ex2_approx(fmaf(__uint_as_float(ra[2 * e]), sl2, -lse_h[c]));
          float a1 = ex2_approx(fmaf(__uint_as_float(ra[2 * e + 1]), sl2, -lse_h[c + 1]));
          float b0 = ex2_approx(fmaf(__uint_as_float(rb[2 * e]), sl2, -lse_h[c + 32]));
          float b1 = ex2_approx(fmaf(__uint_as_float(rb[2 * e + 1]), sl2, -lse_h[c + 33]));
          if (diag) {
            const int cg = cw * 64 + c;  // query column within the tile
            a0 = cg < r ? 0.f : a0;
            a1 = cg + 1 < r ? 0.f : a1;
            b0 = cg + 32 < r ? 0.f : b0;
            b1 = cg + 33 < r ? 0.f : b1;
          }
          if (key_pad) a0 = a1 = b0 = b1 = 0.f;  // zero-filled K row: score 0, not −∞
          pk[e] = pack_bf16x2(a0, a1);
          pk[16 + e] = pack_bf16x2(b0, b1);
        }
      }
      tmem_st32(tmem + lane_base + kColS + cw * 64, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->p_ready);

      ok = mbar_wait(&bars->dp_full, ph, abort_flag, p.err, site(9)) &&
           mbar_wait(&bars->ds_free, ph ^ 1, abort_flag, p.err, site(10));
      if (!__all_sync(0xffffffffu, ok)) { ok = false; continue; }
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t rd[32];
        tmem_ld32(tmem + lane_base + kColDP + cw * 64 + cc * 32, rd);
        tmem_wait_ld();
        reg_fence(rd);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t w[4];
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            const int c = cc * 32 + q4 * 8 + 2 * e2;  // local query column
            const uint32_t pw = pk[c >> 1];
            const float d0 = bf16lo(pw) * (__uint_as_float(rd[q4 * 8 + 2 * e2]) - del_h[c]);
            const float d1 = bf16hi(pw) * (__uint_as_float(rd[q4 * 8 + 2 * e2 + 1]) - del_h[c + 1]);
            w[e2] = pack_bf16x2(d0, d1);
          }
          const int c8 = cw * 8 + cc * 4 + q4;  // 16-byte chunk (8 query columns) within the row
          *reinterpret_cast<uint4*>(sDST + (c8 >> 3) * kTileBytes + r * 128 + (((c8 & 7) ^ (r & 7)) << 4)) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->ds_ready);
    }
    // Warpgroup 0 writes dV, warpgroup 1 dK (with σ), through shared memory and
    // TMA: once every MMA is complete (acc_done) the Q buffers are free.  Each
    // thread writes its key row into 128-byte-swizzled [128 rows][64 columns]
    // blocks and one thread per warpgroup stores them (rows past N are clipped).
    // Every warp reaches the barrier once, even after an abort (the store is
    // then skipped).
    bool eok = false;
    if (ok) {
      ok = mbar_wait(&bars->acc_done, 0, abort_flag, p.err, site(11));
      eok = __all_sync(0xffffffffu, ok);
    }
    uint8_t* ob = smem + kOffQ + cw * (D / 64) * kTileBytes;
    if (eok) {
      tc_fence_after();
      const uint32_t col = cw == 0 ? kColDV : kColDK;
      const float mul = cw == 0 ? 1.f : p.scale;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t rr[32];
        tmem_ld32(tmem + lane_base + col + cc * 32, rr);
        tmem_wait_ld();
        reg_fence(rr);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint4 v;
          v.x = pack_bf16x2(__uint_as_float(rr[8 * q4 + 0]) * mul, __uint_as_float(rr[8 * q4 + 1]) * mul);
          v.y = pack_bf16x2(__uint_as_float(rr[8 * q4 + 2]) * mul, __uint_as_float(rr[8 * q4 + 3]) * mul);
          v.z = pack_bf16x2(__uint_as_float(rr[8 * q4 + 4]) * mul, __uint_as_float(rr[8 * q4 + 5]) * mul);
          v.w = pack_bf16x2(__uint_as_float(rr[8 * q4 + 6]) * mul, __uint_as_float(rr[8 * q4 + 7]) * mul);
          const int ch = cc * 4 + q4;  // 16-byte chunk of the row
          *reinterpret_cast<uint4*>(ob + (ch >> 3) * kTileBytes + r * 128 + (((ch & 7) ^ (r & 7)) << 4)) = v;
        }
      }
    }
    fence_proxy_async_smem();
    named_sync(bar_id, 128);
    if (wq == 0 && lane == 0 && !*abort_flag) {
      const CUtensorMap* map = cw == 0 ? &p.tm_dv : &p.tm_dk;
      for (int kb = 0; kb < D / 64; ++kb) tma_store_4d(map, ob + kb * kTileBytes, kb * 64, j * kTile, h, b);
      bulk_commit();
      bulk_wait_read();  // the source must stay until read; the writes complete with the grid
    }
    tc_fence_before();
    named_sync(2, kThreads);
  } else {
    reg_dealloc<kRegsDrain>();
    // ------------------------------------------------------ dQ_iᵀ drain
    // Thread = head-dim index (TMEM lane); warpgroup `half` owns query columns
    // 64·half … 64·half+63.  Each warp loads its 64 columns of dQ_iᵀ, frees them
    // for the next dPᵀ (once both warpgroups have), then adds them: a 4 × 4
    // exchange among neighbouring lanes turns "lane = head-dim index" into
    // four consecutive head dims of one query row per lane, so every reduction
    // instruction adds 16 bytes per lane: four full 128-byte lines per warp.
    // With D < 128 the warps of lane quarters at or past D have nothing to
    // drain (they hold the zero rows) and sit this out.
    const int half = (warp - 12) >> 2;
    const int wq = warp & 3;
    const int r4 = lane & 3;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    for (int it = 0; wq * 32 < D && it < nT; ++it) {
      const int i = i0 + it;
      const bool ok = mbar_wait_inl(&bars->dq_full, it & 1, abort_flag, p.err, site(12));
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      uint32_t r0[32], r1[32];
      tmem_ld32(tmem + lane_base + kColDP + half * 64, r0);
      tmem_ld32(tmem + lane_base + kColDP + half * 64 + 32, r1);
      tmem_wait_ld();
      reg_fence(r0);
      reg_fence(r1);
      tc_fence_before();
      mbar_arrive(&bars->dq_free);
      // Column c of dQ_iᵀ is query row i·128 + c; lane 4g + r4 ends up with query
      // row c0 + r4, head dims wq·32 + 4g … +3.
      float* dst = p.dq_acc + (bh * p.N + static_cast<int64_t>(i) * kTile) * D + wq * 32 + (lane & ~3);
      const int rows_valid = p.N - i * kTile;
      reduce_cols<D>(r0, dst, half * 64, r4, rows_valid);
      reduce_cols<D>(r1, dst, half * 64 + 32, r4, rows_valid);
    }
    tc_fence_before();
    named_sync(2, kThreads);
  }
}

}  // namespace

namespace {

template <int D>
cudaError_t launch_bwd_d(const BwdParams& p, cudaStream_t stream, int* launches) {
  const int64_t rows = static_cast<int64_t>(p.B) * p.H * p.N;
  cudaError_t e = cudaMemsetAsync(p.dq_acc, 0, static_cast<size_t>(rows) * D * sizeof(float), stream);
  if (e != cudaSuccess) return e;
  const int pre_blocks = static_cast<int>(std::min<int64_t>((rows + 15) / 16, 152 * 16));
  bwd_preprocess_kernel<D><<<pre_blocks, 256, 0, stream>>>(p);
  ++*launches;
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  auto kern = p.causal ? bwd_main_kernel<D, true> : bwd_main_kernel<D, false>;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem)) != cudaSuccess) return e;
  // setmaxnreg.inc waits until the block's pool can supply the registers: refuse
  // to launch unless ptxas gave the kernel the count the split assumes.
  cudaFuncAttributes attr;
  if ((e = cudaFuncGetAttributes(&attr, kern)) != cudaSuccess) return e;
  if (attr.numRegs < kRegsLaunch) return cudaErrorInvalidConfiguration;
  const unsigned n_kt = (p.N + kTile - 1) / kTile;
  dim3 grid(n_kt, p.H, p.B);
  if (p.causal) {
    // Heads per group: Q, dO (bf16) and the fp32 dQ accumulator about 32 MiB.
    const int64_t bh = static_cast<int64_t>(p.B) * p.H;
    const int64_t per_head = static_cast<int64_t>(p.N) * D * (2 + 2 + 4);
    int64_t g = std::max<int64_t>(1, (int64_t{32} << 20) / per_head);
    g = std::min(g, bh);
    g = std::max(g, (bh + 65534) / 65535);  // the group count must fit the z axis
    grid = dim3(static_cast<unsigned>(g), n_kt, static_cast<unsigned>((bh + g - 1) / g));
  }
  kern<<<grid, kThreads, kSmem, stream>>>(p);
  ++*launches;
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t n4 = rows * D / 4;
  const int cv_blocks = static_cast<int>(std::min<int64_t>((n4 + 255) / 256, 152 * 8));
  bwd_dq_convert_kernel<D><<<cv_blocks, 256, 0, stream>>>(p);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_bf16(int d, const BwdParams& p, cudaStream_t stream, int* launches) {
  *launches = 0;
  if (d == 128) return launch_bwd_d<128>(p, stream, launches);
  if (d == 64) return launch_bwd_d<64>(p, stream, launches);
  return cudaErrorInvalidValue;
}

}  // namespace fa
