// fa_decode_tc.cu — grouped-query split-KV decode on tcgen05 tensor cores.
//
// With G query heads per key/value head, each key costs 2·G·d multiply-adds
// per byte pair of K and V read, which at G ≥ 2 outgrows what CUDA cores hide
// under the HBM stream.  Here the G query rows of one (b, key/value head) form
// the first rows of a 128-row A tile (the rest are neighbouring rows that never
// leave the CTA), and each key tile goes through the tensor cores:
//   S = Q_g K_jᵀ (tcgen05.mma → TMEM), online softmax of §3.2 of
//   "FlashAttention：IO-aware 的注意力 kernel" on rows 0..G−1, O += P̃ V_j.
// The CTA covers one chunk of the key range (FlashDecoding's split, §3.3 and
// §9 of the same lesson) and writes unnormalised (m, ℓ, o) triples that the
// split-KV merge kernel folds with the block-merge rule (omica.com.cn news
// 1422242, §二.3).
//
// Warp roles (224 threads): warps 0..3 softmax and epilogue for TMEM lanes
// 32·w … 32·w+31 (rows of the A tile; rows ≥ G are padding, and only the
// ⌈G/32⌉ warps that hold query rows take part); warp 5 TMA producer (Q once,
// then K_0, K_1, V_0, K_2, V_1, … into a 5-slot ring); warp 6 TMEM owner and
// MMA issuer; warp 4 idle.  Warp w runs on SM sub-partition w % 4, so with
// G ≤ 32 softmax, producer and MMA issuer each have a sub-partition of their own.  TMEM: S buffers at columns 0 and 128, O at 256.
// P̃ is written as bf16 pairs over its S buffer and read from TMEM by the P̃V
// MMA; S(j) is issued after P̃V(j−2), so the in-order tensor pipe has read
// P̃(j−2) before S(j) overwrites it.  Keeping P̃ out of shared memory leaves
// room for five ring slots, which is what keeps enough copies in flight.
// Rows keep their reference max until a tile's max exceeds it by 2^8 (base 2),
// exactly as in the forward kernel; the merge accepts any reference m.
//
// Paged cache (PAGED): k and v are [num_blocks, H_kv, bs, d] with bs dividing
// 128; logical key t of sequence b is row t % bs of page block_table[b][t / bs].
// Each 128-key tile is loaded as 128/bs page boxes; pages past the sequence are
// requested at an out-of-range row so TMA fills them with zeros, and on a
// split's last, partial tile the softmax warp zeroes the V rows past the end
// (slots of a partly filled page hold stale data) before P̃V runs.
// The boxes of one tile are issued by different lanes of the producer warp at
// once; small pages need that to keep enough copies in flight.  At d = 128 a
// page of one head is a single box of a 5-D view (64 columns, 8 rows, 2 column
// halves, bs/8 row groups, page·H_kv + head) that lands as [row group][half]
// [8 rows][128 bytes]: the tile's 8-row groups are 2 KB apart and its column
// halves 1 KB apart for any page size, and one box per page (4 KB at 16 keys)
// replaces two half-width boxes.  The MMA descriptors follow that layout.
#include "fa_kernels.h"
#include "sm103.cuh"

namespace fa {
namespace {

constexpr int kBN = 128;
constexpr int kTileBytes = 128 * 128;    // [128 rows][64 bf16], 128-byte swizzle
constexpr int kThreads = 224;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;
constexpr float kRescaleLog2 = 8.0f;
constexpr int kMaxStagedPages = 1024;
constexpr int kMaxRing = 10;

// Shared-memory layout for head dim D: a Q, K or V tile is D/64 swizzled
// [128 rows][64 columns] blocks; the ring holds about 160 KB of K/V tiles
// (5 slots at d = 128, 10 at d = 64), which keeps enough copies in flight.
template <int D>
struct TcCfg {
  static constexpr int kNKB = D / 64;
  // Paged d = 128 tiles use the grouped layout above: byte offsets of the next
  // 8-row group and of the second column half.
  static constexpr int kPgGroup = 2048;
  static constexpr int kPgHalf = 1024;
  static constexpr int kSlot = kNKB * kTileBytes;
  static constexpr int kRing = D == 64 ? 10 : 5;
  static constexpr int kOffQ = 0;
  static constexpr int kOffR = kOffQ + kSlot;
  static constexpr int kOffPages = kOffR + kRing * kSlot;  // paged cache: staged page ids
  static constexpr int kOffBar = kOffPages + kMaxStagedPages * 4;
  static constexpr int kSmem = kOffBar + 256 + 1024;
  static_assert(kRing <= kMaxRing, "ring barriers");
};

struct Bars {
  uint64_t q_full;
  uint64_t r_full[kMaxRing], r_empty[kMaxRing];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full, p_free;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

__device__ __forceinline__ unsigned int site(unsigned int s) { return (kKernDecode << 8) | (0x80u | s); }
__device__ __forceinline__ int seq_k(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int seq_v(int j, int T) { return min(2 * j + 2, 2 * T - 1); }

template <int D, bool PAGED>
__global__ void __launch_bounds__(kThreads, 1) decode_gqa_tc_kernel(const __grid_constant__ DecodeTcParams p) {
  using C = TcCfg<D>;
  constexpr int kSlot = C::kSlot, kRing = C::kRing, kOffQ = C::kOffQ, kOffR = C::kOffR;
  constexpr bool kPg5 = PAGED && D == 128;  // K/V tiles in the grouped page layout
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kOffBar);
  volatile int* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  const int hkv = blockIdx.y;
  const int b = blockIdx.z;
  const int qrow0 = b * p.Hq + hkv * p.G;  // first query row in the [B·H_q, d] view
  int len = p.Nkv;
  int chunk = p.chunk;
  if (PAGED) {
    len = p.seq_lens[b];
    if (len < 1 || len > p.max_blocks * p.block_size) {
      if (threadIdx.x == 0) atomicCAS(p.err, 0u, (kKernDecode << 8) | kSiteBadLength);
      len = min(max(len, 1), p.max_blocks * p.block_size);
    }
    chunk = (((len + p.n_splits - 1) / p.n_splits) + 127) & ~127;
  }
  const int key0 = c * chunk;
  const int kend = min(len, key0 + chunk);
  const int nkeys = max(0, kend - key0);
  const int T = (nkeys + kBN - 1) / kBN;
  const int nsw = (p.G + 31) >> 5;  // softmax warps holding query rows (1..4)

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&bars->r_full[s], 1);
      mbar_init(&bars->r_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->s_free[s], 32 * nsw);
    }
    mbar_init(&bars->p_full, 32 * nsw);
    mbar_init(&bars->p_free, 1);
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 6) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 5) {
    // ------------------------------------------------------------ producer
    int* staged = reinterpret_cast<int*>(smem + C::kOffPages);
    const int page0 = PAGED ? key0 / p.block_size : 0;
    if (PAGED && T > 0) {
      // The warp stages this range's page ids with one coalesced, checked load.
      const int npages = min(kMaxStagedPages, (kend - 1) / p.block_size - page0 + 1);
      for (int i = lane; i < npages; i += 32) {
        int blk = p.block_table[static_cast<int64_t>(b) * p.max_blocks + page0 + i];
        if (blk < 0 || blk >= p.num_blocks) {
          atomicCAS(p.err, 0u, (kKernDecode << 8) | kSiteBadBlock);
          blk = 0;
        }
        staged[i] = blk;
      }
      __syncwarp();
    }
    // Page holding key t0 (a multiple of the page size), checked.
    auto page_id = [&](int t0) -> int {
      const int rel = t0 / p.block_size - page0;
      if (rel < kMaxStagedPages) return staged[rel];
      int blk = p.block_table[static_cast<int64_t>(b) * p.max_blocks + t0 / p.block_size];
      if (blk < 0 || blk >= p.num_blocks) {
        atomicCAS(p.err, 0u, (kKernDecode << 8) | kSiteBadBlock);
        blk = 0;
      }
      return blk;
    };
    if (T > 0) {
      // TMA boxes, issued warp-wide: lane 0 waits for the slot and arms its
      // byte count, then lane kb (contiguous cache) or lane pg (one page,
      // both 64-column halves) issues its boxes.
      if (lane == 0) {
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_v);
        mbar_arrive_expect_tx(&bars->q_full, kSlot);
        for (int kb = 0; kb < C::kNKB; ++kb)
          tma_load_4d(smem + kOffQ + kb * kTileBytes, &p.tm_q, &bars->q_full, kb * 64, qrow0, 0, 0);
      }
      int issued = 0;
      for (int t = 0; t < 2 * T; ++t) {
        const int slot = t % kRing;
        const bool is_v = t != 0 && (t == 2 * T - 1 || !(t & 1));
        const int jt = t == 0 ? 0 : (t == 2 * T - 1 ? T - 1 : ((t & 1) ? (t + 1) >> 1 : (t - 2) >> 1));
        bool ok = true;
        if (lane == 0) {
          ok = mbar_wait(&bars->r_empty[slot], ((t / kRing) & 1) ^ 1, abort_flag, p.err, site(1));
          if (ok) mbar_arrive_expect_tx(&bars->r_full[slot], kSlot);
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        __syncwarp();
        const CUtensorMap* tm = is_v ? &p.tm_v : &p.tm_k;
        if (!PAGED) {
          if (lane < C::kNKB)
            tma_load_4d(smem + kOffR + slot * kSlot + lane * kTileBytes, tm, &bars->r_full[slot], lane * 64,
                        key0 + jt * kBN, hkv, b);
        } else {
          const int bs = p.block_size;
          if (lane < kBN / bs) {
            const int t0 = key0 + jt * kBN + lane * bs;  // a multiple of bs
            int blk = 0, row = 0;
            if (t0 < kend)
              blk = page_id(t0);
            else
              row = bs;  // wholly out of range: zero fill
            if constexpr (D == 128) {
              tma_load_5d(smem + kOffR + slot * kSlot + lane * bs * 256, tm, &bars->r_full[slot], 0, 0, 0,
                          row >> 3, blk * p.Hkv + hkv);
            } else {
              for (int kb = 0; kb < C::kNKB; ++kb)
                tma_load_4d(smem + kOffR + slot * kSlot + kb * kTileBytes + lane * bs * 128, tm,
                            &bars->r_full[slot], kb * 64, row, hkv, blk);
            }
          }
        }
        ++issued;
      }
      if (lane == 0 && *abort_flag) {
        mbar_wait_drain(&bars->q_full, 0, 200000000ull);
        for (int t = (issued > kRing ? issued - kRing : 0); t < issued; ++t)
          mbar_wait_drain(&bars->r_full[t % kRing], (t / kRing) & 1, 200000000ull);
      }
    }
  } else if (warp == 6) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && T > 0) {
      constexpr uint32_t kIdescS = idesc_bf16_f32(128, kBN, false, false);
      constexpr uint32_t kIdescO = idesc_bf16_f32(128, D, false, true);
      const uint32_t sQ = smem_u32(smem + kOffQ);
      const uint32_t sR = smem_u32(smem + kOffR);
      auto issue_pv = [&](int jj) -> bool {
        const int t = seq_v(jj, T);
        const int slot = t % kRing;
        if (!mbar_wait(&bars->p_full, jj & 1, abort_flag, p.err, site(2))) return false;
        if (!mbar_wait(&bars->r_full[slot], (t / kRing) & 1, abort_flag, p.err, site(3))) return false;
        tc_fence_after();
        const uint32_t vb = sR + slot * kSlot;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {  // A = P̃(jj) from its S buffer's TMEM columns
          // 16 keys per k-step: two 8-key groups; the head dim's 64-column halves are the MN blocks.
          const uint64_t bd = kPg5 ? sdesc_sw128(vb + kk * 2 * C::kPgGroup, C::kPgHalf, C::kPgGroup)
                                   : sdesc_sw128(vb + kk * 2048, kTileBytes, 1024);
          mma_bf16_ts(tmem + kColO, tmem + (jj & 1) * kBN + kk * 8, bd, kIdescO, (jj > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&bars->p_free);
        mma_commit(&bars->r_empty[slot]);
        return true;
      };
      bool ok = mbar_wait(&bars->q_full, 0, abort_flag, p.err, site(4));
      for (int j = 0; ok && j < T; ++j) {
        const int t = seq_k(j);
        const int slot = t % kRing;
        const int sb = j & 1;
        ok = mbar_wait(&bars->r_full[slot], (t / kRing) & 1, abort_flag, p.err, site(5)) &&
             mbar_wait(&bars->s_free[sb], ((j >> 1) & 1) ^ 1, abort_flag, p.err, site(6));
        if (!ok) break;
        tc_fence_after();
        const uint32_t kb = sR + slot * kSlot;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kTileBytes + (kk & 3) * 32;
          const uint64_t bd = kPg5 ? sdesc_sw128(kb + (kk >> 2) * C::kPgHalf + (kk & 3) * 32, 16, C::kPgGroup)
                                   : sdesc_sw128(kb + off, 16, 1024);
          mma_bf16_ss(tmem + sb * kBN, sdesc_sw128(sQ + off, 16, 1024), bd, kIdescS, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars->s_full[sb]);
        mma_commit(&bars->r_empty[slot]);
        if (j >= 1) ok = issue_pv(j - 1);
      }
      if (ok) issue_pv(T - 1);
      if (*abort_flag) {
        mma_commit(&bars->drain);
        mbar_wait_drain(&bars->drain, 0, 200000000ull);
      }
    }
  } else if (warp < nsw) {
    // ------------------------------- softmax for rows 32·warp … +31, epilogue
    const int row = warp * 32 + lane;  // TMEM lane; rows < G are the group's query heads
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const float sl2 = p.scale_log2;
    float m_run = -INFINITY;
    float l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < T; ++j) {
      const int sb = j & 1;
      ok = mbar_wait(&bars->s_full[sb], (j >> 1) & 1, abort_flag, p.err, site(7));
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
      for (int e = 0; e < 32; ++e) {
        s[e] = __uint_as_float(r0[e]);
        s[32 + e] = __uint_as_float(r1[e]);
        s[64 + e] = __uint_as_float(r2[e]);
        s[96 + e] = __uint_as_float(r3[e]);
      }
      const int valid = kend - (key0 + j * kBN);  // keys past the chunk belong to the next split
      if (valid < kBN) {
#pragma unroll
        for (int e = 0; e < 128; ++e)
          if (e >= valid) s[e] = -INFINITY;
      }
      float mx8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx8[i] = s[i];
#pragma unroll
      for (int e = 8; e < 128; e += 8)
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(mx8[i], s[e + i]);
      const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      const float m_cand = fmaxf(m_run, mx * sl2);
      const bool need = m_cand > m_run + kRescaleLog2;
      const float m_new = need ? m_cand : m_run;
      const float corr = need ? ex2_approx(m_run - m_new) : 1.f;
      float rs8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) rs8[i] = 0.f;
#pragma unroll
      for (int e = 0; e < 128; e += 8)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          s[e + i] = ex2_approx(fmaf(s[e + i], sl2, -m_new));
          rs8[i] += s[e + i];
        }
      l_run = l_run * corr + (((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7])));

      {
        uint32_t w0[32], w1[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          w0[e] = pack_bf16x2(s[2 * e], s[2 * e + 1]);
          w1[e] = pack_bf16x2(s[64 + 2 * e], s[64 + 2 * e + 1]);
        }
        tmem_st32(tmem + lane_base + sb * kBN, w0);
        tmem_st32(tmem + lane_base + sb * kBN + 32, w1);
      }
      // Wait for P̃V(j−1) on every tile, not only before a rescale of O: the
      // final wait below tells phases apart by parity, which is only sound if
      // p_free is never more than one phase ahead of the last one waited for.
      ok = mbar_wait(&bars->p_free, (j & 1) ^ 1, abort_flag, p.err, site(8));
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      if (j >= 1 && __any_sync(0xffffffffu, need)) {
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t r[32];
          const uint32_t oa = tmem + lane_base + kColO + cc * 32;
          tmem_ld32(oa, r);
          tmem_wait_ld();
          reg_fence(r);
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * corr);
          tmem_st32(oa, r);
        }
      }
      tmem_wait_st();
      if (PAGED && valid < kBN && warp == 0) {
        // Zero the V rows past the sequence end once V_j has landed (warp 0
        // does it before its p_full arrival, which P̃V waits for).
        const int t = seq_v(j, T);
        ok = mbar_wait(&bars->r_full[t % kRing], (t / kRing) & 1, abort_flag, p.err, site(10));
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        uint8_t* vt = smem + kOffR + (t % kRing) * kSlot;
        for (int rr = max(valid, 0) + lane; rr < kBN; rr += 32)
#pragma unroll
          for (int kb = 0; kb < C::kNKB; ++kb) {
            // Byte offset of key row rr's 128 bytes in column half kb.
            const int ro = kPg5 ? (rr >> 3) * C::kPgGroup + kb * C::kPgHalf + (rr & 7) * 128 : kb * kTileBytes + rr * 128;
#pragma unroll
            for (int q = 0; q < 8; ++q) *reinterpret_cast<uint4*>(vt + ro + q * 16) = make_uint4(0, 0, 0, 0);
          }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->p_full);
      m_run = m_new;
    }
    // Unnormalised triple for each query head of the group.
    if (T == 0) {
      if (row < p.G) {
        const int64_t slot = static_cast<int64_t>(qrow0 + row) * p.n_splits + c;
        for (int e = 0; e < D; ++e) p.part_o[slot * D + e] = 0.f;
        p.part_ml[slot * 2 + 0] = -INFINITY;
        p.part_ml[slot * 2 + 1] = 0.f;
      }
    } else if (ok) {
      ok = mbar_wait(&bars->p_free, (T - 1) & 1, abort_flag, p.err, site(9));
      if (__all_sync(0xffffffffu, ok)) {
        tc_fence_after();
        const int64_t slot = static_cast<int64_t>(qrow0 + row) * p.n_splits + c;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_base + kColO + cc * 32, r);
          tmem_wait_ld();
          reg_fence(r);
          if (row < p.G) {
            float4* dst = reinterpret_cast<float4*>(p.part_o + slot * D + cc * 32);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              dst[q4] = make_float4(__uint_as_float(r[4 * q4]), __uint_as_float(r[4 * q4 + 1]),
                                    __uint_as_float(r[4 * q4 + 2]), __uint_as_float(r[4 * q4 + 3]));
          }
        }
        if (row < p.G) {
          p.part_ml[slot * 2 + 0] = m_run;
          p.part_ml[slot * 2 + 1] = l_run;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 6) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool PAGED>
cudaError_t launch_gqa_d(const DecodeTcParams& p, cudaStream_t stream) {
  constexpr int kSmem = TcCfg<D>::kSmem;
  cudaError_t e =
      cudaFuncSetAttribute(decode_gqa_tc_kernel<D, PAGED>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  decode_gqa_tc_kernel<D, PAGED><<<dim3(p.n_splits, p.Hkv, p.B), kThreads, kSmem, stream>>>(p);
  return cudaGetLastError();
}

template <bool PAGED>
cudaError_t launch_gqa(const DecodeTcParams& p, cudaStream_t stream) {
  if (p.d == 128) return launch_gqa_d<128, PAGED>(p, stream);
  if (p.d == 64) return launch_gqa_d<64, PAGED>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_decode_gqa_tc(const DecodeTcParams& p, cudaStream_t stream) {
  return launch_gqa<false>(p, stream);
}

cudaError_t launch_decode_gqa_tc_paged(const DecodeTcParams& p, cudaStream_t stream) {
  if (p.block_size < 16 || p.block_size > kBN || (kBN % p.block_size) != 0) return cudaErrorInvalidValue;
  return launch_gqa<true>(p, stream);
}

}  // namespace fa
