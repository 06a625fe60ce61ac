// fa_decode.cu — split-KV decode (one query row per head), bf16 in, fp32 math.
//
// Decode reads the whole key/value cache once per step and is bound by device
// memory bandwidth, not by arithmetic ("FlashAttention：IO-aware 的注意力 kernel"
// §3.3 and §9: the single query's scores are a 1×N vector; FlashDecoding
// splits the key range across SMs to keep them all busy).
//
// Kernel 1 (grid = splits × H × B, 128 threads): CTA c streams keys
// [c·chunk, (c+1)·chunk) of one (b, h) in sub-chunks of 64 keys.  K and V rows
// of a sub-chunk are contiguous in memory, so each arrives with one untiled bulk
// copy per tensor into a 2-stage shared-memory ring.  The CTA runs the online
// softmax over its keys and writes the unnormalised triple (m_c, ℓ_c, o_c).
// Kernel 2 (grid = B·H, d threads) folds the triples with the block-merge rule
// of the FlashAttention interview notes (omica.com.cn news 1422242, §二.3)
// and writes O = o/ℓ and LSE = m + ln ℓ.
#include <mutex>

#include "fa_kernels.h"
#include "sm103.cuh"

namespace fa {
namespace {

constexpr int kSub = 64;                      // keys per sub-chunk
constexpr int kThreads = 128;

// Sizes for head dim D (64 or 128).  A key's D values are spread over D/8
// lanes (8 values each), so a warp covers 256/D keys at once, and the P·V sums
// of the 4·256/D (warp, key slot) groups are combined at the end.
template <int D>
struct DecCfg {
  static constexpr int kRowBytes = D * 2;                   // one bf16 key row
  static constexpr int kStageBytes = 2 * kSub * kRowBytes;  // K then V
  static constexpr int kSmem = 2 * kStageBytes + 1024;
  static constexpr int kLanesPerKey = D / 8;
  static constexpr int kKeysPerStep = 32 / kLanesPerKey;
  static constexpr int kGroups = 4 * kKeysPerStep;
  static_assert(kGroups * D == 1024, "partial sums fill the reduction buffer");
};

constexpr int kMaxStagedPages = 256;  // page ids of a CTA's key range held in shared memory

struct DecodeSmem {
  float scores[kSub];
  float probs[kSub];
  float red[1024];  // [kGroups][D] partial P·V sums
  uint64_t full[2];
  int abort_flag;
  int pages[kMaxStagedPages];  // paged cache only: validated page ids of this CTA's range
};

__device__ __forceinline__ unsigned int site(unsigned int s) { return (kKernDecode << 8) | s; }

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Page id of logical page `page` of sequence b, checked against the pool; an
// out-of-range id is reported and replaced by page 0 so no address leaves it.
__device__ __forceinline__ int checked_page(const DecodeParams& p, int b, int page) {
  int blk = p.block_table[static_cast<int64_t>(b) * p.max_blocks + page];
  if (blk < 0 || blk >= p.num_blocks) {
    atomicCAS(p.err, 0u, (kKernDecode << 8) | kSiteBadBlock);
    blk = 0;
  }
  return blk;
}

// Device address of logical key `t` of head h in a paged cache [num_blocks, H,
// bs, d], and how many rows of that page follow it.  `staged` holds the ids of
// pages page0 … page0 + kMaxStagedPages − 1; later pages are read directly.
__device__ __forceinline__ const uint8_t* paged_row(const void* cache, const DecodeParams& p, const int* staged,
                                                    int page0, int b, int h, int t, int row_bytes, int* piece_rows) {
  const int page = t / p.block_size;
  const int slot = t - page * p.block_size;
  const int rel = page - page0;
  const int blk = rel < kMaxStagedPages ? staged[rel] : checked_page(p, b, page);
  *piece_rows = p.block_size - slot;
  return reinterpret_cast<const uint8_t*>(cache) +
         ((static_cast<int64_t>(blk) * p.H + h) * p.block_size + slot) * row_bytes;
}

template <int D, bool PAGED>
__global__ void __launch_bounds__(kThreads) decode_split_kernel(const DecodeParams p) {
  using C = DecCfg<D>;
  constexpr int kRowBytes = C::kRowBytes;
  constexpr int kStageBytes = C::kStageBytes;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (128u - (smem_u32(smem_raw) & 127u)) & 127u;
  uint8_t* ring = smem_raw + pad;
  __shared__ DecodeSmem sm;

  const int c = blockIdx.x;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int dchunk = lane % C::kLanesPerKey;  // 8 head-dim values per lane
  const int kpar = lane / C::kLanesPerKey;    // which of the warp's keys this lane works on
  const int64_t bh = static_cast<int64_t>(b) * p.H + h;
  int len = p.Nkv;
  int chunk = p.chunk;
  if (PAGED) {
    // Per-sequence length; splits are whole 128-key multiples of it.
    len = p.seq_lens[b];
    if (len < 1 || len > p.max_blocks * p.block_size) {
      if (tid == 0) atomicCAS(p.err, 0u, (kKernDecode << 8) | kSiteBadLength);
      len = min(max(len, 1), p.max_blocks * p.block_size);
    }
    chunk = (((len + p.n_splits - 1) / p.n_splits) + 127) & ~127;
  }
  const int key0 = c * chunk;
  const int nkeys = max(0, min(len, key0 + chunk) - key0);
  const int nsub = (nkeys + kSub - 1) / kSub;
  const int page0 = PAGED ? key0 / max(p.block_size, 1) : 0;
  if (PAGED && nkeys > 0) {
    // Stage this range's page ids with one coalesced, checked load.
    const int npages = min(kMaxStagedPages, (key0 + nkeys - 1) / p.block_size - page0 + 1);
    for (int i = tid; i < npages; i += kThreads) sm.pages[i] = checked_page(p, b, page0 + i);
  }

  const uint8_t* kbase = reinterpret_cast<const uint8_t*>(p.k) + (bh * p.Nkv + key0) * kRowBytes;
  const uint8_t* vbase = reinterpret_cast<const uint8_t*>(p.v) + (bh * p.Nkv + key0) * kRowBytes;

  if (tid == 0) {
    mbar_init(&sm.full[0], 1);
    mbar_init(&sm.full[1], 1);
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  // Called by all of warp 0: lane 0 arms the stage's byte count, then every
  // lane issues its own copies, so a paged stage's pieces go out together.
  auto issue = [&](int i) {
    const int st = i & 1;
    const int n = min(kSub, nkeys - i * kSub);
    const uint32_t bytes = static_cast<uint32_t>(n) * kRowBytes;
    if (lane == 0) mbar_arrive_expect_tx(&sm.full[st], 2 * bytes);
    __syncwarp();
    if (!PAGED) {
      if (lane == 0) {
        bulk_load(ring + st * kStageBytes, kbase + static_cast<int64_t>(i) * kSub * kRowBytes, bytes, &sm.full[st]);
        bulk_load(ring + st * kStageBytes + kSub * kRowBytes, vbase + static_cast<int64_t>(i) * kSub * kRowBytes,
                  bytes, &sm.full[st]);
      }
    } else {
      // Lane r copies piece r: min(block_size, 64) rows starting at a piece
      // boundary, which is also a page boundary or the middle of a 128-row page.
      const int ps = min(p.block_size, kSub);
      const int r = lane * ps;
      if (r < n) {
        int rows;
        const uint8_t* ksrc = paged_row(p.k, p, sm.pages, page0, b, h, key0 + i * kSub + r, kRowBytes, &rows);
        const uint8_t* vsrc = paged_row(p.v, p, sm.pages, page0, b, h, key0 + i * kSub + r, kRowBytes, &rows);
        rows = min(min(rows, ps), n - r);
        bulk_load(ring + st * kStageBytes + r * kRowBytes, ksrc, rows * kRowBytes, &sm.full[st]);
        bulk_load(ring + st * kStageBytes + kSub * kRowBytes + r * kRowBytes, vsrc, rows * kRowBytes, &sm.full[st]);
      }
    }
  };
  if (warp == 0) {
    if (nsub > 0) issue(0);
    if (nsub > 1) issue(1);
  }

  // This lane's slice of q (8 values), widened to fp32.
  float qf[8];
  {
    const uint4 u = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(p.q) + bh * kRowBytes +
                                                    dchunk * 16);
    bf16x8_to_f32(u, qf);
  }
  const float sl2 = p.scale_log2;
  float m_run = -INFINITY, l_run = 0.f;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;

  int issued = min(nsub, 2);
  bool ok = true;
  for (int i = 0; i < nsub; ++i) {
    const int st = i & 1;
    const int n = min(kSub, nkeys - i * kSub);
    ok = mbar_wait(&sm.full[st], (i >> 1) & 1, &sm.abort_flag, p.err, site(1));
    if (!__syncthreads_and(ok)) { ok = false; break; }
    const uint8_t* sK = ring + st * kStageBytes;
    const uint8_t* sV = sK + kSub * kRowBytes;

    // Scores: each warp takes 16 keys, kKeysPerStep at a time.
#pragma unroll
    for (int pr = 0; pr < 16 / C::kKeysPerStep; ++pr) {
      const int key = warp * 16 + pr * C::kKeysPerStep + kpar;
      float kf[8];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(sK + key * kRowBytes + dchunk * 16), kf);
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) dot = fmaf(qf[e], kf[e], dot);
#pragma unroll
      for (int o = C::kLanesPerKey / 2; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
      if (dchunk == 0) sm.scores[key] = (key < n) ? dot * sl2 : -INFINITY;
    }
    __syncthreads();

    // Online softmax over this sub-chunk (every warp computes the same values).
    const float s0 = sm.scores[lane];
    const float s1 = sm.scores[lane + 32];
    float mx = fmaxf(s0, s1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float m_new = fmaxf(m_run, mx);
    const float corr = ex2_approx(m_run - m_new);
    const float p0 = ex2_approx(s0 - m_new);
    const float p1 = ex2_approx(s1 - m_new);
    float ps = p0 + p1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
    l_run = l_run * corr + ps;
    m_run = m_new;
    if (warp == 0) {
      sm.probs[lane] = p0;
      sm.probs[lane + 32] = p1;
    }
    __syncthreads();

    // P·V: lane owns 8 head-dim values; the kGroups (warp, key slot) groups split the keys.
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] *= corr;
#pragma unroll
    for (int ii = 0; ii < kSub / C::kGroups; ++ii) {
      const int key = ii * C::kGroups + warp * C::kKeysPerStep + kpar;
      if (key < n) {
        const float pk = sm.probs[key];
        float vf[8];
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(sV + key * kRowBytes + dchunk * 16), vf);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = fmaf(pk, vf[e], acc[e]);
      }
    }
    __syncthreads();
    if (i + 2 < nsub) {
      if (warp == 0) issue(i + 2);
      ++issued;
    }
  }
  if (!ok) {
    if (tid == 0) {
      for (int t = max(0, issued - 2); t < issued; ++t) mbar_wait_drain(&sm.full[t & 1], (t >> 1) & 1, 200000000ull);
    }
    return;
  }

  // Combine the key groups, then write the unnormalised triple.
  const int g = warp * C::kKeysPerStep + kpar;
#pragma unroll
  for (int e = 0; e < 8; ++e) sm.red[g * D + dchunk * 8 + e] = acc[e];
  __syncthreads();
  const int64_t slot = bh * p.n_splits + c;
  if (tid < D) {
    float o = 0.f;
#pragma unroll
    for (int gg = 0; gg < C::kGroups; ++gg) o += sm.red[gg * D + tid];
    p.part_o[slot * D + tid] = o;
  }
  if (tid == 0) {
    p.part_ml[slot * 2 + 0] = m_run;  // −∞ and ℓ = 0 for a split with no keys
    p.part_ml[slot * 2 + 1] = l_run;
  }
}

template <int D>
__global__ void __launch_bounds__(D) decode_merge_kernel(const DecodeParams p) {
  const int64_t bh = blockIdx.x;
  const int t = threadIdx.x;
  const float* ml = p.part_ml + bh * p.n_splits * 2;
  const float* po = p.part_o + bh * p.n_splits * D;
  float m = -INFINITY;
  for (int c = 0; c < p.n_splits; ++c) m = fmaxf(m, ml[2 * c]);
  float l = 0.f, o = 0.f;
  for (int c = 0; c < p.n_splits; ++c) {
    const float mc = ml[2 * c];
    const float w = (mc == -INFINITY) ? 0.f : ex2_approx(mc - m);
    l = fmaf(ml[2 * c + 1], w, l);
    o = fmaf(po[static_cast<int64_t>(c) * D + t], w, o);
  }
  reinterpret_cast<__nv_bfloat16*>(p.o)[bh * D + t] = __float2bfloat16_rn(o / l);
  if (t == 0 && p.lse != nullptr) p.lse[bh] = (m + __log2f(l)) * 0.69314718055994531f;
}

template <int D, bool PAGED>
cudaError_t launch_split(const DecodeParams& p, cudaStream_t stream) {
  constexpr int kSmem = DecCfg<D>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<D, PAGED>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  decode_split_kernel<D, PAGED><<<dim3(p.n_splits, p.H, p.B), kThreads, kSmem, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  decode_merge_kernel<D><<<p.B * p.H, D, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_paged_bf16(const DecodeParams& p, cudaStream_t stream) {
  if (p.G != 1) return cudaErrorInvalidValue;
  if (p.d == 128) return launch_split<128, true>(p, stream);
  if (p.d == 64) return launch_split<64, true>(p, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_merge(const DecodeParams& p, cudaStream_t stream) {
  if (p.d == 128)
    decode_merge_kernel<128><<<p.B * p.H, 128, 0, stream>>>(p);
  else if (p.d == 64)
    decode_merge_kernel<64><<<p.B * p.H, 64, 0, stream>>>(p);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_decode_bf16(int d, const DecodeParams& p, cudaStream_t stream) {
  if (p.G != 1 || d != p.d) return cudaErrorInvalidValue;  // groups go to the tensor-core kernel
  if (d == 128) return launch_split<128, false>(p, stream);
  if (d == 64) return launch_split<64, false>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa

// ----------------------------------------------------- library-owned scratch
// Scratch for fa_decode_splitkv_noalloc: the partial triples live in this
// fixed buffer instead of a caller workspace.  Every device that loads the
// library holds it until the process exits.  In host code the name is only a
// stand-in; the device address comes from cudaGetSymbolAddress below.
namespace fa {
namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[kDecodeStaticScratchBytes];

}  // namespace

cudaError_t decode_static_scratch(void** out) {
  static std::mutex mu;
  static void* cache[64] = {};
  static void* cache_ctx[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  void* ctx = nullptr;
  if ((e = current_context(&ctx)) != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == nullptr || ctx == nullptr || cache_ctx[dev] != ctx) {
    // Once per device (and again after a device reset gave it a new context),
    // with that device current.
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    if ((e = current_context(&ctx)) != cudaSuccess) return e;
    cache[dev] = p;
    cache_ctx[dev] = ctx;
  }
  *out = cache[dev];
  return cudaSuccess;
}

}  // namespace fa
