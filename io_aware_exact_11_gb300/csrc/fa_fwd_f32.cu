// fa_fwd_f32.cu — fp32 forward attention on CUDA cores, for exact checks.
//
// Same online-softmax recurrence as the tensor-core kernel ("FlashAttention：
// IO-aware 的注意力 kernel" §3.2): each query row keeps a running max m, a
// running normaliser ℓ and an unnormalised accumulator, rescaled by
// e^(m − m_new) as each key tile is consumed; O/ℓ and LSE = m + ln ℓ are
// written once at the end.  Everything is fp32 with correctly rounded expf,
// so it meets a 1e-5 bound where the tf32 tensor path (10-bit mantissa) cannot.
//
// With the causal mask (bottom-right aligned) row i sees keys j <= i + N_kv − N_q.
// CTA = 16 query rows of one (b, h), 4 warps × 4 rows.  Key/value tiles of 32
// keys are staged in shared memory; lane = key for the scores, lane = head-dim
// slice for the P·V accumulation.
#include "fa_kernels.h"

namespace fa {
namespace {

constexpr int kRows = 16;
constexpr int kKeys = 32;
constexpr int kThreads = 128;

template <int D>
__global__ void __launch_bounds__(kThreads) fwd_f32_kernel(const FwdF32Params p) {
  constexpr int kDL = D / 32;  // head-dim values per lane
  __shared__ float sQ[kRows][D];
  __shared__ float sK[kKeys][D + 1];
  __shared__ float sV[kKeys][D];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int r0 = blockIdx.x * kRows;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const float* q = p.q + b * p.q_sb + h * p.q_sh;
  const float* k = p.k + b * p.k_sb + h * p.k_sh;
  const float* v = p.v + b * p.v_sb + h * p.v_sh;

  for (int i = threadIdx.x; i < kRows * D; i += kThreads) {
    const int r = i / D, t = i % D;
    sQ[r][t] = (r0 + r < p.Nq) ? q[static_cast<int64_t>(r0 + r) * p.q_sn + t] : 0.f;
  }

  float m[4], l[4], acc[4][kDL];
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    m[rr] = -INFINITY;
    l[rr] = 0.f;
#pragma unroll
    for (int t = 0; t < kDL; ++t) acc[rr][t] = 0.f;
  }

  for (int j0 = 0; j0 < p.Nkv; j0 += kKeys) {
    __syncthreads();
    for (int i = threadIdx.x; i < kKeys * D; i += kThreads) {
      const int r = i / D, t = i % D;
      const bool ok = j0 + r < p.Nkv;
      sK[r][t] = ok ? k[static_cast<int64_t>(j0 + r) * p.k_sn + t] : 0.f;
      sV[r][t] = ok ? v[static_cast<int64_t>(j0 + r) * p.v_sn + t] : 0.f;
    }
    __syncthreads();
    const bool key_ok = j0 + lane < p.Nkv;
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int r = warp * 4 + rr;
      float dot = 0.f;
#pragma unroll 8
      for (int t = 0; t < D; ++t) dot = fmaf(sQ[r][t], sK[lane][t], dot);
      const bool vis = key_ok && (!p.causal || j0 + lane <= r0 + r + (p.Nkv - p.Nq));
      const float s = vis ? dot * p.scale : -INFINITY;
      float mx = s;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float m_new = fmaxf(m[rr], mx);
      const float corr = (m[rr] == -INFINITY) ? 0.f : expf(m[rr] - m_new);
      const float pk = vis ? expf(s - m_new) : 0.f;
      float ps = pk;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
      l[rr] = l[rr] * corr + ps;
#pragma unroll
      for (int t = 0; t < kDL; ++t) acc[rr][t] *= corr;
      for (int kk = 0; kk < kKeys; ++kk) {
        const float pj = __shfl_sync(0xffffffffu, pk, kk);
#pragma unroll
        for (int t = 0; t < kDL; ++t) acc[rr][t] = fmaf(pj, sV[kk][lane + 32 * t], acc[rr][t]);
      }
      m[rr] = m_new;
    }
  }

#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    const int gr = r0 + warp * 4 + rr;
    if (gr >= p.Nq) continue;
    float* orow = p.o + b * p.o_sb + h * p.o_sh + static_cast<int64_t>(gr) * p.o_sn;
    const float inv = 1.f / l[rr];
#pragma unroll
    for (int t = 0; t < kDL; ++t) orow[lane + 32 * t] = acc[rr][t] * inv;
    if (lane == 0 && p.lse != nullptr)
      p.lse[(static_cast<int64_t>(b) * p.H + h) * p.Nq + gr] = m[rr] + logf(l[rr]);
  }
}

}  // namespace

cudaError_t launch_fwd_f32(int d, const FwdF32Params& p, cudaStream_t stream) {
  dim3 grid((p.Nq + kRows - 1) / kRows, p.H, p.B);
  if (d == 128) {
    fwd_f32_kernel<128><<<grid, kThreads, 0, stream>>>(p);
  } else if (d == 64) {
    fwd_f32_kernel<64><<<grid, kThreads, 0, stream>>>(p);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace fa
