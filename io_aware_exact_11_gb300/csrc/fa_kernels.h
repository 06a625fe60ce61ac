// fa_kernels.h — launch interface between the C ABI (fa_api.cu) and the
// kernel translation units.  Internal to libfa.so.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fa {

// Watchdog codes written to the device error word: (kernel << 8) | wait site.
enum : unsigned int {
  kKernFwd = 1,
  kKernDecode = 2,
  kKernBwd = 3,
  kKernSelftest = 15,  // fa_watchdog_selftest
};

struct FwdParams {
  CUtensorMap tm_q;  // 4-D maps {d, N, H, B}, box {64, 128, 1, 1}, 128-byte swizzle
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  void* o;
  float* lse;  // may be null
  int B, H, Nq, Nkv;
  int64_t o_sb, o_sh, o_sn;  // element strides of O
  float scale_log2;          // σ·log2(e) (FP8: also × the Q and K descale factors)
  int causal;                // query i sees keys j <= i + (Nkv − Nq); needs Nq <= Nkv
  unsigned int* err;
  float o_scale = 1.f;       // multiplies O before the 1/ℓ (FP8: the V descale factor)
  CUtensorMap tm_o;          // O as {d, N_q, H, B} (its strides), box {64, 128, 1, 1}, 128-byte swizzle
};

struct FwdF32Params {
  const float* q;
  const float* k;
  const float* v;
  float* o;
  float* lse;
  int B, H, Nq, Nkv;
  int64_t q_sb, q_sh, q_sn, k_sb, k_sh, k_sn, v_sb, v_sh, v_sn, o_sb, o_sh, o_sn;
  float scale;
  int causal;
};

struct DecodeParams {
  const void* q;  // [B,H,d] bf16 (H query heads)
  const void* k;  // [B,Hkv,N,d] bf16
  const void* v;
  void* o;        // [B,H,d] bf16
  float* lse;     // [B,H] or null
  float* part_o;  // [B,H,S,d] fp32
  float* part_ml; // [B,H,S,2] fp32: (m in log2 units, ℓ)
  int B, H, Nkv, n_splits, chunk;
  float scale_log2;
  unsigned int* err;
  int Hkv = 0;    // key/value heads (informational; this kernel needs Hkv = H)
  int G = 1;      // query heads per key/value head; the CUDA-core kernel handles G = 1
  // Paged cache (k, v are [num_blocks, H, block_size, d]); null block_table = contiguous.
  const int* block_table = nullptr;  // [B, max_blocks]
  const int* seq_lens = nullptr;     // [B]
  int max_blocks = 0, block_size = 0, num_blocks = 0;
  int d = 128;  // head dim: 64 or 128
};

// Device-side argument checks report through the status word with these sites.
enum : unsigned int { kSiteBadBlock = 0xE1, kSiteBadLength = 0xE2 };

// Grouped-query split-KV decode on tensor cores (fa_decode_tc.cu).
struct DecodeTcParams {
  CUtensorMap tm_q;  // q viewed as [B·Hq rows, d]: 4-D map {d, B·Hq, 1, 1}, box {64, 128, 1, 1}
  CUtensorMap tm_k;  // {d, N, Hkv, B}, box {64, 128, 1, 1}; paged: {d, bs, Hkv, num_blocks}, box {64, bs, 1, 1}
  CUtensorMap tm_v;
  const int* block_table;  // paged cache only: [B, max_blocks]
  const int* seq_lens;     // paged cache only: [B]
  int max_blocks, block_size, num_blocks;
  float* part_o;     // [B,Hq,S,d] fp32
  float* part_ml;    // [B,Hq,S,2] fp32
  int B, Hq, Hkv, G, Nkv, n_splits, chunk;
  int d;             // head dim: 64 or 128
  float scale_log2;
  unsigned int* err;
};

struct BwdParams {
  CUtensorMap tm_q;   // {d, N, H, B}, box {64, 128, 1, 1}
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  CUtensorMap tm_do;
  const void* q;
  const void* o;
  const void* dout;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  float* dq_acc;      // [B,H,N,d] fp32, zeroed before the main kernel
  float* delta;       // [B,H,N]   D_i
  float* lse_log2;    // [B,H,N]   LSE·log2(e)
  int B, H, N;
  float scale;        // σ
  float scale_log2;   // σ·log2(e)
  int causal;         // key j visible to query i when j <= i
  unsigned int* err;
  CUtensorMap tm_dk;  // dK, dV as {d, N, H, B}, box {64, 128, 1, 1}, 128-byte swizzle (TMA stores)
  CUtensorMap tm_dv;
};

cudaError_t launch_fwd_bf16(int d, const FwdParams& p, cudaStream_t s);
// Unmasked bf16 forward at d = 64 with 3 or 4 query tiles of 128 rows per CTA
// (fa_fwd_d64.cu); K/V maps with 64-row boxes.
cudaError_t launch_fwd_d64_tiles(int query_tiles, const FwdParams& p, cudaStream_t s);
cudaError_t launch_fwd_fp8(int d, const FwdParams& p, cudaStream_t s);  // E4M3 Q/K/V, bf16 O
cudaError_t launch_fwd_f32(int d, const FwdF32Params& p, cudaStream_t s);
cudaError_t launch_decode_bf16(int d, const DecodeParams& p, cudaStream_t s);
cudaError_t launch_decode_merge(const DecodeParams& p, cudaStream_t s);
cudaError_t launch_decode_gqa_tc(const DecodeTcParams& p, cudaStream_t s);
cudaError_t launch_decode_paged_bf16(const DecodeParams& p, cudaStream_t s);
cudaError_t launch_decode_gqa_tc_paged(const DecodeTcParams& p, cudaStream_t s);
cudaError_t launch_bwd_bf16(int d, const BwdParams& p, cudaStream_t s, int* launches);

// Size of the library-owned decode scratch (fa_decode_splitkv_noalloc).
constexpr size_t kDecodeStaticScratchBytes = static_cast<size_t>(36) << 20;
// Device address of that scratch on the current device (looked up once per
// device and context).
cudaError_t decode_static_scratch(void** out);
// The calling thread's current CUDA context (null if the runtime has not bound
// one to the thread yet); keys the per-device caches of symbol addresses.
cudaError_t current_context(void** ctx);

}  // namespace fa
