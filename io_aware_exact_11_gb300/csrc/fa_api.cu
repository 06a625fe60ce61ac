// fa_api.cu — the C ABI declared in include/fa.h: argument checks, TMA
// descriptor construction and kernel dispatch.  No device memory is allocated
// here; every buffer, including workspaces, belongs to the caller.  The only
// resources the library creates are, per device, the two copy streams and the
// events fa_forward_host pipelines its transfers with.
#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/fa.h"
#include "fa_kernels.h"
#include "sm103.cuh"

namespace fa {
// One thread waits, with the same bounded wait every pipeline kernel uses, on
// an mbarrier that nothing completes.  The wait gives up after its limit,
// records (kKernSelftest << 8) | 1 in the watchdog word and the kernel returns:
// the failure path of a stuck pipeline, with nothing faulting or hanging.
__global__ void watchdog_selftest_kernel(unsigned int* err) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
    mbar_wait(&bar, 0, &abort_flag, err, (kKernSelftest << 8) | 1u);
  }
}

cudaError_t current_context(void** ctx) {
  typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
  static std::once_flag once;
  static CtxGetCurrentFn fn = nullptr;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    err = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q);
    if (err == cudaSuccess && q != cudaDriverEntryPointSuccess) err = cudaErrorSymbolNotFound;
    if (err == cudaSuccess) fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  if (fn == nullptr) return err != cudaSuccess ? err : cudaErrorSymbolNotFound;
  CUcontext c = nullptr;
  if (fn(&c) != CUDA_SUCCESS) return cudaErrorContextIsDestroyed;
  *ctx = c;  // null while the runtime has not yet bound a context to this thread
  return cudaSuccess;
}
}  // namespace fa

namespace {

thread_local char g_last_error[512] = "";
std::atomic<uint64_t> g_launches{0};

// One watchdog word per device: kernels write the site of a wait that gave up.
__device__ unsigned int g_watchdog_word;

fa_status fail(fa_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return s;
}

fa_status ok() {
  g_last_error[0] = '\0';
  return FA_OK;
}

fa_status cuda_fail(cudaError_t e, const char* where) {
  return fail(FA_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Device address of this device's watchdog word, looked up once per device and
// context: a device reset (a new primary context) triggers a fresh lookup.
fa_status watchdog_ptr(unsigned int** out) {
  static std::mutex mu;
  static unsigned int* cache[64] = {};
  static void* cache_ctx[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(FA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  void* ctx = nullptr;
  if ((e = fa::current_context(&ctx)) != cudaSuccess) return cuda_fail(e, "cuCtxGetCurrent");
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == nullptr || ctx == nullptr || cache_ctx[dev] != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_watchdog_word);  // binds the device's context if none was
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(watchdog)");
    if ((e = fa::current_context(&ctx)) != cudaSuccess) return cuda_fail(e, "cuCtxGetCurrent");
    cache[dev] = static_cast<unsigned int*>(p);
    cache_ctx[dev] = ctx;
  }
  *out = cache[dev];
  return FA_OK;
}

// ------------------------------------------------------------ tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

fa_status get_encoder(EncodeTiledFn* fn) {
  static std::once_flag once;
  static EncodeTiledFn cached = nullptr;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (err == cudaSuccess && q == cudaDriverEntryPointSuccess) cached = reinterpret_cast<EncodeTiledFn>(p);
  });
  if (cached == nullptr) {
    return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (%s)",
                err == cudaSuccess ? "symbol not found" : cudaGetErrorString(err));
  }
  *fn = cached;
  return FA_OK;
}

// 4-D bf16 map over a [B, H, N, d] tensor with element strides (sb, sh, sn),
// d contiguous; box = 64 head-dim values × 128 rows, 128-byte swizzle; rows
// past N read as zero.
fa_status make_map(CUtensorMap* tm, const void* base, int B, int H, int N, int d, int64_t sb, int64_t sh,
                   int64_t sn, const char* name, int box_rows = 128, bool fp8 = false) {
  EncodeTiledFn enc;
  fa_status s = get_encoder(&enc);
  if (s != FA_OK) return s;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(B)};
  // One box row is 128 bytes (the swizzle width): 64 bf16 or 128 E4M3 values.
  const int esz = fp8 ? 1 : 2;
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(sn) * esz, static_cast<cuuint64_t>(sh) * esz,
                           static_cast<cuuint64_t>(sb) * esz};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / esz), static_cast<cuuint32_t>(box_rows), 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(tm, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                   const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FA_ERR_INVALID_ARG, "cuTensorMapEncodeTiled(%s) failed with %d", name, (int)r);
  return FA_OK;
}

// 5-D bf16 map over a paged cache [num_blocks, H_kv, bs, 128] that loads one
// page of one head as a single box laid out for the tensor cores: dimensions
// (64 columns, 8 rows, 2 column halves, bs/8 row groups, page·H_kv + head), so
// a page lands as [row group][half][8 rows][128 bytes] and every 8-row group of
// a key tile is 2 KB from the next whatever the page size.  The column halves
// (stride 128 bytes) come after the rows (stride 256 bytes); page and head
// merge into one dimension because a page's heads are contiguous.
fa_status make_page_map5(CUtensorMap* tm, const void* base, int num_blocks, int H_kv, int bs, const char* name) {
  EncodeTiledFn enc;
  fa_status s = get_encoder(&enc);
  if (s != FA_OK) return s;
  cuuint64_t dims[5] = {64, 8, 2, static_cast<cuuint64_t>(bs / 8),
                        static_cast<cuuint64_t>(num_blocks) * static_cast<cuuint64_t>(H_kv)};
  cuuint64_t strides[4] = {256, 128, 8 * 256, static_cast<cuuint64_t>(bs) * 256};
  cuuint32_t box[5] = {64, 8, 2, static_cast<cuuint32_t>(bs / 8), 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FA_ERR_INVALID_ARG, "cuTensorMapEncodeTiled(%s) failed with %d", name, (int)r);
  return FA_OK;
}

bool bad_scale(float scale) { return !(std::isfinite(scale) && scale > 0.f); }

fa_status check_launch(const char* what, int n) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, what);
  g_launches.fetch_add(static_cast<uint64_t>(n), std::memory_order_relaxed);
  return ok();
}

}  // namespace

extern "C" {

int fa_abi_version(void) { return 1; }

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported configuration";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_DEVICE_TIMEOUT: return "device pipeline wait timed out";
  }
  return "unknown status";
}

const char* fa_get_last_error(void) { return g_last_error; }

uint64_t fa_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"

namespace {

fa_status forward_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N_q,
                       int N_kv, int d, fa_dtype dtype, float scale, const int64_t* strides, int causal,
                       void* stream) {
  if (!q || !k || !v || !o) return fail(FA_ERR_INVALID_ARG, "fa_forward: null tensor pointer");
  if (B <= 0 || H <= 0 || N_q <= 0 || N_kv <= 0 || d <= 0)
    return fail(FA_ERR_INVALID_ARG, "fa_forward: sizes must be positive (B=%d H=%d N_q=%d N_kv=%d d=%d)", B, H,
                N_q, N_kv, d);
  if (dtype != FA_BF16 && dtype != FA_FP32) return fail(FA_ERR_INVALID_ARG, "fa_forward: unknown dtype %d", dtype);
  if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED, "fa_forward: head dim %d not built (64, 128)", d);
  if (bad_scale(scale)) return fail(FA_ERR_INVALID_ARG, "fa_forward: scale must be finite and > 0");
  if (B > 65535 || H > 65535) return fail(FA_ERR_UNSUPPORTED, "fa_forward: B and H must be <= 65535");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
    return fail(FA_ERR_INVALID_ARG, "fa_forward: q, k, v, o must be 16-byte aligned");
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u))
    return fail(FA_ERR_INVALID_ARG, "fa_forward: lse must be 4-byte aligned");
  if (causal && N_q > N_kv)
    return fail(FA_ERR_INVALID_ARG, "fa_forward: causal attention needs N_q <= N_kv (got %d > %d)", N_q, N_kv);
  if (causal && (N_q + 255) / 256 > 65535)  // the causal grid puts the 256-row query blocks on its y axis
    return fail(FA_ERR_UNSUPPORTED, "fa_forward: causal attention needs N_q <= %d", 65535 * 256);
  const int esz = dtype == FA_BF16 ? 2 : 4;
  int64_t st[12];
  if (strides == nullptr) {
    const int64_t nq = static_cast<int64_t>(N_q) * d, nk = static_cast<int64_t>(N_kv) * d;
    const int64_t def[12] = {H * nq, nq, d, H * nk, nk, d, H * nk, nk, d, H * nq, nq, d};
    memcpy(st, def, sizeof(st));
  } else {
    memcpy(st, strides, sizeof(st));
    for (int i = 0; i < 12; ++i) {
      if (st[i] < 0 || (st[i] * esz) % 16 != 0)
        return fail(FA_ERR_INVALID_ARG, "fa_forward: stride[%d]=%lld must be >= 0 and a multiple of 16 bytes", i,
                    static_cast<long long>(st[i]));
    }
    if (st[2] < d || st[5] < d || st[8] < d || st[11] < d)
      return fail(FA_ERR_INVALID_ARG, "fa_forward: row strides must be >= d");
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == FA_BF16) {
    fa::FwdParams p;
    memset(&p, 0, sizeof(p));
    fa_status r;
    if ((r = make_map(&p.tm_q, q, B, H, N_q, d, st[0], st[1], st[2], "q")) != FA_OK) return r;
    // The unmasked d = 64 kernel streams 64-key tiles; every other case 128.
    const bool d64_tiles = d == 64 && !causal;
    const int kv_rows = d64_tiles ? 64 : 128;
    if ((r = make_map(&p.tm_k, k, B, H, N_kv, d, st[3], st[4], st[5], "k", kv_rows)) != FA_OK) return r;
    if ((r = make_map(&p.tm_v, v, B, H, N_kv, d, st[6], st[7], st[8], "v", kv_rows)) != FA_OK) return r;
    if ((r = make_map(&p.tm_o, o, B, H, N_q, d, st[9], st[10], st[11], "o")) != FA_OK) return r;
    if ((r = watchdog_ptr(&p.err)) != FA_OK) return r;
    p.o = o;
    p.lse = lse;
    p.B = B;
    p.H = H;
    p.Nq = N_q;
    p.Nkv = N_kv;
    p.o_sb = st[9];
    p.o_sh = st[10];
    p.o_sn = st[11];
    p.scale_log2 = scale * 1.4426950408889634f;
    p.causal = causal;
    p.o_scale = 1.f;
    cudaError_t e = d64_tiles ? fa::launch_fwd_d64_tiles(4, p, s) : fa::launch_fwd_bf16(d, p, s);
    if (e != cudaSuccess) return cuda_fail(e, "fa_forward launch");
    return check_launch("fa_forward", 1);
  }
  fa::FwdF32Params p;
  p.q = static_cast<const float*>(q);
  p.k = static_cast<const float*>(k);
  p.v = static_cast<const float*>(v);
  p.o = static_cast<float*>(o);
  p.lse = lse;
  p.B = B;
  p.H = H;
  p.Nq = N_q;
  p.Nkv = N_kv;
  p.q_sb = st[0]; p.q_sh = st[1]; p.q_sn = st[2];
  p.k_sb = st[3]; p.k_sh = st[4]; p.k_sn = st[5];
  p.v_sb = st[6]; p.v_sh = st[7]; p.v_sn = st[8];
  p.o_sb = st[9]; p.o_sh = st[10]; p.o_sn = st[11];
  p.scale = scale;
  p.causal = causal;
  cudaError_t e = fa::launch_fwd_f32(d, p, s);
  if (e != cudaSuccess) return cuda_fail(e, "fa_forward (fp32) launch");
  return check_launch("fa_forward", 1);
}

}  // namespace

extern "C" {

fa_status fa_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N_q,
                     int N_kv, int d, fa_dtype dtype, float scale, const int64_t* strides, void* stream) {
  return forward_impl(q, k, v, o, lse, B, H, N_q, N_kv, d, dtype, scale, strides, 0, stream);
}

fa_status fa_forward_masked(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N_q,
                            int N_kv, int d, fa_dtype dtype, float scale, const int64_t* strides, fa_mask mask,
                            void* stream) {
  if (mask != FA_MASK_NONE && mask != FA_MASK_CAUSAL)
    return fail(FA_ERR_INVALID_ARG, "fa_forward_masked: unknown mask %d", static_cast<int>(mask));
  return forward_impl(q, k, v, o, lse, B, H, N_q, N_kv, d, dtype, scale, strides, mask == FA_MASK_CAUSAL ? 1 : 0,
                      stream);
}

fa_status fa_forward_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N_q,
                         int N_kv, int d, float scale, float q_descale, float k_descale, float v_descale,
                         fa_mask mask, void* stream) {
  if (!q || !k || !v || !o) return fail(FA_ERR_INVALID_ARG, "fa_forward_fp8: null tensor pointer");
  if (B <= 0 || H <= 0 || N_q <= 0 || N_kv <= 0 || d <= 0)
    return fail(FA_ERR_INVALID_ARG, "fa_forward_fp8: sizes must be positive");
  if (mask != FA_MASK_NONE && mask != FA_MASK_CAUSAL)
    return fail(FA_ERR_INVALID_ARG, "fa_forward_fp8: unknown mask %d", static_cast<int>(mask));
  if (d != 128) return fail(FA_ERR_UNSUPPORTED, "fa_forward_fp8: only d=128 is built (got %d)", d);
  if (bad_scale(scale) || bad_scale(q_descale) || bad_scale(k_descale) || bad_scale(v_descale))
    return fail(FA_ERR_INVALID_ARG, "fa_forward_fp8: scale and descale factors must be finite and > 0");
  if (B > 65535 || H > 65535) return fail(FA_ERR_UNSUPPORTED, "fa_forward_fp8: B and H must be <= 65535");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
    return fail(FA_ERR_INVALID_ARG, "fa_forward_fp8: q, k, v, o must be 16-byte aligned");
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u))
    return fail(FA_ERR_INVALID_ARG, "fa_forward_fp8: lse must be 4-byte aligned");
  if (mask == FA_MASK_CAUSAL && N_q > N_kv)
    return fail(FA_ERR_INVALID_ARG, "fa_forward_fp8: causal attention needs N_q <= N_kv");
  if (mask == FA_MASK_CAUSAL && (N_q + 255) / 256 > 65535)
    return fail(FA_ERR_UNSUPPORTED, "fa_forward_fp8: causal attention needs N_q <= %d", 65535 * 256);
  fa::FwdParams p;
  memset(&p, 0, sizeof(p));
  const int64_t nq = static_cast<int64_t>(N_q) * d, nk = static_cast<int64_t>(N_kv) * d;
  fa_status r;
  if ((r = make_map(&p.tm_q, q, B, H, N_q, d, H * nq, nq, d, "q", 128, true)) != FA_OK) return r;
  if ((r = make_map(&p.tm_k, k, B, H, N_kv, d, H * nk, nk, d, "k", 128, true)) != FA_OK) return r;
  if ((r = make_map(&p.tm_v, v, B, H, N_kv, d, H * nk, nk, d, "v", 128, true)) != FA_OK) return r;
  if ((r = make_map(&p.tm_o, o, B, H, N_q, d, H * nq, nq, d, "o")) != FA_OK) return r;
  if ((r = watchdog_ptr(&p.err)) != FA_OK) return r;
  p.o = o;
  p.lse = lse;
  p.B = B;
  p.H = H;
  p.Nq = N_q;
  p.Nkv = N_kv;
  p.o_sb = H * nq;
  p.o_sh = nq;
  p.o_sn = d;
  // True scores are q_descale·k_descale·(Q₈K₈ᵀ); true O is v_descale·(P̃V₈)/ℓ.
  p.scale_log2 = scale * q_descale * k_descale * 1.4426950408889634f;
  p.o_scale = v_descale;
  p.causal = mask == FA_MASK_CAUSAL ? 1 : 0;
  cudaError_t e = fa::launch_fwd_fp8(d, p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fa_forward_fp8 launch");
  return check_launch("fa_forward_fp8", 1);
}

}  // extern "C"

namespace {

// ------------------------------------------------ host-buffer forward
// Per-device copy streams and events for fa_forward_host, created on first use
// and kept for the life of the process.  The mutex serialises calls on one
// device: they share the events (a stream wait captures the event's latest
// record when it is queued, so reuse across chunks and calls is safe).
struct HostPipe {
  std::mutex mu;
  bool ready = false;
  int sms = 1;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr;
  cudaEvent_t in_done[2] = {nullptr, nullptr};   // chunk's q, k, v are on the device
  cudaEvent_t fwd_done[2] = {nullptr, nullptr};  // chunk's forward has finished
  cudaEvent_t out_done[2] = {nullptr, nullptr};  // chunk's o, lse are back on the host
  bool last_eager = false;                       // out_done last recorded outside a graph capture
};
HostPipe g_pipes[64];

fa_status init_pipe(HostPipe& hp, int dev) {
  cudaError_t e;
  if ((e = cudaDeviceGetAttribute(&hp.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return cuda_fail(e, "fa_forward_host: SM count");
  if ((e = cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking)) != cudaSuccess ||
      (e = cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking)) != cudaSuccess ||
      (e = cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming)) != cudaSuccess)
    return cuda_fail(e, "fa_forward_host: stream/event creation");
  for (int b = 0; b < 2; ++b) {
    if ((e = cudaEventCreateWithFlags(&hp.in_done[b], cudaEventDisableTiming)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&hp.fwd_done[b], cudaEventDisableTiming)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&hp.out_done[b], cudaEventDisableTiming)) != cudaSuccess)
      return cuda_fail(e, "fa_forward_host: event creation");
  }
  hp.ready = true;
  return FA_OK;
}

// Byte offsets of one chunk buffer inside the workspace.
struct HostChunk {
  size_t q, k, v, o, lse, bytes;
};

HostChunk host_chunk(int N_q, int N_kv, int d, int esz, int heads) {
  HostChunk c;
  const size_t hq = static_cast<size_t>(heads) * N_q * d * esz, hk = static_cast<size_t>(heads) * N_kv * d * esz;
  c.q = 0;
  c.k = c.q + round256(hq);
  c.v = c.k + round256(hk);
  c.o = c.v + round256(hk);
  c.lse = c.o + round256(hq);
  c.bytes = c.lse + round256(static_cast<size_t>(heads) * N_q * 4);
  return c;
}

// Heads per chunk: the caller's choice, or about eight chunks with at least
// two waves of 256-row blocks each.
int64_t chunk_heads(int64_t heads, int N_q, int requested, int sms) {
  int64_t hpc = requested;
  if (hpc == 0) {
    const int64_t blocks_per_head = (N_q + 255) / 256;
    hpc = std::max<int64_t>((heads + 7) / 8, (2 * static_cast<int64_t>(sms) + blocks_per_head - 1) / blocks_per_head);
  }
  return std::min<int64_t>(std::min<int64_t>(hpc, heads), 65535);
}

}  // namespace

extern "C" {

size_t fa_forward_host_workspace_size(int B, int H, int N_q, int N_kv, int d, fa_dtype dtype, int heads_per_chunk) {
  if (B <= 0 || H <= 0 || N_q <= 0 || N_kv <= 0 || d <= 0 || heads_per_chunk < 0) return 0;
  if (dtype != FA_BF16 && dtype != FA_FP32) return 0;
  int sms = 1;
  if (heads_per_chunk == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return 0;
  }
  const int64_t hpc = chunk_heads(static_cast<int64_t>(B) * H, N_q, heads_per_chunk, sms);
  return 2 * host_chunk(N_q, N_kv, d, dtype == FA_BF16 ? 2 : 4, static_cast<int>(hpc)).bytes;
}

fa_status fa_forward_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N_q,
                          int N_kv, int d, fa_dtype dtype, float scale, fa_mask mask, int heads_per_chunk,
                          void* workspace, size_t workspace_bytes, void* stream) {
  // Every check fa_forward_masked makes on a chunk is made here first, so a
  // bad argument returns before any copy is queued.
  if (!q || !k || !v || !o) return fail(FA_ERR_INVALID_ARG, "fa_forward_host: null tensor pointer");
  if (!workspace) return fail(FA_ERR_INVALID_ARG, "fa_forward_host: null workspace");
  if (B <= 0 || H <= 0 || N_q <= 0 || N_kv <= 0 || d <= 0)
    return fail(FA_ERR_INVALID_ARG, "fa_forward_host: sizes must be positive (B=%d H=%d N_q=%d N_kv=%d d=%d)", B, H,
                N_q, N_kv, d);
  if (dtype != FA_BF16 && dtype != FA_FP32) return fail(FA_ERR_INVALID_ARG, "fa_forward_host: unknown dtype %d", dtype);
  if (mask != FA_MASK_NONE && mask != FA_MASK_CAUSAL)
    return fail(FA_ERR_INVALID_ARG, "fa_forward_host: unknown mask %d", static_cast<int>(mask));
  if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED, "fa_forward_host: head dim %d not built (64, 128)", d);
  if (bad_scale(scale)) return fail(FA_ERR_INVALID_ARG, "fa_forward_host: scale must be finite and > 0");
  if (mask == FA_MASK_CAUSAL && N_q > N_kv)
    return fail(FA_ERR_INVALID_ARG, "fa_forward_host: causal attention needs N_q <= N_kv (got %d > %d)", N_q, N_kv);
  if (heads_per_chunk < 0) return fail(FA_ERR_INVALID_ARG, "fa_forward_host: heads_per_chunk must be >= 0");
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return fail(FA_ERR_INVALID_ARG, "fa_forward_host: workspace must be 256-byte aligned");
  const int64_t heads = static_cast<int64_t>(B) * H;
  const int esz = dtype == FA_BF16 ? 2 : 4;
  if (heads_per_chunk > 0) {  // the size is known without asking the device
    const int hpc = static_cast<int>(chunk_heads(heads, N_q, heads_per_chunk, 1));
    const size_t need = 2 * host_chunk(N_q, N_kv, d, esz, hpc).bytes;
    if (workspace_bytes < need)
      return fail(FA_ERR_INVALID_ARG, "fa_forward_host: workspace of %zu bytes is smaller than the %zu needed",
                  workspace_bytes, need);
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(FA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  HostPipe& hp = g_pipes[dev];
  std::lock_guard<std::mutex> lock(hp.mu);
  if (!hp.ready) {
    fa_status r = init_pipe(hp, dev);
    if (r != FA_OK) return r;
  }
  const int64_t hpc = chunk_heads(heads, N_q, heads_per_chunk, hp.sms);
  const HostChunk L = host_chunk(N_q, N_kv, d, esz, static_cast<int>(hpc));
  if (workspace_bytes < 2 * L.bytes)
    return fail(FA_ERR_INVALID_ARG, "fa_forward_host: workspace of %zu bytes is smaller than the %zu needed",
                workspace_bytes, 2 * L.bytes);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t q_head = static_cast<size_t>(N_q) * d * esz, kv_head = static_cast<size_t>(N_kv) * d * esz;
  const int64_t chunks = (heads + hpc - 1) / hpc;
#define FA_HOST_CUDA(call, what)                  \
  do {                                            \
    cudaError_t ce_ = (call);                     \
    if (ce_ != cudaSuccess) return cuda_fail(ce_, what); \
  } while (0)
  FA_HOST_CUDA(cudaEventRecord(hp.start, s), "fa_forward_host: event record");
  FA_HOST_CUDA(cudaStreamWaitEvent(hp.h2d, hp.start, 0), "fa_forward_host: stream wait");
  FA_HOST_CUDA(cudaStreamWaitEvent(hp.d2h, hp.start, 0), "fa_forward_host: stream wait");
  // The previous call on this device (perhaps from another thread, on another
  // stream, with the same workspace) must have copied its results out before
  // this call's first copy in: its last copy-out events cover all of its work.
  // Only eager calls are ordered this way; a wait across a graph capture's edge
  // is not allowed, and a captured call is ordered by whoever replays it.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  FA_HOST_CUDA(cudaStreamIsCapturing(s, &cap), "fa_forward_host: capture query");
  const bool eager = cap == cudaStreamCaptureStatusNone;
  if (eager && hp.last_eager)
    for (int b = 0; b < 2; ++b)
      FA_HOST_CUDA(cudaStreamWaitEvent(hp.h2d, hp.out_done[b], 0), "fa_forward_host: stream wait");
  hp.last_eager = eager;
  for (int64_t c = 0; c < chunks; ++c) {
    const int b = static_cast<int>(c & 1);
    const int64_t h0 = c * hpc;
    const int nh = static_cast<int>(std::min<int64_t>(hpc, heads - h0));
    uint8_t* buf = ws + b * L.bytes;
    // Buffer b was last used by chunk c − 2: its results must be home first.
    if (c >= 2) FA_HOST_CUDA(cudaStreamWaitEvent(hp.h2d, hp.out_done[b], 0), "fa_forward_host: stream wait");
    FA_HOST_CUDA(cudaMemcpyAsync(buf + L.q, static_cast<const uint8_t*>(q) + h0 * q_head, nh * q_head,
                                 cudaMemcpyHostToDevice, hp.h2d), "fa_forward_host: copy q in");
    FA_HOST_CUDA(cudaMemcpyAsync(buf + L.k, static_cast<const uint8_t*>(k) + h0 * kv_head, nh * kv_head,
                                 cudaMemcpyHostToDevice, hp.h2d), "fa_forward_host: copy k in");
    FA_HOST_CUDA(cudaMemcpyAsync(buf + L.v, static_cast<const uint8_t*>(v) + h0 * kv_head, nh * kv_head,
                                 cudaMemcpyHostToDevice, hp.h2d), "fa_forward_host: copy v in");
    FA_HOST_CUDA(cudaEventRecord(hp.in_done[b], hp.h2d), "fa_forward_host: event record");
    FA_HOST_CUDA(cudaStreamWaitEvent(s, hp.in_done[b], 0), "fa_forward_host: stream wait");
    fa_status r = forward_impl(buf + L.q, buf + L.k, buf + L.v, buf + L.o,
                               lse ? reinterpret_cast<float*>(buf + L.lse) : nullptr, 1, nh, N_q, N_kv, d, dtype,
                               scale, nullptr, mask == FA_MASK_CAUSAL ? 1 : 0, s);
    if (r != FA_OK) return r;
    FA_HOST_CUDA(cudaEventRecord(hp.fwd_done[b], s), "fa_forward_host: event record");
    FA_HOST_CUDA(cudaStreamWaitEvent(hp.d2h, hp.fwd_done[b], 0), "fa_forward_host: stream wait");
    FA_HOST_CUDA(cudaMemcpyAsync(static_cast<uint8_t*>(o) + h0 * q_head, buf + L.o, nh * q_head,
                                 cudaMemcpyDeviceToHost, hp.d2h), "fa_forward_host: copy o out");
    if (lse)
      FA_HOST_CUDA(cudaMemcpyAsync(lse + h0 * N_q, buf + L.lse, static_cast<size_t>(nh) * N_q * 4,
                                   cudaMemcpyDeviceToHost, hp.d2h), "fa_forward_host: copy lse out");
    FA_HOST_CUDA(cudaEventRecord(hp.out_done[b], hp.d2h), "fa_forward_host: event record");
  }
  // The copy-out stream runs the chunks in order: its last event covers them all.
  FA_HOST_CUDA(cudaStreamWaitEvent(s, hp.out_done[(chunks - 1) & 1], 0), "fa_forward_host: stream wait");
#undef FA_HOST_CUDA
  return ok();
}

int fa_decode_choose_splits(int B, int H_q, int H_kv, int N_kv) {
  if (B <= 0 || H_q <= 0 || H_kv <= 0 || N_kv <= 0 || H_q % H_kv != 0) return 0;
  int sms = 152;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 152;
  cudaGetLastError();  // a failed query on a machine without a device is not an error here
  const bool grouped = H_q > H_kv;
  const double heads = static_cast<double>(B) * (grouped ? H_kv : H_q);
  const double want = (grouped ? 1.0 : 27.0) * sms / heads;  // splits that give the target CTA count
  int s = 1;
  while (s < 256 && 2.0 * s <= want * 1.41421356) s *= 2;  // nearest power of two (geometric)
  while (s > 1 && static_cast<int64_t>(s) * 256 > N_kv) s /= 2;
  return s;
}

size_t fa_decode_workspace_size(int B, int H, int d, int n_splits) {
  if (B <= 0 || H <= 0 || d <= 0 || n_splits <= 0) return 0;
  const size_t slots = static_cast<size_t>(B) * H * n_splits;
  return round256(slots * d * 4) + round256(slots * 2 * 4);
}

fa_status fa_decode_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                            int N_kv, int d, fa_dtype dtype, float scale, int n_splits, void* workspace,
                            size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !o || !workspace) return fail(FA_ERR_INVALID_ARG, "fa_decode_splitkv: null pointer");
  if (B <= 0 || H <= 0 || N_kv <= 0 || d <= 0 || n_splits <= 0)
    return fail(FA_ERR_INVALID_ARG, "fa_decode_splitkv: sizes must be positive");
  if (dtype != FA_BF16 && dtype != FA_FP32) return fail(FA_ERR_INVALID_ARG, "fa_decode_splitkv: unknown dtype");
  if (dtype != FA_BF16 || (d != 64 && d != 128))
    return fail(FA_ERR_UNSUPPORTED, "fa_decode_splitkv: only bf16 with d = 64 or 128 is built");
  if (n_splits > 256) return fail(FA_ERR_UNSUPPORTED, "fa_decode_splitkv: n_splits must be <= 256");
  if (B > 65535 || H > 65535) return fail(FA_ERR_UNSUPPORTED, "fa_decode_splitkv: B and H must be <= 65535");
  if (bad_scale(scale)) return fail(FA_ERR_INVALID_ARG, "fa_decode_splitkv: scale must be finite and > 0");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(workspace))
    return fail(FA_ERR_INVALID_ARG, "fa_decode_splitkv: pointers must be 16-byte aligned");
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u))
    return fail(FA_ERR_INVALID_ARG, "fa_decode_splitkv: lse must be 4-byte aligned");
  const size_t need = fa_decode_workspace_size(B, H, d, n_splits);
  if (workspace_bytes < need)
    return fail(FA_ERR_INVALID_ARG, "fa_decode_splitkv: workspace %zu bytes, need %zu", workspace_bytes, need);
  fa::DecodeParams p;
  p.q = q;
  p.k = k;
  p.v = v;
  p.o = o;
  p.lse = lse;
  const size_t slots = static_cast<size_t>(B) * H * n_splits;
  p.part_o = static_cast<float*>(workspace);
  p.part_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) + round256(slots * d * 4));
  p.B = B;
  p.H = H;
  p.Nkv = N_kv;
  p.n_splits = n_splits;
  p.d = d;
  p.chunk = (N_kv + n_splits - 1) / n_splits;
  p.scale_log2 = scale * 1.4426950408889634f;
  fa_status r = watchdog_ptr(&p.err);
  if (r != FA_OK) return r;
  cudaError_t e = fa::launch_decode_bf16(d, p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fa_decode_splitkv launch");
  return check_launch("fa_decode_splitkv", 2);
}

// Same kernels as fa_decode_splitkv; the partial triples live in the library's
// own scratch buffer (fa_decode.cu) instead of a caller workspace.
fa_status fa_decode_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                    int N_kv, int d, fa_dtype dtype, float scale, int n_splits, void* stream) {
  if (!q || !k || !v || !o) return fail(FA_ERR_INVALID_ARG, "fa_decode_splitkv_noalloc: null pointer");
  if (B <= 0 || H <= 0 || N_kv <= 0 || d <= 0 || n_splits <= 0)
    return fail(FA_ERR_INVALID_ARG, "fa_decode_splitkv_noalloc: sizes must be positive");
  if (dtype != FA_BF16 && dtype != FA_FP32)
    return fail(FA_ERR_INVALID_ARG, "fa_decode_splitkv_noalloc: unknown dtype");
  if (dtype != FA_BF16 || (d != 64 && d != 128))
    return fail(FA_ERR_UNSUPPORTED, "fa_decode_splitkv_noalloc: only bf16 with d = 64 or 128 is built");
  if (n_splits > 256) return fail(FA_ERR_UNSUPPORTED, "fa_decode_splitkv_noalloc: n_splits must be <= 256");
  if (B > 65535 || H > 65535) return fail(FA_ERR_UNSUPPORTED, "fa_decode_splitkv_noalloc: B and H must be <= 65535");
  if (bad_scale(scale)) return fail(FA_ERR_INVALID_ARG, "fa_decode_splitkv_noalloc: scale must be finite and > 0");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
    return fail(FA_ERR_INVALID_ARG, "fa_decode_splitkv_noalloc: pointers must be 16-byte aligned");
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u))
    return fail(FA_ERR_INVALID_ARG, "fa_decode_splitkv_noalloc: lse must be 4-byte aligned");
  const size_t need = fa_decode_workspace_size(B, H, d, n_splits);
  if (need > fa::kDecodeStaticScratchBytes)
    return fail(FA_ERR_UNSUPPORTED,
                "fa_decode_splitkv_noalloc: needs %zu bytes of scratch, the built-in buffer holds %zu "
                "(use fa_decode_splitkv with a workspace)",
                need, fa::kDecodeStaticScratchBytes);
  void* scratch = nullptr;
  cudaError_t e = fa::decode_static_scratch(&scratch);
  if (e != cudaSuccess) return cuda_fail(e, "fa_decode_splitkv_noalloc: scratch address");
  fa::DecodeParams p;
  p.q = q;
  p.k = k;
  p.v = v;
  p.o = o;
  p.lse = lse;
  const size_t slots = static_cast<size_t>(B) * H * n_splits;
  p.part_o = static_cast<float*>(scratch);
  p.part_ml = reinterpret_cast<float*>(static_cast<char*>(scratch) + round256(slots * d * 4));
  p.B = B;
  p.H = H;
  p.Nkv = N_kv;
  p.n_splits = n_splits;
  p.d = d;
  p.chunk = (N_kv + n_splits - 1) / n_splits;
  p.scale_log2 = scale * 1.4426950408889634f;
  fa_status r = watchdog_ptr(&p.err);
  if (r != FA_OK) return r;
  e = fa::launch_decode_bf16(d, p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fa_decode_splitkv_noalloc launch");
  return check_launch("fa_decode_splitkv_noalloc", 2);
}

fa_status fa_decode_splitkv_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H_q,
                                int H_kv, int N_kv, int d, fa_dtype dtype, float scale, int n_splits, void* workspace,
                                size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !o || !workspace) return fail(FA_ERR_INVALID_ARG, "fa_decode_splitkv_gqa: null pointer");
  if (B <= 0 || H_q <= 0 || H_kv <= 0 || N_kv <= 0 || d <= 0 || n_splits <= 0)
    return fail(FA_ERR_INVALID_ARG, "fa_decode_splitkv_gqa: sizes must be positive");
  if (H_q % H_kv != 0)
    return fail(FA_ERR_INVALID_ARG, "fa_decode_splitkv_gqa: H_q (%d) must be a multiple of H_kv (%d)", H_q, H_kv);
  if (dtype != FA_BF16 && dtype != FA_FP32) return fail(FA_ERR_INVALID_ARG, "fa_decode_splitkv_gqa: unknown dtype");
  if (dtype != FA_BF16 || (d != 64 && d != 128))
    return fail(FA_ERR_UNSUPPORTED, "fa_decode_splitkv_gqa: only bf16 with d = 64 or 128 is built");
  if (H_q / H_kv > 128)  // the group's rows share one 128-row MMA tile
    return fail(FA_ERR_UNSUPPORTED, "fa_decode_splitkv_gqa: at most 128 query heads per key/value head (got %d)",
                H_q / H_kv);
  if (n_splits > 256) return fail(FA_ERR_UNSUPPORTED, "fa_decode_splitkv_gqa: n_splits must be <= 256");
  if (B > 65535 || H_q > 65535) return fail(FA_ERR_UNSUPPORTED, "fa_decode_splitkv_gqa: B and H must be <= 65535");
  if (bad_scale(scale)) return fail(FA_ERR_INVALID_ARG, "fa_decode_splitkv_gqa: scale must be finite and > 0");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(workspace))
    return fail(FA_ERR_INVALID_ARG, "fa_decode_splitkv_gqa: pointers must be 16-byte aligned");
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u))
    return fail(FA_ERR_INVALID_ARG, "fa_decode_splitkv_gqa: lse must be 4-byte aligned");
  const size_t need = fa_decode_workspace_size(B, H_q, d, n_splits);
  if (workspace_bytes < need)
    return fail(FA_ERR_INVALID_ARG, "fa_decode_splitkv_gqa: workspace %zu bytes, need %zu", workspace_bytes, need);
  fa::DecodeParams p;
  p.q = q;
  p.k = k;
  p.v = v;
  p.o = o;
  p.lse = lse;
  const size_t slots = static_cast<size_t>(B) * H_q * n_splits;
  p.part_o = static_cast<float*>(workspace);
  p.part_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) + round256(slots * d * 4));
  p.B = B;
  p.H = H_q;
  p.Hkv = H_kv;
  p.G = H_q / H_kv;
  p.Nkv = N_kv;
  p.n_splits = n_splits;
  p.d = d;
  p.chunk = (N_kv + n_splits - 1) / n_splits;
  p.scale_log2 = scale * 1.4426950408889634f;
  fa_status r = watchdog_ptr(&p.err);
  if (r != FA_OK) return r;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p.G == 1) {
    cudaError_t e = fa::launch_decode_bf16(d, p, s);
    if (e != cudaSuccess) return cuda_fail(e, "fa_decode_splitkv_gqa launch");
    return check_launch("fa_decode_splitkv_gqa", 2);
  }
  // Groups of two or more query heads: tensor-core split kernel, then the merge.
  fa::DecodeTcParams t;
  memset(&t, 0, sizeof(t));
  const int64_t qspan = static_cast<int64_t>(B) * H_q * d;  // q as one [B·H_q, d] matrix
  if ((r = make_map(&t.tm_q, q, 1, 1, B * H_q, d, qspan, qspan, d, "q")) != FA_OK) return r;
  const int64_t nd = static_cast<int64_t>(N_kv) * d;
  if ((r = make_map(&t.tm_k, k, B, H_kv, N_kv, d, H_kv * nd, nd, d, "k")) != FA_OK) return r;
  if ((r = make_map(&t.tm_v, v, B, H_kv, N_kv, d, H_kv * nd, nd, d, "v")) != FA_OK) return r;
  t.part_o = p.part_o;
  t.part_ml = p.part_ml;
  t.B = B;
  t.Hq = H_q;
  t.Hkv = H_kv;
  t.G = p.G;
  t.Nkv = N_kv;
  t.n_splits = n_splits;
  t.d = d;
  t.chunk = p.chunk;
  t.scale_log2 = p.scale_log2;
  t.err = p.err;
  cudaError_t e = fa::launch_decode_gqa_tc(t, s);
  if (e != cudaSuccess) return cuda_fail(e, "fa_decode_splitkv_gqa launch");
  e = fa::launch_decode_merge(p, s);
  if (e != cudaSuccess) return cuda_fail(e, "fa_decode_splitkv_gqa merge launch");
  return check_launch("fa_decode_splitkv_gqa", 2);
}

fa_status fa_decode_paged(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                          const int32_t* seq_lens, void* o, float* lse, int B, int H_q, int H_kv, int num_blocks,
                          int block_size, int max_blocks, int d, fa_dtype dtype, float scale, int n_splits,
                          void* workspace, size_t workspace_bytes, void* stream) {
  if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !o || !workspace)
    return fail(FA_ERR_INVALID_ARG, "fa_decode_paged: null pointer");
  if (B <= 0 || H_q <= 0 || H_kv <= 0 || num_blocks <= 0 || block_size <= 0 || max_blocks <= 0 || d <= 0 ||
      n_splits <= 0)
    return fail(FA_ERR_INVALID_ARG, "fa_decode_paged: sizes must be positive");
  if (H_q % H_kv != 0)
    return fail(FA_ERR_INVALID_ARG, "fa_decode_paged: H_q (%d) must be a multiple of H_kv (%d)", H_q, H_kv);
  if (dtype != FA_BF16 && dtype != FA_FP32) return fail(FA_ERR_INVALID_ARG, "fa_decode_paged: unknown dtype");
  if (dtype != FA_BF16 || (d != 64 && d != 128))
    return fail(FA_ERR_UNSUPPORTED, "fa_decode_paged: only bf16 with d = 64 or 128 is built");
  if (block_size != 16 && block_size != 32 && block_size != 64 && block_size != 128)
    return fail(FA_ERR_UNSUPPORTED, "fa_decode_paged: block_size must be 16, 32, 64 or 128 (got %d)", block_size);
  if (H_q / H_kv > 128)
    return fail(FA_ERR_UNSUPPORTED, "fa_decode_paged: at most 128 query heads per key/value head");
  if (n_splits > 256) return fail(FA_ERR_UNSUPPORTED, "fa_decode_paged: n_splits must be <= 256");
  if (B > 65535 || H_q > 65535) return fail(FA_ERR_UNSUPPORTED, "fa_decode_paged: B and H must be <= 65535");
  if (static_cast<int64_t>(max_blocks) * block_size > (1 << 30))
    return fail(FA_ERR_UNSUPPORTED, "fa_decode_paged: max_blocks * block_size too large");
  // The grouped kernel addresses a page of one head as page·H_kv + head in a 32-bit TMA coordinate.
  if (static_cast<int64_t>(num_blocks) * H_kv > INT32_MAX)
    return fail(FA_ERR_UNSUPPORTED, "fa_decode_paged: num_blocks * H_kv too large");
  if (bad_scale(scale)) return fail(FA_ERR_INVALID_ARG, "fa_decode_paged: scale must be finite and > 0");
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return fail(FA_ERR_INVALID_ARG, "fa_decode_paged: tensors must be 16-byte aligned (tables 4-byte)");
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u))
    return fail(FA_ERR_INVALID_ARG, "fa_decode_paged: lse must be 4-byte aligned");
  const size_t need = fa_decode_workspace_size(B, H_q, d, n_splits);
  if (workspace_bytes < need)
    return fail(FA_ERR_INVALID_ARG, "fa_decode_paged: workspace %zu bytes, need %zu", workspace_bytes, need);
  fa::DecodeParams p;
  p.q = q;
  p.k = k_cache;
  p.v = v_cache;
  p.o = o;
  p.lse = lse;
  const size_t slots = static_cast<size_t>(B) * H_q * n_splits;
  p.part_o = static_cast<float*>(workspace);
  p.part_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) + round256(slots * d * 4));
  p.B = B;
  p.H = H_q;
  p.Nkv = 0;
  p.n_splits = n_splits;
  p.d = d;
  p.chunk = 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.Hkv = H_kv;
  p.G = H_q / H_kv;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.max_blocks = max_blocks;
  p.block_size = block_size;
  p.num_blocks = num_blocks;
  fa_status r = watchdog_ptr(&p.err);
  if (r != FA_OK) return r;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p.G == 1) {
    cudaError_t e = fa::launch_decode_paged_bf16(p, s);
    if (e != cudaSuccess) return cuda_fail(e, "fa_decode_paged launch");
    return check_launch("fa_decode_paged", 2);
  }
  fa::DecodeTcParams t;
  memset(&t, 0, sizeof(t));
  const int64_t qspan = static_cast<int64_t>(B) * H_q * d;
  if ((r = make_map(&t.tm_q, q, 1, 1, B * H_q, d, qspan, qspan, d, "q")) != FA_OK) return r;
  if (d == 128) {  // one box per page of one head, both 64-column halves
    if ((r = make_page_map5(&t.tm_k, k_cache, num_blocks, H_kv, block_size, "k_cache")) != FA_OK) return r;
    if ((r = make_page_map5(&t.tm_v, v_cache, num_blocks, H_kv, block_size, "v_cache")) != FA_OK) return r;
  } else {  // d = 64: pages as a 4-D tensor {d, block_size, H_kv, num_blocks}
    const int64_t page = static_cast<int64_t>(block_size) * d;
    if ((r = make_map(&t.tm_k, k_cache, num_blocks, H_kv, block_size, d, H_kv * page, page, d, "k_cache",
                      block_size)) != FA_OK)
      return r;
    if ((r = make_map(&t.tm_v, v_cache, num_blocks, H_kv, block_size, d, H_kv * page, page, d, "v_cache",
                      block_size)) != FA_OK)
      return r;
  }
  t.block_table = block_table;
  t.seq_lens = seq_lens;
  t.max_blocks = max_blocks;
  t.block_size = block_size;
  t.num_blocks = num_blocks;
  t.part_o = p.part_o;
  t.part_ml = p.part_ml;
  t.B = B;
  t.Hq = H_q;
  t.Hkv = H_kv;
  t.G = p.G;
  t.Nkv = 0;
  t.n_splits = n_splits;
  t.d = d;
  t.chunk = 0;
  t.scale_log2 = p.scale_log2;
  t.err = p.err;
  cudaError_t e = fa::launch_decode_gqa_tc_paged(t, s);
  if (e != cudaSuccess) return cuda_fail(e, "fa_decode_paged launch");
  e = fa::launch_decode_merge(p, s);
  if (e != cudaSuccess) return cuda_fail(e, "fa_decode_paged merge launch");
  return check_launch("fa_decode_paged", 2);
}

size_t fa_backward_workspace_size(int B, int H, int N, int d) {
  if (B <= 0 || H <= 0 || N <= 0 || d <= 0) return 0;
  const size_t rows = static_cast<size_t>(B) * H * N;
  return round256(rows * d * 4) + 2 * round256(rows * 4);
}

}  // extern "C"

namespace {

fa_status backward_impl(const void* q, const void* k, const void* v, const void* o, const float* lse,
                        const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d, fa_dtype dtype,
                        float scale, void* workspace, size_t workspace_bytes, int causal, void* stream) {
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !workspace)
    return fail(FA_ERR_INVALID_ARG, "fa_backward: null pointer");
  if (B <= 0 || H <= 0 || N <= 0 || d <= 0) return fail(FA_ERR_INVALID_ARG, "fa_backward: sizes must be positive");
  if (dtype != FA_BF16 && dtype != FA_FP32) return fail(FA_ERR_INVALID_ARG, "fa_backward: unknown dtype");
  if (dtype != FA_BF16 || (d != 64 && d != 128))
    return fail(FA_ERR_UNSUPPORTED, "fa_backward: only bf16 with d = 64 or 128 is built");
  if (B > 65535 || H > 65535) return fail(FA_ERR_UNSUPPORTED, "fa_backward: B and H must be <= 65535");
  if (causal && (N + 127) / 128 > 65535)  // the causal grid puts the 128-key tiles on its y axis
    return fail(FA_ERR_UNSUPPORTED, "fa_backward: causal backward needs N <= %d", 65535 * 128);
  if (bad_scale(scale)) return fail(FA_ERR_INVALID_ARG, "fa_backward: scale must be finite and > 0");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv) || !aligned16(workspace) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return fail(FA_ERR_INVALID_ARG, "fa_backward: pointers must be 16-byte aligned (lse 4-byte)");
  const size_t need = fa_backward_workspace_size(B, H, N, d);
  if (workspace_bytes < need)
    return fail(FA_ERR_INVALID_ARG, "fa_backward: workspace %zu bytes, need %zu", workspace_bytes, need);
  fa::BwdParams p;
  memset(&p, 0, sizeof(p));
  const int64_t nd = static_cast<int64_t>(N) * d;
  fa_status r;
  if ((r = make_map(&p.tm_q, q, B, H, N, d, H * nd, nd, d, "q")) != FA_OK) return r;
  if ((r = make_map(&p.tm_k, k, B, H, N, d, H * nd, nd, d, "k")) != FA_OK) return r;
  if ((r = make_map(&p.tm_v, v, B, H, N, d, H * nd, nd, d, "v")) != FA_OK) return r;
  if ((r = make_map(&p.tm_do, dout, B, H, N, d, H * nd, nd, d, "dout")) != FA_OK) return r;
  if ((r = make_map(&p.tm_dk, dk, B, H, N, d, H * nd, nd, d, "dk")) != FA_OK) return r;
  if ((r = make_map(&p.tm_dv, dv, B, H, N, d, H * nd, nd, d, "dv")) != FA_OK) return r;
  if ((r = watchdog_ptr(&p.err)) != FA_OK) return r;
  const size_t rows = static_cast<size_t>(B) * H * N;
  char* ws = static_cast<char*>(workspace);
  p.q = q;
  p.o = o;
  p.dout = dout;
  p.lse = lse;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.dq_acc = reinterpret_cast<float*>(ws);
  p.delta = reinterpret_cast<float*>(ws + round256(rows * d * 4));
  p.lse_log2 = reinterpret_cast<float*>(ws + round256(rows * d * 4) + round256(rows * 4));
  p.B = B;
  p.H = H;
  p.N = N;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.causal = causal;
  int launches = 0;
  cudaError_t e = fa::launch_bwd_bf16(d, p, static_cast<cudaStream_t>(stream), &launches);
  if (e != cudaSuccess) return cuda_fail(e, "fa_backward launch");
  return check_launch("fa_backward", launches);
}

}  // namespace

extern "C" {

fa_status fa_backward(const void* q, const void* k, const void* v, const void* o, const float* lse,
                      const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d, fa_dtype dtype,
                      float scale, void* workspace, size_t workspace_bytes, void* stream) {
  return backward_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, dtype, scale, workspace, workspace_bytes, 0,
                       stream);
}

fa_status fa_backward_masked(const void* q, const void* k, const void* v, const void* o, const float* lse,
                             const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                             fa_dtype dtype, float scale, void* workspace, size_t workspace_bytes, fa_mask mask,
                             void* stream) {
  if (mask != FA_MASK_NONE && mask != FA_MASK_CAUSAL)
    return fail(FA_ERR_INVALID_ARG, "fa_backward_masked: unknown mask %d", static_cast<int>(mask));
  return backward_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, dtype, scale, workspace, workspace_bytes,
                       mask == FA_MASK_CAUSAL ? 1 : 0, stream);
}

fa_status fa_watchdog_selftest(void* stream) {
  unsigned int* word = nullptr;
  fa_status r = watchdog_ptr(&word);
  if (r != FA_OK) return r;
  fa::watchdog_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(word);
  return check_launch("fa_watchdog_selftest", 1);
}

fa_status fa_device_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fa_device_status: stream sync");
  unsigned int* word = nullptr;
  fa_status r = watchdog_ptr(&word);
  if (r != FA_OK) return r;
  unsigned int code = 0;
  e = cudaMemcpy(&code, word, sizeof(code), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "fa_device_status: read watchdog");
  if (code != 0) {
    const unsigned int zero = 0;
    cudaMemcpy(word, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    if ((code & 0xFFu) == fa::kSiteBadBlock)
      return fail(FA_ERR_INVALID_ARG, "paged decode: a block-table entry is outside [0, num_blocks) (page 0 was read)");
    if ((code & 0xFFu) == fa::kSiteBadLength)
      return fail(FA_ERR_INVALID_ARG, "paged decode: a sequence length is outside [1, max_blocks * block_size]");
    return fail(FA_ERR_DEVICE_TIMEOUT, "kernel %u gave up waiting at site %u", code >> 8, code & 0xFFu);
  }
  return ok();
}

}  // extern "C"
