// C ABI of the attention library: argument validation, TMA tensor-map
// encoding, launch of the forward and backward kernels, status reporting.
// The declarations and their contracts are in include/attn.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/attn.h"
#include "attn_common.cuh"
#include "attn_sparse.cuh"

namespace attn {
namespace {

// Status word of the forward kernels (one per device that loads the library).
__device__ int g_fwd_status;

constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;
// Rows of the forward's output TMA stores: each epilogue warp stores its own
// 32 rows of a query tile.
constexpr int kFwdStoreRows = 32;
unsigned long long g_timeout_ns = kDefaultTimeoutNs;
int g_inject_stall = 0;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool check_status_env() {
  static int v = -1;
  if (v < 0) {
    const char* e = std::getenv("ATTN_CHECK_STATUS");
    v = (e && e[0] == '1') ? 1 : 0;
  }
  return v == 1;
}

// 0 = unknown, 1 = supported, 2 = not supported.
int g_dev_ok[64];

attn_status_t check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev >= 0 && dev < 64 && g_dev_ok[dev]) return g_dev_ok[dev] == 1 ? ATTN_OK : ATTN_ERR_UNSUPPORTED;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return ATTN_ERR_CUDA;
  // The kernels are built for sm_103a only.
  const bool ok = (major == 10 && minor == 3);
  if (dev >= 0 && dev < 64) g_dev_ok[dev] = ok ? 1 : 2;
  return ok ? ATTN_OK : ATTN_ERR_UNSUPPORTED;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

attn_status_t validate_sizes(int B, int Hq, int Hkv, int S, int D) {
  if (B < 0 || S < 0 || Hq <= 0 || Hkv <= 0) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  // Element offsets stay within what the TMA coordinates and 64-bit indices hold.
  if (static_cast<long long>(S) > (1ll << 24)) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

// Tensor maps already encoded, keyed by every argument of the encoding (the
// base address, element type, sizes, strides, box and swizzle), so a key
// that matches gives the identical map. A map only describes addresses, so it
// stays valid after its memory is freed and reused. Fixed capacity, replaced
// round-robin; guarded by a mutex.
struct MapKey {
  const void* base;
  int dtype, rank, swizzle;
  cuuint64_t dims[4], strides[3];
  cuuint32_t box[4];
};
constexpr int kMapCache = 256;
struct MapCache {
  std::mutex mu;
  uint64_t hash[kMapCache];
  MapKey key[kMapCache];
  CUtensorMap map[kMapCache];
  int n = 0, next = 0;
};
MapCache g_map_cache;

bool encode_cached(CUtensorMap* m, CUtensorMapDataType dtype, int rank, const void* base,
                   const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                   CUtensorMapSwizzle swizzle) {
  MapKey k;
  std::memset(&k, 0, sizeof(k));
  k.base = base;
  k.dtype = static_cast<int>(dtype);
  k.rank = rank;
  k.swizzle = static_cast<int>(swizzle);
  for (int i = 0; i < rank; ++i) {
    k.dims[i] = dims[i];
    k.box[i] = box[i];
    if (i + 1 < rank) k.strides[i] = strides[i];
  }
  uint64_t h = 1469598103934665603ull;  // FNV-1a over the key's bytes
  const unsigned char* kb = reinterpret_cast<const unsigned char*>(&k);
  for (size_t i = 0; i < sizeof(k); ++i) h = (h ^ kb[i]) * 1099511628211ull;
  std::lock_guard<std::mutex> lock(g_map_cache.mu);
  for (int i = 0; i < g_map_cache.n; ++i)
    if (g_map_cache.hash[i] == h && std::memcmp(&g_map_cache.key[i], &k, sizeof(k)) == 0) {
      *m = g_map_cache.map[i];
      return true;
    }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t es[4] = {1, 1, 1, 1};
  if (fn(m, dtype, rank, const_cast<void*>(base), dims, strides, box, es,
         CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  const int slot = g_map_cache.next;
  g_map_cache.hash[slot] = h;
  g_map_cache.key[slot] = k;
  g_map_cache.map[slot] = *m;
  g_map_cache.next = (slot + 1) % kMapCache;
  if (g_map_cache.n < kMapCache) ++g_map_cache.n;
  return true;
}

// 4-D bf16 map over a [B, S, H, D] tensor; a box is `rows` sequence rows of
// one head and 64 columns (128 bytes), stored with 128-byte swizzle.
bool make_bshd_map(CUtensorMap* m, const void* base, int B, int S, int H, int D, int rows) {
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2,
                                 static_cast<cuuint64_t>(H) * D * 2,
                                 static_cast<cuuint64_t>(S) * H * D * 2};
  const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(rows), 1};
  return encode_cached(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box,
                       CU_TENSOR_MAP_SWIZZLE_128B);
}

// 4-D fp32 map over the [B, S, Hq, D] dq output; a box is 32 sequence rows of
// one head, all D columns, unswizzled (the layout the dQ staging tile uses).
bool make_dq_map(CUtensorMap* m, void* base, int B, int S, int H, int D) {
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 4,
                                 static_cast<cuuint64_t>(H) * D * 4,
                                 static_cast<cuuint64_t>(S) * H * D * 4};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(D), 1,
                             static_cast<cuuint32_t>(BwdCfg<128>::DQ_ROWS), 1};
  return encode_cached(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, dims, strides, box,
                       CU_TENSOR_MAP_SWIZZLE_NONE);
}

// 2-D bf16 map over `rows` rows of `cols` columns (row-major, contiguous); a
// box is `box_rows` rows of 64 columns (128 bytes), 128-byte swizzle.
bool make_rows_map(CUtensorMap* m, const void* base, long long rows, int cols, int box_rows) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  return encode_cached(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box,
                       CU_TENSOR_MAP_SWIZZLE_128B);
}

int* fwd_status_ptr() {
  static int* ptrs[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return nullptr;
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fwd_status) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<int*>(p);
  }
  return ptrs[dev];
}

// Reads and clears a status word: the forward's device global (tagless) or a
// backward workspace's tagged word (counted only once a backward call has
// started it). Returns the code it held, or -1 if the read failed.
int read_clear_status(int* status_dev, bool tagged) {
  int w[2] = {0, 0};
  if (cudaMemcpy(w, status_dev, (tagged ? 2 : 1) * sizeof(int), cudaMemcpyDeviceToHost) !=
      cudaSuccess)
    return -1;
  if (tagged && w[1] != kStatusTag) return 0;
  if (w[0] != 0 && cudaMemset(status_dev, 0, sizeof(int)) != cudaSuccess) return -1;
  return w[0];
}

attn_status_t finish(cudaError_t e, cudaStream_t stream, int* status_dev, bool tagged) {
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  if (check_status_env()) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ERR_CUDA;
    const int st = status_dev ? read_clear_status(status_dev, tagged) : 0;
    if (st < 0) return ATTN_ERR_CUDA;
    if (st == ATTN_ERR_BOUNDS) return ATTN_ERR_BOUNDS;
    if (st != 0) return ATTN_ERR_TIMEOUT;
  }
  return ATTN_OK;
}

attn_status_t check_workspace(void* ws, size_t bytes, int B, int Hq, int S, int D) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return ATTN_ERR_WORKSPACE;
  (void)D;
  if (bytes < bwd_workspace_layout(B, Hq, S).total) return ATTN_ERR_WORKSPACE;
  return ATTN_OK;
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" {

const char* attn_status_string(attn_status_t s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration or device";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_TIMEOUT: return "kernel pipeline wait timed out";
    case ATTN_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case ATTN_ERR_BOUNDS: return "index check failed (bounds-checked build)";
  }
  return "unknown status";
}

void attn_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns = ns ? ns : kDefaultTimeoutNs; }

void attn_set_fault_injection(int mask) { g_inject_stall = mask & 3; }

size_t attn_bwd_workspace_size(int B, int Hq, int Hkv, int S, int D) {
  if (validate_sizes(B, Hq, Hkv, S, D) != ATTN_OK || B == 0 || S == 0) return 0;
  return bwd_workspace_layout(B, Hq, S).total;
}

// A sliding window (window > 0) is defined for causal attention only.
static attn_status_t validate_window(int causal, int window) {
  if (window < 0 || (window > 0 && !causal)) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

static attn_status_t fwd_impl(const void* q, const void* k, const void* v, void* o, void* o_lo,
                              float* lse, int B, int Hq, int Hkv, int S, int D, int causal,
                              int window, float scale, void* stream) {
  attn_status_t st = validate_sizes(B, Hq, Hkv, S, D);
  if (st != ATTN_OK) return st;
  if ((st = validate_window(causal, window)) != ATTN_OK) return st;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (B == 0 || S == 0) return ATTN_OK;
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(o_lo))
    return ATTN_ERR_INVALID_ARG;
  if ((st = check_device()) != ATTN_OK) return st;
  CUtensorMap tq, tk, tv, to, tolo;
  if (!make_bshd_map(&tq, q, B, S, Hq, D, FwdCfg<128>::BQ) ||
      !make_bshd_map(&tk, k, B, S, Hkv, D, FwdCfg<128>::BK) ||
      !make_bshd_map(&tv, v, B, S, Hkv, D, FwdCfg<128>::BK) ||
      !make_bshd_map(&to, o, B, S, Hq, D, kFwdStoreRows) ||
      !make_bshd_map(&tolo, o_lo ? o_lo : o, B, S, Hq, D, kFwdStoreRows))
    return ATTN_ERR_CUDA;
  int* status = fwd_status_ptr();
  if (!status) return ATTN_ERR_CUDA;
  FwdParams p;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.o_lo = static_cast<__nv_bfloat16*>(o_lo);
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.S = S;
  p.G = Hq / Hkv;
  p.causal = causal ? 1 : 0;
  p.window = window;
  // The kernel masks a key by giving it an infinite score, which a zero scale
  // would turn into NaN. A scale below 2^-100 in magnitude is taken as
  // +-2^-100: that moves no exponent by one fp32 ulp unless |q.k| > 2^70.
  float sl2 = scale * kLog2e;
  if (std::fabs(sl2) < 0x1p-100f) sl2 = std::signbit(sl2) ? -0x1p-100f : 0x1p-100f;
  p.scale_log2 = sl2;
  p.n_qblocks = (S + 2 * FwdCfg<128>::BQ - 1) / (2 * FwdCfg<128>::BQ);
  p.status = status;
  p.timeout_ns = g_timeout_ns;
  p.inject_stall = g_inject_stall & 1;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return finish(launch_fwd(D, tq, tk, tv, to, tolo, p, s), s, status, false);
}

attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int Hq, int Hkv, int S, int D, int causal, float scale, void* stream) {
  return fwd_impl(q, k, v, o, nullptr, lse, B, Hq, Hkv, S, D, causal, 0, scale, stream);
}

attn_status_t attn_fwd_residual(const void* q, const void* k, const void* v, void* o, void* o_lo,
                                float* lse, int B, int Hq, int Hkv, int S, int D, int causal,
                                float scale, void* stream) {
  if (B > 0 && S > 0 && !o_lo) return ATTN_ERR_INVALID_ARG;
  return fwd_impl(q, k, v, o, o_lo, lse, B, Hq, Hkv, S, D, causal, 0, scale, stream);
}

attn_status_t attn_fwd_ex(const void* q, const void* k, const void* v, void* o, void* o_lo,
                          float* lse, int B, int Hq, int Hkv, int S, int D, int causal, int window,
                          float scale, void* stream) {
  return fwd_impl(q, k, v, o, o_lo, lse, B, Hq, Hkv, S, D, causal, window, scale, stream);
}

attn_status_t attn_bwd_preprocess(const void* o, const void* o_lo, const void* dO,
                                  const float* lse, void* dq, int B, int Hq, int Hkv, int S, int D,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  attn_status_t st = validate_sizes(B, Hq, Hkv, S, D);
  if (st != ATTN_OK) return st;
  if (B == 0 || S == 0) return ATTN_OK;
  if (!o || !dO || !lse || !dq) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(o) || !aligned16(o_lo) || !aligned16(dO) || !aligned16(lse) || !aligned16(dq))
    return ATTN_ERR_INVALID_ARG;
  if ((st = check_workspace(workspace, workspace_bytes, B, Hq, S, D)) != ATTN_OK) return st;
  if ((st = check_device()) != ATTN_OK) return st;
  const BwdWorkspace w = bwd_workspace_layout(B, Hq, S);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_bwd_preprocess(
      static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(o_lo),
      static_cast<const __nv_bfloat16*>(dO), lse, reinterpret_cast<float*>(ws + w.off_nlse2),
      reinterpret_cast<float*>(ws + w.off_dvec), static_cast<float*>(dq),
      reinterpret_cast<int*>(ws + w.off_status), B, Hq, S, D, s);
  return finish(e, s, nullptr, true);
}

// The Dvec pass (attn_bwd_dvec): reads the log2-scaled LSE rows the
// preprocess left in the workspace, writes exact Dvec rows over them.
static attn_status_t dvec_impl(const void* q, const void* k, const void* v, const void* dO,
                               int B, int Hq, int Hkv, int S, int D, int causal, int window,
                               float scale, void* workspace, size_t workspace_bytes,
                               void* stream) {
  attn_status_t st = validate_sizes(B, Hq, Hkv, S, D);
  if (st != ATTN_OK) return st;
  if ((st = validate_window(causal, window)) != ATTN_OK) return st;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (B == 0 || S == 0) return ATTN_OK;
  if (!q || !k || !v || !dO) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO)) return ATTN_ERR_INVALID_ARG;
  if ((st = check_workspace(workspace, workspace_bytes, B, Hq, S, D)) != ATTN_OK) return st;
  if ((st = check_device()) != ATTN_OK) return st;
  const BwdWorkspace w = bwd_workspace_layout(B, Hq, S);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int BQ = DvecCfg<128>::BQ;
  CUtensorMap tq, tk, tv, tdo;
  if (!make_bshd_map(&tq, q, B, S, Hq, D, BQ) || !make_bshd_map(&tdo, dO, B, S, Hq, D, BQ) ||
      !make_bshd_map(&tk, k, B, S, Hkv, D, 128) || !make_bshd_map(&tv, v, B, S, Hkv, D, 128))
    return ATTN_ERR_CUDA;
  DvecParams p;
  p.nlse2 = reinterpret_cast<const float*>(ws + w.off_nlse2);
  p.dvec = reinterpret_cast<float*>(ws + w.off_dvec);
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.S = S;
  p.S_pad = seq_pad(S);
  p.G = Hq / Hkv;
  p.causal = causal ? 1 : 0;
  p.window = window;
  p.scale_log2 = scale * kLog2e;
  p.n_qblocks = (S + 2 * BQ - 1) / (2 * BQ);
  p.status = reinterpret_cast<int*>(ws + w.off_status);
  p.timeout_ns = g_timeout_ns;
  p.inject_stall = (g_inject_stall >> 1) & 1;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return finish(launch_bwd_dvec(D, tq, tk, tv, tdo, p, s), s, p.status, true);
}

attn_status_t attn_bwd_dvec(const void* q, const void* k, const void* v, const void* dO, int B,
                            int Hq, int Hkv, int S, int D, int causal, int window, float scale,
                            void* workspace, size_t workspace_bytes, void* stream) {
  return dvec_impl(q, k, v, dO, B, Hq, Hkv, S, D, causal, window, scale, workspace,
                   workspace_bytes, stream);
}

attn_status_t attn_bwd_main_ex(const void* q, const void* k, const void* v, const void* dO,
                               void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int S, int D,
                               int causal, int window, float scale, void* workspace,
                               size_t workspace_bytes, void* stream) {
  attn_status_t st = validate_sizes(B, Hq, Hkv, S, D);
  if (st != ATTN_OK) return st;
  if ((st = validate_window(causal, window)) != ATTN_OK) return st;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (B == 0 || S == 0) return ATTN_OK;
  if (!q || !k || !v || !dO || !dq || !dk || !dv) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv))
    return ATTN_ERR_INVALID_ARG;
  if ((st = check_workspace(workspace, workspace_bytes, B, Hq, S, D)) != ATTN_OK) return st;
  if ((st = check_device()) != ATTN_OK) return st;
  const BwdWorkspace w = bwd_workspace_layout(B, Hq, S);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int BQ = BwdCfg<128>::BQ;
  CUtensorMap tq, tk, tv, tdo, tdq;
  if (!make_bshd_map(&tq, q, B, S, Hq, D, BQ) || !make_bshd_map(&tdo, dO, B, S, Hq, D, BQ) ||
      !make_bshd_map(&tk, k, B, S, Hkv, D, 128) || !make_bshd_map(&tv, v, B, S, Hkv, D, 128) ||
      !make_dq_map(&tdq, dq, B, S, Hq, D))
    return ATTN_ERR_CUDA;
  BwdParams p;
  p.nlse2 = reinterpret_cast<const float*>(ws + w.off_nlse2);
  p.dvec = reinterpret_cast<const float*>(ws + w.off_dvec);
  p.dk = static_cast<float*>(dk);
  p.dv = static_cast<float*>(dv);
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.S = S;
  p.S_pad = seq_pad(S);
  p.G = Hq / Hkv;
  p.causal = causal ? 1 : 0;
  p.window = window;
  p.scale_log2 = scale * kLog2e;
  p.scale = scale;
  p.n_ktiles = (S + 127) / 128;
  p.split = 1;  // chosen by the launcher
  p.status = reinterpret_cast<int*>(ws + w.off_status);
  p.timeout_ns = g_timeout_ns;
  p.inject_stall = (g_inject_stall >> 1) & 1;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return finish(launch_bwd_main(D, tq, tk, tv, tdo, tdq, p, s), s, p.status, true);
}

attn_status_t attn_bwd_main(const void* q, const void* k, const void* v, const void* dO, void* dq,
                            void* dk, void* dv, int B, int Hq, int Hkv, int S, int D, int causal,
                            float scale, void* workspace, size_t workspace_bytes, void* stream) {
  return attn_bwd_main_ex(q, k, v, dO, dq, dk, dv, B, Hq, Hkv, S, D, causal, 0, scale, workspace,
                          workspace_bytes, stream);
}

attn_status_t attn_bwd_ex(const void* q, const void* k, const void* v, const void* o,
                          const void* dO, const float* lse, void* dq, void* dk, void* dv,
                          const void* o_lo, int B, int Hq, int Hkv, int S, int D, int causal,
                          int window, float scale, void* workspace, size_t workspace_bytes,
                          void* stream) {
  // Validate everything up front so a failure launches nothing.
  attn_status_t st = validate_sizes(B, Hq, Hkv, S, D);
  if (st != ATTN_OK) return st;
  if ((st = validate_window(causal, window)) != ATTN_OK) return st;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (B == 0 || S == 0) return ATTN_OK;
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) ||
      !aligned16(lse) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(o_lo))
    return ATTN_ERR_INVALID_ARG;
  if ((st = check_workspace(workspace, workspace_bytes, B, Hq, S, D)) != ATTN_OK) return st;
  if ((st = check_device()) != ATTN_OK) return st;
  if (o_lo) {
    // Dvec = rowsum(dO * (o + o_lo)) in the preprocess.
    st = attn_bwd_preprocess(o, o_lo, dO, lse, dq, B, Hq, Hkv, S, D, workspace, workspace_bytes,
                             stream);
  } else {
    // Without the residual, bf16 o gives Dvec to about 8 bits only: the
    // preprocess writes the LSE rows and zeroes dq, and the Dvec pass
    // computes Dvec = rowsum(P * dP) from its definition.
    const BwdWorkspace w = bwd_workspace_layout(B, Hq, S);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    st = finish(launch_bwd_preprocess(nullptr, nullptr, static_cast<const __nv_bfloat16*>(dO), lse,
                                      reinterpret_cast<float*>(ws + w.off_nlse2),
                                      reinterpret_cast<float*>(ws + w.off_dvec),
                                      static_cast<float*>(dq),
                                      reinterpret_cast<int*>(ws + w.off_status), B, Hq, S, D, s),
                s, nullptr, true);
    if (st == ATTN_OK)
      st = dvec_impl(q, k, v, dO, B, Hq, Hkv, S, D, causal, window, scale, workspace,
                     workspace_bytes, stream);
  }
  if (st != ATTN_OK) return st;
  return attn_bwd_main_ex(q, k, v, dO, dq, dk, dv, B, Hq, Hkv, S, D, causal, window, scale,
                          workspace, workspace_bytes, stream);
}

attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
                       const float* lse, void* dq, void* dk, void* dv, const void* o_lo, int B,
                       int Hq, int Hkv, int S, int D, int causal, float scale, void* workspace,
                       size_t workspace_bytes, void* stream) {
  return attn_bwd_ex(q, k, v, o, dO, lse, dq, dk, dv, o_lo, B, Hq, Hkv, S, D, causal, 0, scale,
                     workspace, workspace_bytes, stream);
}

attn_status_t attn_sparse_fwd(const void* q, const void* kp, const void* vp, const int* idx,
                              void* o, void* o_lo, float* lse, int B, int T, int H, int P, int K,
                              int DK, int DV, float scale, void* stream) {
  if (B < 0 || T < 0 || H <= 0 || H > 128 || P <= 0 || K <= 0 || (K % 4) != 0)
    return ATTN_ERR_INVALID_ARG;
  if ((DK != 64 && DK != 128) || (DV != 64 && DV != 128)) return ATTN_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  // Row counts of the 2-D views stay within what the TMA coordinates hold.
  if (static_cast<long long>(B) * T * H >= (1ll << 31) || static_cast<long long>(B) * P >= (1ll << 31))
    return ATTN_ERR_UNSUPPORTED;
  if (B == 0 || T == 0) return ATTN_OK;
  if (!q || !kp || !vp || !idx || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kp) || !aligned16(vp) || !aligned16(idx) || !aligned16(o) ||
      !aligned16(o_lo) || !aligned16(lse))
    return ATTN_ERR_INVALID_ARG;
  attn_status_t st = check_device();
  if (st != ATTN_OK) return st;
  const long long qrows = static_cast<long long>(B) * T * H, prows = static_cast<long long>(B) * P;
  CUtensorMap tq, tk, to, tolo;
  if (!make_rows_map(&tq, q, qrows, DK, 128) || !make_rows_map(&tk, kp, prows, DK, 1) ||
      !make_rows_map(&to, o, qrows, DV, H) || !make_rows_map(&tolo, o_lo ? o_lo : o, qrows, DV, H))
    return ATTN_ERR_CUDA;
  int* status = fwd_status_ptr();
  if (!status) return ATTN_ERR_CUDA;
  SparseFwdParams p;
  p.kp = static_cast<const __nv_bfloat16*>(kp);
  p.vp = static_cast<const __nv_bfloat16*>(vp);
  p.idx = idx;
  p.lse = lse;
  p.B = B;
  p.T = T;
  p.H = H;
  p.P = P;
  p.K = K;
  p.n_chunks = (K + 127) / 128;
  // As in the dense forward: empty slots get an infinite score, which a zero
  // scale would turn into NaN, so a scale below 2^-100 is taken as +-2^-100.
  float sl2 = scale * kLog2e;
  if (std::fabs(sl2) < 0x1p-100f) sl2 = std::signbit(sl2) ? -0x1p-100f : 0x1p-100f;
  p.scale_log2 = sl2;
  p.status = status;
  p.timeout_ns = g_timeout_ns;
  p.inject_stall = g_inject_stall & 1;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return finish(launch_sparse_fwd(DK, DV, tq, tk, to, tolo, o_lo != nullptr, p, s), s, status,
                false);
}

size_t attn_sparse_bwd_workspace_size(int B, int T, int H) {
  if (B <= 0 || T <= 0 || H <= 0 || H > 128) return 0;
  return sparse_bwd_workspace_bytes(static_cast<long long>(B) * T * H);
}

attn_status_t attn_sparse_bwd(const void* q, const void* kp, const void* vp, const int* idx,
                              const void* o, const void* o_lo, const void* dO, const float* lse,
                              float* dq, float* dkp, float* dvp, int B, int T, int H, int P, int K,
                              int DK, int DV, float scale, void* workspace, size_t workspace_bytes,
                              void* stream) {
  if (B < 0 || T < 0 || H <= 0 || H > 128 || P <= 0 || K <= 0 || (K % 4) != 0)
    return ATTN_ERR_INVALID_ARG;
  if ((DK != 64 && DK != 128) || (DV != 64 && DV != 128)) return ATTN_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * T * H >= (1ll << 31) || static_cast<long long>(B) * P >= (1ll << 31))
    return ATTN_ERR_UNSUPPORTED;
  if (B == 0 || T == 0) return ATTN_OK;
  if (!q || !kp || !vp || !idx || !o || !dO || !lse || !dq || !dkp || !dvp) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kp) || !aligned16(vp) || !aligned16(idx) || !aligned16(o) ||
      !aligned16(o_lo) || !aligned16(dO) || !aligned16(lse) || !aligned16(dq) || !aligned16(dkp) ||
      !aligned16(dvp))
    return ATTN_ERR_INVALID_ARG;
  const long long rows = static_cast<long long>(B) * T * H;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < sparse_bwd_workspace_bytes(rows))
    return ATTN_ERR_WORKSPACE;
  attn_status_t st = check_device();
  if (st != ATTN_OK) return st;
  CUtensorMap tq, tdo, tk;
  if (!make_rows_map(&tq, q, rows, DK, 128) || !make_rows_map(&tdo, dO, rows, DV, 128) ||
      !make_rows_map(&tk, kp, static_cast<long long>(B) * P, DK, 1))
    return ATTN_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t vec_bytes = (static_cast<size_t>(rows) * 4 + 255) / 256 * 256;
  float* nlse2 = reinterpret_cast<float*>(ws + 256);
  float* dvec = reinterpret_cast<float*>(ws + 256 + vec_bytes);
  SparseBwdParams p;
  p.kp = static_cast<const __nv_bfloat16*>(kp);
  p.vp = static_cast<const __nv_bfloat16*>(vp);
  p.idx = idx;
  p.nlse2 = nlse2;
  p.dvec = dvec;
  p.dq = dq;
  p.dkp = dkp;
  p.dvp = dvp;
  p.B = B;
  p.T = T;
  p.H = H;
  p.P = P;
  p.K = K;
  p.n_chunks = (K + 127) / 128;
  float sl2 = scale * kLog2e;
  if (std::fabs(sl2) < 0x1p-100f) sl2 = std::signbit(sl2) ? -0x1p-100f : 0x1p-100f;
  p.scale_log2 = sl2;
  p.scale = scale;
  p.status = static_cast<int*>(workspace);
  p.timeout_ns = g_timeout_ns;
  p.inject_stall = (g_inject_stall >> 1) & 1;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return finish(launch_sparse_bwd(DK, DV, static_cast<const __nv_bfloat16*>(o),
                                  static_cast<const __nv_bfloat16*>(o_lo),
                                  static_cast<const __nv_bfloat16*>(dO), lse, nlse2, dvec, tq, tdo, tk,
                                  p, s),
                s, p.status, true);
}

attn_status_t attn_check_status(void* workspace) {
  if (cudaDeviceSynchronize() != cudaSuccess) return ATTN_ERR_CUDA;
  int* fs = fwd_status_ptr();
  if (!fs) return ATTN_ERR_CUDA;
  const int a = read_clear_status(fs, false);
  // Without a workspace: the no-allocation backward's word as well, once a
  // call on this device has looked up its scratch array.
  int* ws_word = workspace ? static_cast<int*>(workspace) : noalloc_status_word();
  const int b = ws_word ? read_clear_status(ws_word, true) : 0;
  if (a < 0 || b < 0) return ATTN_ERR_CUDA;
  if (a == ATTN_ERR_BOUNDS || b == ATTN_ERR_BOUNDS) return ATTN_ERR_BOUNDS;
  return (a != 0 || b != 0) ? ATTN_ERR_TIMEOUT : ATTN_OK;
}

}  // extern "C"
