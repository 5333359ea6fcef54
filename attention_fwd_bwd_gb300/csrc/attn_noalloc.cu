// attn_bwd_noalloc: the backward pass for callers that cannot allocate device
// memory. Its scratch space is a fixed array compiled into the library instead
// of a caller-provided workspace; see the declaration in include/attn.h.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/attn.h"
#include "attn_common.cuh"

namespace attn {
namespace {

// Scratch of the backward pass (status word, log2-scaled LSE rows, Dvec rows)
// for every attn_bwd_noalloc call on a device. It lives as long as the library
// is loaded, on every device that loads it.
constexpr size_t kNoAllocScratchBytes = 16u << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch per device. Host code cannot use the
// array's name as a device pointer: on the host it names a stand-in object.
void* g_scratch_ptr[64];
std::mutex g_scratch_mu;

attn_status_t scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return ATTN_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return ATTN_OK;
}

}  // namespace

int* noalloc_status_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  return static_cast<int*>(g_scratch_ptr[dev]);
}

}  // namespace attn

extern "C" attn_status_t attn_bwd_noalloc(const void* q, const void* k, const void* v,
                                          const void* o, const void* dO, const float* lse,
                                          void* dq, void* dk, void* dv, const void* o_lo, int B,
                                          int Hq, int Hkv, int S, int D, int causal, float scale,
                                          void* stream) {
  if (B == 0 || S == 0)  // empty problem: same no-op (and checks) as attn_bwd
    return attn_bwd(q, k, v, o, dO, lse, dq, dk, dv, o_lo, B, Hq, Hkv, S, D, causal, scale,
                    nullptr, 0, stream);
  const size_t need = attn_bwd_workspace_size(B, Hq, Hkv, S, D);
  if (need == 0)  // invalid or unsupported sizes: let attn_bwd report which
    return attn_bwd(q, k, v, o, dO, lse, dq, dk, dv, o_lo, B, Hq, Hkv, S, D, causal, scale,
                    nullptr, 0, stream);
  if (need > attn::kNoAllocScratchBytes) return ATTN_ERR_WORKSPACE;
  void* scratch = nullptr;
  const attn_status_t st = attn::scratch_for_current_device(&scratch);
  if (st != ATTN_OK) return st;
  // The preprocess kernel rewrites every word of the scratch this call reads
  // (LSE and Dvec rows including padding), so nothing left from an earlier
  // call leaks in; the status word keeps a timeout that an earlier call
  // recorded until attn_check_status(NULL) reads it.
  return attn_bwd(q, k, v, o, dO, lse, dq, dk, dv, o_lo, B, Hq, Hkv, S, D, causal, scale, scratch,
                  attn::kNoAllocScratchBytes, stream);
}
