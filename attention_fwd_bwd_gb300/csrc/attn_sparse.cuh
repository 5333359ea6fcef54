// Shared definitions of the sparse top-k gather attention kernels (device
// code and the host side of the C ABI).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace attn {

// Forward: one work item per (batch, token). The token's H <= 128 query heads
// form the 128-row tile (rows past H belong to the next token, or are zero
// past the end, and are never stored); its K slots stream through in chunks
// of 128 gathered pool rows.
template <int DK, int DV>
struct SparseFwdCfg {
  static constexpr int BQ = 128;  // head rows of the tile
  static constexpr int BK = 128;  // slots per chunk
  static constexpr int KCH = DK / 64;
  static constexpr int VCH = DV / 64;
  static constexpr int Q_BYTES = BQ * DK * 2;
  static constexpr int K_BYTES = BK * DK * 2;
  static constexpr int V_BYTES = BK * DV * 2;
  static constexpr int SLOT_BYTES = K_BYTES > V_BYTES ? K_BYTES : V_BYTES;
  static constexpr int STG_BYTES = BQ * 64 * 2;  // one 64-column bf16 output tile
  static constexpr int MERGE_BYTES = 2 * BQ * 4;  // second warpgroup's (m, l) per row
  static constexpr int IDX_BYTES = BK * 4;         // the chunk's pool rows, for the producer
  static constexpr int FIXED = Q_BYTES + 2 * STG_BYTES + MERGE_BYTES + IDX_BYTES + 1024;
  static constexpr int NSLOT_FIT = (232448 - FIXED) / SLOT_BYTES;
  static constexpr int NSLOT = NSLOT_FIT > 8 ? 8 : NSLOT_FIT;  // ring slots (K or V chunks)
  static constexpr int SMEM_Q = 0;
  static constexpr int SMEM_RING = Q_BYTES;
  static constexpr int SMEM_STG = SMEM_RING + NSLOT * SLOT_BYTES;
  static constexpr int SMEM_MERGE = SMEM_STG + 2 * STG_BYTES;
  static constexpr int SMEM_IDX = SMEM_MERGE + MERGE_BYTES;
  static constexpr int SMEM_BYTES = SMEM_IDX + IDX_BYTES;
  // Ring positions whose copies may still be in flight while the producer
  // issues the next one. Releasing position x needs positions up to x + 1
  // (the MMA warp issues S(c+1) before P.V(c)), so it stays below NSLOT - 1.
  static constexpr int COPY_DEPTH = 2;
  static constexpr int SMEM_ALLOC = SMEM_BYTES + 1024;
  // Tensor memory per softmax warpgroup w: scores S_w (128 columns, later P_w
  // as bf16 hi/lo pairs) and the output accumulator O_w (DV columns).
  __host__ __device__ static constexpr int tm_s(int w) { return 256 * w; }
  __host__ __device__ static constexpr int tm_o(int w) { return 256 * w + 128; }
  static constexpr int TMEM_COLS = 512;
  static constexpr int THREADS = 320;
  static_assert(NSLOT >= 4, "the ring needs at least two chunks of K and V");
  static_assert(COPY_DEPTH < NSLOT - 1, "copies in flight would block the ring");
  static_assert(SMEM_ALLOC <= 232448, "shared-memory plan exceeds 227 KB");
};

struct SparseFwdParams {
  const __nv_bfloat16* kp;  // [B, P, DK]
  const __nv_bfloat16* vp;  // [B, P, DV]
  const int* idx;  // [B, T, K] pool rows; entries outside [0, P) are empty slots
  float* lse;      // [B, H, T]
  int B, T, H, P, K;
  int n_chunks;      // ceil(K / 128)
  float scale_log2;  // scale * log2(e)
  int* status;
  unsigned long long timeout_ns;
  int inject_stall;  // testing hook: the MMA warp issues nothing (waits then run out)
};

// tq: [B*T*H, DK] rows, box 128 x 64; to / tolo: [B*T*H, DV] rows, box H x 64.
cudaError_t launch_sparse_fwd(int DK, int DV, const CUtensorMap& tq, const CUtensorMap& to,
                              const CUtensorMap& tolo, bool write_lo, const SparseFwdParams& p,
                              cudaStream_t stream);

}  // namespace attn
