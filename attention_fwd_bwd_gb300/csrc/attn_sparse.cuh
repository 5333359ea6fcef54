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
  static constexpr int SMEM_ALLOC = SMEM_BYTES + 1024;
  // Tensor memory per softmax warpgroup w: scores S_w (128 columns, later P_w
  // as bf16 hi/lo pairs) and the output accumulator O_w (DV columns).
  __host__ __device__ static constexpr int tm_s(int w) { return 256 * w; }
  __host__ __device__ static constexpr int tm_o(int w) { return 256 * w + 128; }
  static constexpr int TMEM_COLS = 512;
  // K and V come from two producers, so they use separate slots: slots
  // 0..KSLOTS-1 hold K chunks in turn, the rest V chunks in turn, and each
  // producer's closing wait for its last copies finds those slots' last
  // phases its own.
  static constexpr int KSLOTS = 2;
  static constexpr int VSLOTS = NSLOT - KSLOTS;
  // V chunks whose copies stay in flight while the V producer issues the
  // next one. Its next chunk waits for the release of the chunk VSLOTS back,
  // which must not be one of them.
  static constexpr int V_IN_FLIGHT = 1;
  static constexpr int THREADS = 352;  // 8 softmax warps, K producer, MMA issuer, V producer
  static_assert(NSLOT >= 4, "the ring needs at least two chunks of K and V");
  static_assert(V_IN_FLIGHT < VSLOTS, "copies in flight would block the V slots");
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

// tq: [B*T*H, DK] rows, box 128 x 64; tk: [B*P, DK] rows, box 1 x 64 (gathered
// four rows at a time); to / tolo: [B*T*H, DV] rows, box H x 64.
cudaError_t launch_sparse_fwd(int DK, int DV, const CUtensorMap& tq, const CUtensorMap& tk,
                              const CUtensorMap& to, const CUtensorMap& tolo, bool write_lo,
                              const SparseFwdParams& p, cudaStream_t stream);

}  // namespace attn

namespace attn {

// Backward: one work item per (batch, token), as in the forward. The token's
// Q (H x DK) and dO (H x DV) rows stay in shared memory; the gathered K and V
// rows of each 128-slot chunk stream through the ring. Products are taken
// slot-major (TMEM lane = slot): S^T = K_c Q^T, dP^T = V_c dO^T, then
// dV_c = P^T dO and dK_c = dS^T Q (A from TMEM), scatter-added into the pool
// gradients, and dQ^T += K_c^T dS^T (dS^T from shared memory), which stays in
// TMEM over the token's chunks.
template <int DK, int DV>
struct SparseBwdCfg {
  static constexpr int BQ = 128;  // head rows
  static constexpr int BK = 128;  // slots per chunk
  static constexpr int KCH = DK / 64;
  static constexpr int VCH = DV / 64;
  static constexpr int Q_BYTES = BQ * DK * 2;
  static constexpr int DO_BYTES = BQ * DV * 2;
  static constexpr int K_BYTES = BK * DK * 2;
  static constexpr int V_BYTES = BK * DV * 2;
  // A K slot is read as a 128-row (two 64-column block) MN-major operand by
  // the dQ^T product even when DK = 64 (rows past DK are ignored), so a slot
  // is never smaller than two blocks.
  static constexpr int SLOT_BYTES = 2 * BK * 128;
  static constexpr int DS_BYTES = BK * BQ * 2;     // one bf16 dS^T tile (hi or lo)
  static constexpr int ROWS_BYTES = 2 * BQ * 4;    // -LSE*log2(e) and Dvec per head
  static constexpr int IDX_BYTES = BK * 4;
  static constexpr int SMEM_Q = 0;
  static constexpr int SMEM_DO = SMEM_Q + Q_BYTES;
  static constexpr int SMEM_DS = SMEM_DO + DO_BYTES;  // hi tile, then lo tile
  static constexpr int SMEM_RING = SMEM_DS + 2 * DS_BYTES;
  static constexpr int FIXED = SMEM_RING + ROWS_BYTES + IDX_BYTES + 1024;
  static constexpr int NSLOT_FIT = (232448 - FIXED) / SLOT_BYTES;
  static constexpr int NSLOT = NSLOT_FIT > 8 ? 8 : NSLOT_FIT;
  static constexpr int SMEM_ROWS = SMEM_RING + NSLOT * SLOT_BYTES;
  static constexpr int SMEM_IDX = SMEM_ROWS + ROWS_BYTES;
  static constexpr int SMEM_BYTES = SMEM_IDX + IDX_BYTES;
  static constexpr int SMEM_ALLOC = SMEM_BYTES + 1024;
  // Slot NSLOT - 1 holds V chunks (one slot: V_c is free again after dP^T(c),
  // early in chunk c), the others K chunks in turn (K_c is read until dQ^T(c),
  // at the end of chunk c). So V_{c+1} and K_{c+1} both load while chunk c is
  // processed. K comes from one producer warp, V from another; each slot set
  // has a single producer, so its barriers see their phases in order. The V
  // producer reports each chunk as soon as it has landed: with one V slot, its
  // next load waits for the release of the chunk it has just issued.
  static constexpr int KSLOTS = NSLOT - 1;
  static constexpr int VSLOT = NSLOT - 1;
  // TMEM columns: S^T (then P^T, then dK_c), dP^T (then dS^T), dV_c, dQ^T.
  static constexpr int TM_S = 0, TM_DP = 128, TM_DV = 256, TM_DQ = 384;
  static constexpr int TMEM_COLS = 512;
  // Warps 0-7 compute (warps w and w + 4 share TMEM lanes and split the
  // heads, then the gradient columns), then the K producer, the MMA issuer
  // and the V producer.
  static constexpr int W_KPROD = 8, W_MMA = 9, W_VPROD = 10;
  static constexpr int THREADS = 352;
  static_assert(NSLOT >= 3, "the ring needs K and V of one chunk plus one");
  static_assert(SMEM_ALLOC <= 232448, "shared-memory plan exceeds 227 KB");
};

struct SparseBwdParams {
  const __nv_bfloat16* kp;  // [B, P, DK]
  const __nv_bfloat16* vp;  // [B, P, DV]
  const int* idx;           // [B, T, K]
  const float* nlse2;       // [B, T, H] -LSE * log2(e) (-inf for a token without filled slots)
  const float* dvec;        // [B, T, H] rowsum(dO * O)
  float* dq;                // [B, T, H, DK]
  float* dkp;               // [B, P, DK] (zeroed by the preprocess)
  float* dvp;               // [B, P, DV] (zeroed by the preprocess)
  int B, T, H, P, K;
  int n_chunks;
  float scale_log2, scale;
  int* status;
  unsigned long long timeout_ns;
  int inject_stall;
};

// Workspace of the sparse backward: status word, then nlse2 and dvec rows.
inline size_t sparse_bwd_workspace_bytes(long long rows) {
  return 256 + 2 * ((static_cast<size_t>(rows) * 4 + 255) / 256 * 256);
}

cudaError_t launch_sparse_bwd(int DK, int DV, const __nv_bfloat16* o, const __nv_bfloat16* o_lo,
                              const __nv_bfloat16* dO, const float* lse, float* nlse2, float* dvec,
                              const CUtensorMap& tq, const CUtensorMap& tdo, const CUtensorMap& tk,
                              const SparseBwdParams& p, cudaStream_t stream);

}  // namespace attn
