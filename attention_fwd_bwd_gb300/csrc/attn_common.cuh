// Shared definitions of the attention kernels: tile shapes, shared-memory and
// tensor-memory plans, kernel parameter blocks, and the host-side launchers
// the C ABI calls.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace attn {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Rows of a tile in the sequence dimension are padded up to this multiple in
// the backward workspace arrays (Dvec, log2-scaled LSE, dQ accumulator).
constexpr int kSeqPad = 128;
__host__ __device__ constexpr int seq_pad(int S) { return (S + kSeqPad - 1) / kSeqPad * kSeqPad; }

// ---------------------------------------------------------------- forward
// One CTA per (batch, query head, block of two 128-row query tiles); K/V tiles
// of 128 keys stream through a ring of shared-memory slots (K_j and V_j take
// one slot each) and serve both query tiles. Warps 0-3 / 4-7: softmax, rescale
// and epilogue of query tile A / B (one query row per thread, the row's TMEM
// lane); warp 8: TMA producer; warp 9: MMA issuer.
template <int D>
struct FwdCfg {
  static constexpr int BQ = 128;                     // rows per query tile (two per CTA)
  static constexpr int BK = 128;
  static constexpr int KCH = D / 64;                 // 64-wide (128-byte) column chunks
  static constexpr int Q_BYTES = BQ * D * 2;         // one query tile
  static constexpr int KV_BYTES = BK * D * 2;        // one K or V tile
  static constexpr int NSLOT = (D == 128) ? 4 : 8;   // ring slots
  static constexpr int SMEM_Q = 0;
  static constexpr int SMEM_RING = 2 * Q_BYTES;
  // Output staging, one 128-row x 64-column bf16 tile (128-byte swizzle) per
  // query tile: the epilogue writes O (and o_lo) through it with TMA stores.
  static constexpr int STG_BYTES = BQ * 64 * 2;
  static constexpr int SMEM_STG = SMEM_RING + NSLOT * KV_BYTES;
  static constexpr int SMEM_BYTES = SMEM_STG + 2 * STG_BYTES;
  static constexpr int SMEM_ALLOC = SMEM_BYTES + 1024;  // slack for 1024-byte alignment
  // Tensor-memory columns per query tile t: scores S_t (128 fp32 columns,
  // for D = 128 later overwritten by P_t: for keys 16k..16k+15, bf16 pairs in
  // columns 16k..16k+7) and the output accumulator O_t (D fp32 columns).
  __host__ __device__ static constexpr int tm_s(int t) { return 256 * t; }
  __host__ __device__ static constexpr int tm_o(int t) { return 256 * t + 128; }
  // D = 64: O_t uses 64 of its 128 columns and P_t (keys 16k..16k+15 as bf16
  // pairs in columns 8k..8k+7) the other 64, so the softmax frees S_t as soon
  // as it has read it and the next score product runs while the exponentials
  // are computed. D = 128: P_t is written over S_t.
  // Also D = 64: one MMA-issuing warp per query tile (measured faster there;
  // at D = 128 one warp alternating the tiles is faster).
  static constexpr bool SEP_P = (D == 64);
  static constexpr int N_MMA = SEP_P ? 2 : 1;  // MMA-issuing warps
  __host__ __device__ static constexpr int tm_p(int t) { return SEP_P ? 256 * t + 192 : 256 * t; }
  static constexpr int TMEM_COLS = 512;
  static constexpr int THREADS = 32 * (9 + N_MMA);  // 8 softmax warps, producer, MMA warps
  static_assert(SMEM_ALLOC <= 232448, "shared-memory plan exceeds 227 KB");
};

struct FwdParams {
  __nv_bfloat16* o;
  __nv_bfloat16* o_lo;  // optional: bf16(O - o), the part of O that bf16 o drops
  float* lse;
  int B, Hq, Hkv, S, G;
  int causal;
  int window;        // > 0: query i sees keys i-window+1..i (needs causal); 0: no window
  float scale_log2;  // scale * log2(e)
  int n_qblocks;     // blocks of two 128-row query tiles
  int* status;
  unsigned long long timeout_ns;
  int inject_stall;  // testing hook: the MMA warp issues nothing (waits then run out)
};

// Work items of the query-tile-parallel kernels (the forward, and the
// backward's Dvec pass): batch b, query head hq, and the two 128-row query
// tiles starting at q0; tile t needs K/V tiles [j_lo[t], n_kv[t]). A sliding
// window of W keys starts row r's keys at r - W + 1.
struct FwdItem {
  int b, hq, g, q0;
  int n_kv[2], j_lo[2];
};

// Items in longest-first order: index i takes head i % (B Hq) of query-block
// pair n_qblocks - 1 - i / (B Hq) (the causal rows get shorter down the list).
// P is a parameter block with B, Hq, G, S, causal, window and n_qblocks;
// WIN: sliding-window instantiation (without it the window code compiles
// away).
template <bool WIN, class P>
__device__ __forceinline__ FwdItem fwd_item(const P& p, int i) {
  constexpr int BQ = 128, BK = 128;
  FwdItem it;
  const int bhq = p.B * p.Hq;
  const int bh = i % bhq;
  it.hq = bh % p.Hq;
  it.b = bh / p.Hq;
  it.g = it.hq / p.G;
  it.q0 = (p.n_qblocks - 1 - i / bhq) * (2 * BQ);
  const int nkv_all = (p.S + BK - 1) / BK;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int qt0 = it.q0 + t * BQ;
    it.n_kv[t] = p.causal ? min(qt0 / BK + 1, nkv_all) : nkv_all;
    // (A tile wholly past S still runs one K/V tile; its rows are not stored.)
    it.j_lo[t] = WIN ? min(max(0, qt0 - p.window + 1) / BK, it.n_kv[t] - 1) : 0;
  }
  return it;
}

// The r-th item of CTA c among G CTAs: round r hands items r G .. r G + G - 1
// to the CTAs, in reverse order on odd rounds, which balances the
// longest-first list (a negative result: no item left).
__device__ __forceinline__ int fwd_item_index(int r, int c, int G, int n_items) {
  const int i = r * G + ((r & 1) ? (G - 1 - c) : c);
  return i < n_items ? i : -1;
}

// ---------------------------------------------------------------- backward Dvec pass
// The backward's Dvec without the forward's output: Dvec_i = sum_j P_ij dP_ij
// with P_ij = exp2(scale log2(e) q_i.k_j - LSE_i log2(e)) and dP = dO V^T,
// per query row (the definition that rowsum(dO * O) equals). Items as the
// forward's: two 128-row query tiles of one head per item, K/V tiles
// streaming through a ring. Warps 0-3 / 4-7: rows of tile A / B (one row per
// thread, its TMEM lane); warp 8: TMA producer; warp 9: MMA issuer.
template <int D>
struct DvecCfg {
  static constexpr int BQ = 128;
  static constexpr int BK = 128;
  static constexpr int KCH = D / 64;
  static constexpr int Q_BYTES = BQ * D * 2;         // one Q or dO tile
  static constexpr int KV_BYTES = BK * D * 2;        // one K or V tile
  static constexpr int NSLOT = (D == 128) ? 3 : 8;   // ring slots
  static constexpr int SMEM_Q = 0;                   // Q_A, Q_B, dO_A, dO_B
  static constexpr int SMEM_RING = 4 * Q_BYTES;
  static constexpr int SMEM_BYTES = SMEM_RING + NSLOT * KV_BYTES;
  static constexpr int SMEM_ALLOC = SMEM_BYTES + 1024;
  // Tensor-memory columns per query tile t: S_t (128 fp32) and dP_t (128 fp32).
  __host__ __device__ static constexpr int tm_s(int t) { return 256 * t; }
  __host__ __device__ static constexpr int tm_dp(int t) { return 256 * t + 128; }
  static constexpr int TMEM_COLS = 512;
  static constexpr int THREADS = 320;
  static_assert(SMEM_ALLOC <= 232448, "shared-memory plan exceeds 227 KB");
};

struct DvecParams {
  const float* nlse2;  // [B, Hq, S_pad] -lse * log2(e)
  float* dvec;         // [B, Hq, S_pad] out (rows < S)
  int B, Hq, Hkv, S, S_pad, G;
  int causal;
  int window;
  float scale_log2;
  int n_qblocks;
  int* status;
  unsigned long long timeout_ns;
  int inject_stall;
};

// ---------------------------------------------------------------- backward
// One CTA per (batch, kv head, 128-key tile): K_j and V_j stay resident, the
// group's query heads and their 64-row query tiles stream through a three-stage
// ring holding Q_i, dO_i and the rows' log2-scaled LSE and Dvec. dK_j and dV_j
// accumulate in TMEM over the whole loop; dQ tiles are added into the fp32
// dq output with TMA tensor reductions.
// Warps 0-7: P^T / dS^T and the dK/dV epilogue (one key row per thread; warps
// w and w+4 share TMEM lanes and split the 64 query columns); the dQ warps
// from 8 on (see DQ_IN_COMPUTE); then the TMA producer and the MMA issuer.
//
// P and dS enter the gradient MMAs as a pair of bf16 values (hi = bf16(x),
// lo = bf16(x - hi)), i.e. with about 16 significant bits: dV += P_hi^T dO +
// P_lo^T dO and likewise for dK and dQ. dQ is produced transposed
// (dQ^T = K_j^T dS^T, M = 128 head-dim rows) so every MMA has M = 128; for
// D = 64 the upper 64 rows of K^T are zero in shared memory and ignored.
template <int D>
struct BwdCfg {
  static constexpr int BK = 128;
  static constexpr int BQ = 64;
  static constexpr int KCH = D / 64;
  static constexpr int K_BYTES = BK * 128 * 2;       // always two 64-column chunks
  static constexpr int V_BYTES = BK * D * 2;
  static constexpr int Q_BYTES = BQ * D * 2;
  static constexpr int STAGES = 3;
  static constexpr int ROWVEC_BYTES = BQ * 4;
  // Who reads dQ^T out of TMEM. D = 64: the P^T / dS^T warps, just before
  // storing P^T / dS^T over it, each staging its 32-row half tile in its own
  // shared-memory tile, and one warp issues the reductions. D = 128: four
  // drain warps, which also stage the tile, so that the twice larger staging
  // stores stay off the P^T / dS^T warps (measured faster there).
  static constexpr bool DQ_IN_COMPUTE = (D == 64);
  // Per stage: Q, dO, then -LSE*log2(e) and Dvec of the stage's BQ query rows
  // (1024-byte multiple) when the row vectors sit in the stage, as for D = 128.
  static constexpr int STAGE_BYTES =
      DQ_IN_COMPUTE ? 2 * Q_BYTES : (2 * Q_BYTES + 2 * ROWVEC_BYTES + 1023) / 1024 * 1024;
  static constexpr int DS_BYTES = BK * BQ * 2;       // one bf16 dS^T tile (hi or lo)
  static constexpr int DQ_ROWS = BQ / 2;            // dQ leaves in two halves of 32 rows
  static constexpr int DQS_BYTES = DQ_ROWS * D * 4;  // dQ staging half-tile, fp32
  static constexpr int SMEM_K = 0;
  static constexpr int SMEM_V = SMEM_K + K_BYTES;
  static constexpr int SMEM_STAGE = SMEM_V + V_BYTES;
  static constexpr int SMEM_DS_HI = SMEM_STAGE + STAGES * STAGE_BYTES;
  static constexpr int SMEM_DS_LO = SMEM_DS_HI + DS_BYTES;
  static constexpr int N_DQS = DQ_IN_COMPUTE ? 2 : 1;  // dQ staging tiles
  static constexpr int SMEM_DQS = SMEM_DS_LO + DS_BYTES;
  // D = 64: the row vectors of every stage, after the staging tiles.
  static constexpr int SMEM_ROWS = SMEM_DQS + N_DQS * DQS_BYTES;
  static constexpr int SMEM_BYTES = SMEM_ROWS + (DQ_IN_COMPUTE ? STAGES * 2 * ROWVEC_BYTES : 0);
  static constexpr int SMEM_ALLOC = SMEM_BYTES + 1024;
  // Tensor-memory columns. dQ^T is produced as one N = 128 product over the
  // adjacent [dS_hi^T | dS_lo^T] tiles: its columns 0..63 hold K^T dS_hi^T and
  // 64..127 hold K^T dS_lo^T, summed when read back. P^T and dS^T (hi/lo,
  // bf16 pairs) live in that region between the read of dQ^T(i-1) and the
  // dQ MMA of tile i, which runs after dV(i) and dK(i) have read them. dV and
  // dK take their A operand from tensor memory, so only their B operand
  // (dO, Q) is read from shared memory.
  static constexpr int TM_ST = 0;       // S^T  fp32 (64 cols)
  static constexpr int TM_DPT = 64;     // dP^T fp32 (64 cols)
  static constexpr int TM_DV = 128;     // dV   fp32 (D cols)
  static constexpr int TM_DK = 256;     // dK   fp32 (D cols)
  static constexpr int TM_DQ = 384;     // dQ^T fp32 (2 x 64 cols: hi part, lo part)
  // P^T and dS^T, bf16 pairs, 64 cols each: query columns 32c..32c+31 take
  // 32 cols from 32c on, hi pairs first (16 cols) then lo pairs (16 cols).
  static constexpr int TM_P = 384;
  static constexpr int TM_DS = 448;
  static constexpr int TMEM_COLS = 512;
  static constexpr int N_DQW = DQ_IN_COMPUTE ? 1 : 4;  // warps 8 .. 8 + N_DQW - 1
  static constexpr int W_PROD = 8 + N_DQW;               // TMA producer warp
  static constexpr int W_MMA = W_PROD + 1;               // MMA issuer warp
#ifdef ATTN_TRACE
  static constexpr int THREADS = 32 * (W_MMA + 2);  // + one warp that timestamps MMA completions
#else
  static constexpr int THREADS = 32 * (W_MMA + 1);
#endif
  static_assert(SMEM_ALLOC <= 232448, "shared-memory plan exceeds 227 KB");
};

struct BwdParams {
  const float* nlse2;  // [B, Hq, S_pad] -lse * log2(e); -inf on padding rows
  const float* dvec;   // [B, Hq, S_pad] rowsum(dO * O); 0 on padding rows
  float* dk;           // [B, S, Hkv, D] fp32
  float* dv;           // [B, S, Hkv, D] fp32
  int B, Hq, Hkv, S, S_pad, G;
  int causal;
  int window;  // > 0: query i sees keys i-window+1..i (needs causal); 0: no window
  float scale_log2;
  float scale;
  int n_ktiles;
  // Query heads of a kv head's group are split over `split` items per key
  // tile (1 or 2), each taking G / split consecutive heads; with 2 the dK and
  // dV rows are added into zeroed dk and dv. Set by the launcher.
  int split;
  // Persistent launch: the work counter (the status region's word
  // kBwdWorkWord, zeroed by the preprocess) and the number of item codes.
  int* work;
  int n_items;
  int* status;
  unsigned long long timeout_ns;
  int inject_stall;  // testing hook: the MMA warp issues nothing (waits then run out)
};

// Status word of a backward workspace (the first 8 bytes of it): int 0 holds
// the status code (0, or 4 after a bounded wait ran out), int 1 a tag that
// marks the word as started by this library. A backward call starts a
// workspace that lacks the tag at status 0; on a tagged workspace it leaves
// the code as it is, so that a timeout an earlier call recorded stays there
// until attn_check_status reads (and clears) it, instead of being erased.
constexpr int kStatusTag = 0x41544E31;
__device__ __forceinline__ void init_status_word(int* status) {
  volatile int* w = status;
  if (w[1] != kStatusTag) {
    w[0] = 0;
    w[1] = kStatusTag;
  }
}

// Workspace layout of the backward pass (all offsets 256-byte aligned).
struct BwdWorkspace {
  size_t off_status, off_nlse2, off_dvec, total;
};
// Word of the workspace's 256-byte status region that counts the items the
// persistent backward main kernel has taken (words 0 and 1: status word and
// its tag).
constexpr int kBwdWorkWord = 4;

inline BwdWorkspace bwd_workspace_layout(int B, int Hq, int S) {
  auto al = [](size_t x) { return (x + 255) / 256 * 256; };
  BwdWorkspace w;
  const size_t rows = static_cast<size_t>(B) * Hq * seq_pad(S);
  w.off_status = 0;
  w.off_nlse2 = 256;
  w.off_dvec = w.off_nlse2 + al(rows * 4);
  w.total = w.off_dvec + al(rows * 4);
  return w;
}

// ---------------------------------------------------------------- tracing
// Timeline tracing for kernel tuning, compiled in only with -DATTN_TRACE (the
// regular build has none of it). Each traced CTA (a 2-D grid: blockIdx.x ==
// 0 and the first kTraceCtas values of blockIdx.y; a 1-D grid: the first
// kTraceCtas blocks) gets kTraceRoles streams of
// kTraceEvents 64-bit records: event code (bits 56..63), iteration
// (bits 40..55) and the SM clock (bits 0..39).
constexpr int kTraceCtas = 32;
constexpr int kTraceRoles = 16;
constexpr int kTraceEvents = 2048;
#ifdef ATTN_TRACE
// Each kernel source that traces defines its own buffer named g_attn_trace.
struct TraceCursor {
  unsigned long long* base = nullptr;
  int n = 0;
  __device__ void init(unsigned long long* buf, int role) {
    const unsigned idx = gridDim.y > 1 ? (blockIdx.x == 0 ? blockIdx.y : kTraceCtas) : blockIdx.x;
    if (idx < kTraceCtas) base = buf + (static_cast<size_t>(idx) * kTraceRoles + role) * kTraceEvents;
  }
  __device__ void ev(int code, int it) {
    if (base && n < kTraceEvents) {
      const unsigned long long c = clock64();
      base[n++] = (static_cast<unsigned long long>(code) << 56) |
                  (static_cast<unsigned long long>(it & 0xFFFF) << 40) | (c & 0xFFFFFFFFFFull);
    }
  }
};
#define ATTN_TRACE_INIT(tc, role) (tc).init(g_attn_trace, role)
#define ATTN_TRACE_EV(tc, code, it) (tc).ev((code), (it))
#else
struct TraceCursor {};
#define ATTN_TRACE_INIT(tc, role) ((void)0)
#define ATTN_TRACE_EV(tc, code, it) ((void)0)
#endif

// Status word of attn_bwd_noalloc's scratch array on the current device, or
// nullptr if no call on this device has looked the array up yet.
int* noalloc_status_word();

// ---------------------------------------------------------------- launchers
cudaError_t launch_fwd(int D, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, const CUtensorMap& tolo, const FwdParams& p,
                       cudaStream_t stream);
cudaError_t launch_bwd_preprocess(const __nv_bfloat16* o, const __nv_bfloat16* o_lo,
                                  const __nv_bfloat16* dO, const float* lse, float* nlse2,
                                  float* dvec, float* dq, int* status, int B, int Hq, int S,
                                  int D, cudaStream_t stream);
cudaError_t launch_bwd_dvec(int D, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo, const DvecParams& p,
                            cudaStream_t stream);
cudaError_t launch_bwd_main(int D, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                            const BwdParams& p, cudaStream_t stream);

}  // namespace attn
