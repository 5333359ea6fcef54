// Backward attention kernels for sm_103a: the exact gradient of
// O = softmax(scale * Q K^T) V ("Scheduling Data to Compute: Hierarchical Data
// Pipelining for LLM Training on AMD GPUs", section 2.1, Eq. (1)) for the loss
// L = sum(dO * O). With P = exp(scale * Q K^T - LSE):
//   dV = P^T dO,  dP = dO V^T,  Dvec_i = rowsum(dO * O)_i,  dS = P * (dP - Dvec),
//   dK = scale * dS^T Q,  dQ = scale * dS K.
// The paper's Table 3 lists the scores, query-gradient and key-gradient
// products with their transposed operands; here every transposed operand is a
// shared-memory descriptor in MN-major form, so no tile is ever transposed.
//
// Two kernels run in order on one stream:
//   1. preprocess: Dvec (from o, plus the forward's low-order residual o_lo
//      when given) and log2-scaled LSE rows into the workspace; the fp32 dq
//      output zeroed (HBM-bound).
//   2. main: one CTA per (batch, kv head, 128-key tile). K_j and V_j stay in
//      shared memory while Q_i, dO_i, LSE_i and Dvec_i of every 64-row query
//      tile of the group's query heads stream through a three-stage TMA ring:
//        S^T = K_j Q_i^T and dP^T = V_j dO_i^T         (TMEM)
//        P^T (TMEM) and scale * dS^T (shared memory) as bf16 hi/lo pairs
//        dV += P^T dO_i, dK += dS^T Q_i                 (TMEM, whole loop)
//        dQ_i^T = K_j^T dS^T                            (TMEM)
//      dQ^T(i) is read out of TMEM (D = 64: by the P^T / dS^T warps, just
//      before they store P^T(i+1) / dS^T(i+1) over it; D = 128: by four drain
//      warps), staged in shared memory and added into dq with asynchronous
//      TMA tensor reductions (fp32 add in L2).
#include <algorithm>
#include <type_traits>
#include <utility>

#include "attn_common.cuh"
#include "sm100_ptx.cuh"

namespace attn {
using namespace ptx;

namespace {

// The main kernel's waits sleep until their phase completes (suspend-time
// hint): its 14 warps share four schedulers, and a polling warp would take
// issue slots from the P/dS and drain warps (1-2% faster, same-box A/B).
constexpr bool kBwdSuspend = true;

#ifdef ATTN_TRACE
static __device__ unsigned long long g_attn_trace[kTraceCtas * kTraceRoles * kTraceEvents];
// Per CTA of the main kernel (linear block index, up to kSpanCtas): global
// timer at entry and at exit (ns), and the SM it ran on.
constexpr int kSpanCtas = 16384;
static __device__ unsigned long long g_attn_spans[kSpanCtas * 4];
#endif

// ------------------------------------------------------------------ preprocess
// Dvec_i = sum_d dO_id (o_id + o_lo_id) and -LSE_i log2(e) per row, the
// padding rows of both, and dq zeroed: an HBM-bound pass. A row of D bf16
// values is read by D/8 threads, 16 bytes each. Each warp step takes
// kPreU row groups: it issues all their loads first, then zeroes the dq rows
// of the same rows (so reads and writes stay interleaved over the pass), then
// reduces. With o = NULL the Dvec rows (not their padding) are left to the
// Dvec pass. Measured at the Llama-3-8B shape against variants with four row
// groups in flight, streaming cache hints, or the zeroing on blocks of its
// own: two row groups with eight blocks per SM launched was the fastest.
constexpr int kPreU = 2;

template <int D>
__global__ void __launch_bounds__(256) attn_bwd_preprocess_kernel(
    const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ o_lo,
    const __nv_bfloat16* __restrict__ dO, const float* __restrict__ lse, float* __restrict__ nlse2,
    float* __restrict__ dvec, float4* __restrict__ dq, int* __restrict__ status, int B, int Hq,
    int S, int S_pad) {
  constexpr int TPR = D / 8;        // threads per row, 8 bf16 (16 bytes) each
  constexpr int RPW = 32 / TPR;     // rows per warp and row group
  constexpr int RPI = RPW * kPreU;  // rows per warp step
  constexpr int Z4 = RPI * D / 4 / 32;  // float4 zero stores per lane and step
  const long long nrows = static_cast<long long>(B) * S * Hq;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    init_status_word(status);
    status[kBwdWorkWord] = 0;  // the main kernel's work counter
  }
  const long long gthreads = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long gwarp = tid / 32, nwarps = gthreads / 32;
  const int lane = threadIdx.x % 32;
  const int sub = lane % TPR;
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  // Rows in [B, S, Hq] order, so a warp reads consecutive memory. The loop
  // condition is warp-uniform so the shuffles below see the whole warp.
  for (long long base = gwarp * RPI; base < nrows; base += nwarps * RPI) {
    uint4 a[kPreU], c[kPreU], r[kPreU];
#pragma unroll
    for (int u = 0; u < kPreU; ++u) {
      const long long row = base + u * RPW + lane / TPR;
      a[u] = c[u] = r[u] = make_uint4(0u, 0u, 0u, 0u);
      if (row < nrows && o) {
        a[u] = reinterpret_cast<const uint4*>(o + row * D)[sub];
        c[u] = reinterpret_cast<const uint4*>(dO + row * D)[sub];
        if (o_lo) r[u] = reinterpret_cast<const uint4*>(o_lo + row * D)[sub];
      }
    }
    // dq rows base .. base + RPI - 1 (the reductions of the main kernel add into them).
    const long long f_end = min(nrows, base + RPI) * (D / 4);
#pragma unroll
    for (int u = 0; u < Z4; ++u) {
      const long long f = base * (D / 4) + u * 32 + lane;
      if (f < f_end) dq[f] = z;
    }
#pragma unroll
    for (int u = 0; u < kPreU; ++u) {
      const long long row = base + u * RPW + lane / TPR;
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a[u]);
      const __nv_bfloat162* c2 = reinterpret_cast<const __nv_bfloat162*>(&c[u]);
      const __nv_bfloat162* r2 = reinterpret_cast<const __nv_bfloat162*>(&r[u]);
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 fa = __bfloat1622float2(a2[i]);
        const float2 fr = __bfloat1622float2(r2[i]);
        const float2 fc = __bfloat1622float2(c2[i]);
        acc = fmaf(fa.x + fr.x, fc.x, acc);
        acc = fmaf(fa.y + fr.y, fc.y, acc);
      }
#pragma unroll
      for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (row < nrows && sub == 0) {
        const int h = static_cast<int>(row % Hq);
        const long long bs = row / Hq;
        const int s = static_cast<int>(bs % S);
        const int b = static_cast<int>(bs / S);
        const long long bh = static_cast<long long>(b) * Hq + h;
        if (o) dvec[bh * S_pad + s] = acc;
        nlse2[bh * S_pad + s] = -lse[bh * S + s] * kLog2e;
      }
    }
  }
  // Padding rows S..S_pad-1 of every (b, h): probability 0 (nlse2 = -inf), Dvec 0.
  const long long npad = static_cast<long long>(B) * Hq * (S_pad - S);
  for (long long i = tid; i < npad; i += gthreads) {
    const long long bh = i / (S_pad - S);
    const int s = S + static_cast<int>(i % (S_pad - S));
    dvec[bh * S_pad + s] = 0.f;
    nlse2[bh * S_pad + s] = -INFINITY;
  }
}

// ------------------------------------------------------------------ main
// Adds a [rows x D] fp32 box from shared memory into the 4-D (D, H, S, B) map.
__device__ __forceinline__ void tma_reduce_add_4d(const CUtensorMap* m, int c0, int c1, int c2,
                                                  int c3, uint32_t src) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.4d.global.shared::cta.add.tile.bulk_group"
      " [%0, {%1, %2, %3, %4}], [%5];" ::"l"(reinterpret_cast<uint64_t>(m)),
      "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(src)
      : "memory");
}

// dk and dv zeroed before a split backward adds into them.
__global__ void __launch_bounds__(256) zero_f32x4_kernel(float4* __restrict__ a,
                                                         float4* __restrict__ b, long long n4) {
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    a[i] = z;
    b[i] = z;
  }
}

// Writes 16 bytes to unit `u` (0..7) of 128-byte row `row` of a tile stored
// with 128-byte swizzle (8-row atoms on 1024-byte boundaries).
__device__ __forceinline__ void st_sw128(uint32_t tile, int row, int u, uint4 v) {
  const uint32_t addr = tile + row * 128 + ((u ^ (row & 7)) << 4);
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// One item of the backward main kernel: key tile j of one (batch b, kv head
// g) and `hpc` consecutive query heads h0.. of its group (all of them, or
// one half when the group is split), over the query tiles that see the tile.
// Item code = (j * B * Hkv + b * Hkv + g) * split + part.
struct BwdItem {
  int b, g, h0, hpc, k0, i_start, niq, n_it;
};
template <bool WIN>
__host__ __device__ __forceinline__ BwdItem bwd_item(const BwdParams& p, int code, int bq, int bk) {
  BwdItem t;
  const int part = code % p.split;
  const int rest = code / p.split;
  const int bg = rest % (p.B * p.Hkv);
  const int j = rest / (p.B * p.Hkv);
  t.g = bg % p.Hkv;
  t.b = bg / p.Hkv;
  t.hpc = p.G / p.split;
  t.h0 = t.g * p.G + part * t.hpc;
  t.k0 = j * bk;
  const int nq = (p.S + bq - 1) / bq;
  t.i_start = p.causal ? t.k0 / bq : 0;
  // With a window of W keys, the last row that sees this tile's keys is
  // k0 + BK - 1 + W - 1.
  const int i_last = (t.k0 + bk + p.window - 2) / bq + 1;
  const int i_end = WIN ? (i_last < nq ? i_last : nq) : nq;
  t.niq = i_end - t.i_start;
  t.n_it = t.hpc * t.niq;
  return t;
}

// Head and query tile of an item's iteration `it`: heads outer, query tiles
// inner (measured as fast as or faster than query-tile-outer orders).
__device__ __forceinline__ int bwd_head(const BwdItem& t, int it) { return t.h0 + it / t.niq; }
__device__ __forceinline__ int bwd_qtile(const BwdItem& t, int it) { return t.i_start + it % t.niq; }

// WIN: sliding-window instantiation (p.window > 0). PERSIST: one CTA per SM
// taking items from the work counter until none is left; otherwise one CTA
// per item, named by the block index.
template <int D, bool WIN, bool PERSIST>
__global__ void __launch_bounds__(BwdCfg<D>::THREADS, 1)
    attn_bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_do,
                         const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
  using C = BwdCfg<D>;
  constexpr int BQ = C::BQ, BK = C::BK, ST = C::STAGES;
  constexpr int HALF = BQ / 2;  // query columns per compute warpgroup
#ifdef ATTN_TRACE
  const unsigned long long t_entry = globaltimer();
#endif
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  __shared__ uint64_t bar_kv_full, bar_kv_free, bar_mma_done, bar_dkv_free, bar_fin;
  __shared__ uint64_t bar_st_full[ST], bar_st_empty[ST];
  __shared__ uint64_t bar_sdp_full, bar_sdp_free, bar_pds_full, bar_pds_free, bar_dq_full,
      bar_dq_free, bar_stg_full[2], bar_stg_free[2];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;
  // Persistent launch: the codes of this CTA's items, in the order taken, in
  // a 4-slot ring (bar_item[s] completes when slot s holds the next code; -1
  // ends the run). Four slots suffice: the producer starts item ii + 4 only
  // after the MMA warp has issued all of item ii + 3 (kv_free), by when the
  // compute and dQ warps have passed the start of item ii + 2.
  __shared__ int item_code_s[4];
  __shared__ uint64_t bar_item[4];
#ifdef ATTN_TRACE
  __shared__ int trace_iters;  // iterations the MMA warp issued (for the observer)
#endif

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  const uint32_t sK = smem_u32(smem + C::SMEM_K);
  const uint32_t sV = smem_u32(smem + C::SMEM_V);
  const uint32_t sStage = smem_u32(smem + C::SMEM_STAGE);
  const uint32_t sDsHi = smem_u32(smem + C::SMEM_DS_HI);
  const uint32_t sDsLo = smem_u32(smem + C::SMEM_DS_LO);
  const uint32_t sDQS = smem_u32(smem + C::SMEM_DQS);

  if (D == 64) {
    // Rows 64..127 of K^T (the second 64-column chunk of K) are zero, so the
    // M = 128 dQ^T product carries zeros in its unused upper half. The K
    // loads fill only the first chunk, so this holds for every item.
    uint4* z = reinterpret_cast<uint4*>(smem + C::SMEM_K + BK * 128);
    for (int i = threadIdx.x; i < BK * 128 / 16; i += blockDim.x) z[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_async_smem();
  }
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar_kv_full), 1);
    mbar_init(smem_u32(&bar_kv_free), 1);
    mbar_init(smem_u32(&bar_mma_done), 1);
    mbar_init(smem_u32(&bar_dkv_free), 256);
    mbar_init(smem_u32(&bar_fin), 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(smem_u32(&bar_st_full[s]), 1);
      mbar_init(smem_u32(&bar_st_empty[s]), 1);
    }
    mbar_init(smem_u32(&bar_sdp_full), 1);
    mbar_init(smem_u32(&bar_sdp_free), 256);
    mbar_init(smem_u32(&bar_pds_full), 256);
    mbar_init(smem_u32(&bar_pds_free), 1);
    mbar_init(smem_u32(&bar_dq_full), 1);
    mbar_init(smem_u32(&bar_dq_free), 128);
    for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&bar_item[i]), 1);
#ifdef ATTN_TRACE
    trace_iters = -1;
#endif
    for (int h = 0; h < 2; ++h) {
      mbar_init(smem_u32(&bar_stg_full[h]), 128);
      mbar_init(smem_u32(&bar_stg_free[h]), 1);
    }
    fence_barrier_init();
  }
  if (warp == C::W_MMA) {
    tmem_alloc(smem_u32(&tmem_base_s), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  const WaitCtl ctl{&abort_flag, p.status, p.timeout_ns};

  // Code of this CTA's item ii, -1 past its last item, -2 if the wait for it
  // gave up. Grid launch: the one item the block index names. Persistent
  // launch: items are taken in code order (key tiles longest first) from a
  // work counter that the preprocess zeroes; the producer takes the next one
  // when it starts an item (take_item) and the other roles read it from the
  // ring (item_code).
  auto item_code = [&](int ii) -> int {
    if constexpr (PERSIST) {
      if (!mbar_wait_warp<kBwdSuspend>(smem_u32(&bar_item[ii & 3]), (ii >> 2) & 1, ctl)) return -2;
      return reinterpret_cast<volatile int*>(item_code_s)[ii & 3];
    } else {
      return ii == 0 ? static_cast<int>(blockIdx.y * gridDim.x + blockIdx.x) : -1;
    }
  };
  auto take_item = [&](int ii) -> int {
    if constexpr (PERSIST) {
      int code = 0;
      if (lane == 0) {
        code = atomicAdd(p.work, 1);
        if (code >= p.n_items) code = -1;
        reinterpret_cast<volatile int*>(item_code_s)[ii & 3] = code;
        mbar_arrive(smem_u32(&bar_item[ii & 3]));
      }
      return __shfl_sync(0xffffffffu, code, 0);
    } else {
      return item_code(ii);
    }
  };

  auto stage_q = [&](int s) { return sStage + s * C::STAGE_BYTES; };
  auto stage_do = [&](int s) { return sStage + s * C::STAGE_BYTES + C::Q_BYTES; };
  auto stage_rows = [&](int s) {  // nlse2 then dvec, BQ floats each
    return reinterpret_cast<const float*>(
        C::DQ_IN_COMPUTE ? smem + C::SMEM_ROWS + s * 2 * C::ROWVEC_BYTES
                         : smem + C::SMEM_STAGE + s * C::STAGE_BYTES + 2 * C::Q_BYTES);
  };
  // Barrier phases run on across items: `git` counts the (head, query tile)
  // iterations of earlier items, `ii` the items.

  if (warp == C::W_PROD) {
    // ------------------------------------------------------------ producer
    // The whole warp runs this loop; each copy is issued by one elected lane.
    // An item's K and V replace the previous item's once its last MMA has
    // run (kv_free); its first query stages are issued before that wait, so
    // they load while the previous item finishes.
    {
      TraceCursor tc;
      if (lane == 0) ATTN_TRACE_INIT(tc, 0);
      ATTN_TRACE_EV(tc, 1, 0);
      if (lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_do);
      }
      bool ok = true;
      int issued = 0, kv_issued = 0, git = 0;
      auto load_kv = [&](const BwdItem& t) {
        mbar_arrive_expect_tx_el(smem_u32(&bar_kv_full), 2 * C::V_BYTES);
        for (int c = 0; c < C::KCH; ++c) {
          tma_load_4d_el(sK + c * (BK * 128), &tm_k, smem_u32(&bar_kv_full), c * 64, t.g, t.k0, t.b);
          tma_load_4d_el(sV + c * (BK * 128), &tm_v, smem_u32(&bar_kv_full), c * 64, t.g, t.k0, t.b);
        }
      };
      for (int ii = 0; ok && (PERSIST || ii == 0); ++ii) {
        const int code = take_item(ii);
        if (code < 0) break;
        const BwdItem t = bwd_item<WIN>(p, code, BQ, BK);
        if (!bounds_ok(t.b < p.B && t.g < p.Hkv && t.k0 < p.S, ctl)) {
          ok = false;
          break;
        }
        const int n_early = ii == 0 ? 0 : min(ST, t.n_it);  // stages issued before K/V
        if (ii == 0) {
          load_kv(t);
          ++kv_issued;
        }
        for (int it = 0; it < t.n_it; ++it) {
          if (ii > 0 && it == n_early) {
            ok = mbar_wait_warp<kBwdSuspend>(smem_u32(&bar_kv_free), (ii - 1) & 1, ctl);
            if (!ok) break;
            load_kv(t);
            ++kv_issued;
          }
          const int gi = git + it;
          const int s = gi % ST, round = gi / ST;
          if (round > 0) ok = mbar_wait_warp<kBwdSuspend>(smem_u32(&bar_st_empty[s]), (round - 1) & 1, ctl);
          if (!ok) break;
          ATTN_TRACE_EV(tc, 2, gi);  // stage free, issuing loads
          const int h = bwd_head(t, it);
          const int q0 = bwd_qtile(t, it) * BQ;
          if (!bounds_ok(h < p.Hq && q0 >= 0 && q0 + BQ <= p.S_pad && s < ST, ctl)) {
            ok = false;
            break;
          }
          const uint32_t full = smem_u32(&bar_st_full[s]);
          mbar_arrive_expect_tx_el(full, 2 * C::Q_BYTES + 2 * C::ROWVEC_BYTES);
          for (int c = 0; c < C::KCH; ++c) {
            tma_load_4d_el(stage_q(s) + c * (BQ * 128), &tm_q, full, c * 64, h, q0, t.b);
            tma_load_4d_el(stage_do(s) + c * (BQ * 128), &tm_do, full, c * 64, h, q0, t.b);
          }
          const size_t rowoff = (static_cast<size_t>(t.b) * p.Hq + h) * p.S_pad + q0;
          const uint32_t rows = smem_u32(stage_rows(s));
          bulk_load_el(rows, p.nlse2 + rowoff, C::ROWVEC_BYTES, full);
          bulk_load_el(rows + C::ROWVEC_BYTES, p.dvec + rowoff, C::ROWVEC_BYTES, full);
          issued = gi + 1;
        }
        if (ok && ii > 0 && t.n_it <= n_early) {  // an item of at most ST iterations
          ok = mbar_wait_warp<kBwdSuspend>(smem_u32(&bar_kv_free), (ii - 1) & 1, ctl);
          if (!ok) break;
          load_kv(t);
          ++kv_issued;
        }
        git += t.n_it;
      }
      if (lane == 0) {
        // Let every copy issued land before the CTA's shared memory goes away
        // (immediate in a normal run, where the MMA warp consumed them all).
        for (int gi = max(0, issued - ST); gi < issued; ++gi)
          mbar_wait_drain(smem_u32(&bar_st_full[gi % ST]), (gi / ST) & 1, 50000000ull);
        if (kv_issued > 0) mbar_wait_drain(smem_u32(&bar_kv_full), (kv_issued - 1) & 1, 50000000ull);
      }
      (void)ok;
      __syncwarp();
    }
  } else if (warp == C::W_MMA) {
    // ------------------------------------------------------------ MMA issuer
    TraceCursor tc;
    if (lane == 0) ATTN_TRACE_INIT(tc, 1);
    // The whole warp runs this loop and builds the (warp-uniform) descriptors;
    // each MMA and commit is issued by one elected lane.
    bool ok = !p.inject_stall;
    constexpr uint32_t idesc_sdp = idesc_bf16_f32(128, BQ, 0, 0);
    constexpr uint32_t idesc_kv = idesc_bf16_f32(128, D, 0, 1);
    constexpr uint32_t idesc_dq = idesc_bf16_f32(128, 2 * BQ, 1, 1);
    // Descriptor bases; each step below only adds a constant byte offset
    // (>> 4) to the start-address field.
    const uint64_t dK_kmaj = sw128_desc(sK, 16, 1024);
    const uint64_t dV_kmaj = sw128_desc(sV, 16, 1024);
    const uint64_t dK_mn = sw128_desc(sK, BK * 128, 1024);
    // [dS_hi^T | dS_lo^T] as one MN-major operand of N = 128: the second
    // 64-column block (dS_lo^T) sits DS_BYTES after the first.
    const uint64_t dDs_mn = sw128_desc(sDsHi, C::DS_BYTES, 1024);
    auto add = [](uint64_t d, uint32_t bytes) { return d + (bytes >> 4); };
    auto issue_sdp = [&](int s) {
      const uint64_t dq_k = sw128_desc(stage_q(s), 16, 1024);
      const uint64_t ddo_k = sw128_desc(stage_do(s), 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t ka = (kk >> 2) * (BK * 128) + (kk & 3) * 32;
        const uint32_t kb = (kk >> 2) * (BQ * 128) + (kk & 3) * 32;
        mma_ss_el(tmem + C::TM_ST, add(dK_kmaj, ka), add(dq_k, kb), idesc_sdp, kk > 0);
        mma_ss_el(tmem + C::TM_DPT, add(dV_kmaj, ka), add(ddo_k, kb), idesc_sdp, kk > 0);
      }
      mma_commit_el(smem_u32(&bar_sdp_full));
    };
    int git = 0;
    for (int ii = 0; ok && (PERSIST || ii == 0); ++ii) {
      const int code = item_code(ii);
      if (code < 0) {
        ok = code == -1;
        break;
      }
      const int n_it = bwd_item<WIN>(p, code, BQ, BK).n_it;
      ok = mbar_wait_warp<kBwdSuspend>(smem_u32(&bar_kv_full), ii & 1, ctl);
      ATTN_TRACE_EV(tc, 1, ii);
      // The item's first S^T/dP^T: once its stage has landed and the compute
      // warps have read the previous S^T/dP^T out of their columns.
      if (ok) ok = mbar_wait_warp<kBwdSuspend>(smem_u32(&bar_st_full[git % ST]), (git / ST) & 1, ctl);
      if (ok && git > 0) ok = mbar_wait_warp<kBwdSuspend>(smem_u32(&bar_sdp_free), (git - 1) & 1, ctl);
      if (!ok) break;
      tc_fence_after();
      issue_sdp(git % ST);
      for (int it = 0; it < n_it && ok; ++it) {  // ok is warp-uniform
        const int gi = git + it;
        const int s = gi % ST;
        if (it + 1 < n_it) {
          const int s1 = (gi + 1) % ST;
          ATTN_TRACE_EV(tc, 7, gi + 1);  // start waiting for stage / sdp_free
          ok = mbar_wait_warp<kBwdSuspend>(smem_u32(&bar_st_full[s1]), ((gi + 1) / ST) & 1, ctl);
          ATTN_TRACE_EV(tc, 10, gi + 1);  // stage landed
          if (ok) ok = mbar_wait_warp<kBwdSuspend>(smem_u32(&bar_sdp_free), gi & 1, ctl);
          if (!ok) break;
          tc_fence_after();
          issue_sdp(s1);
          ATTN_TRACE_EV(tc, 3, gi + 1);  // S^T, dP^T issued
        }
        ATTN_TRACE_EV(tc, 8, gi);  // start waiting for P, dS
        ok = mbar_wait_warp<kBwdSuspend>(smem_u32(&bar_pds_full), gi & 1, ctl);
        // The item's first dV/dK products overwrite the accumulators: the
        // compute warps must have read the previous item's dK/dV out.
        if (ok && it == 0 && ii > 0) ok = mbar_wait_warp<kBwdSuspend>(smem_u32(&bar_dkv_free), (ii - 1) & 1, ctl);
        if (!ok) break;
        ATTN_TRACE_EV(tc, 4, gi);  // P, dS ready seen
        tc_fence_after();
        const uint64_t dq_mn = sw128_desc(stage_q(s), BQ * 128, 1024);
        const uint64_t ddo_mn = sw128_desc(stage_do(s), BQ * 128, 1024);
        // dV += (P_hi + P_lo)^T dO_i and dK += (dS_hi + dS_lo)^T Q_i, A from
        // TMEM: 16 query columns = 8 TMEM columns a step.
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk) {
          const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
          const uint64_t bdo = add(ddo_mn, kk * 2048);
          const uint64_t bq = add(dq_mn, kk * 2048);
          const uint32_t hi = (kk >> 1) * 32 + (kk & 1) * 8, lo = hi + 16;
          mma_ts_el(tmem + C::TM_DV, tmem + C::TM_P + hi, bdo, idesc_kv, acc);
          mma_ts_el(tmem + C::TM_DV, tmem + C::TM_P + lo, bdo, idesc_kv, 1u);
          mma_ts_el(tmem + C::TM_DK, tmem + C::TM_DS + hi, bq, idesc_kv, acc);
          mma_ts_el(tmem + C::TM_DK, tmem + C::TM_DS + lo, bq, idesc_kv, 1u);
        }
        // Q_i and dO_i are not read again: hand the stage back to the producer.
        mma_commit_el(smem_u32(&bar_st_empty[s]));
        ATTN_TRACE_EV(tc, 5, gi);  // dV, dK issued
        if constexpr (!C::DQ_IN_COMPUTE) {
          if (gi >= 1) {
            ok = mbar_wait_warp<kBwdSuspend>(smem_u32(&bar_dq_free), (gi - 1) & 1, ctl);
            if (!ok) break;
            tc_fence_after();
          }
        }
        ATTN_TRACE_EV(tc, 9, gi);  // issuing dQ
        // dQ^T[d][q] (+ 64 columns for the lo part) = sum over keys of
        // K[key][d] [dS_hi^T | dS_lo^T][key][q]. It overwrites P^T and dS^T,
        // which dV(gi) and dK(gi) above have read (MMAs run in issue order).
        // dQ^T(gi-1) has been read out of these columns before P/dS(gi) were
        // stored (pds_full above) or, with drain warps, before dq_free.
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          mma_ss_el(tmem + C::TM_DQ, add(dK_mn, kk * 2048), add(dDs_mn, kk * 2048), idesc_dq,
                    kk > 0);
        if constexpr (!C::DQ_IN_COMPUTE) mma_commit_el(smem_u32(&bar_dq_full));
        mma_commit_el(smem_u32(&bar_pds_free));
        ATTN_TRACE_EV(tc, 6, gi);  // dQ issued
      }
      if (!ok) break;
      // The item's last products are issued: K and V may be replaced, and
      // dK/dV are complete once these run.
      mma_commit_el(smem_u32(&bar_kv_free));
      mma_commit_el(smem_u32(&bar_mma_done));
      git += n_it;
    }
#ifdef ATTN_TRACE
    if (lane == 0) reinterpret_cast<volatile int*>(&trace_iters)[0] = git;
#endif
    mma_commit_el(smem_u32(&bar_fin));
    // Every MMA issued finishes before TMEM is released.
    mbar_wait_drain(smem_u32(&bar_fin), 0, 50000000ull);
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------------------ P^T / dS^T warps 0-7
    const int r = threadIdx.x % 128;  // key row within the tile == TMEM lane
    const int cg = warp / 4;          // query-column half
    const uint32_t lane_base = static_cast<uint32_t>((warp % 4) * 32) << 16;
    bool ok = true;
    TraceCursor tc;
    if (lane == 0) ATTN_TRACE_INIT(tc, 2 + warp);
    float* stg = reinterpret_cast<float*>(smem + C::SMEM_DQS + cg * C::DQS_BYTES);
    // dQ^T = hi part (columns TM_DQ..+63) + lo part (TM_DQ+64..+127); this
    // thread takes TMEM lane r (head dim d = r) and this half's 32 query
    // columns of each part. The hi part sits where P^T goes and the lo part
    // where dS^T goes, so each store below follows the read of its cells.
    static_assert(C::TM_DQ == C::TM_P && C::TM_DQ + BQ == C::TM_DS, "dQ^T shares P^T/dS^T columns");
    auto read_dq_part = [&](int part, float (&v)[HALF], bool add) {
      uint32_t a[HALF];
      tmem_ld32(tmem + lane_base + C::TM_DQ + part * BQ + cg * HALF, a);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < HALF; ++i) v[i] = add ? v[i] + __uint_as_float(a[i]) : __uint_as_float(a[i]);
    };
    // Hand dQ(gq)'s rows cg*32.. (this half) to the reduction warp through
    // this half's staging tile [32 q][D] fp32, once the reduction has read
    // the half's previous tile out of it.
    auto stage_dq = [&](int gq, const float (&v)[HALF]) {
      if (gq >= 1 && !mbar_wait_warp<kBwdSuspend>(smem_u32(&bar_stg_free[cg]), (gq - 1) & 1, ctl))
        return false;
      if (r < D) {
#pragma unroll
        for (int i = 0; i < HALF; ++i) stg[i * D + r] = v[i];
      }
      fence_async_smem();
      mbar_arrive(smem_u32(&bar_stg_full[cg]));
      return true;
    };
    int git = 0;
    for (int ii = 0; ok && (PERSIST || ii == 0); ++ii) {
      const int code = item_code(ii);
      if (code < 0) {
        ok = code == -1;
        break;
      }
      const BwdItem t = bwd_item<WIN>(p, code, BQ, BK);
      const int key = t.k0 + r;
      const bool key_valid = key < p.S;
      for (int it = 0; it < t.n_it; ++it) {
        const int gi = git + it;
        const int s = gi % ST;
        const int q0 = bwd_qtile(t, it) * BQ;
        ATTN_TRACE_EV(tc, 1, gi);
        ok = mbar_wait_warp<kBwdSuspend>(smem_u32(&bar_sdp_full), gi & 1, ctl);
        if (ok) ok = mbar_wait_warp<kBwdSuspend>(smem_u32(&bar_st_full[s]), (gi / ST) & 1, ctl);
        if (!ok) break;
        tc_fence_after();
        // This warpgroup's query columns of -LSE*log2(e) and Dvec, four at a time.
        const float4* nl4 = reinterpret_cast<const float4*>(stage_rows(s) + cg * HALF);
        const float4* dv4 = reinterpret_cast<const float4*>(stage_rows(s) + BQ + cg * HALF);
        // Only tiles that cross the causal diagonal, hold keys past S, or hold
        // keys below some row's window mask.
        const bool need_mask = (p.causal && (q0 < t.k0 + BK - 1)) || (t.k0 + BK > p.S) ||
                               (WIN && t.k0 <= q0 + BQ - 1 - p.window);
        uint32_t us[HALF], ud[HALF];
        tmem_ld32(tmem + lane_base + C::TM_ST + cg * HALF, us);
        tmem_ld32(tmem + lane_base + C::TM_DPT + cg * HALF, ud);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(smem_u32(&bar_sdp_free));
        ATTN_TRACE_EV(tc, 2, gi);  // S^T, dP^T loaded
        // bf16 pairs of this half's 32 query columns: P hi then P lo, dS hi then dS lo.
        uint32_t pp[HALF], dd[HALF];
        // P = exp2(S * scale*log2(e) - LSE*log2(e)); dS = scale * P * (dP - Dvec),
        // two query columns per packed instruction.
        const uint64_t sl2 = f32x2(p.scale_log2, p.scale_log2);
        const uint64_t sc2 = f32x2(p.scale, p.scale);
        // Key position relative to this half's first query row, and the first
        // query column past the key's window (no window: never).
        const int rel = key - (q0 + cg * HALF);
        const int relw = WIN ? rel + p.window : (1 << 30);
        auto p_ds = [&](auto masked) {
#pragma unroll
          for (int c = 0; c < HALF; c += 4) {
            const float4 nl = nl4[c / 4];
            const float4 dv = dv4[c / 4];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int cc = c + 2 * h;  // columns cc, cc + 1 of this half
              float x0, x1;
              unpack_f32x2(fma_f32x2(f32x2(__uint_as_float(us[cc]), __uint_as_float(us[cc + 1])), sl2,
                                     h ? f32x2(nl.z, nl.w) : f32x2(nl.x, nl.y)),
                           x0, x1);
              float p0 = ex2(x0), p1 = ex2(x1);
              // Query column cc of this half sees the key iff rel <= cc
              // (causal) and cc < rel + W (window); rel, relw above.
              constexpr int MODE = decltype(masked)::value;
              if (MODE == 1) {  // every condition
                if (!key_valid || (p.causal && cc < rel) || cc >= relw) p0 = 0.f;
                if (!key_valid || (p.causal && cc + 1 < rel) || cc + 1 >= relw) p1 = 0.f;
              } else if (MODE == 2) {  // the causal side only
                if (cc < rel) p0 = 0.f;
                if (cc + 1 < rel) p1 = 0.f;
              } else if (MODE == 3) {  // the window side only
                if (cc >= relw) p0 = 0.f;
                if (cc + 1 >= relw) p1 = 0.f;
              }
              const uint64_t dpv = sub_f32x2(f32x2(__uint_as_float(ud[cc]), __uint_as_float(ud[cc + 1])),
                                             h ? f32x2(dv.z, dv.w) : f32x2(dv.x, dv.y));
              float d0, d1;
              unpack_f32x2(mul_f32x2(mul_f32x2(f32x2(p0, p1), sc2), dpv), d0, d1);
              split_bf16x2(p0, p1, pp[cc / 2], pp[HALF / 2 + cc / 2]);
              split_bf16x2(d0, d1, dd[cc / 2], dd[HALF / 2 + cc / 2]);
            }
          }
        };
        // Mask modes, decided per warp: 0 none, 1 every condition, 2 the
        // causal side only (the diagonal tiles), 3 the window's far side only.
        int mode = 0;
        if (need_mask) {
          const bool all_valid = __all_sync(0xffffffffu, key_valid);
          const bool c_side = p.causal && __any_sync(0xffffffffu, rel > 0);
          const bool w_side = WIN && __any_sync(0xffffffffu, relw < HALF);
          mode = (!all_valid || (c_side && w_side)) ? 1 : c_side ? 2 : w_side ? 3 : 0;
        }
        if (mode == 0)
          p_ds(std::integral_constant<int, 0>{});
        else if (mode == 2)
          p_ds(std::integral_constant<int, 2>{});
        else if (WIN && mode == 3)
          p_ds(std::integral_constant<int, 3>{});
        else
          p_ds(std::integral_constant<int, 1>{});
        ATTN_TRACE_EV(tc, 3, gi);  // P, dS computed
        // pds_free(gi-1): the MMAs of iteration gi-1 are done, so dS^T in
        // shared memory is free and dQ^T(gi-1) is complete in TMEM. With
        // D = 64 this thread reads its part of dQ^T(gi-1) (lane = head dim d,
        // this half's query columns) before storing P/dS(gi) over those same
        // TMEM cells; the item's last dQ^T is read after its loop.
        float dqv[HALF];
        if (gi >= 1) {
          ok = mbar_wait_warp<kBwdSuspend>(smem_u32(&bar_pds_free), (gi - 1) & 1, ctl);
          if (!ok) break;
        }
        // Row r of dS^T, K-major with 128-byte swizzle: 64 query columns per
        // 128-byte row, 8 per 16-byte unit; this half owns units cg*4..cg*4+3.
#pragma unroll
        for (int u = 0; u < HALF / 8; ++u) {
          const int unit = cg * (HALF / 8) + u;
          const uint32_t* h = dd + u * 4;
          const uint32_t* lo = dd + HALF / 2 + u * 4;
          st_sw128(sDsHi, r, unit, make_uint4(h[0], h[1], h[2], h[3]));
          st_sw128(sDsLo, r, unit, make_uint4(lo[0], lo[1], lo[2], lo[3]));
        }
        ATTN_TRACE_EV(tc, 4, gi);  // previous MMAs done
        if constexpr (!C::DQ_IN_COMPUTE) {
          // The drain warps hand back the dQ^T(gi-1) columns.
          if (gi >= 1) {
            ok = mbar_wait_warp<kBwdSuspend>(smem_u32(&bar_dq_free), (gi - 1) & 1, ctl);
            if (!ok) break;
          }
        }
        tc_fence_after();
        if (C::DQ_IN_COMPUTE && it >= 1) read_dq_part(0, dqv, false);
        tmem_st32(tmem + lane_base + C::TM_P + cg * HALF, pp);
        if (C::DQ_IN_COMPUTE && it >= 1) read_dq_part(1, dqv, true);
        tmem_st32(tmem + lane_base + C::TM_DS + cg * HALF, dd);
        tmem_wait_st();
        fence_async_smem();
        tc_fence_before();
        mbar_arrive(smem_u32(&bar_pds_full));
        ATTN_TRACE_EV(tc, 5, gi);  // P, dS stored and signalled
        if (C::DQ_IN_COMPUTE && it >= 1) {
          ok = stage_dq(gi - 1, dqv);
          if (!ok) break;
        }
      }
      if (!ok) break;
      // The item's last dQ^T, once its MMA has run.
      if (C::DQ_IN_COMPUTE && t.n_it > 0) {
        const int gl = git + t.n_it - 1;
        ok = mbar_wait_warp<kBwdSuspend>(smem_u32(&bar_pds_free), gl & 1, ctl);
        if (ok) {
          tc_fence_after();
          float dqv[HALF];
          read_dq_part(0, dqv, false);
          read_dq_part(1, dqv, true);
          ok = stage_dq(gl, dqv);
        }
        if (!ok) break;
      }
      ok = mbar_wait_warp<kBwdSuspend>(smem_u32(&bar_mma_done), ii & 1, ctl);
      if (!ok) break;
      // dK and dV rows in fp32; this warpgroup stores columns [cg*D/2, (cg+1)*D/2).
      const size_t rowoff = ((static_cast<size_t>(t.b) * p.S + key) * p.Hkv + t.g) * D;
      {
        // (warp-uniform outcome: the TMEM loads below are .sync.aligned)
        const bool row_in =
            !key_valid || bounds_ok(rowoff + D <= static_cast<size_t>(p.B) * p.S * p.Hkv * D, ctl);
        if (!__all_sync(0xffffffffu, row_in)) ok = false;
      }
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int tt = 0; tt < 2; ++tt) {
        const uint32_t col0 = (tt == 0 ? C::TM_DK : C::TM_DV) + cg * (D / 2);
        float* dst = (tt == 0 ? p.dk : p.dv) + rowoff + cg * (D / 2);
#pragma unroll
        for (int c = 0; c < D / 2; c += 32) {
          uint32_t u[32];
          tmem_ld32(tmem + lane_base + col0 + c, u);
          tmem_wait_ld();
          if (tt == 1 && c + 32 >= D / 2) {
            // The last read of this thread's dK/dV cells: the next item's
            // first dV/dK products may overwrite them.
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_dkv_free));
          }
          if (key_valid) {
            if (p.split > 1) {
              // Two CTAs add their head halves into the zeroed row: two
              // additions onto zero give the same sum in either order.
#pragma unroll
              for (int i = 0; i < 8; ++i)
                red_add_v4(dst + c + 4 * i, __uint_as_float(u[4 * i]), __uint_as_float(u[4 * i + 1]),
                           __uint_as_float(u[4 * i + 2]), __uint_as_float(u[4 * i + 3]));
            } else {
              float4* d4 = reinterpret_cast<float4*>(dst + c);
#pragma unroll
              for (int i = 0; i < 8; ++i)
                d4[i] = make_float4(__uint_as_float(u[4 * i]), __uint_as_float(u[4 * i + 1]),
                                    __uint_as_float(u[4 * i + 2]), __uint_as_float(u[4 * i + 3]));
            }
          }
        }
      }
      git += t.n_it;
    }
#ifdef ATTN_TRACE
  } else if (warp == C::W_MMA + 1) {
    // ------------------------------------------------------------ trace observer
    // Timestamps the completion of S^T/dP^T (1), dV/dK (2) and dQ^T (3) of
    // every iteration by polling their barriers without blocking.
    TraceCursor tc;
    if (lane == 0) ATTN_TRACE_INIT(tc, 14);
    auto done = [](uint32_t bar, uint32_t parity) {
      uint32_t ok;
      asm volatile(
          "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
          "selp.u32 %0, 1, 0, p;\n\t}"
          : "=r"(ok)
          : "r"(bar), "r"(parity)
          : "memory");
      return ok != 0;
    };
    // Runs until the MMA warp has published its iteration count and every
    // iteration has been seen (or the CTA aborts, or 2 s pass).
    int i1 = 0, i2 = 0, i3 = 0;
    const uint64_t t0 = globaltimer();
    for (;;) {
      const int total = reinterpret_cast<volatile int*>(&trace_iters)[0];
      if (total >= 0 && i1 >= total && i2 >= total && i3 >= total) break;
      if ((total < 0 || i1 < total) && done(smem_u32(&bar_sdp_full), i1 & 1)) ATTN_TRACE_EV(tc, 1, i1++);
      if ((total < 0 || i2 < total) && done(smem_u32(&bar_st_empty[i2 % ST]), (i2 / ST) & 1))
        ATTN_TRACE_EV(tc, 2, i2++);
      if ((total < 0 || i3 < total) && done(smem_u32(&bar_pds_free), i3 & 1)) ATTN_TRACE_EV(tc, 3, i3++);
      if (abort_flag || globaltimer() - t0 > 2000000000ull) break;
    }
#endif
  } else if (C::DQ_IN_COMPUTE) {
    // ------------------------------------------------------------ dQ reduction warp
    // Adds each staged half tile of dQ into dq with an fp32 TMA reduction,
    // then hands the staging tile back once the reduction has read it.
    bool ok = true;
    TraceCursor tc;
    if (lane == 0) ATTN_TRACE_INIT(tc, 10);
    int git = 0;
    for (int ii = 0; ok && (PERSIST || ii == 0); ++ii) {
      const int code = item_code(ii);
      if (code < 0) {
        ok = code == -1;
        break;
      }
      const BwdItem t = bwd_item<WIN>(p, code, BQ, BK);
      // Half 0 of each tile, then half 1; each half's staging tile cycles
      // through its own pair of barriers.
      for (int n = 0; n < 2 * t.n_it && ok; ++n) {
        const int it = n >> 1, half = n & 1;
        const int gq = git + it;
        ok = mbar_wait_warp<kBwdSuspend>(smem_u32(&bar_stg_full[half]), gq & 1, ctl);
        if (!ok) break;
        ATTN_TRACE_EV(tc, 1, 2 * gq + half);  // half staged
        if (lane == 0) {
          const int h = bwd_head(t, it);
          const int q0 = bwd_qtile(t, it) * BQ;
          if (bounds_ok(h < p.Hq && q0 + (half + 1) * C::DQ_ROWS <= p.S_pad, ctl))
            tma_reduce_add_4d(&tm_dq, 0, h, q0 + half * C::DQ_ROWS, t.b, sDQS + half * C::DQS_BYTES);
          bulk_commit_group();
          bulk_wait_read_all();
          mbar_arrive(smem_u32(&bar_stg_free[half]));
        }
        __syncwarp();
      }
      git += t.n_it;
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  } else {
    // ------------------------------------------------------------ dQ drain warps 8-11
    const int tid = threadIdx.x - 256;  // TMEM lane = head-dim index d of dQ^T
    const uint32_t lane_base = static_cast<uint32_t>((warp % 4) * 32) << 16;
    bool ok = true;
    TraceCursor tc;
    if (lane == 0) ATTN_TRACE_INIT(tc, 10 + (warp - 8));
    int git = 0;
    for (int ii = 0; ok && (PERSIST || ii == 0); ++ii) {
      const int code = item_code(ii);
      if (code < 0) {
        ok = code == -1;
        break;
      }
      const BwdItem t = bwd_item<WIN>(p, code, BQ, BK);
      for (int it = 0; it < t.n_it; ++it) {
        const int gi = git + it;
        const int h = bwd_head(t, it);
        const int q0 = bwd_qtile(t, it) * BQ;
        ok = mbar_wait_warp<kBwdSuspend>(smem_u32(&bar_dq_full), gi & 1, ctl);
        // The four drain warps meet at bar.sync below: agree first on going on.
        ok = named_bar_and(1, 128, ok);
        if (!ok) break;
        ATTN_TRACE_EV(tc, 1, gi);  // dQ landed
        tc_fence_after();
        // dQ^T = hi part (columns 0..63) + lo part (64..127).
        float u[BQ];
#pragma unroll
        for (int c = 0; c < BQ; c += 32) {
          uint32_t a[32], bl[32];
          tmem_ld32(tmem + lane_base + C::TM_DQ + c, a);
          tmem_ld32(tmem + lane_base + C::TM_DQ + BQ + c, bl);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) u[c + i] = __uint_as_float(a[i]) + __uint_as_float(bl[i]);
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&bar_dq_free));
        ATTN_TRACE_EV(tc, 3, gi);  // dQ^T read, TMEM handed back
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          if (tid == 0) bulk_wait_read_all();  // the previous reduction has read the staging tile
          named_bar_sync(1, 128);
          float* stg = reinterpret_cast<float*>(smem + C::SMEM_DQS);
          if (tid < D) {
            // staging [32 q][D] fp32, row-major (the TMA box layout); lane tid holds column d = tid.
#pragma unroll
            for (int q = 0; q < C::DQ_ROWS; ++q) stg[q * D + tid] = u[half * C::DQ_ROWS + q];
          }
          fence_async_smem();
          named_bar_sync(1, 128);
          if (tid == 0 && bounds_ok(h < p.Hq && q0 + (half + 1) * C::DQ_ROWS <= p.S_pad, ctl)) {
            tma_reduce_add_4d(&tm_dq, 0, h, q0 + half * C::DQ_ROWS, t.b, sDQS);
            bulk_commit_group();
          }
        }
        ATTN_TRACE_EV(tc, 2, gi);  // both halves handed to the reduction
      }
      git += t.n_it;
    }
    if (tid == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::W_MMA) tmem_dealloc(tmem, C::TMEM_COLS);
#ifdef ATTN_TRACE
  if (threadIdx.x == 0) {
    const unsigned lin = blockIdx.y * gridDim.x + blockIdx.x;
    if (lin < kSpanCtas) {
      unsigned smid;
      asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
      const int total = trace_iters;
      g_attn_spans[4 * lin] = t_entry;
      g_attn_spans[4 * lin + 1] = globaltimer();
      g_attn_spans[4 * lin + 2] = smid;
      g_attn_spans[4 * lin + 3] = total;
    }
  }
#endif
}

// The grid launch's head split (CTAs per key tile, 1 or 2): 2 splits the
// group's query heads in halves, so the longest key tiles, which the grid
// starts first but which end last, take half as long. It pays only where that
// tail is a large part of the run and the extra prologue/epilogue per key
// tile and the zeroing of dk/dv are small against a CTA's work: measured
// (same-box A/B, causal, D = 128) 3-5% faster at B = 1, Hq = 64, Hkv = 8,
// S = 8192 (512 CTAs unsplit, 1024 iterations in the longest); 0-1% slower at
// B = 2, Hq = 32, S = 4096 (256 iterations), and 1-3% slower at S = 16384 and
// 32768 (1024 and 2048 CTAs). Hence: an even group, at least 512 (head,
// query tile) iterations in the longest CTA, and at most four waves.
int bwd_grid_split(const BwdParams& p, int bq, int sms) {
  const int nq = (p.S + bq - 1) / bq;
  const int niq0 = p.window > 0 ? std::min(nq, (128 + p.window - 2) / bq + 1) : nq;
  const long long ctas = static_cast<long long>(p.B) * p.Hkv * p.n_ktiles;
  return (p.G % 2 == 0 && p.G * niq0 >= 512 && ctas <= 4LL * sms) ? 2 : 1;
}

template <int D, bool WIN, bool PERSIST>
cudaError_t set_bwd_smem(int dev) {
  static bool attr_set[64] = {};
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_main_kernel<D, WIN, PERSIST>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         BwdCfg<D>::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  return cudaSuccess;
}

// Items of at most this many (head, query tile) iterations on average run on
// a persistent grid (one CTA per SM taking items from the work counter): a
// CTA's own prologue and epilogue (about 9 us at D = 128 against 1.8 us per
// iteration) then outweigh what a launch of one CTA per item gives. Measured
// (same-box A/B): persistent 7% faster at D = 64, B = 8, H = 16, S = 2048 (16
// iterations per item) and 6% faster with a 128-key window at D = 128 (32
// per item); 3% slower at the Llama-3-8B, 70B and S = 32768 shapes (132 to
// 1028 per item), where the grid launch of one CTA per item stays.
constexpr int kBwdPersistMaxMeanIters = 64;

template <int D, bool WIN>
cudaError_t launch_bwd_main_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdParams& p,
                              cudaStream_t stream) {
  using C = BwdCfg<D>;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  BwdParams pp = p;
  pp.split = bwd_grid_split(p, C::BQ, sms);
  const int per_tile = p.B * p.Hkv * pp.split;  // items per key tile
  pp.n_items = per_tile * p.n_ktiles;
  pp.work = p.status + kBwdWorkWord;
  // Iterations of all items: those of the first item of each key tile (all
  // items of a key tile have the same count) times the items per key tile.
  long long total = 0;
  for (int j = 0; j < p.n_ktiles; ++j) total += bwd_item<WIN>(pp, j * per_tile, C::BQ, C::BK).n_it;
  total *= per_tile;
  const bool persist = total <= static_cast<long long>(kBwdPersistMaxMeanIters) * pp.n_items;
  if (pp.split > 1) {
    const long long n4 = static_cast<long long>(p.B) * p.S * p.Hkv * D / 4;
    zero_f32x4_kernel<<<4 * sms, 256, 0, stream>>>(reinterpret_cast<float4*>(p.dk),
                                                   reinterpret_cast<float4*>(p.dv), n4);
  }
  if (persist) {
    cudaError_t e = set_bwd_smem<D, WIN, true>(dev);
    if (e != cudaSuccess) return e;
    const int grid = pp.n_items < sms ? pp.n_items : sms;
    attn_bwd_main_kernel<D, WIN, true><<<grid, C::THREADS, C::SMEM_ALLOC, stream>>>(tq, tk, tv, tdo, tdq, pp);
    return cudaGetLastError();
  }
  cudaError_t e = set_bwd_smem<D, WIN, false>(dev);
  if (e != cudaSuccess) return e;
  const dim3 grid(per_tile, p.n_ktiles);
  attn_bwd_main_kernel<D, WIN, false><<<grid, C::THREADS, C::SMEM_ALLOC, stream>>>(tq, tk, tv, tdo, tdq, pp);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_preprocess(const __nv_bfloat16* o, const __nv_bfloat16* o_lo,
                                  const __nv_bfloat16* dO, const float* lse, float* nlse2,
                                  float* dvec, float* dq, int* status, int B, int Hq, int S,
                                  int D, cudaStream_t stream) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // Eight 256-thread blocks per SM: about two waves at the kernel's register
  // use (measured faster than one wave of four, or one of six).
  const int nblk = 8 * sms;
  const int S_pad = seq_pad(S);
  if (D == 128)
    attn_bwd_preprocess_kernel<128><<<nblk, 256, 0, stream>>>(
        o, o_lo, dO, lse, nlse2, dvec, reinterpret_cast<float4*>(dq), status, B, Hq, S, S_pad);
  else
    attn_bwd_preprocess_kernel<64><<<nblk, 256, 0, stream>>>(
        o, o_lo, dO, lse, nlse2, dvec, reinterpret_cast<float4*>(dq), status, B, Hq, S, S_pad);
  return cudaGetLastError();
}

cudaError_t launch_bwd_main(int D, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                            const BwdParams& p, cudaStream_t stream) {
  const bool win = p.window > 0;
  if (D == 128)
    return win ? launch_bwd_main_t<128, true>(tq, tk, tv, tdo, tdq, p, stream)
               : launch_bwd_main_t<128, false>(tq, tk, tv, tdo, tdq, p, stream);
  return win ? launch_bwd_main_t<64, true>(tq, tk, tv, tdo, tdq, p, stream)
             : launch_bwd_main_t<64, false>(tq, tk, tv, tdo, tdq, p, stream);
}

}  // namespace attn

#ifdef ATTN_TRACE
// Trace build only: copies the backward main kernel's per-CTA spans out and clears them.
extern "C" int attn_trace_copy_spans(void* host, size_t bytes) {
  const size_t total = sizeof(attn::g_attn_spans);
  if (bytes < total) return 1;
  if (cudaDeviceSynchronize() != cudaSuccess) return 3;
  if (cudaMemcpyFromSymbol(host, attn::g_attn_spans, total) != cudaSuccess) return 3;
  static unsigned long long zeros[4096];
  for (size_t off = 0; off < total; off += sizeof(zeros))
    if (cudaMemcpyToSymbol(attn::g_attn_spans, zeros, sizeof(zeros), off) != cudaSuccess) return 3;
  return 0;
}
// Trace build only: copies the backward main kernel's timeline records out and clears them.
extern "C" int attn_trace_copy_bwd(void* host, size_t bytes) {
  const size_t total = sizeof(attn::g_attn_trace);
  if (bytes < total) return 1;
  if (cudaDeviceSynchronize() != cudaSuccess) return 3;
  if (cudaMemcpyFromSymbol(host, attn::g_attn_trace, total) != cudaSuccess) return 3;
  static unsigned long long zeros[4096];
  for (size_t off = 0; off < total; off += sizeof(zeros))
    if (cudaMemcpyToSymbol(attn::g_attn_trace, zeros, sizeof(zeros), off) != cudaSuccess) return 3;
  return 0;
}
#endif
