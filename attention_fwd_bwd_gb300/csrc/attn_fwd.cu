// Forward attention kernel for sm_103a: O = softmax(scale * Q K^T) V and the
// row log-sum-exp, per (batch, query head) -- "Scheduling Data to Compute:
// Hierarchical Data Pipelining for LLM Training on AMD GPUs", section 2.1,
// Eq. (1), computed as that section's Algorithm 0 describes (K/V tiles stream
// through on-chip memory, online softmax, output accumulator kept on chip),
// with the query-tile loop outside and the key/value loop inside so the state
// never leaves the SM.
//
// Per CTA (one 128-row query tile of one head):
//   warp 4 (TMA producer): Q once, then K_0, V_0, K_1, V_1, ... into a ring of
//       shared-memory slots, each slot guarded by a full/empty mbarrier pair
//       (the GB300 counterpart of the paper's "issue N+1 loads, wait until at
//       most N are outstanding" rule for its Tensor Data Mover, section 3.1.1).
//   warp 5 (MMA issuer): S_j = Q K_j^T into one of two TMEM score buffers
//       (both operands K-major, so K^T needs no transpose -- Table 3's first
//       row), then O += P_j V_j with P read from TMEM and V_j described
//       MN-major (the transposed-operand case of section 3.1.2, handled by
//       the descriptor instead of a transpose).
//   warps 0-3 (softmax): thread r owns query row r (TMEM lane r); it reads its
//       score row, updates the running max m and sum l, writes bf16 P to TMEM
//       and, when m grew by more than 2^8, rescales its O row in TMEM first.
//       The final m and l give O = acc / l and LSE = (m + log2 l) ln 2.
// When the caller asks for the output residual o_lo = bf16(O - o) (training,
// where the backward needs rowsum(dO * O) beyond bf16 accuracy), P is split
// into bf16 hi (P truncated) and lo (the truncated residual) parts and goes
// through a second MMA, O += P_lo V_j, so O carries about 16 significant bits.
#include "attn_common.cuh"
#include "sm100_ptx.cuh"

namespace attn {
using namespace ptx;

namespace {

#ifdef ATTN_TRACE
static __device__ unsigned long long g_attn_trace[kTraceCtas * kTraceRoles * kTraceEvents];
#endif

// Rescale threshold in log2 units: the running max used for exponentiation
// only moves when the true max exceeds it by more than this, which keeps every
// p <= 2^8 and leaves the result exact after the final division by l.
constexpr float kRescaleThreshold = 8.0f;

template <int D, bool SPLIT>
__global__ void __launch_bounds__(FwdCfg<D>::THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  __shared__ uint64_t bar_q_full;
  __shared__ uint64_t bar_kv_full[C::NSLOT], bar_kv_empty[C::NSLOT];
  __shared__ uint64_t bar_s_full[2], bar_p_full[2], bar_pv_done[2];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  const int bh = blockIdx.x;  // b * Hq + hq
  const int hq = bh % p.Hq;
  const int b = bh / p.Hq;
  const int g = hq / p.G;
  const int qt = p.n_qtiles - 1 - static_cast<int>(blockIdx.y);  // longest causal rows first
  const int q0 = qt * C::BQ;
  const int nkv_all = (p.S + C::BK - 1) / C::BK;
  const int n_kv = p.causal ? min(qt + 1, nkv_all) : nkv_all;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar_q_full), 1);
    for (int i = 0; i < C::NSLOT; ++i) {
      mbar_init(smem_u32(&bar_kv_full[i]), 1);
      mbar_init(smem_u32(&bar_kv_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bar_s_full[i]), 1);
      mbar_init(smem_u32(&bar_p_full[i]), 128);
      mbar_init(smem_u32(&bar_pv_done[i]), 1);
    }
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(&tmem_base_s), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  const WaitCtl ctl{&abort_flag, p.status, p.timeout_ns};
  // SPLIT (the residual output o_lo is requested): P enters O += P V as a
  // bf16 hi/lo pair, so O (and o + o_lo) carries about 16 significant bits.
  constexpr bool split = SPLIT;

  const uint32_t sQ = smem_u32(smem + C::SMEM_Q);
  const uint32_t sRing = smem_u32(smem + C::SMEM_RING);

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    // The whole warp runs this loop; each copy is issued by one elected lane.
    TraceCursor tc;
    if (lane == 0) ATTN_TRACE_INIT(tc, 0);
    ATTN_TRACE_EV(tc, 1, 0);
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
    }
    const uint64_t keep = policy_evict_last();  // K/V tiles are re-read by G heads x tiles
    mbar_arrive_expect_tx_el(smem_u32(&bar_q_full), C::Q_BYTES);
    for (int c = 0; c < C::KCH; ++c)
      tma_load_4d_el(sQ + c * (C::BQ * 128), &tm_q, smem_u32(&bar_q_full), c * 64, hq, q0, b);
    int issued = 0;
    bool ok = true;
    for (int idx = 0; idx < 2 * n_kv; ++idx) {
      const int slot = idx % C::NSLOT, round = idx / C::NSLOT;
      if (round > 0) ok = mbar_wait_warp(smem_u32(&bar_kv_empty[slot]), (round - 1) & 1, ctl);
      if (!ok) break;
      ATTN_TRACE_EV(tc, 2, idx);  // slot free, issuing the load
      const uint32_t full = smem_u32(&bar_kv_full[slot]);
      const uint32_t dst = sRing + slot * C::KV_BYTES;
      const CUtensorMap* m = (idx & 1) ? &tm_v : &tm_k;
      mbar_arrive_expect_tx_el(full, C::KV_BYTES);
      for (int c = 0; c < C::KCH; ++c)
        tma_load_4d_hint_el(dst + c * (C::BK * 128), m, full, c * 64, g, (idx >> 1) * C::BK, b,
                            keep);
      issued = idx + 1;
    }
    if (!ok && lane == 0) {
      // Let in-flight copies land before the CTA's shared memory goes away.
      for (int idx = max(0, issued - C::NSLOT); idx < issued; ++idx)
        mbar_wait_drain(smem_u32(&bar_kv_full[idx % C::NSLOT]), (idx / C::NSLOT) & 1,
                        50000000ull);
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop and builds the (warp-uniform) descriptors;
    // each MMA and commit is issued by one elected lane.
    TraceCursor tc;
    if (lane == 0) ATTN_TRACE_INIT(tc, 1);
    bool ok = mbar_wait_warp(smem_u32(&bar_q_full), 0, ctl);
    if (ok) {
      ATTN_TRACE_EV(tc, 1, 0);
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, 0, 1);
      const uint64_t dq_desc = sw128_desc(sQ, 16, 1024);
      for (int j = 0; j <= n_kv; ++j) {
        if (j < n_kv) {
          const int idx = 2 * j, slot = idx % C::NSLOT;
          ok = mbar_wait_warp(smem_u32(&bar_kv_full[slot]), (idx / C::NSLOT) & 1, ctl);
          if (!ok) break;
          tc_fence_after();
          const uint64_t dk = sw128_desc(sRing + slot * C::KV_BYTES, 16, 1024);
          const uint32_t d_s = tmem + ((j & 1) ? C::TM_S1 : C::TM_S0);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = ((kk >> 2) * (128 * 128) + (kk & 3) * 32) >> 4;
            mma_ss_el(d_s, dq_desc + koff, dk + koff, idesc_s, kk > 0);
          }
          mma_commit_el(smem_u32(&bar_s_full[j & 1]));
          mma_commit_el(smem_u32(&bar_kv_empty[slot]));
          ATTN_TRACE_EV(tc, 3, j);  // S_j issued
        }
        if (j >= 1) {
          const int jj = j - 1, pb = jj & 1;
          ok = mbar_wait_warp(smem_u32(&bar_p_full[pb]), (jj >> 1) & 1, ctl);
          if (!ok) break;
          ATTN_TRACE_EV(tc, 4, jj);  // P_jj ready seen
          const int idx = 2 * jj + 1, slot = idx % C::NSLOT;
          ok = mbar_wait_warp(smem_u32(&bar_kv_full[slot]), (idx / C::NSLOT) & 1, ctl);
          if (!ok) break;
          tc_fence_after();
          const uint64_t dv = sw128_desc(sRing + slot * C::KV_BYTES, C::BK * 128, 1024);
          const uint32_t a_p = tmem + (pb ? C::TM_P1 : C::TM_P0);
#pragma unroll
          for (int kk = 0; kk < C::BK / 16; ++kk) {
            mma_ts_el(tmem + C::TM_O, a_p + kk * 8, dv + ((kk * 2048) >> 4), idesc_o,
                      (jj > 0 || kk > 0) ? 1u : 0u);
          }
          if constexpr (SPLIT) {
            // O += P_lo V_j: the low-order bf16 part of P, stored over the
            // first 64 columns of the score buffer it was computed from.
            const uint32_t a_lo = tmem + (pb ? C::TM_S1 : C::TM_S0);
#pragma unroll
            for (int kk = 0; kk < C::BK / 16; ++kk)
              mma_ts_el(tmem + C::TM_O, a_lo + kk * 8, dv + ((kk * 2048) >> 4), idesc_o, 1u);
          }
          mma_commit_el(smem_u32(&bar_pv_done[pb]));
          mma_commit_el(smem_u32(&bar_kv_empty[slot]));
          ATTN_TRACE_EV(tc, 5, jj);  // PV_jj issued
        }
      }
      if (!ok) {
        // Wait for the MMAs already issued before TMEM is released. bar_q_full
        // has completed its only phase, so this commit completes phase 1.
        mma_commit_el(smem_u32(&bar_q_full));
        mbar_wait_drain(smem_u32(&bar_q_full), 1, 50000000ull);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warps 0-3
    const int r = threadIdx.x;  // query row within the tile == TMEM lane
    const int qrow = q0 + r;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    float m = -INFINITY;  // running max in log2 units (scaled scores)
    float l = 0.f;
    const float sl2 = p.scale_log2;
    const bool pos = sl2 >= 0.f;
    TraceCursor tc;
    if (lane == 0) ATTN_TRACE_INIT(tc, 2 + warp);
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int sb = j & 1;
      ATTN_TRACE_EV(tc, 1, j);  // start waiting for S_j
      ok = mbar_wait_warp(smem_u32(&bar_s_full[sb]), (j >> 1) & 1, ctl);
      if (!ok) break;
      ATTN_TRACE_EV(tc, 2, j);  // S_j landed
      tc_fence_after();
      // Raw scores of this row; the scale is folded into the exponent below.
      float x[C::BK];
      {
        const uint32_t ts = tmem + lane_base + (sb ? C::TM_S1 : C::TM_S0);
        uint32_t u[C::BK];
#pragma unroll
        for (int c = 0; c < C::BK; c += 32)
          tmem_ld32(ts + c, *reinterpret_cast<uint32_t(*)[32]>(&u[c]));
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < C::BK; ++c) x[c] = __uint_as_float(u[c]);
      }
      const int k0 = j * C::BK;
      const bool need_mask = (p.causal && k0 + C::BK - 1 > q0) || (k0 + C::BK > p.S);
      const int lim = p.causal ? min(qrow, p.S - 1) : (p.S - 1);  // last visible key
      // Largest scaled score: the max of the raw scores for scale >= 0, the min
      // for scale < 0 (masked keys pushed to the losing end).
      float mraw;
      {
        const float lose = pos ? -INFINITY : INFINITY;
        if (need_mask) {
#pragma unroll
          for (int c = 0; c < C::BK; ++c)
            if (k0 + c > lim) x[c] = lose;
        }
        float a[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] = x[i];
        if (pos) {
#pragma unroll
          for (int c = 8; c < C::BK; c += 8)
#pragma unroll
            for (int i = 0; i < 8; ++i) a[i] = fmaxf(a[i], x[c + i]);
#pragma unroll
          for (int w = 4; w > 0; w >>= 1)
#pragma unroll
            for (int i = 0; i < w; ++i) a[i] = fmaxf(a[i], a[i + w]);
        } else {
#pragma unroll
          for (int c = 8; c < C::BK; c += 8)
#pragma unroll
            for (int i = 0; i < 8; ++i) a[i] = fminf(a[i], x[c + i]);
#pragma unroll
          for (int w = 4; w > 0; w >>= 1)
#pragma unroll
            for (int i = 0; i < w; ++i) a[i] = fminf(a[i], a[i + w]);
        }
        mraw = a[0];
      }
      const float mx = mraw * sl2;
      float alpha = 1.f;
      const bool rescale = mx > m + kRescaleThreshold;
      if (rescale) {
        alpha = ex2(m - mx);  // m = -inf on the first tile gives 0
        m = mx;
      }
      const float neg_m = -m;
      // P buffer sb was last read by PV_{j-2}.
      if (j >= 2) {
        ok = mbar_wait_warp(smem_u32(&bar_pv_done[sb]), ((j - 2) >> 1) & 1, ctl);
        if (!ok) break;
      }
      float sums[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) sums[i] = 0.f;
      const uint32_t tp = tmem + lane_base + (sb ? C::TM_P1 : C::TM_P0);
      // With SPLIT, P_lo goes over columns 0..63 of this tile's score buffer,
      // whose scores this thread has already read; the next MMA to write that
      // buffer (S_{j+2}) issues after PV_j and tcgen05 MMAs run in issue order.
      const uint32_t tl = tmem + lane_base + (sb ? C::TM_S1 : C::TM_S0);
#pragma unroll
      for (int ch = 0; ch < C::BK; ch += 32) {
        uint32_t pk[16];
        uint32_t pl[SPLIT ? 16 : 1];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float p0 = ex2(fmaf(x[ch + c], sl2, neg_m));
          float p1 = ex2(fmaf(x[ch + c + 1], sl2, neg_m));
          if (need_mask) {
            if (k0 + ch + c > lim) p0 = 0.f;
            if (k0 + ch + c + 1 > lim) p1 = 0.f;
          }
          sums[(c / 2) & 7] += p0 + p1;
          if constexpr (SPLIT) {
            split_bf16x2_trunc(p0, p1, pk[c / 2], pl[c / 2]);
          } else {
            pk[c / 2] = pack_bf16x2(p0, p1);
          }
        }
        tmem_st16(tp + ch / 2, pk);
        if constexpr (SPLIT) tmem_st16(tl + ch / 2, *reinterpret_cast<uint32_t(*)[16]>(&pl[0]));
      }
#pragma unroll
      for (int w = 4; w > 0; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) sums[i] += sums[i + w];
      const float sum = sums[0];
      l = l * alpha + sum;
      ATTN_TRACE_EV(tc, 3, j);  // exponentials done
      // Rescale this warp's O rows once PV_{j-1} has landed in TMEM.
      if (j >= 1 && __any_sync(0xffffffffu, rescale)) {
        ok = mbar_wait_warp(smem_u32(&bar_pv_done[(j - 1) & 1]), ((j - 1) >> 1) & 1, ctl);
        if (!ok) break;
        tc_fence_after();
        const uint32_t to = tmem + lane_base + C::TM_O;
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t u[32];
          tmem_ld32(to + c, u);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha);
          tmem_st32(to + c, u);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(smem_u32(&bar_p_full[sb]));
      ATTN_TRACE_EV(tc, 4, j);  // P_j stored and signalled
    }
    if (ok && n_kv > 0) {
      const int jl = n_kv - 1;
      ok = mbar_wait_warp(smem_u32(&bar_pv_done[jl & 1]), (jl >> 1) & 1, ctl);
    }
    if (ok) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      const bool valid = qrow < p.S;
      const size_t rowoff = ((static_cast<size_t>(b) * p.S + qrow) * p.Hq + hq) * D;
      const uint32_t to = tmem + lane_base + C::TM_O;
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        uint32_t u[32];
        tmem_ld32(to + c, u);
        tmem_wait_ld();
        uint4 w[4], wl[4];
        uint32_t* wp = reinterpret_cast<uint32_t*>(w);
        uint32_t* wlp = reinterpret_cast<uint32_t*>(wl);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float x0 = __uint_as_float(u[2 * i]) * inv_l;
          const float x1 = __uint_as_float(u[2 * i + 1]) * inv_l;
          wp[i] = pack_bf16x2(x0, x1);
          // what bf16 rounding dropped, itself rounded to bf16
          wlp[i] = pack_bf16x2(x0 - __uint_as_float(wp[i] << 16),
                               x1 - __uint_as_float(wp[i] & 0xFFFF0000u));
        }
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(p.o + rowoff + c);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = w[i];
          if (p.o_lo) {
            uint4* dl = reinterpret_cast<uint4*>(p.o_lo + rowoff + c);
#pragma unroll
            for (int i = 0; i < 4; ++i) dl[i] = wl[i];
          }
        }
      }
      if (valid)
        p.lse[(static_cast<size_t>(b) * p.Hq + hq) * p.S + qrow] = (m + __log2f(l)) * kLn2;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int D, bool SPLIT>
cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const FwdParams& p, cudaStream_t stream) {
  using C = FwdCfg<D>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D, SPLIT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  dim3 grid(p.B * p.Hq, p.n_qtiles);
  attn_fwd_kernel<D, SPLIT><<<grid, C::THREADS, C::SMEM_ALLOC, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(int D, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdParams& p, cudaStream_t stream) {
  const bool split = p.o_lo != nullptr;
  if (D == 128)
    return split ? launch_fwd_t<128, true>(tq, tk, tv, p, stream)
                 : launch_fwd_t<128, false>(tq, tk, tv, p, stream);
  return split ? launch_fwd_t<64, true>(tq, tk, tv, p, stream)
               : launch_fwd_t<64, false>(tq, tk, tv, p, stream);
}

}  // namespace attn

#ifdef ATTN_TRACE
// Trace build only: copies the forward kernel's timeline records out and clears them.
extern "C" int attn_trace_copy_fwd(void* host, size_t bytes) {
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
