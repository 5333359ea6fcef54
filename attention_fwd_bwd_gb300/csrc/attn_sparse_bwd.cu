// Sparse top-k gather attention, backward, for sm_103a ("Scheduling Data to
// Compute: Hierarchical Data Pipelining for LLM Training on AMD GPUs", section
// 2.1: the backward gathers the same sparse vectors to form dQ, produces a
// per-slot intermediate for dKV and reduces it through the inverse of the
// top-k map). The gradient of sum(dO * O) for
// O[t, h] = softmax_j(scale * q[t, h] . kp[idx[t, j]]) vp[idx[t, j]]:
//   P = softmax, dP = dO V^T, Dvec = rowsum(dO * O), dS = P * (dP - Dvec),
//   dq = scale * dS K, per-slot dK = scale * dS^T Q and dV = P^T dO,
//   dkp / dvp of a pool row = sum of the per-slot terms of every slot naming it.
//
// Two kernels on one stream:
//   1. preprocess: Dvec from o (+ o_lo) and dO, -LSE*log2(e) per (token, head),
//      and zeroed dkp / dvp (HBM-bound).
//   2. main, one persistent CTA per SM over (batch, token) items:
//      warp 8 (K producer): the token's Q and dO rows (TMA tiles) and row
//          vectors, then each chunk's K rows through the tensor engine's
//          four-row gather, into K slots used in turn.
//      warp 10 (V producer): each chunk's V rows through cp.async, into one V
//          slot. (Two copy paths at once, as in the forward.)
//      warp 9 (MMA issuer), per chunk c: S^T = K_c Q^T and dP^T = V_c dO^T
//          (slot-major: TMEM lane = slot), then dV_c = P^T dO and
//          dK_c = dS^T Q with A from TMEM, and dQ^T += K_c^T dS^T with dS^T
//          from shared memory (dQ^T stays in TMEM over the token's chunks).
//      warps 0-7 (thread = slot; warps w and w + 4 take one half of the heads
//          each): P^T and scale * dS^T as bf16 hi/lo pairs into TMEM and
//          (dS^T) shared memory; then (one half of the columns each) the
//          per-slot dK_c and dV_c rows are added into the pool gradients with
//          vector fp32 reductions (red.global.add.v4.f32); after the token's
//          last chunk, dQ^T (thread = head-dim index) is written to dq.
// A chunk's products wait for its P^T / dS^T; the next chunk's S^T and dP^T
// start once dK_c (which sits in the S^T columns) has been read out, so they
// run while dV_c is drained. The gathers of the next chunks overlap it all.
#include <type_traits>

#include "attn_common.cuh"
#include "attn_sparse.cuh"
#include "sm100_ptx.cuh"

namespace attn {
using namespace ptx;

namespace {

#ifdef ATTN_TRACE
static __device__ unsigned long long g_attn_trace[kTraceCtas * kTraceRoles * kTraceEvents];
#endif

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}
// Four rows r0..r3 of a 2-D map (box: one row of 64 columns), columns
// col..col+63, into 4 consecutive 128-byte rows of shared memory.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                            int col, int r0, int r1, int r2, int r3,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5, %6, %7}], [%2], %8;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(col), "r"(r0), "r"(r1), "r"(r2), "r"(r3),
      "l"(policy)
      : "memory");
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------------------------ preprocess
// One warp per (batch, token, head) row: Dvec = sum_k dO * (o + o_lo) and
// -LSE*log2(e) (-inf when LSE is -inf: no filled slot), plus the zeroing of
// dkp and dvp by a grid-stride loop, and the start of the status word.
__global__ void __launch_bounds__(256) attn_sparse_bwd_preprocess_kernel(
    const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ o_lo,
    const __nv_bfloat16* __restrict__ dO, const float* __restrict__ lse, float* __restrict__ nlse2,
    float* __restrict__ dvec, float4* __restrict__ dkp, long long n_dkp4, float4* __restrict__ dvp,
    long long n_dvp4, int* __restrict__ status, int B, int T, int H, int DV) {
  const long long gt = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long nthreads = static_cast<long long>(gridDim.x) * blockDim.x;
  if (gt == 0) init_status_word(status);
  for (long long i = gt; i < n_dkp4; i += nthreads) dkp[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (long long i = gt; i < n_dvp4; i += nthreads) dvp[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  const long long rows = static_cast<long long>(B) * T * H;
  const int lane = threadIdx.x % 32;
  for (long long row = gt / 32; row < rows; row += nthreads / 32) {
    const __nv_bfloat16* orow = o + row * DV;
    const __nv_bfloat16* drow = dO + row * DV;
    float acc = 0.f;
    for (int k = lane; k < DV; k += 32) {
      float ov = __bfloat162float(orow[k]);
      if (o_lo) ov += __bfloat162float(o_lo[row * DV + k]);
      acc = fmaf(__bfloat162float(drow[k]), ov, acc);
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
    if (lane == 0) {
      const long long bt = row / H;
      const int h = static_cast<int>(row % H);
      const int b = static_cast<int>(bt / T), t = static_cast<int>(bt % T);
      const float l = lse[(static_cast<long long>(b) * H + h) * T + t];
      dvec[row] = acc;
      nlse2[row] = (l == -INFINITY) ? -INFINITY : -l * kLog2e;
    }
  }
}

// ------------------------------------------------------------------ main
template <int DK, int DV>
__global__ void __launch_bounds__(SparseBwdCfg<DK, DV>::THREADS, 1)
    attn_sparse_bwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_do,
                           const __grid_constant__ CUtensorMap tm_k, const SparseBwdParams p) {
  using C = SparseBwdCfg<DK, DV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  __shared__ uint64_t bar_q_full, bar_q_empty, bar_mma_done;
  __shared__ uint64_t bar_kv_full[C::NSLOT], bar_kv_empty[C::NSLOT];
  __shared__ uint64_t bar_sdp_full, bar_pds_full, bar_grads_full, bar_dk_drained, bar_dv_drained;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int n_items = p.B * p.T;
  const int nch = p.n_chunks;
  const int cta = blockIdx.x, n_cta = gridDim.x;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar_q_full), 1);
    mbar_init(smem_u32(&bar_q_empty), 1);
    mbar_init(smem_u32(&bar_mma_done), 1);
    for (int i = 0; i < C::NSLOT; ++i) {
      mbar_init(smem_u32(&bar_kv_full[i]), 1);
      mbar_init(smem_u32(&bar_kv_empty[i]), 1);
    }
    mbar_init(smem_u32(&bar_sdp_full), 1);
    mbar_init(smem_u32(&bar_pds_full), 256);
    mbar_init(smem_u32(&bar_grads_full), 1);
    mbar_init(smem_u32(&bar_dk_drained), 256);
    mbar_init(smem_u32(&bar_dv_drained), 256);
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

  const uint32_t sQ = smem_u32(smem + C::SMEM_Q);
  const uint32_t sDO = smem_u32(smem + C::SMEM_DO);
  const uint32_t sDsHi = smem_u32(smem + C::SMEM_DS);
  const uint32_t sDsLo = sDsHi + C::DS_BYTES;
  const uint32_t sRing = smem_u32(smem + C::SMEM_RING);
  float* rows_s = reinterpret_cast<float*>(smem + C::SMEM_ROWS);  // nlse2[128], then dvec[128]

  if (warp == C::W_KPROD) {
    // ------------------------------------------------------------ K producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_do);
      prefetch_tmap(&tm_k);
    }
    const uint64_t keep = policy_evict_last();  // pool rows recur in nearby tokens' lists
    TraceCursor tc;
    if (lane == 0) ATTN_TRACE_INIT(tc, 0);
    int q_loads = 0, last_k = -1;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int item = r * n_cta + cta;
      if (item >= n_items) break;
      const int b = item / p.T;
      const int* lst = p.idx + static_cast<size_t>(item) * p.K;
      const int row0 = b * p.P;
      auto load_k = [&](int c) {
        const int gc = r * nch + c;  // chunk index over this CTA's items
        const int slot = gc % C::KSLOTS, round = gc / C::KSLOTS;
        const int s0 = c * C::BK + 4 * lane;
        int4 e = make_int4(-1, -1, -1, -1);
        if (s0 < p.K) e = __ldg(reinterpret_cast<const int4*>(lst + s0));
        // Empty slots fetch row 0; the compute warps give them P = dS = 0.
        auto row = [&](int x) { return row0 + ((x >= 0 && x < p.P) ? x : 0); };
        if (round > 0) ok = mbar_wait_warp(smem_u32(&bar_kv_empty[slot]), (round - 1) & 1, ctl);
        if (!ok) return;
        ATTN_TRACE_EV(tc, 1, gc);  // K slot free, gather issued
        const uint32_t full = smem_u32(&bar_kv_full[slot]);
        const uint32_t dst = sRing + slot * C::SLOT_BYTES + lane * 4 * 128;
        mbar_arrive_expect_tx_el(full, C::K_BYTES);
        __syncwarp();
#pragma unroll
        for (int cb = 0; cb < C::KCH; ++cb)
          tma_gather4(dst + cb * (C::BK * 128), &tm_k, full, cb * 64, row(e.x), row(e.y), row(e.z),
                      row(e.w), keep);
        last_k = gc;
      };
      // The first chunk's K, then Q, dO and the row vectors once the previous
      // item's products are done with them, then the remaining chunks' K.
      if (r > 0) load_k(0);
      if (!ok) break;
      if (r > 0) ok = mbar_wait_warp(smem_u32(&bar_q_empty), (r - 1) & 1, ctl);
      if (!ok) break;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int h = 4 * lane + k;
        const bool in = h < p.H;
        const size_t rr = static_cast<size_t>(item) * p.H + h;
        // Heads past H (the next token's rows, or zeros) get P = 0 and dS = 0.
        rows_s[h] = in ? p.nlse2[rr] : -INFINITY;
        rows_s[C::BQ + h] = in ? p.dvec[rr] : 0.f;
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(smem_u32(&bar_q_full), C::Q_BYTES + C::DO_BYTES);
        for (int cb = 0; cb < C::KCH; ++cb)
          tma_load_2d(sQ + cb * (C::BQ * 128), &tm_q, smem_u32(&bar_q_full), cb * 64, item * p.H);
        for (int cb = 0; cb < C::VCH; ++cb)
          tma_load_2d(sDO + cb * (C::BQ * 128), &tm_do, smem_u32(&bar_q_full), cb * 64, item * p.H);
      }
      __syncwarp();
      ++q_loads;
      for (int c = (r > 0 ? 1 : 0); c < nch && ok; ++c) load_k(c);
    }
    if (lane == 0) {
      // Let every copy issued land before the CTA's shared memory goes away.
      for (int g = max(0, last_k - C::KSLOTS + 1); g <= last_k; ++g)
        mbar_wait_drain(smem_u32(&bar_kv_full[g % C::KSLOTS]), (g / C::KSLOTS) & 1, 50000000ull);
      if (q_loads > 0) mbar_wait_drain(smem_u32(&bar_q_full), (q_loads - 1) & 1, 50000000ull);
    }
    __syncwarp();
  } else if (warp == C::W_VPROD) {
    // ------------------------------------------------------------ V producer
    // Row j's 16-byte unit u lands at j * 128 + ((u % 8) ^ (j % 8)) * 16 in
    // 64-column block u / 8 (the 128-byte swizzle the MMA descriptors expect).
    int* idx_s = reinterpret_cast<int*>(smem + C::SMEM_IDX);
    TraceCursor tc;
    if (lane == 0) ATTN_TRACE_INIT(tc, 10);
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int item = r * n_cta + cta;
      if (item >= n_items) break;
      const int b = item / p.T;
      const int* lst = p.idx + static_cast<size_t>(item) * p.K;
      for (int c = 0; c < nch && ok; ++c) {
        const int gc = r * nch + c;
        __syncwarp();
        const int s0 = c * C::BK + 4 * lane;
        int4 e = make_int4(-1, -1, -1, -1);
        if (s0 < p.K) e = __ldg(reinterpret_cast<const int4*>(lst + s0));
        auto chk = [&](int x) { return (x >= 0 && x < p.P) ? x : -1; };
        reinterpret_cast<int4*>(idx_s)[lane] = make_int4(chk(e.x), chk(e.y), chk(e.z), chk(e.w));
        __syncwarp();
        if (gc > 0) ok = mbar_wait_warp(smem_u32(&bar_kv_empty[C::VSLOT]), (gc - 1) & 1, ctl);
        if (!ok) break;
        ATTN_TRACE_EV(tc, 1, gc);  // V slot free, copies issued
        const uint32_t dst = sRing + C::VSLOT * C::SLOT_BYTES;
        constexpr int UNITS = DV / 8;
        constexpr int RPI = 32 / UNITS;
        const int u = lane % UNITS, jr = lane / UNITS;
        const uint32_t ublk = (u / 8) * (C::BK * 128);
        const __nv_bfloat16* base = p.vp + static_cast<size_t>(b) * p.P * DV + u * 8;
#pragma unroll 8
        for (int j0 = 0; j0 < C::BK; j0 += RPI) {
          const int j = j0 + jr;
          const int x = idx_s[j];
          const uint32_t d = dst + ublk + j * 128 + (((u % 8) ^ (j & 7)) << 4);
          cp_async16(d, base + static_cast<size_t>(x < 0 ? 0 : x) * DV, x < 0 ? 0u : 16u);
        }
        cp_async_commit();
        cp_async_wait<0>();
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bar_kv_full[C::VSLOT]));
        ATTN_TRACE_EV(tc, 2, gc);  // V landed
      }
    }
    cp_async_wait<0>();
    __syncwarp();
  } else if (warp == C::W_MMA) {
    // ------------------------------------------------------------ MMA issuer
    bool ok = !p.inject_stall;
    TraceCursor tc;
    if (lane == 0) ATTN_TRACE_INIT(tc, 1);
    constexpr uint32_t idesc_sdp = idesc_bf16_f32(128, 128, 0, 0);  // K-major A and B
    constexpr uint32_t idesc_dv = idesc_bf16_f32(128, DV, 0, 1);    // B = dO, MN-major
    constexpr uint32_t idesc_dk = idesc_bf16_f32(128, DK, 0, 1);    // B = Q, MN-major
    constexpr uint32_t idesc_dq = idesc_bf16_f32(128, 128, 1, 1);   // A = K^T, B = dS^T, MN-major
    const uint64_t dq_k = sw128_desc(sQ, 16, 1024);
    const uint64_t ddo_k = sw128_desc(sDO, 16, 1024);
    const uint64_t dq_mn = sw128_desc(sQ, C::BQ * 128, 1024);
    const uint64_t ddo_mn = sw128_desc(sDO, C::BQ * 128, 1024);
    const uint64_t dds_hi = sw128_desc(sDsHi, C::BK * 128, 1024);
    const uint64_t dds_lo = sw128_desc(sDsLo, C::BK * 128, 1024);
    auto add = [](uint64_t d, uint32_t bytes) { return d + (bytes >> 4); };
    int chunk = 0;  // chunk count over this CTA's items
    for (int r = 0; ok; ++r) {
      const int item = r * n_cta + cta;
      if (item >= n_items) break;
      ok = mbar_wait_warp(smem_u32(&bar_q_full), r & 1, ctl);
      if (!ok) break;
      for (int c = 0; c < nch && ok; ++c, ++chunk) {
        const int sk = chunk % C::KSLOTS, sv = C::VSLOT;
        // The S^T / P^T / dK columns are free once the compute warps have
        // read the previous chunk's dK_c out of them.
        if (chunk > 0) ok = mbar_wait_warp(smem_u32(&bar_dk_drained), (chunk - 1) & 1, ctl);
        if (ok) ok = mbar_wait_warp(smem_u32(&bar_kv_full[sk]), (chunk / C::KSLOTS) & 1, ctl);
        if (ok) ok = mbar_wait_warp(smem_u32(&bar_kv_full[sv]), chunk & 1, ctl);
        if (!ok) break;
        ATTN_TRACE_EV(tc, 1, chunk);  // dK drained, K and V landed: issuing S^T, dP^T
        tc_fence_after();
        const uint32_t kb = sRing + sk * C::SLOT_BYTES, vb = sRing + sv * C::SLOT_BYTES;
        const uint64_t dk_k = sw128_desc(kb, 16, 1024), dv_k = sw128_desc(vb, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < DK / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (128 * 128) + (kk & 3) * 32;
          mma_ss_el(tmem + C::TM_S, add(dk_k, off), add(dq_k, off), idesc_sdp, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < DV / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (128 * 128) + (kk & 3) * 32;
          mma_ss_el(tmem + C::TM_DP, add(dv_k, off), add(ddo_k, off), idesc_sdp, kk > 0);
        }
        mma_commit_el(smem_u32(&bar_sdp_full));
        mma_commit_el(smem_u32(&bar_kv_empty[sv]));  // V_c is not read again
        ok = mbar_wait_warp(smem_u32(&bar_pds_full), chunk & 1, ctl);
        // dV_c's columns (and, at a token's first chunk, dQ^T's) are free once
        // the previous chunk's dV_c (and the token's dq) have been read out.
        if (ok && chunk > 0) ok = mbar_wait_warp(smem_u32(&bar_dv_drained), (chunk - 1) & 1, ctl);
        if (!ok) break;
        ATTN_TRACE_EV(tc, 2, chunk);  // P/dS stored, dV drained: issuing dV, dK, dQ
        tc_fence_after();
        // dV_c = P^T dO and dK_c = dS^T Q: heads 16kk..16kk+15 are TMEM columns
        // 16kk..16kk+7 (hi pairs) and 16kk+8..16kk+15 (lo pairs). dK_c goes into
        // the S^T columns, which dV_c above has read (MMAs run in issue order).
#pragma unroll
        for (int kk = 0; kk < C::BQ / 16; ++kk) {
          const uint32_t acc = kk > 0 ? 1u : 0u;
          mma_ts_el(tmem + C::TM_DV, tmem + C::TM_S + 16 * kk, add(ddo_mn, kk * 2048), idesc_dv, acc);
          mma_ts_el(tmem + C::TM_DV, tmem + C::TM_S + 16 * kk + 8, add(ddo_mn, kk * 2048), idesc_dv, 1u);
        }
#pragma unroll
        for (int kk = 0; kk < C::BQ / 16; ++kk) {
          const uint32_t acc = kk > 0 ? 1u : 0u;
          mma_ts_el(tmem + C::TM_S, tmem + C::TM_DP + 16 * kk, add(dq_mn, kk * 2048), idesc_dk, acc);
          mma_ts_el(tmem + C::TM_S, tmem + C::TM_DP + 16 * kk + 8, add(dq_mn, kk * 2048), idesc_dk, 1u);
        }
        // dQ^T[d][h] += sum over slots of K_c[slot][d] (dS_hi + dS_lo)^T[slot][h].
        const uint64_t dk_mn = sw128_desc(kb, C::BK * 128, 1024);
#pragma unroll
        for (int kk = 0; kk < C::BK / 16; ++kk) {
          const uint32_t acc = (c > 0 || kk > 0) ? 1u : 0u;
          mma_ss_el(tmem + C::TM_DQ, add(dk_mn, kk * 2048), add(dds_hi, kk * 2048), idesc_dq, acc);
          mma_ss_el(tmem + C::TM_DQ, add(dk_mn, kk * 2048), add(dds_lo, kk * 2048), idesc_dq, 1u);
        }
        mma_commit_el(smem_u32(&bar_grads_full));
        mma_commit_el(smem_u32(&bar_kv_empty[sk]));  // K_c is not read again
        if (c + 1 == nch) mma_commit_el(smem_u32(&bar_q_empty));
      }
    }
    mma_commit_el(smem_u32(&bar_mma_done));
    mbar_wait_drain(smem_u32(&bar_mma_done), 0, 50000000ull);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ compute warps 0-7
    const int j = threadIdx.x % 128;  // slot within the chunk == TMEM lane (later: head-dim index)
    const int cg = warp / 4;          // this warp's half: heads 64 cg.., gradient columns
    const uint32_t lane_base = static_cast<uint32_t>((warp % 4) * 32) << 16;
    const uint64_t sl2 = f32x2(p.scale_log2, p.scale_log2);
    const uint64_t sc2 = f32x2(p.scale, p.scale);
    const float4* nl4 = reinterpret_cast<const float4*>(rows_s);        // -LSE*log2(e) per head
    const float4* dv4 = reinterpret_cast<const float4*>(rows_s + C::BQ);  // Dvec per head
    // This warp's part of the dS^T tiles: rows j of head block cg, 4 KB in the
    // hi tile and 4 KB in the lo tile. Only this warp writes them, so it can
    // stage its gradient rows there once the chunk's dQ^T product has read
    // them, with no other warp touching them until its own next stores.
    const uint32_t stA = sDsHi + cg * (C::BK * 128) + (warp % 4) * 4096;
    const uint32_t stB = sDsLo + cg * (C::BK * 128) + (warp % 4) * 4096;
    bool ok = true;
    TraceCursor tc;
    if (lane == 0 && warp % 4 == 0) ATTN_TRACE_INIT(tc, 2 + cg);
    int chunk = 0;
    for (int r = 0; ok; ++r) {
      const int item = r * n_cta + cta;
      if (item >= n_items) break;
      const int b = item / p.T;
      const int* lst = p.idx + static_cast<size_t>(item) * p.K;
      ok = mbar_wait_warp(smem_u32(&bar_q_full), r & 1, ctl);  // the row vectors are in
      if (!ok) break;
      for (int c = 0; c < nch && ok; ++c, ++chunk) {
        const int s = c * C::BK + j;
        const int e = s < p.K ? __ldg(lst + s) : -1;
        const bool filled = e >= 0 && e < p.P;
        ok = mbar_wait_warp(smem_u32(&bar_sdp_full), chunk & 1, ctl);
        if (!ok) break;
        ATTN_TRACE_EV(tc, 1, chunk);  // S^T, dP^T landed
        tc_fence_after();
        // Row j of S^T and dP^T, 16 heads at a time: P^T and scale * dS^T as
        // bf16 hi/lo pairs into TMEM over the scores, and dS^T into shared
        // memory (row j of the MN-major B operand of dQ^T: heads 0..63 in the
        // first 64-column block, 64..127 in the second, 128-byte swizzle).
#pragma unroll 1
        for (int h0 = 64 * cg; h0 < 64 * cg + 64; h0 += 16) {
          uint32_t su[16], du[16];
          tmem_ld16(tmem + lane_base + C::TM_S + h0, su);
          tmem_ld16(tmem + lane_base + C::TM_DP + h0, du);
          tmem_wait_ld();
          uint32_t pp[16], dd[16];
#pragma unroll
          for (int k = 0; k < 16; k += 4) {
            const float4 nl = nl4[(h0 + k) / 4];
            const float4 dv = dv4[(h0 + k) / 4];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int kk = k + 2 * hh;  // heads h0 + kk, h0 + kk + 1
              float x0, x1;
              unpack_f32x2(fma_f32x2(f32x2(__uint_as_float(su[kk]), __uint_as_float(su[kk + 1])), sl2,
                                     hh ? f32x2(nl.z, nl.w) : f32x2(nl.x, nl.y)),
                           x0, x1);
              float p0 = ex2(x0), p1 = ex2(x1);
              if (!filled) p0 = p1 = 0.f;
              const uint64_t dpv = sub_f32x2(f32x2(__uint_as_float(du[kk]), __uint_as_float(du[kk + 1])),
                                             hh ? f32x2(dv.z, dv.w) : f32x2(dv.x, dv.y));
              float d0, d1;
              unpack_f32x2(mul_f32x2(mul_f32x2(f32x2(p0, p1), sc2), dpv), d0, d1);
              split_bf16x2_fma(p0, p1, pp[kk / 2], pp[8 + kk / 2]);
              split_bf16x2_fma(d0, d1, dd[kk / 2], dd[8 + kk / 2]);
            }
          }
          tmem_st16(tmem + lane_base + C::TM_S + h0, pp);
          tmem_st16(tmem + lane_base + C::TM_DP + h0, dd);
          // Heads h0..h0+15: two 16-byte units of row j in block h0 / 64.
          const uint32_t blk = (h0 / 64) * (C::BK * 128) + j * 128;
          const int u0 = (h0 % 64) / 8;
#pragma unroll
          for (int q2 = 0; q2 < 2; ++q2) {
            const uint32_t off = blk + (((u0 + q2) ^ (j & 7)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sDsHi + off),
                         "r"(dd[4 * q2]), "r"(dd[4 * q2 + 1]), "r"(dd[4 * q2 + 2]), "r"(dd[4 * q2 + 3])
                         : "memory");
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sDsLo + off),
                         "r"(dd[8 + 4 * q2]), "r"(dd[8 + 4 * q2 + 1]), "r"(dd[8 + 4 * q2 + 2]),
                         "r"(dd[8 + 4 * q2 + 3])
                         : "memory");
          }
        }
        tmem_wait_st();
        fence_async_smem();
        tc_fence_before();
        mbar_arrive(smem_u32(&bar_pds_full));
        ATTN_TRACE_EV(tc, 2, chunk);  // P^T, dS^T stored
        // The chunk's products are done: add row j of dK_c and dV_c (this
        // warp's half of the columns) into the pool gradients of pool row e.
        ok = mbar_wait_warp(smem_u32(&bar_grads_full), chunk & 1, ctl);
        if (!ok) break;
        ATTN_TRACE_EV(tc, 3, chunk);  // dV_c, dK_c, dQ^T done
        tc_fence_after();
        // Staging: the warp's 32 rows in its own 8 KB of the dS^T tiles, row i
        // (HC fp32 columns) in piece stA or stB, 16-byte unit u at unit
        // position u ^ (i mod UNITS); then each reduction instruction adds
        // RPI whole rows, lane l taking unit l mod UNITS of row l / UNITS, so
        // each one covers contiguous row segments instead of scattered words.
        auto drain = [&](uint32_t col, float* pool, auto dcols) {
          constexpr int DC = decltype(dcols)::value;
          constexpr int HC = DC / 2;        // this warp's columns: cg * HC ..
          constexpr int ROWB = HC * 4;      // bytes of a staged row
          constexpr int UNITS = HC / 4;     // 16-byte units of a staged row
          constexpr int RPP = 4096 / ROWB;  // rows per 4 KB piece
          constexpr int RPI = 32 / UNITS;   // rows per reduction instruction
          auto row_addr = [&](int i) { return (i < RPP ? stA : stB) + (i % RPP) * ROWB; };
#pragma unroll
          for (int k0 = 0; k0 < HC; k0 += 32) {
            uint32_t u[32];
            tmem_ld32(tmem + lane_base + col + cg * HC + k0, u);
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const int unit = k0 / 4 + q;
              const uint32_t addr = row_addr(lane) + ((unit ^ (lane & (UNITS - 1))) << 4);
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(u[4 * q]),
                           "r"(u[4 * q + 1]), "r"(u[4 * q + 2]), "r"(u[4 * q + 3])
                           : "memory");
            }
          }
          __syncwarp();
          const int sub = lane % UNITS, rr = lane / UNITS;
#pragma unroll 4
          for (int i0 = 0; i0 < 32; i0 += RPI) {
            const int i = i0 + rr;
            const int ei = __shfl_sync(0xffffffffu, e, i);
            const bool fi = __shfl_sync(0xffffffffu, filled ? 1 : 0, i) != 0;
            if (fi) {
              const uint32_t addr = row_addr(i) + ((sub ^ (i & (UNITS - 1))) << 4);
              float4 v;
              asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                           : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                           : "r"(addr));
              red_add_v4(pool + (static_cast<size_t>(b) * p.P + ei) * DC + cg * HC + 4 * sub, v.x, v.y,
                         v.z, v.w);
            }
          }
          __syncwarp();
        };
        drain(C::TM_S, p.dkp, std::integral_constant<int, DK>{});
        // dK_c is read: the next chunk's S^T may overwrite its columns.
        tc_fence_before();
        mbar_arrive(smem_u32(&bar_dk_drained));
        ATTN_TRACE_EV(tc, 4, chunk);  // dK_c drained
        drain(C::TM_DV, p.dvp, std::integral_constant<int, DV>{});
        if (c + 1 == nch) {
          // dQ^T is complete for this token: thread j < DK writes column j of
          // dq for this warp's heads (row j of dQ^T). j < DK is warp-uniform.
          if (j < DK) {
            float* dqb = p.dq + static_cast<size_t>(item) * p.H * DK + j;
#pragma unroll 1
            for (int h0 = 64 * cg; h0 < 64 * cg + 64; h0 += 32) {
              uint32_t u[32];
              tmem_ld32(tmem + lane_base + C::TM_DQ + h0, u);
              tmem_wait_ld();
#pragma unroll
              for (int k = 0; k < 32; ++k)
                if (h0 + k < p.H) dqb[static_cast<size_t>(h0 + k) * DK] = __uint_as_float(u[k]);
            }
          }
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&bar_dv_drained));
        ATTN_TRACE_EV(tc, 5, chunk);  // dV_c (and dq) drained
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::W_MMA) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int DK, int DV>
cudaError_t launch_sparse_bwd_t(const CUtensorMap& tq, const CUtensorMap& tdo, const CUtensorMap& tk,
                                const SparseBwdParams& p, cudaStream_t stream) {
  using C = SparseBwdCfg<DK, DV>;
  static bool attr_set[64] = {};
  static int sm_count[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attn_sparse_bwd_kernel<DK, DV>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  if (dev < 64 && sm_count[dev] == 0)
    cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
  const long long n_items = static_cast<long long>(p.B) * p.T;
  const int sms = (dev < 64 && sm_count[dev] > 0) ? sm_count[dev] : 148;
  const dim3 grid(static_cast<unsigned>(n_items < sms ? n_items : sms));
  attn_sparse_bwd_kernel<DK, DV><<<grid, C::THREADS, C::SMEM_ALLOC, stream>>>(tq, tdo, tk, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sparse_bwd(int DK, int DV, const __nv_bfloat16* o, const __nv_bfloat16* o_lo,
                              const __nv_bfloat16* dO, const float* lse, float* nlse2, float* dvec,
                              const CUtensorMap& tq, const CUtensorMap& tdo, const CUtensorMap& tk,
                              const SparseBwdParams& p, cudaStream_t stream) {
  const long long n_dkp4 = static_cast<long long>(p.B) * p.P * DK / 4;
  const long long n_dvp4 = static_cast<long long>(p.B) * p.P * DV / 4;
  attn_sparse_bwd_preprocess_kernel<<<1024, 256, 0, stream>>>(
      o, o_lo, dO, lse, nlse2, dvec, reinterpret_cast<float4*>(p.dkp), n_dkp4,
      reinterpret_cast<float4*>(p.dvp), n_dvp4, p.status, p.B, p.T, p.H, DV);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (DK == 128 && DV == 128) return launch_sparse_bwd_t<128, 128>(tq, tdo, tk, p, stream);
  if (DK == 128 && DV == 64) return launch_sparse_bwd_t<128, 64>(tq, tdo, tk, p, stream);
  if (DK == 64 && DV == 128) return launch_sparse_bwd_t<64, 128>(tq, tdo, tk, p, stream);
  if (DK == 64 && DV == 64) return launch_sparse_bwd_t<64, 64>(tq, tdo, tk, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attn

#ifdef ATTN_TRACE
// Copies the sparse backward's timeline records to the host and clears them
// (traced build only).
extern "C" int attn_trace_copy_sparse_bwd(void* host, size_t bytes) {
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
