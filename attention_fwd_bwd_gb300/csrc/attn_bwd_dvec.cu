// The backward's Dvec pass for sm_103a, used when the forward's low-order
// output residual is not available. The gradient of O = softmax(scale Q K^T) V
// ("Scheduling Data to Compute: Hierarchical Data Pipelining for LLM Training
// on AMD GPUs", section 2.1, Eq. (1)) needs, per query row,
//   Dvec_i = sum_j P_ij dP_ij,   dP = dO V^T,
// which equals rowsum(dO * O)_i. From a bf16 o that sum keeps only about 8
// significant bits of O, and with a sharp softmax the error it leaves in dQ
// exceeds the gradient tolerance; this pass computes the sum from its
// definition instead, in fp32, at the cost of two GEMM units (Q K^T and
// dO V^T).
//
// Per CTA (persistent, items as the forward's: two 128-row query tiles that
// share their K/V tiles, longest first; see TileItem):
//   warp 8 (TMA producer): Q_A, Q_B, dO_A, dO_B once per item, then K_j and
//       V_j into a ring of shared-memory slots (full/empty mbarrier pairs).
//   warp 9 (MMA issuer): S_t = Q_t K_j^T and dP_t = dO_t V_j^T into tile t's
//       two TMEM buffers (all operands K-major); the tiles alternate on the
//       tensor core, so one tile's rows are read while the other's products
//       run.
//   warps 0-3 / 4-7 (rows of tile A / B): thread r owns query row r (TMEM
//       lane r): P = exp2(S scale log2(e) - LSE log2(e)) with the mask, and
//       the row sum of P dP, accumulated over the row's key tiles.
#include "attn_common.cuh"
#include "attn_items.cuh"
#include "sm100_ptx.cuh"

namespace attn {
using namespace ptx;

namespace {

template <int D, bool WIN>
__global__ void __launch_bounds__(DvecCfg<D>::THREADS, 1)
    attn_bwd_dvec_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_do, const DvecParams p,
                         const int pair) {
  using C = DvecCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  __shared__ uint64_t bar_q_full, bar_q_empty, bar_mma_done;
  __shared__ uint64_t bar_kv_full[C::NSLOT], bar_kv_empty[C::NSLOT];
  __shared__ uint64_t bar_sdp_full[2], bar_sdp_free[2];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int n_items = tile_n_items(p, pair != 0);
  const int cta = blockIdx.x, n_cta = gridDim.x;
  auto jlo = [&](const TileItem& it, int t) { return WIN ? it.j_lo[t] : 0; };

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar_q_full), 1);
    mbar_init(smem_u32(&bar_q_empty), 1);
    mbar_init(smem_u32(&bar_mma_done), 1);
    for (int i = 0; i < C::NSLOT; ++i) {
      mbar_init(smem_u32(&bar_kv_full[i]), 1);
      mbar_init(smem_u32(&bar_kv_empty[i]), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_u32(&bar_sdp_full[t]), 1);
      mbar_init(smem_u32(&bar_sdp_free[t]), 128);
    }
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(&tmem_base_s), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  const WaitCtl ctl{&abort_flag, p.status, p.timeout_ns};

  // Q_A, Q_B, dO_A, dO_B at sQ + n * Q_BYTES, n = 0..3.
  const uint32_t sQ = smem_u32(smem + C::SMEM_Q);
  const uint32_t sRing = smem_u32(smem + C::SMEM_RING);

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    // Per item: the first K/V tile pair, then Q and dO of both tiles once the
    // previous item's last products have read them, then the remaining K/V
    // tiles. Ring positions run on across items: K_j at 2 (j - jb), V_j after.
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      prefetch_tmap(&tm_do);
    }
    const uint64_t keep = policy_evict_last();  // K/V tiles are re-read by G heads x tiles
    int issued = 0;
    int q_loads = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int ii = fwd_item_index(r, cta, n_cta, n_items);
      if (ii < 0) break;
      const TileItem it = tile_item<WIN>(p, pair != 0, ii);
      const int jb = jlo(it, 0);
      const int n_pos = 2 * (it.n_kv[1] - jb);
      auto load_kv = [&](int idx) {
        const int pos = issued;
        const int slot = pos % C::NSLOT, round = pos / C::NSLOT;
        if (round > 0) ok = mbar_wait_warp(smem_u32(&bar_kv_empty[slot]), (round - 1) & 1, ctl);
        if (!ok) return;
        if (!bounds_ok(jb + (idx >> 1) >= 0 && (jb + (idx >> 1)) * C::BK < p.S && it.b < p.B &&
                           it.g < p.Hkv, ctl)) {
          ok = false;
          return;
        }
        const uint32_t full = smem_u32(&bar_kv_full[slot]);
        const uint32_t dst = sRing + slot * C::KV_BYTES;
        const CUtensorMap* m = (idx & 1) ? &tm_v : &tm_k;
        mbar_arrive_expect_tx_el(full, C::KV_BYTES);
        for (int c = 0; c < C::KCH; ++c)
          tma_load_4d_hint_el(dst + c * (C::BK * 128), m, full, c * 64, it.g,
                              (jb + (idx >> 1)) * C::BK, it.b, keep);
        issued = pos + 1;
      };
      const int pre = (r == 0) ? 0 : min(2, n_pos);
      for (int idx = 0; idx < pre && ok; ++idx) load_kv(idx);
      if (!ok) break;
      if (r > 0) ok = mbar_wait_warp(smem_u32(&bar_q_empty), (r - 1) & 1, ctl);
      if (!ok) break;
      mbar_arrive_expect_tx_el(smem_u32(&bar_q_full), 4 * C::Q_BYTES);
      for (int n = 0; n < 4; ++n)
        for (int c = 0; c < C::KCH; ++c)
          tma_load_4d_el(sQ + n * C::Q_BYTES + c * (C::BQ * 128), n < 2 ? &tm_q : &tm_do,
                         smem_u32(&bar_q_full), c * 64, it.hq[n & 1], it.qs[n & 1], it.b);
      ++q_loads;
      for (int idx = pre; idx < n_pos && ok; ++idx) load_kv(idx);
    }
    if (lane == 0) {
      // Let every copy issued land before the CTA's shared memory goes away
      // (immediate in a normal run, where the MMA warp consumed them all).
      for (int pos = max(0, issued - C::NSLOT); pos < issued; ++pos)
        mbar_wait_drain(smem_u32(&bar_kv_full[pos % C::NSLOT]), (pos / C::NSLOT) & 1, 50000000ull);
      if (q_loads > 0) mbar_wait_drain(smem_u32(&bar_q_full), (q_loads - 1) & 1, 50000000ull);
    }
    (void)ok;
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    bool ok = !p.inject_stall;
    constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
    const uint64_t dq_desc = sw128_desc(sQ, 16, 1024);
    int ring = 0;             // ring position of the item's first K/V tile
    int n_sdp[2] = {0, 0};    // S/dP products issued per tile, over all items
    for (int r = 0; ok; ++r) {
      const int ii = fwd_item_index(r, cta, n_cta, n_items);
      if (ii < 0) break;
      const TileItem it = tile_item<WIN>(p, pair != 0, ii);
      const int jb = jlo(it, 0);
      const int n_kv = it.n_kv[1];
      ok = mbar_wait_warp(smem_u32(&bar_q_full), r & 1, ctl);
      if (!ok) break;
      // Product pairs left in this item; the last one hands Q/dO back.
      int left = (it.n_kv[0] - jlo(it, 0)) + (it.n_kv[1] - jlo(it, 1));
      auto wait_kv = [&](int idx) {
        const int pos = ring + idx;
        return mbar_wait_warp(smem_u32(&bar_kv_full[pos % C::NSLOT]), (pos / C::NSLOT) & 1, ctl);
      };
      auto kv_slot = [&](int idx) { return (ring + idx) % C::NSLOT; };
      // Per key tile j: both tiles' S products (K_j), then both tiles' dP
      // products (V_j). K_j's slot is handed back after the S products, so
      // the load of V_{j+1} into it overlaps the dP products of j.
      for (int j = jb; j < n_kv && ok; ++j) {
        // Every ring tile is waited for before its slot is handed back, so no
        // copy is in flight then (each tile also has a use: the two tiles'
        // ranges leave no gap, with a window too).
        ok = wait_kv(2 * (j - jb));
        if (!ok) break;
        const uint64_t dk = sw128_desc(sRing + kv_slot(2 * (j - jb)) * C::KV_BYTES, 16, 1024);
        for (int t = 0; t < 2 && ok; ++t) {
          if (j < jlo(it, t) || j >= it.n_kv[t]) continue;
          // Tile t's rows have read S_t and dP_t of its previous product pair.
          if (n_sdp[t] > 0) ok = mbar_wait_warp(smem_u32(&bar_sdp_free[t]), (n_sdp[t] - 1) & 1, ctl);
          if (!ok) break;
          tc_fence_after();
          const uint64_t dq = dq_desc + ((t * C::Q_BYTES) >> 4);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = ((kk >> 2) * (128 * 128) + (kk & 3) * 32) >> 4;
            mma_ss_el(tmem + C::tm_s(t), dq + koff, dk + koff, idesc, kk > 0);
          }
        }
        if (!ok) break;
        mma_commit_el(smem_u32(&bar_kv_empty[kv_slot(2 * (j - jb))]));
        ok = wait_kv(2 * (j - jb) + 1);
        if (!ok) break;
        tc_fence_after();
        const uint64_t dv = sw128_desc(sRing + kv_slot(2 * (j - jb) + 1) * C::KV_BYTES, 16, 1024);
        for (int t = 0; t < 2; ++t) {
          if (j < jlo(it, t) || j >= it.n_kv[t]) continue;
          const uint64_t ddo = dq_desc + (((2 + t) * C::Q_BYTES) >> 4);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = ((kk >> 2) * (128 * 128) + (kk & 3) * 32) >> 4;
            mma_ss_el(tmem + C::tm_dp(t), ddo + koff, dv + koff, idesc, kk > 0);
          }
          mma_commit_el(smem_u32(&bar_sdp_full[t]));
          ++n_sdp[t];
          if (--left == 0) mma_commit_el(smem_u32(&bar_q_empty));
        }
        mma_commit_el(smem_u32(&bar_kv_empty[kv_slot(2 * (j - jb) + 1)]));
      }
      ring += 2 * (n_kv - jb);
    }
    // Every MMA issued finishes before TMEM is released.
    mma_commit_el(smem_u32(&bar_mma_done));
    mbar_wait_drain(smem_u32(&bar_mma_done), 0, 50000000ull);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ row warps 0-7
    const int t = warp / 4;
    const int r = threadIdx.x % 128;
    const uint32_t lane_base = static_cast<uint32_t>((warp % 4) * 32) << 16;
    const uint32_t ts = tmem + lane_base + C::tm_s(t);
    const uint32_t tdp = tmem + lane_base + C::tm_dp(t);
    const uint64_t sl2 = f32x2(p.scale_log2, p.scale_log2);
    bool ok = true;
    int n_seen = 0;  // product pairs of this tile, over all items
    for (int item = 0; ok; ++item) {
      const int ii = fwd_item_index(item, cta, n_cta, n_items);
      if (ii < 0) break;
      const TileItem it = tile_item<WIN>(p, pair != 0, ii);
      const int qt0 = it.qs[t];
      const int qrow = qt0 + r;
      const size_t rowoff = (static_cast<size_t>(it.b) * p.Hq + it.hq[t]) * p.S_pad;
      // Rows past S (padding) have -LSE log2(e) = -inf: P = 0; they are not stored.
      const float nl = p.nlse2[rowoff + min(qrow, p.S_pad - 1)];
      const uint64_t nl2 = f32x2(nl, nl);
      uint64_t acc[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};
      for (int j = jlo(it, t); j < it.n_kv[t]; ++j) {
        ok = mbar_wait_warp(smem_u32(&bar_sdp_full[t]), n_seen & 1, ctl);
        if (!ok) break;
        ++n_seen;
        tc_fence_after();
        const int k0 = j * C::BK;
        // Tiles that cross the causal diagonal, hold keys past S, or hold keys
        // below some row's window mask; the rest skip masking.
        const bool need_mask = (p.causal && k0 + C::BK - 1 > qt0) || (k0 + C::BK > p.S) ||
                               (WIN && k0 < qt0 + C::BQ - p.window);
        // Visible columns of this tile for this row: c_lo <= c <= c_hi.
        const int c_hi = (p.causal ? min(qrow, p.S - 1) : (p.S - 1)) - k0;
        const int c_lo = WIN ? qrow - p.window + 1 - k0 : 0;
        // Two halves of 64 columns; the buffers are handed back once the
        // second half is read, before its arithmetic.
#pragma unroll
        for (int c = 0; c < C::BK; c += 64) {
          uint32_t us[64], ud[64];
          tmem_ld32(ts + c, *reinterpret_cast<uint32_t(*)[32]>(&us[0]));
          tmem_ld32(ts + c + 32, *reinterpret_cast<uint32_t(*)[32]>(&us[32]));
          tmem_ld32(tdp + c, *reinterpret_cast<uint32_t(*)[32]>(&ud[0]));
          tmem_ld32(tdp + c + 32, *reinterpret_cast<uint32_t(*)[32]>(&ud[32]));
          tmem_wait_ld();
          if (c + 64 == C::BK) {
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_sdp_free[t]));
          }
#pragma unroll
          for (int i = 0; i < 64; i += 2) {
            float p0, p1;
            unpack_f32x2(fma_f32x2(f32x2(__uint_as_float(us[i]), __uint_as_float(us[i + 1])), sl2, nl2),
                         p0, p1);
            p0 = ex2(p0);
            p1 = ex2(p1);
            if (need_mask) {
              if (c + i > c_hi || (WIN && c + i < c_lo)) p0 = 0.f;
              if (c + i + 1 > c_hi || (WIN && c + i + 1 < c_lo)) p1 = 0.f;
            }
            acc[(i / 2) & 1] = fma_f32x2(f32x2(p0, p1),
                                         f32x2(__uint_as_float(ud[i]), __uint_as_float(ud[i + 1])),
                                         acc[(i / 2) & 1]);
          }
        }
      }
      if (!ok) break;
      float a0, a1, b0, b1;
      unpack_f32x2(acc[0], a0, a1);
      unpack_f32x2(acc[1], b0, b1);
      if (qrow < p.S && bounds_ok(rowoff + qrow < static_cast<size_t>(p.B) * p.Hq * p.S_pad, ctl))
        p.dvec[rowoff + qrow] = (a0 + a1) + (b0 + b1);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int D, bool WIN>
cudaError_t launch_dvec_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const DvecParams& p, cudaStream_t stream) {
  using C = DvecCfg<D>;
  static bool attr_set[64] = {};
  static int sm_count[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_dvec_kernel<D, WIN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  if (dev < 64 && sm_count[dev] == 0)
    cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
  const bool pair = tile_pair_heads(p);  // see TileItem
  const long long n_items = tile_n_items(p, pair);
  const int sms = (dev < 64 && sm_count[dev] > 0) ? sm_count[dev] : 148;
  const dim3 grid(static_cast<unsigned>(n_items < sms ? n_items : sms));
  attn_bwd_dvec_kernel<D, WIN><<<grid, C::THREADS, C::SMEM_ALLOC, stream>>>(tq, tk, tv, tdo, p,
                                                                           pair ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dvec(int D, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo, const DvecParams& p,
                            cudaStream_t stream) {
  const bool win = p.window > 0;
  if (D == 128)
    return win ? launch_dvec_t<128, true>(tq, tk, tv, tdo, p, stream)
               : launch_dvec_t<128, false>(tq, tk, tv, tdo, p, stream);
  return win ? launch_dvec_t<64, true>(tq, tk, tv, tdo, p, stream)
             : launch_dvec_t<64, false>(tq, tk, tv, tdo, p, stream);
}

}  // namespace attn
