// Sparse top-k gather attention, forward, for sm_103a. Each query token t
// carries a list of K pool rows (its top-k list: a sliding window plus
// compressed rows), and every one of its H query heads attends over exactly
// those rows: O[t, h] = softmax_j(scale * q[t, h] . kp[idx[t, j]]) vp[idx[t, j]]
// ("Scheduling Data to Compute: Hierarchical Data Pipelining for LLM Training
// on AMD GPUs", section 2.1: the forward gathers the listed vectors, computes
// scores and streams the values into the output accumulator; section 3: a
// token's top-k list is a list of KV row indices, fetched by a gather-mode
// tensor load; Table 7 for the list shapes).
//
// Per work item (batch b, token t), in a persistent CTA:
//   warp 8 (K producer): the token's H x DK query rows once (one TMA tile),
//       then every chunk's 128 K rows, gathered four pool rows per TMA
//       instruction (tile::gather4) straight into the 128-byte-swizzled
//       layout the MMAs read; empty slots fetch row 0 and are masked.
//   warp 10 (V producer): every chunk's V rows, gathered with 16-byte
//       cp.async copies into the same layout (empty slots copy nothing).
//       K and V thus arrive through two separate copy paths, each of which
//       moves about as many bytes per clock as one path alone did. K chunks
//       go through KSLOTS slots in turn and V chunks through the others, each
//       slot with a full/empty mbarrier pair.
//   warp 9 (MMA issuer): S_w = Q K_c^T for chunk c into warpgroup w = c % 2,
//       O_w += P_w V_c (P hi and lo bf16 parts from TMEM, V described
//       MN-major). The warpgroups alternate on the tensor core.
//   warps 0-3 / 4-7 (softmax of the even / odd chunks): thread r owns head row
//       r, keeps its own running max and sum, masks empty slots, writes P over
//       the scores in TMEM. At the item's end warpgroup 1 hands its (m, l)
//       over through shared memory and warpgroup 0 merges both partial
//       outputs -- read from both accumulators in TMEM -- into O and LSE, and
//       stores O (and o_lo) with TMA.
#include <type_traits>

#include "attn_common.cuh"
#include "attn_sparse.cuh"
#include "sm100_ptx.cuh"

namespace attn {
using namespace ptx;

namespace {

// 2-D tile load issued by one elected lane.
__device__ __forceinline__ void tma_load_2d_el(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                               int c0, int c1) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];\n\t}" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

// Four rows r0..r3 of a 2-D map (box: one row of 64 columns), columns
// col..col+63, into 4 consecutive 128-byte rows of shared memory. Issued by
// the calling thread.
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

// 16-byte global -> shared copy that bypasses L1; src_bytes = 0 copies
// nothing and zero-fills the 16 bytes.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* m, int c0, int c1, uint32_t src) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
          reinterpret_cast<uint64_t>(m)),
      "r"(c0), "r"(c1), "r"(src)
      : "memory");
}

// Largest (MAX) or smallest value of a 128-entry row.
template <bool MAX>
__device__ __forceinline__ float extreme128(const float (&x)[128]) {
  auto f3 = [](float a, float b, float c) { return MAX ? fmax3(a, b, c) : fmin3(a, b, c); };
  float a[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) a[i] = f3(x[i], x[16 + i], x[32 + i]);
#pragma unroll
  for (int c = 48; c < 112; c += 32)
#pragma unroll
    for (int i = 0; i < 16; ++i) a[i] = f3(a[i], x[c + i], x[c + 16 + i]);
#pragma unroll
  for (int i = 0; i < 16; ++i) a[i] = MAX ? fmaxf(a[i], x[112 + i]) : fminf(a[i], x[112 + i]);
  const float b0 = f3(a[0], a[1], a[2]), b1 = f3(a[3], a[4], a[5]), b2 = f3(a[6], a[7], a[8]);
  const float b3 = f3(a[9], a[10], a[11]), b4 = f3(a[12], a[13], a[14]);
  const float c0 = f3(b0, b1, b2), c1 = f3(b3, b4, a[15]);
  return MAX ? fmaxf(c0, c1) : fminf(c0, c1);
}

// Same rescale rule as the dense forward: the running max used for the
// exponentials moves only when the chunk's max exceeds it by more than 2^8.
constexpr float kSparseRescale = 8.0f;

// Chunks of warpgroup w in an item of n chunks (it takes c = w, w + 2, ...).
__device__ __forceinline__ int chunks_of(int n, int w) { return n > w ? (n - w + 1) / 2 : 0; }

template <int DK, int DV>
__global__ void __launch_bounds__(SparseFwdCfg<DK, DV>::THREADS, 1)
    attn_sparse_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_o,
                           const __grid_constant__ CUtensorMap tm_olo, const int write_lo,
                           const SparseFwdParams p) {
  using C = SparseFwdCfg<DK, DV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  __shared__ uint64_t bar_q_full, bar_q_empty, bar_mma_done, bar_merge, bar_o1_free;
  __shared__ uint64_t bar_kv_full[C::NSLOT], bar_kv_empty[C::NSLOT];
  __shared__ uint64_t bar_s_full[2], bar_p_full[2], bar_pv_done[2];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_flag;
  __shared__ uint4 filled_s[8];  // per softmax warp: filled-slot bits of its current chunk

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
    mbar_init(smem_u32(&bar_merge), 128);
    mbar_init(smem_u32(&bar_o1_free), 128);
    for (int i = 0; i < C::NSLOT; ++i) {
      mbar_init(smem_u32(&bar_kv_full[i]), 1);
      mbar_init(smem_u32(&bar_kv_empty[i]), 1);
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(smem_u32(&bar_s_full[w]), 1);
      mbar_init(smem_u32(&bar_p_full[w]), 128);
      mbar_init(smem_u32(&bar_pv_done[w]), 1);
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

  const uint32_t sQ = smem_u32(smem + C::SMEM_Q);
  const uint32_t sRing = smem_u32(smem + C::SMEM_RING);
  const uint32_t sStg = smem_u32(smem + C::SMEM_STG);
  float* merge_m = reinterpret_cast<float*>(smem + C::SMEM_MERGE);
  float* merge_l = merge_m + C::BQ;

  if (warp == 8) {
    // ------------------------------------------------------------ K producer
    // Chunk c of this CTA's item r is its chunk r n + c: K slot (r n + c) % KSLOTS.
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
    }
    const uint64_t keep = policy_evict_last();  // pool rows recur in nearby tokens' lists
    int q_loads = 0, last_k = -1;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int item = r * n_cta + cta;
      if (item >= n_items) break;
      const int b = item / p.T;
      const int* lst = p.idx + static_cast<size_t>(item) * p.K;
      const int row0 = b * p.P;
      auto load_k = [&](int c) {
        const int g = r * nch + c;  // chunk index over this CTA's items
        const int slot = g % C::KSLOTS, round = g / C::KSLOTS;
        const int s0 = c * C::BK + 4 * lane;
        int4 e = make_int4(-1, -1, -1, -1);
        if (s0 < p.K) e = __ldg(reinterpret_cast<const int4*>(lst + s0));
        auto row = [&](int x) { return row0 + ((x >= 0 && x < p.P) ? x : 0); };
        if (round > 0) ok = mbar_wait_warp(smem_u32(&bar_kv_empty[slot]), (round - 1) & 1, ctl);
        if (!ok) return;
        const uint32_t full = smem_u32(&bar_kv_full[slot]);
        const uint32_t dst = sRing + slot * C::SLOT_BYTES + lane * 4 * 128;
        mbar_arrive_expect_tx_el(full, C::K_BYTES);
        __syncwarp();
#pragma unroll
        for (int cb = 0; cb < C::KCH; ++cb)
          tma_gather4(dst + cb * (C::BK * 128), &tm_k, full, cb * 64, row(e.x), row(e.y), row(e.z),
                      row(e.w), keep);
        last_k = g;
      };
      // The first chunk's K, then Q once the previous item's last S product
      // has read the Q buffer, then the remaining chunks' K.
      if (r > 0) load_k(0);
      if (!ok) break;
      if (r > 0) ok = mbar_wait_warp(smem_u32(&bar_q_empty), (r - 1) & 1, ctl);
      if (!ok) break;
      mbar_arrive_expect_tx_el(smem_u32(&bar_q_full), C::Q_BYTES);
      for (int cb = 0; cb < C::KCH; ++cb)
        tma_load_2d_el(sQ + cb * (C::BQ * 128), &tm_q, smem_u32(&bar_q_full), cb * 64,
                       item * p.H);
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
  } else if (warp == 10) {
    // ------------------------------------------------------------ V producer
    // Each copy instruction of the warp moves UNITS 16-byte units of each of
    // 32 / UNITS rows (whole rows, contiguous in global memory); row j's unit
    // u lands at j * 128 + ((u % 8) ^ (j % 8)) * 16 in 64-column block u / 8.
    // V_IN_FLIGHT chunks' copies stay in flight: V_c is reported once V_{c+1}
    // has been issued (releasing an earlier V chunk needs nothing later).
    int* idx_s = reinterpret_cast<int*>(smem + C::SMEM_IDX);
    int issued = 0, signalled = 0;
    int pend[4];
    bool ok = true;
    auto signal_oldest = [&]() {
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bar_kv_full[pend[signalled & 3]]));
      ++signalled;
    };
    for (int r = 0; ok; ++r) {
      const int item = r * n_cta + cta;
      if (item >= n_items) break;
      const int b = item / p.T;
      const int* lst = p.idx + static_cast<size_t>(item) * p.K;
      for (int c = 0; c < nch && ok; ++c) {
        const int g = r * nch + c;
        const int slot = C::KSLOTS + g % C::VSLOTS, round = g / C::VSLOTS;
        __syncwarp();
        const int s0 = c * C::BK + 4 * lane;
        int4 e = make_int4(-1, -1, -1, -1);
        if (s0 < p.K) e = __ldg(reinterpret_cast<const int4*>(lst + s0));
        auto chk = [&](int x) { return (x >= 0 && x < p.P) ? x : -1; };
        reinterpret_cast<int4*>(idx_s)[lane] = make_int4(chk(e.x), chk(e.y), chk(e.z), chk(e.w));
        __syncwarp();
        if (round > 0) ok = mbar_wait_warp(smem_u32(&bar_kv_empty[slot]), (round - 1) & 1, ctl);
        if (!ok) break;
        const uint32_t dst = sRing + slot * C::SLOT_BYTES;
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
        pend[issued & 3] = slot;
        ++issued;
        if (issued - signalled > C::V_IN_FLIGHT) {
          cp_async_wait<C::V_IN_FLIGHT>();
          signal_oldest();
        }
      }
    }
    cp_async_wait<0>();
    while (signalled < issued) signal_oldest();
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    bool ok = !p.inject_stall;
    constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 0);
    constexpr uint32_t idesc_o = idesc_bf16_f32(128, DV, 0, 1);
    const uint64_t dq_desc = sw128_desc(sQ, 16, 1024);
    int p_cnt[2] = {0, 0};  // P tiles consumed per warpgroup, over all items
    for (int r = 0; ok; ++r) {
      const int item = r * n_cta + cta;
      if (item >= n_items) break;
      ok = mbar_wait_warp(smem_u32(&bar_q_full), r & 1, ctl);
      if (!ok) break;
      int s_left = nch;  // the last S product of the item hands the Q buffer back
      // Chunk c of this item is chunk r n + c of the CTA: its K slot and V slot.
      auto kslot = [&](int c) { return (r * nch + c) % C::KSLOTS; };
      auto vslot = [&](int c) { return C::KSLOTS + (r * nch + c) % C::VSLOTS; };
      auto wait_k = [&](int c) {
        return mbar_wait_warp(smem_u32(&bar_kv_full[kslot(c)]), ((r * nch + c) / C::KSLOTS) & 1, ctl);
      };
      auto wait_v = [&](int c) {
        return mbar_wait_warp(smem_u32(&bar_kv_full[vslot(c)]), ((r * nch + c) / C::VSLOTS) & 1, ctl);
      };
      // S_w = Q K_c^T; K_c's slot is released once the product has run.
      auto issue_s = [&](int c) {
        const int w = c & 1;
        const uint64_t dk = sw128_desc(sRing + kslot(c) * C::SLOT_BYTES, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < DK / 16; ++kk) {
          const uint32_t koff = ((kk >> 2) * (128 * 128) + (kk & 3) * 32) >> 4;
          mma_ss_el(tmem + C::tm_s(w), dq_desc + koff, dk + koff, idesc_s, kk > 0);
        }
        mma_commit_el(smem_u32(&bar_s_full[w]));
        mma_commit_el(smem_u32(&bar_kv_empty[kslot(c)]));
        if (--s_left == 0) mma_commit_el(smem_u32(&bar_q_empty));
      };
      for (int c = 0; c < 2 && c < nch && ok; ++c) {
        ok = wait_k(c);
        if (!ok) break;
        tc_fence_after();
        issue_s(c);
      }
      for (int c = 0; c < nch && ok; ++c) {
        const int w = c & 1;
        ok = mbar_wait_warp(smem_u32(&bar_p_full[w]), p_cnt[w] & 1, ctl);
        if (!ok) break;
        ++p_cnt[w];
        ok = wait_v(c);
        if (!ok) break;
        tc_fence_after();
        // O_w += P_hi V_c + P_lo V_c: slots 16kk..16kk+15 hold P hi pairs in
        // score columns 16kk..16kk+7 and lo pairs in 16kk+8..16kk+15.
        const uint64_t dv = sw128_desc(sRing + vslot(c) * C::SLOT_BYTES, C::BK * 128, 1024);
        const uint32_t a_p = tmem + C::tm_s(w);
#pragma unroll
        for (int kk = 0; kk < C::BK / 16; ++kk)
          mma_ts_el(tmem + C::tm_o(w), a_p + kk * 16, dv + ((kk * 2048) >> 4), idesc_o,
                    (c >= 2 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < C::BK / 16; ++kk)
          mma_ts_el(tmem + C::tm_o(w), a_p + kk * 16 + 8, dv + ((kk * 2048) >> 4), idesc_o, 1u);
        mma_commit_el(smem_u32(&bar_kv_empty[vslot(c)]));
        if (c + 2 >= nch) mma_commit_el(smem_u32(&bar_pv_done[w]));
        // The next score tile of w overwrites P_w; MMAs run in issue order.
        if (c + 2 < nch) {
          ok = wait_k(c + 2);
          if (!ok) break;
          tc_fence_after();
          issue_s(c + 2);
        }
      }
    }
    mma_commit_el(smem_u32(&bar_mma_done));
    mbar_wait_drain(smem_u32(&bar_mma_done), 0, 50000000ull);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warps 0-7
    const int w = warp / 4;           // chunk parity of this warpgroup
    const int r = threadIdx.x % 128;  // head row == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp % 4) * 32) << 16;
    const uint32_t ts = tmem + lane_base + C::tm_s(w);
    const float sl2 = p.scale_log2;
    const bool pos = sl2 >= 0.f;
    const float lose = pos ? -INFINITY : INFINITY;
    const int my_n = chunks_of(nch, w);
    bool ok = true;
    int s_cnt = 0, pv_cnt = 0;
    for (int rr = 0; ok; ++rr) {
      const int item = rr * n_cta + cta;
      if (item >= n_items) break;
      const int b = item / p.T, t = item % p.T;
      const int* lst = p.idx + static_cast<size_t>(item) * p.K;
      float m = -INFINITY;  // running max in log2 units
      float l = 0.f;
      bool o1_checked = (w == 0) || rr == 0;
      for (int i = 0; i < my_n; ++i) {
        const int c = w + 2 * i;
        // Filled-slot bits of this chunk (bit s of word g is slot 32g + s),
        // parked in shared memory while the scores are in registers.
        bool all_filled;
        {
          uint32_t ball[4];
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const int s = c * C::BK + 32 * g + lane;
            const int e = s < p.K ? __ldg(lst + s) : -1;
            ball[g] = __ballot_sync(0xffffffffu, e >= 0 && e < p.P);
          }
          all_filled = (ball[0] & ball[1] & ball[2] & ball[3]) == 0xffffffffu;
          if (lane == 0) filled_s[warp] = make_uint4(ball[0], ball[1], ball[2], ball[3]);
          __syncwarp();
        }
        ok = mbar_wait_warp(smem_u32(&bar_s_full[w]), s_cnt & 1, ctl);
        if (!ok) break;
        ++s_cnt;
        tc_fence_after();
        float x[C::BK];
        {
          uint32_t u[C::BK];
#pragma unroll
          for (int cc = 0; cc < C::BK; cc += 32)
            tmem_ld32(ts + cc, *reinterpret_cast<uint32_t(*)[32]>(&u[cc]));
          tmem_wait_ld();
#pragma unroll
          for (int cc = 0; cc < C::BK; ++cc) x[cc] = __uint_as_float(u[cc]);
        }
        if (!all_filled) {
          const uint4 f4 = filled_s[warp];
          const uint32_t fw[4] = {f4.x, f4.y, f4.z, f4.w};
#pragma unroll
          for (int cc = 0; cc < C::BK; ++cc)
            if (!((fw[cc >> 5] >> (cc & 31)) & 1u)) x[cc] = lose;
        }
        const float mraw = pos ? extreme128<true>(x) : extreme128<false>(x);
        const float mx = mraw * sl2;
        float alpha = 1.f;
        const bool rescale = mx > m + kSparseRescale;
        if (rescale) {
          alpha = ex2(m - mx);  // m = -inf before the first filled chunk gives 0
          m = mx;
        }
        // A row with no filled slot so far keeps m = -inf; an offset of 0 then
        // gives its masked scores p = 0.
        const float neg_m = (m == -INFINITY) ? 0.f : -m;
        const uint64_t sl2x2 = f32x2(sl2, sl2), negm2 = f32x2(neg_m, neg_m);
        uint64_t sums[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) sums[k] = f32x2(0.f, 0.f);
#pragma unroll
        for (int ch = 0; ch < C::BK; ch += 16) {
          uint32_t pkl[16];  // P hi pairs, then P lo pairs
#pragma unroll
          for (int cc = 0; cc < 16; cc += 2) {
            float e0, e1;
            unpack_f32x2(fma_f32x2(f32x2(x[ch + cc], x[ch + cc + 1]), sl2x2, negm2), e0, e1);
            const float p0 = ex2(e0), p1 = ex2(e1);
            sums[(cc / 2) & 3] = add_f32x2(sums[(cc / 2) & 3], f32x2(p0, p1));
            split_bf16x2_fma(p0, p1, pkl[cc / 2], pkl[8 + cc / 2]);
          }
          tmem_st16(ts + ch, pkl);
        }
        float s0, s1;
        unpack_f32x2(add_f32x2(add_f32x2(sums[0], sums[1]), add_f32x2(sums[2], sums[3])), s0, s1);
        l = l * alpha + (s0 + s1);
        // Rescale this row of O_w (the commit of S_w(c) covered PV_w(c - 2)).
        if (i > 0 && __any_sync(0xffffffffu, rescale)) {
          const uint32_t to = tmem + lane_base + C::tm_o(w);
#pragma unroll
          for (int cc = 0; cc < DV; cc += 32) {
            uint32_t u[32];
            tmem_ld32(to + cc, u);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) u[k] = __float_as_uint(__uint_as_float(u[k]) * alpha);
            tmem_st32(to + cc, u);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        if (!o1_checked) {
          // Warpgroup 0 has read O_1 of the previous item: the first PV of
          // this item may overwrite it.
          ok = mbar_wait_warp(smem_u32(&bar_o1_free), (rr - 1) & 1, ctl);
          if (!ok) break;
          o1_checked = true;
        }
        mbar_arrive(smem_u32(&bar_p_full[w]));
      }
      if (ok && my_n > 0) {
        ok = mbar_wait_warp(smem_u32(&bar_pv_done[w]), pv_cnt & 1, ctl);
        ++pv_cnt;
      }
      if (w == 1) {
        // Hand (m, l) to warpgroup 0, which merges and stores the item.
        if (ok && !o1_checked) ok = mbar_wait_warp(smem_u32(&bar_o1_free), (rr - 1) & 1, ctl);
        if (!ok) break;
        merge_m[r] = m;
        merge_l[r] = l;
        tc_fence_before();
        mbar_arrive(smem_u32(&bar_merge));
        continue;
      }
      // ---- warpgroup 0: merge, normalise, store. Every warp of the group
      // reaches this consensus, also after one of its waits gave up, so none
      // can be left at the named barriers below.
      if (ok) ok = mbar_wait_warp(smem_u32(&bar_merge), rr & 1, ctl);
      ok = named_bar_and(1, 128, ok);
      if (!ok) break;
      tc_fence_after();
      const float m1 = merge_m[r], l1 = merge_l[r];
      const float mt = fmaxf(m, m1);
      const float f0 = l > 0.f ? ex2(m - mt) : 0.f;
      const float f1 = l1 > 0.f ? ex2(m1 - mt) : 0.f;
      const float lt = l * f0 + l1 * f1;
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      const float g0 = f0 * inv, g1 = f1 * inv;
      const bool use1 = chunks_of(nch, 1) > 0;
      const uint32_t to0 = tmem + lane_base + C::tm_o(0);
      const uint32_t to1 = tmem + lane_base + C::tm_o(1);
      const bool leader = (r == 0);
      // 64 columns at a time: both staging tiles (o, o_lo) are free once the
      // previous stores have read them; each 32-column half is combined and
      // written straight into them.
#pragma unroll
      for (int cb = 0; cb < DV; cb += 64) {
        if (leader) bulk_wait_read_all();
        named_bar_sync(1, 128);
#pragma unroll
        for (int h = 0; h < 4; ++h) {  // 16 columns: two 16-byte units per row
          uint32_t u[16], v[16];
          tmem_ld16(to0 + cb + 16 * h, u);
          if (use1) tmem_ld16(to1 + cb + 16 * h, v);
          tmem_wait_ld();
          uint32_t hi[8], lo[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            float x0 = __uint_as_float(u[2 * k]) * g0, x1 = __uint_as_float(u[2 * k + 1]) * g0;
            if (use1) {
              x0 = fmaf(__uint_as_float(v[2 * k]), g1, x0);
              x1 = fmaf(__uint_as_float(v[2 * k + 1]), g1, x1);
            }
            const uint32_t wv = pack_bf16x2(x0, x1);
            hi[k] = wv;
            lo[k] = pack_bf16x2(x0 - __uint_as_float(wv << 16),
                                x1 - __uint_as_float(wv & 0xFFFF0000u));
          }
          if (r < p.H) {
            // Row r: 128 bytes, 16-byte unit u8 at (u8 ^ (r % 8)) (128-byte swizzle).
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
              const uint32_t off = r * 128 + (((2 * h + q2) ^ (r & 7)) << 4);
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sStg + off),
                           "r"(hi[4 * q2]), "r"(hi[4 * q2 + 1]), "r"(hi[4 * q2 + 2]),
                           "r"(hi[4 * q2 + 3])
                           : "memory");
              if (write_lo)
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                 sStg + C::STG_BYTES + off),
                             "r"(lo[4 * q2]), "r"(lo[4 * q2 + 1]), "r"(lo[4 * q2 + 2]),
                             "r"(lo[4 * q2 + 3])
                             : "memory");
            }
          }
        }
        fence_async_smem();
        named_bar_sync(1, 128);
        if (leader) {
          tma_store_2d(&tm_o, cb, item * p.H, sStg);
          if (write_lo) tma_store_2d(&tm_olo, cb, item * p.H, sStg + C::STG_BYTES);
          bulk_commit_group();
        }
      }
      if (r < p.H)
        p.lse[(static_cast<size_t>(b) * p.H + r) * p.T + t] =
            lt > 0.f ? (mt + __log2f(lt)) * kLn2 : -INFINITY;
      // O_1 (and O_0) are read: the next item's first PV may overwrite them.
      tc_fence_before();
      mbar_arrive(smem_u32(&bar_o1_free));
    }
  }

  // The epilogue's TMA stores finish before the CTA's shared memory goes away.
  if (warp < 4 && threadIdx.x % 128 == 0) bulk_wait_all();
  tc_fence_before();
  __syncthreads();
  if (warp == 9) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int DK, int DV>
cudaError_t launch_sparse_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& to,
                                const CUtensorMap& tolo, bool write_lo,
                                const SparseFwdParams& p, cudaStream_t stream) {
  using C = SparseFwdCfg<DK, DV>;
  static bool attr_set[64] = {};
  static int sm_count[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attn_sparse_fwd_kernel<DK, DV>,
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
  attn_sparse_fwd_kernel<DK, DV><<<grid, C::THREADS, C::SMEM_ALLOC, stream>>>(
      tq, tk, to, tolo, write_lo ? 1 : 0, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sparse_fwd(int DK, int DV, const CUtensorMap& tq, const CUtensorMap& tk,
                              const CUtensorMap& to, const CUtensorMap& tolo, bool write_lo,
                              const SparseFwdParams& p, cudaStream_t stream) {
  if (DK == 128 && DV == 128) return launch_sparse_fwd_t<128, 128>(tq, tk, to, tolo, write_lo, p, stream);
  if (DK == 128 && DV == 64) return launch_sparse_fwd_t<128, 64>(tq, tk, to, tolo, write_lo, p, stream);
  if (DK == 64 && DV == 128) return launch_sparse_fwd_t<64, 128>(tq, tk, to, tolo, write_lo, p, stream);
  if (DK == 64 && DV == 64) return launch_sparse_fwd_t<64, 64>(tq, tk, to, tolo, write_lo, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attn
