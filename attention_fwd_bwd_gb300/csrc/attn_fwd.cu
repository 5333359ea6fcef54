// Forward attention kernel for sm_103a: O = softmax(scale * Q K^T) V and the
// row log-sum-exp, per (batch, query head) -- "Scheduling Data to Compute:
// Hierarchical Data Pipelining for LLM Training on AMD GPUs", section 2.1,
// Eq. (1), computed as that section's Algorithm 0 describes (K/V tiles stream
// through on-chip memory, online softmax, output accumulator kept on chip),
// with the query-tile loop outside and the key/value loop inside so the state
// never leaves the SM.
//
// Per item: two 128-row query tiles (A and B) that share every K/V tile that
// streams in -- the same rows of two query heads of one kv group under causal
// GQA, else consecutive rows of one head (TileItem).
//   warp 8 (TMA producer): Q_A and Q_B once, then K_0, V_0, K_1, V_1, ... into
//       a ring of shared-memory slots, each guarded by a full/empty mbarrier
//       pair (the GB300 counterpart of the paper's "issue N+1 loads, wait
//       until at most N are outstanding" rule for its Tensor Data Mover,
//       section 3.1.1).
//   warp 9 (MMA issuer): S_t = Q_t K_j^T into tile t's TMEM score buffer (both
//       operands K-major, so K^T needs no transpose -- Table 3's first row),
//       and O_t += P_t V_j with P read from TMEM and V_j described MN-major
//       (the transposed-operand case of section 3.1.2, handled by the
//       descriptor instead of a transpose). The two tiles alternate on the
//       tensor core: while one tile's softmax runs, the other tile's MMAs do.
//       At D = 64, where each product is half as long and the issuer's own
//       waits dominate, warps 9 and 10 issue tile A's and tile B's products.
//   warps 0-3 / 4-7 (softmax of tile A / B): thread r owns query row r of its
//       tile (TMEM lane r); it reads its score row, updates the running max m
//       and writes P, rounded to bf16, over the scores in TMEM (at D = 64 into
//       TMEM columns of its own, so that the next score product need not wait
//       for the exponentials); when m grew by
//       more than 2^8 it first rescales its O row. It keeps two row sums: l,
//       of the fp32 probabilities, gives LSE = (m + log2 l) ln 2, and l_b, of
//       the bf16 values that actually enter P V, gives O = acc / l_b. Dividing
//       by l_b makes O an exact weighted mean of V rows whose weights are
//       within bf16 rounding of the softmax weights; dividing by l would add
//       the rounding's mean as a common scale error, which the backward's
//       Dvec = rowsum(dO * O) turns into a dQ error for sharp rows.
// When the caller asks for the output residual o_lo = bf16(O - o) (training,
// where the backward needs rowsum(dO * O) beyond bf16 accuracy), the epilogue
// also stores what the bf16 rounding of O dropped.
#include "attn_common.cuh"
#include "attn_items.cuh"
#include "sm100_ptx.cuh"

namespace attn {
using namespace ptx;

namespace {

#ifdef ATTN_TRACE
static __device__ unsigned long long g_attn_trace[kTraceCtas * kTraceRoles * kTraceEvents];
#endif

// Rescale threshold in log2 units: the running max used for exponentiation
// only moves when the true max exceeds it by more than this, which keeps every
// p <= 2^8 and leaves the result exact after the final division by l (or l_b).
constexpr float kRescaleThreshold = 8.0f;

// Largest (MAX) or smallest value of a 128-entry row, mostly with
// three-input max / min instructions.
template <bool MAX>
__device__ __forceinline__ float row_extreme128(const float (&x)[128]) {
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

// Eight K-steps of S = Q K^T (M = N = 128, D = 128) issued by one elected lane
// in a single asm block (one election, no branch): the descriptors advance
// 32 bytes per step inside a 128-byte swizzle row (+2 in the descriptor's
// 16-byte address units) and 16 KB per 64-column chunk (+1024).
__device__ __forceinline__ void mma_s8_el(uint32_t d, uint64_t a0, uint64_t b0, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred e, t, f;\n\t.reg .b64 a, b;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.eq.u32 t, 1, 1;\n\tsetp.eq.u32 f, 1, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, f;\n\t"
      "add.s64 a, %1, 2;\n\tadd.s64 b, %2, 2;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n\t"
      "add.s64 a, %1, 4;\n\tadd.s64 b, %2, 4;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n\t"
      "add.s64 a, %1, 6;\n\tadd.s64 b, %2, 6;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n\t"
      "add.s64 a, %1, 1024;\n\tadd.s64 b, %2, 1024;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n\t"
      "add.s64 a, %1, 1026;\n\tadd.s64 b, %2, 1026;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n\t"
      "add.s64 a, %1, 1028;\n\tadd.s64 b, %2, 1028;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n\t"
      "add.s64 a, %1, 1030;\n\tadd.s64 b, %2, 1030;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n\t}"
      ::"r"(d), "l"(a0), "l"(b0), "r"(idesc)
      : "memory");
}
// Eight K-steps of O += P V (A = P from tensor memory, 16 columns a step; B = V,
// 2048 bytes a step), one elected lane, one asm block; acc0 enables the
// accumulation of the first step.
__device__ __forceinline__ void mma_pv8_el(uint32_t d, uint32_t a0, uint64_t b0, uint32_t idesc,
                                           uint32_t acc0) {
  asm volatile(
      "{\n\t.reg .pred e, t, p;\n\t.reg .b32 a;\n\t.reg .b64 b;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.eq.u32 t, 1, 1;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
      "add.u32 a, %1, 16;\n\tadd.s64 b, %2, 128;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, t;\n\t"
      "add.u32 a, %1, 32;\n\tadd.s64 b, %2, 256;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, t;\n\t"
      "add.u32 a, %1, 48;\n\tadd.s64 b, %2, 384;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, t;\n\t"
      "add.u32 a, %1, 64;\n\tadd.s64 b, %2, 512;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, t;\n\t"
      "add.u32 a, %1, 80;\n\tadd.s64 b, %2, 640;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, t;\n\t"
      "add.u32 a, %1, 96;\n\tadd.s64 b, %2, 768;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, t;\n\t"
      "add.u32 a, %1, 112;\n\tadd.s64 b, %2, 896;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, t;\n\t}"
      ::"r"(d), "r"(a0), "l"(b0), "r"(idesc), "r"(acc0)
      : "memory");
}

// RESID: the epilogue also stores o_lo. WIN: sliding-window instantiation
// (p.window > 0); without it the window code compiles away. The kernel is
// persistent: each CTA loops over its work items, and every barrier keeps
// counting phases across items.
template <int D, bool RESID, bool WIN>
__global__ void __launch_bounds__(FwdCfg<D>::THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_o,
                    const __grid_constant__ CUtensorMap tm_olo, const FwdParams p,
                    const int pair) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  __shared__ uint64_t bar_q_full, bar_q_empty, bar_mma_done;
  __shared__ uint64_t bar_kv_full[C::NSLOT], bar_kv_empty[C::NSLOT];
  __shared__ uint64_t bar_s_full[2], bar_p_full[2], bar_pv_done[2];
  // Separate P columns only: S_t read out (s_free) and each P_t V done (pv_step).
  __shared__ uint64_t bar_s_free[2], bar_pv_step[2];
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
    mbar_init(smem_u32(&bar_q_empty), C::N_MMA);  // one commit per MMA warp
    mbar_init(smem_u32(&bar_mma_done), C::N_MMA);
    for (int i = 0; i < C::NSLOT; ++i) {
      mbar_init(smem_u32(&bar_kv_full[i]), 1);
      mbar_init(smem_u32(&bar_kv_empty[i]), C::N_MMA);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_u32(&bar_s_full[t]), 1);
      mbar_init(smem_u32(&bar_p_full[t]), 128);
      mbar_init(smem_u32(&bar_pv_done[t]), 1);
      mbar_init(smem_u32(&bar_s_free[t]), 128);
      mbar_init(smem_u32(&bar_pv_step[t]), 1);
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
  // At D = 64 the waits sleep until their phase completes (suspend-time hint),
  // so that waiting warps leave issue slots to the softmax warps (1% faster
  // there; no change at D = 128, which polls).

  const uint32_t sQ = smem_u32(smem + C::SMEM_Q);  // tile t at sQ + t * Q_BYTES
  const uint32_t sRing = smem_u32(smem + C::SMEM_RING);
  const uint32_t sStg = smem_u32(smem + C::SMEM_STG);  // tile t at sStg + t * STG_BYTES

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    // The whole warp runs this loop; each copy is issued by one elected lane.
    // Per item: the first K/V tile pair, then Q_A and Q_B once the previous
    // item's last S product has read the Q buffer, then the remaining K/V
    // tiles. Ring positions run on across items.
    TraceCursor tc;
    if (lane == 0) ATTN_TRACE_INIT(tc, 0);
    ATTN_TRACE_EV(tc, 1, 0);
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
    }
    const uint64_t keep = policy_evict_last();  // K/V tiles are re-read by G heads x tiles
    const int nkv_all = (p.S + C::BK - 1) / C::BK;
    (void)nkv_all;
    int issued = 0;   // ring positions issued
    int q_loads = 0;  // Q loads issued
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
        if (round > 0) ok = mbar_wait_warp<C::SEP_P>(smem_u32(&bar_kv_empty[slot]), (round - 1) & 1, ctl);
        if (!ok) return;
        ATTN_TRACE_EV(tc, 2, pos);  // slot free, issuing the load
        const int jl = jb + (idx >> 1);
        if (!bounds_ok(jl >= 0 && jl < nkv_all && it.b < p.B && it.g < p.Hkv, ctl)) {
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
      if (r > 0) ok = mbar_wait_warp<C::SEP_P>(smem_u32(&bar_q_empty), (r - 1) & 1, ctl);
      if (!ok) break;
      if (!bounds_ok(it.hq[0] >= 0 && it.hq[1] < p.Hq && it.qs[0] >= 0 &&
                         it.qs[1] < p.n_qblocks * 2 * C::BQ, ctl))
        break;
      mbar_arrive_expect_tx_el(smem_u32(&bar_q_full), 2 * C::Q_BYTES);
      for (int t = 0; t < 2; ++t)
        for (int c = 0; c < C::KCH; ++c)
          tma_load_4d_el(sQ + t * C::Q_BYTES + c * (C::BQ * 128), &tm_q, smem_u32(&bar_q_full),
                         c * 64, it.hq[t], it.qs[t], it.b);
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
  } else if (warp == 9 || (C::SEP_P && warp == 10)) {
    if constexpr (!C::SEP_P) {
      // ------------------------------------------------------------ MMA issuer
      // The whole warp runs this loop and builds the (warp-uniform) descriptors;
      // each MMA and commit is issued by one elected lane.
      TraceCursor tc;
      if (lane == 0) ATTN_TRACE_INIT(tc, 1);
      bool ok = !p.inject_stall;
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, 0, 1);
      const uint64_t dq_desc = sw128_desc(sQ, 16, 1024);
      int ring = 0;                // ring position of the item's first K/V tile
      int p_cnt[2] = {0, 0};       // P tiles consumed per query tile, over all items
      for (int r = 0; ok; ++r) {
        const int ii = fwd_item_index(r, cta, n_cta, n_items);
        if (ii < 0) break;
        const TileItem it = tile_item<WIN>(p, pair != 0, ii);
        const int jb = jlo(it, 0);
        const int n_kv = it.n_kv[1];  // tile B ends last; tile A starts first
        ok = mbar_wait_warp<C::SEP_P>(smem_u32(&bar_q_full), r & 1, ctl);
        if (!ok) break;
        ATTN_TRACE_EV(tc, 1, r);
        // S products left in this item; the last one hands the Q buffer back.
        int s_left = (it.n_kv[0] - jlo(it, 0)) + (it.n_kv[1] - jlo(it, 1));
        // Ring position of K_j is ring + 2 (j - jb), of V_j the one after it.
        // S_t = Q_t K_j^T into tile t's score buffer.
        auto issue_s = [&](int t, int j) {
          const int slot = (ring + 2 * (j - jb)) % C::NSLOT;
          const uint64_t dk = sw128_desc(sRing + slot * C::KV_BYTES, 16, 1024);
          const uint64_t dq = dq_desc + ((t * C::Q_BYTES) >> 4);
          static_assert(D == 128, "the batched issue covers D = 128");
          mma_s8_el(tmem + C::tm_s(t), dq, dk, idesc_s);
          mma_commit_el(smem_u32(&bar_s_full[t]));
          if (--s_left == 0) mma_commit_el(smem_u32(&bar_q_empty));
        };
        auto wait_kv = [&](int idx) {
          const int pos = ring + idx;
          return mbar_wait_warp<C::SEP_P>(smem_u32(&bar_kv_full[pos % C::NSLOT]), (pos / C::NSLOT) & 1, ctl);
        };
        auto kv_slot = [&](int idx) { return (ring + idx) % C::NSLOT; };
        ok = wait_kv(0);
        if (!ok) break;
        tc_fence_after();
        issue_s(0, jb);
        if (jlo(it, 1) == jb) issue_s(1, jb);
        mma_commit_el(smem_u32(&bar_kv_empty[kv_slot(0)]));  // K_jb is done once its S products ran
        ATTN_TRACE_EV(tc, 3, r);
        for (int j = jb; j < n_kv && ok; ++j) {
          bool v_ready = false, k_next_ready = false;
          for (int t = 0; t < 2 && ok; ++t) {
            if (j >= jlo(it, t) && j < it.n_kv[t]) {
              ok = mbar_wait_warp<C::SEP_P>(smem_u32(&bar_p_full[t]), p_cnt[t] & 1, ctl);
              if (!ok) break;
              ++p_cnt[t];
              ATTN_TRACE_EV(tc, 4 + t, j);  // P_t(j) ready seen
              if (!v_ready) {
                ok = wait_kv(2 * (j - jb) + 1);
                if (!ok) break;
                v_ready = true;
              }
              tc_fence_after();
              if (!bounds_ok(j >= 0 && j * C::BK < p.S, ctl)) {
                ok = false;
                break;
              }
              const int vslot = kv_slot(2 * (j - jb) + 1);
              const uint64_t dv = sw128_desc(sRing + vslot * C::KV_BYTES, C::BK * 128, 1024);
              // Keys 16kk..16kk+15: bf16 P pairs in score columns 16kk..16kk+7.
              const uint32_t a_p = tmem + C::tm_s(t);
              mma_pv8_el(tmem + C::tm_o(t), a_p, dv, idesc_o, j > jlo(it, t) ? 1u : 0u);
              if (j + 1 == it.n_kv[t]) mma_commit_el(smem_u32(&bar_pv_done[t]));
              ATTN_TRACE_EV(tc, 6 + t, j);  // PV_t(j) issued
            }
            // The next score tile of t overwrites P_t(j) in TMEM; MMAs execute in
            // issue order, so it runs after PV_t(j) has read P_t(j).
            if (j + 1 < it.n_kv[t] && j + 1 >= jlo(it, t)) {
              if (!k_next_ready) {
                ok = wait_kv(2 * (j - jb) + 2);
                if (!ok) break;
                k_next_ready = true;
                tc_fence_after();
              }
              issue_s(t, j + 1);
            }
          }
          if (!ok) break;
          // Release V_j and K_{j+1} when the MMAs issued on them complete. Every
          // ring tile has a use (with a window too, the tiles' ranges leave no
          // gap), so with a window these waits only make sure that no copy is in
          // flight when its slot is handed back.
          if constexpr (WIN) {
            if (!v_ready) ok = wait_kv(2 * (j - jb) + 1);
            if (ok && j + 1 < n_kv && !k_next_ready) {
              ok = wait_kv(2 * (j - jb) + 2);
              k_next_ready = ok;
            }
            if (!ok) break;
          }
          mma_commit_el(smem_u32(&bar_kv_empty[kv_slot(2 * (j - jb) + 1)]));
          if (k_next_ready) mma_commit_el(smem_u32(&bar_kv_empty[kv_slot(2 * (j - jb) + 2)]));
        }
        ring += 2 * (n_kv - jb);
      }
      // Every MMA issued finishes before TMEM is released (in a normal run the
      // epilogues have already waited for them).
      mma_commit_el(smem_u32(&bar_mma_done));
      mbar_wait_drain(smem_u32(&bar_mma_done), 0, 50000000ull);
      __syncwarp();
    } else {
      // ------------------------------------------------------------ MMA issuers (D = 64)
      // Warp 9 issues query tile A's products, warp 10 tile B's, so that each
      // tile's chain of waits and issues runs on its own and the two overlap on
      // the tensor core. The whole warp runs the loop and builds the
      // (warp-uniform) descriptors; one elected lane issues each run of MMAs
      // and commits. Ring slots and the Q buffer are handed back when both
      // warps' commits have arrived (barrier count 2).
      const int t = warp - 9;
      TraceCursor tc;
      if (lane == 0) ATTN_TRACE_INIT(tc, t == 0 ? 1 : 4);
      bool ok = !p.inject_stall;
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, 0, 1);
      const uint64_t dq = sw128_desc(sQ + t * C::Q_BYTES, 16, 1024);
      int ring = 0;   // ring position of the item's first K/V tile
      int p_cnt = 0;  // P tiles of this query tile consumed, over all items
      int s_iss = 0;  // score products of this query tile issued, over all items
      for (int r = 0; ok; ++r) {
        const int ii = fwd_item_index(r, cta, n_cta, n_items);
        if (ii < 0) break;
        const TileItem it = tile_item<WIN>(p, pair != 0, ii);
        const int jb = jlo(it, 0);
        const int n_kv = it.n_kv[1];  // tile B ends last; tile A starts first
        const int my_lo = jlo(it, t), my_n = it.n_kv[t];
        ok = mbar_wait_warp<C::SEP_P>(smem_u32(&bar_q_full), r & 1, ctl);
        if (!ok) break;
        ATTN_TRACE_EV(tc, 1, r);
        // This tile's S products left in the item; its last one hands this
        // warp's share of the Q buffer back.
        int s_left = my_n - my_lo;
        // Ring position of K_j is ring + 2 (j - jb), of V_j the one after it.
        // S_t = Q_t K_j^T into the tile's score columns, once the softmax has
        // read the previous S_t out of them.
        auto issue_s = [&](int j) {
          if (s_iss > 0) {
            ok = mbar_wait_warp<C::SEP_P>(smem_u32(&bar_s_free[t]), (s_iss - 1) & 1, ctl);
            if (!ok) return;
            tc_fence_after();
          }
          ++s_iss;
          const int slot = (ring + 2 * (j - jb)) % C::NSLOT;
          const uint64_t dk = sw128_desc(sRing + slot * C::KV_BYTES, 16, 1024);
          const bool last_s = --s_left == 0;
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t koff = ((kk >> 2) * (128 * 128) + (kk & 3) * 32) >> 4;
              mma_ss(tmem + C::tm_s(t), dq + koff, dk + koff, idesc_s, kk > 0);
            }
            mma_commit(smem_u32(&bar_s_full[t]));
            if (last_s) mma_commit(smem_u32(&bar_q_empty));
          }
          __syncwarp();
          ATTN_TRACE_EV(tc, 8, j);  // S_t(j) issued
        };
        auto wait_kv = [&](int idx) {
          const int pos = ring + idx;
          return mbar_wait_warp<C::SEP_P>(smem_u32(&bar_kv_full[pos % C::NSLOT]), (pos / C::NSLOT) & 1, ctl);
        };
        auto kv_slot = [&](int idx) { return (ring + idx) % C::NSLOT; };
        // S_t(j+1), if this tile has it.
        bool k_done = false;  // this step's K_{j+1} copy waited for
        auto next_s = [&](int j) {
          if (j + 1 < my_n && j + 1 >= my_lo) {
            ok = wait_kv(2 * (j - jb) + 2);
            if (!ok) return;
            k_done = true;
            tc_fence_after();
            issue_s(j + 1);
          }
        };
        // A slot is handed back once both warps have committed its release
        // (count 2). Each warp first waits for the copy of every ring tile it
        // releases, the tiles it does not read included: that copy lands only
        // after both warps released the slot's previous tile, so a warp that
        // runs ahead cannot arrive twice on one phase of the slot's barrier
        // (and hand back a tile the other warp has still to read).
        ok = wait_kv(0);
        if (!ok) break;
        tc_fence_after();
        if (my_lo == jb) {
          issue_s(jb);
          if (!ok) break;
        }
        // K_jb is done once the S products on it ran.
        mma_commit_el(smem_u32(&bar_kv_empty[kv_slot(0)]));
        ATTN_TRACE_EV(tc, 3, r);
        for (int j = jb; j < n_kv && ok; ++j) {
          k_done = false;
          bool v_done = false;
          // The next score product goes first, as soon as the softmax has read
          // the current scores.
          next_s(j);
          if (!ok) break;
          if (j >= my_lo && j < my_n) {
            // V_j first: it landed long before P_t(j) is ready.
            ok = wait_kv(2 * (j - jb) + 1);
            if (!ok) break;
            v_done = true;
            ok = mbar_wait_warp<C::SEP_P>(smem_u32(&bar_p_full[t]), p_cnt & 1, ctl);
            if (!ok) break;
            ++p_cnt;
            ATTN_TRACE_EV(tc, 4, j);  // P_t(j) ready seen
            tc_fence_after();
            if (!bounds_ok(j >= 0 && j * C::BK < p.S, ctl)) {
              ok = false;
              break;
            }
            const int vslot = kv_slot(2 * (j - jb) + 1);
            const uint64_t dv = sw128_desc(sRing + vslot * C::KV_BYTES, C::BK * 128, 1024);
            // Keys 16kk..16kk+15: bf16 P pairs in P columns 8kk..8kk+7.
            const uint32_t a_p = tmem + C::tm_p(t);
            const uint32_t acc0 = j > my_lo ? 1u : 0u;
            const bool last_pv = j + 1 == my_n;
            if (elect_one()) {
#pragma unroll
              for (int kk = 0; kk < C::BK / 16; ++kk)
                mma_ts(tmem + C::tm_o(t), a_p + kk * 8, dv + ((kk * 2048) >> 4), idesc_o,
                       kk > 0 ? 1u : acc0);
              mma_commit(smem_u32(&bar_pv_step[t]));
              if (last_pv) mma_commit(smem_u32(&bar_pv_done[t]));
            }
            __syncwarp();
            ATTN_TRACE_EV(tc, 6, j);  // PV_t(j) issued
          }
          if (!ok) break;
          // This warp's share of handing back V_j and K_{j+1} (arrives when the
          // MMAs it issued so far complete), after waiting for their copies if
          // it did not read them.
          if (!v_done) ok = wait_kv(2 * (j - jb) + 1);
          if (ok && j + 1 < n_kv && !k_done) ok = wait_kv(2 * (j - jb) + 2);
          if (!ok) break;
          if (elect_one()) {
            mma_commit(smem_u32(&bar_kv_empty[kv_slot(2 * (j - jb) + 1)]));
            if (j + 1 < n_kv) mma_commit(smem_u32(&bar_kv_empty[kv_slot(2 * (j - jb) + 2)]));
          }
          __syncwarp();
        }
        ring += 2 * (n_kv - jb);
      }
      // Every MMA issued finishes before TMEM is released (in a normal run the
      // epilogues have already waited for them); the barrier completes once
      // both warps' commits have arrived.
      mma_commit_el(smem_u32(&bar_mma_done));
      mbar_wait_drain(smem_u32(&bar_mma_done), 0, 50000000ull);
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ softmax warps 0-7
    const int t = warp / 4;           // query tile of this warpgroup
    const int r = threadIdx.x % 128;  // query row within the tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp % 4) * 32) << 16;
    const uint32_t ts = tmem + lane_base + C::tm_s(t);
    const float sl2 = p.scale_log2;
    const bool pos = sl2 >= 0.f;
    TraceCursor tc;
    if (lane == 0 && (warp == 0 || warp == 4)) ATTN_TRACE_INIT(tc, 2 + t);
    bool ok = true;
    int s_cnt = 0;  // score tiles of this query tile, over all items
    for (int item = 0; ok; ++item) {
      const int ii = fwd_item_index(item, cta, n_cta, n_items);
      if (ii < 0) break;
      const TileItem it = tile_item<WIN>(p, pair != 0, ii);
      const int qt0 = it.qs[t], b = it.b, hq = it.hq[t];  // this tile's first row, its head
      const int qrow = qt0 + r;
      const int my_kv = it.n_kv[t];
      float m = -INFINITY;  // running max in log2 units (scaled scores)
      float l = 0.f;        // row sum of the fp32 probabilities (for LSE)
      float lb = 0.f;       // row sum of the bf16 probabilities that enter P V (for O)
      for (int j = jlo(it, t); j < my_kv; ++j) {
        ATTN_TRACE_EV(tc, 1, j);  // start waiting for S_t(j)
        // S_t(j) landed. With P over S its commit also covers PV_t(j-1), so O_t
        // is current; with separate P columns that is waited for below.
        ok = mbar_wait_warp<C::SEP_P>(smem_u32(&bar_s_full[t]), s_cnt & 1, ctl);
        if (!ok) break;
        ++s_cnt;
        ATTN_TRACE_EV(tc, 2, j);  // S_t(j) landed
        tc_fence_after();
        // Raw scores of this row; the scale is folded into the exponent below.
        float x[C::BK];
        {
          uint32_t u[C::BK];
#pragma unroll
          for (int c = 0; c < C::BK; c += 32)
            tmem_ld32(ts + c, *reinterpret_cast<uint32_t(*)[32]>(&u[c]));
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < C::BK; ++c) x[c] = __uint_as_float(u[c]);
        }
        if constexpr (C::SEP_P) {
          // S_t(j) is in registers: the next score product may overwrite it.
          tc_fence_before();
          mbar_arrive(smem_u32(&bar_s_free[t]));
          ATTN_TRACE_EV(tc, 7, j);  // S_t(j) read out
        }
        const int k0 = j * C::BK;
        // Tiles that cross the causal diagonal, hold keys past S, or hold keys
        // below some row's window mask; the rest skip masking.
        const bool need_mask = (p.causal && k0 + C::BK - 1 > qt0) || (k0 + C::BK > p.S) ||
                               (WIN && k0 < qt0 + C::BQ - p.window);
        // Visible columns of this tile for this row: c_lo <= c <= c_hi.
        const int c_hi = (p.causal ? min(qrow, p.S - 1) : (p.S - 1)) - k0;
        const int c_lo = WIN ? qrow - p.window + 1 - k0 : 0;
        float alpha = 1.f;
        bool rescale = false, o_rescale = false;
        uint32_t pk[C::BK / 2];  // bf16 P pairs of the tile's keys
        // One tile of the online softmax: row max, exponentials, both row sums
        // and bf16 P; with P over S it goes into TMEM 16 columns at a time
        // (this thread has read all its scores already).
        {
          const bool MASKED = need_mask;
          // Largest scaled score: the max of the raw scores for scale >= 0, the
          // min for scale < 0 (masked keys pushed to the losing end).
          if (MASKED) {
            const float lose = pos ? -INFINITY : INFINITY;
            if constexpr (WIN) {
              // A window tile usually needs one side of the interval only (the
              // diagonal tile the causal end, the tile before it the window's
              // start): test only the sides some row of the warp needs.
              const bool lo_side = __any_sync(0xffffffffu, c_lo > 0);
              const bool hi_side = __any_sync(0xffffffffu, c_hi < C::BK - 1);
              if (lo_side && hi_side) {
#pragma unroll
                for (int c = 0; c < C::BK; ++c)
                  if (c > c_hi || c < c_lo) x[c] = lose;
              } else if (lo_side) {
#pragma unroll
                for (int c = 0; c < C::BK; ++c)
                  if (c < c_lo) x[c] = lose;
              } else if (hi_side) {
#pragma unroll
                for (int c = 0; c < C::BK; ++c)
                  if (c > c_hi) x[c] = lose;
              }
            } else {
#pragma unroll
              for (int c = 0; c < C::BK; ++c)
                if (c > c_hi) x[c] = lose;
            }
          }
          static_assert(C::BK == 128, "row_extreme128 covers one 128-key tile");
          const float mraw = pos ? row_extreme128<true>(x) : row_extreme128<false>(x);
          const float mx = mraw * sl2;
          rescale = mx > m + kRescaleThreshold;
          if (rescale) {
            // A row whose max was still -inf has O = 0 (all its p were 0), so
            // only rows with a finite max need their O rescaled below.
            o_rescale = m > -INFINITY;
            alpha = ex2(m - mx);  // m = -inf on the first tile gives 0
            m = mx;
          }
          const uint64_t sl2x2 = f32x2(sl2, sl2);
          // A row whose keys in this tile are all outside its window keeps
          // m = -inf; an offset of 0 then gives its masked scores p = 0.
          const float neg_m = (WIN && m == -INFINITY) ? 0.f : -m;
          const uint64_t negm2 = f32x2(neg_m, neg_m);
          uint64_t sums[2];
          float sb[4] = {0.f, 0.f, 0.f, 0.f};  // the bf16 values' sums, same grouping as sums
#pragma unroll
          for (int i = 0; i < 2; ++i) sums[i] = f32x2(0.f, 0.f);
#pragma unroll
          for (int ch = 0; ch < C::BK; ch += 16) {
#pragma unroll
            for (int c = 0; c < 16; c += 2) {
              float e0, e1;
              unpack_f32x2(fma_f32x2(f32x2(x[ch + c], x[ch + c + 1]), sl2x2, negm2), e0, e1);
              // A masked score is -inf (or +inf with a negative scale): its
              // exponent is -inf and its probability 0 (the scale is never 0).
              const float p0 = ex2(e0), p1 = ex2(e1);
              sums[(c / 2) & 1] = add_f32x2(sums[(c / 2) & 1], f32x2(p0, p1));
              const uint32_t w = pack_bf16x2(p0, p1);  // round to nearest even
              pk[(ch + c) / 2] = w;
              add_bf16x2_f32(w, sb[2 * ((c / 2) & 1)], sb[2 * ((c / 2) & 1) + 1]);
            }
            // Columns ch..ch+7 of the scores (already read) take these keys' P.
            if constexpr (!C::SEP_P)
              tmem_st8(ts + ch, *reinterpret_cast<const uint32_t(*)[8]>(&pk[ch / 2]));
          }
          float s0, s1, b0, b1;
          unpack_f32x2(add_f32x2(sums[0], sums[1]), s0, s1);
          b0 = sb[0] + sb[2];
          b1 = sb[1] + sb[3];
          l = l * alpha + (s0 + s1);
          lb = lb * alpha + (b0 + b1);
        }
        ATTN_TRACE_EV(tc, 3, j);  // exponentials done
        if constexpr (C::SEP_P) {
          // PV_t of the previous P (this item's or, for its first tile, the
          // previous item's last) has read the P columns and written O_t.
          if (s_cnt > 1) {
            ok = mbar_wait_warp<C::SEP_P>(smem_u32(&bar_pv_step[t]), (s_cnt - 2) & 1, ctl);
            if (!ok) break;
            tc_fence_after();
          }
          ATTN_TRACE_EV(tc, 8, j);  // PV_t(j-1) seen done
          const uint32_t tp = tmem + lane_base + C::tm_p(t);
#pragma unroll
          for (int c = 0; c < C::BK / 2; c += 32)
            tmem_st32(tp + c, *reinterpret_cast<const uint32_t(*)[32]>(&pk[c]));
        }
        // Rescale this warp's O rows (PV_t(j-1) has completed, see above).
        if (j > jlo(it, t) && __any_sync(0xffffffffu, o_rescale)) {
          const uint32_t to = tmem + lane_base + C::tm_o(t);
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
        mbar_arrive(smem_u32(&bar_p_full[t]));
        ATTN_TRACE_EV(tc, 4, j);  // P_t(j) stored and signalled
      }
      // The item's last P.V product of this tile has run: O_t is final. (Its
      // TMEM columns are free again once this epilogue has read them, which
      // is before this warpgroup signals the next item's first P.)
      if (ok) ok = mbar_wait_warp<C::SEP_P>(smem_u32(&bar_pv_done[t]), item & 1, ctl);
      ATTN_TRACE_EV(tc, 5, item);  // the item's O_t final: epilogue starts
      // The tile's four warps meet at named barriers in the epilogue: agree
      // first on going on.
      ok = named_bar_and(1 + t, 128, ok);
      if (ok) {
        tc_fence_after();
        // O = acc / l_b (and o_lo, what bf16 rounding of O dropped, itself in
        // bf16) leave 64 columns at a time through this tile's staging buffer
        // and TMA stores; rows past S are clipped by the store. (One 128-row
        // store per round after two 128-thread barriers measured up to 2%
        // slower than these per-warp rounds.)
        const float inv_l = 1.f / lb;
        const uint32_t to = tmem + lane_base + C::tm_o(t);
        // Each warp stages its own 32 rows (4 KB of the tile's staging buffer)
        // and stores them with its own 32-row TMA store.
        const int wr = (warp % 4) * 32;  // this warp's first row of the tile
        const uint32_t stg = sStg + t * C::STG_BYTES + wr * 128;
        const bool leader = (lane == 0);
#pragma unroll
        for (int c = 0; c < D; c += 64) {
          uint32_t hi[32], lo[32];  // bf16 pairs of this row's 64 columns
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t u[32];
            tmem_ld32(to + c + 32 * h, u);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float x0 = __uint_as_float(u[2 * i]) * inv_l;
              const float x1 = __uint_as_float(u[2 * i + 1]) * inv_l;
              const uint32_t w = pack_bf16x2(x0, x1);
              hi[16 * h + i] = w;
              lo[16 * h + i] = pack_bf16x2(x0 - __uint_as_float(w << 16),
                                           x1 - __uint_as_float(w & 0xFFFF0000u));
            }
          }
#pragma unroll
          for (int part = 0; part < (RESID ? 2 : 1); ++part) {
            const uint32_t* v = part ? lo : hi;
            // This warp's previous store has read its rows.
            if (leader) bulk_wait_read_all();
            __syncwarp();
            // Row r: 128 bytes, 16-byte unit u at (u ^ (r % 8)) (128-byte swizzle).
#pragma unroll
            for (int u8 = 0; u8 < 8; ++u8) {
              const uint32_t addr = stg + lane * 128 + ((u8 ^ (r & 7)) << 4);
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v[4 * u8]),
                           "r"(v[4 * u8 + 1]), "r"(v[4 * u8 + 2]), "r"(v[4 * u8 + 3])
                           : "memory");
            }
            fence_async_smem();
            __syncwarp();
            if (leader && bounds_ok(hq < p.Hq && b < p.B && qt0 >= 0, ctl)) {
              tma_store_4d(part ? &tm_olo : &tm_o, c, hq, qt0 + wr, b, stg);
              bulk_commit_group();
            }
          }
        }
        if (qrow < p.S && bounds_ok(b < p.B && hq < p.Hq && qrow >= 0, ctl))
          p.lse[(static_cast<size_t>(b) * p.Hq + hq) * p.S + qrow] = (m + __log2f(l)) * kLn2;
        ATTN_TRACE_EV(tc, 6, item);  // epilogue done
      }
    }
  }

  // The epilogue's TMA stores finish before the CTA (and its staging buffers) go away.
  if (warp < 8 && lane == 0) bulk_wait_all();
  tc_fence_before();
  __syncthreads();
  if (warp == 9) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int D, bool RESID, bool WIN>
cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& to, const CUtensorMap& tolo, const FwdParams& p,
                         cudaStream_t stream) {
  using C = FwdCfg<D>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D, RESID, WIN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  // Persistent: one CTA per SM (or per item, if fewer), each looping over its
  // items.
  static int sm_count[64] = {};
  if (dev < 64 && sm_count[dev] == 0)
    cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
  const bool pair = tile_pair_heads(p);  // see TileItem
  const long long n_items = tile_n_items(p, pair);
  const int sms = (dev < 64 && sm_count[dev] > 0) ? sm_count[dev] : 148;
  const dim3 grid(static_cast<unsigned>(n_items < sms ? n_items : sms));
  attn_fwd_kernel<D, RESID, WIN><<<grid, C::THREADS, C::SMEM_ALLOC, stream>>>(tq, tk, tv, to, tolo,
                                                                                 p, pair ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(int D, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, const CUtensorMap& tolo, const FwdParams& p,
                       cudaStream_t stream) {
  const bool split = p.o_lo != nullptr, win = p.window > 0;  // split: store o_lo
  if (D == 128) {
    if (win)
      return split ? launch_fwd_t<128, true, true>(tq, tk, tv, to, tolo, p, stream)
                   : launch_fwd_t<128, false, true>(tq, tk, tv, to, tolo, p, stream);
    return split ? launch_fwd_t<128, true, false>(tq, tk, tv, to, tolo, p, stream)
                 : launch_fwd_t<128, false, false>(tq, tk, tv, to, tolo, p, stream);
  }
  if (win)
    return split ? launch_fwd_t<64, true, true>(tq, tk, tv, to, tolo, p, stream)
                 : launch_fwd_t<64, false, true>(tq, tk, tv, to, tolo, p, stream);
  return split ? launch_fwd_t<64, true, false>(tq, tk, tv, to, tolo, p, stream)
               : launch_fwd_t<64, false, false>(tq, tk, tv, to, tolo, p, stream);
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
