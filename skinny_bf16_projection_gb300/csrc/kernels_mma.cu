// Warp split-K skinny projection on mma.sync (m16n8k16) fed by TMA.
//
//   out[M, N] = x[M, K] @ W[N, K]^T,  M <= 32, swap-AB: the weight tile is
//   the MMA's A operand (16 weight rows per fragment), the tokens its B
//   operand (8 tokens per fragment).
//
// Prior art: page "vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.
// gemm.warp_splitk", module docstring (weight streamed with an L2 evict_first
// hint, one tile issued before the PDL wait, activations after it, four MMA
// warps, small output tiles so many CTAs share an SM) and its fragment
// helpers (A = 16 weight rows x 16 k per ldmatrix.x4, 16-byte chunks XORed
// with row % 8).  Differences here: the weight and the activations both come
// through TMA boxes written with the hardware 128-byte swizzle (same XOR
// pattern) instead of per-thread cp.async, every stage's weight box count is
// a tactic parameter, and the four compute warps split the tile's ROWS (each
// warp 16*MT rows, all K of the stage) so no intra-CTA reduction is needed;
// the split-K across CTAs goes through the cluster reduction below.
//
//   warp 0 lane 0  TMA producer (same protocol as the tcgen05 kernel)
//   warps 1-4      ldmatrix + mma.sync over every box of each stage, fp32
//                  accumulators in registers; then push partial sums to the
//                  owning CTA of the cluster (st.async) and reduce in rank order.
#include "device_common.cuh"

namespace skg {

template <int MT, int TOK, int NBOX, typename OutT, bool kFp16>
__global__ void __launch_bounds__(160) skinny_mma_kernel(const __grid_constant__ CUtensorMap wmap,
                                                       const __grid_constant__ CUtensorMap xmap,
                                                       const KParams p) {
  constexpr int kComputeWarps = 4;
  constexpr int ROWS = 16 * MT * kComputeWarps;
  constexpr int NT = TOK / 8;
  constexpr uint32_t kWBox = ROWS * kBoxRowBytes;
  constexpr uint32_t kXBox = TOK * kBoxRowBytes;
  constexpr uint32_t kStage = stage_bytes(ROWS, TOK, NBOX);
  static_assert(TOK == 8 || TOK % 16 == 0, "token tile");

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + kSmemAlign - 1) & ~static_cast<uint32_t>(kSmemAlign - 1);
  uint8_t* const gbase = smem_raw + (base - raw);
  const int S = p.stages;
  const uint32_t red = base + static_cast<uint32_t>(S) * kStage;
  const uint32_t stages_end = red;  // (checked build only)
  const uint32_t red_words = static_cast<uint32_t>(ROWS * TOK);
  float* const red_g = reinterpret_cast<float*>(gbase + static_cast<uint32_t>(S) * kStage);
  const uint32_t bars = red + red_bytes(ROWS, TOK);
  const uint32_t recv_bar = bars + 8u * (2 * S) + 8u;
  const uint32_t dbg_bar = recv_bar + 8u;
  auto full_bar = [&](int s) { return bars + 8u * static_cast<uint32_t>(s); };
  auto empty_bar = [&](int s) { return bars + 8u * static_cast<uint32_t>(S + s); };

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();

  if (p.debug_wait) {
    // Checked-build self-test: one failed check, reported like a real one; no access.
    if (p.debug_wait == 2) {
      if (threadIdx.x == 0) skg_check(false, p.status, kCheckSelfTest);
      return;
    }
    if (threadIdx.x == 0) {
      mbar_init(dbg_bar, 1);
      fence_mbar_init();
    }
    __syncthreads();
    if (!mbar_wait_bounded(dbg_bar, 0, p.timeout_ns)) report_status(p.status, kStatusTimeoutDebug);
    return;
  }

  const uint32_t csize = cluster_nctarank();
  const uint32_t rank = cluster_ctarank();
  const int n0 = static_cast<int>(blockIdx.x / csize) * ROWS;
  const int kb0 = static_cast<int>(static_cast<int64_t>(rank) * p.kboxes / csize);
  const int kb1 = static_cast<int>(static_cast<int64_t>(rank + 1) * p.kboxes / csize);
  const int nb = kb1 - kb0;
  const int iters = (nb + NBOX - 1) / NBOX;
  const int RS = ROWS / static_cast<int>(csize);
  const int M = p.M;
  // Run-time K sharing: the first stages hold fixed boxes (stage j of rank r:
  // boxes starting at (j * csize + r) * NBOX), later ones whatever the
  // cluster's counter hands out, so the CTAs of a cluster finish together.
  const bool dyn = p.dyn_k != 0 && csize > 1;
  const uint32_t dyn_area = bars + 8u * (2 * S + 4) + 16u;  // [counter | pad | counts[16]]
  volatile uint32_t* const stage_boxes =
      reinterpret_cast<volatile uint32_t*>(gbase + (dyn_area + 16u - base));

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), kComputeWarps);
    }
    mbar_init(recv_bar, 1);
    if (csize > 1) mbar_arrive_expect_tx(recv_bar, (csize - 1) * RS * M * 4u);
    if (dyn && rank == 0)  // boxes below S * csize * NBOX belong to the first stages
      *reinterpret_cast<volatile uint32_t*>(gbase + (dyn_area - base)) =
          static_cast<uint32_t>(S) * csize * NBOX;
    fence_mbar_init();
  }
  __syncthreads();
  if (csize > 1) cluster_arrive_release();  // counter and receive barrier initialised
  bool start_waited = false;  // the producer waits for that before its first counter use
  int n_armed = 0;            // producer: pipeline iterations armed (the drain below)

  float acc[MT][NT][4];
#pragma unroll
  for (int a = 0; a < MT; ++a)
#pragma unroll
    for (int b = 0; b < NT; ++b)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[a][b][c] = 0.0f;

  if (warp == 0) {
    // Producer state (lane 0's copy is the one used).
    int pro = 0, trig = 0;
    bool triggered = false;
    uint64_t policy = 0;
    if (lane == 0) {
      prefetch_tensormap(&wmap);
      prefetch_tensormap(&xmap);
      policy = l2_policy_evict_first();
      // First box and box count of pipeline iteration `it` (fixed assignment;
      // with dyn only the first S iterations, the prologue, are fixed).
      auto fixed_box = [&](int it) {
        return dyn ? (it * static_cast<int>(csize) + static_cast<int>(rank)) * NBOX : kb0 + it * NBOX;
      };
      auto fixed_count = [&](int it, int b0) {
        return dyn ? max(0, min(NBOX, p.kboxes - b0)) : min(NBOX, nb - it * NBOX);
      };
      for (; pro < S && (dyn || pro < iters); ++pro) {
        const int b0 = fixed_box(pro);
        const int nbi = fixed_count(pro, b0);
        if (nbi <= 0) break;
        if (dyn) stage_boxes[pro] = static_cast<uint32_t>(nbi);
        const uint32_t st = base + static_cast<uint32_t>(pro) * kStage;
        mbar_arrive_expect_tx(full_bar(pro), nbi * (kWBox + kXBox));
        for (int b = 0; b < nbi; ++b)
          if (skg_check(st + (b + 1) * kWBox <= stages_end && ((b0 + b) * kBoxK) % 8 == 0, p.status,
                        kCheckTmaW))
            tma_load_2d_hint(st + b * kWBox, &wmap, (b0 + b) * kBoxK, n0, full_bar(pro), policy);
      }
      // The weight boxes of the next l2_pre stages go to L2 now: these requests
      // queue behind the previous grid's last loads and are served while it
      // finishes, and the refills after the wait then read them from L2.
      if (!dyn)
        for (int it = pro; it < iters && it < pro + p.l2_pre; ++it)
          for (int b = 0; b < min(NBOX, nb - it * NBOX); ++b)
            tma_prefetch_2d(&wmap, (kb0 + it * NBOX + b) * kBoxK, n0);
      // Let the next kernel on the stream launch: its CTAs prefetch their own
      // weight tiles into whatever shared memory is free (they still wait for
      // our completion in griddepcontrol.wait before touching x or out).  By
      // default that happens now; with pdl_late it waits until this CTA has
      // issued (nearly) all of its weight loads, so the next grid's first
      // loads queue up behind ours instead of competing with them (with dyn
      // the iteration count is estimated by the fixed split's).
      trig = p.pdl_late > 0 ? max(pro, iters - p.pdl_late + 1) : pro;
      triggered = trig == pro;
      if (triggered) pdl_launch_dependents();
      pdl_wait();
      for (int it = 0; it < pro; ++it) {
        const int b0 = fixed_box(it);
        const int nbi = fixed_count(it, b0);
        const uint32_t st = base + static_cast<uint32_t>(it) * kStage + NBOX * kWBox;
        for (int b = 0; b < nbi; ++b)
          if (skg_check(st + (b + 1) * kXBox <= stages_end, p.status, kCheckTmaX))
            tma_load_2d(st + b * kXBox, &xmap, (b0 + b) * kBoxK, 0, full_bar(it));
      }
    }
    __syncwarp();
    if (dyn) {
      // The whole warp, converged (the cluster barrier is only ever used by
      // complete warps): rank 0's counter is initialised.
      cluster_wait_acquire();
      start_waited = true;
    }
    if (lane == 0) {
      const uint32_t counter = dyn ? mapa_shared(dyn_area, 0) : 0u;
      // (dyn) the next chunk is taken from the counter as soon as the previous
      // one's loads are issued, so the remote atomic's round trip overlaps the
      // wait for a free stage instead of delaying the refill
      int next_b0 = dyn ? static_cast<int>(atom_add_cluster_u32(counter, NBOX)) : 0;
      int it = pro;
      for (;; ++it) {
        if (!dyn && it >= iters) break;
        if (it == trig && !triggered) {
          pdl_launch_dependents();
          triggered = true;
        }
        const int s = it % S;
        if (it >= S) {
          const uint32_t ph = static_cast<uint32_t>((it / S) - 1) & 1u;
          if (!mbar_wait_bounded(empty_bar(s), ph, p.timeout_ns))
            report_status(p.status, kStatusTimeoutEmpty);
        }
        const int b0 = dyn ? next_b0 : kb0 + it * NBOX;
        const int nbi = dyn ? max(0, min(NBOX, p.kboxes - b0)) : min(NBOX, nb - it * NBOX);
        if (nbi <= 0) {  // (dyn) the cluster's boxes are all handed out: tell the consumers
          stage_boxes[s] = 0u;
          mbar_arrive(full_bar(s));
          ++it;
          break;
        }
        if (dyn) stage_boxes[s] = static_cast<uint32_t>(nbi);
        const uint32_t st = base + static_cast<uint32_t>(s) * kStage;
        mbar_arrive_expect_tx(full_bar(s), nbi * (kWBox + kXBox));
        for (int b = 0; b < nbi; ++b)
          if (skg_check(st + (b + 1) * kWBox <= stages_end && ((b0 + b) * kBoxK) % 8 == 0, p.status,
                        kCheckTmaW))
            tma_load_2d_hint(st + b * kWBox, &wmap, (b0 + b) * kBoxK, n0, full_bar(s), policy);
        for (int b = 0; b < nbi; ++b)
          if (skg_check(st + NBOX * kWBox + (b + 1) * kXBox <= stages_end, p.status, kCheckTmaX))
            tma_load_2d(st + NBOX * kWBox + b * kXBox, &xmap, (b0 + b) * kBoxK, 0, full_bar(s));
        if (dyn) next_b0 = static_cast<int>(atom_add_cluster_u32(counter, NBOX));
      }
      n_armed = it;
      if (!triggered) pdl_launch_dependents();
    }
    __syncwarp();
  } else {
    pdl_wait();
    const int cw = static_cast<int>(warp) - 1;
    const int row_base = cw * MT * 16;
    // (dyn: a CTA consumes at most every box of the K range, plus the end marker)
    const int max_it = dyn ? (p.kboxes + NBOX - 1) / NBOX + 1 : iters;
    for (int it = 0; it < max_it; ++it) {
      const int s = it % S;
      const uint32_t ph = static_cast<uint32_t>(it / S) & 1u;
      // (one decision per warp, so the warp stays converged for the cluster barrier)
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(full_bar(s), ph, p.timeout_ns))) {
        report_status(p.status, kStatusTimeoutFull);
        if (dyn) break;  // the stage's box count cannot be trusted
      }
      const int nbi = dyn ? static_cast<int>(stage_boxes[s]) : min(NBOX, nb - it * NBOX);
      if (nbi <= 0) break;
      const uint32_t wst = base + static_cast<uint32_t>(s) * kStage;
      const uint32_t xst = wst + NBOX * kWBox;
      for (int b = 0; b < nbi; ++b) {
        const uint32_t wb = wst + b * kWBox;
        const uint32_t xb = xst + b * kXBox;
#pragma unroll
        for (int j = 0; j < kBoxK / 16; ++j) {
          uint32_t a[MT][4];
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const uint32_t row = static_cast<uint32_t>(row_base + mt * 16) + (lane & 15u);
            const uint32_t chunk = static_cast<uint32_t>(2 * j) + (lane >> 4);
            const uint32_t aaddr = wb + row * 128u + ((chunk ^ (row & 7u)) << 4);
            // (a failing lane reads the box start instead, so the collective stays warp-wide)
            const bool aok = skg_check(aaddr >= wb && aaddr + 16u <= wb + kWBox, p.status, kCheckMmaOperand);
            ldsm_x4(aok ? aaddr : wb, a[mt][0], a[mt][1], a[mt][2], a[mt][3]);
          }
          if constexpr (TOK == 8) {
            const uint32_t tr = lane & 7u;
            const uint32_t chunk = static_cast<uint32_t>(2 * j) + ((lane >> 3) & 1u);
            uint32_t b0, b1;
            const uint32_t baddr = xb + tr * 128u + ((chunk ^ (tr & 7u)) << 4);
            const bool bok = skg_check(baddr >= xb && baddr + 16u <= xb + kXBox, p.status, kCheckMmaOperand);
            ldsm_x2(bok ? baddr : xb, b0, b1);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) mma_16816<kFp16>(acc[mt][0], a[mt], b0, b1);
          } else {
#pragma unroll
            for (int np = 0; np < NT / 2; ++np) {
              const uint32_t tr = static_cast<uint32_t>(np * 16) + ((lane >> 4) << 3) + (lane & 7u);
              const uint32_t chunk = static_cast<uint32_t>(2 * j) + ((lane >> 3) & 1u);
              uint32_t b00, b01, b10, b11;
              const uint32_t baddr = xb + tr * 128u + ((chunk ^ (tr & 7u)) << 4);
              const bool bok =
                  skg_check(baddr >= xb && baddr + 16u <= xb + kXBox, p.status, kCheckMmaOperand);
              ldsm_x4(bok ? baddr : xb, b00, b01, b10, b11);
#pragma unroll
              for (int mt = 0; mt < MT; ++mt) {
                mma_16816<kFp16>(acc[mt][2 * np], a[mt], b00, b01);
                mma_16816<kFp16>(acc[mt][2 * np + 1], a[mt], b10, b11);
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(s));
    }
  }

  // ------------------------------------------------------------ epilogue
  pdl_wait();  // every thread that reads residual / writes out is ordered after the previous grid
  if (csize > 1 && !start_waited) cluster_wait_acquire();
  if (warp > 0) {
    // Accumulator fragment: c0,c1 -> row g, tokens 2q, 2q+1; c2,c3 -> row g+8.
    const int cw = static_cast<int>(warp) - 1;
    const int g = static_cast<int>(lane >> 2);
    const int q = static_cast<int>(lane & 3u);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int row = cw * MT * 16 + mt * 16 + g + 8 * h;
        const uint32_t owner = static_cast<uint32_t>(row / RS);
        const int rs = row % RS;
        if (owner == rank) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const int t = nt * 8 + 2 * q;
            const uint32_t i0 = static_cast<uint32_t>((rank * TOK + t) * RS + rs);
            if (!skg_check(i0 + static_cast<uint32_t>(RS) < red_words, p.status, kCheckRedLocal)) continue;
            if (t < M) red_g[i0] = acc[mt][nt][2 * h];
            if (t + 1 < M) red_g[i0 + RS] = acc[mt][nt][2 * h + 1];
          }
        } else {
          const uint32_t raddr = mapa_shared(red + ((rank * TOK) * RS + rs) * 4u, owner);
          const uint32_t rbar = mapa_shared(recv_bar, owner);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const int t = nt * 8 + 2 * q;
            if (!skg_check(owner < csize &&
                               static_cast<uint32_t>((rank * TOK + t + 1) * RS + rs) < red_words,
                           p.status, kCheckRedRemote))
              continue;
            if (t < M) st_async_b32(raddr + static_cast<uint32_t>(t * RS * 4), acc[mt][nt][2 * h], rbar);
            if (t + 1 < M)
              st_async_b32(raddr + static_cast<uint32_t>((t + 1) * RS * 4), acc[mt][nt][2 * h + 1],
                           rbar);
          }
        }
      }
    }
  }
  __syncthreads();
  if (csize > 1 && !mbar_wait_bounded<true>(recv_bar, 0, p.timeout_ns)) {
    report_status(p.status, kStatusTimeoutRecv);
    // A live peer pushes after at most one bounded wait per pipeline stage of
    // its K range (at most iters + 1 stages; with dyn, every box of K): keep
    // waiting that many more rounds, so this CTA does not exit while a peer may
    // still push into it.
    const int rounds = (dyn ? (p.kboxes + NBOX - 1) / NBOX : iters) + 2;
    for (int r = 0; r < rounds; ++r)
      if (mbar_wait_bounded<true>(recv_bar, 0, p.timeout_ns)) break;
  }
  const int nbase = n0 + static_cast<int>(rank) * RS;
  for (int idx = threadIdx.x; idx < RS * M; idx += blockDim.x) {
    const int rs2 = idx % RS;
    const int t = idx / RS;
    float sum = 0.0f;
    if (!skg_check(static_cast<uint32_t>(((csize - 1) * TOK + t) * RS + rs2) < red_words, p.status,
                   kCheckRedRead))
      continue;
    for (uint32_t k = 0; k < csize; ++k) sum += red_g[(k * TOK + t) * RS + rs2];
    const int n = nbase + rs2;
    if (n < p.N) store_out<OutT>(p, t, n, sum);
  }
  if (threadIdx.x == 0) {  // the producer thread: every armed stage's last phase has landed
    const int used = n_armed < S ? n_armed : S;
    for (int s = 0; s < used; ++s) {
      const int last = s + ((n_armed - 1 - s) / S) * S;
      if (!mbar_wait_bounded(full_bar(s), static_cast<uint32_t>(last / S) & 1u, p.timeout_ns))
        report_status(p.status, kStatusTimeoutDrain);
    }
  }
}

#define SKG_MMA_ENTRY(MT, TOK, NBOX, OUTT, OUTCODE, FP16)                                   \
  KernelEntry {                                                                              \
    kVariantMma, 64 * MT, TOK, NBOX, FP16 ? 1 : 0, OUTCODE, 160,                             \
        reinterpret_cast<const void*>(&skinny_mma_kernel<MT, TOK, NBOX, OUTT, FP16>)         \
  }

#define SKG_MMA_ROW(MT, OUTT, OUTCODE)                                                       \
  SKG_MMA_ENTRY(MT, 8, 1, OUTT, OUTCODE, false), SKG_MMA_ENTRY(MT, 16, 1, OUTT, OUTCODE, false), \
      SKG_MMA_ENTRY(MT, 32, 1, OUTT, OUTCODE, false),                                       \
      SKG_MMA_ENTRY(MT, 8, 2, OUTT, OUTCODE, false), SKG_MMA_ENTRY(MT, 8, 4, OUTT, OUTCODE, false), \
      SKG_MMA_ENTRY(MT, 16, 2, OUTT, OUTCODE, false),                                        \
      SKG_MMA_ENTRY(MT, 16, 4, OUTT, OUTCODE, false),                                        \
      SKG_MMA_ENTRY(MT, 32, 2, OUTT, OUTCODE, false), SKG_MMA_ENTRY(MT, 32, 4, OUTT, OUTCODE, false)

// fp16 operands (both x and W): two 64-wide boxes per stage only.
#define SKG_MMA_ROW16(MT, OUTT, OUTCODE)                                                     \
  SKG_MMA_ENTRY(MT, 8, 2, OUTT, OUTCODE, true), SKG_MMA_ENTRY(MT, 16, 2, OUTT, OUTCODE, true), \
      SKG_MMA_ENTRY(MT, 32, 2, OUTT, OUTCODE, true)

static const KernelEntry kMmaTable[] = {
    SKG_MMA_ROW(1, __nv_bfloat16, 0), SKG_MMA_ROW(2, __nv_bfloat16, 0), SKG_MMA_ROW(1, float, 2),
    SKG_MMA_ROW(2, float, 2),         SKG_MMA_ROW16(1, __half, 1),      SKG_MMA_ROW16(2, __half, 1),
    SKG_MMA_ROW16(1, float, 2),       SKG_MMA_ROW16(2, float, 2)};

const KernelEntry* mma_kernel_table(int* count) {
  *count = static_cast<int>(sizeof(kMmaTable) / sizeof(kMmaTable[0]));
  return kMmaTable;
}

}  // namespace skg
