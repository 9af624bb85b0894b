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
  float* const red_g = reinterpret_cast<float*>(gbase + static_cast<uint32_t>(S) * kStage);
  const uint32_t bars = red + red_bytes(ROWS, TOK);
  const uint32_t recv_bar = bars + 8u * (2 * S) + 8u;
  const uint32_t dbg_bar = recv_bar + 8u;
  auto full_bar = [&](int s) { return bars + 8u * static_cast<uint32_t>(s); };
  auto empty_bar = [&](int s) { return bars + 8u * static_cast<uint32_t>(S + s); };

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();

  if (p.debug_wait) {
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

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), kComputeWarps);
    }
    mbar_init(recv_bar, 1);
    if (csize > 1) mbar_arrive_expect_tx(recv_bar, (csize - 1) * RS * M * 4u);
    fence_mbar_init();
  }
  __syncthreads();
  if (csize > 1) cluster_arrive_release();

  float acc[MT][NT][4];
#pragma unroll
  for (int a = 0; a < MT; ++a)
#pragma unroll
    for (int b = 0; b < NT; ++b)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[a][b][c] = 0.0f;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tensormap(&wmap);
      prefetch_tensormap(&xmap);
      const uint64_t policy = l2_policy_evict_first();
      const int pro = iters < S ? iters : S;
      for (int it = 0; it < pro; ++it) {
        const int nbi = min(NBOX, nb - it * NBOX);
        const uint32_t st = base + static_cast<uint32_t>(it) * kStage;
        mbar_arrive_expect_tx(full_bar(it), nbi * (kWBox + kXBox));
        for (int b = 0; b < nbi; ++b)
          tma_load_2d_hint(st + b * kWBox, &wmap, (kb0 + it * NBOX + b) * kBoxK, n0, full_bar(it),
                           policy);
      }
      // Let the next kernel on the stream launch: its CTAs prefetch their own
      // weight tiles into whatever shared memory is free (they still wait for
      // our completion in griddepcontrol.wait before touching x or out).  By
      // default that happens now; with pdl_late it waits until this CTA has
      // issued (nearly) all of its weight loads, so the next grid's first
      // loads queue up behind ours instead of competing with them.
      const int trig = p.pdl_late > 0 ? max(pro, iters - p.pdl_late + 1) : pro;
      if (trig == pro) pdl_launch_dependents();
      pdl_wait();
      for (int it = 0; it < pro; ++it) {
        const int nbi = min(NBOX, nb - it * NBOX);
        const uint32_t st = base + static_cast<uint32_t>(it) * kStage + NBOX * kWBox;
        for (int b = 0; b < nbi; ++b)
          tma_load_2d(st + b * kXBox, &xmap, (kb0 + it * NBOX + b) * kBoxK, 0, full_bar(it));
      }
      for (int it = pro; it < iters; ++it) {
        if (it == trig) pdl_launch_dependents();
        const int s = it % S;
        const uint32_t ph = static_cast<uint32_t>((it / S) - 1) & 1u;
        if (!mbar_wait_bounded(empty_bar(s), ph, p.timeout_ns))
          report_status(p.status, kStatusTimeoutEmpty);
        const int nbi = min(NBOX, nb - it * NBOX);
        const uint32_t st = base + static_cast<uint32_t>(s) * kStage;
        mbar_arrive_expect_tx(full_bar(s), nbi * (kWBox + kXBox));
        for (int b = 0; b < nbi; ++b)
          tma_load_2d_hint(st + b * kWBox, &wmap, (kb0 + it * NBOX + b) * kBoxK, n0, full_bar(s),
                           policy);
        for (int b = 0; b < nbi; ++b)
          tma_load_2d(st + NBOX * kWBox + b * kXBox, &xmap, (kb0 + it * NBOX + b) * kBoxK, 0,
                      full_bar(s));
      }
      if (trig == iters && trig != pro) pdl_launch_dependents();
    }
    __syncwarp();
  } else {
    pdl_wait();
    const int cw = static_cast<int>(warp) - 1;
    const int row_base = cw * MT * 16;
    for (int it = 0; it < iters; ++it) {
      const int s = it % S;
      const uint32_t ph = static_cast<uint32_t>(it / S) & 1u;
      if (!mbar_wait_bounded(full_bar(s), ph, p.timeout_ns))
        report_status(p.status, kStatusTimeoutFull);
      const int nbi = min(NBOX, nb - it * NBOX);
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
            ldsm_x4(wb + row * 128u + ((chunk ^ (row & 7u)) << 4), a[mt][0], a[mt][1], a[mt][2],
                    a[mt][3]);
          }
          if constexpr (TOK == 8) {
            const uint32_t tr = lane & 7u;
            const uint32_t chunk = static_cast<uint32_t>(2 * j) + ((lane >> 3) & 1u);
            uint32_t b0, b1;
            ldsm_x2(xb + tr * 128u + ((chunk ^ (tr & 7u)) << 4), b0, b1);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) mma_16816<kFp16>(acc[mt][0], a[mt], b0, b1);
          } else {
#pragma unroll
            for (int np = 0; np < NT / 2; ++np) {
              const uint32_t tr = static_cast<uint32_t>(np * 16) + ((lane >> 4) << 3) + (lane & 7u);
              const uint32_t chunk = static_cast<uint32_t>(2 * j) + ((lane >> 3) & 1u);
              uint32_t b00, b01, b10, b11;
              ldsm_x4(xb + tr * 128u + ((chunk ^ (tr & 7u)) << 4), b00, b01, b10, b11);
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
  if (csize > 1) cluster_wait_acquire();
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
            if (t < M) red_g[(rank * TOK + t) * RS + rs] = acc[mt][nt][2 * h];
            if (t + 1 < M) red_g[(rank * TOK + t + 1) * RS + rs] = acc[mt][nt][2 * h + 1];
          }
        } else {
          const uint32_t raddr = mapa_shared(red + ((rank * TOK) * RS + rs) * 4u, owner);
          const uint32_t rbar = mapa_shared(recv_bar, owner);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const int t = nt * 8 + 2 * q;
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
    // its K range (at most iters + 1 stages): keep waiting that many more
    // rounds, so this CTA does not exit while a peer may still push into it.
    for (int r = 0; r < iters + 2; ++r)
      if (mbar_wait_bounded<true>(recv_bar, 0, p.timeout_ns)) break;
  }
  const int nbase = n0 + static_cast<int>(rank) * RS;
  for (int idx = threadIdx.x; idx < RS * M; idx += blockDim.x) {
    const int rs2 = idx % RS;
    const int t = idx / RS;
    float sum = 0.0f;
    for (uint32_t k = 0; k < csize; ++k) sum += red_g[(k * TOK + t) * RS + rs2];
    const int n = nbase + rs2;
    if (n < p.N) store_out<OutT>(p, t, n, sum);
  }
  if (threadIdx.x == 0) {
    const int used = iters < S ? iters : S;
    for (int s = 0; s < used; ++s) {
      const int last = s + ((iters - 1 - s) / S) * S;
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
