// Split-K skinny projection on the 5th-generation tensor cores (tcgen05/TMEM).
//
//   out[M, N] = x[M, K] @ W[N, K]^T,  M <= 64, computed swap-AB: the MMA's M
//   dimension is 128 weight rows, its N dimension the token tile, so the
//   accumulator D[128 rows][TOK tokens] (fp32) lives in TMEM and the weight
//   tile is the MMA's A operand straight from TMA-written shared memory.
//
// Design points taken from the pages (page "vllm.models.glm5next.nvidia.
// specialized_decode.gemm", module docstring: split-K tcgen05 GEMM with a
// cluster DSMEM reduction and an evict-first weight TMA; page "vllm.models.
// kimi_k3.nvidia.specialized_decode.cutedsl.gemm.projection", weight_map: a
// TMA map of W with box {64, rows} and 128-byte swizzle; output view
// (cols, rows): the kernel holds C^T).  The kernel body is our own design:
//
//   warp 0 lane 0  TMA producer: W boxes for the first `stages` stages are
//                  issued BEFORE griddepcontrol.wait (the weight does not
//                  depend on the previous kernel), x boxes after it.
//   warp 1 lane 0  MMA issuer: 4 x tcgen05.mma (K = 16 each) per 64-wide box,
//                  tcgen05.commit releases the stage back to the producer.
//   warps 0-3      epilogue: tcgen05.ld of the 128 x TOK accumulator (warp w
//                  owns TMEM lanes 32w..32w+31 = weight rows), then either a
//                  direct store (cluster of 1) or the cluster split-K
//                  reduction: each CTA pushes the rows owned by peer j into
//                  j's shared memory with st.async (counted on j's mbarrier),
//                  and every CTA sums its ROWS/cluster rows over the cluster
//                  in rank order (deterministic) and writes them.
//
// The CTAs of one cluster hold disjoint K ranges of the same 128-row tile.
#include "device_common.cuh"

namespace skg {

template <int TOK, int NBOX, typename OutT, bool kFp16, int ROWS = 128>
__global__ void __launch_bounds__(128) skinny_tc_kernel(const __grid_constant__ CUtensorMap wmap,
                                                      const __grid_constant__ CUtensorMap xmap,
                                                      const KParams p) {
  constexpr uint32_t kWBox = ROWS * kBoxRowBytes;
  constexpr uint32_t kXBox = TOK * kBoxRowBytes;
  constexpr uint32_t kStage = stage_bytes(ROWS, TOK, NBOX);
  // TMEM is allocated in powers of two of at least 32 columns (48 tokens: 64)
  constexpr uint32_t kTmemCols = TOK <= 32 ? 32u : TOK <= 64 ? 64u : TOK <= 128 ? 128u : 256u;
  constexpr uint32_t kIdesc = mma_idesc<kFp16>(ROWS, TOK);
  constexpr uint32_t kStageRed = static_cast<uint32_t>(ROWS * TOK) * 4u;
  static_assert(TOK % 16 == 0 && TOK >= 16 && TOK <= 256, "MMA needs N % 16 == 0, N <= 256");
  static_assert(ROWS == 128 || ROWS == 64, "MMA M is 128 or 64 weight rows");

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + kSmemAlign - 1) & ~static_cast<uint32_t>(kSmemAlign - 1);
  uint8_t* const gbase = smem_raw + (base - raw);
  const int S = p.stages;
  const uint32_t csize = cluster_nctarank();
  // With red_alias the cluster receive buffer lives in the pipeline stages,
  // which are idle once every MMA has completed; peers push into it only after
  // the cluster barrier that each CTA arrives at from that point on.
  const bool alias = p.red_alias != 0 && csize > 1;
  const uint32_t stages_end = base + static_cast<uint32_t>(S) * kStage;
  const uint32_t smem_end = raw + dynamic_smem_bytes();  // (checked build only)
  const uint32_t bars = stages_end + (csize > 1 && !alias ? tc_red_bytes(TOK, ROWS) : 0u);
  const uint32_t done_bar = bars + 8u * (2 * S);
  const uint32_t recv_bar = done_bar + 8u;
  const uint32_t dbg_bar = done_bar + 16u;
  const uint32_t tmem_slot = bars + 8u * (2 * S + 4);
  volatile uint32_t* const tmem_slot_g =
      reinterpret_cast<volatile uint32_t*>(gbase + (tmem_slot - base));
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
    // Watchdog self-test: wait on a barrier nothing will complete, report, return.
    if (threadIdx.x == 0) {
      mbar_init(dbg_bar, 1);
      fence_mbar_init();
    }
    __syncthreads();
    if (!mbar_wait_bounded(dbg_bar, 0, p.timeout_ns)) report_status(p.status, kStatusTimeoutDebug);
    return;
  }

  const uint32_t rank = cluster_ctarank();
  const int n0 = static_cast<int>(blockIdx.x / csize) * ROWS;
  const int kb0 = static_cast<int>(static_cast<int64_t>(rank) * p.kboxes / csize);
  const int kb1 = static_cast<int>(static_cast<int64_t>(rank + 1) * p.kboxes / csize);
  const int nb = kb1 - kb0;
  const int iters = (nb + NBOX - 1) / NBOX;
  const int RS = ROWS / static_cast<int>(csize);
  // Token tile of this CTA (gridDim.y > 1 when M exceeds the tile): rows
  // m0 .. m0 + M - 1 of x and out.
  const int m0 = static_cast<int>(blockIdx.y) * TOK;
  const int M = min(TOK, p.M - m0);
  // Cluster reduction: for token tiles of 64 and more, bulk DSMEM copies of
  // [TOK][RS] fp32 blocks staged in the idle pipeline buffers (when they are
  // large enough), unless the tactic asks for per-thread st.async pushes
  // (red_stores), which smaller tiles always use.
  const bool bulk = csize > 1 && TOK >= 64 && p.red_stores == 0 &&
                    static_cast<uint32_t>(S) * kStage >= (alias ? 2u : 1u) * kStageRed;
  // Receive buffer: after the stages, or (aliased) at their start, or right
  // after the bulk path's staging area.
  const uint32_t red = !alias ? stages_end : (bulk ? base + kStageRed : base);
  // Run-time K sharing (not with the aliased receive buffer): the first stages
  // hold fixed boxes (stage j of rank r: boxes from (j * csize + r) * NBOX),
  // later ones whatever the cluster's counter in rank 0 hands out, so the CTAs
  // of a cluster finish their K work together.
  const bool dyn = p.dyn_k != 0 && csize > 1 && !alias;
  const uint32_t dyn_area = bars + 8u * (2 * S + 4) + 16u;  // [counter | pad | counts[16]]
  volatile uint32_t* const stage_boxes =
      reinterpret_cast<volatile uint32_t*>(gbase + (dyn_area + 16u - base));
  // (dyn: a CTA whose first fixed box lies beyond K gets no box at all)
  const bool has_work = dyn ? static_cast<int>(rank) * NBOX < p.kboxes : iters > 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(done_bar, 1);
    mbar_init(recv_bar, 1);
    if (csize > 1)
      mbar_arrive_expect_tx(recv_bar, bulk ? (csize - 1) * static_cast<uint32_t>(M * RS) * 4u
                                           : (csize - 1) * RS * ((M + 3) / 4) * 16u);
    if (dyn && rank == 0)  // boxes below S * csize * NBOX belong to the first stages
      *reinterpret_cast<volatile uint32_t*>(gbase + (dyn_area - base)) =
          static_cast<uint32_t>(S) * csize * NBOX;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot_g;
  // matched by the wait before the pushes (aliased: arrive once the MMAs are done)
  if (csize > 1 && !alias) cluster_arrive_release();
  bool start_waited = false;  // the producer waits for it before its first counter use
  int n_armed = 0;            // producer: pipeline iterations armed (the drain below)

  if (warp == 0) {
    // Producer state (lane 0's copy is the one used).
    int pro = 0, trig = 0;
    bool triggered = false;
    uint64_t policy = 0;
    if (lane == 0) {
      prefetch_tensormap(&wmap);
      prefetch_tensormap(&xmap);
      // Weight tiles are streamed once (evict first), unless other token tiles'
      // CTAs read the same tiles again (then keep them at normal priority).
      policy = gridDim.y > 1 ? l2_policy_evict_normal() : l2_policy_evict_first();
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
      pdl_wait();  // x is produced by the previous kernel on the stream
      for (int it = 0; it < pro; ++it) {
        const int b0 = fixed_box(it);
        const int nbi = fixed_count(it, b0);
        const uint32_t st = base + static_cast<uint32_t>(it) * kStage + NBOX * kWBox;
        for (int b = 0; b < nbi; ++b)
          if (skg_check(st + (b + 1) * kXBox <= stages_end, p.status, kCheckTmaX))
            tma_load_2d(st + b * kXBox, &xmap, (b0 + b) * kBoxK, m0, full_bar(it));
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
        if (nbi <= 0) {  // (dyn) the cluster's boxes are all handed out: tell the MMA issuer
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
            tma_load_2d(st + NBOX * kWBox + b * kXBox, &xmap, (b0 + b) * kBoxK, m0, full_bar(s));
        if (dyn) next_b0 = static_cast<int>(atom_add_cluster_u32(counter, NBOX));
      }
      n_armed = it;
      if (!triggered) pdl_launch_dependents();
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      pdl_wait();
      // (dyn: at most every box of the K range, plus the end marker)
      const int max_it = dyn ? (p.kboxes + NBOX - 1) / NBOX + 1 : iters;
      bool first = true;
      for (int it = 0; it < max_it; ++it) {
        const int s = it % S;
        const uint32_t ph = static_cast<uint32_t>(it / S) & 1u;
        if (!mbar_wait_bounded(full_bar(s), ph, p.timeout_ns)) {
          report_status(p.status, kStatusTimeoutFull);
          if (dyn) break;  // the stage's box count cannot be trusted
        }
        tc_fence_after_sync();
        const int nbi = dyn ? static_cast<int>(stage_boxes[s]) : min(NBOX, nb - it * NBOX);
        if (nbi <= 0) break;
        const uint32_t wst = base + static_cast<uint32_t>(s) * kStage;
        const uint32_t xst = wst + NBOX * kWBox;
        for (int b = 0; b < nbi; ++b) {
          if (!skg_check(wst + (b + 1) * kWBox <= stages_end && xst + (b + 1) * kXBox <= stages_end,
                         p.status, kCheckMmaOperand))
            continue;
#pragma unroll
          for (int j = 0; j < kBoxK / 16; ++j) {
            const uint64_t ad = sw128_kmajor_desc(wst + b * kWBox + j * 32);
            const uint64_t bd = sw128_kmajor_desc(xst + b * kXBox + j * 32);
            tc_mma_f16kind(tmem, ad, bd, kIdesc, first ? 0u : 1u);
            first = false;
          }
        }
        tc_commit(empty_bar(s));
      }
      // A CTA that got no K box (possible with run-time sharing) issued no MMA:
      // arrive directly rather than through a commit with nothing to track.
      if (first)
        mbar_arrive(done_bar);
      else
        tc_commit(done_bar);
    }
    __syncwarp();
  }

  // ------------------------------------------------------------ epilogue
  pdl_wait();
  if (!mbar_wait_bounded(done_bar, 0, p.timeout_ns)) report_status(p.status, kStatusTimeoutDone);
  tc_fence_after_sync();
  if (alias) cluster_arrive_release();  // this CTA's stages may now receive peers' partials
  // The accumulator is read 32 TMEM columns (tokens) at a time, so registers
  // stay bounded for token tiles up to 256.
  constexpr int CH = TOK < 32 ? TOK : 32;
  // Accumulator row r lives in TMEM lane r (M = 128) or, for M = 64, in lane
  // 16 * (r / 16) + r (the first 16 lanes of each warp's quarter); warp w
  // reads its own quarter, lanes 32w .. 32w + 31.
  const uint32_t row_taddr = tmem + ((warp * 32u) << 16);
  const bool row_ok = ROWS == 128 || lane < 16u;
  const int r = ROWS == 128 ? static_cast<int>(warp * 32u + lane) : static_cast<int>(warp * 16u + (lane & 15u));
  auto load_chunk = [&](int c0, float (&v)[CH]) {
#pragma unroll
    for (int c = 0; c < CH / 16; ++c) {
      float t16[16];
      // (c0 and c are the same in every lane: the collective load stays warp-wide)
      if (skg_check(c0 + c * 16 + 16 <= static_cast<int>(kTmemCols), p.status, kCheckTmem)) {
        tmem_ld_32x32b_x16(row_taddr + static_cast<uint32_t>(c0 + c * 16), t16);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) t16[i] = 0.0f;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) v[c * 16 + i] = has_work ? t16[i] : 0.0f;
    }
  };

  if (csize == 1) {
    const int n = n0 + r;
    for (int c0 = 0; c0 < TOK && c0 < M; c0 += CH) {
      float v[CH];
      load_chunk(c0, v);
      if (row_ok && n < p.N) {
#pragma unroll
        for (int i = 0; i < CH; ++i)
          if (c0 + i < M) store_out<OutT>(p, m0 + c0 + i, n, v[i]);
      }
    }
  } else if (bulk) {
    if (!start_waited) cluster_wait_acquire();  // every peer's receive barrier is initialised
    // Token-major blocks [owner][TOK][RS]: each row's partial sums go to the
    // block of the CTA that owns the row, staged in this CTA's idle pipeline
    // buffers (every TMA load has landed and every MMA has read its operands
    // once done_bar fired); the own block is written straight into `red`,
    // which receives the peers' blocks in the same layout at [rank].
    const uint32_t blk = static_cast<uint32_t>(TOK * RS) * 4u;
    const uint32_t owner = static_cast<uint32_t>(r / RS);
    const uint32_t dst = (owner == rank ? red : base) + owner * blk + static_cast<uint32_t>(r % RS) * 4u;
    for (int c0 = 0; c0 < TOK && c0 < M; c0 += CH) {
      float v[CH];
      load_chunk(c0, v);
#pragma unroll
      for (int i = 0; i < CH; ++i)
        if (row_ok && c0 + i < M &&
            skg_check(dst >= base && dst + static_cast<uint32_t>((c0 + i) * RS + 1) * 4u <= smem_end,
                      p.status, kCheckRedLocal))
          asm volatile("st.shared.f32 [%0], %1;" ::"r"(dst + static_cast<uint32_t>((c0 + i) * RS) * 4u),
                       "f"(v[i])
                       : "memory");
    }
    fence_proxy_async_shared();
    __syncthreads();
    if (threadIdx.x == 0) {
      const uint32_t bytes = static_cast<uint32_t>(M * RS) * 4u;
      for (uint32_t j = 1; j < csize; ++j) {
        const uint32_t o = (rank + j) % csize;
        if (skg_check(bytes <= blk && red + (rank + 1) * blk <= smem_end && base + (o + 1) * blk <= smem_end,
                      p.status, kCheckBulk))
          bulk_copy_to_peer(mapa_shared(red + rank * blk, o), base + o * blk, bytes,
                            mapa_shared(recv_bar, o));
      }
    }
    if (!mbar_wait_bounded<true>(recv_bar, 0, p.timeout_ns))
      report_status(p.status, kStatusTimeoutRecv);
    // Once every CTA of the cluster has received its blocks, no copy still reads
    // this CTA's staging buffers: arrive now, wait before exiting.
    cluster_arrive_release();
    // Reduce in rank order (deterministic) 8 rows x 1 token per step and store
    // the 8 outputs, contiguous in out[t], with 16-byte stores where aligned.
    const int RB = RS / 8;
    const int nbase = n0 + static_cast<int>(rank) * RS;
    const bool vec = rows_vectorizable<OutT>(p);
    for (int idx = threadIdx.x; idx < M * RB; idx += blockDim.x) {
      const int t = idx / RB;
      const int rb = idx % RB;
      float acc[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
      for (uint32_t k = 0; k < csize; ++k) {
        const uint32_t a = red + k * blk + static_cast<uint32_t>(t * RS + rb * 8) * 4u;
        if (!skg_check(a + 32u <= smem_end, p.status, kCheckRedRead)) continue;
        float4 q0, q1;
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(q0.x), "=f"(q0.y), "=f"(q0.z), "=f"(q0.w)
                     : "r"(a)
                     : "memory");
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(q1.x), "=f"(q1.y), "=f"(q1.z), "=f"(q1.w)
                     : "r"(a + 16u)
                     : "memory");
        acc[0] += q0.x; acc[1] += q0.y; acc[2] += q0.z; acc[3] += q0.w;
        acc[4] += q1.x; acc[5] += q1.y; acc[6] += q1.z; acc[7] += q1.w;
      }
      const int n = nbase + rb * 8;
      if (vec && n + 8 <= p.N) {
        store_out8<OutT>(p, m0 + t, n, acc);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (n + j < p.N) store_out<OutT>(p, m0 + t, n + j, acc[j]);
      }
    }
    cluster_wait_acquire();
  } else {
    if (!start_waited) cluster_wait_acquire();  // every peer's receive barrier is initialised
    // Receive buffer [rank][RS][TP]: each row's tokens contiguous (16-byte pushes),
    // rows padded by 4 floats so the reduce's 16-byte reads do not collide.
    constexpr int TP = TOK + 4;
    const int MG = (M + 3) / 4;  // groups of 4 tokens carried
    const uint32_t owner = static_cast<uint32_t>(r / RS);
    const int rs = r % RS;
    const uint32_t row_off = ((rank * RS + rs) * TP) * 4u;
    const uint32_t raddr = owner == rank ? 0u : mapa_shared(red + row_off, owner);
    const uint32_t rbar = owner == rank ? 0u : mapa_shared(recv_bar, owner);
    for (int c0 = 0; c0 < TOK && c0 < M; c0 += CH) {
      float v[CH];
      load_chunk(c0, v);
#pragma unroll
      for (int g = 0; g < CH / 4; ++g) {
        const int gg = c0 / 4 + g;
        if (gg >= MG || !row_ok) continue;
        if (!skg_check(owner < csize && red + row_off + (gg + 1) * 16u <= smem_end, p.status,
                       owner == rank ? kCheckRedLocal : kCheckRedRemote))
          continue;
        if (owner == rank)
          asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(red + row_off + gg * 16u),
                       "f"(v[4 * g]), "f"(v[4 * g + 1]), "f"(v[4 * g + 2]), "f"(v[4 * g + 3])
                       : "memory");
        else
          st_async_v4(raddr + static_cast<uint32_t>(gg * 16), v[4 * g], v[4 * g + 1], v[4 * g + 2],
                      v[4 * g + 3], rbar);
      }
    }
    __syncthreads();
    if (!mbar_wait_bounded<true>(recv_bar, 0, p.timeout_ns)) {
      report_status(p.status, kStatusTimeoutRecv);
      // A live peer pushes after at most one bounded wait per pipeline stage of
      // its K range (at most iters + 1 stages) and one for its MMAs: keep
      // waiting that many more rounds, so this CTA does not exit while a peer
      // may still push into it.
      const int rounds = (dyn ? (p.kboxes + NBOX - 1) / NBOX : iters) + 3;
      for (int r = 0; r < rounds; ++r)
        if (mbar_wait_bounded<true>(recv_bar, 0, p.timeout_ns)) break;
    }
    // Reduce in rank order (deterministic) 8 rows x 1 token per step (lanes
    // walk the token index: conflict-free reads) and store the 8 outputs,
    // contiguous in out[t], with 16-byte stores where aligned.
    const int RB = RS / 8;
    const int nbase = n0 + static_cast<int>(rank) * RS;
    const bool vec = rows_vectorizable<OutT>(p);
    const float* redf = reinterpret_cast<const float*>(gbase + (red - base));
    for (int idx = threadIdx.x; idx < M * RB; idx += blockDim.x) {
      const int t = idx % M;
      const int rb = idx / M;
      float acc[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
      if (!skg_check(red + static_cast<uint32_t>(((static_cast<int>(csize) - 1) * RS + rb * 8 + 7) * TP + t + 1) * 4u <=
                         smem_end,
                     p.status, kCheckRedRead))
        continue;
      for (uint32_t k = 0; k < csize; ++k)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] += redf[(k * RS + rb * 8 + j) * TP + t];
      const int n = nbase + rb * 8;
      if (vec && n + 8 <= p.N) {
        store_out8<OutT>(p, m0 + t, n, acc);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (n + j < p.N) store_out<OutT>(p, m0 + t, n + j, acc[j]);
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  if (threadIdx.x == 0) {
    // Drain (the producer thread): every armed stage's last phase must have
    // landed before exit (immediate on the normal path, where the MMA issuer
    // waited for them).
    const int used = n_armed < S ? n_armed : S;
    for (int s = 0; s < used; ++s) {
      const int last = s + ((n_armed - 1 - s) / S) * S;
      if (!mbar_wait_bounded(full_bar(s), static_cast<uint32_t>(last / S) & 1u, p.timeout_ns))
        report_status(p.status, kStatusTimeoutDrain);
    }
  }
}

#define SKG_TC_ENTRY_R(ROWS, TOK, NBOX, OUTT, OUTCODE, FP16)                               \
  KernelEntry {                                                                             \
    kVariantTc, ROWS, TOK, NBOX, FP16 ? 1 : 0, OUTCODE, 128,                                \
        reinterpret_cast<const void*>(&skinny_tc_kernel<TOK, NBOX, OUTT, FP16, ROWS>)       \
  }
#define SKG_TC_ENTRY(TOK, NBOX, OUTT, OUTCODE, FP16) SKG_TC_ENTRY_R(128, TOK, NBOX, OUTT, OUTCODE, FP16)

// 64-row tiles (MMA M = 64): twice the CTAs of a 128-row tiling for the same
// cluster size, half the partial sums per CTA in the cluster reduction.
#define SKG_TC_ROW64(OUTT, OUTCODE)                                                         \
  SKG_TC_ENTRY_R(64, 16, 1, OUTT, OUTCODE, false), SKG_TC_ENTRY_R(64, 16, 2, OUTT, OUTCODE, false), \
      SKG_TC_ENTRY_R(64, 16, 4, OUTT, OUTCODE, false),                                      \
      SKG_TC_ENTRY_R(64, 32, 1, OUTT, OUTCODE, false), SKG_TC_ENTRY_R(64, 32, 2, OUTT, OUTCODE, false), \
      SKG_TC_ENTRY_R(64, 32, 4, OUTT, OUTCODE, false),                                      \
      SKG_TC_ENTRY_R(64, 48, 1, OUTT, OUTCODE, false), SKG_TC_ENTRY_R(64, 48, 2, OUTT, OUTCODE, false), \
      SKG_TC_ENTRY_R(64, 64, 1, OUTT, OUTCODE, false), SKG_TC_ENTRY_R(64, 64, 2, OUTT, OUTCODE, false)

#define SKG_TC_ROW(OUTT, OUTCODE)                                                           \
  SKG_TC_ENTRY(16, 1, OUTT, OUTCODE, false), SKG_TC_ENTRY(16, 2, OUTT, OUTCODE, false),     \
      SKG_TC_ENTRY(16, 4, OUTT, OUTCODE, false), SKG_TC_ENTRY(32, 1, OUTT, OUTCODE, false), \
      SKG_TC_ENTRY(32, 2, OUTT, OUTCODE, false), SKG_TC_ENTRY(32, 4, OUTT, OUTCODE, false), \
      SKG_TC_ENTRY(48, 1, OUTT, OUTCODE, false), SKG_TC_ENTRY(48, 2, OUTT, OUTCODE, false), \
      SKG_TC_ENTRY(64, 1, OUTT, OUTCODE, false), SKG_TC_ENTRY(64, 2, OUTT, OUTCODE, false), \
      SKG_TC_ENTRY(64, 4, OUTT, OUTCODE, false), SKG_TC_ENTRY(128, 1, OUTT, OUTCODE, false), \
      SKG_TC_ENTRY(128, 2, OUTT, OUTCODE, false), SKG_TC_ENTRY(256, 1, OUTT, OUTCODE, false)

// fp16 operands: one or two boxes per stage.
#define SKG_TC_ROW16(OUTT, OUTCODE)                                                         \
  SKG_TC_ENTRY(16, 1, OUTT, OUTCODE, true), SKG_TC_ENTRY(16, 2, OUTT, OUTCODE, true),       \
      SKG_TC_ENTRY(32, 1, OUTT, OUTCODE, true), SKG_TC_ENTRY(32, 2, OUTT, OUTCODE, true),   \
      SKG_TC_ENTRY(48, 1, OUTT, OUTCODE, true), SKG_TC_ENTRY(48, 2, OUTT, OUTCODE, true),   \
      SKG_TC_ENTRY(64, 1, OUTT, OUTCODE, true), SKG_TC_ENTRY(64, 2, OUTT, OUTCODE, true),   \
      SKG_TC_ENTRY(128, 1, OUTT, OUTCODE, true), SKG_TC_ENTRY(256, 1, OUTT, OUTCODE, true)

static const KernelEntry kTcTable[] = {SKG_TC_ROW(__nv_bfloat16, 0), SKG_TC_ROW(float, 2),
                                       SKG_TC_ROW64(__nv_bfloat16, 0), SKG_TC_ROW64(float, 2),
                                       SKG_TC_ROW16(__half, 1), SKG_TC_ROW16(float, 2)};

const KernelEntry* tc_kernel_table(int* count) {
  *count = static_cast<int>(sizeof(kTcTable) / sizeof(kTcTable[0]));
  return kTcTable;
}

}  // namespace skg
