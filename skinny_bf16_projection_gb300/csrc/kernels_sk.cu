// Stream-K skinny projection on tcgen05/TMEM, without thread-block clusters.
//
//   out[M, N] = x[M, K] @ W[N, K]^T,  M <= 64, swap-AB as in the cluster
//   kernel: 128 weight rows are the MMA's M, the token tile its N.
//
// Work: the weight is cut into units of 128 rows x 64 K (one TMA box); units
// are ordered tile-major (all K boxes of row tile 0, then tile 1, ...) and
// CTA c of G takes units [c*U/G, (c+1)*U/G), so every CTA streams the same
// number of weight bytes (within one box) and the grid is one wave (G = the
// SM count or twice it).  A CTA's range cuts the tiles into segments; a tile
// held whole by one CTA is written directly, a tile cut between CTAs is
// finished by the last CTA to arrive on the tile's counter: every CTA writes
// its fp32 partial sum to the workspace; after a CTA barrier one thread
// releases those writes and increments the counter (acq_rel, GPU scope);
// the one that sees all other parts summed them in CTA order (fixed order, so
// the bits do not depend on arrival order) and resets the counter.  No CTA
// ever waits for another one.
//
// This replaces the pages' cluster/DSMEM split-K reduction (page
// "vllm.models.glm5next.nvidia.specialized_decode.gemm", module docstring)
// where cluster residency limits how many CTAs run at once; the weight
// stream itself (TMA boxes {64, 128} with 128-byte swizzle and an
// evict_first policy, issued before the PDL wait) is the same as in the
// cluster kernels.
//
//   warp 0 lane 0  TMA producer over this CTA's stages
//   warp 1         TMEM allocation; lane 0 issues the MMAs into one of two
//                  accumulators (segment j uses accumulator j % 2)
//   warps 2-5      epilogue: tcgen05.ld of the finished accumulator (warp w
//                  reads TMEM lanes 32*(w%4)..+31), release it, then store or
//                  run the split-tile protocol above
#include "device_common.cuh"

namespace skg {

namespace {

// This CTA's segments: maximal runs of its units inside one row tile.
struct SegmentIter {
  int u, u1, kb;
  __device__ bool next(int& tile, int& ka, int& kend) {
    if (u >= u1) return false;
    tile = u / kb;
    const int end = min(u1, (tile + 1) * kb);
    ka = u - tile * kb;
    kend = end - tile * kb;
    u = end;
    return true;
  }
};

// Pipeline stages: up to NBOX consecutive boxes of one segment per stage.
template <int NBOX>
struct StageIter {
  SegmentIter seg;
  int tile = 0, k = 0, kend = 0;
  __device__ bool next(int& t, int& kbox, int& nbox) {
    if (k >= kend) {
      if (!seg.next(tile, k, kend)) return false;
    }
    t = tile;
    kbox = k;
    nbox = min(NBOX, kend - k);
    k += nbox;
    return true;
  }
};

// a / b for non-negative a, positive b: a 32-bit division when both fit (a
// 64-bit one is a long dependent instruction sequence, and these sit on the
// epilogue's critical path).
__device__ __forceinline__ int64_t udiv_fast(int64_t a, int64_t b) {
  if (((static_cast<uint64_t>(a) | static_cast<uint64_t>(b)) >> 32) == 0)
    return static_cast<int64_t>(static_cast<uint32_t>(a) / static_cast<uint32_t>(b));
  return a / b;
}

// First unit of CTA c when U units are split over G CTAs as floor(c*U/G).
__device__ __forceinline__ int first_unit(int64_t c, int64_t U, int64_t G) {
  return static_cast<int>(udiv_fast(c * U, G));
}

// CTA owning unit u under that split.
__device__ __forceinline__ int cta_of_unit(int64_t u, int64_t U, int64_t G) {
  return static_cast<int>(udiv_fast((u + 1) * G + U - 1, U) - 1);
}

}  // namespace

template <int TOK, int NBOX, typename OutT, bool kFp16>
__global__ void __launch_bounds__(192) skinny_sk_kernel(const __grid_constant__ CUtensorMap wmap,
                                                      const __grid_constant__ CUtensorMap xmap,
                                                      const KParams p) {
  constexpr int ROWS = 128;
  constexpr uint32_t kWBox = ROWS * kBoxRowBytes;
  constexpr uint32_t kXBox = TOK * kBoxRowBytes;
  constexpr uint32_t kStage = stage_bytes(ROWS, TOK, NBOX);
  constexpr uint32_t kTmemCols = 2 * TOK <= 32 ? 32u : (2 * TOK <= 64 ? 64u : 128u);
  constexpr uint32_t kIdesc = mma_idesc<kFp16>(ROWS, TOK);
  static_assert(TOK % 16 == 0 && TOK >= 16 && TOK <= 64, "M=128 MMA needs N % 16 == 0");

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + kSmemAlign - 1) & ~static_cast<uint32_t>(kSmemAlign - 1);
  uint8_t* const gbase = smem_raw + (base - raw);
  const int S = p.stages;
  const uint32_t bars = base + static_cast<uint32_t>(S) * kStage;
  const uint32_t stages_end = bars;  // (checked build only)
  const uint32_t tfull_bar = bars + 8u * (2 * S);     // [2]
  const uint32_t tempty_bar = tfull_bar + 16u;        // [2]
  const uint32_t dbg_bar = tempty_bar + 16u;
  const uint32_t flag_slot = dbg_bar + 8u;            // u32: "this CTA finishes the tile"
  const uint32_t tmem_slot = flag_slot + 4u;
  volatile uint32_t* const tmem_slot_g =
      reinterpret_cast<volatile uint32_t*>(gbase + (tmem_slot - base));
  volatile uint32_t* const flag_g = reinterpret_cast<volatile uint32_t*>(gbase + (flag_slot - base));
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

  const int kb = p.kboxes;
  const int ntiles = (p.N + ROWS - 1) / ROWS;
  const int64_t U = static_cast<int64_t>(ntiles) * kb;
  const int64_t G = gridDim.x;
  const int c = blockIdx.x;
  const int u0 = first_unit(c, U, G);
  const int u1 = first_unit(c + 1, U, G);
  const int first_tile = u0 / kb;
  const int M = p.M;

  // Number of stages this CTA runs (for the drain at exit).
  int total_stages = 0;
  {
    StageIter<NBOX> si{SegmentIter{u0, u1, kb}};
    int t, k, n;
    while (si.next(t, k, n)) ++total_stages;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar + 8u * a, 1);
      mbar_init(tempty_bar + 8u * a, 4);
    }
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

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tensormap(&wmap);
      prefetch_tensormap(&xmap);
      const uint64_t policy = l2_policy_evict_first();
      const int pro = total_stages < S ? total_stages : S;
      StageIter<NBOX> si{SegmentIter{u0, u1, kb}};
      int t, k, n;
      for (int it = 0; it < pro && si.next(t, k, n); ++it) {
        const uint32_t st = base + static_cast<uint32_t>(it) * kStage;
        mbar_arrive_expect_tx(full_bar(it), n * (kWBox + kXBox));
        for (int b = 0; b < n; ++b)
          if (skg_check(st + (b + 1) * kWBox <= stages_end && ((k + b) * kBoxK) % 8 == 0, p.status,
                        kCheckTmaW))
            tma_load_2d_hint(st + b * kWBox, &wmap, (k + b) * kBoxK, t * ROWS, full_bar(it), policy);
      }
      // Let the next kernel on the stream launch now: its CTAs can prefetch their
      // own weight tiles while this grid streams (they still wait for our
      // completion in griddepcontrol.wait before touching x or out).
      pdl_launch_dependents();
      pdl_wait();  // x is produced by the previous kernel on the stream
      StageIter<NBOX> sx{SegmentIter{u0, u1, kb}};
      for (int it = 0; it < pro && sx.next(t, k, n); ++it) {
        const uint32_t st = base + static_cast<uint32_t>(it) * kStage + NBOX * kWBox;
        for (int b = 0; b < n; ++b)
          if (skg_check(st + (b + 1) * kXBox <= stages_end, p.status, kCheckTmaX))
            tma_load_2d(st + b * kXBox, &xmap, (k + b) * kBoxK, 0, full_bar(it));
      }
      for (int it = pro; si.next(t, k, n); ++it) {
        const int s = it % S;
        const uint32_t ph = static_cast<uint32_t>((it / S) - 1) & 1u;
        if (!mbar_wait_bounded(empty_bar(s), ph, p.timeout_ns))
          report_status(p.status, kStatusTimeoutEmpty);
        const uint32_t st = base + static_cast<uint32_t>(s) * kStage;
        mbar_arrive_expect_tx(full_bar(s), n * (kWBox + kXBox));
        for (int b = 0; b < n; ++b)
          if (skg_check(st + (b + 1) * kWBox <= stages_end && ((k + b) * kBoxK) % 8 == 0, p.status,
                        kCheckTmaW))
            tma_load_2d_hint(st + b * kWBox, &wmap, (k + b) * kBoxK, t * ROWS, full_bar(s), policy);
        for (int b = 0; b < n; ++b)
          if (skg_check(st + NBOX * kWBox + (b + 1) * kXBox <= stages_end, p.status, kCheckTmaX))
            tma_load_2d(st + NBOX * kWBox + b * kXBox, &xmap, (k + b) * kBoxK, 0, full_bar(s));
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      pdl_wait();
      SegmentIter sg{u0, u1, kb};
      int t, ka, kend;
      int it = 0;
      for (int j = 0; sg.next(t, ka, kend); ++j) {
        const int acc = j & 1;
        if (j >= 2 && !mbar_wait_bounded(tempty_bar + 8u * acc,
                                         static_cast<uint32_t>((j >> 1) - 1) & 1u, p.timeout_ns))
          report_status(p.status, kStatusTimeoutDone);
        tc_fence_after_sync();
        const uint32_t dcol = tmem + static_cast<uint32_t>(acc * TOK);
        for (int k = ka; k < kend; k += NBOX, ++it) {
          const int n = min(NBOX, kend - k);
          const int s = it % S;
          if (!mbar_wait_bounded(full_bar(s), static_cast<uint32_t>(it / S) & 1u, p.timeout_ns))
            report_status(p.status, kStatusTimeoutFull);
          tc_fence_after_sync();
          const uint32_t wst = base + static_cast<uint32_t>(s) * kStage;
          const uint32_t xst = wst + NBOX * kWBox;
          for (int b = 0; b < n; ++b) {
#pragma unroll
            for (int q = 0; q < kBoxK / 16; ++q) {
              const uint64_t ad = sw128_kmajor_desc(wst + b * kWBox + q * 32);
              const uint64_t bd = sw128_kmajor_desc(xst + b * kXBox + q * 32);
              tc_mma_f16kind(dcol, ad, bd, kIdesc, (k > ka || b > 0 || q > 0) ? 1u : 0u);
            }
          }
          tc_commit(empty_bar(s));
        }
        tc_commit(tfull_bar + 8u * acc);
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue warps 2..5
    pdl_wait();
    const uint32_t quarter = warp & 3u;
    const int row = static_cast<int>(quarter * 32u + lane);
    const uint32_t ep_tid = threadIdx.x - 64u;  // 0..127
    SegmentIter sg{u0, u1, kb};
    int t, ka, kend;
    for (int j = 0; sg.next(t, ka, kend); ++j) {
      const int acc = j & 1;
      if (!mbar_wait_bounded(tfull_bar + 8u * acc, static_cast<uint32_t>(j >> 1) & 1u,
                             p.timeout_ns))
        report_status(p.status, kStatusTimeoutDone);
      tc_fence_after_sync();
      float v[TOK];
      const uint32_t taddr = tmem + ((quarter * 32u) << 16) + static_cast<uint32_t>(acc * TOK);
#pragma unroll
      for (int cc = 0; cc < TOK / 16; ++cc) {
        float t16[16];
        // (acc and cc are the same in every lane: the collective load stays warp-wide)
        if (skg_check(acc * TOK + cc * 16 + 16 <= static_cast<int>(kTmemCols), p.status, kCheckTmem)) {
          tmem_ld_32x32b_x16(taddr + static_cast<uint32_t>(cc * 16), t16);
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) t16[i] = 0.0f;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) v[cc * 16 + i] = t16[i];
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar + 8u * acc);

      const int n = t * ROWS + row;
      if (ka == 0 && kend == kb) {  // whole tile in this CTA
        if (n < p.N) {
#pragma unroll
          for (int tk = 0; tk < TOK; ++tk)
            if (tk < M) store_out<OutT>(p, tk, n, v[tk]);
        }
        continue;
      }
      // Split tile: publish this part, count arrivals, the last one finishes.
      const int slot_self = c * 2 + (t == first_tile ? 0 : 1);
      float* const ws_self = p.workspace + static_cast<int64_t>(slot_self) * TOK * ROWS;
      const bool ws_ok = skg_check(slot_self >= 0 && slot_self < 2 * static_cast<int>(gridDim.x) &&
                                       row < ROWS && t >= 0 && t < ntiles,
                                   p.status, kCheckWorkspace);
#pragma unroll
      for (int tk = 0; tk < TOK; ++tk)
        if (tk < M && ws_ok) __stcg(ws_self + tk * ROWS + row, v[tk]);
      named_barrier_sync(1, 128);  // all parts of this CTA written before the release below
      const int c_first = cta_of_unit(static_cast<int64_t>(t) * kb, U, G);
      const int c_last = cta_of_unit(static_cast<int64_t>(t + 1) * kb - 1, U, G);
      if (ep_tid == 0) {
        const uint32_t prev = arrive_count_acq_rel(p.counters + t);
        *flag_g = (prev + 1u == static_cast<uint32_t>(c_last - c_first + 1)) ? 1u : 0u;
      }
      named_barrier_sync(1, 128);
      if (*flag_g != 0u) {
        // Sum every part in CTA order (the same order whichever CTA arrives
        // last).  The parts are CTAs c_first..c_last; each wrote its slot
        // 2 * cq, except c_first when its range began in the previous tile
        // (then this tile is its second segment: slot 2 * cq + 1).  Work items
        // are (token, 4 consecutive rows); a thread keeps kIB items x kPB
        // parts of loads in flight, then adds them in part order, so each
        // batch costs one L2 round trip.
        constexpr int kPB = 8;
        constexpr int kIB = 2;
        const int parts = c_last - c_first + 1;
        const int first_slot =
            2 * c_first + (first_unit(c_first, U, G) / kb == t ? 0 : 1);
        const int items = M * (ROWS / 4);
        for (int i0 = static_cast<int>(ep_tid); i0 < items; i0 += 128 * kIB) {
          float4 acc[kIB];
          int off[kIB];
#pragma unroll
          for (int ii = 0; ii < kIB; ++ii) {
            acc[ii] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            const int item = i0 + ii * 128;
            off[ii] = (item / (ROWS / 4)) * ROWS + (item % (ROWS / 4)) * 4;
          }
          for (int q0 = 0; q0 < parts; q0 += kPB) {
            float4 pv[kIB][kPB];
#pragma unroll
            for (int q = 0; q < kPB; ++q) {
              const int slot = q0 + q == 0 ? first_slot : 2 * (c_first + q0 + q);
              const bool slot_ok = q0 + q < parts &&
                                   skg_check(slot >= 0 && slot < 2 * static_cast<int>(gridDim.x),
                                             p.status, kCheckWorkspace);
              const float* const part = p.workspace + static_cast<int64_t>(slot_ok ? slot : 0) * TOK * ROWS;
#pragma unroll
              for (int ii = 0; ii < kIB; ++ii) {
                pv[ii][q] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                if (slot_ok && i0 + ii * 128 < items &&
                    skg_check(off[ii] >= 0 && off[ii] + 4 <= TOK * ROWS, p.status, kCheckWorkspace))
                  pv[ii][q] = __ldcg(reinterpret_cast<const float4*>(part + off[ii]));
              }
            }
#pragma unroll
            for (int ii = 0; ii < kIB; ++ii)
#pragma unroll
              for (int q = 0; q < kPB; ++q)
                if (q0 + q < parts) {
                  acc[ii].x += pv[ii][q].x;
                  acc[ii].y += pv[ii][q].y;
                  acc[ii].z += pv[ii][q].z;
                  acc[ii].w += pv[ii][q].w;
                }
          }
#pragma unroll
          for (int ii = 0; ii < kIB; ++ii) {
            const int item = i0 + ii * 128;
            if (item >= items) continue;
            const int tk = item / (ROWS / 4);
            const int nb0 = t * ROWS + (item % (ROWS / 4)) * 4;
            if (nb0 + 0 < p.N) store_out<OutT>(p, tk, nb0 + 0, acc[ii].x);
            if (nb0 + 1 < p.N) store_out<OutT>(p, tk, nb0 + 1, acc[ii].y);
            if (nb0 + 2 < p.N) store_out<OutT>(p, tk, nb0 + 2, acc[ii].z);
            if (nb0 + 3 < p.N) store_out<OutT>(p, tk, nb0 + 3, acc[ii].w);
          }
        }
        if (ep_tid == 0) p.counters[t] = 0u;  // ready for the next launch
      }
      named_barrier_sync(1, 128);  // the flag word is reused by the next segment
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  if (threadIdx.x == 0) {
    const int used = total_stages < S ? total_stages : S;
    for (int s = 0; s < used; ++s) {
      const int last = s + ((total_stages - 1 - s) / S) * S;
      if (!mbar_wait_bounded(full_bar(s), static_cast<uint32_t>(last / S) & 1u, p.timeout_ns))
        report_status(p.status, kStatusTimeoutDrain);
    }
  }
}

#define SKG_SK_ENTRY(TOK, NBOX, OUTT, OUTCODE, FP16)                                    \
  KernelEntry {                                                                         \
    kVariantSk, 128, TOK, NBOX, FP16 ? 1 : 0, OUTCODE, 192,                             \
        reinterpret_cast<const void*>(&skinny_sk_kernel<TOK, NBOX, OUTT, FP16>)         \
  }

#define SKG_SK_ROW(OUTT, OUTCODE)                                                       \
  SKG_SK_ENTRY(16, 1, OUTT, OUTCODE, false), SKG_SK_ENTRY(16, 2, OUTT, OUTCODE, false), \
      SKG_SK_ENTRY(16, 4, OUTT, OUTCODE, false), SKG_SK_ENTRY(32, 1, OUTT, OUTCODE, false), \
      SKG_SK_ENTRY(32, 2, OUTT, OUTCODE, false), SKG_SK_ENTRY(32, 4, OUTT, OUTCODE, false), \
      SKG_SK_ENTRY(64, 1, OUTT, OUTCODE, false), SKG_SK_ENTRY(64, 2, OUTT, OUTCODE, false), \
      SKG_SK_ENTRY(64, 4, OUTT, OUTCODE, false)

#define SKG_SK_ROW16(OUTT, OUTCODE)                                                     \
  SKG_SK_ENTRY(16, 2, OUTT, OUTCODE, true), SKG_SK_ENTRY(32, 2, OUTT, OUTCODE, true),   \
      SKG_SK_ENTRY(64, 2, OUTT, OUTCODE, true)

static const KernelEntry kSkTable[] = {SKG_SK_ROW(__nv_bfloat16, 0), SKG_SK_ROW(float, 2),
                                       SKG_SK_ROW16(__half, 1), SKG_SK_ROW16(float, 2)};

const KernelEntry* sk_kernel_table(int* count) {
  *count = static_cast<int>(sizeof(kSkTable) / sizeof(kSkTable[0]));
  return kSkTable;
}

}  // namespace skg
