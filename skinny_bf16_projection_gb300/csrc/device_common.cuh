// Device-side building blocks shared by the two kernel families: mbarriers
// with bounded waits, TMA tile loads with an L2 evict_first policy, thread
// block cluster / distributed shared memory primitives, tcgen05 (TMEM) and
// legacy mma.sync wrappers.  All inline PTX for sm_103a.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernel_params.h"

namespace skg {

// ---------------------------------------------------------------- basics
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

// First error wins; the host reads and clears the word.
__device__ __forceinline__ void report_status(uint32_t* status, uint32_t code) {
  if (status != nullptr) atomicCAS(status, 0u, code);
}

// Checked build (-DSKG_DEVICE_CHECKS=1): an access guarded by skg_check is
// tested first; a failed test records kStatusCheck | site (first error wins)
// and the caller skips the access.  In the normal build the test compiles away.
#ifndef SKG_DEVICE_CHECKS
#define SKG_DEVICE_CHECKS 0
#endif
__device__ __forceinline__ bool skg_check(bool ok, uint32_t* status, uint32_t site) {
  if constexpr (SKG_DEVICE_CHECKS != 0) {
    if (!ok) report_status(status, kStatusCheck | site);
    return ok;
  } else {
    (void)ok;
    (void)status;
    (void)site;
    return true;
  }
}
// Bytes of dynamic shared memory this launch was given.
__device__ __forceinline__ uint32_t dynamic_smem_bytes() {
  uint32_t r;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(r));
  return r;
}

// Barrier among `nthreads` threads (whole warps) of the CTA, separate from __syncthreads.
__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// L2-coherent load (bypasses L1), issued in program order so a run of them is in flight together.
__device__ __forceinline__ float ld_cg_f32(const float* ptr) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(ptr) : "memory");
  return v;
}

__device__ __forceinline__ float4 ld_cg_f32x4(const float* ptr) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(ptr)
               : "memory");
  return v;
}

// Release this CTA's prior writes (ordered before by a CTA barrier), count one
// arrival on *ctr at GPU scope, acquire the other arrivals' writes.
__device__ __forceinline__ uint32_t arrive_count_acq_rel(uint32_t* ctr) {
  uint32_t prev;
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(prev) : "l"(ctr) : "memory");
  return prev;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the async proxy and to the cluster.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, P;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0u;
}

// Acquire at cluster scope: used where the phase is completed by remote
// st.async writes from other CTAs of the cluster.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 P, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, P;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0u;
}

// Every spin in these kernels is bounded: after timeout_ns the wait gives up,
// the caller records a status code and carries on with the protocol, so the
// kernel always terminates and the context stays usable.
template <bool kClusterScope = false>
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t timeout_ns) {
  auto probe = [&]() {
    return kClusterScope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
  };
  if (probe()) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (probe()) return true;
    if (globaltimer_ns() - t0 > timeout_ns) return false;
  }
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// A runtime-created policy: every weight line is marked first to evict, so
// the one-pass weight stream does not push the reused activations out of L2.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, int32_t c0,
                                                 int32_t c1, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t c0,
                                            int32_t c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// Bring one box of a tiled tensor into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int32_t c0, int32_t c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1)
               : "memory");
}

// ---------------------------------------------------------------- PDL
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}
// Shared-memory writes by this thread become visible to the async proxy (bulk copies).
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Bulk copy of `bytes` (multiple of 16) from this CTA's shared memory into a
// peer CTA's shared memory, counted on the peer's mbarrier (both addresses
// already mapped into the cluster window with mapa).
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst_cluster, uint32_t src_cta,
                                                  uint32_t bytes, uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst_cluster),
      "r"(src_cta), "r"(bytes), "r"(bar_cluster)
      : "memory");
}
// Atomic add on a 32-bit word in the shared memory of a CTA of this cluster
// (address mapped with mapa); returns the previous value.  Relaxed: only the
// uniqueness of the returned values matters.
__device__ __forceinline__ uint32_t atom_add_cluster_u32(uint32_t addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.relaxed.cluster.shared::cluster.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "r"(addr), "r"(v)
               : "memory");
  return old;
}

// Address of the same shared-memory variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Remote 4-byte store whose arrival is counted on the remote CTA's mbarrier.
__device__ __forceinline__ void st_async_b32(uint32_t remote_addr, float v, uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(
                   remote_addr),
               "r"(__float_as_uint(v)), "r"(remote_bar)
               : "memory");
}

// Remote 16-byte store (four fp32) counted on the remote CTA's mbarrier.
__device__ __forceinline__ void st_async_v4(uint32_t remote_addr, float a, float b, float c,
                                            float d, uint32_t remote_bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::
          "r"(remote_addr),
      "r"(__float_as_uint(a)), "r"(__float_as_uint(b)), "r"(__float_as_uint(c)),
      "r"(__float_as_uint(d)), "r"(remote_bar)
      : "memory");
}

// ---------------------------------------------------------------- output
template <typename T>
__device__ __forceinline__ T to_out(float v);
template <>
__device__ __forceinline__ float to_out<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ __nv_bfloat16 to_out<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}
template <>
__device__ __forceinline__ __half to_out<__half>(float v) {
  return __float2half_rn(v);
}
__device__ __forceinline__ float from_out(float v) { return v; }
__device__ __forceinline__ float from_out(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float from_out(__half v) { return __half2float(v); }

// out[t][n] = round(v + residual[t][n]) (residual optional, in the output type):
// the residual joins the fp32 sum before the single rounding to the output type.
template <typename OutT>
__device__ __forceinline__ void store_out(const KParams& p, int t, int n, float v) {
  if (!skg_check(t >= 0 && t < p.M && n >= 0 && n < p.N, p.status, kCheckOut)) return;
  if (p.residual != nullptr)
    v += from_out(static_cast<const OutT*>(p.residual)[static_cast<int64_t>(t) * p.ldr + n]);
  static_cast<OutT*>(p.out)[static_cast<int64_t>(t) * p.ldo + n] = to_out<OutT>(v);
}

// Two 2-byte output values packed into / unpacked from one 32-bit word (low half first).
template <typename OutT>
__device__ __forceinline__ uint32_t pack2(float a, float b);
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}
template <typename OutT>
__device__ __forceinline__ float2 unpack2(uint32_t u);
template <>
__device__ __forceinline__ float2 unpack2<__nv_bfloat16>(uint32_t u) {
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}
template <>
__device__ __forceinline__ float2 unpack2<__half>(uint32_t u) {
  __half2 h;
  *reinterpret_cast<uint32_t*>(&h) = u;
  return __half22float2(h);
}

// Eight consecutive outputs out[t][n..n+7] with one (bf16/fp16) or two (fp32)
// 16-byte stores; same arithmetic as store_out per element.  The caller checks
// that out (and residual) rows are 16-byte aligned at n and n + 8 <= N.
template <typename OutT>
__device__ __forceinline__ void store_out8(const KParams& p, int t, int n, const float (&v)[8]) {
  if (!skg_check(t >= 0 && t < p.M && n >= 0 && n + 8 <= p.N, p.status, kCheckOut)) return;
  float w[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) w[j] = v[j];
  if (p.residual != nullptr) {
    const OutT* rp = static_cast<const OutT*>(p.residual) + static_cast<int64_t>(t) * p.ldr + n;
    if constexpr (sizeof(OutT) == 2) {
      const uint4 q = *reinterpret_cast<const uint4*>(rp);
      const float2 a = unpack2<OutT>(q.x), b = unpack2<OutT>(q.y), c = unpack2<OutT>(q.z),
                   d = unpack2<OutT>(q.w);
      w[0] += a.x; w[1] += a.y; w[2] += b.x; w[3] += b.y;
      w[4] += c.x; w[5] += c.y; w[6] += d.x; w[7] += d.y;
    } else {
      const float4 a = *reinterpret_cast<const float4*>(rp);
      const float4 b = *reinterpret_cast<const float4*>(rp + 4);
      w[0] += a.x; w[1] += a.y; w[2] += a.z; w[3] += a.w;
      w[4] += b.x; w[5] += b.y; w[6] += b.z; w[7] += b.w;
    }
  }
  OutT* op = static_cast<OutT*>(p.out) + static_cast<int64_t>(t) * p.ldo + n;
  if constexpr (sizeof(OutT) == 2) {
    *reinterpret_cast<uint4*>(op) = make_uint4(pack2<OutT>(w[0], w[1]), pack2<OutT>(w[2], w[3]),
                                               pack2<OutT>(w[4], w[5]), pack2<OutT>(w[6], w[7]));
  } else {
    *reinterpret_cast<float4*>(op) = make_float4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<float4*>(op + 4) = make_float4(w[4], w[5], w[6], w[7]);
  }
}

// True when every row of out (and of residual, if any) starts 16-byte aligned
// for 8-element column blocks, so store_out8 may be used at n % 8 == 0.
template <typename OutT>
__device__ __forceinline__ bool rows_vectorizable(const KParams& p) {
  constexpr int64_t e = static_cast<int64_t>(sizeof(OutT));
  bool ok = (reinterpret_cast<uintptr_t>(p.out) % 16 == 0) && ((p.ldo * e) % 16 == 0);
  if (p.residual != nullptr)
    ok = ok && (reinterpret_cast<uintptr_t>(p.residual) % 16 == 0) && ((p.ldr * e) % 16 == 0);
  return ok;
}

// ---------------------------------------------------------------- mma.sync (legacy path)
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr)
               : "memory");
}
template <bool kFp16>
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  if constexpr (kFp16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

// ---------------------------------------------------------------- tcgen05 / TMEM
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile written by TMA
// with the 128-byte swizzle: rows of 128 B, 8-row (1024 B) swizzle atoms
// stacked along M/N (stride byte offset 1024), leading byte offset unused for
// swizzled K-major tiles, descriptor version 1, swizzle mode 2 (128 B).
// Stepping K by 16 elements inside the 128-byte row is a +32 B start offset.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

// Instruction descriptor, kind::f16: D fp32, A/B bf16 (or fp16), both K-major,
// N >> 3 at bit 17, M >> 4 at bit 24.
template <bool kFp16>
__host__ __device__ constexpr uint32_t mma_idesc(int m, int n) {
  return (1u << 4) | ((kFp16 ? 0u : 1u) << 7) | ((kFp16 ? 0u : 1u) << 10) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void tc_mma_f16kind(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 op issued so far by this thread is done.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 32 lanes x 16 columns of 32-bit TMEM cells -> 16 registers per thread, then
// wait for the load; the wait names the registers so no use moves above it.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace skg
