// Host side of the C ABI declared in include/skinny_gemm.h: validation,
// TMA map encoding, the per-M tactic plan, launches (clusters + programmatic
// dependent launch), the on-device autotuner, the two-stream overlap step and
// the device watchdog word.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <unordered_set>
#include <vector>

#include "kernel_params.h"
#include "skinny_gemm.h"

// 1 in the checked build (libskinny_gemm_checked.so), whose kernels test their accesses.
#ifndef SKG_DEVICE_CHECKS
#define SKG_DEVICE_CHECKS 0
#endif

using namespace skg;

// ------------------------------------------------------------------ errors
namespace {

thread_local std::string g_err;
thread_local int g_last_status = 0;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  g_last_status = code;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  if (e == cudaErrorStreamCaptureUnsupported || e == cudaErrorStreamCaptureImplicit ||
      e == cudaErrorStreamCaptureInvalidated)
    return fail(SKG_ECAPTURING, "%s: not allowed while a stream is capturing (%s)", what,
                cudaGetErrorString(e));
  return fail(SKG_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

int ok() {
  g_err.clear();
  return SKG_OK;
}

// ECAPTURING when a capture that this call's allocations or synchronous copies
// would disturb is visible from the calling thread: the per-thread default
// stream capturing, or the legacy stream capturing or tied to a capturing
// blocking stream (the legacy-stream query reports that without invalidating
// the capture).  The per-thread stream is asked first, so a capture on it is
// refused before the legacy stream is touched.  A capture on a non-blocking
// stream is not visible here.
int refuse_if_capturing(const char* what) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(cudaStreamPerThread, &cs);
  if (e == cudaSuccess && cs == cudaStreamCaptureStatusNone)
    e = cudaStreamIsCapturing(cudaStreamLegacy, &cs);
  if (e == cudaErrorStreamCaptureImplicit ||
      (e == cudaSuccess && cs != cudaStreamCaptureStatusNone)) {
    (void)cudaGetLastError();
    return fail(SKG_ECAPTURING, "%s must not be called while a stream is capturing", what);
  }
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
  return SKG_OK;
}

bool log_enabled() {
  static const bool on = [] {
    const char* v = getenv("SKINNY_GEMM_LOG");
    return v != nullptr && v[0] != '\0' && v[0] != '0';
  }();
  return on;
}

// ------------------------------------------------------------------ driver entry point
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D tile map over a row-major [rows, cols] matrix with row pitch `pitch`
// elements: box {64, box_rows}, 128-byte swizzle, zero fill outside.
int encode_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int64_t pitch,
               int box_rows, int dtype, CUtensorMapL2promotion promo) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return fail(SKG_ECUDA, "cuTensorMapEncodeTiled unavailable from the driver");
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch) * 2u};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBoxK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt =
      dtype == SKG_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = fn(map, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, promo,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(SKG_EINVAL, "cuTensorMapEncodeTiled failed (%d) for [%lld, %lld] pitch %lld box %d",
                static_cast<int>(r), static_cast<long long>(rows), static_cast<long long>(cols),
                static_cast<long long>(pitch), box_rows);
  return SKG_OK;
}

// Tensor map of the activations x [M, K] (pitch ldx, box {64, tok}).  A decode
// loop passes the same activation buffers call after call, so the encoded maps
// are kept in a small per-thread cache keyed by everything the encoding reads
// (a map holds no device state: reusing one for the same key is exact).
struct XMapEntry {
  const void* x = nullptr;
  int64_t M = 0, K = 0, ldx = 0;
  int tok = 0, dtype = -1;
  CUtensorMap map{};
};
thread_local XMapEntry t_xmaps[16];

int x_map(CUtensorMap* out, const void* x, int64_t M, int64_t K, int64_t ldx, int tok, int dtype) {
  const uintptr_t key = reinterpret_cast<uintptr_t>(x) ^ static_cast<uintptr_t>(M * 0x9E3779B1ull) ^
                        static_cast<uintptr_t>(tok << 3);
  XMapEntry& e = t_xmaps[(key ^ (key >> 7) ^ (key >> 13)) & 15u];
  if (e.x == x && e.M == M && e.K == K && e.ldx == ldx && e.tok == tok && e.dtype == dtype) {
    *out = e.map;
    return SKG_OK;
  }
  const int rc = encode_map(out, x, M, K, ldx, tok, dtype, CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
  if (rc != SKG_OK) return rc;
  e.x = x;
  e.M = M;
  e.K = K;
  e.ldx = ldx;
  e.tok = tok;
  e.dtype = dtype;
  e.map = *out;
  return SKG_OK;
}

// ------------------------------------------------------------------ kernels / tactics
// cl: cluster size (tc, mma); for stream-K, CTAs per SM (mode 0, "g") or
// parts per row tile (mode 1, "p").
struct Tactic {
  int variant = 0, rows = 0, tok = 0, nbox = 0, stages = 0, cl = 0, mode = 0;
  int lt = 0;  // k >= 1: launch dependents only with k-1 stages' loads left to issue (mma / tc)
  int al = 0;  // 1: tcgen05 cluster receive buffer aliases the pipeline stages
  int dy = 0;  // 1: K boxes after the first stages shared out at run time within the cluster
  int pf = 0;  // k >= 1: the next k stages' weight boxes prefetched into L2 before the PDL wait
  int rs = 0;  // 1: tcgen05 cluster reduction by per-thread stores at >= 64 tokens (no bulk copies)
  bool valid() const { return variant != 0; }
};

// "tc:r128:t16:b2:s4:c8" (c = cluster size) or "sk:r128:t16:b2:s5:g1" (g = CTAs per SM),
// with ":d<k>" appended for a late PDL trigger (mma / tc), ":a" for a tcgen05
// cluster reduction buffer aliased onto the pipeline stages, ":w" for K boxes
// shared out at run time within a cluster and ":p<k>" for k stages of weight
// boxes prefetched into L2 before the PDL wait; ":s" makes a tcgen05 cluster
// reduction at >= 64 tokens use per-thread stores instead of bulk copies.
std::string tactic_str(const Tactic& t) {
  char b[96];
  const char* kind = t.variant == kVariantTc ? "tc" : (t.variant == kVariantSk ? "sk" : "mma");
  const char last = t.variant != kVariantSk ? 'c' : (t.mode == 1 ? 'p' : 'g');
  char lt[16] = "", pf[16] = "";
  if (t.lt > 0) snprintf(lt, sizeof lt, ":d%d", t.lt);
  if (t.pf > 0) snprintf(pf, sizeof pf, ":p%d", t.pf);
  snprintf(b, sizeof b, "%s:r%d:t%d:b%d:s%d:%c%d%s%s%s%s%s", kind, t.rows, t.tok, t.nbox, t.stages,
           last, t.cl, lt, pf, t.al ? ":a" : "", t.rs ? ":s" : "", t.dy ? ":w" : "");
  return b;
}

bool tactic_parse(const char* s, Tactic* t) {
  char kind[16] = {0};
  char last = 0;
  Tactic x;
  int used = 0;
  if (s == nullptr || sscanf(s, "%15[^:]:r%d:t%d:b%d:s%d:%c%d%n", kind, &x.rows, &x.tok, &x.nbox,
                             &x.stages, &last, &x.cl, &used) != 7)
    return false;
  // optional suffixes, in any order, each at most once: ":d<k>", ":p<k>", ":a", ":s", ":w"
  const char* rest = s + used;
  while (*rest != '\0') {
    if (strncmp(rest, ":d", 2) == 0 && x.lt == 0) {
      int k = 0, n2 = 0;
      if (sscanf(rest, ":d%d%n", &k, &n2) != 1 || k < 1 || k > 64) return false;
      x.lt = k;
      rest += n2;
    } else if (strncmp(rest, ":p", 2) == 0 && x.pf == 0) {
      int k = 0, n2 = 0;
      if (sscanf(rest, ":p%d%n", &k, &n2) != 1 || k < 1 || k > 16) return false;
      x.pf = k;
      rest += n2;
    } else if (strncmp(rest, ":a", 2) == 0 && (rest[2] == '\0' || rest[2] == ':') && x.al == 0) {
      x.al = 1;
      rest += 2;
    } else if (strncmp(rest, ":s", 2) == 0 && (rest[2] == '\0' || rest[2] == ':') && x.rs == 0) {
      x.rs = 1;
      rest += 2;
    } else if (strncmp(rest, ":w", 2) == 0 && (rest[2] == '\0' || rest[2] == ':') && x.dy == 0) {
      x.dy = 1;
      rest += 2;
    } else {
      return false;
    }
  }
  if (strcmp(kind, "tc") == 0 && last == 'c')
    x.variant = kVariantTc;
  else if (strcmp(kind, "mma") == 0 && last == 'c')
    x.variant = kVariantMma;
  else if (strcmp(kind, "sk") == 0 && (last == 'g' || last == 'p')) {
    x.variant = kVariantSk;
    x.mode = last == 'p' ? 1 : 0;
  } else
    return false;
  if (x.lt && x.variant == kVariantSk) return false;
  if (x.al && x.variant != kVariantTc) return false;
  if (x.dy && x.variant == kVariantSk) return false;
  if (x.pf && (x.variant == kVariantSk || x.dy)) return false;
  if (x.rs && x.variant != kVariantTc) return false;
  *t = x;
  return true;
}

const KernelEntry* find_kernel(const Tactic& t, int in_dtype, int out_dtype) {
  int n = 0;
  const KernelEntry* tab = t.variant == kVariantTc   ? tc_kernel_table(&n)
                           : t.variant == kVariantSk ? sk_kernel_table(&n)
                                                     : mma_kernel_table(&n);
  for (int i = 0; i < n; ++i)
    if (tab[i].rows == t.rows && tab[i].tok == t.tok && tab[i].nbox == t.nbox &&
        tab[i].in_dtype == in_dtype && tab[i].out_dtype == out_dtype)
      return &tab[i];
  return nullptr;
}

std::vector<const KernelEntry*> all_kernels() {
  std::vector<const KernelEntry*> v;
  int n = 0;
  const KernelEntry* a = tc_kernel_table(&n);
  for (int i = 0; i < n; ++i) v.push_back(&a[i]);
  a = mma_kernel_table(&n);
  for (int i = 0; i < n; ++i) v.push_back(&a[i]);
  a = sk_kernel_table(&n);
  for (int i = 0; i < n; ++i) v.push_back(&a[i]);
  return v;
}

struct DeviceInfo {
  int sm_count = 0, smem_optin = 0, l2_bytes = 0, major = 0, minor = 0;
  int smem_per_sm = 0, smem_reserved = 0, regs_per_sm = 0, threads_per_sm = 0;
  char name[256] = {0};
  bool attrs_set = false;
};

std::mutex g_dev_mu;
DeviceInfo g_dev[64];

int device_info(int dev, DeviceInfo** out) {
  if (dev < 0 || dev >= 64) return fail(SKG_EDEVICE, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.attrs_set) {
    cudaDeviceProp prop;
    cudaError_t e = cudaGetDeviceProperties(&prop, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
    d.sm_count = prop.multiProcessorCount;
    d.smem_optin = static_cast<int>(prop.sharedMemPerBlockOptin);
    d.l2_bytes = prop.l2CacheSize;
    d.smem_per_sm = static_cast<int>(prop.sharedMemPerMultiprocessor);
    d.smem_reserved = static_cast<int>(prop.reservedSharedMemPerBlock);
    d.regs_per_sm = prop.regsPerMultiprocessor;
    d.threads_per_sm = prop.maxThreadsPerMultiProcessor;
    d.major = prop.major;
    d.minor = prop.minor;
    snprintf(d.name, sizeof d.name, "%s", prop.name);
    if (!(d.major == 10 && d.minor == 3))
      return fail(SKG_EDEVICE, "device %d is sm_%d%d; this library is built for sm_103a only", dev,
                  d.major, d.minor);
    for (const KernelEntry* k : all_kernels()) {
      e = cudaFuncSetAttribute(k->func, cudaFuncAttributeMaxDynamicSharedMemorySize, d.smem_optin);
      if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(max dynamic smem)");
      e = cudaFuncSetAttribute(k->func, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(non-portable cluster)");
      // Operands arrive through TMA into shared memory; L1 is barely used.
      e = cudaFuncSetAttribute(k->func, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
      if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(carveout)");
    }
    d.attrs_set = true;
  }
  *out = &d;
  return SKG_OK;
}

uint64_t env_u64(const char* name, uint64_t dflt) {
  const char* v = getenv(name);
  if (v == nullptr || *v == '\0') return dflt;
  return strtoull(v, nullptr, 10);
}

const int kTcToks[] = {16, 32, 48, 64, 128, 256};
const int kSkToks[] = {16, 32, 64};
const int kMmaToks[] = {8, 16, 32};
const int kClusters[] = {1, 2, 4, 8, 16};

}  // namespace

// ------------------------------------------------------------------ handle
struct skinny_gemm_plan {
  const void* W = nullptr;
  int64_t N = 0, K = 0, ldw = 0;
  int dtype = SKG_BF16, out_dtype = SKG_BF16;
  int device = 0;
  DeviceInfo* dev = nullptr;
  int kboxes = 0;
  CUtensorMap wmap64{}, wmap128{};
  Tactic plan[SKINNY_GEMM_MAX_M + 1];
  uint32_t* status = nullptr;
  float* workspace = nullptr;      // stream-K partial sums (allocated when a tactic needs it)
  size_t workspace_bytes = 0;
  uint32_t* counters = nullptr;    // stream-K per-tile arrival counters, zero between launches
  size_t counters_bytes = 0;
  void* x_stage = nullptr;
  void* out_stage = nullptr;
  uint64_t timeout_ns = 2000000000ull;
  int debug_count = 0;
  int debug_kind = 1;  // KParams::debug_wait of the injected launches (1 timeout, 2 check)
  bool pdl = true;  // programmatic dependent launch attribute on every launch
  bool deterministic = false;  // the tuner keeps a fixed summation order (no :w tactics)
  uint64_t debug_timeout_ns = 0;
};

namespace {

int out_elem_bytes(const skinny_gemm_plan* h) { return h->out_dtype == SKG_FP32 ? 4 : 2; }

int ntiles_of(const skinny_gemm_plan* h, const Tactic& t) {
  return static_cast<int>((h->N + t.rows - 1) / t.rows);
}
uint32_t tactic_smem(const Tactic& t) {
  if (t.variant == kVariantSk) return sk_smem_bytes(t.tok, t.nbox, t.stages);
  const uint32_t dyn = t.dy ? kDynBytes : 0u;
  if (t.variant == kVariantTc)
    return tc_smem_bytes(t.tok, t.nbox, t.stages, t.cl, t.al != 0, t.rows) + dyn;
  return smem_bytes(t.rows, t.tok, t.nbox, t.stages) + dyn;
}
// CTAs launched: row tiles x cluster size, or (stream-K) CTAs-per-SM x SMs,
// capped at the number of work units.
int tactic_grid(const skinny_gemm_plan* h, const Tactic& t) {
  if (t.variant != kVariantSk) return ntiles_of(h, t) * t.cl;
  const int64_t units = static_cast<int64_t>(ntiles_of(h, t)) * h->kboxes;
  const int64_t want = t.mode == 1 ? static_cast<int64_t>(ntiles_of(h, t)) * t.cl
                                   : static_cast<int64_t>(t.cl) * h->dev->sm_count;
  return static_cast<int>(std::min<int64_t>(want, units));
}
int tactic_cluster(const Tactic& t) { return t.variant == kVariantSk ? 1 : t.cl; }
// Stream-K scratch: two fp32 [TOK][128] partial-sum slots per CTA, one counter per tile.
void workspace_need(const skinny_gemm_plan* h, const Tactic& t, size_t* ws, size_t* cnt) {
  if (t.variant != kVariantSk) {
    *ws = *cnt = 0;
    return;
  }
  *ws = static_cast<size_t>(tactic_grid(h, t)) * 2 * t.tok * t.rows * sizeof(float);
  *cnt = static_cast<size_t>(ntiles_of(h, t)) * sizeof(uint32_t);
}

// Validity of tactic t for this weight at token count M (M = 0: any M <= tok).
bool tactic_fits(const skinny_gemm_plan* h, const Tactic& t, int64_t M, std::string* why) {
  auto no = [&](const char* w) {
    if (why) *why = w;
    return false;
  };
  if (!t.valid()) return no("empty tactic");
  const KernelEntry* k = find_kernel(t, h->dtype, h->out_dtype);
  if (k == nullptr) return no("no compiled kernel for this rows/tok/box/dtype combination");
  // tcgen05 tactics cover M > tok with ceil(M / tok) token tiles (grid y);
  // the others need one tile of at least M tokens.
  if (M > t.tok && t.variant != kVariantTc) return no("token tile smaller than M");
  if (t.variant == kVariantSk) {
    if (t.mode == 0 && t.cl != 1 && t.cl != 2) return no("stream-K runs 1 or 2 CTAs per SM");
    if (t.mode == 1 && (t.cl < 1 || t.cl > 64 || t.cl > h->kboxes))
      return no("parts per tile must be 1..64 and at most the number of 64-wide K blocks");
  } else {
    bool pow2 = false;
    for (int c : kClusters) pow2 |= (c == t.cl);
    if (!pow2) return no("cluster size must be 1, 2, 4, 8 or 16");
    if (t.cl > h->kboxes) return no("cluster larger than the number of 64-wide K blocks");
    if (t.rows % t.cl != 0) return no("cluster size must divide the row tile");
  }
  if (t.stages < 1 || t.stages > 16) return no("stages out of range 1..16");
  if (t.variant == kVariantTc && t.rows / t.cl < 8)
    return no("tcgen05 cluster reduction needs at least 8 rows per CTA (rows / cluster)");
  if (t.al && (t.cl < 2 || static_cast<uint32_t>(t.stages) * stage_bytes(t.rows, t.tok, t.nbox) <
                               tc_red_bytes(t.tok, t.rows)))
    return no("an aliased receive buffer needs a cluster and stages at least as large");
  if (t.dy && (t.cl < 2 || t.al))
    return no("run-time K sharing (:w) needs a cluster and no aliased receive buffer");
  if (t.rs && (t.cl < 2 || t.tok < 64))
    return no("per-thread reduction stores (:s) apply to tcgen05 clusters at >= 64 tokens");
  if (static_cast<int>(tactic_smem(t)) > h->dev->smem_optin)
    return no("shared memory footprint exceeds the per-block limit");
  return true;
}

// Grow the handle's stream-K workspace and counters to fit tactic t.  Only
// called from prepare / set_tactic / autotune (never from run): it may
// synchronize the device and allocate.
int ensure_workspace(skinny_gemm_plan* h, const Tactic& t) {
  size_t ws = 0, cnt = 0;
  workspace_need(h, t, &ws, &cnt);
  if (ws <= h->workspace_bytes && cnt <= h->counters_bytes) return SKG_OK;
  cudaError_t e = cudaDeviceSynchronize();  // no launch may still use the old buffers
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  if (ws > h->workspace_bytes) {
    if (h->workspace) cudaFree(h->workspace);
    h->workspace = nullptr;
    h->workspace_bytes = 0;
    e = cudaMalloc(&h->workspace, ws);
    if (e != cudaSuccess) return h->workspace = nullptr, cuda_fail(e, "cudaMalloc(workspace)");
    h->workspace_bytes = ws;
  }
  if (cnt > h->counters_bytes) {
    if (h->counters) cudaFree(h->counters);
    h->counters = nullptr;
    h->counters_bytes = 0;
    e = cudaMalloc(&h->counters, cnt);
    if (e != cudaSuccess) return h->counters = nullptr, cuda_fail(e, "cudaMalloc(counters)");
    e = cudaMemset(h->counters, 0, cnt);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(counters)");
    h->counters_bytes = cnt;
  }
  return SKG_OK;
}

int launch_tactic(skinny_gemm_plan* h, const Tactic& t, const void* x, int64_t ldx, int64_t M,
                  void* out, int64_t ldo, cudaStream_t st, const void* residual = nullptr,
                  int64_t ldr = 0) {
  const KernelEntry* k = find_kernel(t, h->dtype, h->out_dtype);
  if (k == nullptr) return fail(SKG_EINVAL, "no kernel for tactic %s", tactic_str(t).c_str());
  if (t.variant == kVariantSk) {
    size_t ws = 0, cnt = 0;
    workspace_need(h, t, &ws, &cnt);
    if (ws > h->workspace_bytes || cnt > h->counters_bytes)
      return fail(SKG_EINVAL, "tactic %s needs a workspace this handle has not prepared",
                  tactic_str(t).c_str());
  }
  CUtensorMap xmap;
  int rc = x_map(&xmap, x, M, h->K, ldx, t.tok, h->dtype);
  if (rc != SKG_OK) return rc;
  KParams p{};
  p.out = out;
  p.ldo = ldo;
  p.M = static_cast<int32_t>(M);
  p.N = static_cast<int32_t>(h->N);
  p.kboxes = h->kboxes;
  p.stages = t.stages;
  p.status = h->status;
  p.timeout_ns = h->timeout_ns;
  p.workspace = h->workspace;
  p.counters = h->counters;
  p.residual = residual;
  p.ldr = ldr;
  p.pdl_late = t.lt;
  p.red_alias = t.al;
  p.dyn_k = t.dy;
  p.l2_pre = t.pf;
  p.red_stores = t.rs;
  if (h->debug_count > 0) {
    --h->debug_count;
    p.debug_wait = h->debug_kind;
    p.timeout_ns = h->debug_timeout_ns;
  }
  cudaLaunchConfig_t cfg{};
  const unsigned ty = t.variant == kVariantTc ? static_cast<unsigned>((M + t.tok - 1) / t.tok) : 1u;
  cfg.gridDim = dim3(static_cast<unsigned>(tactic_grid(h, t)), ty, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(k->threads), 1, 1);
  cfg.dynamicSmemBytes = tactic_smem(t);
  cfg.stream = st;
  // A cluster attribute, even of size 1, makes the launch a cluster launch,
  // which was measured to allow only one cluster per SM: attach it only for
  // real clusters.
  cudaLaunchAttribute attrs[2];
  int na = 0;
  if (h->pdl) {
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (tactic_cluster(t) > 1) {
    attrs[na].id = cudaLaunchAttributeClusterDimension;
    attrs[na].val.clusterDim.x = static_cast<unsigned>(tactic_cluster(t));
    attrs[na].val.clusterDim.y = 1;
    attrs[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = static_cast<unsigned>(na);
  const CUtensorMap* wmap = t.rows == 64 ? &h->wmap64 : &h->wmap128;
  void* args[3] = {const_cast<CUtensorMap*>(wmap), &xmap, &p};
  cudaError_t e = cudaLaunchKernelExC(&cfg, k->func, args);
  if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchKernelExC");
  return SKG_OK;
}

// CTAs of this tactic one SM holds at once, counted from shared memory,
// registers, threads and tensor-memory columns (0: cannot launch).  Counted
// here rather than by cudaOccupancyMaxActiveBlocksPerMultiprocessor, which
// answers one block per SM for any kernel that allocates tensor memory
// (measured: four such blocks of 32 columns ran at once per SM).
int resident_per_sm(const skinny_gemm_plan* h, const Tactic& t) {
  const KernelEntry* k = find_kernel(t, h->dtype, h->out_dtype);
  if (k == nullptr) return 0;
  cudaFuncAttributes fa{};
  if (cudaFuncGetAttributes(&fa, k->func) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  const DeviceInfo& d = *h->dev;
  const int regs = ((fa.numRegs + 7) / 8) * 8 * k->threads;
  int per_sm = std::min(32, d.threads_per_sm / k->threads);
  per_sm = std::min(per_sm, regs > 0 ? d.regs_per_sm / regs : per_sm);
  per_sm = std::min(per_sm, d.smem_per_sm / static_cast<int>(tactic_smem(t) + d.smem_reserved));
  const int tmem_cols = t.variant == kVariantSk  ? (2 * t.tok <= 32 ? 32 : (2 * t.tok <= 64 ? 64 : 128))
                        : t.variant == kVariantTc ? (t.tok <= 32 ? 32 : t.tok <= 64 ? 64 : t.tok <= 128 ? 128 : 256)
                                                  : 0;
  if (tmem_cols > 0) per_sm = std::min(per_sm, 512 / tmem_cols);
  return std::max(per_sm, 0);
}

// Clusters of this tactic that fit on the GPU at once (0: cannot launch).
// Without clusters this is resident CTAs per SM x SMs.
int active_clusters(const skinny_gemm_plan* h, const Tactic& t) {
  const KernelEntry* k = find_kernel(t, h->dtype, h->out_dtype);
  if (k == nullptr) return 0;
  if (tactic_cluster(t) == 1) return resident_per_sm(h, t) * h->dev->sm_count;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(tactic_grid(h, t)), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(k->threads), 1, 1);
  cfg.dynamicSmemBytes = tactic_smem(t);
  cudaLaunchAttribute a[1];
  a[0].id = cudaLaunchAttributeClusterDimension;
  a[0].val.clusterDim.x = static_cast<unsigned>(tactic_cluster(t));
  a[0].val.clusterDim.y = 1;
  a[0].val.clusterDim.z = 1;
  cfg.attrs = a;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k->func, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

// Number of refill stages of a CTA's K range after its first `stages` (the
// late-trigger settings 1..span launch dependents at distinct points).
int late_trigger_span(const skinny_gemm_plan* h, const Tactic& t) {
  if (t.variant == kVariantSk || t.cl < 1) return 0;
  const int nb = static_cast<int>((h->kboxes + t.cl - 1) / t.cl);
  const int iters = (nb + t.nbox - 1) / t.nbox;
  return std::max(0, iters - std::min(iters, t.stages));
}

// Candidate tactics for M: the smallest token tile >= M of each variant (for
// M > 64 also tcgen05 tiles of 64 and 128 tokens repeated over ceil(M / tok)
// token tiles), every stage count / box count / cluster size that fits and
// can launch.
std::vector<Tactic> candidates(const skinny_gemm_plan* h, int64_t M) {
  std::vector<Tactic> out;
  std::vector<std::pair<int, int>> vt;  // (variant, token tile)
  for (int variant : {kVariantTc, kVariantMma, kVariantSk}) {
    const int* toks = variant == kVariantMma ? kMmaToks : (variant == kVariantSk ? kSkToks : kTcToks);
    const int ntok = variant == kVariantTc ? 6 : 3;
    for (int i = 0; i < ntok; ++i)
      if (toks[i] >= M) {
        vt.push_back({variant, toks[i]});
        break;
      }
    if (variant == kVariantTc && M > 64)
      for (int tok : {64, 128})
        if (tok < M) vt.push_back({variant, tok});
  }
  for (const auto& [variant, tok] : vt) {
    for (const KernelEntry* k : all_kernels()) {
      if (k->variant != variant || k->tok != tok || k->in_dtype != h->dtype ||
          k->out_dtype != h->out_dtype)
        continue;
      std::vector<std::pair<int, int>> grids;  // (cl, mode)
      if (variant == kVariantSk) {
        for (int g : {1, 2}) grids.push_back({g, 0});
        for (int pp : {1, 2, 3, 4, 6, 8, 12, 16}) grids.push_back({pp, 1});
      } else {
        for (int cl : kClusters) grids.push_back({cl, 0});
      }
      for (const auto& gm : grids)
        for (int s = 2; s <= 8; ++s) {
          Tactic t{variant, k->rows, tok, k->nbox, s, gm.first, gm.second};
          if (!tactic_fits(h, t, M, nullptr)) continue;
          const int act = active_clusters(h, t);
          // stream-K: every CTA of the grid must be resident at once (one wave)
          if (act <= 0 || (variant == kVariantSk && act < tactic_grid(h, t))) {
            if (log_enabled())
              fprintf(stderr, "[skinny_gemm] candidate %s rejected: %d resident of %d (smem %u)\n",
                      tactic_str(t).c_str(), act * tactic_cluster(t), tactic_grid(h, t),
                      tactic_smem(t));
            continue;
          }
          out.push_back(t);
          // tcgen05 clusters: the variant whose receive buffer aliases the stages,
          // when that lets more CTAs share an SM, and always at >= 48 tokens,
          // where it timed fastest on the 3584x7168 weight at equal residency (it
          // waits for the whole cluster's MMAs before reducing).
          if (variant == kVariantTc && t.cl > 1) {
            Tactic ta = t;
            ta.al = 1;
            const int per = h->dev->smem_per_sm;
            const int rsv = h->dev->smem_reserved;
            if (tactic_fits(h, ta, M, nullptr) &&
                (tok >= 48 || per / static_cast<int>(tactic_smem(ta) + rsv) >
                                  per / static_cast<int>(tactic_smem(t) + rsv)) &&
                active_clusters(h, ta) > 0)
              out.push_back(ta);
          }
        }
    }
  }
  return out;
}

// Default (untuned) choice, from what the autotuner picked on GB300 for the
// 3584x7168 and 6288x7168 weights with every weight read from HBM:
//   M <= 8   mma.sync, 128-row tiles, 8-token tile, 1 box x 2 stages with a
//            16-way cluster where that keeps <= 3 CTAs/SM, else 2 boxes x 3 stages
//   M <= 16  mma.sync, 64-row tiles, 16-token tile, 2 boxes x 2 stages
//   M <= 32  tcgen05, 32-token tile, 2 boxes x 2 stages
//   M <= 64  tcgen05, 64-token tile, 1 box x 3 stages
// with the cluster split (split-K factor) that gives about 1.4 CTAs per SM
// (64-row tiles and the one-box 8-token tiles: the largest giving at most 3),
// at most 8 (16 for the latter); fewer stages where shared memory or
// the K range is short, or where the grid would not be resident in one wave
// (then 3 -> 2 stages, then half the cluster: e.g. the 6288x7168 weight runs
// 2 stages for its 8-token tile and clusters of 4 for its 32/64-token tiles).  Any
// choice that does not fit falls back to fewer stages, then to the tcgen05
// kernel with the same rule.  Every default issues its PDL trigger late (3
// stages before the end for mma.sync, 2 for tcgen05) and prefetches into L2 the
// weight stages after its first ones before it waits on the previous kernel
// (one stage, two above 32 tokens, within the K range).
Tactic default_tactic(const skinny_gemm_plan* h, int64_t M) {
  Tactic best;
  // Split-K cluster size: the smallest giving at least 1.4 CTAs per SM, or
  // (cap3, the 64-row tiles) the largest giving at most 3 CTAs per SM.
  auto with_cluster = [&](Tactic t, bool cap3 = false) {
    const int ntiles = static_cast<int>((h->N + t.rows - 1) / t.rows);
    const int sms = h->dev->sm_count;
    int cl = 1;
    const int cl_max = cap3 && t.nbox == 1 ? 16 : 8;
    while (cl < cl_max && cl * 2 <= h->kboxes && t.rows % (cl * 2) == 0 &&
           (cap3 ? ntiles * cl * 2 <= 3 * sms : ntiles * cl * 10 < sms * 14))
      cl *= 2;
    t.cl = cl;
    const int iters = ((h->kboxes + cl - 1) / cl + t.nbox - 1) / t.nbox;
    t.stages = std::max(1, std::min(t.stages, iters));
    // Late PDL trigger (measured on the 3584x7168 and 6288x7168 weights): with
    // 2 (tcgen05) or 3 (mma.sync) stages still to issue.
    t.lt = t.variant == kVariantMma ? 3 : 2;
    // Fewer stages (down to 2), then a smaller cluster, until the whole grid is
    // resident at once (one wave); else the first tactic that fits.
    Tactic fit;
    const int s0 = t.stages;
    for (; t.cl >= 1; t.cl /= 2) {
      for (t.stages = s0; t.stages >= 1; --t.stages) {
        // L2 prefetch of the stages after the first ones before the PDL wait
        // (measured on both weights: every default tactic gains 0.1-1.1 us with
        // one stage, those above 32 tokens more with two), within the K range
        t.pf = std::min(M > 32 ? 2 : 1, late_trigger_span(h, t));
        if (!tactic_fits(h, t, M, nullptr)) continue;
        if (!fit.valid()) fit = t;
        // (per-SM count: the cluster occupancy query undercounts tensor-memory kernels)
        const int64_t resident = static_cast<int64_t>(resident_per_sm(h, t)) * h->dev->sm_count;
        if (resident >= tactic_grid(h, t)) return t;
        if (t.stages <= 2) break;
      }
    }
    return fit;
  };
  Tactic t;
  if (M <= 8) {
    // one-box stages pay off with 16-way clusters (measured on 3584x7168: 9.4 us
    // vs 9.6); where the weight has too many row tiles for that (6288x7168) the
    // two-box stages with a 1.4 CTAs/SM cluster stay ahead.
    t = with_cluster(Tactic{kVariantMma, 128, 8, 1, 2, 1, 0}, true);
    if (!t.valid() || t.cl < 16) t = with_cluster(Tactic{kVariantMma, 128, 8, 2, 3, 1, 0});
  }
  else if (M <= 16)
    t = with_cluster(Tactic{kVariantMma, 64, 16, 2, 2, 1, 0}, true);
  else if (M <= 32)
    t = with_cluster(Tactic{kVariantTc, 128, 32, 2, 2, 1, 0});
  else if (M <= 48)
    t = with_cluster(Tactic{kVariantTc, 128, 48, 1, 3, 1, 0});
  else if (M <= 64)
    t = with_cluster(Tactic{kVariantTc, 128, 64, 1, 3, 1, 0});
  else if (M <= 128)
    t = with_cluster(Tactic{kVariantTc, 128, 128, 1, 2, 1, 0});
  else
    t = with_cluster(Tactic{kVariantTc, 128, 256, 1, 2, 1, 0});
  if (t.valid()) return t;
  for (int tok : kTcToks)
    if (tok >= M) {
      t = with_cluster(Tactic{kVariantTc, 128, tok, 1, 2, 1, 0});
      if (t.valid()) return t;
    }
  return best;
}

// ------------------------------------------------------------------ tactic file
const char* out_name(int d) { return d == SKG_FP32 ? "fp32" : (d == SKG_FP16 ? "fp16" : "bf16"); }

// One whitespace-free word (a tactic-file line is "<key> <M> <tactic> <us>"):
// blanks in the device name ("NVIDIA GB300") become '_'.
std::string cache_key(const skinny_gemm_plan* h) {
  char b[512];
  snprintf(b, sizeof b, "%s|sm%d|N%lld|K%lld|in%s|out%s|abi%d", h->dev->name, h->dev->sm_count,
           static_cast<long long>(h->N), static_cast<long long>(h->K), out_name(h->dtype),
           out_name(h->out_dtype), SKINNY_GEMM_ABI_VERSION);
  std::string k = b;
  for (char& c : k)
    if (c == ' ' || c == '\t' || c == '\n' || c == '\r') c = '_';
  return k;
}

// SKINNY_GEMM_TUNE, read at prepare: "off" (the default plan only; the tactic
// file is ignored), "cache" (the default: entries of SKINNY_GEMM_TACTIC_FILE
// replace the default plan's), "full" (as "cache", then the decode token
// counts the file has no entry for are autotuned at prepare and appended).
// Returns 0, 1 or 2, or -1 for any other value.
int tune_mode() {
  const char* v = getenv("SKINNY_GEMM_TUNE");
  if (v == nullptr || *v == '\0' || strcmp(v, "cache") == 0) return 1;
  if (strcmp(v, "off") == 0) return 0;
  if (strcmp(v, "full") == 0) return 2;
  return -1;
}

// Applies the tactic file's entries for this weight to the plan and marks the
// token counts it set in loaded[1..SKINNY_GEMM_MAX_M].
void load_tactic_file(skinny_gemm_plan* h, bool* loaded) {
  const char* path = getenv("SKINNY_GEMM_TACTIC_FILE");
  if (path == nullptr || *path == '\0') return;
  FILE* f = fopen(path, "r");
  if (f == nullptr) return;
  const std::string key = cache_key(h);
  char line[1024];
  while (fgets(line, sizeof line, f) != nullptr) {
    // line: <key> <M> <tactic> <us>
    char k[600], ts[96];
    int m = 0;
    double us = 0;
    if (sscanf(line, "%599s %d %95s %lf", k, &m, ts, &us) < 3) continue;
    Tactic t;
    if (key != k || m < 1 || m > SKINNY_GEMM_MAX_M || !tactic_parse(ts, &t)) continue;
    if (tactic_fits(h, t, m, nullptr) && active_clusters(h, t) > 0) {  // last wins
      h->plan[m] = t;
      loaded[m] = true;
    }
  }
  fclose(f);
}

// Token counts without an entry of their own take the tactic of the smallest
// M' > M that has one (known[M']), when it fits M: the rule skinny_gemm_autotune
// applies to the token counts it did not time, so a plan rebuilt from the
// tactic file matches the tuned one.
void propagate_plan(skinny_gemm_plan* h, const bool* known) {
  for (int m = 1; m <= SKINNY_GEMM_MAX_M; ++m) {
    if (known[m]) continue;
    for (int mp = m + 1; mp <= SKINNY_GEMM_MAX_M; ++mp)
      if (known[mp]) {
        if (tactic_fits(h, h->plan[mp], m, nullptr)) h->plan[m] = h->plan[mp];
        break;
      }
  }
}

void append_tactic_file(const skinny_gemm_plan* h, int64_t M, const Tactic& t, double us) {
  const char* path = getenv("SKINNY_GEMM_TACTIC_FILE");
  if (path == nullptr || *path == '\0') return;
  FILE* f = fopen(path, "a");
  if (f == nullptr) return;
  fprintf(f, "%s %lld %s %.3f\n", cache_key(h).c_str(), static_cast<long long>(M),
          tactic_str(t).c_str(), us);
  fclose(f);
}

// Live handles (prepare inserts, destroy erases), so that a destroyed or
// foreign pointer is refused with EINVAL instead of being dereferenced.  An
// address reused by a later prepare is indistinguishable from that handle.
std::mutex g_handles_mu;
std::unordered_set<const skinny_gemm_plan*>& live_handles() {
  static std::unordered_set<const skinny_gemm_plan*> s;
  return s;
}
void register_handle(const skinny_gemm_plan* h) {
  std::lock_guard<std::mutex> lk(g_handles_mu);
  live_handles().insert(h);
}
bool unregister_handle(const skinny_gemm_plan* h) {
  std::lock_guard<std::mutex> lk(g_handles_mu);
  return live_handles().erase(h) > 0;
}

int check_handle(const skinny_gemm_plan* h) {
  if (h == nullptr) return fail(SKG_EINVAL, "null handle");
  {
    std::lock_guard<std::mutex> lk(g_handles_mu);
    if (live_handles().count(h) == 0) return fail(SKG_EINVAL, "unknown or destroyed handle");
  }
  return SKG_OK;
}

// Argument checks of a run on a plan (the handle itself is checked by callers
// of the public entry points; the tuners pass private copies of a plan).
int validate_args(const skinny_gemm_plan* h, const void* x, int64_t ldx, int64_t M, const void* out,
                  int64_t ldo) {
  if (M < 1 || M > SKINNY_GEMM_MAX_M)
    return fail(SKG_EUNSUPPORTED_M, "M = %lld outside 1..%d: fall back", static_cast<long long>(M),
                SKINNY_GEMM_MAX_M);
  if (x == nullptr || out == nullptr) return fail(SKG_EINVAL, "null x or out");
  if (ldx < h->K || ldo < h->N)
    return fail(SKG_EINVAL, "row pitch too small: ldx %lld (K %lld), ldo %lld (N %lld)",
                static_cast<long long>(ldx), static_cast<long long>(h->K),
                static_cast<long long>(ldo), static_cast<long long>(h->N));
  if (reinterpret_cast<uintptr_t>(x) % 16 || reinterpret_cast<uintptr_t>(out) % 16)
    return fail(SKG_EALIGN, "x and out must be 16-byte aligned");
  if ((ldx * 2) % 16) return fail(SKG_EALIGN, "x row pitch must be a multiple of 16 bytes");
  return SKG_OK;
}

int validate_run(const skinny_gemm_plan* h, const void* x, int64_t ldx, int64_t M, const void* out,
                 int64_t ldo) {
  if (check_handle(h) != SKG_OK) return SKG_EINVAL;
  return validate_args(h, x, ldx, M, out, ldo);
}

}  // namespace

// ------------------------------------------------------------------ C ABI
extern "C" {

int skinny_gemm_abi_version(void) { return SKINNY_GEMM_ABI_VERSION; }

const char* skinny_gemm_last_error(void) { return g_err.c_str(); }

int skinny_gemm_last_status(void) { return g_last_status; }

skinny_gemm_t skinny_gemm_prepare_ex(const void* W, int64_t N, int64_t K, int64_t ldw, int dtype,
                                     int out_dtype, unsigned flags) {
  g_last_status = 0;
  if (W == nullptr) return fail(SKG_EINVAL, "null weight pointer"), nullptr;
  if (dtype != SKG_BF16 && dtype != SKG_FP16)
    return fail(SKG_EINVAL, "weight dtype %d unsupported: BF16 or FP16", dtype), nullptr;
  // Output: FP32, or the operands' own 16-bit type.
  if (out_dtype != SKG_FP32 && out_dtype != dtype)
    return fail(SKG_EINVAL,
                "unsupported projection output dtype %d for %s operands (%s or FP32)", out_dtype,
                dtype == SKG_FP16 ? "FP16" : "BF16", dtype == SKG_FP16 ? "FP16" : "BF16"),
           nullptr;
  if (N < 1 || K < 8 || N > (1ll << 31) - 1 || K > (1ll << 31) - 1)
    return fail(SKG_EINVAL, "weight shape [%lld, %lld] out of range", static_cast<long long>(N),
                static_cast<long long>(K)),
           nullptr;
  if (K % 8 != 0)
    return fail(SKG_EALIGN, "K = %lld: rows need a 16-byte multiple length (K %% 8 == 0)",
                static_cast<long long>(K)),
           nullptr;
  if (ldw < K || ldw % 8 != 0)
    return fail(SKG_EALIGN, "weight rows need unit stride and a 16 B TMA pitch (ldw %lld)",
                static_cast<long long>(ldw)),
           nullptr;
  if (reinterpret_cast<uintptr_t>(W) % 16 != 0)
    return fail(SKG_EALIGN, "weight base must be 16-byte aligned"), nullptr;
  const int mode = (flags & SKG_PREPARE_NO_TUNE_CACHE) ? 0 : tune_mode();
  if (mode < 0)
    return fail(SKG_EINVAL, "SKINNY_GEMM_TUNE must be off, cache or full"), nullptr;
  // prepare allocates and clears device memory, which a capture must not see
  if (refuse_if_capturing("skinny_gemm_prepare") != SKG_OK) return nullptr;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice"), nullptr;
  DeviceInfo* di = nullptr;
  if (device_info(dev, &di) != SKG_OK) return nullptr;

  auto* h = new skinny_gemm_plan();
  h->W = W;
  h->N = N;
  h->K = K;
  h->ldw = ldw;
  h->dtype = dtype;
  h->out_dtype = out_dtype;
  h->device = dev;
  h->dev = di;
  h->kboxes = static_cast<int>((K + kBoxK - 1) / kBoxK);
  h->timeout_ns = env_u64("SKINNY_GEMM_TIMEOUT_NS", 2000000000ull);
  if (encode_map(&h->wmap64, W, N, K, ldw, 64, dtype, CU_TENSOR_MAP_L2_PROMOTION_L2_256B) != SKG_OK ||
      encode_map(&h->wmap128, W, N, K, ldw, 128, dtype, CU_TENSOR_MAP_L2_PROMOTION_L2_256B) != SKG_OK) {
    delete h;
    return nullptr;
  }
  e = cudaMalloc(&h->status, sizeof(uint32_t));
  if (e != cudaSuccess) {
    h->status = nullptr;
    cuda_fail(e, "cudaMalloc(status word)");
    delete h;
    return nullptr;
  }
  e = cudaMemset(h->status, 0, sizeof(uint32_t));
  if (e != cudaSuccess) {
    cuda_fail(e, "cudaMemset(status word)");
    skinny_gemm_destroy(h);
    return nullptr;
  }
  for (int m = 1; m <= SKINNY_GEMM_MAX_M; ++m) h->plan[m] = default_tactic(h, m);
  h->pdl = !(flags & SKG_PREPARE_NO_PDL);
  h->deterministic = (flags & SKG_PREPARE_DETERMINISTIC) != 0;
  bool loaded[SKINNY_GEMM_MAX_M + 1] = {};
  if (mode >= 1) {
    load_tactic_file(h, loaded);
    propagate_plan(h, loaded);
  }
  bool forced = false;
  if (const char* f = getenv("SKINNY_GEMM_FORCE_TACTIC")) {
    Tactic t;
    if (tactic_parse(f, &t))
      for (int m = 1; m <= SKINNY_GEMM_MAX_M; ++m)
        if (tactic_fits(h, t, m, nullptr)) {
          h->plan[m] = t;
          forced = true;
        }
  }
  for (int m = 1; m <= SKINNY_GEMM_MAX_M; ++m) {
    if (!h->plan[m].valid()) {
      fail(SKG_EINVAL, "no valid tactic for M = %d on this weight", m);
      skinny_gemm_destroy(h);
      return nullptr;
    }
    if (ensure_workspace(h, h->plan[m]) != SKG_OK) {
      const int code = g_last_status;
      const std::string msg = g_err;
      skinny_gemm_destroy(h);
      fail(code, "%s", msg.c_str());
      return nullptr;
    }
  }
  if (log_enabled()) {
    fprintf(stderr, "[skinny_gemm] prepared N=%lld K=%lld on %s (%d SMs):", static_cast<long long>(N),
            static_cast<long long>(K), di->name, di->sm_count);
    for (int m : {1, 2, 4, 8, 16, 32, 48, 64}) fprintf(stderr, " M%d=%s", m, tactic_str(h->plan[m]).c_str());
    fprintf(stderr, "\n");
  }
  register_handle(h);
  if (mode == 2 && !forced) {
    std::vector<int64_t> want;
    for (int m : {1, 2, 4, 8, 16, 32, 48, 64})
      if (!loaded[m]) want.push_back(m);
    std::vector<Tactic> from_file(h->plan, h->plan + SKINNY_GEMM_MAX_M + 1);
    int rc = SKG_OK;
    if (!want.empty())
      rc = skinny_gemm_autotune(h, want.data(), static_cast<int>(want.size()), nullptr);
    if (rc == SKG_OK) {
      // The tuner spreads its picks over the token counts it did not time; the
      // file's entries stay, and the rest follow the nearest entry above.
      bool known[SKINNY_GEMM_MAX_M + 1] = {};
      for (int m = 1; m <= SKINNY_GEMM_MAX_M; ++m)
        if (loaded[m]) {
          h->plan[m] = from_file[m];
          known[m] = true;
        }
      for (int64_t m : want) known[m] = true;
      propagate_plan(h, known);
      for (int m = 1; m <= SKINNY_GEMM_MAX_M && rc == SKG_OK; ++m) rc = ensure_workspace(h, h->plan[m]);
    }
    if (rc != SKG_OK) {
      const int code = g_last_status;
      const std::string msg = g_err;
      skinny_gemm_destroy(h);
      fail(code, "SKINNY_GEMM_TUNE=full: %s", msg.c_str());
      return nullptr;
    }
  }
  ok();
  return h;
}

skinny_gemm_t skinny_gemm_prepare(const void* W, int64_t N, int64_t K, int dtype, int out_dtype) {
  return skinny_gemm_prepare_ex(W, N, K, K, dtype, out_dtype, 0u);
}

int skinny_gemm_run_strided(skinny_gemm_t h, const void* x, int64_t ldx, int64_t M, void* out,
                            int64_t ldo, void* stream) {
  int rc = validate_run(h, x, ldx, M, out, ldo);
  if (rc != SKG_OK) return rc;
  rc = launch_tactic(h, h->plan[M], x, ldx, M, out, ldo, static_cast<cudaStream_t>(stream));
  return rc == SKG_OK ? ok() : rc;
}

int skinny_gemm_run_residual(skinny_gemm_t h, const void* x, int64_t ldx, int64_t M,
                             const void* residual, int64_t ldr, void* out, int64_t ldo,
                             void* stream) {
  int rc = validate_run(h, x, ldx, M, out, ldo);
  if (rc != SKG_OK) return rc;
  if (residual == nullptr) return fail(SKG_EINVAL, "null residual (use skinny_gemm_run)");
  if (ldr < h->N) return fail(SKG_EINVAL, "residual row pitch %lld < N %lld",
                               static_cast<long long>(ldr), static_cast<long long>(h->N));
  if (reinterpret_cast<uintptr_t>(residual) % out_elem_bytes(h) != 0)
    return fail(SKG_EALIGN, "residual must be aligned to its element size");
  const char* r0 = static_cast<const char*>(residual);
  const char* o0 = static_cast<const char*>(out);
  const size_t esz = static_cast<size_t>(out_elem_bytes(h));
  const char* r1 = r0 + (static_cast<size_t>(M - 1) * ldr + h->N) * esz;
  const char* o1 = o0 + (static_cast<size_t>(M - 1) * ldo + h->N) * esz;
  if (!(r0 == o0 && ldr == ldo) && r0 < o1 && o0 < r1)
    return fail(SKG_EINVAL, "residual overlaps out without being exactly out (in place)");
  rc = launch_tactic(h, h->plan[M], x, ldx, M, out, ldo, static_cast<cudaStream_t>(stream),
                     residual, ldr);
  return rc == SKG_OK ? ok() : rc;
}

int skinny_gemm_run(skinny_gemm_t h, const void* x, int64_t M, void* out, void* stream) {
  if (check_handle(h) != SKG_OK) return SKG_EINVAL;
  int rc = validate_args(h, x, h->K, M, out, h->N);
  if (rc != SKG_OK) return rc;
  rc = launch_tactic(h, h->plan[M], x, h->K, M, out, h->N, static_cast<cudaStream_t>(stream));
  return rc == SKG_OK ? ok() : rc;
}

namespace {
// H2D of x into the handle's staging buffer, the projection, D2H of out, all
// enqueued on `st` (staging allocated on first use).
int enqueue_host(skinny_gemm_t h, const void* x_host, int64_t M, void* out_host, cudaStream_t st) {
  if (check_handle(h) != SKG_OK) return SKG_EINVAL;
  if (x_host == nullptr || out_host == nullptr) return fail(SKG_EINVAL, "null host buffer");
  if (M < 1 || M > SKINNY_GEMM_MAX_M)
    return fail(SKG_EUNSUPPORTED_M, "M = %lld outside 1..%d", static_cast<long long>(M),
                SKINNY_GEMM_MAX_M);
  cudaError_t e;
  if (h->x_stage == nullptr) {
    e = cudaMalloc(&h->x_stage, static_cast<size_t>(SKINNY_GEMM_MAX_M) * h->K * 2);
    if (e != cudaSuccess) return h->x_stage = nullptr, cuda_fail(e, "cudaMalloc(x staging)");
  }
  if (h->out_stage == nullptr) {
    e = cudaMalloc(&h->out_stage, static_cast<size_t>(SKINNY_GEMM_MAX_M) * h->N * out_elem_bytes(h));
    if (e != cudaSuccess) return h->out_stage = nullptr, cuda_fail(e, "cudaMalloc(out staging)");
  }
  e = cudaMemcpyAsync(h->x_stage, x_host, static_cast<size_t>(M) * h->K * 2, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync(x)");
  int rc = launch_tactic(h, h->plan[M], h->x_stage, h->K, M, h->out_stage, h->N, st);
  if (rc != SKG_OK) return rc;
  e = cudaMemcpyAsync(out_host, h->out_stage, static_cast<size_t>(M) * h->N * out_elem_bytes(h),
                      cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync(out)");
  return SKG_OK;
}
}  // namespace

int skinny_gemm_run_host(skinny_gemm_t h, const void* x_host, int64_t M, void* out_host,
                         void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int rc = enqueue_host(h, x_host, M, out_host, st);
  if (rc != SKG_OK) return rc;
  const cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  return ok();
}

int skinny_gemm_run_host_async(skinny_gemm_t h, const void* x_host, int64_t M, void* out_host,
                               void* stream) {
  const int rc = enqueue_host(h, x_host, M, out_host, static_cast<cudaStream_t>(stream));
  return rc != SKG_OK ? rc : ok();
}

namespace {
// The two-stream step on plans already known to be valid (public entry point
// below; the overlap tuner passes private copies of the main plan).
int overlap_impl(skinny_gemm_t h_main, skinny_gemm_t h_fa, skinny_gemm_t h_fb, int chain,
                 const void* x, int64_t M, void* out_main, void* fa, void* out_fb,
                 void* main_stream, void* aux_stream, void* fork_event, void* join_event) {
  if (chain < 1) return fail(SKG_EINVAL, "chain must be >= 1");
  if (h_fa->K != h_main->K) return fail(SKG_EINVAL, "F_A and main weights need the same K");
  if (h_fa->out_dtype != SKG_BF16) return fail(SKG_EINVAL, "F_A output must be bf16 (it feeds F_B)");
  if (h_fb->K != h_fa->N) return fail(SKG_EINVAL, "F_B K must equal F_A N");
  if (chain > 1 && (h_fb->out_dtype != SKG_BF16 || h_fb->N < h_fb->K))
    return fail(SKG_EINVAL, "a chain needs bf16 F_B output with N_fb >= K_fb");
  if (fork_event == nullptr || join_event == nullptr || aux_stream == nullptr)
    return fail(SKG_EINVAL, "overlap needs an aux stream and two events");
  // Every launch's arguments are checked before the fork is recorded, so a
  // refused step enqueues nothing (a capture stays consistent).
  int rc = validate_args(h_main, x, h_main->K, M, out_main, h_main->N);
  if (rc != SKG_OK) return rc;
  rc = validate_args(h_fa, x, h_fa->K, M, fa, h_fa->N);
  if (rc != SKG_OK) return rc;
  rc = validate_args(h_fb, fa, h_fb->K, M, out_fb, h_fb->N);  // link 1 reads fa
  if (rc != SKG_OK) return rc;
  const size_t blk = static_cast<size_t>(M) * h_fb->N * out_elem_bytes(h_fb);
  char* fb = static_cast<char*>(out_fb);
  if (chain > 1) {
    // link i > 1 reads the first K_fb columns of link i-1's block (pitch N_fb)
    if (blk % 16 != 0) return fail(SKG_EALIGN, "out_fb blocks of a chain must be 16-byte multiples");
    rc = validate_args(h_fb, fb, h_fb->N, M, fb + blk, h_fb->N);
    if (rc != SKG_OK) return rc;
  }
  cudaStream_t ms = static_cast<cudaStream_t>(main_stream);
  cudaStream_t as = static_cast<cudaStream_t>(aux_stream);
  cudaEvent_t fork = static_cast<cudaEvent_t>(fork_event);
  cudaEvent_t join = static_cast<cudaEvent_t>(join_event);
  cudaError_t e = cudaEventRecord(fork, ms);
  if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord(fork)");
  e = cudaStreamWaitEvent(as, fork, 0);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent(aux, fork)");
  // Aux chain first so its small grids are queued before the big one fills the GPU.
  rc = launch_tactic(h_fa, h_fa->plan[M], x, h_fa->K, M, fa, h_fa->N, as);
  if (rc == SKG_OK) rc = launch_tactic(h_fb, h_fb->plan[M], fa, h_fb->K, M, fb, h_fb->N, as);
  for (int i = 1; i < chain && rc == SKG_OK; ++i)
    rc = launch_tactic(h_fb, h_fb->plan[M], fb + (i - 1) * blk, h_fb->N, M, fb + i * blk, h_fb->N, as);
  if (rc == SKG_OK) rc = launch_tactic(h_main, h_main->plan[M], x, h_main->K, M, out_main, h_main->N, ms);
  // The join is recorded even after a failed launch, so the aux stream is
  // always joined back into main (a capture would otherwise be left unjoined).
  const std::string why = g_err;
  const int code = rc;
  e = cudaEventRecord(join, as);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ms, join, 0);
  if (code != SKG_OK) return fail(code, "%s", why.c_str());
  if (e != cudaSuccess) return cuda_fail(e, "overlap join");
  return ok();
}
}  // namespace

int skinny_gemm_run_overlap(skinny_gemm_t h_main, skinny_gemm_t h_fa, skinny_gemm_t h_fb, int chain,
                            const void* x, int64_t M, void* out_main, void* fa, void* out_fb,
                            void* main_stream, void* aux_stream, void* fork_event,
                            void* join_event) {
  if (check_handle(h_main) != SKG_OK || check_handle(h_fa) != SKG_OK || check_handle(h_fb) != SKG_OK)
    return SKG_EINVAL;
  return overlap_impl(h_main, h_fa, h_fb, chain, x, M, out_main, fa, out_fb, main_stream,
                      aux_stream, fork_event, join_event);
}

int skinny_gemm_autotune_overlap(skinny_gemm_t h_main, skinny_gemm_t h_fa, skinny_gemm_t h_fb,
                                 int chain, const int64_t* Ms, int nM, void* stream) {
  if (check_handle(h_main) != SKG_OK || check_handle(h_fa) != SKG_OK || check_handle(h_fb) != SKG_OK)
    return SKG_EINVAL;
  if (chain < 1) return fail(SKG_EINVAL, "chain must be >= 1");
  if (h_fa->K != h_main->K || h_fb->K != h_fa->N || h_fa->out_dtype != SKG_BF16 ||
      h_main->dtype != h_fa->dtype)
    return fail(SKG_EINVAL, "handles do not form an overlap step (see skinny_gemm_run_overlap)");
  if (chain > 1 && (h_fb->out_dtype != SKG_BF16 || h_fb->N < h_fb->K))
    return fail(SKG_EINVAL, "a chain needs bf16 F_B output with N_fb >= K_fb");
  if (Ms == nullptr || nM < 1) return fail(SKG_EINVAL, "no token counts to tune");
  for (int i = 0; i < nM; ++i)
    if (Ms[i] < 1 || Ms[i] > SKINNY_GEMM_MAX_M)
      return fail(SKG_EUNSUPPORTED_M, "M = %lld outside 1..%d", static_cast<long long>(Ms[i]),
                  SKINNY_GEMM_MAX_M);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(st, &cs);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
  if (cs != cudaStreamCaptureStatusNone)
    return fail(SKG_ECAPTURING, "autotune must run before CUDA graph capture");
  e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");

  // The whole step is timed as a CUDA graph of back-to-back steps; the main
  // projection rotates over scratch copies of its weight layout (>= 4.5x L2).
  const size_t wbytes = static_cast<size_t>(h_main->N) * h_main->ldw * 2;
  const size_t l2 = static_cast<size_t>(std::max(h_main->dev->l2_bytes, 1 << 20));
  const int R = static_cast<int>(std::min<size_t>(64, std::max<size_t>(2, (9 * l2 / 2 + wbytes - 1) / wbytes)));
  const int L = R * std::max(1, (12 + R - 1) / R);
  void *rot = nullptr, *xb = nullptr, *om = nullptr, *fo = nullptr, *fbo = nullptr;
  cudaStream_t ts = nullptr, as = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr, e0 = nullptr, e1 = nullptr;
  auto cleanup = [&]() {
    if (ts) cudaStreamSynchronize(ts);
    if (as) cudaStreamSynchronize(as);
    for (void* p : {rot, xb, om, fo, fbo})
      if (p) cudaFree(p);
    for (cudaEvent_t ev : {fork, join, e0, e1})
      if (ev) cudaEventDestroy(ev);
    if (ts) cudaStreamDestroy(ts);
    if (as) cudaStreamDestroy(as);
  };
  int lo_pri = 0, hi_pri = 0;
  cudaDeviceGetStreamPriorityRange(&lo_pri, &hi_pri);
  const size_t mx = SKINNY_GEMM_MAX_M;
  if ((e = cudaMalloc(&rot, wbytes * R)) != cudaSuccess ||
      (e = cudaMalloc(&xb, mx * h_main->K * 2)) != cudaSuccess ||
      (e = cudaMalloc(&om, mx * h_main->N * out_elem_bytes(h_main))) != cudaSuccess ||
      (e = cudaMalloc(&fo, mx * h_fa->N * 2)) != cudaSuccess ||
      (e = cudaMalloc(&fbo, static_cast<size_t>(chain) * mx * h_fb->N * out_elem_bytes(h_fb))) != cudaSuccess ||
      (e = cudaMemset(rot, 0, wbytes * R)) != cudaSuccess ||
      (e = cudaMemset(xb, 0, mx * h_main->K * 2)) != cudaSuccess ||
      (e = cudaMemset(fo, 0, mx * h_fa->N * 2)) != cudaSuccess ||
      (e = cudaStreamCreateWithFlags(&ts, cudaStreamNonBlocking)) != cudaSuccess ||
      (e = cudaStreamCreateWithPriority(&as, cudaStreamNonBlocking, hi_pri)) != cudaSuccess ||
      (e = cudaEventCreateWithFlags(&fork, cudaEventDisableTiming)) != cudaSuccess ||
      (e = cudaEventCreateWithFlags(&join, cudaEventDisableTiming)) != cudaSuccess ||
      (e = cudaEventCreate(&e0)) != cudaSuccess || (e = cudaEventCreate(&e1)) != cudaSuccess) {
    cleanup();
    return cuda_fail(e, "autotune_overlap setup");
  }
  std::vector<skinny_gemm_plan> shadow(R, *h_main);
  for (int r = 0; r < R; ++r) {
    skinny_gemm_plan& sh = shadow[r];
    sh.W = static_cast<char*>(rot) + r * wbytes;
    sh.debug_count = 0;
    sh.x_stage = sh.out_stage = nullptr;
    if (encode_map(&sh.wmap64, sh.W, h_main->N, h_main->K, h_main->ldw, 64, h_main->dtype,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B) != SKG_OK ||
        encode_map(&sh.wmap128, sh.W, h_main->N, h_main->K, h_main->ldw, 128, h_main->dtype,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B) != SKG_OK) {
      const int code = g_last_status;
      cleanup();
      return code;
    }
  }
  // One step = the whole two-stream step, timed as a graph of L back-to-back
  // steps (the main projection rotating over the scratch copies).
  // mult x L steps per graph, `reps` timed replays, the fastest kept
  auto time_step = [&](int64_t M, double* us_out, int mult = 1, int reps = 3) -> int {
    const int LL = L * mult;
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    cudaError_t ce = cudaStreamBeginCapture(ts, cudaStreamCaptureModeThreadLocal);
    if (ce != cudaSuccess) return cuda_fail(ce, "cudaStreamBeginCapture(autotune_overlap)");
    int trc = SKG_OK;
    for (int l = 0; l < LL && trc == SKG_OK; ++l)
      trc = overlap_impl(&shadow[l % R], h_fa, h_fb, chain, xb, M, om, fo, fbo, ts, as, fork, join);
    ce = cudaStreamEndCapture(ts, &graph);
    if (trc != SKG_OK || ce != cudaSuccess) {
      if (graph) cudaGraphDestroy(graph);
      return trc != SKG_OK ? trc : cuda_fail(ce, "cudaStreamEndCapture(autotune_overlap)");
    }
    ce = cudaGraphInstantiate(&exec, graph, 0);
    if (ce != cudaSuccess) {
      cudaGraphDestroy(graph);
      return cuda_fail(ce, "cudaGraphInstantiate(autotune_overlap)");
    }
    float best_ms = 1e30f;
    ce = cudaGraphLaunch(exec, ts);
    for (int r = 0; r < reps && ce == cudaSuccess; ++r) {
      cudaEventRecord(e0, ts);
      ce = cudaGraphLaunch(exec, ts);
      cudaEventRecord(e1, ts);
      if (ce == cudaSuccess) ce = cudaEventSynchronize(e1);
      float ms = 0;
      if (ce == cudaSuccess && cudaEventElapsedTime(&ms, e0, e1) == cudaSuccess)
        best_ms = std::min(best_ms, ms);
    }
    cudaGraphExecDestroy(exec);
    cudaGraphDestroy(graph);
    if (ce != cudaSuccess) return cuda_fail(ce, "autotune_overlap timing");
    *us_out = 1000.0 * best_ms / LL;
    return SKG_OK;
  };
  // The main projection's tactic for M, on the handle and on every shadow.
  auto set_main = [&](int64_t M, const Tactic& t) -> int {
    const int wrc = ensure_workspace(h_main, t);
    if (wrc != SKG_OK) return wrc;
    h_main->plan[M] = t;
    for (skinny_gemm_plan& sh : shadow) {
      sh.plan[M] = t;
      sh.workspace = h_main->workspace;
      sh.workspace_bytes = h_main->workspace_bytes;
      sh.counters = h_main->counters;
      sh.counters_bytes = h_main->counters_bytes;
    }
    return SKG_OK;
  };
  int rc = SKG_OK;
  std::vector<int64_t> tuned;
  for (int i = 0; i < nM && rc == SKG_OK; ++i) {
    const int64_t M = Ms[i];
    double step_us = 0;
    // Passes: F_A's tactic (main fixed), the main projection's (F_A fixed), F_A's again.
    for (int pass = 0; pass < 3 && rc == SKG_OK; ++pass) {
      const bool fa_pass = pass != 1;
      skinny_gemm_t hp = fa_pass ? h_fa : h_main;
      const Tactic keep = hp->plan[M];
      auto install = [&](const Tactic& t) -> int {
        if (!fa_pass) return set_main(M, t);
        const int wrc = ensure_workspace(h_fa, t);
        if (wrc == SKG_OK) h_fa->plan[M] = t;
        return wrc;
      };
      std::vector<std::pair<double, Tactic>> timed;
      for (const Tactic& t : candidates(hp, M)) {
        rc = install(t);
        if (rc != SKG_OK) break;
        double us = 0;
        rc = time_step(M, &us);
        if (rc != SKG_OK) break;
        if (log_enabled())
          fprintf(stderr, "[skinny_gemm] tune overlap M=%lld %s %s: step %.3f us\n",
                  static_cast<long long>(M), fa_pass ? "F_A" : "main", tactic_str(t).c_str(), us);
        timed.push_back({us, t});
      }
      // The four fastest again, twice as long and five times: a single short
      // timing of many candidates favours whichever was timed luckily.
      double best_us = 1e30;
      Tactic best;
      std::stable_sort(timed.begin(), timed.end(),
                       [](const auto& a, const auto& b) { return a.first < b.first; });
      for (size_t c = 0; c < timed.size() && c < 4 && rc == SKG_OK; ++c) {
        rc = install(timed[c].second);
        double us = 0;
        if (rc == SKG_OK) rc = time_step(M, &us, 2, 5);
        if (rc == SKG_OK && us < best_us) {
          best_us = us;
          best = timed[c].second;
        }
      }
      const Tactic pick = (rc == SKG_OK && best.valid()) ? best : keep;
      if (fa_pass) {
        h_fa->plan[M] = pick;
      } else {
        const int src = set_main(M, pick);
        if (rc == SKG_OK) rc = src;
      }
      step_us = best_us;
    }
    // Last pass: the main projection's pick with later PDL triggers and with
    // weight stages prefetched into L2, timed inside the step.
    if (rc == SKG_OK && h_main->plan[M].variant != kVariantSk) {
      const Tactic base = h_main->plan[M];
      std::vector<std::pair<double, Tactic>> timed{{step_us, base}};
      const int span = late_trigger_span(h_main, base);
      for (int lt = 0; lt <= 4 && rc == SKG_OK; ++lt)
        for (int pf : {0, 1, 2}) {
          Tactic t = base;
          t.lt = lt;
          t.pf = t.dy ? 0 : pf;
          if ((t.lt == base.lt && t.pf == base.pf) || lt > span || t.pf > span ||
              !tactic_fits(h_main, t, M, nullptr))
            continue;
          rc = set_main(M, t);
          double us = 0;
          if (rc == SKG_OK) rc = time_step(M, &us);
          if (rc != SKG_OK) break;
          timed.push_back({us, t});
        }
      // the three fastest (the base among them if it still is) timed longer, as above
      std::stable_sort(timed.begin(), timed.end(),
                       [](const auto& a, const auto& b) { return a.first < b.first; });
      double best_us = 1e30;
      Tactic best = base;
      for (size_t c = 0; c < timed.size() && c < 3 && rc == SKG_OK; ++c) {
        rc = set_main(M, timed[c].second);
        double us = 0;
        if (rc == SKG_OK) rc = time_step(M, &us, 2, 5);
        if (rc == SKG_OK && us < best_us) {
          best_us = us;
          best = timed[c].second;
        }
      }
      const int src = set_main(M, best);
      if (rc == SKG_OK) rc = src;
      step_us = best_us;
    }
    if (rc == SKG_OK) tuned.push_back(M);
    if (log_enabled() && rc == SKG_OK)
      fprintf(stderr, "[skinny_gemm] overlap M=%lld: main %s, F_A %s, step %.3f us\n",
              static_cast<long long>(M), tactic_str(h_main->plan[M]).c_str(),
              tactic_str(h_fa->plan[M]).c_str(), step_us);
  }
  cleanup();
  if (rc != SKG_OK) return rc;
  std::sort(tuned.begin(), tuned.end());
  for (int m = 1; m <= SKINNY_GEMM_MAX_M; ++m) {
    if (std::binary_search(tuned.begin(), tuned.end(), static_cast<int64_t>(m))) continue;
    for (int64_t mp : tuned)
      if (mp >= m) {
        if (tactic_fits(h_fa, h_fa->plan[mp], m, nullptr)) h_fa->plan[m] = h_fa->plan[mp];
        if (tactic_fits(h_main, h_main->plan[mp], m, nullptr)) h_main->plan[m] = h_main->plan[mp];
        break;
      }
  }
  return ok();
}

int skinny_gemm_tactic_normalize(const char* tactic, char* buf, size_t len) {
  if (buf == nullptr || len == 0) return fail(SKG_EINVAL, "null buffer");
  Tactic t;
  if (!tactic_parse(tactic, &t)) return fail(SKG_EINVAL, "cannot parse tactic '%s'", tactic ? tactic : "");
  snprintf(buf, len, "%s", tactic_str(t).c_str());
  return ok();
}

int skinny_gemm_set_tactic(skinny_gemm_t h, int64_t M, const char* tactic) {
  if (check_handle(h) != SKG_OK) return SKG_EINVAL;
  if (M < 1 || M > SKINNY_GEMM_MAX_M)
    return fail(SKG_EUNSUPPORTED_M, "M = %lld outside 1..%d", static_cast<long long>(M),
                SKINNY_GEMM_MAX_M);
  Tactic t;
  if (!tactic_parse(tactic, &t)) return fail(SKG_EINVAL, "cannot parse tactic '%s'", tactic ? tactic : "");
  std::string why;
  if (!tactic_fits(h, t, M, &why))
    return fail(SKG_EINVAL, "tactic %s does not fit: %s", tactic, why.c_str());
  if (active_clusters(h, t) <= 0)
    return fail(SKG_EINVAL, "tactic %s cannot be resident on this GPU", tactic);
  if (ensure_workspace(h, t) != SKG_OK) return g_last_status;
  h->plan[M] = t;
  return ok();
}

int skinny_gemm_plan_query(skinny_gemm_t h, int64_t M, char* buf, size_t len) {
  if (check_handle(h) != SKG_OK) return SKG_EINVAL;
  if (M < 1 || M > SKINNY_GEMM_MAX_M)
    return fail(SKG_EUNSUPPORTED_M, "M = %lld outside 1..%d", static_cast<long long>(M),
                SKINNY_GEMM_MAX_M);
  if (buf == nullptr || len == 0) return fail(SKG_EINVAL, "null buffer");
  snprintf(buf, len, "%s", tactic_str(h->plan[M]).c_str());
  return ok();
}

int skinny_gemm_list_tactics(skinny_gemm_t h, int64_t M, char* buf, size_t len) {
  if (check_handle(h) != SKG_OK) return -SKG_EINVAL;
  if (M < 1 || M > SKINNY_GEMM_MAX_M) return -fail(SKG_EUNSUPPORTED_M, "M out of range");
  std::vector<Tactic> c = candidates(h, M);
  std::string s;
  for (size_t i = 0; i < c.size(); ++i) {
    if (i) s += ';';
    s += tactic_str(c[i]);
  }
  if (buf != nullptr && len > 0) snprintf(buf, len, "%s", s.c_str());
  ok();
  return static_cast<int>(c.size());
}

int skinny_gemm_autotune(skinny_gemm_t h, const int64_t* Ms, int nM, void* stream) {
  if (check_handle(h) != SKG_OK) return SKG_EINVAL;
  if (Ms == nullptr || nM < 1) return fail(SKG_EINVAL, "no token counts to tune");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(st, &cs);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
  if (cs != cudaStreamCaptureStatusNone)
    return fail(SKG_ECAPTURING, "autotune must run before CUDA graph capture");
  for (int i = 0; i < nM; ++i)
    if (Ms[i] < 1 || Ms[i] > SKINNY_GEMM_MAX_M)
      return fail(SKG_EUNSUPPORTED_M, "M = %lld outside 1..%d", static_cast<long long>(Ms[i]),
                  SKINNY_GEMM_MAX_M);
  e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");

  // Steady-state timing, the way decode steps run: each candidate is captured
  // as a CUDA graph of back-to-back launches (programmatic dependent launch
  // between them) that rotate over R scratch copies of the weight's layout,
  // R * weight bytes >= 4.5x L2, so every launch streams its weight from HBM.
  // The copies' contents do not matter for timing; they are zero-filled.
  const size_t wbytes = static_cast<size_t>(h->N) * h->ldw * 2;
  const size_t l2 = static_cast<size_t>(std::max(h->dev->l2_bytes, 1 << 20));
  // >= 4.5x L2: a cyclic read of only ~2x L2 was measured still partly L2-fed.
  const int R = static_cast<int>(std::min<size_t>(64, std::max<size_t>(2, (9 * l2 / 2 + wbytes - 1) / wbytes)));
  const int L = R * std::max(1, (24 + R - 1) / R);  // launches per timed graph
  const int reps = std::max(1, static_cast<int>(env_u64("SKINNY_GEMM_TUNE_REPS", 3)));
  void *rot = nullptr, *xbuf = nullptr, *obuf = nullptr;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  cudaStream_t ts = nullptr;
  auto cleanup = [&]() {
    if (ts) cudaStreamSynchronize(ts);
    if (rot) cudaFree(rot);
    if (xbuf) cudaFree(xbuf);
    if (obuf) cudaFree(obuf);
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    if (ts) cudaStreamDestroy(ts);
  };
  const size_t xbytes = static_cast<size_t>(SKINNY_GEMM_MAX_M) * h->K * 2;
  const size_t obytes = static_cast<size_t>(SKINNY_GEMM_MAX_M) * h->N * 4;
  if ((e = cudaMalloc(&rot, wbytes * R)) != cudaSuccess ||
      (e = cudaMalloc(&xbuf, xbytes)) != cudaSuccess ||
      (e = cudaMalloc(&obuf, obytes)) != cudaSuccess ||
      (e = cudaMemset(rot, 0, wbytes * R)) != cudaSuccess ||
      (e = cudaMemset(xbuf, 0, xbytes)) != cudaSuccess ||
      (e = cudaStreamCreateWithFlags(&ts, cudaStreamNonBlocking)) != cudaSuccess ||
      (e = cudaEventCreate(&e0)) != cudaSuccess || (e = cudaEventCreate(&e1)) != cudaSuccess) {
    cleanup();
    return cuda_fail(e, "autotune setup");
  }
  std::vector<skinny_gemm_plan> shadow(R, *h);
  for (int r = 0; r < R; ++r) {
    skinny_gemm_plan& sh = shadow[r];
    sh.W = static_cast<char*>(rot) + r * wbytes;
    sh.debug_count = 0;
    sh.x_stage = sh.out_stage = nullptr;
    if (encode_map(&sh.wmap64, sh.W, h->N, h->K, h->ldw, 64, h->dtype,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B) != SKG_OK ||
        encode_map(&sh.wmap128, sh.W, h->N, h->K, h->ldw, 128, h->dtype,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B) != SKG_OK) {
      const int code = g_last_status;
      cleanup();
      return code;
    }
  }
  int rc = SKG_OK;
  std::vector<int64_t> tuned;
  // Token counts with identical candidate lists (the same token tiles) are tuned
  // together: phases 1-2 at the largest of them, phase 3 summed over all of them,
  // one tactic installed for the group (the same kernel for, e.g., M = 1..8).
  std::vector<std::string> group_keys;
  std::vector<std::vector<int64_t>> groups;
  for (int i = 0; i < nM; ++i) {
    std::string key;
    for (const Tactic& t : candidates(h, Ms[i])) key += tactic_str(t) + ";";
    size_t g = 0;
    while (g < group_keys.size() && group_keys[g] != key) ++g;
    if (g == group_keys.size()) {
      group_keys.push_back(key);
      groups.emplace_back();
    }
    if (std::find(groups[g].begin(), groups[g].end(), Ms[i]) == groups[g].end())
      groups[g].push_back(Ms[i]);
  }
  for (size_t gi = 0; gi < groups.size() && rc == SKG_OK; ++gi) {
    const std::vector<int64_t>& grp = groups[gi];
    const int64_t Mmax = *std::max_element(grp.begin(), grp.end());
    int64_t M = Mmax;  // token count the next timing runs at
    // Time one tactic as a graph of L back-to-back launches over the rotated copies.
    auto time_tactic = [&](const Tactic& t, double* us_out, int nrep = 0, int mult = 1) -> int {
      const int LL = L * mult;
      const int RR = nrep > 0 ? nrep : reps;
      int trc = ensure_workspace(h, t);
      if (trc != SKG_OK) return trc;
      for (skinny_gemm_plan& sh : shadow) {
        sh.workspace = h->workspace;
        sh.workspace_bytes = h->workspace_bytes;
        sh.counters = h->counters;
        sh.counters_bytes = h->counters_bytes;
      }
      cudaGraph_t graph = nullptr;
      cudaGraphExec_t exec = nullptr;
      cudaError_t ce = cudaStreamBeginCapture(ts, cudaStreamCaptureModeThreadLocal);
      if (ce != cudaSuccess) return cuda_fail(ce, "cudaStreamBeginCapture(autotune)");
      for (int l = 0; l < LL && trc == SKG_OK; ++l)
        trc = launch_tactic(&shadow[l % R], t, xbuf, h->K, M, obuf, h->N, ts);
      ce = cudaStreamEndCapture(ts, &graph);
      if (trc != SKG_OK || ce != cudaSuccess) {
        if (graph) cudaGraphDestroy(graph);
        return trc != SKG_OK ? trc : cuda_fail(ce, "cudaStreamEndCapture(autotune)");
      }
      ce = cudaGraphInstantiate(&exec, graph, 0);
      if (ce != cudaSuccess) {
        cudaGraphDestroy(graph);
        return cuda_fail(ce, "cudaGraphInstantiate(autotune)");
      }
      float best_ms = 1e30f;
      ce = cudaGraphLaunch(exec, ts);  // warm-up
      for (int r = 0; r < RR && ce == cudaSuccess; ++r) {
        cudaEventRecord(e0, ts);
        ce = cudaGraphLaunch(exec, ts);
        cudaEventRecord(e1, ts);
        if (ce == cudaSuccess) ce = cudaEventSynchronize(e1);
        float ms = 0;
        if (ce == cudaSuccess) {
          cudaEventElapsedTime(&ms, e0, e1);
          best_ms = std::min(best_ms, ms);
        }
      }
      cudaGraphExecDestroy(exec);
      cudaGraphDestroy(graph);
      if (ce != cudaSuccess) return cuda_fail(ce, "autotune timing");
      *us_out = 1000.0 * best_ms / LL;
      if (log_enabled())
        fprintf(stderr, "[skinny_gemm] tune N=%lld K=%lld M=%lld %s %.3f us\n",
                static_cast<long long>(h->N), static_cast<long long>(h->K),
                static_cast<long long>(M), tactic_str(t).c_str(), *us_out);
      return SKG_OK;
    };
    // Phase 1: every candidate with the PDL trigger right after the first stages.
    std::vector<std::pair<double, Tactic>> timed;
    for (const Tactic& t : candidates(h, M)) {
      double us = 0;
      rc = time_tactic(t, &us);
      if (rc != SKG_OK) break;
      timed.push_back({us, t});
    }
    // Phase 2: the six fastest of phase 1, each with every later PDL trigger
    // (:d1-:d4) and L2 prefetch depth (:p1, :p2, :p4) and their combinations,
    // tcgen05 cluster tactics at >= 64 tokens also with per-thread reduction
    // stores (:s) (a tactic that is not the fastest alone can gain the most);
    // unless the handle is deterministic, the six fastest cluster tactics also
    // with run-time K sharing (:w), and the best two of those with later triggers.
    if (rc == SKG_OK) {
      std::stable_sort(timed.begin(), timed.end(),
                       [](const auto& a, const auto& b) { return a.first < b.first; });
      const std::vector<std::pair<double, Tactic>> base_timed = timed;
      auto later_triggers = [&](const Tactic& t0) {
        for (int lt = 1; lt <= 4 && rc == SKG_OK; ++lt) {
          Tactic t = t0;
          if (t.variant == kVariantSk || late_trigger_span(h, t) < lt) break;
          t.lt = lt;
          double us = 0;
          rc = time_tactic(t, &us);
          if (rc == SKG_OK) timed.push_back({us, t});
        }
      };
      for (size_t c = 0; c < std::min<size_t>(base_timed.size(), 6) && rc == SKG_OK; ++c) {
        const Tactic t0 = base_timed[c].second;
        if (t0.variant == kVariantSk) continue;
        const int span = late_trigger_span(h, t0);
        for (int rs = 0; rs <= 1 && rc == SKG_OK; ++rs)
          for (int lt = 0; lt <= 4 && lt <= span && rc == SKG_OK; ++lt)
            for (int pf : {0, 1, 2, 4}) {
              Tactic t = t0;
              t.rs = rs;
              t.lt = lt;
              t.pf = pf;
              if ((rs == 0 && lt == 0 && pf == 0) || pf > span) continue;
              if (rs == 1 && !tactic_fits(h, t, M, nullptr)) break;
              double us = 0;
              rc = time_tactic(t, &us);
              if (rc != SKG_OK) break;
              timed.push_back({us, t});
            }
      }
      if (!h->deterministic) {
        std::vector<std::pair<double, Tactic>> shared;
        for (size_t c = 0; c < base_timed.size() && shared.size() < 6 && rc == SKG_OK; ++c) {
          Tactic t = base_timed[c].second;
          t.dy = 1;
          if (!tactic_fits(h, t, M, nullptr) || active_clusters(h, t) <= 0) continue;
          double us = 0;
          rc = time_tactic(t, &us);
          if (rc == SKG_OK) shared.push_back({us, t});
        }
        std::stable_sort(shared.begin(), shared.end(),
                         [](const auto& a, const auto& b) { return a.first < b.first; });
        for (size_t c = 0; c < shared.size(); ++c) {
          timed.push_back(shared[c]);
          if (c < 2 && rc == SKG_OK) later_triggers(shared[c].second);
        }
      }
    }
    // Phase 3: the six fastest so far timed again, longer (twice the launches,
    // five repetitions) and at every token count of the group (times summed), so
    // that near-ties are not decided by timing noise.
    if (rc == SKG_OK && (timed.size() > 1 || grp.size() > 1)) {
      std::stable_sort(timed.begin(), timed.end(),
                       [](const auto& a, const auto& b) { return a.first < b.first; });
      std::vector<std::pair<double, Tactic>> fin;
      for (size_t c = 0; c < timed.size() && c < 6 && rc == SKG_OK; ++c) {
        double sum = 0;
        for (size_t k = 0; k < grp.size() && rc == SKG_OK; ++k) {
          if (!tactic_fits(h, timed[c].second, grp[k], nullptr)) {
            sum = 1e30;
            break;
          }
          M = grp[k];
          double us = 0;
          rc = time_tactic(timed[c].second, &us, 5, 2);
          sum += us;
        }
        M = Mmax;
        if (rc == SKG_OK) fin.push_back({sum / static_cast<double>(grp.size()), timed[c].second});
      }
      if (rc == SKG_OK) timed = fin;
    }
    double best_us = 1e30;
    Tactic best;
    for (const auto& ut : timed)
      if (ut.first < best_us) {
        best_us = ut.first;
        best = ut.second;
      }
    if (rc == SKG_OK && best.valid() && best_us < 1e29) {
      for (int64_t m : grp) {
        h->plan[m] = best;
        tuned.push_back(m);
        append_tactic_file(h, m, best, best_us);
      }
    }
  }
  cleanup();
  if (rc != SKG_OK) return rc;
  // Untuned M take the tuned tactic of the smallest tuned M' >= M.
  std::sort(tuned.begin(), tuned.end());
  for (int m = 1; m <= SKINNY_GEMM_MAX_M; ++m) {
    if (std::binary_search(tuned.begin(), tuned.end(), static_cast<int64_t>(m))) continue;
    for (int64_t mp : tuned)
      if (mp >= m) {
        if (tactic_fits(h, h->plan[mp], m, nullptr)) h->plan[m] = h->plan[mp];
        break;
      }
  }
  return ok();
}

int skinny_gemm_check_status(skinny_gemm_t h, void* stream) {
  if (check_handle(h) != SKG_OK) return SKG_EINVAL;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  uint32_t v = 0;
  e = cudaMemcpy(&v, h->status, sizeof v, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(status)");
  if (v != 0) {
    cudaMemset(h->status, 0, sizeof v);
    // a kernel that gave up may have left split-tile counters mid-count
    if (h->counters) cudaMemset(h->counters, 0, h->counters_bytes);
    if ((v & 0xffff0000u) == kStatusCheck)
      return fail(SKG_ECHECK, "device check failed: access %u out of bounds (code 0x%08x)",
                  v & 0xffffu, v);
    return fail(SKG_ETIMEOUT, "device watchdog: bounded wait expired (code 0x%08x)", v);
  }
  return ok();
}

int skinny_gemm_debug_inject_timeout(skinny_gemm_t h, int count, uint64_t timeout_ns) {
  if (check_handle(h) != SKG_OK) return SKG_EINVAL;
  if (count < 0) return fail(SKG_EINVAL, "negative count");
  h->debug_count = count;
  h->debug_kind = 1;
  h->debug_timeout_ns = timeout_ns;
  return ok();
}

int skinny_gemm_debug_inject_check(skinny_gemm_t h, int count) {
  if (check_handle(h) != SKG_OK) return SKG_EINVAL;
  if (count < 0) return fail(SKG_EINVAL, "negative count");
  if (SKG_DEVICE_CHECKS == 0)
    return fail(SKG_EINVAL, "not a checked build (libskinny_gemm_checked.so has the device checks)");
  h->debug_count = count;
  h->debug_kind = 2;
  return ok();
}

void skinny_gemm_destroy(skinny_gemm_t h) {
  if (h == nullptr || !unregister_handle(h)) return;  // null, unknown or already destroyed
  if (h->status) cudaFree(h->status);
  if (h->workspace) cudaFree(h->workspace);
  if (h->counters) cudaFree(h->counters);
  if (h->x_stage) cudaFree(h->x_stage);
  if (h->out_stage) cudaFree(h->out_stage);
  delete h;
}

}  // extern "C"

// ------------------------------------------------------------------ no-allocation entry point
// skinny_gemm_run_noalloc is for callers that cannot allocate device memory
// (see its declaration in skinny_gemm.h).  The only scratch the kernels need
// is the watchdog status word; here it lives in this file-scope array instead
// of a cudaMalloc'd word owned by a handle.  Every GPU that loads the library
// holds these 256 bytes until the process exits.
namespace {
constexpr size_t kNoAllocScratchBytes = 256;
}  // namespace

static __device__ __align__(256) uint32_t g_noalloc_scratch[kNoAllocScratchBytes / sizeof(uint32_t)];

namespace {

std::mutex g_noalloc_mu;
uint32_t* g_noalloc_addr[64] = {};

// Device address of the scratch array on device `dev` (which must be current).
// Host code cannot pass `g_noalloc_scratch` itself to a kernel: on the host
// that name is a stand-in, not a device address.  Looked up once per device;
// the array is zeroed then, with a synchronous memset (set-up happens outside
// any capture), so no later call has to clear it.
int noalloc_scratch_address(int dev, uint32_t** out) {
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_addr[dev] == nullptr) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(no-alloc scratch)");
    e = cudaMemset(p, 0, kNoAllocScratchBytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(no-alloc scratch)");
    g_noalloc_addr[dev] = static_cast<uint32_t*>(p);
  }
  *out = g_noalloc_addr[dev];
  return SKG_OK;
}

}  // namespace

extern "C" int skinny_gemm_run_noalloc(const void* W, int64_t N, int64_t K, int64_t ldw,
                                       int out_dtype, const void* x, int64_t ldx, int64_t M,
                                       void* out, int64_t ldo, void* stream) {
  if (W == nullptr) return fail(SKG_EINVAL, "null weight pointer");
  if (out_dtype != SKG_BF16 && out_dtype != SKG_FP32)
    return fail(SKG_EINVAL, "unsupported projection output dtype %d (BF16 or FP32)", out_dtype);
  if (N < 1 || K < 8 || N > (1ll << 31) - 1 || K > (1ll << 31) - 1)
    return fail(SKG_EINVAL, "weight shape [%lld, %lld] out of range", static_cast<long long>(N),
                static_cast<long long>(K));
  if (K % 8 != 0 || ldw < K || ldw % 8 != 0 || reinterpret_cast<uintptr_t>(W) % 16 != 0)
    return fail(SKG_EALIGN, "weight rows need a 16-byte aligned base and pitch (K %% 8 == 0)");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  DeviceInfo* di = nullptr;
  if (device_info(dev, &di) != SKG_OK) return g_last_status;
  uint32_t* scratch = nullptr;
  if (noalloc_scratch_address(dev, &scratch) != SKG_OK) return g_last_status;

  // A plan on the stack (host memory, gone at return): no handle, no allocation.
  skinny_gemm_plan p;
  p.W = W;
  p.N = N;
  p.K = K;
  p.ldw = ldw;
  p.dtype = SKG_BF16;
  p.out_dtype = out_dtype;
  p.device = dev;
  p.dev = di;
  p.kboxes = static_cast<int>((K + kBoxK - 1) / kBoxK);
  p.status = scratch;
  p.timeout_ns = env_u64("SKINNY_GEMM_TIMEOUT_NS", 2000000000ull);
  int rc = validate_args(&p, x, ldx, M, out, ldo);  // p is a private plan, not a handle
  if (rc != SKG_OK) return rc;
  const Tactic t = default_tactic(&p, M);
  if (!t.valid()) return fail(SKG_EINVAL, "no valid tactic for M = %lld", static_cast<long long>(M));
  const size_t need = sizeof(uint32_t);  // the launched kernels' scratch: one status word
  if (need > kNoAllocScratchBytes)
    return fail(SKG_EINVAL, "needs %zu bytes of scratch, more than the %zu-byte static buffer", need,
                kNoAllocScratchBytes);
  rc = encode_map(t.rows == 64 ? &p.wmap64 : &p.wmap128, W, N, K, ldw, t.rows, SKG_BF16,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  if (rc != SKG_OK) return rc;
  // The array keeps the previous call's contents.  The status word is the
  // only part a kernel touches, it only ever goes from zero to a code (first
  // expiry wins) and nothing reads it back, so no call needs it cleared; with
  // no clearing node between them, consecutive calls on a stream still overlap
  // under programmatic dependent launch.
  rc = launch_tactic(&p, t, x, ldx, M, out, ldo, static_cast<cudaStream_t>(stream));
  return rc == SKG_OK ? ok() : rc;
}
