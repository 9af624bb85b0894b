// Launch parameters and the kernel registry shared by the host library and
// the kernel translation units.
#pragma once

#include <cstdint>

namespace skg {

constexpr int kBoxK = 64;            // bf16 elements per TMA box row (128 bytes)
constexpr int kBoxRowBytes = 128;
constexpr int kSmemAlign = 1024;     // 128-byte swizzle atoms are 8 rows x 128 B

// Status codes written into the device status word (first error wins).
enum : uint32_t {
  kStatusTimeoutFull = 0x10000001u,   // waiting for a stage's TMA data
  kStatusTimeoutEmpty = 0x10000002u,  // producer waiting for a stage to drain
  kStatusTimeoutDone = 0x10000003u,   // waiting for the MMAs to finish
  kStatusTimeoutRecv = 0x10000004u,   // waiting for cluster peers' partial sums
  kStatusTimeoutDebug = 0x10000005u,  // injected watchdog self-test
  kStatusTimeoutDrain = 0x10000006u,  // final drain of in-flight copies
  // checked build (SKG_DEVICE_CHECKS): an access failed its bounds test and was
  // skipped; the low 16 bits name the access (kCheck* below)
  kStatusCheck = 0x20000000u,
};

// Accesses tested in a checked build.
enum : uint32_t {
  kCheckTmaW = 1,       // weight box destination inside the pipeline stages
  kCheckTmaX = 2,       // x box destination inside the pipeline stages
  kCheckMmaOperand = 3, // MMA / ldmatrix operand inside its stage box
  kCheckTmem = 4,       // TMEM column range inside the allocation
  kCheckRedLocal = 5,   // write into this CTA's receive / staging buffer
  kCheckRedRemote = 6,  // push into a peer's receive buffer
  kCheckRedRead = 7,    // reduction read of the receive buffer
  kCheckOut = 8,        // output element inside [M, N]
  kCheckWorkspace = 9,  // stream-K partial-sum slot / tile counter
  kCheckBulk = 10,      // bulk DSMEM copy source / destination range
  kCheckSelfTest = 11,  // injected by skinny_gemm_debug_inject_check (no access is made)
};

struct KParams {
  void* out;              // [M, ldo] row-major, output element type of the kernel
  int64_t ldo;            // output row pitch (elements)
  int32_t M;              // valid tokens, 1..TOK
  int32_t N;              // valid weight rows
  int32_t kboxes;         // ceil(K / 64): 64-wide K blocks of the weight
  int32_t stages;         // pipeline depth (shared-memory stages)
  uint32_t* status;       // device status word (watchdog)
  uint64_t timeout_ns;    // bound of every spin wait
  int32_t debug_wait;     // 1: watchdog self-test, wait on a dead barrier and return;
                          // 2 (checked build): record a failed kCheckSelfTest and return
  int32_t pdl_late;       // 0: launch dependents right after the first stages' weight loads;
                          // k >= 1: only once all but the last k-1 stages' loads are issued
  int32_t red_alias;      // tcgen05 clusters: the reduction buffer reuses the pipeline stages
  int32_t dyn_k;          // clusters: K boxes after the first stages are shared out at run time
                          // through a counter in the cluster's rank-0 CTA (see kDynBytes)
  int32_t l2_pre;         // stages after the first ones whose weight boxes are prefetched
                          // into L2 before the PDL wait (0: none)
  int32_t red_stores;     // tcgen05 clusters, >= 64 tokens: per-thread st.async pushes
                          // instead of bulk DSMEM copies
  // stream-K kernel only: fp32 partial sums of split tiles and per-tile arrival counters
  float* workspace;       // [gridDim.x][2][TOK][128]
  uint32_t* counters;     // [ceil(N / 128)], zero between launches
  // optional residual added before the output rounding: [M, ldr], output type
  const void* residual;   // nullptr: none
  int64_t ldr;
};

// Run-time K sharing (dyn_k): a 16-byte slot holding the cluster's work counter
// (used in rank 0) and one 32-bit box count per pipeline stage (at most 16),
// placed after the barriers; added to the footprints below when dyn_k is set.
constexpr uint32_t kDynBytes = 16 + 16 * 4;

// Shared-memory footprint of one configuration (bytes, including 1 KB of
// alignment slack).  Same formula on host and device.
__host__ __device__ constexpr uint32_t stage_bytes(int rows, int tok, int nbox) {
  return static_cast<uint32_t>(nbox * (rows + tok) * kBoxRowBytes);
}
__host__ __device__ constexpr uint32_t red_bytes(int rows, int tok) {
  return static_cast<uint32_t>(rows * tok * 4);
}
__host__ __device__ constexpr uint32_t smem_bytes(int rows, int tok, int nbox, int stages) {
  return kSmemAlign + stages * stage_bytes(rows, tok, nbox) + red_bytes(rows, tok) +
         static_cast<uint32_t>((2 * stages + 4) * 8) + 16;
}

enum Variant : int { kVariantMma = 1, kVariantTc = 2, kVariantSk = 3 };

struct KernelEntry {
  int variant;    // kVariantMma (mma.sync) or kVariantTc (tcgen05 / TMEM)
  int rows;       // weight rows per CTA tile
  int tok;        // token tile (MMA N)
  int nbox;       // 64-wide K boxes per pipeline stage
  int in_dtype;   // 0 bf16, 1 fp16 (skinny_gemm_dtype)
  int out_dtype;  // 0 bf16, 2 fp32
  int threads;    // CTA size
  const void* func;
};

// Defined in kernels_mma.cu, kernels_tc.cu and kernels_sk.cu.
const KernelEntry* mma_kernel_table(int* count);
const KernelEntry* tc_kernel_table(int* count);
const KernelEntry* sk_kernel_table(int* count);

// tcgen05 cluster kernel: the receive buffer is [cluster][rows/cluster][TOK + 4]
// fp32 (token-contiguous rows, padded so 16-byte reads of consecutive rows
// fall in different banks).
__host__ __device__ constexpr uint32_t tc_red_bytes(int tok, int rows = 128) {
  return static_cast<uint32_t>(rows * (tok + 4) * 4);
}
// (The receive buffer exists only for clusters of more than one CTA, and takes
// no space of its own when it aliases the pipeline stages.)
__host__ __device__ constexpr uint32_t tc_smem_bytes(int tok, int nbox, int stages, int cluster,
                                                     bool alias = false, int rows = 128) {
  return kSmemAlign + stages * stage_bytes(rows, tok, nbox) +
         (cluster > 1 && !alias ? tc_red_bytes(tok, rows) : 0u) +
         static_cast<uint32_t>((2 * stages + 4) * 8) + 16;
}

// Stream-K shared memory: stages plus barriers (no cluster receive buffer).
__host__ __device__ constexpr uint32_t sk_smem_bytes(int tok, int nbox, int stages) {
  return kSmemAlign + stages * stage_bytes(128, tok, nbox) +
         static_cast<uint32_t>((2 * stages + 6) * 8) + 16;
}

}  // namespace skg
