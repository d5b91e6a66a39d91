// Device-side helpers shared by the chord_moe kernels (sm_103a).
//
// Inline PTX for mbarriers, bulk async copies (TMA 1D), ldmatrix and the
// register-operand BF16 MMA, plus bounded waits: every spin on an mbarrier
// gives up after a fixed number of polls, records CHORD_ERR_TIMEOUT in the
// caller's status word and lets the kernel return.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "chord_moe.h"

namespace chord {

constexpr int kGroup = 32;            // INT4 scale group along K
constexpr int kTileRows = 64;         // weight rows per packed tile (4 slabs of 16)
constexpr int kSlabs = kTileRows / 16;
constexpr int kUnitK = 64;            // K per packed unit
constexpr int kUnitQBytes = kTileRows * kUnitK / 2;          // 2048
constexpr int kUnitSBytes = kTileRows * (kUnitK / kGroup) * 2; // 256
constexpr int kUnitBytes = kUnitQBytes + kUnitSBytes;        // 2304
constexpr uint32_t kPackMagic = 0x57344843u;   // "CH4W"
constexpr uint32_t kPackVersion = 2u;
constexpr int kPackHeaderBytes = 256;
constexpr uint32_t kPackFlagGateUp = 1u;

// Packed-weight header (first 256 bytes of a prepacked blob).
struct PackHeader {
  uint32_t magic, version;
  int32_t E, N, K, group, tile_rows, unit_k;
  uint32_t flags;
  int32_t n_tiles;
  int64_t tile_bytes;   // bytes of one 128-row tile over all of K
  int64_t expert_bytes; // n_tiles * tile_bytes
};
static_assert(sizeof(PackHeader) <= kPackHeaderBytes, "header too large");

// Programmatic dependent launch.  A kernel launched with
// launch_kernel(..., pdl = true) may start while the previous kernel in the
// stream is still running; grid_dep_wait() returns once that kernel has
// completed and its writes are visible (at once for an ordinary launch), so
// it must come before any read of what the previous kernels wrote.  Those
// reads must not use __ldg / ld.global.nc: the compiler treats such a load
// as invariant and may move it above the wait (measured: stale block counts
// in the GEMM after the wait); they use ld_ca / ld_cg / ld_cg_v4 below,
// which stay in program order.
// grid_dep_launch() lets the next programmatic launch be scheduled once
// every CTA of this grid has issued it or exited; the kernels here issue it
// only after their own grid_dep_wait(), so a kernel two launches later
// always finds the outputs of the one before its predecessor complete.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Global loads cached in L2 only (no L1 or texture-cache copy), kept in
// program order relative to the other inline-assembly statements.
__device__ __forceinline__ int ld_cg(const int32_t* p) {
  int v;
  asm volatile("ld.global.cg.b32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
// Same, cached in L1 as well: for small data read many times after the wait
// (the wait makes the preceding grid's writes visible to ordinary loads).
__device__ __forceinline__ int ld_ca(const int32_t* p) {
  int v;
  asm volatile("ld.global.ca.b32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ float ld_ca(const float* p) {
  float v;
  asm volatile("ld.global.ca.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ float ld_cg(const float* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint4 ld_cg_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Four FP32 values, cached in L2 only: for data another CTA wrote (after a
// fence and an atomic that orders it), which this SM's L1 may hold stale.
__device__ __forceinline__ float4 ld_cg_f4(const float* p) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

// Split-K workspace of the decode GEMM: kSplitSlots slots of partial
// accumulators (4 consumer warps x 32 lanes x 4 x up to 4 token tiles, FP32)
// and one arrival counter per (item, consumer warp).
constexpr int kSplitSlots = 512;
constexpr int kSplitSlotFloats = 4 * 32 * 4 * 4;
constexpr size_t kSplitCntBytes = static_cast<size_t>(kSplitSlots) * 4 * sizeof(int);
constexpr size_t kSplitPartialBytes = static_cast<size_t>(kSplitSlots) * kSplitSlotFloats * sizeof(float);

// Launch a kernel, with programmatic stream serialization when pdl is set.
template <typename... P, typename... A>
inline cudaError_t launch_kernel(void (*kern)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                 bool pdl, A&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<A&&>(args)...);
}

__device__ __forceinline__ void set_status(int* st, int code) {
  if (st) atomicCAS(st, 0, code);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Poll limit: each try_wait may suspend the thread for a while, so this is
// seconds of waiting, far beyond any legitimate stall.
constexpr uint32_t kWaitPolls = 1u << 24;
// Poll limit of the waits a test of the timeout path makes run out.
constexpr uint32_t kTestWaitPolls = 1024;

// Returns false (and records a timeout) if the phase did not complete
// within `polls` probes.  Waits for a CTA's own copies in flight before it
// exits always use the full kWaitPolls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status,
                                          uint32_t polls = kWaitPolls) {
  for (uint32_t i = 0; i < polls; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  set_status(status, CHORD_ERR_TIMEOUT);
  return false;
}

// Both barriers' phases complete (parity p0 of b0 and p1 of b1).  The two
// probes are issued back to back and their results combined, so a warp that
// waits for two phases which have usually completed already pays one probe
// latency instead of two.
__device__ __forceinline__ bool mbar_try_wait2(uint64_t* b0, uint32_t p0, uint64_t* b1, uint32_t p1) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 q, [%3], %4;\n\t"
      "and.pred p, p, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(b0)), "r"(p0), "r"(smem_u32(b1)), "r"(p1)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait2(uint64_t* b0, uint32_t p0, uint64_t* b1, uint32_t p1, int* status,
                                           uint32_t polls = kWaitPolls) {
  for (uint32_t i = 0; i < polls; ++i)
    if (mbar_try_wait2(b0, p0, b1, p1)) return true;
  set_status(status, CHORD_ERR_TIMEOUT);
  return false;
}

// Same, for a thread that is not latency critical (a producer waiting for a
// free slot): sleeps briefly between probes instead of spinning.
__device__ __forceinline__ bool mbar_wait_backoff(uint64_t* bar, uint32_t parity, int* status,
                                                  uint32_t polls = kWaitPolls) {
  for (uint32_t i = 0; i < polls; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    __nanosleep(64);
  }
  set_status(status, CHORD_ERR_TIMEOUT);
  return false;
}

// Zero n ints at p (p may be NULL) with the whole grid: a layer's first
// kernel clears the counters its later kernels use (they start after it has
// completed, through the launch chain), instead of a separate memset.
__device__ __forceinline__ void zero_ints(int* p, int n) {
  if (!p) return;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) p[i] = 0;
}

// ------------------------------------------------------- bulk async copies
// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------- MMA
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// D = A(16x16, row) * B(16x8, col) + C, BF16 inputs, FP32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1, const float (&c)[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
        "f"(c[2]), "f"(c[3]));
}

// ------------------------------------------------------------ INT4 decode
// A packed word holds 8 offset-binary nibbles u = q + 8.  Nibble positions
// j and j+4 form register j of an m16n8k16 A fragment.  OR-ing a nibble into
// the mantissa of BF16 128.0 gives the exact value 128 + u = q + 136; the
// constant 136 is removed after the MMA (136 * sum of the activations).
// `mask` (0x000F000F) and `magic` (0x43004300, bf16x2 (128, 128)) are passed
// in registers so that each register costs one 3-input LOP3.
__device__ __forceinline__ void decode_word_offset136(uint32_t w, uint32_t mask, uint32_t magic,
                                                      uint32_t (&a)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j)
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(a[j]) : "r"(w >> (4 * j)), "r"(mask), "r"(magic));
}
constexpr uint32_t kBf16x2Neg136 = 0xC308C308u;  // bf16x2 (-136, -136)


__device__ __forceinline__ float bf16lo_to_f32(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Raise a kernel's dynamic shared-memory limit once per (kernel, device):
// the first call must precede any stream capture; later calls make no CUDA
// call.  Keyed by the kernel itself (a template argument), not its type.
template <auto Kern>
inline cudaError_t ensure_smem_limit(int bytes) {
  static int done_bytes[64] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (done_bytes[dev] >= bytes) return cudaSuccess;
  err = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (err == cudaSuccess) done_bytes[dev] = bytes;
  return err;
}

}  // namespace chord
