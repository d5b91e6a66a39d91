// Small-M (decode) indexed W4A16 MoE GEMM: weight streaming with register MMA.
//
// [Humming] "워크로드별 튜닝 및 JIT 컴파일": at small batch a multistage
// async-copy + MMA pipeline beats TMA + UMMA; [Chord] "인덱스 커널 기법":
// decode is a weight-streaming problem.  Design on sm_103a:
//   * grid (weight tile, local expert); a CTA streams one expert's 128-row
//     weight tile over all of K once per pass of up to NT*8 of the expert's
//     rows, so each weight byte is read once per expert (not once per block);
//   * one producer warp issues 1-D bulk async copies (TMA engine) of the
//     contiguous packed units and of the expert's activation rows into a
//     STAGES-deep ring, completing on mbarriers;
//   * four consumer warps each own 32 weight rows (two 16-row slabs),
//     decode INT4 nibbles straight into m16n8k16 A fragments (the packed
//     order is the fragment order), take B fragments with ldmatrix, and run
//     mma.sync with weights as the M side and tokens as N ("swap AB");
//   * scales are applied in FP32 per 32-wide group to a per-group partial
//     sum, so the dequantised weights q*s are never rounded;
//   * epilogue: SiLU(gate) * up (gate/up blobs pair the two slabs of a warp)
//     or a plain store, BF16, rows in sorted order.
#include "common.cuh"
#include "kernels.h"

namespace chord {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kUnitsPerStage = 4;                          // 256 of K per stage
constexpr int kXRowBytes = kUnitsPerStage * kUnitK * 2;    // 512
constexpr int kXPitch = kXRowBytes + 16;                   // conflict-free ldmatrix rows

template <int NT>
struct SmallCfg {
  static constexpr int kRowsPerPass = NT * 8;
  static constexpr int kWBytes = kUnitsPerStage * kUnitBytes;
  static constexpr int kStageBytes = kWBytes + kRowsPerPass * kXPitch;
};

struct SmallArgs {
  const uint16_t* A;
  const uint8_t* packed;
  const int32_t* sorted;
  const int32_t* counts;
  const int32_t* offsets;
  uint16_t* C;
  int* status;
  int N, K, topk, ldc, n_tiles, E_local;
  int64_t tile_bytes;
  uint32_t need_flags;
};

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ float silu_f32(float z) { return z / (1.0f + __expf(-z)); }

__device__ bool header_ok(const SmallArgs& a) {
  const PackHeader* h = reinterpret_cast<const PackHeader*>(a.packed);
  return h->magic == kPackMagic && h->version == kPackVersion && h->N == a.N && h->K == a.K &&
         h->group == kGroup && h->E >= a.E_local && h->tile_bytes == a.tile_bytes &&
         (h->flags & a.need_flags) == a.need_flags;
}

template <int NT, int STAGES, bool GATHER, int EPI>
__global__ void __launch_bounds__(kThreads) gemm_small_kernel(SmallArgs a) {
  using Cfg = SmallCfg<NT>;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[STAGES];
  __shared__ __align__(8) uint64_t empty_bar[STAGES];
  __shared__ int hdr_ok;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nt = blockIdx.x, e = blockIdx.y;
  const int cnt = __ldg(a.counts + e);
  if (cnt == 0) return;
  const int off = __ldg(a.offsets + e);
  if (tid == 0) {
    hdr_ok = header_ok(a);
    if (!hdr_ok) set_status(a.status, CHORD_ERR_PREPACK_MISMATCH);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (!hdr_ok) return;

  const int n_units = a.K / kUnitK;
  const int k_stages = (n_units + kUnitsPerStage - 1) / kUnitsPerStage;
  const int passes = (cnt + Cfg::kRowsPerPass - 1) / Cfg::kRowsPerPass;
  const int iters = passes * k_stages;
  const uint8_t* wtile = a.packed + kPackHeaderBytes +
                         (static_cast<size_t>(e) * a.n_tiles + nt) * static_cast<size_t>(a.tile_bytes);

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    int issued = 0;
    bool ok = true;
    for (int it = 0; it < iters && ok; ++it) {
      const int s = it % STAGES;
      if (it >= STAGES) ok = mbar_wait(&empty_bar[s], ((it / STAGES) - 1) & 1, a.status);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      const int pass = it / k_stages, ks = it - pass * k_stages;
      const int units = min(kUnitsPerStage, n_units - ks * kUnitsPerStage);
      const int rows = min(Cfg::kRowsPerPass, cnt - pass * Cfg::kRowsPerPass);
      const uint32_t xbytes = units * kUnitK * 2;
      uint8_t* st = smem + s * Cfg::kStageBytes;
      if (lane == 0) {
        mbar_arrive_expect_tx(&full_bar[s], units * kUnitBytes + rows * xbytes);
        bulk_g2s(st, wtile + static_cast<size_t>(ks) * kUnitsPerStage * kUnitBytes,
                 units * kUnitBytes, &full_bar[s]);
      }
      __syncwarp();
      for (int j = lane; j < rows; j += 32) {
        const int r = off + pass * Cfg::kRowsPerPass + j;
        const int row = GATHER ? __ldg(a.sorted + r) / a.topk : r;
        const uint16_t* src = a.A + static_cast<size_t>(row) * a.K + ks * kUnitsPerStage * kUnitK;
        bulk_g2s(st + Cfg::kWBytes + j * kXPitch, src, xbytes, &full_bar[s]);
      }
      issued = it + 1;
    }
    // Before leaving, make sure no copy into this CTA's smem is in flight.
    if (lane == 0) {
      for (int it = max(0, issued - STAGES); it < issued; ++it)
        mbar_wait(&full_bar[it % STAGES], (it / STAGES) & 1, a.status);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, t = lane & 3;
  const uint32_t smem_base = smem_u32(smem);
  const int slab0 = 2 * warp;
  for (int pass = 0; pass < passes; ++pass) {
    const int rows = min(Cfg::kRowsPerPass, cnt - pass * Cfg::kRowsPerPass);
    const int active = (rows + 7) >> 3;
    float acc[2][NT][4];
#pragma unroll
    for (int sl = 0; sl < 2; ++sl)
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[sl][n][i] = 0.f;

    for (int ks = 0; ks < k_stages; ++ks) {
      const int it = pass * k_stages + ks;
      const int s = it % STAGES;
      if (!mbar_wait(&full_bar[s], (it / STAGES) & 1, a.status)) return;
      const int units = min(kUnitsPerStage, n_units - ks * kUnitsPerStage);
      const uint32_t st = smem_base + s * Cfg::kStageBytes;
      const uint32_t xs = st + Cfg::kWBytes + (lane & 7) * kXPitch + (lane >> 3) * 16;
#pragma unroll
      for (int u = 0; u < kUnitsPerStage; ++u) {
        if (u >= units) break;
        const uint32_t ub = st + u * kUnitBytes;
        const uint4 q0 = lds128(ub + slab0 * 512 + lane * 16);
        const uint4 q1 = lds128(ub + (slab0 + 1) * 512 + lane * 16);
        const uint2 s0 = lds64(ub + kUnitQBytes + slab0 * 64 + g * 8);
        const uint2 s1 = lds64(ub + kUnitQBytes + (slab0 + 1) * 64 + g * 8);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t bf[NT][4];
#pragma unroll
          for (int n = 0; n < NT; ++n)
            if (n < active) ldmatrix_x4(bf[n], xs + n * 8 * kXPitch + (u * kUnitK + half * 32) * 2);
          float tmp[2][NT][4];
#pragma unroll
          for (int sl = 0; sl < 2; ++sl)
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
              for (int i = 0; i < 4; ++i) tmp[sl][n][i] = 0.f;
#pragma unroll
          for (int stp = 0; stp < 2; ++stp) {
            const int j = half * 2 + stp;
            const uint32_t w0 = j == 0 ? q0.x : j == 1 ? q0.y : j == 2 ? q0.z : q0.w;
            const uint32_t w1 = j == 0 ? q1.x : j == 1 ? q1.y : j == 2 ? q1.z : q1.w;
            uint32_t a0[4], a1[4];
            dequant_word(w0, a0);
            dequant_word(w1, a1);
#pragma unroll
            for (int n = 0; n < NT; ++n) {
              if (n < active) {
                mma_bf16_16816(tmp[0][n], a0, bf[n][2 * stp], bf[n][2 * stp + 1], tmp[0][n]);
                mma_bf16_16816(tmp[1][n], a1, bf[n][2 * stp], bf[n][2 * stp + 1], tmp[1][n]);
              }
            }
          }
          const uint32_t sw0 = half ? s0.y : s0.x;
          const uint32_t sw1 = half ? s1.y : s1.x;
          const float sg0 = bf16lo_to_f32(sw0), sh0 = bf16hi_to_f32(sw0);
          const float sg1 = bf16lo_to_f32(sw1), sh1 = bf16hi_to_f32(sw1);
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            acc[0][n][0] = fmaf(sg0, tmp[0][n][0], acc[0][n][0]);
            acc[0][n][1] = fmaf(sg0, tmp[0][n][1], acc[0][n][1]);
            acc[0][n][2] = fmaf(sh0, tmp[0][n][2], acc[0][n][2]);
            acc[0][n][3] = fmaf(sh0, tmp[0][n][3], acc[0][n][3]);
            acc[1][n][0] = fmaf(sg1, tmp[1][n][0], acc[1][n][0]);
            acc[1][n][1] = fmaf(sg1, tmp[1][n][1], acc[1][n][1]);
            acc[1][n][2] = fmaf(sh1, tmp[1][n][2], acc[1][n][2]);
            acc[1][n][3] = fmaf(sh1, tmp[1][n][3], acc[1][n][3]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[s]);
    }

    // ------------------------------------------------------------ epilogue
    const int r0 = off + pass * Cfg::kRowsPerPass;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int tok = n * 8 + 2 * t + (i & 1);
        if (tok >= rows) continue;
        const size_t r = static_cast<size_t>(r0 + tok);
        const int rr = g + 8 * (i >> 1);
        if (EPI == CHORD_EPI_SILU_MUL) {
          const int col = 64 * nt + 16 * warp + rr;
          const float h = silu_f32(acc[0][n][i]) * acc[1][n][i];
          a.C[r * a.ldc + col] = f32_to_bf16_rn(h);
        } else {
#pragma unroll
          for (int sl = 0; sl < 2; ++sl) {
            const int col = kTileRows * nt + 32 * warp + 16 * sl + rr;
            if (col < a.N) a.C[r * a.ldc + col] = f32_to_bf16_rn(acc[sl][n][i]);
          }
        }
      }
    }
  }
}

template <int NT, int STAGES, bool GATHER, int EPI>
cudaError_t launch_small(const SmallArgs& a, cudaStream_t st) {
  auto kern = gemm_small_kernel<NT, STAGES, GATHER, EPI>;
  const int smem = STAGES * SmallCfg<NT>::kStageBytes;
  cudaError_t err = ensure_smem_limit<gemm_small_kernel<NT, STAGES, GATHER, EPI>>(smem);
  if (err != cudaSuccess) return err;
  dim3 grid(a.n_tiles, a.E_local);
  kern<<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

template <int NT, int STAGES>
cudaError_t dispatch_mode(const SmallArgs& a, bool gather, int epi, cudaStream_t st) {
  if (gather) {
    return epi == CHORD_EPI_SILU_MUL ? launch_small<NT, STAGES, true, CHORD_EPI_SILU_MUL>(a, st)
                                     : launch_small<NT, STAGES, true, CHORD_EPI_STORE>(a, st);
  }
  return epi == CHORD_EPI_SILU_MUL ? launch_small<NT, STAGES, false, CHORD_EPI_SILU_MUL>(a, st)
                                   : launch_small<NT, STAGES, false, CHORD_EPI_STORE>(a, st);
}

}  // namespace

cudaError_t gemm_small_launch(const GemmLaunch& g, int rows_per_pass, cudaStream_t st) {
  SmallArgs a;
  a.A = g.A;
  a.packed = static_cast<const uint8_t*>(g.packed);
  a.sorted = g.sorted;
  a.counts = g.counts;
  a.offsets = g.offsets;
  a.C = g.C;
  a.status = g.status;
  a.N = g.N;
  a.K = g.K;
  a.topk = g.topk;
  a.E_local = g.E_local;
  const PackHeader h = make_pack_header(g.E_local, g.N, g.K, g.epilogue == CHORD_EPI_SILU_MUL);
  a.n_tiles = h.n_tiles;
  a.tile_bytes = h.tile_bytes;
  a.need_flags = g.epilogue == CHORD_EPI_SILU_MUL ? kPackFlagGateUp : 0u;
  a.ldc = g.epilogue == CHORD_EPI_SILU_MUL ? g.N / 2 : g.N;
  if (rows_per_pass <= 8) return dispatch_mode<1, 4>(a, g.gather, g.epilogue, st);
  if (rows_per_pass <= 16) return dispatch_mode<2, 4>(a, g.gather, g.epilogue, st);
  return dispatch_mode<4, 6>(a, g.gather, g.epilogue, st);
}

}  // namespace chord
