// Large-M (prefill) indexed W4A16 MoE GEMM on the 5th-generation tensor cores.
//
// [Humming] "워크로드별 튜닝 및 JIT 컴파일": at larger batch a TMA + UMMA
// pipeline gives the better throughput; [Chord] "그룹 SM90 커널 기법": a
// persistent warp-specialised main loop pipelining TMA loads, dequantisation
// and the MMA.  Design on sm_103a (one CTA per SM, persistent):
//   * work item = (local expert, 128 weight rows, pass of up to 256 of the
//     expert's rows); items are dealt round-robin to the CTAs;
//   * the MMA is "swap AB": the 128 weight rows are M, the expert's rows
//     (tokens) are N (a multiple of 16 up to 256), so an expert's rows are
//     padded to 16, not to 128;
//   * warp 0 (producer): 1-D bulk copies of the two packed 64-row units of
//     each 64-wide K step, and 2-D TMA loads (128-byte swizzle) of the
//     expert's activation rows, into a 4-stage ring;
//   * warps 2-5 (dequant): INT4 -> BF16 q*s (rounded once) written into the
//     K-major 128-byte-swizzled A tile, then a proxy fence;
//   * warp 1 (MMA): TMEM allocation, one thread issues tcgen05.mma
//     (M=128, K=16 x4 per stage) into one of two TMEM accumulators and
//     commits stage and item completion to mbarriers;
//   * warps 6-9 (epilogue): tcgen05.ld of the accumulator, SiLU(gate) * up
//     (gate and up rows of one index sit 8 TMEM lanes apart) or a plain
//     store, BF16, rows in sorted order; the second accumulator lets the next
//     item's MMAs run meanwhile.
// Every mbarrier wait is bounded; on a timeout the CTA records
// CHORD_ERR_TIMEOUT, drains its own copies and MMAs, frees TMEM and exits.
#include "common.cuh"
#include "kernels.h"
#include "tc5.cuh"

namespace chord {
namespace {

constexpr int kStages = 4;
constexpr int kMRows = 128;                      // weight rows per item (2 packed tiles)
constexpr int kMaxTok = 256;                     // tokens per pass (MMA N)
constexpr int kBoxRows = 32;                     // activation rows per TMA box
constexpr int kABytes = kMRows * kUnitK * 2;     // 16 KB
constexpr int kBBytes = kMaxTok * kUnitK * 2;    // 32 KB
constexpr int kPBytes = 2 * kUnitBytes;          // 4608
constexpr int kStageBytes = kABytes + kBBytes + 5120;
constexpr int kSmemBytes = kStages * kStageBytes + 1024;   // + alignment slack
constexpr int kThreads = 320;
constexpr int kTmemCols = 512;
constexpr int kMaxExperts = 1024;
static_assert(kSmemBytes + (kMaxExperts + 1) * 4 + 256 <= 232448, "shared memory budget");

struct LargeArgs {
  const uint8_t* packed;
  const int32_t* counts;
  const int32_t* offsets;
  uint16_t* C;
  int* status;
  int N, K, ldc, E_local, n_blob_tiles;
  int64_t tile_bytes;
  uint32_t need_flags;
  int gate_up;
};

struct Item {
  int e, wt, row0, rows;
};

__device__ __forceinline__ bool header_ok(const LargeArgs& a) {
  const PackHeader* h = reinterpret_cast<const PackHeader*>(a.packed);
  return h->magic == kPackMagic && h->version == kPackVersion && h->N == a.N && h->K == a.K &&
         h->group == kGroup && h->E >= a.E_local && h->tile_bytes == a.tile_bytes &&
         (h->flags & a.need_flags) == a.need_flags;
}

// Item i of the global list (experts in order; per expert, passes, then
// 128-row weight tiles).  prefix[e] = first item of expert e.
__device__ __forceinline__ Item item_of(int i, const int* prefix, const int32_t* counts,
                                        const int32_t* offsets, int E, int n_wt) {
  int lo = 0, hi = E - 1;  // largest e with prefix[e] <= i
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= i) lo = mid; else hi = mid - 1;
  }
  const int e = lo, cnt = __ldg(counts + e);
  const int local = i - prefix[e];
  const int p = local / n_wt, wt = local - p * n_wt;
  const int n_pass = (cnt + kMaxTok - 1) / kMaxTok;
  const int tp = ((cnt + n_pass - 1) / n_pass + 15) & ~15;
  Item it;
  it.e = e;
  it.wt = wt;
  it.row0 = __ldg(offsets + e) + p * tp;
  it.rows = min(tp, cnt - p * tp);
  return it;
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_large_kernel(const __grid_constant__ CUtensorMap tmap_b, LargeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kStages], afull_bar[kStages], empty_bar[kStages];
  __shared__ __align__(8) uint64_t tfull_bar[2], tempty_bar[2], done_bar;
  __shared__ uint32_t tmem_base_s;
  __shared__ int prefix[kMaxExperts + 1];
  __shared__ int hdr_ok;
  __shared__ volatile int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t smem0 = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (smem0 - smem_u32(smem_raw));
  const int E = a.E_local, K = a.K;
  const int n_wt = a.N / kMRows;
  const int k_steps = K / kUnitK;

  if (tid == 0) {
    hdr_ok = header_ok(a);
    if (!hdr_ok) set_status(a.status, CHORD_ERR_PREPACK_MISMATCH);
    abort_flag = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&afull_bar[s], 4);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], 4);
    }
    mbar_init(&done_bar, 1);
    fence_mbar_init();
  }
  // the item prefix over experts
  if (warp == 0) {
    int run = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      int items = 0;
      const int cnt = e < E ? __ldg(a.counts + e) : 0;
      if (cnt > 0) items = n_wt * ((cnt + kMaxTok - 1) / kMaxTok);
      int inc = items;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
      }
      if (e < E) prefix[e] = run + inc - items;
      run += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) prefix[E] = run;
  }
  if (warp == 1) tmem_alloc(&tmem_base_s, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_s;
  const int total_items = hdr_ok ? prefix[E] : 0;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int it = 0;
      for (int i = blockIdx.x; i < total_items && !abort_flag; i += gridDim.x) {
        const Item item = item_of(i, prefix, a.counts, a.offsets, E, n_wt);
        const int nbox = (item.rows + kBoxRows - 1) / kBoxRows;
        const uint8_t* t0 = a.packed + kPackHeaderBytes +
                            (static_cast<size_t>(item.e) * a.n_blob_tiles + 2 * item.wt) *
                                static_cast<size_t>(a.tile_bytes);
        for (int ks = 0; ks < k_steps; ++ks, ++it) {
          const int s = it % kStages;
          if (it >= kStages && !mbar_wait(&empty_bar[s], ((it / kStages) - 1) & 1, a.status)) {
            abort_flag = 1;
            break;
          }
          uint8_t* st = smem + s * kStageBytes;
          mbar_arrive_expect_tx(&full_bar[s], kPBytes + nbox * kBoxRows * kUnitK * 2);
          bulk_g2s(st + kABytes + kBBytes, t0 + static_cast<size_t>(ks) * kUnitBytes, kUnitBytes,
                   &full_bar[s]);
          bulk_g2s(st + kABytes + kBBytes + kUnitBytes,
                   t0 + a.tile_bytes + static_cast<size_t>(ks) * kUnitBytes, kUnitBytes, &full_bar[s]);
          for (int b = 0; b < nbox; ++b)
            tma_load_2d(st + kABytes + b * kBoxRows * kUnitK * 2, &tmap_b, ks * kUnitK,
                        item.row0 + b * kBoxRows, &full_bar[s]);
        }
      }
      // drain: every issued copy must land before the CTA can exit
      for (int j = max(0, it - kStages); j < it; ++j)
        mbar_wait(&full_bar[j % kStages], (j / kStages) & 1, a.status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int it = 0, j = 0;
      bool issued_any = false;
      for (int i = blockIdx.x; i < total_items && !abort_flag; i += gridDim.x, ++j) {
        const Item item = item_of(i, prefix, a.counts, a.offsets, E, n_wt);
        const int acc = j & 1, use = j >> 1;
        if (use >= 1 && !mbar_wait(&tempty_bar[acc], (use - 1) & 1, a.status)) {
          abort_flag = 1;
          break;
        }
        tc_fence_after();
        const int n_mma = (item.rows + 15) & ~15;
        const uint32_t idesc = idesc_bf16_f32(kMRows, n_mma);
        const uint32_t d_tmem = tmem_base + acc * kMaxTok;
        for (int ks = 0; ks < k_steps; ++ks, ++it) {
          const int s = it % kStages;
          if (!mbar_wait(&afull_bar[s], (it / kStages) & 1, a.status) ||
              !mbar_wait(&full_bar[s], (it / kStages) & 1, a.status)) {
            abort_flag = 1;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem0 + s * kStageBytes;
          const uint64_t a_desc = sw128_kmajor_desc(st);
          const uint64_t b_desc = sw128_kmajor_desc(st + kABytes);
#pragma unroll
          for (int kk = 0; kk < kUnitK / 16; ++kk)
            tc_mma_bf16(d_tmem, a_desc + 2 * kk, b_desc + 2 * kk, idesc, (ks | kk) != 0);
          tc_commit(&empty_bar[s]);
          issued_any = true;
        }
        if (abort_flag) break;
        tc_commit(&tfull_bar[acc]);
      }
      // all issued MMAs complete before TMEM can be freed
      if (issued_any) {
        tc_commit(&done_bar);
        mbar_wait(&done_bar, 0, a.status);
      }
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ dequant
    const int d = warp - 2;
    const int g = lane >> 2, t = lane & 3;
    const uint32_t mask = 0x000F000Fu, magic = 0x43004300u;
    const __nv_bfloat162 k136 = __floats2bfloat162_rn(136.f, 136.f);
    int it = 0;
    for (int i = blockIdx.x; i < total_items && !abort_flag; i += gridDim.x) {
      for (int ks = 0; ks < k_steps; ++ks, ++it) {
        const int s = it % kStages;
        if (!mbar_wait(&full_bar[s], (it / kStages) & 1, a.status)) {
          abort_flag = 1;
          break;
        }
        uint8_t* st = smem + s * kStageBytes;
        const uint8_t* pk = st + kABytes + kBBytes;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int S = 2 * d + h;                      // 16-row slab of the 128-row tile
          const uint8_t* unit = pk + (S >> 2) * kUnitBytes;
          const uint4 q = *reinterpret_cast<const uint4*>(unit + (S & 3) * 512 + lane * 16);
          const uint2 sc = *reinterpret_cast<const uint2*>(unit + kUnitQBytes + (S & 3) * 64 + g * 8);
          const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
          const int r_lo = 16 * S + g;                  // rows r_lo and r_lo + 8; (row & 7) == g
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t sw = (j >> 1) ? sc.y : sc.x;
            const uint32_t s_lo = __byte_perm(sw, sw, 0x1010);   // {s[g], s[g]}
            const uint32_t s_hi = __byte_perm(sw, sw, 0x3232);   // {s[g+8], s[g+8]}
            uint32_t v[4];
            decode_word_offset136(w4[j], mask, magic, v);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162*>(&v[r]);
              x = __hsub2(x, k136);
              const uint32_t sr = (r & 1) ? s_hi : s_lo;
              x = __hmul2(x, *reinterpret_cast<const __nv_bfloat162*>(&sr));
              v[r] = *reinterpret_cast<uint32_t*>(&x);
            }
            // v[0]: row r_lo, k 16j+2t; v[1]: row r_lo+8; v[2]: row r_lo, k +8; v[3]: row r_lo+8, k +8
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              const int row = r_lo + 8 * (r & 1);
              const int chunk = 2 * j + (r >> 1);
              const uint32_t off = row * 128 + ((chunk ^ g) << 4) + 4 * t;
              *reinterpret_cast<uint32_t*>(st + off) = v[r];
            }
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&afull_bar[s]);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int qw = warp & 3;                 // TMEM lane quarter of this warp
    int j = 0;
    for (int i = blockIdx.x; i < total_items && !abort_flag; i += gridDim.x, ++j) {
      const Item item = item_of(i, prefix, a.counts, a.offsets, E, n_wt);
      const int acc = j & 1, use = j >> 1;
      if (!mbar_wait(&tfull_bar[acc], use & 1, a.status)) {
        abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + acc * kMaxTok + (static_cast<uint32_t>(32 * qw) << 16);
      const int row_in = 32 * qw + lane;     // A row = TMEM lane
      for (int c0 = 0; c0 < item.rows; c0 += 32) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(taddr + c0, v);
        tmem_ld_wait();
        const int ncol = min(32, item.rows - c0);
        if (a.gate_up) {
          // rows 0-7 of a 16-row slab are gate, rows 8-15 the matching up rows
          const int bt = 2 * item.wt + (row_in >> 6);
          const int p = row_in & 63;
          const int col = 32 * bt + 8 * (p >> 4) + (p & 7);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float mine = __uint_as_float(v[c]);
            const float other = __shfl_xor_sync(0xffffffffu, mine, 8);
            if (!(lane & 8) && c < ncol) {
              const float h = mine / (1.0f + __expf(-mine)) * other;
              a.C[static_cast<size_t>(item.row0 + c0 + c) * a.ldc + col] = f32_to_bf16_rn(h);
            }
          }
        } else {
          const int col = kMRows * item.wt + row_in;
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            if (c < ncol)
              a.C[static_cast<size_t>(item.row0 + c0 + c) * a.ldc + col] =
                  f32_to_bf16_rn(__uint_as_float(v[c]));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty_bar[acc]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

}  // namespace

size_t gemm_large_smem_bytes() { return kSmemBytes; }

cudaError_t gemm_large_launch(const GemmLaunch& g, const uint16_t* B, size_t b_rows,
                              cudaStream_t st) {
  if (g.N % kMRows != 0 || g.K % kUnitK != 0 || g.E_local > kMaxExperts) return cudaErrorInvalidValue;
  EncodeTiledFn encode = get_encode_fn();
  if (!encode) return cudaErrorNotSupported;
  CUtensorMap map;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(g.K), static_cast<cuuint64_t>(b_rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(g.K) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kUnitK), static_cast<cuuint32_t>(kBoxRows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(B), dims,
                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  LargeArgs a;
  a.packed = static_cast<const uint8_t*>(g.packed);
  a.counts = g.counts;
  a.offsets = g.offsets;
  a.C = g.C;
  a.status = g.status;
  a.N = g.N;
  a.K = g.K;
  a.E_local = g.E_local;
  const bool gate_up = g.epilogue == CHORD_EPI_SILU_MUL;
  const PackHeader h = make_pack_header(g.E_local, g.N, g.K, gate_up);
  a.n_blob_tiles = h.n_tiles;
  a.tile_bytes = h.tile_bytes;
  a.need_flags = gate_up ? kPackFlagGateUp : 0u;
  a.gate_up = gate_up ? 1 : 0;
  a.ldc = gate_up ? g.N / 2 : g.N;
  cudaError_t err = ensure_smem_limit<gemm_large_kernel>(kSmemBytes);
  if (err != cudaSuccess) return err;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  gemm_large_kernel<<<sms, kThreads, kSmemBytes, st>>>(map, a);
  return cudaGetLastError();
}

// ------------------------------------------------------------ row gather
// x_sorted[r] = x[sorted[r] / topk] for r < num_tokens_post_padded (padding
// rows become zeros), so the activation rows of an expert are contiguous for
// the tensor-map loads.
__global__ void gather_rows_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ sorted,
                                   const int32_t* __restrict__ ntpp, int topk, int sentinel, int K,
                                   uint16_t* __restrict__ out) {
  const int n = __ldg(ntpp);
  const int vec_per_row = K / 8;
  for (int r = blockIdx.x; r < n; r += gridDim.x) {
    const int f = __ldg(sorted + r);
    uint4* dst = reinterpret_cast<uint4*>(out + static_cast<size_t>(r) * K);
    if (f >= sentinel) {
      for (int c = threadIdx.x; c < vec_per_row; c += blockDim.x) dst[c] = make_uint4(0, 0, 0, 0);
    } else {
      const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(f / topk) * K);
      for (int c = threadIdx.x; c < vec_per_row; c += blockDim.x) dst[c] = __ldg(src + c);
    }
  }
}

cudaError_t gather_rows_launch(const uint16_t* x, const int32_t* sorted, const int32_t* ntpp,
                               int topk, int sentinel, int K, size_t capacity, uint16_t* out,
                               cudaStream_t st) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long want = static_cast<long long>(capacity);
  const int grid = static_cast<int>(want < 8LL * sms ? (want > 0 ? want : 1) : 8LL * sms);
  gather_rows_kernel<<<grid, 256, 0, st>>>(x, sorted, ntpp, topk, sentinel, K, out);
  return cudaGetLastError();
}

}  // namespace chord
