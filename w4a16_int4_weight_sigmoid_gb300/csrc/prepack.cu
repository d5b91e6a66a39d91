// INT4 weight prepack into the kernel layout.
//
// Preprocessing that validates, pads N and repacks for the target kernel
// ([Humming] "워크로드별 튜닝 및 JIT 컴파일"; auto padding: [HumPR]
// "왜 이게 좋은가" 2).  Layout of a blob:
//
//   header (256 B) | expert 0: tile 0: unit 0 | unit 1 | ... | tile 1 ... | expert 1 ...
//
// A tile is 64 weight rows ("physical rows", 4 slabs of 16) over all of K; a
// unit is the tile's 64-wide K slice, 2304 bytes, contiguous so one bulk copy
// moves any run of units:
//   q part, 2048 B: [slab 0..3][lane 0..31][4 words]; word j (k16 step j of
//     the unit) holds the lane's m16n8k16 A fragment as 8 offset-binary
//     nibbles u = q + 8: nibble p (p & 3 = pp, p >> 2 = hi) is row
//     g + 8*(pp & 1), column 2t + 8*(pp >> 1) + hi of the 16x16 block,
//     with g = lane / 4, t = lane % 4.
//   s part, 256 B: [slab][g 0..7][group 0..1][row half 0..1] BF16 scales of
//     rows g and g+8 for the unit's two 32-wide groups.
// Physical -> logical rows: plain weights: tile nt row p = logical 64*nt + p
// (rows >= N are zero).  Gate/up weights (N = 2I): slab s of tile nt holds
// intermediate indices i = 32*nt + 8*s + (0..7), gate rows in its first 8
// rows and the matching up rows in its last 8, so one MMA thread holds the
// gate and up values of the same (i, token).
#include "common.cuh"
#include "kernels.h"

namespace chord {
namespace {

__device__ __forceinline__ int logical_row(int nt, int p, int N, bool gate_up) {
  if (gate_up) {
    const int I = N / 2;
    const int r = p & 15;
    return (r >> 3) * I + 32 * nt + 8 * (p >> 4) + (r & 7);
  }
  const int n = kTileRows * nt + p;
  return n < N ? n : -1;
}

__global__ void prepack_kernel(const uint8_t* __restrict__ q, const uint16_t* __restrict__ s, int E,
                               int N, int K, int n_tiles, bool gate_up, uint8_t* __restrict__ out) {
  const int n_units = K / kUnitK;
  const long long total = static_cast<long long>(E) * n_tiles * n_units * kSlabs * 32;
  const long long gid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= total) return;
  const int lane = static_cast<int>(gid & 31);
  const int slab = static_cast<int>((gid >> 5) % kSlabs);
  long long rest = (gid >> 5) / kSlabs;
  const int kt = static_cast<int>(rest % n_units);
  rest /= n_units;
  const int nt = static_cast<int>(rest % n_tiles);
  const int e = static_cast<int>(rest / n_tiles);
  const int g = lane >> 2, t = lane & 3;
  const int row_lo = logical_row(nt, 16 * slab + g, N, gate_up);
  const int row_hi = logical_row(nt, 16 * slab + g + 8, N, gate_up);
  const size_t qrow = static_cast<size_t>(K / 2);
  const uint8_t* qe = q + static_cast<size_t>(e) * N * qrow;
  uint32_t words[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t w = 0;
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      const int pp = p & 3, hi = p >> 2;
      const int row = (pp & 1) ? row_hi : row_lo;
      const int col = kt * kUnitK + 16 * j + 2 * t + 8 * (pp >> 1) + hi;
      uint32_t nib = 8u;  // u = q + 8 with q = 0 for padding rows
      if (row >= 0) {
        const uint8_t byte = qe[static_cast<size_t>(row) * qrow + (col >> 1)];
        nib = ((col & 1) ? (byte >> 4) : (byte & 0xF)) ^ 8u;
      }
      w |= nib << (4 * p);
    }
    words[j] = w;
  }
  const size_t unit_off = kPackHeaderBytes +
                          ((static_cast<size_t>(e) * n_tiles + nt) * n_units + kt) * kUnitBytes;
  uint4 v = make_uint4(words[0], words[1], words[2], words[3]);
  *reinterpret_cast<uint4*>(out + unit_off + slab * 512 + lane * 16) = v;
  static_assert(kUnitQBytes == kSlabs * 512, "q part is 512 B per slab");
  if (t == 0) {
    const int ng = K / kGroup;
    const uint16_t* se = s + static_cast<size_t>(e) * N * ng;
    uint16_t sv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int grp = 2 * kt + (i >> 1);
      const int row = (i & 1) ? row_hi : row_lo;
      sv[i] = row >= 0 ? se[static_cast<size_t>(row) * ng + grp] : 0;
    }
    uint2 sw = make_uint2(sv[0] | (uint32_t(sv[1]) << 16), sv[2] | (uint32_t(sv[3]) << 16));
    *reinterpret_cast<uint2*>(out + unit_off + kUnitQBytes + slab * 64 + g * 8) = sw;
  }
}

__global__ void prepack_header_kernel(PackHeader h, uint8_t* out) {
  uint32_t* dst = reinterpret_cast<uint32_t*>(out);
  const uint32_t* src = reinterpret_cast<const uint32_t*>(&h);
  for (int i = threadIdx.x; i < kPackHeaderBytes / 4; i += blockDim.x)
    dst[i] = i < static_cast<int>(sizeof(PackHeader) / 4) ? src[i] : 0u;
}

}  // namespace

PackHeader make_pack_header(int E, int N, int K, bool gate_up) {
  PackHeader h{};
  h.magic = kPackMagic;
  h.version = kPackVersion;
  h.E = E;
  h.N = N;
  h.K = K;
  h.group = kGroup;
  h.tile_rows = kTileRows;
  h.unit_k = kUnitK;
  h.flags = gate_up ? kPackFlagGateUp : 0u;
  h.n_tiles = (N + kTileRows - 1) / kTileRows;
  h.tile_bytes = static_cast<int64_t>(K / kUnitK) * kUnitBytes;
  h.expert_bytes = h.n_tiles * h.tile_bytes;
  return h;
}

size_t prepack_bytes(int E, int N, int K) {
  PackHeader h = make_pack_header(E, N, K, false);
  return kPackHeaderBytes + static_cast<size_t>(E) * h.expert_bytes;
}

cudaError_t prepack_launch(const uint8_t* q, const uint16_t* s, int E, int N, int K, bool gate_up,
                           uint8_t* out, cudaStream_t st) {
  PackHeader h = make_pack_header(E, N, K, gate_up);
  prepack_header_kernel<<<1, 64, 0, st>>>(h, out);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const long long total = static_cast<long long>(E) * h.n_tiles * (K / kUnitK) * kSlabs * 32;
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  const long long blocks = (total + threads - 1) / threads;
  prepack_kernel<<<static_cast<unsigned>(blocks), threads, 0, st>>>(q, s, E, N, K, h.n_tiles,
                                                                    gate_up, out);
  return cudaGetLastError();
}

}  // namespace chord
