// Dense W4A16 GEMM support: the one-expert block map of the indexed GEMM
// (every row is "expert 0", no routing), written on the device each call so
// the dense entry point captures into a CUDA graph like the others.
#include "common.cuh"
#include "kernels.h"

namespace chord {
namespace {

__global__ void dense_setup_kernel(int M, int bm, int32_t* counts, int32_t* offsets, int32_t* ntpp,
                                   int32_t* expert_ids) {
  const int m_pad = (M + bm - 1) / bm * bm;
  const int nblk = m_pad / bm;
  for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < nblk; b += gridDim.x * blockDim.x) expert_ids[b] = 0;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    counts[0] = M;
    offsets[0] = 0;
    offsets[1] = m_pad;
    ntpp[0] = m_pad;
  }
}

}  // namespace

cudaError_t dense_setup_launch(int M, int bm, int32_t* counts, int32_t* offsets, int32_t* ntpp,
                               int32_t* expert_ids, cudaStream_t st) {
  const int nblk = (M + bm - 1) / bm;
  const int grid = nblk > 256 * 8 ? 8 : (nblk + 255) / 256 > 0 ? (nblk + 255) / 256 : 1;
  dense_setup_kernel<<<grid, 256, 0, st>>>(M, bm, counts, offsets, ntpp, expert_ids);
  return cudaGetLastError();
}

}  // namespace chord
