// Backward pass of blocked GQA flash attention on sm_103a (placeholder until
// the tcgen05 kernels land): the D preprocess only.
#include <cuda_bf16.h>
#include "kernels.h"
#include "ptx.cuh"

namespace fa {
namespace {

// D[row] = sum_h dO[row, h] * o[row, h] in fp32; one warp per row.
__global__ void bwd_preprocess_kernel(const __nv_bfloat16* __restrict__ o,
                                      const __nv_bfloat16* __restrict__ dO, float* __restrict__ delta,
                                      long rows, int H) {
  const long row = (long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const uint4* po = reinterpret_cast<const uint4*>(o + row * H);
  const uint4* pd = reinterpret_cast<const uint4*>(dO + row * H);
  float acc = 0.f;
  for (int i = lane; i < H / 8; i += 32) {
    const uint4 a = __ldg(po + i), d = __ldg(pd + i);
    const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&d);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 fa2 = __bfloat1622float2(a2[j]);
      const float2 fd2 = __bfloat1622float2(d2[j]);
      acc = fmaf(fa2.x, fd2.x, acc);
      acc = fmaf(fa2.y, fd2.y, acc);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) delta[row] = acc;
}

}  // namespace

cudaError_t launch_bwd_preprocess(const void* o, const void* dO, float* delta, long rows, int H,
                                  cudaStream_t st) {
  const int warps = 8;
  const long blocks = (rows + warps - 1) / warps;
  bwd_preprocess_kernel<<<(unsigned)blocks, warps * 32, 0, st>>>(
      reinterpret_cast<const __nv_bfloat16*>(o), reinterpret_cast<const __nv_bfloat16*>(dO), delta,
      rows, H);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv(const BwdArgs&, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_bwd_dq(const BwdArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace fa
