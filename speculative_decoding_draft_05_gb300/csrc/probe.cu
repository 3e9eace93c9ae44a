// probe.cu -- a streaming kernel used to measure the bandwidth ceiling of the
// draft step's traffic mix (2 bytes read, 4 bytes written per element) on this
// GPU: bf16 in, fp32 out, contiguous 16-byte pieces, grid-stride over four
// CTAs of 256 threads per SM.  A measurement aid; no step of the path uses it.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace dspark {

namespace {

__global__ void __launch_bounds__(256)
stream_probe_kernel(const uint4* __restrict__ in, float4* __restrict__ out, size_t n8) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n8;
       i += (size_t)gridDim.x * blockDim.x) {
    const uint4 q = __ldcs(in + i);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    float f[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      f[2 * j] = __uint_as_float(w[j] << 16);
      f[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
    }
    __stcs(out + 2 * i, make_float4(f[0], f[1], f[2], f[3]));
    __stcs(out + 2 * i + 1, make_float4(f[4], f[5], f[6], f[7]));
  }
}

}  // namespace

cudaError_t launch_stream_probe(const void* in, float* out, size_t n, cudaStream_t s) {
  int dev = 0, sms = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const size_t n8 = n / 8;
  size_t grid = (size_t)sms * 4;
  const size_t need = (n8 + 255) / 256;
  if (need < grid) grid = need > 0 ? need : 1;
  stream_probe_kernel<<<(unsigned)grid, 256, 0, s>>>((const uint4*)in, (float4*)out, n8);
  return cudaGetLastError();
}

}  // namespace dspark
