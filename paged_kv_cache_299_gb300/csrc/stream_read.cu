// Read-only streaming kernel: the in-run HBM read reference that the decode kernel's
// achieved bandwidth is compared with (same bytes, same launch conditions).  It reads a
// buffer once with 16-byte vector loads and XORs every 32-bit word into a result word, so
// none of the loads can be dropped and a caller can check the result.
//
// Grid: eight 1024-thread CTAs per SM (two resident per SM, so four waves), four loads in
// flight per thread, streaming cache hint; the fastest shape of a sweep on this GPU.
#include "common.cuh"
#include "internal.h"

namespace pkv {

namespace {

constexpr int kStreamThreads = 1024;
constexpr int kStreamCtasPerSm = 8;

__global__ void __launch_bounds__(kStreamThreads)
stream_read_kernel(const uint4* __restrict__ p, size_t n16, uint32_t* __restrict__ x) {
  __shared__ uint32_t warp_x[kStreamThreads / 32];
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  uint32_t acc = 0;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    const uint4 a = __ldcs(p + i);
    const uint4 b = __ldcs(p + i + stride);
    const uint4 c = __ldcs(p + i + 2 * stride);
    const uint4 d = __ldcs(p + i + 3 * stride);
    acc ^= (a.x ^ a.y ^ a.z ^ a.w) ^ (b.x ^ b.y ^ b.z ^ b.w) ^ (c.x ^ c.y ^ c.z ^ c.w) ^
           (d.x ^ d.y ^ d.z ^ d.w);
  }
  for (; i < n16; i += stride) {
    const uint4 a = __ldcs(p + i);
    acc ^= a.x ^ a.y ^ a.z ^ a.w;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, off);
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) warp_x[warp] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t v = 0;
    for (int w = 0; w < kStreamThreads / 32; ++w) v ^= warp_x[w];
    atomicXor(x, v);
  }
}

}  // namespace

cudaError_t launch_stream_read(const void* buf, size_t bytes, uint32_t* x, cudaStream_t stream) {
  if (bytes == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  stream_read_kernel<<<sms * kStreamCtasPerSm, kStreamThreads, 0, stream>>>(
      static_cast<const uint4*>(buf), bytes / 16, x);
  return cudaGetLastError();
}

}  // namespace pkv
