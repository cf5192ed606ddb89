// Measurement helper for the roofline's L2 term (not part of the attention method).
//
// Streams a device buffer `reps` times with 16-byte loads that bypass L1 (ld.global.cg),
// from four 512-thread blocks per SM.  With a buffer well inside L2 (at most half of it)
// every load after the first pass is an L2 hit, so reps * bytes / time is the L2-to-SM
// read bandwidth that a kernel gathering L2-resident tiles can draw on.
#include "common.cuh"

namespace sba {
namespace {

constexpr int kProbeThreads = 512;

__global__ void __launch_bounds__(kProbeThreads)
l2_read_kernel(const uint4* __restrict__ buf, long long n16, int reps, unsigned* __restrict__ sink) {
  unsigned acc = 0u;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long first = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  for (int r = 0; r < reps; ++r) {
    long long i = first;
    // four independent loads in flight per thread
    for (; i + 3 * stride < n16; i += 4 * stride) {
      const uint4 a = __ldcg(buf + i), b = __ldcg(buf + i + stride);
      const uint4 c = __ldcg(buf + i + 2 * stride), d = __ldcg(buf + i + 3 * stride);
      acc ^= (a.x ^ a.y ^ a.z ^ a.w) ^ (b.x ^ b.y ^ b.z ^ b.w) ^ (c.x ^ c.y ^ c.z ^ c.w) ^
             (d.x ^ d.y ^ d.z ^ d.w);
    }
    for (; i < n16; i += stride) {
      const uint4 v = __ldcg(buf + i);
      acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
  }
  // one word per warp keeps every load live
  acc = __reduce_xor_sync(0xffffffffu, acc);
  if ((threadIdx.x & 31) == 0) atomicXor(sink, acc);
}

}  // namespace

int launch_l2_read_probe(const void* buf, size_t bytes, int reps, unsigned* sink,
                         cudaStream_t stream) {
  const int grid = 4 * num_sms();
  l2_read_kernel<<<grid, kProbeThreads, 0, stream>>>(static_cast<const uint4*>(buf),
                                                     static_cast<long long>(bytes / 16), reps, sink);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "l2_read_probe launch");
  return SBA_OK;
}

}  // namespace sba
