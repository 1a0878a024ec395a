// copy: a plain device-to-device byte copy used as the measured HBM roofline.
// Each thread moves four 16-byte vectors per trip (grid-stride), so a launch
// reads and writes every byte exactly once; the tail below 16 bytes is copied
// bytewise.  Both pointers must be 16-byte aligned.
#include "common.cuh"
#include "kernels.h"

namespace gbf {
namespace {

constexpr int kCopyBlock = 256;
constexpr int kCopyUnroll = 4;

__global__ void __launch_bounds__(kCopyBlock) copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                          int64_t nvec, const uint8_t* __restrict__ tail_src,
                                                          uint8_t* __restrict__ tail_dst, int tail) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kCopyBlock;
  int64_t i = static_cast<int64_t>(blockIdx.x) * kCopyBlock + threadIdx.x;
  for (; i + (kCopyUnroll - 1) * stride < nvec; i += kCopyUnroll * stride) {
    uint4 v[kCopyUnroll];
#pragma unroll
    for (int k = 0; k < kCopyUnroll; ++k) v[k] = ld_stream(src + i + k * stride);
#pragma unroll
    for (int k = 0; k < kCopyUnroll; ++k) dst[i + k * stride] = v[k];
  }
  for (; i < nvec; i += stride) dst[i] = ld_stream(src + i);
  if (blockIdx.x == 0 && threadIdx.x < tail) tail_dst[threadIdx.x] = tail_src[threadIdx.x];
}

}  // namespace

cudaError_t launch_copy(const void* src, void* dst, int64_t bytes, cudaStream_t stream) {
  if (bytes == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t nvec = bytes / 16;
  const int tail = static_cast<int>(bytes - nvec * 16);
  int64_t want = (nvec + kCopyBlock * kCopyUnroll - 1) / (kCopyBlock * kCopyUnroll);
  const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 148) * 8;
  if (want > cap) want = cap;
  if (want < 1) want = 1;
  copy_kernel<<<static_cast<unsigned>(want), kCopyBlock, 0, stream>>>(
      static_cast<const uint4*>(src), static_cast<uint4*>(dst), nvec,
      static_cast<const uint8_t*>(src) + nvec * 16, static_cast<uint8_t*>(dst) + nvec * 16, tail);
  return cudaGetLastError();
}

}  // namespace gbf
