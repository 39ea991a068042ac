// Query input of the decode step when the queries sit in page-locked host memory
// (okvq_decode_host).
//
// The decode kernel stages each segment's queries from device memory by bulk copy,
// and it is launched as a programmatic dependent of the kernel before it on the
// stream (the previous step's merge), so that its prologue runs while that merge
// finishes. An upload on another stream would end that overlap: the decode would
// have to wait on an event. So page-locked queries come in through this kernel,
// launched on the decode's own stream right before the decode, itself a
// programmatic dependent of the previous kernel:
//  - it reads the host words through their mapped device address (zero-copy)
//    before griddepcontrol.wait: the host wrote them before the launch, and no
//    kernel writes them;
//  - it writes the device staging buffer after the wait, when every earlier kernel
//    on the stream, the decode that last read that buffer included, has completed.
// The decode then waits (griddepcontrol.wait) for this kernel alone.

#include "okvq_hostio.h"

#include <cstdint>

namespace okvq {
namespace {

constexpr int SQ_THREADS = 256;
constexpr int SQ_PER = 4;   // 16-byte words per thread

__global__ void __launch_bounds__(SQ_THREADS) stage_queries_kernel(const uint4 *src, uint4 *dst, long long n16) {
  const long long base = (long long)blockIdx.x * (SQ_THREADS * SQ_PER) + threadIdx.x;
  uint4 v[SQ_PER];
#pragma unroll
  for (int k = 0; k < SQ_PER; ++k) {
    const long long i = base + (long long)k * SQ_THREADS;
    if (i < n16) v[k] = src[i];
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
#pragma unroll
  for (int k = 0; k < SQ_PER; ++k) {
    const long long i = base + (long long)k * SQ_THREADS;
    if (i < n16) dst[i] = v[k];
  }
}

}  // namespace

cudaError_t launch_stage_queries(const void *src, void *dst, long long n16, cudaStream_t s) {
  if (n16 <= 0) return cudaSuccess;
  const long long per_cta = (long long)SQ_THREADS * SQ_PER;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((n16 + per_cta - 1) / per_cta));
  cfg.blockDim = dim3(SQ_THREADS);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, stage_queries_kernel, static_cast<const uint4 *>(src), static_cast<uint4 *>(dst),
                            n16);
}

}  // namespace okvq
