// Query input of okvq_decode_host from page-locked host memory (okvq_hostio.cu).
#pragma once

#include <cuda_runtime.h>

namespace okvq {

// Copies n16 16-byte words from `src` (the device address of page-locked, mapped
// host memory, 16-byte aligned) to `dst` (device memory) on stream s, launched as a
// programmatic dependent of the previous kernel on s: the host words are read
// before griddepcontrol.wait, `dst` is written after it.
cudaError_t launch_stage_queries(const void *src, void *dst, long long n16, cudaStream_t s);

}  // namespace okvq
