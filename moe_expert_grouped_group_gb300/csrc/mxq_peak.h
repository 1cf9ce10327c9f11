// The MXFP8 tensor-pipe ceiling probe (mxq_peak.cu): a measurement utility
// beside the MXFP8 path, exported as mxq_probe_mma_stream.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace mxq {
// One CTA per SM issues mmas_per_sm block-scaled 128x256x32 MMAs from
// resident shared memory; a bounded-wait timeout sets MXQ_STATUS_WAIT_TIMEOUT.
cudaError_t run_mma_stream(int64_t mmas_per_sm, int32_t* status, cudaStream_t s);
}  // namespace mxq
