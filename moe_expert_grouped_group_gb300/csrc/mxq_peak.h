// Utilities beside the MXFP8 path (mxq_peak.cu): the tensor-pipe ceiling
// probe (mxq_probe_mma_stream) and the bounded-wait self-test
// (mxq_selftest_wait_timeout).
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace mxq {
// One CTA per SM issues mmas_per_sm block-scaled 128x256x32 MMAs from
// resident shared memory (zeros, or pseudo-random E4M3 with unit scales when
// random != 0); a bounded-wait timeout sets MXQ_STATUS_WAIT_TIMEOUT.
cudaError_t run_mma_stream(int64_t mmas_per_sm, int random, int32_t* status, cudaStream_t s);
// One CTA waits limit_ns on an mbarrier nothing arrives on, then reports
// MXQ_STATUS_WAIT_TIMEOUT in *status.
cudaError_t run_wait_timeout(int64_t limit_ns, int32_t* status, cudaStream_t s);
}  // namespace mxq
