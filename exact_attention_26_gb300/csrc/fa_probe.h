// Unit-rate and read-bandwidth probes (fa_probe.cu), behind fa_probe_unit_rates and
// fa_probe_read_bandwidth.
#pragma once

#include <cuda_runtime.h>

namespace fa {

// Wait site recorded by the probes' bounded MMA completion waits (after the
// attention kernels' sites).
constexpr int SITE_PROBE = 31;

// Runs the N = 256 MMA, N = 64 MMA and ex2 probes (one CTA per SM each),
// synchronises `stream` and writes the median per-SM rates (FLOP, FLOP, ex2 per SM
// clock) to rates[3].
int run_unit_probes(int num_sms, int iters, int *status, cudaStream_t stream, double *rates);

// Times `iters` streaming reads of `bytes` (a multiple of 16) at `buf` after one
// untimed read, CUDA events on `stream`; writes the read rate in GB/s.
int run_read_probe(int num_sms, const void *buf, size_t bytes, int iters, cudaStream_t stream,
                   double *gbs);

}  // namespace fa
