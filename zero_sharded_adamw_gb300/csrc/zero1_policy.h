// zero1_policy.h -- host-side choices about how a launch runs (never what
// it computes), shared by the C-ABI host code (zero1_host.cu,
// zero1_noalloc.cu).  Not installed.
#pragma once

namespace zero1 {

// The device-wide rate (GB/s) that sets the update kernel's load period, or
// 0 for free-running loads.  option: zero1_options.load_phase_gbs (0 = the
// built-in rule, > 0 = this rate, < 0 = never).  reread: the launch re-reads
// the gradients (W <= 2 without a scratch) instead of reading the fp32
// scratch.  Phasing needs every SM in the grid (a period shared by fewer
// CTAs, or by CTAs that share the device with other work, is not the one
// measured; callers whose launch runs beside other work pass no rate) and
// fp32 moments.
//
// Built-in rule, from sweeps on GB300 (update-kernel time against
// free-running loads):
//  - scratch path: below W = 16 the loads are too large a share of the
//    bytes (16 against 12 + 2W stored per parameter) and every period tried
//    was slower; at 16 <= W < 20 a period of half a tile's time (14000
//    GB/s) was 3.7% faster and a whole tile's barely faster; from W = 20 a
//    whole tile's time at 7000 GB/s was 4-13% faster and within 2.5% of the
//    best rate on every box measured;
//  - re-read path (W = 2: 16 bytes in, 16 out per parameter): a whole
//    tile's period was 9-18% slower, but a period of about 0.4 of a tile
//    (17500 GB/s) was 1.2% faster, and every rate from 14000 to 21000 GB/s
//    faster than free-running, in two separate runs.
inline double load_rate_gbs(double option, int world, bool moments_bf16, bool reread, int grid, int num_sms)
{
    if (option < 0.0 || moments_bf16 || num_sms <= 0 || grid < num_sms) return 0.0;
    if (option > 0.0) return option;
    if (reread) return 17500.0;
    if (world < 16) return 0.0;
    return world < 20 ? 14000.0 : 7000.0;
}

}  // namespace zero1
