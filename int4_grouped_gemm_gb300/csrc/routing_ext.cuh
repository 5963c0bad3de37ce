// Routing-table launch that also clears a buffer on the side (declared apart
// from the other launches of kernels.cuh).
#pragma once

#include "kernels.cuh"

namespace moe {

// launch_routing_tables from the router's partial sums, with the top-k kernel
// zeroing clear[0 .. clear_elems) (fp32, 16-byte aligned, clear_elems % 4 == 0)
// while it waits on its loads.
cudaError_t launch_routing_tables_clearing(const float *logits_part, int ld, const float *bias, int T, int E, int k,
                                           int has_shared, const RouteOpts &opts, const RoutingBufs &rb, float *clear,
                                           int64_t clear_elems, cudaStream_t s);

}  // namespace moe
