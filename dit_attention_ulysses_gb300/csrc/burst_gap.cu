// Burst-Gap microbenchmark of the store path (single GPU).
//
// X-Stage (arXiv 2607.23264), gist.science technical summary, "Methodology:
// The X-Stage Abstraction and Burst-Gap Model": K producers each issue a burst
// of stores, the aggregate burst volume being V, then compute for a gap G before
// the next burst; the sender-visible issue time of a burst is
//     T_iss(G; K, V) = max(T0_iss(K, V), V / R - G)
// with T0_iss the backpressure-free issue time, R the effective drain rate of
// the path and Q its outstanding capacity.  On the pages the stores are remote
// (NVLink); here the path is the local one of the fused epilogue: SM -> L2 ->
// HBM, into a destination buffer larger than L2 so that sustained bursts reach
// HBM.
//
// One CTA per producer (the dynamic shared memory request keeps one CTA per
// SM).  After a lead-in spin (the path drains while the SMs stay busy), per
// burst r, CTA c stores its V/K bytes as 16-byte chunks into its own
// contiguous window of the destination (windows rotate through the buffer); all
// threads of the CTA issue, then thread 0 records the issue time (from before
// the first store to after the last thread has issued its last store:
// %globaltimer around two CTA barriers), spins for the gap, and the next burst
// starts.  Every loop is bounded by its arguments (checked on the host).
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace xs {
namespace {

constexpr int BG_THREADS = 256;
constexpr int BG_SMEM = 120 * 1024;   // one CTA per SM

// The 16-byte chunk stored at index i of the window of burst r, CTA c.
__device__ __forceinline__ uint4 bg_chunk(int r, int c, int64_t i) {
    const uint32_t lo = static_cast<uint32_t>(i);
    return make_uint4(lo, static_cast<uint32_t>(r), static_cast<uint32_t>(c), lo ^ 0x9E3779B9u);
}

__global__ void __launch_bounds__(BG_THREADS, 1) burst_gap_kernel(const BurstGapArgs a) {
    const int c = blockIdx.x;
    uint4* dst = reinterpret_cast<uint4*>(a.dst);
    if (threadIdx.x == 0) {   // a lead-in gap: the path drains while the SM stays busy
        const uint64_t t = globaltimer_ns();
        while (globaltimer_ns() - t < static_cast<uint64_t>(a.lead_ns)) {
        }
    }
    for (int r = 0; r < a.bursts; ++r) {
        // window of (r, c): windows laid end to end, wrapping around the buffer
        const int64_t w = (static_cast<int64_t>(r) * gridDim.x + c) % a.windows;
        uint4* win = dst + w * a.chunks_per_producer;
        __syncthreads();
        uint64_t t0 = 0;
        if (threadIdx.x == 0) t0 = globaltimer_ns();
        for (int64_t i = threadIdx.x; i < a.chunks_per_producer; i += BG_THREADS) win[i] = bg_chunk(r, c, i);
        __syncthreads();
        if (threadIdx.x == 0) {
            const uint64_t t1 = globaltimer_ns();
            a.issue_ns[static_cast<int64_t>(r) * gridDim.x + c] = static_cast<long long>(t1 - t0);
            // the producer-side gap: a bounded spin on the clock
            while (globaltimer_ns() - t1 < static_cast<uint64_t>(a.gap_ns)) {
            }
        }
    }
}

}  // namespace

cudaError_t launch_burst_gap(const BurstGapArgs& a, int producers, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(burst_gap_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, BG_SMEM);
    if (e != cudaSuccess) return e;
    burst_gap_kernel<<<producers, BG_THREADS, BG_SMEM, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace xs
