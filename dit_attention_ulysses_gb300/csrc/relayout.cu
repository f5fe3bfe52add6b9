// The separate Ulysses All-to-All re-layouts (single GPU): after attention,
// head shards [B, S, H/P, D] of the P virtual ranks -> sequence shards
// [B, S/P, H, D]; before attention, the inverse.
//
// X-Stage (arXiv 2607.23264), abstract: "serial execution" is attention followed
// by a separate All-to-All; this kernel is that separate step, used as the
// unfused baseline that the fused store is measured against.
//
// Pure data movement: every thread copies 16-byte chunks (8 bf16) with
// read-only vector loads and vector stores, walking the OUTPUT linearly so both
// sides stay coalesced (a destination row of D elements comes from one source
// row of D elements).  Grid-stride loop; the grid is a multiple of the SM count.
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace xs {
namespace {

struct alignas(16) Chunk {
    uint4 v;
};

__global__ void __launch_bounds__(256) relayout_kernel(const RelayoutArgs a) {
    const int64_t chunks_per_row = a.D / 8;
    const int64_t Sl = a.S / a.P;
    const int64_t Hl = a.H / a.P;
    const int64_t per_shard = static_cast<int64_t>(a.B) * Sl * a.H * chunks_per_row;
    const int64_t total = per_shard * a.P;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        // output coordinates (p, b, s', h, chunk)
        int64_t rem = i;
        const int64_t dc = rem % chunks_per_row;
        rem /= chunks_per_row;
        const int64_t h = rem % a.H;
        rem /= a.H;
        const int64_t s2 = rem % Sl;
        rem /= Sl;
        const int64_t b = rem % a.B;
        const int64_t p = rem / a.B;
        // source: rank r = h / Hl holds local head j = h % Hl for all s
        const int64_t r = h / Hl;
        const int64_t j = h % Hl;
        const int64_t s = p * Sl + s2;
        const uint4* src = reinterpret_cast<const uint4*>(a.heads[r]) + ((b * a.S + s) * Hl + j) * chunks_per_row + dc;
        uint4* dst = reinterpret_cast<uint4*>(a.out[p]) + ((b * Sl + s2) * a.H + h) * chunks_per_row + dc;
        *dst = __ldg(src);
    }
}

// The pre-attention exchange: sequence shards [B, S/P, H, D] (read from
// a.heads[p]) -> head shards [B, S, H/P, D] (written to a.out[r]):
//     heads[r][b, s, j, :] = seq[s / Sl][b, s % Sl, r*Hl + j, :]
// Again 16-byte chunks, walking the output linearly.
__global__ void __launch_bounds__(256) relayout_inverse_kernel(const RelayoutArgs a) {
    const int64_t chunks_per_row = a.D / 8;
    const int64_t Sl = a.S / a.P;
    const int64_t Hl = a.H / a.P;
    const int64_t per_rank = static_cast<int64_t>(a.B) * a.S * Hl * chunks_per_row;
    const int64_t total = per_rank * a.P;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        // output coordinates (r, b, s, j, chunk)
        int64_t rem = i;
        const int64_t dc = rem % chunks_per_row;
        rem /= chunks_per_row;
        const int64_t j = rem % Hl;
        rem /= Hl;
        const int64_t s = rem % a.S;
        rem /= a.S;
        const int64_t b = rem % a.B;
        const int64_t r = rem / a.B;
        const int64_t p = s / Sl;
        const int64_t s2 = s - p * Sl;
        const int64_t h = r * Hl + j;
        const uint4* src = reinterpret_cast<const uint4*>(a.heads[p]) + ((b * Sl + s2) * a.H + h) * chunks_per_row + dc;
        uint4* dst = reinterpret_cast<uint4*>(a.out[r]) + ((b * a.S + s) * Hl + j) * chunks_per_row + dc;
        *dst = __ldg(src);
    }
}

}  // namespace

cudaError_t launch_relayout_inverse(const RelayoutArgs& a, int num_sms, cudaStream_t stream) {
    const int64_t total = static_cast<int64_t>(a.B) * a.S * a.H * (a.D / 8);
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    relayout_inverse_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_relayout(const RelayoutArgs& a, int num_sms, cudaStream_t stream) {
    const int64_t total = static_cast<int64_t>(a.B) * a.S * a.H * (a.D / 8);
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;  // 8 resident blocks of 256 per SM
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    relayout_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace xs
