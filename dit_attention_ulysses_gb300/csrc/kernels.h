// Internal interface between the C-ABI layer and the CUDA kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <cstdint>

namespace xs {

constexpr int MAX_PTRS = 16;              // == XS_MAX_P
constexpr int XS_DEVICE_TIMEOUT_CODE = 1; // value a kernel writes to the device error word

// Where each output row (b, s, h) of the attention kernel goes:
//   p = s / Sl + h / Hl,  ptr[p] + ((b * Sl + s % Sl) * Hl + h % Hl) * D
// contiguous:   Sl = S,   Hl = H,   one pointer
// A2A shards:   Sl = S/P, Hl = H,   P pointers (sequence shards)
// head shards:  Sl = S,   Hl = H/P, P pointers (Ulysses head shards)
struct EpiParams {
    void* ptr[MAX_PTRS];
    int Sl;
    int Hl;
};

struct AttnArgs {
    int B, S, H;
    int n_kv;       // ceil(S / 128) key blocks
    int n_qt;       // ceil(S / 128) query tiles (work units) per (b, h)
    int units;      // B * H * n_qt
    float c;        // scale * log2(e)
    EpiParams epi;
    unsigned long long timeout_ns;  // limit for every wait inside the kernel
};

template <int D>
int attn_smem_bytes();

template <int D>
cudaError_t launch_attn(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        const AttnArgs& args, int grid, cudaStream_t stream);

cudaError_t read_and_clear_device_error(int* value);

struct RelayoutArgs {
    const void* heads[MAX_PTRS];
    void* out[MAX_PTRS];
    int B, S, H, D, P;
};

cudaError_t launch_relayout(const RelayoutArgs& a, int num_sms, cudaStream_t stream);

}  // namespace xs
