// Internal interface between the C-ABI layer and the CUDA kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <cstdint>

namespace xs {

constexpr int MAX_PTRS = 16;              // == XS_MAX_P
// Values a kernel writes to the device error word (the first one wins).
constexpr int XS_DEVICE_TIMEOUT_CODE = 1; // a bounded wait expired; the launch was abandoned
constexpr int XS_DEVICE_BOUNDS_CODE = 3;  // a per-piece index check failed; the access was skipped
// Where the first device error of a launch happened (see report_error).
struct DeviceErrorInfo {
    int code;       // XS_DEVICE_*_CODE
    int cta;        // blockIdx.x
    int warp;       // threadIdx.x / 32
    int lane;
    int site;       // waits: shared-memory address of the mbarrier (split-tile flags: 0x40000 + slot);
                    // index checks: 1 packed-sequence table entry, 2 destination shard
    int detail[3];  // waits: phase parity, piece index, key block; index checks: the values checked
};

// Division by a launch-constant divisor d >= 1 without a divide instruction, for
// dividends 0 <= n < 2^31 (round-up method of division by invariant integers):
// with l = ceil(log2 d) and m = ceil(2^(31+l) / d) (< 2^32), floor(n / d) =
// floor(n * m / 2^(31+l)).  The error n*(m*d - 2^(31+l)) / (d * 2^(31+l)) of the
// product is below 2^-l <= 1/d, too small to reach the next integer.
struct FastDiv {
    unsigned m;
    unsigned shift;   // 31 + l
    int d;
};

inline FastDiv make_fastdiv(int d) {
    FastDiv f{};
    unsigned l = 0;
    while ((1ull << l) < static_cast<unsigned long long>(d)) ++l;
    f.shift = 31 + l;
    f.m = static_cast<unsigned>(((1ull << f.shift) + static_cast<unsigned long long>(d) - 1) /
                                static_cast<unsigned long long>(d));
    f.d = d;
    return f;
}

__host__ __device__ __forceinline__ int fdiv(int n, const FastDiv& f) {
    return static_cast<int>((static_cast<unsigned long long>(static_cast<unsigned>(n)) * f.m) >> f.shift);
}
// n / d and n % d
__host__ __device__ __forceinline__ void fdivmod(int n, const FastDiv& f, int& q, int& r) {
    q = fdiv(n, f);
    r = n - q * f.d;
}

// Where each output row (b, s, h) of the attention kernel goes:
//   p = s / Sl + h / Hl,  ptr[p] + ((b * Sl + s % Sl) * Hl + h % Hl) * D
// contiguous:   Sl = S,   Hl = H,   one pointer
// A2A shards:   Sl = S/P, Hl = H,   P pointers (sequence shards)
// head shards:  Sl = S,   Hl = H/P, P pointers (Ulysses head shards)
struct EpiParams {
    void* ptr[MAX_PTRS];
    int Sl;
    int Hl;
    int row0;   // output row of the launch's row 0 (one sequence of a packed batch; else 0)
    FastDiv fd_Sl, fd_Hl;   // set by the launch functions from Sl and Hl
};

// Balanced ("stream-K") schedule of the tiles left over after the whole waves.
// Tiles [0, dp_tiles) run whole, tile = cta + w * grid.  The key-block
// iterations of tiles [dp_tiles, units) (sk_iters = their count * n_kv,
// tile-major) are cut into sk_ctas contiguous ranges, range i for CTA i; a range
// may start or end inside a tile, and a tile may be cut among several CTAs.
// Every piece that starts inside a tile (a "part") writes its unnormalised
// partial result to slot `its CTA index` of the workspace and publishes it with
// the launch's epoch in one flag per softmax warp; the piece that starts the
// tile (the "head", done last by its CTA) waits for the parts of the CTAs after
// it whose ranges start inside the tile and merges them.  sk_iters == 0: no split.
// The epoch lives in the workspace, not in the launch arguments: launch_count[0]
// counts the launches that have finished on this workspace, and a launch uses
// launch_count[0] + 1 (0 skipped), read by every CTA at its start; the last CTA
// to finish (counted in launch_count[1]) advances it.  A replayed launch
// therefore never takes flags left by an earlier one for its own.
struct SplitParams {
    int dp_tiles;
    int sk_ctas;
    long long sk_iters;
    float* part_o;         // [grid][128][D] fp32 partial numerators
    float2* part_ml;       // [grid][128] (running max in log2 units, row sum)
    unsigned* part_flag;   // [grid][8] epoch of the publishing softmax warp
    unsigned* launch_count;  // [2]: finished launches, CTAs finished in this launch
};

struct AttnArgs {
    int B, S, H;
    int n_kv;       // ceil(S / 128) key blocks
    int n_qt;       // ceil(S / 128) query tiles per (b, h)
    int units;      // B * H * n_qt tiles
    float c;        // scale * log2(e)
    EpiParams epi;
    unsigned long long timeout_ns;  // limit for every wait inside the kernel
    SplitParams sp;
    int in_Sl;      // inputs as sequence shards: rows per shard (a multiple of 128);
                    // 0: one [B, S, H, D] tensor per operand
    unsigned in_magic;  // shard lookup without division: shard = umulhi(2 * (row / 128), in_magic)
    int in_shift;       //   >> in_shift (see pick_map); set with in_Sl
    int causal_head_major;  // causal tile order: 0 longest first with the B*H tiles of one
                            // query tile side by side; 1 head-major (a head's query tiles
                            // side by side, longest first within the head)
    int h0;         // the launch's head h is head h0 + h of the input tensor maps ...
    int h0_out;     // ... and head h0_out + h of the output layout (both 0: all heads;
                    // a head group of larger tensors: both the group's first head; a
                    // Ulysses rank r with H/P local heads: 0 and r * H/P)
    // divisors of the tile decode, set by the launch functions (callers leave them)
    FastDiv fd_nqt, fd_H, fd_BH, fd_grid;
};

// Packed variable-length sequences (B = 1, S = T rows in total): the sequence
// boundaries and the list of query tiles, built on the host and passed by value
// in the launch's parameter space (about 20 KB), so a call needs no device memory.
constexpr int MAX_VARLEN_SEQS = 1024;
constexpr int MAX_VARLEN_TILES = 4096;
struct VarlenTable {
    int n_seqs;
    int n_tiles;                          // entries of `tile` (units = n_tiles * H)
    int cu[MAX_VARLEN_SEQS + 1];          // packed row of each sequence start; cu[n_seqs] = T
    unsigned tile[MAX_VARLEN_TILES];      // (sequence << 16) | query tile, longest first
};

// Tensor maps of Q, K, V given as P sequence shards [B, S/P, H, D] each (the
// layout every Ulysses rank holds before the pre-attention All-to-All).
struct ShardMaps {
    CUtensorMap q[MAX_PTRS];
    CUtensorMap k[MAX_PTRS];
    CUtensorMap v[MAX_PTRS];
};

template <int D>
int attn_smem_bytes();

// cooperative: launch with the co-residency guarantee (needed whenever
// args.sp.sk_iters != 0, because CTAs then wait for each other).
template <int D>
cudaError_t launch_attn(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        const AttnArgs& args, int grid, bool cooperative, cudaStream_t stream);

// Causal attention (row s attends to keys 0 .. s): tiles run whole, longest
// first (args.sp is ignored; no workspace, no co-residency needed).
template <int D>
cudaError_t launch_attn_causal(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const AttnArgs& args, int grid, cudaStream_t stream);

// Packed variable-length sequences, bidirectional: tiles of vt run whole in the
// listed order; args.B = 1, args.S = T, args.units = vt.n_tiles * H.  (The
// causal packed form runs as one launch_attn_causal per sequence, with
// args.epi.row0 = the sequence's first packed row.)
template <int D>
cudaError_t launch_attn_varlen(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const AttnArgs& args, const VarlenTable& vt, int grid, cudaStream_t stream);

// The same kernel reading Q, K, V from P sequence shards (args.in_Sl = S / P).
template <int D>
cudaError_t launch_attn_sharded(const ShardMaps& maps, int P, const AttnArgs& args, int grid, bool cooperative,
                                cudaStream_t stream);

// Reads and clears the device error word, the record of the first error and the
// flag of abort drains that gave up (copies or MMAs possibly still in flight when
// a CTA exited).
cudaError_t read_and_clear_device_error(int* value, DeviceErrorInfo* info, int* drain_failed);

#ifdef XS_TILE_SPANS
// Instrumented build only: where the per-tile timestamps go (device buffer of
// ctas * (per_cta * 6 + 32 * 10) words; NULL stops recording).
cudaError_t set_tile_spans(unsigned long long* buf, int ctas, int per_cta);
#endif

struct RelayoutArgs {
    const void* heads[MAX_PTRS];
    void* out[MAX_PTRS];
    int B, S, H, D, P;
};

cudaError_t launch_relayout(const RelayoutArgs& a, int num_sms, cudaStream_t stream);

// The inverse exchange (the pre-attention All-to-All): a.heads[p] are read as the
// sequence shards [B, S/P, H, D], a.out[r] are written as the head shards
// [B, S, H/P, D].
cudaError_t launch_relayout_inverse(const RelayoutArgs& a, int num_sms, cudaStream_t stream);

// Burst-Gap microbenchmark of the store path (csrc/burst_gap.cu).
struct BurstGapArgs {
    void* dst;                   // destination buffer, 16-byte aligned
    int64_t chunks_per_producer; // 16-byte chunks each producer stores per burst (V / K / 16)
    int64_t windows;             // dst holds this many producer windows (rotated through)
    int bursts;
    long long lead_ns;           // spin before the first burst
    long long gap_ns;            // producer-side gap after each burst
    long long* issue_ns;         // device [bursts][producers]: issue time of each burst
};

cudaError_t launch_burst_gap(const BurstGapArgs& a, int producers, cudaStream_t stream);

}  // namespace xs
