// Fused attention + post-attention Ulysses All-to-All store, sm_103a: the
// bidirectional kernel (one [B, S, H, D] tensor per operand, or the P sequence
// shards of the Ulysses ranks), the causal kernel, and the packed-sequence
// kernel (bidirectional; the causal packed form runs as one causal launch per
// sequence, with the output row offset EpiParams::row0).
//
// X-Stage (arXiv 2607.23264), abstract and the gist.science technical summary,
// "Key Contributions" item 3 (FlashAttention-A2A piggybacking): the role that
// owns an output tile stores it straight to the rank owning the tile's sequence
// block and immediately resumes the next tile's Q-loop; no dedicated
// communication warp and no separate All-to-All kernel.  On one GPU the ranks are
// P device buffers, so the "remote store" is a 16-byte vector store into the
// owner's [B, S/P, H, D] shard.
//
// Kernel organisation (one persistent CTA per SM, 12 warps; warp w runs on SM
// sub-partition w % 4):
//   warps 0-7  softmax + epilogue of the current 128-row Q tile; two threads per
//              row, both in one warp: warp w owns the 16 rows 32*(w%4) + 16*(w/4)
//              .. +15 (half of its TMEM lane quarter); lane i takes key columns
//              64*(i/16) .. +63 of row i%16 of every score block
//   warp  8    idle (keeps the three single-thread roles on three different
//              sub-partitions without changing the register budget: at most
//              three warps per sub-partition either way)
//   warp  9    issuer of the S = Q K^T MMAs (one lane) and TMEM owner
//   warp 10    issuer of the O += P V MMAs (one lane)
//   warp 11    TMA producer (one lane): Q tile of each piece of work, then the
//              K/V ring in consumption order K0, K1, V0, K2, V1, K3, ...
//              (D = 128: one Q buffer, reloaded as soon as the piece's last S MMA
//              has read it, the next one prefetched into L2 meanwhile, and 4 ring
//              stages of 32 KB; D = 64: two Q buffers and 10 stages of 16 KB)
// The tcgen05 issue queue is shallow, so any control work an issuing thread
// does between MMAs (waits, commits) leaves the tensor core idle; with two
// issuers, one thread's control work overlaps the other thread's MMAs.  The
// single-thread roles share their sub-partitions with softmax warps, so their
// instruction latency matters: sharing one sub-partition between two of them
// measured 1-2 % slower.
// A tile is (b, h, 128 query rows), numbered head-major so that the CTAs running
// at the same time share K/V through L2.  Q, K, V come from one [B,S,H,D]
// tensor each, or from the P sequence shards of the Ulysses ranks (one TMA
// tensor map per shard: the pre-attention exchange fused into the loads).
//
// TMEM (512 columns x 128 lanes, fp32):
//   [  0,128) S buffer 0    [128,256) S buffer 1    [256,384) S buffer 2
//   [384,384+D) O accumulator
// Block g's scores go to S buffer g % 3; once the softmax has read them it writes
// P(g) (bf16, two per column) over the buffer's first 64 columns, where the PV
// MMA reads it.  S(g+3) overwrites the buffer only after PV(g) has completed,
// and that wait is the S issuer's, not the softmax's: the softmax never waits
// for a PV except in the rare O rescale (PV(g-1)).  With three buffers the S
// MMAs run up to three blocks ahead, and the tensor core computes S(g+1),
// S(g+2) and PV(g-1) while the softmax works on block g.
// Softmax (base 2, c = scale*log2(e) folded into one FMA, MUFU ex2):
//   each thread takes the max of its 64 scores; the two threads of a row are
//   lanes i and i + 16 of one warp (TMEM 16x32bx2 accesses) and combine them with
//   one shuffle;
//   lazy rescale: the running max moves (and O, l are multiplied by
//   2^(m_run - m_new)) only when the block max exceeds it by more than 8;
//   p = 2^(s*c - m) -> bf16 -> TMEM, over the S buffer; l accumulates the fp32 p.
// Epilogue (the fused A2A): after the last PV each thread normalises its half of
// the O row by 1/l and stores it with 16-byte st.global.v4 into the destination
// row of the owning shard, then goes on to the next work unit.
//
// Every wait is bounded by a time limit; on expiry the kernel records
// XS_ERR_DEVICE_TIMEOUT in the device error word, raises a CTA-wide abort flag,
// lets each role drain what it has in flight (again bounded), frees TMEM and
// returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace xs {

__device__ int g_device_error = 0;
__device__ DeviceErrorInfo g_error_info;
__device__ int g_drain_failed = 0;

// Per-tile timestamps (a build with XS_TILE_SPANS only; the library's normal
// build compiles the stamps to nothing).  Warp 0, lane 0 of the softmax records,
// for the k-th piece of work of its CTA, SPAN_WORDS words at
// g_spans[(cta * g_spans_per_cta + k) * SPAN_WORDS]:
//   0 %globaltimer when the piece's first scores are seen   1 clock64 then
//   2 clock64 when the piece's last P is written            3 clock64 when its last PV is done
//   4 clock64 after the epilogue's stores are issued        5 (key blocks << 32) | piece kind
// (clock64 is the SM's cycle counter: differences within one CTA are cycles).
// After those words, for the first piece of each CTA and its key blocks
// PHASE_J0 .. PHASE_J0 + PHASE_BLOCKS - 1 (past the pipeline fill of the launch),
// PHASE_WORDS clock64 stamps per block (see phase_stamp's callers): the
// softmax's steps (warp 0, lane 0), the time each softmax warp signals its P,
// the MMA issuers' waits and issue times and the producer's load issue times.
// Last, EPI_WORDS clock64 stamps per CTA of warp 0's epilogue of its first
// piece (see epi_stamp's callers).
#ifdef XS_TILE_SPANS
constexpr int SPAN_WORDS = 6;
constexpr int PHASE_J0 = 8;
constexpr int PHASE_BLOCKS = 32;
constexpr int PHASE_WORDS = 24;
constexpr int EPI_WORDS = 8;
__device__ unsigned long long* g_spans = nullptr;
__device__ int g_spans_ctas = 0;      // CTA slots of the buffer
__device__ int g_spans_per_cta = 0;   // piece slots per CTA
__device__ __forceinline__ void span_stamp(int k, int slot, unsigned long long v) {
    unsigned long long* s = g_spans;
    if (s != nullptr && k < g_spans_per_cta && static_cast<int>(blockIdx.x) < g_spans_ctas && threadIdx.x == 0)
        s[(static_cast<size_t>(blockIdx.x) * g_spans_per_cta + k) * SPAN_WORDS + slot] = v;
}
// The block-phase rows of piece k for a thread that stamps (nullptr when it does
// not): looked up once per piece, so that a stamp costs a clock read and a store.
__device__ __forceinline__ unsigned long long* phase_rows(int k, bool stamps) {
    unsigned long long* s = g_spans;
    if (s == nullptr || k != 0 || !stamps || static_cast<int>(blockIdx.x) >= g_spans_ctas) return nullptr;
    return s + static_cast<size_t>(g_spans_ctas) * g_spans_per_cta * SPAN_WORDS +
           static_cast<size_t>(blockIdx.x) * PHASE_BLOCKS * PHASE_WORDS;
}
// A block-phase stamp of key block j.
__device__ __forceinline__ void phase_stamp(unsigned long long* rows, int j, int slot) {
    if (rows != nullptr && static_cast<unsigned>(j - PHASE_J0) < static_cast<unsigned>(PHASE_BLOCKS))
        rows[(j - PHASE_J0) * PHASE_WORDS + slot] = static_cast<unsigned long long>(clock64());
}
// The epilogue stamps of piece k for a thread that stamps (nullptr when it does not).
__device__ __forceinline__ unsigned long long* epi_rows(int k, bool stamps) {
    unsigned long long* s = g_spans;
    if (s == nullptr || k != 0 || !stamps || static_cast<int>(blockIdx.x) >= g_spans_ctas) return nullptr;
    return s + static_cast<size_t>(g_spans_ctas) * (g_spans_per_cta * SPAN_WORDS + PHASE_BLOCKS * PHASE_WORDS) +
           static_cast<size_t>(blockIdx.x) * EPI_WORDS;
}
__device__ __forceinline__ void epi_stamp(unsigned long long* rows, int slot) {
    if (rows != nullptr) rows[slot] = static_cast<unsigned long long>(clock64());
}
__device__ __forceinline__ unsigned long long span_clock() { return static_cast<unsigned long long>(clock64()); }
#else
__device__ __forceinline__ void span_stamp(int, int, unsigned long long) {}
__device__ __forceinline__ unsigned long long* phase_rows(int, bool) { return nullptr; }
__device__ __forceinline__ void phase_stamp(unsigned long long*, int, int) {}
__device__ __forceinline__ unsigned long long* epi_rows(int, bool) { return nullptr; }
__device__ __forceinline__ void epi_stamp(unsigned long long*, int) {}
__device__ __forceinline__ unsigned long long span_clock() { return 0; }
#endif

// Records the first device error of the launch (later ones only find the word
// set).  Out of line: it runs at most once per launch and must not weigh on the
// register allocation of the loops that call it.
__device__ __noinline__ void report_error(int code, int site, int d0, int d1, int d2) {
    if (atomicCAS(&g_device_error, 0, code) == 0) {
        DeviceErrorInfo r;
        r.code = code;
        r.cta = static_cast<int>(blockIdx.x);
        r.warp = static_cast<int>(threadIdx.x >> 5);
        r.lane = static_cast<int>(threadIdx.x & 31u);
        r.site = site;
        r.detail[0] = d0;
        r.detail[1] = d1;
        r.detail[2] = d2;
        g_error_info = r;
        __threadfence();
    }
}

// Time since t0 has reached the limit.  Signed, so that a timer read that
// comes out below t0 counts as no time passed rather than as a huge one.
__device__ __forceinline__ bool expired(uint64_t t0, uint64_t limit_ns) {
    return static_cast<long long>(globaltimer_ns() - t0) >= static_cast<long long>(limit_ns);
}

namespace {

constexpr int BLOCK_M = 128;
constexpr int BLOCK_N = 128;
constexpr int NUM_THREADS = 384;
constexpr int NUM_SOFTMAX_WARPS = 8;
constexpr int WARP_TMA = 11;
constexpr int WARP_MMA_S = 9;
constexpr int WARP_MMA_PV = 10;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t S_COL = 0;     // + 128 * buffer; P(g) over the first 64 columns of buffer g % 3
constexpr int S_BUFS = 3;
constexpr uint32_t O_COL = 384;
constexpr int PANEL_BYTES = BLOCK_M * 128;  // 128 rows x 64 bf16
constexpr float RESCALE_THRESHOLD = 8.0f;   // log2 units
constexpr uint32_t WAIT_CHECK_EVERY = 16;   // probes between time-limit checks (a power of two)

template <int D>
struct Cfg {
    static constexpr int TILE_BYTES = BLOCK_M * D * 2;
    static constexpr int PANELS = D / 64;
    static constexpr int Q_BUFS = (D == 128) ? 1 : 2;
    static constexpr int KV_STAGES = (D == 128) ? 4 : 10;
    static constexpr int Q_OFF = 0;
    static constexpr int KV_OFF = Q_BUFS * TILE_BYTES;
    static constexpr int STAGE_OFF = KV_OFF + KV_STAGES * TILE_BYTES;  // epilogue staging, 2 KB per softmax warp
    static constexpr int STAGE_BYTES = NUM_SOFTMAX_WARPS * 2048;
    static constexpr int BAR_OFF = STAGE_OFF + STAGE_BYTES;
    // barrier indices
    static constexpr int B_Q_FULL = 0;                 // [2]  TMA -> MMA, per Q buffer
    static constexpr int B_Q_FREE = 2;                 // [2]  MMA -> TMA
    static constexpr int B_S_FULL = 4;                 // [3]  S MMA -> softmax, per S buffer
    static constexpr int B_P_FULL = 7;                 // [3]  softmax -> PV MMA (P written over the buffer)
    static constexpr int B_P_FREE = 10;                // [3]  PV MMA -> S MMA / rescale (PV done: buffer free)
    static constexpr int B_O_FINAL = 13;               // [1]  MMA -> epilogue
    static constexpr int B_O_FREE = 14;                // [1]  epilogue -> MMA
    static constexpr int B_DRAIN = 15;                 // [1]  both issuers
    static constexpr int B_KV_FULL = 16;               // [NS] TMA -> MMA
    static constexpr int B_KV_FREE = 16 + KV_STAGES;   // [NS] MMA -> TMA
    static constexpr int NUM_BARS = 16 + 2 * KV_STAGES;
    static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
    static constexpr int SMEM_BYTES = MISC_OFF + 16;
    static constexpr int SMEM_ALLOC = SMEM_BYTES + 1024;
};

// Bounded wait, executed by a whole warp; the result is warp-uniform.  The
// first probe is a non-blocking test; the further probes are mbarrier.try_wait
// without a time hint (the hardware's own short suspend limit: a waiting role
// resumes as soon as the phase completes, which measured 1-5 % faster per launch
// than a 200 us hint).  The abort flag and the time limit are looked at before
// the first try_wait's retry and then every WAIT_CHECK_EVERY probes: a
// %globaltimer read costs more than a probe, and a read between the phase's
// completion and the next probe delays the waiter by that much.  A limit of 0
// gives up after the first try_wait of the first wait that is not already over.  On expiry the wait records (barrier, parity, piece, block) as
// the launch's first error, unless one is recorded already.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t timeout_ns, int unit = -1, int blk = -1) {
    bool ok = mbar_test_wait(bar, parity);
    if (!__all_sync(0xffffffffu, ok)) {
        uint64_t t0 = 0;
        for (uint32_t n = 0; !ok; ++n) {
            ok = mbar_try_wait(bar, parity);
            if (ok || (n & (WAIT_CHECK_EVERY - 1)) != 0) continue;
            if (*abort_flag) break;
            if (n == 0) t0 = globaltimer_ns();
            if (expired(t0, timeout_ns)) {
                *abort_flag = 1;
                report_error(XS_DEVICE_TIMEOUT_CODE, static_cast<int>(bar), static_cast<int>(parity), unit, blk);
                break;
            }
        }
        ok = __all_sync(0xffffffffu, ok);
    }
    return ok;
}

// Suspend hint of the single-thread roles' probes (ns): a suspended thread is
// woken by the phase's completion, and while it sleeps it takes no issue slots
// from the softmax warps on its sub-partition (measured +1 ... +1.4 % at the long
// power-limited shapes, no change at the short ones, against hint-free probes).
constexpr uint32_t ROLE_WAIT_HINT_NS = 2000;

// The same bounded wait for a single thread (the issuing lanes of the producer
// and MMA roles), without warp votes.
__device__ __forceinline__ bool thread_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                            uint64_t timeout_ns, int unit = -1, int blk = -1) {
    if (mbar_test_wait(bar, parity)) return true;
    uint64_t t0 = 0;
    for (uint32_t n = 0;; ++n) {
        if (mbar_try_wait_sleep(bar, parity, ROLE_WAIT_HINT_NS)) return true;
        if ((n & (WAIT_CHECK_EVERY - 1)) != 0) continue;
        if (*abort_flag) return false;
        if (n == 0) t0 = globaltimer_ns();
        if (expired(t0, timeout_ns)) {
            *abort_flag = 1;
            report_error(XS_DEVICE_TIMEOUT_CODE, static_cast<int>(bar), static_cast<int>(parity), unit, blk);
            return false;
        }
    }
}

// Wait of the abort path for an asynchronous operation already issued (a TMA
// copy, the MMAs before a commit): bounded by `limit_ns`; if it gives up, the
// operation may still be in flight when the CTA frees its tensor memory and
// exits, so that is flagged for the host (XS_ERR_DEVICE_DRAIN), beside the
// error that caused the abort.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_test_wait(bar, parity)) return;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait_sleep(bar, parity, 200000u)) {
        if (expired(t0, limit_ns)) {
            atomicOr(&g_drain_failed, 1);
            return;
        }
    }
}

// Ring position of K(j) / V(j) within a unit of n key blocks (consumption order
// K0, K1, V0, K2, V1, K3, ..., V(n-3), K(n-1), V(n-2), V(n-1)).
__device__ __forceinline__ uint32_t ring_pos_k(int j) { return j < 2 ? j : 2 * j - 1; }
__device__ __forceinline__ uint32_t ring_pos_v(int j, int n) { return (j + 2 < n) ? 2 * j + 2 : n + j; }

// One arrival for a whole warp: every lane has finished its part (its own
// fences included) once __syncwarp returns; lane 0 then arrives.  Replaces 32
// arrivals on the same shared-memory word, which serialise.
__device__ __forceinline__ void warp_arrive(uint32_t bar) {
    __syncwarp();
    if (lane_id() == 0) mbar_arrive(bar);
}

__device__ __forceinline__ void decode_unit(int u, const AttnArgs& a, int& b, int& h, int& qt) {
    int bh;
    fdivmod(u, a.fd_nqt, bh, qt);
    fdivmod(bh, a.fd_H, b, h);
}

// One piece of work of a CTA: key blocks [k0, k0 + nb) of query tile (b, h, qt).
enum WorkKind { WORK_FULL = 0, WORK_HEAD = 1, WORK_PART = 2 };
struct Work {
    int b, h, qt;
    int k0, nb;
    int kind;   // WORK_FULL: the whole tile; WORK_HEAD: blocks [0, k) of a split
                // tile, merged with the parts of the following CTAs and stored;
                // WORK_PART: blocks [k0, k0 + nb), k0 > 0, of a split tile,
                // published as a partial result
    int t_sk;   // index of the tile among the split-scheduled tiles (-1: whole wave)
    int row0;   // VARLEN: packed row of the tile's sequence start (b = 0)
    int len;    // VARLEN: the sequence's length
};

// Start of CTA i's range of split-scheduled key-block iterations.
__device__ __forceinline__ long long sk_start(const AttnArgs& a, int i) {
    return a.sp.sk_iters * i / a.sp.sk_ctas;
}

// The idx-th piece of work of this CTA (every role walks the same sequence):
// first its whole tiles cta, cta + grid, ... below dp_tiles, then the pieces of
// its range [sk_start(cta), sk_start(cta + 1)) of the remaining tiles'
// key-block iterations (CTAs from sk_ctas on have none).  A range holds at most
// one part (its first piece, when it starts inside a tile) and at most one head
// (its last piece, when it ends inside a tile that it entered at block 0).
//
// CAUSAL: query tile qt needs key blocks 0 .. qt only, so tiles differ in
// length.  They run whole, longest first (query tiles in descending order, the
// B*H tiles of one query tile side by side), dealt out in waves of one tile per
// CTA in snake order: CTAs 0 .. G-1 in even waves, G-1 .. 0 in odd ones, so
// that the CTA given the longest tile of a wave gets the shortest of the next.
// The sequence of a CTA ends at the first index past the last tile, since the
// tile index grows with idx.  With a.causal_head_major the tiles go head by
// head instead (query tiles descending within a head): concurrent CTAs then
// share one head's keys and values in L2, at some cost in balance, which the
// host accepts only where it is small (long sequences).
//
// VARLEN: packed sequences (B = 1, S = their total length).  vt->tile lists the
// query tiles (sequence, query tile) longest first, dealt out in the same snake
// order.  CAUSAL: unit u is entry u / H for head u % H.  Otherwise every tile of
// a sequence has the same length, the list holds a sequence's tiles together
// (query tile 0 first), and the sequence's units [H * first, H * (first + nq))
// run head-major, the query tiles of one head side by side, so that the CTAs
// working at once share that head's keys and values in L2.  A tile of sequence
// i reads the key blocks of that sequence only: ceil(len_i / 128) of them, or
// (CAUSAL) qt + 1.
template <bool CAUSAL, bool VARLEN>
__device__ __forceinline__ bool get_work(const AttnArgs& a, const VarlenTable* vt, int idx, Work& w) {
    const int G = static_cast<int>(gridDim.x);
    const int i = static_cast<int>(blockIdx.x);
    if constexpr (VARLEN) {
        const long long u = static_cast<long long>(idx) * G + ((idx & 1) ? G - 1 - i : i);
        if (u >= a.units) return false;
        const int t = fdiv(static_cast<int>(u), a.fd_H);
        // index checks on the host-built table (every role takes the same exit)
        if (t >= vt->n_tiles) {
            report_error(XS_DEVICE_BOUNDS_CODE, 1, t, vt->n_tiles, idx);
            return false;
        }
        const unsigned e = vt->tile[t];
        const int seq = static_cast<int>(e >> 16);
        if (seq >= vt->n_seqs) {
            report_error(XS_DEVICE_BOUNDS_CODE, 1, t, static_cast<int>(e), idx);
            return false;
        }
        w.b = 0;
        w.row0 = vt->cu[seq];
        w.len = vt->cu[seq + 1] - w.row0;
        if constexpr (CAUSAL) {
            w.h = static_cast<int>(u) - t * a.H;
            w.qt = static_cast<int>(e & 0xffffu);
        } else {
            const int nq = (w.len + BLOCK_M - 1) / BLOCK_M;
            const int first = t - static_cast<int>(e & 0xffffu);   // list index of the sequence's tile 0
            const int v = static_cast<int>(u) - first * a.H;      // unit within the sequence, < nq * H
            w.h = v / nq;
            w.qt = v - w.h * nq;
        }
        if (w.row0 < 0 || w.len < 1 || w.row0 + w.len > a.S || w.qt * BLOCK_M >= w.len || w.h < 0 || w.h >= a.H) {
            report_error(XS_DEVICE_BOUNDS_CODE, 1, t, static_cast<int>(e), w.row0);
            return false;
        }
        w.k0 = 0;
        w.nb = CAUSAL ? w.qt + 1 : (w.len + BLOCK_N - 1) / BLOCK_N;
        w.kind = WORK_FULL;
        w.t_sk = -1;
        return true;
    }
    if constexpr (CAUSAL) {
        const long long u = static_cast<long long>(idx) * G + ((idx & 1) ? G - 1 - i : i);
        if (u >= a.units) return false;
        const int t = static_cast<int>(u);
        int bh, r;
        if (a.causal_head_major) {
            fdivmod(t, a.fd_nqt, bh, r);     // r: position within the head, longest first
            w.qt = a.n_qt - 1 - r;
        } else {
            fdivmod(t, a.fd_BH, r, bh);      // r: rank of the query tile, longest first
            w.qt = a.n_qt - 1 - r;
        }
        fdivmod(bh, a.fd_H, w.b, w.h);
        w.k0 = 0;
        w.nb = w.qt + 1;
        w.kind = WORK_FULL;
        w.t_sk = -1;
        return true;
    }
    const int n = a.n_kv;
    const int dp = a.sp.dp_tiles;
    const int ndp = dp > i ? fdiv(dp - i + G - 1, a.fd_grid) : 0;
    int tile, k0 = 0, k1 = n;
    if (idx < ndp) {
        tile = i + idx * G;
        w.kind = WORK_FULL;
        w.t_sk = -1;
    } else {
        if (a.sp.sk_iters == 0 || i >= a.sp.sk_ctas) return false;
        const long long it0 = sk_start(a, i), it1 = sk_start(a, i + 1);
        if (it1 <= it0) return false;
        const long long t = it0 / n + (idx - ndp);
        if (t > (it1 - 1) / n) return false;
        const long long lo = it0 - t * n, hi = it1 - t * n;
        k0 = lo > 0 ? static_cast<int>(lo) : 0;
        k1 = hi < n ? static_cast<int>(hi) : n;
        tile = dp + static_cast<int>(t);
        w.kind = k0 > 0 ? WORK_PART : (k1 == n ? WORK_FULL : WORK_HEAD);
        w.t_sk = static_cast<int>(t);
    }
    decode_unit(tile, a, w.b, w.h, w.qt);
    w.k0 = k0;
    w.nb = k1 - k0;
    return true;
}

// Ring item `i` of a unit with n key blocks, in the consumption order
// K0, K1, V0, K2, V1, K3, ..., V(n-3), K(n-1), V(n-2), V(n-1): the block index
// and whether it is a V block.
__device__ __forceinline__ void ring_item(int i, int n, int& blk, bool& is_v) {
    if (n == 1) {
        blk = 0;
        is_v = (i == 1);
        return;
    }
    if (i < 2) {
        blk = i;
        is_v = false;
        return;
    }
    const int r = i - 2;  // pairs (V_j, K_{j+2}) for j + 2 < n, then V(n-2), V(n-1)
    const int pairs = n - 2;
    if (r < 2 * pairs) {
        is_v = (r & 1) == 0;
        blk = is_v ? (r >> 1) : (r >> 1) + 2;
    } else {
        is_v = true;
        blk = n - 2 + (r - 2 * pairs);
    }
}

// ---------------------------------------------------------------- producer
// Tensor map and row coordinate of sequence row `row` (a multiple of 128): one
// map for the whole tensor, or, for sequence-sharded inputs, the map of shard
// row / in_Sl and the row within it (a tile never straddles two shards because
// in_Sl is a multiple of 128).
__device__ __forceinline__ const CUtensorMap* pick_map(const AttnArgs& a, const CUtensorMap* maps, int row,
                                                      int& row_in_map) {
    if (a.in_Sl == 0) {
        row_in_map = row;
        return maps;
    }
    // No division: this runs in the single producer thread, whose instruction
    // latency is on the pipeline's critical path.  Shard = (row / 128) / bps with
    // bps = in_Sl / 128 blocks per shard, as a multiply-high by the host's
    // reciprocal in_magic = ceil(2^(31 + k) / bps), k = floor(log2 bps), and a
    // shift: exact for row / 128 < 2^16 (the host checks).
    const unsigned blk2 = (static_cast<unsigned>(row) >> 7) << 1;
    const int p = static_cast<int>(__umulhi(blk2, a.in_magic) >> a.in_shift);
    row_in_map = row - p * a.in_Sl;
    return maps + p;
}

// Run by one thread.
template <int D, bool CAUSAL, bool VARLEN>
__device__ void producer_role(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                              const AttnArgs& a, const VarlenTable* vt, uint8_t* smem, uint32_t bar0,
                              volatile int* abort_flag) {
    using C = Cfg<D>;
    const uint32_t sbase = smem_addr(smem);
    auto bar = [&](int i) { return bar0 + static_cast<uint32_t>(i) * 8u; };
    uint32_t item = 0;        // ring items issued over the CTA's lifetime
    int u_iter = 0;
    int q_last = -1;          // u_iter of the last Q load issued
    bool ok = true;
    Work w;
    for (; ok && get_work<CAUSAL, VARLEN>(a, vt, u_iter, w); ++u_iter) {
        const int b = w.b, h = w.h, qt = w.qt;
        unsigned long long* const ph = phase_rows(u_iter, true);
        const int qb = u_iter % C::Q_BUFS;
        if (u_iter >= C::Q_BUFS)
            ok = thread_wait(bar(C::B_Q_FREE + qb), ((u_iter / C::Q_BUFS) - 1) & 1, abort_flag, a.timeout_ns, u_iter);
        if (!ok) break;
        mbar_arrive_expect_tx(bar(C::B_Q_FULL + qb), C::TILE_BYTES);
        const int row_base = VARLEN ? w.row0 : 0;   // packed row of the sequence start
        int q_row;
        const CUtensorMap* q_map = pick_map(a, tq, row_base + qt * BLOCK_M, q_row);
        for (int pnl = 0; pnl < C::PANELS; ++pnl)
            tma_load_4d(sbase + C::Q_OFF + qb * C::TILE_BYTES + pnl * PANEL_BYTES, q_map, bar(C::B_Q_FULL + qb),
                        pnl * 64, a.h0 + h, q_row, b);
        q_last = u_iter;
        {   // start the next piece's Q towards L2: its load waits for this piece's
            // last S MMA (one Q buffer at D = 128) and then hits L2, not HBM
            Work wn;
            if (get_work<CAUSAL, VARLEN>(a, vt, u_iter + 1, wn)) {
                int r;
                const CUtensorMap* m = pick_map(a, tq, (VARLEN ? wn.row0 : 0) + wn.qt * BLOCK_M, r);
                for (int pnl = 0; pnl < C::PANELS; ++pnl) tma_prefetch_l2_4d(m, pnl * 64, a.h0 + wn.h, r, wn.b);
            }
        }
        for (int i = 0; i < 2 * w.nb && ok; ++i) {
            int blk;
            bool is_v;
            ring_item(i, w.nb, blk, is_v);
            blk += w.k0;
            const uint32_t stage = item % C::KV_STAGES;
            const uint32_t round = item / C::KV_STAGES;
            if (round > 0)
                ok = thread_wait(bar(C::B_KV_FREE + stage), (round - 1) & 1, abort_flag, a.timeout_ns, u_iter, blk);
            if (!ok) break;
            mbar_arrive_expect_tx(bar(C::B_KV_FULL + stage), C::TILE_BYTES);
            int kv_row;
            const CUtensorMap* kv_map = pick_map(a, is_v ? tv : tk, row_base + blk * BLOCK_N, kv_row);
            for (int pnl = 0; pnl < C::PANELS; ++pnl)
                tma_load_4d(sbase + C::KV_OFF + stage * C::TILE_BYTES + pnl * PANEL_BYTES, kv_map,
                            bar(C::B_KV_FULL + stage), pnl * 64, a.h0 + h, kv_row, b);
            ++item;
            phase_stamp(ph, blk - w.k0, is_v ? 14 : 13);
        }
    }
    if (!ok) {
        // Let the copies already issued land before the CTA exits: wait (bounded)
        // for the newest phase of every ring stage used and for the last Q load.
        for (uint32_t back = 1; back <= C::KV_STAGES && back <= item; ++back) {
            const uint32_t it = item - back;
            drain_wait(bar(C::B_KV_FULL + it % C::KV_STAGES), (it / C::KV_STAGES) & 1, 20000000ull);
        }
        if (q_last >= 0) drain_wait(bar(C::B_Q_FULL + q_last % C::Q_BUFS), (q_last / C::Q_BUFS) & 1, 20000000ull);
    }
}

// --------------------------------------------------------------------- MMA
// Shared-memory operand descriptors (128-byte swizzle) are built once per role;
// a k-step or a ring stage only moves the start address (desc_add, one 32-bit
// add), which keeps the issuing threads to a few instructions per MMA.
// Q / K operand (K-major): k-step kk covers 16 columns of D, 32 B within the
// 128-B rows of a 64-column panel; panels are PANEL_BYTES apart.
__device__ __forceinline__ constexpr uint32_t k_step16(int kk) {
    return static_cast<uint32_t>((kk >> 2) * (PANEL_BYTES >> 4) + (kk & 3) * 2);
}
// V operand (MN-major = D contiguous): k-step kk covers 16 keys = two 8-key
// groups of 1024 B (SBO); 64-wide D panels are PANEL_BYTES apart (LBO).
__device__ __forceinline__ constexpr uint32_t v_step16(int kk) { return static_cast<uint32_t>(kk * (2048 >> 4)); }

// Issuer of S(j) = Q K_j^T (SS) into S buffer (block index) % 3.  One thread.
template <int D, bool CAUSAL, bool VARLEN>
__device__ void mma_s_role(const AttnArgs& a, const VarlenTable* vt, uint8_t* smem, uint32_t bar0,
                           uint32_t tmem_base, volatile int* abort_flag) {
    using C = Cfg<D>;
    const uint32_t sbase = smem_addr(smem);
    auto bar = [&](int i) { return bar0 + static_cast<uint32_t>(i) * 8u; };
    constexpr uint32_t IDESC_QK = idesc_bf16_f32(BLOCK_M, BLOCK_N, 0);
    const uint64_t qdesc0 = smem_desc_sw128(sbase + C::Q_OFF, 16, 1024);   // Q buffer 0
    const uint64_t kdesc0 = smem_desc_sw128(sbase + C::KV_OFF, 16, 1024);  // ring stage 0, as K
    uint32_t g = 0;      // key blocks over the CTA's lifetime
    uint32_t sb = 0, sph = 0;   // S buffer of block g (g % 3) and its phase parity ((g / 3) & 1)
    uint32_t item0 = 0;  // first ring item of the current piece of work
    int u_iter = 0;
    bool ok = true;
    Work w;
    for (; ok && get_work<CAUSAL, VARLEN>(a, vt, u_iter, w); ++u_iter) {
        unsigned long long* const ph = phase_rows(u_iter, true);
        const int n = w.nb;
        const int qb = u_iter % C::Q_BUFS;
        const uint64_t qdesc = desc_add(qdesc0, qb * (C::TILE_BYTES >> 4));
        ok = thread_wait(bar(C::B_Q_FULL + qb), (u_iter / C::Q_BUFS) & 1, abort_flag, a.timeout_ns, u_iter);
        // the previous piece's last PV first: its epilogue waits for it, while
        // this piece's first scores are only read after that epilogue
        if (ok && u_iter > 0) ok = thread_wait(bar(C::B_O_FINAL), (u_iter - 1) & 1, abort_flag, a.timeout_ns, u_iter);
        for (int j = 0; j < n && ok; ++j) {
            const uint32_t gs = g + j;
            // the buffer's previous block (gs-3) is done: its P has been read by PV(gs-3)
            if (gs >= S_BUFS)
                ok = thread_wait(bar(C::B_P_FREE + sb), sph ^ 1u, abort_flag, a.timeout_ns, u_iter, j);
            phase_stamp(ph, j, 11);
            const uint32_t item = item0 + ring_pos_k(j);
            const uint32_t stage = item % C::KV_STAGES;
            if (ok)
                ok = thread_wait(bar(C::B_KV_FULL + stage), (item / C::KV_STAGES) & 1, abort_flag, a.timeout_ns, u_iter, j);
            phase_stamp(ph, j, 12);
            if (!ok) break;
            tc_fence_after();
            const uint64_t kdesc = desc_add(kdesc0, stage * (C::TILE_BYTES >> 4));
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                mma_ss(tmem_base + S_COL + sb * 128u, desc_add(qdesc, k_step16(kk)), desc_add(kdesc, k_step16(kk)),
                       IDESC_QK, kk > 0);
            phase_stamp(ph, j, 7);
            mma_commit(bar(C::B_S_FULL + sb));
            mma_commit(bar(C::B_KV_FREE + stage));
            if (j == n - 1) mma_commit(bar(C::B_Q_FREE + qb));
            if (++sb == S_BUFS) {
                sb = 0;
                sph ^= 1u;
            }
        }
        g += n;
        item0 += 2u * n;
    }
    // Drain: B_DRAIN completes when both issuers' MMAs have all completed (TMEM
    // is freed after it).  The limit is at least 20 ms whatever the wait limit.
    mma_commit(bar(C::B_DRAIN));
    drain_wait(bar(C::B_DRAIN), 0, a.timeout_ns > 20000000ull ? a.timeout_ns : 20000000ull);
}

// Issuer of PV(j): O += P(j) V_j (A = P(j), over the first 64 columns of S buffer
// j % 3 in TMEM).  One thread.
template <int D, bool CAUSAL, bool VARLEN>
__device__ void mma_pv_role(const AttnArgs& a, const VarlenTable* vt, uint8_t* smem, uint32_t bar0,
                            uint32_t tmem_base, volatile int* abort_flag) {
    using C = Cfg<D>;
    const uint32_t sbase = smem_addr(smem);
    auto bar = [&](int i) { return bar0 + static_cast<uint32_t>(i) * 8u; };
    constexpr uint32_t IDESC_PV = idesc_bf16_f32(BLOCK_M, D, 1);
    const uint64_t vdesc0 = smem_desc_sw128(sbase + C::KV_OFF, PANEL_BYTES, 1024);  // ring stage 0, as V
    uint32_t g = 0;
    uint32_t pb = 0, pph = 0;   // buffer of block g (g % 3) and its phase parity ((g / 3) & 1)
    uint32_t item0 = 0;
    int u_iter = 0;
    bool ok = true;
    Work w;
    for (; ok && get_work<CAUSAL, VARLEN>(a, vt, u_iter, w); ++u_iter) {
        unsigned long long* const ph = phase_rows(u_iter, true);
        const int n = w.nb;
        for (int j = 0; j < n && ok; ++j) {
            ok = thread_wait(bar(C::B_P_FULL + pb), pph, abort_flag, a.timeout_ns, u_iter, j);
            phase_stamp(ph, j, 9);
            // the epilogue has read the previous unit's O (PV(0) overwrites it)
            if (ok && j == 0 && u_iter > 0)
                ok = thread_wait(bar(C::B_O_FREE), (u_iter - 1) & 1, abort_flag, a.timeout_ns, u_iter, j);
            const uint32_t item = item0 + ring_pos_v(j, n);
            const uint32_t stage = item % C::KV_STAGES;
            if (ok)
                ok = thread_wait(bar(C::B_KV_FULL + stage), (item / C::KV_STAGES) & 1, abort_flag, a.timeout_ns, u_iter, j);
            phase_stamp(ph, j, 10);
            if (!ok) break;
            tc_fence_after();
            const uint64_t vdesc = desc_add(vdesc0, stage * (C::TILE_BYTES >> 4));
#pragma unroll
            for (int kk = 0; kk < BLOCK_N / 16; ++kk)
                mma_ts(tmem_base + O_COL, tmem_base + S_COL + pb * 128u + kk * 8, desc_add(vdesc, v_step16(kk)),
                       IDESC_PV, (j > 0) || (kk > 0));
            phase_stamp(ph, j, 8);
            mma_commit(bar(C::B_P_FREE + pb));
            mma_commit(bar(C::B_KV_FREE + stage));
            if (j == n - 1) mma_commit(bar(C::B_O_FINAL));
            if (++pb == S_BUFS) {
                pb = 0;
                pph ^= 1u;
            }
        }
        g += n;
        item0 += 2u * n;
    }
    mma_commit(bar(C::B_DRAIN));
    drain_wait(bar(C::B_DRAIN), 0, a.timeout_ns > 20000000ull ? a.timeout_ns : 20000000ull);
}

// ------------------------------------------------------- softmax + epilogue
// Bounded wait (whole warp) until every softmax warp of CTA `slot` has published
// its part of a split tile in this launch (flag == this launch's epoch).  Each
// lane polls the eight flags itself with acquire loads, so its later loads of
// the partial are ordered after them.  The result is warp-uniform.
__device__ __forceinline__ bool wait_partial(const AttnArgs& a, int slot, unsigned epoch, volatile int* abort_flag) {
    const unsigned* f = a.sp.part_flag + slot * NUM_SOFTMAX_WARPS;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        bool mine = true;
#pragma unroll
        for (int i = 0; i < NUM_SOFTMAX_WARPS; ++i) mine = mine && (ld_acquire_gpu(f + i) == epoch);
        if (__all_sync(0xffffffffu, mine)) return true;
        if (*abort_flag) return false;
        if (expired(t0, a.timeout_ns)) {
            *abort_flag = 1;
            report_error(XS_DEVICE_TIMEOUT_CODE, 0x40000 + slot, static_cast<int>(epoch), -1, -1);
            return false;
        }
        __nanosleep(256);
    }
}

// Maximum of a thread's 64 scores: four independent 3-input chains.
__device__ __forceinline__ float max64(const uint32_t (&sr)[2][32]) {
    float mx[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) mx[r] = __uint_as_float(sr[r >> 1][(r & 1) * 16]);
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
            const int r = q * 2 + (i >> 4);
            mx[r] = fmax3(mx[r], __uint_as_float(sr[q][i]), __uint_as_float(sr[q][i + 1]));
            mx[r] = fmax3(mx[r], __uint_as_float(sr[q][i + 2]), __uint_as_float(sr[q][i + 3]));
        }
    return fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
}

// p = 2^(s*c - m) for a thread's 64 scores: one packed f32x2 FMA per pair of
// scores and one MUFU ex2 each, packed to bf16 pairs; the fp32 values are summed
// with packed f32x2 adds in two independent chains (half the FP32-pipe
// instructions of scalar FMAs and adds).
// TAIL: columns at or past `valid` (keys past the sequence) get p = 0.
template <bool TAIL>
__device__ __forceinline__ float exp64(const uint32_t (&sr)[2][32], float c, float m, int col0, int valid,
                                       uint32_t (&pk)[32]) {
    const float neg_m = -m;
    const uint64_t cc = f2_pack(c, c), mm = f2_pack(neg_m, neg_m);
    uint64_t acc2[2] = {f2_pack(0.0f, 0.0f), f2_pack(0.0f, 0.0f)};
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const int q = i >> 4;
        const int e = (i & 15) * 2;
        float x0, x1;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[q][e]), __uint_as_float(sr[q][e + 1])), cc, mm), x0, x1);
        float p0 = ex2_approx(x0);
        float p1 = ex2_approx(x1);
        if (TAIL) {
            const int col = col0 + q * 32 + e;
            if (col >= valid) p0 = 0.0f;
            if (col + 1 >= valid) p1 = 0.0f;
        }
        acc2[i & 1] = f2_add(acc2[i & 1], f2_pack(p0, p1));
        pk[i] = pack_bf16x2(p0, p1);
    }
    float a0, a1, b0, b1;
    f2_unpack(acc2[0], a0, a1);
    f2_unpack(acc2[1], b0, b1);
    return (a0 + a1) + (b0 + b1);
}

// Epilogue of a piece of a split tile (rare: at most two per CTA and launch),
// kept out of line so that it does not weigh on the register allocation of the
// softmax loop.  The calling thread owns query row `row` of the tile and its DH
// output columns of half `half`, which it reads with the 16x32bx2 TMEM accesses
// at o_base (the O accumulator at the warp's lanes); m, l are the row's running
// max (log2 units) and sum over this piece's key blocks.
//   WORK_PART: publish the unnormalised O, m and l in this CTA's workspace slot,
//              then this warp's flag (release) with the launch epoch.
//   WORK_HEAD: wait for the parts of the tile (slots of the following CTAs whose
//              ranges start inside it) and store
//              (sum_k O_k 2^(m_k - M)) / (sum_k l_k 2^(m_k - M)),  M = max_k m_k,
//              over this piece and the parts.
template <int D>
__device__ __noinline__ bool split_epilogue(const AttnArgs& a, const Work& w, uint32_t o_base, int row, int half,
                                            int warp, float m, float l, unsigned epoch, volatile int* abort_flag) {
    constexpr int DH = D / 2;
    if (w.kind == WORK_PART) {
        float* po = a.sp.part_o + (static_cast<size_t>(blockIdx.x) * BLOCK_M + row) * D + half * DH;
#pragma unroll 1
        for (int q = 0; q < DH / 32; ++q) {
            uint32_t orr[32];
            tmem_ld16x2_32<DH>(o_base + q * 32, orr);
            tmem_wait_ld();
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
                st_global_v4(po + q * 32 + v4 * 4, orr[4 * v4], orr[4 * v4 + 1], orr[4 * v4 + 2], orr[4 * v4 + 3]);
        }
        if (half == 0) a.sp.part_ml[static_cast<size_t>(blockIdx.x) * BLOCK_M + row] = make_float2(m, l);
        __syncwarp();
        if (lane_id() == 0) {
            __threadfence();
            st_release_gpu(a.sp.part_flag + blockIdx.x * NUM_SOFTMAX_WARPS + warp, epoch);
        }
        return true;
    }
    // the parts: CTAs j = blockIdx.x + 1, ... whose ranges start before the tile's end
    const long long tile_end = static_cast<long long>(w.t_sk + 1) * a.n_kv;
    const int j0 = blockIdx.x + 1;
    int j1 = j0;
    while (j1 < a.sp.sk_ctas && sk_start(a, j1) < tile_end) ++j1;
    float m_all = m;
    for (int j = j0; j < j1; ++j) {
        if (!wait_partial(a, j, epoch, abort_flag)) return false;
        m_all = fmaxf(m_all, a.sp.part_ml[static_cast<size_t>(j) * BLOCK_M + row].x);
    }
    const float f_own = ex2_approx(m - m_all);
    float l_all = l * f_own;
    for (int j = j0; j < j1; ++j) {
        const float2 ml = a.sp.part_ml[static_cast<size_t>(j) * BLOCK_M + row];
        l_all += ml.y * ex2_approx(ml.x - m_all);
    }
    const float inv_l = 1.0f / l_all;
    const int s_loc = w.qt * BLOCK_M + row;
    const int s_row = a.epi.row0 + s_loc;
    bool store = s_loc < a.S;
    __nv_bfloat16* dst = nullptr;
    if (store) {
        const int hg = a.h0_out + w.h;   // head in the output layout
        int ps, s_dst, ph, h_dst;
        fdivmod(s_row, a.epi.fd_Sl, ps, s_dst);
        fdivmod(hg, a.epi.fd_Hl, ph, h_dst);
        const int p = ps + ph;
        if (p < MAX_PTRS && a.epi.ptr[p] != nullptr) {
            dst = reinterpret_cast<__nv_bfloat16*>(a.epi.ptr[p]) +
                  ((static_cast<size_t>(w.b) * a.epi.Sl + s_dst) * a.epi.Hl + h_dst) * D + half * DH;
        } else {
            report_error(XS_DEVICE_BOUNDS_CODE, 2, p, s_row, w.h);
            store = false;
        }
    }
#pragma unroll 1
    for (int q = 0; q < DH / 32; ++q) {
        uint32_t orr[32];
        tmem_ld16x2_32<DH>(o_base + q * 32, orr);
        tmem_wait_ld();
        float acc[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[i] = __uint_as_float(orr[i]) * f_own;
        for (int j = j0; j < j1; ++j) {
            const float f = ex2_approx(a.sp.part_ml[static_cast<size_t>(j) * BLOCK_M + row].x - m_all);
            const float* po = a.sp.part_o + (static_cast<size_t>(j) * BLOCK_M + row) * D + half * DH + q * 32;
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4) {
                const float4 pv = *reinterpret_cast<const float4*>(po + v4 * 4);
                acc[4 * v4 + 0] += pv.x * f;
                acc[4 * v4 + 1] += pv.y * f;
                acc[4 * v4 + 2] += pv.z * f;
                acc[4 * v4 + 3] += pv.w * f;
            }
        }
        uint32_t wv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) wv[i] = pack_bf16x2(acc[2 * i] * inv_l, acc[2 * i + 1] * inv_l);
        if (store) {
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
                st_global_v4(dst + q * 32 + v4 * 8, wv[4 * v4], wv[4 * v4 + 1], wv[4 * v4 + 2], wv[4 * v4 + 3]);
        }
    }
    return true;
}

template <int D, bool CAUSAL, bool VARLEN>
__device__ void softmax_role(const AttnArgs& a, const VarlenTable* vt, uint8_t* smem, uint32_t bar0,
                             uint32_t tmem_base, volatile int* abort_flag) {
    using C = Cfg<D>;
    constexpr int DH = D / 2;  // O columns owned by each of a row's two threads
    const int warp = threadIdx.x >> 5;
    const int lane = static_cast<int>(lane_id());
    const int quarter = warp & 3;             // TMEM lane quarter this warp may access
    const int half = lane >> 4;               // key columns [64*half, 64*half + 64), O columns [DH*half, +DH)
    // rows 32*quarter + 16*(warp/4) .. +15: the warp's half of its lane quarter
    const int row = quarter * 32 + (warp >> 2) * 16 + (lane & 15);
    const uint32_t t_base = tmem_base + (static_cast<uint32_t>(quarter * 32 + (warp >> 2) * 16) << 16);
    auto bar = [&](int i) { return bar0 + static_cast<uint32_t>(i) * 8u; };
    const float c = a.c;

    uint32_t g = 0;
    uint32_t sb = 0, sph = 0;    // S buffer of block g (g % 3) and its phase parity ((g / 3) & 1)
    uint32_t pb = 2, pph = 1;    // the same for block g - 1 (the O rescale waits for PV(g-1))
    int u_iter = 0;
    bool ok = true;
    while (ok) {
        int n, valid0;   // only these two stay live through the block loop
        {
            Work w;
            if (!get_work<CAUSAL, VARLEN>(a, vt, u_iter, w)) break;
            n = w.nb;
            // key columns of the piece this row attends to: keys below S, and
            // (causal) keys up to the row's own position
            const int seq_len = VARLEN ? w.len : a.S;
            if constexpr (CAUSAL)
                valid0 = min(seq_len, w.qt * BLOCK_M + row + 1) - w.k0 * BLOCK_N;
            else
                valid0 = seq_len - w.k0 * BLOCK_N;
        }
        float m_run = 0.0f, l_run = 0.0f;
        unsigned long long* const ph = phase_rows(u_iter, threadIdx.x == 0);
        unsigned long long* const phw = phase_rows(u_iter, lane == 0);   // every softmax warp's lane 0
        for (int j = 0; j < n; ++j, ++g) {
            phase_stamp(ph, j, 0);
            ok = warp_wait(bar(C::B_S_FULL + sb), sph, abort_flag, a.timeout_ns, u_iter, j);
            if (!ok) break;
            phase_stamp(ph, j, 1);
            if (j == 0) {
                span_stamp(u_iter, 0, globaltimer_ns());
                span_stamp(u_iter, 1, span_clock());
            }
            tc_fence_after();
            uint32_t sr[2][32];
            tmem_ld16x2_32<64>(t_base + S_COL + sb * 128u, sr[0]);
            tmem_ld16x2_32<64>(t_base + S_COL + sb * 128u + 32, sr[1]);
            tmem_wait_ld();
            phase_stamp(ph, j, 2);
            const int valid = valid0 - j * BLOCK_N;
            // Warp-uniform whenever the tail is (no causal mask).  On the causal
            // diagonal block the rows of a warp differ, and one vote keeps the
            // warp on one path (columns at or past `valid` are masked either way).
            bool tail = valid < BLOCK_N;
            if constexpr (CAUSAL) tail = __any_sync(0xffffffffu, tail);
            if (tail) {
#pragma unroll
                for (int q = 0; q < 2; ++q)
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (half * 64 + q * 32 + i >= valid) sr[q][i] = 0xff800000u;  // -inf
            }
            // row max: the two halves of the row are lanes i and i ^ 16
            const float m_half = max64(sr);
            const float m_blk = fmaxf(m_half, __shfl_xor_sync(0xffffffffu, m_half, 16)) * c;
            phase_stamp(ph, j, 3);
            float m_use, alpha = 1.0f;
            bool rescale = false;
            if (j == 0) {
                m_use = m_blk;
            } else if (m_blk - m_run > RESCALE_THRESHOLD) {
                m_use = m_blk;
                alpha = ex2_approx(m_run - m_blk);
                rescale = true;
            } else {
                m_use = m_run;
            }
            uint32_t pk[32];
            const float sum = tail ? exp64<true>(sr, c, m_use, half * 64, valid, pk)
                                   : exp64<false>(sr, c, m_use, half * 64, valid, pk);
            phase_stamp(ph, j, 4);
            const bool redo = __any_sync(0xffffffffu, rescale);  // warp-uniform
            // Rescale of this thread's half of the O row (rare); PV(g-1) must have
            // completed first.  Warp-uniform: TMEM access is collective.
            if (redo) {
                ok = warp_wait(bar(C::B_P_FREE + pb), pph, abort_flag, a.timeout_ns, u_iter, j);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int q = 0; q < DH / 32; ++q) {
                    uint32_t orr[32];
                    tmem_ld16x2_32<DH>(t_base + O_COL + q * 32, orr);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
                    tmem_st16x2_32<DH>(t_base + O_COL + q * 32, orr);
                }
            }
            // P(g) over the first 64 columns of the scores just read (both halves
            // of every row loaded: the loads above were warp-collective and waited)
            phase_stamp(ph, j, 5);
            tmem_st16x2_32<32>(t_base + S_COL + sb * 128u, pk);
            tmem_wait_st();
            tc_fence_before();
            warp_arrive(bar(C::B_P_FULL + sb));
            phase_stamp(ph, j, 6);
            phase_stamp(phw, j, 16 + warp);
            if (j == n - 1) span_stamp(u_iter, 2, span_clock());
            l_run = l_run * alpha + sum;
            m_run = m_use;
            pb = sb;
            pph = sph;
            if (++sb == S_BUFS) {
                sb = 0;
                sph ^= 1u;
            }
        }
        if (!ok) break;
        // ---- epilogue: the owner of this tile stores it to the destination shard
        const float l_row = l_run + __shfl_xor_sync(0xffffffffu, l_run, 16);
        Work w;
        get_work<CAUSAL, VARLEN>(a, vt, u_iter, w);   // the same piece of work as above (recomputed, not kept live)
        const int b = w.b, h = a.h0_out + w.h, qt = w.qt;   // h: head in the output layout
        ok = warp_wait(bar(C::B_O_FINAL), u_iter & 1, abort_flag, a.timeout_ns, u_iter);
        if (!ok) break;
        span_stamp(u_iter, 3, span_clock());
        unsigned long long* const pe = epi_rows(u_iter, threadIdx.x == 0);
        epi_stamp(pe, 0);
        tc_fence_after();
        if (w.kind == WORK_FULL) {
            // Each lane holds half a row; stores straight from the lanes would
            // scatter 32 pieces per instruction.  A 2 KB per-warp stage (32 half
            // rows x 64 B, 16-byte chunks XOR-swizzled against bank conflicts) lets
            // 4 lanes write 64 contiguous bytes: each store instruction covers 8 pieces.
            const int s_loc = qt * BLOCK_M + row;   // row within the sequence
            unsigned long long dst_row = 0;   // this lane's half row in the destination (0: past the sequence)
            if (s_loc < (VARLEN ? w.len : a.S)) {
                const int s_row = (VARLEN ? w.row0 : a.epi.row0) + s_loc;
                int ps, s_dst, ph, h_dst;
                fdivmod(s_row, a.epi.fd_Sl, ps, s_dst);
                fdivmod(h, a.epi.fd_Hl, ph, h_dst);
                const int p = ps + ph;
                if (p < MAX_PTRS && a.epi.ptr[p] != nullptr)
                    dst_row = reinterpret_cast<unsigned long long>(
                        reinterpret_cast<__nv_bfloat16*>(a.epi.ptr[p]) +
                        ((static_cast<size_t>(b) * a.epi.Sl + s_dst) * a.epi.Hl + h_dst) * D + half * DH);
                else
                    report_error(XS_DEVICE_BOUNDS_CODE, 2, p, s_row, h);
            }
            epi_stamp(pe, 1);
            uint4* stage = reinterpret_cast<uint4*>(smem + C::STAGE_OFF + warp * 2048);
            const float inv_l = 1.0f / l_row;
#pragma unroll
            for (int q = 0; q < DH / 32; ++q) {
                uint32_t orr[32];
                tmem_ld16x2_32<DH>(t_base + O_COL + q * 32, orr);
                tmem_wait_ld();
                epi_stamp(pe, 2 + 3 * q);
                uint32_t wv[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    wv[i] = pack_bf16x2(__uint_as_float(orr[2 * i]) * inv_l, __uint_as_float(orr[2 * i + 1]) * inv_l);
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4)
                    stage[lane * 4 + (c4 ^ (lane & 3))] =
                        make_uint4(wv[4 * c4], wv[4 * c4 + 1], wv[4 * c4 + 2], wv[4 * c4 + 3]);
                __syncwarp();
                epi_stamp(pe, 3 + 3 * q);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int r = k * 8 + (lane >> 2);   // lane whose half row this lane stores a chunk of
                    const int c4 = lane & 3;
                    const uint4 v = stage[r * 4 + (c4 ^ (r & 3))];
                    const unsigned long long rp = __shfl_sync(0xffffffffu, dst_row, r);
                    if (rp)
                        st_global_v4(reinterpret_cast<__nv_bfloat16*>(rp) + q * 32 + c4 * 8, v.x, v.y, v.z, v.w);
                }
                __syncwarp();   // the stage is rewritten by the next chunk
                epi_stamp(pe, 4 + 3 * q);
            }
        } else {
            ok = split_epilogue<D>(a, w, t_base + O_COL, row, half, warp, m_run, l_row,
                                   *reinterpret_cast<const volatile unsigned*>(smem + C::MISC_OFF + 8), abort_flag);
            if (!ok) break;
        }
        span_stamp(u_iter, 4, span_clock());
        span_stamp(u_iter, 5, (static_cast<unsigned long long>(w.nb) << 32) | static_cast<unsigned>(w.kind));
        tc_fence_before();
        warp_arrive(bar(C::B_O_FREE));
        ++u_iter;
    }
}

// The whole kernel; tq, tk, tv point to one tensor map each, or to n_maps maps
// (one per input sequence shard, args.in_Sl != 0).
template <int D, bool CAUSAL, bool VARLEN>
__device__ __forceinline__ void attn_body(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                                          int n_maps, const AttnArgs& args, const VarlenTable* vt) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t bar0 = smem_addr(smem + C::BAR_OFF);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);
    const int warp = threadIdx.x >> 5;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar0 + 8 * (C::B_Q_FULL + i), 1);   // (index 1 unused when Q_BUFS == 1)
            mbar_init(bar0 + 8 * (C::B_Q_FREE + i), 1);
        }
        for (int i = 0; i < S_BUFS; ++i) {
            mbar_init(bar0 + 8 * (C::B_S_FULL + i), 1);
            mbar_init(bar0 + 8 * (C::B_P_FULL + i), NUM_SOFTMAX_WARPS);
            mbar_init(bar0 + 8 * (C::B_P_FREE + i), 1);
        }
        mbar_init(bar0 + 8 * C::B_O_FINAL, 1);
        mbar_init(bar0 + 8 * C::B_O_FREE, NUM_SOFTMAX_WARPS);
        mbar_init(bar0 + 8 * C::B_DRAIN, 2);
        for (int s = 0; s < C::KV_STAGES; ++s) {
            mbar_init(bar0 + 8 * (C::B_KV_FULL + s), 1);
            mbar_init(bar0 + 8 * (C::B_KV_FREE + s), 1);
        }
        *abort_flag = 0;
        // this launch's split-tile epoch: one more than the launches finished on
        // the workspace (never 0, the value of a flag nobody has written)
        unsigned epoch = 0;
        if (args.sp.sk_iters != 0) {
            epoch = *reinterpret_cast<volatile unsigned*>(args.sp.launch_count) + 1u;
            if (epoch == 0) epoch = 1;
        }
        *reinterpret_cast<volatile unsigned*>(smem + C::MISC_OFF + 8) = epoch;
        fence_mbar_init();
    }
    if (warp == WARP_TMA && lane_id() < n_maps) {
        tma_prefetch_desc(tq + lane_id());
        tma_prefetch_desc(tk + lane_id());
        tma_prefetch_desc(tv + lane_id());
    }
    if (warp == WARP_MMA_S) {
        tmem_alloc(smem_addr(tmem_holder), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp < 8) {
        softmax_role<D, CAUSAL, VARLEN>(args, vt, smem, bar0, tmem_base, abort_flag);
    } else if (lane_id() == 0) {
        // single-thread roles; the other lanes of these warps wait at the end
        if (warp == WARP_TMA)
            producer_role<D, CAUSAL, VARLEN>(tq, tk, tv, args, vt, smem, bar0, abort_flag);
        else if (warp == WARP_MMA_S)
            mma_s_role<D, CAUSAL, VARLEN>(args, vt, smem, bar0, tmem_base, abort_flag);
        else if (warp == WARP_MMA_PV)
            mma_pv_role<D, CAUSAL, VARLEN>(args, vt, smem, bar0, tmem_base, abort_flag);
    }
    __syncwarp();

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == WARP_MMA_S) tmem_dealloc(tmem_base, TMEM_COLS);
    // The last CTA of a split launch to get here advances the workspace's launch
    // count (every CTA has read it by then), so the next launch uses a new epoch.
    if (threadIdx.x == 0 && args.sp.sk_iters != 0) {
        __threadfence();
        if (atomicAdd(args.sp.launch_count + 1, 1u) == gridDim.x - 1) {
            args.sp.launch_count[1] = 0;
            __threadfence();
            atomicAdd(args.sp.launch_count, 1u);
        }
    }
}

template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_a2a_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ AttnArgs args) {
    attn_body<D, false, false>(&tmap_q, &tmap_k, &tmap_v, 1, args, nullptr);
}

// Q, K, V read straight from the P sequence shards of the Ulysses ranks: the
// pre-attention All-to-All is fused into the loads (each tile's TMA box comes
// from the shard that holds its rows), as the post-attention one is into the
// epilogue stores.
template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_ulysses_kernel(const __grid_constant__ AttnArgs args, const __grid_constant__ ShardMaps maps) {
    attn_body<D, false, false>(maps.q, maps.k, maps.v, args.S / args.in_Sl, args, nullptr);
}

// Causal attention (row s attends to keys 0 .. s), one [B, S, H, D] tensor per
// operand; the tile order and key-block counts are get_work's causal ones.
template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_causal_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                       const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ AttnArgs args) {
    attn_body<D, true, false>(&tmap_q, &tmap_k, &tmap_v, 1, args, nullptr);
}

// Packed variable-length sequences: one [1, T, H, D] tensor per operand holding
// the sequences of vt back to back; every row attends to its own sequence
// (CAUSAL: up to its own position).  The table travels in parameter space.
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_varlen_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                       const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ AttnArgs args,
                       const __grid_constant__ VarlenTable vt) {
    attn_body<D, CAUSAL, true>(&tmap_q, &tmap_k, &tmap_v, 1, args, &vt);
}

}  // namespace

template <int D>
int attn_smem_bytes() {
    return Cfg<D>::SMEM_ALLOC;
}

// The arguments with the tile-decode and destination divisors filled in (every
// launch goes through here, so the kernel never sees stale ones).
static AttnArgs with_divisors(const AttnArgs& args, int grid) {
    AttnArgs a = args;
    a.fd_nqt = make_fastdiv(a.n_qt > 0 ? a.n_qt : 1);
    a.fd_H = make_fastdiv(a.H > 0 ? a.H : 1);
    a.fd_BH = make_fastdiv(a.B * a.H > 0 ? a.B * a.H : 1);
    a.fd_grid = make_fastdiv(grid > 0 ? grid : 1);
    a.epi.fd_Sl = make_fastdiv(a.epi.Sl > 0 ? a.epi.Sl : 1);
    a.epi.fd_Hl = make_fastdiv(a.epi.Hl > 0 ? a.epi.Hl : 1);
    return a;
}

static_assert(Cfg<128>::SMEM_ALLOC <= 232448, "shared memory budget (D = 128)");
static_assert(Cfg<64>::SMEM_ALLOC <= 232448, "shared memory budget (D = 64)");

template <int D>
cudaError_t launch_attn(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const AttnArgs& args,
                        int grid, bool cooperative, cudaStream_t stream) {
    auto kern = attn_a2a_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    if (!cooperative) {
        kern<<<grid, NUM_THREADS, Cfg<D>::SMEM_ALLOC, stream>>>(tq, tk, tv, with_divisors(args, grid));
        return cudaGetLastError();
    }
    // CTAs of a split tile wait for each other: all of them must be resident at
    // once, which a cooperative launch guarantees (or refuses to launch).
    CUtensorMap q = tq, k = tk, v = tv;
    AttnArgs a = with_divisors(args, grid);
    void* params[] = {&q, &k, &v, &a};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kern), dim3(grid), dim3(NUM_THREADS), params,
                                       Cfg<D>::SMEM_ALLOC, stream);
}

template <int D>
cudaError_t launch_attn_sharded(const ShardMaps& maps, int P, const AttnArgs& args, int grid, bool cooperative,
                                cudaStream_t stream) {
    (void)P;
    auto kern = attn_ulysses_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    if (!cooperative) {
        kern<<<grid, NUM_THREADS, Cfg<D>::SMEM_ALLOC, stream>>>(with_divisors(args, grid), maps);
        return cudaGetLastError();
    }
    ShardMaps m = maps;
    AttnArgs a = with_divisors(args, grid);
    void* params[] = {&a, &m};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kern), dim3(grid), dim3(NUM_THREADS), params,
                                       Cfg<D>::SMEM_ALLOC, stream);
}

template <int D>
cudaError_t launch_attn_causal(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const AttnArgs& args, int grid, cudaStream_t stream) {
    auto kern = attn_causal_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    kern<<<grid, NUM_THREADS, Cfg<D>::SMEM_ALLOC, stream>>>(tq, tk, tv, with_divisors(args, grid));
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_attn_varlen(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const AttnArgs& args, const VarlenTable& vt, int grid, cudaStream_t stream) {
    auto kern = attn_varlen_kernel<D, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    kern<<<grid, NUM_THREADS, Cfg<D>::SMEM_ALLOC, stream>>>(tq, tk, tv, with_divisors(args, grid), vt);
    return cudaGetLastError();
}

template cudaError_t launch_attn_varlen<64>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                            const AttnArgs&, const VarlenTable&, int, cudaStream_t);
template cudaError_t launch_attn_varlen<128>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                             const AttnArgs&, const VarlenTable&, int, cudaStream_t);
template cudaError_t launch_attn_causal<64>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                            const AttnArgs&, int, cudaStream_t);
template cudaError_t launch_attn_causal<128>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                             const AttnArgs&, int, cudaStream_t);
template cudaError_t launch_attn_sharded<64>(const ShardMaps&, int, const AttnArgs&, int, bool, cudaStream_t);
template cudaError_t launch_attn_sharded<128>(const ShardMaps&, int, const AttnArgs&, int, bool, cudaStream_t);
template int attn_smem_bytes<64>();
template int attn_smem_bytes<128>();
template cudaError_t launch_attn<64>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const AttnArgs&, int,
                                     bool, cudaStream_t);
template cudaError_t launch_attn<128>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const AttnArgs&,
                                      int, bool, cudaStream_t);

#ifdef XS_TILE_SPANS
cudaError_t set_tile_spans(unsigned long long* buf, int ctas, int per_cta) {
    cudaError_t e = cudaMemcpyToSymbol(g_spans, &buf, sizeof buf);
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_spans_ctas, &ctas, sizeof ctas);
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_spans_per_cta, &per_cta, sizeof per_cta);
}
#endif

cudaError_t read_and_clear_device_error(int* value, DeviceErrorInfo* info, int* drain_failed) {
    int zero = 0;
    DeviceErrorInfo none{};
    cudaError_t e = cudaMemcpyFromSymbol(value, g_device_error, sizeof(int));
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(drain_failed, g_drain_failed, sizeof(int));
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(info, g_error_info, sizeof(DeviceErrorInfo));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_drain_failed, &zero, sizeof(int));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_error_info, &none, sizeof(DeviceErrorInfo));
    return e;
}

}  // namespace xs
