/*
 * xsattn: fused sequence-parallel attention + post-attention Ulysses All-to-All
 * layout for one GB300 (sm_103a).
 *
 * The method (X-Stage, arXiv 2607.23264, abstract; gist.science technical
 * summary, "Key Contributions" item 3, "FlashAttention-A2A (Piggybacking)"):
 * in Ulysses sequence-parallel DiT attention, the output-tile owner of the
 * attention kernel writes every finished output tile straight to the rank that
 * owns the tile's sequence block, then goes on to the next tile's Q-loop, so no
 * separate All-to-All (transpose / copy) step runs after attention.
 *
 * On one GPU the P ranks are "virtual": P plain device buffers.  Shard p owns the
 * contiguous sequence block [p*S/P, (p+1)*S/P) and holds all H heads at their
 * global head index.
 *
 * Layout conventions (all entry points):
 *   - bf16 tensors, row-major [B, S, H, D] with D fastest ("BSHD"), contiguous
 *     (xs_attn_varlen_fwd: packed [T, H, D]).
 *   - Attention is bidirectional (non-causal): O = softmax(Q K^T * scale) V per
 *     (b, h), no mask, no bias, no dropout, except in xs_attn_causal_fwd and,
 *     when asked, xs_attn_varlen_fwd.  Accumulation is fp32, the
 *     probabilities are rounded to bf16 before the PV product, the output is
 *     rounded to bf16 (round to nearest even).
 *   - D must be 64 or 128.  S, B, H >= 1; S need not be a multiple of the tile.
 *   - All device pointers must be 16-byte aligned.
 *
 * Ownership and synchronisation:
 *   - The caller owns every buffer and the stream.  The library allocates no
 *     device memory per call; on each device it keeps one error word and the
 *     scratch array of xs_attn_fwd_balanced_noalloc (static device data).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  Outputs are valid once the stream reaches the end of
 *     the call.  Inputs are never modified.
 *   - Host pointer arrays (out_ptrs, heads) are read before the call returns;
 *     the library keeps no reference to them.
 *
 * Errors: every entry point returns XS_OK (0) or a negative XS_ERR_* code.
 * Argument checks run on the host before anything is launched; a failed check
 * launches nothing.  NaN/Inf in the inputs give undefined (but memory-safe)
 * results.
 */
#ifndef XSATTN_H
#define XSATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Maximum number of virtual ranks (output shards). */
#define XS_MAX_P 16

enum {
    XS_OK = 0,
    XS_ERR_NULL = -1,            /* a required pointer is NULL                         */
    XS_ERR_SHAPE = -2,           /* B, S, H or P < 1, or a size overflows               */
    XS_ERR_HEAD_DIM = -3,        /* D is not 64 or 128                                  */
    XS_ERR_DIVISIBILITY = -4,    /* S % P != 0 or H % P != 0                            */
    XS_ERR_TOO_MANY_RANKS = -5,  /* P > XS_MAX_P                                        */
    XS_ERR_ALIGNMENT = -6,       /* a device pointer is not 16-byte aligned             */
    XS_ERR_OVERLAP = -7,         /* an output buffer overlaps another output or input   */
    XS_ERR_SCALE = -8,           /* scale is NaN or infinite                            */
    XS_ERR_CUDA = -9,            /* a CUDA runtime/driver call or launch failed         */
    XS_ERR_DEVICE_TIMEOUT = -10, /* a bounded wait inside a kernel ran out; see below   */
    XS_ERR_UNSUPPORTED_DEVICE = -11, /* the current device is not sm_103 (GB300)       */
    XS_ERR_WORKSPACE = -12,      /* the workspace is smaller than required              */
    XS_ERR_LAYOUT = -13,         /* unknown output layout                               */
    XS_ERR_DEVICE_DRAIN = -14,   /* after an expired wait, a copy or MMA may still have
                                    been in flight when a CTA freed its tensor memory   */
    XS_ERR_DEVICE_BOUNDS = -15,  /* a kernel's index check failed; the access was skipped */
    XS_ERR_UNAVAILABLE = -16     /* reserved for a variant disabled in a build; no entry
                                    point of this build returns it                      */
};

/* Output layouts of xs_attn_fwd_balanced (the three layouts of the entry points
 * below: sequence shards, one contiguous tensor, Ulysses head shards). */
enum {
    XS_LAYOUT_A2A = 0,         /* outs[p]: [B, S/P, H, D], as xs_attn_a2a_fwd      */
    XS_LAYOUT_CONTIGUOUS = 1,  /* outs[0]: [B, S, H, D], as xs_attn_fwd (P ignored) */
    XS_LAYOUT_HEADS = 2        /* outs[r]: [B, S, H/P, D], as xs_attn_heads_fwd    */
};

/*
 * xs_attn_a2a_fwd -- the fused path.
 *
 * Computes O = softmax(Q K^T * scale) V for q, k, v of shape [B,S,H,D] and stores
 * every output row (b, s, h) directly into the sequence shard of its owner:
 *     p  = s / (S/P),   s' = s - p*(S/P)
 *     out_ptrs[p][b, s', h, :]   (each out_ptrs[p] is a [B, S/P, H, D] bf16 buffer)
 * This is the layout the post-attention Ulysses All-to-All produces (X-Stage,
 * abstract: tile-granular fusion of the post-attention All-to-All with
 * FlashAttention; the output-tile owner issues the stores and resumes the next
 * tile).  Every element of every shard is written exactly once.
 *
 *   q, k, v   device, bf16 [B,S,H,D], read only.
 *   out_ptrs  host array of P device pointers, each a distinct [B,S/P,H,D] bf16
 *             buffer that must not overlap q, k, v or another shard.
 *   P         1 <= P <= XS_MAX_P, S % P == 0, H % P == 0.
 *   scale     finite softmax scale (1/sqrt(D) for standard attention).
 *   stream    cudaStream_t to launch on.
 */
int xs_attn_a2a_fwd(const void* q, const void* k, const void* v, void* const* out_ptrs,
                    int B, int S, int H, int D, int P, float scale, void* stream);

/*
 * xs_attn_fwd -- the same attention kernel storing one contiguous [B,S,H,D]
 * output ("attention alone").  The arithmetic is identical to xs_attn_a2a_fwd;
 * only the destination address of each output row differs, so
 * out[b, p*S/P + s', h] == out_ptrs[p][b, s', h] bit for bit.
 */
int xs_attn_fwd(const void* q, const void* k, const void* v, void* out,
                int B, int S, int H, int D, float scale, void* stream);

/*
 * xs_attn_heads_fwd -- the same attention kernel storing the head shards a
 * Ulysses rank holds before the post-attention All-to-All:
 *     r = h / (H/P), j = h % (H/P),   heads[r][b, s, j, :]
 * each heads[r] a [B, S, H/P, D] bf16 buffer.  Together with xs_relayout_a2a
 * this is the unfused "serial" path: attention, then a separate exchange.
 */
int xs_attn_heads_fwd(const void* q, const void* k, const void* v, void* const* heads,
                      int B, int S, int H, int D, int P, float scale, void* stream);

/*
 * xs_relayout_a2a -- the separate All-to-All re-layout kernel (single GPU):
 *     out_ptrs[p][b, s', r*(H/P) + j, :] = heads[r][b, p*(S/P) + s', j, :]
 * heads: host array of P device pointers to [B,S,H/P,D] bf16 buffers;
 * out_ptrs: host array of P device pointers to [B,S/P,H,D] bf16 buffers.
 * Outputs must not overlap the inputs or each other.  Pure data movement,
 * 16-byte vector copies; bit-exact.
 */
int xs_relayout_a2a(const void* const* heads, void* const* out_ptrs,
                    int B, int S, int H, int D, int P, void* stream);

/*
 * xs_attn_ulysses_fwd -- the whole Ulysses attention step of P virtual ranks in
 * one launch, both exchanges fused.  Ulysses (DeepSpeed-Ulysses, the sequence
 * parallelism the X-Stage paper's DiT inference uses) gives every rank a
 * sequence shard of Q, K and V; a pre-attention All-to-All turns them into head
 * shards (all S rows of H/P heads), every rank runs attention on its heads, and
 * the post-attention All-to-All returns sequence shards.  Here the kernel loads
 * each Q tile and each K/V block straight from the sequence shard that holds its
 * rows (one TMA tensor map per shard), so the pre-attention exchange becomes the
 * loads, and stores the output as xs_attn_a2a_fwd does, so the post-attention
 * exchange becomes the stores.  The X-Stage summary ("Key Contributions" item 3)
 * fuses only the post-attention exchange; fusing the pre-attention one into the
 * loads is this library's extension of the same idea.
 *   q_shards, k_shards, v_shards  host arrays of P device pointers, shard p a
 *             [B, S/P, H, D] bf16 buffer holding sequence rows [p*S/P, (p+1)*S/P);
 *             read only (they may alias each other).
 *   out_shards host array of P device pointers, [B, S/P, H, D] bf16 each, the
 *             layout of xs_attn_a2a_fwd; must not overlap any input, each other
 *             or the workspace.
 *   P         1 <= P <= XS_MAX_P, H % P == 0 and (S/P) % 128 == 0 (a 128-row
 *             tile must lie in one shard), else XS_ERR_DIVISIBILITY.
 *   workspace, workspace_bytes  as in xs_attn_fwd_balanced (NULL, 0: whole
 *             tiles only).
 * Arithmetic identical to xs_attn_a2a_fwd on the concatenated inputs: the
 * outputs are bit-identical to it for the same schedule.
 */
int xs_attn_ulysses_fwd(const void* const* q_shards, const void* const* k_shards, const void* const* v_shards,
                        void* const* out_shards, int B, int S, int H, int D, int P, float scale,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * xs_attn_ulysses_rank_fwd -- the attention of ONE Ulysses rank with the
 * post-attention All-to-All fused into its epilogue, in the form a multi-GPU
 * deployment runs (X-Stage, abstract; gist.science technical summary, "Key
 * Contributions" item 3: the output-tile owner stores each finished tile to the
 * rank that owns the tile's sequence block and resumes its next tile).  Rank
 * `rank` of P holds, after the pre-attention exchange, all S rows of its H/P
 * heads; it computes exact attention over them and stores each output row
 * (b, s, j) straight into out_shards[s / (S/P)] at row (b, s % (S/P)) and global
 * head rank * H/P + j.  Called once per rank with every rank's pointers, the P
 * calls together fill the P sequence shards exactly as xs_attn_a2a_fwd does on
 * the whole tensors (bit for bit without a workspace).
 *   q_heads, k_heads, v_heads  device bf16 [B, S, H/P, D]: this rank's heads.
 *   out_shards  host array of P device pointers, out_shards[p] = rank p's
 *               sequence shard [B, S/P, H, D] (bf16).  Pointers into another
 *               process's memory (CUDA IPC) or a peer GPU's are plain
 *               addresses to the kernel: its 16-byte stores go there directly.
 *               The call only writes the rows of heads [rank*H/P, (rank+1)*H/P).
 *   B, S, H, D  global shape (H = total heads, H % P == 0, S % P == 0).
 *   rank        0 .. P-1.
 *   workspace, workspace_bytes  as in xs_attn_fwd_balanced, sized for H/P heads
 *               (xs_attn_workspace_bytes(B, S, H/P, D)); NULL, 0: whole tiles.
 * Completion: the stores are visible to the owners of the shards once `stream`
 * has passed the call (for other processes: after an event recorded there);
 * the library adds no flag or barrier of its own.
 * Returns XS_OK or XS_ERR_NULL / _SHAPE (rank out of range) / _HEAD_DIM /
 * _DIVISIBILITY / _TOO_MANY_RANKS / _ALIGNMENT / _OVERLAP / _SCALE /
 * _WORKSPACE / _CUDA.
 */
int xs_attn_ulysses_rank_fwd(const void* q_heads, const void* k_heads, const void* v_heads,
                             void* const* out_shards, int B, int S, int H, int D, int P, int rank,
                             float scale, void* workspace, size_t workspace_bytes, void* stream);

/*
 * xs_relayout_a2a_inverse -- the separate pre-attention All-to-All re-layout
 * (single GPU), the inverse of xs_relayout_a2a:
 *     heads[r][b, s, j, :] = seq_shards[s / (S/P)][b, s % (S/P), r*(H/P) + j, :]
 * seq_shards: host array of P device pointers to [B,S/P,H,D] bf16 buffers;
 * heads: host array of P device pointers to [B,S,H/P,D] bf16 buffers.  Outputs
 * must not overlap the inputs or each other.  Pure data movement; bit-exact.
 * With xs_attn_fwd (per rank) and xs_relayout_a2a it forms the unfused Ulysses
 * step that xs_attn_ulysses_fwd is measured against.
 */
int xs_relayout_a2a_inverse(const void* const* seq_shards, void* const* heads,
                            int B, int S, int H, int D, int P, void* stream);

/*
 * xs_attn_a2a_fwd_staged -- xs_attn_a2a_fwd for host-resident data.
 * Copies q, k, v from host memory into the caller's device buffers q_dev,
 * k_dev, v_dev, runs the fused kernel into the caller's device shards
 * out_dev[p], and copies every shard back into the host buffers out_host[p].
 * The work is pipelined over groups of heads (min(H, 8) equal groups, the first
 * and the last cut in two, since their copies are the ones no kernel hides; up
 * to 10 groups): the kernel of group g
 * runs on `stream` while the host-to-device copies of group g + 1 run on one
 * library stream and the device-to-host copies of group g - 1 on another (one
 * pitched cudaMemcpy2DAsync per tensor and group: a group's heads are a
 * contiguous run of every [.., H, D] row).  Each group's launch computes only its
 * heads (the schedule planned for them; the workspace is used when it is large
 * enough for the group's plan, else whole tiles run); the results are those of
 * xs_attn_a2a_fwd.  `stream` waits for the last copy before the call's end, and
 * the copies wait for the work queued on `stream` before the call, so the call
 * is ordered on `stream` like any other.  Host buffers should be pinned (page-
 * locked); otherwise the copies do not overlap.  They must stay alive and
 * untouched until the stream has finished.  The library keeps two streams and
 * 18 events per device for this (created at the first call, kept until exit);
 * calls from several host threads are enqueued one at a time.  Device-side
 * rules are those of xs_attn_a2a_fwd; workspace / workspace_bytes those of
 * xs_attn_fwd_balanced (NULL, 0: whole tiles).
 */
int xs_attn_a2a_fwd_staged(const void* q_host, const void* k_host, const void* v_host,
                           void* const* out_host,
                           void* q_dev, void* k_dev, void* v_dev, void* const* out_dev,
                           int B, int S, int H, int D, int P, float scale,
                           void* workspace, size_t workspace_bytes, void* stream);

/*
 * xs_attn_workspace_bytes -- device workspace that xs_attn_fwd_balanced needs
 * for this shape on the current device (0 when the tiles already fill whole
 * waves and nothing is split).  The value depends only on the device's SM
 * count, D and whether the shape splits: with G SMs it is about
 * G * (512*D + 1056) bytes (10.1 MB at D = 128 on 152 SMs).
 *   bytes  host pointer that receives the size.
 * Returns XS_OK, XS_ERR_NULL, a shape error, XS_ERR_UNSUPPORTED_DEVICE or
 * XS_ERR_CUDA.
 */
int xs_attn_workspace_bytes(int B, int S, int H, int D, size_t* bytes);

/*
 * xs_attn_fwd_balanced -- the attention kernel of the three entry points above
 * (layout XS_LAYOUT_A2A, _CONTIGUOUS or _HEADS, same outputs and rules) with
 * the last, partial wave of query tiles balanced over all SMs.
 * The kernel is persistent, one CTA per SM, and a 128-row query tile is its unit
 * of work; when the tile count is not a multiple of the SM count, the plain
 * schedule leaves SMs idle in the last wave.  Here the first
 * floor(tiles/SMs) - 1 waves run whole tiles and the key blocks of the
 * remaining tiles are divided evenly over all SMs ("stream-K"); a tile whose
 * key range is cut between two CTAs is completed by both: the later CTA writes
 * its unnormalised partial output (fp32), running max and row sum to the
 * workspace and publishes them with the launch's epoch, the earlier CTA waits
 * for them (a bounded wait) and merges:
 *     O = (O_1 2^(m_1-m) + O_2 2^(m_2-m)) / (l_1 2^(m_1-m) + l_2 2^(m_2-m)),
 *     m = max(m_1, m_2).
 * The merge reorders fp32 sums, so results agree with the plain schedule to
 * rounding, not bit for bit; the three layouts stay bit-identical to each other.
 *   workspace        device buffer, 256-byte aligned, of at least
 *                    xs_attn_workspace_bytes(B, S, H, D) bytes, not overlapping
 *                    any input or output; NULL selects the plain schedule.
 *                    Contents: scratch owned by the library during the call.
 *                    It must be zero-filled once before its first use, and it
 *                    keeps state between calls at fixed offsets from its start
 *                    (a launch count and the flags), so reuse it for any shape
 *                    at the same address.  A launch takes one more than the
 *                    launches finished on it as the epoch of its flags, and
 *                    its last CTA to finish advances the count.  No epoch is
 *                    baked into the launch arguments, so a launch captured in a
 *                    CUDA graph and replayed never mistakes an earlier replay's
 *                    flags for its own.  Two calls may share a workspace only
 *                    if they are ordered (same stream, or synchronised);
 *                    concurrent calls on one workspace race.
 *   workspace_bytes  its size in bytes; smaller than required ->
 *                    XS_ERR_WORKSPACE (nothing launched).
 * When a tile is split the kernel is launched cooperatively (all CTAs resident
 * at once); CTAs then wait for each other only through bounded waits.
 */
int xs_attn_fwd_balanced(const void* q, const void* k, const void* v, int layout, void* const* outs,
                         int B, int S, int H, int D, int P, float scale,
                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * xs_attn_fwd_balanced_noalloc -- xs_attn_fwd_balanced with the workspace taken
 * from a scratch array inside the library instead of from the caller.  The
 * X-Stage paper has no counterpart to this entry point: it exists for callers
 * that may not allocate device memory on their call path (for example a serving
 * loop that reserves all memory at start-up; cudaMalloc may fail there and
 * cudaFree synchronises the whole device), so that they need not size, allocate
 * and keep a workspace of their own.
 *   Scratch: one array of 11 MiB (11,534,336 bytes) per device, a file-scope
 *   device variable of the library, zero-filled when the library's module is
 *   loaded; nothing else must start at zero.  A shape whose workspace
 *   (xs_attn_workspace_bytes) exceeds it gets XS_ERR_WORKSPACE and nothing is
 *   launched; on a 152-SM GB300 the largest need is about 10.1 MB (D = 128).
 *   No device or host memory is allocated by the call.
 *   Setup: the first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress, which may load the library's device code); make that
 *   first call before any stream capture begins.
 *   Concurrency: all calls on a device share the one array.  Calls that may run
 *   at the same time (other streams, other host threads) race on it and give
 *   wrong results; order them (one stream, or events/synchronisation).
 * Arguments, outputs, checks and errors are those of xs_attn_fwd_balanced
 * (without workspace / workspace_bytes); the results are bit-identical to
 * xs_attn_fwd_balanced's for the same inputs.
 */
int xs_attn_fwd_balanced_noalloc(const void* q, const void* k, const void* v, int layout, void* const* outs,
                                 int B, int S, int H, int D, int P, float scale, void* stream);

/*
 * xs_attn_causal_fwd -- causal attention with the same fused output layouts:
 *     O[b,s,h,:] = sum_{t<=s} exp(x_t - m) V[b,t,h,:] / sum_{t<=s} exp(x_t - m),
 *     x_t = scale * <Q[b,s,h,:], K[b,t,h,:]>,  m = max_{t<=s} x_t,
 * i.e. query row s attends to keys 0 .. s only.  The X-Stage pages treat
 * bidirectional DiT attention and define no masked form; this variant is the
 * masked self-attention of autoregressive models, with the epilogue stores of
 * the fused Ulysses layout unchanged.
 *   layout  XS_LAYOUT_A2A (outs = P sequence shards [B, S/P, H, D]),
 *           XS_LAYOUT_CONTIGUOUS (outs[0] = one [B, S, H, D] tensor, P ignored)
 *           or XS_LAYOUT_HEADS (outs = P head shards [B, S, H/P, D]); the same
 *           buffers, ownership and checks as xs_attn_a2a_fwd, xs_attn_fwd and
 *           xs_attn_heads_fwd.
 * Query tile t (rows [128t, 128t + 128)) reads key blocks 0 .. t; the block on
 * the diagonal is masked per row.  Tiles are scheduled longest first over all
 * SMs; no workspace is used.  The three layouts are bit-identical to each
 * other.  Returns as xs_attn_a2a_fwd (XS_ERR_LAYOUT for an unknown layout);
 * asynchronous on `stream`.
 */
int xs_attn_causal_fwd(const void* q, const void* k, const void* v, int layout, void* const* outs,
                       int B, int S, int H, int D, int P, float scale, void* stream);

/*
 * xs_attn_varlen_fwd -- attention over packed variable-length sequences with the
 * same fused output layouts.  The X-Stage pages batch equal-length DiT
 * sequences and define no packed form; this is the usual variable-length batch:
 * n_seqs sequences of lengths seqlens[0..n_seqs) lie back to back along the
 * rows of one [T, H, D] tensor per operand (T = their sum; sequence i holds rows
 * [c_i, c_i + seqlens[i]), c_i = seqlens[0] + ... + seqlens[i-1]), and row s of
 * sequence i attends only to that sequence's keys:
 *     O[s,h,:] = sum_t exp(x_t - m) V[t,h,:] / sum_t exp(x_t - m),
 *     t over [c_i, c_i + seqlens[i])  (causal != 0: over [c_i, s]).
 *   q, k, v   device bf16 [T, H, D] (16-byte aligned), read only.
 *   seqlens   HOST int array of n_seqs lengths, each >= 0 (empty sequences are
 *             skipped), read before the call returns.
 *   n_seqs    1 .. 1024.
 *   causal    0: attend to the whole sequence, in one launch over all the
 *             sequences' tiles.  Any other value: the causal form, run as one
 *             launch of the causal kernel (xs_attn_causal_fwd's) per non-empty
 *             sequence, each reading that sequence's rows and storing its row s
 *             at packed row c_i + s of the layout.  (A single launch over all
 *             sequences' causal tiles ended, at 75,776 packed tokens in four
 *             sequences with 40 heads, in an unspecified launch failure whose
 *             cause is not established; that form is not launched.)  Each
 *             launch is a separate kernel, so many short sequences pay one
 *             launch each.  Sequences whose launch fills every SM run on
 *             `stream` one after the other; shorter ones run on the two library
 *             streams of xs_attn_a2a_fwd_staged (forked from and joined back to
 *             `stream`), so that they fill the SMs the long launches leave idle;
 *             the call stays ordered on `stream`.
 *   layout    XS_LAYOUT_A2A: outs = P sequence shards [T/P, H, D] of the packed
 *             rows (shard p holds rows [p*T/P, (p+1)*T/P), whichever sequences
 *             they belong to; T % P == 0 and H % P == 0);
 *             XS_LAYOUT_CONTIGUOUS: outs[0] = [T, H, D] (P ignored);
 *             XS_LAYOUT_HEADS: outs = P head shards [T, H/P, D].
 * Limits: at most 4096 query tiles of 128 rows in all (sum of ceil(len/128));
 * a sequence at most 8,388,608 rows; tiles x H at most 2^31 - 1.  The library builds the tile list on the
 * host (longest first) and passes it in the launch's parameter space (about
 * 20 KB): the call allocates no device memory.  With equal lengths the result is
 * bit-identical to xs_attn_a2a_fwd on the [B, S, H, D] view of the same memory.
 * Returns XS_OK; XS_ERR_NULL (q, k, v, outs, an out pointer or seqlens);
 * XS_ERR_SHAPE (n_seqs out of range, a negative or too long length, lengths not
 * summing to T, too many tiles or tiles x H, H < 1); the checks of
 * xs_attn_a2a_fwd otherwise (with B = 1, S = T); asynchronous on `stream`.
 */
int xs_attn_varlen_fwd(const void* q, const void* k, const void* v, const int* seqlens, int n_seqs,
                       int causal, int layout, void* const* outs, int T, int H, int D, int P, float scale,
                       void* stream);

/*
 * xs_burst_gap -- Burst-Gap microbenchmark of the store path the fused epilogue
 * uses (SM -> L2 -> HBM on one GPU).  X-Stage (arXiv 2607.23264), gist.science
 * technical summary, "Methodology: The X-Stage Abstraction and Burst-Gap
 * Model": K producers issue bursts of stores of aggregate volume V separated
 * by a producer-side gap G; the sender-visible issue time of a burst is
 *     T_iss(G; K, V) = max(T0_iss(K, V), V / R - G),
 * with T0_iss the backpressure-free issue time, R the effective drain rate and
 * Q the outstanding capacity of the path.  This kernel produces the raw issue
 * times; the fit is dit_attention_ulysses_gb300/burst_gap.py.
 *   dst         device buffer the bursts are stored to (16-byte aligned),
 *               dst_bytes long; producer windows of burst_bytes/producers bytes
 *               rotate through it (use one larger than L2 to reach HBM).
 *               Contents afterwards: the 16-byte pattern
 *               {i, r, c, i ^ 0x9E3779B9} at chunk i of the window of burst r,
 *               producer c (later bursts overwrite earlier ones).
 *   producers   K, 1 <= K <= the SM count (one CTA per SM).
 *   burst_bytes V, a multiple of 16 * producers; dst_bytes / (V/K) >= K.
 *   bursts      1 <= bursts <= 65536;  gap_ns  0 <= G <= 1e8, bursts * G <= 1e10.
 *   lead_ns     0 <= lead_ns <= 1e8: a spin before the first burst (the path
 *               drains from earlier work while the SMs stay busy).
 *   issue_ns    device int64 array [bursts][producers] (8-byte aligned, not
 *               inside dst): the issue time of burst r at producer c, from
 *               before its first store to after its last thread issued its
 *               last store (%globaltimer, ns).
 * Returns XS_OK or XS_ERR_NULL / _SHAPE / _ALIGNMENT / _OVERLAP /
 * _UNSUPPORTED_DEVICE / _CUDA; asynchronous on `stream`.
 */
int xs_burst_gap(void* dst, size_t dst_bytes, int producers, size_t burst_bytes, int bursts,
                 long long lead_ns, long long gap_ns, long long* issue_ns, void* stream);

/*
 * xs_attn_get_device_error -- synchronises `stream`, then reads and clears the
 * library's device error state on the current device (the error word, the
 * record of the first error and the drain flag).  Returns XS_OK;
 * XS_ERR_DEVICE_DRAIN if, after an expired wait, a CTA's bounded wait for its
 * own copies or MMAs in flight also gave up (the CTA then freed its tensor
 * memory and exited with them possibly outstanding: treat the context as
 * suspect); else XS_ERR_DEVICE_TIMEOUT if a bounded wait inside a kernel expired
 * (the kernel abandoned its work and returned; its outputs are unspecified);
 * XS_ERR_DEVICE_BOUNDS if an index check inside a kernel failed (the access was
 * skipped: an internal error); or XS_ERR_CUDA if synchronisation itself failed.
 */
int xs_attn_get_device_error(void* stream);

/*
 * xs_attn_get_device_error_info -- as xs_attn_get_device_error (same return
 * value, same clearing), and also copies the record of the first device error
 * since the last clear into info[0 .. n_info) (n_info <= 8; missing fields are
 * not written; all zero when there was none):
 *   info[0]  kind: 0 none, 1 expired wait, 3 failed index check
 *   info[1]  CTA index, info[2] warp, info[3] lane of the thread that recorded it
 *   info[4]  site: for a wait, the shared-memory address of its mbarrier (the
 *            split-tile flags of CTA slot s: 0x40000 + s); for an index check,
 *            1 = packed-sequence table entry, 2 = destination shard
 *   info[5..7]  details: for a wait, the phase parity, the piece index and the
 *            key block it waited in (-1: none); for an index check, the values
 *            that failed it.
 *   info  host array of n_info ints (may be NULL when n_info == 0).
 */
int xs_attn_get_device_error_info(void* stream, int* info, int n_info);

/* Human-readable text for an XS_* code (static storage; never NULL). */
const char* xs_attn_error_string(int code);

/*
 * The most recent CUDA error seen by the library on this thread (a
 * cudaError_t value; 0 if none), for reports after XS_ERR_CUDA.
 */
int xs_attn_last_cuda_error(void);

/* Library version as major*10000 + minor*100 + patch. */
int xs_attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* XSATTN_H */
