// Fused non-causal attention + post-attention Ulysses All-to-All store, sm_103a.
//
// X-Stage (arXiv 2607.23264), abstract and the gist.science technical summary,
// "Key Contributions" item 3 (FlashAttention-A2A piggybacking): the role that
// owns an output tile stores it straight to the rank owning the tile's sequence
// block and immediately resumes the next tile's Q-loop; no dedicated
// communication warp and no separate All-to-All kernel.  On one GPU the ranks are
// P device buffers, so the "remote store" is a 16-byte vector store into the
// owner's [B, S/P, H, D] shard.
//
// Kernel organisation (one persistent CTA per SM, 10 warps):
//   warps 0-3  softmax + epilogue for Q tile 0 of the current work unit
//   warps 4-7  softmax + epilogue for Q tile 1
//   warp  8    TMA producer: Q tiles, then the K/V ring (K_0, V_0, K_1, V_1, ...)
//   warp  9    tcgen05 MMA issuer (one elected lane) and TMEM owner
// A work unit is (b, h, 256 query rows) = two 128-row Q tiles that share every
// K/V block.  MMA order per K/V block j:  PV0_{j-1}, S0_j, PV1_{j-1}, S1_j, so
// each tile's softmax runs while the tensor core works on the other tile.
//
// TMEM (512 columns x 128 lanes, fp32):
//   [  0,128)  S0 (scores of tile 0); P0 (bf16, 2 per column) overwrites [0,64)
//   [128,256)  S1 / P1
//   [256,256+D) O0 accumulator,  [256+D, 256+2D) O1 accumulator
//
// Shared memory (128-byte swizzled, 1024-byte aligned):
//   Q0, Q1 tiles [128 x D] as D/64 panels of [128 rows x 128 B]
//   KV ring of NS stages, each one K or V block [128 x D] in the same panel form
//   mbarriers, TMEM base address, abort flag
//
// Softmax (per row, one thread per row, base-2 domain with c = scale*log2(e)):
//   m_blk = max_j s_j * c;  m_new = max(m_run, m_blk)
//   lazy rescale: only if m_new - m_run > 8 is the running max moved (and O, l
//   multiplied by 2^(m_run - m_new)); otherwise the stale max is kept, which
//   bounds p by 2^8 and changes nothing after the final division by l.
//   p_j = 2^(s_j*c - m),  l = l*alpha + sum_j p_j,  P -> bf16 into TMEM.
// Epilogue: O / l -> bf16 -> st.global.v4 into the destination row.
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

namespace {

constexpr int BLOCK_M = 128;
constexpr int BLOCK_N = 128;
constexpr int Q_TILES = 2;
constexpr int UNIT_ROWS = BLOCK_M * Q_TILES;
constexpr int NUM_THREADS = 320;
constexpr int WARP_TMA = 8;
constexpr int WARP_MMA = 9;
constexpr uint32_t TMEM_COLS = 512;
constexpr int PANEL_BYTES = BLOCK_M * 128;  // 128 rows x 64 bf16
constexpr float RESCALE_THRESHOLD = 8.0f;   // log2 units

template <int D>
struct Cfg {
    static constexpr int TILE_BYTES = BLOCK_M * D * 2;
    static constexpr int PANELS = D / 64;
    static constexpr int KV_STAGES = (D == 128) ? 5 : 8;
    static constexpr int Q_OFF = 0;
    static constexpr int KV_OFF = Q_TILES * TILE_BYTES;
    static constexpr int BAR_OFF = KV_OFF + KV_STAGES * TILE_BYTES;
    // barrier indices
    static constexpr int B_Q_FULL = 0;                 // [2]
    static constexpr int B_Q_FREE = 2;                 // [2]
    static constexpr int B_S_READY = 4;                // [2]
    static constexpr int B_P_READY = 6;                // [2]
    static constexpr int B_O_FINAL = 8;                // [2]
    static constexpr int B_O_FREE = 10;                // [2]
    static constexpr int B_DRAIN = 12;                 // [1]
    static constexpr int B_KV_FULL = 13;               // [NS]
    static constexpr int B_KV_FREE = 13 + KV_STAGES;   // [NS]
    static constexpr int NUM_BARS = 13 + 2 * KV_STAGES;
    static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
    static constexpr int SMEM_BYTES = MISC_OFF + 16;
    static constexpr int SMEM_ALLOC = SMEM_BYTES + 1024;
    static constexpr uint32_t O_COL = 256;
};

// Bounded wait, executed by a whole warp; the result is warp-uniform.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t timeout_ns) {
    bool ok = mbar_try_wait(bar, parity);
    if (!__all_sync(0xffffffffu, ok)) {
        const uint64_t t0 = globaltimer_ns();
        while (!ok) {
            for (int i = 0; i < 32 && !ok; ++i) ok = mbar_try_wait(bar, parity);
            if (ok) break;
            if (*abort_flag) break;
            if (globaltimer_ns() - t0 > timeout_ns) {
                *abort_flag = 1;
                atomicCAS(&g_device_error, 0, XS_DEVICE_TIMEOUT_CODE);
                break;
            }
        }
        ok = __all_sync(0xffffffffu, ok);
    }
    return ok;
}

template <int D>
__device__ __forceinline__ void decode_unit(int u, const AttnArgs& a, int& b, int& h, int& qu) {
    qu = u % a.n_qu;
    const int bh = u / a.n_qu;
    h = bh % a.H;
    b = bh / a.H;
}

// ---------------------------------------------------------------- producer
template <int D>
__device__ void producer_role(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                              const AttnArgs& a, uint8_t* smem, uint32_t bar0, volatile int* abort_flag) {
    using C = Cfg<D>;
    const bool leader = lane_id() == 0;
    const uint32_t sbase = smem_addr(smem);
    auto bar = [&](int i) { return bar0 + static_cast<uint32_t>(i) * 8u; };
    uint32_t item = 0;
    int u_iter = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x, ++u_iter) {
        int b, h, qu;
        decode_unit<D>(u, a, b, h, qu);
        for (int t = 0; t < Q_TILES && ok; ++t) {
            if (u_iter > 0) ok = warp_wait(bar(C::B_Q_FREE + t), (u_iter - 1) & 1, abort_flag, a.timeout_ns);
            if (!ok) break;
            if (leader) {
                int s0 = qu * UNIT_ROWS + t * BLOCK_M;
                if (s0 >= a.S) s0 = 0;  // tile entirely past the end: load any in-bounds rows, never stored
                mbar_arrive_expect_tx(bar(C::B_Q_FULL + t), C::TILE_BYTES);
                for (int pnl = 0; pnl < C::PANELS; ++pnl)
                    tma_load_4d(sbase + C::Q_OFF + t * C::TILE_BYTES + pnl * PANEL_BYTES, tq,
                                bar(C::B_Q_FULL + t), pnl * 64, h, s0, b);
            }
            __syncwarp();
        }
        for (int j = 0; j < a.n_kv && ok; ++j) {
            for (int kv = 0; kv < 2 && ok; ++kv, ++item) {
                const uint32_t stage = item % C::KV_STAGES;
                const uint32_t round = item / C::KV_STAGES;
                if (round > 0) ok = warp_wait(bar(C::B_KV_FREE + stage), (round - 1) & 1, abort_flag, a.timeout_ns);
                if (!ok) break;
                if (leader) {
                    mbar_arrive_expect_tx(bar(C::B_KV_FULL + stage), C::TILE_BYTES);
                    for (int pnl = 0; pnl < C::PANELS; ++pnl)
                        tma_load_4d(sbase + C::KV_OFF + stage * C::TILE_BYTES + pnl * PANEL_BYTES,
                                    kv ? tv : tk, bar(C::B_KV_FULL + stage), pnl * 64, h, j * BLOCK_N, b);
                }
                __syncwarp();
            }
        }
    }
    if (!ok) {
        // Let the copies already issued land before the CTA exits: wait (bounded)
        // for the newest phase of every ring stage that was used.
        volatile int no_abort = 0;
        for (uint32_t back = 1; back <= C::KV_STAGES && back <= item; ++back) {
            const uint32_t it = item - back;
            warp_wait(bar(C::B_KV_FULL + it % C::KV_STAGES), (it / C::KV_STAGES) & 1, &no_abort, 20000000ull);
        }
    }
}

// --------------------------------------------------------------------- MMA
template <int D>
__device__ void mma_role(const AttnArgs& a, uint8_t* smem, uint32_t bar0, uint32_t tmem_base,
                         volatile int* abort_flag) {
    using C = Cfg<D>;
    const bool leader = lane_id() == 0;
    const uint32_t sbase = smem_addr(smem);
    auto bar = [&](int i) { return bar0 + static_cast<uint32_t>(i) * 8u; };
    constexpr uint32_t IDESC_QK = idesc_bf16_f32(BLOCK_M, BLOCK_N, 0);
    constexpr uint32_t IDESC_PV = idesc_bf16_f32(BLOCK_M, D, 1);

    // Q / K operand (K-major, 128-B swizzle): k-step kk covers 16 columns of D.
    auto kmajor_desc = [&](uint32_t tile_addr, int kk) {
        return smem_desc_sw128(tile_addr + (kk >> 2) * PANEL_BYTES + (kk & 3) * 32, 16, 1024);
    };
    // V operand (MN-major = D contiguous, 128-B swizzle): k-step kk covers 16 keys;
    // 8-key groups are 1024 B apart (SBO), 64-wide D panels PANEL_BYTES apart (LBO).
    auto vdesc = [&](uint32_t tile_addr, int kk) {
        return smem_desc_sw128(tile_addr + kk * 2048, PANEL_BYTES, 1024);
    };
    auto s_tmem = [&](int t) { return tmem_base + static_cast<uint32_t>(t) * 128u; };
    auto o_tmem = [&](int t) { return tmem_base + C::O_COL + static_cast<uint32_t>(t) * D; };

    uint32_t item = 0;
    uint32_t p_count[2] = {0, 0};
    int u_iter = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x, ++u_iter) {
        const int n = a.n_kv;
        for (int t = 0; t < Q_TILES && ok; ++t)
            ok = warp_wait(bar(C::B_Q_FULL + t), u_iter & 1, abort_flag, a.timeout_ns);
        if (!ok) break;
        // K_0 -> S_t_0 for both tiles
        uint32_t k_stage = item % C::KV_STAGES;
        ok = warp_wait(bar(C::B_KV_FULL + k_stage), (item / C::KV_STAGES) & 1, abort_flag, a.timeout_ns);
        if (!ok) break;
        ++item;
        tc_fence_after();
        if (leader) {
            const uint32_t kaddr = sbase + C::KV_OFF + k_stage * C::TILE_BYTES;
            for (int t = 0; t < Q_TILES; ++t) {
                const uint32_t qaddr = sbase + C::Q_OFF + t * C::TILE_BYTES;
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(s_tmem(t), kmajor_desc(qaddr, kk), kmajor_desc(kaddr, kk), IDESC_QK, kk > 0);
                mma_commit(bar(C::B_S_READY + t));
                if (n == 1) mma_commit(bar(C::B_Q_FREE + t));
            }
            mma_commit(bar(C::B_KV_FREE + k_stage));
        }
        __syncwarp();
        for (int j = 0; j < n && ok; ++j) {
            const uint32_t v_stage = item % C::KV_STAGES;
            ok = warp_wait(bar(C::B_KV_FULL + v_stage), (item / C::KV_STAGES) & 1, abort_flag, a.timeout_ns);
            if (!ok) break;
            ++item;
            const bool has_next = (j + 1) < n;
            k_stage = item % C::KV_STAGES;
            const uint32_t k_round = item / C::KV_STAGES;
            if (has_next) ++item;
            for (int t = 0; t < Q_TILES && ok; ++t) {
                ok = warp_wait(bar(C::B_P_READY + t), p_count[t] & 1, abort_flag, a.timeout_ns);
                ++p_count[t];
                if (ok && j == 0 && u_iter > 0)
                    ok = warp_wait(bar(C::B_O_FREE + t), (u_iter - 1) & 1, abort_flag, a.timeout_ns);
                if (!ok) break;
                tc_fence_after();
                if (leader) {
                    const uint32_t vaddr = sbase + C::KV_OFF + v_stage * C::TILE_BYTES;
                    for (int kk = 0; kk < BLOCK_N / 16; ++kk)
                        mma_ts(o_tmem(t), s_tmem(t) + kk * 8, vdesc(vaddr, kk), IDESC_PV, (j > 0) || (kk > 0));
                    if (j == n - 1) mma_commit(bar(C::B_O_FINAL + t));
                    if (t == Q_TILES - 1) mma_commit(bar(C::B_KV_FREE + v_stage));
                }
                __syncwarp();
                if (has_next) {
                    if (t == 0) {
                        ok = warp_wait(bar(C::B_KV_FULL + k_stage), k_round & 1, abort_flag, a.timeout_ns);
                        if (!ok) break;
                        tc_fence_after();
                    }
                    if (leader) {
                        const uint32_t kaddr = sbase + C::KV_OFF + k_stage * C::TILE_BYTES;
                        const uint32_t qaddr = sbase + C::Q_OFF + t * C::TILE_BYTES;
                        for (int kk = 0; kk < D / 16; ++kk)
                            mma_ss(s_tmem(t), kmajor_desc(qaddr, kk), kmajor_desc(kaddr, kk), IDESC_QK, kk > 0);
                        mma_commit(bar(C::B_S_READY + t));
                        if (j + 1 == n - 1) mma_commit(bar(C::B_Q_FREE + t));
                        if (t == Q_TILES - 1) mma_commit(bar(C::B_KV_FREE + k_stage));
                    }
                    __syncwarp();
                }
            }
        }
    }
    // Drain: every MMA this warp issued has completed once B_DRAIN flips.
    if (leader) mma_commit(bar(C::B_DRAIN));
    __syncwarp();
    volatile int no_abort = 0;
    warp_wait(bar(C::B_DRAIN), 0, &no_abort, ok ? a.timeout_ns : 20000000ull);
}

// ------------------------------------------------------- softmax + epilogue
template <int D>
__device__ void softmax_role(const AttnArgs& a, uint32_t bar0, uint32_t tmem_base, volatile int* abort_flag) {
    using C = Cfg<D>;
    const int warp = threadIdx.x >> 5;
    const int t = warp >> 2;                  // Q tile of this warpgroup
    const int quarter = warp & 3;             // TMEM lane quarter this warp may access
    const int row = quarter * 32 + static_cast<int>(lane_id());
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t s_t = tmem_base + lane_off + static_cast<uint32_t>(t) * 128u;
    const uint32_t o_t = tmem_base + lane_off + C::O_COL + static_cast<uint32_t>(t) * D;
    auto bar = [&](int i) { return bar0 + static_cast<uint32_t>(i) * 8u; };
    const float c = a.c;

    uint32_t s_count = 0;
    int u_iter = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x, ++u_iter) {
        int b, h, qu;
        decode_unit<D>(u, a, b, h, qu);
        float m_run = 0.0f, l_run = 0.0f;
        for (int j = 0; j < a.n_kv; ++j) {
            ok = warp_wait(bar(C::B_S_READY + t), s_count & 1, abort_flag, a.timeout_ns);
            ++s_count;
            if (!ok) break;
            tc_fence_after();
            uint32_t sr[4][32];
#pragma unroll
            for (int q = 0; q < 4; ++q) tmem_ld32(s_t + q * 32, sr[q]);
            tmem_wait_ld();
            const int valid = a.S - j * BLOCK_N;  // keys of this block inside the sequence
            const bool tail = valid < BLOCK_N;
            if (tail) {
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (q * 32 + i >= valid) sr[q][i] = 0xff800000u;  // -inf
            }
            float mx = __uint_as_float(sr[0][0]);
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int i = 0; i < 32; ++i) mx = fmaxf(mx, __uint_as_float(sr[q][i]));
            const float m_blk = mx * c;
            float m_use, alpha = 1.0f;
            bool rescale = false;
            if (j == 0) {
                m_use = m_blk;
            } else {
                const float m_new = fmaxf(m_run, m_blk);
                if (m_new - m_run > RESCALE_THRESHOLD) {
                    m_use = m_new;
                    alpha = ex2_approx(m_run - m_new);
                    rescale = true;
                } else {
                    m_use = m_run;
                }
            }
            const float neg_m = -m_use;
            float sum = 0.0f;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int q = half * 2 + (i >> 4);
                    const int e = (i & 15) * 2;
                    float p0 = ex2_approx(fmaf(__uint_as_float(sr[q][e]), c, neg_m));
                    float p1 = ex2_approx(fmaf(__uint_as_float(sr[q][e + 1]), c, neg_m));
                    if (tail) {
                        const int col = q * 32 + e;
                        if (col >= valid) p0 = 0.0f;
                        if (col + 1 >= valid) p1 = 0.0f;
                    }
                    sum += p0 + p1;
                    pk[i] = pack_bf16x2(p0, p1);
                }
                tmem_st32(s_t + half * 32, pk);
            }
            if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
                for (int q = 0; q < D / 32; ++q) {
                    uint32_t orr[32];
                    tmem_ld32(o_t + q * 32, orr);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
                    tmem_st32(o_t + q * 32, orr);
                }
            }
            l_run = l_run * alpha + sum;
            m_run = m_use;
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(C::B_P_READY + t));
        }
        if (!ok) break;
        // ---- epilogue: the owner of this tile stores it to the destination shard
        ok = warp_wait(bar(C::B_O_FINAL + t), u_iter & 1, abort_flag, a.timeout_ns);
        if (!ok) break;
        tc_fence_after();
        const int s_row = qu * UNIT_ROWS + t * BLOCK_M + row;
        const bool store = s_row < a.S;
        __nv_bfloat16* dst = nullptr;
        if (store) {
            const int p = s_row / a.epi.Sl + h / a.epi.Hl;
            const int s_dst = s_row % a.epi.Sl;
            const int h_dst = h % a.epi.Hl;
            dst = reinterpret_cast<__nv_bfloat16*>(a.epi.ptr[p]) +
                  ((static_cast<size_t>(b) * a.epi.Sl + s_dst) * a.epi.Hl + h_dst) * D;
        }
        const float inv_l = 1.0f / l_run;
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
            uint32_t orr[32];
            tmem_ld32(o_t + q * 32, orr);
            tmem_wait_ld();
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                w[i] = pack_bf16x2(__uint_as_float(orr[2 * i]) * inv_l, __uint_as_float(orr[2 * i + 1]) * inv_l);
            if (store) {
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4)
                    st_global_v4(dst + q * 32 + v4 * 8, w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
            }
        }
        tc_fence_before();
        mbar_arrive(bar(C::B_O_FREE + t));
    }
}

template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_a2a_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ AttnArgs args) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t bar0 = smem_addr(smem + C::BAR_OFF);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);
    const int warp = threadIdx.x >> 5;

    if (threadIdx.x == 0) {
        for (int t = 0; t < Q_TILES; ++t) {
            mbar_init(bar0 + 8 * (C::B_Q_FULL + t), 1);
            mbar_init(bar0 + 8 * (C::B_Q_FREE + t), 1);
            mbar_init(bar0 + 8 * (C::B_S_READY + t), 1);
            mbar_init(bar0 + 8 * (C::B_P_READY + t), 128);
            mbar_init(bar0 + 8 * (C::B_O_FINAL + t), 1);
            mbar_init(bar0 + 8 * (C::B_O_FREE + t), 128);
        }
        mbar_init(bar0 + 8 * C::B_DRAIN, 1);
        for (int s = 0; s < C::KV_STAGES; ++s) {
            mbar_init(bar0 + 8 * (C::B_KV_FULL + s), 1);
            mbar_init(bar0 + 8 * (C::B_KV_FREE + s), 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == WARP_TMA && lane_id() == 0) {
        tma_prefetch_desc(&tmap_q);
        tma_prefetch_desc(&tmap_k);
        tma_prefetch_desc(&tmap_v);
    }
    if (warp == WARP_MMA) {
        tmem_alloc(smem_addr(tmem_holder), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp < 8) {
        softmax_role<D>(args, bar0, tmem_base, abort_flag);
    } else if (warp == WARP_TMA) {
        producer_role<D>(&tmap_q, &tmap_k, &tmap_v, args, smem, bar0, abort_flag);
    } else {
        mma_role<D>(args, smem, bar0, tmem_base, abort_flag);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == WARP_MMA) tmem_dealloc(tmem_base, TMEM_COLS);
}

}  // namespace

template <int D>
int attn_smem_bytes() {
    return Cfg<D>::SMEM_ALLOC;
}

template <int D>
cudaError_t launch_attn(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const AttnArgs& args,
                        int grid, cudaStream_t stream) {
    auto kern = attn_a2a_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    kern<<<grid, NUM_THREADS, Cfg<D>::SMEM_ALLOC, stream>>>(tq, tk, tv, args);
    return cudaGetLastError();
}

template int attn_smem_bytes<64>();
template int attn_smem_bytes<128>();
template cudaError_t launch_attn<64>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const AttnArgs&, int,
                                     cudaStream_t);
template cudaError_t launch_attn<128>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const AttnArgs&,
                                      int, cudaStream_t);

cudaError_t read_and_clear_device_error(int* value) {
    int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(value, g_device_error, sizeof(int));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
}

}  // namespace xs
