// C ABI of the fused attention + Ulysses All-to-All layout library.
//
// Host-side argument validation (everything is checked before any CUDA call, so
// an invalid call launches nothing), TMA tensor-map encoding, and launches.
// The declarations and their contracts are in include/xsattn.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <vector>

#include "../../include/xsattn.h"
#include "kernels.h"

namespace {

thread_local int g_last_cuda_error = 0;

int cuda_fail(cudaError_t e) {
    g_last_cuda_error = static_cast<int>(e);
    return XS_ERR_CUDA;
}

struct DeviceInfo {
    bool known = false;
    int sms = 0;
    int major = 0;
    int minor = 0;
    int coop = 0;   // cooperative launches supported
};

constexpr int MAX_DEVICES = 64;
std::mutex g_dev_mutex;
DeviceInfo g_dev[MAX_DEVICES];

int device_info(DeviceInfo* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= MAX_DEVICES) return XS_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceInfo& d = g_dev[dev];
    if (!d.known) {
        if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
            return cuda_fail(e);
        if ((e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
            return cuda_fail(e);
        if ((e = cudaDeviceGetAttribute(&d.coop, cudaDevAttrCooperativeLaunch, dev)) != cudaSuccess)
            return cuda_fail(e);
        d.known = true;
    }
    *out = d;
    if (d.major != 10 || d.minor != 3) return XS_ERR_UNSUPPORTED_DEVICE;
    return XS_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

int get_encoder(PFN_cuTensorMapEncodeTiled_v12000* fn) {
    std::call_once(g_encode_once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
        if (g_encode_err == cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    if (!g_encode) return cuda_fail(g_encode_err != cudaSuccess ? g_encode_err : cudaErrorSymbolNotFound);
    *fn = g_encode;
    return XS_OK;
}

// [B, S, H, D] bf16 as a 4-D tensor (D, H, S, B); box = 64 channels x 1 head x 128 rows.
int encode_bshd(CUtensorMap* m, const void* base, int B, int S, int H, int D) {
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    int rc = get_encoder(&enc);
    if (rc != XS_OK) return rc;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(S),
                                static_cast<cuuint64_t>(B)};
    const cuuint64_t row = static_cast<cuuint64_t>(D) * 2;
    const cuuint64_t strides[3] = {row, row * H, row * H * S};
    const cuuint32_t box[4] = {64, 1, 128, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
    return XS_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};

bool overlaps(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

// Shape checks shared by every attention entry point.
int check_shape(int B, int S, int H, int D, int P, bool need_div) {
    if (B < 1 || S < 1 || H < 1 || P < 1) return XS_ERR_SHAPE;
    if (D != 64 && D != 128) return XS_ERR_HEAD_DIM;
    if (P > XS_MAX_P) return XS_ERR_TOO_MANY_RANKS;
    if (need_div && (S % P != 0 || H % P != 0)) return XS_ERR_DIVISIBILITY;
    // sizes: elements per tensor and the work-unit count must fit the kernels' index types
    const int64_t elems = static_cast<int64_t>(B) * S * H * D;
    if (elems > (int64_t(1) << 40)) return XS_ERR_SHAPE;
    const int64_t units = static_cast<int64_t>(B) * H * ((S + 127) / 128);
    if (units > INT32_MAX) return XS_ERR_SHAPE;
    return XS_OK;
}

int check_scale(float scale) {
    if (!std::isfinite(scale) || scale < 0.0f) return XS_ERR_SCALE;
    return XS_OK;
}

// Outputs must be pairwise disjoint and disjoint from every input.
int check_disjoint(const Range* outs, int n_out, const Range* ins, int n_in) {
    for (int i = 0; i < n_out; ++i) {
        for (int j = i + 1; j < n_out; ++j)
            if (overlaps(outs[i], outs[j])) return XS_ERR_OVERLAP;
        for (int j = 0; j < n_in; ++j)
            if (overlaps(outs[i], ins[j])) return XS_ERR_OVERLAP;
    }
    return XS_OK;
}

Range range_of(const void* p, int64_t bytes) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Range{lo, lo + static_cast<uintptr_t>(bytes)};
}

// Validation of (q, k, v, P output buffers of out_bytes each).
int validate_attn(const void* q, const void* k, const void* v, void* const* outs, int n_out, int B, int S, int H,
                  int D, int P, float scale, int64_t out_bytes, bool need_div) {
    if (!q || !k || !v || !outs) return XS_ERR_NULL;
    int rc = check_shape(B, S, H, D, P, need_div);
    if (rc != XS_OK) return rc;
    for (int i = 0; i < n_out; ++i)
        if (!outs[i]) return XS_ERR_NULL;
    if ((rc = check_scale(scale)) != XS_OK) return rc;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return XS_ERR_ALIGNMENT;
    for (int i = 0; i < n_out; ++i)
        if (!aligned16(outs[i])) return XS_ERR_ALIGNMENT;
    const int64_t in_bytes = static_cast<int64_t>(B) * S * H * D * 2;
    Range ins[3] = {range_of(q, in_bytes), range_of(k, in_bytes), range_of(v, in_bytes)};
    Range o[XS_MAX_P];
    for (int i = 0; i < n_out; ++i) o[i] = range_of(outs[i], out_bytes);
    return check_disjoint(o, n_out, ins, 3);
}

// Limit for every wait inside the kernels.  One second by default: no single
// wait of a healthy launch takes more than microseconds.  XSATTN_WAIT_TIMEOUT_NS
// overrides it (a test sets 0 to make the first unfinished wait expire and
// check that the launch reports XS_ERR_DEVICE_TIMEOUT and the context stays
// usable).
unsigned long long timeout_ns() {
    const char* env = std::getenv("XSATTN_WAIT_TIMEOUT_NS");
    if (env && *env) {
        char* end = nullptr;
        const unsigned long long v = std::strtoull(env, &end, 10);
        if (end && *end == '\0') return v;
    }
    return 1000000000ull;
}

// Work schedule of one attention launch.  Plain: grid = min(tiles, SMs), tile
// u runs whole on CTA u % grid.  Balanced (needs a workspace): the whole waves
// of tiles run as in the plain schedule, and the key-block iterations of the
// tiles left over (tiles % SMs of them) are divided evenly over up to SMs CTAs,
// at least MIN_PIECE blocks each; a tile cut among CTAs is merged in the kernel
// through the workspace.  Used only when it shortens the last wave by at least
// max(MIN_GAIN, n/8) key blocks per CTA.
struct Plan {
    int grid = 0;
    bool split = false;
    int dp_tiles = 0;
    int sk_ctas = 0;
    long long sk_iters = 0;
    size_t off_count = 0, off_flag = 0, off_ml = 0, off_o = 0, ws_bytes = 0;   // workspace layout (split only)
};

constexpr long long MIN_PIECE = 8;    // key blocks per CTA range, at least
constexpr long long MIN_GAIN = 16;    // key blocks a split must save per CTA, at least

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

Plan make_plan(int B, int S, int H, int D, const DeviceInfo& dev) {
    Plan pl;
    const int n = (S + 127) / 128;
    const int tiles = B * H * n;
    const int G = dev.sms;
    pl.grid = tiles < G ? tiles : G;
    pl.dp_tiles = tiles;
    const int rem = tiles % G;
    if (!dev.coop || rem == 0) return pl;
    const long long sk = static_cast<long long>(rem) * n;
    long long ctas = sk / MIN_PIECE;
    if (ctas > G) ctas = G;
    if (ctas <= rem) return pl;   // no more CTAs busy than with whole tiles
    // Each piece of work costs a fixed start (its Q tile, the pipeline fill) and a
    // split tile its merge, a few key blocks' worth; measured on GB300 this eats
    // the gain unless a range is shorter than a tile by max(16, n/8) blocks.
    const long long range = (sk + ctas - 1) / ctas;
    const long long gain_min = n / 8 > MIN_GAIN ? n / 8 : MIN_GAIN;
    if (n - range < gain_min) return pl;
    pl.split = true;
    pl.dp_tiles = tiles - rem;
    pl.sk_iters = sk;
    pl.sk_ctas = static_cast<int>(ctas);
    pl.grid = tiles >= G ? G : pl.sk_ctas;
    // launch count [2] u32 | part_flag [SMs][8] u32 | part_ml [grid][128] float2 | part_o [grid][128][D] fp32.
    // The count and the flags come first, at offsets that depend on the device
    // only: whatever shapes share a workspace, a flag word only ever holds an
    // epoch of an earlier launch on it (or zero), never stale partial data.
    const size_t slots = static_cast<size_t>(pl.grid);
    pl.off_count = 0;
    pl.off_flag = 256;
    pl.off_ml = pl.off_flag + align256(static_cast<size_t>(G) * 8 * 4);
    pl.off_o = pl.off_ml + align256(slots * 128 * 8);
    pl.ws_bytes = pl.off_o + align256(slots * 128 * D * 4);
    return pl;
}

// ws == nullptr: plain schedule.  Otherwise the balanced schedule whenever it
// splits tiles; ws must then hold plan.ws_bytes bytes (256-byte aligned).
// Inputs: q, k, v each one [B,S,H,D] tensor, or (shards != nullptr) the P
// sequence shards [B,S/P,H,D] of each operand: shards[0..P) = q, [P..2P) = k,
// [2P..3P) = v, with (S/P) % 128 == 0.
// Causal tile order.  Tiles are dealt in waves of `grid`, in snake order; a tile of
// query tile t costs t + 1 key blocks plus a fixed start worth about 1.5 blocks
// (measured: ~3 us per tile against ~0.9 us per block).  Longest first with the
// B*H tiles of one query tile side by side balances best; head-major keeps the
// concurrent CTAs on one head's keys and values in L2.  Head-major is taken when
// its modelled makespan is within 2 % of longest-first's.  The model walks every
// tile once, so its answer is kept per (B*H, tiles per head, grid).
bool causal_order_model(int BH, int n_qt, int grid) {
    std::vector<double> lpt(grid, 0.0), hm(grid, 0.0);
    const long long units = static_cast<long long>(BH) * n_qt;
    for (long long u = 0; u < units; ++u) {
        const long long w = u / grid, p = u % grid;
        const int cta = static_cast<int>((w & 1) ? grid - 1 - p : p);
        lpt[cta] += (n_qt - u / BH) + 1.5;          // query tile n_qt-1-u/BH: n_qt-u/BH blocks
        hm[cta] += (n_qt - u % n_qt) + 1.5;         // query tile n_qt-1-u%n_qt
    }
    const double a = *std::max_element(lpt.begin(), lpt.end()), b = *std::max_element(hm.begin(), hm.end());
    return b <= 1.02 * a;
}

struct OrderKey {
    int bh, n_qt, grid;
    bool operator<(const OrderKey& o) const {
        return bh != o.bh ? bh < o.bh : n_qt != o.n_qt ? n_qt < o.n_qt : grid < o.grid;
    }
};
std::mutex g_order_mutex;
std::map<OrderKey, bool> g_order_cache;

bool causal_head_major(int BH, int n_qt, int grid) {
    if (grid < 1) return false;
    const OrderKey key{BH, n_qt, grid};
    {
        std::lock_guard<std::mutex> lock(g_order_mutex);
        auto it = g_order_cache.find(key);
        if (it != g_order_cache.end()) return it->second;
    }
    const bool hm = causal_order_model(BH, n_qt, grid);
    std::lock_guard<std::mutex> lock(g_order_mutex);
    if (g_order_cache.size() >= 256) g_order_cache.clear();
    g_order_cache[key] = hm;
    return hm;
}

// causal: row s attends to keys 0 .. s (one tensor per operand, plain schedule
// in the kernel's causal tile order; ws is not used).
// Head range: the launch computes heads [h0, h0 + Hg) of input tensors with H
// heads (Hg = 0: all of them) and stores head h0 + h at head h0_out + h of the
// output layout (h0_out < 0: the same as h0); the schedule is planned for the
// Hg heads.  ws_optional: a workspace too small for the plan selects whole tiles
// instead of an error.
int run_attention(const void* q, const void* k, const void* v, const void* const* shards, int P,
                  const xs::EpiParams& epi, int B, int S, int H, int D, float scale, void* ws, size_t ws_bytes,
                  cudaStream_t stream, bool causal = false, int h0 = 0, int Hg = 0, bool ws_optional = false,
                  int h0_out = -1) {
    DeviceInfo dev;
    int rc = device_info(&dev);
    if (rc != XS_OK) return rc;
    const int Hw = Hg > 0 ? Hg : H;
    const Plan pl = make_plan(B, S, Hw, D, dev);
    bool split = !causal && ws != nullptr && pl.split;
    if (split && ws_bytes < pl.ws_bytes) {
        if (!ws_optional) return XS_ERR_WORKSPACE;
        split = false;
    }
    xs::AttnArgs a;
    std::memset(&a, 0, sizeof a);
    a.B = B;
    a.S = S;
    a.H = Hw;
    a.h0 = h0;
    a.h0_out = h0_out < 0 ? h0 : h0_out;
    a.n_kv = (S + 127) / 128;
    a.n_qt = (S + 127) / 128;
    a.units = B * Hw * a.n_qt;
    a.c = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    a.epi = epi;
    a.timeout_ns = timeout_ns();
    int grid = pl.grid;
    if (split) {
        char* base = static_cast<char*>(ws);
        a.sp.dp_tiles = pl.dp_tiles;
        a.sp.sk_iters = pl.sk_iters;
        a.sp.sk_ctas = pl.sk_ctas;
        a.sp.part_o = reinterpret_cast<float*>(base + pl.off_o);
        a.sp.part_ml = reinterpret_cast<float2*>(base + pl.off_ml);
        a.sp.part_flag = reinterpret_cast<unsigned*>(base + pl.off_flag);
        a.sp.launch_count = reinterpret_cast<unsigned*>(base + pl.off_count);
    } else {
        a.sp.dp_tiles = a.units;
        grid = a.units < dev.sms ? a.units : dev.sms;
    }
    if (causal) a.causal_head_major = causal_head_major(B * Hw, a.n_qt, grid) ? 1 : 0;
    cudaError_t e;
    if (shards) {
        static thread_local xs::ShardMaps maps;   // 6 KB: kept off the stack
        const int Sl = S / P;
        for (int p = 0; p < P; ++p) {
            if ((rc = encode_bshd(&maps.q[p], shards[p], B, Sl, H, D)) != XS_OK) return rc;
            if ((rc = encode_bshd(&maps.k[p], shards[P + p], B, Sl, H, D)) != XS_OK) return rc;
            if ((rc = encode_bshd(&maps.v[p], shards[2 * P + p], B, Sl, H, D)) != XS_OK) return rc;
        }
        a.in_Sl = Sl;
        // shard of key block x (< 2^16): floor(x / bps) = umulhi(2x, m) >> k with
        // k = floor(log2 bps) and m = ceil(2^(31 + k) / bps) < 2^32: the error of
        // m is below x / 2^31 < 2^-15 after the shift, below the 2^k / bps >= 1/2
        // gap to the next multiple
        const unsigned bps = static_cast<unsigned>(Sl / 128);
        int k = 0;
        while ((2u << k) <= bps) ++k;
        a.in_magic = static_cast<unsigned>(((1ull << (31 + k)) + bps - 1) / bps);
        a.in_shift = k;
        e = (D == 128) ? xs::launch_attn_sharded<128>(maps, P, a, grid, split, stream)
                       : xs::launch_attn_sharded<64>(maps, P, a, grid, split, stream);
    } else {
        CUtensorMap tq, tk, tv;
        if ((rc = encode_bshd(&tq, q, B, S, H, D)) != XS_OK) return rc;
        if ((rc = encode_bshd(&tk, k, B, S, H, D)) != XS_OK) return rc;
        if ((rc = encode_bshd(&tv, v, B, S, H, D)) != XS_OK) return rc;
        if (causal)
            e = (D == 128) ? xs::launch_attn_causal<128>(tq, tk, tv, a, grid, stream)
                           : xs::launch_attn_causal<64>(tq, tk, tv, a, grid, stream);
        else
            e = (D == 128) ? xs::launch_attn<128>(tq, tk, tv, a, grid, split, stream)
                           : xs::launch_attn<64>(tq, tk, tv, a, grid, split, stream);
    }
    if (e != cudaSuccess) return cuda_fail(e);
    return XS_OK;
}

// Output layout -> destination parameters and per-buffer byte size.
int layout_epi(int layout, void* const* outs, int B, int S, int H, int D, int P, xs::EpiParams* epi, int* n_out,
               int64_t* out_bytes, bool* need_div) {
    std::memset(epi, 0, sizeof *epi);
    const int np = (P >= 1 && P <= XS_MAX_P) ? P : 0;
    switch (layout) {
        case XS_LAYOUT_A2A:
            *n_out = np;
            *out_bytes = P >= 1 ? static_cast<int64_t>(B) * (S / P) * H * D * 2 : 0;
            *need_div = true;
            epi->Sl = P >= 1 ? S / P : S;
            epi->Hl = H;
            break;
        case XS_LAYOUT_CONTIGUOUS:
            *n_out = 1;
            *out_bytes = static_cast<int64_t>(B) * S * H * D * 2;
            *need_div = false;
            epi->Sl = S;
            epi->Hl = H;
            break;
        case XS_LAYOUT_HEADS:
            *n_out = np;
            *out_bytes = P >= 1 ? static_cast<int64_t>(B) * S * (H / P) * D * 2 : 0;
            *need_div = true;
            epi->Sl = S;
            epi->Hl = P >= 1 ? H / P : H;
            break;
        default:
            return XS_ERR_LAYOUT;
    }
    for (int i = 0; i < *n_out && outs; ++i) epi->ptr[i] = outs[i];
    return XS_OK;
}

// Checks of a workspace given to a balanced call (after the shape checks).
int check_workspace(const void* ws, size_t ws_bytes, const void* q, const void* k, const void* v, void* const* outs,
                    int n_out, int64_t out_bytes, int B, int S, int H, int D) {
    if (!ws) return XS_OK;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return XS_ERR_ALIGNMENT;
    const int64_t in_bytes = static_cast<int64_t>(B) * S * H * D * 2;
    const Range w = range_of(ws, static_cast<int64_t>(ws_bytes));
    if (overlaps(w, range_of(q, in_bytes)) || overlaps(w, range_of(k, in_bytes)) || overlaps(w, range_of(v, in_bytes)))
        return XS_ERR_OVERLAP;
    for (int i = 0; i < n_out; ++i)
        if (overlaps(w, range_of(outs[i], out_bytes))) return XS_ERR_OVERLAP;
    return XS_OK;
}

int attn_layout_call(const void* q, const void* k, const void* v, int layout, void* const* outs, int B, int S, int H,
                     int D, int P, float scale, void* ws, size_t ws_bytes, cudaStream_t stream) {
    if (!outs) return XS_ERR_NULL;
    xs::EpiParams epi;
    int n_out = 0;
    int64_t out_bytes = 0;
    bool need_div = false;
    int rc = layout_epi(layout, outs, B, S, H, D, P, &epi, &n_out, &out_bytes, &need_div);
    if (rc != XS_OK) return rc;
    rc = validate_attn(q, k, v, outs, n_out, B, S, H, D, layout == XS_LAYOUT_CONTIGUOUS ? 1 : P, scale, out_bytes,
                       need_div);
    if (rc != XS_OK) return rc;
    if ((rc = check_workspace(ws, ws_bytes, q, k, v, outs, n_out, out_bytes, B, S, H, D)) != XS_OK) return rc;
    return run_attention(q, k, v, nullptr, 0, epi, B, S, H, D, scale, ws, ws_bytes, stream);
}

// ---- scratch of xs_attn_fwd_balanced_noalloc
// Callers that may not allocate device memory on their call path (a serving
// loop that reserves all memory at start-up and forbids allocation afterwards:
// cudaMalloc can fail there, and cudaFree synchronises the whole device) get the
// balanced schedule's workspace from this file-scope array instead of from a
// buffer of their own.  It is zero-filled when the module is loaded, which is
// all the split-tile flags and the launch count need (a zero flag never matches
// a launch epoch).
// 11 MiB covers the largest workspace the schedule asks for on a 152-SM GB300
// (D = 128: 152 slots x 66,592 B ~ 10.1 MB); a larger need is refused with
// XS_ERR_WORKSPACE.
constexpr size_t NOALLOC_SCRATCH_BYTES = size_t(11) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mutex;
struct ScratchAddr {
    unsigned long long ctx_id = 0;   // unique id of the context the address belongs to (0: none yet)
    void* addr = nullptr;
};
ScratchAddr g_scratch_addr[MAX_DEVICES];

using PFN_ctxGetCurrent = CUresult (*)(CUcontext*);
using PFN_ctxGetId = CUresult (*)(CUcontext, unsigned long long*);
PFN_ctxGetCurrent g_ctx_get_current = nullptr;
PFN_ctxGetId g_ctx_get_id = nullptr;
std::once_flag g_ctx_fn_once;

// Unique id of the calling thread's current context (cuCtxGetId: never reused
// within the process, unlike the context handle), 0 when there is none.
int current_context_id(unsigned long long* id) {
    std::call_once(g_ctx_fn_once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_current = reinterpret_cast<PFN_ctxGetCurrent>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_id = reinterpret_cast<PFN_ctxGetId>(p);
    });
    if (!g_ctx_get_current || !g_ctx_get_id) return cuda_fail(cudaErrorSymbolNotFound);
    CUcontext ctx = nullptr;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS) return cuda_fail(cudaErrorDeviceUninitialized);
    *id = 0;
    if (ctx && g_ctx_get_id(ctx, id) != CUDA_SUCCESS) return cuda_fail(cudaErrorDeviceUninitialized);
    return XS_OK;
}

// Address of g_noalloc_scratch in the current device's context.  It is looked
// up (cudaGetSymbolAddress, which also loads the module into the context if
// needed) the first time a device is used and again whenever the device's
// current context is a different one than at the last lookup (after
// cudaDeviceReset, say, the module is loaded anew and the array may move).
int noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= MAX_DEVICES) return XS_ERR_UNSUPPORTED_DEVICE;
    unsigned long long id = 0;
    int rc = current_context_id(&id);
    if (rc != XS_OK) return rc;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    ScratchAddr& s = g_scratch_addr[dev];
    if (id == 0 || s.ctx_id != id || !s.addr) {
        void* p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_noalloc_scratch)) != cudaSuccess) return cuda_fail(e);
        if ((rc = current_context_id(&id)) != XS_OK) return rc;   // the lookup made the context current
        s.ctx_id = id;
        s.addr = p;
    }
    *out = s.addr;
    return XS_OK;
}

// Streams and events of the host-buffer pipeline (xs_attn_a2a_fwd_staged):
// created once per device on first use and kept for the life of the process.
constexpr int PIPE_BASE_GROUPS = 8;                     // equal head groups of the host-buffer pipeline,
constexpr int PIPE_MAX_GROUPS = PIPE_BASE_GROUPS + 2;   // the first and the last halved
struct PipeStreams {
    bool ready = false;
    std::mutex mutex;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t in_done[PIPE_MAX_GROUPS] = {}, kernel_done[PIPE_MAX_GROUPS] = {};
};
PipeStreams g_pipe[MAX_DEVICES];
std::mutex g_pipe_mutex;

int pipe_streams(PipeStreams** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= MAX_DEVICES) return XS_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_pipe_mutex);
    PipeStreams& p = g_pipe[dev];
    if (!p.ready) {
        const unsigned ef = cudaEventDisableTiming;
        if ((e = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaEventCreateWithFlags(&p.start, ef)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaEventCreateWithFlags(&p.done, ef)) != cudaSuccess) return cuda_fail(e);
        for (int g = 0; g < PIPE_MAX_GROUPS; ++g) {
            if ((e = cudaEventCreateWithFlags(&p.in_done[g], ef)) != cudaSuccess) return cuda_fail(e);
            if ((e = cudaEventCreateWithFlags(&p.kernel_done[g], ef)) != cudaSuccess) return cuda_fail(e);
        }
        p.ready = true;
    }
    *out = &p;
    return XS_OK;
}

}  // namespace

extern "C" {

int xs_attn_a2a_fwd(const void* q, const void* k, const void* v, void* const* out_ptrs, int B, int S, int H, int D,
                    int P, float scale, void* stream) {
    return attn_layout_call(q, k, v, XS_LAYOUT_A2A, out_ptrs, B, S, H, D, P, scale, nullptr, 0,
                            static_cast<cudaStream_t>(stream));
}

int xs_attn_fwd(const void* q, const void* k, const void* v, void* out, int B, int S, int H, int D, float scale,
                void* stream) {
    void* outs[1] = {out};
    return attn_layout_call(q, k, v, XS_LAYOUT_CONTIGUOUS, outs, B, S, H, D, 1, scale, nullptr, 0,
                            static_cast<cudaStream_t>(stream));
}

int xs_attn_heads_fwd(const void* q, const void* k, const void* v, void* const* heads, int B, int S, int H, int D,
                      int P, float scale, void* stream) {
    return attn_layout_call(q, k, v, XS_LAYOUT_HEADS, heads, B, S, H, D, P, scale, nullptr, 0,
                            static_cast<cudaStream_t>(stream));
}

int xs_attn_workspace_bytes(int B, int S, int H, int D, size_t* bytes) {
    if (!bytes) return XS_ERR_NULL;
    int rc = check_shape(B, S, H, D, 1, false);
    if (rc != XS_OK) return rc;
    DeviceInfo dev;
    if ((rc = device_info(&dev)) != XS_OK) return rc;
    *bytes = make_plan(B, S, H, D, dev).ws_bytes;
    return XS_OK;
}

int xs_attn_fwd_balanced_noalloc(const void* q, const void* k, const void* v, int layout, void* const* outs, int B,
                                 int S, int H, int D, int P, float scale, void* stream) {
    // argument checks first, so that an invalid call touches no CUDA state
    if (!outs) return XS_ERR_NULL;
    xs::EpiParams epi;
    int n_out = 0;
    int64_t out_bytes = 0;
    bool need_div = false;
    int rc = layout_epi(layout, outs, B, S, H, D, P, &epi, &n_out, &out_bytes, &need_div);
    if (rc != XS_OK) return rc;
    rc = validate_attn(q, k, v, outs, n_out, B, S, H, D, layout == XS_LAYOUT_CONTIGUOUS ? 1 : P, scale, out_bytes,
                       need_div);
    if (rc != XS_OK) return rc;
    size_t need = 0;
    if ((rc = xs_attn_workspace_bytes(B, S, H, D, &need)) != XS_OK) return rc;
    if (need > NOALLOC_SCRATCH_BYTES) return XS_ERR_WORKSPACE;
    void* scratch = nullptr;
    if ((rc = noalloc_scratch(&scratch)) != XS_OK) return rc;
    return attn_layout_call(q, k, v, layout, outs, B, S, H, D, P, scale, scratch, NOALLOC_SCRATCH_BYTES,
                            static_cast<cudaStream_t>(stream));
}

int xs_attn_causal_fwd(const void* q, const void* k, const void* v, int layout, void* const* outs, int B, int S,
                       int H, int D, int P, float scale, void* stream) {
    if (!outs) return XS_ERR_NULL;
    xs::EpiParams epi;
    int n_out = 0;
    int64_t out_bytes = 0;
    bool need_div = false;
    int rc = layout_epi(layout, outs, B, S, H, D, P, &epi, &n_out, &out_bytes, &need_div);
    if (rc != XS_OK) return rc;
    rc = validate_attn(q, k, v, outs, n_out, B, S, H, D, layout == XS_LAYOUT_CONTIGUOUS ? 1 : P, scale, out_bytes,
                       need_div);
    if (rc != XS_OK) return rc;
    return run_attention(q, k, v, nullptr, 0, epi, B, S, H, D, scale, nullptr, 0, static_cast<cudaStream_t>(stream),
                         true);
}

int xs_attn_varlen_fwd(const void* q, const void* k, const void* v, const int* seqlens, int n_seqs, int causal,
                       int layout, void* const* outs, int T, int H, int D, int P, float scale, void* stream) {
    if (!outs || !seqlens) return XS_ERR_NULL;
    if (n_seqs < 1 || n_seqs > xs::MAX_VARLEN_SEQS) return XS_ERR_SHAPE;
    int64_t total = 0, tiles = 0;
    for (int i = 0; i < n_seqs; ++i) {
        if (seqlens[i] < 0 || seqlens[i] > 65536 * 128) return XS_ERR_SHAPE;
        total += seqlens[i];
        tiles += (seqlens[i] + 127) / 128;
    }
    if (total != T || tiles > xs::MAX_VARLEN_TILES) return XS_ERR_SHAPE;
    if (tiles * static_cast<int64_t>(H) > INT32_MAX) return XS_ERR_SHAPE;   // units must fit an int
    xs::EpiParams epi;
    int n_out = 0;
    int64_t out_bytes = 0;
    bool need_div = false;
    int rc = layout_epi(layout, outs, 1, T, H, D, P, &epi, &n_out, &out_bytes, &need_div);
    if (rc != XS_OK) return rc;
    rc = validate_attn(q, k, v, outs, n_out, 1, T, H, D, layout == XS_LAYOUT_CONTIGUOUS ? 1 : P, scale, out_bytes,
                       need_div);
    if (rc != XS_OK) return rc;
    if (causal) {
        // The packed kernel's causal form is not launched (at 75,776 packed tokens
        // it ended in an unspecified launch failure whose cause is not
        // established).  The causal packed call runs as one causal launch per
        // sequence instead: the sequence's rows of Q, K and V as [1, len, H, D]
        // tensors, its output row s stored at packed row start + s of the layout.
        // A sequence whose launch fills every SM runs on `stream`, one after the
        // other (concurrent long launches interleave their CTAs and share less
        // K/V in L2: measured 4 % slower); the shorter ones run on the library's
        // two side streams (forked from and joined back to `stream`), so that
        // they fill the SMs the long launches leave idle at their ends.
        const size_t row_bytes = static_cast<size_t>(H) * D * 2;
        const cudaStream_t st = static_cast<cudaStream_t>(stream);
        int starts[xs::MAX_VARLEN_SEQS], order[xs::MAX_VARLEN_SEQS], n_live = 0;
        for (int i = 0, start = 0; i < n_seqs; start += seqlens[i], ++i) {
            starts[i] = start;
            if (seqlens[i] > 0) order[n_live++] = i;
        }
        std::stable_sort(order, order + n_live, [&](int x, int y) { return seqlens[x] > seqlens[y]; });
        auto launch = [&](int i, cudaStream_t s) {
            xs::EpiParams es = epi;
            es.row0 = starts[i];
            const size_t off = static_cast<size_t>(starts[i]) * row_bytes;
            return run_attention(static_cast<const char*>(q) + off, static_cast<const char*>(k) + off,
                                 static_cast<const char*>(v) + off, nullptr, 0, es, 1, seqlens[i], H, D, scale,
                                 nullptr, 0, s, true);
        };
        if (n_live == 1) return launch(order[0], st);
        DeviceInfo dev;
        if ((rc = device_info(&dev)) != XS_OK) return rc;
        auto fills_gpu = [&](int i) { return static_cast<int64_t>((seqlens[i] + 127) / 128) * H >= dev.sms; };
        if (std::all_of(order, order + n_live, fills_gpu)) {   // nothing for the side streams
            for (int n = 0; n < n_live && rc == XS_OK; ++n) rc = launch(order[n], st);
            return rc;
        }
        PipeStreams* ps = nullptr;
        if ((rc = pipe_streams(&ps)) != XS_OK) return rc;
        std::lock_guard<std::mutex> lock(ps->mutex);
        const cudaStream_t lanes[2] = {ps->in, ps->out};
        cudaError_t e = cudaEventRecord(ps->start, st);
        for (int j = 0; j < 2 && e == cudaSuccess; ++j) e = cudaStreamWaitEvent(lanes[j], ps->start, 0);
        if (e != cudaSuccess) return cuda_fail(e);
        double work[2] = {0.0, 0.0};
        for (int n = 0; n < n_live; ++n) {
            const int i = order[n];
            if (fills_gpu(i)) {
                rc = launch(i, st);
            } else {
                const int j = work[1] < work[0] ? 1 : 0;
                work[j] += static_cast<double>(seqlens[i]) * (seqlens[i] + 1);
                rc = launch(i, lanes[j]);
            }
            if (rc != XS_OK) break;
        }
        // join even after a failed launch, so that `stream` stays ordered after what was queued
        for (int j = 0; j < 2; ++j) {
            if ((e = cudaEventRecord(ps->kernel_done[j], lanes[j])) != cudaSuccess) return cuda_fail(e);
            if ((e = cudaStreamWaitEvent(st, ps->kernel_done[j], 0)) != cudaSuccess) return cuda_fail(e);
        }
        return rc;
    }
    DeviceInfo dev;
    if ((rc = device_info(&dev)) != XS_OK) return rc;

    // The tile list, longest first: tile (i, t) reads ceil(len_i / 128) key blocks;
    // ties keep sequence order, then query-tile order (the sort is stable), so a
    // sequence's tiles stay together, tile 0 first, which the kernel's head-major
    // order within a sequence relies on.
    static thread_local xs::VarlenTable vt;   // 20 KB: kept off the stack
    vt.n_seqs = n_seqs;
    vt.cu[0] = 0;
    for (int i = 0; i < n_seqs; ++i) vt.cu[i + 1] = vt.cu[i] + seqlens[i];
    int n = 0;
    for (int i = 0; i < n_seqs; ++i)
        for (int t = 0; t * 128 < seqlens[i]; ++t) vt.tile[n++] = (static_cast<unsigned>(i) << 16) | static_cast<unsigned>(t);
    vt.n_tiles = n;
    auto blocks = [&](unsigned e) { return (seqlens[e >> 16] + 127) / 128; };
    std::stable_sort(vt.tile, vt.tile + n, [&](unsigned x, unsigned y) { return blocks(x) > blocks(y); });

    xs::AttnArgs a;
    std::memset(&a, 0, sizeof a);
    a.B = 1;
    a.S = T;
    a.H = H;
    a.n_kv = (T + 127) / 128;
    a.n_qt = (T + 127) / 128;
    a.units = n * H;
    a.c = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    a.epi = epi;
    a.timeout_ns = timeout_ns();
    a.sp.dp_tiles = a.units;
    const int grid = a.units < dev.sms ? a.units : dev.sms;
    CUtensorMap tq, tk, tv;
    if ((rc = encode_bshd(&tq, q, 1, T, H, D)) != XS_OK) return rc;
    if ((rc = encode_bshd(&tk, k, 1, T, H, D)) != XS_OK) return rc;
    if ((rc = encode_bshd(&tv, v, 1, T, H, D)) != XS_OK) return rc;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const cudaError_t e = (D == 128) ? xs::launch_attn_varlen<128>(tq, tk, tv, a, vt, grid, st)
                                     : xs::launch_attn_varlen<64>(tq, tk, tv, a, vt, grid, st);
    if (e != cudaSuccess) return cuda_fail(e);
    return XS_OK;
}

int xs_attn_ulysses_fwd(const void* const* q_shards, const void* const* k_shards, const void* const* v_shards,
                        void* const* out_shards, int B, int S, int H, int D, int P, float scale, void* workspace,
                        size_t workspace_bytes, void* stream) {
    if (!q_shards || !k_shards || !v_shards || !out_shards) return XS_ERR_NULL;
    int rc = check_shape(B, S, H, D, P, true);
    if (rc != XS_OK) return rc;
    const int Sl = S / P;
    if (Sl % 128 != 0) return XS_ERR_DIVISIBILITY;
    if ((S + 127) / 128 > 65536) return XS_ERR_SHAPE;   // the kernel's shard lookup covers 2^16 key blocks
    const void* in[3 * XS_MAX_P];
    for (int p = 0; p < P; ++p) {
        in[p] = q_shards[p];
        in[P + p] = k_shards[p];
        in[2 * P + p] = v_shards[p];
    }
    for (int i = 0; i < 3 * P; ++i)
        if (!in[i]) return XS_ERR_NULL;
    for (int p = 0; p < P; ++p)
        if (!out_shards[p]) return XS_ERR_NULL;
    if ((rc = check_scale(scale)) != XS_OK) return rc;
    for (int i = 0; i < 3 * P; ++i)
        if (!aligned16(in[i])) return XS_ERR_ALIGNMENT;
    for (int p = 0; p < P; ++p)
        if (!aligned16(out_shards[p])) return XS_ERR_ALIGNMENT;
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return XS_ERR_ALIGNMENT;
    const int64_t shard_bytes = static_cast<int64_t>(B) * Sl * H * D * 2;
    Range ins[3 * XS_MAX_P + 1], outs[XS_MAX_P + 1];
    for (int i = 0; i < 3 * P; ++i) ins[i] = range_of(in[i], shard_bytes);
    for (int p = 0; p < P; ++p) outs[p] = range_of(out_shards[p], shard_bytes);
    int n_out = P;
    if (workspace) outs[n_out++] = range_of(workspace, static_cast<int64_t>(workspace_bytes));
    if ((rc = check_disjoint(outs, n_out, ins, 3 * P)) != XS_OK) return rc;
    xs::EpiParams epi;
    std::memset(&epi, 0, sizeof epi);
    for (int p = 0; p < P; ++p) epi.ptr[p] = out_shards[p];
    epi.Sl = Sl;
    epi.Hl = H;
    return run_attention(nullptr, nullptr, nullptr, in, P, epi, B, S, H, D, scale, workspace, workspace_bytes,
                         static_cast<cudaStream_t>(stream));
}

int xs_attn_ulysses_rank_fwd(const void* q_heads, const void* k_heads, const void* v_heads, void* const* out_shards,
                             int B, int S, int H, int D, int P, int rank, float scale, void* workspace,
                             size_t workspace_bytes, void* stream) {
    if (!q_heads || !k_heads || !v_heads || !out_shards) return XS_ERR_NULL;
    int rc = check_shape(B, S, H, D, P, true);
    if (rc != XS_OK) return rc;
    if (rank < 0 || rank >= P) return XS_ERR_SHAPE;
    for (int p = 0; p < P; ++p)
        if (!out_shards[p]) return XS_ERR_NULL;
    if ((rc = check_scale(scale)) != XS_OK) return rc;
    if (!aligned16(q_heads) || !aligned16(k_heads) || !aligned16(v_heads)) return XS_ERR_ALIGNMENT;
    for (int p = 0; p < P; ++p)
        if (!aligned16(out_shards[p])) return XS_ERR_ALIGNMENT;
    const int Hl = H / P;
    const int64_t in_bytes = static_cast<int64_t>(B) * S * Hl * D * 2;
    const int64_t shard_bytes = static_cast<int64_t>(B) * (S / P) * H * D * 2;
    Range ins[3] = {range_of(q_heads, in_bytes), range_of(k_heads, in_bytes), range_of(v_heads, in_bytes)};
    Range outs[XS_MAX_P];
    for (int p = 0; p < P; ++p) outs[p] = range_of(out_shards[p], shard_bytes);
    if ((rc = check_disjoint(outs, P, ins, 3)) != XS_OK) return rc;
    if ((rc = check_workspace(workspace, workspace_bytes, q_heads, k_heads, v_heads, out_shards, P, shard_bytes, B, S,
                              Hl, D)) != XS_OK)
        return rc;
    xs::EpiParams epi;
    std::memset(&epi, 0, sizeof epi);
    for (int p = 0; p < P; ++p) epi.ptr[p] = out_shards[p];
    epi.Sl = S / P;
    epi.Hl = H;
    return run_attention(q_heads, k_heads, v_heads, nullptr, 0, epi, B, S, Hl, D, scale, workspace, workspace_bytes,
                         static_cast<cudaStream_t>(stream), false, 0, 0, false, rank * Hl);
}

int xs_relayout_a2a_inverse(const void* const* seq_shards, void* const* heads, int B, int S, int H, int D, int P,
                            void* stream) {
    if (!seq_shards || !heads) return XS_ERR_NULL;
    int rc = check_shape(B, S, H, D, P, true);
    if (rc != XS_OK) return rc;
    for (int p = 0; p < P; ++p)
        if (!seq_shards[p] || !heads[p]) return XS_ERR_NULL;
    for (int p = 0; p < P; ++p)
        if (!aligned16(seq_shards[p]) || !aligned16(heads[p])) return XS_ERR_ALIGNMENT;
    const int64_t head_bytes = static_cast<int64_t>(B) * S * (H / P) * D * 2;
    const int64_t shard_bytes = static_cast<int64_t>(B) * (S / P) * H * D * 2;
    Range ins[XS_MAX_P], outs[XS_MAX_P];
    for (int p = 0; p < P; ++p) {
        ins[p] = range_of(seq_shards[p], shard_bytes);
        outs[p] = range_of(heads[p], head_bytes);
    }
    if ((rc = check_disjoint(outs, P, ins, P)) != XS_OK) return rc;
    DeviceInfo dev;
    if ((rc = device_info(&dev)) != XS_OK) return rc;
    xs::RelayoutArgs a;
    std::memset(&a, 0, sizeof a);
    for (int p = 0; p < P; ++p) {
        a.heads[p] = seq_shards[p];   // inverse direction: read sequence shards,
        a.out[p] = heads[p];          // write head shards
    }
    a.B = B;
    a.S = S;
    a.H = H;
    a.D = D;
    a.P = P;
    cudaError_t e = xs::launch_relayout_inverse(a, dev.sms, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return XS_OK;
}

int xs_attn_fwd_balanced(const void* q, const void* k, const void* v, int layout, void* const* outs, int B, int S,
                         int H, int D, int P, float scale, void* workspace, size_t workspace_bytes, void* stream) {
    return attn_layout_call(q, k, v, layout, outs, B, S, H, D, P, scale, workspace, workspace_bytes,
                            static_cast<cudaStream_t>(stream));
}

int xs_relayout_a2a(const void* const* heads, void* const* out_ptrs, int B, int S, int H, int D, int P,
                    void* stream) {
    if (!heads || !out_ptrs) return XS_ERR_NULL;
    int rc = check_shape(B, S, H, D, P, true);
    if (rc != XS_OK) return rc;
    for (int p = 0; p < P; ++p)
        if (!heads[p] || !out_ptrs[p]) return XS_ERR_NULL;
    for (int p = 0; p < P; ++p)
        if (!aligned16(heads[p]) || !aligned16(out_ptrs[p])) return XS_ERR_ALIGNMENT;
    const int64_t head_bytes = static_cast<int64_t>(B) * S * (H / P) * D * 2;
    const int64_t shard_bytes = static_cast<int64_t>(B) * (S / P) * H * D * 2;
    Range ins[XS_MAX_P], outs[XS_MAX_P];
    for (int p = 0; p < P; ++p) {
        ins[p] = range_of(heads[p], head_bytes);
        outs[p] = range_of(out_ptrs[p], shard_bytes);
    }
    if ((rc = check_disjoint(outs, P, ins, P)) != XS_OK) return rc;
    DeviceInfo dev;
    if ((rc = device_info(&dev)) != XS_OK) return rc;
    xs::RelayoutArgs a;
    std::memset(&a, 0, sizeof a);
    for (int p = 0; p < P; ++p) {
        a.heads[p] = heads[p];
        a.out[p] = out_ptrs[p];
    }
    a.B = B;
    a.S = S;
    a.H = H;
    a.D = D;
    a.P = P;
    cudaError_t e = xs::launch_relayout(a, dev.sms, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return XS_OK;
}

int xs_attn_a2a_fwd_staged(const void* q_host, const void* k_host, const void* v_host, void* const* out_host,
                           void* q_dev, void* k_dev, void* v_dev, void* const* out_dev, int B, int S, int H, int D,
                           int P, float scale, void* workspace, size_t workspace_bytes, void* stream) {
    if (!q_host || !k_host || !v_host || !out_host || !out_dev) return XS_ERR_NULL;
    if (P >= 1 && P <= XS_MAX_P)
        for (int p = 0; p < P; ++p)
            if (!out_host[p]) return XS_ERR_NULL;
    const int n_out = (P >= 1 && P <= XS_MAX_P) ? P : 0;
    const int64_t shard_bytes = (P >= 1) ? static_cast<int64_t>(B) * (S / P) * H * D * 2 : 0;
    int rc = validate_attn(q_dev, k_dev, v_dev, out_dev, n_out, B, S, H, D, P, scale, shard_bytes, true);
    if (rc != XS_OK) return rc;
    if ((rc = check_workspace(workspace, workspace_bytes, q_dev, k_dev, v_dev, out_dev, n_out, shard_bytes, B, S, H,
                              D)) != XS_OK)
        return rc;
    PipeStreams* ps = nullptr;
    if ((rc = pipe_streams(&ps)) != XS_OK) return rc;
    std::lock_guard<std::mutex> lock(ps->mutex);   // one call's enqueues at a time on the shared streams
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    xs::EpiParams epi;
    std::memset(&epi, 0, sizeof epi);
    for (int p = 0; p < P; ++p) epi.ptr[p] = out_dev[p];
    epi.Sl = S / P;
    epi.Hl = H;
    // Head groups: the copies of group g + 1 in and of group g - 1 out overlap the
    // kernel of group g.  Every copy is one pitched cudaMemcpy2DAsync: the group's
    // heads are hg * D contiguous elements of every [.., H, D] row.
    // Group bounds: PIPE_BASE_GROUPS equal groups, the first and the last cut in
    // two, since their copies (the first group's in, the last group's out) are the
    // ones no kernel hides.
    int bounds[PIPE_MAX_GROUPS + 1];
    int ng = 0;
    {
        const int nb = H < PIPE_BASE_GROUPS ? H : PIPE_BASE_GROUPS;
        bounds[0] = 0;
        for (int i = 0; i < nb; ++i) {
            const int lo = H * i / nb, hi = H * (i + 1) / nb;
            if (nb >= 2 && (i == 0 || i == nb - 1) && hi - lo >= 2) bounds[++ng] = lo + (hi - lo) / 2;
            bounds[++ng] = hi;
        }
    }
    const size_t row = static_cast<size_t>(H) * D * 2;       // bytes per (b, s) row
    const size_t rows_in = static_cast<size_t>(B) * S, rows_out = static_cast<size_t>(B) * (S / P);
    cudaError_t e;
    if ((e = cudaEventRecord(ps->start, st)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaStreamWaitEvent(ps->in, ps->start, 0)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaStreamWaitEvent(ps->out, ps->start, 0)) != cudaSuccess) return cuda_fail(e);
    const void* hin[3] = {q_host, k_host, v_host};
    void* din[3] = {q_dev, k_dev, v_dev};
    for (int g = 0; g < ng; ++g) {
        const int h_lo = bounds[g], h_hi = bounds[g + 1];
        const size_t off = static_cast<size_t>(h_lo) * D * 2, width = static_cast<size_t>(h_hi - h_lo) * D * 2;
        for (int t = 0; t < 3; ++t)
            if ((e = cudaMemcpy2DAsync(static_cast<char*>(din[t]) + off, row, static_cast<const char*>(hin[t]) + off,
                                       row, width, rows_in, cudaMemcpyHostToDevice, ps->in)) != cudaSuccess)
                return cuda_fail(e);
        if ((e = cudaEventRecord(ps->in_done[g], ps->in)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaStreamWaitEvent(st, ps->in_done[g], 0)) != cudaSuccess) return cuda_fail(e);
        if ((rc = run_attention(q_dev, k_dev, v_dev, nullptr, 0, epi, B, S, H, D, scale, workspace, workspace_bytes,
                                st, false, h_lo, h_hi - h_lo, true)) != XS_OK)
            return rc;
        if ((e = cudaEventRecord(ps->kernel_done[g], st)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaStreamWaitEvent(ps->out, ps->kernel_done[g], 0)) != cudaSuccess) return cuda_fail(e);
        for (int p = 0; p < P; ++p)
            if ((e = cudaMemcpy2DAsync(static_cast<char*>(out_host[p]) + off, row,
                                       static_cast<const char*>(out_dev[p]) + off, row, width, rows_out,
                                       cudaMemcpyDeviceToHost, ps->out)) != cudaSuccess)
                return cuda_fail(e);
    }
    if ((e = cudaEventRecord(ps->done, ps->out)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaStreamWaitEvent(st, ps->done, 0)) != cudaSuccess) return cuda_fail(e);
    return XS_OK;
}

int xs_burst_gap(void* dst, size_t dst_bytes, int producers, size_t burst_bytes, int bursts, long long lead_ns,
                 long long gap_ns, long long* issue_ns, void* stream) {
    if (!dst || !issue_ns) return XS_ERR_NULL;
    if (producers < 1 || bursts < 1 || bursts > 65536 || gap_ns < 0 || gap_ns > 100000000LL) return XS_ERR_SHAPE;
    if (lead_ns < 0 || lead_ns > 100000000LL) return XS_ERR_SHAPE;
    if (static_cast<double>(bursts) * static_cast<double>(gap_ns) > 1e10) return XS_ERR_SHAPE;  // <= 10 s of gaps
    const size_t per = burst_bytes / static_cast<size_t>(producers);
    if (burst_bytes == 0 || burst_bytes % (16u * static_cast<size_t>(producers)) != 0) return XS_ERR_SHAPE;
    const size_t windows = dst_bytes / per;
    if (windows < static_cast<size_t>(producers)) return XS_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(dst) & 15u) != 0 || (reinterpret_cast<uintptr_t>(issue_ns) & 7u) != 0)
        return XS_ERR_ALIGNMENT;
    const int64_t times_bytes = static_cast<int64_t>(bursts) * producers * 8;
    if (overlaps(range_of(dst, static_cast<int64_t>(dst_bytes)), range_of(issue_ns, times_bytes)))
        return XS_ERR_OVERLAP;
    DeviceInfo dev;
    int rc = device_info(&dev);
    if (rc != XS_OK) return rc;
    if (producers > dev.sms) return XS_ERR_SHAPE;
    xs::BurstGapArgs a;
    a.dst = dst;
    a.chunks_per_producer = static_cast<int64_t>(per / 16);
    a.windows = static_cast<int64_t>(windows);
    a.bursts = bursts;
    a.lead_ns = lead_ns;
    a.gap_ns = gap_ns;
    a.issue_ns = issue_ns;
    cudaError_t e = xs::launch_burst_gap(a, producers, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return XS_OK;
}

int xs_attn_get_device_error_info(void* stream, int* info, int n_info) {
    if (n_info < 0 || n_info > 8 || (n_info > 0 && !info)) return XS_ERR_NULL;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    int v = 0, drain = 0;
    xs::DeviceErrorInfo r{};
    if ((e = xs::read_and_clear_device_error(&v, &r, &drain)) != cudaSuccess) return cuda_fail(e);
    const int fields[8] = {v ? r.code : 0, r.cta, r.warp, r.lane, r.site, r.detail[0], r.detail[1], r.detail[2]};
    for (int i = 0; i < n_info; ++i) info[i] = v ? fields[i] : 0;
    if (drain) return XS_ERR_DEVICE_DRAIN;
    if (v == 0) return XS_OK;
    return v == xs::XS_DEVICE_BOUNDS_CODE ? XS_ERR_DEVICE_BOUNDS : XS_ERR_DEVICE_TIMEOUT;
}

int xs_attn_get_device_error(void* stream) { return xs_attn_get_device_error_info(stream, nullptr, 0); }

const char* xs_attn_error_string(int code) {
    switch (code) {
        case XS_OK: return "success";
        case XS_ERR_NULL: return "a required pointer is NULL";
        case XS_ERR_SHAPE: return "B, S, H and P must be >= 1 and the tensor sizes must fit the kernel's index types";
        case XS_ERR_HEAD_DIM: return "head dimension D must be 64 or 128";
        case XS_ERR_DIVISIBILITY: return "S and H must be divisible by the number of virtual ranks P";
        case XS_ERR_TOO_MANY_RANKS: return "P exceeds XS_MAX_P (16)";
        case XS_ERR_ALIGNMENT: return "device pointers must be 16-byte aligned";
        case XS_ERR_OVERLAP: return "an output buffer overlaps another output or an input";
        case XS_ERR_SCALE: return "scale must be finite and non-negative";
        case XS_ERR_CUDA: return "a CUDA call or kernel launch failed (see xs_attn_last_cuda_error)";
        case XS_ERR_DEVICE_TIMEOUT: return "a bounded wait inside a kernel expired; the launch was abandoned";
        case XS_ERR_UNSUPPORTED_DEVICE: return "the current device is not an sm_103 (GB300) GPU";
        case XS_ERR_WORKSPACE: return "the workspace is smaller than xs_attn_workspace_bytes reports";
        case XS_ERR_LAYOUT: return "unknown output layout";
        case XS_ERR_DEVICE_DRAIN:
            return "after an expired wait, a kernel gave up waiting for its own copies or MMAs in flight";
        case XS_ERR_DEVICE_BOUNDS: return "an index check inside a kernel failed; the access was skipped";
        case XS_ERR_UNAVAILABLE: return "this variant is disabled in this build";
        default: return "unknown xsattn error code";
    }
}

int xs_attn_last_cuda_error(void) { return g_last_cuda_error; }

#ifdef XS_TILE_SPANS
// Exported by the instrumented build only (libxsattn_spans.so), not declared in
// the public header: point the kernels' per-tile timestamps at `buf` (device,
// ctas * (per_cta * 6 + 32 * 10) unsigned 64-bit words: the per-piece words of
// CTAs 0 .. ctas-1, then their block phases), or stop with NULL.
int xs_attn_set_tile_spans(void* buf, int ctas, int per_cta) {
    if (ctas < 0 || per_cta < 0 || (buf && (ctas == 0 || per_cta == 0))) return XS_ERR_SHAPE;
    const cudaError_t e = xs::set_tile_spans(static_cast<unsigned long long*>(buf), ctas, per_cta);
    return e == cudaSuccess ? XS_OK : cuda_fail(e);
}
#endif

int xs_attn_version(void) { return 100; }

}  // extern "C"
