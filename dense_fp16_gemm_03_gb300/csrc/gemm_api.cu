// C ABI of the fp16 NT GEMM (declared in include/gemm_f16.h): argument
// validation, planning (variant, raster width, grid, stream-K tail or
// rotated K walk), the host-buffer pipeline and the allocation-free form;
// the variant table, the launch and the TMA tensor maps are in
// gemm_launch.cuh.
//
// The interface mirrors the call of "1. WGMMA: Hopper's Asynchronous Tensor
// Core" (section "The Full Kernel": m, n, k and the a, b, c fp16 pointers)
// plus a stream, a plan query and a workspace query.  The capability gate
// answers the one on the "wgmma_gemm.cu" page (refuse a device the code was
// not built for with a clear status instead of failing inside the driver).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <chrono>
#include <mutex>
#include <random>
#include <string.h>

#include "gemm_f16.h"
#include "gemm_launch.cuh"

using namespace gemm_f16;

// The device error word: set by a kernel whose pipeline wait timed out,
// read and cleared by gemm_f16_take_device_error.
__device__ uint32_t g_gemm_f16_error_word = 0u;

#ifdef GEMM_F16_PHASE_TRACE
// Phase-trace buffer of the following launches (trace build only).
static std::atomic<unsigned long long *> g_trace_buffer{nullptr};
#endif

namespace {

constexpr int kMaxDevices = 64;

// ---------------------------------------------------- per-device state

// Identity of the calling thread's current CUDA context (cuCtxGetCurrent +
// cuCtxGetId through the runtime's driver entry points).  Per-device state
// below is kept per context: after cudaDeviceReset the primary context, the
// module and every address looked up in it are new, so state made for an
// earlier context is made again instead of reused.
typedef CUresult (*PfnCtxGetCurrent)(CUcontext *);
typedef CUresult (*PfnCtxGetId)(CUcontext, unsigned long long *);
PfnCtxGetCurrent g_ctx_get_current = nullptr;
PfnCtxGetId g_ctx_get_id = nullptr;

gemm_status_t current_context_id(unsigned long long *id)
{
    static std::once_flag once;
    std::call_once(once, []() {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_current = reinterpret_cast<PfnCtxGetCurrent>(f);
        else
            cudaGetLastError();
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_id = reinterpret_cast<PfnCtxGetId>(f);
        else
            cudaGetLastError();
    });
    if (!g_ctx_get_current || !g_ctx_get_id) return GEMM_ERR_CUDA;
    CUcontext ctx = nullptr;
    // no context yet on this thread: let the runtime make the device's primary context current
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) {
        if (cudaFree(nullptr) != cudaSuccess || g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
    }
    return g_ctx_get_id(ctx, id) == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_CUDA;
}

struct DeviceInfo {
    bool ready = false;
    unsigned long long ctx_id = 0;  // the context the entries below were made in
    bool arch_ok = false;
    int num_sms = 0;
    int max_clusters[kNumVariants] = {};
    uint32_t *error_word = nullptr;  // device address of g_gemm_f16_error_word in that context
};

std::mutex g_mutex;
DeviceInfo g_devices[kMaxDevices];

gemm_status_t device_info(DeviceInfo **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    unsigned long long ctx = 0;
    gemm_status_t st = current_context_id(&ctx);
    if (st != GEMM_OK) return st;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo &d = g_devices[dev];
    if (!d.ready || d.ctx_id != ctx) {
        DeviceInfo made;
        made.ctx_id = ctx;
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        made.arch_ok = (major == 10 && minor == 3);
        made.num_sms = sms;
        if (made.arch_ok) {
            for (int v = 0; v < kNumVariants; ++v) {
                const Variant &var = kVariants[v];
                if (cudaFuncSetAttribute(var.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, var.smem) !=
                    cudaSuccess) {
                    cudaGetLastError();
                    return GEMM_ERR_CUDA;
                }
                const int cs = cluster_of(var);
                made.max_clusters[v] = sms / cs;
                if (cs > 1) {
                    cudaLaunchConfig_t cfg;
                    memset(&cfg, 0, sizeof(cfg));
                    cfg.gridDim = dim3(unsigned(cs * (sms / cs)), 1, 1);
                    cfg.blockDim = dim3(unsigned(var.threads), 1, 1);
                    cfg.dynamicSmemBytes = size_t(var.smem);
                    cudaLaunchAttribute attr;
                    attr.id = cudaLaunchAttributeClusterDimension;
                    attr.val.clusterDim.x = unsigned(cs);
                    attr.val.clusterDim.y = 1;
                    attr.val.clusterDim.z = 1;
                    cfg.attrs = &attr;
                    cfg.numAttrs = 1;
                    int clusters = 0;
                    if (cudaOccupancyMaxActiveClusters(&clusters, var.fn, &cfg) == cudaSuccess && clusters > 0)
                        made.max_clusters[v] = clusters;
                    else
                        cudaGetLastError();
                }
            }
            void *err_ptr = nullptr;
            if (cudaGetSymbolAddress(&err_ptr, g_gemm_f16_error_word) != cudaSuccess || err_ptr == nullptr) {
                cudaGetLastError();
                return GEMM_ERR_CUDA;
            }
            made.error_word = static_cast<uint32_t *>(err_ptr);
        }
        made.ready = true;
        d = made;
    }
    *out = &d;
    return d.arch_ok ? GEMM_OK : GEMM_ERR_ARCH;
}

// ---------------------------------------------------------- validation

int current_device()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    return dev;
}

bool aligned16(const void *p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

gemm_status_t check_shape(int64_t m, int64_t n, int64_t k)
{
    if (m < 0 || n < 0 || k < 0) return GEMM_ERR_INVALID_ARG;
    const int64_t lim = int64_t(1) << 31;
    if (m >= lim || n >= lim || k >= lim) return GEMM_ERR_UNSUPPORTED_SHAPE;
    if (k % 8 != 0 || n % 8 != 0) return GEMM_ERR_UNSUPPORTED_SHAPE;
    return GEMM_OK;
}

gemm_status_t check_pointers(int64_t m, int64_t n, int64_t k, const void *a, const void *b, const void *c)
{
    if (m > 0 && n > 0) {
        if (!c) return GEMM_ERR_INVALID_ARG;
        if (!aligned16(c)) return GEMM_ERR_ALIGNMENT;
        if (k > 0) {
            if (!a || !b) return GEMM_ERR_INVALID_ARG;
            if (!aligned16(a) || !aligned16(b)) return GEMM_ERR_ALIGNMENT;
        }
    }
    return GEMM_OK;
}

int64_t cdiv(int64_t a, int64_t b)
{
    return (a + b - 1) / b;
}

// --------------------------------------------------------------- plans

// Raster width: tile columns per raster group, so that a group spans 2048
// columns of C.  Measured on GB300 (interleaved runs under the power cap):
// 256-column pair tiles at 8192^3 did best with widths 8-16 (fewest DRAM
// re-reads, highest clock), 512-column tiles with width 4 (8192^3: +1% over
// width 8; 4096^3 and 6144^3 level or slightly ahead); narrower groups re-read
// A from DRAM more often.
int32_t auto_raster_width(int64_t tiles_n, int32_t block_n)
{
    int64_t w = 2048 / (block_n > 0 ? block_n : 256);
    if (w > tiles_n) w = tiles_n;
    return int32_t(w < 1 ? 1 : w);
}

// Fraction of the resident slots the data-parallel waves keep busy.
double wave_efficiency(int64_t tiles, int64_t slots)
{
    if (tiles <= 0 || slots <= 0) return 1.0;
    const int64_t waves = (tiles + slots - 1) / slots;
    return double(tiles) / double(waves * slots);
}

// A stream-K tail pays when the data-parallel schedule would leave the last
// wave badly short of the resident clusters: measured, it wins when less
// than about 86% of the slots are busy over the waves (ragged 3000x5000),
// and loses above that, because under the power cap keeping the idle SMs of
// a nearly full last wave busy costs clock for the whole launch.
// Rotating the K walk of whole tiles pays when no operand strip is shared by
// two tiles (a single row or column of tiles, e.g. 128 x 16384 x 16384:
// measured +10%); when strips are shared, tiles that read them in K
// lockstep hit L2 instead of DRAM, and rotation loses (8192^3: -6%).
bool rotate_pays(int64_t tiles_m, int64_t tiles_n, int64_t k_blocks)
{
    return (tiles_m == 1 || tiles_n == 1) && k_blocks >= 8;
}

// Neither pays with 32 K blocks per tile or fewer: each cluster's K range is then short and the
// partial fix-up (and, for split K, the reduction launch) costs more than the work it spreads.
// Device time on GB300 against the best data-parallel plan: 1024 x 1024 x 448 (7 K blocks) 9.05
// against 4.62 us; 1024^3 (16) 12.16 (tail) and 9.82 (split) against 6.89; 2048^3 (32) 22.19 and
// 27.16 against 13.30.  Every tail and split measured to pay had 47 K blocks or more.  With more,
// even very few tiles are split (the parts keep at least 4 K blocks each): two 128 x 128 tiles with
// K = 8192 would otherwise run on two SMs.
bool streamk_pays(int64_t num_tiles, int64_t k_blocks, int64_t slots)
{
    if (k_blocks <= 32) return false;
    return wave_efficiency(num_tiles, slots) < 0.86;
}

// The wide tiles (256 x 512, 256 x 448, 256 x 320) can take a stream-K tail
// over the partial last wave only (every whole wave data-parallel), but the
// automatic plans never give them one: measured on GB300 (burst, 400-launch
// blocks) it lost everywhere -- 8192^3 575 against 565 us, 4096^3 85.3
// against 79.7 us, 3000 x 5000 x 4096 78.4 against 68.6 us for the 448-column
// tile -- even with the owner's partials bulk-copied into the idle ring.
// With one accumulator filling tensor memory, about half the tail tiles are
// cut three ways; the owner then waits for a middle contributor that ends
// its whole range and publishes 256 KB per CTA through its ~95 GB/s port,
// and adds one or two such partials, which costs more than the third of a
// tile the tail saves.  A request for it (stream_k = 1) is honoured.
bool wide_tail_pays(int64_t, int64_t, int64_t)
{
    return false;
}

// Clusters that share a stream-K tail of `tiles` tiles when no whole wave is
// left to run data-parallel.  A tile split over w clusters is finished by its
// owner adding the other w - 1 partials one after another (~2,800 cycles each
// for a CTA's 128 KB at 256 columns), while the split shortens every
// cluster's K range (512 cycles per K block); both scale with the tile width.
// Balancing tiles * k_blocks / W blocks against W / tiles partials gives
// W = tiles * sqrt(0.18 * k_blocks), at most the resident clusters.  (Using
// every cluster made a 256 x 256 x 65536 product split its one tile 76 ways
// and spend most of its time in the owner's fix-up.)
int64_t tail_workers(int64_t tiles, int64_t k_blocks, int64_t slots)
{
    int64_t w = int64_t(double(tiles) * sqrt(0.18 * double(k_blocks)) + 0.5);
    if (w < 1) w = 1;
    return w < slots ? w : slots;
}

// Rotation and a stream-K tail exclude each other (the tail does not rotate).
// Rotation wins where it was measured to (one row or column of tiles filling
// most of one wave, e.g. 128 x 16384 x 16384); when fewer than half of the
// slots would have a tile (e.g. one 256 x 256 tile with K = 2^20), only
// splitting K over the clusters keeps the machine busy, and when the tiles
// spill into a second, partial wave (157 tiles of 128 x 128 for 152 SMs:
// 100 x 20000 x 8192), the few clusters of that wave would run alone for a
// whole tile, so the tail wins.
void tail_choice(int64_t tiles_m, int64_t tiles_n, int64_t k_blocks, int64_t slots, bool *rotate, bool *stream_k)
{
    const int64_t tiles = tiles_m * tiles_n;
    const bool sk = streamk_pays(tiles, k_blocks, slots);
    *rotate = rotate_pays(tiles_m, tiles_n, k_blocks) && !(sk && (wave_efficiency(tiles, slots) < 0.5 || tiles > slots));
    *stream_k = sk && !*rotate;
}

// Tile-shape choice, from interleaved measurements on GB300 under the power
// cap:
//  - M <= 128: one 128-row tile of A.  With enough rows of B to give at
//    least half the CTA pairs a tile, the swapped pair tile (variant 13:
//    256 rows of B on the MMA's M side, A's 128 rows on N) brings 24 KB per
//    K block into each SM against 32 KB for the single-CTA 128 x 128 tile
//    (variant 1), measured +0.5 to +4% on products that stream B from HBM
//    (128 x 16384 x 16384: 785 against 767 TFLOP/s; -0.7 to -1.4% on two
//    with K = 4096); with fewer, variant 1, whose K can be split;
//  - otherwise the cheapest of the wide pair tiles, 256 x 512 (variant 15)
//    and 256 x 448 (variant 16), and an alternative with 256-column tiles:
//    the 256 x 256 pair tile (variant 2) for M <= 256 or when its waves keep
//    >= 95% of the pair slots busy, else two pairs sharing B by multicast
//    (variant 4, whole clusters of four SMs only).
// The estimate is waves x work per SM in units of a 256 x 256 pair tile
// (variants 2 and 4: 1 per tile).  A 256 x 512 tile is 2 units but moves 25%
// less data per flop, which under the power cap bought ~6% more clock
// (8192^3: +4-5%); it counts 1.88.  A 256 x 448 tile counts 1.69 (8192^3:
// 8 of its waves ran 3% longer than 7 of the 512-column ones); it pays where
// N / 512 leaves the last wave mostly idle and N / 448 fills it
// (3000 x 5000 x 4096: 1486 against 1433 TFLOP/s; 4096 x 8192 x 4096: 1581
// against 1573 for the 256 x 256 tile).  An alternative whose tail stream-K
// balances counts its tiles / slots plus 3% for the fix-up.  This picked
// the faster plan on 12 of 13 measured shapes (4096^3, 8192^3, 6144^3,
// 3000 x 5000 x 4096, 4096 x 8192 x 4096, ...; the miss, 7168^3, by 0.7%).
int32_t auto_variant(int64_t m, int64_t n, int64_t k_blocks, int32_t num_sms, const int32_t *slots_by_variant,
                     int32_t layout)
{
    if (layout == 1) return m <= 128 ? 6 : 7;  // B stored [K, N], fp32 result
    auto slots_of = [&](int v) -> int64_t {
        const int64_t s = slots_by_variant ? slots_by_variant[v] : num_sms / cluster_of(kVariants[v]);
        return s < 1 ? 1 : s;
    };
    // Small products with fewer than 8 K blocks whose single-CTA tiles fit one wave: the launch is
    // latency-bound, and the smallest tile that still fits one wave shortens each CTA's main loop and
    // its share of C to store.  Device time per launch on GB300 (CUDA graph, 128 x 64 / 128 x 128 /
    // 256 x 256 pair): 256^3 3.66 / 3.89 / 5.74 us; 512 x 512 x 256 3.45 / 3.92; 256 x 1024 x 384
    // 4.02 / 4.47; 128 x 2048 x 256 3.48 / 3.95; 1024 x 1024 x 448 4.62 / 4.81.  Once the 128 x 64
    // tiles need a second wave they lose (2048 x 1024 x 256: 5.01 against 4.08).
    const bool short_k = k_blocks < 8;
    // Few tiles and 16 to 64 K blocks: each SM brings in its operand boxes at a fixed rate (~90
    // GB/s), so a launch whose tiles fit one wave is as long as one tile's K loop.  Sharing each
    // tile's K blocks across a cluster (K split: 4 CTAs of 128 x 64, 2 of 128 x 64 or 2 of 128 x 128)
    // shortens it, at ~2 us for the exchange of partials.  Device time per launch on GB300 (CUDA
    // graph; this choice / the plan chosen before): 256 x 256 x 2048 6.08 / 10.16 us,
    // 128 x 1024 x 2048 6.27 / 10.65, 512 x 512 x 1024 5.54 / 6.30, 512 x 512 x 2048 7.02 / 10.35,
    // 512 x 1024 x 2048 8.32 / 10.45, 768 x 768 x 2048 8.61 / 10.46, 1024 x 1024 x 2048 9.45 / 10.91,
    // 1024 x 1024 x 4096 13.45 / 16.59.  It lost with fewer K blocks (512^3 4.63 / 4.31; 1024^3 on
    // 128 x 128 pairs 8.57 / 6.89) and, with more than 64, to a split K over all the SMs
    // (256 x 256 x 8192 11.98 against 8.29 us).
    if (k_blocks >= 16 && k_blocks <= 64) {
        const int64_t tiles64 = cdiv(m, 128) * cdiv(n, 64), tiles128 = cdiv(m, 128) * cdiv(n, 128);
        if (k_blocks >= 24 && tiles64 <= slots_of(19)) return 19;
        if (tiles64 <= slots_of(20)) return 20;  // (1024 x 512 x 1024: 6.03 against 6.42 us unsplit)
        // (one strip of A rows keeps its split K over more SMs: 100 x 5000 x 3000 12.86 against 13.65 us)
        if (k_blocks >= 32 && m > 128 && tiles128 <= slots_of(21)) return 21;
    }
    // (128 x 32 tiles, variant 22, wherever twice as many tiles still fit one wave: each SM then takes in
    // 20 KB per K block against 24 KB; 256^3 3.00 against 3.21 us, 128^3 2.38 against 2.65, 512^3 4.08
    // against 4.30, 512 x 512 x 256 3.07 against 3.28)
    if (m <= 128) {
        if (short_k && cdiv(n, 32) <= int64_t(num_sms)) return 22;
        if (short_k && cdiv(n, 64) <= int64_t(num_sms)) return 18;
        return 2 * cdiv(n, 256) >= slots_of(13) ? 13 : 1;
    }
    if (short_k && cdiv(m, 128) * cdiv(n, 32) <= int64_t(num_sms)) return 22;
    if (short_k && cdiv(m, 128) * cdiv(n, 64) <= int64_t(num_sms)) return 18;
    if (short_k && cdiv(m, 128) * cdiv(n, 128) <= int64_t(num_sms)) return 1;
    if (n <= 128) return 3;  // a 256-column tile would be half empty: the 256 x 128 pair tile
    // Few tiles and more than 64 K blocks: the single-CTA 128 x 128 tile, its K split over the SMs,
    // up to 4096 tile-K-blocks in all.  Device time per launch on GB300 (CUDA graph; this choice /
    // the pair or multicast tile with split K chosen before): 256 x 256 x 8192 9.93 / 11.54 us,
    // 256 x 256 x 32768 12.83 / 16.99, 512 x 512 x 8192 13.09 / 16.75, 512 x 256 x 16384 11.08 / 15.88,
    // 384 x 384 x 16384 12.89 / 16.38, 256 x 1024 x 16384 17.07 / 19.32.  Beyond (512 x 512 x 32768
    // 24.84 / 23.92) or with more tiles (768 x 768 x 8192 17.07 / 16.21) the larger tiles win.
    {
        const int64_t tiles128 = cdiv(m, 128) * cdiv(n, 128);
        if (k_blocks > 64 && tiles128 <= 16 && tiles128 * k_blocks <= 4096) return 1;
    }
    const int64_t pair_tiles_m = cdiv(m, 256), tiles_n = cdiv(n, 256);
    // Mid-size products (up to 32 K blocks) whose 256 x 256 pair tiles would not fill one wave: the
    // smallest single-CTA tile that still fits one wave, data-parallel.  Device time per launch on
    // GB300 (CUDA graph; this choice / the best other plan / the pair or multicast tile with split K
    // chosen before): 512^3 4.39 / 4.84 / 6.95 us, 1024^3 6.91 / 6.89 / 13.09, 1536^3 9.56 / 9.96 /
    // 18.46, 2048^3 13.30 / 15.20 / 15.42, 1024 x 2048 x 512 5.25 / 5.74 / 7.02.
    if (k_blocks <= 32 && pair_tiles_m * tiles_n < slots_of(2)) {
        for (int32_t v : {22, 18, 1, 0})
            if (cdiv(m, 128) * cdiv(n, kVariants[v].bn) <= int64_t(num_sms)) return v;
    }
    int32_t alt = 2;
    int64_t alt_tiles_m = pair_tiles_m;
    if (m > 256 && wave_efficiency(pair_tiles_m * tiles_n, slots_of(2)) < 0.95) {
        alt = 4;
        alt_tiles_m = cdiv(m, 512);
    }
    const int64_t alt_tiles = alt_tiles_m * tiles_n, alt_slots = slots_of(alt);
    bool alt_rotate = false, alt_sk = false;
    tail_choice(alt_tiles_m, tiles_n, k_blocks, alt_slots, &alt_rotate, &alt_sk);
    const double alt_cost = alt_sk ? 1.03 * double(alt_tiles) / double(alt_slots) : double(cdiv(alt_tiles, alt_slots));
    int32_t best = alt;
    double best_cost = alt_cost;
    for (int32_t v : {15, 16}) {  // on a tie the 512-column tile (fewer, fuller tiles) stays
        const double per_wave = v == 15 ? 1.88 : 1.69;
        const double cost = per_wave * double(cdiv(pair_tiles_m * cdiv(n, kVariants[v].bn), slots_of(v)));
        if (cost < best_cost) {
            best = v;
            best_cost = cost;
        }
    }
    return best;
}

int64_t round_up(int64_t x, int64_t a)
{
    return (x + a - 1) / a * a;
}

// Stream-K workspace: one fp32 partial tile per CTA, then one flag per CTA.
int64_t streamk_partials_bytes(int64_t grid, int32_t block_n)
{
    return round_up(grid * 128 * int64_t(block_n) * 4, 256);
}

int64_t streamk_workspace_bytes(int64_t grid, int32_t block_n)
{
    return streamk_partials_bytes(grid, block_n) + round_up(grid * 8, 256);
}

// Split-K workspace: one fp32 part of 128 x block_n per CTA of every (tile, part).
int64_t splitk_workspace_bytes(int64_t tiles, int64_t parts, int32_t cluster, int32_t block_n)
{
    return round_up(tiles * parts * cluster * 128 * int64_t(block_n) * 4, 256);
}

// Split-K needs the fp16 [N,K] layout without operand swap and tiles of whole 64-column chunks up to
// 256 columns (not the wide tiles).
bool split_capable(const Variant &var)
{
    return var.layout == 0 && !var.swap && var.bn % 64 == 0 && var.bn <= 256 && var.ks == 1;
}

// Parts per tile: about one (tile, part) per resident cluster, each part at least 4 K blocks; a
// forced split takes at least 2 parts.  0: no split.
int64_t split_parts(int64_t tiles, int64_t k_blocks, int64_t slots, bool forced)
{
    int64_t s = tiles > 0 ? slots / tiles : 0;
    if (s > k_blocks / 4) s = k_blocks / 4;
    if (forced && s < 2) s = k_blocks >= 2 ? 2 : 0;
    return s >= 2 ? s : 0;
}

// Stamps of stream-K launches: a per-process random high word and a counter,
// so a flag left by an earlier launch (or found in fresh memory) does not
// equal the current launch's stamp; no clearing launch is needed.
std::atomic<uint64_t> g_sk_counter{0};
uint64_t g_sk_nonce = 0;
std::once_flag g_sk_nonce_once;

uint64_t next_sk_stamp()
{
    std::call_once(g_sk_nonce_once, []() {
        std::random_device rd;
        uint64_t r = (uint64_t(rd()) << 32) ^ uint64_t(rd()) ^
                     uint64_t(std::chrono::steady_clock::now().time_since_epoch().count());
        g_sk_nonce = (r & 0xFFFFFFFF00000000ull) | 0x100000000ull;  // high word, never zero
    });
    const uint64_t c = (g_sk_counter.fetch_add(1) + 1) & 0xFFFFFFFFull;
    return g_sk_nonce | (c ? c : 1u);
}

gemm_status_t make_plan(int64_t m, int64_t n, int64_t k, int32_t num_sms, int32_t max_clusters_in,
                        int32_t variant, int32_t raster_width, int32_t stream_k, gemm_f16_plan_t *out,
                        const int32_t *slots_by_variant = nullptr, int32_t layout = -1)
{
    if (!out) return GEMM_ERR_INVALID_ARG;
    gemm_status_t st = check_shape(m, n, k);
    if (st != GEMM_OK) return st;
    if (num_sms < 1) return GEMM_ERR_INVALID_ARG;
    if (variant >= kNumVariants || stream_k > 2 || layout > 1) return GEMM_ERR_INVALID_ARG;
    if (variant < 0) variant = auto_variant(m, n, cdiv(k, kBlockK), num_sms, slots_by_variant, layout < 0 ? 0 : layout);
    const Variant &var = kVariants[variant];
    if (layout >= 0 && var.layout != layout) return GEMM_ERR_INVALID_ARG;
    const int32_t cs = cluster_of(var);  // CTAs per cluster
    int32_t max_clusters = max_clusters_in > 0 ? max_clusters_in : num_sms / cs;
    if (slots_by_variant) max_clusters = slots_by_variant[variant];
    gemm_f16_plan_t p;
    memset(&p, 0, sizeof(p));
    p.variant = variant;
    p.cta_group = var.cg;
    p.block_m = 128 * var.cg * (var.cg == 2 ? var.mc : 1);  // rows per cluster tile
    p.block_n = var.bn * (var.cg == 1 ? var.mc : 1);      // columns per cluster tile
    p.block_k = kBlockK;
    p.stages = var.stages;
    p.layout = var.layout;
    p.m = m;
    p.n = n;
    p.k = k;
    // a swapped variant tiles the transposed problem: B's n rows on the MMA's M side
    p.tiles_m = cdiv(var.swap ? n : m, p.block_m);
    p.tiles_n = cdiv(var.swap ? m : n, p.block_n);
    p.num_tiles = p.tiles_m * p.tiles_n;
    p.k_blocks = cdiv(k, kBlockK);
    p.cluster = cs;
    p.smem_bytes = var.smem;
    p.num_sms = num_sms;
    if (p.num_tiles >= (int64_t(1) << 31)) return GEMM_ERR_UNSUPPORTED_SHAPE;
    int64_t slots = (cs > 1) ? max_clusters : num_sms;
    if (slots < 1) slots = 1;
    // Data-parallel: as many clusters as the waves need and no more -- 128 tiles on 76 resident CTA
    // pairs take two waves either way, and on 64 pairs both waves are full (4096^3: 79.8 against
    // 80.8 us, the idle SMs' share of the power going to the busy ones).
    const int64_t dp_waves_all = p.num_tiles > 0 ? cdiv(p.num_tiles, slots) : 1;
    int64_t clusters = p.num_tiles > 0 ? cdiv(p.num_tiles, dp_waves_all) : 0;
    p.stream_k = 0;
    p.dp_tiles = p.num_tiles;
    p.sk_iters = 0;
    p.workspace_bytes = 0;
    // rotation or a stream-K tail (tail_choice; the wide tiles' own rule, wide_tail_pays); with the tail
    // forbidden, rotation alone
    const bool wide = is_wide(var);
    bool rotate = false, tail = false;
    tail_choice(p.tiles_m, p.tiles_n, p.k_blocks, slots, &rotate, &tail);
    if (wide) {
        tail = wide_tail_pays(p.num_tiles, p.k_blocks, slots);
        rotate = rotate_pays(p.tiles_m, p.tiles_n, p.k_blocks) && !tail;
    }
    if (var.ks > 1) {
        // K split: whole tiles only, data-parallel (the cluster already shares each tile's K blocks)
        if (stream_k == 1 || stream_k == 2) return GEMM_ERR_INVALID_ARG;
        tail = false;
    }
    if (stream_k == 0) rotate = rotate_pays(p.tiles_m, p.tiles_n, p.k_blocks);
    if (stream_k == 1) rotate = false;
    p.k_rotate = rotate ? 1 : 0;
    const bool want_sk = stream_k == 1 || (stream_k < 0 && tail);
    if (want_sk && p.num_tiles > 0) {
        // whole waves but the last one or two stay data-parallel; the rest is split evenly.  For the
        // wide tiles every whole wave stays data-parallel (a 256 x 512 fp32 partial is 512 KB, so only
        // the partial last wave is worth splitting)
        const int64_t full_waves = p.num_tiles / slots;
        int64_t dp = full_waves >= 1 ? (full_waves - 1) * slots : 0;
        if (wide) dp = full_waves * slots;
        const int64_t sk_iters = (p.num_tiles - dp) * p.k_blocks;
        const int64_t workers = dp == 0 ? tail_workers(p.num_tiles, p.k_blocks, slots) : slots;
        // the tail must shorten the longest cluster's work: data-parallel, the tail's tiles take
        // ceil(left / min(left, slots)) tiles on some cluster; the tail gives each left / workers
        const int64_t left = p.num_tiles - dp;
        const int64_t dp_waves = left > 0 ? cdiv(left, left < slots ? left : slots) : 0;
        if (left > 0 && sk_iters >= workers && left < dp_waves * workers) {
            clusters = workers;
            p.stream_k = 1;
            p.dp_tiles = dp;
            p.sk_iters = sk_iters;
            p.workspace_bytes = uint64_t(streamk_workspace_bytes(clusters * cs, var.bn));
        }
    }
    // Split-K instead of a tail that has no whole wave in front of it (fewer tiles than clusters),
    // or when asked for (stream_k == 2).  Measured on GB300 against the tail sized by tail_workers
    // (sustained TFLOP/s): 256x256x65536 385 vs 132, 512x512x65536 929 vs 429, 1024x1024x16384
    // 1051 vs 895, 200x1000x3000 84 vs 60, 1024^3 150 vs 122, 8192x128x8192 493 vs 476: every
    // split tile's parts are added by the whole GPU instead of one owner after another.
    p.split_k = 0;
    if (stream_k == 2 && !split_capable(var)) return GEMM_ERR_INVALID_ARG;
    const bool split_candidate = stream_k < 0 && split_capable(var) && p.stream_k == 1 && p.dp_tiles == 0;
    if ((stream_k == 2 || split_candidate) && p.num_tiles > 0) {
        const int64_t parts = split_parts(p.num_tiles, p.k_blocks, slots, stream_k == 2);
        if (parts > 1) {
            const int64_t units = p.num_tiles * parts;
            clusters = units < slots ? units : slots;
            p.split_k = int32_t(parts);
            p.stream_k = 0;
            p.dp_tiles = p.num_tiles;
            p.sk_iters = 0;
            p.k_rotate = 0;
            p.workspace_bytes = uint64_t(splitk_workspace_bytes(p.num_tiles, parts, cs, var.bn));
        }
    }
    p.grid = int32_t(clusters * cs);
    if (raster_width <= 0) raster_width = auto_raster_width(p.tiles_n, p.block_n);
    if (p.tiles_n > 0 && raster_width > p.tiles_n) raster_width = int32_t(p.tiles_n);
    if (raster_width < 1) raster_width = 1;
    p.raster_width = raster_width;
    *out = p;
    return GEMM_OK;
}

// Launch a plan this library made for the current device (device_plan) or one run_plan has
// validated: the workspace the caller passed is checked, the plan itself is not checked again.
gemm_status_t launch_plan(const gemm_f16_plan_t &plan, const DeviceInfo *dev, const void *a, const void *b, void *c,
                          void *ws, size_t ws_bytes, cudaStream_t stream, uint32_t skip_fill, long long wait_limit);

gemm_status_t run_plan(const gemm_f16_plan_t &plan, const void *a, const void *b, void *c, void *ws,
                       size_t ws_bytes, cudaStream_t stream, uint32_t skip_fill, long long wait_limit)
{
    gemm_status_t st = check_shape(plan.m, plan.n, plan.k);
    if (st != GEMM_OK) return st;
    st = check_pointers(plan.m, plan.n, plan.k, a, b, c);
    if (st != GEMM_OK) return st;
    if (plan.m == 0 || plan.n == 0) return GEMM_OK;
    if (plan.workspace_bytes > 0 && (ws == nullptr || ws_bytes < plan.workspace_bytes)) return GEMM_ERR_WORKSPACE;
    DeviceInfo *dev = nullptr;
    st = device_info(&dev);
    if (st != GEMM_OK) return st;
    if (plan.variant < 0 || plan.variant >= kNumVariants) return GEMM_ERR_INVALID_ARG;
    if (plan.k == 0) return launch_plan(plan, dev, a, b, c, ws, ws_bytes, stream, skip_fill, wait_limit);
    // the plan must be consistent with what this library computes for its shape
    gemm_f16_plan_t check;
    st = make_plan(plan.m, plan.n, plan.k, plan.num_sms, 0, plan.variant, plan.raster_width, 0, &check);
    if (st != GEMM_OK) return st;
    if (check.variant != plan.variant || check.tiles_m != plan.tiles_m || check.tiles_n != plan.tiles_n ||
        check.k_blocks != plan.k_blocks || check.smem_bytes != plan.smem_bytes || plan.cluster != check.cluster ||
        plan.grid < plan.cluster || plan.grid % plan.cluster != 0)
        return GEMM_ERR_INVALID_ARG;
    const int64_t workers = plan.grid / plan.cluster;
    if (plan.k_rotate != 0 && plan.k_rotate != 1) return GEMM_ERR_INVALID_ARG;
    if (kVariants[plan.variant].ks > 1 && (plan.stream_k != 0 || plan.split_k > 1)) return GEMM_ERR_INVALID_ARG;
    if (plan.split_k > 1) {
        // clusters walk the (tile, part) units persistently and wait for nobody: any grid works
        if (plan.stream_k != 0 || !split_capable(kVariants[plan.variant]) || plan.dp_tiles != plan.num_tiles ||
            plan.sk_iters != 0 || plan.split_k > plan.k_blocks || workers > plan.num_tiles * plan.split_k ||
            int64_t(plan.workspace_bytes) !=
                splitk_workspace_bytes(plan.num_tiles, plan.split_k, plan.cluster, kVariants[plan.variant].bn))
            return GEMM_ERR_INVALID_ARG;
        if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return GEMM_ERR_ALIGNMENT;
        // the reduction runs one thread per float4 of every part: its grid must fit the launch limit
        const int64_t reduce_blocks = cdiv(plan.num_tiles * plan.cluster * 32 * kVariants[plan.variant].bn, 256);
        if (reduce_blocks > 0x7FFFFFFF) return GEMM_ERR_UNSUPPORTED_SHAPE;
    } else if (plan.split_k != 0 && plan.split_k != 1) {
        return GEMM_ERR_INVALID_ARG;
    } else if (plan.stream_k == 0) {
        // any grid of whole clusters is correct: the kernel walks the tiles persistently
        if (plan.dp_tiles != plan.num_tiles || plan.sk_iters != 0 || workers > plan.num_tiles)
            return GEMM_ERR_INVALID_ARG;
    } else {
        // owners wait for contributors: every cluster must be resident at once
        if (plan.stream_k != 1 || plan.dp_tiles < 0 || plan.dp_tiles > plan.num_tiles ||
            plan.sk_iters != (plan.num_tiles - plan.dp_tiles) * plan.k_blocks || plan.sk_iters < workers ||
            workers > dev->max_clusters[plan.variant] ||
            int64_t(plan.workspace_bytes) != streamk_workspace_bytes(plan.grid, kVariants[plan.variant].bn))
            return GEMM_ERR_INVALID_ARG;
    }
    return launch_plan(plan, dev, a, b, c, ws, ws_bytes, stream, skip_fill, wait_limit);
}

// The kernel parameters of one launch of `plan` (k > 0): workspace and pointer checks, the tensor
// maps and the schedule; everything but the stream-K stamp, which every launch draws afresh.
gemm_status_t build_params(const gemm_f16_plan_t &plan, const DeviceInfo *dev, const void *a, const void *b, void *c,
                           void *ws, size_t ws_bytes, uint32_t skip_fill, long long wait_limit, KernelParams *params)
{
    if (plan.workspace_bytes > 0) {
        if (ws == nullptr || ws_bytes < plan.workspace_bytes) return GEMM_ERR_WORKSPACE;
        if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return GEMM_ERR_ALIGNMENT;
    }
    const Variant &var = kVariants[plan.variant];
    if (var.mc > 1) {
        // Cluster multicast loads deliver one copy of a tile to several CTAs of this GPU; they are
        // only used on this GPU's own device memory (never on a peer's or on host-mapped memory).
        const int cur = current_device();
        for (const void *ptr : {a, b}) {
            cudaPointerAttributes at;
            if (cudaPointerGetAttributes(&at, ptr) != cudaSuccess) {
                cudaGetLastError();
                return GEMM_ERR_INVALID_ARG;
            }
            if (at.type != cudaMemoryTypeDevice || at.device != cur) return GEMM_ERR_INVALID_ARG;
        }
    }
    memset(params, 0, sizeof(*params));
    gemm_status_t st = encode_tensor_maps(var, plan, a, b, c, params);
    if (st != GEMM_OK) return st;
    // kernel-side problem: the transposed one for a swapped variant
    const int64_t km = var.swap ? plan.n : plan.m;
    const int64_t kn = var.swap ? plan.m : plan.n;
    params->raster = make_raster(uint32_t(plan.tiles_m), uint32_t(plan.tiles_n), uint32_t(plan.raster_width));
    params->m = uint32_t(km);
    params->n = uint32_t(kn);
    params->k = uint32_t(plan.k);
    params->num_tiles = uint32_t(plan.num_tiles);
    params->k_blocks = uint32_t(plan.k_blocks);
    params->dp_tiles = uint32_t(plan.dp_tiles);
    params->k_rotate = plan.k_rotate ? 1u : 0u;
    params->sk_iters = uint64_t(plan.sk_iters);
    if (plan.split_k > 1) {
        params->split_k = uint32_t(plan.split_k);
        params->partials = static_cast<float *>(ws);
    }
    if (plan.stream_k) {
        params->partials = static_cast<float *>(ws);
        params->flags = reinterpret_cast<uint64_t *>(static_cast<char *>(ws) +
                                                     streamk_partials_bytes(plan.grid, var.bn));
    }
    params->skip_fill = skip_fill;
    params->wait_limit = wait_limit;
    params->error_word = dev->error_word;
    return GEMM_OK;
}

// Launch `plan` with parameters from build_params (a fresh stream-K stamp when it has a tail), and its
// split-K reduction.
gemm_status_t launch_params(const gemm_f16_plan_t &plan, KernelParams &params, void *c, cudaStream_t stream)
{
    const Variant &var = kVariants[plan.variant];
    if (plan.stream_k) params.sk_stamp = next_sk_stamp();
#ifdef GEMM_F16_PHASE_TRACE
    params.trace = g_trace_buffer.load();
#endif
    if (var.launch(plan, params, stream) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    if (plan.split_k > 1 && launch_split_reduce(plan, var, params.raster, params.partials, c, stream) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    return GEMM_OK;
}

gemm_status_t launch_plan(const gemm_f16_plan_t &plan, const DeviceInfo *dev, const void *a, const void *b, void *c,
                          void *ws, size_t ws_bytes, cudaStream_t stream, uint32_t skip_fill, long long wait_limit)
{
    if (plan.m == 0 || plan.n == 0) return GEMM_OK;
    if (plan.k == 0) {
        if (plan.workspace_bytes > 0 && (ws == nullptr || ws_bytes < plan.workspace_bytes)) return GEMM_ERR_WORKSPACE;
        const size_t c_elem = kVariants[plan.variant].layout == 1 ? 4u : 2u;
        if (cudaMemsetAsync(c, 0, size_t(plan.m) * size_t(plan.n) * c_elem, stream) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_LAUNCH;
        }
        return GEMM_OK;
    }
    KernelParams params;
    gemm_status_t st = build_params(plan, dev, a, b, c, ws, ws_bytes, skip_fill, wait_limit, &params);
    if (st != GEMM_OK) return st;
    return launch_params(plan, params, c, stream);
}

// A wait may legitimately last one whole tile's main loop: allow ~1 s plus
// a generous per-K-block allowance.
long long default_wait_limit(int64_t k_blocks)
{
    return 2000000000LL + k_blocks * 65536LL;
}

}  // namespace

extern "C" {

const char *gemm_f16_status_string(gemm_status_t s)
{
    switch (s) {
    case GEMM_OK: return "GEMM_OK";
    case GEMM_ERR_INVALID_ARG: return "GEMM_ERR_INVALID_ARG: invalid argument";
    case GEMM_ERR_ALIGNMENT: return "GEMM_ERR_ALIGNMENT: pointer not 16-byte aligned";
    case GEMM_ERR_UNSUPPORTED_SHAPE: return "GEMM_ERR_UNSUPPORTED_SHAPE: k and n must be multiples of 8, sizes < 2^31";
    case GEMM_ERR_ARCH: return "GEMM_ERR_ARCH: device is not compute capability 10.3 (sm_103a)";
    case GEMM_ERR_WORKSPACE: return "GEMM_ERR_WORKSPACE: workspace missing or too small";
    case GEMM_ERR_LAUNCH: return "GEMM_ERR_LAUNCH: kernel launch failed";
    case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT: a pipeline wait in the kernel timed out";
    case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA: CUDA runtime call failed";
    }
    return "unknown gemm_status_t";
}

// The name the boundary's specification gives the same function.
const char *gemm_status_string(gemm_status_t s)
{
    return gemm_f16_status_string(s);
}

#ifdef GEMM_F16_PHASE_TRACE
void gemm_f16_trace_set(unsigned long long *buffer)
{
    g_trace_buffer.store(buffer);
}
#endif

int32_t gemm_f16_variant_count(void)
{
    return kNumVariants;
}

gemm_status_t gemm_f16_variant_info(int32_t v, int32_t *cta_group, int32_t *block_n, int32_t *stages,
                                    int32_t *smem_bytes, int32_t *cluster, int32_t *layout, int32_t *swapped,
                                    int32_t *k_split)
{
    if (v < 0 || v >= kNumVariants) return GEMM_ERR_INVALID_ARG;
    if (k_split) *k_split = kVariants[v].ks;
    if (swapped) *swapped = kVariants[v].swap;
    if (cluster) *cluster = cluster_of(kVariants[v]);
    if (layout) *layout = kVariants[v].layout;
    if (cta_group) *cta_group = kVariants[v].cg;
    if (block_n) *block_n = kVariants[v].bn;
    if (stages) *stages = kVariants[v].stages;
    if (smem_bytes) *smem_bytes = kVariants[v].smem;
    return GEMM_OK;
}

gemm_status_t gemm_f16_nt_plan_for(int64_t m, int64_t n, int64_t k, int32_t num_sms, int32_t max_clusters,
                                   int32_t variant, int32_t raster_width, int32_t stream_k, gemm_f16_plan_t *out)
{
    return make_plan(m, n, k, num_sms, max_clusters, variant, raster_width, stream_k, out);
}

gemm_status_t gemm_f16_nt_plan_for_clusters(int64_t m, int64_t n, int64_t k, int32_t num_sms,
                                            const int32_t *clusters_by_variant, int32_t count, int32_t variant,
                                            int32_t raster_width, int32_t stream_k, gemm_f16_plan_t *out)
{
    if (!clusters_by_variant || count != kNumVariants) return GEMM_ERR_INVALID_ARG;
    for (int v = 0; v < kNumVariants; ++v)
        if (clusters_by_variant[v] < 1) return GEMM_ERR_INVALID_ARG;
    return make_plan(m, n, k, num_sms, 0, variant, raster_width, stream_k, out, clusters_by_variant);
}

}  // extern "C"

namespace {

// Plan for the current device; arguments as in gemm_f16_nt_plan_for.
gemm_status_t device_plan(int64_t m, int64_t n, int64_t k, int32_t variant, int32_t raster_width, int32_t stream_k,
                          gemm_f16_plan_t *out, int32_t layout = 0, DeviceInfo **dev_out = nullptr)
{
    if (!out) return GEMM_ERR_INVALID_ARG;
    gemm_status_t st = check_shape(m, n, k);
    if (st != GEMM_OK) return st;
    if (variant >= kNumVariants) return GEMM_ERR_INVALID_ARG;
    DeviceInfo *dev = nullptr;
    st = device_info(&dev);
    if (st != GEMM_OK) return st;
    if (dev_out) *dev_out = dev;
    return make_plan(m, n, k, dev->num_sms, 0, variant, raster_width, stream_k, out, dev->max_clusters, layout);
}

// Launches of the automatic entry points repeat: a caller runs the same shapes on the same buffers
// step after step.  Each host thread keeps its last few launches -- plan and encoded parameters --
// keyed on the context, the entry point, the shape, every pointer and the workspace size, so that a
// repeat skips planning and the tensor-map encodes (the parameters depend on nothing else; the
// stream-K stamp is drawn again at every launch).
struct LaunchCacheEntry {
    bool valid;
    int entry;  // 0: gemm_f16_nt, 1: gemm_f16_nt_ws
    unsigned long long ctx;
    int64_t m, n, k;
    const void *a, *b;
    void *c, *ws;
    size_t ws_bytes;
    gemm_f16_plan_t plan;
    KernelParams params;
};
constexpr int kLaunchCacheEntries = 4;
thread_local LaunchCacheEntry t_launch_cache[kLaunchCacheEntries];
thread_local int t_launch_cache_next = 0;

// The automatic plan of (m, n, k) launched on a, b, c (m, n, k > 0, arguments already checked).
gemm_status_t launch_auto(int entry, int64_t m, int64_t n, int64_t k, const void *a, const void *b, void *c, void *ws,
                          size_t ws_bytes, cudaStream_t stream)
{
    unsigned long long ctx = 0;
    gemm_status_t st = current_context_id(&ctx);
    if (st != GEMM_OK) return st;
    for (LaunchCacheEntry &e : t_launch_cache) {
        if (e.valid && e.entry == entry && e.ctx == ctx && e.m == m && e.n == n && e.k == k && e.a == a &&
            e.b == b && e.c == c && e.ws == ws && e.ws_bytes == ws_bytes)
            return launch_params(e.plan, e.params, c, stream);
    }
    gemm_f16_plan_t p;
    DeviceInfo *dev = nullptr;
    st = device_plan(m, n, k, -1, 0, entry == 0 ? 0 : -1, &p, 0, &dev);
    if (st != GEMM_OK) return st;
    LaunchCacheEntry &e = t_launch_cache[t_launch_cache_next];
    e.valid = false;
    st = build_params(p, dev, a, b, c, ws, ws_bytes, ~0u, default_wait_limit(p.k_blocks), &e.params);
    if (st != GEMM_OK) return st;
    e.entry = entry;
    e.ctx = dev->ctx_id;
    e.m = m;
    e.n = n;
    e.k = k;
    e.a = a;
    e.b = b;
    e.c = c;
    e.ws = ws;
    e.ws_bytes = ws_bytes;
    e.plan = p;
    e.valid = true;
    t_launch_cache_next = (t_launch_cache_next + 1) % kLaunchCacheEntries;
    return launch_params(e.plan, e.params, c, stream);
}

// ---------------------------------------------- host-buffer pipeline

// gemm_f16_nt_host moves the rows of A and C through in chunks so that the
// copies of one chunk overlap the GEMM of another: B and the first rows of A
// go in first; then chunk i's GEMM runs on the caller's stream while chunk
// i+1's rows of A come in on one copy stream and chunk i-1's rows of C go out
// on another.  On GB300 the copy engines move ~210 GB/s in and ~190 GB/s out
// (~170 each way at once) and run beside the GEMM at full speed, so the step
// time falls from copies + GEMM towards the inbound copy time.
constexpr int kHostChunksMax = 8;
constexpr int64_t kHostChunkRowsMin = 1024;

struct HostPipe {
    bool ready = false;
    unsigned long long ctx_id = 0;  // the context the streams and events belong to
    cudaStream_t in = nullptr, out = nullptr;  // inbound and outbound copy streams
    cudaEvent_t start = nullptr, in_done = nullptr, out_done = nullptr;
    cudaEvent_t landed[kHostChunksMax] = {};    // chunk i's rows of A (and all of B) are on the device
    cudaEvent_t computed[kHostChunksMax] = {};  // chunk i's rows of C are computed
};

std::mutex g_pipe_mutex;
HostPipe g_pipes[kMaxDevices];

// The current device's copy streams and events, created on first use; call
// with g_pipe_mutex held.
gemm_status_t host_pipe(HostPipe **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    unsigned long long ctx = 0;
    gemm_status_t st = current_context_id(&ctx);
    if (st != GEMM_OK) return st;
    HostPipe &hp = g_pipes[dev];
    if (!hp.ready || hp.ctx_id != ctx) {
        // (streams and events of an earlier, reset context are gone with it)
        HostPipe made;
        made.ctx_id = ctx;
        bool ok = cudaStreamCreateWithFlags(&made.in, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&made.out, cudaStreamNonBlocking) == cudaSuccess;
        cudaEvent_t *events[3 + 2 * kHostChunksMax] = {&made.start, &made.in_done, &made.out_done};
        for (int i = 0; i < kHostChunksMax; ++i) {
            events[3 + 2 * i] = &made.landed[i];
            events[4 + 2 * i] = &made.computed[i];
        }
        for (cudaEvent_t *e : events)
            ok = ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
        if (!ok) {
            cudaGetLastError();
            for (cudaEvent_t *e : events)
                if (*e) cudaEventDestroy(*e);
            if (made.in) cudaStreamDestroy(made.in);
            if (made.out) cudaStreamDestroy(made.out);
            return GEMM_ERR_CUDA;
        }
        made.ready = true;
        hp = made;
    }
    *out = &hp;
    return GEMM_OK;
}

// Rows per chunk: whole 256-row tiles, at least 1024 rows, at most 8 chunks.
int64_t host_chunk_rows(int64_t m)
{
    int64_t chunks = m / kHostChunkRowsMin;
    if (chunks < 1) chunks = 1;
    if (chunks > kHostChunksMax) chunks = kHostChunksMax;
    return round_up(cdiv(m, chunks), 256);
}

// The automatic plan for a chunk, without a stream-K tail when the caller's
// workspace cannot hold one.
gemm_status_t chunk_plan(int64_t m, int64_t n, int64_t k, const void *workspace, size_t ws_bytes,
                         gemm_f16_plan_t *p)
{
    gemm_status_t st = device_plan(m, n, k, -1, 0, -1, p);
    if (st == GEMM_OK && p->workspace_bytes > 0 && (!workspace || ws_bytes < p->workspace_bytes))
        st = device_plan(m, n, k, -1, 0, 0, p);
    return st;
}

}  // namespace

extern "C" {

gemm_status_t gemm_f16_nt_plan(int64_t m, int64_t n, int64_t k, gemm_f16_plan_t *out)
{
    return device_plan(m, n, k, -1, 0, -1, out);
}

gemm_status_t gemm_f16_nt_plan_ex(int64_t m, int64_t n, int64_t k, int32_t variant, int32_t raster_width,
                                  int32_t stream_k, gemm_f16_plan_t *out)
{
    return device_plan(m, n, k, variant, raster_width, stream_k, out);
}

gemm_status_t gemm_f16_nt_workspace_size(int64_t m, int64_t n, int64_t k, size_t *bytes)
{
    if (!bytes) return GEMM_ERR_INVALID_ARG;
    gemm_f16_plan_t p;
    gemm_status_t st = device_plan(m, n, k, -1, 0, -1, &p);
    if (st != GEMM_OK) return st;
    *bytes = size_t(p.workspace_bytes);
    return GEMM_OK;
}

gemm_status_t gemm_f16_nt_ws(int64_t m, int64_t n, int64_t k, const void *a, const void *b, void *c,
                             void *workspace, size_t ws_bytes, gemm_stream_t stream)
{
    gemm_status_t st = check_shape(m, n, k);
    if (st != GEMM_OK) return st;
    st = check_pointers(m, n, k, a, b, c);
    if (st != GEMM_OK) return st;
    if (m == 0 || n == 0) return GEMM_OK;
    if (k == 0) {
        gemm_f16_plan_t p;
        DeviceInfo *dev = nullptr;
        st = device_plan(m, n, k, -1, 0, -1, &p, 0, &dev);
        if (st != GEMM_OK) return st;
        return launch_plan(p, dev, a, b, c, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream), ~0u,
                           default_wait_limit(p.k_blocks));
    }
    return launch_auto(1, m, n, k, a, b, c, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_f16_nt(int64_t m, int64_t n, int64_t k, const void *a, const void *b, void *c,
                          gemm_stream_t stream)
{
    gemm_status_t st = check_shape(m, n, k);
    if (st != GEMM_OK) return st;
    st = check_pointers(m, n, k, a, b, c);
    if (st != GEMM_OK) return st;
    if (m == 0 || n == 0) return GEMM_OK;
    if (k == 0) {
        gemm_f16_plan_t p;
        DeviceInfo *dev = nullptr;
        st = device_plan(m, n, k, -1, 0, 0, &p, 0, &dev);
        if (st != GEMM_OK) return st;
        return launch_plan(p, dev, a, b, c, nullptr, 0, reinterpret_cast<cudaStream_t>(stream), ~0u,
                           default_wait_limit(p.k_blocks));
    }
    return launch_auto(0, m, n, k, a, b, c, nullptr, 0, reinterpret_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_f16_nt_run(const gemm_f16_plan_t *plan, const void *a, const void *b, void *c, void *workspace,
                              size_t ws_bytes, gemm_stream_t stream)
{
    if (!plan) return GEMM_ERR_INVALID_ARG;
    return run_plan(*plan, a, b, c, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream), ~0u,
                    default_wait_limit(plan->k_blocks));
}

gemm_status_t gemm_f16_nn_f32_plan_ex(int64_t m, int64_t n, int64_t k, int32_t variant, int32_t raster_width,
                                      int32_t stream_k, gemm_f16_plan_t *out)
{
    return device_plan(m, n, k, variant, raster_width, stream_k, out, 1);
}

gemm_status_t gemm_f16_nn_f32_ws(int64_t m, int64_t n, int64_t k, const void *a, const void *b, void *d,
                                 void *workspace, size_t ws_bytes, gemm_stream_t stream)
{
    gemm_status_t st = check_shape(m, n, k);
    if (st != GEMM_OK) return st;
    st = check_pointers(m, n, k, a, b, d);
    if (st != GEMM_OK) return st;
    if (m == 0 || n == 0) return GEMM_OK;
    gemm_f16_plan_t p;
    DeviceInfo *dev = nullptr;
    st = device_plan(m, n, k, -1, 0, workspace ? -1 : 0, &p, 1, &dev);
    if (st != GEMM_OK) return st;
    return launch_plan(p, dev, a, b, d, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream), ~0u,
                       default_wait_limit(p.k_blocks));
}

gemm_status_t gemm_f16_nn_f32(int64_t m, int64_t n, int64_t k, const void *a, const void *b, void *d,
                              gemm_stream_t stream)
{
    return gemm_f16_nn_f32_ws(m, n, k, a, b, d, nullptr, 0, stream);
}

// Failure-detection hook: the producer of CTA 0 leaves fill number
// `skip_fill` undone and waits are limited to `wait_limit_cycles`, so the
// kernel's bounded waits expire and report GEMM_ERR_TIMEOUT through
// gemm_f16_take_device_error.
gemm_status_t gemm_f16_nt_run_stall_test(const gemm_f16_plan_t *plan, const void *a, const void *b, void *c,
                                         uint32_t skip_fill, long long wait_limit_cycles, gemm_stream_t stream)
{
    if (!plan || wait_limit_cycles <= 0) return GEMM_ERR_INVALID_ARG;
    return run_plan(*plan, a, b, c, nullptr, 0, reinterpret_cast<cudaStream_t>(stream), skip_fill,
                    wait_limit_cycles);
}

gemm_status_t gemm_f16_nt_host(int64_t m, int64_t n, int64_t k, const void *a_host, const void *b_host,
                               void *c_host, void *a_dev, void *b_dev, void *c_dev, void *workspace,
                               size_t ws_bytes, gemm_stream_t stream)
{
    gemm_status_t st = check_shape(m, n, k);
    if (st != GEMM_OK) return st;
    st = check_pointers(m, n, k, a_dev, b_dev, c_dev);
    if (st != GEMM_OK) return st;
    if (m == 0 || n == 0) return GEMM_OK;
    if (!c_host || (k > 0 && (!a_host || !b_host))) return GEMM_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t rows = host_chunk_rows(m);
    const int64_t chunks = cdiv(m, rows);
    if (k == 0 || chunks == 1) {
        // one chunk: copies in, GEMM, copy out, in stream order
        if (k > 0) {
            if (cudaMemcpyAsync(a_dev, a_host, size_t(m) * size_t(k) * 2u, cudaMemcpyHostToDevice, s) !=
                    cudaSuccess ||
                cudaMemcpyAsync(b_dev, b_host, size_t(n) * size_t(k) * 2u, cudaMemcpyHostToDevice, s) !=
                    cudaSuccess) {
                cudaGetLastError();
                return GEMM_ERR_CUDA;
            }
        }
        st = workspace ? gemm_f16_nt_ws(m, n, k, a_dev, b_dev, c_dev, workspace, ws_bytes, stream)
                       : gemm_f16_nt(m, n, k, a_dev, b_dev, c_dev, stream);
        if (st != GEMM_OK) return st;
        if (cudaMemcpyAsync(c_host, c_dev, size_t(m) * size_t(n) * 2u, cudaMemcpyDeviceToHost, s) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        return GEMM_OK;
    }
    // the plans first, so that a planning error enqueues nothing
    gemm_f16_plan_t plan_full, plan_last;
    const int64_t last_rows = m - (chunks - 1) * rows;
    st = chunk_plan(rows, n, k, workspace, ws_bytes, &plan_full);
    if (st == GEMM_OK) st = chunk_plan(last_rows, n, k, workspace, ws_bytes, &plan_last);
    if (st != GEMM_OK) return st;
    std::lock_guard<std::mutex> lock(g_pipe_mutex);
    HostPipe *hp = nullptr;
    st = host_pipe(&hp);
    if (st != GEMM_OK) return st;
    const char *ah = static_cast<const char *>(a_host);
    char *ad = static_cast<char *>(a_dev), *ch = static_cast<char *>(c_host), *cd = static_cast<char *>(c_dev);
    const size_t a_row = size_t(k) * 2u, c_row = size_t(n) * 2u;
    bool ok = true;
    auto cuda_ok = [&](cudaError_t e) {
        if (e != cudaSuccess) ok = false;
        return ok;
    };
    // both copy streams start after the work the caller has already enqueued on `stream`
    cuda_ok(cudaEventRecord(hp->start, s)) && cuda_ok(cudaStreamWaitEvent(hp->in, hp->start, 0)) &&
        cuda_ok(cudaStreamWaitEvent(hp->out, hp->start, 0)) &&
        cuda_ok(cudaMemcpyAsync(b_dev, b_host, size_t(n) * size_t(k) * 2u, cudaMemcpyHostToDevice, hp->in));
    for (int64_t i = 0; ok && i < chunks; ++i) {
        const int64_t r = (i + 1 < chunks) ? rows : last_rows;
        cuda_ok(cudaMemcpyAsync(ad + size_t(i * rows) * a_row, ah + size_t(i * rows) * a_row, size_t(r) * a_row,
                                cudaMemcpyHostToDevice, hp->in)) &&
            cuda_ok(cudaEventRecord(hp->landed[i], hp->in));
    }
    for (int64_t i = 0; ok && i < chunks; ++i) {
        const bool last = (i + 1 == chunks);
        const gemm_f16_plan_t &p = last ? plan_last : plan_full;
        const int64_t r = last ? last_rows : rows;
        if (!cuda_ok(cudaStreamWaitEvent(s, hp->landed[i], 0))) break;
        st = run_plan(p, ad + size_t(i * rows) * a_row, b_dev, cd + size_t(i * rows) * c_row, workspace, ws_bytes, s,
                      ~0u, default_wait_limit(p.k_blocks));
        if (st != GEMM_OK) {
            ok = false;
            break;
        }
        cuda_ok(cudaEventRecord(hp->computed[i], s)) && cuda_ok(cudaStreamWaitEvent(hp->out, hp->computed[i], 0)) &&
            cuda_ok(cudaMemcpyAsync(ch + size_t(i * rows) * c_row, cd + size_t(i * rows) * c_row, size_t(r) * c_row,
                                    cudaMemcpyDeviceToHost, hp->out));
    }
    // the caller's stream continues after the last copy in and the last copy out (joined even
    // after an error, so that nothing enqueued here outlives the call's place in the stream)
    const bool joined = cudaEventRecord(hp->in_done, hp->in) == cudaSuccess &&
                        cudaEventRecord(hp->out_done, hp->out) == cudaSuccess &&
                        cudaStreamWaitEvent(s, hp->in_done, 0) == cudaSuccess &&
                        cudaStreamWaitEvent(s, hp->out_done, 0) == cudaSuccess;
    if (!ok || !joined) {
        cudaGetLastError();
        return st != GEMM_OK ? st : GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

gemm_status_t gemm_f16_take_device_error(gemm_stream_t stream, uint32_t *code)
{
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    const uint32_t zero = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess ||
        cudaMemcpyFromSymbol(&word, g_gemm_f16_error_word, sizeof(word)) != cudaSuccess ||
        (word != 0 && cudaMemcpyToSymbol(g_gemm_f16_error_word, &zero, sizeof(zero)) != cudaSuccess)) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (code) *code = word;
    return word ? GEMM_ERR_TIMEOUT : GEMM_OK;
}

gemm_status_t gemm_f16_raster_coord(int64_t tiles_m, int64_t tiles_n, int32_t raster_width, int64_t tile,
                                    int64_t *m_block, int64_t *n_block)
{
    if (!m_block || !n_block || tiles_m < 1 || tiles_n < 1 || raster_width < 1) return GEMM_ERR_INVALID_ARG;
    if (tiles_m * tiles_n >= (int64_t(1) << 31) || tile < 0 || tile >= tiles_m * tiles_n)
        return GEMM_ERR_INVALID_ARG;
    Raster r = make_raster(uint32_t(tiles_m), uint32_t(tiles_n), uint32_t(raster_width));
    uint32_t mb, nb;
    raster_coord(r, uint32_t(tile), mb, nb);
    *m_block = mb;
    *n_block = nb;
    return GEMM_OK;
}

gemm_status_t gemm_f16_fast_divmod(uint32_t d, uint32_t n, uint32_t *q, uint32_t *r)
{
    if (d == 0 || !q || !r) return GEMM_ERR_INVALID_ARG;
    FastDiv f = make_fastdiv(d);
    *q = fast_div(f, n);
    *r = n - *q * d;
    return GEMM_OK;
}

}  // extern "C"

// ------------------------------------------------- allocation-free form

// Scratch of gemm_f16_nt_noalloc: the stream-K partial tiles and flags of
// one call at a time, inside the library's device image.
static __device__ __align__(256) unsigned char g_noalloc_scratch[GEMM_F16_STATIC_SCRATCH_BYTES];

namespace {

struct NoallocScratch {
    unsigned long long ctx_id = 0;  // the context the address was looked up in
    void *ptr = nullptr;
};
NoallocScratch g_noalloc[kMaxDevices];

// Device address of g_noalloc_scratch on the current device, looked up with
// that device current once per context (host code must not pass the symbol
// itself to a kernel: in host code it names a host-side stand-in).  After
// cudaDeviceReset the module is loaded anew and the address is looked up
// again.
gemm_status_t noalloc_scratch(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    unsigned long long ctx = 0;
    gemm_status_t st = current_context_id(&ctx);
    if (st != GEMM_OK) return st;
    std::lock_guard<std::mutex> lock(g_mutex);
    NoallocScratch &s = g_noalloc[dev];
    if (s.ptr == nullptr || s.ctx_id != ctx) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        s.ctx_id = ctx;
        s.ptr = ptr;
    }
    *out = s.ptr;
    return GEMM_OK;
}

}  // namespace

extern "C" gemm_status_t gemm_f16_nt_noalloc(int64_t m, int64_t n, int64_t k, const void *a, const void *b,
                                             void *c, gemm_stream_t stream)
{
    gemm_status_t st = check_shape(m, n, k);
    if (st != GEMM_OK) return st;
    st = check_pointers(m, n, k, a, b, c);
    if (st != GEMM_OK) return st;
    if (m == 0 || n == 0) return GEMM_OK;
    gemm_f16_plan_t p;
    DeviceInfo *dev = nullptr;
    st = device_plan(m, n, k, -1, 0, -1, &p, 0, &dev);
    if (st != GEMM_OK) return st;
    if (p.workspace_bytes > uint64_t(GEMM_F16_STATIC_SCRATCH_BYTES)) return GEMM_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (p.workspace_bytes > 0) {
        st = noalloc_scratch(&scratch);
        if (st != GEMM_OK) return st;
    }
    return launch_plan(p, dev, a, b, c, scratch, size_t(GEMM_F16_STATIC_SCRATCH_BYTES),
                       reinterpret_cast<cudaStream_t>(stream), ~0u, default_wait_limit(p.k_blocks));
}
