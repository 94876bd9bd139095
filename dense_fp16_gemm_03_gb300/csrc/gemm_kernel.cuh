// Persistent, warp-specialised sm_103a kernel for C[M,N] = A[M,K] . B[N,K]^T
// (fp16 operands, fp32 accumulation in tensor memory, fp16 result).
//
// What it computes is the product of "1. WGMMA: Hopper's Asynchronous
// Tensor Core" (section "The Full Kernel"); how it is organised takes the
// ideas of "4. Pipeline Abstraction and Two Consumer Warp Groups" -- a
// producer feeding a multi-stage shared-memory ring through full/empty
// mbarriers ("Pipeline Abstraction"), role-specialised warps ("Producer
// Warp", "Consumer Warp Groups"), grouped tile rasterization ("Tile
// Rasterization") -- and rebuilds them for the fifth-generation tensor
// cores:
//
//   warp 0      TMA producer: one thread streams A and B K-blocks into a
//               STAGES-deep ring of 128-byte-swizzled shared-memory tiles.
//   warp 1      MMA issuer: owns the tensor-memory allocation; one thread
//               issues tcgen05.mma (kind::f16, fp32 accumulate) on each
//               ring stage and frees the stage with tcgen05.commit, so the
//               issue loop never waits for an MMA to finish (the "keep MMA
//               work in flight" step the Hopper tutorial leaves for later).
//   warps 2..5  epilogue: tensor memory -> registers -> fp16 (round to
//               nearest even) -> swizzled shared staging -> TMA store, on
//               one of two accumulator buffers while the MMA warp already
//               fills the other one for the next tile.
//
// CG == 2 runs a cluster of two CTAs as one MMA of M = 256 (cta_group::2):
// each CTA loads its own 128 rows of A and half of the B tile, the first
// CTA of the pair issues the MMA for both, and each CTA's tensor memory
// holds its own 128 output rows.
//
// MC > 1 with CG == 1 puts MC single CTAs side by side along N in one
// cluster: they need the same A rows, so each loads 1/MC of the A tile and
// multicasts it to all of them (A + B per CTA becomes A/MC + B).
//
// MC > 1 with CG == 2 stacks MC CTA pairs along M in one cluster: the
// pairs work on vertically adjacent tiles that need the same B columns, so
// each CTA loads only 1/MC of its half of the B tile and multicasts it to
// the CTAs with the same rank-in-pair of the other pairs; a ring stage is
// refilled only after every pair's MMAs have released it.  This cuts each
// CTA's L2-to-shared traffic from A + B/2 to A + B/(2 MC) per K block.
//
// Stream-K tail (optional): the first dp_tiles tiles (whole waves) are
// walked data-parallel, one tile per cluster at a time; the K iterations of
// the remaining tiles are cut into equal contiguous ranges, one per cluster,
// so the last wave is not partly idle.  A cluster whose range starts inside
// a tile publishes its fp32 partial tile to the caller's workspace and sets
// its flag to this launch's stamp; the cluster that holds the tile's first K block adds the
// published partials in its epilogue.  That owning segment is the last one
// in its range while the publishing segments are the first ones in theirs,
// so no cluster ever waits on a cluster that waits on it.
//
// Ragged edges: loads outside [0,M)x[0,K) / [0,N)x[0,K) are zero-filled by
// the TMA unit (so a partial K block adds zeros), stores outside [0,M)x[0,N)
// are dropped by it, and store boxes that start outside C are skipped.
//
// Every mbarrier wait is bounded: past `wait_limit` cycles the waiting
// thread records an error code in a device word, raises a block-wide abort
// flag, and all roles leave their loops, drain what they issued, free the
// tensor memory and return.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <type_traits>

#include "ptx.cuh"
#include "sched.cuh"

namespace gemm_f16 {

constexpr int kBlockK = 64;          // fp16 elements per 128-byte swizzled row
constexpr int kNumThreads = 192;     // 6 warps
constexpr int kEpiWarps = 4;         // one per 32-lane quarter of tensor memory
constexpr int kStoreRows = 32;       // rows per epilogue store box (one warp)
constexpr int kStoreCols = 64;       // columns per store box (128 bytes)
constexpr int kStoreBufBytes = kStoreRows * kStoreCols * 2;
constexpr int kMaxSmem = 232448;     // 227 KB opt-in dynamic shared memory per CTA
// A rotated K walk starts tile t at K block (t * kRotateStride) mod k_blocks.  The stride decides how
// the strips' concurrent reads fall on DRAM channels; measured on GB300 over eight single-strip
// products and three allocations of B each, 67 was fastest on six (128 x 16384 x 16384: 86.4 us
// against 88.4 for 37; 16384 x 128 x 16384 86.6 against 89.6) and within 1.4% on the other two.
constexpr uint32_t kRotateStride = 67u;

// Device error word codes (low byte); bits 8.. hold the CTA index.
enum : uint32_t {
    kErrWaitEmpty = 1,
    kErrWaitFull = 2,
    kErrWaitAccEmpty = 3,
    kErrWaitAccFull = 4,
    kErrWaitDrain = 5,
    kErrWaitPartial = 6,
    kErrWaitRingDrain = 7,   // after an abort, a ring stage's loads did not all land in time
    kErrWaitRecv = 8,        // K split: the partners' partial slices of a tile did not arrive in time
    kErrWaitPeerFree = 9,    // K split: the partners did not free their receive slots in time
};

struct KernelParams {
    CUtensorMap tmap_a;   // A [M, K]: box {64, 128}
    CUtensorMap tmap_b;   // B [N, K]: box {64, BN / CG}
    CUtensorMap tmap_c;   // C [M, N]: fp16 box {64, 32} (fp32 box {32, 32}), 128-byte swizzle
    CUtensorMap tmap_c32; // C [M, N]: box {32, 32}, 64-byte swizzle (last chunk of a tile N % 64 == 32)
    Raster raster;
    uint32_t m, n, k;
    uint32_t num_tiles;
    uint32_t k_blocks;
    uint32_t dp_tiles;    // tiles [0, dp_tiles) are walked data-parallel
    uint32_t k_rotate;    // 1: a whole tile starts its K walk at a per-tile offset (see the producer)
    uint64_t sk_iters;    // K iterations of tiles [dp_tiles, num_tiles), split evenly over the clusters
    uint32_t split_k;     // > 1: split-K, tile t's K blocks cut into split_k parts, each published
    float *partials;      // stream-K workspace: one 128 x BN fp32 partial tile per CTA (split-K: per part and CTA)
    uint64_t *flags;      // stream-K workspace: one "partial published" stamp per CTA
    uint64_t sk_stamp;    // this launch's stamp: a flag equal to it marks a partial of this launch
    uint32_t skip_fill;   // test hook: k-block fill (counted across CTA 0's tiles) the producer
                          // of CTA 0 leaves undone, to exercise the bounded waits; ~0u = none
    long long wait_limit; // cycles a single barrier wait may take before it gives up
    uint32_t *error_word;
    void *c_out;          // C [M, N] fp16, row-major (the K-split epilogue stores it directly)
#ifdef GEMM_F16_PHASE_TRACE
    unsigned long long *trace;  // null, or kTraceSlots global-timer stamps per CTA
#endif
};

// Phase trace (a separate build with GEMM_F16_PHASE_TRACE defined; compiled out otherwise): one
// thread per phase stores %globaltimer (ns) into its CTA's slot each time it passes the phase, so a
// CTA that runs several segments keeps its last segment's stamps.  The store is not waited on;
// reading the slot first would put a global-load round trip into the traced thread's path.
enum TracePhase : int {
    kTraceEntry = 0,       // thread 0 enters the kernel
    kTraceSetUp = 1,       // barriers initialised, tensor memory allocated, CTA (cluster) synchronised
    kTraceDepWait = 2,     // the previous launch in the stream has completed (griddepcontrol.wait)
    kTraceFirstFull = 3,   // the MMA issuer sees a segment's first ring stage full
    kTraceMmaDone = 4,     // a segment's last MMA is committed
    kTraceAccReady = 5,    // the epilogue sees a segment's accumulator complete
    kTraceStored = 6,      // a segment's stores (or published partial) are issued
    kTraceStoresDone = 7,  // the epilogue's bulk stores have all completed
    kTraceTeardown = 8,    // the teardown barrier is passed
    kTraceExit = 9,        // tensor memory is freed; the CTA exits
    kTraceKsSent = 10,     // K split: a tile's partner slices are sent
    kTraceKsReceived = 11, // K split: the partners' slices of a tile have arrived
    kTraceSlots = 16,
};
#ifdef GEMM_F16_PHASE_TRACE
__device__ __forceinline__ void trace_mark(const KernelParams &p, int phase)
{
    if (p.trace == nullptr) return;
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    p.trace[size_t(blockIdx.x) * kTraceSlots + phase] = t;
}
#define GEMM_TRACE(phase) trace_mark(p, phase)
#else
#define GEMM_TRACE(phase) ((void)0)
#endif

// KS > 1 (K split): a cluster of KS single CTAs computes one 128 x BN tile, CTA r accumulating the
// r-th of KS runs of the tile's K blocks; the CTAs then trade fp32 partials through distributed
// shared memory so that CTA r adds all KS partials of columns [r BN / KS, (r + 1) BN / KS) and
// stores them.  It lets the K blocks of few tiles be loaded by more SMs at once: each SM brings in
// its operand boxes at a fixed rate, which bounds a launch with fewer tiles than SMs.
template <int CG, int BN, int STAGES, int MC = 1, bool B_KMAJOR = true, bool C_F16 = true, bool C_TRANS = false,
          int EPI = 2, int KS = 1>
struct KernelCfg {
    static_assert(CG == 1 || CG == 2, "cta group");
    static_assert(MC == 1 || MC == 2 || MC == 4, "cluster multicast width");
    static_assert(KS == 1 || KS == 2 || KS == 4, "K split across the cluster");
    static_assert(KS == 1 || (CG == 1 && MC == 1 && B_KMAJOR && C_F16 && !C_TRANS), "K split: single-CTA fp16 tiles");
    static constexpr bool kAMC = (CG == 1 && MC > 1);  // single CTAs along N share A by multicast
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "tile N");
    static constexpr int kFullChunks = BN / 64;      // 64-column epilogue chunks
    static constexpr bool kTail = (BN % 64) != 0;   // plus one 32-column chunk
    static constexpr int kCS = CG * MC * KS;        // CTAs per cluster
    static constexpr int kKsCols = BN / KS;         // K split: columns of a tile one CTA adds up and stores
    static_assert(KS == 1 || (BN % 64 == 0 && kKsCols % 16 == 0), "K split slices");
    static constexpr int kRecvSlotBytes = 128 * kKsCols * 4;  // K split: one partner's fp32 slice of 128 rows
    static constexpr int kBM = 128 * CG;            // MMA M (one pair)
    static constexpr int kBMCluster = kAMC ? kBM : kBM * MC;  // output rows per scheduling unit
    static constexpr int kBNCluster = kAMC ? BN * MC : BN;    // output columns per scheduling unit
    static constexpr int kBNCta = BN / CG;                    // B rows in one CTA's ring stage
    static constexpr int kBSlice = kAMC ? kBNCta : kBNCta / MC;  // B rows one CTA loads per stage
    static constexpr int kASlice = kAMC ? 128 / MC : 128;        // A rows one CTA loads per stage
    static constexpr int kABytes = 128 * kBlockK * 2;
    static constexpr int kBBytes = kBNCta * kBlockK * 2;
    static constexpr int kStageTx = (kABytes + kBBytes) * CG;  // bytes landing on one full barrier
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + STAGES * kABytes;
    static constexpr int kOffStore = kOffB + STAGES * kBBytes;
    // full, empty, acc_full x2, acc_empty x2, drain; K split: recv_full, peer_free
    static constexpr int kNumBars = 2 * STAGES + 5 + (KS > 1 ? 2 : 0);
    // EPI staging buffers per epilogue warp: 2 lets a warp fill one while the other is being stored;
    // 1 frees 16 KB for one more ring stage
    static_assert(EPI == 1 || EPI == 2, "epilogue staging buffers");
    // K split: where the other variants stage their stores, one receive slot per partner (its slice
    // of this CTA's columns) and one send slot per partner (this CTA's slice of the partner's
    // columns, moved by bulk copies); C is stored from registers
    static constexpr int kEpiBytes = KS > 1 ? 2 * (KS - 1) * kRecvSlotBytes : kEpiWarps * EPI * kStoreBufBytes;
    static constexpr int kOffSend = kOffStore + (KS - 1) * kRecvSlotBytes;
    static constexpr int kOffBar = kOffStore + kEpiBytes;
    static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
    static constexpr int kOffAbort = kOffTmemSlot + 4;
    static constexpr int kOffFills = kOffAbort + 4;  // ring fills the producer walked (read by the abort drain)
    // K split: tiles whose partner slices the epilogue armed / received (read by the abort drain)
    static constexpr int kOffRecvArmed = kOffFills + 4;
    static constexpr int kOffRecvDone = kOffRecvArmed + 4;
    static constexpr int kSmemUsed = kOffFills + 4 + (KS > 1 ? 8 : 0);
    static constexpr int kSmemBytes = kSmemUsed + 1024;  // room to align the base to 1024
    static constexpr int kAccCols = (BN + 63) / 64 * 64;  // accumulator buffer stride (64-column aligned)
    static constexpr int kTmemCols = (2 * kAccCols <= 128) ? 128 : (2 * kAccCols <= 256 ? 256 : 512);
    static_assert(kBBytes % 1024 == 0 && kABytes % 1024 == 0 && (kBSlice * 128) % 1024 == 0 &&
                      (kASlice * 128) % 1024 == 0, "swizzle atoms");
    static_assert(!kAMC || B_KMAJOR, "A multicast with K-major B only");
    // C_TRANS: the kernel computes the transposed product (operands swapped by the host) and
    // the epilogue writes each tile transposed
    static_assert(!C_TRANS || (C_F16 && B_KMAJOR && BN % 64 == 0), "transposed store: fp16, K-major");
    static_assert(BN % (16 * CG) == 0, "MMA N");
    // B stored [K, N] (MN-major operand): whole 64-column swizzle atoms, no multicast slices
    static_assert(B_KMAJOR || (MC == 1 && kBNCta % 64 == 0), "MN-major B tile");
    static constexpr int kBAtomBytes = 64 * kBlockK * 2;  // one 64-column x 64-K-row MN-major atom column
    static_assert(kSmemBytes <= kMaxSmem, "shared memory budget");
};

// tcgen05 shared-memory matrix descriptor for a K-major operand tile written
// by TMA with 128-byte swizzling: rows of 128 bytes, 8-row swizzle atoms of
// 1024 bytes stacked along M/N (stride byte offset 1024); the leading byte
// offset is not used by swizzled K-major layouts.  Fields: start address
// >> 4 (bits 0-13), leading byte offset >> 4 (16-29), stride byte offset
// >> 4 (32-45), descriptor version 1 (46-48), base offset 0 (49-51, tiles
// are 1024-byte aligned), swizzle mode 2 = 128-byte (61-63).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr)
{
    return uint64_t((addr & 0x3FFFFu) >> 4) | (uint64_t(1) << 16) | (uint64_t(1024 >> 4) << 32) |
           (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// Descriptor for an MN-major operand tile written by TMA as 64-element-wide
// (128-byte) columns of 64 K rows each, 128-byte swizzled: the leading byte
// offset is the distance between consecutive 64-element MN atoms (one
// 64 x 64 box, 8 KB), the stride byte offset the distance between groups of
// 8 K rows (1024 bytes); other fields as for the K-major form.
__device__ __forceinline__ uint64_t smem_desc_sw128_mn(uint32_t addr)
{
    return uint64_t((addr & 0x3FFFFu) >> 4) | (uint64_t(8192 >> 4) << 16) | (uint64_t(1024 >> 4) << 32) |
           (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// tcgen05 instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B
// fp16 (bits 7-9, 10-12 = 0), A K-major (bit 15 = 0), B K-major (bit 16 = 0)
// or MN-major (bit 16 = 1), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N, bool b_mn_major = false)
{
    return (1u << 4) | (b_mn_major ? (1u << 16) : 0u) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// After an abort, make sure no TMA load can still write into the ring once
// the CTAs exit.  Run by one thread of every CTA whose full barriers count
// the ring's bytes (every CTA for single-CTA MMAs, the first CTA of each
// pair otherwise), between two cluster barriers of the teardown.
//   fills[x]:  ring fills the producer of cluster CTA x walked (loads issued
//              for each, except the test hook's skipped fill of block 0);
//   share(x):  bytes the loads of one fill by CTA x complete on this CTA's
//              full barrier; stage_tx the bytes this CTA arms per fill.
// A producer issues fill f only after every MMA consumed fill f - STAGES of
// that stage, so only the last STAGES fills can have loads in flight.  For
// each: bytes armed here but never issued are completed by hand, a fill
// never armed here whose loads were issued elsewhere is armed now for just
// those bytes, and then the stage's phase is awaited (bounded).
template <int STAGES, int CS, class Share>
__device__ __forceinline__ void drain_ring(uint32_t bar_full0, const uint32_t (&fills)[CS], uint32_t self, uint32_t first_block,
                           uint32_t stage_tx, Share share, const KernelParams &p)
{
    uint32_t fmax = 0;
#pragma unroll
    for (int x = 0; x < CS; ++x) fmax = fills[x] > fmax ? fills[x] : fmax;
    const uint32_t f0 = fmax > uint32_t(STAGES) ? fmax - uint32_t(STAGES) : 0u;
    for (uint32_t f = f0; f < fmax; ++f) {
        auto issued = [&](uint32_t x) { return f < fills[x] && !(first_block + x == 0u && f == p.skip_fill); };
        uint32_t landing = 0;
#pragma unroll
        for (int x = 0; x < CS; ++x)
            if (issued(uint32_t(x))) landing += share(uint32_t(x));
        const uint32_t bar = bar_full0 + 8u * (f % uint32_t(STAGES));
        if (issued(self)) {
            if (stage_tx > landing) ptx::mbar_complete_tx(bar, stage_tx - landing);
        } else if (landing > 0) {
            ptx::mbar_arrive_expect_tx(bar, landing);
        } else {
            continue;
        }
        const uint32_t parity = (f / uint32_t(STAGES)) & 1u;
        const long long t0 = clock64();
        while (!ptx::mbar_try_wait(bar, parity)) {
            if (clock64() - t0 > p.wait_limit) {
                atomicCAS(p.error_word, 0u, kErrWaitRingDrain | (blockIdx.x << 8));
                break;
            }
        }
    }
}

// Bounded wait on phase `parity` of the barrier at `bar` (cluster-scope
// acquire when the cluster has more than one CTA).
template <int CS>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const KernelParams &p,
                                             volatile uint32_t *abort_flag, uint32_t code)
{
    auto try_once = [&]() {
        if constexpr (CS > 1) return ptx::mbar_try_wait_cluster(bar, parity);
        else return ptx::mbar_try_wait(bar, parity);
    };
    if (try_once()) return true;
    const long long t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (try_once()) return true;
        if ((it & 31u) == 0) {
            if (*abort_flag) return false;
            if (clock64() - t0 > p.wait_limit) {
                *abort_flag = 1u;
                atomicCAS(p.error_word, 0u, code | (blockIdx.x << 8));
                return false;
            }
        }
    }
}

// First stream-K iteration of cluster w (of `workers`).
__device__ __forceinline__ uint64_t sk_begin(const KernelParams &p, uint32_t w, uint32_t workers)
{
    return uint64_t(w) * p.sk_iters / workers;
}

// Every role walks the same sequence of segments (tile, [k_lo, k_hi)):
// data-parallel tiles first, then this cluster's stream-K range; with split-K
// instead the parts u = tile * split_k + s, s-th of split_k equal K ranges,
// one after another per cluster.  f_dp receives the data-parallel tiles,
// f_sk the stream-K segments (and split-K parts); either returns false to
// stop early (abort).  A kernel that never runs split-K plans instantiates
// it with kSplitK = false.
template <bool kSplitK = true, class FD, class FS>
__device__ __forceinline__ void for_each_segment2(const KernelParams &p, uint32_t worker, uint32_t workers, FD &&f_dp,
                                                  FS &&f_sk)
{
    if (kSplitK && p.split_k > 1) {
        const uint64_t units = uint64_t(p.num_tiles) * p.split_k;
        for (uint64_t u = worker; u < units; u += workers) {
            const uint32_t tile = uint32_t(u / p.split_k), part = uint32_t(u % p.split_k);
            const uint32_t k_lo = uint32_t(uint64_t(part) * p.k_blocks / p.split_k);
            const uint32_t k_hi = uint32_t(uint64_t(part + 1) * p.k_blocks / p.split_k);
            if (!f_sk(tile, k_lo, k_hi)) return;
        }
        return;
    }
    for (uint32_t tile = worker; tile < p.dp_tiles; tile += workers)
        if (!f_dp(tile, 0u, p.k_blocks)) return;
    if (p.sk_iters == 0) return;
    uint64_t it = sk_begin(p, worker, workers);
    const uint64_t end = sk_begin(p, worker + 1, workers);
    while (it < end) {
        const uint64_t u = it / p.k_blocks;
        const uint32_t k_lo = uint32_t(it - u * p.k_blocks);
        const uint64_t left = end - it;
        const uint32_t k_hi = (left >= uint64_t(p.k_blocks - k_lo)) ? p.k_blocks : k_lo + uint32_t(left);
        if (!f_sk(p.dp_tiles + uint32_t(u), k_lo, k_hi)) return;
        it += k_hi - k_lo;
    }
}

// As for_each_segment2, with this cluster's last data-parallel tile handed to
// f_last instead of f_dp when no stream-K segment follows it (then nothing
// of this cluster uses the operand ring or tensor memory after that tile).
// The last tile is peeled off the loop, so the three functions' bodies do
// not share live ranges.
template <bool kSplitK = true, class FD, class FL, class FS>
__device__ __forceinline__ void for_each_segment3(const KernelParams &p, uint32_t worker, uint32_t workers, FD &&f_dp,
                                                  FL &&f_last, FS &&f_sk)
{
    if ((kSplitK && p.split_k > 1) || p.sk_iters != 0) {
        for_each_segment2<kSplitK>(p, worker, workers, f_dp, f_sk);
        return;
    }
    if (worker >= p.dp_tiles) return;
    const uint32_t last = worker + (p.dp_tiles - 1u - worker) / workers * workers;
    for (uint32_t tile = worker; tile < last; tile += workers)
        if (!f_dp(tile, 0u, p.k_blocks)) return;
    f_last(last, 0u, p.k_blocks);
}

// The same walk with one function for every segment.
template <bool kSplitK = true, class F>
__device__ __forceinline__ void for_each_segment(const KernelParams &p, uint32_t worker, uint32_t workers, F &&f)
{
    for_each_segment2<kSplitK>(p, worker, workers, f, f);
}

__device__ __forceinline__ uint32_t pack_half2(uint32_t lo_bits, uint32_t hi_bits)
{
    __half2 h = __floats2half2_rn(__uint_as_float(lo_bits), __uint_as_float(hi_bits));
    return *reinterpret_cast<uint32_t *>(&h);
}

// The teardown's abort drain (see drain_ring), run by one thread of every
// CTA that owns full barriers, between two cluster barriers: if any CTA of
// the cluster gave up a wait, wait for the ring loads still in flight.  Kept
// out of line, and recomputing its addresses, so that it costs the main
// loops no registers.
template <int CG, int BN, int STAGES, int MC, bool B_KMAJOR, bool C_F16, bool C_TRANS, int EPI, int KS>
__device__ __noinline__ void nt_abort_drain(const KernelParams &p)
{
    using Cfg = KernelCfg<CG, BN, STAGES, MC, B_KMAJOR, C_F16, C_TRANS, EPI, KS>;
    constexpr int CS = Cfg::kCS;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t cta_rank = (CS > 1) ? ptx::cluster_ctarank() : 0u;
    const uint32_t pair = (KS > 1) ? 0u : cta_rank / CG;
    uint32_t fills[CS];
    bool aborted = false;
    if constexpr (KS > 1) {
        // K split: no CTA loads into another's ring, and a CTA that did not give up received every
        // partner slice sent to it, so this CTA's own state decides
        aborted = *reinterpret_cast<volatile uint32_t *>(smem_raw + (base - raw) + Cfg::kOffAbort) != 0u;
#pragma unroll
        for (int x = 0; x < CS; ++x)
            fills[x] = uint32_t(x) == cta_rank
                           ? *reinterpret_cast<volatile uint32_t *>(smem_raw + (base - raw) + Cfg::kOffFills)
                           : 0u;
    } else if constexpr (CS > 1) {
#pragma unroll
        for (int x = 0; x < CS; ++x) {
            aborted |= ptx::ld_shared_cluster_u32(ptx::map_to_rank(base + Cfg::kOffAbort, uint32_t(x))) != 0u;
            fills[x] = ptx::ld_shared_cluster_u32(ptx::map_to_rank(base + Cfg::kOffFills, uint32_t(x)));
        }
    } else {
        aborted = *reinterpret_cast<volatile uint32_t *>(smem_raw + (base - raw) + Cfg::kOffAbort) != 0u;
        fills[0] = *reinterpret_cast<volatile uint32_t *>(smem_raw + (base - raw) + Cfg::kOffFills);
    }
    if (!aborted) return;
    // bytes one fill of cluster CTA x lands on this CTA's full barriers (see the producer)
    auto share = [&](uint32_t x) -> uint32_t {
        if constexpr (KS > 1) return x == cta_rank ? uint32_t(Cfg::kABytes + Cfg::kBBytes) : 0u;  // own loads only
        else if constexpr (Cfg::kAMC) return uint32_t(Cfg::kASlice * 128) + (x == cta_rank ? uint32_t(Cfg::kBBytes) : 0u);
        else if constexpr (MC == 1) return uint32_t(Cfg::kABytes + Cfg::kBBytes);
        else return ((x / CG) == pair ? uint32_t(Cfg::kABytes) : 0u) + uint32_t(Cfg::kBSlice * 128);
    };
    drain_ring<STAGES, CS>(base + Cfg::kOffBar, fills, cta_rank, blockIdx.x - cta_rank, uint32_t(Cfg::kStageTx),
                           share, p);
    if constexpr (KS > 1) {
        // Partners may have sent their slices of a tile whose arrival this CTA never waited for (the
        // one after the last it received; they send the next only once it has summed the one before).
        // Arm that phase if the epilogue did not and wait for it, bounded: it completes once every
        // partner's bytes have landed, or the wait gives up.
        const uint8_t *smem = smem_raw + (base - raw);
        const uint32_t done = *reinterpret_cast<const volatile uint32_t *>(smem + Cfg::kOffRecvDone);
        const uint32_t armed = *reinterpret_cast<const volatile uint32_t *>(smem + Cfg::kOffRecvArmed);
        const uint32_t bar = base + Cfg::kOffBar + 8u * (2 * STAGES + 5);
        if (armed == done) ptx::mbar_arrive_expect_tx(bar, uint32_t(KS - 1) * uint32_t(Cfg::kRecvSlotBytes));
        const long long t0 = clock64();
        while (!ptx::mbar_try_wait_cluster(bar, done & 1u)) {
            if (clock64() - t0 > p.wait_limit) {
                atomicCAS(p.error_word, 0u, kErrWaitRecv | (blockIdx.x << 8));
                break;
            }
        }
    }
}

template <int CG, int BN, int STAGES, int MC, bool B_KMAJOR, bool C_F16, bool C_TRANS, int EPI, int KS>
__global__ void __launch_bounds__(kNumThreads, 1) gemm_f16_nt_kernel(const __grid_constant__ KernelParams p)
{
    using Cfg = KernelCfg<CG, BN, STAGES, MC, B_KMAJOR, C_F16, C_TRANS, EPI, KS>;
    constexpr int CS = Cfg::kCS;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);

    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t cta_rank = (CS > 1) ? ptx::cluster_ctarank() : 0u;  // rank in the cluster
    const uint32_t ks_rank = (KS > 1) ? cta_rank : 0u;                  // K split: this CTA's run of K blocks
    const uint32_t mc_rank = (KS > 1) ? 0u : cta_rank;                  // rank among CTAs sharing by multicast
    const uint32_t pair_rank = (CG == 2) ? (mc_rank & 1u) : 0u;         // rank in the CTA pair
    const uint32_t pair = mc_rank / CG;                                   // pair index in the cluster
    const uint32_t pair_leader = cta_rank - pair_rank;                    // cluster rank of the pair's first CTA
    const bool leader = (pair_rank == 0);
    const uint32_t cluster_id = blockIdx.x / CS;
    const uint32_t num_clusters = gridDim.x / CS;
    // CTAs whose B slices land in this CTA's stage: same rank-in-pair, every pair
    uint16_t same_rank_mask = 0;
#pragma unroll
    for (int q = 0; q < MC; ++q) same_rank_mask |= uint16_t(1u << (q * CG + pair_rank));

    auto bar_full = [&](uint32_t s) { return base + Cfg::kOffBar + 8u * s; };
    auto bar_empty = [&](uint32_t s) { return base + Cfg::kOffBar + 8u * (STAGES + s); };
    auto bar_acc_full = [&](uint32_t b) { return base + Cfg::kOffBar + 8u * (2 * STAGES + b); };
    auto bar_acc_empty = [&](uint32_t b) { return base + Cfg::kOffBar + 8u * (2 * STAGES + 2 + b); };
    const uint32_t bar_drain = base + Cfg::kOffBar + 8u * (2 * STAGES + 4);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + Cfg::kOffAbort);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Cfg::kOffTmemSlot);
    volatile uint32_t *fills_slot = reinterpret_cast<volatile uint32_t *>(smem + Cfg::kOffFills);
    if (threadIdx.x == 0) GEMM_TRACE(kTraceEntry);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(bar_full(s), 1);
            ptx::mbar_init(bar_empty(s), MC);  // released by the MMA issuer of every pair
        }
        *fills_slot = 0u;
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar_acc_full(b), 1);
            ptx::mbar_init(bar_acc_empty(b), kEpiWarps * CG);
        }
        ptx::mbar_init(bar_drain, 1);
        if constexpr (KS > 1) {
            ptx::mbar_init(base + Cfg::kOffBar + 8u * (2 * STAGES + 5), 1);  // recv_full: armed by the epilogue
            // peer_free: one arrival per epilogue warp of every partner
            ptx::mbar_init(base + Cfg::kOffBar + 8u * (2 * STAGES + 6), uint32_t(KS - 1) * kEpiWarps);
            *reinterpret_cast<volatile uint32_t *>(smem + Cfg::kOffRecvArmed) = 0u;
            *reinterpret_cast<volatile uint32_t *>(smem + Cfg::kOffRecvDone) = 0u;
        }
        *abort_flag = 0u;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&p.tmap_a);
        ptx::prefetch_tmap(&p.tmap_b);
        ptx::prefetch_tmap(&p.tmap_c);
        if constexpr (Cfg::kTail) ptx::prefetch_tmap(&p.tmap_c32);
    }
    if (warp == 1) {
        ptx::tmem_alloc<CG>(ptx::smem_addr(tmem_slot), Cfg::kTmemCols);
        ptx::tmem_relinquish<CG>();
    }
    ptx::tc_fence_before_sync();
    if constexpr (CS > 1) ptx::cluster_sync();
    else __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    if (threadIdx.x == 0) GEMM_TRACE(kTraceSetUp);
    bool arrived = false;  // K split: this thread has already arrived on the teardown's cluster barrier

    // Where this CTA's boxes of a segment start: the A rows m0, the B rows (or, B stored [K, N], the
    // columns) n0, and the K-walk rotation.  With k_rotate, a whole tile walks its K blocks from a
    // per-tile offset, wrapping around: when no operand strip is shared between tiles, lockstep K
    // walks make every CTA read the same K column of rows a power-of-two pitch apart, which piles the
    // requests onto the same DRAM channels.  The MMA consumes stages in order either way.
    auto segment_origin = [&](uint32_t tile, uint32_t k_lo, uint32_t k_hi, int32_t &m0, int32_t &n0, uint32_t &rot) {
        uint32_t mb, nb;
        raster_coord(p.raster, tile, mb, nb);
        m0 = Cfg::kAMC ? int32_t(mb * 128u + cta_rank * Cfg::kASlice)
                       : int32_t(mb * Cfg::kBMCluster + pair * Cfg::kBM + pair_rank * 128u);
        n0 = Cfg::kAMC ? int32_t((nb * MC + cta_rank) * BN)
                       : int32_t(nb * BN + pair_rank * Cfg::kBNCta + pair * Cfg::kBSlice);
        const bool whole = (k_lo == 0u) && (k_hi == p.k_blocks);
        rot = (p.k_rotate && whole) ? uint32_t((uint64_t(tile) * kRotateStride) % p.k_blocks) : 0u;
    };
    // The K blocks [lo, hi) of a segment that this CTA loads and accumulates: all of them, or with a
    // K split the ks_rank-th of KS contiguous runs of the walk (empty when the segment is shorter)
    auto k_share = [&](uint32_t k_lo, uint32_t k_hi, uint32_t &lo, uint32_t &hi) {
        if constexpr (KS > 1) {
            const uint32_t len = k_hi - k_lo;
            lo = k_lo + len * ks_rank / uint32_t(KS);
            hi = k_lo + len * (ks_rank + 1u) / uint32_t(KS);
        } else {
            lo = k_lo;
            hi = k_hi;
        }
    };

    // Launched as a programmatic dependent: the set-up above overlaps the tail of the previous
    // kernel in the stream, and nothing is read or written through the generic or the TMA load path
    // before that kernel has completed (griddepcontrol.wait).  Before the wait, the producer only asks
    // L2 to prefetch the boxes of its first ring fills: a prefetch is a hint with no effect on
    // results (L2 is where every write lands, so a line the previous kernel writes afterwards is
    // still read as written), and it lets this launch's first reads from DRAM overlap the previous
    // launch's last tiles.  The next launch in the stream is let in once this CTA's first
    // accumulator is complete (the epilogue below), not here: triggered at entry, every launch of a
    // long run of small products becomes resident at once, each waiting on its predecessor, and
    // the hand-over from one to the next slows down (one-tile launches replayed from a CUDA graph:
    // 2.51 against 2.32 us at 64^3, 3.71 against 3.43 us at 256^3; level from 512^3 up).
    if (warp == 0 && lane == 0) {
        for_each_segment(p, cluster_id, num_clusters, [&](uint32_t tile, uint32_t k_lo, uint32_t k_hi) {
            int32_t m0, n0;
            uint32_t rot;
            segment_origin(tile, k_lo, k_hi, m0, n0, rot);
            uint32_t lo, hi;
            k_share(k_lo, k_hi, lo, hi);
            for (uint32_t kb = lo; kb < hi && kb < lo + uint32_t(STAGES); ++kb) {
                uint32_t kr = kb + rot;
                if (kr >= p.k_blocks) kr -= p.k_blocks;
                const int32_t k0 = int32_t(kr * kBlockK);
                ptx::tma_prefetch_2d(&p.tmap_a, k0, m0);
                if constexpr (B_KMAJOR) {
                    ptx::tma_prefetch_2d(&p.tmap_b, k0, n0);
                } else {
#pragma unroll
                    for (int h = 0; h < Cfg::kBNCta / 64; ++h) ptx::tma_prefetch_2d(&p.tmap_b, n0 + 64 * h, k0);
                }
            }
            return false;  // the first segment only
        });
    }
    ptx::griddep_wait();
    if (threadIdx.x == 0) GEMM_TRACE(kTraceDepWait);

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, fills = 0;
            bool ok = true;
            for_each_segment(p, cluster_id, num_clusters, [&](uint32_t tile, uint32_t k_lo, uint32_t k_hi) {
                int32_t m0, n0;
                uint32_t rot;
                segment_origin(tile, k_lo, k_hi, m0, n0, rot);
                uint32_t lo, hi;
                k_share(k_lo, k_hi, lo, hi);
                for (uint32_t kb = lo; kb < hi; ++kb, ++fills) {
                    if (!wait_bounded<CS>(bar_empty(stage), phase ^ 1u, p, abort_flag, kErrWaitEmpty)) {
                        ok = false;
                        return false;
                    }
                    const bool skip = (blockIdx.x == 0) && (fills == p.skip_fill);
                    if (!skip) {
                        const uint32_t fb = bar_full(stage);
                        const uint32_t a_dst = base + Cfg::kOffA + stage * Cfg::kABytes;
                        const uint32_t b_dst = base + Cfg::kOffB + stage * Cfg::kBBytes;
                        uint32_t kr = kb + rot;
                        if (kr >= p.k_blocks) kr -= p.k_blocks;
                        const int32_t k0 = int32_t(kr * kBlockK);
                        if constexpr (!B_KMAJOR) {
                            // B stored [K, N]: 64-column boxes of 64 K rows (tensor coordinates {n, k})
                            const uint32_t fbl = (CG == 1) ? fb : ptx::map_to_rank(fb, pair_leader);
                            if (leader) ptx::mbar_arrive_expect_tx(fb, Cfg::kStageTx);
                            if constexpr (CG == 1) ptx::tma_load_2d(a_dst, &p.tmap_a, fbl, k0, m0);
                            else ptx::tma_load_2d_pair(a_dst, &p.tmap_a, fbl, k0, m0);
#pragma unroll
                            for (int h = 0; h < Cfg::kBNCta / 64; ++h) {
                                if constexpr (CG == 1)
                                    ptx::tma_load_2d(b_dst + h * Cfg::kBAtomBytes, &p.tmap_b, fbl, n0 + 64 * h, k0);
                                else
                                    ptx::tma_load_2d_pair(b_dst + h * Cfg::kBAtomBytes, &p.tmap_b, fbl, n0 + 64 * h, k0);
                            }
                        } else if constexpr (Cfg::kAMC) {
                            // every CTA of the cluster receives the whole A tile, 1/MC from each
                            ptx::mbar_arrive_expect_tx(fb, Cfg::kStageTx);
                            ptx::tma_load_2d_mc(a_dst + cta_rank * Cfg::kASlice * 128u, &p.tmap_a, fb, k0, m0,
                                                uint16_t((1u << CS) - 1u));
                            ptx::tma_load_2d(b_dst, &p.tmap_b, fb, k0, n0);
                        } else if constexpr (CG == 1) {
                            ptx::mbar_arrive_expect_tx(fb, Cfg::kStageTx);
                            ptx::tma_load_2d(a_dst, &p.tmap_a, fb, k0, m0);
                            ptx::tma_load_2d(b_dst, &p.tmap_b, fb, k0, n0);
                        } else {
                            const uint32_t fb_leader = ptx::map_to_rank(fb, pair_leader);
                            if (leader) ptx::mbar_arrive_expect_tx(fb, Cfg::kStageTx);
                            ptx::tma_load_2d_pair(a_dst, &p.tmap_a, fb_leader, k0, m0);
                            if constexpr (MC == 1)
                                ptx::tma_load_2d_pair(b_dst, &p.tmap_b, fb_leader, k0, n0);
                            else
                                ptx::tma_load_2d_pair_mc(b_dst + pair * Cfg::kBSlice * 128u, &p.tmap_b, fb_leader, k0,
                                                         n0, same_rank_mask);
                        }
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                return true;
            });
            *fills_slot = fills;  // read by the teardown's abort drain
            (void)ok;
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (leader && lane == 0) {
            constexpr uint32_t idesc = idesc_f16_f32(Cfg::kBM, BN, !B_KMAJOR);
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            for_each_segment(p, cluster_id, num_clusters, [&](uint32_t, uint32_t k_lo, uint32_t k_hi) {
                if (!wait_bounded<CS>(bar_acc_empty(acc), acc_phase ^ 1u, p, abort_flag, kErrWaitAccEmpty))
                    return false;
                ptx::tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + acc * Cfg::kAccCols;
                uint32_t lo, hi;
                k_share(k_lo, k_hi, lo, hi);
                for (uint32_t kb = lo; kb < hi; ++kb) {
                    if (!wait_bounded<CS>(bar_full(stage), phase, p, abort_flag, kErrWaitFull)) return false;
                    ptx::tc_fence_after_sync();
                    if (kb == lo) GEMM_TRACE(kTraceFirstFull);
                    const uint64_t a_desc = smem_desc_sw128(base + Cfg::kOffA + stage * Cfg::kABytes);
                    const uint32_t b_addr = base + Cfg::kOffB + stage * Cfg::kBBytes;
                    const uint64_t b_desc = B_KMAJOR ? smem_desc_sw128(b_addr) : smem_desc_sw128_mn(b_addr);
                    // per 16-element K step: +32 bytes inside a K-major swizzle atom; +2048 bytes
                    // (two 8-row groups) in an MN-major tile
                    constexpr uint64_t kBStep = B_KMAJOR ? 2u : (2048u >> 4);
#pragma unroll
                    for (int kk = 0; kk < kBlockK / 16; ++kk) {
                        ptx::mma_f16<CG>(d_tmem, a_desc + uint64_t(2 * kk), b_desc + kBStep * uint64_t(kk), idesc,
                                         (kb != lo || kk != 0) ? 1u : 0u);
                    }
                    // the stage is free in every CTA whose producer writes into this pair's stage
                    if constexpr (Cfg::kAMC) ptx::mma_commit_mc(bar_empty(stage), uint16_t((1u << CS) - 1u));
                    else if constexpr (CG == 1) ptx::mma_commit(bar_empty(stage));
                    else ptx::mma_commit_pair(bar_empty(stage), uint16_t((1u << CS) - 1u));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if constexpr (CG == 1) ptx::mma_commit(bar_acc_full(acc));
                else ptx::mma_commit_pair(bar_acc_full(acc), uint16_t(0x3u << pair_leader));
                GEMM_TRACE(kTraceMmaDone);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
                return true;
            });
            // No MMA may still be running when the tensor memory is freed.
            if constexpr (CG == 1) ptx::mma_commit(bar_drain);
            else ptx::mma_commit_pair(bar_drain, uint16_t(1u << cta_rank));
            const long long t0 = clock64();
            while (!ptx::mbar_try_wait(bar_drain, 0)) {
                if (clock64() - t0 > p.wait_limit) {
                    atomicCAS(p.error_word, 0u, kErrWaitDrain | (blockIdx.x << 8));
                    break;
                }
            }
        }
    } else {
        // ------------------------------------------------ epilogue
        const uint32_t quarter = warp & 3u;  // tensor-memory lanes [32q, 32q + 32) belong to this warp
        const uint32_t stage_base = base + Cfg::kOffStore + (warp - 2u) * uint32_t(EPI) * kStoreBufBytes;
        const uint32_t lane_sel = (quarter * 32u) << 16;
        constexpr uint32_t kSlotFloats = 128u * BN;          // one CTA's partial tile
        constexpr uint32_t kChunkFloats = 32u * kStoreCols;  // one warp's 32 x 64 piece
        const bool first_epi_thread = (threadIdx.x == 64u);
        uint32_t acc = 0, acc_phase = 0, stores = 0;
        bool released = false;
        // K split: the partners' slots in this CTA, the barrier their bytes complete (armed once per
        // tile) and the one on which the partners report that this CTA's slots in them are free again
        const uint32_t recv_base = base + Cfg::kOffStore;
        const uint32_t bar_recv_full = base + Cfg::kOffBar + 8u * (2 * STAGES + 5);
        const uint32_t bar_peer_free = base + Cfg::kOffBar + 8u * (2 * STAGES + 6);
        uint32_t recv_phase = 0, peer_phase = 0, ks_tiles = 0;
        for_each_segment(p, cluster_id, num_clusters, [&](uint32_t tile, uint32_t k_lo, uint32_t k_hi) {
            uint32_t mb, nb;
            raster_coord(p.raster, tile, mb, nb);
            const uint32_t row0 = Cfg::kAMC ? mb * 128u + quarter * 32u
                                            : mb * Cfg::kBMCluster + pair * Cfg::kBM + pair_rank * 128u + quarter * 32u;
            const uint32_t col0 = Cfg::kAMC ? (nb * MC + cta_rank) * BN : nb * BN;
            const bool ok = wait_bounded<CS>(bar_acc_full(acc), acc_phase, p, abort_flag, kErrWaitAccFull);
            // A stream-K split tile meets the other epilogue warps at named barrier 1 below, so the
            // decision to stop must be the same in all four warps; otherwise it is per warp.
            const bool split = (p.split_k <= 1) && ((k_lo != 0) || (k_hi != p.k_blocks));
            const bool all_ok = split ? ptx::named_barrier_and(1, 32 * kEpiWarps, ok) : __all_sync(0xffffffffu, ok);
            if (!all_ok) return false;
            ptx::tc_fence_after_sync();
            if (!released) {
                ptx::griddep_launch_dependents();  // the first accumulator is ready
                released = true;
            }
            if (first_epi_thread) GEMM_TRACE(kTraceAccReady);
            const uint32_t acc_col = tmem_base + acc * Cfg::kAccCols + lane_sel;
            if constexpr (KS > 1) {
                // ---- K split: every CTA of the cluster holds a partial of the whole tile.  Send the
                // partners their columns, keep this CTA's, add the KS partials of those in rank order
                // (so the sum does not depend on which CTA finishes first) and store them.
                constexpr int W = Cfg::kKsCols;
                constexpr uint32_t kChunks = uint32_t(W) / 4u;  // 16-byte chunks of one row of a slice
                const uint32_t row_local = quarter * 32u + lane;
                const uint32_t len = k_hi - k_lo;
                const bool have = len * (ks_rank + 1u) / uint32_t(KS) > len * ks_rank / uint32_t(KS);
                // this thread's row, columns [j W, j W + W) of the partial (zero: no K block here)
                auto slice = [&](uint32_t j, uint32_t (&v)[W]) {
                    if (have) {
                        if constexpr (W == 16) ptx::tmem_ld_32x32b_x16_wait(acc_col + j * uint32_t(W), v);
                        else if constexpr (W == 32) ptx::tmem_ld_32x32b_x32_wait(acc_col + j * uint32_t(W), v);
                        else ptx::tmem_ld_32x32b_x64_wait(acc_col + j * uint32_t(W), v);
                    } else {
#pragma unroll
                        for (int i = 0; i < W; ++i) v[i] = 0u;
                    }
                };
                // a slot row holds the 16-byte chunks rotated by the row, so that a warp's accesses to
                // one chunk of 32 consecutive rows spread over the banks
                auto chunk_at = [&](uint32_t c) { return ((c ^ (row_local & (kChunks - 1u))) * 16u); };
                // (each wait's outcome is made warp-uniform: the tensor-memory loads and __syncwarp
                // below need the whole warp)
                if (ks_tiles > 0u) {  // the partners have added up this CTA's previous slices
                    const bool free_ok = wait_bounded<CS>(bar_peer_free, peer_phase, p, abort_flag, kErrWaitPeerFree);
                    if (!__all_sync(0xffffffffu, free_ok)) return false;
                    peer_phase ^= 1u;
                }
                // Stage this row of every partner's columns in the send slots (free again: the
                // partners have consumed the previous tile's copies), then one bulk copy per partner
                // moves the warp's 32 rows into the partner's slot for this CTA.
                const uint32_t send_base = base + Cfg::kOffSend;
#pragma unroll
                for (uint32_t j = 0; j < uint32_t(KS); ++j) {
                    if (j == ks_rank) continue;
                    uint32_t v[W];
                    slice(j, v);
                    const uint32_t q = j < ks_rank ? j : j - 1u;  // send slot of partner j
                    const uint32_t row_addr = send_base + q * uint32_t(Cfg::kRecvSlotBytes) + row_local * uint32_t(W * 4);
#pragma unroll
                    for (uint32_t c = 0; c < kChunks; ++c)
                        ptx::st_shared_v4(row_addr + chunk_at(c), v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    constexpr uint32_t kWarpBytes = 32u * uint32_t(W * 4);  // a warp's 32 rows of one slot
                    const uint32_t off = quarter * kWarpBytes;
#pragma unroll
                    for (uint32_t j = 0; j < uint32_t(KS); ++j) {
                        if (j == ks_rank) continue;
                        const uint32_t q = j < ks_rank ? j : j - 1u;
                        const uint32_t slot = ks_rank < j ? ks_rank : ks_rank - 1u;  // this CTA's slot in CTA j
                        ptx::bulk_copy_to_cluster(
                            ptx::map_to_rank(recv_base + slot * uint32_t(Cfg::kRecvSlotBytes) + off, j),
                            send_base + q * uint32_t(Cfg::kRecvSlotBytes) + off, kWarpBytes,
                            ptx::map_to_rank(bar_recv_full, j));
                    }
                }
                if (first_epi_thread) GEMM_TRACE(kTraceKsSent);
                uint32_t own[W];
                slice(ks_rank, own);
                ptx::tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar_acc_empty(acc));  // the accumulator is free for the MMA
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
                if (first_epi_thread) {
                    ptx::mbar_arrive_expect_tx(bar_recv_full, uint32_t(KS - 1) * uint32_t(Cfg::kRecvSlotBytes));
                    *reinterpret_cast<volatile uint32_t *>(smem + Cfg::kOffRecvArmed) = ks_tiles + 1u;
                }
                const bool recv_ok = wait_bounded<CS>(bar_recv_full, recv_phase, p, abort_flag, kErrWaitRecv);
                if (!__all_sync(0xffffffffu, recv_ok)) return false;
                recv_phase ^= 1u;
                if (first_epi_thread) GEMM_TRACE(kTraceKsReceived);
                ++ks_tiles;
                if (first_epi_thread) *reinterpret_cast<volatile uint32_t *>(smem + Cfg::kOffRecvDone) = ks_tiles;
                float sum[W];
#pragma unroll
                for (uint32_t r = 0; r < uint32_t(KS); ++r) {
                    if (r == ks_rank) {
#pragma unroll
                        for (int i = 0; i < W; ++i) sum[i] = r == 0 ? __uint_as_float(own[i]) : sum[i] + __uint_as_float(own[i]);
                    } else {
                        const uint32_t slot = r < ks_rank ? r : r - 1u;
                        const uint32_t src = recv_base + slot * uint32_t(Cfg::kRecvSlotBytes) + row_local * uint32_t(W * 4);
#pragma unroll
                        for (uint32_t c = 0; c < kChunks; ++c) {
                            const float4 x = ptx::ld_shared_f4(src + chunk_at(c));
                            const float t[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) sum[4 * c + e] = r == 0 ? t[e] : sum[4 * c + e] + t[e];
                        }
                    }
                }
                // Every warp has read its rows of the partners' slices: they may refill this CTA's
                // receive slots (a next tile: the reads must be ordered before their copies, a
                // cluster-scope release), or, after the last tile, exit (their copies out of the send
                // slots completed before this CTA's receive barrier did: a plain signal suffices)
                const bool next = tile + num_clusters < p.dp_tiles;
                __syncwarp();
                if (lane == 0) {
#pragma unroll
                    for (uint32_t j = 0; j < uint32_t(KS); ++j) {
                        if (j == ks_rank) continue;
                        if (next) ptx::mbar_arrive_cluster(ptx::map_to_rank(bar_peer_free, j));
                        else ptx::mbar_arrive_cluster_signal(ptx::map_to_rank(bar_peer_free, j));
                    }
                }
                if (!next) {
                    // This warp touches no other CTA's shared memory from here on: arrive on the
                    // teardown's cluster barrier now, so that its latency overlaps the stores of C
                    // instead of waiting for them.  The release covers the signals above; the bulk
                    // copies have landed before any partner arrives (each waits for them first).
                    __syncwarp();
                    ptx::tc_fence_before_sync();
                    ptx::cluster_arrive_release();
                    arrived = true;
                }
                const uint32_t row = row0 + lane;
                const uint32_t col = col0 + ks_rank * uint32_t(W);
                if (row < p.m) {
                    __half *dst = static_cast<__half *>(p.c_out) + size_t(row) * p.n + col;
#pragma unroll
                    for (int g = 0; g < W / 8; ++g) {
                        if (col + uint32_t(8 * g) >= p.n) break;
                        const float *q = sum + 8 * g;
                        ptx::st_global_v4(dst + 8 * g, pack_half2(__float_as_uint(q[0]), __float_as_uint(q[1])),
                                          pack_half2(__float_as_uint(q[2]), __float_as_uint(q[3])),
                                          pack_half2(__float_as_uint(q[4]), __float_as_uint(q[5])),
                                          pack_half2(__float_as_uint(q[6]), __float_as_uint(q[7])));
                    }
                }
                if (first_epi_thread) GEMM_TRACE(kTraceStored);
                return true;
            }
            // Partial-tile layout in the workspace: per warp quarter and 64-column chunk, 16 float4
            // slots x 32 lanes, so every warp-wide 16-byte access is one contiguous 512-byte run.
            const uint32_t piece = quarter * 32u * BN + lane * 4u;
            if (p.split_k > 1 || k_lo != 0) {
                // ---- publish this partial tile: a split-K part to its own slot (the reduction
                // kernel adds the parts), a stream-K part for the owner of the tile to add.  Part s
                // of tile t starts at floor(s * k_blocks / split_k), so s = ceil(k_lo * split_k / k_blocks)
                // (split_k <= k_blocks)
                size_t slot_index = blockIdx.x;
                if (p.split_k > 1) {
                    const uint64_t part = (uint64_t(k_lo) * p.split_k + p.k_blocks - 1) / p.k_blocks;
                    slot_index = (uint64_t(tile) * p.split_k + part) * CS + cta_rank;
                }
                float *slot = p.partials + slot_index * kSlotFloats + piece;
                if (row0 < p.m) {
                    auto publish = [&](auto width, int c) {
                        constexpr int W = decltype(width)::value;
                        if (col0 + uint32_t(c * kStoreCols) >= p.n) return;
                        uint32_t r[W];
                        if constexpr (W == 64) ptx::tmem_ld_32x32b_x64_wait(acc_col + uint32_t(c * kStoreCols), r);
                        else ptx::tmem_ld_32x32b_x32_wait(acc_col + uint32_t(c * kStoreCols), r);
                        float *dst = slot + c * kChunkFloats;
#pragma unroll
                        for (int j = 0; j < W / 4; ++j)
                            ptx::st_global_cg_f4(dst + j * 128, __uint_as_float(r[4 * j]),
                                                 __uint_as_float(r[4 * j + 1]), __uint_as_float(r[4 * j + 2]),
                                                 __uint_as_float(r[4 * j + 3]));
                    };
#pragma unroll 1
                    for (int c = 0; c < Cfg::kFullChunks; ++c) publish(std::integral_constant<int, 64>{}, c);
                    if constexpr (Cfg::kTail) publish(std::integral_constant<int, 32>{}, Cfg::kFullChunks);
                }
                if (p.split_k <= 1) {
                    __threadfence();
                    ptx::named_barrier_sync(1, 32 * kEpiWarps);
                    if (first_epi_thread) ptx::st_release_gpu_u64(p.flags + blockIdx.x, p.sk_stamp);
                }
            } else {
                // ---- a whole tile, or the owning segment of a split tile
                uint32_t first_w = 0, last_w = 0;  // contributors [first_w, last_w)
                if (k_hi != p.k_blocks) {
                    const uint64_t tile_end = uint64_t(tile - p.dp_tiles + 1) * p.k_blocks;
                    first_w = cluster_id + 1;
                    last_w = first_w;
                    while (last_w < num_clusters && sk_begin(p, last_w, num_clusters) < tile_end) ++last_w;
                    if (first_epi_thread) {
                        for (uint32_t w = first_w; w < last_w; ++w) {
                            if (sk_begin(p, w, num_clusters) >= sk_begin(p, w + 1, num_clusters)) continue;
                            const uint64_t *flag = p.flags + w * CS + cta_rank;
                            const long long t0 = clock64();
                            while (ptx::ld_acquire_gpu_u64(flag) != p.sk_stamp) {
                                if (*abort_flag || clock64() - t0 > p.wait_limit) {
                                    *abort_flag = 1u;
                                    atomicCAS(p.error_word, 0u, kErrWaitPartial | (blockIdx.x << 8));
                                    break;
                                }
                            }
                        }
                    }
                    ptx::named_barrier_sync(1, 32 * kEpiWarps);
                }
                if (row0 < p.m) {
                    auto store = [&](auto width, int c) {
                        constexpr int W = decltype(width)::value;
                        const uint32_t col = col0 + uint32_t(c * kStoreCols);
                        if (col >= p.n) return;
                        uint32_t r[W];
                        if constexpr (W == 64) ptx::tmem_ld_32x32b_x64_wait(acc_col + uint32_t(c * kStoreCols), r);
                        else ptx::tmem_ld_32x32b_x32_wait(acc_col + uint32_t(c * kStoreCols), r);
                        for (uint32_t w = first_w; w < last_w; ++w) {
                            if (sk_begin(p, w, num_clusters) >= sk_begin(p, w + 1, num_clusters)) continue;
                            const float *src =
                                p.partials + size_t(w * CS + cta_rank) * kSlotFloats + piece + c * kChunkFloats;
#pragma unroll
                            for (int j = 0; j < W / 4; ++j) {
                                const float4 v = ptx::ld_global_cg_f4(src + j * 128);
                                r[4 * j] = __float_as_uint(__uint_as_float(r[4 * j]) + v.x);
                                r[4 * j + 1] = __float_as_uint(__uint_as_float(r[4 * j + 1]) + v.y);
                                r[4 * j + 2] = __float_as_uint(__uint_as_float(r[4 * j + 2]) + v.z);
                                r[4 * j + 3] = __float_as_uint(__uint_as_float(r[4 * j + 3]) + v.w);
                            }
                        }
                        if constexpr (C_TRANS) {
                            // The tile is D' = C^T: lane = a column n of C, register j = row m of C.
                            // Stage a [64 m][32 n] fp16 block (64-byte rows, unswizzled), store it
                            // with a {32 n, 64 m} box at (n = row0, m = col).
                            const uint32_t buf = stage_base + (EPI == 2 ? (stores & 1u) : 0u) * kStoreBufBytes;
                            if (lane == 0) ptx::bulk_wait_group_read<EPI - 1>();
                            __syncwarp();
#pragma unroll
                            for (int j = 0; j < W; ++j)
                                ptx::st_shared_u16(buf + uint32_t(j) * 64u + lane * 2u,
                                                   __half_as_ushort(__float2half_rn(__uint_as_float(r[j]))));
                            ptx::fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                ptx::tma_store_2d(&p.tmap_c, buf, int32_t(row0), int32_t(col));
                                ptx::bulk_commit_group();
                            }
                            ++stores;
                            return;
                        }
                        if constexpr (!C_F16) {
                            // fp32 result: 32-column (128-byte) swizzled boxes
#pragma unroll
                            for (int h = 0; h < W / 32; ++h) {
                                if (col + 32u * h >= p.n) break;
                                const uint32_t buf = stage_base + (EPI == 2 ? (stores & 1u) : 0u) * kStoreBufBytes;
                                if (lane == 0) ptx::bulk_wait_group_read<EPI - 1>();
                                __syncwarp();
                                const uint32_t row_addr = buf + lane * 128u;
#pragma unroll
                                for (int j = 0; j < 8; ++j)
                                    ptx::st_shared_v4(row_addr + ((uint32_t(j) ^ (lane & 7u)) << 4), r[32 * h + 4 * j],
                                                      r[32 * h + 4 * j + 1], r[32 * h + 4 * j + 2],
                                                      r[32 * h + 4 * j + 3]);
                                ptx::fence_proxy_async_smem();
                                __syncwarp();
                                if (lane == 0) {
                                    ptx::tma_store_2d(&p.tmap_c, buf, int32_t(col + 32u * h), int32_t(row0));
                                    ptx::bulk_commit_group();
                                }
                                ++stores;
                            }
                            return;
                        }
                        const uint32_t buf = stage_base + (EPI == 2 ? (stores & 1u) : 0u) * kStoreBufBytes;
                        if (lane == 0) ptx::bulk_wait_group_read<EPI - 1>();  // this buffer's previous store has read it
                        __syncwarp();
                        if constexpr (W == 64) {
                            const uint32_t row_addr = buf + lane * 128u;
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const uint32_t w0 = pack_half2(r[8 * j + 0], r[8 * j + 1]);
                                const uint32_t w1 = pack_half2(r[8 * j + 2], r[8 * j + 3]);
                                const uint32_t w2 = pack_half2(r[8 * j + 4], r[8 * j + 5]);
                                const uint32_t w3 = pack_half2(r[8 * j + 6], r[8 * j + 7]);
                                // 128-byte swizzle: 16-byte chunk j of row r sits at chunk j ^ (r mod 8)
                                ptx::st_shared_v4(row_addr + ((uint32_t(j) ^ (lane & 7u)) << 4), w0, w1, w2, w3);
                            }
                        } else {
                            // 64-byte rows, 64-byte swizzle: 16-byte chunk j of row r sits at chunk
                            // j ^ ((r / 2) mod 4), so each quarter warp's stores hit distinct banks
                            const uint32_t row_addr = buf + lane * 64u;
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                ptx::st_shared_v4(row_addr + ((uint32_t(j) ^ ((lane >> 1) & 3u)) << 4),
                                                  pack_half2(r[8 * j + 0], r[8 * j + 1]),
                                                  pack_half2(r[8 * j + 2], r[8 * j + 3]),
                                                  pack_half2(r[8 * j + 4], r[8 * j + 5]),
                                                  pack_half2(r[8 * j + 6], r[8 * j + 7]));
                        }
                        ptx::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            ptx::tma_store_2d(W == 64 ? static_cast<const void *>(&p.tmap_c)
                                                      : static_cast<const void *>(&p.tmap_c32),
                                              buf, int32_t(col), int32_t(row0));
                            ptx::bulk_commit_group();
                        }
                        ++stores;
                    };
#pragma unroll 1
                    for (int c = 0; c < Cfg::kFullChunks; ++c) store(std::integral_constant<int, 64>{}, c);
                    if constexpr (Cfg::kTail) store(std::integral_constant<int, 32>{}, Cfg::kFullChunks);
                }
            }
            if (first_epi_thread) GEMM_TRACE(kTraceStored);
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if constexpr (CG == 1) ptx::mbar_arrive(bar_acc_empty(acc));
                else ptx::mbar_arrive_cluster(ptx::map_to_rank(bar_acc_empty(acc), pair_leader));
            }
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
            return true;
        });
        if (lane == 0) ptx::bulk_wait_group<0>();
        if constexpr (KS > 1) {
            // The partners have consumed this CTA's last slices: the bulk copies out of its send
            // slots are complete, so the CTA may exit (bounded: after an abort the wait gives up)
            if (ks_tiles > 0u) (void)wait_bounded<CS>(bar_peer_free, peer_phase, p, abort_flag, kErrWaitPeerFree);
        }
        if (threadIdx.x == 64u) GEMM_TRACE(kTraceStoresDone);
    }

    // ---------------------------------------------------- teardown
    ptx::griddep_launch_dependents();  // a CTA whose epilogue stored nothing still lets the next launch in
    __syncwarp();
    ptx::tc_fence_before_sync();
    if constexpr (KS > 1) {
        if (!arrived) ptx::cluster_arrive_release();  // (arrived: K-split epilogue warps after their last tile)
        ptx::cluster_wait_acquire();
    } else if constexpr (CS > 1) {
        ptx::cluster_sync();
    } else {
        __syncthreads();
    }
    ptx::tc_fence_after_sync();
    if (threadIdx.x == 0) GEMM_TRACE(kTraceTeardown);
    // Between two cluster barriers every CTA of the cluster is still running, so the owners of full
    // barriers may read the other CTAs' flags: after an abort anywhere in the cluster they wait for
    // the ring loads still in flight before any CTA exits.
    if (threadIdx.x == 0 && (CG == 1 || leader))
        nt_abort_drain<CG, BN, STAGES, MC, B_KMAJOR, C_F16, C_TRANS, EPI, KS>(p);
    // (a K-split CTA's drain reads nothing of the other CTAs, and nothing of the cluster touches its
    // shared memory once all have passed the barrier above: no second barrier)
    if constexpr (CS > 1 && KS == 1) ptx::cluster_sync();
    if (warp == 1) ptx::tmem_dealloc<CG>(tmem_base, Cfg::kTmemCols);
    if (threadIdx.x == 32u) GEMM_TRACE(kTraceExit);
}

// Split-K reduction: for every tile, adds its split_k fp32 parts in part
// order and writes the fp16 result (round to nearest even) to C.  The parts
// use the epilogue's publish layout: per CTA, 128 x bn floats in which float4
// number i = (q * bn / 4 + c * 16 + j) * 32 + lane holds row 32 q + lane of
// the CTA's rows and columns 64 c + 4 j .. + 3 of its columns.  One thread per
// float4; rows at or past M and columns at or past N are skipped (the
// epilogue never wrote them), so C outside [0, M) x [0, N) is untouched.
struct SplitReduceParams {
    const float *parts;
    __half *c;
    Raster raster;
    uint32_t m, n;
    uint32_t split_k;
    uint32_t bn;          // columns of one CTA's part (multiple of 64)
    uint32_t cs;          // CTAs per cluster (parts per tile and split)
    uint32_t block_m;     // rows of a cluster tile
    uint32_t block_n;     // columns of a cluster tile
    uint32_t cta_rows;    // row offset between the CTAs of a cluster (128, or 0 when they sit along N)
    uint64_t threads;     // num_tiles * cs * 32 * bn
};

__global__ void __launch_bounds__(256) splitk_reduce_kernel(const __grid_constant__ SplitReduceParams p)
{
    // Launched as a programmatic dependent of the GEMM that wrote the parts: blocks may start on SMs
    // the GEMM has left, and wait here until that whole grid has completed and its writes are visible.
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();
    const uint64_t g = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (g >= p.threads) return;
    const uint64_t per_cta = 32ull * p.bn;  // float4s in one CTA's part
    const uint32_t i = uint32_t(g % per_cta);
    const uint32_t cta = uint32_t((g / per_cta) % p.cs);
    const uint32_t tile = uint32_t(g / (per_cta * p.cs));
    const uint32_t lane = i & 31u, r = i >> 5;
    const uint32_t q = r / (p.bn / 4u), rr = r % (p.bn / 4u);
    const uint32_t chunk = rr / 16u, j = rr % 16u;
    uint32_t mb, nb;
    raster_coord(p.raster, tile, mb, nb);
    const uint32_t row = mb * p.block_m + (p.cta_rows ? cta * p.cta_rows : 0u) + q * 32u + lane;
    const uint32_t col = nb * p.block_n + (p.cta_rows ? 0u : cta * p.bn) + chunk * 64u + j * 4u;
    if (row >= p.m || col >= p.n) return;  // n % 8 == 0, col % 4 == 0: the whole float4 is inside
    const float4 *src = reinterpret_cast<const float4 *>(p.parts) + (uint64_t(tile) * p.split_k * p.cs + cta) * per_cta + i;
    float4 acc = src[0];
    for (uint32_t s = 1; s < p.split_k; ++s) {
        const float4 v = src[uint64_t(s) * p.cs * per_cta];
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
    }
    const __half2 lo = __floats2half2_rn(acc.x, acc.y), hi = __floats2half2_rn(acc.z, acc.w);
    uint2 out;
    out.x = *reinterpret_cast<const uint32_t *>(&lo);
    out.y = *reinterpret_cast<const uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(p.c + uint64_t(row) * p.n + col) = out;
}

}  // namespace gemm_f16
