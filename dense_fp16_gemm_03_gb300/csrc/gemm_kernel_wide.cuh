// Wide-tile variant of the persistent sm_103a kernel: a CTA pair computes a
// 256 x (2 HALF_N) tile of C[M,N] = A[M,K] . B[N,K]^T (fp16 in, fp32
// accumulate, fp16 out) as two cta_group::2 MMAs of N = HALF_N per K step
// (HALF_N = 256: 256 x 512 tiles; 224: 256 x 448; 160: 256 x 320).
//
// Why a wider tile: every byte of A and B reaches a CTA's shared memory
// through the SM's port on the L2 crossbar.  On GB300 that delivery measured
// near 95 GB/s per SM, independent of the SM clock and not relieved by
// cluster multicast (a multicast copy still arrives at each destination SM).
// A 256 x 256 pair tile brings in (128 + 128) x 128 bytes per K block for
// 2 x 128 x 256 x 64 flops per SM (128 flop/byte); a 256 x 512 tile brings in
// (128 + 256) x 128 bytes for twice the flops (171 flop/byte), 25% less
// crossbar traffic per flop.  The accumulator then fills the tensor memory
// (half h at column 256 h), so there is no second buffer for the epilogue to
// drain while the next tile accumulates; instead the epilogue empties tensor
// memory into registers (converted to fp16) at once, releases it to the MMA
// warp, and only then writes the tile out through shared memory and TMA.
// The 448-column form trades 5% of that intensity for wave quantization:
// where N / 512 leaves the last wave of tiles mostly idle, N / 448 can fill
// it (3000 x 5000: 144 tiles for 152 SMs instead of 120).
//
// Roles (320 threads):
//   warp 0      TMA producer: per K block, A (128 rows) and two HALF_N / 2-row
//               B sub-tiles per CTA into a STAGES-deep ring.
//   warp 1      MMA issuer of the pair (first CTA) and tensor-memory owner.
//   warps 2..9  epilogue: warp w reads tensor-memory lanes [32 (w mod 4), +32)
//               and accumulator half (w - 2) / 4, i.e. a 32 x HALF_N piece,
//               stored as 64-column boxes and, when HALF_N mod 64 = 32, one
//               last 32-column box.
//
// The pipeline, the raster order, the K rotation, the ragged-edge rules and
// the bounded waits are those of gemm_kernel.cuh.  A stream-K tail covers only
// the partial last wave (every whole wave stays data-parallel, because a
// partial of a 256 x 512 tile is 512 KB): a segment that ends a tile's K walk
// publishes its fp32 partial straight from tensor memory, and the tile's
// owner, whose segment is the last of its range, adds the partials chunk by
// chunk on the way out.  There is no split-K.
#pragma once

#include "gemm_kernel.cuh"

namespace gemm_f16 {

constexpr int kWideEpiWarps = 8;
constexpr int kWideThreads = 64 + 32 * kWideEpiWarps;

// Shared memory one epilogue warp stages its whole 32 x HALF_N piece in, on a cluster's last tile:
// one 4 KB box per 64-column chunk (and one for a 32-column tail).
template <int HALF_N>
__host__ __device__ constexpr int wide_final_bytes()
{
    return ((HALF_N + 63) / 64) * 4096;
}

template <int STAGES, int HALF_N>
struct WideCfg {
    static_assert(HALF_N % 32 == 0 && HALF_N >= 128 && HALF_N <= 256, "one MMA's N: whole 32-column chunks");
    static constexpr int kHalfN = HALF_N;                 // columns per MMA
    static constexpr int kBN = 2 * HALF_N;                // tile columns: two MMAs
    static constexpr int kBM = 256;                       // tile rows: the pair's MMA M
    static constexpr int kHalfCol = 256;                  // tensor-memory column of accumulator half 1
    static constexpr int kFullChunks = HALF_N / 64;       // 64-column epilogue chunks per half
    static constexpr bool kTail = (HALF_N % 64) != 0;     // plus one 32-column chunk
    static constexpr int kABytes = 128 * kBlockK * 2;     // one CTA's 128 rows of A
    static constexpr int kBBoxRows = HALF_N / 2;          // the rank's share of one MMA's B rows
    static constexpr int kBSubBytes = kBBoxRows * kBlockK * 2;
    static constexpr int kBBytes = 2 * kBSubBytes;
    static constexpr int kStageTx = (kABytes + kBBytes) * 2;  // both CTAs' bytes land on the leader's barrier
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + STAGES * kABytes;
    static constexpr int kOffStore = kOffB + STAGES * kBBytes;
    // full, empty, acc_full, acc_empty, drain, then two per epilogue warp for the stream-K owner's
    // partial pieces
    static constexpr int kNumBars = 2 * STAGES + 3 + 2 * kWideEpiWarps;
    static constexpr int kOffBar = kOffStore + kWideEpiWarps * kStoreBufBytes;
    static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
    static constexpr int kOffAbort = kOffTmemSlot + 4;
    static constexpr int kOffFills = kOffAbort + 4;  // ring fills the producer walked (read by the abort drain)
    static constexpr int kSmemUsed = kOffFills + 4;
    static constexpr int kSmemBytes = kSmemUsed + 1024;  // room to align the base to 1024
    static constexpr int kTmemCols = 512;
    static_assert(kBSubBytes % 1024 == 0, "B sub-tiles stay 1024-byte aligned for the 128-byte swizzle");
    static_assert(STAGES * (kABytes + kBBytes) >= kWideEpiWarps * 2 * 4096, "partial pieces land in the idle ring");
    static_assert(STAGES * (kABytes + kBBytes) >= kWideEpiWarps * wide_final_bytes<HALF_N>(),
                  "the last tile's pieces are staged in the idle ring");
    static_assert(kHalfCol + kHalfN <= kTmemCols, "both accumulator halves fit tensor memory");
    static_assert(kSmemBytes <= kMaxSmem, "shared memory budget");
};

// Write 64 fp16 columns (32 packed words) of one row into a 128-byte-swizzled
// staging row: 16-byte chunk j of row r sits at chunk j ^ (r mod 8).
__device__ __forceinline__ void stage_row_sw128(uint32_t row_addr, uint32_t row, const uint32_t (&w)[32])
{
#pragma unroll
    for (int j = 0; j < 8; ++j)
        ptx::st_shared_v4(row_addr + ((uint32_t(j) ^ (row & 7u)) << 4), w[4 * j], w[4 * j + 1], w[4 * j + 2],
                          w[4 * j + 3]);
}

// The teardown's abort drain of the wide kernel (see drain_ring), run by the
// pair's first CTA between two cluster barriers: if either CTA gave up a
// wait, wait for the ring loads still in flight.  Kept out of line, and
// recomputing its addresses, so that it costs the main loops no registers.
template <int STAGES, int HALF_N>
__device__ __noinline__ void wide_abort_drain(const KernelParams &p)
{
    using Cfg = WideCfg<STAGES, HALF_N>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t abort_addr = base + Cfg::kOffAbort;
    if (ptx::ld_shared_cluster_u32(ptx::map_to_rank(abort_addr, 0u)) == 0u &&
        ptx::ld_shared_cluster_u32(ptx::map_to_rank(abort_addr, 1u)) == 0u)
        return;
    const uint32_t fills_addr = base + Cfg::kOffFills;
    const uint32_t fills[2] = {ptx::ld_shared_cluster_u32(ptx::map_to_rank(fills_addr, 0u)),
                               ptx::ld_shared_cluster_u32(ptx::map_to_rank(fills_addr, 1u))};
    // each CTA's loads of one fill (its A rows, its two B sub-tiles) land on the leader's barrier
    drain_ring<STAGES, 2>(base + Cfg::kOffBar, fills, 0u, blockIdx.x, uint32_t(Cfg::kStageTx),
                          [](uint32_t) { return uint32_t(Cfg::kABytes + Cfg::kBBytes); }, p);
}

template <int STAGES, int HALF_N>
__global__ void __launch_bounds__(kWideThreads, 1) gemm_f16_nt_wide_kernel(const __grid_constant__ KernelParams p)
{
    using Cfg = WideCfg<STAGES, HALF_N>;
    constexpr int CS = 2;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);

    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t pair_rank = ptx::cluster_ctarank();  // the cluster is one CTA pair
    const bool leader = (pair_rank == 0);
    const uint32_t cluster_id = blockIdx.x / CS;
    const uint32_t num_clusters = gridDim.x / CS;

    auto bar_full = [&](uint32_t s) { return base + Cfg::kOffBar + 8u * s; };
    auto bar_empty = [&](uint32_t s) { return base + Cfg::kOffBar + 8u * (STAGES + s); };
    const uint32_t bar_acc_full = base + Cfg::kOffBar + 8u * (2 * STAGES);
    const uint32_t bar_acc_empty = base + Cfg::kOffBar + 8u * (2 * STAGES + 1);
    const uint32_t bar_drain = base + Cfg::kOffBar + 8u * (2 * STAGES + 2);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + Cfg::kOffAbort);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Cfg::kOffTmemSlot);
    volatile uint32_t *fills_slot = reinterpret_cast<volatile uint32_t *>(smem + Cfg::kOffFills);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(bar_full(s), 1);
            ptx::mbar_init(bar_empty(s), 1);
        }
        *fills_slot = 0u;
        ptx::mbar_init(bar_acc_full, 1);
        ptx::mbar_init(bar_acc_empty, kWideEpiWarps * CS);
        ptx::mbar_init(bar_drain, 1);
        for (int b = 0; b < 2 * kWideEpiWarps; ++b) ptx::mbar_init(bar_drain + 8u * (1 + b), 1);
        *abort_flag = 0u;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&p.tmap_a);
        ptx::prefetch_tmap(&p.tmap_b);
        ptx::prefetch_tmap(&p.tmap_c);
        if constexpr (Cfg::kTail) ptx::prefetch_tmap(&p.tmap_c32);
    }
    if (warp == 1) {
        ptx::tmem_alloc<2>(ptx::smem_addr(tmem_slot), Cfg::kTmemCols);
        ptx::tmem_relinquish<2>();
    }
    ptx::tc_fence_before_sync();
    ptx::cluster_sync();
    ptx::tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // As in gemm_kernel.cuh: before waiting for the previous kernel, only L2 prefetches of the first
    // ring fills' boxes (hints, no effect on results).
    ptx::griddep_launch_dependents();
    if (warp == 0 && lane == 0) {
        for_each_segment<false>(p, cluster_id, num_clusters, [&](uint32_t tile, uint32_t k_lo, uint32_t k_hi) {
            uint32_t mb, nb;
            raster_coord(p.raster, tile, mb, nb);
            const int32_t m0 = int32_t(mb * Cfg::kBM + pair_rank * 128u);
            const int32_t n0 = int32_t(nb * Cfg::kBN + pair_rank * uint32_t(Cfg::kBBoxRows));
            const bool whole = (k_lo == 0u) && (k_hi == p.k_blocks);
            const uint32_t rot = (p.k_rotate && whole) ? uint32_t((uint64_t(tile) * kRotateStride) % p.k_blocks) : 0u;
            for (uint32_t kb = k_lo; kb < k_hi && kb < k_lo + uint32_t(STAGES); ++kb) {
                uint32_t kr = kb + rot;
                if (kr >= p.k_blocks) kr -= p.k_blocks;
                const int32_t k0 = int32_t(kr * kBlockK);
                ptx::tma_prefetch_2d(&p.tmap_a, k0, m0);
                ptx::tma_prefetch_2d(&p.tmap_b, k0, n0);
                ptx::tma_prefetch_2d(&p.tmap_b, k0, n0 + Cfg::kHalfN);
            }
            return false;  // the first segment only
        });
    }
    ptx::griddep_wait();

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, fills = 0;
            bool ok = true;
            for_each_segment<false>(p, cluster_id, num_clusters, [&](uint32_t tile, uint32_t k_lo, uint32_t k_hi) {
                uint32_t mb, nb;
                raster_coord(p.raster, tile, mb, nb);
                const int32_t m0 = int32_t(mb * Cfg::kBM + pair_rank * 128u);
                // sub-tile h of this CTA: B rows [nb*BN + HALF_N*h + (HALF_N/2)*rank, +HALF_N/2), the rank's
                // half of MMA h
                const int32_t n0 = int32_t(nb * Cfg::kBN + pair_rank * uint32_t(Cfg::kBBoxRows));
                const bool whole = (k_lo == 0u) && (k_hi == p.k_blocks);
                const uint32_t rot = (p.k_rotate && whole) ? uint32_t((uint64_t(tile) * kRotateStride) % p.k_blocks) : 0u;
                for (uint32_t kb = k_lo; kb < k_hi; ++kb, ++fills) {
                    if (!wait_bounded<CS>(bar_empty(stage), phase ^ 1u, p, abort_flag, kErrWaitEmpty)) {
                        ok = false;
                        return false;
                    }
                    const bool skip = (blockIdx.x == 0) && (fills == p.skip_fill);
                    if (!skip) {
                        const uint32_t fb = bar_full(stage);
                        const uint32_t fb_leader = ptx::map_to_rank(fb, 0u);
                        const uint32_t a_dst = base + Cfg::kOffA + stage * Cfg::kABytes;
                        const uint32_t b_dst = base + Cfg::kOffB + stage * Cfg::kBBytes;
                        uint32_t kr = kb + rot;
                        if (kr >= p.k_blocks) kr -= p.k_blocks;
                        const int32_t k0 = int32_t(kr * kBlockK);
                        if (leader) ptx::mbar_arrive_expect_tx(fb, Cfg::kStageTx);
                        ptx::tma_load_2d_pair(a_dst, &p.tmap_a, fb_leader, k0, m0);
                        ptx::tma_load_2d_pair(b_dst, &p.tmap_b, fb_leader, k0, n0);
                        ptx::tma_load_2d_pair(b_dst + Cfg::kBSubBytes, &p.tmap_b, fb_leader, k0, n0 + Cfg::kHalfN);
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
            constexpr uint32_t idesc = idesc_f16_f32(Cfg::kBM, Cfg::kHalfN);
            uint32_t stage = 0, phase = 0, acc_phase = 0;
            for_each_segment<false>(p, cluster_id, num_clusters, [&](uint32_t, uint32_t k_lo, uint32_t k_hi) {
                if (!wait_bounded<CS>(bar_acc_empty, acc_phase ^ 1u, p, abort_flag, kErrWaitAccEmpty)) return false;
                ptx::tc_fence_after_sync();
                for (uint32_t kb = k_lo; kb < k_hi; ++kb) {
                    if (!wait_bounded<CS>(bar_full(stage), phase, p, abort_flag, kErrWaitFull)) return false;
                    ptx::tc_fence_after_sync();
                    const uint64_t a_desc = smem_desc_sw128(base + Cfg::kOffA + stage * Cfg::kABytes);
                    const uint32_t b_addr = base + Cfg::kOffB + stage * Cfg::kBBytes;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint64_t b_desc = smem_desc_sw128(b_addr + uint32_t(h) * Cfg::kBSubBytes);
#pragma unroll
                        for (int kk = 0; kk < kBlockK / 16; ++kk)
                            ptx::mma_f16<2>(tmem_base + uint32_t(h * Cfg::kHalfCol), a_desc + uint64_t(2 * kk),
                                            b_desc + uint64_t(2 * kk), idesc, (kb != k_lo || kk != 0) ? 1u : 0u);
                    }
                    ptx::mma_commit_pair(bar_empty(stage), uint16_t(0x3u));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                ptx::mma_commit_pair(bar_acc_full, uint16_t(0x3u));
                acc_phase ^= 1u;
                return true;
            });
            // No MMA may still be running when the tensor memory is freed.
            ptx::mma_commit_pair(bar_drain, uint16_t(1u));
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
        const uint32_t quarter = warp & 3u;         // tensor-memory lanes [32q, 32q + 32)
        const uint32_t half = (warp - 2u) >> 2;     // accumulator columns [256 half, +256)
        const uint32_t buf = base + Cfg::kOffStore + (warp - 2u) * kStoreBufBytes;
        const uint32_t row_addr = buf + lane * 128u;
        const uint32_t t_col = tmem_base + ((quarter * 32u) << 16) + half * uint32_t(Cfg::kHalfCol);
        constexpr int kHeld = Cfg::kFullChunks - 1;
        constexpr int kFinalBytes = wide_final_bytes<HALF_N>();
        // Stream-K partial tile of one CTA in the workspace: 128 rows x kBN fp32.  Warp piece
        // (half, quarter) = 32 rows x HALF_N columns at (half * 4 + quarter) * 32 * HALF_N; inside it,
        // 32-column chunk c, float4 j (columns 32c + 4j ..) of lane l at ((c * 8 + j) * 32 + l) * 4,
        // so every warp-wide 16-byte access is one contiguous 512-byte run.
        constexpr uint32_t kSlotFloats = 128u * uint32_t(Cfg::kBN);
        uint32_t acc_phase = 0;
        // a stream-K segment of the tail: publish its fp32 partial (it ends a tile's K walk) or finish a
        // tile as its owner (it starts the tile's K walk; the last segment of this cluster's range)
        auto sk_segment = [&](uint32_t tile, uint32_t k_lo, uint32_t k_hi) {
            uint32_t mb, nb;
            raster_coord(p.raster, tile, mb, nb);
            const uint32_t row0 = mb * Cfg::kBM + pair_rank * 128u + quarter * 32u;
            const uint32_t col0 = nb * Cfg::kBN + half * uint32_t(Cfg::kHalfN);
            const bool ok = wait_bounded<CS>(bar_acc_full, acc_phase, p, abort_flag, kErrWaitAccFull);
            // the owner meets the other epilogue warps at named barrier 1, so the decision to stop
            // must be the same in all eight warps
            if (!ptx::named_barrier_and(1, 32 * kWideEpiWarps, ok)) return false;
            acc_phase ^= 1u;
            ptx::tc_fence_after_sync();
            const bool live = (row0 < p.m) && (col0 < p.n);
            if (k_lo != 0u) {
                // ---- publish: this segment ends the tile's K walk; its fp32 partial goes to this
                // CTA's workspace slot for the tile's owner to add, then the flag gets the stamp
                const uint32_t piece = (half * 4u + quarter) * 32u * uint32_t(Cfg::kHalfN) + lane * 4u;
                float *slot = p.partials + size_t(blockIdx.x) * kSlotFloats + piece;
                if (live) {
#pragma unroll 1
                    for (int c = 0; c < Cfg::kHalfN / 32; ++c) {
                        uint32_t r[32];
                        ptx::tmem_ld_32x32b_x32_wait(t_col + uint32_t(32 * c), r);
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            ptx::st_global_cg_f4(slot + (c * 8 + j) * 128, __uint_as_float(r[4 * j]),
                                                 __uint_as_float(r[4 * j + 1]), __uint_as_float(r[4 * j + 2]),
                                                 __uint_as_float(r[4 * j + 3]));
                    }
                }
                ptx::tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive_cluster_signal(ptx::map_to_rank(bar_acc_empty, 0u));
                __threadfence();
                ptx::named_barrier_sync(1, 32 * kWideEpiWarps);
                if (threadIdx.x == 64u) ptx::st_release_gpu_u64(p.flags + blockIdx.x, p.sk_stamp);
                return true;
            }
            {
                // ---- owner of a tile (always the last segment of this cluster's range): wait
                // for the clusters that hold the rest of the tile's K walk, then add their partials
                // to the accumulator chunk by chunk on the way out; tensor memory is released at the
                // end (nothing of this cluster waits for it)
                const uint64_t tile_end = uint64_t(tile - p.dp_tiles + 1) * p.k_blocks;
                const uint32_t first_w = cluster_id + 1;
                uint32_t last_w = first_w;
                while (last_w < num_clusters && sk_begin(p, last_w, num_clusters) < tile_end) ++last_w;
                if (threadIdx.x == 64u) {
                    for (uint32_t w = first_w; w < last_w; ++w) {
                        if (sk_begin(p, w, num_clusters) >= sk_begin(p, w + 1, num_clusters)) continue;
                        const uint64_t *flag = p.flags + w * CS + pair_rank;
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
                ptx::named_barrier_sync(1, 32 * kWideEpiWarps);
                if (live) {
                    const uint32_t piece = (half * 4u + quarter) * 32u * uint32_t(Cfg::kHalfN) + lane * 4u;
                    auto contributes = [&](uint32_t w) {
                        return sk_begin(p, w, num_clusters) < sk_begin(p, w + 1, num_clusters);
                    };
                    // The owner's segment is this cluster's last: its main loop is done, so the operand
                    // ring is idle.  Each 32-column piece of the first contributor's partial is one
                    // contiguous 4 KB block; it is bulk-copied into one of two 4 KB buffers of this
                    // warp in the ring, one piece ahead, and read from there (lane l, float4 j at
                    // (j * 32 + l) * 16 bytes).  Other contributors, rare, are loaded in turn.
                    uint32_t w0 = first_w;
                    while (w0 < last_w && !contributes(w0)) ++w0;
                    const bool have0 = w0 < last_w;
                    const float *src0 = p.partials + size_t(w0 * CS + pair_rank) * kSlotFloats +
                                        (half * 4u + quarter) * 32u * uint32_t(Cfg::kHalfN);
                    const uint32_t land = base + Cfg::kOffA + (warp - 2u) * 8192u;
                    const uint32_t bar_land = bar_drain + 8u * (1u + 2u * (warp - 2u));
                    constexpr int kPieces = Cfg::kHalfN / 32;
                    auto fetch = [&](int c) {  // lane 0: piece c into buffer c mod 2
                        if (have0 && c < kPieces) {
                            const uint32_t b = uint32_t(c) & 1u;
                            ptx::mbar_arrive_expect_tx(bar_land + 8u * b, 4096u);
                            ptx::bulk_load(land + 4096u * b, src0 + c * 1024, 4096u, bar_land + 8u * b);
                        }
                    };
                    if (lane == 0) {
                        ptx::fence_proxy_async_global();
                        fetch(0);
                        fetch(1);
                    }
                    int used = 0;  // pieces consumed, in order
                    auto wait_piece = [&](int c) {
                        const long long t0 = clock64();
                        while (!ptx::mbar_try_wait(bar_land + 8u * (uint32_t(c) & 1u), (uint32_t(c) >> 1) & 1u)) {
                            if (clock64() - t0 > p.wait_limit) {
                                *abort_flag = 1u;
                                atomicCAS(p.error_word, 0u, kErrWaitPartial | (blockIdx.x << 8));
                                break;
                            }
                        }
                    };
                    // 32 columns at a time: load, add every contributor's partial, round to fp16
                    auto chunk32 = [&](int c, uint32_t (&packed)[16]) {
                        uint32_t r[32];
                        ptx::tmem_ld_32x32b_x32_wait(t_col + uint32_t(32 * c), r);
                        used = c + 1;
                        if (have0) {
                            const uint32_t b = uint32_t(c) & 1u;
                            wait_piece(c);
                            const uint32_t from = land + 4096u * b + lane * 16u;
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const float4 v = ptx::ld_shared_f4(from + uint32_t(j) * 512u);
                                r[4 * j] = __float_as_uint(__uint_as_float(r[4 * j]) + v.x);
                                r[4 * j + 1] = __float_as_uint(__uint_as_float(r[4 * j + 1]) + v.y);
                                r[4 * j + 2] = __float_as_uint(__uint_as_float(r[4 * j + 2]) + v.z);
                                r[4 * j + 3] = __float_as_uint(__uint_as_float(r[4 * j + 3]) + v.w);
                            }
                            // every lane has read the buffer: refill it with the piece after next
                            ptx::fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) fetch(c + 2);
                        }
                        for (uint32_t w = w0 + 1; w < last_w; ++w) {
                            if (!contributes(w)) continue;
                            const float *src = p.partials + size_t(w * CS + pair_rank) * kSlotFloats + piece;
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const float4 v = ptx::ld_global_cg_f4(src + (c * 8 + j) * 128);
                                r[4 * j] = __float_as_uint(__uint_as_float(r[4 * j]) + v.x);
                                r[4 * j + 1] = __float_as_uint(__uint_as_float(r[4 * j + 1]) + v.y);
                                r[4 * j + 2] = __float_as_uint(__uint_as_float(r[4 * j + 2]) + v.z);
                                r[4 * j + 3] = __float_as_uint(__uint_as_float(r[4 * j + 3]) + v.w);
                            }
                        }
#pragma unroll
                        for (int j = 0; j < 16; ++j) packed[j] = pack_half2(r[2 * j], r[2 * j + 1]);
                    };
#pragma unroll 1
                    for (int c = 0; c < Cfg::kFullChunks; ++c) {
                        const uint32_t col = col0 + uint32_t(64 * c);
                        if (col >= p.n) break;
                        uint32_t lo[16], hi[16];
                        chunk32(2 * c, lo);
                        chunk32(2 * c + 1, hi);
                        if (lane == 0) ptx::bulk_wait_group_read<0>();
                        __syncwarp();
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            ptx::st_shared_v4(row_addr + ((uint32_t(j) ^ (lane & 7u)) << 4), lo[4 * j], lo[4 * j + 1],
                                              lo[4 * j + 2], lo[4 * j + 3]);
                            ptx::st_shared_v4(row_addr + ((uint32_t(j + 4) ^ (lane & 7u)) << 4), hi[4 * j],
                                              hi[4 * j + 1], hi[4 * j + 2], hi[4 * j + 3]);
                        }
                        ptx::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            ptx::tma_store_2d(&p.tmap_c, buf, int32_t(col), int32_t(row0));
                            ptx::bulk_commit_group();
                        }
                    }
                    if constexpr (Cfg::kTail) {
                        const uint32_t col = col0 + uint32_t(64 * Cfg::kFullChunks);
                        if (col < p.n) {
                            uint32_t w[16];
                            chunk32(2 * Cfg::kFullChunks, w);
                            if (lane == 0) ptx::bulk_wait_group_read<0>();
                            __syncwarp();
                            const uint32_t row32 = buf + lane * 64u;
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                ptx::st_shared_v4(row32 + ((uint32_t(j) ^ ((lane >> 1) & 3u)) << 4), w[4 * j],
                                                  w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
                            ptx::fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                ptx::tma_store_2d(&p.tmap_c32, buf, int32_t(col), int32_t(row0));
                                ptx::bulk_commit_group();
                            }
                        }
                    }
                    // pieces fetched ahead but not consumed (columns past N): let them land before the
                    // CTA can exit
                    if (have0 && lane == 0)
                        for (int c = used; c < used + 2 && c < kPieces; ++c) wait_piece(c);
                }
                ptx::tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive_cluster_signal(ptx::map_to_rank(bar_acc_empty, 0u));
                return true;
            }
        };
        // this cluster's last tile (no stream-K segment after it): its MMAs consumed every ring stage
        // and no load follows, so the ring is idle.  Each warp stages its whole piece there (one 4 KB box
        // per 64-column chunk, 128-byte swizzled, then the 32-column tail box) and issues all its
        // stores at once instead of one at a time through its staging buffer.
        auto last_tile = [&](uint32_t tile, uint32_t, uint32_t) {
            uint32_t mb, nb;
            raster_coord(p.raster, tile, mb, nb);
            const uint32_t row0 = mb * Cfg::kBM + pair_rank * 128u + quarter * 32u;
            const uint32_t col0 = nb * Cfg::kBN + half * uint32_t(Cfg::kHalfN);
            const bool ok = wait_bounded<CS>(bar_acc_full, acc_phase, p, abort_flag, kErrWaitAccFull);
            if (!__all_sync(0xffffffffu, ok)) return false;
            acc_phase ^= 1u;
            ptx::tc_fence_after_sync();
            const bool live = (row0 < p.m) && (col0 < p.n);
            if (live) {
                const uint32_t area = base + Cfg::kOffA + (warp - 2u) * uint32_t(kFinalBytes);
#pragma unroll 1
                for (int c = 0; c < Cfg::kFullChunks; ++c) {
                    const uint32_t col = col0 + uint32_t(64 * c);
                    if (col >= p.n) break;
                    uint32_t w[32];
#pragma unroll
                    for (int s = 0; s < 2; ++s) {
                        uint32_t r[32];
                        ptx::tmem_ld_32x32b_x32_wait(t_col + uint32_t(64 * c + 32 * s), r);
#pragma unroll
                        for (int j = 0; j < 16; ++j) w[16 * s + j] = pack_half2(r[2 * j], r[2 * j + 1]);
                    }
                    const uint32_t box = area + uint32_t(c) * uint32_t(kStoreBufBytes);
                    stage_row_sw128(box + lane * 128u, lane, w);
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) ptx::tma_store_2d(&p.tmap_c, box, int32_t(col), int32_t(row0));
                }
                if constexpr (Cfg::kTail) {
                    const uint32_t col = col0 + uint32_t(64 * Cfg::kFullChunks);
                    if (col < p.n) {
                        uint32_t r[32];
                        ptx::tmem_ld_32x32b_x32_wait(t_col + uint32_t(64 * Cfg::kFullChunks), r);
                        const uint32_t box = area + uint32_t(Cfg::kFullChunks) * uint32_t(kStoreBufBytes);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            ptx::st_shared_v4(box + lane * 64u + ((uint32_t(j) ^ ((lane >> 1) & 3u)) << 4),
                                              pack_half2(r[8 * j + 0], r[8 * j + 1]),
                                              pack_half2(r[8 * j + 2], r[8 * j + 3]),
                                              pack_half2(r[8 * j + 4], r[8 * j + 5]),
                                              pack_half2(r[8 * j + 6], r[8 * j + 7]));
                        ptx::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) ptx::tma_store_2d(&p.tmap_c32, box, int32_t(col), int32_t(row0));
                    }
                }
                if (lane == 0) ptx::bulk_commit_group();
            }
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_cluster_signal(ptx::map_to_rank(bar_acc_empty, 0u));
            return true;
        };
        for_each_segment3<false>(p, cluster_id, num_clusters, [&](uint32_t tile, uint32_t, uint32_t) {
            uint32_t mb, nb;
            raster_coord(p.raster, tile, mb, nb);
            const uint32_t row0 = mb * Cfg::kBM + pair_rank * 128u + quarter * 32u;
            const uint32_t col0 = nb * Cfg::kBN + half * uint32_t(Cfg::kHalfN);
            const bool ok = wait_bounded<CS>(bar_acc_full, acc_phase, p, abort_flag, kErrWaitAccFull);
            if (!__all_sync(0xffffffffu, ok)) return false;
            acc_phase ^= 1u;
            ptx::tc_fence_after_sync();
            const bool live = (row0 < p.m) && (col0 < p.n);
            uint32_t held[kHeld][32];             // 64-column chunks 1.. of this warp's piece, packed fp16 pairs
            uint32_t tail[Cfg::kTail ? 16 : 1];   // the last 32 columns when HALF_N mod 64 = 32
            if (live) {
                // Columns 0..63 go straight to the staging buffer (its previous store was issued a
                // whole main loop ago); the rest wait in registers.  32 columns per load keep the
                // registers live at once near 128 words a thread.
                if (lane == 0) ptx::bulk_wait_group_read<0>();
                __syncwarp();
                {
                    uint32_t w[32];
#pragma unroll
                    for (int s = 0; s < 2; ++s) {
                        uint32_t r[32];
                        ptx::tmem_ld_32x32b_x32_wait(t_col + uint32_t(32 * s), r);
#pragma unroll
                        for (int j = 0; j < 16; ++j) w[16 * s + j] = pack_half2(r[2 * j], r[2 * j + 1]);
                    }
                    stage_row_sw128(row_addr, lane, w);
                }
#pragma unroll
                for (int c = 1; c <= kHeld; ++c) {
#pragma unroll
                    for (int s = 0; s < 2; ++s) {
                        uint32_t r[32];
                        ptx::tmem_ld_32x32b_x32_wait(t_col + uint32_t(64 * c + 32 * s), r);
#pragma unroll
                        for (int j = 0; j < 16; ++j) held[c - 1][16 * s + j] = pack_half2(r[2 * j], r[2 * j + 1]);
                    }
                }
                if constexpr (Cfg::kTail) {
                    uint32_t r[32];
                    ptx::tmem_ld_32x32b_x32_wait(t_col + uint32_t(64 * Cfg::kFullChunks), r);
#pragma unroll
                    for (int j = 0; j < 16; ++j) tail[j] = pack_half2(r[2 * j], r[2 * j + 1]);
                }
            }
            // tensor memory is free for the next tile as soon as every warp has read its piece; the
            // loads are complete (tcgen05.wait::ld), so the arrival only signals, with CTA-scope
            // release: a cluster-scope one stalled each warp ~950 cycles while the MMA warp waited
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_cluster_signal(ptx::map_to_rank(bar_acc_empty, 0u));
            if (live) {
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    ptx::tma_store_2d(&p.tmap_c, buf, int32_t(col0), int32_t(row0));
                    ptx::bulk_commit_group();
                }
#pragma unroll
                for (int c = 1; c <= kHeld; ++c) {
                    const uint32_t col = col0 + uint32_t(64 * c);
                    if (col < p.n) {
                        if (lane == 0) ptx::bulk_wait_group_read<0>();
                        __syncwarp();
                        stage_row_sw128(row_addr, lane, held[c - 1]);
                        ptx::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            ptx::tma_store_2d(&p.tmap_c, buf, int32_t(col), int32_t(row0));
                            ptx::bulk_commit_group();
                        }
                    }
                }
                if constexpr (Cfg::kTail) {
                    const uint32_t col = col0 + uint32_t(64 * Cfg::kFullChunks);
                    if (col < p.n) {
                        if (lane == 0) ptx::bulk_wait_group_read<0>();
                        __syncwarp();
                        // box {32, 32}: 64-byte rows, 64-byte swizzle (chunk j of row r at j ^ ((r / 2) mod 4))
                        const uint32_t row32 = buf + lane * 64u;
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            ptx::st_shared_v4(row32 + ((uint32_t(j) ^ ((lane >> 1) & 3u)) << 4), tail[4 * j],
                                              tail[4 * j + 1], tail[4 * j + 2], tail[4 * j + 3]);
                        ptx::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            ptx::tma_store_2d(&p.tmap_c32, buf, int32_t(col), int32_t(row0));
                            ptx::bulk_commit_group();
                        }
                    }
                }
            }
            return true;
        }, last_tile, sk_segment);
        if (lane == 0) ptx::bulk_wait_group<0>();
    }

    // ---------------------------------------------------- teardown
    __syncwarp();
    ptx::tc_fence_before_sync();
    ptx::cluster_sync();
    ptx::tc_fence_after_sync();
    // Both CTAs stay until the second barrier, so the first CTA may read the second's flags: after an
    // abort in either, it waits for every ring load still in flight before either CTA exits.
    if (threadIdx.x == 0 && leader) wide_abort_drain<STAGES, HALF_N>(p);
    ptx::cluster_sync();
    if (warp == 1) ptx::tmem_dealloc<2>(tmem_base, Cfg::kTmemCols);
}

}  // namespace gemm_f16
