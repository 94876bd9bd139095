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
// the bounded waits are those of gemm_kernel.cuh; this variant has neither a
// stream-K tail nor split-K (its plans are always data-parallel).
#pragma once

#include "gemm_kernel.cuh"

namespace gemm_f16 {

constexpr int kWideEpiWarps = 8;
constexpr int kWideThreads = 64 + 32 * kWideEpiWarps;

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
    static constexpr int kNumBars = 2 * STAGES + 3;  // full, empty, acc_full, acc_empty, drain
    static constexpr int kOffBar = kOffStore + kWideEpiWarps * kStoreBufBytes;
    static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
    static constexpr int kOffAbort = kOffTmemSlot + 4;
    static constexpr int kOffFills = kOffAbort + 4;  // ring fills the producer walked (read by the abort drain)
    static constexpr int kSmemUsed = kOffFills + 4;
    static constexpr int kSmemBytes = kSmemUsed + 1024;  // room to align the base to 1024
    static constexpr int kTmemCols = 512;
    static_assert(kBSubBytes % 1024 == 0, "B sub-tiles stay 1024-byte aligned for the 128-byte swizzle");
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
    ptx::griddep_launch_dependents();
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
                const uint32_t rot = (p.k_rotate && whole) ? uint32_t((uint64_t(tile) * 37u) % p.k_blocks) : 0u;
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
        uint32_t acc_phase = 0;
        for_each_segment<false>(p, cluster_id, num_clusters, [&](uint32_t tile, uint32_t, uint32_t) {
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
        });
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
