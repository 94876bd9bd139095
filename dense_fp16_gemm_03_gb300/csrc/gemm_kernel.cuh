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

// Device error word codes (low byte); bits 8.. hold the CTA index.
enum : uint32_t {
    kErrWaitEmpty = 1,
    kErrWaitFull = 2,
    kErrWaitAccEmpty = 3,
    kErrWaitAccFull = 4,
    kErrWaitDrain = 5,
};

struct KernelParams {
    CUtensorMap tmap_a;   // A [M, K]: box {64, 128}
    CUtensorMap tmap_b;   // B [N, K]: box {64, BN / CG}
    CUtensorMap tmap_c;   // C [M, N]: box {64, 32}
    Raster raster;
    uint32_t m, n, k;
    uint32_t num_tiles;
    uint32_t k_blocks;
    uint32_t skip_fill;   // test hook: k-block fill (counted across CTA 0's tiles) the producer
                          // of CTA 0 leaves undone, to exercise the bounded waits; ~0u = none
    long long wait_limit; // cycles a single barrier wait may take before it gives up
    uint32_t *error_word;
};

template <int CG, int BN, int STAGES>
struct KernelCfg {
    static_assert(CG == 1 || CG == 2, "cta group");
    static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "tile N");
    static constexpr int kBM = 128 * CG;            // MMA M
    static constexpr int kBNCta = BN / CG;          // B rows loaded per CTA
    static constexpr int kABytes = 128 * kBlockK * 2;
    static constexpr int kBBytes = kBNCta * kBlockK * 2;
    static constexpr int kStageTx = (kABytes + kBBytes) * CG;  // bytes landing on one full barrier
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + STAGES * kABytes;
    static constexpr int kOffStore = kOffB + STAGES * kBBytes;
    static constexpr int kNumBars = 2 * STAGES + 5;  // full, empty, acc_full x2, acc_empty x2, drain
    static constexpr int kOffBar = kOffStore + kEpiWarps * 2 * kStoreBufBytes;
    static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
    static constexpr int kOffAbort = kOffTmemSlot + 4;
    static constexpr int kSmemUsed = kOffAbort + 4;
    static constexpr int kSmemBytes = kSmemUsed + 1024;  // room to align the base to 1024
    static constexpr int kTmemCols = (2 * BN <= 128) ? 128 : (2 * BN <= 256 ? 256 : 512);
    static_assert(kBBytes % 1024 == 0 && kABytes % 1024 == 0, "swizzle atoms");
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

// tcgen05 instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B
// fp16 (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0), N >> 3 in
// bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N)
{
    return (1u << 4) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// Bounded wait on phase `parity` of the barrier at `bar`.
template <int CG>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const KernelParams &p,
                                             volatile uint32_t *abort_flag, uint32_t code)
{
    auto try_once = [&]() {
        if constexpr (CG == 2) return ptx::mbar_try_wait_cluster(bar, parity);
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

__device__ __forceinline__ uint32_t pack_half2(uint32_t lo_bits, uint32_t hi_bits)
{
    __half2 h = __floats2half2_rn(__uint_as_float(lo_bits), __uint_as_float(hi_bits));
    return *reinterpret_cast<uint32_t *>(&h);
}

template <int CG, int BN, int STAGES>
__global__ void __launch_bounds__(kNumThreads, 1) gemm_f16_nt_kernel(const __grid_constant__ KernelParams p)
{
    using Cfg = KernelCfg<CG, BN, STAGES>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);

    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t cta_rank = (CG == 2) ? ptx::cluster_ctarank() : 0u;
    const bool leader = (cta_rank == 0);
    const uint32_t cluster_id = blockIdx.x / CG;
    const uint32_t num_clusters = gridDim.x / CG;

    auto bar_full = [&](uint32_t s) { return base + Cfg::kOffBar + 8u * s; };
    auto bar_empty = [&](uint32_t s) { return base + Cfg::kOffBar + 8u * (STAGES + s); };
    auto bar_acc_full = [&](uint32_t b) { return base + Cfg::kOffBar + 8u * (2 * STAGES + b); };
    auto bar_acc_empty = [&](uint32_t b) { return base + Cfg::kOffBar + 8u * (2 * STAGES + 2 + b); };
    const uint32_t bar_drain = base + Cfg::kOffBar + 8u * (2 * STAGES + 4);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + Cfg::kOffAbort);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Cfg::kOffTmemSlot);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(bar_full(s), 1);
            ptx::mbar_init(bar_empty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar_acc_full(b), 1);
            ptx::mbar_init(bar_acc_empty(b), kEpiWarps * CG);
        }
        ptx::mbar_init(bar_drain, 1);
        *abort_flag = 0u;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&p.tmap_a);
        ptx::prefetch_tmap(&p.tmap_b);
        ptx::prefetch_tmap(&p.tmap_c);
    }
    if (warp == 1) {
        ptx::tmem_alloc<CG>(ptx::smem_addr(tmem_slot), Cfg::kTmemCols);
        ptx::tmem_relinquish<CG>();
    }
    ptx::tc_fence_before_sync();
    if constexpr (CG == 2) ptx::cluster_sync();
    else __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_a = ptx::policy_evict_normal();
            const uint64_t pol_b = ptx::policy_evict_normal();
            uint32_t stage = 0, phase = 0, fills = 0;
            bool ok = true;
            for (uint32_t tile = cluster_id; ok && tile < p.num_tiles; tile += num_clusters) {
                uint32_t mb, nb;
                raster_coord(p.raster, tile, mb, nb);
                const int32_t m0 = int32_t(mb * Cfg::kBM + cta_rank * 128u);
                const int32_t n0 = int32_t(nb * BN + cta_rank * Cfg::kBNCta);
                for (uint32_t kb = 0; kb < p.k_blocks; ++kb, ++fills) {
                    if (!wait_bounded<CG>(bar_empty(stage), phase ^ 1u, p, abort_flag, kErrWaitEmpty)) {
                        ok = false;
                        break;
                    }
                    const bool skip = (blockIdx.x == 0) && (fills == p.skip_fill);
                    if (!skip) {
                        const uint32_t fb = bar_full(stage);
                        const uint32_t a_dst = base + Cfg::kOffA + stage * Cfg::kABytes;
                        const uint32_t b_dst = base + Cfg::kOffB + stage * Cfg::kBBytes;
                        const int32_t k0 = int32_t(kb * kBlockK);
                        if constexpr (CG == 1) {
                            ptx::mbar_arrive_expect_tx(fb, Cfg::kStageTx);
                            ptx::tma_load_2d(a_dst, &p.tmap_a, fb, k0, m0, pol_a);
                            ptx::tma_load_2d(b_dst, &p.tmap_b, fb, k0, n0, pol_b);
                        } else {
                            const uint32_t fb_leader = ptx::map_to_rank(fb, 0);
                            if (leader) ptx::mbar_arrive_expect_tx(fb, Cfg::kStageTx);
                            ptx::tma_load_2d_pair(a_dst, &p.tmap_a, fb_leader, k0, m0, pol_a);
                            ptx::tma_load_2d_pair(b_dst, &p.tmap_b, fb_leader, k0, n0, pol_b);
                        }
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) __nanosleep(100000);  // let copies already issued land before teardown
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (leader && lane == 0) {
            constexpr uint32_t idesc = idesc_f16_f32(Cfg::kBM, BN);
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            for (uint32_t tile = cluster_id; ok && tile < p.num_tiles; tile += num_clusters) {
                if (!wait_bounded<CG>(bar_acc_empty(acc), acc_phase ^ 1u, p, abort_flag, kErrWaitAccEmpty)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (uint32_t kb = 0; kb < p.k_blocks; ++kb) {
                    if (!wait_bounded<CG>(bar_full(stage), phase, p, abort_flag, kErrWaitFull)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after_sync();
                    const uint64_t a_desc = smem_desc_sw128(base + Cfg::kOffA + stage * Cfg::kABytes);
                    const uint64_t b_desc = smem_desc_sw128(base + Cfg::kOffB + stage * Cfg::kBBytes);
#pragma unroll
                    for (int kk = 0; kk < kBlockK / 16; ++kk) {
                        // +32 bytes along K inside the swizzle atom per 16-element step
                        ptx::mma_f16<CG>(d_tmem, a_desc + uint64_t(2 * kk), b_desc + uint64_t(2 * kk), idesc,
                                         (kb | uint32_t(kk)) != 0u);
                    }
                    if constexpr (CG == 1) ptx::mma_commit(bar_empty(stage));
                    else ptx::mma_commit_pair(bar_empty(stage), uint16_t(0x3));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if constexpr (CG == 1) ptx::mma_commit(bar_acc_full(acc));
                else ptx::mma_commit_pair(bar_acc_full(acc), uint16_t(0x3));
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // No MMA may still be running when the tensor memory is freed.
            if constexpr (CG == 1) ptx::mma_commit(bar_drain);
            else ptx::mma_commit_pair(bar_drain, uint16_t(0x1));
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
        const uint32_t stage_base = base + Cfg::kOffStore + (warp - 2u) * 2u * kStoreBufBytes;
        const uint32_t lane_sel = (quarter * 32u) << 16;
        uint32_t acc = 0, acc_phase = 0, stores = 0;
        for (uint32_t tile = cluster_id; tile < p.num_tiles; tile += num_clusters) {
            uint32_t mb, nb;
            raster_coord(p.raster, tile, mb, nb);
            const uint32_t row0 = mb * Cfg::kBM + cta_rank * 128u + quarter * 32u;
            const uint32_t col0 = nb * BN;
            const bool ok = wait_bounded<CG>(bar_acc_full(acc), acc_phase, p, abort_flag, kErrWaitAccFull);
            if (!__all_sync(0xffffffffu, ok)) break;
            ptx::tc_fence_after_sync();
            if (row0 < p.m) {
#pragma unroll 1
                for (int c = 0; c < BN / kStoreCols; ++c) {
                    const uint32_t col = col0 + uint32_t(c * kStoreCols);
                    if (col >= p.n) break;
                    uint32_t r[64];
                    ptx::tmem_ld_32x32b_x64_wait(tmem_base + acc * BN + uint32_t(c * kStoreCols) + lane_sel, r);
                    const uint32_t buf = stage_base + (stores & 1u) * kStoreBufBytes;
                    if (lane == 0) ptx::bulk_wait_group_read<1>();  // this buffer's previous store has read it
                    __syncwarp();
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
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        ptx::tma_store_2d(&p.tmap_c, buf, int32_t(col), int32_t(row0));
                        ptx::bulk_commit_group();
                    }
                    ++stores;
                }
            }
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if constexpr (CG == 1) ptx::mbar_arrive(bar_acc_empty(acc));
                else ptx::mbar_arrive_cluster(ptx::map_to_rank(bar_acc_empty(acc), 0));
            }
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (lane == 0) ptx::bulk_wait_group<0>();
    }

    // ---------------------------------------------------- teardown
    __syncwarp();
    ptx::tc_fence_before_sync();
    if constexpr (CG == 2) ptx::cluster_sync();
    else __syncthreads();
    ptx::tc_fence_after_sync();
    if (warp == 1) ptx::tmem_dealloc<CG>(tmem_base, Cfg::kTmemCols);
}

}  // namespace gemm_f16
