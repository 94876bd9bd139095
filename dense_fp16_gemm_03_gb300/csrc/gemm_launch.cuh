// Launch side of the C ABI: the table of compiled kernel variants, the
// persistent cluster launch (programmatic dependent launch), and the TMA
// tensor maps each variant reads and writes.  Together with the kernels this
// fixes what a plan moves through memory; planning, validation and the
// host-buffer pipeline live in gemm_api.cu.  Included by gemm_api.cu only.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>
#include <string.h>

#include "gemm_f16.h"
#include "gemm_kernel.cuh"
#include "gemm_kernel_wide.cuh"

namespace gemm_f16 {

// ------------------------------------------------------------ variants

struct Variant {
    int cg, bn, stages, mc;
    int layout;  // 0: B [N,K], fp16 C; 1: B [K,N], fp32 D
    int swap;    // 1: computes C^T = B . A^T (operands swapped, tiles stored transposed)
    int smem;
    const void *fn;
    cudaError_t (*launch)(const gemm_f16_plan_t &, const KernelParams &, cudaStream_t);
    int threads;  // threads per CTA
    int b_box;    // B rows per TMA box (B [N,K] layout)
    int ks;       // > 1: the K blocks of each tile split across a cluster of ks single CTAs
};

// CTAs per cluster
int cluster_of(const Variant &var)
{
    return var.cg * var.mc * var.ks;
}

// Launch `kernel` persistently with clusters of `cs` CTAs, as a programmatic dependent launch.
cudaError_t launch_persistent(const void *kernel, const gemm_f16_plan_t &plan, const KernelParams &params,
                              cudaStream_t stream, int threads, int smem, int cs)
{
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(unsigned(plan.grid), 1, 1);
    cfg.blockDim = dim3(unsigned(threads), 1, 1);
    cfg.dynamicSmemBytes = size_t(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (cs > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = unsigned(cs);
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    // programmatic dependent launch: the kernel's set-up may overlap the previous kernel's tail;
    // it waits (griddepcontrol.wait) for that kernel before touching global memory
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    cfg.attrs = attr;
    cfg.numAttrs = na;
    void *args[1] = {const_cast<KernelParams *>(&params)};
    return cudaLaunchKernelExC(&cfg, kernel, args);
}

template <int CG, int BN, int ST, int MC, bool BK, bool CF, bool CT, int EP, int KS>
cudaError_t launch_variant(const gemm_f16_plan_t &plan, const KernelParams &params, cudaStream_t stream)
{
    return launch_persistent(reinterpret_cast<const void *>(&gemm_f16_nt_kernel<CG, BN, ST, MC, BK, CF, CT, EP, KS>),
                             plan, params, stream, kNumThreads,
                             KernelCfg<CG, BN, ST, MC, BK, CF, CT, EP, KS>::kSmemBytes, CG * MC * KS);
}

template <int ST, int HN>
cudaError_t launch_wide(const gemm_f16_plan_t &plan, const KernelParams &params, cudaStream_t stream)
{
    return launch_persistent(reinterpret_cast<const void *>(&gemm_f16_nt_wide_kernel<ST, HN>), plan, params, stream,
                             kWideThreads, WideCfg<ST, HN>::kSmemBytes, 2);
}

#define GEMM_VARIANT_K(CG, BN, ST, MC, BK, CF, CT, EP, KS)                                                    \
    Variant                                                                                                   \
    {                                                                                                         \
        CG, BN, ST, MC, (BK ? 0 : 1), (CT ? 1 : 0), KernelCfg<CG, BN, ST, MC, BK, CF, CT, EP, KS>::kSmemBytes, \
            reinterpret_cast<const void *>(&gemm_f16_nt_kernel<CG, BN, ST, MC, BK, CF, CT, EP, KS>),          \
            &launch_variant<CG, BN, ST, MC, BK, CF, CT, EP, KS>, kNumThreads,                                 \
            KernelCfg<CG, BN, ST, MC, BK, CF, CT, EP, KS>::kBSlice, KS                                        \
    }
#define GEMM_VARIANT_E(CG, BN, ST, MC, BK, CF, CT, EP) GEMM_VARIANT_K(CG, BN, ST, MC, BK, CF, CT, EP, 1)
#define GEMM_VARIANT_X(CG, BN, ST, MC, BK, CF, CT) GEMM_VARIANT_E(CG, BN, ST, MC, BK, CF, CT, 2)
#define GEMM_VARIANT_L(CG, BN, ST, MC, BK, CF) GEMM_VARIANT_X(CG, BN, ST, MC, BK, CF, false)
#define GEMM_VARIANT(CG, BN, ST, MC) GEMM_VARIANT_L(CG, BN, ST, MC, true, true)
#define GEMM_VARIANT_WIDE(ST, HN)                                                                              \
    Variant                                                                                                    \
    {                                                                                                          \
        2, WideCfg<ST, HN>::kBN, ST, 1, 0, 0, WideCfg<ST, HN>::kSmemBytes,                                     \
            reinterpret_cast<const void *>(&gemm_f16_nt_wide_kernel<ST, HN>), &launch_wide<ST, HN>,            \
            kWideThreads, WideCfg<ST, HN>::kBBoxRows, 1                                                        \
    }

const Variant kVariants[] = {
    GEMM_VARIANT(1, 256, 4, 1),  // 0: 128 x 256 tile, one CTA
    GEMM_VARIANT(1, 128, 6, 1),  // 1: 128 x 128 tile, one CTA
    GEMM_VARIANT(2, 256, 6, 1),  // 2: 256 x 256 tile on a CTA pair
    GEMM_VARIANT(2, 128, 8, 1),  // 3: 256 x 128 tile on a CTA pair
    GEMM_VARIANT(2, 256, 6, 2),  // 4: two pairs stacked along M share B by multicast (512 x 256 per cluster)
    GEMM_VARIANT(2, 224, 6, 2),  // 5: as 4 with 224-column tiles (512 x 224 per cluster)
    // B stored [K, N] (MN-major operand), fp32 result
    GEMM_VARIANT_L(1, 128, 6, 1, false, false),  // 6: 128 x 128 tile, one CTA
    GEMM_VARIANT_L(2, 256, 6, 1, false, false),  // 7: 256 x 256 tile on a CTA pair
    // shallow rings, for the pipeline-depth ablation only
    GEMM_VARIANT(1, 128, 1, 1),  // 8: single stage: load, then compute, then load
    GEMM_VARIANT(1, 128, 2, 1),  // 9: two stages
    GEMM_VARIANT(2, 256, 3, 1),  // 10: CTA pair, three stages
    GEMM_VARIANT(1, 128, 6, 2),  // 11: two CTAs along N share A by multicast (128 x 256 per cluster)
    GEMM_VARIANT(1, 128, 6, 4),  // 12: four CTAs along N share A by multicast (128 x 512 per cluster)
    // operands swapped (C^T = B . A^T, tiles stored transposed), for few rows of A
    GEMM_VARIANT_X(2, 128, 8, 1, true, true, true),  // 13: B rows on the pair's M = 256, A rows on N = 128
    GEMM_VARIANT_X(1, 128, 6, 1, true, true, true),  // 14: one CTA, 128 B rows x 128 A rows
    // wide tiles on a CTA pair, one accumulator filling tensor memory (no stream-K tail)
    GEMM_VARIANT_WIDE(4, 256),  // 15: 256 x 512
    GEMM_VARIANT_WIDE(4, 224),  // 16: 256 x 448 (fills the last wave where N / 512 would leave it idle)
    GEMM_VARIANT_WIDE(5, 160),  // 17: 256 x 320, five stages (4096^3: 208 tiles, 2.7 waves, where 512 columns
                                //     make 128 tiles, 1.7 waves)
    GEMM_VARIANT(1, 64, 8, 1),  // 18: 128 x 64 tile, one CTA (small, latency-bound products)
    // K split: each tile's K blocks shared by a cluster of single CTAs, partials traded through
    // distributed shared memory (products with fewer tiles than SMs)
    GEMM_VARIANT_K(1, 64, 4, 1, true, true, false, 2, 4),   // 19: 128 x 64 tile on four CTAs
    GEMM_VARIANT_K(1, 64, 6, 1, true, true, false, 2, 2),   // 20: 128 x 64 tile on two CTAs
    GEMM_VARIANT_K(1, 128, 4, 1, true, true, false, 2, 2),  // 21: 128 x 128 tile on two CTAs
    GEMM_VARIANT(1, 32, 8, 1),  // 22: 128 x 32 tile, one CTA (small products: 20 KB per K block into each SM)
};
constexpr int kNumVariants = int(sizeof(kVariants) / sizeof(kVariants[0]));

bool is_wide(const Variant &var)
{
    return var.threads == kWideThreads;
}

// Columns per MMA: a wide tile runs two MMAs side by side.
int mma_n(const Variant &var)
{
    return is_wide(var) ? var.bn / 2 : var.bn;
}

// ------------------------------------------------------- tensor maps

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

gemm_status_t get_encoder(PFN_cuTensorMapEncodeTiled_v12000 *fn)
{
    static std::once_flag once;
    std::call_once(once, []() {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        else
            cudaGetLastError();
    });
    *fn = g_encode;
    return g_encode ? GEMM_OK : GEMM_ERR_CUDA;
}

// Row-major fp16 (or, with elem_bytes 4, fp32) matrix of `rows` x `cols`
// (cols contiguous), boxes of box_cols x box_rows in shared memory laid out
// with `swizzle`, zero fill outside the matrix.
gemm_status_t encode_matrix(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap *map, const void *ptr,
                            uint64_t rows, uint64_t cols, uint32_t box_cols, uint32_t box_rows,
                            CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B, uint32_t elem_bytes = 2)
{
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * elem_bytes};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt = elem_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUresult r = enc(map, dt, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_INVALID_ARG;
}

// The tensor maps of one launch of `plan` (a, b, c as the caller passed them;
// a swapped variant computes the transposed product).
gemm_status_t encode_tensor_maps(const Variant &var, const gemm_f16_plan_t &plan, const void *a, const void *b,
                                 void *c, KernelParams *params)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    gemm_status_t st = get_encoder(&enc);
    if (st != GEMM_OK) return st;
    // kernel-side problem: the transposed one for a swapped variant
    const void *ka = var.swap ? b : a;
    const void *kb = var.swap ? a : b;
    params->c_out = c;
    const int64_t km = var.swap ? plan.n : plan.m;
    const int64_t kn = var.swap ? plan.m : plan.n;
    st = encode_matrix(enc, &params->tmap_a, ka, uint64_t(km), uint64_t(plan.k), kBlockK,
                       uint32_t((var.cg == 1 && var.mc > 1) ? 128 / var.mc : 128));
    if (st != GEMM_OK) return st;
    if (var.layout == 0) {
        st = encode_matrix(enc, &params->tmap_b, kb, uint64_t(kn), uint64_t(plan.k), kBlockK, uint32_t(var.b_box));
        if (st != GEMM_OK) return st;
        if (var.swap)  // C [m, n] written in transposed tiles: boxes of 32 columns x 64 rows, unswizzled
            st = encode_matrix(enc, &params->tmap_c, c, uint64_t(plan.m), uint64_t(plan.n), 32, 64,
                               CU_TENSOR_MAP_SWIZZLE_NONE);
        else
            st = encode_matrix(enc, &params->tmap_c, c, uint64_t(plan.m), uint64_t(plan.n), kStoreCols, kStoreRows);
    } else {
        // B [K, N]: 64-column boxes of 64 K rows; D [M, N] fp32: 32-column boxes
        st = encode_matrix(enc, &params->tmap_b, b, uint64_t(plan.k), uint64_t(plan.n), 64, kBlockK);
        if (st != GEMM_OK) return st;
        st = encode_matrix(enc, &params->tmap_c, c, uint64_t(plan.m), uint64_t(plan.n), 32, kStoreRows,
                           CU_TENSOR_MAP_SWIZZLE_128B, 4);
    }
    if (st != GEMM_OK) return st;
    if (mma_n(var) % 64 != 0 && var.layout == 0) {  // a last 32-column store box per tile (or tile half)
        st = encode_matrix(enc, &params->tmap_c32, c, uint64_t(plan.m), uint64_t(plan.n), 32, kStoreRows,
                           CU_TENSOR_MAP_SWIZZLE_64B);
        if (st != GEMM_OK) return st;
    }
    return GEMM_OK;
}

// The split-K reduction of a plan with split_k > 1, after its GEMM launch on the same stream.
cudaError_t launch_split_reduce(const gemm_f16_plan_t &plan, const Variant &var, const Raster &raster,
                                const void *parts, void *c, cudaStream_t stream)
{
    SplitReduceParams r;
    memset(&r, 0, sizeof(r));
    r.parts = static_cast<const float *>(parts);
    r.c = static_cast<__half *>(c);
    r.raster = raster;
    r.m = uint32_t(plan.m);
    r.n = uint32_t(plan.n);
    r.split_k = uint32_t(plan.split_k);
    r.bn = uint32_t(var.bn);
    r.cs = uint32_t(cluster_of(var));
    r.block_m = uint32_t(plan.block_m);
    r.block_n = uint32_t(plan.block_n);
    r.cta_rows = (var.cg == 1 && var.mc > 1) ? 0u : 128u;  // single CTAs sharing A sit along N
    r.threads = uint64_t(plan.num_tiles) * r.cs * 32u * r.bn;
    const uint64_t blocks = (r.threads + 255u) / 256u;  // within the grid limit (run_plan checks)
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(unsigned(blocks), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;  // overlaps the GEMM's tail
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, splitk_reduce_kernel, r);
}

}  // namespace gemm_f16
