// MXFP8 GEMM kernel for sm_103a, CTA-pair version.
//
// Same result as fp8bs_mxfp8_kernel (mx_kernel.cu). Two CTAs of a cluster share
// one 256 x 256 tile: each CTA owns 128 rows of A and C and holds 128 of the
// 256 rows of the B tile; the even CTA issues
// tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale (M256 x N256 x K32),
// which reads A from each CTA's own shared memory, exchanges the B halves and
// writes each CTA's 128 x 256 accumulator into that CTA's tensor memory.
//
// Why: the one-CTA kernel is bound by its stage count. A stage is refilled only
// after its MMAs complete and its data lands ~2000 clocks later, so with four
// 49.5 KiB stages a 128-K step takes ~(512 + 300 + 2000) / 4 clocks. Here a
// CTA's stage is 16 KiB (A) + 16 KiB (B half) + 1.5 KiB (scale atoms), so six
// fit, which is enough for the tensor pipe to stay busy.
//
// Scale factors: each CTA stages the atom of its own 128 A rows and the atoms
// of both 128-row B blocks of the tile in its shared memory (loaded by tensor
// copies that complete on the even CTA's barrier); the even CTA's issuer copies
// them into tensor memory with tcgen05.cp.cta_group::2, which moves each CTA's
// shared-memory atoms into that CTA's own tensor memory at the same address.
//
// Per CTA, 11 warps:
//   warp 0      TMA producer: own A rows, own B half, scale atoms of a K step
//               into stage s; the pair's bytes complete on the even CTA's
//               full[s], which the even CTA's producer alone arms.
//   warp 1      pair TMEM allocation and, in the even CTA only, the
//               single-thread MMA issuer; tcgen05.commit multicasts the stage
//               release and "accumulator ready" to both CTAs.
//   warps 2..9  epilogue for this CTA's 128 rows (128 columns per thread),
//               releasing the accumulator on the even CTA's acc_empty barrier
//               (16 arrivals: 8 warps from each CTA).
//   warp 10     in the even CTA, the scale-factor copier: for each K step it
//               waits for the stage, copies its three atoms into that stage's
//               tensor-memory columns and signals sf_full[s]. The copies run
//               ahead of the MMAs (up to the ring depth), so the issuer's
//               thread spends its issue slots on the four MMAs of a step only:
//               issuing three copies and four MMAs from one thread cost ~950
//               clocks per step in a ring probe, against ~665 for the MMAs alone.
#include "common.cuh"

namespace fp8bs {

constexpr int kMx2Threads = (3 + kEpiWarps) * 32;
constexpr int kMx2CopierWarp = 2 + kEpiWarps;   // warp 10
constexpr int kMx2BN = 256;   // N of the pair tile (each CTA holds half of its B rows)

template <int STAGES>
struct Mx2Layout {
    static constexpr int A_BYTES = kBlockM * kBlockK;              // own 128 rows
    static constexpr int B_BYTES = (kMx2BN / 2) * kBlockK;         // own 128 B rows
    static constexpr int SFA_BYTES = 512;                          // own rows' atom
    static constexpr int SFB_BYTES = 512 * (kMx2BN / 128);         // both B blocks' atoms
    static constexpr int SF_BYTES = SFA_BYTES + SFB_BYTES;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SF_BYTES;   // one CTA's share of a stage
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_SF = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_C = (OFF_SF + STAGES * SF_BYTES + 1023) / 1024 * 1024;
    static constexpr int OFF_BAR = OFF_C + kEpiWarps * kCStageBytes;
    static constexpr int NBAR = 3 * STAGES + 4;     // full[S], empty[S], sf_full[S], acc_full, acc_empty, mma_done, sf_done
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int BYTES = OFF_MISC + 16;
    static constexpr int DYN_SMEM = BYTES + 1024;
    // TMEM: accumulator columns [0, 256), then 16 scale-factor columns per stage
    // (A atom: 4 columns, B atoms: 4 columns per 128 rows).
    static constexpr int SF_COL0 = kMx2BN;
    static constexpr int SF_COLS_PER_STAGE = 16;
    static constexpr int TMEM_COLS = 512;
    static_assert(SF_COL0 + STAGES * SF_COLS_PER_STAGE <= TMEM_COLS, "tensor memory budget");
    static_assert(DYN_SMEM <= 232448, "shared memory budget");
};

// Copy of a scale-factor atom for the pair: each CTA's shared memory at `sdesc`
// into that CTA's tensor memory at `taddr`.
__device__ __forceinline__ void tc_cp_32x128b_warpx4_pair(uint32_t taddr, uint64_t sdesc)
{
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Pair block-scaled MMA (M = 256 over the two CTAs), issued by one thread of the
// even CTA; scale factors at the same tensor-memory addresses in both CTAs.
__device__ __forceinline__ void mma_mxf8f6f4_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                 uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "setp.ne.b32 p, %6, 0;\n"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

template <int STAGES>
__global__ void __launch_bounds__(kMx2Threads, 1)
    fp8bs_mxfp8_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
                            const __grid_constant__ CUtensorMap tmC, const GemmArgs args)
{
    using L = Mx2Layout<STAGES>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = ptx::smem_u32(smem_raw);
    const uint32_t sbase = (raw_s + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw_s);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();   // 0 = even CTA (issues the MMAs)
    const int cluster = static_cast<int>(blockIdx.x) >> 1;
    const int num_clusters = static_cast<int>(gridDim.x) >> 1;
    const int KS = args.K / kBlockK;
    const int num_tiles = args.raster.num_tiles();   // pair tiles (256 x 256)

    auto full_bar = [&](int s) { return sbase + L::OFF_BAR + 8u * s; };
    auto empty_bar = [&](int s) { return sbase + L::OFF_BAR + 8u * (STAGES + s); };
    auto sf_full_bar = [&](int s) { return sbase + L::OFF_BAR + 8u * (2 * STAGES + s); };
    const uint32_t acc_full_bar = sbase + L::OFF_BAR + 8u * (3 * STAGES);
    const uint32_t acc_empty_bar = sbase + L::OFF_BAR + 8u * (3 * STAGES + 1);
    const uint32_t mma_done_bar = sbase + L::OFF_BAR + 8u * (3 * STAGES + 2);
    const uint32_t sf_done_bar = sbase + L::OFF_BAR + 8u * (3 * STAGES + 3);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full_bar(s), 1);     // even CTA's producer (expect_tx of both CTAs' bytes)
            ptx::mbar_init(empty_bar(s), 1);    // multicast MMA commit
            ptx::mbar_init(sf_full_bar(s), 1);  // the copier's commit (even CTA)
        }
        ptx::mbar_init(sf_done_bar, 1);
        ptx::mbar_init(acc_full_bar, 1);                  // multicast MMA commit
        ptx::mbar_init(acc_empty_bar, 2 * kEpiWarps);     // epilogue warps of both CTAs (even CTA's copy)
        ptx::mbar_init(mma_done_bar, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc_pair(ptx::smem_u32(tmem_holder), L::TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    ptx::cluster_sync();   // barriers of both CTAs initialised before any remote arrive
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            ptx::prefetch_tmap(&tmA);
            ptx::prefetch_tmap(&tmB);
            ptx::prefetch_tmap(&tmSFA);
            ptx::prefetch_tmap(&tmSFB);
            const int n_blocks = (args.N + 127) / 128;   // 128-row B blocks with a packed atom per K step
            int it = 0;
            bool ok = true;
            for (int t = cluster; t < num_tiles && ok; t += num_clusters) {
                int mb, nb;
                args.raster.coords(t, mb, nb);
                const int row0 = mb * 2 * kBlockM + static_cast<int>(rank) * kBlockM;
                const int brow0 = nb * kMx2BN + static_cast<int>(rank) * (kMx2BN / 2);
                for (int ks = 0; ks < KS; ++ks, ++it) {
                    const int s = it % STAGES;
                    if (!wait_bounded(empty_bar(s), ((it / STAGES) & 1) ^ 1, abort_flag, args)) {
                        ok = false;
                        break;
                    }
                    const uint32_t leader_full = ptx::mapa_shared(full_bar(s), 0);
                    if (rank == 0)
                        ptx::mbar_arrive_expect_tx(full_bar(s), 2 * L::STAGE_BYTES);
                    ptx::tma_load_2d_pair(sbase + L::OFF_A + s * L::A_BYTES, &tmA, leader_full, ks * kBlockK, row0);
                    ptx::tma_load_2d_pair(sbase + L::OFF_B + s * L::B_BYTES, &tmB, leader_full, ks * kBlockK, brow0);
                    // scale atoms: 4 rows of 128 bytes each in the atom tensors
                    const uint32_t sf_smem = sbase + L::OFF_SF + s * L::SF_BYTES;
                    ptx::tma_load_2d_pair(sf_smem, &tmSFA, leader_full, 0, ((row0 / 128) * KS + ks) * 4);
#pragma unroll
                    for (int h = 0; h < kMx2BN / 128; ++h) {
                        const int bblk = nb * (kMx2BN / 128) + h < n_blocks ? nb * (kMx2BN / 128) + h : n_blocks - 1;
                        ptx::tma_load_2d_pair(sf_smem + L::SFA_BYTES + 512 * h, &tmSFB, leader_full, 0,
                                              (bblk * KS + ks) * 4);
                    }
                }
            }
            if (rank == 0) {
                for (int s = 0; s < STAGES; ++s) {
                    const int uses = it > s ? (it - s + STAGES - 1) / STAGES : 0;
                    if (uses > 0)
                        wait_teardown(full_bar(s), (uses - 1) & 1, args);
                }
            } else {
                // the even CTA's MMAs consumed (or abandoned) every stage; its
                // multicast releases say this CTA's loads have landed
                for (int s = 0; s < STAGES; ++s) {
                    const int uses = it > s ? (it - s + STAGES - 1) / STAGES : 0;
                    if (uses > 0)
                        wait_teardown(empty_bar(s), (uses - 1) & 1, args);
                }
            }
        }
    } else if (warp == 1) {
        // --------------------------------------------------- MMA issuer (even CTA)
        if (lane == 0 && rank == 0) {
            int it = 0, titer = 0;
            bool ok = true;
            for (int t = cluster; t < num_tiles && ok; t += num_clusters, ++titer) {
                if (!wait_bounded(acc_empty_bar, (titer & 1) ^ 1, abort_flag, args))
                    break;
                ptx::tc_fence_after();
                for (int ks = 0; ks < KS; ++ks, ++it) {
                    const int s = it % STAGES;
                    if (!wait_bounded(full_bar(s), (it / STAGES) & 1, abort_flag, args)) {
                        ok = false;
                        break;
                    }
                    // the copier's atoms for this step are in tensor memory (which
                    // also means the stage's data has landed)
                    if (!wait_bounded(sf_full_bar(s), (it / STAGES) & 1, abort_flag, args)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sfa_t = tmem_base + static_cast<uint32_t>(L::SF_COL0 + s * L::SF_COLS_PER_STAGE);
                    const uint32_t sfb_t = sfa_t + 4;
                    const uint64_t adesc = ptx::desc_kmajor_sw128(sbase + L::OFF_A + s * L::A_BYTES);
                    const uint64_t bdesc = ptx::desc_kmajor_sw128(sbase + L::OFF_B + s * L::B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < kBlockK / kMmaK; ++kk)
                        mma_mxf8f6f4_pair(tmem_base, adesc + 2 * kk, bdesc + 2 * kk,
                                          ptx::idesc_mxf8f6f4_e4m3(2 * kBlockM, kMx2BN, kk, kk), sfa_t, sfb_t,
                                          (ks | kk) != 0 ? 1u : 0u);
                    ptx::tc_commit_pair_mc(empty_bar(s), 0x3);
                }
                if (!ok)
                    break;
                ptx::tc_commit_pair_mc(acc_full_bar, 0x3);
            }
            ptx::tc_commit_pair_mc(mma_done_bar, 0x3);
        }
    } else if (warp == kMx2CopierWarp) {
        // ---------------------------------------- scale-factor copier (even CTA)
        // Stage s's tensor-memory columns are free when its data lands: the
        // producer refilled s only after the MMAs that read them committed.
        if (lane == 0 && rank == 0) {
            int it = 0;
            bool ok = true;
            for (int t = cluster; t < num_tiles && ok; t += num_clusters) {
                for (int ks = 0; ks < KS; ++ks, ++it) {
                    const int s = it % STAGES;
                    if (!wait_bounded(full_bar(s), (it / STAGES) & 1, abort_flag, args)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sf_smem = sbase + L::OFF_SF + s * L::SF_BYTES;
                    const uint32_t sfa_t = tmem_base + static_cast<uint32_t>(L::SF_COL0 + s * L::SF_COLS_PER_STAGE);
                    tc_cp_32x128b_warpx4_pair(sfa_t, ptx::desc_noswizzle(sf_smem, 16, 128));
#pragma unroll
                    for (int h = 0; h < kMx2BN / 128; ++h)
                        tc_cp_32x128b_warpx4_pair(sfa_t + 4 + 4 * h,
                                                  ptx::desc_noswizzle(sf_smem + L::SFA_BYTES + 512 * h, 16, 128));
                    ptx::tc_commit_pair_mc(sf_full_bar(s), 0x1);
                }
            }
            // every copy into either CTA's tensor memory has completed before
            // this CTA joins the final cluster barrier
            ptx::tc_commit_pair_mc(sf_done_bar, 0x1);
            wait_teardown(sf_done_bar, 0, args);
        }
    } else {
        // ------------------------------------------------------ epilogue
        constexpr int HALF = kMx2BN / 2;
        const int ew = warp - 2;                // 0..7
        const int wg = ew >> 2;
        const int q = warp & 3;
        const uint32_t cstage = sbase + L::OFF_C + ew * kCStageBytes;
        const uint32_t leader_acc_empty = ptx::mapa_shared(acc_empty_bar, 0);
        int titer = 0;
        for (int t = cluster; t < num_tiles; t += num_clusters, ++titer) {
            int mb, nb;
            args.raster.coords(t, mb, nb);
            if (!wait_bounded_warp(acc_full_bar, titer & 1, abort_flag, args))
                break;
            ptx::tc_fence_after();
            float v[HALF];
            const uint32_t taddr =
                tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(wg * HALF);
#pragma unroll
            for (int c = 0; c < HALF / 32; ++c) {
                uint32_t r[32];
                ptx::tmem_ld_32x32b_x32(taddr + c * 32, r);
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    v[c * 32 + j] = __uint_as_float(r[j]);
            }
            ptx::tmem_wait_ld();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (rank == 0)
                    ptx::mbar_arrive(acc_empty_bar);
                else
                    ptx::mbar_arrive_cluster_relaxed(leader_acc_empty);
            }
            const int x0 = nb * kMx2BN + wg * HALF;
            const int y0 = mb * 2 * kBlockM + static_cast<int>(rank) * kBlockM + q * 32;
#pragma unroll
            for (int c = 0; c < HALF / kCChunkCols; ++c)
                store_c_chunk(&tmC, cstage, lane, v + c * kCChunkCols, x0 + c * kCChunkCols, y0, args.M, args.N);
        }
        if (lane == 0)
            ptx::bulk_wait_all();
    }

    ptx::tc_fence_before();
    __syncthreads();
    // No pair MMA may still write this CTA's tensor memory when it is freed.
    if (warp == 1 && lane == 0)
        wait_teardown(mma_done_bar, 0, args);
    ptx::cluster_sync();   // no remote arrive or multicast commit may target an exited CTA
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, L::TMEM_COLS);
    }
}

template <int STAGES>
cudaError_t launch_mxfp8_pair(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmSFA,
                              const CUtensorMap &tmSFB, const CUtensorMap &tmC, const GemmArgs &args,
                              int max_clusters, cudaStream_t stream)
{
    using L = Mx2Layout<STAGES>;
    auto kern = fp8bs_mxfp8_pair_kernel<STAGES>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::DYN_SMEM);
    if (e != cudaSuccess)
        return e;
    const int tiles = args.raster.num_tiles();
    const int clusters = tiles < max_clusters ? tiles : max_clusters;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(kMx2Threads);
    cfg.dynamicSmemBytes = L::DYN_SMEM;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmSFA, tmSFB, tmC, args);
}

// Co-resident clusters of two CTAs for this kernel on the current device.
template <int STAGES>
cudaError_t max_mx_pair_clusters(int *out)
{
    using L = Mx2Layout<STAGES>;
    auto kern = fp8bs_mxfp8_pair_kernel<STAGES>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::DYN_SMEM);
    if (e != cudaSuccess)
        return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(kMx2Threads);
    cfg.dynamicSmemBytes = L::DYN_SMEM;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(out, kern, &cfg);
}

template cudaError_t launch_mxfp8_pair<6>(const CUtensorMap &, const CUtensorMap &, const CUtensorMap &,
                                          const CUtensorMap &, const CUtensorMap &, const GemmArgs &, int,
                                          cudaStream_t);
template cudaError_t max_mx_pair_clusters<6>(int *);

} // namespace fp8bs
