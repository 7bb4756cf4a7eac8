// FP8 block-scaled GEMM kernel for sm_103a, CTA-pair version.
//
// Same result as fp8bs_blockscale_kernel (bs_kernel.cu):
//   C[m,n] = bf16( sum_kb P_kb[m,n] * a_scale[m,kb] * b_scale[n/128,kb] ),
// P_kb the unscaled fp8 product of 128-wide K block kb, promoted in fp32 after
// the matrix unit (skill card "FlyDSL fp8 blockscale GEMM", "Mechanism A").
//
// Two CTAs of a cluster (two SMs) share one 256 x 128 tile: each CTA owns 128
// rows of A and C and holds half (64 rows) of the B tile; the even CTA issues
// tcgen05.mma.cta_group::2 (M256 x N128 x K32), which reads A from each CTA's
// own shared memory, exchanges the B halves, and writes each CTA's 128 x 128
// partial into that CTA's tensor memory. A stage is then 16 KiB (A) + 8 KiB
// (B) per CTA, and one 128-column partial buffer leaves room for four in TMEM,
// so the MMA can run three K blocks ahead of the fp32 promote.
//
// Per CTA, 12 warps (3 warpgroups):
//   warp 0      TMA producer: own A rows and own B half of a K block into stage
//               s. Both CTAs' bytes complete on the even CTA's full[s] barrier,
//               which the even CTA's producer alone arms with the pair's total
//               (the odd CTA's copies may land first: the barrier cannot complete
//               before that arrive). The a_scale slice [128] goes to a local ring.
//   warp 1      TMEM allocation for the pair (both CTAs) and, in the even CTA
//               only, the single-thread MMA issuer; tcgen05.commit multicasts the
//               stage release and "partial ready" to both CTAs.
//   warps 2,3   idle (complete warpgroup 0, which gives its registers away).
//   warps 4..11 promote + epilogue for this CTA's 128 rows: thread = one row,
//               64 columns; releases a partial buffer on the even CTA's
//               tempty barrier (16 arrivals: 8 warps from each CTA; the odd
//               CTA's are relaxed remote arrives, see mbar_arrive_cluster_relaxed).
#include "common.cuh"

namespace fp8bs {

constexpr int kPairThreads = (4 + kEpiWarps) * 32;
constexpr int kPairBN = 128;            // N of the pair tile (= of each CTA's partial)
constexpr int kPairNBuf = 4;            // TMEM partial buffers per CTA
constexpr int kPairSaSlots = 16;
// Registers: 168 per thread at launch (3 warps per SM sub-partition); warpgroup
// 0 drops to 80, the promote warpgroups rise to 208: 80 + 208 + 208 = 496 <= 512.
constexpr int kPairRegsLow = 80;
constexpr int kPairRegsHigh = 208;

template <int STAGES>
struct PairLayout {
    static constexpr int A_BYTES = kBlockM * kBlockK;             // own 128 rows
    static constexpr int B_BYTES = (kPairBN / 2) * kBlockK;       // own 64 rows of B
    static constexpr int SA_BYTES = kBlockM * 4;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_SA = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_C = (OFF_SA + kPairSaSlots * SA_BYTES + 1023) / 1024 * 1024;
    static constexpr int OFF_BAR = OFF_C + kEpiWarps * kCStageBytes;
    // full[S], empty[S], tfull[NBUF], tempty[NBUF], mma_done, sa_full[SA], sa_empty[SA]
    static constexpr int NBAR = 2 * STAGES + 2 * kPairNBuf + 1 + 2 * kPairSaSlots;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int BYTES = OFF_MISC + 16;
    static constexpr int DYN_SMEM = BYTES + 1024;
    static constexpr int TMEM_COLS = kPairNBuf * kPairBN;
    static_assert(TMEM_COLS == 512, "tensor memory");
    static_assert(DYN_SMEM <= 232448, "shared memory budget");
};

template <int STAGES>
__global__ void __launch_bounds__(kPairThreads, 1)
    fp8bs_blockscale_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                                 const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmC,
                                 const GemmArgs args)
{
    using L = PairLayout<STAGES>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = ptx::smem_u32(smem_raw);
    const uint32_t sbase = (raw_s + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw_s);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();   // 0 = even CTA (issues the MMAs)
    const int cluster = static_cast<int>(blockIdx.x) >> 1;
    const int num_clusters = static_cast<int>(gridDim.x) >> 1;
    const int KB = args.K / kBlockK;
    const int num_tiles = args.raster.num_tiles();   // pair tiles (256 x 128)

    auto full_bar = [&](int s) { return sbase + L::OFF_BAR + 8u * s; };
    auto empty_bar = [&](int s) { return sbase + L::OFF_BAR + 8u * (STAGES + s); };
    auto tfull_bar = [&](int b) { return sbase + L::OFF_BAR + 8u * (2 * STAGES + b); };
    auto tempty_bar = [&](int b) { return sbase + L::OFF_BAR + 8u * (2 * STAGES + kPairNBuf + b); };
    const uint32_t mma_done_bar = sbase + L::OFF_BAR + 8u * (2 * STAGES + 2 * kPairNBuf);
    auto sa_full_bar = [&](int a) { return sbase + L::OFF_BAR + 8u * (2 * STAGES + 2 * kPairNBuf + 1 + a); };
    auto sa_empty_bar = [&](int a) {
        return sbase + L::OFF_BAR + 8u * (2 * STAGES + 2 * kPairNBuf + 1 + kPairSaSlots + a);
    };
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full_bar(s), 1);                 // even CTA's producer (expect_tx of both CTAs' bytes)
            ptx::mbar_init(empty_bar(s), 1);                // multicast MMA commit
        }
        for (int b = 0; b < kPairNBuf; ++b) {
            ptx::mbar_init(tfull_bar(b), 1);                // multicast MMA commit
            ptx::mbar_init(tempty_bar(b), 2 * kEpiWarps);   // promote warps of both CTAs (even CTA's copy)
        }
        ptx::mbar_init(mma_done_bar, 1);
        for (int a = 0; a < kPairSaSlots; ++a) {
            ptx::mbar_init(sa_full_bar(a), 1);
            ptx::mbar_init(sa_empty_bar(a), kEpiWarps);
        }
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

    if (warp < 4) {
        ptx::setmaxnreg_dec<kPairRegsLow>();
        if (warp == 0 && lane == 0) {
            // ------------------------------------------------------------ producer
            ptx::prefetch_tmap(&tmA);
            ptx::prefetch_tmap(&tmB);
            ptx::prefetch_tmap(&tmSA);
            int it = 0;
            bool ok = true;
            for (int t = cluster; t < num_tiles && ok; t += num_clusters) {
                int mb, nb;
                args.raster.coords(t, mb, nb);
                const int row0 = mb * 2 * kBlockM + static_cast<int>(rank) * kBlockM;
                const int brow0 = nb * kPairBN + static_cast<int>(rank) * (kPairBN / 2);
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1;
                    const int a = it % kPairSaSlots;
                    const uint32_t aph = (it / kPairSaSlots) & 1;
                    if (!wait_bounded(empty_bar(s), ph ^ 1, abort_flag, args) ||
                        !wait_bounded(sa_empty_bar(a), aph ^ 1, abort_flag, args)) {
                        ok = false;
                        break;
                    }
                    const uint32_t leader_full = ptx::mapa_shared(full_bar(s), 0);
                    if (rank == 0)
                        ptx::mbar_arrive_expect_tx(full_bar(s), 2 * (L::A_BYTES + L::B_BYTES));
                    ptx::tma_load_2d_pair(sbase + L::OFF_A + s * L::A_BYTES, &tmA, leader_full, kb * kBlockK, row0);
                    ptx::tma_load_2d_pair(sbase + L::OFF_B + s * L::B_BYTES, &tmB, leader_full, kb * kBlockK, brow0);
                    ptx::mbar_arrive_expect_tx(sa_full_bar(a), L::SA_BYTES);
                    ptx::tma_load_2d(sbase + L::OFF_SA + a * L::SA_BYTES, &tmSA, sa_full_bar(a), row0, kb);
                }
            }
            // every load issued must have landed before the CTA exits
            for (int a = 0; a < kPairSaSlots; ++a) {
                const int uses = it > a ? (it - a + kPairSaSlots - 1) / kPairSaSlots : 0;
                if (uses > 0)
                    wait_teardown(sa_full_bar(a), (uses - 1) & 1, args);
            }
            if (rank == 0) {
                for (int s = 0; s < STAGES; ++s) {
                    const int uses = it > s ? (it - s + STAGES - 1) / STAGES : 0;
                    if (uses > 0)
                        wait_teardown(full_bar(s), (uses - 1) & 1, args);
                }
            } else {
                // the even CTA's MMA consumed (or abandoned) every stage; its
                // multicast releases say this CTA's loads have landed
                for (int s = 0; s < STAGES; ++s) {
                    const int uses = it > s ? (it - s + STAGES - 1) / STAGES : 0;
                    if (uses > 0)
                        wait_teardown(empty_bar(s), (uses - 1) & 1, args);
                }
            }
        } else if (warp == 1 && lane == 0) {
            if (rank == 0) {
                // --------------------------------------------------- MMA issuer
                constexpr uint32_t idesc = ptx::idesc_f8f6f4_e4m3(2 * kBlockM, kPairBN);
                int it = 0;
                bool ok = true;
                for (int t = cluster; t < num_tiles && ok; t += num_clusters) {
                    for (int kb = 0; kb < KB; ++kb, ++it) {
                        const int s = it % STAGES;
                        const uint32_t ph = (it / STAGES) & 1;
                        const int buf = it % kPairNBuf;
                        const uint32_t tph = (it / kPairNBuf) & 1;
                        if (!wait_bounded(tempty_bar(buf), tph ^ 1, abort_flag, args) ||
                            !wait_bounded(full_bar(s), ph, abort_flag, args)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        const uint64_t adesc = ptx::desc_kmajor_sw128(sbase + L::OFF_A + s * L::A_BYTES);
                        const uint64_t bdesc = ptx::desc_kmajor_sw128(sbase + L::OFF_B + s * L::B_BYTES);
                        const uint32_t d = tmem_base + static_cast<uint32_t>(buf * kPairBN);
#pragma unroll
                        for (int kk = 0; kk < kBlockK / kMmaK; ++kk)
                            ptx::mma_f8f6f4_pair(d, adesc + 2 * kk, bdesc + 2 * kk, idesc, kk > 0 ? 1u : 0u);
                        ptx::tc_commit_pair_mc(empty_bar(s), 0x3);
                        ptx::tc_commit_pair_mc(tfull_bar(buf), 0x3);
                    }
                }
                ptx::tc_commit_pair_mc(mma_done_bar, 0x3);
            }
        }
    } else {
        ptx::setmaxnreg_inc<kPairRegsHigh>();
        // ------------------------------------------------- promote + epilogue
        constexpr int HALF = kPairBN / 2;            // columns per thread
        const int ew = warp - 4;
        const int wg = ew >> 2;                      // column half
        const int q = warp & 3;                      // TMEM lane quadrant
        const int row = q * 32 + lane;
        const int NB = (args.N + 127) / 128;
        const uint32_t cstage = sbase + L::OFF_C + ew * kCStageBytes;
        const int my_tiles = cluster < num_tiles ? (num_tiles - cluster + num_clusters - 1) / num_clusters : 0;
        const int total = my_tiles * KB;

        auto sb_lane_load = [&](int g) -> float {
            if (g >= total)
                return 0.f;
            const int ti = g / KB;
            const int kb = g - ti * KB;
            int mb, nb;
            args.raster.coords(cluster + ti * num_clusters, mb, nb);
            const int nblk = (nb * kPairBN) >> 7;
            if (nblk >= NB)
                return 0.f;
            return ptx::ldg_nc_f32(args.b_scale + static_cast<size_t>(nblk) * KB + kb);
        };
        float sb_cur = sb_lane_load(lane);
        float sb_next = sb_lane_load(32 + lane);

        float acc[HALF];
        int it = 0;
        bool ok = true;
        for (int t = cluster; t < num_tiles; t += num_clusters) {
            int mb, nb;
            args.raster.coords(t, mb, nb);
#pragma unroll
            for (int j = 0; j < HALF; ++j)
                acc[j] = 0.f;
            for (int kb = 0; kb < KB; ++kb, ++it) {
                const float sb = __shfl_sync(0xffffffffu, sb_cur, it & 31);
                if ((it & 31) == 31) {
                    sb_cur = sb_next;
                    sb_next = sb_lane_load(it + 33 + lane);
                }
                const int a = it % kPairSaSlots;
                const uint32_t aph = (it / kPairSaSlots) & 1;
                const int buf = it % kPairNBuf;
                const uint32_t tph = (it / kPairNBuf) & 1;
                if (!wait_bounded_warp(tfull_bar(buf), tph, abort_flag, args) ||
                    !wait_bounded_warp(sa_full_bar(a), aph, abort_flag, args)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const float sa = reinterpret_cast<const float *>(smem + L::OFF_SA + a * L::SA_BYTES)[row];
                const float scale = sa * sb;
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                       static_cast<uint32_t>(buf * kPairBN + wg * HALF);
                // load the whole 64-column slice, release the buffer, then promote
                uint32_t r0[32], r1[32];
                ptx::tmem_ld_32x32b_x32(taddr, r0);
                ptx::tmem_ld_32x32b_x32(taddr + 32, r1);
                ptx::tmem_wait_ld();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (rank == 0)
                        ptx::mbar_arrive(tempty_bar(buf));
                    else
                        ptx::mbar_arrive_cluster_relaxed(ptx::mapa_shared(tempty_bar(buf), 0));
                    ptx::mbar_arrive(sa_empty_bar(a));
                }
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    acc[j] = fmaf(__uint_as_float(r0[j]), scale, acc[j]);
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    acc[32 + j] = fmaf(__uint_as_float(r1[j]), scale, acc[32 + j]);
            }
            if (!ok)
                break;
            const int x0 = nb * kPairBN + wg * HALF;
            const int y0 = mb * 2 * kBlockM + static_cast<int>(rank) * kBlockM + q * 32;
#pragma unroll
            for (int c = 0; c < HALF / kCChunkCols; ++c)
                store_c_chunk(&tmC, cstage, lane, acc + c * kCChunkCols, x0 + c * kCChunkCols, y0, args.M,
                              args.N);
        }
        if (lane == 0)
            ptx::bulk_wait_all();
    }

    ptx::tc_fence_before();
    __syncthreads();
    // No pair MMA may still write this CTA's tensor memory when it is freed (the
    // promote warps have consumed every partial by now, so this wait is short).
    if (warp == 1 && lane == 0)
        wait_teardown(mma_done_bar, 0, args);
    ptx::cluster_sync();   // no remote arrive or multicast commit may target an exited CTA
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, L::TMEM_COLS);
    }
}

template <int STAGES>
cudaError_t launch_blockscale_pair(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmSA,
                                   const CUtensorMap &tmC, const GemmArgs &args, int max_clusters, cudaStream_t stream)
{
    using L = PairLayout<STAGES>;
    auto kern = fp8bs_blockscale_pair_kernel<STAGES>;
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
    cfg.blockDim = dim3(kPairThreads);
    cfg.dynamicSmemBytes = L::DYN_SMEM;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmSA, tmC, args);
}

// Co-resident clusters of two CTAs for this kernel on the current device.
template <int STAGES>
cudaError_t max_pair_clusters(int *out)
{
    using L = PairLayout<STAGES>;
    auto kern = fp8bs_blockscale_pair_kernel<STAGES>;
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
    cfg.blockDim = dim3(kPairThreads);
    cfg.dynamicSmemBytes = L::DYN_SMEM;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(out, kern, &cfg);
}

template cudaError_t launch_blockscale_pair<8>(const CUtensorMap &, const CUtensorMap &, const CUtensorMap &,
                                               const CUtensorMap &, const GemmArgs &, int, cudaStream_t);
template cudaError_t max_pair_clusters<8>(int *);

} // namespace fp8bs
