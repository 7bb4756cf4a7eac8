// MXFP8 decode GEMM for sm_103a: few rows of A (M <= 128, one row of tiles).
//
// Computes C[m,n] = bf16( sum_k A[m,k] 2^(ea[m,k/32]-127) * B[n,k] 2^(eb[n,k/32]-127) ),
// as the MXFP8 kernel does, for the decode shapes that the PR "1x32 ue8m0
// (MXFP8) 8-wave FlyDSL GEMM for gfx950" (section "Not included") leaves to a
// separate GEMV-style op for M <= 32.
//
// With one row of tiles the work is streaming B once: there are only
// ceil(N/128) tiles, and the persistent kernel gives each tile to one SM that
// refills a six-stage ring again and again (16 K steps at K = 2048). Here a
// tile's K steps are cut into S slices, [s*KS/S, (s+1)*KS/S) for slice s, with
// S chosen so that a slice fits in shared memory whole (at most kMxdMaxSteps
// steps) and the grid fills the SMs. Every load of a CTA is issued at once, so
// its bytes are in flight together and no stage is ever refilled.
//
// The S CTAs of a tile form one thread-block cluster, and their fp32 partials
// meet in distributed shared memory: each CTA writes its partial (the rows
// below M only) into its own shared memory, the cluster synchronises, and the
// CTA of slice 0 adds the partials of slices 1..S-1 in slice order, so the sum
// and C do not depend on timing, and stores C. A second cluster barrier keeps
// every CTA's shared memory alive until it has been read. Nothing goes through
// global memory but A, B, the scales and C, so the kernel needs no workspace.
//
// Warps (192 threads, one CTA per SM by shared memory):
//   warp 0     TMA producer: for each K step of the slice, A [128 x 128] (rows
//              past M are zero-filled), B [128 x 128] and the two 512-byte scale
//              atoms, each step on a barrier of its own.
//   warp 1     TMEM allocator + single-thread issuer: tcgen05.cp of the atoms,
//              four tcgen05.mma.kind::mxf8f6f4.block_scale (M128 N128 K32) per
//              step into one accumulator, then one commit.
//   warps 2-5  epilogue, one TMEM lane quadrant each (32 rows of the tile);
//              warps whose rows all lie past M only take part in the barriers.
#include <type_traits>

#include "common.cuh"

namespace fp8bs {

constexpr int kMxdThreads = 6 * 32;
constexpr int kMxdEpiWarps = 4;

template <int MAXS>
struct MxdLayout {
    static constexpr int A_BYTES = kBlockM * kBlockK;       // 16 KiB
    static constexpr int B_BYTES = 128 * kBlockK;           // 16 KiB
    static constexpr int SF_BYTES = 1024;                   // A atom, then B atom
    static constexpr int OFF_A = 0;                          // after the MMAs: the partial [32][rows][4] fp32
    static constexpr int OFF_B = OFF_A + MAXS * A_BYTES;
    static constexpr int OFF_SF = OFF_B + MAXS * B_BYTES;
    static constexpr int OFF_BAR = OFF_SF + MAXS * SF_BYTES;
    static constexpr int NBAR = MAXS + 2;                    // full[MAXS], acc_full, mma_done
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;      // TMEM holder, abort flag, partial-valid flag
    static constexpr int BYTES = OFF_MISC + 16;
    static constexpr int DYN_SMEM = BYTES + 1024;
    // TMEM: accumulator columns [0, 128), then 8 scale-factor columns per step.
    static constexpr int SF_COL0 = 128;
    static constexpr int TMEM_COLS = 256;
    static_assert(SF_COL0 + 8 * MAXS <= TMEM_COLS, "tensor memory budget");
    static_assert(DYN_SMEM <= 232448, "shared memory budget");
    static_assert(MAXS * A_BYTES >= 128 * 128 * 4, "the partial of 128 rows fits where the A tiles were");
};

template <int MAXS>
__global__ void __launch_bounds__(kMxdThreads, 1)
    fp8bs_mxfp8_decode_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                              const GemmArgs args)
{
    using L = MxdLayout<MAXS>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = ptx::smem_u32(smem_raw);
    const uint32_t sbase = (raw_s + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw_s);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int KS = args.K / kBlockK;
    const int S = args.kslices;                                  // = the cluster size
    const int tile = static_cast<int>(blockIdx.x) / S;
    const int slice = S > 1 ? static_cast<int>(ptx::cluster_ctarank()) : 0;
    const int ks0 = static_cast<int>((static_cast<long long>(slice) * KS) / S);
    const int steps = static_cast<int>((static_cast<long long>(slice + 1) * KS) / S) - ks0;
    // The host sizes S so that every slice has 1..MAXS steps (1 <= S <= KS and
    // ceil(KS/S) <= MAXS). The check depends on K and S only, so every CTA of a
    // cluster returns here or none does.
    if (S < 1 || S > KS || (KS + S - 1) / S > MAXS) {
        if (threadIdx.x == 0)
            atomicExch(args.status, kStatusTimeout);
        return;
    }

    auto full_bar = [&](int s) { return sbase + L::OFF_BAR + 8u * s; };
    const uint32_t acc_full_bar = sbase + L::OFF_BAR + 8u * MAXS;
    const uint32_t mma_done_bar = sbase + L::OFF_BAR + 8u * (MAXS + 1);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 4);
    volatile int *valid_flag = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 8);

    if (threadIdx.x == 0) {
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB);
        for (int s = 0; s < MAXS; ++s)
            ptx::mbar_init(full_bar(s), 1);
        ptx::mbar_init(acc_full_bar, 1);
        ptx::mbar_init(mma_done_bar, 1);
        *abort_flag = 0;
        *valid_flag = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();

    // Live rows of this CTA's epilogue warps; the partial is [32][RP][4] fp32.
    const int RP = (args.M + 31) / 32 * 32;
    const uint32_t part_smem = sbase + L::OFF_A;
    float v[128];                 // epilogue: this thread's row of the accumulator
    bool epi_live = false;        // epilogue thread of a warp with a row below M, holding v
    bool epi_ok = false;          // epilogue thread: no epilogue warp of this CTA gave up

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // Every step of the slice at once: nothing is refilled.
        if (lane == 0) {
            for (int s = 0; s < steps; ++s) {
                const int ks = ks0 + s;
                const uint32_t sf = sbase + L::OFF_SF + s * L::SF_BYTES;
                ptx::mbar_arrive_expect_tx(full_bar(s), L::A_BYTES + L::B_BYTES + L::SF_BYTES);
                ptx::tma_load_2d(sbase + L::OFF_B + s * L::B_BYTES, &tmB, full_bar(s), ks * kBlockK, tile * 128);
                ptx::tma_load_2d(sbase + L::OFF_A + s * L::A_BYTES, &tmA, full_bar(s), ks * kBlockK, 0);
                ptx::bulk_load(sf, args.a_sf + static_cast<size_t>(ks) * 512, 512, full_bar(s));
                ptx::bulk_load(sf + 512, args.b_sf + (static_cast<size_t>(tile) * KS + ks) * 512, 512, full_bar(s));
            }
            // Every load issued must have landed before the CTA exits.
            for (int s = 0; s < steps; ++s)
                wait_teardown(full_bar(s), 0, args);
        }
        __syncwarp();
    } else {
        // TMEM for the issuer and the epilogue (the producer never touches it).
        if (warp == 1) {
            ptx::tmem_alloc(ptx::smem_u32(tmem_holder), L::TMEM_COLS);
            ptx::tmem_relinquish();
        }
        ptx::tc_fence_before();
        asm volatile("bar.sync 1, %0;" ::"n"(kMxdThreads - 32) : "memory");
        ptx::tc_fence_after();
        const uint32_t tmem_base = *tmem_holder;

        if (warp == 1) {
            // -------------------------------------------------------- MMA issuer
            if (lane == 0) {
                bool ok = true;
                for (int s = 0; s < steps; ++s) {
                    if (!wait_bounded(full_bar(s), 0, abort_flag, args)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sf = sbase + L::OFF_SF + s * L::SF_BYTES;
                    const uint32_t sfa_t = tmem_base + static_cast<uint32_t>(L::SF_COL0 + 8 * s);
                    const uint32_t sfb_t = sfa_t + 4;
                    ptx::tc_cp_32x128b_warpx4(sfa_t, ptx::desc_noswizzle(sf, 16, 128));
                    ptx::tc_cp_32x128b_warpx4(sfb_t, ptx::desc_noswizzle(sf + 512, 16, 128));
                    const uint64_t adesc = ptx::desc_kmajor_sw128(sbase + L::OFF_A + s * L::A_BYTES);
                    const uint64_t bdesc = ptx::desc_kmajor_sw128(sbase + L::OFF_B + s * L::B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < kBlockK / kMmaK; ++kk)
                        ptx::mma_mxf8f6f4(tmem_base, adesc + 2 * kk, bdesc + 2 * kk,
                                          ptx::idesc_mxf8f6f4_e4m3(kBlockM, 128, kk, kk), sfa_t, sfb_t,
                                          (s > 0 || kk > 0) ? 1u : 0u);
                }
                if (ok)
                    ptx::tc_commit(acc_full_bar);
                // No MMA may still be running when the tensor memory is freed.
                ptx::tc_commit(mma_done_bar);
                wait_teardown(mma_done_bar, 0, args);
            }
            __syncwarp();
        } else {
            // ---------------------------------------------------------- epilogue
            const int q = warp & 3;                   // TMEM lane quadrant of this warp
            const int row = q * 32 + lane;            // row of A / C
            const bool live = q * 32 < args.M;        // some row of this warp is below M
            const bool ok = wait_bounded_warp(acc_full_bar, 0, abort_flag, args);
            ptx::tc_fence_after();
            if (ok && live) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t r[32];
                    ptx::tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + c * 32, r);
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        v[c * 32 + j] = __uint_as_float(r[j]);
                }
                ptx::tmem_wait_ld();
                epi_live = true;
                // The MMAs have completed (acc_full), so the A tiles are free: a
                // CTA of a cluster leaves its partial there for slice 0 to read,
                // [column/4][row] float4 (a warp's store is 512 contiguous bytes).
                if (S > 1 && slice > 0) {
#pragma unroll
                    for (int c4 = 0; c4 < 32; ++c4)
                        ptx::st_shared_v4(part_smem + static_cast<uint32_t>((c4 * RP + row) * 16),
                                          __float_as_uint(v[4 * c4]), __float_as_uint(v[4 * c4 + 1]),
                                          __float_as_uint(v[4 * c4 + 2]), __float_as_uint(v[4 * c4 + 3]));
                }
            }
            // The partial of this CTA is whole only if no epilogue warp gave up.
            // Every epilogue thread gets the answer from the barrier; the flag
            // in shared memory is for slice 0 of the cluster, which reads it
            // after the cluster barrier.
            epi_ok = ptx::bar_red_and<2, kMxdEpiWarps * 32>(ok);
            if (threadIdx.x == 64)
                *valid_flag = epi_ok ? 1 : 0;
        }
    }

    // C row `row`, columns tile*128 + 8*j0 .. + 8*NJ - 1 from x[0 .. 8*NJ)
    // (N is a multiple of 8).
    const int row = (warp & 3) * 32 + lane;
    auto store_row = [&](const float *x, int j0, auto nj) {
        constexpr int NJ = decltype(nj)::value;
        if (row >= args.M)
            return;
        const int n0 = tile * 128;
        uint16_t *dst = static_cast<uint16_t *>(args.c_out) + static_cast<size_t>(row) * args.N + n0;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            if (n0 + 8 * (j0 + j) >= args.N)
                break;
            const uint32_t w0 = ptx::pack_bf16x2(x[8 * j + 0], x[8 * j + 1]);
            const uint32_t w1 = ptx::pack_bf16x2(x[8 * j + 2], x[8 * j + 3]);
            const uint32_t w2 = ptx::pack_bf16x2(x[8 * j + 4], x[8 * j + 5]);
            const uint32_t w3 = ptx::pack_bf16x2(x[8 * j + 6], x[8 * j + 7]);
            asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(dst + 8 * (j0 + j)), "r"(w0), "r"(w1),
                         "r"(w2), "r"(w3)
                         : "memory");
        }
    };

    if (S == 1) {
        if (epi_live && epi_ok)
            store_row(v, 0, std::integral_constant<int, 16>{});
    } else {
        // Every CTA of the cluster, every thread, on every path (all waits
        // above are bounded): the partials and their valid flags are visible.
        ptx::cluster_sync();
        if (slice == 0 && epi_live) {
            bool all_valid = epi_ok;
            for (int r = 1; r < S; ++r)
                all_valid = all_valid && ptx::ld_cluster_u32(ptx::mapa_shared(sbase + L::OFF_MISC + 8, r)) != 0;
            if (all_valid) {
                // C = slice 0 (registers) + slice 1 + ... + slice S-1, in that
                // order, 32 columns at a time.
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    float t[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        t[j] = v[g * 32 + j];
                    for (int r = 1; r < S; ++r) {
                        const uint32_t rbase = ptx::mapa_shared(part_smem, r);
                        float4 p[8];
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            p[c] = ptx::ld_cluster_v4_f32(rbase + static_cast<uint32_t>(((g * 8 + c) * RP + row) * 16));
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            t[4 * c] += p[c].x;
                            t[4 * c + 1] += p[c].y;
                            t[4 * c + 2] += p[c].z;
                            t[4 * c + 3] += p[c].w;
                        }
                    }
                    store_row(t, 4 * g, std::integral_constant<int, 4>{});
                }
            }
        }
        // No CTA leaves (freeing its shared memory) before slice 0 has read it.
        ptx::cluster_sync();
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(*tmem_holder, L::TMEM_COLS);
    }
}

// Launch of the decode kernel: clusters of args.kslices CTAs (the slices of a
// tile), ceil(N/128) clusters.
template <int MAXS>
cudaError_t launch_mxfp8_decode(const CUtensorMap &tmA, const CUtensorMap &tmB, const GemmArgs &args,
                                cudaStream_t stream)
{
    using L = MxdLayout<MAXS>;
    auto kern = fp8bs_mxfp8_decode_kernel<MAXS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::DYN_SMEM);
    if (e != cudaSuccess)
        return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(args.kslices);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(((args.N + 127) / 128) * args.kslices);
    cfg.blockDim = dim3(kMxdThreads);
    cfg.dynamicSmemBytes = L::DYN_SMEM;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tmA, tmB, args);
}

// Clusters of `slices` CTAs of the decode kernel that fit on the device at once (0: none).
template <int MAXS>
cudaError_t max_mxfp8_decode_clusters(int slices, int *out)
{
    using L = MxdLayout<MAXS>;
    auto kern = fp8bs_mxfp8_decode_kernel<MAXS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::DYN_SMEM);
    if (e != cudaSuccess)
        return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(slices);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(slices);
    cfg.blockDim = dim3(kMxdThreads);
    cfg.dynamicSmemBytes = L::DYN_SMEM;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(out, kern, &cfg);
}

template cudaError_t launch_mxfp8_decode<kMxdMaxSteps>(const CUtensorMap &, const CUtensorMap &, const GemmArgs &,
                                                      cudaStream_t);
template cudaError_t max_mxfp8_decode_clusters<kMxdMaxSteps>(int, int *);

} // namespace fp8bs
