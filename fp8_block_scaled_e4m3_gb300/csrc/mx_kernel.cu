// MXFP8 GEMM kernel for sm_103a.
//
// Computes C[m,n] = bf16( sum_k A[m,k] 2^(ea[m,k/32]-127) * B[n,k] 2^(eb[n,k/32]-127) ).
// The PR "1x32 ue8m0 (MXFP8) 8-wave FlyDSL GEMM for gfx950" (section "Why it is
// faster") feeds the ue8m0 scales to the matrix instruction as operands, so
// there is no software promote: here tcgen05.mma.kind::mxf8f6f4.block_scale
// (scale_vec::1X: one scale byte per row per 32-wide K slice) accumulates over
// the whole K extent in tensor memory.
//
// Persistent, warp-specialised, one CTA per SM, 12 warps:
//   warp 0       TMA producer: A [128 x 128] and B [BN x 128] e4m3 per 128-wide K
//                step, plus the step's scale-factor atoms (512 bytes per 128 rows)
//                from the packed scale layout, all on one mbarrier.
//   warp 1       TMEM allocator + single-thread issuer: tcgen05.cp of the atoms
//                into TMEM (32x128b.warpx4), then four block-scaled MMAs (scale
//                byte id = the 32-wide slice inside the step).
//   warps 2, 3   idle (they complete the control warpgroup of the register split).
//   warps 4..11  epilogue: drain the fp32 accumulator (BN/2 columns per thread),
//                release it to the next accumulation, bf16 convert, TMA store.
//
// Work schedule (WorkSpan in common.cuh), as in the blockscale kernel: one CTA
// per tile, or stream-K for shapes whose last wave of tiles is partial. A tile
// cut between CTAs is accumulated in pieces; the CTAs holding its later K steps
// publish their fp32 partial sums, and the CTA holding K step 0 adds them
// before it stores the tile.
//
// The same body, compiled without the scale atoms and with plain fp8 MMAs, is
// the blockscale GEMM's promote-free ceiling twin: identical tiles and MMA work,
// one per-tensor scale applied in the epilogue (fp8bs_tensorscale_kernel).
//
// Packed scale layout (written by fp8mx_pack_scales from the quantiser's
// row-major [rows][K/32] bytes, which are not TMA-addressable because a row of
// K/32 bytes is not a 16-byte multiple in general): for 128-row block rb and
// K step ks, a 512-byte atom at ((rb * K/128) + ks) * 512 holding byte j of row
// r at sf_atom_offset(r, j), i.e. the shared-memory image one tcgen05.cp
// 32x128b.warpx4 moves into four TMEM columns.
#include "common.cuh"

namespace fp8bs {

// Kernel variants (one instance each, so that the common path carries no code
// it does not run: with the stream-K hand-off and the E4M3 store compiled into
// one kernel, 16384x5120x2048 measured 136.9 us against 125.3 us without
// either, and the stream-K register split below cost another 3.6%):
//   kMxPlain  one CTA per tile, bf16 C: 10 warps (producer, issuer, 8 epilogue)
//   kMxSplitK stream-K, bf16 C: 12 warps with a register split (the epilogue
//             holds a thread's accumulator columns through the hand-off)
//   kMxE4m3   one CTA per tile, E4M3 C (MXFP8 only): 10 warps
constexpr int kMxPlain = 0;
constexpr int kMxSplitK = 1;
constexpr int kMxE4m3 = 2;
template <int V> constexpr int kMxCtrlWarps = V == kMxSplitK ? 4 : 2;
template <int V> constexpr int kMxThreads = (kMxCtrlWarps<V> + kEpiWarps) * 32;
// Register split of the stream-K variant (setmaxnreg) out of the launch
// allotment of 384 threads x 168: the control warpgroup drops to kMxRegsLow,
// the two epilogue warpgroups rise to kMxRegsHigh.
constexpr int kMxRegsLow = 64;
constexpr int kMxRegsHigh = 216;
static_assert(128 * kMxRegsLow + 256 * kMxRegsHigh <= kMxThreads<kMxSplitK> * 168, "register split");

template <int BN, int STAGES, bool MX = true>
struct MxLayout {
    static constexpr int A_BYTES = kBlockM * kBlockK;
    static constexpr int B_BYTES = BN * kBlockK;
    static constexpr int SFA_BYTES = MX ? 512 : 0;   // one atom: 128 rows x 4 groups
    static constexpr int SFB_BYTES = MX ? 512 * (BN / 128) : 0;
    static constexpr int SF_BYTES = SFA_BYTES + SFB_BYTES;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_SF = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_C = (OFF_SF + STAGES * SF_BYTES + 1023) / 1024 * 1024;
    static constexpr int OFF_BAR = OFF_C + kEpiWarps * kCStageBytes;
    static constexpr int NBAR = 2 * STAGES + 3;     // full[S], empty[S], acc_full, acc_empty, mma_done
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int BYTES = OFF_MISC + 16;
    static constexpr int DYN_SMEM = BYTES + 1024;
    // TMEM: accumulator columns [0, BN), then 16 scale-factor columns per stage
    // (A atom: 4 columns, B atoms: 4 columns per 128 rows).
    static constexpr int SF_COL0 = BN;
    static constexpr int SF_COLS_PER_STAGE = 16;
    static constexpr int TMEM_COLS = 512;
    static_assert(SF_COL0 + STAGES * SF_COLS_PER_STAGE <= TMEM_COLS, "tensor memory budget");
    static_assert(4 + 4 * (BN / 128) <= SF_COLS_PER_STAGE, "scale columns per stage");
    static_assert(DYN_SMEM <= 232448, "shared memory budget");
    static_assert(BN == 128 || BN == 256, "tile width");
};

// Body of both kernels below. MX: block-scaled MMAs with the ue8m0 scale atoms
// staged per K step; !MX: plain fp8 MMAs and one per-tensor scale (args.alpha)
// applied in the epilogue, i.e. the same MMA work with no per-block scaling.
template <int BN, int STAGES, bool MX, int V>
__device__ __forceinline__ void mx_gemm_body(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC,
                                             const GemmArgs &args)
{
    using L = MxLayout<BN, STAGES, MX>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = ptx::smem_u32(smem_raw);
    const uint32_t sbase = (raw_s + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw_s);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int KS = args.K / kBlockK;
    const int num_tiles = args.raster.num_tiles();

    auto full_bar = [&](int s) { return sbase + L::OFF_BAR + 8u * s; };
    auto empty_bar = [&](int s) { return sbase + L::OFF_BAR + 8u * (STAGES + s); };
    const uint32_t acc_full_bar = sbase + L::OFF_BAR + 8u * (2 * STAGES);
    const uint32_t acc_empty_bar = sbase + L::OFF_BAR + 8u * (2 * STAGES + 1);
    const uint32_t mma_done_bar = sbase + L::OFF_BAR + 8u * (2 * STAGES + 2);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full_bar(s), 1);      // producer (with tx bytes)
            ptx::mbar_init(empty_bar(s), 1);     // MMA commit
        }
        ptx::mbar_init(acc_full_bar, 1);
        ptx::mbar_init(acc_empty_bar, kEpiWarps);
        ptx::mbar_init(mma_done_bar, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_holder), L::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    constexpr int CTRL = kMxCtrlWarps<V>;
    if (warp < CTRL) {
    if constexpr (V == kMxSplitK)
        ptx::setmaxnreg_dec<kMxRegsLow>();
    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            ptx::prefetch_tmap(&tmA);
            ptx::prefetch_tmap(&tmB);
            const int n_blocks = (args.N + 127) / 128;   // packed atoms per K step of B
            // Stage s <- K step ks of tile (mb, nb).
            auto load_step = [&](int s, int ks, int mb, int nb) {
                ptx::mbar_arrive_expect_tx(full_bar(s), L::A_BYTES + L::B_BYTES + L::SF_BYTES);
                ptx::tma_load_2d(sbase + L::OFF_A + s * L::A_BYTES, &tmA, full_bar(s), ks * kBlockK, mb * kBlockM);
                ptx::tma_load_2d(sbase + L::OFF_B + s * L::B_BYTES, &tmB, full_bar(s), ks * kBlockK, nb * BN);
                if constexpr (MX) {
                    // Scale atoms. A 128-row B block past N (the second half of a
                    // 256-wide tile when N has an odd number of 128-row blocks) reads
                    // the last real atom instead: those B rows are zero-filled by the
                    // tensor copy and their C columns are never stored.
                    const uint32_t sf_smem = sbase + L::OFF_SF + s * L::SF_BYTES;
                    ptx::bulk_load(sf_smem, args.a_sf + (static_cast<size_t>(mb) * KS + ks) * 512, 512, full_bar(s));
#pragma unroll
                    for (int h = 0; h < BN / 128; ++h) {
                        const int bblk = nb * (BN / 128) + h < n_blocks ? nb * (BN / 128) + h : n_blocks - 1;
                        ptx::bulk_load(sf_smem + L::SFA_BYTES + 512 * h,
                                       args.b_sf + (static_cast<size_t>(bblk) * KS + ks) * 512, 512, full_bar(s));
                    }
                }
            };
            int it = 0;
            if constexpr (V != kMxSplitK) {
                // one CTA per tile: tiles blockIdx.x, + gridDim.x, ...
                bool ok = true;
                for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                    int mb, nb;
                    args.raster.coords(t, mb, nb);
                    for (int ks = 0; ks < KS; ++ks, ++it) {
                        const int s = it % STAGES;
                        if (!wait_bounded(empty_bar(s), ((it / STAGES) & 1) ^ 1, abort_flag, args)) {
                            ok = false;
                            break;
                        }
                        load_step(s, ks, mb, nb);
                    }
                }
            } else {
                WorkSpan span;
                span.init(args, KS);
                int t, ks, mb = 0, nb = 0;
                span.step(0, t, ks);
                for (; it < span.total; ++it, span.advance(it, t, ks)) {
                    if (it == 0 || ks == 0 || it == span.dp_steps)   // a new tile (a range may start mid-tile)
                        args.raster.coords(t, mb, nb);
                    const int s = it % STAGES;
                    if (!wait_bounded(empty_bar(s), ((it / STAGES) & 1) ^ 1, abort_flag, args))
                        break;
                    load_step(s, ks, mb, nb);
                }
            }
            for (int s = 0; s < STAGES; ++s) {
                const int uses = it > s ? (it - s + STAGES - 1) / STAGES : 0;
                if (uses > 0)
                    wait_teardown(full_bar(s), (uses - 1) & 1, args);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        // One accumulation per segment: the K steps of one tile in this CTA's
        // range (a whole tile, or a piece of a tile cut by stream-K).
        if (lane == 0) {
            // The MMAs of the K step in stage s; `first` starts the accumulation.
            auto issue_step = [&](int s, bool first) {
                if constexpr (!MX) {
                    constexpr uint32_t idesc = ptx::idesc_f8f6f4_e4m3(kBlockM, BN);
                    const uint64_t adesc = ptx::desc_kmajor_sw128(sbase + L::OFF_A + s * L::A_BYTES);
                    const uint64_t bdesc = ptx::desc_kmajor_sw128(sbase + L::OFF_B + s * L::B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < kBlockK / kMmaK; ++kk)
                        ptx::mma_f8f6f4(tmem_base, adesc + 2 * kk, bdesc + 2 * kk, idesc,
                                        (!first || kk != 0) ? 1u : 0u);
                } else {
                    const uint32_t sf_smem = sbase + L::OFF_SF + s * L::SF_BYTES;
                    const uint32_t sfa_t = tmem_base + static_cast<uint32_t>(L::SF_COL0 + s * L::SF_COLS_PER_STAGE);
                    const uint32_t sfb_t = sfa_t + 4;
                    ptx::tc_cp_32x128b_warpx4(sfa_t, ptx::desc_noswizzle(sf_smem, 16, 128));
#pragma unroll
                    for (int h = 0; h < BN / 128; ++h)
                        ptx::tc_cp_32x128b_warpx4(sfb_t + 4 * h,
                                                  ptx::desc_noswizzle(sf_smem + L::SFA_BYTES + 512 * h, 16, 128));
                    const uint64_t adesc = ptx::desc_kmajor_sw128(sbase + L::OFF_A + s * L::A_BYTES);
                    const uint64_t bdesc = ptx::desc_kmajor_sw128(sbase + L::OFF_B + s * L::B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < kBlockK / kMmaK; ++kk)
                        ptx::mma_mxf8f6f4(tmem_base, adesc + 2 * kk, bdesc + 2 * kk,
                                          ptx::idesc_mxf8f6f4_e4m3(kBlockM, BN, kk, kk), sfa_t, sfb_t,
                                          (!first || kk != 0) ? 1u : 0u);
                }
                ptx::tc_commit(empty_bar(s));
            };
            bool ok = true;
            if constexpr (V != kMxSplitK) {
                int it = 0, titer = 0;
                for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++titer) {
                    if (!wait_bounded(acc_empty_bar, (titer & 1) ^ 1, abort_flag, args))
                        break;
                    ptx::tc_fence_after();
                    for (int ks = 0; ks < KS; ++ks, ++it) {
                        const int s = it % STAGES;
                        if (!wait_bounded(full_bar(s), (it / STAGES) & 1, abort_flag, args)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        issue_step(s, ks == 0);
                    }
                    if (!ok)
                        break;
                    ptx::tc_commit(acc_full_bar);
                }
            } else {
                WorkSpan span;
                span.init(args, KS);
                for (int it = 0, sg = 0; it < span.total && ok; ++sg) {
                    int t, ks0;
                    span.step(it, t, ks0);
                    const int seg_end = it + ((KS - ks0) < (span.total - it) ? (KS - ks0) : (span.total - it));
                    if (!wait_bounded(acc_empty_bar, (sg & 1) ^ 1, abort_flag, args))
                        break;
                    ptx::tc_fence_after();
                    const int seg_start = it;
                    for (; it < seg_end; ++it) {
                        const int s = it % STAGES;
                        if (!wait_bounded(full_bar(s), (it / STAGES) & 1, abort_flag, args)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        issue_step(s, it == seg_start);
                    }
                    if (!ok)
                        break;
                    ptx::tc_commit(acc_full_bar);
                }
            }
            ptx::tc_commit(mma_done_bar);
            wait_teardown(mma_done_bar, 0, args);
        }
    }
    } else {
        if constexpr (V == kMxSplitK)
            ptx::setmaxnreg_inc<kMxRegsHigh>();
        // ------------------------------------------------------ epilogue
        constexpr int HALF = BN / 2;
        constexpr bool kSk = V == kMxSplitK;    // the stream-K hand-off
        const int ew = warp - CTRL;             // 0..7
        const int wg = ew >> 2;
        const int q = warp & 3;
        const int row = q * 32 + lane;          // row of the tile
        const uint32_t cstage = sbase + L::OFF_C + ew * kCStageBytes;
        WorkSpan span;
        span.init(args, KS);
        bool ok = true;
        for (int it = 0, sg = 0; it < span.total; ++sg) {
            int t, ks0, mb, nb;
            span.step(it, t, ks0);
            const int len = (KS - ks0) < (span.total - it) ? (KS - ks0) : (span.total - it);
            const int ks_last = ks0 + len - 1;
            it += len;
            args.raster.coords(t, mb, nb);
            if (!wait_bounded_warp(acc_full_bar, sg & 1, abort_flag, args))
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
            if (lane == 0)
                ptx::mbar_arrive(acc_empty_bar);
            // Stream-K hand-off, warp by warp, as in the blockscale kernel: warp
            // ew of every CTA owns the same 32 rows x HALF columns of a tile, in
            // slot layout [column/4][row] of float4.
            const size_t slice = static_cast<size_t>(wg * HALF / 4) * kBlockM + static_cast<size_t>(row);
            // Warps whose rows all lie past M skip the hand-off (as in the blockscale kernel).
            const bool rows_live = mb * kBlockM + q * 32 < args.M;
            if (kSk && ks0 > 0) {
                if (!rows_live)
                    continue;
                // Head of a tile begun by an earlier CTA: publish the partial.
                float *dst = args.sk_partial + static_cast<size_t>(blockIdx.x) * (BN * kBlockM) + 4 * slice;
#pragma unroll
                for (int j = 0; j < HALF; j += 4)
                    ptx::st_global_v4_f32(dst + static_cast<size_t>(j / 4) * kBlockM * 4, v[j], v[j + 1], v[j + 2],
                                          v[j + 3]);
                // The warp barrier orders every lane's stores before lane 0's
                // release store of the flag, and a release is cumulative: a
                // finisher that acquires the flag sees the whole slice.
                __syncwarp();
                if (lane == 0)
                    ptx::st_release_gpu_u64(args.sk_flags + static_cast<size_t>(blockIdx.x) * kEpiWarps + ew,
                                            args.sk_token);
                continue;
            }
            if (kSk && ks_last != KS - 1 && rows_live) {
                // This CTA holds K step 0 of a cut tile: add the partials of the
                // CTAs up to the one whose range holds the tile's last unit.
                const long long G = gridDim.x;
                const long long U = static_cast<long long>(num_tiles - span.tile0) * KS;
                const long long tile_end = static_cast<long long>(t + 1 - span.tile0) * KS;
                const int c_last = static_cast<int>((tile_end * G - 1) / U);
                for (int c2 = static_cast<int>(blockIdx.x) + 1; c2 <= c_last; ++c2) {
                    unsigned long long *flag = args.sk_flags + static_cast<size_t>(c2) * kEpiWarps + ew;
                    if (!sk_wait_flag(flag, args.sk_token, abort_flag, args)) {
                        ok = false;
                        break;
                    }
                    const float *src = args.sk_partial + static_cast<size_t>(c2) * (BN * kBlockM) + 4 * slice;
#pragma unroll
                    for (int j = 0; j < HALF; j += 4) {
                        const float4 p = ptx::ld_cg_v4_f32(src + static_cast<size_t>(j / 4) * kBlockM * 4);
                        v[j] += p.x;
                        v[j + 1] += p.y;
                        v[j + 2] += p.z;
                        v[j + 3] += p.w;
                    }
                    __syncwarp();
                    if (lane == 0)
                        *reinterpret_cast<volatile unsigned long long *>(flag) = 0ull;   // ready for the next call
                }
                if (!ok)
                    break;
            }
            if constexpr (!MX) {
#pragma unroll
                for (int j = 0; j < HALF; ++j)
                    v[j] *= args.alpha;
            }
            const int x0 = nb * BN + wg * HALF;
            const int y0 = mb * kBlockM + q * 32;
            if constexpr (MX && V == kMxE4m3) {
#pragma unroll
                for (int c = 0; c < HALF / 64; ++c)
                    store_c8_chunk(&tmC, cstage, lane, v + c * 64, args.c_scale, x0 + c * 64, y0, args.M, args.N);
            } else {
#pragma unroll
                for (int c = 0; c < HALF / kCChunkCols; ++c)
                    store_c_chunk(&tmC, cstage, lane, v + c * kCChunkCols, x0 + c * kCChunkCols, y0, args.M,
                                  args.N);
            }
        }
        if (lane == 0)
            ptx::bulk_wait_all();
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, L::TMEM_COLS);
    }
}

// The MXFP8 GEMM, one CTA per tile: bf16 C (V = kMxPlain) or E4M3 C (kMxE4m3).
template <int BN, int STAGES, int V>
__global__ void __launch_bounds__(kMxThreads<V>, 1)
    fp8bs_mxfp8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmC, const GemmArgs args)
{
    mx_gemm_body<BN, STAGES, true, V>(tmA, tmB, tmC, args);
}

// The MXFP8 GEMM under stream-K.
template <int BN, int STAGES>
__global__ void __launch_bounds__(kMxThreads<kMxSplitK>, 1)
    fp8bs_mxfp8_sk_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmC, const GemmArgs args)
{
    mx_gemm_body<BN, STAGES, true, kMxSplitK>(tmA, tmB, tmC, args);
}

// Promote-free ceiling twin of the blockscale GEMM (skill card "FlyDSL fp8
// blockscale GEMM", section "Bottleneck diagnosis": the same kernel with one
// per-tensor scale, i.e. identical MMA work): C = bf16(alpha * A.B^T).
template <int BN, int STAGES>
__global__ void __launch_bounds__(kMxThreads<kMxPlain>, 1)
    fp8bs_tensorscale_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmC, const GemmArgs args)
{
    mx_gemm_body<BN, STAGES, false, kMxPlain>(tmA, tmB, tmC, args);
}

template <int BN, int STAGES>
__global__ void __launch_bounds__(kMxThreads<kMxSplitK>, 1)
    fp8bs_tensorscale_sk_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                                const __grid_constant__ CUtensorMap tmC, const GemmArgs args)
{
    mx_gemm_body<BN, STAGES, false, kMxSplitK>(tmA, tmB, tmC, args);
}

template <int BN, int STAGES, bool MX, int V, typename Kern>
cudaError_t launch_mx_kernel(Kern kern, const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC,
                             const GemmArgs &args, int grid, cudaStream_t stream)
{
    constexpr int DYN_SMEM = MxLayout<BN, STAGES, MX>::DYN_SMEM;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, DYN_SMEM);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kMxThreads<V>);
    cfg.dynamicSmemBytes = DYN_SMEM;
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmC, args);
}

// kind: 0 MXFP8 bf16 C, 1 MXFP8 E4M3 C, 2 tensor-scale twin; sk: stream-K.
template <int BN, int STAGES>
cudaError_t launch_mx_family(int kind, bool sk, const CUtensorMap &tmA, const CUtensorMap &tmB,
                             const CUtensorMap &tmC, const GemmArgs &args, int grid, cudaStream_t stream)
{
    if (kind == 2)
        return sk ? launch_mx_kernel<BN, STAGES, false, kMxSplitK>(fp8bs_tensorscale_sk_kernel<BN, STAGES>, tmA, tmB, tmC,
                                                             args, grid, stream)
                  : launch_mx_kernel<BN, STAGES, false, kMxPlain>(fp8bs_tensorscale_kernel<BN, STAGES>, tmA, tmB, tmC, args,
                                                            grid, stream);
    if (kind == 1)
        return launch_mx_kernel<BN, STAGES, true, kMxE4m3>(fp8bs_mxfp8_kernel<BN, STAGES, kMxE4m3>, tmA, tmB, tmC, args,
                                                      grid, stream);
    return sk ? launch_mx_kernel<BN, STAGES, true, kMxSplitK>(fp8bs_mxfp8_sk_kernel<BN, STAGES>, tmA, tmB, tmC, args, grid,
                                                         stream)
              : launch_mx_kernel<BN, STAGES, true, kMxPlain>(fp8bs_mxfp8_kernel<BN, STAGES, kMxPlain>, tmA, tmB, tmC, args,
                                                        grid, stream);
}

template cudaError_t launch_mx_family<256, 4>(int, bool, const CUtensorMap &, const CUtensorMap &,
                                              const CUtensorMap &, const GemmArgs &, int, cudaStream_t);
template cudaError_t launch_mx_family<128, 6>(int, bool, const CUtensorMap &, const CUtensorMap &,
                                              const CUtensorMap &, const GemmArgs &, int, cudaStream_t);

} // namespace fp8bs
