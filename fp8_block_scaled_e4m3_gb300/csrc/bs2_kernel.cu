// FP8 block-scaled GEMM kernel for sm_103a, CTA-pair version.
//
// Same result as fp8bs_blockscale_kernel (bs_kernel.cu):
//   C[m,n] = bf16( sum_kb P_kb[m,n] * a_scale[m,kb] * b_scale[n/128,kb] ),
// P_kb the unscaled fp8 product of 128-wide K block kb, promoted in fp32 after
// the matrix unit (skill card "FlyDSL fp8 blockscale GEMM", "Mechanism A").
//
// Two CTAs of a cluster (two SMs) share one 256 x 256 tile. Each CTA owns 128
// rows of A and C and holds 128 of the 256 B rows; the even CTA issues
// tcgen05.mma.cta_group::2 (M256 x N256 x K32), which reads A from each CTA's
// own shared memory, exchanges the B halves and writes each CTA's 128 x 256
// partial P_kb into that CTA's tensor memory (two 256-column buffers per CTA,
// as in the one-CTA kernel). Against the one-CTA kernel on 128 x 256 tiles:
//   - a CTA's stage is A 16 KiB + half of B 16 KiB, so four stages take 128
//     KiB where the one-CTA kernel's take 192, and the shared-memory fill per
//     K block (the L2 -> SM stream) drops from 48 to 32 KiB per SM;
//   - one MMA instruction does two SMs' work, so each SM issues half as many
//     (issuing holds up the promote warps of the issuer's sub-partition).
// The promote (fp32 FMAs on TMEM loads) and the epilogue are the one-CTA
// kernel's, per CTA.
//
// Per CTA, 12 warps (3 warpgroups):
//   warp 0      TMA producer: own A rows and own B half into stage s; both
//               CTAs' bytes complete on the even CTA's full[s], which the even
//               CTA's producer arms with the pair's total (an odd-CTA copy may
//               land first: the phase cannot complete before that arrive). The
//               a_scale slice [128] of the CTA's own rows goes to a local ring.
//   warp 3      C store: four TMA stores per tile from the whole-tile buffer.
//   warps 1, 2  pair TMEM allocation (warp 1) and, in the even CTA only, the MMA
//               issuers of the even and the odd steps (one thread each; each
//               owns one TMEM buffer and every other stage); tcgen05.commit
//               multicasts "partial ready" and the stage release to both CTAs.
//   warps 4..11 promote + epilogue for this CTA's 128 rows: thread = one row,
//               128 columns of one 128-column N block (one b_scale value);
//               a buffer is released on the even CTA's tempty barrier (16
//               arrivals, 8 warps of each CTA; the odd CTA's are relaxed remote
//               arrives).
//   - the shared memory left over holds this CTA's whole 128 x 256 bf16 C
//     tile (64 KiB): every promote warp converts its rows into it, arrives
//     (c_full) and goes on to the next tile; warp 3 stores the tile by four TMA
//     stores of 64 columns x 128 rows and releases the buffer (c_empty) as
//     soon as they have read it. The C store of a tile thus overlaps the next
//     tile's K loop, and the promote warps wait on nothing at a tile boundary
//     but a buffer that was freed long before (the one-CTA four-stage kernel
//     stages C in 2 KiB chunks per warp and has no room for this).
// Schedule: one CTA pair per tile, or (SK = true) stream-K over (tile, K
// block) units with the pair as the worker (WorkSpanT<2> in common.cuh):
//   - a CTA of a pair that holds the head of a tile begun by an earlier pair
//     writes its scaled fp32 partial (its own 128 rows) to its slot of the
//     workspace and raises per-warp flags;
//   - in the CTA of the same rank of the pair holding the tile's K block 0 (its
//     range's last segment), the producer waits for the flags and, once the
//     MMAs have read every stage, copies each partial (128 KiB, the size of the
//     whole operand ring) into the ring by one bulk copy; the promote warps add
//     it from there before the C store.
// Both CTAs of a pair run the same steps, so the pair MMAs need no change. The
// two schedules are separate instances: with the stream-K code in the same
// instance, one-pair-per-tile shapes measured 6-13% slower although the
// hand-off never ran. E4M3 C runs on the one-CTA kernel.
#include "common.cuh"

#include <type_traits>

namespace fp8bs {

constexpr int kBs2Threads = (4 + kEpiWarps) * 32;
constexpr int kBs2BN = 256;             // N of the pair tile and of each CTA's partial
constexpr int kBs2NBuf = 2;             // TMEM partial buffers per CTA (2 x 256 columns)
constexpr int kBs2SaSlots = 16;
// Register split as in the one-CTA kernel's 256-wide tile: 168 per thread at
// launch; warpgroup 0 drops to 40 and the promote warpgroups rise to 232.
constexpr int kBs2RegsLow = 40;
constexpr int kBs2RegsHigh = 232;
static_assert(128 * kBs2RegsLow + 256 * kBs2RegsHigh <= kBs2Threads * 168, "register split");

template <int STAGES>
struct Bs2Layout {
    static constexpr int A_BYTES = kBlockM * kBlockK;             // own 128 rows
    static constexpr int B_BYTES = (kBs2BN / 2) * kBlockK;        // own 128 of the tile's 256 B rows
    static constexpr int SA_BYTES = kBlockM * 4;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_SA = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_C = (OFF_SA + kBs2SaSlots * SA_BYTES + 1023) / 1024 * 1024;
    static constexpr int C_AREA = kBlockM * kBs2BN * 2;   // the whole-tile C buffer (bf16)
    static constexpr int OFF_BAR = OFF_C + C_AREA;
    // full[S], empty[S], tfull[NBUF], tempty[NBUF], mma_done, sa_full[SA], sa_empty[SA], c_full, c_empty,
    // part_full, part_empty
    static constexpr int NBAR = 2 * STAGES + 2 * kBs2NBuf + 1 + 2 * kBs2SaSlots + 4;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int BYTES = OFF_MISC + 32;   // TMEM address, abort flag, stream-K span (4 ints)
    static constexpr int DYN_SMEM = BYTES + 1024;
    static constexpr int TMEM_COLS = kBs2NBuf * kBs2BN;
    static_assert(TMEM_COLS == 512, "tensor memory");
    static_assert(STAGES % 2 == 0 && kBs2SaSlots % 2 == 0 && kBs2NBuf == 2,
                  "producers and issuers split the stages, slots and buffers by step parity");
    static_assert(DYN_SMEM <= 232448, "shared memory budget");
    // stream-K: a finisher copies one CTA's fp32 partial (128 rows x 256
    // columns) into the operand ring once its last K block has been read
    static_assert(OFF_A == 0 && OFF_B == STAGES * A_BYTES && STAGES * (A_BYTES + B_BYTES) == kBlockM * kBs2BN * 4,
                  "the ring holds one partial");
};

template <int STAGES, bool SK>
__global__ void __launch_bounds__(kBs2Threads, 1)
    fp8bs_blockscale_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                                 const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmC,
                                 const GemmArgs args)
{
    using L = Bs2Layout<STAGES>;
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
    const int num_tiles = args.raster.num_tiles();   // pair tiles (256 x 256)
    const int my_tiles = cluster < num_tiles ? (num_tiles - cluster + num_clusters - 1) / num_clusters : 0;
    WorkSpanT<2> span;                               // stream-K: the pair's steps (identical in both CTAs)
    const int total = [&] {                          // K-block steps of this pair
        if constexpr (SK) {
            span.init(args, KB, num_tiles);
            return span.total;
        } else {
            return my_tiles * KB;
        }
    }();

    auto full_bar = [&](int s) { return sbase + L::OFF_BAR + 8u * s; };
    auto empty_bar = [&](int s) { return sbase + L::OFF_BAR + 8u * (STAGES + s); };
    auto tfull_bar = [&](int b) { return sbase + L::OFF_BAR + 8u * (2 * STAGES + b); };
    auto tempty_bar = [&](int b) { return sbase + L::OFF_BAR + 8u * (2 * STAGES + kBs2NBuf + b); };
    const uint32_t mma_done_bar = sbase + L::OFF_BAR + 8u * (2 * STAGES + 2 * kBs2NBuf);
    auto sa_full_bar = [&](int a) { return sbase + L::OFF_BAR + 8u * (2 * STAGES + 2 * kBs2NBuf + 1 + a); };
    auto sa_empty_bar = [&](int a) {
        return sbase + L::OFF_BAR + 8u * (2 * STAGES + 2 * kBs2NBuf + 1 + kBs2SaSlots + a);
    };
    const uint32_t c_full_bar = sbase + L::OFF_BAR + 8u * (2 * STAGES + 2 * kBs2NBuf + 1 + 2 * kBs2SaSlots);
    const uint32_t c_empty_bar = c_full_bar + 8u;
    const uint32_t part_full_bar = c_full_bar + 16u;    // stream-K: a partial copied into the ring
    const uint32_t part_empty_bar = c_full_bar + 24u;   // stream-K: the promote warps have added it
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 4);
    volatile int *span_smem = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 16);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full_bar(s), 1);                 // even CTA's producer (expect_tx of both CTAs' bytes)
            ptx::mbar_init(empty_bar(s), 1);                // multicast MMA commit
        }
        for (int b = 0; b < kBs2NBuf; ++b) {
            ptx::mbar_init(tfull_bar(b), 1);                // multicast MMA commit
            ptx::mbar_init(tempty_bar(b), 2 * kEpiWarps);   // promote warps of both CTAs (even CTA's copy)
        }
        ptx::mbar_init(mma_done_bar, 2);                    // both issuers' multicast commits
        ptx::mbar_init(c_full_bar, kEpiWarps);              // tile C buffer written
        ptx::mbar_init(c_empty_bar, 1);                     // the store warp's TMA stores have read it
        ptx::mbar_init(part_full_bar, 1);                   // the producer's expect_tx
        ptx::mbar_init(part_empty_bar, kEpiWarps);
        for (int a = 0; a < kBs2SaSlots; ++a) {
            ptx::mbar_init(sa_full_bar(a), 1);
            ptx::mbar_init(sa_empty_bar(a), kEpiWarps);     // this CTA's promote warps
        }
        *abort_flag = 0;
        if constexpr (SK) {
            span_smem[0] = span.u0;
            span_smem[1] = span.total;
            span_smem[2] = span.dp_steps;
            span_smem[3] = span.tile0;
        }
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
        ptx::setmaxnreg_dec<kBs2RegsLow>();
        if (warp == 0) {
            // ------------------------------------------------------------ producer
            // One thread fills every stage and a_scale slot, waiting on each
            // phase by phase (three copies per K block of 32 KiB).
            if (lane == 0) {
                ptx::prefetch_tmap(&tmA);
                ptx::prefetch_tmap(&tmB);
                ptx::prefetch_tmap(&tmSA);
                int it = 0;
                if constexpr (SK) {
                    // stream-K: steps in the span's order (a range may start mid-tile)
                    bool ok = true;
                    int t = 0, kb = 0, row0 = 0, brow0 = 0, seg_kb0 = 0;
                    if (total > 0)
                        span.step(0, t, kb);
                    for (; it < total; ++it, span.advance(it, t, kb)) {
                        if (it == 0 || kb == 0 || it == span.dp_steps) {
                            seg_kb0 = kb;
                            int mb, nb;
                            args.raster.coords(t, mb, nb);
                            row0 = mb * 2 * kBlockM + static_cast<int>(rank) * kBlockM;
                            brow0 = nb * kBs2BN + static_cast<int>(rank) * (kBs2BN / 2);
                        }
                        const int s = it % STAGES;
                        const uint32_t ph = (it / STAGES) & 1;
                        const int a = it % kBs2SaSlots;
                        const uint32_t aph = (it / kBs2SaSlots) & 1;
                        if (!wait_bounded(empty_bar(s), ph ^ 1, abort_flag, args) ||
                            !wait_bounded(sa_empty_bar(a), aph ^ 1, abort_flag, args))
                            break;
                        const uint32_t leader_full = ptx::mapa_shared(full_bar(s), 0);
                        if (rank == 0)
                            ptx::mbar_arrive_expect_tx(full_bar(s), 2 * (L::A_BYTES + L::B_BYTES));
                        ptx::tma_load_2d_pair(sbase + L::OFF_A + s * L::A_BYTES, &tmA, leader_full, kb * kBlockK,
                                              row0);
                        ptx::tma_load_2d_pair(sbase + L::OFF_B + s * L::B_BYTES, &tmB, leader_full, kb * kBlockK,
                                              brow0);
                        ptx::mbar_arrive_expect_tx(sa_full_bar(a), L::SA_BYTES);
                        ptx::tma_load_2d(sbase + L::OFF_SA + a * L::SA_BYTES, &tmSA, sa_full_bar(a), row0, kb);
                    }
                    // A range whose last segment holds K block 0 of a cut tile ends
                    // in a finisher: once the MMAs have read every stage, the
                    // partials of the pairs holding the rest of the tile (the CTA
                    // of this rank in each; one 128 KiB slot fills the ring) are
                    // copied into the ring one after another, and the promote
                    // warps add them from there.
                    int kb_last = 0;
                    if (total > 0)
                        span.step(total - 1, t, kb_last);
                    const int n_parts =
                        it == total && total > 0 && seg_kb0 == 0 && kb_last != KB - 1 ? span.last_worker(num_tiles, t) - cluster : 0;
                    for (int p = 0; p < n_parts && ok; ++p) {
                        const size_t cta2 = 2 * static_cast<size_t>(cluster + 1 + p) + rank;
                        for (int w = 0; w < kEpiWarps && ok; ++w)
                            ok = sk_wait_flag_thread(args.sk_flags + cta2 * kEpiWarps + w, args.sk_token, abort_flag,
                                                     args);
                        if (!ok)
                            break;
                        for (int w = 0; w < kEpiWarps; ++w)   // ready for the next call (nothing rewrites the slot in this one)
                            *reinterpret_cast<volatile unsigned long long *>(args.sk_flags + cta2 * kEpiWarps + w) = 0ull;
                        ptx::fence_proxy_async_global();
                        if (p == 0) {
                            for (int s = 0; s < STAGES && ok; ++s) {
                                const int uses = it > s ? (it - s + STAGES - 1) / STAGES : 0;
                                ok = uses == 0 || wait_bounded(empty_bar(s), (uses - 1) & 1, abort_flag, args);
                            }
                        } else {
                            ok = wait_bounded(part_empty_bar, (p - 1) & 1, abort_flag, args);
                        }
                        if (!ok)
                            break;
                        ptx::mbar_arrive_expect_tx(part_full_bar, kBlockM * kBs2BN * 4);
                        ptx::bulk_load(sbase + L::OFF_A, args.sk_partial + cta2 * (kBs2BN * kBlockM),
                                       kBlockM * kBs2BN * 4, part_full_bar);
                        wait_teardown(part_full_bar, p & 1, args);   // landed before the next copy or the exit
                    }
                } else {
                    bool ok = true;
                    for (int t = cluster; t < num_tiles && ok; t += num_clusters) {
                        int mb, nb;
                        args.raster.coords(t, mb, nb);
                        const int row0 = mb * 2 * kBlockM + static_cast<int>(rank) * kBlockM;
                        const int brow0 = nb * kBs2BN + static_cast<int>(rank) * (kBs2BN / 2);
                        for (int kb = 0; kb < KB; ++kb, ++it) {
                            const int s = it % STAGES;
                            const uint32_t ph = (it / STAGES) & 1;
                            const int a = it % kBs2SaSlots;
                            const uint32_t aph = (it / kBs2SaSlots) & 1;
                            if (!wait_bounded(empty_bar(s), ph ^ 1, abort_flag, args) ||
                                !wait_bounded(sa_empty_bar(a), aph ^ 1, abort_flag, args)) {
                                ok = false;
                                break;
                            }
                            const uint32_t leader_full = ptx::mapa_shared(full_bar(s), 0);
                            if (rank == 0)
                                ptx::mbar_arrive_expect_tx(full_bar(s), 2 * (L::A_BYTES + L::B_BYTES));
                            ptx::tma_load_2d_pair(sbase + L::OFF_A + s * L::A_BYTES, &tmA, leader_full, kb * kBlockK,
                                                  row0);
                            ptx::tma_load_2d_pair(sbase + L::OFF_B + s * L::B_BYTES, &tmB, leader_full, kb * kBlockK,
                                                  brow0);
                            ptx::mbar_arrive_expect_tx(sa_full_bar(a), L::SA_BYTES);
                            ptx::tma_load_2d(sbase + L::OFF_SA + a * L::SA_BYTES, &tmSA, sa_full_bar(a), row0, kb);
                        }
                    }
                }
                // Every load this thread issued must have landed before the CTA
                // exits: the last use of each of its stages and slots (earlier
                // uses landed before they could be refilled). The odd CTA learns
                // it from the even CTA's multicast stage release.
                for (int s = 0; s < STAGES; ++s) {
                    const int uses = it > s ? (it - s + STAGES - 1) / STAGES : 0;
                    if (uses > 0)
                        wait_teardown(rank == 0 ? full_bar(s) : empty_bar(s), (uses - 1) & 1, args);
                }
                for (int a = 0; a < kBs2SaSlots; ++a) {
                    const int uses = it > a ? (it - a + kBs2SaSlots - 1) / kBs2SaSlots : 0;
                    if (uses > 0)
                        wait_teardown(sa_full_bar(a), (uses - 1) & 1, args);
                }
            }
        } else if ((warp == 1 || warp == 2) && lane == 0 && rank == 0) {
            // ------------------------------------------------ MMA issuers (even CTA)
            // Warp 1 issues the even steps (TMEM buffer 0, even stages), warp 2
            // the odd steps (buffer 1, odd stages).
            const int par = warp - 1;
            constexpr uint32_t idesc = ptx::idesc_f8f6f4_e4m3(2 * kBlockM, kBs2BN);
            for (int it = par; it < total; it += 2) {
                const int s = it % STAGES;
                const uint32_t ph = (it / STAGES) & 1;
                const int buf = it % kBs2NBuf;
                const uint32_t tph = (it / kBs2NBuf) & 1;
                if (!wait_bounded(full_bar(s), ph, abort_flag, args) ||
                    !wait_bounded(tempty_bar(buf), tph ^ 1, abort_flag, args))
                    break;
                ptx::tc_fence_after();
                const uint64_t adesc = ptx::desc_kmajor_sw128(sbase + L::OFF_A + s * L::A_BYTES);
                const uint64_t bdesc = ptx::desc_kmajor_sw128(sbase + L::OFF_B + s * L::B_BYTES);
                const uint32_t d = tmem_base + static_cast<uint32_t>(buf * kBs2BN);
#pragma unroll
                for (int kk = 0; kk < kBlockK / kMmaK; ++kk)
                    ptx::mma_f8f6f4_pair(d, adesc + 2 * kk, bdesc + 2 * kk, idesc, kk > 0 ? 1u : 0u);
                ptx::tc_commit_pair_mc(tfull_bar(buf), 0x3);
                ptx::tc_commit_pair_mc(empty_bar(s), 0x3);
            }
            ptx::tc_commit_pair_mc(mma_done_bar, 0x3);
        }
        if (warp == 3 && lane == 0) {
            // -------------------------------------------------------- C store
            // Once the eight promote warps have written a tile into the buffer
            // (c_full), four TMA stores of 64 columns x 128 rows; the buffer is
            // released (c_empty) as soon as they have read it.
            // Under stream-K a segment that starts past K block 0 (the head of a
            // tile begun by an earlier pair) ends in a published partial, not in
            // a stored tile.
            auto store_tile = [&](int t) {
                int mb, nb;
                args.raster.coords(t, mb, nb);
                const int y = mb * 2 * kBlockM + static_cast<int>(rank) * kBlockM;
#pragma unroll
                for (int c = 0; c < kBs2BN / 64; ++c) {
                    const int x = nb * kBs2BN + c * 64;
                    if (x < args.N && y < args.M)
                        ptx::tma_store_2d(&tmC, sbase + L::OFF_C + c * (kBlockM * 128), x, y);
                }
                ptx::bulk_commit();
                ptx::bulk_wait_read_all();
                ptx::mbar_arrive(c_empty_bar);
            };
            if constexpr (SK) {
                for (int g = 0, n = 0; g < total;) {
                    int t, kb0;
                    span.step(g, t, kb0);
                    g += (KB - kb0) < (total - g) ? (KB - kb0) : (total - g);
                    if (kb0 != 0)
                        continue;
                    if (!wait_bounded(c_full_bar, n & 1, abort_flag, args))
                        break;
                    ++n;
                    store_tile(t);
                }
            } else {
                for (int t = cluster, n = 0; t < num_tiles; t += num_clusters, ++n) {
                    if (!wait_bounded(c_full_bar, n & 1, abort_flag, args))
                        break;
                    store_tile(t);
                }
            }
            ptx::bulk_wait_all();
        }
        // No pair MMA may still write this CTA's tensor memory when it is freed.
        if (warp == 1 && lane == 0)
            wait_teardown(mma_done_bar, 0, args);
    } else {
        ptx::setmaxnreg_inc<kBs2RegsHigh>();
        // ------------------------------------------------- promote + epilogue
        constexpr int HALF = kBs2BN / 2;             // columns per thread
        const int ew = warp - 4;                     // 0..7
        const int wg = ew >> 2;                      // column half
        const int q = warp & 3;                      // TMEM lane quadrant this warp may access
        const int row = q * 32 + lane;               // row of this CTA's 128
        const int NB = (args.N + 127) / 128;
        int n_stored = 0;   // tiles written to the tile C buffer

        float acc[HALF];
        int it = 0;
        bool ok = true;
        // b_scale of this thread's 128-column N block, 32 K blocks ahead: lane l
        // holds K block 32*c + l of batch c (taken with a shuffle); batch c+1 is
        // requested when batch c starts. Set per tile (per segment under
        // stream-K).
        const float *sbrow = nullptr;
        float sb_cur = 0.f, sb_next = 0.f;
        // One K block: acc (+)= P_kb * (sa * sb). A tile's (segment's) first K
        // block is peeled off the loop and sets the accumulators (an FMA onto
        // zero, no separate reset), so the loop body stays branch-free.
        auto kstep = [&](int kb, auto first) -> bool {
            const float sb = __shfl_sync(0xffffffffu, sb_cur, kb & 31);
            if ((kb & 31) == 31) {
                sb_cur = sb_next;
                sb_next = sbrow && kb + 33 + lane < KB ? ptx::ldg_nc_f32(sbrow + kb + 33 + lane) : 0.f;
            }
            const int a = it % kBs2SaSlots;
            const uint32_t aph = (it / kBs2SaSlots) & 1;
            const int buf = it % kBs2NBuf;
            const uint32_t tph = (it / kBs2NBuf) & 1;
            if (!wait_bounded_warp(tfull_bar(buf), tph, abort_flag, args) ||
                !wait_bounded_warp(sa_full_bar(a), aph, abort_flag, args))
                return false;
            ptx::tc_fence_after();
            const float sa = reinterpret_cast<const float *>(smem + L::OFF_SA + a * L::SA_BYTES)[row];
            const float scale = sa * sb;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(buf * kBs2BN + wg * HALF);
            // Two 64-column rounds; the buffer is released once the second
            // round is loaded.
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t r0[32], r1[32];
                ptx::tmem_ld_32x32b_x32(taddr + h * 64, r0);
                ptx::tmem_ld_32x32b_x32(taddr + h * 64 + 32, r1);
                ptx::tmem_wait_ld();
                if (h == 1) {
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        // the even CTA's barrier, by its cluster address from
                        // either CTA (the loads above have completed)
                        ptx::mbar_arrive_cluster_relaxed(ptx::mapa_shared(tempty_bar(buf), 0));
                        ptx::mbar_arrive(sa_empty_bar(a));
                    }
                }
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    acc[h * 64 + j] = fmaf(__uint_as_float(r0[j]), scale, decltype(first)::value ? 0.f : acc[h * 64 + j]);
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    acc[h * 64 + 32 + j] =
                        fmaf(__uint_as_float(r1[j]), scale, decltype(first)::value ? 0.f : acc[h * 64 + 32 + j]);
            }
            ++it;
            return true;
        };
        // The tile into the tile buffer once the store warp has read out the
        // previous one, then on to the next tile.
        auto stage_tile = [&]() -> bool {
            if (!wait_bounded_warp(c_empty_bar, (n_stored & 1) ^ 1, abort_flag, args))
                return false;
#pragma unroll
            for (int c = 0; c < HALF / 64; ++c)
                stage_c64_row(sbase + L::OFF_C + (wg * (HALF / 64) + c) * (kBlockM * 128), row, acc + c * 64);
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(c_full_bar);
            ++n_stored;
            return true;
        };
        if constexpr (!SK) {
            for (int t = cluster; t < num_tiles && ok; t += num_clusters) {
                {
                    int mb, nb;
                    args.raster.coords(t, mb, nb);
                    const int nblk = (nb * kBs2BN + wg * HALF) >> 7;
                    sbrow = nblk < NB ? args.b_scale + static_cast<size_t>(nblk) * KB : nullptr;
                }
                sb_cur = sbrow && lane < KB ? ptx::ldg_nc_f32(sbrow + lane) : 0.f;
                sb_next = sbrow && 32 + lane < KB ? ptx::ldg_nc_f32(sbrow + 32 + lane) : 0.f;
                ok = kstep(0, std::true_type{});
                for (int kb = 1; kb < KB && ok; ++kb)
                    ok = kstep(kb, std::false_type{});
                if (!ok || !stage_tile())
                    break;
            }
        } else {
            // The span comes from shared memory (written once by thread 0)
            // wherever it is needed, so that only the step index, the loop's
            // K blocks and the segment's first step stay in registers across the
            // K loop, next to the 128 accumulators and the 64 loaded partials.
            auto span_of = [&]() {
                WorkSpanT<2> sp;
                sp.u0 = span_smem[0];
                sp.total = span_smem[1];
                sp.dp_steps = span_smem[2];
                sp.tile0 = span_smem[3];
                sp.KB = KB;
                return sp;
            };
            while (true) {
                // One segment: steps seg_start .., K blocks kb0 .. kb_end-1 of one
                // tile; the tile and its coordinates are recomputed after it.
                const int seg_start = it;
                int kb_first, kb_end;
                {
                    const WorkSpanT<2> sp = span_of();
                    if (seg_start >= sp.total)
                        break;
                    int t, kb0, mb, nb;
                    sp.step(seg_start, t, kb0);
                    kb_end = kb0 + ((KB - kb0) < (sp.total - seg_start) ? (KB - kb0) : (sp.total - seg_start));
                    args.raster.coords(t, mb, nb);
                    const int nblk = (nb * kBs2BN + wg * HALF) >> 7;
                    sbrow = nblk < NB ? args.b_scale + static_cast<size_t>(nblk) * KB : nullptr;
                    const int kb_base = kb0 & ~31;
                    sb_cur = sbrow && kb_base + lane < KB ? ptx::ldg_nc_f32(sbrow + kb_base + lane) : 0.f;
                    sb_next = sbrow && kb_base + 32 + lane < KB ? ptx::ldg_nc_f32(sbrow + kb_base + 32 + lane) : 0.f;
                    ok = kstep(kb0, std::true_type{});
                    kb_first = kb0 + 1;
                }
                for (int kb = kb_first; kb < kb_end && ok; ++kb)
                    ok = kstep(kb, std::false_type{});
                if (!ok)
                    break;
                const WorkSpanT<2> sp = span_of();
                const int num_tiles_ = args.raster.num_tiles();
                int t, kb0, mb, nb;
                sp.step(seg_start, t, kb0);
                const int kb_last = kb_end - 1;
                args.raster.coords(t, mb, nb);
                // The hand-off, warp by warp: warp ew of both CTAs of every pair
                // owns the same 32 rows x 128 columns of its CTA's half of a
                // tile, in slot layout [column/4][row] (a warp's store is 512
                // contiguous bytes). A warp whose 32 rows all lie past M moves
                // no data (its counterpart in the other pair decides the same
                // way) but still raises its flag.
                const uint32_t slice = static_cast<uint32_t>(wg * HALF / 4) * kBlockM + static_cast<uint32_t>(row);
                const bool rows_live = mb * 2 * kBlockM + static_cast<int>(rank) * kBlockM + q * 32 < args.M;
                if (kb0 > 0) {
                    // Head of a tile begun by an earlier pair: publish the scaled partial.
                    if (rows_live) {
                        float *dst = args.sk_partial + static_cast<size_t>(blockIdx.x) * (kBs2BN * kBlockM) + 4 * slice;
#pragma unroll
                        for (int j = 0; j < HALF; j += 4)
                            ptx::st_global_v4_f32(dst + static_cast<size_t>(j / 4) * kBlockM * 4, acc[j], acc[j + 1],
                                                  acc[j + 2], acc[j + 3]);
                    }
                    // The warp barrier orders every lane's stores before lane 0's
                    // release store of the flag, and a release is cumulative: a
                    // finisher that acquires the flag sees the whole slice.
                    __syncwarp();
                    if (lane == 0)
                        ptx::st_release_gpu_u64(args.sk_flags + static_cast<size_t>(blockIdx.x) * kEpiWarps + ew,
                                                args.sk_token);
                    continue;
                }
                if (kb_last != KB - 1) {
                    // This pair holds K block 0 of a cut tile: add the partials of
                    // the pairs that hold the rest of it, which the producer copies
                    // into the operand ring one after another.
                    const int n_parts = sp.last_worker(num_tiles_, t) - (static_cast<int>(blockIdx.x) >> 1);
                    for (int p = 0; p < n_parts; ++p) {
                        if (!wait_bounded_warp(part_full_bar, p & 1, abort_flag, args)) {
                            ok = false;
                            break;
                        }
                        if (rows_live) {
                            const uint32_t src = sbase + L::OFF_A + 16 * slice;
#pragma unroll
                            for (int j = 0; j < HALF; j += 4) {
                                const float4 v = ptx::ld_shared_v4_f32(src + (j / 4) * kBlockM * 16);
                                acc[j] += v.x;
                                acc[j + 1] += v.y;
                                acc[j + 2] += v.z;
                                acc[j + 3] += v.w;
                            }
                        }
                        __syncwarp();
                        if (lane == 0)
                            ptx::mbar_arrive(part_empty_bar);
                    }
                    if (!ok)
                        break;
                }
                if (!stage_tile())
                    break;
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::cluster_sync();   // no remote arrive or multicast commit may target an exited CTA
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, L::TMEM_COLS);
    }
}

// `clusters` CTA pairs, at most the co-resident count (stream-K finishers wait
// for the pairs after them); the stream-K instance when args.sk is set.
template <int STAGES>
cudaError_t launch_blockscale_pair(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmSA,
                                   const CUtensorMap &tmC, const GemmArgs &args, int clusters, cudaStream_t stream)
{
    using L = Bs2Layout<STAGES>;
    auto kern = args.sk ? fp8bs_blockscale_pair_kernel<STAGES, true> : fp8bs_blockscale_pair_kernel<STAGES, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::DYN_SMEM);
    if (e != cudaSuccess)
        return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(kBs2Threads);
    cfg.dynamicSmemBytes = L::DYN_SMEM;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmSA, tmC, args);
}

// Co-resident clusters of two CTAs for this kernel on the current device (both
// instances use the same resources).
template <int STAGES>
cudaError_t max_bs_pair_clusters(int *out)
{
    using L = Bs2Layout<STAGES>;
    for (auto kern : {fp8bs_blockscale_pair_kernel<STAGES, false>, fp8bs_blockscale_pair_kernel<STAGES, true>}) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::DYN_SMEM);
        if (e != cudaSuccess)
            return e;
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(kBs2Threads);
    cfg.dynamicSmemBytes = L::DYN_SMEM;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(out, fp8bs_blockscale_pair_kernel<STAGES, false>, &cfg);
}

template cudaError_t launch_blockscale_pair<4>(const CUtensorMap &, const CUtensorMap &, const CUtensorMap &,
                                               const CUtensorMap &, const GemmArgs &, int, cudaStream_t);
template cudaError_t max_bs_pair_clusters<4>(int *);

} // namespace fp8bs
