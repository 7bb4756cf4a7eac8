// FP8 block-scaled GEMM kernel for sm_103a.
//
// Computes C[m,n] = bf16( sum_kb P_kb[m,n] * a_scale[m,kb] * b_scale[n/128,kb] ),
// P_kb = the unscaled fp8 product over the 128-wide K block kb (skill card
// "FlyDSL fp8 blockscale GEMM", section "Mechanism A": keep the matrix unit
// unscaled and apply the arbitrary fp32 block scales in software after it, one
// promote per K block, because those scales are not powers of two).
//
// Work schedule (WorkSpan in common.cuh): one CTA per tile, or stream-K, where
// every CTA takes an equal share of the (tile, K block) units, so a partial last
// wave of tiles leaves no SM idle. A tile cut between CTAs is summed by the CTA
// holding its first K block: the others publish their scaled fp32 partials
// (global workspace, one release flag per promote warp) before anything else,
// and the finisher adds them after its own last K block. Sums stay in fp32 and
// every partial is scaled before it is added, so the result is the same sum
// in another order.
//
// Persistent, warp-specialised, one CTA per SM, 12 warps (3 warpgroups):
//   warps 0, 3  TMA producers, warp 0 for the even K-block steps and warp 3 for
//               the odd ones (warp 0 alone with an odd stage count):
//               A tile [128 x 128] e4m3 and B tile [BN x 128] e4m3
//               of one K block into stage s of a STAGES-deep shared-memory ring
//               (full/empty mbarriers, a stage is freed by the MMA commit), and
//               the a_scale slice [128] fp32 of the K block into a separate
//               kSaSlots-deep ring freed by the promote warps.
//   warps 1, 2  MMA issuers (one thread each, warp 1 even steps, warp 2 odd
//               steps; warp 1 also allocates TMEM): four
//               tcgen05.mma.kind::f8f6f4 (M128 x BN x K32) overwrite TMEM partial
//               buffer (kb % NBUF) with P_kb, NBUF = 512 / BN buffers (2 for
//               BN = 256, 4 for BN = 128), so the MMA can run NBUF-1 K blocks
//               ahead of the promote; tcgen05.commit releases the stage and
//               signals the buffer. Issuing an MMA while the tensor pipe is busy
//               stalls the issuer's SM sub-partition, and the promote warps on it
//               fall behind the others; splitting the issue (and the TMA issue)
//               over two sub-partitions halves that lag.
//   warps 4..11 promote + epilogue: warp w reads TMEM lanes 32*(w%4).., column half
//               (w-4)/4, so each thread owns one row of C and BN/2 columns, all in
//               one 128-column N block, i.e. one b_scale value. Per K block:
//               acc += P_kb * (sa * sb) in fp32 registers. When the thread's
//               whole slice fits in registers (BN = 128) it is loaded, the TMEM
//               buffer is released, and only then promoted, so the FMAs are off
//               the MMA's critical path; for BN = 256 the buffer is released
//               after the last 64-column round.
//               After the last K block: bf16 convert, 64-byte-swizzled staging
//               of 32 x 32 chunks, TMA store (tails clipped by the tensor map).
//               With three stages (shapes with few K blocks per tile) the freed
//               shared memory holds a whole 128 x 256 bf16 C tile: the promote
//               warps convert their rows into it and go straight on to the next
//               tile, and warp 3 (idle with one producer) stores it by TMA.
//   warp 3 (three stages) C store: waits for the eight promote warps to fill
//               the tile buffer, issues four 64-column x 128-row TMA stores,
//               waits for them to read the buffer, releases it.
// Registers: the launch gives 168 per thread (3 warps per SM sub-partition);
// warpgroup 0 drops to 40 and the two promote warpgroups rise to 232, so one
// sub-partition holds 40 + 232 + 232 = 504 <= 512 registers per lane and the
// 128 fp32 accumulators plus 64 in-flight partials per thread fit without spills.
#include "common.cuh"

namespace fp8bs {

constexpr int kBsThreads = (4 + kEpiWarps) * 32;
// Register split (see the header comment): 40 / 232 for the 256-wide tile,
// whose promote holds 128 accumulators and 64 partials per thread; 56 / 224
// for the narrower tiles (at most 80 + 80), which gives the producer slack.
template <int BN> constexpr int kBsRegsLow = BN == 256 ? 40 : 56;
template <int BN> constexpr int kBsRegsHigh = BN == 256 ? 232 : 224;
constexpr int kSaSlots = 16;   // a_scale ring depth (>= STAGES + NBUF, so it never holds back A/B)

template <int BN, int STAGES>
struct BsLayout {
    // Three stages leave room for a whole C tile (128 x 256 bf16, 64 KiB, four
    // 128-byte-swizzled 64-column chunks), stored by a warp of its own, for
    // shapes with few K blocks per tile, where the epilogue is a large part
    // of each tile. (An E4M3 C keeps the per-warp 2 KiB staging, inside it.)
    static constexpr bool TILE_C = STAGES == 3;
    static constexpr int C_BYTES = kCStageBytes;    // per epilogue warp (per-warp staging)
    static constexpr int C_AREA = TILE_C ? kBlockM * BN * 2 : kEpiWarps * C_BYTES;
    static constexpr int A_BYTES = kBlockM * kBlockK;
    static constexpr int B_BYTES = BN * kBlockK;
    static constexpr int SA_BYTES = kBlockM * 4;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_SA = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_C = (OFF_SA + kSaSlots * SA_BYTES + 1023) / 1024 * 1024;
    static constexpr int OFF_BAR = OFF_C + C_AREA;
    static constexpr int NBUF = 512 / BN;        // TMEM partial buffers
    static_assert(NBUF % 2 == 0, "two MMA issuers split the buffers by parity");
    static_assert(STAGES % 2 == 1 || kSaSlots % 2 == 0, "two producers split the a_scale slots by parity");
    // full[S], empty[S], tfull[NBUF], tempty[NBUF], mma_done, sa_full[kSaSlots], sa_empty[kSaSlots],
    // c_full, c_empty
    static constexpr int NBAR = 2 * STAGES + 2 * NBUF + 1 + 2 * kSaSlots + 2;
    static_assert(!TILE_C || (BN == 256 && C_AREA >= kEpiWarps * C_BYTES), "tile C buffer");
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int BYTES = OFF_MISC + 16;
    static constexpr int DYN_SMEM = BYTES + 1024;   // slack to align the base to 1024
    static constexpr int TMEM_COLS = 512;
    static_assert(DYN_SMEM <= 232448, "shared memory budget");
    static_assert(BN == 128 || BN == 256, "tile width");
};

// SK: the stream-K instance (256-wide dense tile only). The hand-off lives in
// its own instance: compiled into the one-CTA-per-tile instance, where it never
// runs, it made that instance 2-7% slower (4096x2048x7168 63.3 -> 59.1 us
// without it, 4096x65536x1536 406 -> 387 us, 16384x7168x768 at three stages
// 106.3 -> 102.6 us; same bits).
template <int BN, int STAGES, bool MOE, bool SK>
__global__ void __launch_bounds__(kBsThreads, 1)
    fp8bs_blockscale_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmC,
                            const GemmArgs args)
{
    using L = BsLayout<BN, STAGES>;
    static_assert(!SK || (BN == 256 && !MOE), "stream-K runs with the dense 256-wide tile");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = ptx::smem_u32(smem_raw);
    const uint32_t sbase = (raw_s + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw_s);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int KB = args.K / kBlockK;
    // Grouped mode: the leader count is device data (graph-safe), read by every role.
    const int n_leaders = MOE ? moe_leader_count(args) : 1;
    const int tiles = MOE ? n_leaders * args.moe_n_tiles : args.raster.num_tiles();

    auto full_bar = [&](int s) { return sbase + L::OFF_BAR + 8u * s; };
    auto empty_bar = [&](int s) { return sbase + L::OFF_BAR + 8u * (STAGES + s); };
    constexpr int NT = L::NBUF;   // TMEM buffer barriers
    auto tfull_bar = [&](int b) { return sbase + L::OFF_BAR + 8u * (2 * STAGES + b); };
    auto tempty_bar = [&](int b) { return sbase + L::OFF_BAR + 8u * (2 * STAGES + NT + b); };
    const uint32_t mma_done_bar = sbase + L::OFF_BAR + 8u * (2 * STAGES + 2 * NT);
    auto sa_full_bar = [&](int a) { return sbase + L::OFF_BAR + 8u * (2 * STAGES + 2 * NT + 1 + a); };
    auto sa_empty_bar = [&](int a) { return sbase + L::OFF_BAR + 8u * (2 * STAGES + 2 * NT + 1 + kSaSlots + a); };
    const uint32_t c_full_bar = sbase + L::OFF_BAR + 8u * (2 * STAGES + 2 * NT + 1 + 2 * kSaSlots);
    const uint32_t c_empty_bar = c_full_bar + 8u;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);              // MMA commit
        }
        for (int a = 0; a < kSaSlots; ++a) {
            ptx::mbar_init(sa_full_bar(a), 1);
            ptx::mbar_init(sa_empty_bar(a), kEpiWarps);   // every promote warp has read the slice
        }
        for (int b = 0; b < L::NBUF; ++b) {
            ptx::mbar_init(tfull_bar(b), 1);
            ptx::mbar_init(tempty_bar(b), kEpiWarps);     // every promote warp has loaded its slice
        }
        ptx::mbar_init(mma_done_bar, 2);                  // both MMA issuers
        ptx::mbar_init(c_full_bar, kEpiWarps);            // tile C buffer filled (three stages)
        ptx::mbar_init(c_empty_bar, 1);                   // tile C buffer read by its TMA stores
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

    if (warp < 4) {
    ptx::setmaxnreg_dec<kBsRegsLow<BN>>();
    // Parity waits are unambiguous only while a barrier is at most one phase
    // ahead of its waiter, i.e. when one thread waits on it for every phase
    // in turn. With an even stage count each stage (like each a_scale slot and
    // TMEM buffer) belongs to the producer and issuer of one step parity. With
    // an odd count a stage's uses alternate between parities, so one producer
    // thread fills every stage, and each issuer waits for its TMEM buffer
    // before the stage: the buffer is released only after the promote of the
    // step before, hence after the stage's previous use was consumed.
    constexpr bool kOneProducer = STAGES % 2 == 1;
    if (warp == 0 || (warp == 3 && !kOneProducer)) {
        // ----------------------------------------------------------- producers
        // Warp 0 fills the stages of the even steps, warp 3 those of the odd
        // steps (with an even STAGES each stage and a_scale slot belongs to
        // one of them and is waited on by that thread alone, in order of its
        // phases); with an odd STAGES warp 0 fills all of them.
        if (lane == 0) {
            const int par = warp == 3 ? 1 : 0;
            ptx::prefetch_tmap(&tmA);
            ptx::prefetch_tmap(&tmB);
            ptx::prefetch_tmap(&tmSA);
            WorkSpan span;
            span.init(args, KB, tiles);
            int it = 0;
            int t, kb;
            TileGeo geo = {};
            span.step(0, t, kb);
            for (; it < span.total; ++it, span.advance(it, t, kb)) {
                if (it == 0 || kb == 0 || it == span.dp_steps)   // a new tile (a stream-K range may start mid-tile)
                    geo = tile_geo<MOE>(args, t, BN, n_leaders);
                if (!kOneProducer && (it & 1) != par)
                    continue;
                const int s = it % STAGES;
                const uint32_t ph = (it / STAGES) & 1;
                const int a = it % kSaSlots;
                const uint32_t aph = (it / kSaSlots) & 1;
                if (!wait_bounded(empty_bar(s), ph ^ 1, abort_flag, args) ||
                    !wait_bounded(sa_empty_bar(a), aph ^ 1, abort_flag, args))
                    break;
                ptx::mbar_arrive_expect_tx(full_bar(s), L::A_BYTES + L::B_BYTES);
                ptx::tma_load_2d(sbase + L::OFF_A + s * L::A_BYTES, &tmA, full_bar(s), kb * kBlockK, geo.a_row);
                ptx::tma_load_2d(sbase + L::OFF_B + s * L::B_BYTES, &tmB, full_bar(s), kb * kBlockK, geo.b_row);
                ptx::mbar_arrive_expect_tx(sa_full_bar(a), L::SA_BYTES);
                ptx::tma_load_2d(sbase + L::OFF_SA + a * L::SA_BYTES, &tmSA, sa_full_bar(a), geo.a_row, kb);
            }
            // Every load issued must have landed before the CTA exits: wait for
            // the last use of each stage this producer filled (earlier uses
            // landed before the stage could be refilled).
            for (int s = kOneProducer ? 0 : par; s < STAGES; s += kOneProducer ? 1 : 2) {
                const int uses = it > s ? (it - s + STAGES - 1) / STAGES : 0;
                if (uses > 0)
                    wait_teardown(full_bar(s), (uses - 1) & 1, args);
            }
            for (int a = kOneProducer ? 0 : par; a < kSaSlots; a += kOneProducer ? 1 : 2) {
                const int uses = it > a ? (it - a + kSaSlots - 1) / kSaSlots : 0;
                if (uses > 0)
                    wait_teardown(sa_full_bar(a), (uses - 1) & 1, args);
            }
        }
    } else if (warp == 1 || warp == 2) {
        // -------------------------------------------------------- MMA issuers
        // Warp 1 issues the MMAs of the even steps, warp 2 those of the odd
        // steps (NBUF is even, so each TMEM buffer, like each stage, has one
        // issuer). Issuing tcgen05.mma stalls the issuing warp's SM
        // sub-partition while the tensor pipe is busy, and the promote warps
        // beside it fall behind; two issuers halve that per sub-partition.
        // (Three would make two threads wait on one buffer's barrier for
        // different phases, which a parity wait cannot tell apart.)
        if (lane == 0) {
            const int par = warp - 1;
            constexpr uint32_t idesc = ptx::idesc_f8f6f4_e4m3(kBlockM, BN);
            WorkSpan span;
            span.init(args, KB, tiles);
            for (int it = par; it < span.total; it += 2) {
                const int s = it % STAGES;
                const uint32_t ph = (it / STAGES) & 1;
                const int buf = it % L::NBUF;
                const uint32_t tph = (it / L::NBUF) & 1;
                // The stage and the TMEM buffer; with an odd stage count the
                // buffer first, whose release orders the stage wait after the
                // stage's previous use (see kOneProducer).
                if (kOneProducer && !wait_bounded(tempty_bar(buf), tph ^ 1, abort_flag, args))
                    break;
                if (!wait_bounded(full_bar(s), ph, abort_flag, args))
                    break;
                if (!kOneProducer && !wait_bounded(tempty_bar(buf), tph ^ 1, abort_flag, args))
                    break;
                ptx::tc_fence_after();
                // One N = BN MMA per 32-wide K slice: on the 256-wide tile, two
                // N = 128 halves with barriers of their own measured slower
                // (4096x2048x7168 64.1 -> 61.7 us, 16384x1536x7168 153.0 ->
                // 149.1 us without the split): twice the MMA instructions, and
                // issuing them holds up the promote warps of the issuer's SM
                // sub-partition.
                const uint64_t adesc = ptx::desc_kmajor_sw128(sbase + L::OFF_A + s * L::A_BYTES);
                const uint64_t bdesc = ptx::desc_kmajor_sw128(sbase + L::OFF_B + s * L::B_BYTES);
                const uint32_t d = tmem_base + static_cast<uint32_t>(buf * BN);
#pragma unroll
                for (int kk = 0; kk < kBlockK / kMmaK; ++kk)
                    ptx::mma_f8f6f4(d, adesc + 2 * kk, bdesc + 2 * kk, idesc, kk > 0 ? 1u : 0u);
                ptx::tc_commit(tfull_bar(buf));
                ptx::tc_commit(empty_bar(s));
            }
            // No MMA may still be running when the tensor memory is freed.
            ptx::tc_commit(mma_done_bar);
            wait_teardown(mma_done_bar, 0, args);
        }
    } else if (L::TILE_C && warp == 3 && !args.c_e4m3) {
        // ---------------------------------------------- C store (three stages)
        // The tiles this CTA stores are its segments that start at K block 0
        // (whole tiles, and under stream-K the tiles it finishes), in the
        // promote warps' order.
        if (lane == 0) {
            WorkSpan span;
            span.init(args, KB, tiles);
            int n_stored = 0;
            for (int it = 0; it < span.total;) {
                int t, kb0;
                span.step(it, t, kb0);
                it += (KB - kb0) < (span.total - it) ? (KB - kb0) : (span.total - it);
                if (kb0 != 0)
                    continue;
                if (!wait_bounded(c_full_bar, n_stored & 1, abort_flag, args))
                    break;
                const TileGeo geo = tile_geo<MOE>(args, t, BN, n_leaders);
#pragma unroll
                for (int c = 0; c < BN / 64; ++c) {
                    const int x = geo.nb * BN + c * 64;
                    if (x < args.N && geo.a_row < args.M)
                        ptx::tma_store_2d(&tmC, sbase + L::OFF_C + c * (kBlockM * 128), x, geo.a_row);
                }
                ptx::bulk_commit();
                ptx::bulk_wait_read_all();
                ptx::mbar_arrive(c_empty_bar);
                ++n_stored;
            }
            ptx::bulk_wait_all();
        }
    }
    } else {
        ptx::setmaxnreg_inc<kBsRegsHigh<BN>>();
        // ------------------------------------------------- promote + epilogue
        constexpr int HALF = BN / 2;                 // columns per thread
        constexpr int kChunk = 16;                   // columns per TMEM load (narrow tile)
        constexpr int NCH = HALF / kChunk;
        constexpr bool kEarlyRelease = HALF <= 64;   // the slice fits next to the accumulator
        constexpr bool kSk = SK;                     // the instance with the stream-K hand-off
        static_assert(HALF % kCChunkCols == 0, "epilogue chunking");
        const int ew = warp - 4;                     // 0..7
        const int wg = ew >> 2;                      // column half
        const int q = warp & 3;                      // TMEM lane quadrant this warp may access
        const int row = q * 32 + lane;               // row of the tile
        const int NB = (args.N + 127) / 128;
        const uint32_t cstage = sbase + L::OFF_C + ew * L::C_BYTES;
        int n_stored = 0;   // tiles handed to the C store warp (three stages)
        WorkSpan span;
        span.init(args, KB, tiles);
        const int total = span.total;

        // b_scale of flattened step g for the 128-column N block of this thread's
        // columns (a slice of 64 or 128 columns never straddles two). Lane l of
        // the warp loads step 32*b + l of batch b; the value for step g is taken
        // with a shuffle. Batch b+1 is requested when batch b starts, so its
        // loads have 32 K blocks to land.
        auto sb_lane_load = [&](int g) -> float {
            if (g >= total)
                return 0.f;
            int t, kb;
            span.step(g, t, kb);
            const TileGeo gg = tile_geo<MOE>(args, t, BN, n_leaders);
            const int nblk = (gg.nb * BN + wg * HALF) >> 7;
            // grouped mode: b_scale is [expert][ceil(N/128)][K/128]
            return nblk < NB ? ptx::ldg_nc_f32(args.b_scale + (static_cast<size_t>(gg.expert) * NB + nblk) * KB + kb)
                             : 0.f;
        };
        float sb_cur = sb_lane_load(lane);
        float sb_next = sb_lane_load(32 + lane);

        float acc[HALF];
        int it = 0;
        bool ok = true;
        while (it < total) {
            // One segment: steps seg_start .. seg_end-1, the K blocks kb0.. of one
            // tile. Only the two step indices stay live across the K loop; the
            // tile and its coordinates are recomputed after it.
            const int seg_start = it;
            int seg_end;
            {
                int t, kb0;
                span.step(it, t, kb0);
                seg_end = it + ((KB - kb0) < (total - it) ? (KB - kb0) : (total - it));
            }
#pragma unroll
            for (int j = 0; j < HALF; ++j)
                acc[j] = 0.f;
            for (; it < seg_end; ++it) {
                const float sb = __shfl_sync(0xffffffffu, sb_cur, it & 31);
                if ((it & 31) == 31) {
                    sb_cur = sb_next;
                    sb_next = sb_lane_load(it + 33 + lane);
                }
                const int a = it % kSaSlots;
                const uint32_t aph = (it / kSaSlots) & 1;
                const int buf = it % L::NBUF;
                const uint32_t tph = (it / L::NBUF) & 1;
                if (!wait_bounded_warp(tfull_bar(buf), tph, abort_flag, args) ||
                    !wait_bounded_warp(sa_full_bar(a), aph, abort_flag, args)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const float sa = reinterpret_cast<const float *>(smem + L::OFF_SA + a * L::SA_BYTES)[row];
                const float scale = sa * sb;
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                       static_cast<uint32_t>(buf * BN + wg * HALF);
                if constexpr (kEarlyRelease) {
                    uint32_t part[HALF];
#pragma unroll
                    for (int c = 0; c < NCH; ++c)
                        ptx::tmem_ld_32x32b_x16(taddr + kChunk * c, part + kChunk * c);
                    ptx::tmem_wait_ld();
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        ptx::mbar_arrive(tempty_bar(buf));
                        ptx::mbar_arrive(sa_empty_bar(a));
                    }
#pragma unroll
                    for (int j = 0; j < HALF; ++j)
                        acc[j] = fmaf(__uint_as_float(part[j]), scale, acc[j]);
                } else {
                    // One N block per slice (BN = 256): two 64-column rounds; the
                    // buffer is released as soon as the second round is loaded.
                    static_assert(HALF == 128, "wide-tile promote");
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
                                ptx::mbar_arrive(tempty_bar(buf));
                                ptx::mbar_arrive(sa_empty_bar(a));
                            }
                        }
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            acc[h * 64 + j] = fmaf(__uint_as_float(r0[j]), scale, acc[h * 64 + j]);
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            acc[h * 64 + 32 + j] = fmaf(__uint_as_float(r1[j]), scale, acc[h * 64 + 32 + j]);
                    }
                }
            }
            if (!ok)
                break;
            int t, kb0, kb_last, scratch;
            span.step(seg_start, t, kb0);
            span.step(seg_end - 1, scratch, kb_last);
            // Stream-K hand-off, warp by warp: warp ew of every CTA owns the same
            // 32 rows x HALF columns of a tile, in slot layout [column/4][row].
            const size_t slice = static_cast<size_t>(wg * HALF / 4) * kBlockM + static_cast<size_t>(row);
            const TileGeo geo = tile_geo<MOE>(args, t, BN, n_leaders);
            // A warp whose 32 rows all lie past M stores nothing, so it neither
            // publishes nor adds partials (its counterparts in the other CTAs of
            // the tile decide the same way): small-M tiles move only live rows.
            const bool rows_live = geo.a_row + q * 32 < args.M;
            // (Stream-K runs with the 256-wide tile only; the host never sets it for the others.)
            if (kSk && kb0 > 0) {
                if (!rows_live)
                    continue;
                // Head of a tile begun by an earlier CTA: publish the scaled partial.
                float *dst = args.sk_partial + static_cast<size_t>(blockIdx.x) * (BN * kBlockM) + 4 * slice;
#pragma unroll
                for (int j = 0; j < HALF; j += 4)
                    ptx::st_global_v4_f32(dst + static_cast<size_t>(j / 4) * kBlockM * 4, acc[j], acc[j + 1], acc[j + 2],
                                          acc[j + 3]);
                // The warp barrier orders every lane's stores before lane 0's
                // release store of the flag, and a release is cumulative: a
                // finisher that acquires the flag sees the whole slice.
                __syncwarp();
                if (lane == 0)
                    ptx::st_release_gpu_u64(args.sk_flags + static_cast<size_t>(blockIdx.x) * kEpiWarps + ew,
                                            args.sk_token);
                continue;
            }
            if (kSk && kb_last != KB - 1 && rows_live) {
                // This CTA holds K block 0 of a cut tile: add the partials of the
                // CTAs that hold the rest of it, then store the tile.
                // The other CTAs of the tile: up to the one whose range holds the
                // tile's last unit, the largest c with floor(c * U / G) <= unit.
                const long long G = gridDim.x;
                const long long U = static_cast<long long>(tiles - span.tile0) * KB;
                const long long tile_end = static_cast<long long>(t + 1 - span.tile0) * KB;
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
                        const float4 v = ptx::ld_cg_v4_f32(src + static_cast<size_t>(j / 4) * kBlockM * 4);
                        acc[j] += v.x;
                        acc[j + 1] += v.y;
                        acc[j + 2] += v.z;
                        acc[j + 3] += v.w;
                    }
                    __syncwarp();
                    if (lane == 0)
                        *reinterpret_cast<volatile unsigned long long *>(flag) = 0ull;   // ready for the next call
                }
                if (!ok)
                    break;
            }
            const int x0 = geo.nb * BN + wg * HALF;
            const int y0 = geo.a_row + q * 32;
            if (MOE && q * 32 >= geo.rows) {
                // Solo leader: rows 64..127 of the tile are the next sort block's
                // (another expert's): computed, never stored.
            } else if (args.c_e4m3) {
#pragma unroll
                for (int c = 0; c < HALF / 64; ++c)
                    store_c8_chunk(&tmC, cstage, lane, acc + c * 64, args.c_scale, x0 + c * 64, y0, args.M, args.N);
            } else if constexpr (L::TILE_C) {
                // Into the tile buffer once its previous tile has been read out,
                // then on to the next tile; the store warp writes C.
                if (!wait_bounded_warp(c_empty_bar, (n_stored & 1) ^ 1, abort_flag, args)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int c = 0; c < HALF / 64; ++c)
                    stage_c64_row(sbase + L::OFF_C + (wg * (HALF / 64) + c) * (kBlockM * 128), row, acc + c * 64);
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0)
                    ptx::mbar_arrive(c_full_bar);
                ++n_stored;
            } else {
#pragma unroll
                for (int c = 0; c < HALF / kCChunkCols; ++c)
                    store_c_chunk(&tmC, cstage, lane, acc + c * kCChunkCols, x0 + c * kCChunkCols, y0, args.M,
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

// Launch helpers called by the host API (api.cu).
template <int BN, int STAGES, bool MOE>
cudaError_t launch_blockscale_any(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmSA,
                                  const CUtensorMap &tmC, const GemmArgs &args, int grid, cudaStream_t stream)
{
    using L = BsLayout<BN, STAGES>;
    constexpr bool kCanSk = BN == 256 && !MOE;
    auto kern = kCanSk && args.sk ? fp8bs_blockscale_kernel<BN, STAGES, MOE, kCanSk>
                                  : fp8bs_blockscale_kernel<BN, STAGES, MOE, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::DYN_SMEM);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kBsThreads);
    cfg.dynamicSmemBytes = L::DYN_SMEM;
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmSA, tmC, args);
}

template <int BN, int STAGES>
cudaError_t launch_blockscale(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmSA,
                              const CUtensorMap &tmC, const GemmArgs &args, int grid, cudaStream_t stream)
{
    return launch_blockscale_any<BN, STAGES, false>(tmA, tmB, tmSA, tmC, args, grid, stream);
}

template <int BN, int STAGES>
cudaError_t launch_blockscale_moe(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmSA,
                                  const CUtensorMap &tmC, const GemmArgs &args, int grid, cudaStream_t stream)
{
    return launch_blockscale_any<BN, STAGES, true>(tmA, tmB, tmSA, tmC, args, grid, stream);
}

template cudaError_t launch_blockscale<256, 4>(const CUtensorMap &, const CUtensorMap &, const CUtensorMap &,
                                               const CUtensorMap &, const GemmArgs &, int, cudaStream_t);
template cudaError_t launch_blockscale<128, 6>(const CUtensorMap &, const CUtensorMap &, const CUtensorMap &,
                                               const CUtensorMap &, const GemmArgs &, int, cudaStream_t);
template cudaError_t launch_blockscale<256, 3>(const CUtensorMap &, const CUtensorMap &, const CUtensorMap &,
                                               const CUtensorMap &, const GemmArgs &, int, cudaStream_t);
template cudaError_t launch_blockscale_moe<256, 4>(const CUtensorMap &, const CUtensorMap &, const CUtensorMap &,
                                                   const CUtensorMap &, const GemmArgs &, int, cudaStream_t);
template cudaError_t launch_blockscale_moe<128, 6>(const CUtensorMap &, const CUtensorMap &, const CUtensorMap &,
                                                   const CUtensorMap &, const GemmArgs &, int, cudaStream_t);

} // namespace fp8bs
