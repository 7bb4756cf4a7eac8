// Pieces shared by the blockscale and MXFP8 kernels and the host launcher.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ptx.cuh"

namespace fp8bs {

constexpr int kBlockM = 128;   // rows of C per tile = TMEM lanes used by one MMA
constexpr int kBlockK = 128;   // K per pipeline stage (one fp32 scale block / four MX groups)
constexpr int kMmaK = 32;      // K of one fp8 tcgen05.mma
constexpr int kEpiWarps = 8;   // promote / epilogue warps (two column halves x four lane quadrants)
constexpr int kCChunkCols = 32;            // C columns per TMA store of one epilogue warp
constexpr int kCStageBytes = 32 * kCChunkCols * 2;  // per epilogue warp: one 32 x 32 bf16 buffer, 64-byte swizzle

constexpr int kStatusTimeout = 1;   // value the device writes into the status word

// Tile order. Tiles are visited in groups of `group` panels of the "inner"
// operand; raster 0 keeps a group of N panels and walks M inside it (A tiles
// stream past a resident set of B panels), raster 1 the converse.
struct TileRaster {
    int m_tiles, n_tiles, raster, group;

    __host__ __device__ __forceinline__ int num_tiles() const { return m_tiles * n_tiles; }

    __host__ __device__ __forceinline__ void coords(int t, int &mb, int &nb) const
    {
        if (raster == 0) {
            const int per = group * m_tiles;
            const int g = t / per;
            const int r = t - g * per;
            const int n0 = g * group;
            const int gw = (n_tiles - n0) < group ? (n_tiles - n0) : group;
            mb = r / gw;
            nb = n0 + (r - mb * gw);
        } else {
            const int per = group * n_tiles;
            const int g = t / per;
            const int r = t - g * per;
            const int m0 = g * group;
            const int gh = (m_tiles - m0) < group ? (m_tiles - m0) : group;
            nb = r / gh;
            mb = m0 + (r - nb * gh);
        }
    }
};

struct GemmArgs {
    int M, N, K;
    TileRaster raster;
    const float *b_scale;      // blockscale: [ceil(N/128)][K/128]
    const uint8_t *a_sf;       // mxfp8: packed scale atoms of A
    const uint8_t *b_sf;       // mxfp8: packed scale atoms of B
    float alpha;               // tensor-scale twin: C = bf16(alpha * A.B^T)
    int c_e4m3;                // blockscale: C is E4M3, c_scale * sum rounded to nearest, saturated
    float c_scale;
    int *status;               // per-device status word
    unsigned long long wait_limit_ns;       // limit of every pipeline wait
    unsigned long long teardown_limit_ns;   // limit of the waits for work already in flight (>= 1 s)
    // Stream-K schedule of the blockscale kernel (sk != 0): partial tiles are
    // handed from the CTA that computed them to the CTA that stores the tile.
    float *sk_partial;                // [gridDim.x][BN/4][128] float4: one partial tile per CTA
    unsigned long long *sk_flags;     // [gridDim.x]: sk_token once that CTA's partial is written
    unsigned long long sk_token;      // unique per call; a finisher resets the flag to 0
    int sk;
    int sk_dp;                        // stream-K: whole waves of tiles done one per CTA first
    // MXFP8 decode kernel: K slices per tile (its partials use sk_partial, its
    // per-tile arrival counters sk_flags) and the C it writes with plain stores.
    int kslices;
    void *c_out;
    // Grouped (MoE) blockscale GEMM: rows of A and C are sort blocks of
    // kMoeBlockRows rows, each owned by one expert; a tile is a leader (one or
    // two adjacent sort blocks of the same expert) x one N tile of that
    // expert's B. Tile t = nb * n_leaders + leader, so the leaders of one
    // expert, which are adjacent, run side by side on the same B tile.
    const int *moe_leaders;           // [n_blocks]: first block | (covers two blocks) << 30
    const int *moe_n_leaders;         // device-side count (written by the descriptor kernel)
    const int *moe_block_expert;      // [n_blocks]: expert of each sort block
    int moe_n_tiles;                  // N tiles per leader
    int moe_n_blocks;                 // sort blocks; device values are clamped to the launch's
    int moe_num_experts;              // bounds, so a malformed descriptor cannot index out of range
};

constexpr int kMoeBlockRows = 64;     // MoE sort-block granularity (rows)
constexpr int kMxdMaxSteps = 6;       // MXFP8 decode kernel: most K steps a CTA holds in shared memory

// Where tile t sits: first rows of A/C and of B, its N tile, the expert (for
// the b_scale rows) and how many of its 128 rows are stored.
struct TileGeo {
    int a_row, b_row, nb, expert, rows;
};

__device__ __forceinline__ int moe_leader_count(const GemmArgs &a)
{
    return min(max(__ldg(a.moe_n_leaders), 0), a.moe_n_blocks);
}

template <bool MOE>
__device__ __forceinline__ TileGeo tile_geo(const GemmArgs &a, int t, int BN, int n_leaders)
{
    TileGeo g;
    if constexpr (MOE) {
        const int li = t % n_leaders;
        g.nb = t / n_leaders;
        const int v = __ldg(a.moe_leaders + li);
        const int b0 = min(v & 0x3FFFFFFF, a.moe_n_blocks - 1);
        g.expert = min(max(__ldg(a.moe_block_expert + b0), 0), a.moe_num_experts - 1);
        g.a_row = b0 * kMoeBlockRows;
        g.b_row = g.expert * a.N + g.nb * BN;
        g.rows = (v >> 30) & 1 ? 2 * kMoeBlockRows : kMoeBlockRows;
    } else {
        int mb;
        a.raster.coords(t, mb, g.nb);
        g.a_row = mb * kBlockM;
        g.b_row = g.nb * BN;
        g.expert = 0;
        g.rows = kBlockM;
    }
    return g;
}

// Tiles of a launch: the raster's, or leaders x N tiles in the grouped mode.
template <bool MOE>
__device__ __forceinline__ int launch_tiles(const GemmArgs &a)
{
    if constexpr (MOE)
        return moe_leader_count(a) * a.moe_n_tiles;
    else
        return a.raster.num_tiles();
}

// The work of one worker (a CTA, or a cluster of CTAS consecutive CTAs that
// share each tile) as flattened steps g = 0 .. total-1, step g being K block kb
// of tile t (tile order of TileRaster). c = blockIdx.x / CTAS is the worker and
// G = gridDim.x / CTAS the number of workers.
//   sk == 0: one worker per tile, tiles c, c + G, ...
//   sk != 0: stream-K after sk_dp whole waves done one worker per tile (so that
//            a wave's workers share operand panels in L2). The units u = t' * KB
//            + kb of the remaining tiles t' are cut into G contiguous ranges
//            equal to one unit; worker c takes [u_c, u_c+1), u_c = floor(c * U /
//            G). A tile cut between workers is finished (scaled partials added,
//            C stored) by the worker that holds its K block 0, which is that
//            worker's last segment; the workers after it write their partials at
//            the start of their range, so the finisher never waits in practice.
template <int CTAS>
struct WorkSpanT {
    int u0;         // first stream-K unit (tiles * KB < 2^31 is checked by the host)
    int total;      // steps of this worker
    int dp_steps;   // steps done one worker per tile, before the stream-K range (all of them without stream-K)
    int tile0;      // first tile of the stream-K range
    int KB;

    __device__ __forceinline__ static int worker() { return static_cast<int>(blockIdx.x) / CTAS; }
    __device__ __forceinline__ static int workers() { return static_cast<int>(gridDim.x) / CTAS; }

    __device__ __forceinline__ static int unit_begin(int U, int c, int G)
    {
        return static_cast<int>((static_cast<long long>(c) * U) / G);
    }

    __device__ __forceinline__ void init(const GemmArgs &a, int KB_) { init(a, KB_, a.raster.num_tiles()); }

    __device__ __forceinline__ void init(const GemmArgs &a, int KB_, int tiles)
    {
        KB = KB_;
        const int c = worker();
        const int G = workers();
        if (a.sk) {
            dp_steps = a.sk_dp * KB;
            tile0 = a.sk_dp * G;
            const int U = (tiles - tile0) * KB;
            u0 = unit_begin(U, c, G);
            total = dp_steps + unit_begin(U, c + 1, G) - u0;
        } else {
            u0 = 0;
            tile0 = tiles;
            total = c < tiles ? ((tiles - c + G - 1) / G) * KB : 0;
            dp_steps = total;
        }
    }

    __device__ __forceinline__ void step(int g, int &t, int &kb) const
    {
        if (g >= dp_steps) {
            const int u = u0 + g - dp_steps;
            t = u / KB;
            kb = u - t * KB;
            t += tile0;
        } else {
            const int i = g / KB;
            t = worker() + i * workers();
            kb = g - i * KB;
        }
    }

    // (t, kb) of step g from that of step g - 1 (g >= 1).
    __device__ __forceinline__ void advance(int g, int &t, int &kb) const
    {
        if (++kb == KB) {
            kb = 0;
            if (g >= dp_steps)
                step(g, t, kb);   // into or inside the stream-K range
            else
                t += workers();
        }
    }

    // The last worker holding a unit of stream-K tile t: the largest c with
    // floor(c * U / G) <= the tile's last unit.
    __device__ __forceinline__ int last_worker(int tiles, int t) const
    {
        const long long G = workers();
        const long long U = static_cast<long long>(tiles - tile0) * KB;
        const long long tile_end = static_cast<long long>(t + 1 - tile0) * KB;
        return static_cast<int>((tile_end * G - 1) / U);
    }
};

using WorkSpan = WorkSpanT<1>;

// Byte offset of (row r in 0..127, group j in 0..3) in a 512-byte scale-factor
// atom: 32 rows of 16 bytes, row (r % 32) holds rows r%32, r%32+32, r%32+64,
// r%32+96 as four 32-bit words, byte j of each word being K group j. This is
// the shared-memory image that one tcgen05.cp 32x128b.warpx4 moves into four
// tensor-memory columns.
__host__ __device__ __forceinline__ int sf_atom_offset(int r, int j)
{
    return (r & 31) * 16 + ((r >> 5) & 3) * 4 + (j & 3);
}

// Bounded wait on an mbarrier phase. Returns false (and raises the CTA abort
// flag and the device status word) when the wait exceeds the time limit, or
// when another role of the CTA has already aborted.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                             const GemmArgs &a)
{
    if (ptx::mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = ptx::globaltimer();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (*abort_flag)
            return false;
        if (ptx::globaltimer() - t0 > a.wait_limit_ns) {
            *abort_flag = 1;
            atomicExch(a.status, kStatusTimeout);
            return false;
        }
    }
    return true;
}

// Wait used only while tearing down, for copies or MMAs this CTA already
// issued (they complete on their own): no abort check, and a limit of its own
// that is never shorter than a second, so that an aborted CTA does not exit
// while its own asynchronous work still targets its shared or tensor memory.
__device__ __forceinline__ void wait_teardown(uint32_t bar, uint32_t parity, const GemmArgs &a)
{
    if (ptx::mbar_try_wait(bar, parity))
        return;
    const uint64_t t0 = ptx::globaltimer();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer() - t0 > a.teardown_limit_ns) {
            atomicExch(a.status, kStatusTimeout);
            return;
        }
    }
}

// Warp-uniform bounded wait: every lane waits, the result is agreed by vote.
__device__ __forceinline__ bool wait_bounded_warp(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                                  const GemmArgs &a)
{
    const bool ok = wait_bounded(bar, parity, abort_flag, a);
    return __all_sync(0xffffffffu, ok);
}

// Warp-uniform bounded wait until *flag == token, i.e. until another CTA of this
// launch has published its partial tile. Every lane acquires the flag itself,
// so its own later loads of the partial are ordered after the publication.
__device__ __forceinline__ bool sk_wait_flag(const unsigned long long *flag, unsigned long long token,
                                             volatile int *abort_flag, const GemmArgs &a)
{
    bool got = ptx::ld_acquire_gpu_u64(flag) == token;
    if (!got) {
        const uint64_t t0 = ptx::globaltimer();
        while (!(got = (ptx::ld_acquire_gpu_u64(flag) == token))) {
            if (*abort_flag)
                break;
            if (ptx::globaltimer() - t0 > a.wait_limit_ns) {
                *abort_flag = 1;
                atomicExch(a.status, kStatusTimeout);
                break;
            }
        }
    }
    return __all_sync(0xffffffffu, got);
}

// The same wait for one thread (no warp vote).
__device__ __forceinline__ bool sk_wait_flag_thread(const unsigned long long *flag, unsigned long long token,
                                                    volatile int *abort_flag, const GemmArgs &a)
{
    if (ptx::ld_acquire_gpu_u64(flag) == token)
        return true;
    const uint64_t t0 = ptx::globaltimer();
    while (ptx::ld_acquire_gpu_u64(flag) != token) {
        if (*abort_flag)
            return false;
        if (ptx::globaltimer() - t0 > a.wait_limit_ns) {
            *abort_flag = 1;
            atomicExch(a.status, kStatusTimeout);
            return false;
        }
    }
    return true;
}

// Store one epilogue warp's 32 rows x 32 columns of C (row = lane) with one
// TMA store of a 2 KiB box through the warp's staging buffer. `v` are the 32
// fp32 values of this lane's row. The buffer uses the 64-byte swizzle: 16-byte
// quarter j of row r sits at quarter j ^ ((r >> 1) & 3). Before the buffer is
// rewritten, the store that last used it must have read it; that wait, the
// fence and the issue are fixed costs per store, so the chunks are as large as
// the staging space allows (halving their number from 16-column chunks saved
// 1-3% of the GEMM time).
__device__ __forceinline__ void store_c_chunk(const CUtensorMap *tmC, uint32_t stage, int lane, const float *v, int x,
                                              int y, int M, int N)
{
    if (lane == 0)
        ptx::bulk_wait_read_all();
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t w0 = ptx::pack_bf16x2(v[j * 8 + 0], v[j * 8 + 1]);
        const uint32_t w1 = ptx::pack_bf16x2(v[j * 8 + 2], v[j * 8 + 3]);
        const uint32_t w2 = ptx::pack_bf16x2(v[j * 8 + 4], v[j * 8 + 5]);
        const uint32_t w3 = ptx::pack_bf16x2(v[j * 8 + 6], v[j * 8 + 7]);
        const int phys = j ^ ((lane >> 1) & 3);
        ptx::st_shared_v4(stage + lane * 64 + phys * 16, w0, w1, w2, w3);
    }
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        if (x < N && y < M)
            ptx::tma_store_2d(tmC, stage, x, y);
        ptx::bulk_commit();
    }
}

// Write one thread's 64 consecutive C columns (bf16) of tile row `row` (0..127)
// into a 128-row x 64-column chunk of a C tile in shared memory (`chunk`,
// 1024-byte aligned). Rows are 128 bytes with the 128-byte swizzle (16-byte
// unit j of row r at unit j ^ (r & 7)): the image one TMA store of a 64 x 128
// box reads. A warp's 32 rows write 8 distinct units per row group of 8, so
// each store instruction takes the minimum four shared-memory wavefronts.
__device__ __forceinline__ void stage_c64_row(uint32_t chunk, int row, const float *v)
{
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t w0 = ptx::pack_bf16x2(v[j * 8 + 0], v[j * 8 + 1]);
        const uint32_t w1 = ptx::pack_bf16x2(v[j * 8 + 2], v[j * 8 + 3]);
        const uint32_t w2 = ptx::pack_bf16x2(v[j * 8 + 4], v[j * 8 + 5]);
        const uint32_t w3 = ptx::pack_bf16x2(v[j * 8 + 6], v[j * 8 + 7]);
        ptx::st_shared_v4(chunk + row * 128 + ((j ^ (row & 7)) * 16), w0, w1, w2, w3);
    }
}

// E4M3 output: one epilogue warp's 32 rows x 64 columns through the same 2 KiB
// staging buffer and 64-byte swizzle as store_c_chunk (a row of 64 bytes), one
// TMA store. Each value is multiplied by `scale` in fp32 and rounded to the
// nearest E4M3 value (ties to even), saturating at +-448: the store side of the
// fp8 partial of skill card "FlyDSL prefill MoE stage-2 fp8 partial"
// (procedure step 2); the consumer multiplies by 1/scale.
__device__ __forceinline__ void store_c8_chunk(const CUtensorMap *tmC, uint32_t stage, int lane, const float *v,
                                               float scale, int x, int y, int M, int N)
{
    if (lane == 0)
        ptx::bulk_wait_read_all();
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float *u = v + j * 16 + q * 4;
            w[q] = ptx::pack_e4m3x4(u[0] * scale, u[1] * scale, u[2] * scale, u[3] * scale);
        }
        const int phys = j ^ ((lane >> 1) & 3);
        ptx::st_shared_v4(stage + lane * 64 + phys * 16, w[0], w[1], w[2], w[3]);
    }
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        if (x < N && y < M)
            ptx::tma_store_2d(tmC, stage, x, y);
        ptx::bulk_commit();
    }
}

} // namespace fp8bs
