// Host side of libfp8bs: argument checks, shape-class -> kernel configuration,
// tensor-map encoding, launches, the per-device status word, the scale repack
// kernels and the layout helpers declared in include/fp8bs.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>
#include <stdint.h>
#include <string.h>

#include "fp8bs.h"
#include "common.cuh"

namespace fp8bs {

template <int BN, int STAGES>
cudaError_t launch_blockscale(const CUtensorMap &, const CUtensorMap &, const CUtensorMap &, const CUtensorMap &,
                              const GemmArgs &, int, cudaStream_t);
template <int BN, int STAGES>
cudaError_t launch_blockscale_moe(const CUtensorMap &, const CUtensorMap &, const CUtensorMap &, const CUtensorMap &,
                                  const GemmArgs &, int, cudaStream_t);
template <int STAGES>
cudaError_t launch_blockscale_pair(const CUtensorMap &, const CUtensorMap &, const CUtensorMap &, const CUtensorMap &,
                                   const GemmArgs &, int, cudaStream_t);
template <int STAGES>
cudaError_t max_bs_pair_clusters(int *);
template <int STAGES>
cudaError_t launch_mxfp8_pair(const CUtensorMap &, const CUtensorMap &, const CUtensorMap &, const CUtensorMap &,
                              const CUtensorMap &, const GemmArgs &, int, cudaStream_t);
template <int STAGES>
cudaError_t max_mx_pair_clusters(int *);
template <int BN, int STAGES>
cudaError_t launch_mx_family(int kind, bool sk, const CUtensorMap &, const CUtensorMap &, const CUtensorMap &,
                             const GemmArgs &, int, cudaStream_t);
template <int MAXS>
cudaError_t launch_mxfp8_decode(const CUtensorMap &, const CUtensorMap &, const GemmArgs &, cudaStream_t);
template <int MAXS>
cudaError_t max_mxfp8_decode_clusters(int, int *);

namespace host {

__device__ int g_status_word;   // per-device status written by the kernels

constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull;
constexpr int kMxPairStages = 6;
constexpr int kBsPairStages = 4;
constexpr int kPairMinM = 2048;       // rows from which the blockscale pair kernel is chosen

struct DeviceState {
    bool ready = false;
    int status = FP8BS_OK;          // result of the set-up
    int num_sms = 0;
    int *status_ptr = nullptr;      // device address of g_status_word
    cudaMemPool_t pool = nullptr;   // stream-ordered pool for fp8mx_gemm's packed scales
    int mx_pair_clusters = 0;       // co-resident CTA pairs of the MXFP8 pair kernel
    int bs_pair_clusters = 0;       // co-resident CTA pairs of the blockscale pair kernel
};

std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];
std::atomic<unsigned long long> g_wait_limit_ns{kDefaultWaitLimitNs};
std::atomic<int> g_config_override{0};
std::atomic<int> g_raster_group{1};   // panels per raster group (1 = plain M-inner / N-inner order)
std::atomic<unsigned long long> g_sk_token{0};   // stream-K hand-off tokens, unique per call
// Whether clusters of n CTAs (2..8) of the MXFP8 decode kernel fit on a device:
// 0 not yet asked, 1 yes, -1 no. A property of the device and the kernel, so it
// survives fp8bs_shutdown; both entry paths (with and without the pool) use it.
std::atomic<int> g_mxd_fit[kMaxDevices][9];
thread_local int t_last_config = 0;

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// One-time set-up per device, with that device current: capability check, SM
// count, the device address of the status word, the workspace pool, and the
// number of co-resident CTA pairs.
int ensure_device(int &dev, DeviceState *&st)
{
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return FP8BS_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    st = &g_dev[dev];
    if (st->ready)
        return st->status;
    st->ready = true;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&st->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return st->status = FP8BS_ERR_CUDA;
    if (major != 10 || minor != 3)
        return st->status = FP8BS_ERR_UNSUPPORTED_DEVICE;
    if (cudaGetSymbolAddress(reinterpret_cast<void **>(&st->status_ptr), g_status_word) != cudaSuccess)
        return st->status = FP8BS_ERR_CUDA;
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    if (cudaMemPoolCreate(&st->pool, &props) != cudaSuccess)
        return st->status = FP8BS_ERR_CUDA;
    uint64_t keep = UINT64_MAX;   // keep freed workspace in the pool between calls
    if (cudaMemPoolSetAttribute(st->pool, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess)
        return st->status = FP8BS_ERR_CUDA;
    if (max_mx_pair_clusters<kMxPairStages>(&st->mx_pair_clusters) != cudaSuccess || st->mx_pair_clusters < 1)
        return st->status = FP8BS_ERR_CUDA;
    if (max_bs_pair_clusters<kBsPairStages>(&st->bs_pair_clusters) != cudaSuccess || st->bs_pair_clusters < 1)
        return st->status = FP8BS_ERR_CUDA;
    if (!g_encode) {
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return st->status = FP8BS_ERR_CUDA;
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    return st->status = FP8BS_OK;
}

// 2-D row-major tensor [rows][cols], box [box_rows][box_cols].
bool encode_2d(CUtensorMap *tm, CUtensorMapDataType dt, const void *base, uint64_t cols, uint64_t rows,
               uint64_t row_stride_bytes, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swz)
{
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {row_stride_bytes};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return g_encode(tm, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Teardown waits (for work already issued) keep at least the default limit.
unsigned long long teardown_limit()
{
    const unsigned long long w = g_wait_limit_ns.load();
    return w > kDefaultWaitLimitNs ? w : kDefaultWaitLimitNs;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int check_shape(int M, int N, int K)
{
    if (M < 0 || N < 8 || (N % 8) != 0 || K < 128 || (K % 128) != 0 || K > (1 << 20))
        return FP8BS_ERR_SHAPE;
    return FP8BS_OK;
}

// Kernel configuration. kind 1: one-CTA blockscale kernel, 2: MXFP8 kernel,
// 3: CTA-pair blockscale kernel (256 x 256 tiles over two SMs), 4: tensor-scale
// twin (the MXFP8 kernel's pipeline with plain fp8 MMAs), 5: CTA-pair MXFP8
// kernel (256 x 256 tiles over two SMs), 6: MXFP8 decode kernel.
// sched 1: one CTA (pair) per tile; 2: stream-K (256-wide tile of kinds 1, 2,
// 3 and 4).
struct Config {
    int kind, block_n, stages, raster, sched;
};

int config_id(const Config &c)
{
    return c.kind * 1000000 + c.block_n * 1000 + c.stages * 100 + c.raster * 10 + c.sched;
}

// Only the instantiated kernels are valid configurations.
bool decode_config_id(int id, Config &c)
{
    c.kind = id / 1000000;
    c.block_n = (id / 1000) % 1000;
    c.stages = (id / 100) % 10;
    c.raster = (id / 10) % 10;
    c.sched = id % 10;
    // stream-K: the 256-wide tile of kinds 1, 2 and 4, and the MXFP8 kernel's 128-wide tile
    if (c.sched < 1 || c.sched > 2 || c.raster > 1 ||
        (c.sched == 2 && c.block_n != 256 && !(c.kind == 2 && c.block_n == 128)))
        return false;
    if (c.kind == 1)
        return (c.block_n == 256 && (c.stages == 4 || c.stages == 3)) || (c.block_n == 128 && c.stages == 6);
    if (c.kind == 2 || c.kind == 4)
        return (c.block_n == 256 && c.stages == 4) || (c.block_n == 128 && c.stages == 6);
    if (c.kind == 3)
        return c.block_n == 256 && c.stages == kBsPairStages;
    if (c.kind == 5)
        return c.block_n == 256 && c.stages == kMxPairStages && c.sched == 1;
    if (c.kind == 6)
        return c.block_n == 128 && c.stages == kMxdMaxSteps && c.sched == 1 && c.raster == 0;   // no tile raster
    return false;
}

// K slices per 128-column tile of the MXFP8 decode kernel (its cluster size):
// enough that a slice (at most kMxdMaxSteps K steps) fits in shared memory
// whole, and otherwise as many as one wave of CTAs on num_sms SMs allows, at
// most the portable cluster size 8. 0 when the kernel does not apply (more than
// one row of tiles, or a K that needs more than 8 slices).
int mxd_slices(int M, int N, int K, int num_sms)
{
    const int tiles = (N + 127) / 128;
    const int KS = K / 128;
    if (M > 128 || KS < 1)
        return 0;
    const int s_min = (KS + kMxdMaxSteps - 1) / kMxdMaxSteps;
    if (s_min > 8)
        return 0;
    const int s_fill = num_sms / tiles;
    int S = s_fill > s_min ? s_fill : s_min;
    if (S > KS)
        S = KS;
    return S > 8 ? 8 : S;
}

// Stream-K grid: every CTA gets at least max(8, KB/4) K blocks, so a tile is
// cut between at most about five CTAs and its finisher adds few partials. With
// a single row of tiles (M <= 128, decode) the hand-off moves only the live
// rows, so the floor is max(4, KB/8): more CTAs stream the weights.
long long sk_grid(long long units, long long KB, int num_sms, bool one_row = false)
{
    const long long floor_units = one_row ? 4 : 8;
    const long long min_units = KB / (one_row ? 8 : 4) > floor_units ? KB / (one_row ? 8 : 4) : floor_units;
    long long g = units / min_units;
    if (g > num_sms)
        g = num_sms;
    return g < 1 ? 1 : g;
}

// Smallest saving of K steps in the longest CTA for which stream-K is chosen.
// The hand-off costs 5-12 us per launch whatever the shape (publishing a 128 KB
// fp32 partial takes ~3.5 us, the finisher's add ~1.5 us, and each CTA has an
// extra segment boundary), against ~0.5 us per blockscale K block and ~0.35 us
// per MXFP8 K step. Measured on 152 SMs (tile vs stream-K, us): blockscale
// 16384x1536x7168 179/159 (saving 53), 8192x2048x7168 122/110 (35),
// 1024x2048x7168 35.5/32.5 (32), 4096x2048x7168 66.2/67.3 (17),
// 2048x2048x7168 37.6/40.7 (8); MXFP8 1024x5120x2048 28.4/26.4 (15),
// 4096x5120x2048 48.9/48.9 (12), 2048x8192x1280 34.5/36.6 (6).
constexpr long long kSkMinGainBs = 20;
constexpr long long kSkMinGainMx = 13;

// Stream-K set-up shared by the kernels with a 256-wide tile: the number of
// workers (`grid`: CTAs, or CTA pairs for the pair kernel, at most `workers`),
// the whole waves run one worker per tile before the stream-K range (a wave's
// workers share A and B panels in L2), and the workspace from the stream-ordered
// pool: one fp32 partial of 128 x 256 and kEpiWarps flags per CTA. Fresh or
// reused memory never holds this call's token, and finishers reset the flags
// they consume. The caller frees `ws` on the stream after the launch.
int setup_stream_k(int tiles, int KB, int workers, cudaMemPool_t pool, cudaStream_t s, GemmArgs &args, int &grid,
                   void *&ws, int ctas_per_worker = 1)
{
    const long long units = static_cast<long long>(tiles) * KB;
    if (units >= (1ll << 31) || !pool)
        return FP8BS_ERR_SHAPE;
    grid = static_cast<int>(sk_grid(units, KB, workers, args.M <= 128));
    const int full_waves = tiles / grid;
    args.sk_dp = full_waves >= 2 ? full_waves - 1 : 0;
    // Every CTA must hold at least one unit of the stream-K range: a finisher
    // waits for each CTA after it up to the one holding its tile's last unit.
    // (True by construction: the range has at least a wave of tiles, or grid <=
    // units / 4.)
    if (static_cast<long long>(tiles - args.sk_dp * grid) * KB < grid)
        return FP8BS_ERR_SHAPE;
    const size_t ctas = static_cast<size_t>(grid) * ctas_per_worker;
    const size_t slot = static_cast<size_t>(kBlockM) * 256 * sizeof(float);
    const size_t bytes = ctas * (slot + kEpiWarps * sizeof(unsigned long long));
    if (cudaMallocFromPoolAsync(&ws, bytes, pool, s) != cudaSuccess)
        return FP8BS_ERR_CUDA;
    args.sk = 1;
    args.sk_partial = static_cast<float *>(ws);
    args.sk_flags = reinterpret_cast<unsigned long long *>(static_cast<char *>(ws) + ctas * slot);
    args.sk_token = g_sk_token.fetch_add(1) + 1;
    return FP8BS_OK;
}

// Shape class -> configuration before the blockscale stage choice below.
Config choose_config_base(int kind, int M, int N, int K, int num_sms)
{
    Config c;
    // Stream the larger operand once past a resident set of panels of the smaller one.
    c.raster = ((long)M >= (long)N) ? 1 : 0;
    c.sched = 1;
    c.kind = kind;
    // Blockscale and MXFP8 alike: wide one-CTA tiles (128 x 256), which keep
    // shared-memory operand traffic at 96 B/clk per SM and give each tcgen05.mma
    // 128 clocks of work (narrower MMAs are issue-bound).
    c.block_n = 256;
    c.stages = 4;
    const long long tiles256 = (long long)((M + 127) / 128) * ((N + 255) / 256);
    // Stream-K (256-wide tile) when it shortens the longest CTA's K loop by at
    // least kSkMinGain K steps, which pays for the partial hand-off. E.g.
    // blockscale 768 tiles x 56 K blocks on 152 SMs: 336 -> 283; 8 tiles x 56:
    // 56 -> 3. The tensor-scale twin follows the blockscale rule, so that the two
    // run the same tiles.
    const long long KB = K / 128;
    const long long units = tiles256 * KB;
    const long long min_gain = kind == 2 ? kSkMinGainMx : kSkMinGainBs;
    // One row of tiles with more than two live 32-row groups: the hand-off
    // carries most of each partial, and the 128-wide tile measured faster
    // (blockscale 128x2048x7168: 26.7 vs 29.1 us; 32x1536x7168: stream-K 25.8
    // vs 26.6 us, 16x2048x7168: 24.9 vs 26.5 us).
    const bool heavy_decode = M <= 128 && M > 64;
    if (tiles256 > 0 && units < (1ll << 31) && num_sms > 0 && !heavy_decode) {
        const long long g = sk_grid(units, KB, num_sms, M <= 128);
        const long long per_tile = (tiles256 + num_sms - 1) / num_sms * KB;   // one CTA per tile
        const long long per_unit = (units + g - 1) / g;                       // stream-K
        if (per_tile - per_unit >= min_gain) {
            c.sched = 2;
            return c;
        }
    }
    // Otherwise the narrow tile when the wide one leaves most SMs idle.
    if (tiles256 * 2 <= num_sms) {
        c.block_n = 128;
        c.stages = 6;
        return c;
    }
    // MXFP8 with M >= 4096, one CTA per tile: the CTA-pair kernel (256 x 256
    // tiles, half of B per CTA, six stages). Measured against the one-CTA
    // kernel (us): 16384x5120x2048 121.5 -> 119.6, 16384x8192x1280 130.2 ->
    // 126.3, 4096x8192x1280 42.8 -> 41.3, 4096x5120x2048 43.3 -> 42.8; at
    // M <= 2048 it is no better.
    if (kind == 2 && M >= 4096) {
        c.kind = 5;
        c.stages = 6;
    }
    return c;
}

// Blockscale GEMM with few K blocks per tile (K <= 1024), one-CTA kernel: the
// three-stage instance, whose freed shared memory holds a whole C tile that a
// warp of its own stores, so the C store of a tile overlaps the next tile's K
// loop. Same-session times (us, L2 flushed, tile / stream-K schedule, 4 -> 3
// stages, with two alternating 4 KiB C buffers per warp, which the tile buffer
// matches within 0.5%): 16384x7168x768 119.2 -> 109.0 / 123.9 -> 114.8;
// 16384x7168x1024 141.3 -> 133.3; 16384x7168x1536 183.8 -> 180.3;
// 4096x65536x1536 398.5 -> 405.1; 16384x7168x2048 225.4 -> 229.9;
// 4096x2048x7168 63.5 -> 71.7 (one producer thread fills the odd-count ring,
// which deep K loops feel).
constexpr int kWideCMaxKBlocks = 8;

// The one-CTA kernels' rule: shape class -> configuration.
Config choose_config_one_cta(int kind, int M, int N, int K, int num_sms)
{
    Config c = choose_config_base(kind, M, N, K, num_sms);
    if (kind == 1 && c.block_n == 256 && K / 128 <= kWideCMaxKBlocks)
        c.stages = 3;
    return c;
}

// Shape class -> configuration, from (M, N, K) only.
Config choose_config(int kind, int M, int N, int K, int num_sms)
{
    Config c = choose_config_one_cta(kind, M, N, K, num_sms);
    // Blockscale, one CTA per tile, M >= 2048: the CTA-pair kernel (256 x 256
    // tiles, half of B per CTA, four stages and a whole-tile C buffer).
    // Same-session times (us, L2 flushed; one-CTA kernel (three / four stages)
    // -> pair): 16384x7168x768 107.8 / 121.4 -> 105.5; 16384x7168x1024 131.2 /
    // 142.8 -> 125.7; 16384x7168x1536 176.8 / 185.4 -> 166.6; 16384x7168x2048
    // 225.1 / 229.5 -> 206.5; 16384x7168x3072 318.3 / 316.0 -> 288.5;
    // 8192x8192x3072 191.3 / 188.5 -> 173.9; 4096x65536x1536 396.0 / 405.3 ->
    // 362.1; 4096x2048x7168 71.8 / 63.6 -> 61.8. Stream-K shapes keep the
    // one-CTA kernel; the pair's own stream-K instance (config 3256402/12) is no
    // faster (us, one session: 16384x1536x7168 153.1 one-CTA stream-K, 152.9
    // pair stream-K; 4096x2048x7168 pair one per tile 60.4, pair stream-K 67.2).
    if (kind == 1 && c.block_n == 256 && c.sched == 1 && M >= kPairMinM) {
        c.kind = 3;
        c.stages = kBsPairStages;
    }
    return c;
}

bool override_config(int kind_a, int kind_b, Config &cfg, int kind_c = -1)
{
    const int ovr = g_config_override.load();
    if (!ovr)
        return true;
    Config o;
    if (!decode_config_id(ovr, o) || (o.kind != kind_a && o.kind != kind_b && o.kind != kind_c))
        return false;
    cfg = o;
    return true;
}

// Repack ue8m0 bytes [rows][K/32] into 512-byte scale-factor atoms (see
// mx_kernel.cu): one thread per (row, 128-wide K step), K steps fastest so the
// 4-byte reads of a row are contiguous. Two tensors (A and B) in one launch.
__global__ void pack_scales_kernel(const uint8_t *__restrict__ e0, uint8_t *__restrict__ p0, int rows0,
                                   const uint8_t *__restrict__ e1, uint8_t *__restrict__ p1, int rows1, int KS)
{
    const int64_t n0 = static_cast<int64_t>((rows0 + 127) / 128) * 128 * KS;
    const int64_t n1 = static_cast<int64_t>((rows1 + 127) / 128) * 128 * KS;
    const int G = KS * 4;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n0 + n1;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const bool first = i < n0;
        const int64_t idx = first ? i : i - n0;
        const uint8_t *e = first ? e0 : e1;
        uint8_t *p = first ? p0 : p1;
        const int rows = first ? rows0 : rows1;
        const int row = static_cast<int>(idx / KS);
        const int ks = static_cast<int>(idx - static_cast<int64_t>(row) * KS);
        uint32_t v = 0;
        if (row < rows)
            v = *reinterpret_cast<const uint32_t *>(e + static_cast<int64_t>(row) * G + 4 * ks);
        const int64_t atom = static_cast<int64_t>(row / 128) * KS + ks;
        *reinterpret_cast<uint32_t *>(p + atom * 512 + sf_atom_offset(row % 128, 0)) = v;
    }
}

int launch_pack_scales(const uint8_t *e0, uint8_t *p0, int rows0, const uint8_t *e1, uint8_t *p1, int rows1, int K,
                       int num_sms, cudaStream_t stream)
{
    const int KS = K / 128;
    const int64_t total = (static_cast<int64_t>((rows0 + 127) / 128) + (rows1 + 127) / 128) * 128 * KS;
    int64_t blocks = (total + 255) / 256;
    if (blocks > static_cast<int64_t>(num_sms) * 16)
        blocks = static_cast<int64_t>(num_sms) * 16;
    if (blocks < 1)
        blocks = 1;
    pack_scales_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(e0, p0, rows0, e1, p1, rows1, KS);
    return cudaGetLastError() == cudaSuccess ? FP8BS_OK : FP8BS_ERR_LAUNCH;
}

__global__ void pack_a_scale_kernel(const float *__restrict__ src, float *__restrict__ dst, int M, int KB,
                                    int64_t ld)
{
    const int64_t total = ld * KB;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int kb = static_cast<int>(i / ld);
        const int m = static_cast<int>(i - static_cast<int64_t>(kb) * ld);
        dst[i] = m < M ? src[static_cast<int64_t>(m) * KB + kb] : 0.f;
    }
}

// Tensor maps, arguments and launch of the MXFP8 kernel on packed scales
// (cfg.kind 2) or of the tensor-scale twin (cfg.kind 4, no scale atoms, one
// alpha): a persistent grid of min(tiles, SMs) CTAs, or the stream-K grid.
int launch_mx(Config &cfg, const void *A, const uint8_t *a_sf, const void *B, const uint8_t *b_sf, void *C, int M,
              int N, int K, float alpha, int *status_ptr, int num_sms, int mx_pair_clusters, cudaMemPool_t pool,
              cudaStream_t s, bool c_e4m3 = false, float c_scale = 1.f)
{
    if (c_e4m3)
        cfg.sched = 1;   // the E4M3-output MXFP8 kernel runs one CTA per tile (cfg reports what ran)
    if (cfg.kind == 5 && c_e4m3) {
        cfg.kind = 2;     // the pair kernel stores bf16 only: E4M3 C goes through the one-CTA kernel
        cfg.stages = 4;
    }
    int slices = cfg.kind == 6 ? mxd_slices(M, N, K, num_sms) : 0;
    if (slices > 1) {
        // Clusters of that size must fit on the device (queried once per size).
        int dev = 0;
        cudaGetDevice(&dev);
        int fit = dev >= 0 && dev < kMaxDevices ? g_mxd_fit[dev][slices].load() : -1;
        if (fit == 0) {
            int n = 0;
            fit = max_mxfp8_decode_clusters<kMxdMaxSteps>(slices, &n) == cudaSuccess && n >= 1 ? 1 : -1;
            g_mxd_fit[dev][slices].store(fit);
        }
        if (fit < 0)
            slices = 0;
    }
    if (cfg.kind == 6 && (c_e4m3 || slices < 1)) {
        // The decode kernel stores bf16 only and takes one row of tiles and a
        // K of at most 8 slices: the one-CTA 128-wide kernel instead.
        cfg.kind = 2;
        cfg.block_n = 128;
        cfg.stages = 6;
        cfg.sched = 1;
    }
    if (cfg.kind == 6) {
        CUtensorMap tmA, tmB;
        if (!encode_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, K, M, K, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, K, N, K, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B))
            return FP8BS_ERR_LAUNCH;
        GemmArgs args = {};
        args.M = M;
        args.N = N;
        args.K = K;
        args.a_sf = a_sf;
        args.b_sf = b_sf;
        args.c_out = C;
        args.kslices = slices;
        args.status = status_ptr;
        args.wait_limit_ns = g_wait_limit_ns.load();
        args.teardown_limit_ns = teardown_limit();
        return launch_mxfp8_decode<kMxdMaxSteps>(tmA, tmB, args, s) == cudaSuccess ? FP8BS_OK : FP8BS_ERR_LAUNCH;
    }
    if (cfg.kind == 5) {
        const int KS = K / 128;
        const uint64_t atoms_a = static_cast<uint64_t>((M + 127) / 128) * KS;
        const uint64_t atoms_b = static_cast<uint64_t>((N + 127) / 128) * KS;
        CUtensorMap tmA, tmB, tmSFA, tmSFB, tmC;
        // a scale atom is 512 contiguous bytes: 4 rows of 128 in these tensors
        if (!encode_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, K, M, K, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, K, N, K, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_2d(&tmSFA, CU_TENSOR_MAP_DATA_TYPE_UINT8, a_sf, 128, atoms_a * 4, 128, 128, 4,
                       CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !encode_2d(&tmSFB, CU_TENSOR_MAP_DATA_TYPE_UINT8, b_sf, 128, atoms_b * 4, 128, 128, 4,
                       CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !encode_2d(&tmC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, C, N, M, static_cast<uint64_t>(N) * 2, kCChunkCols, 32,
                       CU_TENSOR_MAP_SWIZZLE_64B))
            return FP8BS_ERR_LAUNCH;
        GemmArgs args = {};
        args.M = M;
        args.N = N;
        args.K = K;
        args.raster.m_tiles = (M + 2 * kBlockM - 1) / (2 * kBlockM);
        args.raster.n_tiles = (N + 255) / 256;
        args.raster.raster = cfg.raster;
        args.raster.group = g_raster_group.load();
        args.status = status_ptr;
        args.wait_limit_ns = g_wait_limit_ns.load();
        args.teardown_limit_ns = teardown_limit();
        if (mx_pair_clusters < 1)
            return FP8BS_ERR_LAUNCH;
        const cudaError_t e = launch_mxfp8_pair<kMxPairStages>(tmA, tmB, tmSFA, tmSFB, tmC, args, mx_pair_clusters, s);
        return e == cudaSuccess ? FP8BS_OK : FP8BS_ERR_LAUNCH;
    }
    CUtensorMap tmA, tmB, tmC;
    if (!encode_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, K, M, K, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, K, N, K, 128, cfg.block_n, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !(c_e4m3 ? encode_2d(&tmC, CU_TENSOR_MAP_DATA_TYPE_UINT8, C, N, M, static_cast<uint64_t>(N), 64, 32,
                             CU_TENSOR_MAP_SWIZZLE_64B)
                 : encode_2d(&tmC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, C, N, M, static_cast<uint64_t>(N) * 2,
                             kCChunkCols, 32, CU_TENSOR_MAP_SWIZZLE_64B)))
        return FP8BS_ERR_LAUNCH;
    GemmArgs args = {};
    args.c_e4m3 = c_e4m3 ? 1 : 0;
    args.c_scale = c_scale;
    args.M = M;
    args.N = N;
    args.K = K;
    args.raster.m_tiles = (M + kBlockM - 1) / kBlockM;
    args.raster.n_tiles = (N + cfg.block_n - 1) / cfg.block_n;
    args.raster.raster = cfg.raster;
    args.raster.group = g_raster_group.load();
    args.a_sf = a_sf;
    args.b_sf = b_sf;
    args.alpha = alpha;
    args.status = status_ptr;
    args.wait_limit_ns = g_wait_limit_ns.load();
    args.teardown_limit_ns = teardown_limit();
    const int tiles = args.raster.num_tiles();
    int grid = tiles < num_sms ? tiles : num_sms;
    void *ws = nullptr;
    if (cfg.sched == 2) {
        if (cfg.block_n != 256 && cfg.kind != 2)
            return FP8BS_ERR_SHAPE;
        const int rc = setup_stream_k(tiles, K / 128, num_sms, pool, s, args, grid, ws);
        if (rc)
            return rc;
    }
    const int family = cfg.kind == 4 ? 2 : (c_e4m3 ? 1 : 0);
    const bool sk = cfg.sched == 2;
    const cudaError_t e = cfg.block_n == 256 ? launch_mx_family<256, 4>(family, sk, tmA, tmB, tmC, args, grid, s)
                                             : launch_mx_family<128, 6>(family, sk, tmA, tmB, tmC, args, grid, s);
    const bool freed = !ws || cudaFreeAsync(ws, s) == cudaSuccess;
    return e == cudaSuccess && freed ? FP8BS_OK : FP8BS_ERR_LAUNCH;
}

// The blockscale GEMM with a bf16 (c_e4m3 == false) or an E4M3 C.
int blockscale_gemm(const void *A, const float *a_scale, const void *B, const float *b_scale, void *C, bool c_e4m3,
                    float c_scale, int M, int N, int K, void *stream)
{
    int rc = check_shape(M, N, K);
    if (rc)
        return rc;
    if (c_e4m3 && (N % 16) != 0)   // the E4M3 rows of C must be whole 16-byte units for the tensor copies
        return FP8BS_ERR_SHAPE;
    if (M == 0)
        return FP8BS_OK;
    if (!A || !a_scale || !B || !b_scale || !C)
        return FP8BS_ERR_NULL;
    if (!aligned(A, 16) || !aligned(a_scale, 16) || !aligned(B, 16) || !aligned(b_scale, 4) || !aligned(C, 16))
        return FP8BS_ERR_ALIGN;
    int dev;
    DeviceState *st;
    if ((rc = ensure_device(dev, st)))
        return rc;
    Config cfg = choose_config(1, M, N, K, st->num_sms);
    // The E4M3 store is the one-CTA kernel's four-stage instance (stages 2 KiB
    // E4M3 chunks per warp; the whole-tile bf16 buffer of the three-stage
    // instance does not apply): 16384x7168x768 103.4 us there, 116.8 with
    // three stages.
    if (c_e4m3)
        cfg = choose_config_base(1, M, N, K, st->num_sms);
    if (!override_config(1, 3, cfg))
        return FP8BS_ERR_SHAPE;
    const bool pair = cfg.kind == 3;   // CTA-pair kernel: 256 x 256 tiles, half of the B tile per CTA
    if (pair && c_e4m3)
        return FP8BS_ERR_SHAPE;         // forced by the override
    const int KB = K / 128;
    const uint64_t ld_sa = static_cast<uint64_t>(fp8bs_a_scale_ld(M));
    // whole-tile C buffer (one-CTA three stages, and the pair kernel): 128 x 64 bf16 C boxes, 128-byte swizzle
    const bool tile_c = cfg.block_n == 256 && (pair || cfg.stages == 3);
    CUtensorMap tmA, tmB, tmSA, tmC;
    if (!encode_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, K, M, K, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, K, N, K, 128, pair ? cfg.block_n / 2 : cfg.block_n,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tmSA, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a_scale, ld_sa, KB, ld_sa * 4, 128, 1,
                   CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !(c_e4m3 ? encode_2d(&tmC, CU_TENSOR_MAP_DATA_TYPE_UINT8, C, N, M, static_cast<uint64_t>(N), 64, 32,
                             CU_TENSOR_MAP_SWIZZLE_64B)
                 : encode_2d(&tmC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, C, N, M, static_cast<uint64_t>(N) * 2,
                             tile_c ? 64 : kCChunkCols, tile_c ? 128 : 32,
                             tile_c ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B)))
        return FP8BS_ERR_LAUNCH;
    GemmArgs args = {};
    args.M = M;
    args.N = N;
    args.K = K;
    args.c_e4m3 = c_e4m3 ? 1 : 0;
    args.c_scale = c_scale;
    args.raster.m_tiles = (M + (pair ? 2 * kBlockM : kBlockM) - 1) / (pair ? 2 * kBlockM : kBlockM);
    args.raster.n_tiles = (N + cfg.block_n - 1) / cfg.block_n;
    args.raster.raster = cfg.raster;
    args.raster.group = g_raster_group.load();
    args.b_scale = b_scale;
    args.status = st->status_ptr;
    args.wait_limit_ns = g_wait_limit_ns.load();
    args.teardown_limit_ns = teardown_limit();
    const int tiles = args.raster.num_tiles();
    // workers: CTAs, or CTA pairs for the pair kernel
    const int max_workers = pair ? st->bs_pair_clusters : st->num_sms;
    int grid = tiles < max_workers ? tiles : max_workers;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void *ws = nullptr;
    if (cfg.sched == 2) {
        if (cfg.block_n != 256)
            return FP8BS_ERR_SHAPE;
        if ((rc = setup_stream_k(tiles, KB, max_workers, st->pool, s, args, grid, ws, pair ? 2 : 1)))
            return rc;
    }
    cudaError_t e;
    if (pair)
        e = launch_blockscale_pair<kBsPairStages>(tmA, tmB, tmSA, tmC, args, grid, s);
    else if (cfg.block_n == 256 && cfg.stages == 3)
        e = launch_blockscale<256, 3>(tmA, tmB, tmSA, tmC, args, grid, s);
    else if (cfg.block_n == 256)
        e = launch_blockscale<256, 4>(tmA, tmB, tmSA, tmC, args, grid, s);
    else
        e = launch_blockscale<128, 6>(tmA, tmB, tmSA, tmC, args, grid, s);
    if (ws && cudaFreeAsync(ws, s) != cudaSuccess && e == cudaSuccess)
        e = cudaErrorUnknown;
    if (e != cudaSuccess)
        return FP8BS_ERR_LAUNCH;
    t_last_config = config_id(cfg);
    return FP8BS_OK;
}

// MoE leader descriptor (skill card "FlyDSL decode MoE stage-1 blkmap",
// procedure step 2): for every run of k adjacent sort blocks of one expert,
// ceil(k/2) leaders, each the first block of a pair (bit 30 set) or a trailing
// solo block; with pair == 0 every block is its own leader. One CTA scans the
// table in chunks of 1024 blocks: a max-scan of run starts gives each block's
// position in its run, an exclusive sum-scan of the leader flags its slot.
// Blocks whose expert is outside [0, num_experts) are no one's leader.
constexpr int kScanThreads = 1024;

__device__ __forceinline__ int block_scan_incl(int v, bool is_max, int *s_warp)
{
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o)
            v = is_max ? (n > v ? n : v) : v + n;
    }
    if (lane == 31)
        s_warp[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int w = s_warp[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o)
                w = is_max ? (n > w ? n : w) : w + n;
        }
        s_warp[lane] = w;
    }
    __syncthreads();
    if (warp > 0) {
        const int p = s_warp[warp - 1];
        v = is_max ? (p > v ? p : v) : v + p;
    }
    __syncthreads();   // s_warp is reused by the next scan
    return v;
}

__global__ void __launch_bounds__(kScanThreads) moe_leaders_kernel(const int *__restrict__ block_expert, int n_blocks,
                                                                    int num_experts, int pair,
                                                                    int *__restrict__ leaders,
                                                                    int *__restrict__ n_leaders)
{
    __shared__ int s_warp[32];
    __shared__ int s_count, s_start;
    if (threadIdx.x == 0) {
        s_count = 0;
        s_start = 0;
    }
    __syncthreads();
    for (int base = 0; base < n_blocks; base += kScanThreads) {
        const int b = base + static_cast<int>(threadIdx.x);
        const bool in = b < n_blocks;
        const int e = in ? block_expert[b] : -1;
        const bool starts = in && (b == 0 || block_expert[b - 1] != e);
        const int carry_start = s_start;
        const int carry_count = s_count;
        int run_start = block_scan_incl(starts ? b : -1, true, s_warp);
        run_start = run_start > carry_start ? run_start : carry_start;
        const bool valid = in && e >= 0 && e < num_experts;
        const bool leader = valid && (!pair || ((b - run_start) & 1) == 0);
        const bool two = leader && pair && b + 1 < n_blocks && block_expert[b + 1] == e;
        const int incl = block_scan_incl(leader ? 1 : 0, false, s_warp);
        if (leader)
            leaders[carry_count + incl - 1] = b | (two ? (1 << 30) : 0);
        if (threadIdx.x == kScanThreads - 1) {
            s_count = carry_count + incl;
            s_start = run_start;
        }
        __syncthreads();
    }
    if (threadIdx.x == 0)
        *n_leaders = s_count;
}

// Grouped blockscale GEMM over the leaders (one-CTA kernel, one CTA per tile).
int moe_gemm(const void *A, const float *a_scale, const void *B, const float *b_scale, void *C,
             const int *block_expert, const int *leaders, const int *n_leaders, int n_blocks, int N, int K,
             int num_experts, void *stream)
{
    if (n_blocks < 0 || n_blocks > (1 << 24) || num_experts < 1 || num_experts > (1 << 16))
        return FP8BS_ERR_SHAPE;
    const long long M_pad = static_cast<long long>(n_blocks) * kMoeBlockRows;
    int rc = check_shape(static_cast<int>(M_pad), N, K);
    if (rc)
        return rc;
    if (static_cast<long long>(num_experts) * N >= (1ll << 31))
        return FP8BS_ERR_SHAPE;
    if (n_blocks == 0)
        return FP8BS_OK;
    if (!A || !a_scale || !B || !b_scale || !C || !block_expert || !leaders || !n_leaders)
        return FP8BS_ERR_NULL;
    if (!aligned(A, 16) || !aligned(a_scale, 16) || !aligned(B, 16) || !aligned(b_scale, 4) || !aligned(C, 16) ||
        !aligned(block_expert, 4) || !aligned(leaders, 4) || !aligned(n_leaders, 4))
        return FP8BS_ERR_ALIGN;
    int dev;
    DeviceState *st;
    if ((rc = ensure_device(dev, st)))
        return rc;
    const int M = static_cast<int>(M_pad);
    // Tile width: 128 unless all-paired leaders give more than four waves of
    // 256-wide tiles. At decode sizes the grouped GEMM streams expert weights
    // and the narrow tile balances the waves better (same session, paired
    // segment: 256 tokens x top-8 of 32 experts, N 1536, K 2048: 43.1 -> 39.8 us;
    // 1024 tokens, skewed: 57.5 -> 56.3 us).
    Config cfg;
    cfg.kind = 1;
    cfg.raster = 0;
    cfg.sched = 1;
    cfg.block_n = 256;
    cfg.stages = 4;
    if (static_cast<long long>((n_blocks + 1) / 2) * ((N + 255) / 256) <= 4ll * st->num_sms) {
        cfg.block_n = 128;
        cfg.stages = 6;
    }
    if (!override_config(1, 1, cfg) || cfg.sched != 1)
        return FP8BS_ERR_SHAPE;
    const int KB = K / 128;
    const uint64_t ld_sa = static_cast<uint64_t>(fp8bs_a_scale_ld(M));
    CUtensorMap tmA, tmB, tmSA, tmC;
    if (!encode_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, K, M, K, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, K, static_cast<uint64_t>(num_experts) * N, K, 128,
                   cfg.block_n, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tmSA, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a_scale, ld_sa, KB, ld_sa * 4, 128, 1,
                   CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_2d(&tmC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, C, N, M, static_cast<uint64_t>(N) * 2, kCChunkCols, 32,
                   CU_TENSOR_MAP_SWIZZLE_64B))
        return FP8BS_ERR_LAUNCH;
    GemmArgs args = {};
    args.M = M;
    args.N = N;
    args.K = K;
    args.raster.m_tiles = (M + kBlockM - 1) / kBlockM;
    args.raster.n_tiles = (N + cfg.block_n - 1) / cfg.block_n;
    args.raster.raster = 0;
    args.raster.group = 1;   // unused: the grouped mode orders tiles by leader
    args.b_scale = b_scale;
    args.status = st->status_ptr;
    args.wait_limit_ns = g_wait_limit_ns.load();
    args.teardown_limit_ns = teardown_limit();
    args.moe_leaders = leaders;
    args.moe_n_leaders = n_leaders;
    args.moe_block_expert = block_expert;
    args.moe_n_tiles = args.raster.n_tiles;
    args.moe_n_blocks = n_blocks;
    args.moe_num_experts = num_experts;
    // Persistent grid for the worst case (every block a solo leader); CTAs
    // beyond the device-side tile count find no work.
    const long long worst = static_cast<long long>(n_blocks) * args.moe_n_tiles;
    const int grid = worst < st->num_sms ? static_cast<int>(worst) : st->num_sms;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaError_t e = cfg.block_n == 256 ? launch_blockscale_moe<256, 4>(tmA, tmB, tmSA, tmC, args, grid, s)
                                             : launch_blockscale_moe<128, 6>(tmA, tmB, tmSA, tmC, args, grid, s);
    if (e != cudaSuccess)
        return FP8BS_ERR_LAUNCH;
    t_last_config = config_id(cfg);
    return FP8BS_OK;
}

} // namespace host
} // namespace fp8bs

using namespace fp8bs;
using namespace fp8bs::host;

extern "C" {

int fp8bs_gemm(const void *A, const float *a_scale, const void *B, const float *b_scale, void *C, int M, int N,
               int K, void *stream)
{
    return blockscale_gemm(A, a_scale, B, b_scale, C, false, 1.f, M, N, K, stream);
}

int fp8bs_gemm_e4m3out(const void *A, const float *a_scale, const void *B, const float *b_scale, void *C8,
                       float c_scale, int M, int N, int K, void *stream)
{
    return blockscale_gemm(A, a_scale, B, b_scale, C8, true, c_scale, M, N, K, stream);
}

static int mx_gemm_packed_any(const void *A, const uint8_t *a_sf, const void *B, const uint8_t *b_sf, void *C,
                              bool c_e4m3, float c_scale, int M, int N, int K, void *stream)
{
    int rc = check_shape(M, N, K);
    if (rc)
        return rc;
    if (c_e4m3 && (N % 16) != 0)
        return FP8BS_ERR_SHAPE;
    if (M == 0)
        return FP8BS_OK;
    if (!A || !a_sf || !B || !b_sf || !C)
        return FP8BS_ERR_NULL;
    if (!aligned(A, 16) || !aligned(a_sf, 16) || !aligned(B, 16) || !aligned(b_sf, 16) || !aligned(C, 16))
        return FP8BS_ERR_ALIGN;
    int dev;
    DeviceState *st;
    if ((rc = ensure_device(dev, st)))
        return rc;
    Config cfg = choose_config(2, M, N, K, st->num_sms);
    if (!override_config(2, 5, cfg, 6))
        return FP8BS_ERR_SHAPE;
    if ((rc = launch_mx(cfg, A, a_sf, B, b_sf, C, M, N, K, 1.f, st->status_ptr, st->num_sms, st->mx_pair_clusters,
                        st->pool, static_cast<cudaStream_t>(stream), c_e4m3, c_scale)))
        return rc;
    t_last_config = config_id(cfg);
    return FP8BS_OK;
}

int fp8mx_gemm_packed(const void *A, const uint8_t *a_sf, const void *B, const uint8_t *b_sf, void *C, int M,
                      int N, int K, void *stream)
{
    return mx_gemm_packed_any(A, a_sf, B, b_sf, C, false, 1.f, M, N, K, stream);
}

int fp8bs_moe_leaders(const int *block_expert, int n_blocks, int num_experts, int pair, int *leaders,
                      int *n_leaders, void *stream)
{
    if (n_blocks < 0 || n_blocks > (1 << 24) || num_experts < 1)
        return FP8BS_ERR_SHAPE;
    if (!n_leaders || (n_blocks > 0 && (!block_expert || !leaders)))
        return FP8BS_ERR_NULL;
    if (!aligned(n_leaders, 4) || !aligned(block_expert, 4) || !aligned(leaders, 4))
        return FP8BS_ERR_ALIGN;
    int dev;
    DeviceState *st;
    int rc;
    if ((rc = ensure_device(dev, st)))
        return rc;
    moe_leaders_kernel<<<1, kScanThreads, 0, static_cast<cudaStream_t>(stream)>>>(block_expert, n_blocks,
                                                                                  num_experts, pair ? 1 : 0,
                                                                                  leaders, n_leaders);
    return cudaGetLastError() == cudaSuccess ? FP8BS_OK : FP8BS_ERR_LAUNCH;
}

int fp8bs_moe_gemm(const void *A, const float *a_scale, const void *B, const float *b_scale, void *C,
                   const int *block_expert, const int *leaders, const int *n_leaders, int n_blocks, int N, int K,
                   int num_experts, void *stream)
{
    return moe_gemm(A, a_scale, B, b_scale, C, block_expert, leaders, n_leaders, n_blocks, N, K, num_experts,
                    stream);
}

int fp8bs_gemm_tensorscale(const void *A, const void *B, void *C, int M, int N, int K, float alpha, void *stream)
{
    int rc = check_shape(M, N, K);
    if (rc)
        return rc;
    if (M == 0)
        return FP8BS_OK;
    if (!A || !B || !C)
        return FP8BS_ERR_NULL;
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16))
        return FP8BS_ERR_ALIGN;
    int dev;
    DeviceState *st;
    if ((rc = ensure_device(dev, st)))
        return rc;
    Config cfg = choose_config(4, M, N, K, st->num_sms);
    if (!override_config(4, 4, cfg))
        return FP8BS_ERR_SHAPE;
    if ((rc = launch_mx(cfg, A, nullptr, B, nullptr, C, M, N, K, alpha, st->status_ptr, st->num_sms,
                        st->mx_pair_clusters, st->pool, static_cast<cudaStream_t>(stream))))
        return rc;
    t_last_config = config_id(cfg);
    return FP8BS_OK;
}

int64_t fp8mx_packed_scale_bytes(int rows, int K)
{
    if (rows < 0 || K < 128 || (K % 128) != 0)
        return FP8BS_ERR_SHAPE;
    return static_cast<int64_t>((rows + 127) / 128) * (K / 128) * 512;
}

int fp8mx_pack_scales(const uint8_t *e8m0, uint8_t *packed, int rows, int K, void *stream)
{
    if (rows < 0 || K < 128 || (K % 128) != 0 || K > (1 << 20))
        return FP8BS_ERR_SHAPE;
    if (rows == 0)
        return FP8BS_OK;
    if (!e8m0 || !packed)
        return FP8BS_ERR_NULL;
    if (!aligned(e8m0, 4) || !aligned(packed, 16))
        return FP8BS_ERR_ALIGN;
    int dev;
    DeviceState *st;
    int rc = ensure_device(dev, st);
    if (rc)
        return rc;
    return launch_pack_scales(e8m0, packed, rows, e8m0, packed, 0, K, st->num_sms, static_cast<cudaStream_t>(stream));
}

static int mx_gemm_any(const void *A, const uint8_t *a_e8m0, const void *B, const uint8_t *b_e8m0, void *C,
                       bool c_e4m3, float c_scale, int M, int N, int K, void *stream)
{
    int rc = check_shape(M, N, K);
    if (rc)
        return rc;
    if (c_e4m3 && (N % 16) != 0)
        return FP8BS_ERR_SHAPE;
    if (M == 0)
        return FP8BS_OK;
    if (!A || !a_e8m0 || !B || !b_e8m0 || !C)
        return FP8BS_ERR_NULL;
    if (!aligned(A, 16) || !aligned(a_e8m0, 4) || !aligned(B, 16) || !aligned(b_e8m0, 4) || !aligned(C, 16))
        return FP8BS_ERR_ALIGN;
    int dev;
    DeviceState *st;
    if ((rc = ensure_device(dev, st)))
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t a_bytes = static_cast<size_t>(fp8mx_packed_scale_bytes(M, K));
    const size_t b_bytes = static_cast<size_t>(fp8mx_packed_scale_bytes(N, K));
    void *ws = nullptr;
    if (cudaMallocFromPoolAsync(&ws, a_bytes + b_bytes, st->pool, s) != cudaSuccess)
        return FP8BS_ERR_CUDA;
    uint8_t *a_sf = static_cast<uint8_t *>(ws);
    uint8_t *b_sf = a_sf + a_bytes;
    rc = launch_pack_scales(a_e8m0, a_sf, M, b_e8m0, b_sf, N, K, st->num_sms, s);
    if (rc == FP8BS_OK)
        rc = mx_gemm_packed_any(A, a_sf, B, b_sf, C, c_e4m3, c_scale, M, N, K, stream);
    if (cudaFreeAsync(ws, s) != cudaSuccess && rc == FP8BS_OK)
        rc = FP8BS_ERR_CUDA;
    return rc;
}

int fp8mx_gemm(const void *A, const uint8_t *a_e8m0, const void *B, const uint8_t *b_e8m0, void *C, int M, int N,
               int K, void *stream)
{
    return mx_gemm_any(A, a_e8m0, B, b_e8m0, C, false, 1.f, M, N, K, stream);
}

int fp8mx_gemm_e4m3out(const void *A, const uint8_t *a_e8m0, const void *B, const uint8_t *b_e8m0, void *C8,
                       float c_scale, int M, int N, int K, void *stream)
{
    return mx_gemm_any(A, a_e8m0, B, b_e8m0, C8, true, c_scale, M, N, K, stream);
}

int64_t fp8bs_a_scale_ld(int M) { return (static_cast<int64_t>(M) + 3) / 4 * 4; }

int64_t fp8bs_a_scale_index(int m, int kb, int M) { return static_cast<int64_t>(kb) * fp8bs_a_scale_ld(M) + m; }

int64_t fp8bs_b_scale_index(int n, int kb, int K) { return static_cast<int64_t>(n / 128) * (K / 128) + kb; }

int64_t fp8mx_scale_index(int r, int g, int K) { return static_cast<int64_t>(r) * (K / 32) + g; }

int fp8mx_sf_atom_offset(int r, int j) { return sf_atom_offset(r, j); }

int fp8bs_pack_a_scale(const float *a_scale_rowmajor, float *a_scale_kmajor, int M, int K, void *stream)
{
    if (M < 0 || K < 128 || (K % 128) != 0 || K > (1 << 20))
        return FP8BS_ERR_SHAPE;
    if (M == 0)
        return FP8BS_OK;
    if (!a_scale_rowmajor || !a_scale_kmajor)
        return FP8BS_ERR_NULL;
    if (!aligned(a_scale_rowmajor, 4) || !aligned(a_scale_kmajor, 16))
        return FP8BS_ERR_ALIGN;
    int dev;
    DeviceState *st;
    int rc = ensure_device(dev, st);
    if (rc)
        return rc;
    const int KB = K / 128;
    const int64_t ld = fp8bs_a_scale_ld(M);
    const int64_t total = ld * KB;
    int blocks = static_cast<int>((total + 255) / 256);
    if (blocks > st->num_sms * 8)
        blocks = st->num_sms * 8;
    pack_a_scale_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(a_scale_rowmajor, a_scale_kmajor,
                                                                              M, KB, ld);
    return cudaGetLastError() == cudaSuccess ? FP8BS_OK : FP8BS_ERR_LAUNCH;
}

int fp8bs_get_status(void *stream)
{
    int dev;
    DeviceState *st;
    int rc = ensure_device(dev, st);
    if (rc)
        return rc;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return FP8BS_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, st->status_ptr, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return FP8BS_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpy(st->status_ptr, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
            return FP8BS_ERR_CUDA;
    }
    return v == kStatusTimeout ? FP8BS_ERR_DEVICE_TIMEOUT : (v == 0 ? FP8BS_OK : FP8BS_ERR_CUDA);
}

const char *fp8bs_status_string(int status)
{
    switch (status) {
    case FP8BS_OK: return "ok";
    case FP8BS_ERR_NULL: return "null pointer argument";
    case FP8BS_ERR_ALIGN: return "pointer not aligned as required";
    case FP8BS_ERR_SHAPE: return "shape (or configuration id) outside the supported rules";
    case FP8BS_ERR_UNSUPPORTED_DEVICE: return "device is not compute capability 10.3 (sm_103a)";
    case FP8BS_ERR_LAUNCH: return "tensor-map encoding or kernel launch failed";
    case FP8BS_ERR_DEVICE_TIMEOUT: return "a device-side wait exceeded its time limit";
    case FP8BS_ERR_CUDA: return "CUDA runtime error";
    case FP8BS_ERR_SCRATCH_TOO_SMALL:
        return "the packed scales exceed the fixed scratch array of fp8mx_gemm_noalloc";
    default: return "unknown status";
    }
}

int fp8bs_last_config_id(void) { return t_last_config; }

int fp8bs_select_config(int M, int N, int K, int num_sms)
{
    if (check_shape(M, N, K) || num_sms <= 0)
        return FP8BS_ERR_SHAPE;
    return config_id(choose_config(1, M, N, K, num_sms));
}

int fp8mx_select_config(int M, int N, int K, int num_sms)
{
    if (check_shape(M, N, K) || num_sms <= 0)
        return FP8BS_ERR_SHAPE;
    return config_id(choose_config(2, M, N, K, num_sms));
}

int fp8bs_set_raster_group(int group)
{
    if (group < 0 || group > 4096)
        return FP8BS_ERR_SHAPE;
    g_raster_group.store(group ? group : 1);
    return FP8BS_OK;
}

int fp8bs_set_config_override(int config_id)
{
    if (config_id != 0) {
        Config c;
        if (!decode_config_id(config_id, c))
            return FP8BS_ERR_SHAPE;
    }
    g_config_override.store(config_id);
    return FP8BS_OK;
}

int fp8bs_shutdown(void)
{
    std::lock_guard<std::mutex> lock(g_mutex);
    int cur = -1;
    const bool have_cur = cudaGetDevice(&cur) == cudaSuccess;
    int rc = FP8BS_OK;
    for (int d = 0; d < kMaxDevices; ++d) {
        DeviceState &st = g_dev[d];
        if (!st.ready)
            continue;
        if (cudaSetDevice(d) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
            rc = FP8BS_ERR_CUDA;
        if (st.pool && cudaMemPoolDestroy(st.pool) != cudaSuccess)
            rc = FP8BS_ERR_CUDA;
        st = DeviceState();
    }
    if (have_cur)
        cudaSetDevice(cur);
    return rc;
}

int fp8bs_device_info(int *num_sms, int *pair_clusters)
{
    int dev;
    DeviceState *st;
    int rc = ensure_device(dev, st);
    if (rc)
        return rc;
    if (num_sms)
        *num_sms = st->num_sms;
    if (pair_clusters)
        *pair_clusters = st->mx_pair_clusters;
    return FP8BS_OK;
}

int fp8bs_launches_per_call(void) { return 1; }

int fp8mx_launches_per_call(void) { return 2; }

void fp8bs_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns ? ns : kDefaultWaitLimitNs); }

const char *fp8bs_version(void) { return "fp8bs 0.2.0 (sm_103a)"; }

} // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free MXFP8 entry point (fp8mx_gemm_noalloc). Its packed-scale
// scratch is this fixed device array instead of a pool allocation. The array
// exists in every device context that loads the library, until the process
// exits. Host code must not pass the symbol itself to a kernel (on the host it
// only names a stand-in); the set-up below fetches its device address once per
// device with that device current.

namespace fp8bs {
namespace host {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;   // 8 MiB: packed scales of A and B together
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

struct NoAllocDevice {
    bool ready = false;
    int status = FP8BS_OK;
    int num_sms = 0;
    int *status_ptr = nullptr;
    uint8_t *scratch = nullptr;   // device address of g_noalloc_scratch
    int mx_pair_clusters = 0;     // co-resident CTA pairs of the MXFP8 pair kernel (M >= 4096 shapes)
};
NoAllocDevice g_noalloc_dev[kMaxDevices];

// Once per device, with that device current; allocates nothing.
int noalloc_setup(int &dev, NoAllocDevice *&nd)
{
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return FP8BS_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    nd = &g_noalloc_dev[dev];
    if (nd->ready)
        return nd->status;
    nd->ready = true;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nd->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return nd->status = FP8BS_ERR_CUDA;
    if (major != 10 || minor != 3)
        return nd->status = FP8BS_ERR_UNSUPPORTED_DEVICE;
    if (cudaGetSymbolAddress(reinterpret_cast<void **>(&nd->status_ptr), g_status_word) != cudaSuccess)
        return nd->status = FP8BS_ERR_CUDA;
    if (cudaGetSymbolAddress(reinterpret_cast<void **>(&nd->scratch), g_noalloc_scratch) != cudaSuccess ||
        !nd->scratch)
        return nd->status = FP8BS_ERR_CUDA;
    // The shape rule picks the CTA-pair kernel for M >= 4096; its persistent
    // grid is the number of co-resident pairs (an occupancy query, no allocation).
    if (max_mx_pair_clusters<kMxPairStages>(&nd->mx_pair_clusters) != cudaSuccess || nd->mx_pair_clusters < 1)
        return nd->status = FP8BS_ERR_CUDA;
    if (!g_encode) {
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return nd->status = FP8BS_ERR_CUDA;
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    return nd->status = FP8BS_OK;
}

} // namespace host
} // namespace fp8bs

extern "C" {

int64_t fp8mx_noalloc_scratch_bytes(void) { return static_cast<int64_t>(kNoAllocScratchBytes); }

int fp8mx_gemm_noalloc(const void *A, const uint8_t *a_e8m0, const void *B, const uint8_t *b_e8m0, void *C, int M,
                       int N, int K, void *stream)
{
    int rc = check_shape(M, N, K);
    if (rc)
        return rc;
    if (M == 0)
        return FP8BS_OK;
    if (!A || !a_e8m0 || !B || !b_e8m0 || !C)
        return FP8BS_ERR_NULL;
    if (!aligned(A, 16) || !aligned(a_e8m0, 4) || !aligned(B, 16) || !aligned(b_e8m0, 4) || !aligned(C, 16))
        return FP8BS_ERR_ALIGN;
    const size_t a_bytes = static_cast<size_t>(fp8mx_packed_scale_bytes(M, K));
    const size_t b_bytes = static_cast<size_t>(fp8mx_packed_scale_bytes(N, K));
    if (a_bytes + b_bytes > kNoAllocScratchBytes)
        return FP8BS_ERR_SCRATCH_TOO_SMALL;
    int dev;
    NoAllocDevice *nd;
    if ((rc = noalloc_setup(dev, nd)))
        return rc;
    Config cfg = choose_config(2, M, N, K, nd->num_sms);
    if (!override_config(2, 5, cfg, 6))   // the pair and decode kernels need no workspace either
        return FP8BS_ERR_SHAPE;
    cfg.sched = 1;   // stream-K needs a workspace: one CTA per tile here
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *a_sf = nd->scratch;             // every byte used is rewritten by the pack kernel
    uint8_t *b_sf = nd->scratch + a_bytes;   // a_bytes is a multiple of 512
    rc = launch_pack_scales(a_e8m0, a_sf, M, b_e8m0, b_sf, N, K, nd->num_sms, s);
    if (rc)
        return rc;
    if ((rc = launch_mx(cfg, A, a_sf, B, b_sf, C, M, N, K, 1.f, nd->status_ptr, nd->num_sms, nd->mx_pair_clusters,
                        nullptr, s)))
        return rc;
    t_last_config = config_id(cfg);
    return FP8BS_OK;
}

} // extern "C"
