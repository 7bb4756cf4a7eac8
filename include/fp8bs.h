/*
 * fp8bs — FP8 block-scaled GEMM and MXFP8 GEMM for NVIDIA GB300 (sm_103a).
 *
 * C ABI of libfp8bs.so. Plain pointers and sizes only. Device pointers are
 * CUDA device addresses owned by the caller; `stream` is a cudaStream_t passed
 * as void* (NULL = the legacy default stream). Every GEMM call is asynchronous
 * on `stream`, performs no host synchronisation and no allocation after the
 * first call on a device (except the pooled workspaces of fp8mx_gemm and of
 * the stream-K schedule, see fp8bs_gemm), and can be captured in a CUDA graph.
 *
 * Error behaviour: functions return FP8BS_OK (0) or a negative fp8bs_status.
 * Argument errors are detected on the host before anything is launched.
 * A device-side wait that exceeds its time limit does not trap: the kernel
 * records FP8BS_ERR_DEVICE_TIMEOUT in a per-device status word, releases its
 * resources and returns; fp8bs_get_status() reads and clears that word.
 */
#ifndef FP8BS_H
#define FP8BS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP8BS_OK = 0,
    FP8BS_ERR_NULL = -1,               /* a required pointer is NULL                          */
    FP8BS_ERR_ALIGN = -2,              /* a pointer is not 16-byte aligned                    */
    FP8BS_ERR_SHAPE = -3,              /* M, N or K outside the documented shape rules        */
    FP8BS_ERR_UNSUPPORTED_DEVICE = -4, /* current device is not compute capability 10.3       */
    FP8BS_ERR_LAUNCH = -5,             /* the kernel launch or tensor-map encoding failed     */
    FP8BS_ERR_DEVICE_TIMEOUT = -6,     /* a device wait ran out of time (status word)         */
    FP8BS_ERR_CUDA = -7,               /* another CUDA runtime error                          */
    FP8BS_ERR_SCRATCH_TOO_SMALL = -8   /* fp8mx_gemm_noalloc: problem exceeds its fixed scratch */
} fp8bs_status;

/*
 * FP8 block-scaled GEMM (skill card "FlyDSL fp8 blockscale GEMM", sections
 * "When to use" and "Mechanism A"):
 *
 *   C[m,n] = bf16( sum_kb (sum_{k in kb} A[m,k] * B[n,k]) * a_scale[m,kb] * b_scale[n/128,kb] )
 *
 * with 128-wide K blocks kb. The fp8 products are accumulated unscaled per K
 * block and the arbitrary fp32 scales are applied afterwards in fp32 (they are
 * never rounded to powers of two).
 *
 *   A        E4M3 (OCP E4M3FN) [M][K] row-major, 16-byte aligned.
 *   a_scale  fp32 [K/128][fp8bs_a_scale_ld(M)], K-block-major ("transposed
 *            contiguous [scale_k, M]", skill card section "Procedure" step 6):
 *            a_scale[m,kb] is at kb*fp8bs_a_scale_ld(M) + m. 16-byte aligned.
 *   B        E4M3 [N][K] row-major (the weight, K contiguous), 16-byte aligned.
 *   b_scale  fp32 [ceil(N/128)][K/128] row-major ("[scale_n, scale_k]"), 4-byte aligned.
 *   C        bf16 [M][N] row-major, written (never read), 16-byte aligned.
 *
 * Shape rules: M >= 1; N >= 8 and N % 8 == 0; K >= 128, K % 128 == 0 and
 * K <= 1048576. Otherwise FP8BS_ERR_SHAPE. M = 0 is a no-op returning FP8BS_OK.
 * A partial last N block of 128 rows uses its own b_scale row.
 *
 * Schedule: one CTA per output tile, or, when that shortens the longest CTA's
 * loop by at least 20 K blocks (a partial last wave of tiles, or few tiles
 * with a long K), stream-K: the (tile, K block) units are split
 * evenly over the CTAs and a tile cut between CTAs is summed in fp32 from their
 * scaled partials (the same sum in another order). Stream-K takes a workspace
 * of grid * (128 * 256 * 4 + 64) bytes from a stream-ordered memory pool,
 * allocated and freed on `stream` around the launch (allocation failure:
 * FP8BS_ERR_CUDA). Inside a CUDA graph that workspace is reused by every
 * replay; a replay that ends in FP8BS_ERR_DEVICE_TIMEOUT leaves the results of
 * later replays of the same graph undefined.
 */
int fp8bs_gemm(const void *A, const float *a_scale, const void *B, const float *b_scale, void *C,
               int M, int N, int K, void *stream);

/*
 * fp8bs_gemm with an E4M3 C (epilogue fusion that halves the C write; the
 * store side of skill card "FlyDSL prefill MoE stage-2 fp8 partial",
 * procedure steps 2 and 5):
 *
 *   C8[m,n] = e4m3( c_scale * sum_kb P_kb[m,n] * a_scale[m,kb] * b_scale[n/128,kb] )
 *
 * The sum is the fp32 value fp8bs_gemm rounds to bf16; it is multiplied by
 * c_scale in fp32 and rounded to the nearest E4M3FN value (ties to even),
 * saturating at +-448 (a NaN stays NaN). A consumer recovers the value as
 * decode(C8) / c_scale: c_scale is the single source of truth for both sides,
 * passed as an argument (choose it so that |C| * c_scale sits mid-range in
 * E4M3, e.g. 16 / rms(C)).
 *   C8  E4M3 [M][N] row-major, written, 16-byte aligned.
 * Other arguments, schedule and errors as fp8bs_gemm; in addition N % 16 == 0
 * (FP8BS_ERR_SHAPE otherwise).
 */
int fp8bs_gemm_e4m3out(const void *A, const float *a_scale, const void *B, const float *b_scale, void *C8,
                       float c_scale, int M, int N, int K, void *stream);

/*
 * MXFP8 GEMM (PR "1x32 ue8m0 (MXFP8) 8-wave FlyDSL GEMM for gfx950", sections
 * "Why it is faster" and "Correctness"): both operands E4M3 with one ue8m0
 * scale 2^(e-127) per row and 32-wide K group g = k/32:
 *
 *   C[m,n] = bf16( sum_k A[m,k]*2^(a_e8m0[m,g]-127) * B[n,k]*2^(b_e8m0[n,g]-127) )
 *
 *   A       E4M3 [M][K] row-major, 16-byte aligned.
 *   a_e8m0  uint8 [M][K/32] row-major (the quantiser's own layout), 4-byte aligned.
 *   B       E4M3 [N][K] row-major, 16-byte aligned.
 *   b_e8m0  uint8 [N][K/32] row-major, 4-byte aligned.
 *   C       bf16 [M][N] row-major, written, 16-byte aligned.
 *
 * Shape rules as fp8bs_gemm. The scale bytes 0xFF (NaN) are outside the
 * contract. This entry point and fp8bs_gemm are deliberately separate: the
 * two scale formats cannot be told apart by shape or dtype.
 *
 * Launches two kernels on `stream`: fp8mx_pack_scales for both scale tensors
 * (into a workspace taken from a library-owned stream-ordered memory pool and
 * returned to it on the same stream; the pool keeps the memory between calls),
 * then the GEMM of fp8mx_gemm_packed.
 */
int fp8mx_gemm(const void *A, const uint8_t *a_e8m0, const void *B, const uint8_t *b_e8m0, void *C,
               int M, int N, int K, void *stream);

/*
 * fp8mx_gemm with an E4M3 C: C8[m,n] = e4m3(c_scale * the fp32 sum), rounded
 * and saturated as fp8bs_gemm_e4m3out; N % 16 == 0. Other arguments, launches
 * and errors as fp8mx_gemm, except that it always runs one CTA per tile (a
 * stream-K configuration, chosen or forced, runs as its one-per-tile twin and
 * is reported so).
 */
int fp8mx_gemm_e4m3out(const void *A, const uint8_t *a_e8m0, const void *B, const uint8_t *b_e8m0, void *C8,
                       float c_scale, int M, int N, int K, void *stream);

/*
 * MXFP8 GEMM on scale factors already in the packed layout (one kernel; no
 * allocation except the stream-K workspace, chosen as for fp8bs_gemm when it
 * saves at least 13 K steps of 128, same size, pool and graph caveat). The PR above keeps its scale shuffles as separate weight-prep
 * helpers for the same reason: the kernel wants a layout the quantiser does
 * not produce.
 *   a_sf  fp8mx_packed_scale_bytes(M, K) bytes, 16-byte aligned, from fp8mx_pack_scales.
 *   b_sf  fp8mx_packed_scale_bytes(N, K) bytes, 16-byte aligned.
 * Other arguments as fp8mx_gemm.
 */
int fp8mx_gemm_packed(const void *A, const uint8_t *a_sf, const void *B, const uint8_t *b_sf, void *C,
                      int M, int N, int K, void *stream);

/*
 * Promote-free ceiling twin of fp8bs_gemm (skill card "FlyDSL fp8 blockscale
 * GEMM", section "Bottleneck diagnosis": the same kernel with one per-tensor
 * scale, i.e. identical MMA work):
 *
 *   C[m,n] = bf16( alpha * sum_k A[m,k] * B[n,k] )
 *
 * A, B, C and the shape rules as fp8bs_gemm; alpha is one fp32 scale. The
 * fp32 sums run over the whole K extent in tensor memory and alpha is applied
 * once in the epilogue. Comparing its time with fp8bs_gemm's on the same shape
 * measures the cost of the per-block software scaling. One kernel; config ids
 * of kind 4 (the MXFP8 kernel's tiles, fp8bs_gemm's schedule rule and
 * stream-K workspace).
 */
int fp8bs_gemm_tensorscale(const void *A, const void *B, void *C, int M, int N, int K, float alpha,
                           void *stream);

/*
 * Grouped MoE stage-1 (gate+up) blockscale GEMM with paired same-expert sort
 * blocks (skill card "FlyDSL decode MoE stage-1 blkmap", sections "Mechanism"
 * and "Procedure" steps 2-5).
 *
 * Layout. The routed token rows are sorted by expert and each expert's rows are
 * padded up to whole sort blocks of FP8BS_MOE_BLOCK_ROWS (64) rows, as the MoE
 * align/sort step produces them: n_blocks blocks, M = 64 * n_blocks rows.
 *   block_expert  int32 [n_blocks], device: the expert of each block. Blocks of
 *                 one expert are adjacent. A value outside [0, num_experts)
 *                 (e.g. -1 for unused blocks) marks a block that is not
 *                 computed and whose C rows are left as they are.
 *   A, a_scale    the sorted rows, as fp8bs_gemm with M = 64 * n_blocks.
 *   B             E4M3 [num_experts][N][K], 16-byte aligned.
 *   b_scale       fp32 [num_experts][ceil(N/128)][K/128].
 *   C             bf16 [M][N]: row r of block b is
 *                 fp8bs_gemm(A[r], a_scale[r], B[block_expert[b]], b_scale[block_expert[b]]).
 *
 * fp8bs_moe_leaders writes the leader descriptor, one kernel, device-side and
 * graph-safe (no host synchronisation): for every run of k adjacent blocks of
 * one expert, ceil(k/2) leaders, each the first block of a pair (value b |
 * 1 << 30) or a trailing solo block (value b); with pair == 0 every block is a
 * solo leader (the unpaired arm). leaders: int32 [n_blocks] capacity;
 * n_leaders: one int32, the count. Errors: FP8BS_ERR_SHAPE (n_blocks < 0 or
 * > 2^24, num_experts < 1), FP8BS_ERR_NULL, FP8BS_ERR_ALIGN.
 *
 * fp8bs_moe_gemm computes C from the descriptor (which must come from
 * fp8bs_moe_leaders for the same block_expert): one 128-row compute tile per
 * leader and N tile, so a pair streams its expert's B tile once for both
 * blocks; a solo leader's second 64 rows belong to the next block and are not
 * stored. One kernel, a persistent grid sized for n_blocks solo leaders that
 * reads the leader count on the device. Shape rules as fp8bs_gemm for
 * (64 * n_blocks, N, K), num_experts * N < 2^31; n_blocks = 0 is a no-op.
 */
#define FP8BS_MOE_BLOCK_ROWS 64
int fp8bs_moe_leaders(const int *block_expert, int n_blocks, int num_experts, int pair, int *leaders,
                      int *n_leaders, void *stream);
int fp8bs_moe_gemm(const void *A, const float *a_scale, const void *B, const float *b_scale, void *C,
                   const int *block_expert, const int *leaders, const int *n_leaders, int n_blocks, int N,
                   int K, int num_experts, void *stream);

/* Size in bytes of the packed scale layout of a [rows][K/32] ue8m0 tensor:
 * ceil(rows/128) * (K/128) * 512. Negative (FP8BS_ERR_SHAPE) for bad shapes. */
int64_t fp8mx_packed_scale_bytes(int rows, int K);

/*
 * Repack ue8m0 bytes [rows][K/32] (row-major, 4-byte aligned, device) into the
 * packed layout (device, 16-byte aligned): for 128-row block rb and 128-wide K
 * step ks a 512-byte atom at byte ((rb * (K/128)) + ks) * 512, in which byte j
 * (K group 4*ks + j) of row rb*128 + r sits at fp8mx_sf_atom_offset(r, j);
 * rows past `rows` are zero. Asynchronous on `stream`, one kernel.
 */
int fp8mx_pack_scales(const uint8_t *e8m0, uint8_t *packed, int rows, int K, void *stream);

/*
 * MXFP8 GEMM that allocates nothing (the source pages have no counterpart;
 * this is a library-integration entry point). Same arguments, result and
 * shape rules as fp8mx_gemm.
 *
 * For callers that must not allocate device memory on the calling path:
 * engines that reserve all device memory up front and own the allocator (an
 * allocation here could fail or fragment their arena), plugins inside a host
 * framework that hands them no allocator, and code on latency-critical paths
 * that forbids allocator calls. fp8mx_gemm takes its packed-scale workspace
 * from a memory pool; this entry point uses a fixed device array of
 * fp8mx_noalloc_scratch_bytes() bytes (8 MiB) built into the library instead,
 * which every GPU that loads the library holds until the process exits. It
 * always runs one CTA per tile (stream-K would need a workspace); the CTA-pair
 * kernel (chosen from M = 4096 as in fp8mx_gemm, or forced) and the MXFP8
 * decode kernel (config 6128601, by override), which need none, run too.
 *
 * Limit: fp8mx_packed_scale_bytes(M, K) + fp8mx_packed_scale_bytes(N, K) must
 * not exceed that size, else FP8BS_ERR_SCRATCH_TOO_SMALL (checked on the host,
 * before anything runs). All calls share the one array: two calls whose kernels
 * overlap on the GPU (e.g. on different streams without ordering between them)
 * race on it. The first call on a device looks up the array's device address
 * and the CTA-pair kernel's co-resident cluster count (no allocation), with no
 * other call of this library needed before it; make that first call before any
 * stream capture.
 * Launches two kernels on `stream` (scale pack, GEMM), like fp8mx_gemm.
 */
int fp8mx_gemm_noalloc(const void *A, const uint8_t *a_e8m0, const void *B, const uint8_t *b_e8m0, void *C,
                       int M, int N, int K, void *stream);
/* Size in bytes of the fixed scratch array fp8mx_gemm_noalloc uses (8 MiB). */
int64_t fp8mx_noalloc_scratch_bytes(void);

/* ---- layout helpers (bit-exact; host functions, no CUDA calls) ---------- */

/* Leading dimension of the K-block-major a_scale: M rounded up to 4 (a
 * multiple of 16 bytes, as the tensor-memory-access unit requires). */
int64_t fp8bs_a_scale_ld(int M);
/* Element offset of logical a_scale[m,kb] in the K-block-major buffer. */
int64_t fp8bs_a_scale_index(int m, int kb, int M);
/* Element offset of the scale that applies to B row n in K block kb. */
int64_t fp8bs_b_scale_index(int n, int kb, int K);
/* Element offset of the ue8m0 byte for row r and 32-wide K group g. */
int64_t fp8mx_scale_index(int r, int g, int K);
/* Byte offset, inside one 512-byte scale-factor atom (128 rows x 4 groups),
 * at which the MXFP8 kernel stages the byte of row r (0..127) and group j
 * (0..3) before copying the atom to tensor memory: (r%32)*16 + (r/32)*4 + j. */
int fp8mx_sf_atom_offset(int r, int j);

/* Repack a row-major logical a_scale [M][K/128] (device) into the
 * K-block-major layout above (device, fp8bs_a_scale_ld(M)*(K/128) floats,
 * padding rows zeroed). Asynchronous on `stream`. */
int fp8bs_pack_a_scale(const float *a_scale_rowmajor, float *a_scale_kmajor, int M, int K, void *stream);

/* ---- status and introspection ---------------------------------------------- */

/* Synchronises `stream`, then returns and clears the current device's status
 * word: FP8BS_OK, FP8BS_ERR_DEVICE_TIMEOUT, or FP8BS_ERR_CUDA if the
 * synchronisation itself failed. */
int fp8bs_get_status(void *stream);
/* Static string for a status code. */
const char *fp8bs_status_string(int status);
/* Identifier of the kernel configuration the last successful GEMM call on this
 * host thread launched (0 if none): kind*1000000 + block_n*1000 + stages*100 +
 * raster*10 + schedule; kind 1 = one-CTA blockscale kernel (128 x block_n
 * tiles), 2 = mxfp8 kernel, 3 = CTA-pair blockscale kernel (256 x 256 tiles
 * over two SMs, four stages and a whole-tile C buffer: 3256401 / 3256411 one
 * CTA pair per tile, chosen for bf16 C with one CTA per tile from M = 2048;
 * 3256402 / 3256412 stream-K with the pair as the worker, bf16 C only,
 * selectable by fp8bs_set_config_override, never chosen by the shape rule),
 * 4 = tensor-scale twin (fp8bs_gemm_tensorscale), 5 = CTA-pair
 * mxfp8 kernel (256 x 256 tiles over two SMs), 6 = mxfp8 decode kernel
 * (6128601 only; selectable by fp8bs_set_config_override, never chosen by the
 * shape rule: M <= 128, the K steps of each 128-column tile cut into up to 8
 * slices that run as one thread-block cluster and add their fp32 partials in
 * distributed shared memory, in slice order, so the result is the same on
 * every call; a shape it does not take (M > 128, K > 6144, an E4M3 C) runs the
 * one-CTA 128-wide kernel and reports 2128601); schedule 1 = one CTA per tile,
 * 2 = stream-K (kinds 1, 2, 3 and 4 with block_n 256, and kind 2 with block_n 128). */
int fp8bs_last_config_id(void);
/* Release what the library holds per device: waits for each device it set
 * up (cudaDeviceSynchronize), destroys its stream-ordered workspace pool and
 * forgets the set-up, which the next call repeats. No call of this library may
 * be in flight on another thread, and CUDA graphs captured earlier must not be
 * replayed afterwards (their stream-K or scale workspaces came from that pool).
 * The fixed scratch of fp8mx_gemm_noalloc and the status words are static and
 * stay. Returns FP8BS_OK, or FP8BS_ERR_CUDA if a step failed (the rest is still
 * released). A no-op when nothing was set up. */
int fp8bs_shutdown(void);
/* Configuration id fp8bs_gemm / fp8mx_gemm would choose for a shape on a
 * device with `num_sms` SMs (host-only, no CUDA calls). */
int fp8bs_select_config(int M, int N, int K, int num_sms);
int fp8mx_select_config(int M, int N, int K, int num_sms);
/* Force the configuration of subsequent GEMM calls in this process (a valid
 * configuration id of the matching kind; 0 restores the shape-based choice).
 * Returns FP8BS_ERR_SHAPE for an id that names no built kernel. For tests and
 * measurements of each kernel variant. */
int fp8bs_set_config_override(int config_id);
/* Tile-order group size of subsequent GEMM launches in this process (1..4096;
 * 0 restores the default 1). The raster visits tiles in groups of `group`
 * panels of the smaller operand and walks the larger operand inside a group,
 * so a group's panels stay resident in L2 while the other operand streams
 * past (skill card "FlyDSL fp8 blockscale GEMM", section "Mechanism B": tile
 * order as an L2-locality lever). Any group size gives the same result. For
 * measurements (the default of 1 is what the configuration ids report).
 * FP8BS_ERR_SHAPE for a value outside that range. */
int fp8bs_set_raster_group(int group);
/* SM count of the current device and the number of two-CTA clusters of the
 * CTA-pair MXFP8 kernel that can be resident at once (its persistent grid size). */
int fp8bs_device_info(int *num_sms, int *pair_clusters);
/* Number of kernels one fp8bs_gemm call launches (1). */
int fp8bs_launches_per_call(void);
/* Number of kernels one fp8mx_gemm call launches (2: scale pack + GEMM). */
int fp8mx_launches_per_call(void);
/* Set the per-wait device time limit in nanoseconds (default 2e9) used by
 * subsequent launches from this process; 0 restores the default. A pipeline
 * wait that exceeds it makes the kernel record FP8BS_ERR_DEVICE_TIMEOUT, stop
 * issuing work, wait (with a limit of at least the default) for the copies and
 * MMAs it already issued, free its tensor memory and return. */
void fp8bs_set_wait_limit_ns(uint64_t ns);
/* Library version string. */
const char *fp8bs_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8BS_H */
