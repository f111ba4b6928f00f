/*
 * libquads -- NVFP4 W4A4 linear and MoE-expert layers with residual activation
 * compensation, and TRACE rollout-guided rounding, for sm_103a (GB300).
 *
 * Sources for what each call computes (page title, then section):
 *   [QUADS]  "Technical Summary: QUADS - Stabilizing NVFP4 Reinforcement Learning
 *            for MoE via Quantization-error Alignment" (gist.science): section 1
 *            (NVFP4 is a native W4A4 format, E2M1 grid with 8 levels per sign),
 *            2.1 (activation error Delta X_q), 2.2 B "Residual Activation
 *            Compensation" -- "Mechanism" (second-pass quantization of the
 *            high-residual channels, correction added back to the output) and
 *            "Implementation" (top channels by residual magnitude, fused kernels
 *            that keep the native W4A4 GEMM).
 *   [TRACE]  "TRACE: Rollout-Guided Quantization-Aware Training for FP4
 *            Reinforcement Learning of MoE Language Models" (paper.rainbus.top
 *            digest): "NVFP4 与 E2M1 码本" (global scale + per-block scale, round
 *            to nearest), "核心方法" (q_TRACE, Eq. (3)), "MoE 专家路由敏感性"
 *            (router assigns each token a few experts).
 *
 * Conventions for every call:
 *   - Every data pointer is a DEVICE pointer owned by the caller; the library
 *     never allocates device memory.  Calls that need scratch take a caller
 *     buffer `workspace` of at least quads_workspace_size(...) bytes, 16-byte
 *     aligned (QUADS_ERR_MISALIGNED otherwise; any cudaMalloc'd base is).
 *     The R_sel code outputs (`r_codes`) are 16-byte aligned too.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call
 *     only enqueues work on it and returns; no call synchronises the stream.
 *     The layer-path kernels are launched with programmatic stream
 *     serialization (a launch may be set up while the stream's previous kernel
 *     still runs) and each one first waits (griddepcontrol.wait) until every
 *     kernel it depends on in the stream has completed and its writes are
 *     visible, so stream order holds as for ordinary launches, the caller's
 *     own kernels included.
 *   - Host-side argument checks return QUADS_ERR_INVALID_ARG,
 *     QUADS_ERR_UNSUPPORTED_SHAPE or QUADS_ERR_MISALIGNED before anything is
 *     enqueued; a launch failure returns QUADS_ERR_CUDA.  quads_last_error_detail()
 *     gives a one-line reason (per host thread).  Device-side failures (a GEMM
 *     pipeline wait that exceeded its time limit, a device-side shape check)
 *     are latched in a device word read by quads_device_status().
 *   - bf16 tensors are row-major with a leading dimension in elements that is
 *     a multiple of 8; pointers are 16-byte aligned.
 *   - An empty input (rows, tokens or M of 0) is valid: after the shape
 *     checks the call returns QUADS_OK without enqueueing anything, and its
 *     data pointers may then be NULL (as PyTorch gives for empty tensors).
 *     Nothing is written, not even tensor scales.
 *
 * NVFP4 storage:
 *   codes   uint8 [rows, ld_codes]: two E2M1 codes per byte, element 2i of a row
 *           in the low nibble, 2i+1 in the high nibble; code bit 3 is the sign.
 *   scales  one unsigned E4M3 byte per 16 consecutive elements of a row.
 *           QUADS_SCALES_LINEAR: uint8 [rows, cols/16], row-major.
 *           QUADS_SCALES_TCGEN05: the layout the tensor-core block-scaled MMA
 *           reads: rows in blocks of 128, scale columns in blocks of 4; each
 *           (128-row, 4-column) block is 512 contiguous bytes, the blocks are
 *           ordered row-block major, and inside a block the byte of (row r,
 *           scale column c) is at (r % 32) * 16 + ((r / 32) % 4) * 4 + c % 4.
 *           Requires cols % 64 == 0; the buffer holds ceil(rows/128)*128 rows,
 *           padding rows read as scale 0.
 *   tensor scale: one float per row group, s_t = amax / (6 * 448) (1.0 when 0).
 *
 * Rounding (fixed so that GPU and reference agree bit for bit): per 16-block
 * m = max|x|, u = m / (6 s_t), s = E4M3(u) (nearest, ties to even, saturating
 * at 448), d = E4M3value(s) * s_t, code = E2M1(x * (1/d)) (nearest, ties to
 * even, saturating at 6, sign kept), every step one IEEE float32 operation; a
 * block whose d is 0 or whose 1/d overflows gets codes 0.
 */
#ifndef QUADS_H
#define QUADS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QUADS_OK = 0,
  QUADS_ERR_INVALID_ARG = 1,
  QUADS_ERR_UNSUPPORTED_SHAPE = 2,
  QUADS_ERR_MISALIGNED = 3,
  QUADS_ERR_CUDA = 4,
  QUADS_ERR_DEVICE_TIMEOUT = 5,
  QUADS_ERR_DEVICE_CHECK = 6,
  QUADS_ERR_WORKSPACE = 7
} quads_status_t;

enum { QUADS_SCALES_LINEAR = 0, QUADS_SCALES_TCGEN05 = 1 };
enum { QUADS_OUT_F32 = 0, QUADS_OUT_BF16 = 1 };
enum { QUADS_EPILOGUE_NONE = 0, QUADS_EPILOGUE_SWIGLU = 1 };
enum {
  QUADS_OP_QUANTIZE = 0,
  QUADS_OP_SELECT = 1,
  QUADS_OP_GEMM = 2,
  QUADS_OP_MOE_GEMM = 3,
  QUADS_OP_MOE_ROUTE = 4,
  QUADS_OP_QUANTIZE_SELECT = 5,
  QUADS_OP_QUANTIZE_SELECT_GROUPS = 6
};

/* Rows of the score-partial array are chunks of this many consecutive rows. */
#define QUADS_SCORE_CHUNK_ROWS 32
/* The grouped GEMM's row groups (experts) are padded to multiples of this. */
#define QUADS_MOE_ROW_ALIGN 128

/* Library version as major*10000 + minor*100 + patch. */
int quads_version(void);
/* Number of CUDA kernels this library has launched (or recorded into a graph
 * under stream capture) from the calling process since it was loaded. */
uint64_t quads_kernel_launch_count(void);
const char* quads_status_string(quads_status_t s);
/* One-line reason for the last non-OK status returned on this host thread. */
const char* quads_last_error_detail(void);

/*
 * Reads and clears the device-side error word after synchronising `stream`
 * (this call does synchronise).  *device_code = 0 when no kernel reported a
 * problem; QUADS_ERR_DEVICE_TIMEOUT when a GEMM pipeline wait gave up (the
 * kernel then stopped and released its tensor memory); QUADS_ERR_DEVICE_CHECK
 * when a kernel found a device-resident argument out of range (e.g. a group
 * offset that is not a multiple of 32 in score mode).
 */
quads_status_t quads_device_status(void* stream, int32_t* device_code);

/*
 * Test hook for the GEMM's failure path (no counterpart on the pages).  With
 * enable != 0, the next GEMM launch on any device (quads_w4a4_gemm_comp,
 * quads_moe_grouped_gemm or quads_mx_gemm) runs with a 1 ms wait limit and an
 * MMA issuer that issues nothing: its producers fill the ring and their waits
 * for a free stage run out, as do the epilogue's waits for a full
 * accumulator.  The kernel then latches QUADS_ERR_DEVICE_TIMEOUT, lets its
 * copies in flight land, releases its tensor memory and returns; its output
 * is unspecified.  The switch clears itself at that launch.  Nothing faults,
 * traps or hangs: every wait of the kernel is bounded.
 */
void quads_test_gemm_wait_timeout(int32_t enable);

/*
 * Profiling hook (no counterpart on the pages): the next GEMM launch records
 * the stage timeline of its first CTA -- %globaltimer nanoseconds -- into
 * device_buffer, 7 events x 64 entries of uint64 (event e, iteration i at
 * [e*64 + i]): 0 producer got a free stage, 1 scale warp saw the stage's
 * data, 2 scale warp committed its copies, 3 MMA issuer saw the scales,
 * 4 MMA issuer committed the stage, 5 epilogue saw a full accumulator (per
 * tile), 6 epilogue finished a tile.  Unwritten entries keep their contents.
 * The hook clears itself at that launch.
 */
void quads_test_gemm_timeline(uint64_t* device_buffer);

/*
 * GEMM output tile width (no counterpart on the pages: a tuning choice), set
 * process-wide for quads_w4a4_gemm_comp and quads_moe_grouped_gemm.
 *   QUADS_GEMM_TILES_AUTO (default): 128 x 256 tiles for plain products (no
 *     correction) whose N is a multiple of 256, 128 x 128 otherwise;
 *   QUADS_GEMM_TILES_128: always 128 x 128;
 *   QUADS_GEMM_TILES_256: 128 x 256 wherever N is a multiple of 256,
 *     compensated products included (their k-channel correction is then
 *     folded into the single accumulator: its partial sum is scaled by
 *     s_R / s_X in tensor memory before the main MMAs accumulate on top).
 * MXFP4 products always use 128 x 128 tiles.  Results agree within the GEMM
 * tolerance, not bit for bit, across policies.  Returns the previous policy,
 * or -1 (and changes nothing) for an unknown value.
 */
enum { QUADS_GEMM_TILES_AUTO = 0, QUADS_GEMM_TILES_128 = 1, QUADS_GEMM_TILES_256 = 2 };
int32_t quads_set_gemm_tile_policy(int32_t policy);

/* Bytes of scratch the call `op` needs for the given shape (0 if none).
 *   QUADS_OP_QUANTIZE: num_groups floats of tensor amax.
 *   QUADS_OP_SELECT:   rows*k floats (the residual slice) + num_groups floats
 *                      (its amax) + num_groups*cols floats (channel scores).
 *   QUADS_OP_GEMM:     the requantized selected weight columns Q(W_sel):
 *                      n*kpad/2 code bytes + n*kpad/16 scale bytes (+ alignment).
 *   QUADS_OP_MOE_GEMM: the same for num_groups experts.
 *   QUADS_OP_MOE_ROUTE: two int32 per (32-token block, expert): rows = tokens, cols = experts.
 *   QUADS_OP_QUANTIZE_SELECT: 256 bytes of control words + the score partials
 *                      (ceil(rows/32)*cols floats) + cols floats of scores +
 *                      rows*k floats (the residual slice), each 256-byte aligned.
 *   QUADS_OP_QUANTIZE_SELECT_GROUPS: rows*k floats (the residual slice).
 * `cols` is the channel count (K) and `n` the output width (N, unused for the
 * activation-side ops).  kpad = k rounded up to 64 (k <= 256) or to 256. */
size_t quads_workspace_size(int32_t op, int64_t rows, int64_t cols, int64_t n, int32_t k,
                            int32_t num_groups);

/* kpad for a selection of k channels: the width in elements of the stored
 * residual-slice and selected-weight operands (zero codes in the padding). */
int32_t quads_kpad(int32_t k);

/*
 * quads_quantize_nvfp4 -- online RTN quantization of a bf16 activation (or
 * weight) matrix to NVFP4, one tensor scale per row group, optionally with the
 * per-channel residual energy partials used to pick the high-residual channels.
 * [TRACE] "NVFP4 与 E2M1 码本"; [QUADS] 2.1 (Delta X_q) and 2.2 B "Mechanism".
 *
 *   x [rows, cols] bf16, leading dimension ldx (elements).
 *   row_index      nullable; output row r reads input row row_index[r].
 *   group_offsets  nullable ([0, rows] = one group); else device int32
 *                  [num_groups + 1], ascending, first 0, every offset but the
 *                  last a multiple of 32; the last (<= rows) is the number of
 *                  rows processed -- rows past it are neither read nor written,
 *                  so `rows` may be a capacity (e.g. padded expert rows).
 *   group_counts   nullable device int32 [num_groups] (needs group_offsets):
 *                  rows of group g at or past group_offsets[g] +
 *                  group_counts[g] are taken as zero rows -- not read, their
 *                  codes, scale bytes and score partials written as those of
 *                  zeros, and left out of the group's amax (for per-expert rows
 *                  padded to a tile multiple whose padding is zero anyway, the
 *                  quantizer then reads only the real rows).  A count above
 *                  the group's size means every row is real; a count of 0 or
 *                  below, none.
 *   tensor_scale_in nullable device float [num_groups]: use these tensor
 *                  scales instead of computing amax / 2688.
 *   tensor_amax_in nullable device float [num_groups]: the groups' absolute
 *                  maxima, already known (e.g. from the producing GEMM's
 *                  epilogue); s_t = amax / 2688 without another pass over x.
 *   codes [rows, ld_codes] (ld_codes >= cols/2, multiple of 4); scales in
 *                  scale_layout (LINEAR: [rows, cols/16]); tensor_scale_out
 *                  device float [num_groups] (written even when scales are given).
 *   score_partials nullable device float [ceil(rows/32), cols]: entry
 *                  [c, j] = sum over rows 32c..32c+31 (row order) of R^2 with
 *                  R = x - dequant(code), float32 adds, no fused multiply-add.
 *   workspace      >= quads_workspace_size(QUADS_OP_QUANTIZE, ...).
 * cols % 16 == 0 (cols % 64 == 0 for the TCGEN05 scale layout).
 */
quads_status_t quads_quantize_nvfp4(const void* x, int64_t rows, int64_t cols, int64_t ldx,
                                    const int32_t* row_index, const int32_t* group_offsets,
                                    int32_t num_groups, const int32_t* group_counts,
                                    const float* tensor_scale_in,
                                    const float* tensor_amax_in, uint8_t* codes,
                                    int64_t ld_codes, uint8_t* scales,
                                    int32_t scale_layout, float* tensor_scale_out,
                                    float* score_partials, void* workspace,
                                    size_t workspace_bytes, void* stream);

/*
 * quads_qdq_nvfp4 -- the trainer side's W4A16 fake quantization ([QUADS] 2.2 A
 * "Asymmetric Quantization-Aware Training" and 2.1 "Weights": the trainer runs
 * the same quantize-dequantize path as the rollout engine, so every forward
 * pass sees the weights the rollout uses while activations stay bf16).
 * y = bf16(fl(level * d_b)) with the codes, block scales d_b and tensor scale
 * that quads_quantize_nvfp4 produces for the same input (same rules, same
 * bits); the codes and scales can be written in the same pass, for the copy
 * synchronised to the rollout engine.  The backward pass of fake quantization
 * is the identity (straight-through) and needs no call.
 *
 *   x [rows, cols] bf16 (ldx); group_offsets / num_groups / tensor_scale_in as
 *     for quads_quantize_nvfp4 (one tensor scale per group, e.g. per expert).
 *   y [rows, ldy] bf16 (ldy >= cols, multiple of 8; 16-byte aligned).
 *   codes nullable ([rows, ld_codes]); scales (scale_layout) required when
 *     codes is given; tensor_scale_out device float [num_groups].
 *   workspace >= quads_workspace_size(QUADS_OP_QUANTIZE, rows, cols, 0, 0,
 *     num_groups) unless tensor_scale_in is given.
 * cols % 16 == 0.
 */
quads_status_t quads_qdq_nvfp4(const void* x, int64_t rows, int64_t cols, int64_t ldx,
                               const int32_t* group_offsets, int32_t num_groups,
                               const float* tensor_scale_in, void* y, int64_t ldy,
                               uint8_t* codes, int64_t ld_codes, uint8_t* scales,
                               int32_t scale_layout, float* tensor_scale_out, void* workspace,
                               size_t workspace_bytes, void* stream);

/*
 * quads_select_residual_channels -- per row group: channel score = sum of the
 * group's score-partial rows in ascending order (float32); the k channels with
 * the largest score (ties -> lower channel index) returned ascending in
 * sel[g*k .. g*k+k); the residual slice R[:, sel] recomputed from x and the
 * block scales (R = x - dequant(RTN code)), quantized again to NVFP4 with its
 * own tensor scale per group (16-blocks along the selected channels).
 * [QUADS] 2.2 B "Mechanism" and "Implementation" (binary channel mask over the
 * top channels by residual magnitude; here the mask is stored as the sorted
 * index list).
 *
 *   x, rows, cols, ldx, group_offsets, num_groups, group_counts: as for the
 *                  quantizer call that produced `scales`, `tensor_scale` and
 *                  `score_partials` (group_counts nullable, needs group_offsets:
 *                  rows of group g at or past offsets[g] + counts[g] are zero
 *                  rows, not read, and their R is 0).
 *   k              1..cols, multiple of 16.
 *   sel            device int32 [num_groups, k].
 *   scores_out     nullable device float [num_groups, cols].
 *   r_codes        [rows, kpad/2] bytes (kpad = quads_kpad(k)); columns k..kpad
 *                  are written as code 0.
 *   r_scales       r_scale_layout; LINEAR: [rows, kpad/16]; TCGEN05: kpad
 *                  columns, padding blocks 0.
 *   r_tensor_scale device float [num_groups].
 *   workspace      >= quads_workspace_size(QUADS_OP_SELECT, rows, cols, 0, k, num_groups).
 *   sel_ready_event nullable cudaEvent_t (caller-owned, created): recorded on
 *                  `stream` as soon as sel is written, before the residual
 *                  slice is formed, so that work on another stream needing only
 *                  sel (quads_select_weight_channels) can wait on it and
 *                  overlap the rest of this call.  A failed record returns
 *                  QUADS_ERR_CUDA.
 * Requires cols <= 8192.
 */
quads_status_t quads_select_residual_channels(
    const void* x, int64_t rows, int64_t cols, int64_t ldx, const int32_t* group_offsets,
    int32_t num_groups, const int32_t* group_counts, const uint8_t* scales, int32_t scale_layout,
    const float* tensor_scale, const float* score_partials, int32_t k, int32_t* sel,
    float* scores_out, uint8_t* r_codes, uint8_t* r_scales, int32_t r_scale_layout,
    float* r_tensor_scale, void* workspace, size_t workspace_bytes, void* sel_ready_event,
    void* stream);

/*
 * quads_select_residual_channels_noalloc -- the same computation and outputs as
 * quads_select_residual_channels, for callers that cannot allocate device
 * memory and so cannot pass a workspace: e.g. a host runtime that owns every
 * device buffer and forbids allocation while it runs, a framework capturing a
 * CUDA graph with its memory pool frozen, or a process that never links an
 * allocator.  The pages have no counterpart to this call; it only changes where
 * the scratch lives.
 *
 * The scratch is one array compiled into the library (a file-scope __device__
 * variable of QUADS_NOALLOC_SELECT_SCRATCH_BYTES bytes) that every GPU loading
 * the library holds until the process exits.  The call allocates nothing
 * itself: no cudaMalloc/cudaFree and no allocating library routine.
 *   - Shapes whose scratch, quads_workspace_size(QUADS_OP_SELECT, rows, cols, 0,
 *     k, num_groups), exceeds the array are rejected with QUADS_ERR_WORKSPACE.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make that
 *     first call before any stream capture.  The cached address belongs to the
 *     device's context at that time: calls after cudaDeviceReset (or anything
 *     else that replaces the device's primary context) are not supported.
 *   - Argument checks and their status codes are those of
 *     quads_select_residual_channels; a valid shape whose scratch does not fit
 *     the array then returns QUADS_ERR_WORKSPACE.
 *   - Every call on a device uses the same array, which keeps the previous
 *     call's contents (the parts that must start at zero are cleared by each
 *     call).  Calls that overlap on the GPU -- on different streams, or from
 *     different host threads without ordering -- race on it.
 * Arguments are those of quads_select_residual_channels without the workspace
 * and the sel_ready_event.
 */
#define QUADS_NOALLOC_SELECT_SCRATCH_BYTES (32u << 20)
quads_status_t quads_select_residual_channels_noalloc(
    const void* x, int64_t rows, int64_t cols, int64_t ldx, const int32_t* group_offsets,
    int32_t num_groups, const int32_t* group_counts, const uint8_t* scales, int32_t scale_layout,
    const float* tensor_scale, const float* score_partials, int32_t k, int32_t* sel,
    float* scores_out, uint8_t* r_codes, uint8_t* r_scales, int32_t r_scale_layout,
    float* r_tensor_scale, void* stream);

/*
 * quads_quantize_select_nvfp4 -- quads_quantize_nvfp4 (one group, tensor
 * scale from the amax, score partials) followed by
 * quads_select_residual_channels, in one cooperative launch whose five
 * phases (tensor amax; quantization with the residual-energy partials;
 * channel scores; top-k selection and the residual slice R[:, sel]; the
 * second quantization of that slice) are separated by grid-wide barriers, so
 * x is read from HBM once and the second pass over it is served by L2 when x
 * fits there.  [QUADS] 2.2 B "Mechanism" and "Implementation" (the
 * high-residual channels chosen online; the correction path fused).
 * Outputs are those of the two calls, bit for bit: codes, scales
 * (scale_layout), tensor_scale_out[1], sel[k] ascending, scores_out (nullable,
 * [cols]), R_sel codes [rows, kpad/2], scales (r_scale_layout), r_tensor_scale[1].
 * cols % 16 == 0 and cols <= 8192 (cols % 64 for TCGEN05 scales); 16 <= k <=
 * min(cols, 1024), k % 16 == 0.  All blocks must be resident at once (one per
 * SM): the launch is cooperative, and fails with QUADS_ERR_CUDA when the
 * device cannot hold the grid.  A grid barrier that does not complete within
 * 2 s latches QUADS_ERR_DEVICE_TIMEOUT (quads_device_status).
 */
quads_status_t quads_quantize_select_nvfp4(
    const void* x, int64_t rows, int64_t cols, int64_t ldx, int32_t k, uint8_t* codes,
    int64_t ld_codes, uint8_t* scales, int32_t scale_layout, float* tensor_scale_out, int32_t* sel,
    float* scores_out, uint8_t* r_codes, uint8_t* r_scales, int32_t r_scale_layout,
    float* r_tensor_scale, void* workspace, size_t workspace_bytes, void* stream);

/*
 * quads_quantize_select_groups_nvfp4 -- quads_quantize_nvfp4 (row groups,
 * score partials) followed by quads_select_residual_channels (per-group
 * selection) for every group at once, one thread block per group: the
 * group's rows are quantized chunk by chunk, its channel scores kept on chip,
 * its top-k channels chosen and R[:, sel] quantized a second time in the same
 * block, so a group's rows are read from memory once for the quantization and
 * the chunk partials never reach memory.  Groups are independent, so no block
 * waits on another.  [QUADS] 2.2 B "Mechanism" and "Implementation" (the
 * high-residual channels chosen online per input; the correction path fused),
 * [TRACE] "MoE 专家路由敏感性" (one selection per expert).
 * Outputs are those of the two calls with group_counts given, bit for bit:
 * codes [rows, ld_codes] and scales (scale_layout) of the groups' rows,
 * tensor_scale_out[num_groups], sel[num_groups, k] (ascending per group),
 * scores_out (nullable, [num_groups, cols]), R_sel codes [rows, kpad/2] and
 * scales (r_scale_layout), r_tensor_scale[num_groups]; no score partials.
 *   x, rows, cols, ldx   bf16 device rows, row-major; 16 <= cols <= 1024,
 *                        cols % 16 == 0 (cols % 64 for TCGEN05 scales).
 *   group_offsets        device int32 [num_groups+1], ascending, multiples of
 *                        QUADS_SCORE_CHUNK_ROWS (a group that starts elsewhere
 *                        latches QUADS_ERR_DEVICE_CHECK); rows past the last
 *                        offset get zero R_sel codes and scales and keep their
 *                        Q(x) outputs untouched.
 *   group_counts         nullable device int32 [num_groups]: rows of group g at
 *                        or past offsets[g] + counts[g] are zero rows, not read
 *                        (counts are clamped to [0, group size]).
 *   tensor_scale_in / tensor_amax_in  nullable device float [num_groups], at
 *                        most one: the groups' tensor scales, or their amax
 *                        (scale = amax / 2688, 1 when 0); with neither, each
 *                        block takes its group's amax itself.
 *   k                    16 <= k <= cols, k % 16 == 0; kpad = quads_kpad(k).
 *   workspace            >= quads_workspace_size(QUADS_OP_QUANTIZE_SELECT_GROUPS,
 *                        rows, cols, 0, k, num_groups) bytes, device.
 *   sel_ready_event      nullable cudaEvent_t, recorded on the stream after the
 *                        launch (sel is then written).
 * rows * k < 2^31.  Errors as quads_quantize_nvfp4 and
 * quads_select_residual_channels; nothing is launched on a host-side error.
 */
quads_status_t quads_quantize_select_groups_nvfp4(
    const void* x, int64_t rows, int64_t cols, int64_t ldx, const int32_t* group_offsets,
    int32_t num_groups, const int32_t* group_counts, const float* tensor_scale_in,
    const float* tensor_amax_in, int32_t k, uint8_t* codes, int64_t ld_codes, uint8_t* scales,
    int32_t scale_layout, float* tensor_scale_out, int32_t* sel, float* scores_out,
    uint8_t* r_codes, uint8_t* r_scales, int32_t r_scale_layout, float* r_tensor_scale,
    void* workspace, size_t workspace_bytes, void* sel_ready_event, void* stream);

/*
 * quads_w4a4_gemm_comp -- Y = s_a s_w Q(A) Q(W)^T + s_r s_w Q(R_sel) Q(W_sel)^T
 * in one kernel on the tcgen05 block-scaled tensor cores (two TMEM
 * accumulators summed in the epilogue).  [QUADS] 2.2 B "Mechanism" (correction
 * added back to the quantized output) and section 1 (native W4A4 GEMM).
 * Q(W_sel) is either given (w_sel_codes / w_sel_scales, from
 * quads_select_weight_channels, e.g. made on another stream while R_sel is
 * being formed) or built inside the call (into `workspace`) from the
 * column-major copy of the packed weight (quads_weight_columns): the selected
 * columns of DQ(Q(W)) in units of s_w, requantized in 16-blocks along the
 * selection with s_w kept.
 *
 *   A: a_codes [M, K/2], a_scales TCGEN05 (ceil(M/128)*128 rows), a_tensor_scale device [1].
 *   W: w_codes [N, K/2], w_scales TCGEN05, w_tensor_scale device [1];
 *   w_codes_t / w_scales_t: its column-major copy (needed with compensation
 *   unless Q(W_sel) is given; then not read, nor is the workspace).
 *   w_sel_codes [N, kpad/2] / w_sel_scales TCGEN05 over kpad columns: both or
 *   neither (nullable), 16-byte aligned.
 *   r_codes NULL -> plain W4A4 (sel, r_* ignored); else r_codes [M, kpad/2],
 *   r_scales TCGEN05 over kpad columns, r_tensor_scale [1], sel [k] ascending.
 *   y [M, ldy] float32 or bf16 (y_dtype).
 * K % 64 == 0, N % 128 == 0, M >= 0 (M == 0: nothing is enqueued).
 */
quads_status_t quads_w4a4_gemm_comp(int64_t M, int64_t N, int64_t K, const uint8_t* a_codes,
                                    const uint8_t* a_scales, const float* a_tensor_scale,
                                    const uint8_t* w_codes, const uint8_t* w_scales,
                                    const float* w_tensor_scale, const uint8_t* w_codes_t,
                                    const uint8_t* w_scales_t, const uint8_t* w_sel_codes,
                                    const uint8_t* w_sel_scales, const uint8_t* r_codes,
                                    const uint8_t* r_scales, const float* r_tensor_scale,
                                    const int32_t* sel, int32_t k, void* y, int32_t y_dtype,
                                    int64_t ldy, void* workspace, size_t workspace_bytes,
                                    void* stream);

/*
 * quads_moe_grouped_gemm -- the compensated W4A4 product for every expert of an
 * MoE layer in one persistent kernel.  Rows of the A operands are grouped by
 * expert; group e occupies rows [expert_offsets[e], expert_offsets[e+1]) of the
 * padded row space (offsets multiples of 128), of which the first
 * expert_counts[e] are real tokens.
 *
 *   a_codes [rows_capacity, K/2], a_scales TCGEN05; a_tensor_scale [1] or
 *     [num_experts] (a_scale_per_expert).
 *   w_codes [num_experts * N, K/2] (expert e's rows e*N..), w_scales TCGEN05 over
 *     the same num_experts*N rows, w_tensor_scale [num_experts]; w_codes_t /
 *     w_scales_t its column-major copy per expert (needed with compensation
 *     unless w_sel_codes / w_sel_scales [num_experts*N rows over kpad columns,
 *     as quads_select_weight_channels writes them] are given, as in
 *     quads_w4a4_gemm_comp).
 *   r_codes NULL -> plain; else [rows_capacity, kpad/2] + TCGEN05 scales,
 *     r_tensor_scale [1] or [num_experts] (r_scale_per_expert); sel [k] shared
 *     (sel_per_expert = 0) or [num_experts, k].
 *   epilogue NONE: y [rows_capacity, ldy] (F32 or BF16), rows past a group's
 *     count are not written.  SWIGLU: W's 128-row tiles hold 64 gate rows then
 *     the matching 64 up rows; y bf16 [rows_capacity, N/2] gets
 *     silu(g) * u, and padding rows of each group are written as 0.
 *   y_amax nullable device float [num_experts]: set to the largest |stored
 *     output| of each expert (zeroed by this call first) -- the tensor amax
 *     the next quantization needs, computed in the epilogue.
 * N % 128 == 0, K % 64 == 0.
 */
quads_status_t quads_moe_grouped_gemm(
    int32_t num_experts, int64_t rows_capacity, int64_t N, int64_t K,
    const int32_t* expert_offsets, const int32_t* expert_counts, const uint8_t* a_codes,
    const uint8_t* a_scales, const float* a_tensor_scale, int32_t a_scale_per_expert,
    const uint8_t* w_codes, const uint8_t* w_scales, const float* w_tensor_scale,
    const uint8_t* w_codes_t, const uint8_t* w_scales_t, const uint8_t* w_sel_codes,
    const uint8_t* w_sel_scales, const uint8_t* r_codes, const uint8_t* r_scales,
    const float* r_tensor_scale, int32_t r_scale_per_expert,
    const int32_t* sel, int32_t sel_per_expert, int32_t k, int32_t epilogue, void* y,
    int32_t y_dtype, int64_t ldy, float* y_amax, void* workspace, size_t workspace_bytes,
    void* stream);

/*
 * quads_weight_columns -- column-major copy of NVFP4 weights, made once per
 * weight update, from which the selected input channels are gathered with
 * contiguous reads (the selection changes every batch, the weights do not).
 * For each of num_groups stacked matrices of rows_per_group rows:
 *   codes_t [num_groups][cols][rows_per_group/2]: byte (c, n/2) holds the codes
 *     of rows n (low nibble) and n+1 (high nibble) at column c;
 *   scales_t [num_groups][cols/16][rows_per_group]: the block-scale byte.
 * Input: w_codes [num_groups*rows_per_group, cols/2], w_scales TCGEN05.
 * rows_per_group % 128 == 0, cols % 64 == 0.
 */
quads_status_t quads_weight_columns(const uint8_t* w_codes, const uint8_t* w_scales,
                                    int32_t num_groups, int64_t rows_per_group, int64_t cols,
                                    uint8_t* codes_t, uint8_t* scales_t, void* stream);

/*
 * quads_select_weight_channels -- Q(W_sel), the weight side of the correction
 * term ([QUADS] 2.2 B "Mechanism": the selected input channels of the weight,
 * paired with R_sel).  For each of num_groups stacked matrices of
 * rows_per_group rows and each weight row: the selected columns of DQ(Q(W)),
 * exact in units of the group's tensor scale s_w (E2M1 level x E4M3 block
 * scale), requantized in 16-blocks along the selection with tensor scale 1 --
 * the group's s_w is applied by the GEMM.  The same operand the GEMMs build
 * when no Q(W_sel) is given to them; made by its own call so that it can run
 * on another stream while R_sel is formed.
 *
 *   codes_t / scales_t: the column-major copy from quads_weight_columns
 *     (16-byte aligned).
 *   sel [k] shared by every group (sel_per_group = 0) or [num_groups, k];
 *     entries are column indices in [0, cols) (ascending, as
 *     quads_select_residual_channels writes them).
 *   w_sel_codes [num_groups*rows_per_group, kpad/2], w_sel_scales TCGEN05
 *     over kpad columns (both 16-byte aligned), kpad = quads_kpad(k); columns
 *     k..kpad-1 get zero codes and scales.  Caller-owned.
 * rows_per_group % 128 == 0, cols % 64 == 0, 16 <= k <= cols, k % 16 == 0,
 * num_groups <= 65535.
 */
quads_status_t quads_select_weight_channels(int32_t num_groups, int64_t rows_per_group,
                                            int64_t cols, const uint8_t* codes_t,
                                            const uint8_t* scales_t, const int32_t* sel,
                                            int32_t sel_per_group, int32_t k,
                                            uint8_t* w_sel_codes, uint8_t* w_sel_scales,
                                            void* stream);

/*
 * quads_trace_round -- TRACE rollout-guided rounding ([TRACE] "核心方法", Eq. (3)):
 * v = x_train * (1/d) under the rollout block's d; q-/q+ = the signed E2M1
 * levels just below/above v (clamped to +-6); emit whichever is nearer the
 * rollout code's value (a zero result takes the sign of v; a block with
 * rollout d == 0 gives 0x0).
 *
 *   x_train [rows, cols] bf16 (ldx); rollout_codes [rows, ld_codes]; rollout
 *   scales LINEAR [rows, cols/16]; rollout_tensor_scale device [1];
 *   codes_out [rows, ld_codes].
 *   counters nullable device uint64 [3], ADDED to: #(RTN code != rollout code),
 *   #(TRACE code != rollout code), #(RTN mismatches one signed level away),
 *   codes compared by value (+0 == -0).
 *   rows * cols / 8 < 2^31 (else QUADS_ERR_UNSUPPORTED_SHAPE).
 */
quads_status_t quads_trace_round(const void* x_train, int64_t rows, int64_t cols, int64_t ldx,
                                 const uint8_t* rollout_codes, int64_t ld_codes,
                                 const uint8_t* rollout_scales,
                                 const float* rollout_tensor_scale, uint8_t* codes_out,
                                 unsigned long long* counters, void* stream);

/*
 * quads_trace_pack_record -- the compact rollout record of TRACE's
 * mantissa-only mode ([TRACE] "核心方法" second innovation, "方法步骤详情"
 * step 2): of each rollout E2M1 code only its mantissa bit (the low bit of the
 * magnitude) is kept; with the E4M3 block scales (kept as they are, 8 bits per
 * 16 values) the record costs 1.5 bits per value.
 *
 *   rollout_codes [rows, ld_codes] packed codes (4-byte aligned, ld_codes >=
 *     cols/2, multiple of 4).
 *   mantissa_bits [rows, ld_bits] bytes (ld_bits >= cols/8): bit j of byte i of
 *     a row is the mantissa bit of element 8i+j.
 * cols % 16 == 0, rows * cols / 8 < 2^31.
 */
quads_status_t quads_trace_pack_record(const uint8_t* rollout_codes, int64_t rows, int64_t cols,
                                       int64_t ld_codes, uint8_t* mantissa_bits, int64_t ld_bits,
                                       void* stream);

/*
 * quads_trace_round_1bit -- TRACE rounding from the 1-bit record: v = x_train *
 * (1/d_b) under the rollout block's d_b; of the two neighbouring signed E2M1
 * levels of v (clamped to +-6) pick the one whose mantissa bit equals the
 * record's -- adjacent levels have opposite mantissa bits, so this is the
 * rollout's code whenever that code is one of the two neighbours, the
 * off-by-one case that makes one bit enough ([TRACE] "核心方法": over 99% of
 * mismatched values differ by one adjacent code).  v on a level has that level
 * alone; a zero result takes the sign of v; a rollout block with d_b == 0
 * gives 0x0.
 *
 *   x_train [rows, cols] bf16 (ldx, 16-byte aligned); mantissa_bits as written
 *   by quads_trace_pack_record; rollout_scales LINEAR [rows, cols/16];
 *   rollout_tensor_scale device [1]; codes_out [rows, ld_codes] (4-byte aligned).
 *   counters nullable device uint64 [2], ADDED to: #(result != RTN code under
 *   the rollout scale), #(result's mantissa bit != record bit).
 * cols % 16 == 0, rows * cols / 8 < 2^31.
 */
quads_status_t quads_trace_round_1bit(const void* x_train, int64_t rows, int64_t cols,
                                      int64_t ldx, const uint8_t* mantissa_bits, int64_t ld_bits,
                                      const uint8_t* rollout_scales,
                                      const float* rollout_tensor_scale, uint8_t* codes_out,
                                      int64_t ld_codes, unsigned long long* counters,
                                      void* stream);

/*
 * MXFP4 variant ([TRACE] "技术新颖性", "实验结果": the method also runs on
 * MXFP4 W4A4 / W4A8 rollouts).  The pages do not define the format; these calls
 * follow the OCP microscaling definition: blocks of 32 consecutive elements of
 * a row share a power-of-two scale 2^e stored as an E8M0 byte (e + 127), with
 * e = floor(log2(block max)) - 2 clamped to >= -127; elements are the E2M1
 * codes (round to nearest even, saturating at +-6) of x / 2^e.  No tensor
 * scale.  The residual compensation stays NVFP4-only.
 *
 * quads_mx_quantize -- x [rows, cols] bf16 (ldx; 16-byte aligned) -> codes
 *   [rows, ld_codes] (8-byte aligned, ld_codes >= cols/2, multiple of 8) and
 *   E8M0 scale bytes: LINEAR [rows, cols/32] or TCGEN05 (the same 128-row x
 *   4-column atoms as NVFP4, a column being a 32-element block; cols % 128;
 *   padding rows 0).  y_qdq nullable: bf16 [rows, ldy] = level * 2^e (the
 *   trainer's fake quantization in this format).
 *   cols % 32 == 0, rows * cols / 16 < 2^31.
 */
quads_status_t quads_mx_quantize(const void* x, int64_t rows, int64_t cols, int64_t ldx,
                                 uint8_t* codes, int64_t ld_codes, uint8_t* scales,
                                 int32_t scale_layout, void* y_qdq, int64_t ldy, void* stream);

/*
 * quads_mx_gemm -- Y = DQ(A) DQ(W)^T for MXFP4 operands on the block-scaled
 * tensor cores (tcgen05.mma kind::mxf4, E8M0 scales, float32 accumulation).
 *   a_codes [M, K/2], a_scales TCGEN05 (ceil(M/128)*128 rows); w_codes [N, K/2],
 *   w_scales TCGEN05; y [M, ldy] float32 or bf16 (y_dtype).
 *   M >= 0 (0: nothing is enqueued), N % 128 == 0, K % 128 == 0; operands
 *   16-byte aligned.
 */
quads_status_t quads_mx_gemm(int64_t M, int64_t N, int64_t K, const uint8_t* a_codes,
                             const uint8_t* a_scales, const uint8_t* w_codes,
                             const uint8_t* w_scales, void* y, int32_t y_dtype, int64_t ldy,
                             void* stream);

/*
 * quads_trace_round_mx -- TRACE rounding (as quads_trace_round) under an MXFP4
 * rollout: v = x_train / 2^e with the rollout block's E8M0 scale
 * (rollout_scales LINEAR [rows, cols/32]); codes 4-byte aligned.  counters
 * nullable device uint64 [3] as in quads_trace_round.
 *   cols % 32 == 0, rows * cols / 8 < 2^31.
 */
quads_status_t quads_trace_round_mx(const void* x_train, int64_t rows, int64_t cols, int64_t ldx,
                                    const uint8_t* rollout_codes, int64_t ld_codes,
                                    const uint8_t* rollout_scales, uint8_t* codes_out,
                                    unsigned long long* counters, void* stream);

/*
 * quads_moe_route -- router top-k and the token -> expert dispatch plan
 * ([TRACE] "MoE 专家路由敏感性").  Per token: the topk largest logits (ties ->
 * lower expert id), kept in ascending expert order; gate = exp(l - lmax) /
 * sum over the chosen (float32); then per expert the rows of its tokens in
 * ascending token order, each group padded to a multiple of 128 rows.
 *
 *   logits [tokens, num_experts] float32 (num_experts <= 256, topk <= 16).
 *   topk_idx int32 [tokens, topk], gates float32 [tokens, topk].
 *   expert_counts int32 [num_experts], expert_offsets int32 [num_experts + 1].
 *   row_token int32 [rows_capacity] (-1 on padding rows), token_row int32
 *   [tokens, topk] (row of each slot).
 *   rows_capacity >= tokens*topk + num_experts*127 (checked on the host).
 *   workspace >= quads_workspace_size(QUADS_OP_MOE_ROUTE, tokens, num_experts, 0, 0, 1).
 */
quads_status_t quads_moe_route(const float* logits, int32_t tokens, int32_t num_experts,
                               int32_t topk, int32_t* topk_idx, float* gates,
                               int32_t* expert_counts, int32_t* expert_offsets,
                               int32_t* row_token, int32_t* token_row, int64_t rows_capacity,
                               void* workspace, size_t workspace_bytes, void* stream);

/*
 * quads_moe_gather -- copy NVFP4 rows into expert order: row r of the output is
 * row row_token[r] of the input (zeros where row_token[r] < 0), for rows
 * r < expert_offsets[num_experts] (as written by quads_moe_route).  Input
 * scales LINEAR, output scales TCGEN05 (the grouped GEMM's operand layout).
 *   in_codes [tokens, cols/2] -> out_codes [rows_capacity, cols/2];
 *   in_scales [tokens, cols/16] -> out_scales TCGEN05 (cols % 64 == 0).
 * Codes and out_scales 16-byte aligned, in_scales 4-byte aligned, else
 * QUADS_ERR_MISALIGNED.
 */
quads_status_t quads_moe_gather(const int32_t* row_token, const int32_t* expert_offsets,
                                int32_t num_experts, int64_t rows_capacity, int64_t cols,
                                const uint8_t* in_codes, const uint8_t* in_scales,
                                uint8_t* out_codes, uint8_t* out_scales, void* stream);

/*
 * quads_moe_combine -- out[t] = bf16( sum_j gates[t, j] * y[token_row[t, j]] )
 * in float32, j ascending (ascending expert id).  y bf16 [rows, ldy].
 * hidden, ldy and ldo multiples of 8 (QUADS_ERR_UNSUPPORTED_SHAPE); y and
 * out 16-byte aligned (QUADS_ERR_MISALIGNED).
 */
quads_status_t quads_moe_combine(const void* y, int64_t ldy, const int32_t* token_row,
                                 const float* gates, int32_t tokens, int32_t topk,
                                 int64_t hidden, void* out, int64_t ldo, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* QUADS_H */
