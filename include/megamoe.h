/*
 * megamoe.h -- C ABI of the GB300 (sm_103a) fused MoE expert layer.
 *
 * One call runs the whole single-GPU hot path of the fused "MegaMoE" expert
 * layer: route the (token, k) assignments to experts, L1 gate/up grouped GEMM
 * (FP8-E4M3 activations x FP4-E2M1 weights, one UE8M0 scale per 32 elements
 * along K), clamp + SwiGLU + FP8 requantisation, L2 down grouped GEMM, and the
 * top-k weighted combine into a bf16 output.
 *
 * Sources (the pages this library follows):
 *  [P1] sglang PR #36657 "[Blackwell] Reserve SMs for DeepGEMM MegaMoE grid
 *       barriers" -- Summary, Root cause, Fix: an even clustered grid with a
 *       whole-grid software barrier; the launch size is the physical SM count
 *       minus a reserve (default 2), floored at 2 and rounded down to even.
 *  [P2] the prhub.com.cn digest of the same PR -- 实现拆解 and 关键源码片段:
 *       the env default of 2 reserved SMs, the reserve arithmetic, the call
 *       fp8_fp4_mega_moe(y, l1_weights, l2_weights, buf, recipe=(1, 1, 32),
 *       activation="swiglu", activation_clamp=swiglu_limit, fast_math=True),
 *       and a symmetric-buffer cache keyed only on the shape.
 *  [P3] DeepGEMM "SM90 MegaMoE 开发日志" -- Phase 1 entry (the buffer views
 *       x, x_sf, topk_idx, topk_weights, l1_acts, l1_acts_sf, l2_acts,
 *       l2_acts_sf; a workspace-size query) and Phase 2 entry (the dispatch
 *       clears its workspace, counts each expert's assignments, records the
 *       source (token, k) of every slot and releases a per-expert arrival
 *       count once the expert's rows are in place).
 *  [P4] DeepGEMM PR #451 "[Bugfix] Reset MegaMoE combine readiness for CUDA
 *       graph replay": readiness flags are reset by every launch, never keyed
 *       on %gridid, so graph replays match eager runs exactly.
 *
 * Conventions for every entry point:
 *  - All tensors are row-major and live in device memory unless a comment says
 *    "host".  The caller owns every buffer; the library allocates no device
 *    memory and keeps no per-call state.
 *  - Calls are stream-ordered on `stream` (a cudaStream_t; 0 = legacy default
 *    stream).  Argument errors are returned synchronously before anything is
 *    enqueued.  Errors found on the device (a bad expert index, a wait that
 *    timed out) are written to the status word at the head of the workspace
 *    and read back with mm_get_status().
 *  - Return values are mm_status codes (0 = success, negative = error) unless
 *    stated otherwise.
 */
#ifndef MEGAMOE_H
#define MEGAMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle (binary-compatible with cudaStream_t / CUstream). */
typedef struct CUstream_st* mm_stream_t;

typedef enum {
  MM_OK = 0,
  MM_ERR_INVALID_ARG = -1,         /* null pointer, misaligned pointer, bad value     */
  MM_ERR_UNSUPPORTED_SHAPE = -2,   /* dimensions outside the supported envelope       */
  MM_ERR_WORKSPACE_TOO_SMALL = -3, /* workspace_bytes < mm_workspace_size(...)        */
  MM_ERR_CUDA = -4,                /* a CUDA runtime/driver call failed               */
  MM_ERR_TIMEOUT = -5,             /* a device wait (readiness counter, pipeline
                                      barrier, tile ring) ran past its time limit     */
  MM_ERR_BAD_INDEX = -6,           /* topk_idx outside [-1, experts)                  */
  MM_ERR_BOUNDS = -7,              /* reserved for checked builds                     */
  MM_ERR_NO_DEVICE = -8            /* no usable sm_103 device                         */
} mm_status;

/* Element formats accepted by mm_quantize_mx. */
typedef enum { MM_FMT_E4M3 = 0, MM_FMT_E2M1 = 1 } mm_format;

/*
 * Supported shapes (checked by every entry point that takes dimensions):
 *   hidden  H : multiple of 128, 128 <= H <= 32768
 *   inter   I : multiple of 128, 128 <= I <= 16384  (the packed-FP4 TMA tile
 *               needs rows of a multiple of 128 elements)
 *   experts E : 1 <= E <= 1024
 *   topk    k : 1 <= k <= 16
 *   tokens  T : 0 <= T, T * k <= 2^24
 */

/*
 * mm_workspace_size -- bytes of device workspace that mm_forward / mm_route
 * need for up to `max_tokens` tokens.  Depends only on the shape, never on the
 * SM count or the reserve (the cache key of [P2] 实现拆解 item 5 holds only
 * shape parameters).  Returns 0 for unsupported arguments.
 * Workspace contents: a control block (status, abort flag, tile counter),
 * per-expert readiness counters, routing results (counts, offsets, permutation), the
 * dispatched tokens and their scales in expert order, the L1 activations
 * (E4M3 + UE8M0/32) and the weighted L2 outputs (fp32) -- the views of [P3].
 */
size_t mm_workspace_size(int max_tokens, int experts, int topk, int hidden, int inter);

/*
 * mm_forward -- the fused layer, y = MoE(x).  ([P2] 关键源码片段, [P3])
 *
 *   num_tokens T, experts E, topk k, hidden H, inter I : the shape
 *   x         E4M3 codes            [T, H]        16-byte aligned
 *   x_sf      UE8M0 bytes           [T, H/32]     4-byte aligned
 *   topk_idx  int32                 [T, k]        expert id, or -1 = empty slot
 *   topk_w    float32               [T, k]        combine weight of each slot
 *   l1_w      E2M1, two per byte    [E, 2I, H/2]  element 2c in the low nibble;
 *             rows [0, I) are the gate projection, rows [I, 2I) the up
 *             projection; 32-byte aligned
 *   l1_sf     UE8M0 scales of l1_w  [E, 2I, H/32] as prepared by
 *             mm_prepare_weight_scales (rows E*2I, K = H); 16-byte aligned
 *   l2_w      E2M1, two per byte    [E, H, I/2]   32-byte aligned
 *   l2_sf     UE8M0 scales of l2_w  [E, H, I/32]  as prepared by
 *             mm_prepare_weight_scales (rows E*H, K = I); 16-byte aligned
 *   y         bfloat16              [T, H]        16-byte aligned; fully written
 *             (a token whose slots are all empty gets a zero row)
 *   clamp     swiglu limit L: applies iff finite and > 0; then
 *             gate = min(gate, L), up = min(max(up, -L), L) before SwiGLU
 *   num_sms   SMs this launch may use; <= 0 means all.  The persistent grid is
 *             min(num_sms, SMs - reserve) rounded down to even, at least 2
 *             ([P1] Fix; [P2] 实现拆解 items 2-3), and never more CTAs than
 *             can be resident at once.
 *   workspace device buffer of at least mm_workspace_size(T', E, k, H, I)
 *             bytes for some T' >= T, 256-byte aligned, owned by the caller;
 *             one workspace must not be used by two launches that overlap.
 *   stream    the stream to enqueue on.
 *
 * Enqueues the routing (one kernel, or three above 2048 assignments), the
 * persistent layer kernel, then the top-k combine, and returns.  T = 0
 * returns MM_OK without launching.  Device-side errors land in
 * the workspace status (mm_get_status); the next mm_forward resets it.  Every
 * device wait is bounded by mm_set_wait_timeout_ns; a wait that runs out sets
 * MM_ERR_TIMEOUT and the kernel returns instead of hanging.  The call makes
 * no host synchronisation and no allocation, so it can be captured in a CUDA
 * graph; all counters and flags are reset by each launch ([P4]).
 */
int mm_forward(int num_tokens, int experts, int topk, int hidden, int inter,
               const void* x, const void* x_sf, const int32_t* topk_idx, const float* topk_w,
               const void* l1_w, const void* l1_sf, const void* l2_w, const void* l2_sf,
               void* y, float clamp, int num_sms,
               void* workspace, size_t workspace_bytes, mm_stream_t stream);

/*
 * mm_forward_bf16 -- mm_forward on bfloat16 activations: the quantisation
 * that precedes the fused call in the pages' pipeline ([P1] Fix, the
 * "pre-dispatch" step; [P2] 关键源码片段, the quantisation done before
 * fp8_fp4_mega_moe) is folded into the layer's dispatch.
 *
 *   x_bf16    bfloat16              [T, H]        16-byte aligned
 *
 * Every other argument, the workspace and the error behaviour are those of
 * mm_forward.  Each token's row is read once; every 32-element block is
 * quantised to E4M3 with one UE8M0 scale by the same rule as mm_quantize_mx
 * (the smallest power of two 2^s with max|v| <= 448 * 2^s, s in [-127, 127];
 * elements round to nearest even, saturating) and written to each of the
 * token's expert slots.  The result equals mm_forward on mm_quantize_mx of
 * the same values, bit for bit.
 */
int mm_forward_bf16(int num_tokens, int experts, int topk, int hidden, int inter,
                    const void* x_bf16, const int32_t* topk_idx, const float* topk_w,
                    const void* l1_w, const void* l1_sf, const void* l2_w, const void* l2_sf,
                    void* y, float clamp, int num_sms,
                    void* workspace, size_t workspace_bytes, mm_stream_t stream);

/*
 * mm_bf16_workspace_size / mm_bf16_forward -- the bf16 x bf16 layer: the
 * second MegaMoE kernel of the pages, the BF16 one whose dispatch, readiness
 * and combine protocol DeepGEMM PR #451 fixes together with the FP8/FP4 one
 * (description: "both FP8/FP4 and BF16 kernels"; validation: BF16 graph
 * replay equal to eager).  The pages give its protocol, not its arithmetic;
 * the layer computed here is that of mm_forward with every quantisation step
 * replaced by bfloat16:
 *
 *   x      bfloat16   [T, H]       16-byte aligned
 *   l1_w   bfloat16   [E, 2I, H]   rows [0, I) gate, [I, 2I) up; 32-byte aligned
 *   l2_w   bfloat16   [E, H, I]    32-byte aligned
 *   a1 = x . W1[e]^T and o = h . W2[e]^T accumulate in fp32; the clamp and
 *   SwiGLU are those of mm_forward; the L1 activations h are rounded to
 *   bfloat16 (nearest even); y = bf16(sum over j ascending of topk_w * o).
 *
 * topk_idx, topk_w, y, clamp, num_sms, stream and the error behaviour are
 * those of mm_forward.  The workspace (mm_bf16_workspace_size bytes, same
 * alignment and ownership rules) holds activations of 2 bytes per element;
 * mm_get_status reads its status word as for mm_forward.
 */
size_t mm_bf16_workspace_size(int max_tokens, int experts, int topk, int hidden, int inter);
int mm_bf16_forward(int num_tokens, int experts, int topk, int hidden, int inter,
                    const void* x, const int32_t* topk_idx, const float* topk_w,
                    const void* l1_w, const void* l2_w, void* y, float clamp, int num_sms,
                    void* workspace, size_t workspace_bytes, mm_stream_t stream);

/*
 * mm_set_reserved_sms -- SMs left free for other streams by every launch
 * ([P1] Summary: two by default; [P2] 实现拆解 item 1: 0 disables it).
 * n < 0 is taken as 0.  Process-wide; read at each launch.  Returns the
 * previous value.  The environment variable MM_RESERVED_SMS, if set when the
 * library loads, replaces the default of 2.
 */
int mm_set_reserved_sms(int n);
int mm_get_reserved_sms(void);

/*
 * mm_set_pair_mma -- whether mm_forward and mm_forward_bf16 run batches of
 * more than 16 assignments per expert (on average) as MMA tiles of 256 tokens
 * shared by a cluster of two CTAs on neighbouring SMs (tcgen05 cta_group::2:
 * M = 256, each CTA loading and holding half of the tile's 256 weight rows),
 * or as 128-token tiles of one CTA.  The pages' kernel runs an even grid of
 * such two-CTA clusters ([P1] Root cause and Fix: the reserve keeps the grid
 * even so that it stays "compatible with the two-CTA cluster").  Applies only
 * when hidden is a multiple of 256 (every weight tile then splits into two
 * 128-row halves); other shapes, decode-sized batches and mm_bf16_forward use
 * one-CTA tiles.  The result is the same either way (same arithmetic, same
 * rounding).  enable != 0 turns it on.  Process-wide; read at each launch.
 * Returns the previous value.  Off by default: on GB300 the two-CTA tiles
 * measured slower than the one-CTA tiles (about 1.85x the step time of the
 * 8192-token batch).  The environment variable MM_PAIR_MMA (0 or 1), if set
 * when the library first needs it, replaces the default of 0.
 */
int mm_set_pair_mma(int enable);
int mm_get_pair_mma(void);

/*
 * mm_layer_variant -- which layer kernel a launch of this shape runs, under
 * the current settings: 0 one-CTA tiles of 128 tokens, 1 one-CTA tiles of
 * 32-token stages (at most 16 assignments per expert on average), 2 and 3 the
 * same two for mm_bf16_forward (bf16_layer != 0), 4 two-CTA tiles of 256
 * tokens (see mm_set_pair_mma).  MM_ERR_INVALID_ARG for a bad shape.  Host
 * only; for tests and reports.
 */
int mm_layer_variant(int num_tokens, int experts, int topk, int hidden, int bf16_layer);

/*
 * mm_grid_size -- the launch-size rule, exposed for tests and callers:
 *   cap    = max(2, device_sms - max(reserved_sms, 0))
 *   want   = num_sms > 0 ? min(num_sms, device_sms) : device_sms
 *   g      = min(cap, want);  g -= g % 2;  g = max(g, 2)
 *   g      = min(g, max_resident) rounded down to even (if max_resident > 0)
 * ([P2] 关键源码片段: _mega_moe_max_num_sms and the context manager).
 * Returns the grid size, or MM_ERR_INVALID_ARG if device_sms < 2.  Host only.
 */
int mm_grid_size(int device_sms, int reserved_sms, int num_sms, int max_resident);

/*
 * mm_set_wait_timeout_ns -- time limit of every device-side wait (default
 * 2e9 ns).  The pages' kernel reports a grid-sync timeout with the SM, the
 * thread and the barrier's index instead of hanging ([P2] 功能与动机); here the wait
 * records MM_ERR_TIMEOUT with the SM and the wait site, raises the abort flag
 * and returns.  ns == 0 restores the default.  Process-wide.
 */
void mm_set_wait_timeout_ns(unsigned long long ns);
unsigned long long mm_get_wait_timeout_ns(void);

/*
 * mm_get_status -- synchronises `stream`, then reads the status word of
 * `workspace`.  *sm (may be NULL) receives the SM id that recorded the error;
 * *info (may be NULL) the wait site ((site << 24) | tile) or the first bad
 * flat index for MM_ERR_BAD_INDEX.  Returns the recorded mm_status (MM_OK if
 * none) or MM_ERR_CUDA if the synchronisation or copy failed.
 */
int mm_get_status(const void* workspace, mm_stream_t stream, int* sm, int* info);

/*
 * mm_route -- runs only the routing of mm_forward (reset, expert histogram,
 * prefix scan, stable permutation) into `workspace` ([P3] Phase 2 entry:
 * the per-expert counts and each slot's source assignment): one kernel up to 2048
 * assignments, else three (per-chunk counts, scan, scatter).  Same argument
 * rules as mm_forward.  Test hook.
 */
int mm_route(int num_tokens, int experts, int topk, int hidden, int inter,
             const int32_t* topk_idx, void* workspace, size_t workspace_bytes,
             mm_stream_t stream);

/*
 * mm_read_routing -- synchronous copy of the routing results left in
 * `workspace` by mm_route / mm_forward for the given shape into HOST buffers
 * (any may be NULL): counts [E], offsets [E+1] (exclusive prefix of counts),
 * perm [T*k] (slot -> flat index t*k+j; entries past offsets[E] are unused),
 * inv [T*k] (flat index -> slot, -1 for an empty slot).  Synchronises the
 * device.  Test hook.
 */
int mm_read_routing(int num_tokens, int experts, int topk, int hidden, int inter,
                    const void* workspace, int32_t* counts, int32_t* offsets,
                    int32_t* perm, int32_t* inv);

/*
 * mm_workspace_region -- byte offset and size of a named region of the
 * workspace for the given shape, so tests can inspect intermediates:
 *   0 control block   1 counts      2 offsets     3 work items  4 arrivals
 *   5 L1-done counts  6 perm        7 inv         8 dispatched x [T*k, H]
 *   9 dispatched x scales           10 l1_acts [T*k, I] (E4M3, slot order)
 *  11 l1_acts scales                12 weighted L2 outputs, fp32 [T*k, H]
 *     indexed by the flat assignment t*k+j
 *  13 routing chunk table: int32 [E][C] then [C], C = 1 up to 2048
 *     assignments, else min(ceil(T*k / 1024), 128) chunks
 *  14 token blocks, in block order: int32 {expert, the expert's first
 *     block, its first slot, its count} per block (room for T*k blocks;
 *     region 3 entry E is the number used)
 * Regions 9 and 11 hold, for the UE8M0 layers, 512-byte scale atoms (the
 * layout of mm_prepare_weight_scales) per token block, 128-row half of the
 * block (two halves for the two-CTA tiles, else one) and 128-wide K stage:
 * atom ((b * halves + h) * K/128 + s); row r of the half at byte
 * 16 (r % 32) + 4 (r / 32).  Blocks are those of region 14.  For
 * mm_f8b_forward they hold fp32 scales [T*k, K/128] in slot order.
 * Returns MM_OK, or MM_ERR_INVALID_ARG for an unknown region or shape.
 */
int mm_workspace_region(int which, int num_tokens, int experts, int topk, int hidden,
                        int inter, size_t* offset, size_t* bytes);

/*
 * mm_prepare_weight_scales -- the one-time transform of a weight matrix's
 * block scales into the layout the layer kernel copies straight into tensor
 * memory (the pages' SM90 work checks such a weight transform in its Phase 1
 * smoke test: DeepGEMM fork, "SM90 MegaMoE 开发日志", Phase 1 entry).
 *   sf    UE8M0 bytes [rows, K/32], row-major (what mm_quantize_mx writes
 *         for an E2M1 matrix [rows, K]); 4-byte aligned
 *   out   rows * K/32 bytes, 16-byte aligned, caller-owned: 512-byte atoms
 *         [rows/128][K/128]; atom (b, s) holds, at byte 16 l + 4 c + j, the
 *         scale of row 128 b + 32 c + l, block 4 s + j (l < 32, c, j < 4)
 *   rows  a multiple of 128; K a multiple of 128
 * The transform is a permutation of bytes: no value changes.  Prepare l1_sf
 * with rows = E*2I, K = H and l2_sf with rows = E*H, K = I once, when the
 * weights are loaded; mm_forward, mm_forward_bf16 and mm_forward_noalloc take
 * the prepared bytes.  Enqueued on `stream`; MM_ERR_INVALID_ARG for bad sizes
 * or alignment.
 */
int mm_prepare_weight_scales(const void* sf, long long rows, long long k, void* out, mm_stream_t stream);

/*
 * mm_quantize_mx -- block quantiser: src float32 [rows, cols] (cols a
 * multiple of 32, 16-byte aligned) -> element codes and one UE8M0 scale per
 * 32 consecutive elements of a row.  For each block with largest magnitude a,
 * the scale exponent is the smallest s with a <= F * 2^s (F = 448 for E4M3,
 * 6 for E2M1), clamped to [-127, 127], and 0 for an all-zero block; elements
 * are round-to-nearest-even of v / 2^s.  dst: E4M3 -> [rows, cols] bytes;
 * E2M1 -> [rows, cols/2] bytes, element 2c in the low nibble (16-byte
 * aligned).  dst_sf: [rows, cols/32] bytes.  This is the quantisation that
 * precedes the fused call ([P1] Fix: "pre-dispatch"; [P2] 关键源码片段) and
 * the rule the layer applies to its L1 activations.
 */
int mm_quantize_mx(const float* src, long long rows, long long cols, int fmt,
                   void* dst, void* dst_sf, mm_stream_t stream);

/*
 * mm_quantize_f8b -- the block quantiser of the (1, 128, 128) recipe, the one
 * the SM90 path of the pages uses with float scale factors ([P3] Phase 1
 * entry): src float32 [rows, cols] (cols a multiple of 128, rows a multiple
 * of block_rows, 16-byte aligned) -> E4M3 codes dst [rows, cols] (4-byte
 * aligned) and one float32 scale per block of block_rows x 128 in dst_sf
 * [rows / block_rows, cols / 128] (4-byte aligned).  block_rows is 1 (token
 * activations: one scale per token and 128 elements) or 128 (weights: one
 * scale per 128 x 128 block).  For a block with largest magnitude a the scale
 * is s = a / 448 rounded to fp32 (1 for an all-zero block) and each element's
 * code is the round-to-nearest-even E4M3 value of the fp32 quotient v / s,
 * saturating.  MM_ERR_INVALID_ARG for bad sizes or pointers.
 */
int mm_quantize_f8b(const float* src, long long rows, long long cols, int block_rows, void* dst, float* dst_sf,
                    mm_stream_t stream);

/*
 * mm_f8b_forward -- the fused layer in the (1, 128, 128) recipe ([P3] Phase 1
 * entry: the SM90 wrapper's recipe (1, 128, 128) with float scale factors):
 *
 *   x      E4M3 codes   [T, H]              16-byte aligned
 *   x_sf   float32      [T, H/128]          one scale per token and 128 elements of H
 *   l1_w   E4M3 codes   [E, 2I, H]          rows [0, I) gate, [I, 2I) up; 32-byte aligned
 *   l1_sf  float32      [E, 2I/128, H/128]  one scale per 128 x 128 block
 *   l2_w   E4M3 codes   [E, H, I]           32-byte aligned
 *   l2_sf  float32      [E, H/128, I/128]
 *   (scale arrays 4-byte aligned; the values as mm_quantize_f8b makes them)
 *
 * a1 = sum over the 128-wide K blocks b of (x_sf[t, b] * l1_sf[e, n/128, b])
 * * (E4M3 dot product of block b), accumulated in fp32; then the clamp and
 * SwiGLU of mm_forward; the L1 activations are requantised by the rule of
 * mm_quantize_f8b with one scale per token and 128 features; L2 likewise with
 * l2_sf; y = bf16(sum over j ascending of topk_w * o), as mm_forward.
 * topk_idx, topk_w, y, clamp, num_sms, the workspace (mm_workspace_size bytes)
 * and stream, and the error behaviour (mm_get_status) are those of mm_forward.
 */
int mm_f8b_forward(int num_tokens, int experts, int topk, int hidden, int inter,
                   const void* x, const float* x_sf, const int32_t* topk_idx, const float* topk_w,
                   const void* l1_w, const float* l1_sf, const void* l2_w, const float* l2_sf,
                   void* y, float clamp, int num_sms,
                   void* workspace, size_t workspace_bytes, mm_stream_t stream);

/*
 * mm_forward_noalloc -- mm_forward without a caller-provided workspace.  The
 * pages have no counterpart to this entry point.
 *
 * Some callers cannot allocate device memory at the point where they run the
 * layer: inference runtimes whose device memory is entirely owned by their
 * own pool allocator (a cudaMalloc behind its back fails or breaks its
 * accounting), plugins that run inside such a host and are handed only their
 * inputs and outputs, and real-time or safety-certified loops that forbid any
 * allocation after start-up.  For them the library keeps one fixed scratch
 * array of 64 MiB in device memory (a file-scope __device__ array, present on
 * every GPU where the library's kernels are loaded until the process exits),
 * enough for a decode batch of the DeepSeek-sized layer (128 tokens, top-8,
 * 256 experts, hidden 7168, inter 2048 needs 56.2 MiB).
 *
 * Arguments are those of mm_forward minus the workspace.  A shape whose
 * workspace (mm_workspace_size) exceeds 64 MiB is rejected with
 * MM_ERR_WORKSPACE_TOO_SMALL before anything is enqueued.  No cudaMalloc,
 * cudaFree or allocating routine is called.  The first call on a device looks
 * up the array's device address (cudaGetSymbolAddress, with that device
 * current); make that first call before any stream capture begins.  Every
 * call on a device shares the same array, and each launch resets what must
 * start at zero; two calls whose kernels overlap on the GPU (different
 * streams, or different host threads) race on it.  Device-side errors are
 * recorded in the array's status word: read them with mm_noalloc_get_status;
 * after such an error the output is undefined, and the next call resets the
 * status.
 */
int mm_forward_noalloc(int num_tokens, int experts, int topk, int hidden, int inter,
                       const void* x, const void* x_sf, const int32_t* topk_idx, const float* topk_w,
                       const void* l1_w, const void* l1_sf, const void* l2_w, const void* l2_sf,
                       void* y, float clamp, int num_sms, mm_stream_t stream);

/*
 * mm_noalloc_get_status -- mm_get_status for the calls of
 * mm_forward_noalloc on the current device: synchronises `stream`, then reads
 * the status word at the head of the library's scratch array.  *sm and *info
 * (either may be NULL) as for mm_get_status.  Returns the recorded mm_status
 * (MM_OK if none, or if mm_forward_noalloc never ran on this device),
 * MM_ERR_NO_DEVICE without a current device, or MM_ERR_CUDA if the address
 * lookup, the synchronisation or the copy failed.  No counterpart on the
 * pages; it allocates nothing.
 */
int mm_noalloc_get_status(mm_stream_t stream, int* sm, int* info);

#ifdef __cplusplus
}
#endif
#endif /* MEGAMOE_H */
