/*
 * moe_mxfp4.h -- C ABI of the MXFP4 mixture-of-experts layer for GB300 (sm_103a).
 *
 * The layer (the MoE block of a gpt-oss-style decoder) is:
 *   router GEMV/GEMM -> top-k with softmax over the selected logits -> per-expert
 *   tile table -> permute -> grouped gate/up GEMM with SwiGLU -> down GEMM with the
 *   weighted top-k combine and unpermute.
 * Sources: "A 297-line kernel file that decodes faster than vLLM" (cloudy.so),
 * section "Where the time went" (rows "Router + top-k", "MoE gate/up + SwiGLU",
 * "MoE down + combine") and section "Optimizations" (rows "MXFP4 MoE on tensor
 * cores", "Per-expert routing tile table", "Fixed decode tiles", "MoE token tile
 * follows tokens per expert"); "triton-kernels" README (bassrehab), section
 * "Quick Start", "Fused MoE Dispatch" (router -> permute -> fused expert FFN ->
 * unpermute, returning output, expert indices and expert weights).
 *
 * Conventions for every entry point:
 *  - Pointers are DEVICE pointers owned by the caller unless stated otherwise.  The
 *    library never allocates or frees device memory on these paths.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and never synchronise the host, except moe_prepare_weights,
 *    moe_get_device_status, moe_route_noalloc_status and moe_tensor_peak.
 *  - The return value is a status: MOE_OK (0) or a negative MOE_ERR_* code.  On an
 *    error nothing has been launched unless the code is MOE_ERR_CUDA.
 *  - Shapes: 1 <= T, T * k <= 2^24, H % 32 == 0 with 32 <= H <= 8192, I % 32 == 0
 *    with 32 <= I <= 16384, 1 <= k <= E <= 256, k <= 32.
 *  - bf16 arrays are raw bf16 bit patterns (uint16_t).
 *  - Expert weights: MXFP4 = FP4 E2M1 codes in blocks of 32 along K sharing one
 *    E8M0 scale, value = E2M1[code] * 2^(scale - 127) (OCP MX v1.0).  Raw layout:
 *    codes [E][rows][K/2] bytes with the even K index in the low nibble, scales
 *    [E][rows][K/32] bytes.  Gate/up rows: gate rows 0..I-1 then up rows I..2I-1
 *    (K = H).  Down rows: H rows (K = I).
 *  - Alignment: every device pointer 16-byte aligned; workspace and prepared
 *    weights 256-byte aligned.
 */
#ifndef MOE_MXFP4_H
#define MOE_MXFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* same type as cudaStream_t */

#define MOE_OK 0
#define MOE_ERR_INVALID_ARG (-1)       /* null pointer, bad alignment, bad flag      */
#define MOE_ERR_UNSUPPORTED_SHAPE (-2) /* shape outside the supported set above      */
#define MOE_ERR_WORKSPACE_TOO_SMALL (-3)
#define MOE_ERR_CUDA (-4)              /* a launch or driver call failed             */
#define MOE_ERR_DEVICE_TIMEOUT (-5)    /* a bounded device-side wait gave up          */
#define MOE_ERR_NAN_SCALE (-6)         /* an E8M0 scale byte of 255 (NaN) in weights */

#define MOE_WEIGHTS_GATEUP 0
#define MOE_WEIGHTS_DOWN 1

#define MOE_ROUTE_FROM_LOGITS 1 /* moe_route: `logits` is an input, skip the GEMV */
/* Gating variants (moe_route flags, moe_forward_gated): the k experts are selected the
 * same way in every one (the k largest logits, ties to the lower index); only their
 * weights differ.  Default (neither flag): softmax over the k selected logits.
 * "triton-kernels" README, "Project Structure" (router: softmax / sigmoid gating +
 * top-k) and "References" (DeepSeek-V3: sigmoid gating).                          */
#define MOE_ROUTE_GATING_SOFTMAX_ALL 2 /* w_j = exp(l_j) / sum over all E of exp(l_e)   */
#define MOE_ROUTE_GATING_SIGMOID 4     /* w_j = sigmoid(l_j) / sum over the k selected  */

/* Static description of a status code; never NULL. */
const char* moe_error_string(int status);

/* ------------------------------------------------------------------ weights
 * One-time re-layout of raw MXFP4 expert weights into the layout the tensor-core
 * kernels stream: the codes stay row major, [E][rows][K/2] (the TMA boxes of 128
 * rows x 256 codes are cut from them directly), and the E8M0 scales are regrouped
 * into 512-byte atoms of 128 rows x 4 MX blocks, the order in which the
 * block-scaled MMA reads them, [E][groups][rows/128][K groups of 128, rounded up to
 * even][512] (groups = 2 for gate/up: gate rows, up rows).  No value is re-quantised;
 * the bytes are only moved ("MXFP4 MoE on tensor cores": weights permuted once at
 * load).
 *   kind  MOE_WEIGHTS_GATEUP: rows = 2*I (gate then up), K = H.
 *         MOE_WEIGHTS_DOWN:   rows = H, K = I.
 *   codes [E][rows][K/2], scales [E][rows][K/32]: device, read only.
 *   dst: device, moe_prepared_weight_bytes(...) bytes, 256-byte aligned, written.
 * Scale bytes of 255 are rejected: the call returns MOE_ERR_NAN_SCALE after the
 * stream has finished (it synchronises `stream`, as a load-time call may).
 */
size_t moe_prepared_weight_bytes(int E, int rows, int K, int kind);
int moe_prepare_weights(const uint8_t* codes, const uint8_t* scales, int E, int rows, int K, int kind,
                        void* dst, size_t dst_bytes, moe_stream_t stream);

/* One-time re-layout of bf16 expert weights for moe_forward_bf16 into the tiles its
 * tensor-core kernels stream, one bulk copy each.  Tile (e, g, m, s) holds rows
 * [128 m, 128 m + 128) of row group g of expert e (gate rows then up rows for
 * gate/up, one group for down) and their values [64 s, 64 s + 64): 128 rows of
 * 128 bytes, the 16-byte chunk c of row r stored at chunk c ^ (r % 8) (the 128-byte
 * swizzle the MMA reads), rows past the group's end zero.  Tiles are ordered
 * [E][groups][ceil(rows per group / 128)][K / 64], followed by one zero tile.  The
 * values are copied unchanged.  The pages' Triton kernels read the weights as
 * stored; this is a layout of this implementation (weights permuted once at load,
 * as for MXFP4).
 *   kind, rows, K: as moe_prepare_weights; rows a multiple of the group count, K a
 *   multiple of 64.
 *   w bf16 [E][rows][K]: device, 16-byte aligned, read only.
 *   dst: device, moe_prepared_weight_bytes_bf16(...) bytes, 256-byte aligned, written.
 * Returns MOE_OK, MOE_ERR_UNSUPPORTED_SHAPE, MOE_ERR_INVALID_ARG,
 * MOE_ERR_WORKSPACE_TOO_SMALL or MOE_ERR_CUDA; asynchronous on `stream`.          */
size_t moe_prepared_weight_bytes_bf16(int E, int rows, int K, int kind);
int moe_prepare_weights_bf16(const uint16_t* w, int E, int rows, int K, int kind, void* dst, size_t dst_bytes,
                             moe_stream_t stream);

/* ------------------------------------------------------------------ sizes
 * Token rows per tile chosen for a shape (16, 64 or 128 from the mean tokens per
 * expert T*k/E; fixed per shape, never autotuned) and the bound on tile count.  */
int moe_tile_rows(int T, int k, int E);
int moe_max_tiles(int T, int k, int E, int tile_rows);

/* Bytes of device workspace needed by moe_forward and the stage calls below for
 * this shape; 0 for an unsupported shape.  The workspace holds routing results,
 * quantised activations, the slot buffer of the combine, arrival counters and a
 * status word.  Zero-fill it once after allocation (cudaMemset); every call leaves
 * its counters at zero again, so it can serve consecutive calls on one stream.
 * Calls that overlap on the GPU must not share a workspace.                       */
size_t moe_workspace_bytes(int T, int H, int I, int E, int k);

/* ------------------------------------------------------------------ stage calls
 * moe_route: logits[t, e] = sum_h x[t, h] * w_router[e, h] (+ router_bias[e]) in
 * fp32; then per token the k largest logits (ties: lower expert index first),
 * listed in that order, and weights = softmax over those k logits (or the gating
 * variant a MOE_ROUTE_GATING_* flag names; both flags at once is invalid).
 *   x bf16 [T, H]; w_router bf16 [E, H]; router_bias f32 [E] or NULL.
 *   logits f32 [T, E]: written, or read when flags has MOE_ROUTE_FROM_LOGITS (then
 *   x, w_router and router_bias may be NULL).
 *   topk_idx i32 [T, k], topk_w f32 [T, k]: written.
 *   workspace: zero-filled once, at least moe_workspace_bytes(T, 32, 32, E, k)
 *   bytes; only its status word and routing arrival counters are used.
 * Source: "Where the time went", row "Router + top-k"; "Quick Start",
 * fused_moe_forward(..., gating="softmax").                                        */
int moe_route(const uint16_t* x, const uint16_t* w_router, const float* router_bias, int T, int H, int E, int k,
              float* logits, int flags, int32_t* topk_idx, float* topk_w, void* workspace, size_t workspace_bytes,
              moe_stream_t stream);

/* moe_route_noalloc: moe_route for callers that cannot allocate device memory.
 * The pages have no counterpart of this entry point; it exists for callers such as
 * a serving runtime that owns a fixed memory pool, or a plugin that is handed only
 * its input and output buffers, which have no way to call cudaMalloc for the
 * workspace moe_route wants.  It computes exactly what moe_route computes, with
 * the same arguments minus the workspace: the small scratch moe_route keeps in
 * the workspace (a status word and the arrival counters of its last-block
 * hand-off) lives instead in a fixed array compiled into the library,
 * 256 + 4 * (8192 / 8 + 1) = 4356 bytes, which every GPU that loads the library
 * holds until the process exits.
 *   T must be <= 8192: larger T returns MOE_ERR_UNSUPPORTED_SHAPE.
 *   The first call on a device looks up the array's device address for that
 *   device (once per device, with it current); make that first call before any
 *   stream capture.  The array is zero when the library loads and every call
 *   leaves its counters at zero again, so no call clears anything before it
 *   launches.
 *   All calls share the one array: calls that overlap on the GPU (on different
 *   streams, or from several threads) race and must be serialised by the caller.
 *   A bounded device wait that gives up sets the array's status word; read it with
 *   moe_route_noalloc_status (a routing whose status is non-zero is not reliable). */
int moe_route_noalloc(const uint16_t* x, const uint16_t* w_router, const float* router_bias, int T, int H, int E,
                      int k, float* logits, int flags, int32_t* topk_idx, float* topk_w, moe_stream_t stream);

/* moe_route_noalloc_status: the device status of moe_route_noalloc on the current
 * device.  The pages have no counterpart of it; it is moe_get_device_status for the
 * fixed array.  Synchronises `stream`, reads the array's status word into *status
 * (bits as in moe_get_device_status; 0 = healthy) and, when it is non-zero, clears
 * the whole array, status word and arrival counters alike.  Returns MOE_OK,
 * MOE_ERR_DEVICE_TIMEOUT when a bit was set, MOE_ERR_INVALID_ARG for a NULL
 * status, or MOE_ERR_CUDA.  Not for the hot path.                                 */
int moe_route_noalloc_status(int* status, moe_stream_t stream);

/* moe_build_tile_table: the per-expert tile table of a routing ("Per-expert
 * routing tile table": each expert writes its own tiles).  Atomic-free counting
 * sort, deterministic:
 *   counts[e] (i32 [E]); offsets (i32 [E+1], exclusive prefix sum, offsets[E] = T*k);
 *   perm[s] (i32 [T*k]) = assignment t*k+j at sorted row s, rows sorted by expert
 *   then ascending t*k+j; inv_perm (i32 [T*k]) its inverse;
 *   tiles (i32 [max_tiles][4]) = {expert, first sorted row, rows (1..tile_rows),
 *   tile*tile_rows}, experts ascending, ceil(counts[e]/tile_rows) tiles each;
 *   num_tiles (i32 [1]).
 *   tile_rows: 16, 64 or 128, or 0 for moe_tile_rows(T, k, E).
 *   topk_idx i32 [T, k] with entries in [0, E): read.                              */
int moe_build_tile_table(const int32_t* topk_idx, int T, int k, int E, int tile_rows, int32_t* counts,
                         int32_t* offsets, int32_t* perm, int32_t* inv_perm, int32_t* tiles, int32_t* num_tiles,
                         moe_stream_t stream);

/* moe_mxfp4_gateup_swiglu: for every tile (expert e, rows of perm) and every
 * hidden feature i: g = x_t . W_gate[e][i], u = x_t . W_up[e][i], h = silu(g) * u.
 * Three launches: every token row of x is encoded once as a sum of four E2M1
 * terms, each with its own E8M0 scale per 32-value block; the encoded rows are
 * gathered by perm (the permute step) into tile order; the GEMM runs.  The
 * weights stay MXFP4 and both operands' scales feed the block-scaled MMA
 * (kind::mxf4) directly.
 * h is left in the workspace, encoded the same way in tile row order, for
 * moe_mxfp4_down_combine.
 *   x bf16 [T, H]; perm, tiles, num_tiles as written by moe_build_tile_table with
 *   the same tile_rows (0 = policy); w_gateup: moe_prepare_weights(MOE_WEIGHTS_GATEUP).
 * Source: "Where the time went", row "MoE gate/up + SwiGLU".                       */
int moe_mxfp4_gateup_swiglu(const uint16_t* x, const int32_t* perm, const int32_t* tiles, const int32_t* num_tiles,
                            int tile_rows, const void* w_gateup, int T, int H, int I, int E, int k, void* workspace,
                            size_t workspace_bytes, moe_stream_t stream);

/* moe_mxfp4_down_combine: y_tj = h_tj . W_down[e_tj]^T for every assignment, then
 * out[t] = sum_{j=0..k-1} topk_w[t, j] * y_tj summed in fp32 in ascending j and
 * rounded once to bf16 -- deterministic run to run.  Reads h from the workspace
 * (written by moe_mxfp4_gateup_swiglu for the same routing).  Two launches: the
 * down GEMM writes w_tj * y_tj into a per-assignment fp32 slot of the workspace,
 * then a combine kernel sums each token's k slots.
 *   topk_w f32 [T, k]; w_down: moe_prepare_weights(MOE_WEIGHTS_DOWN); out bf16 [T, H].
 * Source: "Where the time went", row "MoE down + combine".                         */
int moe_mxfp4_down_combine(const int32_t* perm, const int32_t* tiles, const int32_t* num_tiles, int tile_rows,
                           const float* topk_w, const void* w_down, int T, int H, int I, int E, int k,
                           void* workspace, size_t workspace_bytes, uint16_t* out, moe_stream_t stream);

/* moe_hidden_dequant: expand the workspace's four-term encoded h into f32
 * [T*k, I] rows in assignment order (t*k + j); a test and inspection aid.          */
int moe_hidden_dequant(const int32_t* perm, const int32_t* tiles, const int32_t* num_tiles, int tile_rows, int T,
                       int H, int I, int E, int k, const void* workspace, size_t workspace_bytes, float* h_out,
                       moe_stream_t stream);

/* ------------------------------------------------------------------ whole layer
 * moe_forward_gated: moe_forward with the top-k weights of the gating variant
 * `gating` (0, MOE_ROUTE_GATING_SOFTMAX_ALL or MOE_ROUTE_GATING_SIGMOID; any other
 * value is MOE_ERR_INVALID_ARG).                                                   */
int moe_forward_gated(const uint16_t* x, const uint16_t* w_router, const float* router_bias, const void* w_gateup,
                      const void* w_down, int T, int H, int I, int E, int k, int gating, void* workspace,
                      size_t workspace_bytes, uint16_t* out, int32_t* topk_idx_out, float* topk_w_out,
                      moe_stream_t stream);

/* moe_forward_norm: the step before the layer fused into it, then the layer:
 *   s = bf16(x + residual)                      (the residual stream, returned)
 *   y = bf16(s / sqrt(mean_H(s^2) + eps) * norm_weight)
 *   out = MoE(y)  (moe_forward_gated on y; `gating` as there).
 * Sources: "triton-kernels" README, "Kernels" (rmsnorm_residual_fused) and "Quick
 * Start", "Fused RMSNorm + Residual"; the decode-engine page "A 297-line kernel file
 * that decodes faster than vLLM", "Where the time went", row "RMSNorm + residual".
 * No launch is added: the routing kernel and the encoder each normalise the rows
 * they read (the same bits: one fixed summation order), and the combine kernel
 * writes residual_out.
 *   x, residual bf16 [T, H]; norm_weight bf16 [H]; all 16-byte aligned.
 *   eps: finite and >= 0.
 *   residual_out: bf16 [T, H] or NULL.  It may be x or residual itself: it is
 *   written after every read of both.  It may not be `out`.
 * Errors: MOE_ERR_INVALID_ARG for a NULL or misaligned x, residual or norm_weight,
 * a bad eps or gating value, or residual_out == out.  Everything else is as for
 * moe_forward.                                                                     */
int moe_forward_norm(const uint16_t* x, const uint16_t* residual, const uint16_t* norm_weight, float eps,
                     const uint16_t* w_router, const float* router_bias, const void* w_gateup, const void* w_down,
                     int T, int H, int I, int E, int k, int gating, void* workspace, size_t workspace_bytes,
                     uint16_t* out, uint16_t* residual_out, int32_t* topk_idx_out, float* topk_w_out,
                     moe_stream_t stream);

/* moe_forward_bf16: the same layer with bf16 expert weights instead of MXFP4.
 * This is the "Fused MoE Dispatch" workload of the "triton-kernels" README
 * ("Quick Start"; "MoE Dispatch Results": Mixtral-8x7B, 8 experts, top-2,
 * hidden 4096, ffn 14336): router -> top-k softmax gating -> permute -> gate/up +
 * SwiGLU -> down -> weighted combine + unpermute.
 * Launches:
 *   - routing: as moe_forward;
 *   - permute: bf16 rows of x into tile order;
 *   - gate/up and down: the grouped tcgen05 GEMMs with kind::f16 (bf16 x bf16,
 *     f32 accumulate); h is rounded to bf16 between them.  Tiles are 256 token rows
 *     once T*k >= 256*E (N = 256 MMAs), else moe_tile_rows(T, k, E);
 *   - combine: as moe_forward.
 * Arguments:
 *   x bf16 [T, H]; w_router bf16 [E, H]; router_bias f32 [E] or NULL;
 *   w_gateup: moe_prepare_weights_bf16(MOE_WEIGHTS_GATEUP) of bf16 [E, 2I, H], gate
 *   rows [0, I) then up rows [I, 2I); w_down: moe_prepare_weights_bf16(MOE_WEIGHTS_DOWN)
 *   of bf16 [E, H, I].  All pointers are 16-byte aligned.
 *   workspace: moe_workspace_bytes(T, H, I, E, k) bytes, 256-byte aligned.
 *   out bf16 [T, H].
 *   topk_idx_out / topk_w_out: as moe_forward.
 * Errors:
 *   - MOE_ERR_UNSUPPORTED_SHAPE as moe_forward, and also unless H and I are
 *     multiples of 64;
 *   - MOE_ERR_INVALID_ARG for NULL or misaligned pointers;
 *   - MOE_ERR_WORKSPACE_TOO_SMALL.                                                  */
int moe_forward_bf16(const uint16_t* x, const uint16_t* w_router, const float* router_bias, const uint16_t* w_gateup,
                     const uint16_t* w_down, int T, int H, int I, int E, int k, void* workspace,
                     size_t workspace_bytes, uint16_t* out, int32_t* topk_idx_out, float* topk_w_out,
                     moe_stream_t stream);

/* moe_forward: the whole layer, out = MoE(x), on one stream with no host sync.
 *   x bf16 [T, H]; w_router bf16 [E, H]; router_bias f32 [E] or NULL;
 *   w_gateup / w_down: prepared weights; out bf16 [T, H];
 *   topk_idx_out i32 [T, k] and topk_w_out f32 [T, k]: optional copies (NULL to skip).
 *   workspace: moe_workspace_bytes(T, H, I, E, k) bytes.                           */
int moe_forward(const uint16_t* x, const uint16_t* w_router, const float* router_bias, const void* w_gateup,
                const void* w_down, int T, int H, int I, int E, int k, void* workspace, size_t workspace_bytes,
                uint16_t* out, int32_t* topk_idx_out, float* topk_w_out, moe_stream_t stream);

/* moe_forward_timed: moe_forward that also records caller-created CUDA events
 * (cudaEvent_t, passed as void*) on `stream` around its MOE_FORWARD_STAGES stages:
 * events[i] just before stage i and events[MOE_FORWARD_STAGES] after the last one.
 * The stages are its five launches: route + top-k + tile table, the per-token
 * encoding of x (which waits for routing and writes the tile order itself: the
 * permute step), the gate/up + SwiGLU GEMM, the down GEMM, and the combine.  It
 * gives the per-launch time split ("Where the time went": per-section times of a
 * decode step); an event between two launches also separates them, so the
 * programmatic-launch overlap of consecutive kernels is lost in this form.
 * events must hold MOE_FORWARD_STAGES + 1 valid events.                          */
#define MOE_FORWARD_STAGES 5
int moe_forward_timed(const uint16_t* x, const uint16_t* w_router, const float* router_bias, const void* w_gateup,
                      const void* w_down, int T, int H, int I, int E, int k, void* workspace,
                      size_t workspace_bytes, uint16_t* out, int32_t* topk_idx_out, float* topk_w_out,
                      void* const* events, moe_stream_t stream);

/* Number of kernels moe_forward launches for a shape (for launch accounting):
 * route + top-k + table, encode + permute x, gate/up, down, combine.             */
int moe_forward_launches(int T, int H, int I, int E, int k);

/* moe_tensor_peak: the measured dense tensor-pipe rate of this GPU, in TFLOP/s, for
 * one of the MMA forms the expert GEMMs issue, as the roofline peak of the
 * compute-bound (many-token) workloads.  The pages give no tensor peak for this
 * hardware; the 4096-token prefill case is to be reported against the MXFP4 rate.
 *   kind MOE_PEAK_MXF4: tcgen05 kind::mxf4 block-scaled (E2M1 x E2M1, E8M0 scales,
 *        K = 64 per instruction), the MXFP4 layer's GEMMs;
 *   kind MOE_PEAK_BF16: kind::f16 (bf16 x bf16, K = 16), the bf16-weight layer.
 * One CTA per SM issues mmas_per_sm (8 .. 2^24) MMAs of M = 128, N = 256 back to
 * back into tensor memory; the call times that launch with CUDA events on
 * `stream`, synchronises it and writes 2*M*N*K*mmas*SMs / time to *tflops.
 * Returns MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_CUDA, or MOE_ERR_DEVICE_TIMEOUT when
 * the bounded completion wait gave up.  Not for the hot path.                      */
#define MOE_PEAK_MXF4 0
#define MOE_PEAK_BF16 1
int moe_tensor_peak(int kind, int mmas_per_sm, double* tflops, moe_stream_t stream);

/* moe_set_wait_limit_ns: how long (ns) each pipeline wait of the expert GEMMs may
 * take before it gives up, for launches made after the call (process-wide; 0
 * restores the default of 1 s; at most 10 s, else MOE_ERR_INVALID_ARG).  A wait
 * that gives up sets a bit of the workspace status word (moe_get_device_status), the
 * kernel drops its remaining work, waits (up to 1 s) for the copies and tensor-core
 * operations it has already issued, frees its tensor memory and exits: no trap, and
 * the context stays usable.  Limits under 2 us are polled without suspending the
 * waiting thread, so a limit shorter than the pipeline's own latency (a copy landing
 * takes about a microsecond even from L2) makes waits give up on ordinary calls;
 * that is how failure detection is tested.  The pages have no counterpart of it.   */
int moe_set_wait_limit_ns(unsigned long long ns);

/* Synchronises `stream`, reads the workspace's device status word into *status
 * (bit 0: main-loop wait timed out, bit 1: epilogue wait timed out, bit 2:
 * producer wait timed out; 0 = healthy) and clears it.  Returns MOE_OK, or
 * MOE_ERR_DEVICE_TIMEOUT when any bit was set.  After a timeout the call's outputs
 * are not reliable and the workspace's arrival counters may be left non-zero:
 * zero-fill the workspace again before its next use.  Not for the hot path.        */
int moe_get_device_status(void* workspace, size_t workspace_bytes, int* status, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_MXFP4_H */
