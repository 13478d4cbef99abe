/*
 * moe.h -- C ABI of the GB300 (sm_103a) Mixture-of-Experts SwiGLU FFN layer, forward and backward.
 *
 * One GPU, one CUDA stream per call, no host synchronisation on the compute path.  Every entry
 * point takes plain pointers and sizes; the caller owns and allocates every buffer (device
 * memory unless stated otherwise).  The library never allocates device memory.
 *
 * The layer (the pages give the systems around it, not its formulas; see "readings" below):
 *   logits = x W_r (+ b_r)                          [T,E] fp32
 *   p      = softmax(logits) over the E routed experts
 *   idx    = top-k experts by logit, larger first, a tie going to the lower expert index
 *   gates  = p[idx]  (renormalised over the k selected when cfg.renorm != 0)
 *   dispatch: per-expert queues in token order (histogram, exclusive prefix sum, stable
 *             permutation); with a capacity C = ceil(cf*T*k/E) the positions >= C are dropped
 *   expert e: h = silu(x_r W_gate[e]^T) * (x_r W_up[e]^T),  o = h W_down[e]^T
 *   y_t    = sum over kept slots j of gates[t,j] * o_{t,j}  +  sum over shared experts s of o^s_t
 *
 * Sources on the pages:
 *   - "MoEBlaze: Breaking the Memory Wall for Efficient MoE Training on Modern GPUs" (Korean
 *     summary): Methodology item 1 (dispatch queues instead of a dense token-by-expert routing
 *     matrix), item 2 (fused scatter/gather around the expert FFN; activation checkpointing that
 *     keeps a minimum and recomputes the rest in backward), the training-loop figure (fused
 *     expert kernels forward, checkpoint, fused expert kernels backward, gradient reduce) and
 *     Limitations (static top-k routing).
 *   - "Piper: Efficient Large-Scale MoE Training via Resource Modeling and Pipelined Hybrid
 *     Parallelism" (Japanese explainer, "the problem"): the router picks a few experts per
 *     token; loads can be heavily skewed; fine-grained experts give tall-and-skinny GEMMs.
 *   - "DisagMoE" technical summary, section 2.2: dispatch and combine around the expert FFN.
 *
 * Readings where the pages are silent: softmax over all E then top-k; selection by logit with
 * ties to the lower index; slot order = descending logit; capacity drops in token order (t, then
 * slot); dropped slots contribute zero and get zero gate gradient; kept gates are not
 * renormalised after drops; shared experts have weight 1 and sit outside softmax/top-k; SwiGLU
 * without biases.
 *
 * Data types and layouts (all row-major, contiguous):
 *   bf16 values are passed as raw 16-bit patterns (moe_bf16).
 *   x, y, dy, dx          [T, d_model]          bf16
 *   W_r                   [d_model, E]          fp32       b_r [E] fp32 (nullable)
 *   W_gate, W_up          [E+S, d_ff, d_model]  bf16       (out x in, like torch Linear)
 *   W_down                [E+S, d_model, d_ff]  bf16
 *   experts E..E+S-1 are the S shared (always-on) experts.
 *   idx                   [T, k] int32          gates, dgates [T, k] fp32
 *   dW_r                  [d_model, E] fp32     db_r [E] fp32
 *   dW_gate, dW_up, dW_down: same shapes as the weights, bf16, OVERWRITTEN (not accumulated).
 *
 * Expert-ordered ("permuted") rows.  moe_dispatch writes x_perm in a padded, expert-contiguous
 * layout with room for moe_perm_rows() rows:
 *   segment g (routed experts g < E first, then shared experts) starts at row P_g, a multiple of
 *   256; P_0 = 0, P_{g+1} = P_g + roundup(n_g, 256), where n_g = min(counts[g], C) for routed
 *   experts and n_g = T for shared ones.  Rows P_g + n_g .. P_{g+1}-1 are zero padding.
 *   The kept assignment (t, j) of expert e with queue position q sits at row P_e + q; shared
 *   expert s sees token t at row P_{E+s} + t.
 * The exact (unpadded) numbering is reported as well: offsets[e] is the exclusive prefix sum of
 * the kept counts and row_of_slot[t,j] = offsets[e] + q (or -1 when dropped).
 *
 * Kept activations (MoEBlaze, Methodology item 2: selective checkpointing, here with an adjustable
 * granularity).  By default the backward recomputes the SwiGLU pre-activations a = x W_gate^T and
 * b = x W_up^T from x_perm.  With keep_rows > 0, the forward also writes a and b (bf16) of the
 * first keep_rows expert-ordered rows (rounded down to a multiple of 256, at most all rows), and the
 * backward takes them instead of recomputing those rows: 2 * d_ff * 2 bytes kept per row buy
 * 4 * d_model * d_ff FLOP per row.  moe_layer_fwd / moe_layer_bwd keep them in `saved` (which grows
 * by those bytes: moe_workspace_size), so the workspace stays free for other layers between the
 * forward and the backward; moe_expert_ffn_fwd / moe_expert_ffn_bwd keep them in the workspace,
 * which must then reach the matching backward untouched.  moe_keep_rows_for_budget chooses
 * keep_rows from a byte budget (the adaptive granularity of the MoEBlaze summary's future work).
 *
 * Gathered operand loads (MoEBlaze summary, Methodology item 2, first bullet: the dispatch gather
 * fused with the expert feed-forward).  With gather_in_gemm = 1, moe_layer_fwd and moe_layer_bwd
 * write no x_perm or dY_perm: the dispatch builds its tables and the token of every padded row, and
 * the GEMMs that read those rows (gate/up, dh', the recompute, the weight gradients) fetch them from
 * x and dy in token order, four rows per TMA tile::gather4 copy, from four producer warps.  For
 * finite x and dy the results are those of gather_in_gemm = 0 bit for bit (a pad row reads token 0's
 * row instead of zeros, and its zero gate zeroes every gradient term it feeds).  It is the slower
 * choice on GB300: a stage's
 * 32 gather copies take about twice as long as the tensor cores' work on it, where one TMA box of a
 * contiguous x_perm tile keeps up, so the GEMMs that gather run at about half their speed while the
 * separate gather they save costs 0.1 to 0.5 ms per step.  It saves the x_perm and dY_perm traffic
 * (2 (T + N) d bytes each way) for a workload where that matters more than GEMM time.
 *
 * Workspace.  Size it with moe_workspace_size(), zero its header once with moe_workspace_init(),
 * and pass the same workspace to every call of one layer instance.  moe_dispatch leaves the
 * routing tables in it that moe_expert_ffn_fwd/bwd, moe_combine and moe_combine_bwd read; the
 * fused moe_layer_fwd/bwd keep all their intermediates there.  Calls that share a workspace
 * must be ordered on one stream.
 *
 * Errors.  Argument checks are synchronous: a call that returns anything but MOE_OK enqueued no
 * work.  Errors found on the device (an expert id out of range, a bounded wait that ran out)
 * are recorded in the workspace; moe_check_error() synchronises the stream, returns the first
 * such error since the last check, and clears it.  Device waits never spin unboundedly.
 *
 * Requirements: 1 <= k <= E <= 256; 0 <= S <= 8; d_model and d_ff multiples of 64 and <= 16384;
 * 1 <= T <= 1048576 and T*k <= 2^24; every pointer 16-byte aligned; sm_103a device.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* a null pointer, a misaligned pointer or a shape out of range */
    MOE_ERR_UNSUPPORTED = 2,   /* a valid shape the library does not handle (or not an sm_103 device) */
    MOE_ERR_WORKSPACE = 3,     /* workspace smaller than moe_workspace_size() */
    MOE_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed */
    MOE_ERR_BAD_INDEX = 5,     /* (device) an expert id outside [0, E): the dispatch that saw it
                                * publishes no rows (see moe_dispatch) */
    MOE_ERR_TIMEOUT = 6        /* (device) a bounded wait ran out; outputs of that call are invalid */
} moe_status_t;

typedef struct {
    int32_t T;                 /* tokens */
    int32_t d_model;           /* model width d */
    int32_t d_ff;              /* expert hidden width f */
    int32_t E;                 /* routed experts */
    int32_t k;                 /* experts per token */
    int32_t n_shared;          /* S always-on shared experts */
    int32_t renorm;            /* 1: gates renormalised over the k selected */
    float capacity_factor;     /* cf > 0: capacity ceil(cf*T*k/E) per expert; <= 0: dropless */
    int32_t keep_rows;         /* >= 0: expert-ordered rows whose gate/up pre-activations the forward
                                * keeps for the backward (see "Kept activations"); 0 recomputes all */
    int32_t gather_in_gemm;    /* 0 or 1, moe_layer_fwd / moe_layer_bwd only: 1 gathers the x and dy
                                * rows inside the expert GEMMs' operand loads (TMA tile::gather4 from
                                * token order) instead of copying them to x_perm / dY_perm first;
                                * same results, slower on GB300 (see "Gathered operand loads") */
} moe_config_t;

typedef uint16_t moe_bf16;                 /* raw bf16 bit pattern */
typedef struct CUstream_st* moe_stream_t;  /* a cudaStream_t; NULL is the legacy default stream */

/* Workspace bytes for any call of this configuration, and bytes of the `saved` buffer that
 * moe_layer_fwd fills and moe_layer_bwd reads: idx int32 [T,k], then gates fp32 [T,k], then, when
 * the gates are not renormalised, from the next 256-byte boundary the router logits fp32 [T,E]
 * (bias included: the backward's softmax reads them instead of recomputing x W_r), then, when
 * keep_rows > 0, from the next 256-byte boundary the kept a and b [keep, d_ff] bf16 (keep =
 * keep_rows rounded down to 256, at most moe_perm_rows()).  Host only; touches no device. */
moe_status_t moe_workspace_size(const moe_config_t* cfg, size_t* ws_bytes, size_t* saved_bytes);

/* Where the parts of `saved` after idx and gates sit (the layout above): the logits' byte offset
 * and size (both 0 with renormalised gates, which keep none), and the kept a, b block's offset and
 * size (a first, b right after it; size 0 when keep_rows is 0).  Every pointer is nullable.  Host
 * only; touches no device. */
moe_status_t moe_saved_layout(const moe_config_t* cfg, size_t* logits_off, size_t* logits_bytes, size_t* kept_off,
                              size_t* kept_bytes);

/* Checkpoint granularity from a memory budget (MoEBlaze summary, Limitations and future work:
 * adaptive checkpoint granularity driven by memory pressure at run time; Methodology item 2: keep
 * a minimum and recompute the rest).  *keep_rows receives the largest keep_rows (a multiple of 256,
 * at most moe_perm_rows()) whose kept a and b -- 4 * d_ff bytes per expert-ordered row, the bytes
 * `saved` grows by -- fit in budget_bytes; *kept_bytes (nullable) receives those bytes.  The
 * cfg's own keep_rows is ignored; set it to the result.  Rows kept cost no recompute GEMM work in
 * the backward (4 * d_model * d_ff FLOP each).  Host only; touches no device. */
moe_status_t moe_keep_rows_for_budget(const moe_config_t* cfg, uint64_t budget_bytes, int32_t* keep_rows,
                                      uint64_t* kept_bytes);

/* The same with the budget taken from the current device's free memory at the time of the call
 * (cudaMemGetInfo) less reserve_bytes (0 if free memory is below it): the kept share follows the
 * memory pressure of each step.  MOE_ERR_CUDA if the query fails. */
moe_status_t moe_keep_rows_for_free_memory(const moe_config_t* cfg, uint64_t reserve_bytes, int32_t* keep_rows,
                                           uint64_t* kept_bytes);

/* Rows (capacity) of x_perm / o_perm / dx_perm buffers: each is [rows, d_model] bf16.  Host only. */
moe_status_t moe_perm_rows(const moe_config_t* cfg, int64_t* rows);

/* Zero the workspace header (error word and device counters).  Call once after allocating. */
moe_status_t moe_workspace_init(const moe_config_t* cfg, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Router (Piper explainer, "the problem": a router sends each token to a few experts; MoEBlaze
 * summary, Limitations: a static top-k routing policy): logits, softmax, top-k and gates for every
 * token, by the readings above.  b_r and logits may be NULL.  Writes idx [T,k], gates [T,k], and
 * logits [T,E] when non-NULL.  ws is this configuration's workspace (moe_workspace_size).  For
 * E <= 128 and k <= 8 the logits run on the tensor cores: W_r is split in ws into three bf16 parts
 * whose sum equals it within fp32 rounding, and the products are summed in fp32 over 256-wide
 * slices of d_model (E <= 32: the parts stacked in one MMA and d_model split across CTAs, so that
 * the whole GPU streams x); other shapes use an fp32 tile product with warp-per-token selection. */
moe_status_t moe_route(const moe_config_t* cfg, const moe_bf16* x, const float* W_r, const float* b_r,
                       int32_t* idx, float* gates, float* logits, void* ws, size_t ws_bytes,
                       moe_stream_t stream);

/* Dispatch queues (MoEBlaze, Methodology item 1): per-expert histogram, exclusive prefix sum with
 * a decoupled look-back, stable (token-order) ranks, capacity, and the 16-byte gather of x rows into
 * x_perm (padded layout above; pad rows are zeroed; shared-expert segments hold copies of x).
 * Outputs: counts [E] (raw demand, sums to T*k), offsets [E+1] (exact), row_of_slot [T,k]
 * (exact row or -1), token_of_row [T*k] (entries >= offsets[E] are left untouched),
 * x_perm [moe_perm_rows(), d_model].  Leaves the padded tables in ws for the calls below.
 * An id outside [0,E) anywhere in idx records MOE_ERR_BAD_INDEX (read with moe_check_error) and
 * empties the whole dispatch, since the queue positions of that call cannot be trusted: counts
 * still hold the demand of the valid ids, but every segment is published with no rows (offsets
 * all 0, row_of_slot all -1, token_of_row and x_perm not written), so the calls that follow on
 * this workspace touch no rows.  The next dispatch with valid ids starts afresh. */
moe_status_t moe_dispatch(const moe_config_t* cfg, const int32_t* idx, const moe_bf16* x,
                          int32_t* counts, int32_t* offsets, int32_t* row_of_slot, int32_t* token_of_row,
                          moe_bf16* x_perm, void* ws, size_t ws_bytes, moe_stream_t stream);

/* moe_dispatch for callers that cannot allocate device memory: no workspace argument.  (The
 * pages have no counterpart; this exists for integration.)  Meant for code that runs where
 * cudaMalloc is not available or not allowed: inside a memory arena or pool owned by a host
 * framework that cannot grow at step time, or on a path that must not pay cudaMalloc's implicit
 * synchronisation.  Outputs and their meaning are those of moe_dispatch (counts, offsets,
 * row_of_slot, token_of_row, x_perm with room for moe_perm_rows() rows); the caller still
 * provides every input and output buffer.
 * Scratch: a fixed device array of about 3.6 MB inside the library, which every GPU that loads
 * the library holds until the process exits.  Limits: T*k <= 262144 assignments and
 * moe_perm_rows() <= 393216 rows; larger configurations return MOE_ERR_UNSUPPORTED and enqueue
 * nothing.  The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call before any stream
 * capture.  (The address is looked up again on every call, so a device reset or a re-created
 * primary context between calls is safe.)  The call allocates nothing: no cudaMalloc, cudaFree or
 * allocating library routine.
 * Every call shares the one array and leaves its contents behind (each call clears what must
 * start at zero), so calls that may overlap on the GPU -- on different streams, or from several
 * host threads -- race and must be serialised by the caller.
 * status: nullable device pointer to one int32 (4-byte aligned).  With no workspace there is no
 * error word for moe_check_error, so the call's device-side outcome lands here, written on the
 * stream after the scan: MOE_OK, MOE_ERR_BAD_INDEX (an id outside [0,E); as in moe_dispatch the
 * whole dispatch is then empty: offsets all 0, row_of_slot all -1, token_of_row and x_perm not
 * written) or MOE_ERR_TIMEOUT (a bounded wait ran out; outputs invalid).  Read it after the
 * stream's work completes.  With status NULL a bad id still empties the dispatch, unreported. */
moe_status_t moe_dispatch_noalloc(const moe_config_t* cfg, const int32_t* idx, const moe_bf16* x,
                                  int32_t* counts, int32_t* offsets, int32_t* row_of_slot,
                                  int32_t* token_of_row, moe_bf16* x_perm, int32_t* status,
                                  moe_stream_t stream);

/* Grouped expert SwiGLU FFN on the rows moe_dispatch laid out in ws: tcgen05/TMEM tiles fed by
 * TMA, a per-expert tile scheduler, SwiGLU fused into the first GEMM's epilogue.
 * o_perm [moe_perm_rows(), d_model] bf16 receives every segment's rows (pad rows are zero). */
moe_status_t moe_expert_ffn_fwd(const moe_config_t* cfg, const moe_bf16* x_perm,
                                const moe_bf16* W_gate, const moe_bf16* W_up, const moe_bf16* W_down,
                                moe_bf16* o_perm, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Weighted combine back to token order (MoEBlaze summary, Methodology item 2: the reverse
 * dispatch after the expert FFN; DisagMoE technical summary, section 2.2: combine), by token owner
 * (no atomics, fixed slot order, fp32 sums, one rounding):
 * y[t] = sum_kept gates[t,j] o_perm[row(t,j)] + sum_s o_perm[P_{E+s}+t].  Reads the row tables
 * moe_dispatch left in ws. */
moe_status_t moe_combine(const moe_config_t* cfg, const moe_bf16* o_perm, const float* gates,
                         moe_bf16* y, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Backward of the expert FFN and of the combine's gate weighting, recomputing the SwiGLU
 * activations from x_perm (MoEBlaze, Methodology item 2: selective checkpointing).
 * Reads dy [T,d] in token order; writes dx_perm [moe_perm_rows(), d_model] (gradient of x_perm,
 * padded layout), dgates [T,k] (dy . o, zero for dropped slots), dW_gate, dW_up, dW_down. */
moe_status_t moe_expert_ffn_bwd(const moe_config_t* cfg, const moe_bf16* x_perm, const moe_bf16* dy,
                                const float* gates,
                                const moe_bf16* W_gate, const moe_bf16* W_up, const moe_bf16* W_down,
                                moe_bf16* dx_perm, float* dgates,
                                moe_bf16* dW_gate, moe_bf16* dW_up, moe_bf16* dW_down,
                                void* ws, size_t ws_bytes, moe_stream_t stream);

/* Router backward with the selection held fixed: recompute logits from x, then
 * dlogits [T,E] fp32 from dgates, dW_r = x^T dlogits, db_r = sum_t dlogits (db_r nullable).
 * Without renorm: dl_e = p_e (dg_{slot(e)} [e selected] - sum_j dg_j g_j); with renorm:
 * dl_{idx_j} = g_j (dg_j - sum_m dg_m g_m) and 0 elsewhere.  b_r nullable. */
moe_status_t moe_router_bwd(const moe_config_t* cfg, const moe_bf16* x, const float* W_r, const float* b_r,
                            const int32_t* idx, const float* gates, const float* dgates,
                            float* dlogits, float* dW_r, float* db_r,
                            void* ws, size_t ws_bytes, moe_stream_t stream);

/* Input gradient, by token owner: dx[t] = sum_kept dx_perm[row(t,j)] + sum_s dx_perm[P_{E+s}+t]
 * + dlogits[t] W_r^T.  dlogits may be NULL (no router term).  Uses the tables of moe_dispatch. */
moe_status_t moe_combine_bwd(const moe_config_t* cfg, const moe_bf16* dx_perm, const float* dlogits,
                             const float* W_r, moe_bf16* dx, void* ws, size_t ws_bytes, moe_stream_t stream);

/* FP8 expert GEMMs, forward (the MoEBlaze summary names mixed-precision and quantised experts as
 * future work; the format is this library's reading).  Format: OCP FP8 E4M3 (max 448, no
 * infinities), one fp32 scale per row.  The steps are exposed one by one (quantise, gate/up, down)
 * and composed by moe_layer_fwd_fp8 below.
 *
 * moe_quantize_rows_e4m3: src [rows, cols] bf16 -> codes [rows, cols] uint8 and scales [rows]
 * fp32, with scale = amax / 448 over the row (1 for an all-zero row) and code = e4m3(v / scale),
 * both in fp32, rounded to nearest even and saturated.  cols a multiple of 16, at most 16384;
 * 16-byte-aligned pointers.  Used for token or x_perm rows, h rows, and the rows (output channels)
 * of W_gate, W_up and W_down.  Argument errors are returned before any work is queued. */
moe_status_t moe_quantize_rows_e4m3(const moe_bf16* src, int64_t rows, int32_t cols, uint8_t* codes,
                                    float* scales, moe_stream_t stream);

/* The gate/up projection and SwiGLU of moe_expert_ffn_fwd with e4m3 operands on the tensor cores
 * (kind::f8f6f4): h = silu(a) * b, a = s_x s_g (q_x . q_g), b = s_x s_u (q_x . q_u), accumulated in
 * fp32.  x8 / x_scale: the quantised x_perm rows [moe_perm_rows(), d_model] / [moe_perm_rows()]
 * (pad rows: zero codes); wg8, wu8 [E+S, d_ff, d_model] codes with wg_scale, wu_scale [E+S, d_ff].
 * Writes h [moe_perm_rows(), d_ff] bf16.  Uses the tables of moe_dispatch in ws. */
moe_status_t moe_gate_up_fp8(const moe_config_t* cfg, const uint8_t* x8, const float* x_scale,
                             const uint8_t* wg8, const float* wg_scale, const uint8_t* wu8,
                             const float* wu_scale, moe_bf16* h, void* ws, size_t ws_bytes,
                             moe_stream_t stream);

/* The down projection with e4m3 operands: o = s_h s_d (q_h . q_d) per row and output channel,
 * accumulated in fp32 and stored bf16.  h8 / h_scale: quantised h rows [moe_perm_rows(), d_ff] /
 * [moe_perm_rows()] (moe_quantize_rows_e4m3 of h); wd8 [E+S, d_model, d_ff] codes with wd_scale
 * [E+S, d_model] (one scale per output channel: the rows of W_down).  Writes o_perm
 * [moe_perm_rows(), d_model] bf16.  Uses the tables of moe_dispatch in ws. */
moe_status_t moe_down_fp8(const moe_config_t* cfg, const uint8_t* h8, const float* h_scale, const uint8_t* wd8,
                          const float* wd_scale, moe_bf16* o_perm, void* ws, size_t ws_bytes,
                          moe_stream_t stream);

/* The whole forward with e4m3 expert GEMMs: route as moe_layer_fwd; quantise the T token rows of
 * x once (a row's codes are the same in every expert it visits); dispatch, gathering those codes
 * and row scales into the padded expert rows; moe_gate_up_fp8 (h kept in bf16); quantise the h
 * rows this step fills; moe_down_fp8; and the combine.  The weights come quantised
 * (moe_quantize_rows_e4m3 of every row of W_gate, W_up and W_down, as above).  The router stays
 * fp32.  Fills `saved` like moe_layer_fwd (idx, gates, logits), so moe_layer_bwd can follow with
 * the bf16 weights.
 * keep_rows must be 0 (MOE_ERR_INVALID_ARG otherwise): the call's scratch uses the workspace
 * buffers that would carry kept activations to the backward. */
moe_status_t moe_layer_fwd_fp8(const moe_config_t* cfg, const moe_bf16* x, const float* W_r, const float* b_r,
                               const uint8_t* wg8, const float* wg_scale, const uint8_t* wu8,
                               const float* wu_scale, const uint8_t* wd8, const float* wd_scale, moe_bf16* y,
                               void* saved, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Per-column e4m3 codes, written transposed, for the FP8 backward's weights (same format as
 * moe_quantize_rows_e4m3: scale = amax / 448 over the column, 1 for an all-zero column; code =
 * e4m3(v / scale) rounded to nearest even and saturated, both in fp32).  For each of G experts the
 * source is [top[g]; bottom[g]], rows_top + rows_bottom rows of `cols` bf16 values (bottom NULL when
 * rows_bottom is 0); codes[g] receives its transpose [cols, rows_top + rows_bottom] and scales[g]
 * one scale per column.  Used as
 *   W_down [G, d, f]                     -> codes [G, f, d], scales [G, f]   (top = W_down)
 *   W_gate, W_up [G, f, d] (stacked)     -> codes [G, d, 2f], scales [G, d]  (top = W_gate, bottom = W_up)
 * rows_top + rows_bottom a multiple of 16, at most 32768; 16-byte-aligned pointers.  The column
 * maxima are gathered in `scales` before it receives the scales.  Argument errors return before
 * any work is queued. */
moe_status_t moe_quantize_cols_e4m3(const moe_bf16* top, const moe_bf16* bottom, int64_t G, int32_t rows_top,
                                    int32_t rows_bottom, int32_t cols, uint8_t* codes, float* scales,
                                    moe_stream_t stream);

/* The whole backward with e4m3 expert GEMMs (the MoEBlaze summary names mixed-precision and
 * quantised experts as future work; the format is this library's reading): as moe_layer_bwd, with
 *   dh' = (s_dy q_dy) (s_wd q_wd)^T     dY rows quantised per row; W_down's columns per d_ff channel
 *                                       (wdt8, wdt_scale from moe_quantize_cols_e4m3 of W_down)
 *   a, b = the forward's e4m3 products, recomputed from the x rows (quantised per row) and the
 *          forward's row codes of W_gate and W_up (wg8, wg_scale, wu8, wu_scale)
 *   dA, dB, Hg from the SwiGLU backward in fp32, held in bf16 (dh' too)
 *   dX = (s_ab q_ab) (s_w q_w)^T        the joined row [dA | dB] quantised per row; column i of
 *                                       W_gate and W_up quantised together per d_model channel
 *                                       (wgut8, wgut_scale from moe_quantize_cols_e4m3 of W_gate over W_up)
 * accumulated in fp32.  The weight gradients stay bf16 products of dA, dB, Hg and the bf16 x and dY
 * rows; the router stays fp32.  `saved` comes from moe_layer_fwd or moe_layer_fwd_fp8 of the same
 * configuration; keep_rows must be 0 (MOE_ERR_INVALID_ARG otherwise). */
moe_status_t moe_layer_bwd_fp8(const moe_config_t* cfg, const moe_bf16* x, const float* W_r, const float* b_r,
                               const uint8_t* wg8, const float* wg_scale, const uint8_t* wu8, const float* wu_scale,
                               const uint8_t* wdt8, const float* wdt_scale, const uint8_t* wgut8,
                               const float* wgut_scale, const void* saved, const moe_bf16* dy, moe_bf16* dx,
                               float* dW_r, float* db_r, moe_bf16* dW_gate, moe_bf16* dW_up, moe_bf16* dW_down,
                               void* ws, size_t ws_bytes, moe_stream_t stream);

/* The whole forward: route, dispatch, expert FFN, combine (MoEBlaze summary, the training-loop
 * figure: fused expert kernels forward, then checkpoint).  Fills `saved` with idx and gates, the
 * router logits (gates not renormalised; T * E fp32, small beside x), and the kept a and b of the
 * first keep_rows expert-ordered rows when keep_rows > 0; every other activation is recomputed in
 * the backward (Methodology item 2). */
moe_status_t moe_layer_fwd(const moe_config_t* cfg, const moe_bf16* x, const float* W_r, const float* b_r,
                           const moe_bf16* W_gate, const moe_bf16* W_up, const moe_bf16* W_down,
                           moe_bf16* y, void* saved, void* ws, size_t ws_bytes, moe_stream_t stream);

/* The whole backward from x, the weights, `saved` and dy (MoEBlaze summary, the training-loop
 * figure: fused expert kernels backward, then gradient reduce): rebuilds the dispatch queues from
 * the saved idx, recomputes the expert activations of the rows not kept (Methodology item 2), takes
 * the router's softmax from the saved logits, and writes dx, dW_r, db_r (nullable) and the expert
 * weight gradients.  `saved` must come from moe_layer_fwd of the same configuration (keep_rows
 * included); a caller that writes idx and gates into it by hand writes the logits too. */
moe_status_t moe_layer_bwd(const moe_config_t* cfg, const moe_bf16* x, const float* W_r, const float* b_r,
                           const moe_bf16* W_gate, const moe_bf16* W_up, const moe_bf16* W_down,
                           const void* saved, const moe_bf16* dy,
                           moe_bf16* dx, float* dW_r, float* db_r,
                           moe_bf16* dW_gate, moe_bf16* dW_up, moe_bf16* dW_down,
                           void* ws, size_t ws_bytes, moe_stream_t stream);

/* Synchronise `stream`, return the first device-side error recorded in ws since the last check
 * (MOE_OK if none) and clear it.  Returns MOE_ERR_CUDA if the stream itself reports an error. */
moe_status_t moe_check_error(void* ws, moe_stream_t stream);

/* Test hook: make dispatch scan block `stall_block` never publish its counts (-1: off), make the
 * first CTA pair of every expert GEMM skip its fill number `stall_fill` of the operand ring -- no
 * loads, no expected bytes, so the MMA's wait for that stage never completes (-1: off) -- and bound
 * every device wait of later calls by `timeout_ns` (0: the default, 2 s).  Used to check that a
 * wait that runs out returns MOE_ERR_TIMEOUT through moe_check_error instead of hanging: the kernel
 * that gives up still waits, with the same bound, for the copies and MMAs it has in flight before
 * it frees its shared memory and TMEM, so the next call runs normally.  Outputs of the stalled call
 * are invalid. */
moe_status_t moe_debug_inject(void* ws, int32_t stall_block, int32_t stall_fill, uint64_t timeout_ns,
                              moe_stream_t stream);

/* Kernel timing.  While enabled, every kernel launch of the library is bracketed by two CUDA
 * events recorded on its launching stream.  moe_profile_enable(on) also clears the totals.
 * moe_profile_read(kernel, ...) waits for the recorded events and returns, for kernel id
 * 0..n-1, its name, summed milliseconds and launch count; MOE_ERR_INVALID_ARG past the last id.
 * Host-side state shared by the whole process; not for concurrent use from several threads. */
moe_status_t moe_profile_enable(int32_t on);
moe_status_t moe_profile_read(int32_t kernel, const char** name, double* total_ms, int32_t* launches);

/* The SM clock a tensor-core GEMM kernel actually ran at: while profiling is enabled, one thread of
 * each of its CTAs adds the SM cycles (clock64) and nanoseconds (globaltimer) from its entry to its
 * exit on the current device; *mhz receives cycles / ns x 1000 over all its CTAs since
 * moe_profile_enable (0 when none ran; same kernel ids as moe_profile_read).  Under the GPU's
 * power cap this is the clock the kernel's work ran at, which nvidia-smi's periodic samples miss.
 * moe_profile_enable touches the current device for this (MOE_ERR_CUDA if it cannot);
 * moe_profile_sm_clock synchronises with it.  The other kernels record nothing here. */
moe_status_t moe_profile_sm_clock(int32_t kernel, double* mhz);

/* Static text for a status code. */
const char* moe_status_string(moe_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
