/*
 * moe.h -- C ABI of libmoe_gb300: forward pass of one routed sparse
 * Mixture-of-Experts FFN layer on one NVIDIA GB300 (sm_103a).
 *
 * The layer (per token t with hidden vector x_t of size D):
 *   z_t     = x_t . Wr^T (+ bias)                       router logits over E experts
 *   ids_t   = the k experts with the largest z_t        (exact ties: lower index)
 *   w_t     = softmax(z_t)[ids_t] / sum of the same     renormalised gate weights
 *   y_t     = sum_j w_tj * FFN_{ids_tj}(x_t) + FFN_shared(x_t)
 *   FFN(x)  = W_down . (silu(W_gate . x) * (W_up . x))  SwiGLU expert
 *
 * Source passages (page title, section):
 *   [P1] "Systems engineering playbook: optimizing Qwen 3.5-397B MoE on Ironwood
 *        (TPU7x)", section 1, "Sparse Mixture-of-Experts (MoE)": router gate,
 *        softmax over 512 experts, top-10 routed experts, always-on shared expert.
 *   [P3] same page, section 3, "3-to-2 All-Gather optimisation": ids [T,k] and
 *        weights [T,k] stacked on a new axis, bit-cast, one dense int32 blob.
 *   [P3B] same page, section 3, "Option B": each device filters and computes the
 *        inputs of its own experts (dispatch), then outputs are reduced back.
 *   [PM] same page, executive summary: grouped GEMM and SparseCore unpermute as
 *        reusable building blocks.
 *   [R1] "vLLM TPU Inference v0.31.0: hierarchical MoE dispatch and W4A16",
 *        4-bit weight section: symmetric int4 weights in the pack-quantized
 *        format, group or channel scales, activations not quantised; weights
 *        stay int4 in HBM and the kernel restores only the tiles it needs
 *        on-chip; unsupported formats are rejected when the model loads.
 *   [R1G] same page, section on dispatch shared by two cores: the EP grouped
 *        matmul (GMM) path, with support conditions and a fallback otherwise.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers (except moe_forward_host's x and
 *     y), row-major, contiguous, 16-byte aligned.  bf16 is IEEE bfloat16.
 *   - The caller allocates and owns every buffer, including the workspace; the
 *     library never allocates device memory.  Size the workspace with
 *     moe_workspace_size() for the same entry and config.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  Buffers must stay alive until the stream has passed the call.
 *   - Concurrent calls that share a workspace race; give each stream its own.
 *   - A bf16 grouped GEMM with 256-row token tiles (T >= 2048 or T*k >= 48*E)
 *     and under 512 rows per expert on average (T*k < 512*E) runs its groups
 *     of fewer than 64 rows in a second grid on a stream of the library's,
 *     forked from `stream` and joined back to it with events inside the call:
 *     the call stays ordered on `stream` and can be captured into a CUDA
 *     graph.  The stream and events are created on first use, one set per
 *     host thread and CUDA context, and kept.
 *   - Return 0 on success or a negative MOE_ERR_* code.  Argument and shape
 *     errors are detected on the host and launch nothing.  Device-side wait
 *     timeouts are reported through moe_get_status().
 *   - Index data read from caller buffers (expert ids in a blob, offsets,
 *     perm_pair, a_row_index, inv_row) is checked on the device: a value
 *     outside its range is clamped into it, so every access stays inside the
 *     buffers whatever they hold (the affected tokens' outputs are then
 *     meaningless), and the entries that take a workspace record
 *     MOE_ERR_INVALID_ARG in its status word (moe_get_status).  The data
 *     written by moe_route and moe_permute is always in range.
 *   - NaN logits (from NaN in x, the router weights or the bias) rank below
 *     every number, NaNs among themselves by index: every token gets k
 *     distinct ids; a token whose selected logits include a NaN gets NaN
 *     weights, and a NaN in a token row reaches only that token's output.
 *   - There is no fallback path: unsupported shapes return MOE_ERR_UNSUPPORTED.
 *   - Kernels are built for sm_103a only; other devices get MOE_ERR_UNSUPPORTED.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- error codes ---- */
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG (-1)  /* null pointer, k < 1, k > E, T < 1, ...; on the
                                     device: an index out of range (moe_get_status) */
#define MOE_ERR_UNSUPPORTED (-2)  /* shape/format outside the kernels' envelope     */
#define MOE_ERR_WORKSPACE (-3)    /* workspace null or smaller than required        */
#define MOE_ERR_CUDA (-4)         /* a CUDA runtime call or launch failed           */
#define MOE_ERR_TIMEOUT (-5)      /* a device wait hit its bound (moe_get_status)   */
#define MOE_ERR_ALIGN (-6)        /* a pointer is not 16-byte aligned               */
#define MOE_ERR_SCRATCH_LIMIT (-7) /* too large for moe_permute_static's fixed scratch */

/* ---- weight formats ---- */
#define MOE_QUANT_BF16 0    /* bf16 expert weights                                   */
#define MOE_QUANT_W4A16 1   /* symmetric int4, 8 per int32 in PAIR order (value 2i
                               in bits 4i..4i+3, value 2i+1 in bits 16+4i..19+4i,
                               two's complement); bf16 scales, one per `group` = 128
                               K values ([rows][K/128]) or, with group = 0, one per
                               output row ([rows], channel-wise) [R1].
                               The pair order is this library's storage layout: it
                               is NOT the sequential nibble order of the
                               pack-quantized checkpoint format [R1] (value j in
                               bits 4j..4j+3).  Convert sequential words once, when
                               the weights are loaded, with moe_repack_int4. */

/* ---- grouped GEMM operations ---- */
#define MOE_OP_GATE_UP_SWIGLU 0  /* h = silu(a.Wg^T) * (a.Wu^T) -> bf16               */
#define MOE_OP_DOWN_WEIGHTED 1   /* o = w_row * (h.Wd^T)      -> fp32                 */

/* ---- entries (for moe_workspace_size) ---- */
#define MOE_ENTRY_ROUTE 0
#define MOE_ENTRY_PERMUTE 1
#define MOE_ENTRY_GROUPED_GEMM 2
#define MOE_ENTRY_FORWARD 3
#define MOE_ENTRY_FORWARD_HOST 4
#define MOE_ENTRY_FORWARD_EXPERTS 5

/* ---- source layouts of packed int4 words (moe_repack_int4) ---- */
#define MOE_INT4_SEQUENTIAL 0          /* value j in bits 4j..4j+3, two's complement */
#define MOE_INT4_SEQUENTIAL_OFFSET8 1  /* value j in bits 4j..4j+3, stored as q + 8  */

/*
 * Shapes of one layer call.
 *   T        tokens (1 .. 2^20), D hidden size (multiple of 128),
 *   E        routed experts (1 .. 1024), I / I_shared expert intermediate sizes
 *            (multiples of 64), k experts per token (1 .. min(E, 32)),
 *   quant    MOE_QUANT_*; for W4A16, group = 128 (group scales) or 0
 *            (channel-wise scales), and D, I, I_shared are multiples of 256
 *            (packed K tiles of 256 values).
 */
typedef struct moe_config {
  int T, D, E, I, I_shared, k;
  int quant;
  int group;
} moe_config;

/*
 * Layer weights (device pointers).  Gate/up of an expert is one [2I][D]
 * matrix with the I gate rows first; down is [D][I].  Both are K-major:
 * rows are output features [P1, reading of the expert form].
 *   quant == BF16 : w_gate_up bf16 [E][2I][D], w_down bf16 [E][D][I];
 *                   scale pointers must be NULL.
 *   quant == W4A16: w_gate_up int32 [E][2I][D/8] + s_gate_up bf16 [E][2I][D/group],
 *                   w_down int32 [E][D][I/8] + s_down bf16 [E][D][I/group];
 *                   with group = 0: s_gate_up bf16 [E][2I], s_down bf16 [E][D].
 *   The shared expert (ws_*, ss_*) has the same format with I_shared and no
 *   leading E.  w_router is bf16 [E][D] in both cases; router_bias is fp32 [E]
 *   or NULL.
 */
typedef struct moe_weights {
  const void *w_router;
  const float *router_bias;
  const void *w_gate_up, *w_down, *s_gate_up, *s_down;
  const void *ws_gate_up, *ws_down, *ss_gate_up, *ss_down;
} moe_weights;

/*
 * Arguments of one grouped GEMM over the E routed experts, plus an optional
 * shared-expert group covering all T tokens with weight 1 [P1, PM, R1G].
 * Routed group e owns GEMM rows [offsets[e], offsets[e+1]).
 *   op == GATE_UP_SWIGLU:
 *     a      bf16 [rows][D]; row r of the GEMM reads a[r], or a[a_row_index[r]]
 *            when a_row_index is non-NULL (then `a` is [T][D] and a_row_index
 *            holds token indices; the rows are gathered into the workspace);
 *     w      expert gate/up weights (format per cfg->quant), w_scales or NULL;
 *     out    bf16 [P][I]: h = silu(a.Wg^T) * (a.Wu^T), rounded once to bf16.
 *     a_shared bf16 [T][D] (NULL: no shared group), w_shared/ws_scales the
 *            shared gate/up weights, out_shared bf16 [T][I_shared].
 *   op == DOWN_WEIGHTED:
 *     a      bf16 [P][I] (a_row_index must be NULL);
 *     w      expert down weights; out fp32 [P][D] = wgt(r) * (a_r . Wd^T),
 *            wgt(r) = the blob weight of pair perm_pair[r] (t = p/k, j = p%k).
 *     a_shared bf16 [T][I_shared], w_shared [D][I_shared], out_shared fp32 [T][D]
 *            (weight 1).
 */
typedef struct moe_gemm_args {
  int op;
  const void *a;
  const int32_t *a_row_index;
  const int32_t *offsets;
  const void *w, *w_scales;
  const int32_t *perm_pair;
  const int32_t *blob;
  void *out;
  const void *a_shared;
  const void *w_shared, *ws_scales;
  void *out_shared;
} moe_gemm_args;

/*
 * Workspace bytes an entry needs for `cfg` (0 on invalid config).  The first
 * 256 bytes of every workspace are a status header read by moe_get_status:
 * zero them once when the workspace is created (the status word is then
 * written only by a kernel that records an error, and cleared only by
 * moe_get_status).
 */
size_t moe_workspace_size(const moe_config *cfg, int entry);

/*
 * Router [P1, P3]: logits z = x.Wr^T + bias, top-k by (logit desc, index asc),
 * softmax over all E then renormalised over the k selected, packed into
 *   blob int32 [T][2][k]: blob[t][0][j] = expert id (ascending in j),
 *                         blob[t][1][j] = fp32 bit pattern of its weight.
 * The selected set equals the one decided by fp64 index-order logits: fp32
 * tensor-core logits carry an error radius, and tokens whose boundary it does
 * not certify are re-decided with a compensated fp32 sum and, if still not
 * separated, with the fp64 definition itself.
 *   x bf16 [T][D], w_router bf16 [E][D], bias fp32 [E] or NULL.
 */
int moe_route(const moe_config *cfg, const void *x, const void *w_router,
              const float *bias, int32_t *blob, void *ws, size_t ws_bytes,
              void *stream);

/*
 * Router logits [P1] ("Systems engineering playbook: optimizing Qwen 3.5-397B
 * MoE on Ironwood (TPU7x)", section 1: the router gate projection), the first
 * step of moe_route on its own:
 *   z fp32 [T][E] = x.Wr^T (no bias), computed on the tensor cores with one
 *   fresh fp32 accumulator per 64-wide K chunk and the chunk values added in
 *   K order.  moe_route certifies its decisions assuming
 *   |z - exact| <= 2^-15 * sum_d |x_d Wr_ed| + (D/64 + 2) * 2^-24 * sum_d |x_d Wr_ed|.
 *   x bf16 [T][D], w_router bf16 [E][D]; ws sized for MOE_ENTRY_ROUTE.
 * Errors: as moe_route; a device wait that runs out sets MOE_ERR_TIMEOUT in
 * the status word (moe_get_status).
 */
int moe_router_logits(const moe_config *cfg, const void *x, const void *w_router, float *z,
                      void *ws, size_t ws_bytes, void *stream);

/*
 * Dispatch [P3B]: group the T*k (token, slot) pairs by expert, stable in the
 * pair index p = t*k + j.
 *   counts int32 [E], offsets int32 [E+1] (exclusive scan; offsets[E] = T*k),
 *   perm_pair int32 [T*k]: grouped row r holds pair perm_pair[r],
 *   inv_row int32 [T*k]:   pair p sits in grouped row inv_row[p].
 * If x (bf16 [T][D]) and x_perm (bf16 [T*k][D]) are both non-NULL, the token
 * rows are also copied in grouped order: x_perm[r] = x[perm_pair[r] / k].
 * Bit-exact and deterministic.  Expert ids outside [0, E) are clamped into it
 * and recorded as MOE_ERR_INVALID_ARG in the status word of ws.
 */
int moe_permute(const moe_config *cfg, const int32_t *blob, int32_t *counts,
                int32_t *offsets, int32_t *perm_pair, int32_t *inv_row,
                const void *x, void *x_perm, void *ws, size_t ws_bytes,
                void *stream);

/*
 * moe_permute_static: moe_permute for callers that cannot allocate device
 * memory.  (This entry point has no counterpart in the pages; it is an
 * interface convenience of this library.)
 *
 * Some callers cannot call cudaMalloc or hand the library a workspace: a
 * plug-in or foreign-language caller that holds only the tensors it was given,
 * an engine whose device memory is owned by an allocator this call site cannot
 * reach, or a serving loop that must not allocate once it is running.  This
 * variant needs no workspace: its scratch (the per-chunk expert count table)
 * is a fixed array inside the library, 65536 int32 (256 KiB), kept in every
 * GPU that loads the library until the process exits.  The call allocates
 * nothing and calls no allocating routine.
 *   Same arguments and results as moe_permute, bit for bit, without ws.
 *   Limit: ceil(T*k / 2048) * E <= 65536 (e.g. E = 512: T*k <= 262144);
 *   larger problems return MOE_ERR_SCRATCH_LIMIT and launch nothing.
 *   The array's device address belongs to the CUDA context: the first call
 *   in a context (the primary context of a device, or one made current with
 *   cuCtxCreate / after a reset) looks it up with that context current and
 *   caches it by the context's unique ID; make that first call before any
 *   stream capture.
 *   All calls share the one array: calls that may overlap on the GPU (other
 *   streams, other host threads) race and must be serialised by the caller.
 *   Each call writes every table entry it reads, so no clearing is needed.
 */
int moe_permute_static(const moe_config *cfg, const int32_t *blob,
                       int32_t *counts, int32_t *offsets, int32_t *perm_pair,
                       int32_t *inv_row, const void *x, void *x_perm,
                       void *stream);

/*
 * Persistent grouped GEMM over ragged expert row groups (TMA + tcgen05/TMEM)
 * [PM, R1G, R1]; see moe_gemm_args for operands.  W4A16 weights stay packed
 * and are restored tile by tile on chip just ahead of the MMA (into tensor
 * memory for token tiles of up to 64 rows, into shared memory for 256-row
 * tiles) [R1].  The call first copies `offsets` (clamped into [0, T*k] and
 * made non-decreasing) and `perm_pair` (clamped into [0, T*k)) into ws, and
 * the kernels read those copies; a value that needed clamping is recorded as
 * MOE_ERR_INVALID_ARG in the status word.  ws sized for MOE_ENTRY_GROUPED_GEMM.
 */
int moe_grouped_gemm(const moe_config *cfg, const moe_gemm_args *args, void *ws,
                     size_t ws_bytes, void *stream);

/*
 * Combine / unpermute [PM, P3B]:
 *   y[t][d] = bf16_rne( o_shared[t][d] + sum_j o[inv_row[t*k+j]][d] )
 * with o fp32 [T*k][D] already weighted, o_shared fp32 [T][D] or NULL, y bf16 [T][D].
 */
int moe_combine(const moe_config *cfg, const float *o, const float *o_shared,
                const int32_t *inv_row, void *y, void *stream);

/*
 * Whole layer [P1, P3, P3B, PM]: route (softmax over E, top-k, renormalised,
 * packed blob) -> permute (dispatch by expert) -> grouped gate/up + SiLU.mul
 * (routed experts and the always-on shared expert) -> grouped down with the
 * routing weight -> combine (unpermute, sum, one bf16 rounding).
 *   x bf16 [T][D], y bf16 [T][D]; ws sized for MOE_ENTRY_FORWARD.
 * Errors: as the per-stage calls; nothing is launched on a host-side error.
 */
int moe_forward(const moe_config *cfg, const void *x, const moe_weights *w,
                void *y, void *ws, size_t ws_bytes, void *stream);

/*
 * moe_forward with HOST x and y (pinned memory recommended): copies x into the
 * workspace, runs the layer, copies y back, all ordered on `stream`.  From
 * T >= 512 the combine runs in chunks of tokens and each chunk's copy to the
 * host goes on the library's second stream (forked from and joined back to
 * `stream`), overlapping the combine of the next chunk; from T >= 4096 x is
 * likewise copied in 2048-token chunks, each routed once it has arrived.
 * Results equal moe_forward's bit for bit.  The caller synchronises `stream`
 * before reading y.
 */
int moe_forward_host(const moe_config *cfg, const void *x_host,
                     const moe_weights *w, void *y_host, void *ws,
                     size_t ws_bytes, void *stream);

/*
 * Expert-parallel slice of the layer [P3B, P3]: the part of the layer output
 * that one device of an expert-parallel group computes when it holds only the
 * routed experts [e_begin, e_end) ("Systems engineering playbook: optimizing
 * Qwen 3.5-397B MoE on Ironwood (TPU7x)", section 3, "Option B": every device
 * receives all tokens and the packed routing blob, filters the (token, slot)
 * pairs routed to its own experts, computes them, and the outputs are
 * reduce-scattered back to the devices that own the tokens; "3-to-2
 * All-Gather": ids and weights travel as the one int32 blob of moe_route).
 *   y_partial fp32 [T][D] = sum over slots j with e_begin <= ids[t][j] < e_end
 *                           of w[t][j] * FFN_{ids[t][j]}(x_t)
 *                         + FFN_shared(x_t) for shared_begin <= t < shared_end.
 * Summing y_partial over a partition of [0, E) whose parts give the shared
 * expert disjoint token ranges covering [0, T), and rounding once to bf16,
 * gives the layer output of moe_forward (up to the fp32 summation order).
 *   cfg       T = tokens in x and blob (all devices' tokens), E = ALL experts.
 *   x         bf16 [T][D];  blob int32 [T][2][k] as written by moe_route.
 *   w         routed weights of the LOCAL experts only: w_gate_up / w_down (and
 *             W4A16 scales) hold e_end - e_begin experts, local expert i being
 *             global expert e_begin + i; w_router and router_bias are unused
 *             (may be NULL); shared weights are needed when
 *             shared_end > shared_begin.
 *   0 <= e_begin < e_end <= E; 0 <= shared_begin <= shared_end <= T.
 *   ws sized for MOE_ENTRY_FORWARD_EXPERTS.
 * Errors: MOE_ERR_INVALID_ARG for a bad range or a missing pointer; otherwise
 * as moe_forward.  Expert ids in the blob outside [0, E) are clamped into it
 * and recorded as MOE_ERR_INVALID_ARG in the status word of ws.
 */
int moe_forward_experts(const moe_config *cfg, const void *x, const int32_t *blob,
                        const moe_weights *w, int e_begin, int e_end, int shared_begin,
                        int shared_end, float *y_partial, void *ws, size_t ws_bytes,
                        void *stream);

/*
 * Load-time conversion of packed int4 weights to this library's pair order
 * (MOE_QUANT_W4A16) [R1] ("vLLM TPU Inference v0.31.0: hierarchical MoE
 * dispatch and W4A16", 4-bit weight section: symmetric int4 weights in the
 * pack-quantized format, 8 values per int32).
 *   src       int32 [n_words], eight 4-bit values per word in sequential order
 *             (value j in bits 4j..4j+3, j = 0..7), as two's complement
 *             (MOE_INT4_SEQUENTIAL) or offset binary q + 8
 *             (MOE_INT4_SEQUENTIAL_OFFSET8);
 *   dst       int32 [n_words] in pair order (value 2i in bits 4i..4i+3, value
 *             2i+1 in bits 16+4i..19+4i), two's complement.  dst == src (in
 *             place) is allowed; otherwise the ranges must not overlap.
 * Bit-exact.  Both pointers are device pointers, 16-byte aligned.  Scales are
 * not touched.  MOE_ERR_INVALID_ARG for a null pointer or an unknown layout.
 */
int moe_repack_int4(const int32_t *src, int32_t *dst, size_t n_words, int src_layout,
                    void *stream);

/*
 * Device status of the calls that used `ws` since the status was last read:
 * synchronises `stream`, returns MOE_OK or the first device-side error
 * recorded (MOE_ERR_TIMEOUT when a bounded wait inside a kernel gave up,
 * MOE_ERR_INVALID_ARG when caller index data was out of range and clamped),
 * then clears it.  The status is sticky: no other entry point clears it, so an
 * error recorded by one call is still reported after later calls succeed.  A
 * kernel whose wait gave up stops issuing work, so any output written by a
 * call since the last MOE_OK status is not to be trusted.
 */
int moe_get_status(void *ws, void *stream);

/*
 * Self-test of the device-side timeout path: launches one CTA that holds
 * tensor memory, waits on a barrier that nothing ever completes, gives up after
 * `limit_ms` (1 .. 10000), records MOE_ERR_TIMEOUT in the status word of `ws`
 * (>= 256 bytes), frees the tensor memory and exits.  moe_get_status(ws, ...)
 * then returns MOE_ERR_TIMEOUT and the context stays usable.  This is the same
 * bounded-wait code every pipelined kernel of the library uses.
 */
int moe_selftest_wait_timeout(void *ws, size_t ws_bytes, unsigned int limit_ms,
                              void *stream);

/*
 * Releases what the library keeps between calls for the calling host thread
 * in the current CUDA context: the second stream and the two events that
 * split grouped GEMMs and moe_forward_host's chunked copies use (see the
 * conventions above).  Work already queued on them
 * still completes (the CUDA runtime defers the release), so the call is safe
 * with calls in flight.  The next split call creates them again.  Nothing
 * else is cached across calls except moe_permute_static's address of its
 * fixed array (a few bytes per context, kept for the process).
 * Returns MOE_OK, or MOE_ERR_CUDA if no context could be made current or a
 * destroy call failed.
 */
int moe_release_cache(void);

/* Static description of an error code. */
const char *moe_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
