/*
 * gdn.h -- C ABI of libgdn_gb300.so, the batched Gated DeltaNet (GDN)
 * speculative transaction for MTP speculative decoding, written for GB300
 * (sm_103a).
 *
 * One verify/commit cycle of a hybrid Qwen-style model, per GDN layer:
 *
 *   gdn_conv_verify   conv-ring read + width-4 causal depthwise conv + SiLU +
 *                     L2 norm of q/k + gated delta rule over the T
 *                     draft-plus-verify positions of every row, from the
 *                     pre-verification state, which it never writes.
 *   gdn_commit        once per cycle for all layers: keep the accepted prefix
 *                     keep[b] of every row; keep=0 and inactive rows restore
 *                     the pre-verification state exactly (nothing is
 *                     written); shifts the conv window; advances the per-row
 *                     committed offsets.
 *   gdn_flush         materialise commits that a DEFERRED-mode cycle left
 *                     pending in its workspaces.
 *   gdn_prefill_chunked  the same recurrence over a prompt of L tokens in
 *                     chunked (WY/UT) form, leaving state, conv ring and
 *                     offsets primed for the first verify.
 *
 * Passages this follows (page title, section):
 *  - "MTP inference: review and commit structure", Functional commits, item 2:
 *    GDN speculative transactions with verifier buffers, accepted-prefix state
 *    replay, grouped copies across layers and a compiled short convolution;
 *    item 4: the conv-cache mutation sits behind an operator boundary; Review
 *    fixes: grouped replay checks every input before combining layers.
 *  - "Add request-owned eight-way MTP serving for Qwen 35B", section 2 (per-row
 *    committed offsets; inactive rows use keep=0 and keep their state) and
 *    section 4 (the commit handles keep = 0, 1, 2; keep=0 restores the
 *    pre-verification state; padded and finished rows are inert).
 *  - "perf(qwen): full-context MTP draft prefill and replay-free rewind",
 *    Summary item 4: the rewind reruns only the GDN mixer on captured
 *    verification inputs from the pre-verification state.
 *  - The recurrence is the gated delta rule (Yang, Kautz & Hatamizadeh, "Gated
 *    Delta Networks", ICLR 2025): S_t = a_t S_{t-1} (I - b_t k_t k_t^T) +
 *    b_t v_t k_t^T, a_t = exp(g_t), o_t = S_t q_t with q_t, k_t L2-normalised
 *    and q_t scaled by 1/sqrt(d_k).
 *
 * Conventions shared by every call
 *  - Every pointer argument except `dims` and the host arrays of gdn_commit is
 *    a DEVICE pointer on the current CUDA device, owned by the caller, 16-byte
 *    aligned, to densely packed row-major storage in the layout stated.
 *    The library never allocates device memory and never frees caller memory.
 *  - bf16 tensors are passed as gdn_bf16 (the raw 16-bit pattern).
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every call
 *    only enqueues work; none synchronises the host except gdn_get_status.
 *  - Arguments are validated on the host before anything is launched; on error
 *    nothing is launched, the call returns a negative GDN_ERR_* code and
 *    gdn_last_error() describes it.  Launch failures return GDN_ERR_CUDA.
 *  - All verify/commit calls of one layer must be issued in stream order.
 *
 * Layouts (C = 2*H_k*d_k + H_v*d_v conv channels; R = width - 1 + T_max)
 *  x        [B][T][C]           bf16  raw pre-conv inputs, channels q | k | v:
 *                                     q [H_k][d_k], k [H_k][d_k], v [H_v][d_v]
 *  conv_w   [C][width]          bf16  taps; conv_w[c][width-1] multiplies the
 *                                     current token, conv_w[c][0] the oldest
 *  g, beta  [B][T][H_v]         fp32  log-decay (a = exp(g), g <= 0 expected)
 *                                     and write strength
 *  state    [B][H_v][d_v][d_k]  fp32  S with v ~ S k: row j (d_v) holds a
 *                                     contiguous d_k vector
 *  ring     [B][R][C]           bf16  conv cache: slots 0..2 hold the raw inputs
 *                                     of the three committed positions before the
 *                                     next token (oldest first); slots 3..2+T hold
 *                                     the raw inputs of the latest verify's T
 *                                     positions.  A fresh row has zeros in 0..2.
 *  offsets  [B]                 int32 committed tokens per row (one array shared
 *                                     by all layers); bookkeeping for the caller,
 *                                     advanced by gdn_commit and
 *                                     gdn_prefill_chunked, not read by verify
 *  active   [B]                 uint8 0 = inactive/padding/finished row
 *  out      [B][T][H_v][d_v]    bf16  o_t for each position
 *
 * Value head h reads key head floor(h * H_k / H_v).
 * Supported: d_k == d_v in {32, 64, 128}; width == 4; 1 <= T <= T_max <= 8;
 * H_v % H_k == 0; B <= 65535; H_v <= 65535.
 *
 * Numerics: the state and all arithmetic are fp32; bf16 appears only in the
 * inputs and outputs.  At d = 128 in RECOMPUTE and DEFERRED mode the verify
 * takes the dot products of the state rows with q_t and k_t on the tensor
 * cores in tf32 (the state read truncated to tf32, q and k rounded to it:
 * about 2^-11 of each term's magnitude); these products only enter e_t and
 * o_t through per-head coefficients, and the state itself, every state
 * update, conv, norm, gate and recurrence step stays in fp32.  Its results
 * differ from the CUDA-core path's (d = 32, 64, SNAPSHOT) only by rounding.
 * The chunked prefill takes its products on the tensor cores in bf16: three
 * passes (x = x_hi + x_lo, about 16 bits of each fp32 operand) for every
 * product that reaches the state, one pass for those that only reach the
 * bf16 outputs.  The d = 128 tensor-core verify addresses the state as
 * B * H_v * d_v rows of a tensor map, so it needs B * H_v * 128 < 2^31.
 */
#ifndef GDN_GB300_H
#define GDN_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t gdn_bf16; /* bfloat16 bit pattern */

/* return codes */
#define GDN_OK 0
#define GDN_ERR_INVALID_ARG (-1)   /* null pointer, bad enum, inconsistent sizes */
#define GDN_ERR_UNSUPPORTED (-2)   /* a shape outside the supported set above */
#define GDN_ERR_MISALIGNED (-3)    /* a device pointer not 16-byte aligned */
#define GDN_ERR_WORKSPACE (-4)     /* workspace smaller than the size query */
#define GDN_ERR_CUDA (-5)          /* a CUDA runtime call or launch failed */

/* conv activation */
#define GDN_ACT_NONE 0
#define GDN_ACT_SILU 1

/* commit strategies (chosen per call pair; verify and commit must agree) */
#define GDN_COMMIT_RECOMPUTE 0 /* verify captures k, the per-row delta
                                  coefficients and the cumulative decay; commit
                                  rebuilds S_keep from the untouched S_0 */
#define GDN_COMMIT_SNAPSHOT 1  /* verify writes S_1..S_T to the workspace;
                                  commit copies S_keep back */
#define GDN_COMMIT_DEFERRED 2  /* as RECOMPUTE, but gdn_commit only records
                                  keep and the state update of each (row, head)
                                  is applied by that layer's next verify, which
                                  reads the state anyway: each committed row is
                                  read once and written once per cycle.  The
                                  state buffer then lags the committed state
                                  until that verify or gdn_flush runs.  The
                                  workspace must be zero-filled once before its
                                  first use; dims must not change after that. */

/* flag OR-ed into the mode argument of gdn_conv_verify.  Every kernel of
 * the library is launched with programmatic dependent launch and waits for
 * the preceding kernel on the stream before reading anything it may write.
 * With GDN_VERIFY_OVERLAP the call's kernel also lets the next kernel on the
 * stream start as soon as it has started, and before waiting for its
 * predecessor it stages its own state tiles, reads its conv taps, committed
 * conv window (ring slots 0..2) and active mask, and warms L2 with its x, g
 * and beta (a prefetch only; those values are read after the wait), so
 * consecutive flagged verifies stream their state ahead of one another; in
 * DEFERRED mode it also fetches the captures of the layer's previous verify
 * and applies a pending commit (and writes it back) before that wait.  A
 * kernel of any other library call (including a verify flagged
 * GDN_VERIFY_OVERLAP_STATE) lets the next kernel start only after its own
 * wait, so a chain of flagged verifies never runs ahead of the last call
 * made without this flag.  The caller guarantees that no work issued since
 * that call writes this call's `state`, `conv_w`, ring slots 0..2, `active`
 * or `layer_ws`, and that the previous verify of this layer was issued
 * before that call.  In a verify cycle over a layer stack that means:
 * flag every layer but the first one after a gdn_commit (any mode),
 * gdn_prefill_chunked, gdn_flush, gdn_move_rows or any other write of these
 * buffers.  Never flag a repeated verify of the same layer.  At d = 128 a
 * flagged verify also takes 32 tensor-memory columns per CTA before that
 * wait; so the kernel that precedes it on the stream must not be one that,
 * after letting its dependents start, allocates tensor memory and needs more
 * than 416 of an SM's 512 columns (no kernel of this library does).  It is
 * always safe to omit. */
#define GDN_VERIFY_OVERLAP 0x100

/* A weaker flag for the first layer of a cycle after a DEFERRED gdn_commit
 * (OR-ed into the mode argument instead of GDN_VERIFY_OVERLAP, never with
 * it).  Before waiting for its predecessor the call stages its state tiles,
 * reads its conv taps and active mask and (DEFERRED) fetches the captures of
 * the layer's previous verify whether or not a commit is pending; the
 * pending keep and the conv window are read after the wait, and the next
 * kernel may start only after that wait, as for an unflagged call.  The caller guarantees that the work issued
 * since this layer's previous gdn_conv_verify does not write this call's
 * `state`, `conv_w`, `active` or the capture region of `layer_ws`: a
 * DEFERRED gdn_commit writes none of them (it writes the pending keep, the
 * conv windows and the offsets), while RECOMPUTE and SNAPSHOT commits write
 * the state and gdn_flush, gdn_prefill_chunked and gdn_move_rows write the
 * state and conv cache.  The tensor-memory condition of GDN_VERIFY_OVERLAP
 * applies too.  It acts at d = 128 in RECOMPUTE and DEFERRED mode and is the
 * same as no flag elsewhere.  It is always safe to omit. */
#define GDN_VERIFY_OVERLAP_STATE 0x200

/* sticky device status bits (gdn_get_status) */
#define GDN_STATUS_BAD_KEEP 1u /* an active row passed keep outside [0, T];
                                  that row was committed with keep = 0 */
#define GDN_STATUS_TIMEOUT 2u  /* a kernel gave up waiting for one of its own
                                  bulk copies or products (bounded wait); it
                                  wrote no output, capture or state for that
                                  (row, head) after the wait */
#define GDN_STATUS_BAD_ROW 4u  /* gdn_move_rows got a row index outside its
                                  cohort; that pair was not copied */

#define GDN_MAX_LAYERS 256     /* layers one gdn_commit call may group */

typedef struct gdn_dims {
  int32_t B;      /* rows in the cohort */
  int32_t T;      /* positions per verify, 1..T_max */
  int32_t T_max;  /* ring capacity parameter (R = width - 1 + T_max), <= 8 */
  int32_t H_k;    /* key heads */
  int32_t H_v;    /* value heads, a multiple of H_k */
  int32_t d_k;    /* key head size */
  int32_t d_v;    /* value head size (== d_k) */
  int32_t width;  /* conv width, must be 4 */
  int32_t act;    /* GDN_ACT_SILU or GDN_ACT_NONE */
} gdn_dims;

/* Library version string (static storage).  (The pages describe no such
 * call; it identifies the library build.) */
const char *gdn_version(void);

/* Message for the last error returned on the calling host thread ("" if none;
 * thread-local storage, valid until the next call on that thread).  Every
 * call validates its arguments and fails with a message before it launches
 * anything ("Add request-owned eight-way MTP serving for Qwen 35B",
 * Clean-install public launch verification: an incomplete launch contract
 * fails closed before any work). */
const char *gdn_last_error(void);

/*
 * Bytes of per-layer workspace that gdn_conv_verify fills and gdn_commit reads
 * for `mode`: the captured verification inputs that let the commit rerun the
 * recurrence over the accepted prefix ("perf(qwen): full-context MTP draft
 * prefill and replay-free rewind", Summary item 4); 0 if dims or mode are
 * invalid.  Regions are 256-byte aligned:
 *   RECOMPUTE  e [B][H_v][T][d_v], normalised k [B][H_k][T][d_k] and the
 *              cumulative log-decay [B][H_v][8], fp32:
 *              about 4*B*T*(H_v*d_v + H_k*d_k) + 32*B*H_v bytes;
 *   SNAPSHOT   S_1..S_T: 4*T*B*H_v*d_v*d_k bytes;
 *   DEFERRED   the pending keep [B][H_v] int32, then e and k (one copy per
 *              (row, value head): [B][H_v][T][d]) and the decay:
 *              about 4*B*H_v + 4*B*T*(2*H_v*d) + 32*B*H_v bytes.
 */
size_t gdn_layer_workspace_bytes(const gdn_dims *dims, int mode);

/*
 * Verify one layer: for every active row b run the T positions from the
 * committed window and the pre-verification state, writing o_t to `out`
 * ("MTP inference: review and commit structure", Functional commits item 2:
 * a speculative transaction that verifies from verifier buffers and leaves
 * the committed state to the accepted-prefix commit).
 *  - reads  x, conv_w, g, beta, state, ring slots 0..2, active;
 *  - writes out; ring slots 3..2+T of active rows (never the committed
 *    window); layer_ws (the captured verification quantities the matching
 *    gdn_commit needs).
 *  - RECOMPUTE / SNAPSHOT: never writes `state`.  DEFERRED: first applies the
 *    commit the last gdn_commit left pending for this layer to the state rows
 *    it concerns (also for rows now inactive), then verifies from them.
 *  - inactive rows get out = 0 and no ring access.
 *  - `offsets` is not read (it may be NULL).
 * layer_ws must stay untouched until the matching gdn_commit has run.
 * Errors: GDN_ERR_INVALID_ARG, _UNSUPPORTED, _MISALIGNED, _WORKSPACE
 * (layer_ws_bytes < gdn_layer_workspace_bytes), _CUDA.
 */
int gdn_conv_verify(const gdn_dims *dims, int mode, const gdn_bf16 *x, const gdn_bf16 *conv_w,
                    const float *g, const float *beta, const float *state, gdn_bf16 *ring,
                    const int32_t *offsets, const uint8_t *active, gdn_bf16 *out,
                    void *layer_ws, size_t layer_ws_bytes, void *stream);

/*
 * gdn_conv_verify followed, in the same kernel, by the gated RMSNorm that
 * comes after the GDN mixer in the hybrid-Qwen layer ("MTP inference: review
 * and commit structure", Functional commits item 4, keeps it behind its own
 * operator boundary): per (row, position, value head)
 *   out[j] = o[j] / sqrt(mean_j o[j]^2 + eps) * norm_w[j] * silu(gate_z[j])
 * with o the verify output (fp32 inside the kernel, never rounded).
 *  gate_z  [B][T][H_v][d_v] bf16  device, read only
 *  norm_w  [d_v]            bf16  device, read only (shared by all heads)
 *  eps     finite, >= 0
 * Everything else, including the captures for gdn_commit, is as for
 * gdn_conv_verify; inactive rows get out = 0.
 */
int gdn_conv_verify_gated(const gdn_dims *dims, int mode, const gdn_bf16 *x, const gdn_bf16 *conv_w,
                          const float *g, const float *beta, const float *state, gdn_bf16 *ring,
                          const int32_t *offsets, const uint8_t *active, const gdn_bf16 *gate_z,
                          const gdn_bf16 *norm_w, float eps, gdn_bf16 *out, void *layer_ws,
                          size_t layer_ws_bytes, void *stream);

/*
 * Commit the accepted prefix of every row for n_layers layers in one launch
 * (grouped across layers: "MTP inference: review and commit structure",
 * Functional commits item 2, accepted-prefix state replay with grouped copies;
 * "Add request-owned eight-way MTP serving for Qwen 35B", section 4, keep =
 * 0, 1, 2 per row with keep = 0 restoring the pre-verification state).  keep'[b] = keep[b] if active[b] and
 * 0 <= keep[b] <= T, else 0 (an active row with keep outside [0, T] also sets
 * GDN_STATUS_BAD_KEEP).  For keep' >= 1 the layer's state rows of b become the
 * state after the first keep' positions (RECOMPUTE, SNAPSHOT: now; DEFERRED:
 * recorded, applied by the layer's next verify or gdn_flush) and the conv
 * window becomes ring slots keep'..keep'+2 (written to slots 0..2); for
 * keep' = 0 nothing of row b is written (exact restore).
 * offsets[b] += keep' (once, not per layer).
 *  state    host array [n_layers] of device pointers to each layer's state
 *  ring     host array [n_layers] of device pointers to each layer's ring
 *  layer_ws host array [n_layers] of device pointers to each layer's workspace
 *           (as filled by that layer's gdn_conv_verify with the same dims/mode)
 *  keep, active, offsets  device arrays [B]; keep/active are read on the
 *           device, so the call can be captured in a CUDA graph.
 * Errors: GDN_ERR_INVALID_ARG (n_layers outside 1..GDN_MAX_LAYERS, null
 * entries), _UNSUPPORTED, _MISALIGNED, _CUDA.
 */
int gdn_commit(const gdn_dims *dims, int mode, int n_layers, float *const *state,
               gdn_bf16 *const *ring, void *const *layer_ws, const int32_t *keep,
               const uint8_t *active, int32_t *offsets, void *stream);

/*
 * Apply every commit a DEFERRED cycle left pending in the n_layers layer
 * workspaces to the state buffers, so that they hold the committed state (as
 * an eager commit would have left them: the accepted-prefix state of "MTP
 * inference: review and commit structure", Functional commits item 2).  Call it before reading a state
 * buffer directly, before gdn_prefill_chunked, and before switching a layer
 * to another mode.  Idempotent; a no-op for RECOMPUTE and SNAPSHOT.
 * Errors: as gdn_commit.
 */
int gdn_flush(const gdn_dims *dims, int mode, int n_layers, float *const *state,
              void *const *layer_ws, void *stream);

/*
 * Bytes of workspace gdn_prefill_chunked needs for a prompt of L tokens (the
 * per-chunk operands of the chunked form, "MTP inference: review and commit
 * structure", Verification and limits); 0 if the arguments are invalid.
 */
size_t gdn_prefill_workspace_bytes(const gdn_dims *dims, int L);

/*
 * Prime every row over a prompt of L tokens in chunked form (chunk = 64; "MTP
 * inference: review and commit structure", Verification and limits: the
 * chunked recurrence used for a prompt differs from the sequential one only
 * in its rounding boundaries):
 * conv from the committed window (ring slots 0..2), L2 norm, then per chunk
 * the UT transform of the decay-weighted strictly-lower K K^T block on tensor
 * cores and a sequential pass of the state across chunks.  Equivalent, up to
 * rounding, to gdn_conv_verify with T = L followed by gdn_commit with
 * keep = L for all rows.
 *  x [B][L][C] bf16; g, beta [B][L][H_v] fp32; state [B][H_v][d_v][d_k] fp32
 *  in (initial) / out (final); ring slots 0..2 set to the last three raw
 *  inputs of window ++ prompt; offsets[b] += L; out [B][L][H_v][d_v] bf16.
 * A layer run in DEFERRED mode must be flushed (gdn_flush) first.
 * dims->T and T_max describe the ring the state is primed for (R = 3 + T_max).
 * At d = 128, for prompts of 24 or more chunks with 2 * B * H_v at most the
 * SM count, the sequential state pass of each chunk range runs on `stream`
 * at the device's highest launch priority while the products of the later
 * ranges run on an internal stream of the current device (created on first
 * use), forked from `stream` after the first range's products; events order
 * the two and `stream` ends behind the last state pass, so all work is
 * complete in `stream` order as for any other call (and a call captured into
 * a CUDA graph captures both streams).
 * Errors: as gdn_conv_verify; GDN_ERR_WORKSPACE if ws_bytes is too small.
 */
int gdn_prefill_chunked(const gdn_dims *dims, int L, const gdn_bf16 *x, const gdn_bf16 *conv_w,
                        const float *g, const float *beta, float *state, gdn_bf16 *ring,
                        int32_t *offsets, gdn_bf16 *out, void *ws, size_t ws_bytes,
                        void *stream);

/*
 * gdn_conv_verify_noalloc -- gdn_conv_verify for callers that cannot allocate
 * device memory.  (The pages describe no such call; it exists for hosts of
 * this library.)
 *
 * Some callers have no way to hand the library a workspace: a plug-in running
 * inside a host framework that owns every device allocation and gives the
 * plug-in only its input and output tensors, or a latency-critical serving
 * loop where a cudaMalloc (which can synchronise the device) is not allowed
 * once serving has started.  This entry point does what gdn_conv_verify does,
 * with the same arguments except the workspace: the verify captures go to a
 * scratch array built into the library's device code, GDN_NOALLOC_WS_BYTES
 * (4 MiB) per GPU, which every GPU that loads the library holds until the
 * process exits.  It allocates nothing and frees nothing.
 *  - DEFERRED mode is not accepted (its workspace must persist per layer).
 *  - Shapes whose workspace (gdn_layer_workspace_bytes) exceeds the scratch
 *    are rejected with GDN_ERR_WORKSPACE before anything is launched (e.g. the
 *    B=8, T=2, 32x128 cohort needs about 0.4 MiB in RECOMPUTE mode and fits;
 *    its SNAPSHOT mode needs 32 MiB and does not).
 *  - The first call on each device looks up the scratch's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture begins.
 *  - The scratch's device address is stored in *layer_ws_used (if not NULL):
 *    pass it as this layer's workspace to gdn_commit (n_layers = 1).
 *  - Every call shares the one scratch array and it keeps the last call's
 *    contents; nothing in it needs to start at zero, since verify writes every
 *    entry the commit reads.  The captures of one call are valid only until
 *    the next call of this entry point on the same device, so commit that
 *    layer before verifying another with it.  Calls that overlap on the GPU
 *    (other streams, other host threads) race on the scratch.
 * Errors: as gdn_conv_verify, plus GDN_ERR_WORKSPACE for shapes too large.
 */
#define GDN_NOALLOC_WS_BYTES (4u << 20)
int gdn_conv_verify_noalloc(const gdn_dims *dims, int mode, const gdn_bf16 *x, const gdn_bf16 *conv_w,
                            const float *g, const float *beta, const float *state, gdn_bf16 *ring,
                            const int32_t *offsets, const uint8_t *active, gdn_bf16 *out,
                            void **layer_ws_used, void *stream);

/*
 * Read the sticky device status word of the current device (GDN_STATUS_*
 * bits) into *status; clear it if `clear` is nonzero.  Synchronises the
 * device.  Returns GDN_OK or GDN_ERR_CUDA / GDN_ERR_INVALID_ARG.  Conditions
 * found on the device (a keep outside [0, T], a row index outside its cohort,
 * a bounded wait that ran out) cannot fail the launch that met them; the
 * kernel takes the safe action (commit nothing, copy nothing, write nothing
 * more) and records the condition here ("Add request-owned eight-way MTP
 * serving for Qwen 35B", section 4: keep = 0 restores the pre-verification
 * state; Clean-install public launch verification: fail closed).
 */
int gdn_get_status(int clear, uint32_t *status);

/* ---- joining rows into a cohort ------------------------------------------------
 * Copy, for every layer, the decode state of row src_rows[i] of one cohort
 * into row dst_rows[i] of another (or the same) cohort, i < n_rows: the fp32
 * state, the whole conv cache row and the committed offset.  This is how a
 * row primed by gdn_prefill_chunked (B = 1) joins a verify cohort ("Add
 * request-owned eight-way MTP serving for Qwen 35B", sections 2 and 3: rows
 * enter the eight-way cohort with their own committed offsets).
 *  src_dims, dst_dims  equal H_k, H_v, d_k, T_max, width; B may differ
 *  src_state, dst_state, src_ring, dst_ring  host arrays [n_layers] of device pointers
 *  src_offsets, dst_offsets  [B] int32 device
 *  dst_layer_ws  DEFERRED only: the destination cohort's layer workspaces; the
 *                destination rows' pending keep is cleared.  The source must
 *                have no commit pending (gdn_flush it first).
 *  src_rows, dst_rows  [n_rows] int32 device; destination rows distinct, and
 *                none of them a source row of another pair when the cohorts
 *                share memory.  A pair with an index outside its cohort is
 *                skipped and sets GDN_STATUS_BAD_ROW.
 */
int gdn_move_rows(const gdn_dims *src_dims, const gdn_dims *dst_dims, int mode, int n_layers,
                  const float *const *src_state, const gdn_bf16 *const *src_ring, const int32_t *src_offsets,
                  float *const *dst_state, gdn_bf16 *const *dst_ring, int32_t *dst_offsets,
                  void *const *dst_layer_ws, const int32_t *src_rows, const int32_t *dst_rows, int n_rows,
                  void *stream);

/* ---- on-device greedy acceptance ---------------------------------------------
 * "Add request-owned eight-way MTP serving for Qwen 35B" takes the acceptance
 * decision of the batched decode cycle off the host, so a cycle needs no host
 * synchronisation.  Position 0 of a row's verify holds the last accepted
 * token, positions 1..T-1 the draft tokens.  For every active row b:
 *   target_t = argmax_v logits[b][t][v]   first index of the maximum; NaN never
 *                                          wins; an all-NaN position gives 0
 *   keep[b]  = 1 + the number of leading t in 1..T-1 with
 *              draft[b][t] == target_{t-1}
 *   next[b]  = target_{keep[b]-1}          the token the next cycle feeds
 * Inactive rows get keep 0 and next -1.  keep is what gdn_commit takes, so
 * verify -> accept -> commit runs on one stream with no host round trip.
 *
 *  logits [B][T][V]  bf16   device, read only
 *  draft  [B][T]     int32  device; draft[b][0] is not read
 *  active [B]        uint8  device
 *  keep, next [B]    int32  device, written
 *  ws                device scratch of gdn_accept_workspace_bytes(B, T, V)
 *                    bytes, zero-filled once before its first use (each call
 *                    leaves it ready for the next)
 * Supported: 1 <= T <= 64, V >= 1, B*T <= 65535.  Errors as for every call.
 */
size_t gdn_accept_workspace_bytes(int B, int T, int V);
int gdn_accept_greedy(int B, int T, int V, const gdn_bf16 *logits, const int32_t *draft, const uint8_t *active,
                      int32_t *keep, int32_t *next, void *ws, size_t ws_bytes, void *stream);

/* ---- test hook ---------------------------------------------------------------
 * gdn_conv_verify at d = 128 (RECOMPUTE or DEFERRED) with its failure path
 * forced, for tests of that path.  (The pages describe no such call; it
 * exercises the bounded waits that every kernel of the library puts on its
 * own copies.)  The CTA of (row 0, head 0) announces 16 bytes more on one of
 * its state-tile barriers than its copy delivers, so that barrier's phase
 * never completes; every bounded wait of the call gives up after wait_limit
 * polls instead of the library's default (a poll lasts at most about a
 * microsecond).  That CTA then sets GDN_STATUS_TIMEOUT, waits (bounded) for
 * its own copies, writes no output, no capture and no state (it may already
 * have written its new ring inputs, slots 3..2+T) and leaves; every other
 * CTA completes as in gdn_conv_verify.  Row 0 must be active.  Contract after
 * a timeout: the layer's state is unchanged in RECOMPUTE mode (in DEFERRED
 * mode a commit that was pending for (row 0, head 0) stays pending), and the
 * next ordinary gdn_conv_verify of the layer recomputes everything it
 * writes.  Errors: as gdn_conv_verify, plus GDN_ERR_UNSUPPORTED for another
 * head size or SNAPSHOT mode.
 */
int gdn_test_verify_timeout(const gdn_dims *dims, int mode, const gdn_bf16 *x, const gdn_bf16 *conv_w,
                            const float *g, const float *beta, const float *state, gdn_bf16 *ring,
                            const int32_t *offsets, const uint8_t *active, gdn_bf16 *out, void *layer_ws,
                            size_t layer_ws_bytes, uint32_t wait_limit, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_GB300_H */
