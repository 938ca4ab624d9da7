/*
 * mk.h — C ABI of the GB300 whole-model decode megakernel (libmk.so).
 *
 * One decode step of a whole decoder stack runs as ONE persistent CUDA kernel launch with one CTA per
 * SM: embedding, every layer's RMSNorm, projections, attention (GQA or MLA) or delta-rule recurrence
 * (gated delta net or KDA), SwiGLU feed-forward or MoE (router, shared and routed experts), residual,
 * final norm, LM head and greedy argmax. Weight loads run ahead of compute across op and layer
 * boundaries through a shared-memory ring. The design follows the pages' megakernel idea — one
 * program for the whole layer stack, with a weight load issued as early as on-chip storage allows
 * instead of at the start of the op that uses it (Kimi K3's TPU megakernel, "What a megakernel is,
 * and what it fixes on a TPU"; tpu-megakernels README, intro) — re-designed for one GB300.
 *
 * Conventions for every call:
 *   - Pointers named "device" are CUDA device pointers on the handle's device; "host" pointers are
 *     ordinary (pageable or pinned) host memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream). Device work is
 *     enqueued on it and the call returns without waiting, unless the call says otherwise.
 *   - Host-side argument errors are returned at once and enqueue nothing. Errors found on the device
 *     (a token id outside [0, vocab), a position outside the sequence's valid window, a watchdog
 *     timeout of an inter-SM wait) are recorded in the handle's device status word, the kernel exits
 *     early, and mk_get_status() reports them.
 *   - A handle is not thread-safe: calls on one handle must come from one host thread at a time and
 *     must use streams that are ordered with each other.
 *   - No call falls back to the CPU and no call takes PyTorch types.
 */
#ifndef MK_H_
#define MK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MK_MAX_LAYERS 128

typedef enum mk_status {
  MK_OK = 0,
  MK_ERR_INVALID_ARG = 1,  /* a host-side argument is out of range or inconsistent            */
  MK_ERR_UNSUPPORTED = 2,  /* shape or feature this build does not implement                   */
  MK_ERR_NOMEM = 3,        /* cudaMalloc failed                                                 */
  MK_ERR_CUDA = 4,         /* a CUDA runtime call failed (see mk_last_error)                   */
  MK_ERR_TIMEOUT = 5,      /* device watchdog: an inter-SM wait exceeded its time limit         */
  MK_ERR_DEVICE = 6        /* device-side input check failed (token id, position window)        */
} mk_status;

typedef enum mk_mixer {
  MK_MIXER_GQA = 0, /* grouped-query softmax attention over a bf16 KV cache, RoPE               */
  MK_MIXER_GDN = 1, /* gated delta net: one sigmoid decay per head, fp32 state [dk x dv]/head    */
  MK_MIXER_KDA = 2, /* Kimi delta attention: one sigmoid decay per key channel                   */
  MK_MIXER_MLA = 3  /* multi-head latent attention, absorbed form, bf16 latent cache              */
} mk_mixer;

typedef enum mk_ffn { MK_FFN_DENSE = 0, MK_FFN_MOE = 1 } mk_ffn;
typedef enum mk_expert_format { MK_FMT_BF16 = 0, MK_FMT_NVFP4 = 1 } mk_expert_format;

/* Model shape. Every layer is  x += Mixer(RMSNorm(x)); x += FFN(RMSNorm(x))  (pre-norm, no biases),
 * then a final RMSNorm and the LM head. RMSNorm gains multiply. */
typedef struct mk_model_desc {
  int32_t n_layers;
  int32_t d_model;
  int32_t vocab;
  int32_t tied_embedding;          /* 1: the LM head is the embedding matrix                   */
  float norm_eps;                  /* RMSNorm epsilon (also used for the MLA c_q / c_kv norms) */
  float rope_theta;                /* rotate-half RoPE base                                    */
  int32_t mixer[MK_MAX_LAYERS];    /* mk_mixer per layer                                      */
  /* GQA */
  int32_t n_q_heads, n_kv_heads, head_dim;
  /* GDN / KDA */
  int32_t lin_heads, lin_dk, lin_dv;
  /* MLA */
  int32_t mla_heads, q_lora, kv_lora, qk_nope, qk_rope, v_head;
  /* FFN */
  int32_t ffn_kind;                /* mk_ffn                                                    */
  int32_t ffn_dim;                 /* dense SwiGLU hidden size                                 */
  int32_t n_experts, top_k, n_shared, expert_dim, expert_format;
  float route_scale;               /* routed weights = route_scale * s_sel / sum(s_sel)         */
  /* capacity of the handle */
  int32_t max_batch;               /* sequences the handle holds (at most 256; a call uses 64 at most)*/
  int32_t max_rows;                /* query rows per sequence per call (at most 8; a call's batch x
                                      rows may not exceed 64)                                    */
  int32_t max_ctx;                 /* positions per sequence (KV / latent cache length)         */
} mk_model_desc;

/* Device pointers of one layer's weights. bf16 matrices are row-major [out, in] (the input
 * dimension contiguous) unless stated. Unused entries are NULL. */
typedef struct mk_layer_weights {
  const void* attn_norm;           /* bf16 [d]                                                 */
  const void* ffn_norm;            /* bf16 [d]                                                 */
  /* GQA: wq [Hq*hd, d], wk/wv [Hkv*hd, d], wo [d, Hq*hd]
   * GDN/KDA: wq/wk [H*dk, d], wv [H*dv, d], wa [H, d] (GDN) or [H*dk, d] (KDA), wb [H, d],
   *          wo [d, H*dv]
   * MLA: wo [d, H*v_head] */
  const void *wq, *wk, *wv, *wo, *wa, *wb;
  /* MLA: w_dq [q_lora, d], q_norm [q_lora], w_uq [H*(nope+rope), q_lora] (per head: nope then rope),
   *      w_dkv [kv_lora+rope, d] (latent then rope key), kv_norm [kv_lora],
   *      w_uk [H, kv_lora, nope] (k_nope = w_uk[h]^T c;  absorbed query = w_uk[h] q_nope),
   *      w_uv [H, v_head, kv_lora] (v = w_uv[h] c) */
  const void *w_dq, *q_norm, *w_uq, *w_dkv, *kv_norm, *w_uk, *w_uv;
  /* dense SwiGLU: w_gate/w_up [F, d], w_down [d, F] */
  const void *w_gate, *w_up, *w_down;
  /* MoE: w_router bf16 [E, d]; router_bias fp32 [E] (may be NULL = zero bias)
   * routed experts e_gate/e_up [E, F, d], e_down [E, d, F]; shared s_gate/s_up [S, F, d],
   * s_down [S, d, F]. bf16: the pointers are bf16 tensors and the *_scales / *_gscale entries are
   * NULL. NVFP4: the pointers are packed e2m1 codes (uint8, 2 per byte, element 2i in the low
   * nibble, [.., in/2]), *_scales are e4m3 block scales (uint8 [.., in/16], one per 16 inputs) and
   * *_gscale are fp32 per-expert tensor scales [E] or [S]; w = e2m1 * e4m3 * gscale. */
  const void* w_router;
  const float* router_bias;
  const void *e_gate, *e_up, *e_down, *s_gate, *s_up, *s_down;
  const uint8_t *e_gate_scales, *e_up_scales, *e_down_scales;
  const uint8_t *s_gate_scales, *s_up_scales, *s_down_scales;
  const float *e_gate_gscale, *e_up_gscale, *e_down_gscale;
  const float *s_gate_gscale, *s_up_gscale, *s_down_gscale;
} mk_layer_weights;

typedef struct mk_weights {
  const void* embed;       /* bf16 [vocab, d]                                              */
  const void* final_norm;  /* bf16 [d]                                                     */
  const void* lm_head;     /* bf16 [vocab, d]; NULL when tied_embedding                    */
  mk_layer_weights layers[MK_MAX_LAYERS];
  /* The dense projection matrices (every matrix above except the embedding table, the norms, the
   * routed / shared experts and w_uk / w_uv) in the kernel's tiled layout, written by mk_pack_weights
   * for this model and device; or NULL, and mk_create makes its own copy (mk_decode_step_static needs
   * it). Device memory owned by the caller, 1024-byte aligned, kept alive and unchanged while used. */
  const void* packed;
} mk_weights;

typedef struct mk_handle mk_handle;

/* Read-only facts about a handle (for harnesses and byte accounting). */
typedef struct mk_info {
  int32_t n_sm;             /* CTAs per launch = SMs of the device                          */
  int32_t threads_per_cta;
  int32_t smem_bytes;       /* dynamic shared memory per CTA                                */
  int32_t ring_slots;       /* weight-ring slots per SM                                     */
  int32_t ring_slot_bytes;
  int32_t n_ops_last;       /* ops in the program of the last step                          */
  int64_t device_bytes;     /* device memory owned by the handle                            */
} mk_info;

/* Creates a handle on `device`. The caller keeps ownership of every weight buffer and must keep
 * them alive and unchanged until mk_destroy. The handle allocates (cudaMalloc) and owns the KV /
 * latent caches, the recurrent states, activation scratch, instruction queues, counters and the
 * status word; and, when weights->packed is NULL, a tiled copy of the dense projection matrices
 * (mk_pack_weights' layout; as large as those matrices), made here, which the decode path reads
 * instead of the caller's matrices. Synchronous. Errors: MK_ERR_INVALID_ARG (inconsistent shape, missing weight,
 * alignment: every weight must be 16-byte aligned and every inner dimension a multiple of 8),
 * MK_ERR_UNSUPPORTED, MK_ERR_NOMEM, MK_ERR_CUDA.
 * Passage: the pages define no API for the kernel (their interface is a CLI and an HTTP server); this
 * call holds what their kernel receives as arguments: the model's shapes and every weight as a raw
 * reference into HBM (Kimi K3's TPU megakernel, "How it maps onto a TPU v7"). */
mk_status mk_create(const mk_model_desc* desc, const mk_weights* weights, int device, mk_handle** out);

/* Fills the caches and recurrent states of sequences 0..batch-1 from a context of n_tokens tokens
 * each (device int32 [batch, n_tokens], row-major), discarding whatever they held. Afterwards each
 * sequence has n_tokens committed tokens and the next mk_decode_step must pass positions[b] =
 * n_tokens. Runs ceil(n_tokens / max_rows) launches of the decode kernel with all rows accepted and
 * no LM head. Asynchronous on `stream`; `tokens` must stay valid until the work completes.
 * Errors: MK_ERR_INVALID_ARG (batch outside 1..min(max_batch, 64), n_tokens outside 1..max_ctx).
 * Passage: the pages define no prefill call; their benchmark decodes after a context of about a thousand
 * positions (Kimi K3's TPU megakernel, "Acceptance length and batch size"), and this call builds such a
 * context's caches and states. */
mk_status mk_prefill_kv(mk_handle* h, const int32_t* tokens, int batch, int n_tokens, void* stream);

/* One decode (rows = 1) or speculative-verify (rows = 2..max_rows) step for `batch` sequences.
 *   tokens     device int32 [batch * rows]: row r of sequence b at index b*rows + r
 *   positions  device int32 [batch]: position of row 0 of each sequence. Sequence b has c_b committed
 *              tokens and u_b pending rows from its previous call (u_b = 0 after a prefill). The call
 *              commits the first positions[b] - c_b pending rows and drops the rest, so
 *              c_b <= positions[b] <= c_b + u_b is required (verify: positions advance by the accepted
 *              length). Row r sits at position positions[b] + r and attends causally to positions
 *              0 .. positions[b] + r; recurrent layers advance their state row by row.
 *              After the call c_b = positions[b] and u_b = rows.
 *   logits_out device fp32 [batch * rows, vocab] or NULL (no logits written)
 *   argmax_out device int32 [batch * rows] or NULL: greedy token per row (lowest index on ties)
 * The verify semantics follow the pages' speculative step: an anchor plus seven drafts are checked
 * as eight rows of one sequence and only the accepted prefix is kept (Kimi K3's TPU megakernel,
 * "What DSpark changes per step").
 * One kernel launch. Asynchronous, except that the first call with a given (batch, rows) shape (and the
 * first prefill with a given batch) compiles that shape's program and uploads it with synchronous
 * cudaMalloc / cudaMemcpy; later calls reuse it. Host errors: MK_ERR_INVALID_ARG (batch outside 1..max_batch,
 * rows outside 1..max_rows, both outputs NULL). Device errors via mk_get_status: MK_ERR_DEVICE
 * (token outside [0, vocab), position outside the window, positions[b] + rows > max_ctx; the step is
 * then skipped and no state changes), MK_ERR_TIMEOUT. */
mk_status mk_decode_step(mk_handle* h, const int32_t* tokens, const int32_t* positions, int batch,
                         int rows, float* logits_out, int32_t* argmax_out, void* stream);

/* A speculative-verify step (rows = 2..max_rows: row 0 the anchor, rows 1.. the drafts) that also decides,
 * on the device, how much of each block greedy decoding accepts: draft r + 1 is accepted while it equals the
 * greedy token of row r, so sequence b accepts a_b rows (1 <= a_b <= rows) and emits them plus one bonus
 * token, the greedy token of row a_b - 1 (the accepted prefix plus one bonus token of the pages' verify step:
 * Kimi K3's TPU megakernel, "What DSpark changes per step").
 *   accept_out  device int32 [3][batch]: accept_out[b] = a_b, accept_out[batch + b] = the bonus token (the
 *               next anchor), accept_out[2 * batch + b] = positions[b] + a_b (the next call's position, which
 *               commits exactly the accepted rows).
 * So the next call can take its anchor and positions straight from accept_out without a host round trip.
 * The other arguments and the step itself are mk_decode_step's. One launch, asynchronous.
 * Errors: MK_ERR_INVALID_ARG (rows < 2, missing accept_out, as mk_decode_step). */
mk_status mk_verify_step(mk_handle* h, const int32_t* tokens, const int32_t* positions, int batch, int rows,
                         float* logits_out, int32_t* argmax_out, int32_t* accept_out, void* stream);

/* `n_steps` greedy decode steps of `batch` sequences in ONE kernel launch: step s feeds each sequence the
 * greedy token step s - 1 produced, on the device, so the host is involved once per call (the pages run 24
 * steps inside one device call and meet the host once every 24: Kimi K3's TPU megakernel, "What DSpark
 * changes per step"). Equivalent to n_steps calls of mk_decode_step with rows = 1, the first with `tokens`
 * and `positions`, call s with positions + s and the previous call's greedy tokens.
 *   tokens      device int32 [batch]: the first step's token of each sequence
 *   positions   device int32 [batch]: the first step's position (as for mk_decode_step)
 *   tokens_out  device int32 [n_steps][batch]: the greedy token each step produced (required)
 *   logits_out  device fp32 [batch, vocab] or NULL: the last step's logits
 * Positions + n_steps must stay within max_ctx (checked on the device: MK_ERR_DEVICE, nothing runs).
 * Inside the launch the weight ring runs on from one step into the next. Asynchronous, one launch.
 * Errors: MK_ERR_INVALID_ARG (batch, n_steps, missing tokens_out). */
mk_status mk_decode_steps(mk_handle* h, const int32_t* tokens, const int32_t* positions, int batch, int n_steps,
                          int32_t* tokens_out, float* logits_out, void* stream);

/* mk_decode_steps from HOST buffers: copies tokens_host [batch] and positions_host [batch] in, runs the
 * n_steps launch, copies the greedy tokens [n_steps][batch] back to tokens_out_host and waits for `stream`;
 * returns the device status as mk_get_status would. The first call asking for more steps than before grows
 * the handle's token staging with a synchronous cudaMalloc.
 * Passage: as mk_decode_steps. */
mk_status mk_decode_steps_host(mk_handle* h, const int32_t* tokens_host, const int32_t* positions_host, int batch,
                               int n_steps, int32_t* tokens_out_host, void* stream);

/* The same step from HOST buffers: copies tokens_host [batch*rows] and positions_host [batch] to
 * handle-owned device staging, runs the step, copies the greedy tokens back to argmax_host
 * [batch*rows] (and, when logits_host is not NULL, the logits [batch*rows, vocab]), and waits for
 * `stream`. Returns the device status of the step as mk_get_status would.
 * Passage: none; the pages define no API. This is the end-to-end form of mk_decode_step (inputs and the
 * greedy tokens cross the host boundary every step). */
mk_status mk_decode_step_host(mk_handle* h, const int32_t* tokens_host, const int32_t* positions_host,
                              int batch, int rows, float* logits_host, int32_t* argmax_host, void* stream);

/* Waits for `stream`, returns the device status word of the work enqueued so far and clears it.
 * After MK_ERR_TIMEOUT the handle's inter-SM counters are reset so it can be used again (the state
 * of the interrupted step is undefined: run mk_prefill_kv again).
 * Passage: none; the pages define no API and no error reporting for their kernel. */
mk_status mk_get_status(mk_handle* h, void* stream);

/* Sets the time limit, in nanoseconds, of every wait inside the kernel (an inter-SM dependency counter,
 * a ring slot, a copy in flight); the default is 2 s. A wait that runs past it records MK_ERR_TIMEOUT in
 * the status word and raises the abort flag: every CTA gives up at its next wait, lets its copies in flight
 * land, and returns, so the context stays usable; mk_get_status reports the error and resets the handle's
 * counters. Takes effect at the next launch. Below 1 ms the waits also read the clock on every poll
 * instead of every 64th (what a test of the watchdog uses). Errors: MK_ERR_INVALID_ARG (limit 0).
 * Passage: none; the pages' TPU program has no inter-core waits to bound. */
mk_status mk_set_wait_limit(mk_handle* h, uint64_t limit_ns);

/* Makes sequence `dst` a copy of sequence `src` (both in 0..max_batch-1): its KV / latent caches,
 * recurrent states, pending verify rows and committed / pending counts, so that dst continues exactly as
 * src would. For parallel sampling or beam search from one shared prefix (one prefill, then forks), and
 * for setting up a batch of long contexts quickly. Device-to-device copies of whole per-sequence blocks,
 * asynchronous on `stream`; must not overlap a step that uses either sequence. src == dst does nothing.
 * The pages have no counterpart for this call. Errors: MK_ERR_INVALID_ARG, MK_ERR_CUDA. */
mk_status mk_fork_sequence(mk_handle* h, int src, int dst, void* stream);

/* ---- Program inspection (host only, no GPU needed) -------------------------------------------------
 * Compiles the program of one step shape exactly as mk_decode_step would for a device with `n_sm` SMs,
 * without touching any device, and describes it: one mk_plan_op per op (in program order) and one
 * mk_plan_instr per instruction (grouped by SM, each SM's instructions in the order it runs them). The
 * weight pointers are checked for presence and 16-byte alignment but never dereferenced. For tests and
 * tools that check the scheduler (row coverage, chunking, staging decisions) on a machine without a GPU.
 * The pages have no counterpart. Fills *n_ops / *n_instr with the true counts; writes at most ops_cap /
 * instr_cap records. Errors: MK_ERR_INVALID_ARG, MK_ERR_UNSUPPORTED (as mk_create / mk_decode_step). */
typedef struct mk_plan_op {
  int32_t type;        /* op kind (embed 0, gemv 1, rope/append 2, attention 3, delta rule 4, MLA prep 5,
                          MLA attention 6, route 7, expert up 8, expert down 9, final 10, attention combine
                          11, MLA absorbed query 12, MLA W_UV 13) */
  int32_t n_instr;     /* instructions of the op                                                     */
  int32_t layer;       /* model layer, -1 for embed / LM head / final                                 */
  int32_t rows;        /* GEMV: logical output rows                                                   */
  int32_t K, k_begin, ldw;  /* GEMV: inputs of this op, first input column, full input width         */
  int32_t mma, staged, kc, rg, passes;  /* GEMV / expert path: tensor cores, staged inputs, inputs per
                          chunk, weight rows per group, activation passes                              */
  int32_t out_kind;    /* GEMV epilogue: store 0, residual 1, SwiGLU 2, logits 3                        */
  int32_t nchunk, groups, head_dim, n_heads, n_kv_heads, col_group;  /* attention / delta / MLA       */
  int32_t ncols;       /* GEMV, tcgen05: activation columns per tile (hi / lo pairs, 2 N rounded up to 16);
                          a K-stacked block (P <= 64 rows, ncols 16) takes min(4, 128 / P) x ncols TMEM columns */
  int32_t pa0, patoms; /* GEMV: first packed atom (64 inputs) this op reads, atoms per packed row       */
  int64_t pk_offset;   /* GEMV: byte offset of the op's weight group in the packed copy                */
} mk_plan_op;

typedef struct mk_plan_instr {
  int32_t op, sm, a, b, c;  /* op index, SM, and the op-specific operands (GEMV: rows [a, b))          */
} mk_plan_instr;

mk_status mk_plan(const mk_model_desc* desc, const mk_weights* weights, int n_sm, int batch, int rows,
                  int with_head, mk_plan_op* ops, int ops_cap, int* n_ops, mk_plan_instr* instrs,
                  int instr_cap, int* n_instr);

/* Routing log of MoE models (for checking and analysis; the decode path does not need it). With a
 * non-NULL `device_log` — device int32 [n_layers][max_batch][max_ctx][top_k], owned by the caller and kept
 * alive while set — every later step and prefill writes, for each MoE layer l and each row r of sequence b
 * at position t = positions[b] + r, the ids of the experts that row selected, in pick order, to
 * device_log[((l * max_batch + b) * max_ctx + t) * top_k + k]. Entries of dense layers and of positions
 * no call has reached are left as they were. NULL turns the log off (the default). Takes effect at the
 * next launch. Errors: MK_ERR_INVALID_ARG (no MoE layer in the model, misaligned pointer). */
mk_status mk_set_routing_log(mk_handle* h, int32_t* device_log);

/* Routing replay for MoE models: with a non-NULL `device_ids` — device int32, the routing log's layout
 * [n_layers][max_batch][max_ctx][top_k], owned by the caller and kept alive while set — every later step and
 * prefill makes the row of sequence b at position t of MoE layer l use the experts
 * device_ids[((l * max_batch + b) * max_ctx + t) * top_k + k], k = 0 .. top_k - 1, instead of the ones its
 * router picks, whenever the first of them is >= 0 (an id outside [0, n_experts) falls back to the row's own
 * pick). The weights stay route_scale * s / sum(s) over the sigmoid scores of the experts used. The routing
 * log (mk_set_routing_log) still records each row's own picks. For reproducing another run's routing
 * exactly (comparing two implementations expert for expert, or keeping a rollout and its replay on the same
 * experts); the decode path does not need it. NULL turns it off (the default). Takes effect at the next
 * launch. Errors: MK_ERR_INVALID_ARG (no MoE layer, misaligned pointer).
 * Passage: none; the pages' router always uses its own picks. */
mk_status mk_set_routing_override(mk_handle* h, const int32_t* device_ids);

/* Human-readable description of the last error on this handle ("" if none). Owned by the handle.
 * Passage: none; the pages define no API. */
const char* mk_last_error(const mk_handle* h);

/* Fills `out`. Passage: none; the pages define no API. */
mk_status mk_get_info(const mk_handle* h, mk_info* out);

/* Synchronises the device, frees everything the handle owns. NULL is ignored.
 * Passage: none; the pages define no API. */
void mk_destroy(mk_handle* h);

/* ---- Packed projection weights -------------------------------------------------------------------
 * Every GEMV of the step (projections, output projections, dense FFN, router, LM head) reads its
 * matrices from a tiled copy laid out for the weight ring: each SM's share of the rows (whole 8-row
 * units) is cut into row blocks of at most 128 rows (SwiGLU: 64 gate rows and their 64 up rows), and a
 * block stores 64 inputs of all its rows at a time, each 128-byte row piece swizzled in 16-byte units,
 * so that one contiguous copy fills a ring slot with exactly what the tensor cores read. The layout
 * depends on the model and on the device's SM count only.
 *
 * mk_packed_weight_bytes: size of that copy for `desc` / `weights` on `device`. mk_pack_weights fills
 * `packed` (device memory of that size, 1024-byte aligned, owned by the caller) from the caller's
 * matrices on `stream` (asynchronous; allocates nothing); pass it as weights->packed to mk_create (no
 * second copy is made) or to mk_decode_step_static (which needs it). Errors: MK_ERR_INVALID_ARG
 * (as mk_create, or a misaligned `packed`), MK_ERR_CUDA.
 * Passage: none; the pages read each weight from HBM in its own layout, and this is this library's
 * layout of the same values. */
mk_status mk_packed_weight_bytes(const mk_model_desc* desc, const mk_weights* weights, int device, uint64_t* bytes);
mk_status mk_pack_weights(const mk_model_desc* desc, const mk_weights* weights, int device, void* packed,
                          void* stream);

/* ---- A decode step that allocates no device memory ---------------------------------------------
 * The source pages have no counterpart for this call; it is a convenience of this library.
 * Some callers cannot call cudaMalloc at decode time: a serving process that hands all free HBM to its
 * own pool up front (so a later cudaMalloc fails or breaks the pool's accounting), a plug-in that runs
 * inside a host framework which owns device memory, or a latency-critical loop that cannot afford
 * cudaMalloc's implicit device synchronisation. mk_decode_step_static runs the same kernel as
 * mk_decode_step without a handle: the caller passes the model, the weights (with weights->packed
 * filled by mk_pack_weights), its own persistent buffers
 * (below) and the step's inputs and outputs, and the step's working memory (activations, partial
 * results, inter-SM counters, the instruction queues, the RoPE table) lives in one statically sized
 * device array inside libmk, MK_STATIC_SCRATCH_BYTES long, which every GPU that loads the library keeps
 * until the process exits.
 *
 * Persistent buffers, device memory owned by the caller, zero-filled before the first call for a set of
 * sequences (their sizes use the fields of `desc`; n_gqa / n_lin = number of GQA / GDN+KDA layers):
 *   kcache, vcache  bf16 [n_gqa][max_batch][n_kv_heads][max_ctx][head_dim]      (NULL when n_gqa = 0)
 *   state           fp32 [n_lin][max_batch][lin_heads][lin_dv][lin_dk]           (NULL when n_lin = 0)
 *   pending         fp32 [n_lin][2][max_batch][max_rows][lin_heads][rec], rec = 2*lin_dk + lin_dv + 1
 *                   rounded up to a multiple of 4                                (NULL when n_lin = 0)
 *   seq             int32 [max_batch][4]
 *   epoch           host-side call counter: 0 before the first call; each call advances it
 * The step semantics (positions, committed and pending rows, outputs) are those of mk_decode_step.
 *
 * Behaviour: the first call on a device resolves the device address of the static array (with that
 * device current), so make that first call before any stream capture begins. Every call shares the one
 * array and it keeps the last call's contents; the call clears what must start at zero. Calls whose GPU
 * work overlaps (two host threads, or two streams that are not ordered) race on the array and give
 * wrong results. The call waits for `stream` and returns the device status of the step (as
 * mk_get_status would). Errors: MK_ERR_INVALID_ARG (as mk_create / mk_decode_step, or a missing
 * persistent buffer or weights->packed), MK_ERR_UNSUPPORTED when the step needs more working memory than
 * MK_STATIC_SCRATCH_BYTES (a message on stderr gives both sizes), MK_ERR_CUDA, MK_ERR_DEVICE,
 * MK_ERR_TIMEOUT. MLA and MoE models are refused with MK_ERR_UNSUPPORTED: their latent cache and routing
 * buffers are not among the persistent buffers below. */
#define MK_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)

typedef struct mk_state_buffers {
  void* kcache;
  void* vcache;
  float* state;
  float* pending;
  int32_t* seq;
  uint32_t epoch;
} mk_state_buffers;

mk_status mk_decode_step_static(const mk_model_desc* desc, const mk_weights* weights, mk_state_buffers* state,
                                const int32_t* tokens, const int32_t* positions, int batch, int rows,
                                float* logits_out, int32_t* argmax_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MK_H_ */
