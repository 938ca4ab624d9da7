// Internal layout shared by the host scheduler (mk_host.cu) and the persistent kernel (mk_kernel.cuh).
//
// A decode step is compiled into a PROGRAM: a list of ops in topological order (embedding, then per
// layer: projection GEMV, attention / delta-rule op, output GEMV, FFN GEMVs, then LM head and a final
// op). Each op is split into work items ("instructions") placed on SMs; every SM runs its own queue of
// instructions in op order. An op's instructions wait until the ops it depends on have counted all their
// instructions done (per-op counters in global memory, release/acquire at GPU scope). A producer warp
// per SM walks the same queue ahead of the consumers and streams each instruction's weights (and KV
// prefix) into a shared-memory ring with bulk async copies, so weight traffic for op k+1 and later is
// already in flight while op k computes or waits for its dependencies.
#pragma once
#include <stdint.h>

namespace mk {

constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 32;  // + one producer warp
#ifndef MK_RING_SLOTS
#define MK_RING_SLOTS 4
#endif
constexpr int kSlots = MK_RING_SLOTS;
// shared-memory activation / staging area: 80.25 KB, what is left of the 227 KB a CTA may use after the
// ring and the consumers' bookkeeping; it holds 4 activation rows of width 5120 as bf16 hi/lo pairs with
// their 16-byte row padding (4 x 5128 x 4 bytes), so batch 4 of a d = 5120 model takes the tensor cores
constexpr int kActBytes = 82176;
constexpr int kSlotBytes = 33 * 1024;   // ring slot allocation (payload <= kChunkBytes + row padding)
constexpr int kChunkBytes = 32768;      // weight bytes per chunk
constexpr int kMaxN = 64;        // rows per call (batch * rows)
constexpr int kMaxSeqs = 256;    // sequences a handle can hold
constexpr int kMaxRows = 8;      // query rows per sequence
constexpr int kMaxOpMats = 6;
constexpr int kMaxDeps = 2;
constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 16;

enum OpType : int32_t {
  OP_EMBED = 0,       // x = E[token] (fp32), RMS partials of x
  OP_GEMV = 1,        // y = act(in) W^T, one instruction per SM over a range of output rows
  OP_ROPE_APPEND = 2, // rotate q / k, append bf16 k, v to the KV cache
  OP_ATTN = 3,        // GQA attention over one context chunk of one (sequence, kv head)
  OP_DELTA = 4,       // gated delta rule (GDN / KDA) over a group of value columns of one head
  OP_MLA_PREP = 5,    // MLA: norm + rope of the new latents, append to the latent cache, q rope
  OP_MLA_ATTN = 6,    // MLA absorbed attention over one context chunk of one (sequence, head group)
  OP_ROUTE = 7,       // MoE: sigmoid scores, biased top-k, renormalised weights, expert row lists
  OP_MOE_UP = 8,      // MoE: gate/up GEMV of shared + routed experts, SwiGLU
  OP_MOE_DOWN = 9,    // MoE: down GEMV of shared + routed experts, weighted sum, residual add
  OP_FINAL = 10,      // greedy argmax, sequence bookkeeping, counter reset
  OP_ATTN_COMBINE = 11,  // GQA / MLA: merge the context-chunk partials of one (sequence, row, head)
  OP_MLA_QABS = 12,   // MLA: absorbed query q~_h = W_UK[h] q_nope_h, rotated q_rope (scaled for the softmax)
  OP_MLA_UV = 13,     // MLA: o_h = W_UV[h] o_lat_h
};

enum InKind : int32_t { IN_NORM = 0, IN_BUF = 1 };
enum OutKind : int32_t { OUT_STORE = 0, OUT_RESID = 1, OUT_SWIGLU = 2, OUT_LOGITS = 3 };

struct OpDesc {
  int32_t type;
  int32_t n_instr;          // instructions of this op in one step (its counter's target)
  int32_t n_deps;
  int32_t deps[kMaxDeps];
  int32_t layer;            // model layer (or -1)
  int32_t slot;             // index of the layer among layers of its kind (cache / state slot)
  // ---- GEMV ----
  int32_t K;                // input features
  int32_t rows;             // output rows (logical rows for SwiGLU)
  int32_t rg;               // MoE: physical weight rows per row group (16 or 8)
  int32_t ldw;              // the full input width of the weights (RMSNorm divides by it)
  int32_t k_begin;          // first input column of this op (an op may cover a K range of the matrix)
  int32_t staged;           // MoE: 1 = input rows staged in shared memory (fp32) for the whole instruction
  int32_t mma;              // GEMV tensor-core path: 1 = mma.sync (up to 4 rows; inputs staged whole as bf16
                            // hi/lo pairs), 2 = tcgen05 with TMEM accumulators (inputs staged per K part)
  int32_t ncols;            // mma 2: TMEM columns per accumulator tile = bf16 hi / lo columns, 2 N rounded up to 16
  int32_t kc;               // MoE: inputs per weight slice (chunk width)
  int32_t passes;           // MoE: ceil(N / 8) when 8 activation rows are processed per pass, else 1
  // packed GEMV weights: the group's tiled copy, its atoms per row, and the first atom this op reads
  const uint8_t* wp;
  int32_t patoms;
  int32_t pa0;
  int32_t n_mat;
  int32_t mat_rows[kMaxOpMats];
  const uint16_t* w[kMaxOpMats];
  int32_t in_kind;
  int32_t in_stride;        // floats between activation rows (IN_BUF)
  const float* in;
  const uint16_t* gain;     // bf16 RMSNorm gain (IN_NORM)
  int32_t ssq_in;           // RMS-partial slot read (IN_NORM)
  int32_t out_kind;
  int32_t out_stride;       // floats between output rows
  float* out;
  int32_t ssq_out;          // RMS-partial slot written (OUT_RESID, EMBED); -1 = none
  // ---- attention ----
  int32_t nchunk;           // context chunks per (sequence, kv head)
  int32_t groups;           // q heads per kv head (GQA) or heads per item (MLA)
  int32_t head_dim;
  int32_t n_heads;          // q heads (GQA) / heads (delta, MLA)
  int32_t n_kv_heads;
  // ---- delta rule ----
  int32_t dk, dv;
  int32_t per_channel_decay; // KDA
  int32_t col_group;         // value columns per instruction
  // ---- MoE (OP_ROUTE, OP_MOE_UP, OP_MOE_DOWN) ----
  int32_t n_experts, n_shared, top_k, fp4;
  int32_t route_op;          // index of the op whose routing the expert ops read
  int32_t F;                 // expert hidden size
  float route_scale;
  const float* router_bias;  // [E] or NULL
  const void* ew[2];         // routed experts: gate, up (MOE_UP) or down (MOE_DOWN); bf16 or e2m1 codes
  const void* sw[2];         // shared experts, same layout
  const uint8_t* esc[2];     // e4m3 block scales (NVFP4)
  const uint8_t* ssc[2];
  const float* egs[2];       // fp32 per-expert tensor scales (NVFP4)
  const float* sgs[2];
  // ---- MLA ----
  int32_t q_lora, kv_lora, nope, rope, v_head;
  const uint16_t* w_uk;      // [H, kv_lora, nope]
  const uint16_t* w_uv;      // [H, v_head, kv_lora]
  const uint16_t* q_norm;
  const uint16_t* kv_norm;
  float* aux;                // op-specific second output (MLA: the normalised c_q)
  int32_t aux_stride;
};

// ---- packed GEMV weights -----------------------------------------------------------------------------
// The matrices one GEMV op reads (stacked by rows: q, k, v of a projection; or the gate and up matrices of
// a SwiGLU, paired row by row) are kept in a tiled copy made for the weight ring. Rows are shared out to the
// SMs in whole 8-row units; each SM's share is cut into row blocks of at most 128 logical rows, rounded up to
// whole 8-row runs (SwiGLU: the block's gate rows then its up rows, up to 256 physical rows). A block stores its rows
// atom by atom (64 inputs = 128 bytes of each row, inputs padded with zeros to whole atoms); inside an atom
// row r's eight 16-byte pieces sit at positions (piece ^ (r & 7)). That is the K-major, 128-byte-swizzle
// layout a tcgen05 descriptor reads (8-row groups 1024 bytes apart) and one ldmatrix reads without bank
// conflicts; a ring chunk, one block over a run of atoms, is one contiguous copy. Every logical row before
// a block's first row takes atoms x 128 bytes (x 2 for SwiGLU), so a block starting at logical row r
// starts r x atoms x 128 (x 2) bytes into the copy.
constexpr int kPackAtom = 64;       // inputs per atom
constexpr int kPackBlockRows = 128; // logical rows per block at most
#if defined(__CUDACC__)
#define MK_HD __host__ __device__ __forceinline__
#else
#define MK_HD inline
#endif
MK_HD int pk_atoms(int K) { return (K + kPackAtom - 1) / kPackAtom; }
// first logical row of SM s's share (s = n_sm gives the end)
MK_HD int pk_split(int rows, int n_sm, int s) {
  const long long units = (rows + 7) / 8;
  const int r = 8 * (int)(units * s / n_sm);
  return r < rows ? r : rows;
}
// the SM whose share holds logical row r
MK_HD int pk_sm_of(int rows, int n_sm, int r) {
  const long long units = (rows + 7) / 8;
  return (int)(((long long)n_sm * (r / 8 + 1) - 1) / units);
}
MK_HD int pk_block_lrows(int) { return kPackBlockRows; }
// bytes of the packed copy of a group of `rows` logical rows over K inputs
MK_HD long long pk_bytes(int rows, int K, int swiglu) {
  return (long long)((rows + 7) & ~7) * pk_atoms(K) * 128 * (swiglu ? 2 : 1);
}

// the caller's matrices of one GEMV weight group, as the packing kernel reads them (row-major bf16, K inputs
// per row)
struct PackSrc {
  const uint16_t* w[kMaxOpMats];
  int32_t mat_rows[kMaxOpMats];
  int32_t n_mat;
  int32_t rows;    // logical rows (SwiGLU: rows of each of the two matrices)
  int32_t K;
  int32_t swiglu;  // 1: w[0] gate and w[1] up, paired row by row
  int32_t n_sm;
};

// tcgen05 GEMV geometry: accumulator tiles are 128 TMEM lanes (weight rows) x ncols columns; a packed row
// block is one tile (two for SwiGLU: gate and up); K is covered in K parts of 256 / ncols atoms (the staged
// activations of one part fill one 32 KB buffer).
constexpr int kTcCols = 512;      // TMEM columns allocated per CTA
constexpr int kTcBBytes = 32768;  // one staged-activation buffer (two are used)

struct Instr {
  int32_t op;
  int32_t a, b, c;
};

struct SeqState {
  int32_t c_int;   // tokens absorbed into the recurrent state in HBM
  int32_t u_int;   // pending rows of the previous call (stored for replay)
  int32_t c_spec;  // lowest position the next call may pass (the committed prefix)
  int32_t pad;
};

struct KParams {
  const OpDesc* ops;
  const Instr* instrs;
  const int32_t* qoff;      // [n_sm + 1] per-SM queue offsets into instrs
  uint32_t* counters;       // [n_ops] completed instructions per op in this launch
  int32_t* status;
  int32_t* abort_flag;
  unsigned long long timeout_ns;  // limit of every inter-SM / ring wait
  int32_t use_tc;           // the program has tcgen05 ops: allocate TMEM
  uint32_t spin_mask;             // polls between clock reads, minus one (63, or 0 for limits below 1 ms)
  int32_t n_ops;
  int32_t n_sm;
  // step inputs
  const int32_t* tokens;
  int32_t tok_stride;       // tokens of sequence b start at b * tok_stride
  const int32_t* positions;
  int32_t B, R, N;
  uint32_t epoch;
  int32_t commit_all;       // prefill: the rows of this call count as committed for c_spec
  int32_t n_steps;          // greedy decode steps in this launch (R = 1 when above 1)
  float* logits;            // [N, V] (a multi-step launch leaves the last step's)
  int32_t* argmax;          // [n_steps][N] greedy tokens; step s > 0 embeds the tokens of step s - 1
  int32_t* accept_out;      // verify: [3][B] accepted length, bonus token, next position (or NULL)
  // model
  int32_t d, V, max_ctx, max_batch, max_rows;
  float eps;
  const uint16_t* embed;
  // activations
  float* x;                 // [N, d] residual stream
  float* ssq;               // [slots][kMaxN][n_sm] RMS partials (sum of squares per row and SM)
  float2* amax_part;        // [n_sm][kMaxN] (value, index) LM-head argmax partials
  float* attn_part;         // attention chunk partials
  int32_t attn_part_stride; // floats per partial record
  // GQA caches: [slot][max_batch][Hkv][max_ctx][hd] bf16
  uint16_t* kcache;
  uint16_t* vcache;
  // delta rule: state [slot][max_batch][H][dv][dk] fp32; pending [slot][2][max_batch][max_rows][H][rec]
  float* state;
  float* pend;
  int32_t pend_rec;         // floats per pending record (k_hat, v, alpha, beta)
  // MLA: latent cache [slot][max_batch][max_ctx][kv_lora + rope] bf16
  uint16_t* latent;
  // MoE routing of the current layer: [N][top_k] expert ids and weights; the union of the experts the
  // step selected, ascending: union_list[0] = count, union_list[1..] = experts
  int32_t* route_idx;
  float* route_w;
  int32_t* union_list;
  float* hexp;              // [n_shared + union][N][F] expert SwiGLU outputs
  int32_t* route_log;       // optional [n_layers][max_batch][max_ctx][top_k] expert ids by position
  const int32_t* route_force;  // optional, same layout: expert ids a row must use (replay); < 0 = its own
  SeqState* seq;
  const float2* rope;       // [max_ctx][rot_dim / 2] (cos, sin)
  int32_t rot_dim;
  // model dims needed by several ops
  int32_t n_q_heads, n_kv_heads, head_dim;
  int32_t lin_heads, lin_dk, lin_dv;
  // optional %globaltimer trace, kTraceWords per instruction (NULL = off)
  unsigned long long* trace;
};

// trace words per instruction: consumer begin, dependencies met, done; producer first issue
// (tcgen05 GEMV instructions also: first activation part staged, first weight chunk arrived, last MMA issued,
// last activation part staged)
constexpr int kTraceWords = 9;

}  // namespace mk
