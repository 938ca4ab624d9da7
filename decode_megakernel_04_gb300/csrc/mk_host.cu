// Host side of libmk: the C ABI (include/mk.h), the device memory plan of a handle, and the scheduler
// that compiles one decode step of the layer stack into per-SM instruction queues for the persistent
// kernel (mk_kernel.cuh, built as mk_kernel_dense.cu and mk_kernel_full.cu).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <deque>
#include <mutex>
#include <string>
#include <vector>

#include "mk.h"
#include "mk_internal.h"

namespace mk {
// the two builds of the megakernel: without (dense) and with (full) the MLA and MoE ops
namespace dense {
size_t kernel_smem_bytes();
cudaError_t kernel_configure();
cudaError_t kernel_launch(const KParams& p, int n_sm, cudaStream_t stream);
}  // namespace dense
namespace full {
size_t kernel_smem_bytes();
cudaError_t kernel_configure();
cudaError_t kernel_launch(const KParams& p, int n_sm, cudaStream_t stream);
}  // namespace full
cudaError_t rope_table_launch(float2* tab, int max_ctx, int rot_dim, double theta, cudaStream_t stream);
cudaError_t fill_i32_launch(int32_t* dst, int n, int32_t value, cudaStream_t stream);
cudaError_t pack_gemv_launch(uint8_t* dst, const PackSrc& src, cudaStream_t stream);
}  // namespace mk

using namespace mk;

namespace {

size_t kernel_smem_bytes() { return std::max(dense::kernel_smem_bytes(), full::kernel_smem_bytes()); }
cudaError_t kernel_configure(bool full_ops) { return full_ops ? full::kernel_configure() : dense::kernel_configure(); }
cudaError_t kernel_launch(bool full_ops, const KParams& p, int n_sm, cudaStream_t stream) {
  return full_ops ? full::kernel_launch(p, n_sm, stream) : dense::kernel_launch(p, n_sm, stream);
}

struct Program {
  int B = 0, R = 0;
  bool head = false;  // LM head + argmax partials
  OpDesc* d_ops = nullptr;
  Instr* d_instr = nullptr;
  int32_t* d_qoff = nullptr;
  int n_ops = 0;
  int n_instr = 0;
  bool use_tc = false;  // the program has tcgen05 GEMV ops (the kernel allocates TMEM)
};

int round_up(int v, int m) { return (v + m - 1) / m * m; }

// The packed GEMV weights of a model (layout in mk_internal.h): one group per set of matrices a GEMV op
// reads, in the order the step program first meets them, each at a 1024-byte aligned offset of one copy.
// The groups depend on the model and the SM count only, so every step shape finds its groups here.
struct PackTable {
  struct Group {
    PackSrc src;
    size_t offset;
  };
  std::vector<Group> groups;
  size_t total = 0;
  const uint8_t* base = nullptr;  // device address of the copy (never dereferenced on the host)
  int n_sm = 0;

  // device address of the packed group of GEMV `d` (its first matrix, width, rows, SwiGLU pairing), adding
  // the group on first sight
  const uint8_t* find(const OpDesc& d) {
    const int sw = d.out_kind == OUT_SWIGLU ? 1 : 0;
    for (const Group& g : groups)
      if (g.src.w[0] == d.w[0] && g.src.K == d.K && g.src.rows == d.rows && g.src.swiglu == sw) return base + g.offset;
    Group g;
    std::memset(&g, 0, sizeof(g));
    for (int m = 0; m < d.n_mat; ++m) {
      g.src.w[m] = d.w[m];
      g.src.mat_rows[m] = d.mat_rows[m];
    }
    g.src.n_mat = d.n_mat;
    g.src.rows = d.rows;
    g.src.K = d.K;
    g.src.swiglu = sw;
    g.src.n_sm = n_sm;
    g.offset = total;
    total += (size_t)((pk_bytes(d.rows, d.K, sw) + 1023) / 1024 * 1024);
    groups.push_back(g);
    return base + g.offset;
  }
};

}  // namespace

struct mk_handle {
  mk_model_desc desc{};
  mk_weights w{};
  int device = 0;
  int n_sm = 0;
  std::string err;
  std::vector<void*> allocs;
  int64_t bytes = 0;
  uint32_t epoch = 0;
  unsigned long long wait_limit_ns = 2000000000ull;  // watchdog limit of every device-side wait

  // per-layer slot among layers of the same kind
  std::vector<int> slot;
  int n_gqa = 0, n_delta = 0, n_mla = 0;
  bool full_ops = false;  // the model has MLA or MoE layers: launch the full build of the kernel

  int nmax = 0;
  int proj_stride = 0, attn_stride = 0, hbuf_stride = 0;
  float* x = nullptr;
  float* proj = nullptr;
  float* attn_out = nullptr;
  float* hbuf = nullptr;
  float* ssq = nullptr;
  float2* amax_part = nullptr;
  float* attn_part = nullptr;
  int attn_part_stride = 0;
  uint16_t* kcache = nullptr;
  uint16_t* vcache = nullptr;
  float* state = nullptr;
  float* pend = nullptr;
  int pend_rec = 0;
  // MLA: latent cache and the per-step query / latent-output buffers
  uint16_t* latent = nullptr;
  float* mla_cq = nullptr;    // [N][q_lora] normalised c_q
  float* mla_qf = nullptr;    // [N][H * (nope + rope)] projected queries
  float* mla_qt = nullptr;    // [N][H * (kv_lora + rope)] absorbed, rotated, scaled queries
  float* mla_olat = nullptr;  // [N][H * kv_lora] attention output in latent space
  int mla_qf_stride = 0, mla_qt_stride = 0, mla_olat_stride = 0;
  // MoE routing of the current layer and the expert SwiGLU outputs
  int32_t* route_idx = nullptr;
  float* route_w = nullptr;
  int32_t* union_list = nullptr;
  float* hexp = nullptr;
  size_t hexp_floats = 0;
  int32_t* route_log = nullptr;  // caller's device buffer (mk_set_routing_log) or NULL
  const int32_t* route_force = nullptr;  // caller's device buffer (mk_set_routing_override) or NULL
  uint32_t* counters = nullptr;
  int32_t* status = nullptr;
  int32_t* abort_flag = nullptr;
  SeqState* seq = nullptr;
  float2* rope = nullptr;
  int rot_dim = 0;
  int32_t* pos_buf = nullptr;
  int32_t* stage_tok = nullptr;
  int32_t* stage_pos = nullptr;
  int32_t* stage_argmax = nullptr;
  float* stage_logits = nullptr;
  int32_t* stage_steps = nullptr;  // mk_decode_steps_host: the greedy tokens of every step
  size_t steps_cap = 0;
  int max_ops = 0;
  int n_ops_last = 0;
  std::deque<Program> programs;  // stable addresses: launches and the trace keep pointers into it
  PackTable pk;                  // packed GEMV weights: the groups and the copy's address
  void* packed_own = nullptr;    // the copy when this handle made it (NULL: the caller's mk_weights.packed)
  // optional per-instruction timestamp trace of the last step (env MK_TRACE=<file>), written at destroy
  std::string trace_path;
  unsigned long long* trace = nullptr;
  size_t trace_cap = 0;  // instructions
  const Program* last_prog = nullptr;
};

namespace {

mk_status fail(mk_handle* h, mk_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  if (h) h->err = buf;
  return s;
}

mk_status cuda_fail(mk_handle* h, cudaError_t e, const char* what) {
  return fail(h, e == cudaErrorMemoryAllocation ? MK_ERR_NOMEM : MK_ERR_CUDA, "%s: %s", what,
              cudaGetErrorString(e));
}

template <typename T>
mk_status dev_alloc(mk_handle* h, T** out, size_t count, const char* what) {
  void* p = nullptr;
  const size_t bytes = std::max<size_t>(count * sizeof(T), 16);
  cudaError_t e = cudaMalloc(&p, bytes);
  if (e != cudaSuccess) return cuda_fail(h, e, what);
  e = cudaMemset(p, 0, bytes);
  if (e != cudaSuccess) return cuda_fail(h, e, what);
  h->allocs.push_back(p);
  h->bytes += (int64_t)bytes;
  *out = reinterpret_cast<T*>(p);
  return MK_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool is_delta(int m) { return m == MK_MIXER_GDN || m == MK_MIXER_KDA; }

int delta_proj_cols(const mk_model_desc& d, int mixer) {
  const int H = d.lin_heads;
  return 2 * H * d.lin_dk + H * d.lin_dv + (mixer == MK_MIXER_KDA ? H * d.lin_dk : H) + H;
}

mk_status check_desc(mk_handle* h, const mk_model_desc& d, const mk_weights& w) {
  if (d.n_layers < 1 || d.n_layers > MK_MAX_LAYERS) return fail(h, MK_ERR_INVALID_ARG, "n_layers %d", d.n_layers);
  if (d.d_model < 8 || d.d_model % 8) return fail(h, MK_ERR_INVALID_ARG, "d_model %d must be a multiple of 8", d.d_model);
  if (d.vocab < 1) return fail(h, MK_ERR_INVALID_ARG, "vocab %d", d.vocab);
  // a handle may hold up to kMaxSeqs sequences (caches and states); one call processes at most kMaxN rows
  if (d.max_batch < 1 || d.max_rows < 1 || d.max_rows > kMaxRows || d.max_batch > kMaxSeqs)
    return fail(h, MK_ERR_UNSUPPORTED, "max_batch must be <= %d and max_rows <= %d", kMaxSeqs, kMaxRows);
  if (d.max_ctx < d.max_rows) return fail(h, MK_ERR_INVALID_ARG, "max_ctx %d", d.max_ctx);
  if (!w.embed || !w.final_norm || (!d.tied_embedding && !w.lm_head))
    return fail(h, MK_ERR_INVALID_ARG, "embed / final_norm / lm_head missing");
  if (!aligned16(w.embed) || !aligned16(w.final_norm) || (w.lm_head && !aligned16(w.lm_head)))
    return fail(h, MK_ERR_INVALID_ARG, "weights must be 16-byte aligned");
  for (int i = 0; i < d.n_layers; ++i) {
    const mk_layer_weights& L = w.layers[i];
    const int m = d.mixer[i];
    auto need = [&](const void* p, const char* name) -> mk_status {
      if (!p) return fail(h, MK_ERR_INVALID_ARG, "layer %d: %s missing", i, name);
      if (!aligned16(p)) return fail(h, MK_ERR_INVALID_ARG, "layer %d: %s not 16-byte aligned", i, name);
      return MK_OK;
    };
    mk_status s;
#define NEED(p) if ((s = need(L.p, #p)) != MK_OK) return s
    NEED(attn_norm);
    NEED(ffn_norm);
    if (m == MK_MIXER_GQA) {
      NEED(wq); NEED(wk); NEED(wv); NEED(wo);
      if (d.n_kv_heads < 1 || d.n_q_heads % d.n_kv_heads)
        return fail(h, MK_ERR_INVALID_ARG, "n_q_heads must be a multiple of n_kv_heads");
      if (d.head_dim != 64 && d.head_dim != 128 && d.head_dim != 256)
        return fail(h, MK_ERR_UNSUPPORTED, "head_dim %d (64, 128 or 256)", d.head_dim);
      if (d.n_q_heads / d.n_kv_heads > 8) return fail(h, MK_ERR_UNSUPPORTED, "more than 8 q heads per kv head");
    } else if (is_delta(m)) {
      NEED(wq); NEED(wk); NEED(wv); NEED(wo); NEED(wa); NEED(wb);
      if (d.lin_dk != 32 && d.lin_dk != 64 && d.lin_dk != 128)
        return fail(h, MK_ERR_UNSUPPORTED, "lin_dk %d (32, 64 or 128)", d.lin_dk);
      if (d.lin_dv % 8) return fail(h, MK_ERR_UNSUPPORTED, "lin_dv %d must be a multiple of 8", d.lin_dv);
    } else if (m == MK_MIXER_MLA) {
      NEED(w_dq); NEED(q_norm); NEED(w_uq); NEED(w_dkv); NEED(kv_norm); NEED(w_uk); NEED(w_uv); NEED(wo);
      // the latent attention op gives each lane 16 latent dims and 2 rope dims of a 512 + 64 latent, each
      // warp one head of an 8-head group; the absorbed-query op gives each lane nope / 32 query dims
      if (d.kv_lora != 512 || d.qk_rope != 64)
        return fail(h, MK_ERR_UNSUPPORTED, "MLA latent %d + rope %d (512 + 64)", d.kv_lora, d.qk_rope);
      if (d.qk_nope < 32 || d.qk_nope > 128 || d.qk_nope % 32)
        return fail(h, MK_ERR_UNSUPPORTED, "qk_nope %d (32, 64, 96 or 128)", d.qk_nope);
      if (d.mla_heads < 8 || d.mla_heads % 8) return fail(h, MK_ERR_UNSUPPORTED, "mla_heads %d (multiple of 8)", d.mla_heads);
      if (d.v_head < 16 || d.v_head % 16) return fail(h, MK_ERR_UNSUPPORTED, "v_head %d (multiple of 16)", d.v_head);
      if (d.q_lora < 16 || d.q_lora % 16) return fail(h, MK_ERR_UNSUPPORTED, "q_lora %d (multiple of 16)", d.q_lora);
    } else {
      return fail(h, MK_ERR_INVALID_ARG, "layer %d: mixer %d", i, m);
    }
    if (d.ffn_kind == MK_FFN_DENSE) {
      NEED(w_gate); NEED(w_up); NEED(w_down);
      if (d.ffn_dim < 8 || d.ffn_dim % 8) return fail(h, MK_ERR_INVALID_ARG, "ffn_dim %d", d.ffn_dim);
    } else if (d.ffn_kind == MK_FFN_MOE) {
      NEED(w_router); NEED(e_gate); NEED(e_up); NEED(e_down);
      if (L.router_bias && !aligned16(L.router_bias)) return fail(h, MK_ERR_INVALID_ARG, "layer %d: router_bias alignment", i);
      if (d.n_experts < 1 || d.n_experts > kMaxExperts)
        return fail(h, MK_ERR_UNSUPPORTED, "n_experts %d (1..%d)", d.n_experts, kMaxExperts);
      if (d.top_k < 1 || d.top_k > kMaxTopK || d.top_k > d.n_experts)
        return fail(h, MK_ERR_UNSUPPORTED, "top_k %d (1..min(%d, n_experts))", d.top_k, kMaxTopK);
      if (d.n_shared < 0 || d.n_shared > 8) return fail(h, MK_ERR_UNSUPPORTED, "n_shared %d (0..8)", d.n_shared);
      if (d.n_shared) { NEED(s_gate); NEED(s_up); NEED(s_down); }
      if (d.expert_format == MK_FMT_NVFP4) {
        // NVFP4 rows are copied as 16-byte multiples of codes (2 per byte) and of e4m3 scales (1 per 16)
        if (d.expert_dim < 256 || d.expert_dim % 256 || d.d_model % 256)
          return fail(h, MK_ERR_UNSUPPORTED, "NVFP4 experts need expert_dim and d_model multiples of 256");
        NEED(e_gate_scales); NEED(e_up_scales); NEED(e_down_scales);
        NEED(e_gate_gscale); NEED(e_up_gscale); NEED(e_down_gscale);
        if (d.n_shared) {
          NEED(s_gate_scales); NEED(s_up_scales); NEED(s_down_scales);
          NEED(s_gate_gscale); NEED(s_up_gscale); NEED(s_down_gscale);
        }
      } else if (d.expert_format == MK_FMT_BF16) {
        if (d.expert_dim < 8 || d.expert_dim % 8) return fail(h, MK_ERR_INVALID_ARG, "expert_dim %d", d.expert_dim);
      } else {
        return fail(h, MK_ERR_INVALID_ARG, "expert_format %d", d.expert_format);
      }
    } else {
      return fail(h, MK_ERR_INVALID_ARG, "ffn_kind %d", d.ffn_kind);
    }
#undef NEED
  }
  bool has_gqa = false, has_mla = false;
  for (int i = 0; i < d.n_layers; ++i) {
    has_gqa = has_gqa || d.mixer[i] == MK_MIXER_GQA;
    has_mla = has_mla || d.mixer[i] == MK_MIXER_MLA;
  }
  if (has_gqa && has_mla && d.head_dim != d.qk_rope)
    return fail(h, MK_ERR_UNSUPPORTED, "GQA and MLA layers in one model need head_dim == qk_rope (one RoPE table)");
  return MK_OK;
}

// Layer slots and activation strides of a handle, derived from its model description alone.
void derive_layout(mk_handle* h) {
  const mk_model_desc& D = h->desc;
  h->slot.resize(D.n_layers);
  h->n_gqa = h->n_delta = h->n_mla = 0;
  for (int i = 0; i < D.n_layers; ++i) {
    if (D.mixer[i] == MK_MIXER_GQA) h->slot[i] = h->n_gqa++;
    else if (D.mixer[i] == MK_MIXER_MLA) h->slot[i] = h->n_mla++;
    else h->slot[i] = h->n_delta++;
  }
  h->nmax = std::min(D.max_batch * D.max_rows, kMaxN);  // rows of the largest call
  h->full_ops = h->n_mla > 0 || D.ffn_kind == MK_FFN_MOE;
  int proj = 8, attn = 8;
  for (int i = 0; i < D.n_layers; ++i) {
    const int m = D.mixer[i];
    if (m == MK_MIXER_GQA) {
      proj = std::max(proj, (D.n_q_heads + 2 * D.n_kv_heads) * D.head_dim);
      attn = std::max(attn, D.n_q_heads * D.head_dim);
    } else if (is_delta(m)) {
      proj = std::max(proj, delta_proj_cols(D, m));
      attn = std::max(attn, D.lin_heads * D.lin_dv);
    } else if (m == MK_MIXER_MLA) {
      proj = std::max(proj, D.q_lora + D.kv_lora + D.qk_rope);
      attn = std::max(attn, D.mla_heads * D.v_head);
    }
  }
  h->proj_stride = round_up(proj, 8);
  h->attn_stride = round_up(attn, 8);
  // dense SwiGLU hidden rows, or the MoE router logits
  const int hb = D.ffn_kind == MK_FFN_MOE ? D.n_experts : D.ffn_dim;
  h->hbuf_stride = round_up(std::max(hb, 8), 8);
  h->max_ops = 32 * D.n_layers + 16;
  if (h->n_gqa) {
    h->attn_part_stride = D.head_dim + 4;
    h->rot_dim = D.head_dim;
  }
  if (h->n_mla) {
    h->attn_part_stride = std::max(h->attn_part_stride, D.kv_lora + 4);
    h->rot_dim = D.qk_rope;
    h->mla_qf_stride = D.mla_heads * (D.qk_nope + D.qk_rope);
    h->mla_qt_stride = D.mla_heads * (D.kv_lora + D.qk_rope);
    h->mla_olat_stride = D.mla_heads * D.kv_lora;
  }
  if (h->n_delta) h->pend_rec = round_up(2 * D.lin_dk + D.lin_dv + 1, 4);
  if (D.ffn_kind == MK_FFN_MOE) {
    // the shared experts plus the union of the experts the rows of one step select
    const int64_t uni = std::min<int64_t>(D.n_experts, (int64_t)h->nmax * D.top_k);
    h->hexp_floats = (size_t)(D.n_shared + uni) * h->nmax * D.expert_dim;
  }
}

// Attention partial records of one step (GQA and MLA share the buffer): (sequence, kv head or head group,
// context chunk) triples times rows times heads per group. The chunk count of an op is at most n_sm / the
// other factors, so the triples are at most max(n_sm, sequences x groups).
size_t attn_part_records(const mk_handle* h, int B, int R) {
  const mk_model_desc& D = h->desc;
  size_t recs = 0;
  if (h->n_gqa)
    recs = (size_t)std::max(h->n_sm, B * D.n_kv_heads) * R * (D.n_q_heads / D.n_kv_heads);
  if (h->n_mla)
    recs = std::max(recs, (size_t)std::max(h->n_sm, B * (D.mla_heads / 8)) * R * 8);
  return 2 * recs;
}

// ------------------------------------------------------------------------------------------------
// scheduler
// ------------------------------------------------------------------------------------------------
struct Builder {
  int n_sm;
  PackTable* pk;
  std::vector<OpDesc> ops;
  std::vector<std::vector<Instr>> q;
  Builder(int n, PackTable* table) : n_sm(n), pk(table), q(n) {}

  int add(OpDesc d) {
    const int idx = (int)ops.size();
    if (idx > 0 && d.n_deps == 0) {
      d.n_deps = 1;
      d.deps[0] = idx - 1;
    }
    ops.push_back(d);
    return idx;
  }
  void place(int op, int sm, int a, int b, int c) {
    Instr in;
    in.op = op;
    in.a = a;
    in.b = b;
    in.c = c;
    q[sm].push_back(in);
    ops[op].n_instr += 1;
  }
};

OpDesc blank(int type) {
  OpDesc d;
  std::memset(&d, 0, sizeof(d));
  d.type = type;
  d.layer = -1;
  d.passes = 1;
  return d;
}

// A GEMV op reads the packed copy of its weights. Every SM takes a share of whole 8-row units (the packed row
// blocks are cut from the shares). Up to 4 activation rows take the mma.sync path when their bf16 hi / lo
// columns (and, for a residual add, the SM's slice of x) fit the staging area; a residual-add GEMV whose input
// does not fit is split along K into sequential ops over runs of whole atoms that each add their part to x
// (the last one also writes the RMS partials of the new x). Everything else takes the tcgen05 path.
void gemv_op(Builder& bld, OpDesc d, int N) {
  d.type = OP_GEMV;
  d.ldw = d.K;
  d.k_begin = 0;
  d.wp = bld.pk->find(d);
  d.patoms = pk_atoms(d.K);
  d.pa0 = 0;
  const int A = d.patoms;
  auto place_all = [&](int op) {
    for (int s = 0; s < bld.n_sm; ++s)
      bld.place(op, s, pk_split(d.rows, bld.n_sm, s), pk_split(d.rows, bld.n_sm, s + 1), 0);
  };
  // a residual-add instruction also keeps its slice of x (N x its rows) in the staging area
  int64_t xrows = 0;
  if (d.out_kind == OUT_RESID)
    for (int s = 0; s < bld.n_sm; ++s)
      xrows = std::max<int64_t>(xrows, pk_split(d.rows, bld.n_sm, s + 1) - pk_split(d.rows, bld.n_sm, s));
  const int64_t cap = kActBytes / 4 - 8;  // floats
  auto fits_mma = [&](int atoms) { return N <= 4 && (int64_t)N * (atoms * 64 + 8 + xrows) <= cap; };
  int pa = A;  // atoms per K part
  if (!fits_mma(pa) && N <= 4 && d.out_kind == OUT_RESID) {
    int parts = 2;
    while (parts <= 16 && !fits_mma((A + parts - 1) / parts)) ++parts;
    pa = (A + parts - 1) / parts;
  }
  if (!fits_mma(pa)) {
    d.mma = 2;
    d.ncols = round_up(2 * N, 16);
    place_all(bld.add(d));
    return;
  }
  const int parts = (A + pa - 1) / pa;
  const int ssq_out = d.ssq_out;
  for (int part = 0; part < parts; ++part) {
    OpDesc q = d;
    q.mma = 1;
    q.pa0 = part * pa;
    q.k_begin = q.pa0 * kPackAtom;
    q.K = std::min(pa * kPackAtom, d.ldw - q.k_begin);
    q.ssq_out = (part == parts - 1) ? ssq_out : -1;
    place_all(bld.add(q));
  }
}

OpDesc gemv_desc(int K, std::initializer_list<std::pair<const void*, int>> mats) {
  OpDesc d = blank(OP_GEMV);
  d.K = K;
  for (auto& m : mats) {
    d.w[d.n_mat] = reinterpret_cast<const uint16_t*>(m.first);
    d.mat_rows[d.n_mat] = m.second;
    d.rows += m.second;
    d.n_mat++;
  }
  return d;
}

// Multi-head latent attention, absorbed form, of layer i (the ops are described in mk_kernel.cuh):
//   GEMV [w_dq; w_dkv] on RMSNorm(x) -> proj;  MLA_PREP: c_q norm -> mla_cq, latent (norm + rope) -> cache;
//   GEMV w_uq on c_q -> mla_qf;  MLA_QABS -> mla_qt;  MLA_ATTN over context chunks -> partials;
//   ATTN_COMBINE -> mla_olat;  MLA_UV -> attn_out;  GEMV wo, residual add.
void mla_layer(mk_handle* h, Builder& bld, int i, int B, int R) {
  const mk_model_desc& D = h->desc;
  const mk_layer_weights& L = h->w.layers[i];
  const int N = B * R, d = D.d_model;
  const int H = D.mla_heads, nope = D.qk_nope, rp = D.qk_rope, kl = D.kv_lora, ql = D.q_lora;
  constexpr int G = kConsumerWarps;  // heads per attention group (one per warp)
  const int ngr = H / G;

  OpDesc a = gemv_desc(d, {{L.w_dq, ql}, {L.w_dkv, kl + rp}});
  a.layer = i;
  a.in_kind = IN_NORM;
  a.gain = reinterpret_cast<const uint16_t*>(L.attn_norm);
  a.ssq_in = 2 * i;
  a.out_kind = OUT_STORE;
  a.out = h->proj;
  a.out_stride = h->proj_stride;
  gemv_op(bld, a, N);

  OpDesc pr = blank(OP_MLA_PREP);
  pr.layer = i;
  pr.slot = h->slot[i];
  pr.q_lora = ql;
  pr.kv_lora = kl;
  pr.rope = rp;
  pr.q_norm = reinterpret_cast<const uint16_t*>(L.q_norm);
  pr.kv_norm = reinterpret_cast<const uint16_t*>(L.kv_norm);
  pr.in = h->proj;
  pr.in_stride = h->proj_stride;
  pr.aux = h->mla_cq;
  pr.aux_stride = ql;
  const int op_pr = bld.add(pr);
  // one warp per (row, q or kv half); the op indexes its work by SM, so SM s takes items 8s .. 8s + 7
  const int n_pr = std::min(h->n_sm, (2 * N + kConsumerWarps - 1) / kConsumerWarps);
  for (int s = 0; s < n_pr; ++s) bld.place(op_pr, s, 0, 0, 0);

  OpDesc uq = gemv_desc(ql, {{L.w_uq, h->mla_qf_stride}});
  uq.layer = i;
  uq.in_kind = IN_BUF;
  uq.in = h->mla_cq;
  uq.in_stride = ql;
  uq.out_kind = OUT_STORE;
  uq.out = h->mla_qf;
  uq.out_stride = h->mla_qf_stride;
  gemv_op(bld, uq, N);

  OpDesc qa = blank(OP_MLA_QABS);
  qa.layer = i;
  qa.nope = nope;
  qa.rope = rp;
  qa.kv_lora = kl;
  qa.w_uk = reinterpret_cast<const uint16_t*>(L.w_uk);
  qa.in = h->mla_qf;
  qa.in_stride = h->mla_qf_stride;
  qa.out = h->mla_qt;
  qa.out_stride = h->mla_qt_stride;
  const int op_qa = bld.add(qa);
  int k = 0;
  for (int hh = 0; hh < H; ++hh)
    for (int cb = 0; cb < kl / 128; ++cb, ++k) bld.place(op_qa, k % h->n_sm, hh, cb, 0);

  OpDesc at = blank(OP_MLA_ATTN);
  at.layer = i;
  at.slot = h->slot[i];
  at.kv_lora = kl;
  at.rope = rp;
  at.n_heads = H;
  at.n_kv_heads = ngr;
  at.groups = G;
  at.head_dim = kl;
  at.in = h->mla_qt;
  at.in_stride = h->mla_qt_stride;
  const int rows_per = std::min(R, 2);  // (row, head) pairs per warp
  const int nsplit = (R + rows_per - 1) / rows_per;
  at.nchunk = std::max(1, h->n_sm / (B * ngr * nsplit));
  const int op_at = bld.add(at);
  k = 0;
  for (int b = 0; b < B; ++b)
    for (int g = 0; g < ngr; ++g)
      for (int c = 0; c < at.nchunk; ++c)
        for (int sp = 0; sp < nsplit; ++sp, ++k) {
          const int rlo = sp * rows_per, rhi = std::min(R, rlo + rows_per);
          bld.place(op_at, k % h->n_sm, b * ngr + g, c, rlo | (rhi << 8));
        }

  OpDesc cb = at;
  cb.type = OP_ATTN_COMBINE;
  cb.n_instr = 0;
  cb.n_deps = 0;
  cb.out = h->mla_olat;
  cb.out_stride = h->mla_olat_stride;
  const int op_cb = bld.add(cb);
  k = 0;
  for (int b = 0; b < B; ++b)
    for (int r = 0; r < R; ++r)
      for (int hh = 0; hh < H; ++hh, ++k) bld.place(op_cb, k % h->n_sm, b, r, hh);

  OpDesc uv = blank(OP_MLA_UV);
  uv.layer = i;
  uv.kv_lora = kl;
  uv.v_head = D.v_head;
  uv.w_uv = reinterpret_cast<const uint16_t*>(L.w_uv);
  uv.in = h->mla_olat;
  uv.in_stride = h->mla_olat_stride;
  uv.out = h->attn_out;
  uv.out_stride = h->attn_stride;
  const int op_uv = bld.add(uv);
  k = 0;
  for (int hh = 0; hh < H; ++hh)
    for (int jb = 0; jb < (D.v_head + 63) / 64; ++jb, ++k) bld.place(op_uv, k % h->n_sm, hh, jb, 0);

  OpDesc o = gemv_desc(H * D.v_head, {{L.wo, d}});
  o.layer = i;
  o.in_kind = IN_BUF;
  o.in = h->attn_out;
  o.in_stride = h->attn_stride;
  o.out_kind = OUT_RESID;
  o.ssq_out = 2 * i + 1;
  gemv_op(bld, o, N);
}

// MoE feed-forward of layer i: router GEMV on RMSNorm(x) -> hbuf; ROUTE (one instruction); MOE_UP over
// the F hidden rows and MOE_DOWN over the d output rows, each one instruction per SM covering its row
// range of every selected expert, so an SM's work does not depend on which experts the rows picked.
void moe_layer(mk_handle* h, Builder& bld, int i, int N) {
  const mk_model_desc& D = h->desc;
  const mk_layer_weights& L = h->w.layers[i];
  const int d = D.d_model, E = D.n_experts, F = D.expert_dim;
  const bool fp4 = D.expert_format == MK_FMT_NVFP4;

  OpDesc z = gemv_desc(d, {{L.w_router, E}});
  z.layer = i;
  z.in_kind = IN_NORM;
  z.gain = reinterpret_cast<const uint16_t*>(L.ffn_norm);
  z.ssq_in = 2 * i + 1;
  z.out_kind = OUT_STORE;
  z.out = h->hbuf;
  z.out_stride = h->hbuf_stride;
  gemv_op(bld, z, N);

  OpDesc ro = blank(OP_ROUTE);
  ro.layer = i;
  ro.n_experts = E;
  ro.top_k = D.top_k;
  ro.route_scale = D.route_scale;
  ro.router_bias = L.router_bias;
  ro.in = h->hbuf;
  ro.in_stride = h->hbuf_stride;
  const int op_ro = bld.add(ro);
  bld.place(op_ro, 0, 0, 0, 0);

  OpDesc ex = blank(OP_MOE_UP);
  ex.layer = i;
  ex.n_experts = E;
  ex.n_shared = D.n_shared;
  ex.top_k = D.top_k;
  ex.fp4 = fp4 ? 1 : 0;
  ex.route_op = op_ro;
  ex.F = F;
  // the kernel's expert GEMV: 16 weight rows per group and 4 (bf16) or 8 (NVFP4) inputs per thread for up
  // to 4 activation rows; 8 rows, 8 inputs per thread and ceil(N / 8) passes otherwise
  ex.rg = N <= 4 ? 16 : 8;
  ex.kc = (fp4 || N > 4 ? 8 : 4) * kConsumerThreads;
  ex.passes = N <= 8 ? 1 : (N + 7) / 8;

  OpDesc up = ex;
  up.ew[0] = L.e_gate;
  up.ew[1] = L.e_up;
  up.sw[0] = L.s_gate;
  up.sw[1] = L.s_up;
  up.esc[0] = L.e_gate_scales;
  up.esc[1] = L.e_up_scales;
  up.ssc[0] = L.s_gate_scales;
  up.ssc[1] = L.s_up_scales;
  up.egs[0] = L.e_gate_gscale;
  up.egs[1] = L.e_up_gscale;
  up.sgs[0] = L.s_gate_gscale;
  up.sgs[1] = L.s_up_gscale;
  up.gain = reinterpret_cast<const uint16_t*>(L.ffn_norm);
  up.ssq_in = 2 * i + 1;
  // up to 2 rows: the normalised inputs are staged in shared memory once per instruction
  const int64_t act_floats = kActBytes / 4;
  up.staged = (N <= 2 && (int64_t)N * d <= act_floats) ? 1 : 0;
  const int op_up = bld.add(up);
  for (int s = 0; s < h->n_sm; ++s)
    bld.place(op_up, s, (int)((int64_t)F * s / h->n_sm), (int)((int64_t)F * (s + 1) / h->n_sm), 0);

  OpDesc dn = ex;
  dn.type = OP_MOE_DOWN;
  dn.ew[0] = L.e_down;
  dn.sw[0] = L.s_down;
  dn.esc[0] = L.e_down_scales;
  dn.ssc[0] = L.s_down_scales;
  dn.egs[0] = L.e_down_gscale;
  dn.sgs[0] = L.s_down_gscale;
  dn.ssq_out = 2 * i + 2;
  {  // routing of the rows, the SM's slice of x and two expert input buffers
    const int64_t rt = (N * D.top_k + 3) & ~3;
    const int64_t xr = ((int64_t)N * ((d + h->n_sm - 1) / h->n_sm) + 3) & ~3;
    dn.staged = (N <= 2 && 2 * rt + xr + 2LL * N * F <= act_floats) ? 1 : 0;
  }
  const int op_dn = bld.add(dn);
  for (int s = 0; s < h->n_sm; ++s)
    bld.place(op_dn, s, (int)((int64_t)d * s / h->n_sm), (int)((int64_t)d * (s + 1) / h->n_sm), 0);
}

// Host-side program of one (batch, rows, head) shape: the op list, the flattened per-SM queues and their
// offsets. Reads the handle's shape, weights, slots and activation buffer pointers; touches no device.
struct HostProgram {
  std::vector<OpDesc> ops;
  std::vector<Instr> flat;
  std::vector<int32_t> qoff;
};

mk_status construct_program(mk_handle* h, int B, int R, bool head, HostProgram& hp) {
  const mk_model_desc& D = h->desc;
  const int N = B * R;
  const int d = D.d_model;
  h->pk.n_sm = h->n_sm;
  Builder bld(h->n_sm, &h->pk);

  {  // embedding
    OpDesc e = blank(OP_EMBED);
    e.ssq_out = 0;
    const int op = bld.add(e);
    for (int s = 0; s < h->n_sm; ++s)
      bld.place(op, s, (int)((int64_t)d * s / h->n_sm), (int)((int64_t)d * (s + 1) / h->n_sm), 0);
  }
  for (int i = 0; i < D.n_layers; ++i) {
    const mk_layer_weights& L = h->w.layers[i];
    const int m = D.mixer[i];
    if (m == MK_MIXER_GQA) {
      const int hq = D.n_q_heads, hkv = D.n_kv_heads, hd = D.head_dim, G = hq / hkv;
      OpDesc qkv = gemv_desc(d, {{L.wq, hq * hd}, {L.wk, hkv * hd}, {L.wv, hkv * hd}});
      qkv.layer = i;
      qkv.in_kind = IN_NORM;
      qkv.gain = reinterpret_cast<const uint16_t*>(L.attn_norm);
      qkv.ssq_in = 2 * i;
      qkv.out_kind = OUT_STORE;
      qkv.out = h->proj;
      qkv.out_stride = h->proj_stride;
      gemv_op(bld, qkv, N);

      OpDesc ra = blank(OP_ROPE_APPEND);
      ra.layer = i;
      ra.slot = h->slot[i];
      ra.n_heads = hq;
      ra.n_kv_heads = hkv;
      ra.head_dim = hd;
      ra.out = h->proj;
      ra.out_stride = h->proj_stride;
      const int op_ra = bld.add(ra);
      for (int s = 0; s < h->n_sm; ++s) bld.place(op_ra, s, 0, 0, 0);

      OpDesc at = blank(OP_ATTN);
      at.layer = i;
      at.slot = h->slot[i];
      at.n_heads = hq;
      at.n_kv_heads = hkv;
      at.head_dim = hd;
      at.groups = G;
      at.in = h->proj;
      at.in_stride = h->proj_stride;
      at.out = h->attn_out;
      at.out_stride = h->attn_stride;
      // rows per instruction so that each warp owns at most 4 (row, head) pairs
      const int rows_per = std::max(1, std::min(R, (4 * kConsumerWarps) / G));
      const int nsplit = (R + rows_per - 1) / rows_per;
      at.nchunk = std::max(1, h->n_sm / (B * hkv * nsplit));
      const int op_at = bld.add(at);
      int k = 0;
      for (int b = 0; b < B; ++b)
        for (int g = 0; g < hkv; ++g)
          for (int c = 0; c < at.nchunk; ++c)
            for (int sp = 0; sp < nsplit; ++sp, ++k) {
              const int rlo = sp * rows_per, rhi = std::min(R, rlo + rows_per);
              bld.place(op_at, k % h->n_sm, b * hkv + g, c, rlo | (rhi << 8));
            }

      OpDesc cb = at;
      cb.type = OP_ATTN_COMBINE;
      cb.n_instr = 0;
      cb.n_deps = 0;
      const int op_cb = bld.add(cb);
      k = 0;
      for (int b = 0; b < B; ++b)
        for (int r = 0; r < R; ++r)
          for (int hh = 0; hh < hq; ++hh, ++k) bld.place(op_cb, k % h->n_sm, b, r, hh);

      OpDesc o = gemv_desc(hq * hd, {{L.wo, d}});
      o.layer = i;
      o.in_kind = IN_BUF;
      o.in = h->attn_out;
      o.in_stride = h->attn_stride;
      o.out_kind = OUT_RESID;
      o.ssq_out = 2 * i + 1;
      gemv_op(bld, o, N);
    } else if (is_delta(m)) {  // gated delta net / KDA
      const int H = D.lin_heads, dk = D.lin_dk, dv = D.lin_dv;
      const bool kda = m == MK_MIXER_KDA;
      OpDesc pj = gemv_desc(d, {{L.wq, H * dk}, {L.wk, H * dk}, {L.wv, H * dv}, {L.wa, kda ? H * dk : H}, {L.wb, H}});
      pj.layer = i;
      pj.in_kind = IN_NORM;
      pj.gain = reinterpret_cast<const uint16_t*>(L.attn_norm);
      pj.ssq_in = 2 * i;
      pj.out_kind = OUT_STORE;
      pj.out = h->proj;
      pj.out_stride = h->proj_stride;
      gemv_op(bld, pj, N);

      OpDesc dl = blank(OP_DELTA);
      dl.layer = i;
      dl.slot = h->slot[i];
      dl.n_heads = H;
      dl.dk = dk;
      dl.dv = dv;
      dl.per_channel_decay = kda ? 1 : 0;
      // value columns per instruction: 8 to 64 (1 to 8 per warp), the fewest that keep the instruction
      // count within one per SM (one instruction costs a few dependent memory round trips, whatever its width);
      // 16 columns per warp measured slower than 8 at batch 8 (their serial per-row work outweighs the
      // fewer instructions). The full build of the kernel, with the MLA / MoE handlers, gives this handler
      // fewer registers: up to 32 columns there.
      const int cw_max = h->full_ops ? 4 : 8;
      int cw = 1;
      while (cw < cw_max && (int64_t)B * H * ((dv + kConsumerWarps * cw - 1) / (kConsumerWarps * cw)) > h->n_sm) cw *= 2;
      dl.col_group = kConsumerWarps * cw;
      dl.in = h->proj;
      dl.in_stride = h->proj_stride;
      dl.out = h->attn_out;
      dl.out_stride = h->attn_stride;
      const int op_dl = bld.add(dl);
      const int ngrp = (dv + dl.col_group - 1) / dl.col_group;
      int k = 0;
      for (int b = 0; b < B; ++b)
        for (int hh = 0; hh < H; ++hh)
          for (int jg = 0; jg < ngrp; ++jg, ++k) bld.place(op_dl, k % h->n_sm, b, hh, jg);

      OpDesc o = gemv_desc(H * dv, {{L.wo, d}});
      o.layer = i;
      o.in_kind = IN_BUF;
      o.in = h->attn_out;
      o.in_stride = h->attn_stride;
      o.out_kind = OUT_RESID;
      o.ssq_out = 2 * i + 1;
      gemv_op(bld, o, N);
    } else {
      mla_layer(h, bld, i, B, R);
    }
    if (D.ffn_kind == MK_FFN_MOE) {
      moe_layer(h, bld, i, N);
      continue;
    }
    // dense SwiGLU
    OpDesc up = gemv_desc(d, {{L.w_gate, D.ffn_dim}, {L.w_up, D.ffn_dim}});
    up.rows = D.ffn_dim;  // logical rows: each pairs a gate row with an up row
    up.layer = i;
    up.in_kind = IN_NORM;
    up.gain = reinterpret_cast<const uint16_t*>(L.ffn_norm);
    up.ssq_in = 2 * i + 1;
    up.out_kind = OUT_SWIGLU;
    up.out = h->hbuf;
    up.out_stride = h->hbuf_stride;
    gemv_op(bld, up, N);

    OpDesc dn = gemv_desc(D.ffn_dim, {{L.w_down, d}});
    dn.layer = i;
    dn.in_kind = IN_BUF;
    dn.in = h->hbuf;
    dn.in_stride = h->hbuf_stride;
    dn.out_kind = OUT_RESID;
    dn.ssq_out = 2 * i + 2;
    gemv_op(bld, dn, N);
  }
  if (head) {
    OpDesc lm = gemv_desc(d, {{D.tied_embedding ? h->w.embed : h->w.lm_head, D.vocab}});
    lm.in_kind = IN_NORM;
    lm.gain = reinterpret_cast<const uint16_t*>(h->w.final_norm);
    lm.ssq_in = 2 * D.n_layers;
    lm.out_kind = OUT_LOGITS;
    gemv_op(bld, lm, N);
  }
  {
    OpDesc f = blank(OP_FINAL);
    const int op = bld.add(f);
    bld.place(op, 0, 0, 0, 0);
  }

  if ((int)bld.ops.size() > h->max_ops)
    return fail(h, MK_ERR_UNSUPPORTED, "program has %d ops, more than the %d counters allocated",
                (int)bld.ops.size(), h->max_ops);
  hp.ops = std::move(bld.ops);
  hp.flat.clear();
  hp.qoff.assign(h->n_sm + 1, 0);
  for (int s = 0; s < h->n_sm; ++s) {
    hp.qoff[s] = (int32_t)hp.flat.size();
    hp.flat.insert(hp.flat.end(), bld.q[s].begin(), bld.q[s].end());
  }
  hp.qoff[h->n_sm] = (int32_t)hp.flat.size();
  return MK_OK;
}

Program build_program(mk_handle* h, int B, int R, bool head, mk_status* st) {
  Program prog;
  prog.B = B;
  prog.R = R;
  prog.head = head;
  HostProgram hp;
  *st = construct_program(h, B, R, head, hp);
  if (*st != MK_OK) return prog;
  const std::vector<Instr>& flat = hp.flat;
  const std::vector<int32_t>& qoff = hp.qoff;
  prog.n_ops = (int)hp.ops.size();
  prog.n_instr = (int)flat.size();
  cudaError_t e;
  if ((e = cudaMalloc(&prog.d_ops, sizeof(OpDesc) * prog.n_ops)) != cudaSuccess ||
      (e = cudaMalloc(&prog.d_instr, sizeof(Instr) * std::max(1, prog.n_instr))) != cudaSuccess ||
      (e = cudaMalloc(&prog.d_qoff, sizeof(int32_t) * (h->n_sm + 1))) != cudaSuccess) {
    *st = cuda_fail(h, e, "program allocation");
    return prog;
  }
  if ((e = cudaMemcpy(prog.d_ops, hp.ops.data(), sizeof(OpDesc) * prog.n_ops, cudaMemcpyHostToDevice)) != cudaSuccess ||
      (e = cudaMemcpy(prog.d_instr, flat.data(), sizeof(Instr) * prog.n_instr, cudaMemcpyHostToDevice)) != cudaSuccess ||
      (e = cudaMemcpy(prog.d_qoff, qoff.data(), sizeof(int32_t) * (h->n_sm + 1), cudaMemcpyHostToDevice)) !=
          cudaSuccess) {
    *st = cuda_fail(h, e, "program upload");
    return prog;
  }
  h->bytes += (int64_t)(sizeof(OpDesc) * prog.n_ops + sizeof(Instr) * prog.n_instr + sizeof(int32_t) * (h->n_sm + 1));
  for (const OpDesc& o : hp.ops) prog.use_tc = prog.use_tc || (o.type == OP_GEMV && o.mma == 2);
  return prog;
}

Program* get_program(mk_handle* h, int B, int R, bool head, mk_status* st) {
  for (auto& p : h->programs)
    if (p.B == B && p.R == R && p.head == head) return &p;
  *st = MK_OK;
  Program p = build_program(h, B, R, head, st);
  if (*st != MK_OK) {
    cudaFree(p.d_ops);
    cudaFree(p.d_instr);
    cudaFree(p.d_qoff);
    return nullptr;
  }
  h->programs.push_back(p);
  return &h->programs.back();
}

// Fills the kernel parameters from the handle's buffers and the device copy of a program; launches.
mk_status launch_program(mk_handle* h, const Program* prog, const int32_t* tokens, int tok_stride,
                         const int32_t* positions, int B, int R, float* logits, int32_t* argmax, bool commit_all,
                         cudaStream_t stream, int n_steps = 1, int32_t* accept_out = nullptr) {
  const mk_model_desc& D = h->desc;
  KParams p;
  std::memset(&p, 0, sizeof(p));
  p.ops = prog->d_ops;
  p.instrs = prog->d_instr;
  p.qoff = prog->d_qoff;
  p.counters = h->counters;
  p.status = h->status;
  p.abort_flag = h->abort_flag;
  p.timeout_ns = h->wait_limit_ns;
  p.use_tc = prog->use_tc ? 1 : 0;
  p.spin_mask = h->wait_limit_ns < 1000000ull ? 0u : 63u;
  p.n_ops = prog->n_ops;
  p.n_sm = h->n_sm;
  p.tokens = tokens;
  p.tok_stride = tok_stride;
  p.positions = positions;
  p.B = B;
  p.R = R;
  p.N = B * R;
  p.epoch = h->epoch + 1;  // step s of the launch uses epoch + s: the pending-row halves alternate per step
  h->epoch += (uint32_t)n_steps;
  p.n_steps = n_steps;
  p.commit_all = commit_all ? 1 : 0;
  p.logits = logits;
  p.argmax = argmax;
  p.accept_out = accept_out;
  p.d = D.d_model;
  p.V = D.vocab;
  p.max_ctx = D.max_ctx;
  p.max_batch = D.max_batch;
  p.max_rows = D.max_rows;
  p.eps = D.norm_eps;
  p.embed = reinterpret_cast<const uint16_t*>(h->w.embed);
  p.x = h->x;
  p.ssq = h->ssq;
  p.amax_part = h->amax_part;
  p.attn_part = h->attn_part;
  p.attn_part_stride = h->attn_part_stride;
  p.kcache = h->kcache;
  p.vcache = h->vcache;
  p.state = h->state;
  p.pend = h->pend;
  p.pend_rec = h->pend_rec;
  p.latent = h->latent;
  p.route_idx = h->route_idx;
  p.route_w = h->route_w;
  p.union_list = h->union_list;
  p.hexp = h->hexp;
  p.route_log = h->route_log;
  p.route_force = h->route_force;
  p.seq = h->seq;
  p.rope = h->rope;
  p.rot_dim = h->rot_dim;
  p.n_q_heads = D.n_q_heads;
  p.n_kv_heads = D.n_kv_heads;
  p.head_dim = D.head_dim;
  p.lin_heads = D.lin_heads;
  p.lin_dk = D.lin_dk;
  p.lin_dv = D.lin_dv;
  if (h->trace && (size_t)prog->n_instr <= h->trace_cap) {
    p.trace = h->trace;
    h->last_prog = prog;
  }
  h->n_ops_last = prog->n_ops;
  cudaError_t e = kernel_launch(h->full_ops, p, h->n_sm, stream);
  if (e != cudaSuccess) return cuda_fail(h, e, "megakernel launch");
  return MK_OK;
}

mk_status launch_step(mk_handle* h, const int32_t* tokens, int tok_stride, const int32_t* positions, int B, int R,
                      float* logits, int32_t* argmax, bool commit_all, cudaStream_t stream, int n_steps = 1,
                      int32_t* accept_out = nullptr) {
  mk_status st = MK_OK;
  const bool head = logits != nullptr || argmax != nullptr || accept_out != nullptr;
  Program* prog = get_program(h, B, R, head, &st);
  if (!prog) return st;
  return launch_program(h, prog, tokens, tok_stride, positions, B, R, logits, argmax, commit_all, stream, n_steps,
                        accept_out);
}

// The packed GEMV weights of a handle: the groups are collected from the decode program of one row (every
// step shape reads the same groups), then the caller's copy is taken, or one is made here.
mk_status make_packed(mk_handle* h) {
  HostProgram hp;
  h->pk = PackTable();
  mk_status st = construct_program(h, 1, 1, true, hp);
  if (st != MK_OK) return st;
  if (h->w.packed) {
    if (reinterpret_cast<uintptr_t>(h->w.packed) & 1023u) return fail(h, MK_ERR_INVALID_ARG, "packed weights not 1024-byte aligned");
    h->pk.base = static_cast<const uint8_t*>(h->w.packed);
    return MK_OK;
  }
  cudaError_t e = cudaMalloc(&h->packed_own, std::max<size_t>(h->pk.total, 1024));
  if (e != cudaSuccess) {
    h->packed_own = nullptr;
    return cuda_fail(h, e, "packed weights");
  }
  h->bytes += (int64_t)h->pk.total;
  h->pk.base = static_cast<const uint8_t*>(h->packed_own);
  for (const PackTable::Group& g : h->pk.groups)
    if ((e = pack_gemv_launch(static_cast<uint8_t*>(h->packed_own) + g.offset, g.src, 0)) != cudaSuccess)
      return cuda_fail(h, e, "weight packing");
  return MK_OK;
}

// A shape-only handle for the calls that take a model without creating one (layout and packing).
mk_status shape_handle(mk_handle& tmp, const mk_model_desc* desc, const mk_weights* weights, int device) {
  tmp.desc = *desc;
  tmp.w = *weights;
  tmp.device = device;
  mk_status st = check_desc(&tmp, tmp.desc, tmp.w);
  if (st != MK_OK) return st;
  if (cudaDeviceGetAttribute(&tmp.n_sm, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || tmp.n_sm < 1)
    return MK_ERR_CUDA;
  derive_layout(&tmp);
  HostProgram hp;
  return construct_program(&tmp, 1, 1, true, hp);
}

}  // namespace

// ==================================================================================================
// C ABI
// ==================================================================================================
extern "C" {

mk_status mk_packed_weight_bytes(const mk_model_desc* desc, const mk_weights* weights, int device, uint64_t* bytes) {
  if (!desc || !weights || !bytes) return MK_ERR_INVALID_ARG;
  mk_handle tmp;
  const mk_status st = shape_handle(tmp, desc, weights, device);
  if (st != MK_OK) {
    if (!tmp.err.empty()) fprintf(stderr, "mk_packed_weight_bytes: %s\n", tmp.err.c_str());
    return st;
  }
  *bytes = (uint64_t)tmp.pk.total;
  return MK_OK;
}

mk_status mk_pack_weights(const mk_model_desc* desc, const mk_weights* weights, int device, void* packed,
                          void* stream) {
  if (!desc || !weights || !packed) return MK_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(packed) & 1023u) return MK_ERR_INVALID_ARG;
  mk_handle tmp;
  const mk_status st = shape_handle(tmp, desc, weights, device);
  if (st != MK_OK) {
    if (!tmp.err.empty()) fprintf(stderr, "mk_pack_weights: %s\n", tmp.err.c_str());
    return st;
  }
  int cur = 0;
  if (cudaGetDevice(&cur) != cudaSuccess || cudaSetDevice(device) != cudaSuccess) return MK_ERR_CUDA;
  cudaError_t e = cudaSuccess;
  for (const PackTable::Group& g : tmp.pk.groups) {
    e = pack_gemv_launch(static_cast<uint8_t*>(packed) + g.offset, g.src, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) break;
  }
  cudaSetDevice(cur);
  if (e != cudaSuccess) {
    fprintf(stderr, "mk_pack_weights: %s\n", cudaGetErrorString(e));
    return MK_ERR_CUDA;
  }
  return MK_OK;
}

mk_status mk_create(const mk_model_desc* desc, const mk_weights* weights, int device, mk_handle** out) {
  if (!desc || !weights || !out) return MK_ERR_INVALID_ARG;
  *out = nullptr;
  mk_handle* h = new mk_handle();
  h->desc = *desc;
  h->w = *weights;
  h->device = device;
  mk_status st = check_desc(h, h->desc, h->w);
  if (st != MK_OK) {
    // keep the message for mk_last_error(NULL)-style callers: print it, then fail
    fprintf(stderr, "mk_create: %s\n", h->err.c_str());
    delete h;
    return st;
  }
  cudaError_t e = cudaSetDevice(device);
  if (e != cudaSuccess) {
    delete h;
    return MK_ERR_CUDA;
  }
  int coop = 0;
  cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, device);
  cudaDeviceGetAttribute(&h->n_sm, cudaDevAttrMultiProcessorCount, device);
  int smem_optin = 0;
  cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
  if (!coop || smem_optin < (int)kernel_smem_bytes()) {
    fprintf(stderr, "mk_create: device lacks cooperative launch or %zu bytes of shared memory\n", kernel_smem_bytes());
    delete h;
    return MK_ERR_UNSUPPORTED;
  }
  derive_layout(h);
  if ((e = kernel_configure(h->full_ops)) != cudaSuccess) {
    fprintf(stderr, "mk_create: %s\n", cudaGetErrorString(e));
    delete h;
    return MK_ERR_CUDA;
  }

  const mk_model_desc& D = h->desc;
  const int Bm = D.max_batch, Rm = D.max_rows;

#define ALLOC(ptr, count) \
  if ((st = dev_alloc(h, &h->ptr, (size_t)(count), #ptr)) != MK_OK) goto fail_out
  ALLOC(x, (size_t)kMaxN * D.d_model);
  ALLOC(proj, (size_t)kMaxN * h->proj_stride);
  ALLOC(attn_out, (size_t)kMaxN * h->attn_stride);
  ALLOC(hbuf, (size_t)kMaxN * h->hbuf_stride);
  ALLOC(ssq, (size_t)(2 * D.n_layers + 1) * h->n_sm * kMaxN);
  ALLOC(amax_part, (size_t)h->n_sm * kMaxN);
  ALLOC(counters, h->max_ops);
  ALLOC(status, 4);
  ALLOC(abort_flag, 4);
  ALLOC(seq, Bm);
  ALLOC(pos_buf, std::max(Bm, 8));
  ALLOC(stage_tok, kMaxN);
  ALLOC(stage_pos, std::max(Bm, 8));
  ALLOC(stage_argmax, kMaxN);
  ALLOC(stage_logits, (size_t)h->nmax * D.vocab);
  if (h->n_gqa) {
    const int hkv = D.n_kv_heads, hd = D.head_dim;
    const size_t cache = (size_t)h->n_gqa * Bm * hkv * D.max_ctx * hd;
    ALLOC(kcache, cache);
    ALLOC(vcache, cache);
  }
  if (h->n_gqa || h->n_mla) ALLOC(attn_part, attn_part_records(h, Bm, Rm) * h->attn_part_stride);
  if (h->n_mla) {
    ALLOC(latent, (size_t)h->n_mla * Bm * D.max_ctx * (D.kv_lora + D.qk_rope));
    ALLOC(mla_cq, (size_t)kMaxN * D.q_lora);
    ALLOC(mla_qf, (size_t)kMaxN * h->mla_qf_stride);
    ALLOC(mla_qt, (size_t)kMaxN * h->mla_qt_stride);
    ALLOC(mla_olat, (size_t)kMaxN * h->mla_olat_stride);
  }
  if (D.ffn_kind == MK_FFN_MOE) {
    ALLOC(route_idx, (size_t)kMaxN * kMaxTopK);
    ALLOC(route_w, (size_t)kMaxN * kMaxTopK);
    ALLOC(union_list, (size_t)kMaxExperts + 1);
    ALLOC(hexp, h->hexp_floats);
  }
  if (h->n_delta) {
    const int H = D.lin_heads, dk = D.lin_dk, dv = D.lin_dv;
    ALLOC(state, (size_t)h->n_delta * Bm * H * dv * dk);
    ALLOC(pend, (size_t)h->n_delta * 2 * Bm * Rm * H * h->pend_rec);
  }
  if (h->rot_dim) {
    ALLOC(rope, (size_t)D.max_ctx * (h->rot_dim / 2));
    if ((e = rope_table_launch(h->rope, D.max_ctx, h->rot_dim, (double)D.rope_theta, 0)) != cudaSuccess) {
      st = cuda_fail(h, e, "rope table");
      goto fail_out;
    }
  }
  if (const char* tp = getenv("MK_TRACE")) {
    h->trace_path = tp;
    h->trace_cap = (size_t)h->n_sm * 64 * D.n_layers + 4096;
    ALLOC(trace, h->trace_cap * kTraceWords);
  }
#undef ALLOC
  if ((st = make_packed(h)) != MK_OK) goto fail_out;
  if ((e = cudaDeviceSynchronize()) != cudaSuccess) {
    st = cuda_fail(h, e, "create");
    goto fail_out;
  }
  *out = h;
  return MK_OK;
fail_out:
  fprintf(stderr, "mk_create: %s\n", h->err.c_str());
  mk_destroy(h);
  return st;
}

mk_status mk_prefill_kv(mk_handle* h, const int32_t* tokens, int batch, int n_tokens, void* stream) {
  if (!h || !tokens) return MK_ERR_INVALID_ARG;
  const mk_model_desc& D = h->desc;
  if (batch < 1 || batch > D.max_batch || batch > kMaxN) return fail(h, MK_ERR_INVALID_ARG, "batch %d", batch);
  if (n_tokens < 1 || n_tokens > D.max_ctx) return fail(h, MK_ERR_INVALID_ARG, "n_tokens %d", n_tokens);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSetDevice(h->device);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaSetDevice");
  if ((e = cudaMemsetAsync(h->seq, 0, sizeof(SeqState) * batch, s)) != cudaSuccess) return cuda_fail(h, e, "reset");
  if (h->n_delta) {
    const size_t per_seq = (size_t)D.lin_heads * D.lin_dv * D.lin_dk;
    for (int sl = 0; sl < h->n_delta; ++sl) {
      e = cudaMemsetAsync(h->state + (size_t)sl * D.max_batch * per_seq, 0, sizeof(float) * per_seq * batch, s);
      if (e != cudaSuccess) return cuda_fail(h, e, "state reset");
    }
  }
  const int chunk_rows = std::max(1, std::min(D.max_rows, kMaxN / batch));  // rows per launch: batch x rows <= kMaxN
  for (int c0 = 0; c0 < n_tokens; c0 += chunk_rows) {
    const int rc = std::min(chunk_rows, n_tokens - c0);
    if ((e = fill_i32_launch(h->pos_buf, batch, c0, s)) != cudaSuccess) return cuda_fail(h, e, "positions");
    mk_status st = launch_step(h, tokens + c0, n_tokens, h->pos_buf, batch, rc, nullptr, nullptr,
                               c0 + rc == n_tokens, s);
    if (st != MK_OK) return st;
  }
  return MK_OK;
}

mk_status mk_decode_step(mk_handle* h, const int32_t* tokens, const int32_t* positions, int batch, int rows,
                         float* logits_out, int32_t* argmax_out, void* stream) {
  if (!h || !tokens || !positions) return MK_ERR_INVALID_ARG;
  const mk_model_desc& D = h->desc;
  if (batch < 1 || batch > D.max_batch) return fail(h, MK_ERR_INVALID_ARG, "batch %d outside 1..%d", batch, D.max_batch);
  if (rows < 1 || rows > D.max_rows) return fail(h, MK_ERR_INVALID_ARG, "rows %d outside 1..%d", rows, D.max_rows);
  if (batch * rows > kMaxN) return fail(h, MK_ERR_INVALID_ARG, "batch x rows = %d above %d", batch * rows, kMaxN);
  if (!logits_out && !argmax_out) return fail(h, MK_ERR_INVALID_ARG, "no output requested");
  cudaError_t e = cudaSetDevice(h->device);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaSetDevice");
  return launch_step(h, tokens, rows, positions, batch, rows, logits_out, argmax_out, false,
                     reinterpret_cast<cudaStream_t>(stream));
}

mk_status mk_decode_step_host(mk_handle* h, const int32_t* tokens_host, const int32_t* positions_host, int batch,
                              int rows, float* logits_host, int32_t* argmax_host, void* stream) {
  if (!h || !tokens_host || !positions_host || !argmax_host) return MK_ERR_INVALID_ARG;
  const mk_model_desc& D = h->desc;
  if (batch < 1 || batch > D.max_batch || rows < 1 || rows > D.max_rows || batch * rows > kMaxN)
    return fail(h, MK_ERR_INVALID_ARG, "batch %d / rows %d out of range", batch, rows);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSetDevice(h->device);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaSetDevice");
  const int n = batch * rows;
  if ((e = cudaMemcpyAsync(h->stage_tok, tokens_host, sizeof(int32_t) * n, cudaMemcpyHostToDevice, s)) != cudaSuccess ||
      (e = cudaMemcpyAsync(h->stage_pos, positions_host, sizeof(int32_t) * batch, cudaMemcpyHostToDevice, s)) !=
          cudaSuccess)
    return cuda_fail(h, e, "host to device copy");
  mk_status st = launch_step(h, h->stage_tok, rows, h->stage_pos, batch, rows, logits_host ? h->stage_logits : nullptr,
                             h->stage_argmax, false, s);
  if (st != MK_OK) return st;
  if ((e = cudaMemcpyAsync(argmax_host, h->stage_argmax, sizeof(int32_t) * n, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
    return cuda_fail(h, e, "device to host copy");
  if (logits_host &&
      (e = cudaMemcpyAsync(logits_host, h->stage_logits, sizeof(float) * (size_t)n * D.vocab, cudaMemcpyDeviceToHost,
                           s)) != cudaSuccess)
    return cuda_fail(h, e, "device to host copy");
  return mk_get_status(h, stream);
}

mk_status mk_verify_step(mk_handle* h, const int32_t* tokens, const int32_t* positions, int batch, int rows,
                         float* logits_out, int32_t* argmax_out, int32_t* accept_out, void* stream) {
  if (!h || !tokens || !positions || !accept_out) return MK_ERR_INVALID_ARG;
  const mk_model_desc& D = h->desc;
  if (batch < 1 || batch > D.max_batch) return fail(h, MK_ERR_INVALID_ARG, "batch %d outside 1..%d", batch, D.max_batch);
  if (rows < 2 || rows > D.max_rows) return fail(h, MK_ERR_INVALID_ARG, "rows %d outside 2..%d", rows, D.max_rows);
  if (batch * rows > kMaxN) return fail(h, MK_ERR_INVALID_ARG, "batch x rows = %d above %d", batch * rows, kMaxN);
  cudaError_t e = cudaSetDevice(h->device);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaSetDevice");
  return launch_step(h, tokens, rows, positions, batch, rows, logits_out, argmax_out, false,
                     reinterpret_cast<cudaStream_t>(stream), 1, accept_out);
}

mk_status mk_decode_steps(mk_handle* h, const int32_t* tokens, const int32_t* positions, int batch, int n_steps,
                          int32_t* tokens_out, float* logits_out, void* stream) {
  if (!h || !tokens || !positions || !tokens_out) return MK_ERR_INVALID_ARG;
  const mk_model_desc& D = h->desc;
  if (batch < 1 || batch > D.max_batch || batch > kMaxN)
    return fail(h, MK_ERR_INVALID_ARG, "batch %d outside 1..%d", batch, std::min(D.max_batch, kMaxN));
  if (n_steps < 1 || n_steps > D.max_ctx) return fail(h, MK_ERR_INVALID_ARG, "n_steps %d", n_steps);
  cudaError_t e = cudaSetDevice(h->device);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaSetDevice");
  return launch_step(h, tokens, 1, positions, batch, 1, logits_out, tokens_out, false,
                     reinterpret_cast<cudaStream_t>(stream), n_steps);
}

mk_status mk_decode_steps_host(mk_handle* h, const int32_t* tokens_host, const int32_t* positions_host, int batch,
                               int n_steps, int32_t* tokens_out_host, void* stream) {
  if (!h || !tokens_host || !positions_host || !tokens_out_host) return MK_ERR_INVALID_ARG;
  const mk_model_desc& D = h->desc;
  if (batch < 1 || batch > D.max_batch || batch > kMaxN || n_steps < 1 || n_steps > D.max_ctx)
    return fail(h, MK_ERR_INVALID_ARG, "batch %d / n_steps %d out of range", batch, n_steps);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSetDevice(h->device);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaSetDevice");
  if ((size_t)n_steps * batch > h->steps_cap) {
    // grows the handle's token staging (synchronous cudaMalloc, only when a longer run is asked for)
    if (h->stage_steps) cudaFree(h->stage_steps);
    h->stage_steps = nullptr;
    h->steps_cap = 0;
    if ((e = cudaMalloc(&h->stage_steps, sizeof(int32_t) * (size_t)n_steps * batch)) != cudaSuccess)
      return cuda_fail(h, e, "token staging");
    h->steps_cap = (size_t)n_steps * batch;
  }
  if ((e = cudaMemcpyAsync(h->stage_tok, tokens_host, sizeof(int32_t) * batch, cudaMemcpyHostToDevice, s)) != cudaSuccess ||
      (e = cudaMemcpyAsync(h->stage_pos, positions_host, sizeof(int32_t) * batch, cudaMemcpyHostToDevice, s)) !=
          cudaSuccess)
    return cuda_fail(h, e, "host to device copy");
  mk_status st = launch_step(h, h->stage_tok, 1, h->stage_pos, batch, 1, nullptr, h->stage_steps, false, s, n_steps);
  if (st != MK_OK) return st;
  if ((e = cudaMemcpyAsync(tokens_out_host, h->stage_steps, sizeof(int32_t) * (size_t)n_steps * batch,
                           cudaMemcpyDeviceToHost, s)) != cudaSuccess)
    return cuda_fail(h, e, "device to host copy");
  return mk_get_status(h, stream);
}

mk_status mk_get_status(mk_handle* h, void* stream) {
  if (!h) return MK_ERR_INVALID_ARG;
  cudaError_t e = cudaSetDevice(h->device);
  if (e == cudaSuccess) e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(h, e, "stream synchronize");
  int32_t code = 0;
  if ((e = cudaMemcpy(&code, h->status, sizeof(int32_t), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(h, e, "status read");
  if (code != 0) {
    cudaMemset(h->status, 0, sizeof(int32_t));
    cudaMemset(h->abort_flag, 0, sizeof(int32_t));
    cudaMemset(h->counters, 0, sizeof(uint32_t) * h->max_ops);
    cudaDeviceSynchronize();
    h->err = code == MK_ERR_TIMEOUT ? "device watchdog timeout" : "device input check failed (token or position)";
    return (mk_status)code;
  }
  return MK_OK;
}

mk_status mk_plan(const mk_model_desc* desc, const mk_weights* weights, int n_sm, int batch, int rows,
                  int with_head, mk_plan_op* ops, int ops_cap, int* n_ops, mk_plan_instr* instrs, int instr_cap,
                  int* n_instr) {
  if (!desc || !weights || !n_ops || !n_instr || n_sm < 1 || n_sm > 4096) return MK_ERR_INVALID_ARG;
  mk_handle tmp;  // shape only: no device memory, buffer pointers stay NULL
  tmp.desc = *desc;
  tmp.w = *weights;
  tmp.n_sm = n_sm;
  mk_status st = check_desc(&tmp, tmp.desc, tmp.w);
  if (st != MK_OK) return st;
  if (batch < 1 || batch > desc->max_batch || rows < 1 || rows > desc->max_rows || batch * rows > kMaxN)
    return MK_ERR_INVALID_ARG;
  derive_layout(&tmp);
  HostProgram hp;
  if ((st = construct_program(&tmp, batch, rows, with_head != 0, hp)) != MK_OK) return st;
  *n_ops = (int)hp.ops.size();
  *n_instr = (int)hp.flat.size();
  for (int i = 0; i < (int)hp.ops.size() && ops && i < ops_cap; ++i) {
    const OpDesc& o = hp.ops[i];
    mk_plan_op& r = ops[i];
    r.type = o.type;
    r.n_instr = o.n_instr;
    r.layer = o.layer;
    r.rows = o.rows;
    r.K = o.K;
    r.k_begin = o.k_begin;
    r.ldw = o.ldw;
    r.mma = o.mma;
    r.staged = o.staged;
    r.kc = o.kc;
    r.rg = o.rg;
    r.passes = o.passes;
    r.out_kind = o.out_kind;
    r.nchunk = o.nchunk;
    r.groups = o.groups;
    r.head_dim = o.head_dim;
    r.n_heads = o.n_heads;
    r.n_kv_heads = o.n_kv_heads;
    r.col_group = o.col_group;
    r.ncols = o.ncols;
    r.pa0 = o.pa0;
    r.patoms = o.patoms;
    r.pk_offset = o.type == OP_GEMV ? (int64_t)(o.wp - tmp.pk.base) : 0;
  }
  if (instrs) {
    int k = 0;
    for (int sm = 0; sm < n_sm; ++sm)
      for (int q = hp.qoff[sm]; q < hp.qoff[sm + 1] && k < instr_cap; ++q, ++k) {
        const Instr& in = hp.flat[q];
        instrs[k].op = in.op;
        instrs[k].sm = sm;
        instrs[k].a = in.a;
        instrs[k].b = in.b;
        instrs[k].c = in.c;
      }
  }
  return MK_OK;
}

mk_status mk_fork_sequence(mk_handle* h, int src, int dst, void* stream) {
  if (!h) return MK_ERR_INVALID_ARG;
  const mk_model_desc& D = h->desc;
  const int Bm = D.max_batch;
  if (src < 0 || src >= Bm || dst < 0 || dst >= Bm) return fail(h, MK_ERR_INVALID_ARG, "sequence %d -> %d", src, dst);
  if (src == dst) return MK_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSetDevice(h->device);
  auto copy = [&](void* base, size_t per_seq_bytes, size_t group) {
    // sequence b's block of `per_seq_bytes` inside group `group` of max_batch such blocks
    if (e != cudaSuccess) return;
    char* g = static_cast<char*>(base) + group * Bm * per_seq_bytes;
    e = cudaMemcpyAsync(g + dst * per_seq_bytes, g + src * per_seq_bytes, per_seq_bytes, cudaMemcpyDeviceToDevice, s);
  };
  for (int sl = 0; sl < h->n_gqa; ++sl) {
    const size_t per = sizeof(uint16_t) * D.n_kv_heads * D.max_ctx * D.head_dim;
    copy(h->kcache, per, sl);
    copy(h->vcache, per, sl);
  }
  for (int sl = 0; sl < h->n_mla; ++sl)
    copy(h->latent, sizeof(uint16_t) * D.max_ctx * (D.kv_lora + D.qk_rope), sl);
  for (int sl = 0; sl < h->n_delta; ++sl) {
    copy(h->state, sizeof(float) * D.lin_heads * D.lin_dv * D.lin_dk, sl);
    for (int par = 0; par < 2; ++par)
      copy(h->pend, sizeof(float) * D.max_rows * D.lin_heads * h->pend_rec, 2 * sl + par);
  }
  copy(h->seq, sizeof(SeqState), 0);
  if (e != cudaSuccess) return cuda_fail(h, e, "fork copy");
  return MK_OK;
}

mk_status mk_set_routing_log(mk_handle* h, int32_t* device_log) {
  if (!h) return MK_ERR_INVALID_ARG;
  if (device_log && h->desc.ffn_kind != MK_FFN_MOE) return fail(h, MK_ERR_INVALID_ARG, "the model has no MoE layers");
  if (device_log && (reinterpret_cast<uintptr_t>(device_log) & 3u))
    return fail(h, MK_ERR_INVALID_ARG, "routing log must be 4-byte aligned");
  h->route_log = device_log;
  return MK_OK;
}

mk_status mk_set_wait_limit(mk_handle* h, uint64_t limit_ns) {
  if (!h) return MK_ERR_INVALID_ARG;
  if (limit_ns == 0) return fail(h, MK_ERR_INVALID_ARG, "wait limit must be positive");
  h->wait_limit_ns = limit_ns;
  return MK_OK;
}

mk_status mk_set_routing_override(mk_handle* h, const int32_t* device_ids) {
  if (!h) return MK_ERR_INVALID_ARG;
  if (device_ids && h->desc.ffn_kind != MK_FFN_MOE) return fail(h, MK_ERR_INVALID_ARG, "the model has no MoE layers");
  if (device_ids && (reinterpret_cast<uintptr_t>(device_ids) & 3u))
    return fail(h, MK_ERR_INVALID_ARG, "routing override must be 4-byte aligned");
  h->route_force = device_ids;
  return MK_OK;
}

const char* mk_last_error(const mk_handle* h) { return h ? h->err.c_str() : ""; }

mk_status mk_get_info(const mk_handle* h, mk_info* out) {
  if (!h || !out) return MK_ERR_INVALID_ARG;
  out->n_sm = h->n_sm;
  out->threads_per_cta = kThreads;
  out->smem_bytes = (int32_t)kernel_smem_bytes();
  out->ring_slots = kSlots;
  out->ring_slot_bytes = kSlotBytes;
  out->n_ops_last = h->n_ops_last;
  out->device_bytes = h->bytes;
  return MK_OK;
}

void mk_destroy(mk_handle* h) {
  if (!h) return;
  cudaSetDevice(h->device);
  cudaDeviceSynchronize();
  if (h->trace && h->last_prog && !h->trace_path.empty()) {
    // layout: int32 n_sm, n_ops, n_instr; int32 op type [n_ops]; int32 qoff [n_sm+1]; Instr [n_instr];
    // uint64 trace [n_instr][kTraceWords]
    const Program& pr = *h->last_prog;
    std::vector<OpDesc> ops(pr.n_ops);
    std::vector<Instr> ins(pr.n_instr);
    std::vector<int32_t> qoff(h->n_sm + 1);
    std::vector<unsigned long long> tr((size_t)pr.n_instr * kTraceWords);
    cudaMemcpy(ops.data(), pr.d_ops, sizeof(OpDesc) * pr.n_ops, cudaMemcpyDeviceToHost);
    cudaMemcpy(ins.data(), pr.d_instr, sizeof(Instr) * pr.n_instr, cudaMemcpyDeviceToHost);
    cudaMemcpy(qoff.data(), pr.d_qoff, sizeof(int32_t) * (h->n_sm + 1), cudaMemcpyDeviceToHost);
    cudaMemcpy(tr.data(), h->trace, sizeof(unsigned long long) * tr.size(), cudaMemcpyDeviceToHost);
    if (FILE* f = fopen(h->trace_path.c_str(), "wb")) {
      const int32_t hdr[3] = {h->n_sm, pr.n_ops, pr.n_instr};
      fwrite(hdr, sizeof(hdr), 1, f);
      for (const OpDesc& o : ops) fwrite(&o.type, sizeof(int32_t), 1, f);
      fwrite(qoff.data(), sizeof(int32_t), qoff.size(), f);
      fwrite(ins.data(), sizeof(Instr), ins.size(), f);
      fwrite(tr.data(), sizeof(unsigned long long), tr.size(), f);
      fclose(f);
    }
  }
  for (auto& p : h->programs) {
    cudaFree(p.d_ops);
    cudaFree(p.d_instr);
    cudaFree(p.d_qoff);
  }
  if (h->packed_own) cudaFree(h->packed_own);
  for (void* p : h->allocs) cudaFree(p);
  if (h->stage_steps) cudaFree(h->stage_steps);
  delete h;
}

}  // extern "C"

// ==================================================================================================
// mk_decode_step_static: the same step with no device allocation. Its working memory is one static
// device array of MK_STATIC_SCRATCH_BYTES; the caller owns the persistent buffers (caches, states).
// ==================================================================================================
namespace {

constexpr int kMaxStaticDevices = 64;

// Working memory of mk_decode_step_static. In host code this name is only a host-side stand-in for
// the device array: its device address comes from cudaGetSymbolAddress (static_scratch_address).
static __device__ __align__(256) unsigned char g_static_scratch[MK_STATIC_SCRATCH_BYTES];

std::mutex g_static_mu;
void* g_static_addr[kMaxStaticDevices] = {};

// The RoPE table the last call on each device wrote into the static array: where, for which shape. A call
// whose table would be identical and sits at the same offset skips the rewrite (nothing else a call writes
// can overlap it then: every buffer carved before it ends below it, and every buffer carved after it
// starts above it); any other call rewrites its own table and becomes the record.
struct StaticRope {
  bool valid = false;
  size_t offset = 0;
  int max_ctx = 0, rot_dim = 0;
  float theta = 0.f;
};
StaticRope g_static_rope[kMaxStaticDevices];

// Device address of the static array on `device`, which must be current. Resolved once per device.
mk_status static_scratch_address(int device, void** out) {
  if (device < 0 || device >= kMaxStaticDevices) return MK_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_addr[device]) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess || !ptr) {
      fprintf(stderr, "mk_decode_step_static: cudaGetSymbolAddress failed: %s\n", cudaGetErrorString(e));
      return MK_ERR_CUDA;
    }
    g_static_addr[device] = ptr;
  }
  *out = g_static_addr[device];
  return MK_OK;
}

size_t carve(size_t& off, size_t bytes) {
  off = (off + 255) & ~size_t(255);
  const size_t at = off;
  off += std::max<size_t>(bytes, 16);
  return at;
}

}  // namespace

extern "C" mk_status mk_decode_step_static(const mk_model_desc* desc, const mk_weights* weights,
                                           mk_state_buffers* state, const int32_t* tokens,
                                           const int32_t* positions, int batch, int rows, float* logits_out,
                                           int32_t* argmax_out, void* stream) {
  if (!desc || !weights || !state || !tokens || !positions) return MK_ERR_INVALID_ARG;
  if (!logits_out && !argmax_out) return MK_ERR_INVALID_ARG;
  mk_handle tmp;  // describes the step; every buffer pointer below is the caller's or in the static array
  tmp.desc = *desc;
  tmp.w = *weights;
  mk_status st = check_desc(&tmp, tmp.desc, tmp.w);
  if (st != MK_OK) {
    fprintf(stderr, "mk_decode_step_static: %s\n", tmp.err.c_str());
    return st;
  }
  const mk_model_desc& D = tmp.desc;
  if (batch < 1 || batch > D.max_batch || rows < 1 || rows > D.max_rows || batch * rows > kMaxN)
    return MK_ERR_INVALID_ARG;
  bool has_mla = false;
  for (int i = 0; i < D.n_layers; ++i) has_mla = has_mla || D.mixer[i] == MK_MIXER_MLA;
  if (has_mla || D.ffn_kind == MK_FFN_MOE) {
    fprintf(stderr, "mk_decode_step_static: MLA and MoE models are not accepted by this call\n");
    return MK_ERR_UNSUPPORTED;
  }
  cudaError_t e = cudaGetDevice(&tmp.device);
  if (e != cudaSuccess) return MK_ERR_CUDA;
  int coop = 0, smem_optin = 0;
  cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, tmp.device);
  cudaDeviceGetAttribute(&tmp.n_sm, cudaDevAttrMultiProcessorCount, tmp.device);
  cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, tmp.device);
  if (!coop || smem_optin < (int)kernel_smem_bytes()) return MK_ERR_UNSUPPORTED;
  derive_layout(&tmp);
  if (kernel_configure(tmp.full_ops) != cudaSuccess) return MK_ERR_CUDA;
  if (!state->seq || (tmp.n_gqa && (!state->kcache || !state->vcache)) ||
      (tmp.n_delta && (!state->state || !state->pending))) {
    fprintf(stderr, "mk_decode_step_static: a persistent buffer this model needs is NULL\n");
    return MK_ERR_INVALID_ARG;
  }
  void* base_v = nullptr;
  if ((st = static_scratch_address(tmp.device, &base_v)) != MK_OK) return st;
  unsigned char* base = static_cast<unsigned char*>(base_v);

  // carve the working memory of this step out of the static array
  const int N = batch * rows;
  size_t off = 0;
  const size_t o_counters = carve(off, sizeof(uint32_t) * tmp.max_ops);
  const size_t o_status = carve(off, 16);
  const size_t o_abort = carve(off, 16);
  const size_t o_x = carve(off, sizeof(float) * (size_t)N * D.d_model);
  const size_t o_proj = carve(off, sizeof(float) * (size_t)N * tmp.proj_stride);
  const size_t o_attn = carve(off, sizeof(float) * (size_t)N * tmp.attn_stride);
  const size_t o_hbuf = carve(off, sizeof(float) * (size_t)N * tmp.hbuf_stride);
  const size_t o_ssq = carve(off, sizeof(float) * (size_t)(2 * D.n_layers + 1) * tmp.n_sm * kMaxN);
  const size_t o_amax = carve(off, sizeof(float2) * (size_t)tmp.n_sm * kMaxN);
  size_t o_apart = 0, o_rope = 0;
  if (tmp.n_gqa) o_apart = carve(off, sizeof(float) * attn_part_records(&tmp, batch, rows) * tmp.attn_part_stride);
  if (tmp.rot_dim) o_rope = carve(off, sizeof(float2) * (size_t)D.max_ctx * (tmp.rot_dim / 2));
  tmp.counters = reinterpret_cast<uint32_t*>(base + o_counters);
  tmp.status = reinterpret_cast<int32_t*>(base + o_status);
  tmp.abort_flag = reinterpret_cast<int32_t*>(base + o_abort);
  tmp.x = reinterpret_cast<float*>(base + o_x);
  tmp.proj = reinterpret_cast<float*>(base + o_proj);
  tmp.attn_out = reinterpret_cast<float*>(base + o_attn);
  tmp.hbuf = reinterpret_cast<float*>(base + o_hbuf);
  tmp.ssq = reinterpret_cast<float*>(base + o_ssq);
  tmp.amax_part = reinterpret_cast<float2*>(base + o_amax);
  tmp.attn_part = tmp.n_gqa ? reinterpret_cast<float*>(base + o_apart) : nullptr;
  tmp.rope = tmp.rot_dim ? reinterpret_cast<float2*>(base + o_rope) : nullptr;
  tmp.kcache = static_cast<uint16_t*>(state->kcache);
  tmp.vcache = static_cast<uint16_t*>(state->vcache);
  tmp.state = state->state;
  tmp.pend = state->pending;
  tmp.seq = reinterpret_cast<SeqState*>(state->seq);
  tmp.epoch = state->epoch;

  const bool head = logits_out != nullptr || argmax_out != nullptr;
  if (!weights->packed) {
    fprintf(stderr, "mk_decode_step_static: mk_weights.packed is NULL (fill it once with mk_pack_weights)\n");
    return MK_ERR_INVALID_ARG;
  }
  tmp.pk.base = static_cast<const uint8_t*>(weights->packed);
  HostProgram hp;
  if ((st = construct_program(&tmp, batch, rows, head, hp)) != MK_OK) {
    fprintf(stderr, "mk_decode_step_static: %s\n", tmp.err.c_str());
    return st;
  }
  const size_t o_ops = carve(off, sizeof(OpDesc) * hp.ops.size());
  const size_t o_instr = carve(off, sizeof(Instr) * hp.flat.size());
  const size_t o_qoff = carve(off, sizeof(int32_t) * hp.qoff.size());
  if (off > (size_t)MK_STATIC_SCRATCH_BYTES) {
    fprintf(stderr,
            "mk_decode_step_static: this step needs %zu bytes of working memory, more than the %u-byte static "
            "array (use mk_create / mk_decode_step, or fewer rows per call)\n",
            off, (unsigned)MK_STATIC_SCRATCH_BYTES);
    return MK_ERR_UNSUPPORTED;
  }
  Program prog;
  prog.B = batch;
  prog.R = rows;
  prog.head = head;
  prog.d_ops = reinterpret_cast<OpDesc*>(base + o_ops);
  prog.d_instr = reinterpret_cast<Instr*>(base + o_instr);
  prog.d_qoff = reinterpret_cast<int32_t*>(base + o_qoff);
  prog.n_ops = (int)hp.ops.size();
  prog.n_instr = (int)hp.flat.size();
  for (const OpDesc& o : hp.ops) prog.use_tc = prog.use_tc || (o.type == OP_GEMV && o.mma == 2);

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((e = cudaMemcpyAsync(prog.d_ops, hp.ops.data(), sizeof(OpDesc) * hp.ops.size(), cudaMemcpyHostToDevice, s)) !=
          cudaSuccess ||
      (e = cudaMemcpyAsync(prog.d_instr, hp.flat.data(), sizeof(Instr) * hp.flat.size(), cudaMemcpyHostToDevice,
                           s)) != cudaSuccess ||
      (e = cudaMemcpyAsync(prog.d_qoff, hp.qoff.data(), sizeof(int32_t) * hp.qoff.size(), cudaMemcpyHostToDevice,
                           s)) != cudaSuccess ||
      (e = cudaMemsetAsync(tmp.counters, 0, sizeof(uint32_t) * tmp.max_ops, s)) != cudaSuccess ||
      (e = cudaMemsetAsync(tmp.status, 0, 16, s)) != cudaSuccess ||
      (e = cudaMemsetAsync(tmp.abort_flag, 0, 16, s)) != cudaSuccess) {
    fprintf(stderr, "mk_decode_step_static: %s\n", cudaGetErrorString(e));
    return MK_ERR_CUDA;
  }
  if (tmp.rot_dim) {
    std::lock_guard<std::mutex> lock(g_static_mu);
    StaticRope& rec = g_static_rope[tmp.device];
    const bool same = rec.valid && rec.offset == o_rope && rec.max_ctx == D.max_ctx && rec.rot_dim == tmp.rot_dim &&
                      rec.theta == D.rope_theta;
    if (!same) {
      rec.valid = false;
      if ((e = rope_table_launch(tmp.rope, D.max_ctx, tmp.rot_dim, (double)D.rope_theta, s)) != cudaSuccess) {
        fprintf(stderr, "mk_decode_step_static: %s\n", cudaGetErrorString(e));
        return MK_ERR_CUDA;
      }
      rec.valid = true;
      rec.offset = o_rope;
      rec.max_ctx = D.max_ctx;
      rec.rot_dim = tmp.rot_dim;
      rec.theta = D.rope_theta;
    }
  } else {
    std::lock_guard<std::mutex> lock(g_static_mu);
    g_static_rope[tmp.device].valid = false;  // this call's buffers may cover the recorded table
  }
  st = launch_program(&tmp, &prog, tokens, rows, positions, batch, rows, logits_out, argmax_out, false, s);
  state->epoch = tmp.epoch;
  if (st != MK_OK) {
    fprintf(stderr, "mk_decode_step_static: %s\n", tmp.err.c_str());
    return st;
  }
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return MK_ERR_CUDA;
  int32_t code = 0;
  if ((e = cudaMemcpy(&code, tmp.status, sizeof(int32_t), cudaMemcpyDeviceToHost)) != cudaSuccess) return MK_ERR_CUDA;
  return (mk_status)code;
}
