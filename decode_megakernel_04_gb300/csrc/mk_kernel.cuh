// Persistent decode megakernel for GB300 (sm_103a): one CTA per SM, one launch per decode step.
//
// Each CTA runs 8 consumer warps and 1 producer warp. The producer walks the SM's instruction queue
// ahead of the consumers and streams every weight tile (and every cached-KV block) that an instruction
// will read into a 4-slot shared-memory ring (32 KB of weights per slot) with bulk async copies (cp.async.bulk, completion on an
// mbarrier). Weights never depend on activations, so the producer runs across op and layer boundaries
// while the consumers wait on inter-SM dependency counters: the next op's weights are already arriving
// when its inputs become ready. This is the pages' central idea — a weight load is issued as early as
// on-chip storage allows, not when the op that uses it starts (Kimi K3's TPU megakernel, "What a
// megakernel is, and what it fixes on a TPU"; the cross-layer prefetch of Figure 4) — mapped onto the
// GPU's per-SM shared memory instead of the TPU's single VMEM pool.
//
// Every spin-wait is bounded by %globaltimer; on expiry the kernel records MK_ERR_TIMEOUT, raises an
// abort flag that every other wait also polls, drains its in-flight copies and returns.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <math_constants.h>
#include <float.h>
#include <stdint.h>

#include "mk_internal.h"

// This file is compiled twice (mk_kernel_dense.cu, mk_kernel_full.cu): MK_VARIANT_FULL = 0 leaves out the
// MLA and MoE handlers, so models without them get a kernel whose register allocation those handlers do
// not perturb; MK_VARIANT_NS names the namespace of each copy.
#ifndef MK_VARIANT_FULL
#error "define MK_VARIANT_FULL and MK_VARIANT_NS before including mk_kernel.cuh"
#endif

namespace mk {
namespace MK_VARIANT_NS {

constexpr bool kFull = MK_VARIANT_FULL != 0;

// Every op handler is compiled out of line: each gets its own register allocation within the kernel's
// 168-register budget (288 threads per CTA), and the kernel's main loop stops spilling (measured: the MoE /
// MLA stack runs 2x faster; the dense stack 17% faster at 8 rows and the same at 1 row).
#define MK_OUTLINE __noinline__
constexpr int kStatusTimeout = 5;
constexpr int kStatusDevice = 6;
constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------------------------------------------
// small device helpers
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* ptr) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}
__device__ __forceinline__ unsigned long long global_timer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ float bf2f(uint32_t h16) { return __uint_as_float(h16 << 16); }
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint16_t f2bf(float f) {
  __nv_bfloat16 b = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&b);
}
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* ptr) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add(uint32_t* ptr, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(ptr), "r"(v) : "memory");
}
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
}
// V independent warp sums, their butterfly rounds interleaved; every lane gets every total
template <int V>
__device__ __forceinline__ void warp_sum_n(float (&v)[V]) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
    for (int i = 0; i < V; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], o);
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float sigmoidf_(float z) { return 1.0f / (1.0f + expf(-z)); }

// --- mbarrier / bulk copy -------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// --- bounded waits --------------------------------------------------------------------------------
struct Spin {
  unsigned long long t0 = 0;
  uint32_t n = 0;
  // false = give up (abort raised elsewhere, or this wait timed out and raised it). The clock and the abort
  // flag are read every 64 polls, or on every poll when the limit is below a millisecond (spin_mask 0).
  __device__ __forceinline__ bool ok(const KParams& p) {
    if ((++n & p.spin_mask) != 0u) return true;
    if (*reinterpret_cast<volatile int32_t*>(p.abort_flag) != 0) return false;
    const unsigned long long now = global_timer();
    if (t0 == 0) {
      t0 = now;
      return true;
    }
    if (now - t0 > p.timeout_ns) {
      atomicCAS(p.status, 0, kStatusTimeout);
      atomicExch(p.abort_flag, 1);
      return false;
    }
    return true;
  }
};

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, const KParams& p) {
  Spin s;
  while (!mbar_try_wait(bar, parity)) {
    if (!s.ok(p)) return false;
  }
  return true;
}

__device__ __forceinline__ bool wait_counter(const uint32_t* ctr, uint32_t target, const KParams& p) {
  Spin s;
  while (ld_acquire(ctr) < target) {
    if (!s.ok(p)) return false;
    __nanosleep(20);
  }
  return true;
}

// ------------------------------------------------------------------------------------------------
// shared memory
// ------------------------------------------------------------------------------------------------
struct CSmem {
  float red[kConsumerWarps][64];
  float val[64];
  float sq[64];
  float inv_rms[kMaxN];
  float ssq_acc[kMaxN];
  float best_val[kMaxN];
  int32_t best_idx[kMaxN];
  int32_t flag;
  int32_t last;
  int32_t pad[2];
  float mred[2 * kConsumerWarps * 128];  // tensor-core GEMV: two buffers of 8 warps x 16 rows x 8 cols
  int32_t uni_c[kMaxExperts + 4];        // MoE: the step's expert union, consumers' copy (count, ids)
  int32_t uni_p[kMaxExperts + 4];        // the producer warp's copy of the union during an expert op
  // tcgen05 GEMV: staged-activation buffer ready [2] / free [2], accumulators complete, drain at exit
  uint64_t tcbar[6];
  uint32_t tmem_base;
  uint32_t tmem_pad;
};

struct Ring {
  uint8_t* base;
  uint64_t* full;
  uint64_t* empty;
  __device__ __forceinline__ uint8_t* slot_ptr(uint32_t chunk) const {
    return base + (chunk % kSlots) * kSlotBytes;
  }
};

// ring | activation / staging area (GEMV input rows; the attention block's own K/V rows; the delta rule's
// row inputs; the tcgen05 GEMV's two staged-activation buffers) | ring barriers | consumer scratch.
// Ring slots and the staging area start on 1024-byte boundaries (the 128-byte swizzle atom of the
// tcgen05 operands); an MMA that reads past a short tile at the end of the last slot stays inside the CTA's
// shared memory (in the staging area).
constexpr size_t kActOff = (size_t)kSlots * kSlotBytes;
constexpr size_t kBarOff = kActOff + kActBytes;
constexpr size_t kCSmemOff = kBarOff + 2 * kSlots * sizeof(uint64_t);
constexpr size_t kSmemBytes = kCSmemOff + sizeof(CSmem);
static_assert(kSlotBytes % 1024 == 0 && kActOff % 1024 == 0, "ring slots and staging area must be 1024-byte aligned");
static_assert(2 * kTcBBytes <= kActBytes, "two staged-activation buffers must fit the staging area");
// 227 KB per CTA, less the 1 KB of static shared memory the kernel also uses (the 1024-byte alignment of
// the dynamic array and the launch-state word)
static_assert(kSmemBytes + 1024 <= 232448, "dynamic shared memory above what a CTA may use");
static_assert(kActBytes % 128 == 0, "staging area must keep 128-byte alignment");

// consumer side of one ring chunk
__device__ __forceinline__ bool ring_wait_full(const Ring& rg, uint32_t chunk, const KParams& p) {
  return wait_bar(&rg.full[chunk % kSlots], (chunk / kSlots) & 1u, p);
}
__device__ __forceinline__ void ring_release(const Ring& rg, uint32_t chunk, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(&rg.empty[chunk % kSlots]);
}

// producer side: wait until the slot of `chunk` is free, arm its full barrier with `bytes`
__device__ __forceinline__ bool ring_acquire(const Ring& rg, uint32_t chunk, uint32_t bytes, const KParams& p,
                                             int lane) {
  int ok = 1;
  if (lane == 0) {
    const uint32_t k = chunk / kSlots;
    if (k > 0) ok = wait_bar(&rg.empty[chunk % kSlots], (k - 1) & 1u, p) ? 1 : 0;
    if (ok) mbar_arrive_expect_tx(&rg.full[chunk % kSlots], bytes);
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  return ok != 0;
}

// RMSNorm partials: sum of squares of activation row n over the columns SM `sm` owns, for norm point `slot`;
// laid out [slot][row][SM] so the 32 lanes reading one row's partials read consecutive words
__device__ __forceinline__ size_t ssq_index(const KParams& p, int slot, int n, int sm) {
  return ((size_t)slot * kMaxN + n) * p.n_sm + sm;
}

// ------------------------------------------------------------------------------------------------
// cross-lane reduction of V independent partial sums (V = 16, 32 or 64)
// After the call lane L holds, in v[0 .. F-1] with F = max(V/32, 1), the warp totals of indices
// [L*F, L*F + F) when V >= 32, or of index L / (32/V) when V < 32.
// ------------------------------------------------------------------------------------------------
template <int C, int O>
struct MultiReduce {
  static __device__ __forceinline__ void run(float* v, int lane) {
    if constexpr (O == 0) {
      return;
    } else if constexpr (C > 1) {
      const bool upper = (lane & O) != 0;
#pragma unroll
      for (int i = 0; i < C / 2; ++i) {
        const float send = upper ? v[i] : v[i + C / 2];
        const float keep = upper ? v[i + C / 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
      }
      MultiReduce<C / 2, O / 2>::run(v, lane);
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
      MultiReduce<1, O / 2>::run(v, lane);
    }
  }
};

// block-wide: totals of V values land in cs.val[0..V-1]
template <int V>
__device__ __forceinline__ void block_reduce(float* v, CSmem& cs, int warp, int lane, int ctid) {
  MultiReduce<V, 16>::run(v, lane);
  if constexpr (V >= 32) {
    constexpr int F = V / 32;
#pragma unroll
    for (int f = 0; f < F; ++f) cs.red[warp][lane * F + f] = v[f];
  } else {
    constexpr int S = 32 / V;
    if (lane % S == 0) cs.red[warp][lane / S] = v[0];
  }
  consumer_sync();
  if (ctid < V) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) t += cs.red[w][ctid];
    cs.val[ctid] = t;
  }
  consumer_sync();
}

// ------------------------------------------------------------------------------------------------
// GEMV: out rows [a, b) of  act(in) @ W^T, over the packed row blocks of the weights (mma.sync for up to
// 4 activation rows, tcgen05 otherwise). The routed-expert GEMVs (MoE) stream plain weight rows instead.
// ------------------------------------------------------------------------------------------------
// A packed row block of a GEMV instruction: logical rows [start, end), rounded up to whole 8-row runs; P
// physical rows per atom (SwiGLU: gate rows, then up rows); atoms per ring chunk (at most 32 KB).
struct PkBlock {
  int rows;   // logical rows
  int rows8;  // rows rounded up to 8
  int P;      // physical rows per atom: rows8, or 2 rows8 for SwiGLU
  int atoms;  // atoms per ring chunk
};

// the row block that starts at logical row `start` of an instruction ending at `end`; returns its end
__device__ __forceinline__ int pk_block(const OpDesc& op, int start, int end, PkBlock& blk) {
  const int sw = op.out_kind == OUT_SWIGLU ? 1 : 0;
  const int e = min(end, start + pk_block_lrows(sw));
  blk.rows = e - start;
  blk.rows8 = (blk.rows + 7) & ~7;
  blk.P = blk.rows8 << sw;
  blk.atoms = max(1, 256 / blk.P);
  return e;
}
// the block's first byte in the packed copy: every earlier logical row takes patoms x 128 bytes (x 2 for
// SwiGLU); plus the op's first atom
__device__ __forceinline__ const uint8_t* pk_block_src(const OpDesc& op, int start, const PkBlock& blk) {
  const size_t per_row = (size_t)op.patoms * 128 * (op.out_kind == OUT_SWIGLU ? 2 : 1);
  return op.wp + (size_t)start * per_row + (size_t)op.pa0 * blk.P * 128;
}

// K stacking of a tcgen05 block: with P <= 64 physical rows, one M = 128 MMA reads s = 128 / P consecutive
// atoms of the block (atom a + q lands in TMEM lanes q*P ..), and an N = 16 s operand reads the activations of
// the same s atoms (columns 16 q ..): the diagonal blocks (lanes q*P + r, columns 16 q ..) are row r's partial
// sums over atom a + q, the rest is discarded. This takes s atoms per MMA instead of one. Used for
// non-SwiGLU ops with 16 activation columns (up to 8 rows), at most 4 segments.
__device__ __forceinline__ int tc_stack(const OpDesc& op, const PkBlock& blk) {
  if (op.out_kind == OUT_SWIGLU || op.ncols != 16) return 1;
  return max(1, min(min(4, 128 / blk.P), (op.K + 63) >> 6));
}

// end of the tcgen05 row group that starts at `start`: as many blocks as fit the TMEM columns (a block takes
// ncols per tile, times its K-stacking factor)
__device__ __forceinline__ int tc_group_end(const OpDesc& op, int start, int end) {
  const int tiles = op.out_kind == OUT_SWIGLU ? 2 : 1;
  int cols = 0, r = start;
  while (r < end) {
    PkBlock blk;
    const int e = pk_block(op, r, end, blk);
    const int c = tiles * op.ncols * tc_stack(op, blk);
    if (r > start && cols + c > kTcCols) break;
    cols += c;
    r = e;
  }
  return r;
}

__device__ __forceinline__ int tc_atoms(const OpDesc& op) { return (op.K + 63) >> 6; }
__device__ __forceinline__ int tc_part(const OpDesc& op) { return 256 / op.ncols; }

// ring chunks of one tcgen05 instruction (every consumer thread advances its chunk counter by this)
__device__ __forceinline__ uint32_t tc_instr_chunks(const OpDesc& op, const Instr& in) {
  const int nat = tc_atoms(op), KP = tc_part(op);
  uint32_t n = 0;
  for (int r = in.a; r < in.b;) {
    PkBlock blk;
    r = pk_block(op, r, in.b, blk);
    for (int a0 = 0; a0 < nat; a0 += KP) {
      const int a1 = min(nat, a0 + KP);
      n += (uint32_t)((a1 - a0 + blk.atoms - 1) / blk.atoms);
    }
  }
  return n;
}

// Row groups of an expert GEMV instruction: its rows are split into ceil(n / glog) groups of near-equal size (so no
// group is left with a few rows and tiny chunks), and each group's K range into slices of KC inputs.
__device__ __forceinline__ int gemv_ngroups(int n, int glog) { return (n + glog - 1) / glog; }
__device__ __forceinline__ int gemv_group_row(int r0, int n, int ng, int g) {
  return r0 + (int)((long long)g * n / ng);
}



template <int CPL>
__device__ __forceinline__ void load_f32(const float* src, float (&dst)[CPL]) {
#pragma unroll
  for (int c = 0; c < CPL; c += 4) {
    const float4 v = __ldcg(reinterpret_cast<const float4*>(src + c));
    dst[c] = v.x;
    dst[c + 1] = v.y;
    dst[c + 2] = v.z;
    dst[c + 3] = v.w;
  }
}

template <int CPL>
__device__ __forceinline__ void load_bf16_row(const uint8_t* src, float (&dst)[CPL]) {
  if constexpr (CPL == 8) {
    const uint4 w = *reinterpret_cast<const uint4*>(src);
    dst[0] = bf_lo(w.x); dst[1] = bf_hi(w.x); dst[2] = bf_lo(w.y); dst[3] = bf_hi(w.y);
    dst[4] = bf_lo(w.z); dst[5] = bf_hi(w.z); dst[6] = bf_lo(w.w); dst[7] = bf_hi(w.w);
  } else {
    const uint2 w = *reinterpret_cast<const uint2*>(src);
    dst[0] = bf_lo(w.x); dst[1] = bf_hi(w.x); dst[2] = bf_lo(w.y); dst[3] = bf_hi(w.y);
  }
}

template <int CPL>
__device__ __forceinline__ void load_bf16_global(const uint16_t* src, float (&dst)[CPL]) {
  if constexpr (CPL == 8) {
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(src));
    dst[0] = bf_lo(w.x); dst[1] = bf_hi(w.x); dst[2] = bf_lo(w.y); dst[3] = bf_hi(w.y);
    dst[4] = bf_lo(w.z); dst[5] = bf_hi(w.z); dst[6] = bf_lo(w.w); dst[7] = bf_hi(w.w);
  } else {
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(src));
    dst[0] = bf_lo(w.x); dst[1] = bf_hi(w.x); dst[2] = bf_lo(w.y); dst[3] = bf_hi(w.y);
  }
}

// ------------------------------------------------------------------------------------------------
// Tensor-core GEMV for up to 4 activation rows (mma.sync m16n8k16, bf16 x bf16 -> fp32).
// A = a 16-row weight group straight from the ring (ldmatrix; rows padded by 16 bytes in the slot so the
// eight rows of an 8x8 matrix fall in distinct banks). B = the activations, staged once per instruction
// as a bf16 "hi" and a bf16 "lo" part (hi = bf16(v), lo = bf16(v - hi)), so the pair carries ~16
// mantissa bits and the product keeps fp32-level accuracy: columns 0..3 of the n8 tile are hi of rows
// 0..3, columns 4..7 lo of rows 0..3. Warps split the 16-wide k steps of a chunk; one cross-warp
// reduction (one barrier) per row group.
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 1/rms of activation rows n = warp, warp + 8, .. from the per-SM partial sums of squares of norm point `slot`
// (sum over `width` columns): every partial of a row is loaded at once (8 per lane), so this costs one L2 round
// trip. Writes cs.inv_rms; the caller synchronises.
__device__ __forceinline__ void inv_rms_rows(const KParams& p, int slot, int width, CSmem& cs, int warp, int lane,
                                             int nwarps = kConsumerWarps) {
  for (int n = warp; n < p.N; n += nwarps) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int q = lane + 32 * i;
      v[i] = q < p.n_sm ? __ldcg(&p.ssq[ssq_index(p, slot, n, q)]) : 0.f;
    }
    float s = ((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7]));
    s = warp_sum(s);
    if (lane == 0) cs.inv_rms[n] = rsqrtf(s / (float)width + p.eps);
  }
}

// hi/lo bf16 columns of the staged activations: slot n (n < N) = hi of row n, slot N + n = lo of row n,
// each Kp + 8 elements long (Kp = K rounded up to whole atoms, zeros past K; the 8 pad elements put
// successive slots in different banks). With RMSNorm the 1/rms of each row is computed while the first round
// of input loads is in flight. Loads go out in rounds of kBatch = 4 per thread: deeper rounds (8 to 20 loads in
// flight) measured slower at batch 1 although they need fewer round trips; the unrolled code of a deep round,
// run once per instruction, cost more than the round trips it saved.
template <int kBatch, bool norm>  // kBatch: loads in flight per thread before any of them is converted
__device__ __forceinline__ void stage_hilo(const KParams& p, const OpDesc& op, CSmem& cs, uint16_t* cols, int ctid) {
  const int K = op.K, N = p.N, Kp = tc_atoms(op) * 64, cp = Kp + 8;
  const int total4 = N * Kp / 4;
  const int rounds = (total4 + kConsumerThreads * kBatch - 1) / (kConsumerThreads * kBatch);
  // item i = 4 consecutive inputs of activation row n at column k (N <= 4: no division)
  auto load = [&](int rd, float4 (&v)[kBatch], uint2 (&g)[kBatch]) {
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = rd * kConsumerThreads * kBatch + ctid + u * kConsumerThreads;
      v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      g[u] = make_uint2(0u, 0u);
      if (i < total4) {
        const int e = i * 4;
        const int n = (e >= Kp) + (e >= 2 * Kp) + (e >= 3 * Kp), k = e - n * Kp;
        if (k < K) {
          const float* src =
              norm ? p.x + (size_t)n * p.d + op.k_begin + k : op.in + (size_t)n * op.in_stride + op.k_begin + k;
          v[u] = __ldcg(reinterpret_cast<const float4*>(src));
          if (norm) g[u] = __ldg(reinterpret_cast<const uint2*>(op.gain + op.k_begin + k));
        }
      }
    }
  };
  float4 v[kBatch];
  uint2 g[kBatch];
  load(0, v, g);
  if (norm) {
    inv_rms_rows(p, op.ssq_in, op.ldw, cs, ctid >> 5, ctid & 31);
    consumer_sync();
  }
  // the loads of round rd + 1 are in flight while round rd is converted
#pragma unroll 1
  for (int rd = 0; rd < rounds; ++rd) {
    float4 w[kBatch];
    uint2 h[kBatch];
    load(rd + 1, w, h);
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = rd * kConsumerThreads * kBatch + ctid + u * kConsumerThreads;
      if (i >= total4) break;
      const int e = i * 4;
      const int n = (e >= Kp) + (e >= 2 * Kp) + (e >= 3 * Kp), k = e - n * Kp;
      float4 x = v[u];
      if (norm) {
        const float s = cs.inv_rms[n];
        x.x *= s * bf_lo(g[u].x);
        x.y *= s * bf_hi(g[u].x);
        x.z *= s * bf_lo(g[u].y);
        x.w *= s * bf_hi(g[u].y);
      }
      const float f[4] = {x.x, x.y, x.z, x.w};
      uint16_t hi[4], lo[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        hi[j] = f2bf(f[j]);
        lo[j] = f2bf(f[j] - bf2f(hi[j]));
      }
      *reinterpret_cast<uint2*>(cols + (size_t)n * cp + k) =
          make_uint2(hi[0] | ((uint32_t)hi[1] << 16), hi[2] | ((uint32_t)hi[3] << 16));
      *reinterpret_cast<uint2*>(cols + (size_t)(N + n) * cp + k) =
          make_uint2(lo[0] | ((uint32_t)lo[1] << 16), lo[2] | ((uint32_t)lo[3] << 16));
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      v[u] = w[u];
      g[u] = h[u];
    }
  }
}

// one m16n8k16 step of the mma.sync GEMV: A = 16 packed weight rows of one atom (ldmatrix through the
// 128-byte swizzle), B = this lane's hi / lo activation column
__device__ __forceinline__ void mma_kstep(float (&acc)[4], uint32_t arow, int rx, int lhi, int ks, uint32_t atom_bytes,
                                          const uint16_t* bcol, int kbase, bool bvalid) {
  const int a = ks >> 2, j = ks & 3;
  uint32_t a0, a1, a2, a3;
  ldmatrix_x4(arow + (uint32_t)a * atom_bytes + (uint32_t)(((2 * j + lhi) ^ rx) << 4), a0, a1, a2, a3);
  uint32_t b0 = 0, b1 = 0;
  if (bvalid) {
    const uint16_t* bp = bcol + kbase + ks * 16;
    b0 = *reinterpret_cast<const uint32_t*>(bp);
    b1 = *reinterpret_cast<const uint32_t*>(bp + 8);
  }
  mma_bf16_16816(acc, a0, a1, a2, a3, b0, b1);
}

// GEMV of up to 4 activation rows on mma.sync over packed row blocks. A block's P physical rows form
// G16 = ceil(P / 16) m16 tiles; the 8 warps are split into G16 tiles x (8 / G16) K phases, each warp
// accumulating its tile over every (8 / G16)-th k-step of each chunk, so a block needs one cross-warp sum.
__device__ __noinline__ void gemv_mma_consume(const KParams& p, const OpDesc& op, const Instr& in, const Ring& rg, uint32_t& chunk,
                                 CSmem& cs, float* act, int ctid) {
  const int warp = ctid >> 5, lane = ctid & 31;
  const int sm = blockIdx.x;
  const bool swiglu = op.out_kind == OUT_SWIGLU;
  const bool norm = op.in_kind == IN_NORM;
  const int N = p.N, nat = tc_atoms(op);
  const int cpitch = nat * 64 + 8;
  uint16_t* cols = reinterpret_cast<uint16_t*>(act);
  // the residual slice follows the staged columns
  float* xres = act + (2 * N * cpitch + 1) / 2 + 4;

  // a residual add also stages this SM's slice of x: its first 2 x 256 values load with the inputs' first round
  const int nrows = in.b - in.a;
  const int nx = op.out_kind == OUT_RESID ? N * nrows : 0;
  float xr[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int i = ctid + u * kConsumerThreads;
    xr[u] = i < nx ? __ldcg(p.x + (size_t)(i / nrows) * p.d + in.a + i % nrows) : 0.f;
  }
  if (in.b > in.a) {
    if (norm) stage_hilo<4, true>(p, op, cs, cols, ctid);
    else stage_hilo<4, false>(p, op, cs, cols, ctid);
  }
#pragma unroll
  for (int u = 0; u < 2; ++u)
    if (ctid + u * kConsumerThreads < nx) xres[ctid + u * kConsumerThreads] = xr[u];
  for (int i = ctid + 2 * kConsumerThreads; i < nx; i += kConsumerThreads)
    xres[i] = __ldcg(p.x + (size_t)(i / nrows) * p.d + in.a + i % nrows);
  consumer_sync();

  // this lane's B column: hi of row g, lo of row g - 4, or zero
  const int g = lane >> 2, t = lane & 3;
  const int bslot = (g < N) ? g : ((g >= 4 && g - 4 < N) ? N + (g - 4) : -1);
  const uint16_t* bcol = cols + (size_t)(bslot < 0 ? 0 : bslot) * cpitch + 2 * t;
  // ldmatrix: this lane addresses tile row (lane & 7) + 8 ((lane >> 3) & 1), 16-byte piece parity lane >> 4
  const int lrow = (lane & 7) + ((lane >> 3) & 1) * 8, lhi = lane >> 4;
  const uint32_t ring_s = smem_u32(rg.base);

  // epilogue state: thread ctid serves activation row n = ctid & 3 for logical rows (ctid >> 2) + 64 j
  const int en = ctid & 3;
  float best_v = -CUDART_INF_F, ssq_acc = 0.f;
  int best_i = 0x7fffffff;

  int bno = 0;
  for (int r = in.a; r < in.b; ++bno) {
    PkBlock blk;
    const int r0 = r;
    r = pk_block(op, r, in.b, blk);
    // m16 tiles of the block: up to 8 take one warp each (or 8 / G16 warps splitting the K steps); 9 to 16
    // (SwiGLU blocks over 64 rows) take two per warp, tiles w and w + 8
    const int G16 = (blk.P + 15) >> 4;
    const bool two = G16 > kConsumerWarps;
    const int np = two ? 1 : kConsumerWarps / G16;
    const int tile = two ? warp : warp % G16, ph = two ? 0 : warp / G16;
    const bool active = ph < np, active2 = two && warp + kConsumerWarps < G16;
    // rows past the block's last physical row read that row again (their sums are never used), so the tile
    // never reaches past the chunk
    const int prow = min(tile * 16 + lrow, blk.P - 1);
    const int prow2 = min((tile + kConsumerWarps) * 16 + lrow, blk.P - 1);
    const int rx = prow & 7, rx2 = prow2 & 7;
    const uint32_t atom_bytes = (uint32_t)blk.P * 128u;
    float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
    for (int c0 = 0; c0 < nat; c0 += blk.atoms) {
      const int na = min(blk.atoms, nat - c0);
      ring_wait_full(rg, chunk, p);
      if (active) {
        const uint32_t sbase = ring_s + (chunk % kSlots) * kSlotBytes;
        const uint32_t arow = sbase + (uint32_t)prow * 128u;
        const int nks = 4 * na, kbase = c0 * 64;
        if (two) {
          const uint32_t arow2 = sbase + (uint32_t)prow2 * 128u;
          for (int ks = 0; ks < nks; ++ks) {
            mma_kstep(acc0, arow, rx, lhi, ks, atom_bytes, bcol, kbase, bslot >= 0);
            if (active2) mma_kstep(acc1, arow2, rx2, lhi, ks, atom_bytes, bcol, kbase, bslot >= 0);
          }
        } else {
          int ks = ph;
          for (; ks + np < nks; ks += 2 * np) {
            mma_kstep(acc0, arow, rx, lhi, ks, atom_bytes, bcol, kbase, bslot >= 0);
            mma_kstep(acc1, arow, rx, lhi, ks + np, atom_bytes, bcol, kbase, bslot >= 0);
          }
          if (ks < nks) mma_kstep(acc0, arow, rx, lhi, ks, atom_bytes, bcol, kbase, bslot >= 0);
        }
      }
      ring_release(rg, chunk, lane);
      ++chunk;
    }
    // cross-warp sum: red[buf][warp][row][col] (two tiles a warp: red[tile][row][col] over both buffers);
    // fragment c0/c1 = (row g, cols 2t, 2t+1), c2/c3 = row g+8
    if (two) consumer_sync();  // the whole buffer is rewritten: the previous block's epilogue must be done
    auto put = [&](float* rb, const float (&x)[4], const float (&y)[4]) {
      rb[g * 8 + 2 * t] = x[0] + y[0];
      rb[g * 8 + 2 * t + 1] = x[1] + y[1];
      rb[(g + 8) * 8 + 2 * t] = x[2] + y[2];
      rb[(g + 8) * 8 + 2 * t + 1] = x[3] + y[3];
    };
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
    if (two) {
      if (active) put(cs.mred + tile * 128, acc0, zero4);
      if (active2) put(cs.mred + (tile + kConsumerWarps) * 128, acc1, zero4);
    } else if (active) {
      put(cs.mred + (bno & 1) * (kConsumerWarps * 128) + warp * 128, acc0, acc1);
    }
    consumer_sync();
    const float* rr = two ? cs.mred : cs.mred + (bno & 1) * (kConsumerWarps * 128);
    // physical row pr, activation row n: the hi and lo columns of every K phase of pr's tile
    auto rowval = [&](int pr, int n) -> float {
      const int tl = pr >> 4, i = pr & 15;
      float v = 0.f;
      for (int q = 0; q < np; ++q) v += rr[(q * G16 + tl) * 128 + i * 8 + n] + rr[(q * G16 + tl) * 128 + i * 8 + 4 + n];
      return v;
    };
    if (en < N) {
      for (int i = ctid >> 2; i < blk.rows; i += kConsumerThreads / 4) {
        const int row = r0 + i;
        if (swiglu) {
          const float gv = rowval(i, en), uv = rowval(blk.rows8 + i, en);
          op.out[(size_t)en * op.out_stride + row] = gv / (1.0f + expf(-gv)) * uv;
        } else {
          const float val = rowval(i, en);
          if (op.out_kind == OUT_STORE) {
            op.out[(size_t)en * op.out_stride + row] = val;
          } else if (op.out_kind == OUT_RESID) {
            const float xn = xres[en * nrows + (row - in.a)] + val;
            __stcg(p.x + (size_t)en * p.d + row, xn);
            ssq_acc += xn * xn;
          } else {
            if (p.logits) p.logits[(size_t)en * p.V + row] = val;
            if (val > best_v) { best_v = val; best_i = row; }
          }
        }
      }
    }
    // the other buffer is rewritten two blocks later, after the next block's barrier
    if (two) consumer_sync();
  }
  if (op.out_kind == OUT_RESID || op.out_kind == OUT_LOGITS) {
    // reduce the per-thread state over the threads of each activation row: lanes sharing (lane & 3), then warps
    if (op.out_kind == OUT_RESID) {
      for (int o = 4; o <= 16; o <<= 1) ssq_acc += __shfl_xor_sync(0xffffffffu, ssq_acc, o);
    } else {
      for (int o = 4; o <= 16; o <<= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best_v, o);
        const int oi = __shfl_xor_sync(0xffffffffu, best_i, o);
        if (ov > best_v || (ov == best_v && oi < best_i)) { best_v = ov; best_i = oi; }
      }
    }
    // (cs.red is not used earlier in this instruction, so each warp writes its row without a barrier)
    if (lane < 4) {
      cs.red[warp][lane] = op.out_kind == OUT_RESID ? ssq_acc : best_v;
      cs.red[warp][4 + lane] = __int_as_float(best_i);
    }
    consumer_sync();
    if (ctid < N) {
      if (op.out_kind == OUT_RESID) {
        float s2 = 0.f;
        for (int w = 0; w < kConsumerWarps; ++w) s2 += cs.red[w][ctid];
        if (op.ssq_out >= 0) __stcg(&p.ssq[ssq_index(p, op.ssq_out, ctid, sm)], s2);
      } else {
        float bv = -CUDART_INF_F;
        int bi = 0x7fffffff;
        for (int w = 0; w < kConsumerWarps; ++w) {
          const float v = cs.red[w][ctid];
          const int ix = __float_as_int(cs.red[w][4 + ctid]);
          if (v > bv || (v == bv && ix < bi)) { bv = v; bi = ix; }
        }
        p.amax_part[(size_t)sm * kMaxN + ctid] = make_float2(bv, __int_as_float(bi));
      }
    }
    // the instruction's last writes are warp 0's (N <= 4): ordered before its lane 0's completion signal, which
    // therefore needs no block barrier after this handler
    if (warp == 0) __syncwarp();
  }
}

// ------------------------------------------------------------------------------------------------
// Tensor-core GEMV for 5 to 64 activation rows: tcgen05.mma (kind::f16, bf16 x bf16 -> fp32) with the
// accumulators in tensor memory (TMEM). The weight rows are the M side of the MMA (128 TMEM lanes), the
// activations the N side, split into a bf16 "hi" and "lo" column each (hi = bf16(v), lo = bf16(v - hi)) so
// the product keeps ~16 mantissa bits of the fp32 activations; column 2n + 1 is added to column 2n at the end.
//   * Weight tiles come from the ring: packed row blocks (at most 128 logical rows; SwiGLU: 128 gate rows then
//     128 up rows), stored atom by atom in the canonical K-major 128-byte-swizzle layout the MMA
//     reads directly, one contiguous bulk copy per chunk. One 128-row MMA per 16-input step covers a block
//     (rows past its end read whatever follows and land in TMEM lanes that are never read), and the block
//     accumulates in one TMEM tile of ncols columns (lane i = the block's row i; SwiGLU: a gate and an up
//     tile). One row group (as many blocks as fit 512 columns) keeps all its accumulators in TMEM across the
//     whole K loop, so no cross-warp reduction is needed.
//   * K is covered in parts of 256 / ncols atoms (64 inputs each); the activations of a part are staged by
//     warps 1..7 into one of two 32 KB buffers while lane 0 of warp 0 issues the MMAs of the previous part.
// ------------------------------------------------------------------------------------------------
// --- tcgen05 primitives ---------------------------------------------------------------------
// shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 bytes apart
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// instruction descriptor: D fp32, A and B bf16, both K-major, M = 128, N = ncols
__device__ __forceinline__ uint32_t umma_idesc(int ncols) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(ncols >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive_n(uint64_t* bar, uint32_t n) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(n) : "memory");
}
// 8 consecutive fp32 TMEM columns of this warp's 32 lanes
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// Activations of atoms [a0, a1) as bf16 hi / lo rows (row 2n = hi of activation row n, 2n + 1 = lo; rows
// from 2N to ncols are zero) in the swizzled K-major layout: atom a at buf + (a - a0) * ncols * 128, row r at
// + r * 128, its 16-byte chunk c at + ((c ^ (r & 7)) << 4). Warps 1..7 do this; inputs past K are zero.
// With rms = true (the first K part of an instruction that normalises its input) the staging warps also compute
// 1/rms of every row from the RMS partials while their first loads are in flight, and meet at a barrier of their
// own before converting.
// With ok = false (this warp's wait for the buffer gave up) nothing is staged, but the rms barrier is still
// met, so the staging warps never wait on one another without a limit.
__device__ __forceinline__ void tc_stage(const KParams& p, const OpDesc& op, CSmem& cs, uint8_t* buf, int a0,
                                         int a1, int stid, int nthr, bool rms, bool ok) {
  constexpr int kBatch = 3;  // items whose loads are all in flight before any of them is converted (2 to 8 measured)
  const bool norm = op.in_kind == IN_NORM;
  const int N = p.N, K = op.K, nc = op.ncols;
  const int pairs = nc >> 1;                 // activation rows incl. the zero padding
  const int na = a1 - a0;
  const int items = ok ? pairs * na * 8 : 0;  // (activation row, atom, 16-byte chunk)
  const int rounds = max(rms ? 1 : 0, (items + nthr * kBatch - 1) / (nthr * kBatch));
  for (int rd = 0; rd < rounds; ++rd) {
    const int it0 = rd * nthr * kBatch + stid;
    float4 x0[kBatch], x1[kBatch];
    uint4 g[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int it = it0 + u * nthr;
      const int c = it & 7, rest = it >> 3;
      const int a = a0 + rest % na, n = rest / na;
      const int k = a * 64 + c * 8;
      x0[u] = x1[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      g[u] = make_uint4(0u, 0u, 0u, 0u);
      if (it < items && n < N && k < K) {
        const float* src = norm ? p.x + (size_t)n * p.d + k : op.in + (size_t)n * op.in_stride + k;
        x0[u] = __ldcg(reinterpret_cast<const float4*>(src));
        x1[u] = __ldcg(reinterpret_cast<const float4*>(src + 4));
        if (norm) g[u] = __ldg(reinterpret_cast<const uint4*>(op.gain + k));
      }
    }
    if (rms && rd == 0) {
      inv_rms_rows(p, op.ssq_in, op.ldw, cs, stid >> 5, stid & 31, nthr >> 5);
      asm volatile("bar.sync 2, %0;" ::"r"(nthr) : "memory");  // the staging warps only
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int it = it0 + u * nthr;
      if (it >= items) break;
      const int c = it & 7, rest = it >> 3;
      const int a = a0 + rest % na, n = rest / na;
      float v[8] = {x0[u].x, x0[u].y, x0[u].z, x0[u].w, x1[u].x, x1[u].y, x1[u].z, x1[u].w};
      if (norm && n < N) {
        const float s = cs.inv_rms[n];
        v[0] *= s * bf_lo(g[u].x); v[1] *= s * bf_hi(g[u].x); v[2] *= s * bf_lo(g[u].y); v[3] *= s * bf_hi(g[u].y);
        v[4] *= s * bf_lo(g[u].z); v[5] *= s * bf_hi(g[u].z); v[6] *= s * bf_lo(g[u].w); v[7] *= s * bf_hi(g[u].w);
      }
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint16_t h0 = f2bf(v[2 * e]), h1 = f2bf(v[2 * e + 1]);
        const uint16_t l0 = f2bf(v[2 * e] - bf2f(h0)), l1 = f2bf(v[2 * e + 1] - bf2f(h1));
        hi[e] = h0 | ((uint32_t)h1 << 16);
        lo[e] = l0 | ((uint32_t)l1 << 16);
      }
      uint8_t* atom = buf + (size_t)(a - a0) * nc * 128;
      const int rh = 2 * n, rl = 2 * n + 1;
      *reinterpret_cast<uint4*>(atom + rh * 128 + ((c ^ (rh & 7)) << 4)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(atom + rl * 128 + ((c ^ (rl & 7)) << 4)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
  }
}

// per-CTA state of the tcgen05 path: TMEM base, barriers, running counters (uniform over consumer threads)
struct TcState {
  uint32_t tmem;
  uint32_t kp;   // K parts processed since launch (buffer = kp & 1)
  uint32_t rg;   // row groups completed since launch (accumulator barrier parity)
};

__device__ __noinline__ void gemv_tc_consume(const KParams& p, const OpDesc& op, const Instr& in, const Ring& rg, uint32_t& chunk,
                                CSmem& cs, uint8_t* act, TcState& ts, unsigned long long* tr, int ctid) {
  const int warp = ctid >> 5, lane = ctid & 31;
  const int sm = blockIdx.x;
  const int N = p.N, nc = op.ncols;
  const bool norm = op.in_kind == IN_NORM;
  const bool swiglu = op.out_kind == OUT_SWIGLU;
  const int nat = tc_atoms(op), KP = tc_part(op);
  uint64_t* bready = &cs.tcbar[0];
  uint64_t* bfree = &cs.tcbar[2];
  uint64_t* accb = &cs.tcbar[4];
  float* pred = &cs.red[0][0];                                 // [8 warps][64]: ssq or argmax value partials
  int32_t* pidx = reinterpret_cast<int32_t*>(cs.mred);         // [8 warps][64]: argmax index partials

  for (int i = ctid; i < kConsumerWarps * 64; i += kConsumerThreads) {
    pred[i] = op.out_kind == OUT_LOGITS ? -CUDART_INF_F : 0.f;
    pidx[i] = 0x7fffffff;
  }
  consumer_sync();

  const uint32_t idesc = umma_idesc(nc);
  const uint32_t ring_s = smem_u32(rg.base);
  uint32_t ck = chunk;  // ring position of the MMA thread
  const int nkp = (nat + KP - 1) / KP;  // K parts per row group
  for (int g0 = in.a; g0 < in.b;) {
    const int g1 = tc_group_end(op, g0, in.b);
    const uint32_t kp0 = ts.kp;
    if (warp >= 1) {
      for (int i = 0; i < nkp; ++i) {
        const int a0 = i * KP, a1 = min(nat, a0 + KP);
        const uint32_t buf = (kp0 + i) & 1u, use = (kp0 + i) >> 1;
        uint8_t* bb = act + buf * kTcBBytes;
        bool ok = true;
        if (use > 0) ok = wait_bar(&bfree[buf], (use - 1) & 1u, p);
        tc_stage(p, op, cs, bb, a0, a1, ctid - 32, kConsumerThreads - 32, norm && g0 == in.a && a0 == 0, ok);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive(&bready[buf]);
        if (tr && ctid == 32) tr[8] = global_timer();
      }
    } else {
      // Lane 0 alone walks every K part and chunk of the row group and issues the MMAs; lanes 1..31 wait at the
      // warp barrier below. Entering and leaving a one-lane branch per chunk cost ~300 cycles each time (the
      // MMA stream stalls while the warp reconverges), and lanes left free to run ahead would spin on the
      // accumulator barrier and take the issuing lane's cycles. Descriptors are built once per chunk and
      // stepped by constants (the start address sits in the low bits, in 16-byte units).
      if (lane == 0) {
        const int tiles = swiglu ? 2 : 1;
        for (int i = 0; i < nkp; ++i) {
          const int a0 = i * KP, a1 = min(nat, a0 + KP);
          const uint32_t buf = (kp0 + i) & 1u, use = (kp0 + i) >> 1;
          const bool bok = wait_bar(&bready[buf], use & 1u, p);
          if (tr && g0 == in.a && a0 == 0) tr[5] = global_timer();
          const uint64_t bd0 = umma_desc(smem_u32(act + buf * kTcBBytes));
          const uint64_t b_atom = (uint64_t)((nc * 128) >> 4);
          int col = 0;
          for (int r = g0; r < g1;) {
            PkBlock blk;
            r = pk_block(op, r, g1, blk);
            const uint64_t a_atom = (uint64_t)((blk.P * 128) >> 4);
            const uint64_t a_up = (uint64_t)((blk.rows8 * 128) >> 4);  // SwiGLU: the up rows follow the gate rows
            const uint32_t dg = ts.tmem + (uint32_t)col, du = dg + (uint32_t)nc;
            const int st = tc_stack(op, blk);
            const uint32_t idesc_st = umma_idesc(nc * st);
            for (int c0 = a0; c0 < a1; c0 += blk.atoms) {
              const int na = min(blk.atoms, a1 - c0);
              const bool ok = ring_wait_full(rg, ck, p) && bok;
              if (tr && ck == chunk) tr[6] = global_timer();
              tc_fence_after();
              if (ok) {
                uint64_t ad = umma_desc(ring_s + (ck % kSlots) * kSlotBytes);
                uint64_t bd = bd0 + (uint64_t)(c0 - a0) * b_atom;
                // the block's first MMA starts its accumulators: stacked, so that it covers all 16 st columns
                // (the first chunk of a block always holds st atoms or more)
                uint32_t acc = c0 > 0 ? 1u : 0u;
                int a = 0;
                if (st > 1) {
                  for (; a + st <= na; a += st, ad += st * a_atom, bd += st * b_atom) {
                    umma_bf16(dg, ad, bd, idesc_st, acc);
                    umma_bf16(dg, ad + 2, bd + 2, idesc_st, 1u);
                    umma_bf16(dg, ad + 4, bd + 4, idesc_st, 1u);
                    umma_bf16(dg, ad + 6, bd + 6, idesc_st, 1u);
                    acc = 1u;
                  }
                }
                for (; a < na; ++a, ad += a_atom, bd += b_atom) {
                  umma_bf16(dg, ad, bd, idesc, acc);
                  umma_bf16(dg, ad + 2, bd + 2, idesc, 1u);
                  umma_bf16(dg, ad + 4, bd + 4, idesc, 1u);
                  umma_bf16(dg, ad + 6, bd + 6, idesc, 1u);
                  if (tiles == 2) {
                    const uint64_t au = ad + a_up;
                    umma_bf16(du, au, bd, idesc, acc);
                    umma_bf16(du, au + 2, bd + 2, idesc, 1u);
                    umma_bf16(du, au + 4, bd + 4, idesc, 1u);
                    umma_bf16(du, au + 6, bd + 6, idesc, 1u);
                  }
                  acc = 1u;
                }
              }
              // the slot is free once these MMAs have read it: 7 arrivals now, the 8th from the commit
              mbar_arrive_n(&rg.empty[ck % kSlots], kConsumerWarps - 1);
              umma_commit(&rg.empty[ck % kSlots]);
              ++ck;
            }
            col += tiles * nc * st;
          }
          umma_commit(&bfree[buf]);
          if (tr) tr[7] = global_timer();
        }
        umma_commit(accb);
      }
      __syncwarp();
    }
    ts.kp = kp0 + (uint32_t)nkp;
    wait_bar(accb, ts.rg & 1u, p);
    ++ts.rg;
    tc_fence_after();

    // epilogue: warp w reads TMEM lanes 32 (w & 3) .. + 31 (rows of a tile), columns half (w >> 2) of each tile
    const int q = warp & 3, half = warp >> 2;
    const int hc = nc >> 1;  // columns per half (hi / lo pairs: hc / 2 activation rows)
    // value `val` of output row `row` for activation row n (store, residual + RMS partial, or logits + argmax);
    // every lane of the warp calls it with the same n
    auto emit = [&](int row, int n, float val, bool live) {
      if (op.out_kind == OUT_STORE) {
        if (live) op.out[(size_t)n * op.out_stride + row] = val;
      } else if (op.out_kind == OUT_RESID) {
        float xn = 0.f;
        if (live) {
          xn = __ldcg(p.x + (size_t)n * p.d + row) + val;
          __stcg(p.x + (size_t)n * p.d + row, xn);
        }
        const float s2 = warp_sum(xn * xn);
        if (lane == 0 && n < N) pred[warp * 64 + n] += s2;
      } else {  // OUT_LOGITS
        if (live && p.logits) p.logits[(size_t)n * p.V + row] = val;
        float bv = live ? val : -CUDART_INF_F;
        int bi = live ? row : 0x7fffffff;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
          if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if (lane == 0 && n < N) {
          const float cv = pred[warp * 64 + n];
          const int ci = pidx[warp * 64 + n];
          if (bv > cv || (bv == cv && bi < ci)) { pred[warp * 64 + n] = bv; pidx[warp * 64 + n] = bi; }
        }
      }
    };
    int col = 0;
    for (int r = g0; r < g1;) {
      PkBlock blk;
      const int r0 = r;
      r = pk_block(op, r, g1, blk);
      const int st = tc_stack(op, blk);
      if (st > 1) {
        // K-stacked block (16 columns a segment, N <= 8): lane m = qs*P + rr holds segment qs's partial of row rr
        // in columns 16 qs ..; each lane keeps its own segment's 4 values of this warp's half in shared memory,
        // then the segments are summed per (row, activation row)
        const int P = blk.P;
        float* part = cs.mred + kConsumerWarps * 64;  // [st * P][8], after the argmax index partials
        const int m = q * 32 + lane, qs = m / P;
        for (int qq = 0; qq < st; ++qq) {
          float v[8];
          tmem_ld8(ts.tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(col + qq * nc + half * 8), v);
          if (qs == qq) {
#pragma unroll
            for (int t = 0; t < 4; ++t) part[m * 8 + half * 4 + t] = v[2 * t] + v[2 * t + 1];
          }
        }
        consumer_sync();
        const int n = warp;  // one activation row a warp
        for (int rb = 0; rb < blk.rows; rb += 32) {
          const int rr = rb + lane;
          const bool live = rr < blk.rows && n < N;
          float val = 0.f;
          if (live)
            for (int qq = 0; qq < st; ++qq) val += part[(qq * P + rr) * 8 + n];
          emit(r0 + rr, n, val, live);
        }
        consumer_sync();  // the partials are rewritten by the next stacked block
      } else {
        // lane i of the tile is the block's row i
        const int i = q * 32 + lane;
        const bool valid = i < blk.rows;
        const int row = r0 + i;
        for (int pc = 0; pc < hc; pc += 8) {
          const uint32_t ta = ts.tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(col + half * hc + pc);
          float v[8], u[8];
          tmem_ld8(ta, v);
          if (swiglu) tmem_ld8(ta + (uint32_t)nc, u);
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int n = (half * hc + pc) / 2 + t;
            const float val = v[2 * t] + v[2 * t + 1];
            const bool live = valid && n < N;
            if (swiglu) {
              const float up = u[2 * t] + u[2 * t + 1];
              if (live) op.out[(size_t)n * op.out_stride + row] = val / (1.0f + expf(-val)) * up;
            } else {
              emit(row, n, val, live);
            }
          }
        }
      }
      col += (swiglu ? 2 : 1) * nc * st;
    }
    tc_fence_before();
    consumer_sync();  // TMEM reads done before the next row group's MMAs overwrite the tiles
    g0 = g1;
  }
  chunk += tc_instr_chunks(op, in);

  if (op.out_kind == OUT_RESID || op.out_kind == OUT_LOGITS) {
    if (ctid < N) {
      if (op.out_kind == OUT_RESID) {
        float s = 0.f;
        for (int w = 0; w < kConsumerWarps; ++w) s += pred[w * 64 + ctid];
        if (op.ssq_out >= 0) __stcg(&p.ssq[ssq_index(p, op.ssq_out, ctid, sm)], s);
      } else {
        float bv = -CUDART_INF_F;
        int bi = 0x7fffffff;
        for (int w = 0; w < kConsumerWarps; ++w) {
          const float v = pred[w * 64 + ctid];
          const int ix = pidx[w * 64 + ctid];
          if (v > bv || (v == bv && ix < bi)) { bv = v; bi = ix; }
        }
        p.amax_part[(size_t)sm * kMaxN + ctid] = make_float2(bv, __int_as_float(bi));
      }
    }
  }
}

template <int CPL>
__device__ __forceinline__ void load_f32_smem(const float* src, float (&dst)[CPL]) {
#pragma unroll
  for (int c = 0; c < CPL; c += 4) {
    const float4 v = *reinterpret_cast<const float4*>(src + c);
    dst[c] = v.x;
    dst[c + 1] = v.y;
    dst[c + 2] = v.z;
    dst[c + 3] = v.w;
  }
}

// 16-byte asynchronous global -> shared copy through L2 (cp.async.cg) and its group fences
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int PENDING>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(PENDING) : "memory"); }

// STAGED: activations from shared memory (fp32, N*K*4 <= kActBytes); otherwise each chunk loads
// its activation slice from global memory (L2).
// ------------------------------------------------------------------------------------------------
// embedding: x[n, a:b] = E[token_n, a:b] (fp32) and the RMS partial of this SM's columns
// ------------------------------------------------------------------------------------------------
// A launch may run several greedy decode steps (one row per sequence each): step s sits at position
// positions[b] + s, and its tokens are the greedy tokens step s - 1 wrote (argmax[(s - 1) * N + b]).
__device__ __forceinline__ int seq_pos(const KParams& p, int b, int step) { return p.positions[b] + step; }
__device__ __forceinline__ int token_of(const KParams& p, int n, int step) {
  if (step > 0) return __ldcg(p.argmax + (size_t)(step - 1) * p.N + n);
  return p.tokens[(n / p.R) * p.tok_stride + (n % p.R)];
}

__device__ MK_OUTLINE void embed_consume(const KParams& p, const OpDesc& op, const Instr& in, int step, int ctid) {
  const int warp = ctid >> 5, lane = ctid & 31;
  for (int n = warp; n < p.N; n += kConsumerWarps) {
    const int tok = token_of(p, n, step);
    const uint16_t* e = p.embed + (size_t)tok * p.d;
    float s = 0.f;
    for (int c = in.a + lane; c < in.b; c += 32) {
      const float v = bf2f(e[c]);
      __stcg(&p.x[(size_t)n * p.d + c], v);
      s += v * v;
    }
    s = warp_sum(s);
    if (lane == 0) __stcg(&p.ssq[ssq_index(p, op.ssq_out, n, blockIdx.x)], s);
  }
}

// ------------------------------------------------------------------------------------------------
// GQA: RoPE on q and k of the new rows, bf16 k / v appended to the cache at positions p_b + r
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ size_t kv_index(const KParams& p, const OpDesc& op, int b, int g, int t) {
  return ((((size_t)op.slot * p.max_batch + b) * op.n_kv_heads + g) * p.max_ctx + t) * op.head_dim;
}

__device__ MK_OUTLINE void rope_append_consume(const KParams& p, const OpDesc& op, int step, int ctid) {
  const int warp = ctid >> 5, lane = ctid & 31;
  const int hq = op.n_heads, hkv = op.n_kv_heads, hd = op.head_dim, half = hd / 2;
  const int per_row = hq + 2 * hkv;
  const int total = p.N * per_row;
  for (int it = blockIdx.x * kConsumerWarps + warp; it < total; it += p.n_sm * kConsumerWarps) {
    const int n = it / per_row, h = it % per_row;
    const int b = n / p.R, r = n % p.R;
    const int pos = seq_pos(p, b, step) + r;
    float* vec = op.out + (size_t)n * op.out_stride + (size_t)h * hd;
    const float2* cs = p.rope + (size_t)pos * (p.rot_dim / 2);
    if (h < hq + hkv) {
      for (int i = lane; i < half; i += 32) {
        const float x1 = __ldcg(vec + i), x2 = __ldcg(vec + i + half);
        const float2 t = cs[i];
        const float y1 = x1 * t.x - x2 * t.y, y2 = x2 * t.x + x1 * t.y;
        if (h < hq) {
          __stcg(vec + i, y1);
          __stcg(vec + i + half, y2);
        } else {
          uint16_t* kc = p.kcache + kv_index(p, op, b, h - hq, pos);
          kc[i] = f2bf(y1);
          kc[i + half] = f2bf(y2);
        }
      }
    } else {
      uint16_t* vc = p.vcache + kv_index(p, op, b, h - hq - hkv, pos);
      for (int i = lane; i < hd; i += 32) vc[i] = f2bf(__ldcg(vec + i));
    }
  }
}

// ------------------------------------------------------------------------------------------------
// GQA attention. Instruction (a = b * Hkv + g, b = chunk c, c = first row | last row << 8).
// Chunk c covers prefix positions [c*TC, min((c+1)*TC, p_b)), TC = ceil(p_b / nchunk); the last chunk
// also takes the block's own rows p_b .. p_b + R - 1 (causal). Scores are kept in log2 units.
// Each warp owns up to J (row, head) pairs; lane L owns dims [L*E, L*E + E) of the head.
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ void attn_range(const KParams& p, const OpDesc& op, int b, int c, int step, int& t0,
                                           int& t1) {
  const int pos0 = seq_pos(p, b, step);
  const int tc = (pos0 + op.nchunk - 1) / op.nchunk;
  t0 = min(c * tc, pos0);
  t1 = min(t0 + tc, pos0);
}


template <int E>
__device__ __forceinline__ void load_head_slice(const uint16_t* row, int lane, float (&out)[E]) {
  const uint16_t* s = row + lane * E;
  if constexpr (E == 8) {
    const uint4 w = *reinterpret_cast<const uint4*>(s);
    out[0] = bf_lo(w.x); out[1] = bf_hi(w.x); out[2] = bf_lo(w.y); out[3] = bf_hi(w.y);
    out[4] = bf_lo(w.z); out[5] = bf_hi(w.z); out[6] = bf_lo(w.w); out[7] = bf_hi(w.w);
  } else if constexpr (E == 4) {
    const uint2 w = *reinterpret_cast<const uint2*>(s);
    out[0] = bf_lo(w.x); out[1] = bf_hi(w.x); out[2] = bf_lo(w.y); out[3] = bf_hi(w.y);
  } else {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(s);
    out[0] = bf_lo(w); out[1] = bf_hi(w);
  }
}

// One block of up to 32 keys (rows of K/V in shared memory) folded into the running softmax state.
// causal_base >= 0: key jj is the block row causal_base + jj and row r sees it iff jj <= r - causal_base.
template <int E, int J>
__device__ __forceinline__ void attn_block(const uint16_t* Ks, const uint16_t* Vs, int nb, int hd, int lane,
                                           int npair_w, const int (&prow)[J], int causal_base,
                                           const float (&q)[J][E], float (&m)[J], float (&l)[J],
                                           float (&o)[J][E]) {
#pragma unroll
  for (int j = 0; j < J; ++j) {
    if (j >= npair_w) break;
    float part[32];
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) {
      float acc = 0.f;
      if (jj < nb) {
        float kv[E];
        load_head_slice<E>(Ks + (size_t)jj * hd, lane, kv);
#pragma unroll
        for (int e = 0; e < E; ++e) acc = fmaf(q[j][e], kv[e], acc);
      }
      part[jj] = acc;
    }
    MultiReduce<32, 16>::run(part, lane);
    bool valid = lane < nb;
    if (causal_base >= 0) valid = valid && (lane <= prow[j]);
    const float s = valid ? part[0] : -CUDART_INF_F;
    const float mx = warp_max(s);
    const float m_new = fmaxf(m[j], mx);
    if (m_new == -CUDART_INF_F) continue;
    const float corr = exp2f(m[j] - m_new);
    const float pj = valid ? exp2f(s - m_new) : 0.f;
    l[j] = l[j] * corr + warp_sum(pj);
#pragma unroll
    for (int e = 0; e < E; ++e) o[j][e] *= corr;
    for (int jj = 0; jj < nb; ++jj) {
      const float pp = __shfl_sync(0xffffffffu, pj, jj);
      float vv[E];
      load_head_slice<E>(Vs + (size_t)jj * hd, lane, vv);
#pragma unroll
      for (int e = 0; e < E; ++e) o[j][e] = fmaf(pp, vv[e], o[j][e]);
    }
    m[j] = m_new;
  }
}

template <int E, int J>
__device__ MK_OUTLINE void attn_consume(const KParams& p, const OpDesc& op, const Instr& in, const Ring& rg, uint32_t& chunk,
                             CSmem& cs, uint16_t* stage_u16, int step, int ctid) {
  const int warp = ctid >> 5, lane = ctid & 31;
  const int hd = E * 32;
  const int hkv = op.n_kv_heads, G = op.groups;
  const int b = in.a / hkv, g = in.a % hkv, c = in.b;
  const int rlo = in.c & 0xff, rhi = in.c >> 8;
  const int npairs = (rhi - rlo) * G;
  const int R = p.R;
  int t0, t1;
  attn_range(p, op, b, c, step, t0, t1);
  const int pos0 = seq_pos(p, b, step);
  const int P = kChunkBytes / (4 * hd);
  const float qscale = rsqrtf((float)hd) * kLog2e;

  float q[J][E], o[J][E], m[J], l[J];
  int prow[J];
  int npair_w = 0;
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int pr = warp + j * kConsumerWarps;
    m[j] = -CUDART_INF_F;
    l[j] = 0.f;
    prow[j] = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) { o[j][e] = 0.f; q[j][e] = 0.f; }
    if (pr < npairs) {
      npair_w = j + 1;
      const int r = rlo + pr / G, h = pr % G;
      prow[j] = r;
      const float* qp = op.in + (size_t)(b * R + r) * op.in_stride + (size_t)(g * G + h) * hd + lane * E;
#pragma unroll
      for (int e = 0; e < E; ++e) q[j][e] = __ldcg(qp + e) * qscale;
    }
  }

  for (int t = t0; t < t1; t += P) {
    const int np = min(P, t1 - t);
    ring_wait_full(rg, chunk, p);
    const uint16_t* Ks = reinterpret_cast<const uint16_t*>(rg.slot_ptr(chunk));
    const uint16_t* Vs = Ks + kChunkBytes / 4;
    for (int tb = 0; tb < np; tb += 32)
      attn_block<E, J>(Ks + (size_t)tb * hd, Vs + (size_t)tb * hd, min(32, np - tb), hd, lane, npair_w, prow, -1,
                       q, m, l, o);
    ring_release(rg, chunk, lane);
    ++chunk;
  }
  if (c == op.nchunk - 1) {
    // the block's own rows, written by the RoPE/append op of this step
    uint16_t* knew = stage_u16;
    uint16_t* vnew = knew + kMaxRows * 256;
    for (int i = ctid; i < R * hd; i += kConsumerThreads) {
      const int r = i / hd, e = i % hd;
      knew[i] = __ldcg(p.kcache + kv_index(p, op, b, g, pos0 + r) + e);
      vnew[i] = __ldcg(p.vcache + kv_index(p, op, b, g, pos0 + r) + e);
    }
    consumer_sync();
    attn_block<E, J>(knew, vnew, R, hd, lane, npair_w, prow, 0, q, m, l, o);
    consumer_sync();
  }

  // partial record of every pair: o (hd floats), then m, l
  const int stride = p.attn_part_stride;
  const size_t base_rec = ((size_t)(b * hkv + g) * op.nchunk + c) * R;
#pragma unroll
  for (int j = 0; j < J; ++j) {
    if (j < npair_w) {
      const int pr = warp + j * kConsumerWarps;
      const int r = rlo + pr / G, h = pr % G;
      float* rec = p.attn_part + ((base_rec + r) * G + h) * stride;
#pragma unroll
      for (int e = 0; e < E; ++e) __stcg(rec + lane * E + e, o[j][e]);
      if (lane == 0) {
        __stcg(rec + hd, m[j]);
        __stcg(rec + hd + 1, l[j]);
      }
    }
  }
}

// ------------------------------------------------------------------------------------------------
// GQA attention, combine: instruction (a = b, b = r, c = q head) merges the context-chunk partials
// (m, l, o) of that row and head. Warp w folds chunks w, w+8, ... with the online-softmax rule (one batch
// of independent loads per 4 chunks); the 8 warp results are merged through shared memory.
// ------------------------------------------------------------------------------------------------
template <int E>
__device__ MK_OUTLINE void attn_combine_consume(const KParams& p, const OpDesc& op, const Instr& in, float* stage, int ctid) {
  const int warp = ctid >> 5, lane = ctid & 31;
  const int hd = E * 32;
  const int hkv = op.n_kv_heads, G = op.groups, NC = op.nchunk;
  const int b = in.a, r = in.b, hq = in.c;
  const int g = hq / G, h = hq % G;
  const int R = p.R;
  const int stride = p.attn_part_stride;
  const size_t rec_bg = (size_t)(b * hkv + g) * NC;
  float m = -CUDART_INF_F, l = 0.f, o[E];
#pragma unroll
  for (int e = 0; e < E; ++e) o[e] = 0.f;
  for (int c0 = warp; c0 < NC; c0 += 4 * kConsumerWarps) {
    float mc[4], lc[4], oc[4][E];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int cc = c0 + u * kConsumerWarps;
      mc[u] = -CUDART_INF_F;
      lc[u] = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) oc[u][e] = 0.f;
      if (cc < NC) {
        const float* rec = p.attn_part + (((rec_bg + cc) * R + r) * G + h) * stride;
        mc[u] = __ldcg(rec + hd);
        lc[u] = __ldcg(rec + hd + 1);
#pragma unroll
        for (int e = 0; e < E; ++e) oc[u][e] = __ldcg(rec + lane * E + e);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (mc[u] == -CUDART_INF_F) continue;
      const float mn = fmaxf(m, mc[u]);
      const float sa = exp2f(m - mn), sb = exp2f(mc[u] - mn);
      l = l * sa + lc[u] * sb;
#pragma unroll
      for (int e = 0; e < E; ++e) o[e] = o[e] * sa + oc[u][e] * sb;
      m = mn;
    }
  }
  // merge the warps: stage[w][0..hd) = o, stage[w][hd] = m, stage[w][hd+1] = l
  float* mine = stage + warp * (hd + 2);
#pragma unroll
  for (int e = 0; e < E; ++e) mine[lane * E + e] = o[e];
  if (lane == 0) {
    mine[hd] = m;
    mine[hd + 1] = l;
  }
  consumer_sync();
  for (int i = ctid; i < hd; i += kConsumerThreads) {
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, stage[w * (hd + 2) + hd]);
    float L = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float mw = stage[w * (hd + 2) + hd];
      if (mw == -CUDART_INF_F) continue;
      const float s = exp2f(mw - M);
      L += s * stage[w * (hd + 2) + hd + 1];
      acc += s * stage[w * (hd + 2) + i];
    }
    __stcg(op.out + (size_t)(b * R + r) * op.out_stride + (size_t)hq * hd + i, acc / L);
  }
}

// ------------------------------------------------------------------------------------------------
// Gated delta rule for value columns [j0, j0 + 8*CW) of head h of sequence b (instruction a = b, b = h,
// c = column group; warp w owns columns j0 + w*CW .. + CW; lane L owns key rows [L*E, L*E+E)).
// First the rows the caller accepted from the previous call are replayed into the stored state and the
// result is written back (the committed state); then the new rows advance a register copy, produce the
// outputs, and are stored for replay by the next call.
//   S <- Diag(alpha) S;  u = v - S^T k_hat;  S <- S + beta k_hat u^T;  o = S^T q_hat
// Every input of the instruction (new rows from the projection, accepted rows from the pending store)
// is staged in shared memory by one round of independent loads before the arithmetic starts.
// ------------------------------------------------------------------------------------------------
template <int CW>
__device__ MK_OUTLINE void delta_consume(const KParams& p, const OpDesc& op, const Instr& in, CSmem& cs,
                                          float* stage, int step, int ctid) {
  const int warp = ctid >> 5, lane = ctid & 31;
  const int b = in.a, h = in.b, jg = in.c;
  const int H = op.n_heads, dk = op.dk, dv = op.dv;
  const int E = dk / 32;  // 1, 2 or 4
  const int C = kConsumerWarps * CW;
  const int j0 = jg * C;
  const bool kda = op.per_channel_decay != 0;
  const int na = kda ? dk : 1;
  const int R = p.R;
  const int pos0 = seq_pos(p, b, step);
  const int a = pos0 - __ldcg(&p.seq[b].c_int);  // the previous step of this launch may have moved it
  const int rec = p.pend_rec;
  const uint32_t cur = (p.epoch + (uint32_t)step) & 1u, prev = cur ^ 1u;
  auto pend_at = [&](uint32_t par, int r) -> float* {
    return p.pend + (((((size_t)op.slot * 2 + par) * p.max_batch + b) * p.max_rows + r) * H + h) * rec;
  };
  const int offk = H * dk, offv = 2 * H * dk, offa = 2 * H * dk + H * dv;
  const int offb = offa + (kda ? H * dk : H);

  // staging layout (floats)
  float* sq_ = stage;                 // [R][dk] raw q
  float* sk_ = sq_ + R * dk;          // [R][dk] raw k
  float* sa_ = sk_ + R * dk;          // [R][na] alpha (sigmoid applied)
  float* sb_ = sa_ + R * na;          // [R]     beta (sigmoid applied)
  float* sv_ = sb_ + R;               // [R][C]  v of this instruction's columns
  float* pk_ = sv_ + R * C;           // [a][dk] accepted k_hat
  float* pa_ = pk_ + a * dk;          // [a][na] accepted alpha
  float* pb_ = pa_ + a * na;          // [a]     accepted beta
  float* pv_ = pb_ + a;               // [a][C]  accepted v

  // the state columns this warp owns (independent of the staging); column c at Sp + c * dk
  float S[CW][4];
  float* const Sp = p.state + ((((size_t)op.slot * p.max_batch + b) * H + h) * dv + j0 + warp * CW) * dk + lane * E;
#pragma unroll
  for (int c = 0; c < CW; ++c) {
    const int j = j0 + warp * CW + c;
    if (E == 4) {  // this lane's 4 key rows of the column in one 16-byte load
      const float4 v4 = j < dv ? __ldcg(reinterpret_cast<const float4*>(Sp + c * dk)) : make_float4(0.f, 0.f, 0.f, 0.f);
      S[c][0] = v4.x;
      S[c][1] = v4.y;
      S[c][2] = v4.z;
      S[c][3] = v4.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) S[c][e] = (e < E && j < dv) ? __ldcg(Sp + c * dk + e) : 0.f;
    }
  }
  // All staged values in one flat index space laid out like the staging area (stage[i] is item i), loaded in
  // rounds of 4 per thread: one round trip for the usual 1 to 2 items a thread stages. dk and C are powers of 2.
  const int ldk = __ffs(dk) - 1, lc = __ffs(C) - 1;
  const int e0 = R * dk, e1 = 2 * R * dk, e2 = e1 + R * na, e3 = e2 + R, e4 = e3 + R * C;
  const int e5 = e4 + a * dk, e6 = e5 + a * na, e7 = e6 + a, e8 = e7 + a * C;
  // source of item i (nullptr: zero); the gate sigmoid applies to items [e1, e3)
  auto item_src = [&](int i) -> const float* {
    if (i < e3) {  // new rows: q, k, alpha, beta from the projection output
      int r, off;
      if (i < e1) {
        const int j = i < e0 ? i : i - e0;
        r = j >> ldk;
        off = (i < e0 ? 0 : offk) + h * dk + (j & (dk - 1));
      } else {
        const int j = i < e2 ? i - e1 : i - e2;
        if (i < e2 && kda) {
          r = j >> ldk;
          off = offa + h * dk + (j & (dk - 1));
        } else {
          r = j;
          off = (i < e2 ? offa : offb) + h;
        }
      }
      return op.in + (size_t)(b * R + r) * op.in_stride + off;
    }
    if (i < e4) {  // new rows: v of this instruction's columns
      const int j = i - e3, c = j & (C - 1);
      return j0 + c < dv ? op.in + (size_t)(b * R + (j >> lc)) * op.in_stride + offv + h * dv + j0 + c : nullptr;
    }
    if (i < e7) {  // accepted rows: k_hat, alpha, beta from the pending store
      if (i < e5) return pend_at(prev, (i - e4) >> ldk) + ((i - e4) & (dk - 1));
      if (i < e6) {
        const int j = i - e5;
        return kda ? pend_at(prev, j >> ldk) + dk + dv + (j & (dk - 1)) : pend_at(prev, j) + dk + dv;
      }
      return pend_at(prev, i - e6) + 2 * dk + dv;
    }
    const int j = i - e7, c = j & (C - 1);  // accepted rows: v
    return j0 + c < dv ? pend_at(prev, j >> lc) + dk + j0 + c : nullptr;
  };
  for (int i0 = ctid; i0 < e8; i0 += 4 * kConsumerThreads) {
    float v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * kConsumerThreads;
      const float* src = i < e8 ? item_src(i) : nullptr;
      v[u] = src ? __ldcg(src) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * kConsumerThreads;
      if (i < e8) stage[i] = (i >= e1 && i < e3) ? sigmoidf_(v[u]) : v[u];
    }
  }
  consumer_sync();

  const int jw = j0 + warp * CW;  // first column of this warp
  // replay accepted rows of the previous call
  for (int r = 0; r < a; ++r) {
    float kh[4], al[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      kh[e] = e < E ? pk_[r * dk + lane * E + e] : 0.f;
      al[e] = e < E ? (kda ? pa_[r * dk + lane * E + e] : pa_[r]) : 1.f;
    }
    const float beta = pb_[r];
    float dot[CW];
#pragma unroll
    for (int c = 0; c < CW; ++c) {
      dot[c] = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        S[c][e] *= al[e];
        dot[c] = fmaf(S[c][e], kh[e], dot[c]);
      }
    }
    warp_sum_n(dot);  // the columns' reductions interleaved
#pragma unroll
    for (int c = 0; c < CW; ++c) {
      const float u = pv_[r * C + warp * CW + c] - dot[c];
#pragma unroll
      for (int e = 0; e < 4; ++e) S[c][e] = fmaf(beta * kh[e], u, S[c][e]);
    }
  }
  if (a > 0) {
#pragma unroll
    for (int c = 0; c < CW; ++c)
      if (jw + c < dv) {
        if (E == 4) __stcg(reinterpret_cast<float4*>(Sp + c * dk), make_float4(S[c][0], S[c][1], S[c][2], S[c][3]));
        else
          for (int e = 0; e < E; ++e) __stcg(Sp + c * dk + e, S[c][e]);
      }
  }

  const float qs = rsqrtf((float)dk);
  for (int r = 0; r < R; ++r) {
    const int n = b * R + r;
    float qv[4], kv[4], al[4];
    float sqs = 0.f, sks = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      qv[e] = e < E ? sq_[r * dk + lane * E + e] : 0.f;
      kv[e] = e < E ? sk_[r * dk + lane * E + e] : 0.f;
      al[e] = e < E ? (kda ? sa_[r * dk + lane * E + e] : sa_[r]) : 1.f;
      sqs = fmaf(qv[e], qv[e], sqs);
      sks = fmaf(kv[e], kv[e], sks);
    }
    const float iq = rsqrtf(warp_sum(sqs) + 1e-6f) * qs;
    const float ik = rsqrtf(warp_sum(sks) + 1e-6f);
    const float beta = sb_[r];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      qv[e] *= iq;
      kv[e] *= ik;
    }
    float* pw = pend_at(cur, r);
    float dot[CW], od[CW];
#pragma unroll
    for (int c = 0; c < CW; ++c) {
      dot[c] = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        S[c][e] *= al[e];
        dot[c] = fmaf(S[c][e], kv[e], dot[c]);
      }
    }
    warp_sum_n(dot);
#pragma unroll
    for (int c = 0; c < CW; ++c) {
      const float u = sv_[r * C + warp * CW + c] - dot[c];
      od[c] = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        S[c][e] = fmaf(beta * kv[e], u, S[c][e]);
        od[c] = fmaf(S[c][e], qv[e], od[c]);
      }
    }
    warp_sum_n(od);
    if (lane == 0) {
#pragma unroll
      for (int c = 0; c < CW; ++c) {
        if (jw + c < dv) {
          __stcg(op.out + (size_t)n * op.out_stride + h * dv + jw + c, od[c]);
          __stcg(pw + dk + jw + c, sv_[r * C + warp * CW + c]);  // stored for replay by the next call
        }
      }
    }
    if (jg == 0 && warp == 0) {
      for (int e = 0; e < E; ++e) {
        __stcg(pw + lane * E + e, kv[e]);
        if (kda) __stcg(pw + dk + dv + lane * E + e, al[e]);
      }
      if (lane == 0) {
        if (!kda) __stcg(pw + dk + dv, al[0]);
        __stcg(pw + 2 * dk + dv, beta);
      }
    }
  }
}

// ------------------------------------------------------------------------------------------------
// MoE routing (one instruction): for each row, s = sigmoid(z) over the experts; top_k experts are picked
// by top_k sequential argmax passes over s + bias, the lowest index winning a tie (the pages' router takes
// its top-k as sequential argmax passes: Kimi K3's TPU megakernel, "How it maps onto a TPU v7"); the
// weights are route_scale * s_sel / sum(s_sel). Also the union of the picked experts, ascending.
// ------------------------------------------------------------------------------------------------
__device__ __noinline__ void route_consume(const KParams& p, const OpDesc& op, float* stage, int step, int ctid) {
  const int warp = ctid >> 5, lane = ctid & 31;
  const int E = op.n_experts, K = op.top_k, N = p.N;
  int* flags = reinterpret_cast<int*>(stage);
  for (int e = ctid; e < E; e += kConsumerThreads) flags[e] = 0;
  consumer_sync();
  for (int n = warp; n < N; n += kConsumerWarps) {
    float sc[kMaxExperts / 32], bs[kMaxExperts / 32];
#pragma unroll
    for (int j = 0; j < kMaxExperts / 32; ++j) {
      const int e = lane + 32 * j;
      sc[j] = 0.f;
      bs[j] = -CUDART_INF_F;  // past the last expert, or already picked: never selected
      if (e < E) {
        sc[j] = sigmoidf_(__ldcg(op.in + (size_t)n * op.in_stride + e));
        const float b = sc[j] + (op.router_bias ? __ldg(op.router_bias + e) : 0.f);
        // a selectable expert always beats -inf, so each pass picks a valid id even from NaN scores
        bs[j] = (b == b) ? fmaxf(b, -FLT_MAX) : -FLT_MAX;
      }
    }
    float ssum = 0.f;
    float ssel[kMaxTopK];
    // routing replay: a row with caller-given expert ids uses them (an id outside [0, E) falls back to the
    // row's own pick); its own picks still go to the routing log
    const int b_row = n / p.R, pos_row = seq_pos(p, b_row, step) + n % p.R;
    const int32_t* frow = nullptr;
    if (p.route_force) {
      frow = p.route_force + (((size_t)op.layer * p.max_batch + b_row) * p.max_ctx + pos_row) * K;
      if (__ldg(frow) < 0) frow = nullptr;
    }
    for (int k = 0; k < K; ++k) {
      float bv = -CUDART_INF_F;
      int bi = 0x7fffffff;
#pragma unroll
      for (int j = 0; j < kMaxExperts / 32; ++j) {
        const int e = lane + 32 * j;
        if (bs[j] > bv) { bv = bs[j]; bi = e; }  // ascending e within a lane: first occurrence wins
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
      }
#pragma unroll
      for (int j = 0; j < kMaxExperts / 32; ++j)
        if (lane + 32 * j == bi) bs[j] = -CUDART_INF_F;  // taken
      int use = bi;
      if (frow) {
        const int f = __ldg(frow + k);
        if (f >= 0 && f < E) use = f;
      }
      float s_w = 0.f;
#pragma unroll
      for (int j = 0; j < kMaxExperts / 32; ++j)
        if (lane + 32 * j == use) s_w = sc[j];
      s_w = __shfl_sync(0xffffffffu, s_w, use & 31);
      ssel[k] = s_w;
      ssum += s_w;
      if (lane == 0) {
        __stcg(p.route_idx + n * kMaxTopK + k, use);
        flags[use] = 1;
        if (p.route_log) p.route_log[(((size_t)op.layer * p.max_batch + b_row) * p.max_ctx + pos_row) * K + k] = bi;
      }
    }
    if (lane == 0)
      for (int k = 0; k < K; ++k) __stcg(p.route_w + n * kMaxTopK + k, op.route_scale * ssel[k] / ssum);
  }
  consumer_sync();
  if (warp == 0) {  // compact the picked experts in ascending order, 32 at a time
    int cnt = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const bool f = e0 + lane < E && flags[e0 + lane] != 0;
      const unsigned m = __ballot_sync(0xffffffffu, f);
      if (f) __stcg(p.union_list + 1 + cnt + __popc(m & ((1u << lane) - 1u)), e0 + lane);
      cnt += __popc(m);
    }
    if (lane == 0) __stcg(p.union_list, cnt);
  }
}

__device__ __forceinline__ float e4m3_to_f32(uint8_t b) {
  __nv_fp8_e4m3 v;
  v.__x = b;
  return static_cast<float>(v);
}

// Weight row r of matrix m (0: gate / down, 1: up) of selected expert slot j; for NVFP4 also its scales.
struct ExpertRow {
  const uint8_t* w;
  const uint8_t* s;
};
__device__ __forceinline__ ExpertRow expert_row(const KParams& p, const OpDesc& op, int j, int m, int r, int K,
                                               const int32_t* uni) {
  const int S = op.n_shared;
  const bool shared = j < S;
  const int e = shared ? j : uni[1 + (j - S)];
  const int rows = (op.type == OP_MOE_UP) ? op.F : p.d;
  const size_t row = (size_t)e * rows + r;
  ExpertRow out;
  const void* base = shared ? op.sw[m] : op.ew[m];
  if (op.fp4) {
    out.w = static_cast<const uint8_t*>(base) + row * (K / 2);
    out.s = (shared ? op.ssc[m] : op.esc[m]) + row * (K / 16);
  } else {
    out.w = static_cast<const uint8_t*>(base) + row * K * 2;
    out.s = nullptr;
  }
  return out;
}

__device__ __forceinline__ float expert_gscale(const OpDesc& op, int j, int m, const int32_t* uni) {
  if (!op.fp4) return 1.f;
  const int S = op.n_shared;
  if (j < S) return __ldg(op.sgs[m] + j);
  return __ldg(op.egs[m] + uni[1 + (j - S)]);
}

// Eight e2m1 codes (one 32-bit word, element i in bits 4i..4i+3) times the block scale, without a table:
// one byte permute looks up twice the magnitudes {0, 1, 2, 3, 4, 6, 8, 12} of four codes at once, the
// 2^23 bias trick turns a byte into its float value, and the code's sign bit picks +-scale/2.
__device__ __forceinline__ void e2m1x8_decode(uint32_t codes, float scale, float (&w)[8]) {
  const float hs = 0.5f * scale;
  const uint32_t m03 = __byte_perm(0x03020100u, 0x0C080604u, codes & 0x7777u);
  const uint32_t m47 = __byte_perm(0x03020100u, 0x0C080604u, (codes >> 16) & 0x7777u);
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint32_t mag = ((c < 4 ? m03 : m47) >> (8 * (c & 3))) & 0xffu;
    const float v = __uint_as_float(0x4B000000u | mag) - 8388608.0f;
    w[c] = v * (((codes >> (4 * c + 3)) & 1u) ? -hs : hs);
  }
}

// ------------------------------------------------------------------------------------------------
// MoE expert GEMVs. One instruction per SM covers output rows [a, b) of EVERY selected expert (the shared
// expert(s), then the step's union of routed experts), so the work per SM does not depend on routing.
//   OP_MOE_UP:   hexp[j][n][f] = silu(g) * u,  g / u = rows f of expert j's gate / up times RMSNorm(x)_n
//   OP_MOE_DOWN: x[n][r] += sum_j w[j][n] * (down_j[r] . hexp[j][n]),  w = 1 for shared experts, the
//                router weight for routed ones (0 when row n did not pick expert j)
// Weights stream through the ring like a dense GEMV (bf16 rows, or NVFP4 rows = codes then block
// scales); inputs come from L2 per chunk. NVFP4 decodes as e2m1 * e4m3 (exact in fp32) and the fp32
// tensor scale multiplies the dot product.
// ------------------------------------------------------------------------------------------------
// STG (up to 2 activation rows): the inputs sit in shared memory instead of being read from L2 per chunk —
// for MOE_UP the normalised x rows, staged once; for MOE_DOWN expert j's SwiGLU rows, copied with cp.async
// into one of two buffers while expert j - 1 computes.
template <int RG, int NR, int CPL, bool FP4, bool STG>
__device__ __noinline__ void moe_consume(const KParams& p, const OpDesc& op, const Instr& in, const Ring& rg, uint32_t& chunk,
                            CSmem& cs, float* act, int ctid) {
  constexpr int KC = CPL * kConsumerThreads;
  constexpr int V = RG * NR;
  const int warp = ctid >> 5, lane = ctid & 31;
  const bool up = op.type == OP_MOE_UP;
  const int N = p.N;
  const int K = up ? p.d : op.F;
  const int glog = up ? RG / 2 : RG;
  const int ucount = __ldcg(p.union_list);
  const int nsel = op.n_shared + ucount;
  for (int i = ctid; i <= ucount; i += kConsumerThreads) cs.uni_c[i] = __ldcg(p.union_list + i);
  const int32_t* uni = cs.uni_c;  // read after the consumer_sync below
  const int nrows = in.b - in.a;
  const int ng = gemv_ngroups(nrows, glog);
  const int passes = op.passes;
  // DOWN: each row's routing (expert ids, weights) and this SM's slice of x, in the staging area
  const int rt = (N * op.top_k + 3) & ~3;
  int* ridx = reinterpret_cast<int*>(act);  // [N][top_k]
  float* rw = act + rt;                     // [N][top_k]
  float* xres = act + 2 * rt;               // [N][nrows]
  // staged inputs: UP [N][K] at act; DOWN two [N][F] buffers after xres
  float* hst = act + 2 * rt + ((N * nrows + 3) & ~3);
  if (up) {
    inv_rms_rows(p, op.ssq_in, p.d, cs, warp, lane);
    if constexpr (STG) {
      consumer_sync();
      for (int i = ctid * 4; i < N * K; i += kConsumerThreads * 4) {
        const int n = i / K, k = i % K;
        float4 v = __ldcg(reinterpret_cast<const float4*>(p.x + (size_t)n * p.d + k));
        const uint2 g = __ldg(reinterpret_cast<const uint2*>(op.gain + k));
        const float sc = cs.inv_rms[n];
        v.x *= sc * bf_lo(g.x);
        v.y *= sc * bf_hi(g.x);
        v.z *= sc * bf_lo(g.y);
        v.w *= sc * bf_hi(g.y);
        *reinterpret_cast<float4*>(act + i) = v;
      }
    }
  } else {
    for (int i = ctid; i < N * op.top_k; i += kConsumerThreads) {
      const int n = i / op.top_k, k = i % op.top_k;
      ridx[i] = __ldcg(p.route_idx + n * kMaxTopK + k);
      rw[i] = __ldcg(p.route_w + n * kMaxTopK + k);
    }
    for (int i = ctid; i < N * nrows; i += kConsumerThreads)
      xres[i] = __ldcg(p.x + (size_t)(i / nrows) * p.d + in.a + i % nrows);
  }
  auto stage_down = [&](int jn) {
    const float* src = p.hexp + (size_t)jn * N * op.F;
    float* dst = hst + (jn & 1) * N * op.F;
    for (int i = ctid * 4; i < N * op.F; i += kConsumerThreads * 4) cp_async16(dst + i, src + i);
    cp_async_commit();
  };
  if (STG && !up && ng > 0 && nsel > 0) stage_down(0);
  consumer_sync();

  for (int j = 0; j < nsel && ng > 0; ++j) {
    const float gs0 = expert_gscale(op, j, 0, uni);
    const float gs1 = up ? expert_gscale(op, j, 1, uni) : 1.f;
    const float* hin = p.hexp + (size_t)j * N * op.F;  // DOWN input
    if (STG && !up) {
      // expert j's rows were requested one expert ago; request j + 1's, wait for j's, publish
      if (j + 1 < nsel) {
        stage_down(j + 1);
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
      consumer_sync();
      hin = hst + (j & 1) * N * op.F;
    }
    const int ej = j < op.n_shared ? -1 : uni[1 + (j - op.n_shared)];
    for (int pass = 0; pass < passes; ++pass) {
      const int nbase = pass * NR;
      for (int grp = 0; grp < ng; ++grp) {
        const int g0 = gemv_group_row(in.a, nrows, ng, grp);
        const int nl = gemv_group_row(in.a, nrows, ng, grp + 1) - g0;
        float acc[RG][NR];
#pragma unroll
        for (int i = 0; i < RG; ++i)
#pragma unroll
          for (int n = 0; n < NR; ++n) acc[i][n] = 0.f;
        for (int k0 = 0; k0 < K; k0 += KC) {
          const int kw = min(KC, K - k0);
          const int col = ctid * CPL;
          float a[NR][CPL];
          if (col < kw) {
            float gsc[CPL];
            if (!STG && up) load_bf16_global<CPL>(op.gain + k0 + col, gsc);
#pragma unroll
            for (int n = 0; n < NR; ++n) {
              const int row = nbase + n;
              if (row < N) {
                if (STG) {
                  load_f32_smem<CPL>((up ? act : hin) + (size_t)row * K + k0 + col, a[n]);
                } else if (up) {
                  load_f32<CPL>(p.x + (size_t)row * p.d + k0 + col, a[n]);
                  const float s = cs.inv_rms[row];
#pragma unroll
                  for (int c = 0; c < CPL; ++c) a[n][c] *= s * gsc[c];
                } else {
                  load_f32<CPL>(hin + (size_t)row * op.F + k0 + col, a[n]);
                }
              } else {
#pragma unroll
                for (int c = 0; c < CPL; ++c) a[n][c] = 0.f;
              }
            }
          }
          ring_wait_full(rg, chunk, p);
          if (col < kw) {
            const uint8_t* slot = rg.slot_ptr(chunk);
            if constexpr (FP4) {
              const int pitch = kw / 2 + kw / 16;
#pragma unroll
              for (int i = 0; i < RG; ++i) {
                const uint8_t* rowp = slot + (size_t)i * pitch;
                const uint32_t codes = *reinterpret_cast<const uint32_t*>(rowp + col / 2);
                const float sc = e4m3_to_f32(rowp[kw / 2 + col / 16]);
                float wf[CPL];
                e2m1x8_decode(codes, sc, wf);
#pragma unroll
                for (int c = 0; c < CPL; ++c)
#pragma unroll
                  for (int n = 0; n < NR; ++n) acc[i][n] = fmaf(wf[c], a[n][c], acc[i][n]);
              }
            } else {
              const uint8_t* wbase = slot + col * 2;
              float wf[RG][CPL];
#pragma unroll
              for (int i = 0; i < RG; ++i) load_bf16_row<CPL>(wbase + (size_t)i * kw * 2, wf[i]);
#pragma unroll
              for (int i = 0; i < RG; ++i)
#pragma unroll
                for (int c = 0; c < CPL; ++c)
#pragma unroll
                  for (int n = 0; n < NR; ++n) acc[i][n] = fmaf(wf[i][c], a[n][c], acc[i][n]);
            }
          }
          ring_release(rg, chunk, lane);
          ++chunk;
        }
        float v[V];
#pragma unroll
        for (int i = 0; i < RG; ++i)
#pragma unroll
          for (int n = 0; n < NR; ++n) v[i * NR + n] = acc[i][n];
        block_reduce<V>(v, cs, warp, lane, ctid);
        if (up) {
          if (ctid < nl * NR) {
            const int jj = ctid / NR, n = ctid % NR, row = nbase + n;
            if (row < N) {
              const float g = cs.val[jj * NR + n] * gs0;
              const float u = cs.val[(nl + jj) * NR + n] * gs1;
              __stcg(p.hexp + ((size_t)j * N + row) * op.F + g0 + jj, g / (1.0f + expf(-g)) * u);
            }
          }
        } else if (ctid < V) {
          const int i = ctid / NR, n = ctid % NR, row = nbase + n;
          if (i < nl && row < N) {
            float w = (ej < 0) ? 1.f : 0.f;  // shared experts weigh 1, routed ones their router weight
            for (int k = 0; k < op.top_k; ++k)
              if (ridx[row * op.top_k + k] == ej) w = rw[row * op.top_k + k];
            xres[row * nrows + (g0 - in.a) + i] += w * (cs.val[ctid] * gs0);
          }
        }
        consumer_sync();
      }
    }
  }
  if (!up) {
    // write the SM's slice of x back and the RMS partial of the new x
    for (int n = warp; n < N; n += kConsumerWarps) {
      float s = 0.f;
      for (int i = lane; i < nrows; i += 32) {
        const float xn = xres[n * nrows + i];
        __stcg(p.x + (size_t)n * p.d + in.a + i, xn);
        s += xn * xn;
      }
      s = warp_sum(s);
      if (lane == 0) __stcg(&p.ssq[ssq_index(p, op.ssq_out, n, blockIdx.x)], s);
    }
  }
}

// ------------------------------------------------------------------------------------------------
// Multi-head latent attention, absorbed form. The cache holds one (kv_lora + rope)-wide bf16 latent per
// position (576 = 512 + 64 in the pages' model: Kimi K3's TPU megakernel, "Why one user at a time is a
// bandwidth problem").
//   MLA_PREP : c_q = RMSNorm(proj[0:q_lora]) -> aux;  c_kv = RMSNorm(proj[q_lora : q_lora+kv_lora]),
//              k_r = RoPE(proj[q_lora+kv_lora :]) -> latent cache at positions p_b + r
//   MLA_QABS : q~_h = W_UK[h] q_nope_h (kv_lora), q_r = RoPE(q_rope_h), both times log2(e)/sqrt(nope+rope)
//   MLA_ATTN : per (sequence, 8-head group, context chunk, rows): online softmax of q~.c + q_r.k_r over
//              the chunk, partial (o_lat, m, l) records; the GQA combine op merges them
//   MLA_UV   : o_h = W_UV[h] o_lat_h
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ size_t lat_index(const KParams& p, const OpDesc& op, int b, int t) {
  return (((size_t)op.slot * p.max_batch + b) * p.max_ctx + t) * (op.kv_lora + op.rope);
}

__device__ __noinline__ void mla_prep_consume(const KParams& p, const OpDesc& op, int step, int ctid) {
  const int warp = ctid >> 5, lane = ctid & 31;
  const int total = p.N * 2;
  const int ql = op.q_lora, kl = op.kv_lora, rp = op.rope, half = rp / 2;
  for (int it = blockIdx.x * kConsumerWarps + warp; it < total; it += p.n_sm * kConsumerWarps) {
    const int n = it >> 1, part = it & 1;
    const float* row = op.in + (size_t)n * op.in_stride;
    if (part == 0) {
      float s = 0.f;
      for (int i = lane; i < ql; i += 32) {
        const float v = __ldcg(row + i);
        s += v * v;
      }
      const float inv = rsqrtf(warp_sum(s) / (float)ql + p.eps);
      for (int i = lane; i < ql; i += 32)
        __stcg(op.aux + (size_t)n * op.aux_stride + i, __ldcg(row + i) * inv * bf2f(op.q_norm[i]));
    } else {
      const int b = n / p.R, r = n % p.R;
      const int pos = seq_pos(p, b, step) + r;
      uint16_t* lat = p.latent + lat_index(p, op, b, pos);
      float s = 0.f;
      for (int i = lane; i < kl; i += 32) {
        const float v = __ldcg(row + ql + i);
        s += v * v;
      }
      const float inv = rsqrtf(warp_sum(s) / (float)kl + p.eps);
      for (int i = lane; i < kl; i += 32) lat[i] = f2bf(__ldcg(row + ql + i) * inv * bf2f(op.kv_norm[i]));
      const float2* cs = p.rope + (size_t)pos * (p.rot_dim / 2);
      for (int i = lane; i < half; i += 32) {
        const float x1 = __ldcg(row + ql + kl + i), x2 = __ldcg(row + ql + kl + i + half);
        const float2 t = cs[i];
        lat[kl + i] = f2bf(x1 * t.x - x2 * t.y);
        lat[kl + i + half] = f2bf(x2 * t.x + x1 * t.y);
      }
    }
  }
}

// instruction (a = head h, b = 128-column block of the latent): qt[n][h][c] for c in the block; block 0
// also writes the rotated rope query qt[n][h][kv_lora ..]. Warp w owns 16 latent columns: their W_UK rows
// (lane L holds inputs [L*E, L*E + E) of each) are loaded together up front, then each query row costs 16
// dot products folded across the warp by one multi-value reduction.
__device__ __noinline__ void mla_qabs_consume(const KParams& p, const OpDesc& op, const Instr& in, int step, int ctid) {
  const int warp = ctid >> 5, lane = ctid & 31;
  const int h = in.a, cb = in.b;
  const int nope = op.nope, rp = op.rope, kl = op.kv_lora, half = rp / 2;
  const int qw = nope + rp;  // per-head width of the projected query
  const float qs = rsqrtf((float)(nope + rp)) * kLog2e;
  const int ldq = op.in_stride, ldt = op.out_stride;
  const int N = p.N;
  const int E = nope / 32;  // nope inputs per lane (1 .. 4)
  const int c0 = cb * 128 + warp * 16;
  float w[16][4];
#pragma unroll
  for (int cc = 0; cc < 16; ++cc) {
    const uint16_t* wrow = op.w_uk + ((size_t)h * kl + c0 + cc) * nope + lane * E;
#pragma unroll
    for (int e = 0; e < 4; ++e) w[cc][e] = (e < E) ? bf2f(__ldg(wrow + e)) : 0.f;
  }
  for (int n = 0; n < N; ++n) {
    const float* q = op.in + (size_t)n * ldq + (size_t)h * qw + lane * E;
    float qv[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) qv[e] = (e < E) ? __ldcg(q + e) : 0.f;
    float v[16];
#pragma unroll
    for (int cc = 0; cc < 16; ++cc) {
      float d = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) d = fmaf(w[cc][e], qv[e], d);
      v[cc] = d;
    }
    MultiReduce<16, 16>::run(v, lane);  // lane 2i: column i
    if ((lane & 1) == 0) __stcg(op.out + (size_t)n * ldt + (size_t)h * (kl + rp) + c0 + (lane >> 1), v[0] * qs);
  }
  if (cb == 0) {
    for (int n = warp; n < N; n += kConsumerWarps) {
      const int b = n / p.R, r = n % p.R;
      const int pos = seq_pos(p, b, step) + r;
      const float* q = op.in + (size_t)n * ldq + (size_t)h * qw + nope;
      const float2* cs = p.rope + (size_t)pos * (p.rot_dim / 2);
      float* dst = op.out + (size_t)n * ldt + (size_t)h * (kl + rp) + kl;
      for (int i = lane; i < half; i += 32) {
        const float x1 = __ldcg(q + i), x2 = __ldcg(q + i + half);
        const float2 t = cs[i];
        __stcg(dst + i, (x1 * t.x - x2 * t.y) * qs);
        __stcg(dst + i + half, (x2 * t.x + x1 * t.y) * qs);
      }
    }
  }
}

// Latent attention block: up to 32 positions (rows of the latent chunk in shared memory, 576 bf16 each)
// folded into the online softmax of the warp's J (row, head) pairs. Lane L owns latent dims
// [16L, 16L+16) and rope dims [2L, 2L+2).
template <int J>
__device__ __forceinline__ void mla_block(const uint16_t* lat, int nb, int ldl, int kl, int lane, int npair_w,
                                          const int (&prow)[J], int causal, const float (&q)[J][16],
                                          const float (&qr)[J][2], float (&m)[J], float (&l)[J], float (&o)[J][16]) {
#pragma unroll
  for (int j = 0; j < J; ++j) {
    if (j >= npair_w) break;
    float part[32];
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) {
      float acc = 0.f;
      if (jj < nb) {
        const uint16_t* row = lat + (size_t)jj * ldl;
        const uint4 a0 = *reinterpret_cast<const uint4*>(row + lane * 16);
        const uint4 a1 = *reinterpret_cast<const uint4*>(row + lane * 16 + 8);
        const uint32_t rr = *reinterpret_cast<const uint32_t*>(row + kl + lane * 2);
        const uint32_t ws[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          acc = fmaf(q[j][2 * e], bf_lo(ws[e]), acc);
          acc = fmaf(q[j][2 * e + 1], bf_hi(ws[e]), acc);
        }
        acc = fmaf(qr[j][0], bf_lo(rr), acc);
        acc = fmaf(qr[j][1], bf_hi(rr), acc);
      }
      part[jj] = acc;
    }
    MultiReduce<32, 16>::run(part, lane);
    bool valid = lane < nb;
    if (causal >= 0) valid = valid && (lane <= prow[j]);
    const float s = valid ? part[0] : -CUDART_INF_F;
    const float m_new = fmaxf(m[j], warp_max(s));
    if (m_new == -CUDART_INF_F) continue;
    const float corr = exp2f(m[j] - m_new);
    const float pj = valid ? exp2f(s - m_new) : 0.f;
    l[j] = l[j] * corr + warp_sum(pj);
#pragma unroll
    for (int e = 0; e < 16; ++e) o[j][e] *= corr;
    for (int jj = 0; jj < nb; ++jj) {
      const float pp = __shfl_sync(0xffffffffu, pj, jj);
      const uint16_t* row = lat + (size_t)jj * ldl;
      const uint4 a0 = *reinterpret_cast<const uint4*>(row + lane * 16);
      const uint4 a1 = *reinterpret_cast<const uint4*>(row + lane * 16 + 8);
      const uint32_t ws[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        o[j][2 * e] = fmaf(pp, bf_lo(ws[e]), o[j][2 * e]);
        o[j][2 * e + 1] = fmaf(pp, bf_hi(ws[e]), o[j][2 * e + 1]);
      }
    }
    m[j] = m_new;
  }
}

// instruction (a = b * ngroups + head group, b = chunk, c = first row | last row << 8); warp w owns head
// group*8 + w for the rows of the instruction (J rows per warp)
template <int J>
__device__ __noinline__ void mla_attn_consume(const KParams& p, const OpDesc& op, const Instr& in, const Ring& rg,
                                 uint32_t& chunk, uint16_t* stage, int step, int ctid) {
  const int warp = ctid >> 5, lane = ctid & 31;
  const int ngr = op.n_kv_heads, G = op.groups;  // head groups, heads per group
  const int b = in.a / ngr, hg = in.a % ngr, c = in.b;
  const int rlo = in.c & 0xff, rhi = in.c >> 8;
  const int kl = op.kv_lora, ldl = op.kv_lora + op.rope;
  const int R = p.R;
  const int h = hg * G + warp;
  int t0, t1;
  attn_range(p, op, b, c, step, t0, t1);
  const int pos0 = seq_pos(p, b, step);
  const int P = kChunkBytes / (ldl * 2);
  float q[J][16], qr[J][2], o[J][16], m[J], l[J];
  int prow[J];
  const int npair_w = (warp < G) ? (rhi - rlo) : 0;
#pragma unroll
  for (int j = 0; j < J; ++j) {
    m[j] = -CUDART_INF_F;
    l[j] = 0.f;
    prow[j] = rlo + j;
#pragma unroll
    for (int e = 0; e < 16; ++e) { o[j][e] = 0.f; q[j][e] = 0.f; }
    qr[j][0] = qr[j][1] = 0.f;
    if (j < npair_w) {
      const float* qp = op.in + (size_t)(b * R + rlo + j) * op.in_stride + (size_t)h * ldl;
#pragma unroll
      for (int e = 0; e < 16; ++e) q[j][e] = __ldcg(qp + lane * 16 + e);
      qr[j][0] = __ldcg(qp + kl + lane * 2);
      qr[j][1] = __ldcg(qp + kl + lane * 2 + 1);
    }
  }
  for (int t = t0; t < t1; t += P) {
    const int np = min(P, t1 - t);
    ring_wait_full(rg, chunk, p);
    const uint16_t* lat = reinterpret_cast<const uint16_t*>(rg.slot_ptr(chunk));
    mla_block<J>(lat, np, ldl, kl, lane, npair_w, prow, -1, q, qr, m, l, o);
    ring_release(rg, chunk, lane);
    ++chunk;
  }
  if (c == op.nchunk - 1) {
    for (int i = ctid; i < R * ldl; i += kConsumerThreads) {
      const int r = i / ldl, e = i % ldl;
      stage[i] = __ldcg(p.latent + lat_index(p, op, b, pos0 + r) + e);
    }
    consumer_sync();
    mla_block<J>(stage, R, ldl, kl, lane, npair_w, prow, 0, q, qr, m, l, o);
    consumer_sync();
  }
  // partial records as in GQA: [((b * ngroups + hg) * nchunk + c) * R + r][head in group][o, m, l]
  const int stride = p.attn_part_stride;
  const size_t base_rec = ((size_t)(b * ngr + hg) * op.nchunk + c) * R;
#pragma unroll
  for (int j = 0; j < J; ++j) {
    if (j < npair_w) {
      float* rec = p.attn_part + ((base_rec + rlo + j) * G + warp) * stride;
#pragma unroll
      for (int e = 0; e < 16; ++e) __stcg(rec + lane * 16 + e, o[j][e]);
      if (lane == 0) {
        __stcg(rec + kl, m[j]);
        __stcg(rec + kl + 1, l[j]);
      }
    }
  }
}

// instruction (a = head h, b = 64-row block of v_head): out[n][h * v_head + j] = W_UV[h][j] . o_lat[n][h].
// Warp w owns 8 rows j (v_head is a multiple of 16, so a warp's rows are all valid or all past the end);
// lane L holds latent dims [16L, 16L + 16) of each row, loaded together up front.
__device__ __noinline__ void mla_uv_consume(const KParams& p, const OpDesc& op, const Instr& in, int ctid) {
  const int warp = ctid >> 5, lane = ctid & 31;
  const int h = in.a, jb = in.b;
  const int kl = op.kv_lora, vh = op.v_head;
  const int N = p.N;
  const int j0 = jb * 64 + warp * 8;
  if (j0 >= vh) return;
  uint32_t ws[8][8];
#pragma unroll
  for (int jj = 0; jj < 8; ++jj) {
    const uint16_t* wrow = op.w_uv + ((size_t)h * vh + j0 + jj) * kl + lane * 16;
    const uint4 a0 = __ldg(reinterpret_cast<const uint4*>(wrow));
    const uint4 a1 = __ldg(reinterpret_cast<const uint4*>(wrow + 8));
    ws[jj][0] = a0.x; ws[jj][1] = a0.y; ws[jj][2] = a0.z; ws[jj][3] = a0.w;
    ws[jj][4] = a1.x; ws[jj][5] = a1.y; ws[jj][6] = a1.z; ws[jj][7] = a1.w;
  }
  for (int n = 0; n < N; ++n) {
    const float* ol = op.in + (size_t)n * op.in_stride + (size_t)h * kl + lane * 16;
    float o[16];
#pragma unroll
    for (int e = 0; e < 16; e += 4) {
      const float4 t = __ldcg(reinterpret_cast<const float4*>(ol + e));
      o[e] = t.x; o[e + 1] = t.y; o[e + 2] = t.z; o[e + 3] = t.w;
    }
    float v[8];
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      float d = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        d = fmaf(bf_lo(ws[jj][e]), o[2 * e], d);
        d = fmaf(bf_hi(ws[jj][e]), o[2 * e + 1], d);
      }
      v[jj] = d;
    }
    MultiReduce<8, 16>::run(v, lane);  // lane 4i: row i
    if ((lane & 3) == 0) __stcg(op.out + (size_t)n * op.out_stride + (size_t)h * vh + j0 + (lane >> 2), v[0]);
  }
}

// ------------------------------------------------------------------------------------------------
// Producer: the chunks of an SM's queue, in the order its consumers read them. A cursor walks them and the
// producer loads each chunk into the ring.
// ------------------------------------------------------------------------------------------------
struct ChunkCursor {
  int qi, q0, q1;
  int step;  // decode step of a multi-step launch: the queue is walked once per step
  int kind;  // 0: load the next instruction, 1: GEMV chunks, 2: attention KV chunks, 4: expert rows
  const OpDesc* op;
  // GEMV walk over packed row blocks, in the consumers' order (row groups, K parts, blocks, atoms): the
  // instruction's end row, the row group [g0, g1), the K part (first atom a0, KP atoms; the whole K on the
  // mma.sync path, whose row groups are single blocks), the block [r, rnext) with bP physical rows, bat atoms
  // per chunk and its first byte; the next atom cc and the last chunk's atoms na (adv = 1: step past it)
  int adv, rb, g0, g1, a0, r, rnext, cc, na, nat, KP, tc, bP, bat;
  const uint8_t* bsrc;
  // attention walk: next position, end, positions per chunk, bytes per position, this lane's base,
  // number of copies per chunk (2: K and V of GQA; 1: the MLA latent)
  int t, t1, P, pos_bytes, ncopy;
  const uint16_t* kv;
  // MoE walk: the instruction's rows (first row, count, group rows, groups), K and slice width, passes,
  // selected expert slot, count, format, up / down; pass, row group, first input of the next slice, physical
  // rows of the group; this lane's weight row (codes) and scale row; the step's expert union, copied into
  // shared memory when the walk reaches an expert op
  int a, n, glog, ng, K, kc, passes;
  int j, nsel, fp4, up;
  int pass, grp, k0, nphys;
  int32_t* uni;
  const uint8_t* mw;
  const uint8_t* ms;
};

// the GEMV walk's current block: rows [c.r, ...) of the current row group
__device__ __forceinline__ void cursor_block(ChunkCursor& c) {
  PkBlock blk;
  c.rnext = pk_block(*c.op, c.r, c.g1, blk);
  c.bP = blk.P;
  c.bat = blk.atoms;
  c.bsrc = pk_block_src(*c.op, c.r, blk);
}
// end of the GEMV walk's row group starting at g0: TMEM-sized on the tcgen05 path, one block on mma.sync
__device__ __forceinline__ int cursor_group_end(const ChunkCursor& c) {
  return c.tc ? tc_group_end(*c.op, c.g0, c.rb) : min(c.rb, c.g0 + pk_block_lrows(c.op->out_kind == OUT_SWIGLU));
}

__device__ __forceinline__ void cursor_moe_group(const KParams& p, ChunkCursor& c, int lane) {
  const int g0 = gemv_group_row(c.a, c.n, c.ng, c.grp);
  const int nl = gemv_group_row(c.a, c.n, c.ng, c.grp + 1) - g0;
  c.nphys = c.up ? 2 * nl : nl;
  const int pr = c.fp4 ? (lane & 15) : lane;  // NVFP4: lanes 16..31 copy the scale rows
  c.mw = nullptr;
  c.ms = nullptr;
  if (pr < c.nphys) {
    const int m = (c.up && pr >= nl) ? 1 : 0;
    const int r = g0 + (m ? pr - nl : pr);
    const ExpertRow er = expert_row(p, *c.op, c.j, m, r, c.K, c.uni);
    c.mw = er.w;
    c.ms = er.s;
  }
}

// This lane's copy of the next chunk (bytes = 0: none) and the chunk's total bytes; false at the end.
__device__ __forceinline__ bool cursor_next(const KParams& p, ChunkCursor& c, int lane, const void*& src,
                                            uint32_t& bytes, uint32_t& dst, uint32_t& total) {
  for (;;) {
    if (c.kind == 0) {
      if (c.qi >= c.q1) {
        if (c.step + 1 >= p.n_steps) return false;
        ++c.step;
        c.qi = c.q0;
        continue;
      }
      const Instr in = p.instrs[c.qi];
      const OpDesc& op = p.ops[in.op];
      c.op = &op;
      const int type = op.type;
      if (type == OP_GEMV) {
        if (in.b <= in.a) {
          ++c.qi;
          continue;
        }
        c.rb = in.b;
        c.tc = op.mma == 2 ? 1 : 0;
        c.nat = tc_atoms(op);
        c.KP = c.tc ? tc_part(op) : c.nat;
        c.g0 = in.a;
        c.g1 = cursor_group_end(c);
        c.a0 = 0;
        c.r = in.a;
        cursor_block(c);
        c.cc = 0;
        c.adv = 0;
        c.kind = 1;
      } else if (type == OP_ATTN) {
        const int hkv = op.n_kv_heads, hd = op.head_dim;
        const int b = in.a / hkv, g = in.a % hkv;
        attn_range(p, op, b, in.b, c.step, c.t, c.t1);
        c.P = kChunkBytes / (4 * hd);
        c.pos_bytes = hd * 2;
        c.ncopy = 2;
        c.kv = (lane == 0) ? p.kcache + kv_index(p, op, b, g, 0) : p.vcache + kv_index(p, op, b, g, 0);
        c.kind = 2;
      } else if (kFull && type == OP_MLA_ATTN) {
        const int b = in.a / op.n_kv_heads;
        const int ldl = op.kv_lora + op.rope;
        attn_range(p, op, b, in.b, c.step, c.t, c.t1);
        c.P = kChunkBytes / (2 * ldl);
        c.pos_bytes = ldl * 2;
        c.ncopy = 1;
        c.kv = p.latent + lat_index(p, op, b, 0);
        c.kind = 2;
      } else if (kFull && (type == OP_MOE_UP || type == OP_MOE_DOWN)) {
        // the expert list is known once the router op has finished
        int ok = 1;
        if (lane == 0)
          ok = wait_counter(&p.counters[op.route_op], (uint32_t)p.ops[op.route_op].n_instr * (uint32_t)(c.step + 1), p) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) return false;
        c.up = type == OP_MOE_UP;
        c.fp4 = op.fp4;
        c.glog = c.up ? op.rg / 2 : op.rg;
        c.a = in.a;
        c.n = in.b - in.a;
        c.ng = gemv_ngroups(c.n, c.glog);
        c.K = c.up ? p.d : op.F;
        c.kc = op.kc;
        c.passes = op.passes;
        const int ucount = __ldcg(p.union_list);
        for (int i = lane; i <= ucount; i += 32) c.uni[i] = __ldcg(p.union_list + i);
        __syncwarp();
        c.nsel = op.n_shared + ucount;
        c.j = c.pass = c.grp = c.k0 = 0;
        if (c.ng == 0 || c.nsel == 0) {
          ++c.qi;
          continue;
        }
        cursor_moe_group(p, c, lane);
        c.kind = 4;
      } else {
        ++c.qi;
        continue;
      }
    }
    if (c.kind == 1) {
      if (c.adv) {  // step past the chunk returned last time: atoms, blocks, K parts, row groups
        c.adv = 0;
        c.cc += c.na;
        if (c.cc >= min(c.nat, c.a0 + c.KP)) {
          c.r = c.rnext;
          if (c.r >= c.g1) {
            c.a0 += c.KP;
            if (c.a0 >= c.nat) {
              c.a0 = 0;
              c.g0 = c.g1;
              if (c.g0 >= c.rb) {
                c.kind = 0;
                ++c.qi;
                continue;
              }
              c.g1 = cursor_group_end(c);
            }
            c.r = c.g0;
          }
          cursor_block(c);
          c.cc = c.a0;
        }
      }
      // one contiguous copy of the block's atoms [cc, cc + na)
      c.na = min(c.bat, min(c.nat, c.a0 + c.KP) - c.cc);
      total = (uint32_t)(c.na * c.bP * 128);
      src = c.bsrc + (size_t)c.cc * c.bP * 128;
      bytes = lane == 0 ? total : 0u;
      dst = 0;
      c.adv = 1;
      return true;
    }
    if (kFull && c.kind == 4) {
      const int kw = min(c.kc, c.K - c.k0);
      bytes = 0;
      if (c.fp4) {
        const int pitch = kw / 2 + kw / 16;  // row layout in the slot: codes, then block scales
        total = (uint32_t)(c.nphys * pitch);
        if (c.mw) {
          if (lane < 16) {
            src = c.mw + c.k0 / 2;
            bytes = (uint32_t)(kw / 2);
            dst = (uint32_t)(lane * pitch);
          } else {
            src = c.ms + c.k0 / 16;
            bytes = (uint32_t)(kw / 16);
            dst = (uint32_t)((lane - 16) * pitch + kw / 2);
          }
        }
      } else {
        total = (uint32_t)(c.nphys * kw * 2);
        if (c.mw) {
          src = c.mw + (size_t)c.k0 * 2;
          bytes = (uint32_t)(kw * 2);
          dst = (uint32_t)(lane * kw * 2);
        }
      }
      c.k0 += c.kc;
      if (c.k0 >= c.K) {
        c.k0 = 0;
        if (++c.grp >= c.ng) {
          c.grp = 0;
          if (++c.pass >= c.passes) {
            c.pass = 0;
            if (++c.j >= c.nsel) {
              c.kind = 0;
              ++c.qi;
              return true;
            }
          }
        }
        cursor_moe_group(p, c, lane);
      }
      return true;
    }
    // attention: K then V (GQA) or the latent (MLA) of up to P positions
    if (c.t >= c.t1) {
      c.kind = 0;
      ++c.qi;
      continue;
    }
    const int np = min(c.P, c.t1 - c.t);
    const uint32_t nb = (uint32_t)(np * c.pos_bytes);
    total = c.ncopy * nb;
    bytes = (lane < c.ncopy) ? nb : 0;
    src = reinterpret_cast<const uint8_t*>(c.kv) + (size_t)c.t * c.pos_bytes;
    dst = (lane == 1) ? kChunkBytes / 2 : 0;
    c.t += c.P;
    return true;
  }
}

// ------------------------------------------------------------------------------------------------
// final op: greedy argmax over the LM-head partials, sequence bookkeeping, counter reset
// ------------------------------------------------------------------------------------------------
__device__ MK_OUTLINE void final_consume(const KParams& p, CSmem& cs, int step, int ctid) {
  if (p.argmax || p.accept_out) {
    const int warp = ctid >> 5, lane = ctid & 31;
    for (int n = warp; n < p.N; n += kConsumerWarps) {
      float bv = -CUDART_INF_F;
      int bi = 0x7fffffff;
      for (int q = lane; q < p.n_sm; q += 32) {
        const float2 c = __ldcg(&p.amax_part[(size_t)q * kMaxN + n]);
        const int ci = __float_as_int(c.y);
        if (c.x > bv || (c.x == bv && ci < bi)) { bv = c.x; bi = ci; }
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
      }
      if (lane == 0) {
        if (p.argmax) __stcg(p.argmax + (size_t)step * p.N + n, bi);
        cs.best_idx[n] = bi;
      }
    }
  }
  if (p.accept_out && p.R > 1) {
    // greedy acceptance of a verify block (row 0 the anchor, rows 1.. the drafts): draft r + 1 is accepted
    // while it equals the greedy target of row r; the accepted prefix plus the target after it (the bonus
    // token) is what the block emits (Kimi K3's TPU megakernel, "What DSpark changes per step")
    consumer_sync();
    if (ctid < p.B) {
      const int b = ctid, R = p.R;
      int a = 1;
      while (a < R && cs.best_idx[b * R + a - 1] == p.tokens[b * p.tok_stride + a]) ++a;
      p.accept_out[b] = a;
      p.accept_out[p.B + b] = cs.best_idx[b * R + a - 1];
      p.accept_out[2 * p.B + b] = seq_pos(p, b, step) + a;
    }
  }
  if (ctid < p.B) {
    const int pos = seq_pos(p, ctid, step);
    SeqState s;
    s.c_int = pos;
    s.u_int = p.R;
    s.c_spec = p.commit_all ? pos + p.R : pos;
    s.pad = 0;
    p.seq[ctid] = s;
  }
  // the last step leaves the counters at zero for the next launch (every other CTA is done by now)
  if (step == p.n_steps - 1)
    for (int i = ctid; i < p.n_ops; i += kConsumerThreads) p.counters[i] = 0u;
}

// ------------------------------------------------------------------------------------------------
// the two roles
// ------------------------------------------------------------------------------------------------
__device__ void run_producer(const KParams& p, const Ring& rg, int q0, int q1, int32_t* uni) {
  const int lane = threadIdx.x & 31;
  uint32_t chunk = 0;
  const uint32_t ring_base = smem_u32(rg.base);
  ChunkCursor mc;
  mc.qi = q0;
  mc.q0 = q0;
  mc.q1 = q1;
  mc.step = 0;
  mc.kind = 0;
  mc.uni = uni;
  const void* src = nullptr;
  uint32_t bytes = 0, dst = 0, total = 0;
  int last_qi = -1;
  while (cursor_next(p, mc, lane, src, bytes, dst, total)) {
    if (p.trace && lane == 0 && mc.step == 0 && mc.qi != last_qi) {
      p.trace[(size_t)mc.qi * kTraceWords + 3] = global_timer();
      last_qi = mc.qi;
    }
    if (!ring_acquire(rg, chunk, total, p, lane)) break;
    if (bytes) bulk_g2s(ring_base + (chunk % kSlots) * kSlotBytes + dst, src, bytes, &rg.full[chunk % kSlots]);
    ++chunk;
  }
  // every issued copy must land before the CTA may exit
  if (lane == 0) {
    const uint32_t first = chunk > (uint32_t)kSlots ? chunk - kSlots : 0u;
    for (uint32_t c = first; c < chunk; ++c) {
      const unsigned long long t0 = global_timer();
      while (!mbar_try_wait(&rg.full[c % kSlots], (c / kSlots) & 1u)) {
        if (global_timer() - t0 > 200000000ull) break;
      }
    }
  }
  __syncwarp();
}


// The MLA and MoE ops (full variant only).
__device__ __forceinline__ void run_full_op(const KParams& p, const OpDesc& op, const Instr& in, const Ring& rg,
                                            uint32_t& chunk, CSmem& cs, uint16_t* act, float* actf, int nr, int step,
                                            int ctid) {
  switch (op.type) {
      case OP_ROUTE: route_consume(p, op, actf, step, ctid); break;
      case OP_MOE_UP:
      case OP_MOE_DOWN:
        if (op.fp4) {
          if (op.staged) {
            if (nr == 1) moe_consume<16, 1, 8, true, true>(p, op, in, rg, chunk, cs, actf, ctid);
            else moe_consume<16, 2, 8, true, true>(p, op, in, rg, chunk, cs, actf, ctid);
          } else if (nr == 4) {
            moe_consume<16, 4, 8, true, false>(p, op, in, rg, chunk, cs, actf, ctid);
          } else {
            moe_consume<8, 8, 8, true, false>(p, op, in, rg, chunk, cs, actf, ctid);
          }
        } else {
          if (op.staged) {
            if (nr == 1) moe_consume<16, 1, 4, false, true>(p, op, in, rg, chunk, cs, actf, ctid);
            else moe_consume<16, 2, 4, false, true>(p, op, in, rg, chunk, cs, actf, ctid);
          } else if (nr == 4) {
            moe_consume<16, 4, 4, false, false>(p, op, in, rg, chunk, cs, actf, ctid);
          } else {
            moe_consume<8, 8, 8, false, false>(p, op, in, rg, chunk, cs, actf, ctid);
          }
        }
        break;
      case OP_MLA_PREP: mla_prep_consume(p, op, step, ctid); break;
      case OP_MLA_QABS: mla_qabs_consume(p, op, in, step, ctid); break;
      case OP_MLA_ATTN:
        if (((in.c >> 8) - (in.c & 0xff)) <= 1) mla_attn_consume<1>(p, op, in, rg, chunk, act, step, ctid);
        else mla_attn_consume<2>(p, op, in, rg, chunk, act, step, ctid);
        break;
      case OP_MLA_UV: mla_uv_consume(p, op, in, ctid); break;
    default: break;
  }
}

__device__ void run_consumer(const KParams& p, const Ring& rg, CSmem& cs, uint16_t* act, TcState& ts, int q0, int q1,
                             int ctid) {
  uint32_t chunk = 0;
  float* actf = reinterpret_cast<float*>(act);
  const int nr = p.N <= 1 ? 1 : p.N <= 2 ? 2 : p.N <= 4 ? 4 : 8;
  const bool trace = p.trace != nullptr;
  for (int step = 0; step < p.n_steps; ++step) {
  for (int qi = q0; qi < q1; ++qi) {
    const Instr in = p.instrs[qi];
    const OpDesc& op = p.ops[in.op];
    if (ctid == 0) {
      int ok = 1;
      if (trace && step == 0) p.trace[(size_t)qi * kTraceWords + 0] = global_timer();
      // counters accumulate over the steps of a launch: op k of step s needs n_instr * (s + 1) completions
      for (int d = 0; d < op.n_deps && ok; ++d) {
        const int dop = op.deps[d];
        ok = wait_counter(&p.counters[dop], (uint32_t)p.ops[dop].n_instr * (uint32_t)(step + 1), p) ? 1 : 0;
      }
      // the embedding of step s reads the greedy tokens the final op of step s - 1 wrote
      if (ok && step > 0 && op.type == OP_EMBED)
        ok = wait_counter(&p.counters[p.n_ops - 1], (uint32_t)step, p) ? 1 : 0;
      if (*reinterpret_cast<volatile int32_t*>(p.abort_flag) != 0) ok = 0;
      if (trace && step == 0) p.trace[(size_t)qi * kTraceWords + 1] = global_timer();
      cs.flag = ok;
    }
    consumer_sync();
    if (!cs.flag) return;
    switch (op.type) {
      case OP_EMBED: embed_consume(p, op, in, step, ctid); break;
      case OP_GEMV:
        if (op.mma == 2) {
          gemv_tc_consume(p, op, in, rg, chunk, cs, reinterpret_cast<uint8_t*>(act), ts,
                          (trace && step == 0) ? p.trace + (size_t)qi * kTraceWords : nullptr, ctid);
        } else {
          gemv_mma_consume(p, op, in, rg, chunk, cs, actf, ctid);
        }
        break;
      case OP_ROPE_APPEND: rope_append_consume(p, op, step, ctid); break;
      case OP_ATTN: {
        const int pairs = ((in.c >> 8) - (in.c & 0xff)) * op.groups;
        const int J = (pairs + kConsumerWarps - 1) / kConsumerWarps;
        if (op.head_dim == 256) {
          if (J <= 1) attn_consume<8, 1>(p, op, in, rg, chunk, cs, act, step, ctid);
          else if (J <= 2) attn_consume<8, 2>(p, op, in, rg, chunk, cs, act, step, ctid);
          else attn_consume<8, 4>(p, op, in, rg, chunk, cs, act, step, ctid);
        } else if (op.head_dim == 128) {
          if (J <= 1) attn_consume<4, 1>(p, op, in, rg, chunk, cs, act, step, ctid);
          else if (J <= 2) attn_consume<4, 2>(p, op, in, rg, chunk, cs, act, step, ctid);
          else attn_consume<4, 4>(p, op, in, rg, chunk, cs, act, step, ctid);
        } else {
          if (J <= 1) attn_consume<2, 1>(p, op, in, rg, chunk, cs, act, step, ctid);
          else if (J <= 2) attn_consume<2, 2>(p, op, in, rg, chunk, cs, act, step, ctid);
          else attn_consume<2, 4>(p, op, in, rg, chunk, cs, act, step, ctid);
        }
        break;
      }
      case OP_ATTN_COMBINE:
        if (kFull && op.head_dim == 512) attn_combine_consume<16>(p, op, in, actf, ctid);
        else if (op.head_dim == 256) attn_combine_consume<8>(p, op, in, actf, ctid);
        else if (op.head_dim == 128) attn_combine_consume<4>(p, op, in, actf, ctid);
        else attn_combine_consume<2>(p, op, in, actf, ctid);
        break;
      case OP_ROUTE:
      case OP_MOE_UP:
      case OP_MOE_DOWN:
      case OP_MLA_PREP:
      case OP_MLA_QABS:
      case OP_MLA_ATTN:
      case OP_MLA_UV:
        if constexpr (kFull) run_full_op(p, op, in, rg, chunk, cs, act, actf, nr, step, ctid);
        break;
      case OP_DELTA:
        if (op.col_group == 8) delta_consume<1>(p, op, in, cs, reinterpret_cast<float*>(act), step, ctid);
        else if (op.col_group == 16) delta_consume<2>(p, op, in, cs, reinterpret_cast<float*>(act), step, ctid);
        else if (op.col_group == 32) delta_consume<4>(p, op, in, cs, reinterpret_cast<float*>(act), step, ctid);
        else if constexpr (!kFull)  // (the full build's column groups stop at 32)
          delta_consume<8>(p, op, in, cs, reinterpret_cast<float*>(act), step, ctid);
        break;
      case OP_FINAL: final_consume(p, cs, step, ctid); break;
      default: break;
    }
    // every thread's writes must precede the completion signal; an mma.sync GEMV with a residual or logits
    // output ends with a barrier and warp-0-only writes of its own, so it skips this one
    if (!(op.type == OP_GEMV && op.mma != 2 && (op.out_kind == OUT_RESID || op.out_kind == OUT_LOGITS)))
      consumer_sync();
    if (ctid == 0 && (op.type != OP_FINAL || step + 1 < p.n_steps)) {
      // the release add orders every consumer thread's writes before it: they precede the barrier above, and a
      // release is cumulative over what its thread has synchronised with (a separate fence measured slower)
      red_release_add(&p.counters[in.op], 1u);
    }
    if (ctid == 0 && trace && step == 0) p.trace[(size_t)qi * kTraceWords + 2] = global_timer();
  }
  }
}

// 1 = run, 0 = invalid input, 2 = abort already raised
__device__ int validate(const KParams& p) {
  if (*reinterpret_cast<volatile int32_t*>(p.abort_flag) != 0) return 2;
  for (int b = 0; b < p.B; ++b) {
    const int pos = p.positions[b];
    const SeqState s = p.seq[b];
    if (pos < 0 || pos < s.c_spec || pos > s.c_int + s.u_int || pos + p.R + p.n_steps - 1 > p.max_ctx) return 0;
    for (int r = 0; r < p.R; ++r) {
      const int t = p.tokens[b * p.tok_stride + r];
      if (t < 0 || t >= p.V) return 0;
    }
  }
  return 1;
}

__global__ void __launch_bounds__(kThreads, 1) megakernel(const __grid_constant__ KParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Ring rg;
  rg.base = smem;
  rg.full = reinterpret_cast<uint64_t*>(smem + kBarOff);
  rg.empty = rg.full + kSlots;
  CSmem& cs = *reinterpret_cast<CSmem*>(smem + kCSmemOff);
  uint16_t* act = reinterpret_cast<uint16_t*>(smem + kActOff);
  __shared__ int s_state;
  const int tid = threadIdx.x;
  if (tid == 0) {
    s_state = validate(p);
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&rg.full[i], 1);
      mbar_init(&rg.empty[i], kConsumerWarps);
    }
    if (p.use_tc) {
      mbar_init(&cs.tcbar[0], kConsumerThreads - 32);  // staged-activation buffer ready: warps 1..7 arrive
      mbar_init(&cs.tcbar[1], kConsumerThreads - 32);
      for (int i = 2; i < 6; ++i) mbar_init(&cs.tcbar[i], 1);  // arrivals by tcgen05.commit
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (s_state != 1) {
    if (s_state == 0 && blockIdx.x == 0 && tid == 0) atomicCAS(p.status, 0, kStatusDevice);
    return;
  }
  // TMEM for the tcgen05 GEMV accumulators: one CTA per SM, so the 512 columns are always free here
  if (p.use_tc && tid < 32) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&cs.tmem_base)),
                 "r"(kTcCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int q0 = p.qoff[blockIdx.x], q1 = p.qoff[blockIdx.x + 1];
  if (tid >= kConsumerThreads) {
    run_producer(p, rg, q0, q1, cs.uni_p);
  } else {
    TcState ts;
    ts.tmem = p.use_tc ? cs.tmem_base : 0u;
    ts.kp = 0;
    ts.rg = 0;
    run_consumer(p, rg, cs, act, ts, q0, q1, tid);
    if (p.use_tc) {
      // every MMA this CTA issued has completed (bounded wait, also after an abort), then free the TMEM
      if (tid == 0) {
        umma_commit(&cs.tcbar[5]);
        const unsigned long long t0 = global_timer();
        while (!mbar_try_wait(&cs.tcbar[5], 0)) {
          if (global_timer() - t0 > 200000000ull) break;
        }
      }
      tc_fence_before();
      consumer_sync();
      tc_fence_after();
      if (tid < 32)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(cs.tmem_base), "r"(kTcCols) : "memory");
    }
  }
}

}  // namespace MK_VARIANT_NS

#if !MK_VARIANT_FULL
// ------------------------------------------------------------------------------------------------
// helper kernels (set-up, not on the decode path)
// ------------------------------------------------------------------------------------------------
__global__ void rope_table_kernel(float2* tab, int max_ctx, int rot_dim, double theta) {
  const int half = rot_dim / 2;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= max_ctx * half) return;
  const int pos = i / half, k = i % half;
  const double ang = (double)pos * pow(theta, -2.0 * (double)k / (double)rot_dim);
  double s, c;
  sincos(ang, &s, &c);
  tab[i] = make_float2((float)c, (float)s);
}

// The tiled copy of one GEMV weight group (layout in mk_internal.h): one thread per 16-byte piece, read from
// the caller's row-major matrices; zeros past K and past the group's last row.
__global__ void pack_gemv_kernel(uint8_t* dst, PackSrc s, long long pieces) {
  const long long id = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (id >= pieces) return;
  const int A = pk_atoms(s.K), mc = s.swiglu ? 2 : 1;
  const int c = (int)(id & 7);
  long long rest = id >> 3;
  const int a = (int)(rest % A);
  rest /= A;
  const int m = (int)(rest % mc);
  const int r = (int)(rest / mc);
  // the block holding logical row r: its SM's share is cut into blocks from the share's first row
  const int sm = pk_sm_of(s.rows, s.n_sm, r);
  const int a_s = pk_split(s.rows, s.n_sm, sm), b_s = pk_split(s.rows, s.n_sm, sm + 1);
  const int br = pk_block_lrows(s.swiglu);
  const int bs = a_s + (r - a_s) / br * br;
  const int be = min(b_s, bs + br);
  const int rows8 = (be - bs + 7) & ~7;
  const int P = rows8 * mc;
  const int prow = m * rows8 + (r - bs);
  const size_t off = (size_t)bs * A * 128 * mc + (size_t)a * P * 128 + (size_t)prow * 128 + (size_t)((c ^ (prow & 7)) << 4);
  uint16_t v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  const int k = a * 64 + c * 8;
  if (r < s.rows && k < s.K) {
    const uint16_t* row;
    if (s.swiglu) {
      row = s.w[m] + (size_t)r * s.K;
    } else {
      int rr = r, mm = 0;
      while (mm < s.n_mat - 1 && rr >= s.mat_rows[mm]) rr -= s.mat_rows[mm++];
      row = s.w[mm] + (size_t)rr * s.K;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (k + j < s.K) v[j] = row[k + j];
  }
  uint4 o;
  o.x = v[0] | ((uint32_t)v[1] << 16);
  o.y = v[2] | ((uint32_t)v[3] << 16);
  o.z = v[4] | ((uint32_t)v[5] << 16);
  o.w = v[6] | ((uint32_t)v[7] << 16);
  *reinterpret_cast<uint4*>(dst + off) = o;
}

__global__ void fill_i32_kernel(int32_t* dst, int n, int32_t value) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) dst[i] = value;
}
#endif

}  // namespace mk

// ---- host-side launch wrappers (used by mk_host.cu) ---------------------------------------------
namespace mk {
namespace MK_VARIANT_NS {

size_t kernel_smem_bytes() { return kSmemBytes; }

cudaError_t kernel_configure() {
  return cudaFuncSetAttribute(megakernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
}

cudaError_t kernel_launch(const KParams& p, int n_sm, cudaStream_t stream) {
  void* args[] = {const_cast<KParams*>(&p)};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(megakernel), dim3(n_sm), dim3(kThreads), args,
                                     kSmemBytes, stream);
}

}  // namespace MK_VARIANT_NS

#if !MK_VARIANT_FULL
cudaError_t rope_table_launch(float2* tab, int max_ctx, int rot_dim, double theta, cudaStream_t stream) {
  const int n = max_ctx * (rot_dim / 2);
  rope_table_kernel<<<(n + 255) / 256, 256, 0, stream>>>(tab, max_ctx, rot_dim, theta);
  return cudaGetLastError();
}

cudaError_t pack_gemv_launch(uint8_t* dst, const PackSrc& src, cudaStream_t stream) {
  const long long pieces = pk_bytes(src.rows, src.K, src.swiglu) / 16;
  if (pieces == 0) return cudaSuccess;
  pack_gemv_kernel<<<(unsigned)((pieces + 255) / 256), 256, 0, stream>>>(dst, src, pieces);
  return cudaGetLastError();
}

cudaError_t fill_i32_launch(int32_t* dst, int n, int32_t value, cudaStream_t stream) {
  fill_i32_kernel<<<(n + 255) / 256, 256, 0, stream>>>(dst, n, value);
  return cudaGetLastError();
}
#endif

}  // namespace mk
