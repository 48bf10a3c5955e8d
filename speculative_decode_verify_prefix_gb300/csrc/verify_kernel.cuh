// Device code of the split-KV verify attention for EAGLE target-verify at
// topk = 1, for GB300 (sm_103a): parameters, PTX wrappers and the kernel
// templates.  Each head_dim's kernels are instantiated in their own
// translation unit (vsk_inst_*.cu, compiled in parallel); the host side is
// verify_splitkv.cu.  The operation is defined on the sglang "verify_splitkv.py" page
// (module docstring; "_verify_prefix_stage1" computes per-split partial
// softmaxes over the gathered prefix with qk *= sm_scale * k_scale and
// acc *= v_scale; "_verify_combine_stage2" merges the splits by log-sum-exp,
// adds the causal draft-draft block without scales and merges again).  The
// C ABI is declared in include/verify_splitkv.h.
//
// GB300 design (not the page's two-kernel Triton layout):
//   * ONE persistent kernel per call.  The flattened work space (sequence b,
//     KV-head group hg, prefix token t) is cut into equal contiguous shares,
//     one per CTA; grid = SMs x CTAs-per-SM from static shapes, the split
//     itself is computed on the device from kv_indptr (or seq_lens), so no
//     host synchronisation is needed.
//   * A CTA serves a group of KV heads.  The packed queries of a head (all
//     h_q/h_kv query heads x l_ext draft rows) form 16-row tiles; a warp owns
//     one head and one or two tiles, so each K/V byte is read from HBM once.
//     The warps of a head stream its K and V row slices themselves with
//     16-byte cp.async into the head's XOR-swizzled ring (indices or page ids
//     prefetched by cp.async, completion by wait_group: no producer warp, no
//     mbarrier, no spin-wait) and run mma.sync m16n8k16 for QK and PV (bf16;
//     f16 straight from e4m3 rows for an fp8 pool) with an fp32 online
//     softmax.
//   * Piece ends only write log-sum-exp partials.  After streaming, the CTA
//     that draws a segment's last ticket (atomic, no wait) merges the pieces
//     in CTA order (in two levels for long segments) and continues the same
//     online softmax over the draft keys (causal, tree mask, or drafts read
//     from a paged cache; optionally storing new drafts into the cache), then
//     writes bf16 output.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <climits>
#include <cstdint>
#include <type_traits>

namespace vsk {

// ---------------------------------------------------------------------------
// Constants shared by the host plan and the kernel.
// ---------------------------------------------------------------------------
constexpr int kStageTokens = 16;     // prefix tokens per pipeline stage (one mma k-step)
constexpr int kMaxStages = 7;        // ring depth cap (kIdxAhead >= stages - 1)
constexpr int kIdxAhead = 6;         // stages of kv_indices prefetched ahead of the copies (< kIdxRing)
constexpr int kIdxRing = 8;          // per-warp index ring entries (> kIdxAhead)
// the index of a stage lands before its copies are issued (kIdxAhead >= the
// stages in flight), its ring entry lives until then (kIdxRing > kIdxAhead),
// and the 16-entry valid-token mask ring covers every stage in flight
static_assert(kIdxAhead >= kMaxStages - 1 && kIdxRing > kIdxAhead && kMaxStages <= 16, "ring invariants");
constexpr int kCtlBytes = 256;       // control block before the warp regions
constexpr int kSmemPerSM = 233472;   // 228 KB per SM
constexpr int kSmemPerCTAMax = 232448;  // 227 KB opt-in per CTA
constexpr int kReservedPerCTA = 1024;
constexpr int kTicketBytes = 65536;   // minimum ticket region at the end of a workspace
constexpr float kLazy = 8.f;          // log2 headroom before a running maximum is raised
constexpr int kGroup = 4;             // pieces per group of a two-level merge
constexpr int kTreeMin = 6;           // segments of more pieces merge in two levels

enum : unsigned {
  kErrBadIndex = 1u,
  kErrBadKvIndptr = 2u,
  kErrBadQoIndptr = 4u,
  kErrTimeout = 8u,
  kErrBadMaskIndptr = 16u,
};

struct Params {
  const __nv_bfloat16* q;  long long q_s0, q_s1;
  const __nv_bfloat16* ke; long long ke_s0, ke_s1;
  const __nv_bfloat16* ve; long long ve_s0, ve_s1;
  __nv_bfloat16* o;        long long o_s0, o_s1;
  const unsigned char* kb; long long kb_s0, kb_s1;  // byte strides
  const unsigned char* vb; long long vb_s0, vb_s1;  // byte strides
  const int* qo;
  const int* kvp;
  const void* kvi;
  int idx64;
  long long n_idx, pool, n_rows;
  int B, L, gq, R, HC, MT, n_hg, nwc, nst;
  int ring_off, head_bytes;  // ring of KV head hc at ring_off + hc * head_bytes
  int misc_off, misc_bytes;  // warp w's index / mask rings (and query tiles) at misc_off + w * misc_bytes
  float scale2, dscale2, v_scale;
  float dvs;  // multiplier of draft values (v_scale when drafts come from the cache)
  // drafts already in a paged cache: block table of page ids, prefix lengths
  int paged;
  const int* bt;
  long long bt_s0;
  int bt_cols, page;
  unsigned pg_m;  // division by page: t / page == (umulhi(t, pg_m) + t) >> pg_l for 0 <= t < 2^31
  int pg_l;
  const int* slens;
  // fused store of the new draft K/V (ke / ve) into the cache: 0 none,
  // 1 rows out_cache_loc[s_b + t], 2 paged positions P + t (attention then
  // uses the stored, dequantised values)
  int wmode;
  const void* ocl;
  int ocl64;
  unsigned char* kw;  // the same caches as kb / vb, writable
  unsigned char* vw;
  float kq, vq;       // dequantisation scales the stored codes are divided by
  long long w_min;
  int n_stream;  // CTAs of the stream launch (read by the combine kernel of the two-launch forms)
  int cl;        // cluster form: CTAs per cluster (one cluster per segment); 0 otherwise
  int cl_smem;   // cluster form: shared-memory bytes of one combine group (128 threads)
  int cmb_nb;    // combine: pieces staged per batch (two batches in flight), 1 .. 32
  const unsigned char* cmask;  // tree verify: per-sequence [L][P+L] draft visibility (nullptr: causal)
  const void* mindptr;
  int mindptr64;
  long long n_mask;
  unsigned* err;
  int* cnt;       // [nseg] segment tickets, then [n_cta + nseg] group tickets (one per slot)
  long long nseg;
  float* plse;
  float* po;
};

// ---------------------------------------------------------------------------
// PTX wrappers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// L2 policy for the per-piece partials: kept in L2 until the segment's
// finisher reads them back, while the K/V stream is marked evict-first.
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void st_keep(float* a, float x, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(a), "f"(x), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_keep2(float* a, float x, float y, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v2.f32 [%0], {%1, %2}, %3;" ::"l"(a), "f"(x), "f"(y), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_keep4(float* a, float x, float y, float z, float w, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(a), "f"(x), "f"(y), "f"(z), "f"(w),
               "l"(pol)
               : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void* a) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 16-byte global -> shared copy through L2 only
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
// 16-byte global -> shared copy through L2 only (zero-filled when !valid),
// with an L2 eviction-priority hint.
__device__ __forceinline__ void cp_async_16_zfill(uint32_t dst, const void* src, bool valid, uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// wait_group with a run-time count (0..3)
__device__ __forceinline__ void cp_async_wait_dyn(int n) {
  switch (n) {
    case 0: cp_async_wait<0>(); break;
    case 1: cp_async_wait<1>(); break;
    case 2: cp_async_wait<2>(); break;
    default: cp_async_wait<3>(); break;
  }
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D(16x8 fp32) += A(16x16 f16, row) * B(16x8 f16, col)
__device__ __forceinline__ void mma_f16(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D(16x8 fp32) = A(16x16 f16, row) * B(16x8 f16, col): a chain's first product
// (accumulator input zero, no zero-fill of the registers needed)
__device__ __forceinline__ void mma_f16_z(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
      : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
}

// D(16x8 fp32) = A(16x16 bf16, row) * B(16x8 bf16, col), accumulator input zero
__device__ __forceinline__ void mma_bf16_z(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
      : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
}

// D(16x8 fp32) += A(16x16 bf16, row) * B(16x8 bf16, col)
__device__ __forceinline__ void mma_bf16(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack_bf16(uint32_t w) {
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&w);
  return __bfloat1622float2(v);
}

__device__ __forceinline__ uint32_t ld_u32(const __nv_bfloat16* p) {
  return __ldg(reinterpret_cast<const unsigned int*>(p));
}

__device__ __forceinline__ float quad_max(float x) {
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 1));
  return fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 2));
}
__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  return x + __shfl_xor_sync(0xffffffffu, x, 2);
}

// 2^x with the hardware approximation (ex2.approx.ftz: about 2 ulp, -inf -> +0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// e4m3 x2 -> f16 x2, exactly (every e4m3 value is an f16 value).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(unsigned short two) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two), __NV_E4M3);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// e4m3 x2 -> bf16 x2, exactly (every e4m3 value is a bf16 value).
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(unsigned short two) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two), __NV_E4M3);
  __half2 hv = *reinterpret_cast<__half2*>(&h);
  float2 f = __half22float2(hv);
  return pack_bf16(f.x, f.y);
}

// Cache code of two values stored with dequantisation scale sc: the nearest
// e4m3 (saturating) / bf16 value of the binary32 quotient x / sc.
__device__ __forceinline__ unsigned short store_e4m3x2(float a, float b, float sc) {
  const unsigned lo = __nv_cvt_float_to_fp8(__fdiv_rn(a, sc), __NV_SATFINITE, __NV_E4M3);
  const unsigned hi = __nv_cvt_float_to_fp8(__fdiv_rn(b, sc), __NV_SATFINITE, __NV_E4M3);
  return static_cast<unsigned short>(lo | (hi << 8));
}
__device__ __forceinline__ uint32_t store_bf16x2(float a, float b, float sc) {
  return pack_bf16(__fdiv_rn(a, sc), __fdiv_rn(b, sc));
}

// ---------------------------------------------------------------------------
// Work schedule: segments (b, hg) of virtual length max(P_b, 1), laid end to
// end; CTA c owns positions [c*W, c*W + W).  Both the producer and the
// consumers walk the same sequence deterministically.
// ---------------------------------------------------------------------------
// Prefix length (and kv_indices base) of sequence b; inconsistent entries
// give an empty prefix and return false.
__device__ __forceinline__ bool seq_info(const Params& p, int b, int& P, long long& kv0) {
  if (p.paged) {
    const int n = __ldg(p.slens + b);
    const bool ok = n >= 0 && static_cast<long long>(n) + p.L <= static_cast<long long>(p.bt_cols) * p.page;
    P = ok ? n : 0;
    kv0 = 0;
    return ok;
  }
  const int a = __ldg(p.kvp + b);
  const int e = __ldg(p.kvp + b + 1);
  const bool ok = a >= 0 && e >= a && static_cast<long long>(e) <= p.n_idx;
  P = ok ? e - a : 0;
  kv0 = ok ? a : 0;
  return ok;
}

__device__ __forceinline__ void load_seq(const Params& p, int b, int& P, long long& kv0) { seq_info(p, b, P, kv0); }

// Block-table column of cache position t >= 0: multiply-high division by a
// constant (Granlund and Montgomery, "Division by invariant integers using
// multiplication", 1994), exact for every t < 2^31.
__device__ __forceinline__ int page_of(const Params& p, int t) {
  const unsigned u = static_cast<unsigned>(t);
  return static_cast<int>((__umulhi(u, p.pg_m) + u) >> p.pg_l);
}

// Pool row of cache position pos of sequence b (paged problems), or -1.
__device__ __forceinline__ long long paged_row(const Params& p, int b, int pos) {
  const int col = page_of(p, pos);
  const long long pid = __ldg(p.bt + static_cast<long long>(b) * p.bt_s0 + col);
  const long long r = pid * p.page + (pos - col * p.page);
  return (pid >= 0 && r < p.pool) ? r : -1;
}

struct Seg {
  int b, hg, len, P;
  long long kv0, off;  // off: flattened position of the segment's first token
};

__device__ __forceinline__ void seg_advance(const Params& p, Seg& s) {
  s.off += s.len;
  if (++s.hg == p.n_hg) {
    s.hg = 0;
    if (++s.b < p.B) {
      load_seq(p, s.b, s.P, s.kv0);
      s.len = max(s.P, 1);
    }
  }
}

__device__ __forceinline__ bool seg_live(const Params& p, const Seg& s, long long end) {
  return s.b < p.B && s.off < end;
}

// Stage iterator (producer): successive groups of <= 16 real prefix tokens.
struct StageIt {
  Seg s;
  int tok, te;
  bool valid;
};

__device__ __forceinline__ int piece_real_end(const Seg& s, long long end) {
  const long long t1 = min(end, s.off + s.len) - s.off;
  return static_cast<int>(min(t1, static_cast<long long>(s.P)));
}

__device__ __forceinline__ void sit_settle(const Params& p, StageIt& it, long long end) {
  while (seg_live(p, it.s, end) && it.tok >= it.te) {
    seg_advance(p, it.s);
    it.tok = 0;
    if (seg_live(p, it.s, end)) it.te = piece_real_end(it.s, end);
  }
  it.valid = seg_live(p, it.s, end);
}

// Query fragments (mma A operand, rows r0 and r0 + 8 of the packed tile) of
// one segment, straight from global memory; rows beyond R are zero.  Returns
// the segment's first draft row (qo_indptr[b], validated against l_ext).
template <int KS>
__device__ __forceinline__ int load_q(const Params& p, const Seg& s, int hc, int r0, int r1, int j, bool flag_err,
                                      uint32_t (&qf)[KS][4], int d0 = 0) {
  const int a = p.qo ? __ldg(p.qo + s.b) : s.b * p.L, e = p.qo ? __ldg(p.qo + s.b + 1) : (s.b + 1) * p.L;
  const bool ok = a >= 0 && e - a == p.L && static_cast<long long>(a) + p.L <= p.n_rows;
  if (!ok && flag_err) atomicOr(p.err, kErrBadQoIndptr);
  const int s_b = ok ? a : s.b * p.L;
  const int kvh = s.hg * p.HC + hc;
  const bool v0 = r0 < p.R, v1 = r1 < p.R;
  const __nv_bfloat16* q0 = p.q + (static_cast<long long>(s_b) + (v0 ? r0 / p.gq : 0)) * p.q_s0 +
                            static_cast<long long>(kvh * p.gq + (v0 ? r0 % p.gq : 0)) * p.q_s1 + d0;
  const __nv_bfloat16* q1 = p.q + (static_cast<long long>(s_b) + (v1 ? r1 / p.gq : 0)) * p.q_s0 +
                            static_cast<long long>(kvh * p.gq + (v1 ? r1 % p.gq : 0)) * p.q_s1 + d0;
#pragma unroll
  for (int kk = 0; kk < KS; ++kk) {
    qf[kk][0] = v0 ? ld_u32(q0 + kk * 16 + 2 * j) : 0u;
    qf[kk][1] = v1 ? ld_u32(q1 + kk * 16 + 2 * j) : 0u;
    qf[kk][2] = v0 ? ld_u32(q0 + kk * 16 + 8 + 2 * j) : 0u;
    qf[kk][3] = v1 ? ld_u32(q1 + kk * 16 + 8 + 2 * j) : 0u;
  }
  return s_b;
}

// Query fragments for an e4m3 pool: f16 operands whose contraction index is
// permuted within each 16-wide block (logical k 2j, 2j+1 -> d 4j, 4j+1 and
// k 2j+8, 2j+9 -> d 4j+2, 4j+3), the order in which K fragments come straight
// out of e4m3 rows.  The tile is scaled by 2^-sh (exact), sh chosen so that
// its largest |q| stays below 2^15, inside the f16 range; returns 2^sh.
template <int KS>
__device__ __forceinline__ float load_q_f16(const Params& p, const Seg& s, int hc, int r0, int r1, int j,
                                             bool flag_err, uint32_t (&qf)[KS][4], int d0 = 0) {
  const int a = p.qo ? __ldg(p.qo + s.b) : s.b * p.L, e = p.qo ? __ldg(p.qo + s.b + 1) : (s.b + 1) * p.L;
  const bool ok = a >= 0 && e - a == p.L && static_cast<long long>(a) + p.L <= p.n_rows;
  if (!ok && flag_err) atomicOr(p.err, kErrBadQoIndptr);
  const int s_b = ok ? a : s.b * p.L;
  const int kvh = s.hg * p.HC + hc;
  const bool v0 = r0 < p.R, v1 = r1 < p.R;
  const __nv_bfloat16* q0 = p.q + (static_cast<long long>(s_b) + (v0 ? r0 / p.gq : 0)) * p.q_s0 +
                            static_cast<long long>(kvh * p.gq + (v0 ? r0 % p.gq : 0)) * p.q_s1 + d0;
  const __nv_bfloat16* q1 = p.q + (static_cast<long long>(s_b) + (v1 ? r1 / p.gq : 0)) * p.q_s0 +
                            static_cast<long long>(kvh * p.gq + (v1 ? r1 % p.gq : 0)) * p.q_s1 + d0;
  unsigned mx = 0;
#pragma unroll
  for (int kk = 0; kk < KS; ++kk) {
    qf[kk][0] = v0 ? ld_u32(q0 + kk * 16 + 4 * j) : 0u;
    qf[kk][2] = v0 ? ld_u32(q0 + kk * 16 + 4 * j + 2) : 0u;
    qf[kk][1] = v1 ? ld_u32(q1 + kk * 16 + 4 * j) : 0u;
    qf[kk][3] = v1 ? ld_u32(q1 + kk * 16 + 4 * j + 2) : 0u;
#pragma unroll
    for (int i = 0; i < 4; ++i) mx = max(mx, max(qf[kk][i] & 0x7FFFu, (qf[kk][i] >> 16) & 0x7FFFu));
  }
  mx = __reduce_max_sync(0xffffffffu, mx);
  const int ex = static_cast<int>(mx >> 7) - 127;  // exponent of the largest |q|
  const int sh = ex > 14 ? ex - 14 : 0;
  const float down = __int_as_float((127 - sh) << 23);
#pragma unroll
  for (int kk = 0; kk < KS; ++kk) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = unpack_bf16(qf[kk][i]);
      qf[kk][i] = pack_f16(f.x * down, f.y * down);
    }
  }
  return __int_as_float((127 + sh) << 23);
}

// 16-byte chunk swizzle of a K / V row in a stage: rows of 128 bytes or more
// XOR their chunk index with (token & 7); 64-byte rows (4 chunks) with
// ((token >> 1) & 3).  Either way the 8 rows of an ldmatrix phase hit 8
// distinct bank groups.
template <int CPR>
__device__ __forceinline__ int chunk_swz(int t) {
  return CPR >= 8 ? (t & 7) : ((t >> 1) & 3);
}

// ---------------------------------------------------------------------------
// This CTA's share of the work: the segments (b, hg) of virtual length
// max(P_b, 1) are laid end to end and CTA c owns positions [c W, c W + W),
// W = max(ceil(total / gridDim.x), w_min).  A block scan of the prefix lengths
// (kv_indptr or seq_lens) gives the total and the segment holding `start`; no
// host synchronisation.  Every kernel that writes or reads a call's pieces
// cuts the space this way.  All threads of the block call it (it uses
// __syncthreads and shared memory [0, 256)); false: the CTA has no work.
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool cta_share(const Params& p, unsigned char* smem, long long& start, long long& end,
                                          long long& W, Seg& seg0) {
  long long* ctl_base = reinterpret_cast<long long*>(smem);
  int* ctl_b = reinterpret_cast<int*>(smem + 8);
  long long* scan_ws = reinterpret_cast<long long*>(smem + 128);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) *ctl_b = -1;
  const int nthreads = blockDim.x;
  const int per = (p.B + nthreads - 1) / nthreads;
  const int b_lo = min(p.B, tid * per);
  const int b_hi = min(p.B, b_lo + per);
  long long mysum = 0;
  bool bad_kvp = false;
  for (int b = b_lo; b < b_hi; ++b) {
    int P;
    long long kv0;
    bad_kvp |= !seq_info(p, b, P, kv0);
    mysum += max(P, 1);
  }
  if (bad_kvp && blockIdx.x == 0) atomicOr(p.err, kErrBadKvIndptr);
  long long incl = mysum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  const int nwarps = nthreads >> 5;
  if (lane == 31) scan_ws[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    long long w = lane < nwarps ? scan_ws[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    if (lane < nwarps) scan_ws[lane] = w;
  }
  __syncthreads();
  const long long excl = (warp > 0 ? scan_ws[warp - 1] : 0) + incl - mysum;
  const long long tot = scan_ws[nwarps - 1] * p.n_hg;
  W = (tot + gridDim.x - 1) / gridDim.x;
  if (W < p.w_min) W = p.w_min;
  start = static_cast<long long>(blockIdx.x) * W;
  if (start >= tot) return false;  // uniform
  end = min(tot, start + W);
  {
    long long off = excl;
    for (int b = b_lo; b < b_hi; ++b) {
      int P;
      long long kv0;
      load_seq(p, b, P, kv0);
      const long long len = max(P, 1);
      const long long base = off * p.n_hg;
      if (start >= base && start < base + len * p.n_hg) {
        *ctl_b = b;
        *ctl_base = base;
      }
      off += len;
    }
  }
  __syncthreads();
  seg0.b = *ctl_b;
  if (seg0.b < 0) return false;  // unreachable for consistent inputs; guards the walk
  load_seq(p, seg0.b, seg0.P, seg0.kv0);
  seg0.len = max(seg0.P, 1);
  seg0.hg = static_cast<int>((start - *ctl_base) / seg0.len);
  seg0.off = *ctl_base + static_cast<long long>(seg0.hg) * seg0.len;
  return true;
}

#include "verify_combine.cuh"

// ---------------------------------------------------------------------------
// Cluster form: one thread-block cluster per segment (b, hg), of p.cl CTAs.
// CTA r of the cluster streams tokens [r w, r w + w) of the segment, w = the
// segment's (virtual) length over p.cl in whole stages, and writes its
// partial to slot k (p.cl + 1) + r (k = the cluster, the segment's index);
// after the cluster barrier the cluster's CTAs fold the segment's pieces,
// add the draft block and write o (the combine, in the same launch).  Every
// thread calls it; false: this CTA streams nothing (it still joins the
// barrier and the combine).
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool cluster_share(const Params& p, long long& start, long long& end, Seg& seg0,
                                              long long& slot0, long long& npc) {
  // (also called after streaming, for slot0 / npc alone: recomputing them is
  // cheaper than keeping them in registers across the stream)
  const int C = p.cl;
  const long long k = blockIdx.x / C;
  const int r = static_cast<int>(blockIdx.x % C);
  seg0.b = static_cast<int>(k / p.n_hg);
  seg0.hg = static_cast<int>(k % p.n_hg);
  const bool ok = seq_info(p, seg0.b, seg0.P, seg0.kv0);
  if (!ok && r == 0 && seg0.hg == 0 && threadIdx.x == 0) atomicOr(p.err, kErrBadKvIndptr);
  seg0.len = max(seg0.P, 1);
  seg0.off = 0;
  long long w = (seg0.len + C - 1) / C;
  w = (w + kStageTokens - 1) / kStageTokens * kStageTokens;
  npc = (seg0.len + w - 1) / w;
  slot0 = k * (C + 1);
  start = r * w;
  end = min(static_cast<long long>(seg0.len), start + w);
  return start < seg0.len;
}

// The cluster form's combine unit as a call of its own: its registers are
// allocated apart from the stream's, which are dead by then.
template <int D, bool FP8>
__device__ __noinline__ void combine_unit_cl(const Params& p, unsigned char* smem, int tid, int bar, long long s_idx,
                                             int hc, int tile, int ch, long long slot0, long long npc) {
  combine_unit<D, FP8, true>(p, smem, tid, bar, s_idx, hc, tile, ch, slot0, npc);
}

// Every thread of every CTA of the cluster: what each wrote to global memory
// before is visible to all of them after (release / acquire at cluster scope).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// The kernel.
// Shared memory map (bytes):
//   [0,   128)  control: sched base (i64) @0, sched b @8, ticket flags [2] @16
//   [128, 256)  block-scan scratch (up to 16 x i64)
//   [ring_off + hc * head_bytes, ...)  the ring of KV head hc, shared by the
//        warps that serve it (each copies its share of every stage's tokens):
//        nst stages of K rows [16][D*e] then V rows [16][D*e], XOR-swizzled in
//        16-byte chunks (chunk_swz) so 8-row ldmatrix phases hit 8 distinct
//        bank groups.  After streaming, the first nwc * 32 * D bytes hold each
//        warp's staged new drafts (fused store).
//   [misc_off + w * misc_bytes, ...)  warp w's own kIdxRing x 16 x 8 B of
//        kv_indices, 16 x 4 B valid-token masks and, for two-tile warps and
//        e4m3 pools at head_dim 256, its query tiles (16 x D x 2 B each; its
//        half, 16 x D/2 x 2 B, in the column-split stream, which then adds two
//        1 KB score-exchange slots).
// ---------------------------------------------------------------------------
template <int D>
struct MaxWarps {
  static constexpr int value = (D > 128) ? 4 : 8;
};
template <int A, int B>
struct MaxOf {
  static constexpr int value = A > B ? A : B;
};

// SO (stream only): the kernel ends once its pieces' partials are written; the
// combine kernel folds them in its own launch.  CS = 2 (head_dim 256, one KV
// head per CTA, at most two 16-row tiles; stream only): each 16-row tile is
// shared by a pair of warps that split the QK contraction (exchanging their
// scaled partial scores through shared memory) and own half of the output
// columns each.  Half the accumulator registers per warp, so three CTAs per SM.
// DV: the value head_dim (output columns), D the query / key head_dim.
// CL: the cluster form (stream only, then the combine of the segment by the
// cluster's CTAs after a cluster barrier; one launch, no tickets).
// PIPE: software-pipelined stages (the softmax and PV of stage k run after
// the QK products of stage k + 1 are issued; needs a ring of >= 3 stages).
// The column split with MTW = 2: one warp pair per KV head holding both
// 16-row tiles, each warp half the columns (every K / V element converted
// and loaded once per head); 64-thread CTAs, four per SM.
template <int D, bool FP8, int MTW, int CS = 1, bool SO = (CS == 2), int DV = D, bool CL = false, bool PIPE = false>
__global__ void __launch_bounds__(CS == 2 ? (MTW == 2 ? 64 : 128) : MaxWarps<MaxOf<D, DV>::value>::value * 32,
                                  CS == 2 ? (MTW == 2 ? 4 : 3) : 1)
    vsk_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) unsigned char smem[];
  constexpr int EK = FP8 ? 1 : 2;  // pool element bytes
  constexpr int NT = DV / 8;       // n-tiles of the output row
  constexpr int KS = D / 16;       // k-steps of the QK contraction
  static_assert(CS == 1 || (CS == 2 && D == 256 && DV == 256 && SO),
                "column split: head_dim 256 stream only");
  static_assert(D == DV || (MTW == 1 && CS == 1 && !SO), "head_dim != v_head_dim: one-launch kernel, one tile per warp");
  static_assert(!CL || (SO && MTW == 1 && D == DV), "cluster form: stream-only, one tile per warp");
  static_assert(!PIPE || CS == 1, "pipelined stages: not with the column split");
  constexpr int DH = D / CS;       // contraction length of one warp
  constexpr int DVH = DV / CS;     // output columns of one warp
  constexpr int NTH = NT / CS;     // its n-tiles
  constexpr int KSH = KS / CS;     // its k-steps
  constexpr int KSV = DV / 16 / CS;  // its 16-wide output blocks (e4m3 PV)
  constexpr int ROWB = D * EK;     // bytes of one head's K row
  constexpr int VROWB = DV * EK;   // bytes of one head's V row
  constexpr int CPR = ROWB / 16;   // 16-byte chunks per K row
  constexpr int VCPR = VROWB / 16;  // ... per V row
  constexpr int STAGE_B = kStageTokens * (ROWB + VROWB);

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + 16);  // [2]
  const int nst = p.nst;

  // The stream-only launches are followed by the combine kernel, launched as
  // a programmatic dependent: let it start (its prologue reads only the
  // call's inputs; it waits for this grid before reading any partial).
  if constexpr (SO && !CL) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // ---- prologue: this CTA's share of the flattened space and its first segment ----
  long long start = 0, end = 0, W = 0;
  Seg seg0;
  if constexpr (CL) {
    long long slot0_, npc_;
    // no range (start = end = 0: the stream loop below does nothing) for a
    // CTA past the segment's end
    if (!cluster_share(p, start, end, seg0, slot0_, npc_)) {
      start = 0;
      end = 0;
    }
  } else {
    if (!cta_share(p, smem, start, end, W, seg0)) return;  // uniform: the whole CTA has no work
  }

  // ============================ per-warp pipeline ============================
  // Warp w serves KV head hc = w / WPH of the group and MTW 16-row tiles
  // (from tile mt * MTW) of its packed query rows.  The WPH warps of a head
  // stream its K and V rows themselves with 16-byte cp.async into the head's
  // nst-deep ring, each copying 16/WPH tokens of every stage; with WPH > 1
  // they meet at a named barrier once per stage.  No producer warp.  Indices
  // come kIdxAhead stages ahead, also by cp.async, into each warp's own index
  // ring.
  const int WPH = p.MT / MTW;  // warp groups per KV head; each owns MTW 16-row tiles
  const int WPHC = WPH * CS;   // warps per KV head
  // Cluster form at head_dim <= 128: warps beyond the streaming ones are
  // there only for the combine (it takes four); they take head HC - 1's
  // indices and issue no copy.  (The head_dim 256 cluster form streams with
  // all four warps.)  The range itself stays uniform across the CTA.
  const int hc = (CL && CS == 1) ? min(warp / WPHC, p.HC - 1) : warp / WPHC;
  const bool streamer = !(CL && CS == 1) || warp < p.nwc;
  const int mt = (warp / CS) % WPH;
  const int csi = CS == 2 ? (warp & 1) : 0;  // column half of this warp
  const int cw = warp % WPHC;                // this warp's share of the head's copies
  const int g = lane >> 2;
  const int j = lane & 3;
  const int RM = 16 * p.MT;
  int r0s[MTW], r1s[MTW];  // the packed rows of this lane in each of the warp's tiles
#pragma unroll
  for (int t = 0; t < MTW; ++t) {
    r0s[t] = 16 * (mt * MTW + t) + g;
    r1s[t] = r0s[t] + 8;
  }
  const float NEG_INF = -INFINITY;
  unsigned char* ring = smem + p.ring_off + hc * p.head_bytes;
  unsigned char* idx_ring = smem + p.misc_off + warp * p.misc_bytes;
  unsigned* mask_ring = reinterpret_cast<unsigned*>(idx_ring + kIdxRing * 128);
  const uint32_t ring_s = smem_u32(ring);
  const uint32_t idx_s = smem_u32(idx_ring);
  const uint64_t pol = policy_evict_first();
  const long long Wl = W;
  const int c_self = blockIdx.x;
  const bool flagger = (warp == 0 && lane == 0);

  {
  int dslot = 0;  // ring slot of the next data job (job % nst, kept without a division)
  auto issue_idx = [&](const StageIt& it, long long job) {
    if (streamer && it.valid && lane < min(kStageTokens, it.te - it.tok)) {
      const long long n = it.s.kv0 + it.tok + lane;
      const uint32_t dst = idx_s + static_cast<uint32_t>(job % kIdxRing) * 128u + lane * 8u;
      if (p.paged)  // page id of cache position tok + lane
        cp_async_4(dst, p.bt + static_cast<long long>(it.s.b) * p.bt_s0 + page_of(p, it.tok + lane));
      else if (p.idx64)
        cp_async_8(dst, static_cast<const long long*>(p.kvi) + n);
      else
        cp_async_4(dst, static_cast<const int*>(p.kvi) + n);
    }
  };
  auto issue_data = [&](const StageIt& it, long long job) {
    if (!streamer || !it.valid) return;
    const int n = min(kStageTokens, it.te - it.tok);
    const unsigned char* ie = idx_ring + static_cast<int>(job % kIdxRing) * 128;
    long long myloc = -1;
    if (lane < n) {
      if (p.paged) {
        const long long pid = *reinterpret_cast<const int*>(ie + lane * 8);
        const int t = it.tok + lane;
        myloc = pid >= 0 ? pid * p.page + (t - page_of(p, t) * p.page) : -1;
      } else {
        myloc = p.idx64 ? *reinterpret_cast<const long long*>(ie + lane * 8)
                        : static_cast<long long>(*reinterpret_cast<const int*>(ie + lane * 8));
      }
    }
    const bool ok = lane < n && myloc >= 0 && myloc < p.pool;
    const unsigned mask = __ballot_sync(0xffffffffu, ok) & 0xFFFFu;
    if (lane < n && !ok && hc == 0 && cw == 0) atomicOr(p.err, kErrBadIndex);
    if (lane == 0) mask_ring[job % 16] = mask;
    const long long head = static_cast<long long>(it.s.hg) * p.HC + hc;
    const unsigned char* kbase = p.kb + head * p.kb_s1;
    const unsigned char* vbase = p.vb + head * p.vb_s1;
    const uint32_t slot = ring_s + static_cast<uint32_t>(dslot) * STAGE_B;
    // Two, four or eight warps per KV head (the head's stage split in 8, 4 or
    // 2 tokens per warp): LPN = 32 / TPW lanes serve each token (4, 8 or
    // 16), lane s of a token copying chunks s, s + LPN, ... of its K row and
    // of its V row, so each copy instruction reads runs of 64 bytes or more
    // (smaller runs measured far slower).  A lane forms its token's row
    // addresses once; every further source offset is a compile-time
    // constant.  The swizzle permutes chunks in groups of G = min(8, chunks
    // per row): with LPN < G the lane's destinations repeat every G / LPN
    // chunks (that many precomputed bases plus constants), with LPN >= G one
    // base plus constants covers them.
    auto fast_copy = [&](auto tpw_tag, auto lpn_tag) {
      constexpr int TPW = decltype(tpw_tag)::value;  // tokens this warp copies
      constexpr int LPN = decltype(lpn_tag)::value;  // lanes per token
      constexpr int NPASS = TPW * LPN / 32;          // tokens a lane serves
      const int sl = lane % LPN;
      // all of this warp's tokens present (the common case): no selects
      const unsigned wmask = ((1u << TPW) - 1u) << (cw * TPW);
      const bool full = (mask & wmask) == wmask;
#pragma unroll
      for (int pass = 0; pass < NPASS; ++pass) {
      const int t = cw * TPW + pass * (32 / LPN) + lane / LPN;
      const long long loc = __shfl_sync(0xffffffffu, myloc, t);
      const bool v = (mask >> t) & 1u;
      auto rows = [&](auto rb_tag, const unsigned char* base, long long s0, uint32_t region) {
        constexpr int RB = decltype(rb_tag)::value;  // row bytes
        constexpr int CP = RB / 16;                 // chunks per row
        constexpr int G = CP < 8 ? CP : 8;          // chunks a swizzle permutes together
        constexpr int Q = LPN < G ? G / LPN : 1;    // distinct destination bases
        static_assert(CP % LPN == 0, "lanes per token divide the row");
        const int x = chunk_swz<CP>(t);
        uint32_t db[Q];
#pragma unroll
        for (int q = 0; q < Q; ++q) db[q] = region + static_cast<uint32_t>(t * RB + (((q * LPN + sl) ^ x) << 4));
        const unsigned char* src = v ? base + loc * s0 + sl * 16 : reinterpret_cast<const unsigned char*>(p.q);
        // destination of the lane's r-th chunk (chunk r LPN + sl)
        auto dst = [&](int r) -> uint32_t {
          return LPN < G ? db[r % Q] + ((r * LPN) / G) * G * 16 : db[0] + r * LPN * 16;
        };
        if (full) {
#pragma unroll
          for (int r = 0; r < CP / LPN; ++r) cp_async_16_zfill(dst(r), src + r * LPN * 16, true, pol);
        } else {
#pragma unroll
          for (int r = 0; r < CP / LPN; ++r) cp_async_16_zfill(dst(r), v ? src + r * LPN * 16 : src, v, pol);
        }
      };
      rows(std::integral_constant<int, ROWB>{}, kbase, p.kb_s0, slot);
      rows(std::integral_constant<int, VROWB>{}, vbase, p.vb_s0, slot + 16 * ROWB);
      }
    };
    // (one warp per head keeps the whole-row copies below: with 16 tokens a
    // warp they measured faster than this mapping)
    if (WPHC == 2) {
      // head_dim 256 bf16 rows: eight lanes per token (128-byte runs, two
      // passes) measured 5 % faster; e4m3 rows and the other sizes keep four
      constexpr int LPN2 = (!FP8 && D == 256 && DV == 256) ? 8 : 4;
      fast_copy(std::integral_constant<int, 8>{}, std::integral_constant<int, LPN2>{});
      return;
    }
    if constexpr (CPR % 8 == 0 && VCPR % 8 == 0) {
      if (WPHC == 4) {
        fast_copy(std::integral_constant<int, 4>{}, std::integral_constant<int, 8>{});
        return;
      }
    }
    if constexpr (CPR % 16 == 0 && VCPR % 16 == 0) {
      if (WPHC == 8) {
        fast_copy(std::integral_constant<int, 2>{}, std::integral_constant<int, 16>{});
        return;
      }
    }
    // lane -> (token group, 16-byte chunk): LPT lanes cover one row, so each
    // lane computes a token's K and V addresses once and issues both copies
    if constexpr (D == DV) {
      constexpr int LPT = CPR < 32 ? CPR : 32;  // lanes per row
      constexpr int TSTEP = 32 / LPT;          // tokens covered per pass of the warp
      constexpr int CPL = CPR / LPT;           // chunks of a row per lane
      const int cl = lane % LPT;
      auto copy_token = [&](int t, long long loc) {
        const bool v = (mask >> t) & 1u;
        // an absent token is zero-filled (nothing read); q is a valid, never-empty address
        const unsigned char* ks = v ? kbase + loc * p.kb_s0 : reinterpret_cast<const unsigned char*>(p.q);
        const unsigned char* vs = v ? vbase + loc * p.vb_s0 : reinterpret_cast<const unsigned char*>(p.q);
#pragma unroll
        for (int cj = 0; cj < CPL; ++cj) {
          const int cir = cl + LPT * cj;
          const int pc = cir ^ chunk_swz<CPR>(t);
          const uint32_t d = slot + static_cast<uint32_t>(t * ROWB + pc * 16);
          cp_async_16_zfill(d, v ? ks + cir * 16 : ks, v, pol);
          cp_async_16_zfill(d + 16 * ROWB, v ? vs + cir * 16 : vs, v, pol);
        }
      };
      if (WPHC == 1) {
        // the warp copies the whole stage (token indices known at compile time)
#pragma unroll
        for (int t = lane / LPT; t < kStageTokens; t += TSTEP) copy_token(t, __shfl_sync(0xffffffffu, myloc, t));
      } else {
        // the warps of the head split the stage: tokens [cw * tpw, cw * tpw + tpw)
        const int tpw = kStageTokens / WPHC;
#pragma unroll
        for (int i = 0; i < kStageTokens / TSTEP; ++i) {
          if (i * TSTEP >= tpw) break;  // uniform across the warp
          const int tw = lane / LPT + i * TSTEP;
          const bool act = tw < tpw;    // false only when fewer tokens than one pass of the warp
          const int t = cw * tpw + (act ? tw : 0);
          const long long loc = __shfl_sync(0xffffffffu, myloc, t);
          if (act) copy_token(t, loc);
        }
      }
    } else {
      // K rows and V rows of different sizes: one pass over the stage's K
      // rows, then one over its V rows (region after the 16 K rows)
      auto copy_rows = [&](auto rb_tag, const unsigned char* base, long long s0, uint32_t region) {
        constexpr int RB = decltype(rb_tag)::value;  // row bytes
        constexpr int CP = RB / 16;
        constexpr int LP = CP < 32 ? CP : 32;
        constexpr int TS = 32 / LP;
        constexpr int NCL = CP / LP;
        const int cl = lane % LP;
        auto one = [&](int t, long long loc) {
          const bool v = (mask >> t) & 1u;
          const unsigned char* src = v ? base + loc * s0 : reinterpret_cast<const unsigned char*>(p.q);
#pragma unroll
          for (int cj = 0; cj < NCL; ++cj) {
            const int cir = cl + LP * cj;
            const uint32_t d = region + static_cast<uint32_t>(t * RB + (cir ^ chunk_swz<CP>(t)) * 16);
            cp_async_16_zfill(d, v ? src + cir * 16 : src, v, pol);
          }
        };
        if (WPHC == 1) {
#pragma unroll
          for (int t = lane / LP; t < kStageTokens; t += TS) one(t, __shfl_sync(0xffffffffu, myloc, t));
        } else {
          const int tpw = kStageTokens / WPHC;
#pragma unroll
          for (int i = 0; i < kStageTokens / TS; ++i) {
            if (i * TS >= tpw) break;
            const int tw = lane / LP + i * TS;
            const bool act = tw < tpw;
            const int t = cw * tpw + (act ? tw : 0);
            const long long loc = __shfl_sync(0xffffffffu, myloc, t);
            if (act) one(t, loc);
          }
        }
      };
      copy_rows(std::integral_constant<int, ROWB>{}, kbase, p.kb_s0, slot);
      copy_rows(std::integral_constant<int, VROWB>{}, vbase, p.vb_s0, slot + 16 * ROWB);
    }
  };

  StageIt ii, di;
  ii.s = seg0;
  ii.tok = static_cast<int>(start - seg0.off);
  ii.te = piece_real_end(seg0, end);
  sit_settle(p, ii, end);
  di = ii;
  long long job_i = 0, job_d = 0;
  auto step_idx = [&]() {
    issue_idx(ii, job_i);
    ++job_i;
    if (ii.valid) {
      ii.tok += kStageTokens;
      sit_settle(p, ii, end);
    }
  };
  auto step_data = [&]() {
    issue_data(di, job_d);
    ++job_d;
    if (++dslot == nst) dslot = 0;
    if (di.valid) {
      di.tok += kStageTokens;
      sit_settle(p, di, end);
    }
  };
#pragma unroll 1
  for (int a = 0; a < kIdxAhead; ++a) step_idx();
  cp_async_commit();
  cp_async_wait<0>();
  __syncwarp();
  // stages in flight ahead of the one being consumed: nst - 1, or nst - 2
  // when pipelined (the ring then also holds the stage whose PV is pending)
#pragma unroll 1
  for (int a = 0; a < nst - 1 - (PIPE ? 1 : 0); ++a) {
    step_data();
    step_idx();
    cp_async_commit();
  }

  // ldmatrix lane roles (token row within the 16-token stage, 16-byte chunk)
  const int k_key = ((lane >> 4) << 3) + (lane & 7);
  const int k_chk = (lane >> 3) & 1;
  const int v_key = (((lane >> 3) & 1) << 3) + (lane & 7);
  const int v_chk = lane >> 4;
  const int f_key = lane & 15;  // e4m3 pools: key row of this lane's ldmatrix address
  // This lane's swizzled 16-byte chunk offsets of its ldmatrix rows: the
  // chunk index XOR the row's swizzle only touches the low 3 bits (the low 2
  // with 4-chunk rows), so within each group of four consecutive loads the
  // offsets repeat and the group adds 128 bytes: offset of load i =
  // koff[i & 3] + 128 (i >> 2).
  uint32_t koff[4], voff[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    if constexpr (FP8) {
      koff[r] = static_cast<uint32_t>(((2 * r + (lane >> 4)) ^ chunk_swz<CPR>(f_key)) << 4);
      voff[r] = static_cast<uint32_t>(((2 * r + (lane >> 4)) ^ chunk_swz<VCPR>(f_key)) << 4);
    } else {
      koff[r] = static_cast<uint32_t>(((2 * r + k_chk) ^ (k_key & 7)) << 4);
      voff[r] = static_cast<uint32_t>(((2 * r + v_chk) ^ (v_key & 7)) << 4);
    }
  }

  // The next piece's query fragments are loaded into registers while the
  // current piece streams (head_dim <= 128, one tile per warp), so a piece
  // boundary costs no global round trip.
  constexpr bool kQAhead = D <= 128 && DV <= 128 && MTW == 1;
  uint32_t qf[MTW][KSH][4];  // this warp's columns of the query (all of them unless CS = 2)
  uint32_t qn[kQAhead ? KSH : 1][4];
  // bf16 pool: bf16 q fragments; e4m3 pool: f16 q fragments scaled by 2^-sh
  // (qmul = 2^sh is folded back into the score scale)
  auto load_piece_q = [&](const Seg& sq, bool flag, int ra, int rb, uint32_t (&dst)[KSH][4]) -> float {
    if constexpr (FP8) {
      return load_q_f16<KSH>(p, sq, hc, ra, rb, j, flag, dst, csi * DH);
    } else {
      load_q<KSH>(p, sq, hc, ra, rb, j, flag, dst, csi * DH);
      return 1.f;
    }
  };
  // e4m3 pools at head_dim 256, and warps with two tiles: the piece's query
  // fragments wait in the warp's shared memory (per tile 16 rows x D,
  // 16-byte chunks XOR-swizzled by row) and are re-read by ldmatrix each
  // stage, which frees their registers (for the e4m3 conversions, or for the
  // second tile's accumulators).
  constexpr bool kQSmem = (FP8 && D == 256) || MTW == 2;
  unsigned char* qsm = reinterpret_cast<unsigned char*>(mask_ring) + 128;
  auto q_to_smem = [&]() {
    if constexpr (kQSmem) {
      __syncwarp();  // the previous piece's ldmatrix reads are done
#pragma unroll
      for (int t = 0; t < MTW; ++t) {
#pragma unroll
        for (int kk = 0; kk < KSH; ++kk) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int row = g + ((i & 1) << 3);
            const int e = kk * 16 + ((i >> 1) << 3) + 2 * j;
            *reinterpret_cast<uint32_t*>(qsm + t * 32 * DH + row * (2 * DH) + (((e >> 3) ^ (row & 7)) << 4) +
                                         (e & 7) * 2) = qf[t][kk][i];
          }
        }
      }
      __syncwarp();
    }
  };
  const int q_row = (lane & 7) + (((lane >> 3) & 1) << 3);
  const uint32_t q_lane = smem_u32(qsm) + q_row * (2 * DH);
  // swizzled chunk offsets of this lane's query-fragment loads (as koff)
  uint32_t qoff[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) qoff[r] = static_cast<uint32_t>(((2 * r + (lane >> 4)) ^ (q_row & 7)) << 4);
  // CS = 2: this warp's score exchange buffer (after its query tiles) and the
  // offset, in floats, to its partner's
  float* xbuf = reinterpret_cast<float*>(qsm + (kQSmem ? MTW * 32 * DH : 0));
  const int xpair = (csi ? -1 : 1) * (p.misc_bytes / 4);
  Seg s = seg0;
  float qsc[MTW];
#pragma unroll
  for (int t = 0; t < MTW; ++t) qsc[t] = p.scale2 * load_piece_q(s, flagger && t == 0, r0s[t], r1s[t], qf[t]);
  q_to_smem();
  float qsc_n = p.scale2;
  Seg sn = s;
  seg_advance(p, sn);
  if constexpr (kQAhead) {
    if (seg_live(p, sn, end)) qsc_n = p.scale2 * load_piece_q(sn, false, r0s[0], r1s[0], qn);
  }
  long long k = 0;
  int kslot = 0;  // ring slot of stage k (k % nst, kept without a division)

#pragma unroll 1
  while (streamer && seg_live(p, s, end)) {
    const int t0 = static_cast<int>(max(start, s.off) - s.off);
    const int te = piece_real_end(s, end);
    float acc[MTW][NTH][4];  // this warp's output columns
    float m0[MTW], m1[MTW], l0[MTW], l1[MTW];
#pragma unroll
    for (int t = 0; t < MTW; ++t) {
#pragma unroll
      for (int n = 0; n < NTH; ++n) acc[t][n][0] = acc[t][n][1] = acc[t][n][2] = acc[t][n][3] = 0.f;
      m0[t] = NEG_INF;
      m1[t] = NEG_INF;
      l0[t] = 0.f;
      l1[t] = 0.f;
    }

    // ---------------- prefix: online softmax over this CTA's piece ----------------
    // Pipelined: the previous stage's raw scores, valid-key mask and V rows,
    // finished (softmax, PV) after this stage's QK products are issued.
    [[maybe_unused]] float s_prev[MTW][2][4];
    [[maybe_unused]] unsigned mask_prev = 0u;
    [[maybe_unused]] uint32_t vbase_prev = 0u;
    [[maybe_unused]] bool have_prev = false;
    // softmax of one stage's scores (scaled into the log2 domain here) and its
    // PV products; `sfin` holds the raw QK sums of the stage
    auto finish = [&](float (&sfin)[MTW][2][4], const unsigned mask, const uint32_t vbase) {
      uint32_t pa[MTW][4];
#pragma unroll
      for (int t = 0; t < MTW; ++t)
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
          for (int e = 0; e < 4; ++e) sfin[t][u][e] *= qsc[t];  // scale into the log2 domain
      if constexpr (CS == 2) {
        // the pair's partial scores (each in the log2 domain already) summed
        // by both warps alike, every tile through one barrier; the buffer
        // alternates with the stage parity
        float* xo = xbuf + static_cast<int>(k & 1) * (256 * MTW) + lane * 8;
#pragma unroll
        for (int t = 0; t < MTW; ++t) {
          *reinterpret_cast<float4*>(xo + t * 256) =
              make_float4(sfin[t][0][0], sfin[t][0][1], sfin[t][0][2], sfin[t][0][3]);
          *reinterpret_cast<float4*>(xo + t * 256 + 4) =
              make_float4(sfin[t][1][0], sfin[t][1][1], sfin[t][1][2], sfin[t][1][3]);
        }
        named_bar_sync(10 + (warp >> 1), 64);
#pragma unroll
        for (int t = 0; t < MTW; ++t) {
          const float* xp = xo + t * 256 + xpair;
          const float4 y0 = *reinterpret_cast<const float4*>(xp), y1 = *reinterpret_cast<const float4*>(xp + 4);
          sfin[t][0][0] += y0.x;
          sfin[t][0][1] += y0.y;
          sfin[t][0][2] += y0.z;
          sfin[t][0][3] += y0.w;
          sfin[t][1][0] += y1.x;
          sfin[t][1][1] += y1.y;
          sfin[t][1][2] += y1.z;
          sfin[t][1][3] += y1.w;
        }
      }
#pragma unroll
      for (int t = 0; t < MTW; ++t) {
        // mask absent keys (tail / dropped) only when the stage is not full
        // (the mask is uniform across the warp)
        if (mask != 0xFFFFu) {
#pragma unroll
          for (int u = 0; u < 2; ++u) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int key = u * 8 + 2 * j + (e & 1);
              if (!((mask >> key) & 1u)) sfin[t][u][e] = NEG_INF;
            }
          }
        }
        const float mx0 = quad_max(fmaxf(fmaxf(sfin[t][0][0], sfin[t][0][1]), fmaxf(sfin[t][1][0], sfin[t][1][1])));
        const float mx1 = quad_max(fmaxf(fmaxf(sfin[t][0][2], sfin[t][0][3]), fmaxf(sfin[t][1][2], sfin[t][1][3])));
        // The running maximum is raised only when a stage exceeds it by more
        // than kLazy (log2 units): the weights 2^(s - m) then stay below
        // 2^kLazy, and most stages need no rescale of the accumulator.  The
        // result is the same (weights and sum share the reference m).
        const float mn0 = mx0 > m0[t] + kLazy ? mx0 : m0[t], mn1 = mx1 > m1[t] + kLazy ? mx1 : m1[t];
        const float ms0 = (mn0 == NEG_INF) ? 0.f : mn0;
        const float ms1 = (mn1 == NEG_INF) ? 0.f : mn1;
        float pr[2][4];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          pr[u][0] = fast_exp2(sfin[t][u][0] - ms0);
          pr[u][1] = fast_exp2(sfin[t][u][1] - ms0);
          pr[u][2] = fast_exp2(sfin[t][u][2] - ms1);
          pr[u][3] = fast_exp2(sfin[t][u][3] - ms1);
        }
        const float ps0 = pr[0][0] + pr[0][1] + pr[1][0] + pr[1][1];
        const float ps1 = pr[0][2] + pr[0][3] + pr[1][2] + pr[1][3];
        // rescale only when some row's running maximum moved (rare once the
        // maximum has settled); otherwise alpha is exactly 1
        if (__any_sync(0xffffffffu, (mn0 != m0[t]) || (mn1 != m1[t]))) {
          const float al0 = fast_exp2(m0[t] - ms0), al1 = fast_exp2(m1[t] - ms1);
          l0[t] *= al0;
          l1[t] *= al1;
#pragma unroll
          for (int n = 0; n < NTH; ++n) {
            acc[t][n][0] *= al0;
            acc[t][n][1] *= al0;
            acc[t][n][2] *= al1;
            acc[t][n][3] *= al1;
          }
        }
        l0[t] += ps0;
        l1[t] += ps1;
        m0[t] = mn0;
        m1[t] = mn1;
        if constexpr (FP8) {
          pa[t][0] = pack_f16(pr[0][0], pr[0][1]);
          pa[t][1] = pack_f16(pr[0][2], pr[0][3]);
          pa[t][2] = pack_f16(pr[1][0], pr[1][1]);
          pa[t][3] = pack_f16(pr[1][2], pr[1][3]);
        } else {
          pa[t][0] = pack_bf16(pr[0][0], pr[0][1]);
          pa[t][1] = pack_bf16(pr[0][2], pr[0][3]);
          pa[t][2] = pack_bf16(pr[1][0], pr[1][1]);
          pa[t][3] = pack_bf16(pr[1][2], pr[1][3]);
        }
      }
      if constexpr (FP8) {
        // O += P V for 16 keys.  A transposing x4 load of e4m3 rows gives lane
        // (g, j) the d pair (2g, 2g+1) of keys 2j and 2j+1; a byte permute
        // regroups them by d, so each register feeds two n-tiles: E (even d,
        // column g <-> d 2g) and O (odd d, column g <-> d 2g+1) of a 16-wide
        // block.  acc[2*blk] is E, acc[2*blk+1] is O.
        static_assert(KSV / 2 <= 2 || (KSV / 2) % 4 == 0, "offset groups of four");
        const uint32_t vb = vbase + static_cast<uint32_t>(csi * (KSV / 2) / 4) * 128u;
#pragma unroll
        for (int c2 = 0; c2 < KSV / 2; ++c2) {
          uint32_t r[4];
          ldsm_x4_t(vb + voff[c2 & 3] + (c2 >> 2) * 128, r[0], r[1], r[2], r[3]);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t x0 = __byte_perm(r[2 * h], 0u, 0x3120);      // keys 2j, 2j+1
            const uint32_t x1 = __byte_perm(r[2 * h + 1], 0u, 0x3120);  // keys 2j+8, 2j+9
            const int blk = 2 * c2 + h;
            const uint32_t e0 = e4m3x2_to_f16x2(x0 & 0xFFFF), e1 = e4m3x2_to_f16x2(x1 & 0xFFFF);
            const uint32_t o0 = e4m3x2_to_f16x2(x0 >> 16), o1 = e4m3x2_to_f16x2(x1 >> 16);
#pragma unroll
            for (int t = 0; t < MTW; ++t) {
              mma_f16(acc[t][2 * blk], pa[t], e0, e1);
              mma_f16(acc[t][2 * blk + 1], pa[t], o0, o1);
            }
          }
        }
      } else {
        // O += P V for 16 keys
        static_assert((NTH / 2) % 4 == 0, "offset groups of four");
        const uint32_t vb = vbase + static_cast<uint32_t>(csi * (NTH / 2) / 4) * 128u;
#pragma unroll
        for (int n2 = 0; n2 < NTH / 2; ++n2) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vb + voff[n2 & 3] + (n2 >> 2) * 128, b0, b1, b2, b3);
#pragma unroll
          for (int t = 0; t < MTW; ++t) {
            mma_bf16(acc[t][2 * n2], pa[t], b0, b1);
            mma_bf16(acc[t][2 * n2 + 1], pa[t], b2, b3);
          }
        }
      }
    };
#pragma unroll 1
    for (int tok = t0; tok < te; tok += kStageTokens, ++k, kslot = (kslot + 1 == nst) ? 0 : kslot + 1) {
      cp_async_wait_dyn(nst - 2 - (PIPE ? 1 : 0));  // stage k has landed (this lane's copies)
      __syncwarp();                // ... and every other lane's
      // ... and the other warps' of this head: after this barrier no warp of
      // the head still reads the slot of stage k - 1 (k - 2 when pipelined),
      // which step_data refills
      if (WPHC > 1) named_bar_sync(2 + hc, WPHC * 32);
      step_data();                 // refill the freed slot
      step_idx();
      cp_async_commit();
      const unsigned mask = mask_ring[k % 16];
      unsigned char* slotp = ring + kslot * STAGE_B;
      // ldmatrix row addresses.  bf16: lanes 0-15 / 16-31 take keys 0-7, 8-15
      // of k-chunk 2kk / 2kk+1 ... (k_key, k_chk); e4m3: lane takes key
      // (lane & 15) and chunk 2kk2 + (lane >> 4), so one x4 load gives both
      // 8-key tiles of two 16-wide d blocks.
      const uint32_t kbase = smem_u32(slotp) + (FP8 ? f_key : k_key) * ROWB;
      const uint32_t vbase = smem_u32(slotp) + 16 * ROWB + (FP8 ? f_key : v_key) * VROWB;

      // S = Q K^T for 16 keys: two n-tiles of 8 keys per 16-row tile.
      // Independent accumulator chains per n-tile (k-step mod NCH) cut the
      // dependent mma latency; summed afterwards.  With two tiles per warp the
      // tiles themselves are independent chains.
      // (two chains measured faster than four at head_dim 256, both pools)
      constexpr int NCH = (MTW == 1 && !PIPE) ? ((D == 256 && CS == 1) ? 2 : 4) : 1;
      // (a chain's first product takes a zero accumulator input: nothing to clear)
      float sc[MTW][2][4];
      float sx[MTW][NCH > 1 ? NCH - 1 : 1][2][4];
      auto qk_step = [&](int kk, uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3) {
        const int ch = kk % NCH;
        const bool first = kk < NCH;  // known at compile time in the unrolled loops
#pragma unroll
        for (int t = 0; t < MTW; ++t) {
          float* c0 = ch == 0 ? sc[t][0] : sx[t][ch - 1][0];
          float* c1 = ch == 0 ? sc[t][1] : sx[t][ch - 1][1];
          uint32_t a[4];
          if constexpr (kQSmem) {
            ldsm_x4(q_lane + t * 32 * DH + qoff[kk & 3] + (kk >> 2) * 128, a[0], a[1], a[2], a[3]);
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = qf[t][kk][i];
          }
          if constexpr (FP8) {
            if (first) {
              mma_f16_z(c0, a, b0, b1);
              mma_f16_z(c1, a, b2, b3);
            } else {
              mma_f16(c0, a, b0, b1);
              mma_f16(c1, a, b2, b3);
            }
          } else {
            if (first) {
              mma_bf16_z(c0, a, b0, b1);
              mma_bf16_z(c1, a, b2, b3);
            } else {
              mma_bf16(c0, a, b0, b1);
              mma_bf16(c1, a, b2, b3);
            }
          }
        }
      };
      if constexpr (FP8) {
        // each 32-bit register holds 4 consecutive e4m3 d values of one key:
        // low pair -> b0, high pair -> b1 of the permuted contraction order
        static_assert(KSH / 2 <= 2 || (KSH / 2) % 4 == 0, "offset groups of four");
        const uint32_t kb = kbase + static_cast<uint32_t>(csi * (KSH / 2) / 4) * 128u;
#pragma unroll
        for (int kk2 = 0; kk2 < KSH / 2; ++kk2) {
          uint32_t r0k, r1k, r2k, r3k;
          ldsm_x4(kb + koff[kk2 & 3] + (kk2 >> 2) * 128, r0k, r1k, r2k, r3k);
          qk_step(2 * kk2, e4m3x2_to_f16x2(r0k & 0xFFFF), e4m3x2_to_f16x2(r0k >> 16), e4m3x2_to_f16x2(r1k & 0xFFFF),
                  e4m3x2_to_f16x2(r1k >> 16));
          qk_step(2 * kk2 + 1, e4m3x2_to_f16x2(r2k & 0xFFFF), e4m3x2_to_f16x2(r2k >> 16),
                  e4m3x2_to_f16x2(r3k & 0xFFFF), e4m3x2_to_f16x2(r3k >> 16));
        }
      } else {
        static_assert(KSH % 4 == 0, "offset groups of four");
        const uint32_t kb = kbase + static_cast<uint32_t>(csi * KSH / 4) * 128u;
#pragma unroll
        for (int kk = 0; kk < KSH; ++kk) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kb + koff[kk & 3] + (kk >> 2) * 128, b0, b1, b2, b3);
          qk_step(kk, b0, b1, b2, b3);
        }
      }
      // the stage's raw scores: its accumulation chains summed
      float sr[MTW][2][4];
#pragma unroll
      for (int t = 0; t < MTW; ++t) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float x = sc[t][u][e];
            if constexpr (NCH == 4) {
              x += (sx[t][0][u][e] + sx[t][1][u][e]) + sx[t][2][u][e];
            } else {
#pragma unroll
              for (int c = 0; c < NCH - 1; ++c) x += sx[t][c][u][e];
            }
            sr[t][u][e] = x;
          }
        }
      }
      if constexpr (PIPE) {
        // this stage's QK products are in flight: finish the previous stage
        if (have_prev) finish(s_prev, mask_prev, vbase_prev);
#pragma unroll
        for (int t = 0; t < MTW; ++t)
#pragma unroll
          for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int e = 0; e < 4; ++e) s_prev[t][u][e] = sr[t][u][e];
        mask_prev = mask;
        vbase_prev = vbase;
        have_prev = true;
      } else {
        finish(sr, mask, vbase);
      }
    }
    if constexpr (PIPE) {
      if (have_prev) finish(s_prev, mask_prev, vbase_prev);
    }

    // ---------------- piece end: write the partial and keep streaming ----------------
    // (tickets, merges, drafts and output wait until the whole range is streamed)
    {
      const long long slot_self = c_self + static_cast<long long>(s.b) * p.n_hg + s.hg;
      float* lse_p = p.plse + (slot_self * p.HC + hc) * RM;
      float* o_p = p.po + ((slot_self * p.HC + hc) * RM) * DV;
      const uint64_t keep = policy_evict_last();
#pragma unroll
      for (int t = 0; t < MTW; ++t) {
        const int r0 = r0s[t], r1 = r1s[t];
        const float s0 = quad_sum(l0[t]), s1 = quad_sum(l1[t]);
        const float inv0 = s0 > 0.f ? p.v_scale / s0 : 0.f;
        const float inv1 = s1 > 0.f ? p.v_scale / s1 : 0.f;
        if (j == 0 && csi == 0) {
          st_keep(lse_p + r0, s0 > 0.f ? m0[t] + log2f(s0) : NEG_INF, keep);
          st_keep(lse_p + r1, s1 > 0.f ? m1[t] + log2f(s1) : NEG_INF, keep);
        }
        float* o0p = o_p + r0 * DV + csi * DVH;  // this warp's columns
        float* o1p = o_p + r1 * DV + csi * DVH;
        if constexpr (FP8) {
          // n-tiles E / O of block blk hold d = 16 blk + 4j + {0, 2} / {1, 3}
#pragma unroll
          for (int blk = 0; blk < KSV; ++blk) {
            const float* e = acc[t][2 * blk];
            const float* o = acc[t][2 * blk + 1];
            st_keep4(o0p + blk * 16 + 4 * j, e[0] * inv0, o[0] * inv0, e[1] * inv0, o[1] * inv0, keep);
            st_keep4(o1p + blk * 16 + 4 * j, e[2] * inv1, o[2] * inv1, e[3] * inv1, o[3] * inv1, keep);
          }
        } else {
#pragma unroll
          for (int n = 0; n < NTH; ++n) {
            st_keep2(o0p + n * 8 + 2 * j, acc[t][n][0] * inv0, acc[t][n][1] * inv0, keep);
            st_keep2(o1p + n * 8 + 2 * j, acc[t][n][2] * inv1, acc[t][n][3] * inv1, keep);
          }
        }
      }
    }
    s = sn;
    if (seg_live(p, s, end)) {
      seg_advance(p, sn);
      if constexpr (kQAhead) {
#pragma unroll
        for (int kk = 0; kk < KSH; ++kk) {
          qf[0][kk][0] = qn[kk][0];
          qf[0][kk][1] = qn[kk][1];
          qf[0][kk][2] = qn[kk][2];
          qf[0][kk][3] = qn[kk][3];
        }
        qsc[0] = qsc_n;
        if (seg_live(p, sn, end)) qsc_n = p.scale2 * load_piece_q(sn, false, r0s[0], r1s[0], qn);
      } else {
#pragma unroll
        for (int t = 0; t < MTW; ++t) qsc[t] = p.scale2 * load_piece_q(s, false, r0s[t], r1s[t], qf[t]);
        q_to_smem();
      }
    }
  }
  }  // streaming
  if constexpr (SO) {
    cp_async_wait<0>();  // stream only: the partials are folded by the combine kernel
    if constexpr (CL) {
      // the cluster's pieces are all written: fold them here, 128 threads per
      // (KV head, 16-row tile, 32-column slice) unit, the ring region reused
      // as each group's shared memory
      cluster_sync_all();
      long long cl_slot0, cl_npc, s_, e_;
      Seg g_;
      cluster_share(p, s_, e_, g_, cl_slot0, cl_npc);
      constexpr int kSl = cmb::Geo<D>::kSlices;
      const int C = p.cl;
      const int rank = static_cast<int>(blockIdx.x % C);
      const long long k_seg = blockIdx.x / C;
      const int units = p.HC * p.MT * kSl;
      const int groups = static_cast<int>(blockDim.x) / cmb::kThreads;
      const int gid = warp / (cmb::kThreads / 32);
      unsigned char* gsm = smem + gid * p.cl_smem;
#pragma unroll 1
      for (int u = rank + C * gid; u < units; u += C * groups) {
        const int ch = u % kSl, tile = (u / kSl) % p.MT, hcu = u / (kSl * p.MT);
        combine_unit_cl<D, FP8>(p, gsm, tid % cmb::kThreads, 12 + gid, k_seg, hcu, tile, ch, cl_slot0, cl_npc);
        named_bar_sync(12 + gid, cmb::kThreads);  // the group's shared memory is reused by its next unit
      }
    }
  } else {

  // ================= epilogue: tickets, log-sum-exp merges, drafts, output =================
  // No copy is left in flight, and every partial this thread wrote is made
  // visible device-wide before any ticket of this CTA is taken.
  cp_async_wait<0>();
  __threadfence();
  named_bar_sync(1, p.nwc * 32);
  Seg sg = seg0;
  int nbar = 0;  // ticket rounds so far: selects the flag slot (two slots, one barrier per round)
  // One ticket round: tid 0 draws from ctr; the CTA learns whether it came
  // last (then the ticket is reset to zero for the next call).
  auto take_ticket = [&](int* ctr, int expected) -> bool {
    if (tid == 0) {
      const int old = atomicAdd(ctr, 1);
      const int last = (old == expected - 1) ? 1 : 0;
      if (last) {
        *ctr = 0;
        __threadfence();
      }
      last_flag[nbar & 1] = last;
    }
    named_bar_sync(1, p.nwc * 32);
    const bool r = last_flag[nbar & 1] != 0;
    ++nbar;
    return r;
  };
  float acc[NT][4];
  float m0, m1, l0, l1;
  // Fold `count` partials (slots slot0, slot0 + stride, ...) of this warp's
  // rows in slot order: pass 1 finds each row's largest log-sum-exp, pass 2
  // sums 2^(lse - max) o; two partials per trip of pass 2 at head_dim <= 128
  // keep two partials' loads in flight.
  auto fold = [&](long long slot0, long long stride, long long count, int r0, int r1) {
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
    m0 = NEG_INF;
    m1 = NEG_INF;
    l0 = 0.f;
    l1 = 0.f;
#pragma unroll 4
    for (long long i = 0; i < count; ++i) {
      const float* lq = p.plse + ((slot0 + i * stride) * p.HC + hc) * RM;
      m0 = fmaxf(m0, __ldcg(lq + r0));
      m1 = fmaxf(m1, __ldcg(lq + r1));
    }
    const float ms0 = (m0 == NEG_INF) ? 0.f : m0;
    const float ms1 = (m1 == NEG_INF) ? 0.f : m1;
#pragma unroll(DV <= 128 ? 2 : 1)
    for (long long i = 0; i < count; ++i) {
      const long long sl = slot0 + i * stride;
      const float* lq = p.plse + (sl * p.HC + hc) * RM;
      const float* oq = p.po + ((sl * p.HC + hc) * RM) * DV;
      const float w0 = exp2f(__ldcg(lq + r0) - ms0), w1 = exp2f(__ldcg(lq + r1) - ms1);
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const float2 x0 = __ldcg(reinterpret_cast<const float2*>(oq + r0 * DV + n * 8 + 2 * j));
        const float2 x1 = __ldcg(reinterpret_cast<const float2*>(oq + r1 * DV + n * 8 + 2 * j));
        if (w0 > 0.f) {
          acc[n][0] = fmaf(x0.x, w0, acc[n][0]);
          acc[n][1] = fmaf(x0.y, w0, acc[n][1]);
        }
        if (w1 > 0.f) {
          acc[n][2] = fmaf(x1.x, w1, acc[n][2]);
          acc[n][3] = fmaf(x1.y, w1, acc[n][3]);
        }
      }
      l0 += w0;
      l1 += w1;
    }
  };
#pragma unroll 1
  while (seg_live(p, sg, end)) {
    const long long s_idx = static_cast<long long>(sg.b) * p.n_hg + sg.hg;
    const long long c_first = sg.off / Wl;
    const long long c_last = (sg.off + sg.len - 1) / Wl;
    const long long npc = c_last - c_first + 1;  // pieces of the segment
    // Segments of more than kTreeMin pieces merge in two levels: groups of
    // kGroup consecutive pieces are folded by their group's last arriver into
    // the slot of the group's first piece, then the last group folds the
    // group partials.  Every level folds in slot order, so the result does not
    // depend on which CTA arrived last.
    const bool tree = npc > kTreeMin;
    const long long ng = tree ? (npc + kGroup - 1) / kGroup : npc;
    bool finisher = true;
    if (tree) {
      const long long gfirst = c_first + ((c_self - c_first) / kGroup) * kGroup;
      const long long gcount = min(static_cast<long long>(kGroup), c_last - gfirst + 1);
      finisher = gcount == 1 || take_ticket(p.cnt + p.nseg + gfirst + s_idx, static_cast<int>(gcount));
      if (finisher) {
        // the group partial replaces the partial of the group's first piece
        const long long sl = gfirst + s_idx;
        float* lse_p = p.plse + (sl * p.HC + hc) * RM;
        float* o_p = p.po + ((sl * p.HC + hc) * RM) * DV;
#pragma unroll 1
        for (int t = 0; t < MTW; ++t) {
          const int r0 = r0s[t], r1 = r1s[t];
          fold(gfirst + s_idx, 1, gcount, r0, r1);
          const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
          if (j == 0) {
            lse_p[r0] = l0 > 0.f ? m0 + log2f(l0) : NEG_INF;
            lse_p[r1] = l1 > 0.f ? m1 + log2f(l1) : NEG_INF;
          }
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            *reinterpret_cast<float2*>(o_p + r0 * DV + n * 8 + 2 * j) = make_float2(acc[n][0] * inv0, acc[n][1] * inv0);
            *reinterpret_cast<float2*>(o_p + r1 * DV + n * 8 + 2 * j) = make_float2(acc[n][2] * inv1, acc[n][3] * inv1);
          }
        }
        __threadfence();
        named_bar_sync(1, p.nwc * 32);
        finisher = take_ticket(p.cnt + s_idx, static_cast<int>(ng));
      }
    } else if (npc > 1) {
      finisher = take_ticket(p.cnt + s_idx, static_cast<int>(npc));
    }
    if (finisher) {
      // one 16-row tile of the warp at a time: merge, drafts, output
      auto finish_tile = [&](const int r0, const int r1, const bool first_tile) {
        uint32_t qe[KS][4];  // this tile's query fragments (bf16) for the draft block
      const int kvh = sg.hg * p.HC + hc;
      // the draft rows come from HBM: start them towards L2 now, and (head_dim
      // <= 128) load the query fragments, so both overlap the fold below
      if (first_tile && !p.paged) {
        const int a = p.qo ? __ldg(p.qo + sg.b) : sg.b * p.L;
        if (a >= 0 && static_cast<long long>(a) + p.L <= p.n_rows) {
          constexpr int KL = D * 2 / 128, VL = DV * 2 / 128;  // 128-byte lines of a K / V row
          for (int i = lane; i < p.L * (KL + VL); i += 32) {
            const int t = i / (KL + VL), rest = i % (KL + VL);
            const bool isk = rest < KL;
            const __nv_bfloat16* base = isk ? p.ke + (static_cast<long long>(a) + t) * p.ke_s0
                                            : p.ve + (static_cast<long long>(a) + t) * p.ve_s0;
            prefetch_l2(base + static_cast<long long>(kvh) * (isk ? p.ke_s1 : p.ve_s1) + (isk ? rest : rest - KL) * 64);
          }
        }
      }
      int s_b = 0;
      if constexpr (D <= 128 && DV <= 128) s_b = load_q<KS>(p, sg, hc, r0, r1, j, flagger && first_tile, qe);
      // the pieces (or, for a two-level merge, the group partials) in slot order
      if (tree)
        fold(c_first + s_idx, kGroup, ng, r0, r1);
      else
        fold(c_first + s_idx, 1, npc, r0, r1);
      if constexpr (D > 128 || DV > 128) s_b = load_q<KS>(p, sg, hc, r0, r1, j, flagger && first_tile, qe);
      // ------------- causal draft keys: continue the same online softmax -------------
      const int i0 = r0 / p.gq, i1 = r1 / p.gq;  // draft index of each row
      // tree verify: this sequence's mask rows (row-major [L][P+L], only the
      // draft columns are read); inconsistent offsets fall back to causal
      long long mbase = -1;
      if (p.cmask) {
        const long long m0 = p.mindptr64 ? static_cast<const long long*>(p.mindptr)[sg.b]
                                         : static_cast<long long>(static_cast<const int*>(p.mindptr)[sg.b]);
        const long long span = static_cast<long long>(p.L) * (sg.P + p.L);
        if (m0 >= 0 && m0 + span <= p.n_mask) {
          mbase = m0;
        } else if (flagger) {
          atomicOr(p.err, kErrBadMaskIndptr);
        }
      }
      auto visible = [&](int key, int irow) -> bool {
        if (key >= p.L || irow >= p.L) return false;
        if (mbase < 0) return key <= irow;
        return __ldg(p.cmask + mbase + static_cast<long long>(irow) * (sg.P + p.L) + sg.P + key) != 0;
      };
#pragma unroll 1
      for (int td = 0; td * 8 < p.L; ++td) {
        // fused store (paged): quantise this tile's new draft K and V rows
        // once, store the codes into the cache (the head's first tile) and
        // keep the dequantised values in the warp's idle ring, where the
        // fragment loads below read them
        unsigned char* stK = smem + p.ring_off + warp * (16 * (D + DV));
        unsigned char* stV = stK + 8 * D * 2;
        if (p.wmode == 2) {
          constexpr int PRK = D / 2, PRV = DV / 2;  // bf16 pairs per K / V row
#pragma unroll 1
          for (int idx = lane; idx < 8 * (PRK + PRV); idx += 32) {
            const bool isk = idx < 8 * PRK;
            const int kl = isk ? idx / PRK : (idx - 8 * PRK) / PRV;
            const int c = (isk ? idx % PRK : (idx - 8 * PRK) % PRV) * 2;
            const int key = td * 8 + kl;
            if (key >= p.L) continue;
            const long long row = paged_row(p, sg.b, sg.P + key);
            if (row < 0) continue;
            const long long src = static_cast<long long>(s_b) + key;
            const float2 x = unpack_bf16(isk ? ld_u32(p.ke + src * p.ke_s0 + static_cast<long long>(kvh) * p.ke_s1 + c)
                                             : ld_u32(p.ve + src * p.ve_s0 + static_cast<long long>(kvh) * p.ve_s1 + c));
            unsigned char* dst = isk ? p.kw + row * p.kb_s0 + static_cast<long long>(kvh) * p.kb_s1
                                     : p.vw + row * p.vb_s0 + static_cast<long long>(kvh) * p.vb_s1;
            const float sc = isk ? p.kq : p.vq;
            uint32_t dq;
            if constexpr (FP8) {
              const unsigned short cq = store_e4m3x2(x.x, x.y, sc);
              dq = e4m3x2_to_bf16x2(cq);
              if (first_tile) *reinterpret_cast<unsigned short*>(dst + c) = cq;
            } else {
              dq = store_bf16x2(x.x, x.y, sc);
              if (first_tile) *reinterpret_cast<uint32_t*>(dst + c * 2) = dq;
            }
            if (isk)
              *reinterpret_cast<uint32_t*>(stK + (kl * D + c) * 2) = dq;
            else
              *reinterpret_cast<uint32_t*>(stV + (kl * DV + c) * 2) = dq;
          }
          __syncwarp();
        }
        float sd[4] = {0.f, 0.f, 0.f, 0.f};
        const int tkey = td * 8 + g;  // key whose K row this lane supplies
        bool kv = tkey < p.L;
        unsigned kvm = 0xFFFFFFFFu;  // lane (g, 0) bit set: key td*8+g has a valid row
        if (p.wmode == 2) {
          // the new drafts as stored (staged above)
          const long long krow = kv ? paged_row(p, sg.b, sg.P + tkey) : -1;
          if (tkey < p.L && krow < 0) atomicOr(p.err, kErrBadIndex);
          kv = krow >= 0;
          kvm = __ballot_sync(0xffffffffu, kv);
          const unsigned char* kr = stK + g * D * 2;
#pragma unroll
          for (int kk = 0; kk < KS; ++kk) {
            const uint32_t b0 = kv ? *reinterpret_cast<const uint32_t*>(kr + (kk * 16 + 2 * j) * 2) : 0u;
            const uint32_t b1 = kv ? *reinterpret_cast<const uint32_t*>(kr + (kk * 16 + 8 + 2 * j) * 2) : 0u;
            mma_bf16(sd, qe[kk], b0, b1);
          }
        } else if (p.paged) {
          // drafts are cache positions P + t, dequantised like the prefix
          const long long krow = kv ? paged_row(p, sg.b, sg.P + tkey) : -1;
          if (tkey < p.L && krow < 0) atomicOr(p.err, kErrBadIndex);
          kv = krow >= 0;
          kvm = __ballot_sync(0xffffffffu, kv);
          const unsigned char* kr = p.kb + (kv ? krow : 0) * p.kb_s0 + static_cast<long long>(kvh) * p.kb_s1;
#pragma unroll
          for (int kk = 0; kk < KS; ++kk) {
            uint32_t b0 = 0u, b1 = 0u;
            if (kv) {
              if constexpr (FP8) {
                b0 = e4m3x2_to_bf16x2(*reinterpret_cast<const unsigned short*>(kr + kk * 16 + 2 * j));
                b1 = e4m3x2_to_bf16x2(*reinterpret_cast<const unsigned short*>(kr + kk * 16 + 8 + 2 * j));
              } else {
                b0 = *reinterpret_cast<const uint32_t*>(kr + (kk * 16 + 2 * j) * 2);
                b1 = *reinterpret_cast<const uint32_t*>(kr + (kk * 16 + 8 + 2 * j) * 2);
              }
            }
            mma_bf16(sd, qe[kk], b0, b1);
          }
        } else {
          const __nv_bfloat16* kp = p.ke + (static_cast<long long>(s_b) + (kv ? tkey : 0)) * p.ke_s0 +
                                    static_cast<long long>(kvh) * p.ke_s1;
#pragma unroll
          for (int kk = 0; kk < KS; ++kk) {
            const uint32_t b0 = kv ? ld_u32(kp + kk * 16 + 2 * j) : 0u;
            const uint32_t b1 = kv ? ld_u32(kp + kk * 16 + 8 + 2 * j) : 0u;
            mma_bf16(sd, qe[kk], b0, b1);
          }
          if (p.wmode == 1 && first_tile && kv) {
            // side store of the fresh drafts into rows out_cache_loc[s_b + t]
            const long long dst = p.ocl64 ? static_cast<const long long*>(p.ocl)[s_b + tkey]
                                          : static_cast<long long>(static_cast<const int*>(p.ocl)[s_b + tkey]);
            if (dst >= 0 && dst < p.pool) {
              unsigned char* kr = p.kw + dst * p.kb_s0 + static_cast<long long>(kvh) * p.kb_s1;
#pragma unroll 1
              for (int c2 = 0; c2 < 2 * KS; ++c2) {
                const int c = c2 * 8 + 2 * j;
                const float2 x = unpack_bf16(ld_u32(kp + c));
                if constexpr (FP8)
                  *reinterpret_cast<unsigned short*>(kr + c) = store_e4m3x2(x.x, x.y, p.kq);
                else
                  *reinterpret_cast<uint32_t*>(kr + c * 2) = store_bf16x2(x.x, x.y, p.kq);
              }
            } else if (j == 0) {
              atomicOr(p.err, kErrBadIndex);
            }
          }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = td * 8 + 2 * j + (e & 1);
          const int irow = (e < 2) ? i0 : i1;
          const bool rowok = (kvm >> (((key - td * 8) & 7) * 4)) & 1u;
          sd[e] = (visible(key, irow) && rowok) ? sd[e] * p.dscale2 : NEG_INF;
        }
        const float mx0 = quad_max(fmaxf(sd[0], sd[1]));
        const float mx1 = quad_max(fmaxf(sd[2], sd[3]));
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float ms0 = (mn0 == NEG_INF) ? 0.f : mn0;
        const float ms1 = (mn1 == NEG_INF) ? 0.f : mn1;
        const float a0 = exp2f(m0 - ms0), a1 = exp2f(m1 - ms1);
        float pd[4];
        pd[0] = exp2f(sd[0] - ms0);
        pd[1] = exp2f(sd[1] - ms0);
        pd[2] = exp2f(sd[2] - ms1);
        pd[3] = exp2f(sd[3] - ms1);
        l0 = l0 * a0 + quad_sum(pd[0] + pd[1]);
        l1 = l1 * a1 + quad_sum(pd[2] + pd[3]);
        m0 = mn0;
        m1 = mn1;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          acc[n][0] *= a0;
          acc[n][1] *= a0;
          acc[n][2] *= a1;
          acc[n][3] *= a1;
        }
        // fp32 weighted sum of the draft values of this tile
        bool v_done = false;
        if constexpr (DV <= 128) {
          if (!p.paged && p.wmode == 0) {
            // drafts from v_extend: four keys' value rows per load round trip
#pragma unroll
            for (int kg = 0; kg < 2; ++kg) {
              if (td * 8 + kg * 4 >= p.L) break;  // uniform across the warp
              uint32_t vv[4][NT];
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4) {
                const int key = td * 8 + kg * 4 + q4;
                const bool ok = key < p.L;
                const __nv_bfloat16* vp = p.ve + (static_cast<long long>(s_b) + (ok ? key : 0)) * p.ve_s0 +
                                          static_cast<long long>(kvh) * p.ve_s1 + 2 * j;
#pragma unroll
                for (int n = 0; n < NT; ++n) vv[q4][n] = ok ? ld_u32(vp + n * 8) : 0u;
              }
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4) {
                const int kl = kg * 4 + q4;
                const float w0 = __shfl_sync(0xffffffffu, pd[kl & 1], g * 4 + (kl >> 1)) * p.dvs;
                const float w1 = __shfl_sync(0xffffffffu, pd[2 + (kl & 1)], g * 4 + (kl >> 1)) * p.dvs;
                if (td * 8 + kl >= p.L) continue;  // uniform across the warp
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                  const float2 v = unpack_bf16(vv[q4][n]);
                  acc[n][0] = fmaf(w0, v.x, acc[n][0]);
                  acc[n][1] = fmaf(w0, v.y, acc[n][1]);
                  acc[n][2] = fmaf(w1, v.x, acc[n][2]);
                  acc[n][3] = fmaf(w1, v.y, acc[n][3]);
                }
              }
            }
            v_done = true;
          }
        }
#pragma unroll
        for (int js = 0; js < (v_done ? 0 : 4); ++js) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int key = td * 8 + 2 * js + e;
            if (key >= p.L) continue;  // uniform across the warp
            const float w0 = __shfl_sync(0xffffffffu, pd[e], g * 4 + js) * p.dvs;
            const float w1 = __shfl_sync(0xffffffffu, pd[2 + e], g * 4 + js) * p.dvs;
            if (p.wmode == 2) {
              if (paged_row(p, sg.b, sg.P + key) < 0) continue;  // uniform; its weight is 0
              const unsigned char* vr = stV + ((key - td * 8) * DV + 2 * j) * 2;
#pragma unroll
              for (int n = 0; n < NT; ++n) {
                const float2 v = unpack_bf16(*reinterpret_cast<const uint32_t*>(vr + n * 16));
                acc[n][0] = fmaf(w0, v.x, acc[n][0]);
                acc[n][1] = fmaf(w0, v.y, acc[n][1]);
                acc[n][2] = fmaf(w1, v.x, acc[n][2]);
                acc[n][3] = fmaf(w1, v.y, acc[n][3]);
              }
              continue;
            }
            if (p.paged) {
              const long long vrow = paged_row(p, sg.b, sg.P + key);  // uniform across the warp
              if (vrow < 0) continue;                                   // its weight is 0: never read
              const unsigned char* vr = p.vb + vrow * p.vb_s0 + static_cast<long long>(kvh) * p.vb_s1;
#pragma unroll
              for (int n = 0; n < NT; ++n) {
                float2 v;
                if constexpr (FP8) {
                  v = unpack_bf16(e4m3x2_to_bf16x2(*reinterpret_cast<const unsigned short*>(vr + n * 8 + 2 * j)));
                } else {
                  v = unpack_bf16(*reinterpret_cast<const uint32_t*>(vr + (n * 8 + 2 * j) * 2));
                }
                acc[n][0] = fmaf(w0, v.x, acc[n][0]);
                acc[n][1] = fmaf(w0, v.y, acc[n][1]);
                acc[n][2] = fmaf(w1, v.x, acc[n][2]);
                acc[n][3] = fmaf(w1, v.y, acc[n][3]);
              }
              continue;
            }
            const __nv_bfloat16* vp = p.ve + (static_cast<long long>(s_b) + key) * p.ve_s0 +
                                      static_cast<long long>(kvh) * p.ve_s1 + 2 * j;
            long long vdst = -1;
            if (p.wmode == 1 && first_tile && g == 0) {
              const long long d = p.ocl64 ? static_cast<const long long*>(p.ocl)[s_b + key]
                                          : static_cast<long long>(static_cast<const int*>(p.ocl)[s_b + key]);
              vdst = (d >= 0 && d < p.pool) ? d : -1;  // an out-of-range row is flagged by the K store
            }
            unsigned char* vr = p.vw + (vdst >= 0 ? vdst : 0) * p.vb_s0 + static_cast<long long>(kvh) * p.vb_s1;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
              const float2 v = unpack_bf16(ld_u32(vp + n * 8));
              acc[n][0] = fmaf(w0, v.x, acc[n][0]);
              acc[n][1] = fmaf(w0, v.y, acc[n][1]);
              acc[n][2] = fmaf(w1, v.x, acc[n][2]);
              acc[n][3] = fmaf(w1, v.y, acc[n][3]);
            }
            if (vdst >= 0) {
#pragma unroll 1
              for (int n = 0; n < NT; ++n) {
                const float2 v = unpack_bf16(ld_u32(vp + n * 8));
                if constexpr (FP8)
                  *reinterpret_cast<unsigned short*>(vr + n * 8 + 2 * j) = store_e4m3x2(v.x, v.y, p.vq);
                else
                  *reinterpret_cast<uint32_t*>(vr + (n * 8 + 2 * j) * 2) = store_bf16x2(v.x, v.y, p.vq);
              }
            }
          }
        }
      }
      // ------------------------------ output ------------------------------
      // a row with nothing visible (empty prefix, no visible draft) is 0
      const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
      if (r0 < p.R) {
        __nv_bfloat16* op = p.o + (static_cast<long long>(s_b) + r0 / p.gq) * p.o_s0 +
                            static_cast<long long>(kvh * p.gq + r0 % p.gq) * p.o_s1 + 2 * j;
#pragma unroll
        for (int n = 0; n < NT; ++n)
          *reinterpret_cast<uint32_t*>(op + n * 8) = pack_bf16(acc[n][0] * inv0, acc[n][1] * inv0);
      }
      if (r1 < p.R) {
        __nv_bfloat16* op = p.o + (static_cast<long long>(s_b) + r1 / p.gq) * p.o_s0 +
                            static_cast<long long>(kvh * p.gq + r1 % p.gq) * p.o_s1 + 2 * j;
#pragma unroll
        for (int n = 0; n < NT; ++n)
          *reinterpret_cast<uint32_t*>(op + n * 8) = pack_bf16(acc[n][2] * inv1, acc[n][3] * inv1);
      }
      };
#pragma unroll 1
      for (int t = 0; t < MTW; ++t) finish_tile(r0s[t], r1s[t], mt == 0 && t == 0);
    }
    seg_advance(p, sg);
  }
  }  // !SO
}

#include "verify_tc.cuh"

// Kernel entry points, instantiated per head_dim in vsk_inst_*.cu (nullptr:
// not built).
using KernelFn = void (*)(Params);
// head_dim 64 / 128 (D = Dv): the one-launch kernel (so = false) or the
// stream-only kernel of the two-launch form (so = true), with 1 or 2 tiles
// per warp; cl = true: the cluster form (one tile per warp)
KernelFn kernel_d64(bool fp8, int mtw, bool so, bool cl = false);
KernelFn kernel_d128(bool fp8, int mtw, bool so, bool cl = false);
// head_dim 256 (D = Dv): one-launch kernel (variant 0), column-split stream
// (variant 1), the cluster form streaming by column split (variant 2), the
// one-launch kernel with pipelined stages (variant 3), the column-split
// stream with two tiles per warp (variant 4), the stream-only kernel of the
// two-launch form (variant 5)
KernelFn kernel_d256(bool fp8, int variant);
// tensor-memory stream, head_dim 256, rm = 16 or 32 packed rows
KernelFn kernel_tc(bool fp8, int rm);
// combine kernel of the two-launch forms
KernelFn kernel_combine(int D, bool fp8);
// one-launch kernel with head_dim D != v_head_dim DV
KernelFn kernel_dv(int D, int DV, bool fp8);

}  // namespace vsk
