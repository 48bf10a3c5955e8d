// Split-KV verify attention for EAGLE target-verify at topk = 1, for GB300
// (sm_103a).  The operation is defined on the sglang "verify_splitkv.py" page
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
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/verify_splitkv.h"

#define VSK_VERSION "verify_splitkv-gb300 0.1"

namespace vsk {

// ---------------------------------------------------------------------------
// Constants shared by the host plan and the kernel.
// ---------------------------------------------------------------------------
constexpr int kStageTokens = 16;     // prefix tokens per pipeline stage (one mma k-step)
constexpr int kMaxStages = 5;        // ring depth cap (kIdxAhead >= stages - 1)
constexpr int kIdxAhead = 4;         // stages of kv_indices prefetched ahead of the copies
constexpr int kIdxRing = 8;          // per-warp index ring entries (> kIdxAhead)
constexpr int kCtlBytes = 256;       // control block before the warp regions
constexpr int kSmemPerSM = 233472;   // 228 KB per SM
constexpr int kSmemPerCTAMax = 232448;  // 227 KB opt-in per CTA
constexpr int kReservedPerCTA = 1024;
constexpr int kTicketBytes = 65536;   // minimum ticket region at the end of a workspace
constexpr long long kTwoTileMinTokens = 65536;  // prefix tokens of a call from which warps take two tiles
constexpr long long kColSplitMaxWork = 1LL << 20;  // prefix tokens x KV heads up to which head_dim 256 splits columns
constexpr long long kSplitLaunchMinWork = 2048;        // ... from which head_dim 64 / 128 calls take two launches
constexpr long long kSplitLaunchMaxWork = 1LL << 22;   // ... up to which they do (more than 16 packed rows)
constexpr long long kSplitTwoTileMinTokens = 1LL << 18;  // prefix tokens from which their warps take two tiles
constexpr long long kSplitLaunchMaxWork16 = 1LL << 23;  // ... up to which they do (at most 16 packed rows)
constexpr int kGroup = 4;             // pieces per group of a two-level merge
constexpr int kTreeMin = 6;           // segments of more pieces merge in two levels
constexpr long long kDefaultMinTokens = 64;  // smallest CTA share of the flattened token space
constexpr long long kPiecesPerSegment = 24;    // ... and at least the mean prefix over this many
constexpr long long kPiecesPerSegmentColSplit = 48;  // ... this many for the column-split stream

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

// SO (stream only): the kernel ends once its pieces' partials are written; the
// combine kernel folds them in its own launch.  CS = 2 (head_dim 256, one KV
// head per CTA, at most two 16-row tiles; stream only): each 16-row tile is
// shared by a pair of warps that split the QK contraction (exchanging their
// scaled partial scores through shared memory) and own half of the output
// columns each.  Half the accumulator registers per warp, so three CTAs per SM.
template <int D, bool FP8, int MTW, int CS = 1, bool SO = (CS == 2)>
__global__ void __launch_bounds__(CS == 2 ? 128 : MaxWarps<D>::value * 32, CS == 2 ? 3 : 1)
    vsk_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) unsigned char smem[];
  constexpr int EK = FP8 ? 1 : 2;  // pool element bytes
  constexpr int NT = D / 8;        // n-tiles of the output row
  constexpr int KS = D / 16;       // k-steps of the QK contraction
  static_assert(CS == 1 || (CS == 2 && D == 256 && MTW == 1 && SO), "column split: head_dim 256 stream only");
  constexpr int DH = D / CS;       // output columns (and contraction length) of one warp
  constexpr int NTH = NT / CS;     // its n-tiles
  constexpr int KSH = KS / CS;     // its k-steps
  constexpr int ROWB = D * EK;     // bytes of one head's K (or V) row
  constexpr int CPR = ROWB / 16;   // 16-byte chunks per row
  constexpr int STAGE_B = 2 * kStageTokens * ROWB;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + 16);  // [2]
  const int nst = p.nst;

  // ---- prologue: this CTA's share of the flattened space and its first segment ----
  long long start, end, W;
  Seg seg0;
  if (!cta_share(p, smem, start, end, W, seg0)) return;  // uniform: the whole CTA has no work

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
  const int hc = warp / WPHC;
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
    if (it.valid && lane < min(kStageTokens, it.te - it.tok)) {
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
    if (!it.valid) return;
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
    // lane -> (token group, 16-byte chunk): LPT lanes cover one row, so each
    // lane computes a token's K and V addresses once and issues both copies
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
#pragma unroll 1
  for (int a = 0; a < nst - 1; ++a) {
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

  // The next piece's query fragments are loaded into registers while the
  // current piece streams (head_dim <= 128, one tile per warp), so a piece
  // boundary costs no global round trip.
  constexpr bool kQAhead = D <= 128 && MTW == 1;
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
  while (seg_live(p, s, end)) {
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
#pragma unroll 1
    for (int tok = t0; tok < te; tok += kStageTokens, ++k, kslot = (kslot + 1 == nst) ? 0 : kslot + 1) {
      cp_async_wait_dyn(nst - 2);  // stage k has landed (this lane's copies)
      __syncwarp();                // ... and every other lane's
      // ... and the other warps' of this head: after this barrier no warp of
      // the head still reads the slot of stage k - 1, which step_data refills
      if (WPHC > 1) named_bar_sync(2 + hc, WPHC * 32);
      step_data();                 // refill the slot stage k-1 used
      step_idx();
      cp_async_commit();
      const unsigned mask = mask_ring[k % 16];
      unsigned char* slotp = ring + kslot * STAGE_B;
      // ldmatrix row addresses.  bf16: lanes 0-15 / 16-31 take keys 0-7, 8-15
      // of k-chunk 2kk / 2kk+1 ... (k_key, k_chk); e4m3: lane takes key
      // (lane & 15) and chunk 2kk2 + (lane >> 4), so one x4 load gives both
      // 8-key tiles of two 16-wide d blocks.
      const uint32_t kbase = smem_u32(slotp) + (FP8 ? f_key : k_key) * ROWB;
      const uint32_t vbase = smem_u32(slotp) + 16 * ROWB + (FP8 ? f_key : v_key) * ROWB;

      // S = Q K^T for 16 keys: two n-tiles of 8 keys per 16-row tile.
      // Independent accumulator chains per n-tile (k-step mod NCH) cut the
      // dependent mma latency; summed afterwards.  With two tiles per warp the
      // tiles themselves are independent chains.
      constexpr int NCH = MTW == 1 ? 4 : 1;
      float sc[MTW][2][4];
      float sx[MTW][NCH > 1 ? NCH - 1 : 1][2][4];
#pragma unroll
      for (int t = 0; t < MTW; ++t) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            sc[t][u][e] = 0.f;
#pragma unroll
            for (int c = 0; c < NCH - 1; ++c) sx[t][c][u][e] = 0.f;
          }
        }
      }
      auto qk_step = [&](int kk, uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3) {
        const int ch = kk % NCH;
#pragma unroll
        for (int t = 0; t < MTW; ++t) {
          float* c0 = ch == 0 ? sc[t][0] : sx[t][ch - 1][0];
          float* c1 = ch == 0 ? sc[t][1] : sx[t][ch - 1][1];
          if constexpr (kQSmem) {
            uint32_t a[4];
            ldsm_x4(q_lane + t * 32 * DH + (((2 * kk + (lane >> 4)) ^ (q_row & 7)) << 4), a[0], a[1], a[2], a[3]);
            if constexpr (FP8) {
              mma_f16(c0, a, b0, b1);
              mma_f16(c1, a, b2, b3);
            } else {
              mma_bf16(c0, a, b0, b1);
              mma_bf16(c1, a, b2, b3);
            }
          } else if constexpr (FP8) {
            mma_f16(c0, qf[t][kk], b0, b1);
            mma_f16(c1, qf[t][kk], b2, b3);
          } else {
            mma_bf16(c0, qf[t][kk], b0, b1);
            mma_bf16(c1, qf[t][kk], b2, b3);
          }
        }
      };
      if constexpr (FP8) {
        // each 32-bit register holds 4 consecutive e4m3 d values of one key:
        // low pair -> b0, high pair -> b1 of the permuted contraction order
#pragma unroll
        for (int kk2 = 0; kk2 < KSH / 2; ++kk2) {
          const int c = 2 * (csi * (KSH / 2) + kk2) + (lane >> 4);
          uint32_t r0k, r1k, r2k, r3k;
          ldsm_x4(kbase + ((c ^ chunk_swz<CPR>(f_key)) << 4), r0k, r1k, r2k, r3k);
          qk_step(2 * kk2, e4m3x2_to_f16x2(r0k & 0xFFFF), e4m3x2_to_f16x2(r0k >> 16), e4m3x2_to_f16x2(r1k & 0xFFFF),
                  e4m3x2_to_f16x2(r1k >> 16));
          qk_step(2 * kk2 + 1, e4m3x2_to_f16x2(r2k & 0xFFFF), e4m3x2_to_f16x2(r2k >> 16),
                  e4m3x2_to_f16x2(r3k & 0xFFFF), e4m3x2_to_f16x2(r3k >> 16));
        }
      } else {
#pragma unroll
        for (int kk = 0; kk < KSH; ++kk) {
          uint32_t b0, b1, b2, b3;
          const int lc = (csi * KSH + kk) * 2 + k_chk;
          ldsm_x4(kbase + ((lc ^ (k_key & 7)) << 4), b0, b1, b2, b3);
          qk_step(kk, b0, b1, b2, b3);
        }
      }
      uint32_t pa[MTW][4];
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
            // scale into the log2 domain
            sc[t][u][e] = x * qsc[t];
          }
        }
        if constexpr (CS == 2) {
          // the pair's partial scores (each in the log2 domain already) summed
          // by both warps alike; the buffer alternates with the stage parity
          float* xo = xbuf + static_cast<int>(k & 1) * 256 + lane * 8;
          *reinterpret_cast<float4*>(xo) = make_float4(sc[t][0][0], sc[t][0][1], sc[t][0][2], sc[t][0][3]);
          *reinterpret_cast<float4*>(xo + 4) = make_float4(sc[t][1][0], sc[t][1][1], sc[t][1][2], sc[t][1][3]);
          named_bar_sync(10 + (warp >> 1), 64);
          const float* xp = xo + xpair;
          const float4 y0 = *reinterpret_cast<const float4*>(xp), y1 = *reinterpret_cast<const float4*>(xp + 4);
          sc[t][0][0] += y0.x;
          sc[t][0][1] += y0.y;
          sc[t][0][2] += y0.z;
          sc[t][0][3] += y0.w;
          sc[t][1][0] += y1.x;
          sc[t][1][1] += y1.y;
          sc[t][1][2] += y1.z;
          sc[t][1][3] += y1.w;
        }
        // mask absent keys (tail / dropped) only when the stage is not full
        // (the mask is uniform across the warp)
        if (mask != 0xFFFFu) {
#pragma unroll
          for (int u = 0; u < 2; ++u) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int key = u * 8 + 2 * j + (e & 1);
              if (!((mask >> key) & 1u)) sc[t][u][e] = NEG_INF;
            }
          }
        }
        const float mx0 = quad_max(fmaxf(fmaxf(sc[t][0][0], sc[t][0][1]), fmaxf(sc[t][1][0], sc[t][1][1])));
        const float mx1 = quad_max(fmaxf(fmaxf(sc[t][0][2], sc[t][0][3]), fmaxf(sc[t][1][2], sc[t][1][3])));
        const float mn0 = fmaxf(m0[t], mx0), mn1 = fmaxf(m1[t], mx1);
        const float ms0 = (mn0 == NEG_INF) ? 0.f : mn0;
        const float ms1 = (mn1 == NEG_INF) ? 0.f : mn1;
        float pr[2][4];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          pr[u][0] = fast_exp2(sc[t][u][0] - ms0);
          pr[u][1] = fast_exp2(sc[t][u][1] - ms0);
          pr[u][2] = fast_exp2(sc[t][u][2] - ms1);
          pr[u][3] = fast_exp2(sc[t][u][3] - ms1);
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
#pragma unroll
        for (int c2 = 0; c2 < KSH / 2; ++c2) {
          const int c = 2 * (csi * (KSH / 2) + c2) + (lane >> 4);
          uint32_t r[4];
          ldsm_x4_t(vbase + ((c ^ chunk_swz<CPR>(f_key)) << 4), r[0], r[1], r[2], r[3]);
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
#pragma unroll
        for (int n2 = 0; n2 < NTH / 2; ++n2) {
          uint32_t b0, b1, b2, b3;
          const int lc = (csi * (NTH / 2) + n2) * 2 + v_chk;
          ldsm_x4_t(vbase + ((lc ^ (v_key & 7)) << 4), b0, b1, b2, b3);
#pragma unroll
          for (int t = 0; t < MTW; ++t) {
            mma_bf16(acc[t][2 * n2], pa[t], b0, b1);
            mma_bf16(acc[t][2 * n2 + 1], pa[t], b2, b3);
          }
        }
      }
    }

    // ---------------- piece end: write the partial and keep streaming ----------------
    // (tickets, merges, drafts and output wait until the whole range is streamed)
    {
      const long long slot_self = c_self + static_cast<long long>(s.b) * p.n_hg + s.hg;
      float* lse_p = p.plse + (slot_self * p.HC + hc) * RM;
      float* o_p = p.po + ((slot_self * p.HC + hc) * RM) * D;
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
        float* o0p = o_p + r0 * D + csi * DH;  // this warp's columns
        float* o1p = o_p + r1 * D + csi * DH;
        if constexpr (FP8) {
          // n-tiles E / O of block blk hold d = 16 blk + 4j + {0, 2} / {1, 3}
#pragma unroll
          for (int blk = 0; blk < KSH; ++blk) {
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
#pragma unroll(D <= 128 ? 2 : 1)
    for (long long i = 0; i < count; ++i) {
      const long long sl = slot0 + i * stride;
      const float* lq = p.plse + (sl * p.HC + hc) * RM;
      const float* oq = p.po + ((sl * p.HC + hc) * RM) * D;
      const float w0 = exp2f(__ldcg(lq + r0) - ms0), w1 = exp2f(__ldcg(lq + r1) - ms1);
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const float2 x0 = __ldcg(reinterpret_cast<const float2*>(oq + r0 * D + n * 8 + 2 * j));
        const float2 x1 = __ldcg(reinterpret_cast<const float2*>(oq + r1 * D + n * 8 + 2 * j));
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
        float* o_p = p.po + ((sl * p.HC + hc) * RM) * D;
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
            *reinterpret_cast<float2*>(o_p + r0 * D + n * 8 + 2 * j) = make_float2(acc[n][0] * inv0, acc[n][1] * inv0);
            *reinterpret_cast<float2*>(o_p + r1 * D + n * 8 + 2 * j) = make_float2(acc[n][2] * inv1, acc[n][3] * inv1);
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
          constexpr int LINES = D * 2 / 128;  // 128-byte lines per row
          for (int i = lane; i < p.L * LINES * 2; i += 32) {
            const int t = i / (2 * LINES), rest = i % (2 * LINES);
            const __nv_bfloat16* base = (rest < LINES) ? p.ke + (static_cast<long long>(a) + t) * p.ke_s0
                                                       : p.ve + (static_cast<long long>(a) + t) * p.ve_s0;
            prefetch_l2(base + static_cast<long long>(kvh) * (rest < LINES ? p.ke_s1 : p.ve_s1) + (rest % LINES) * 64);
          }
        }
      }
      int s_b = 0;
      if constexpr (D <= 128) s_b = load_q<KS>(p, sg, hc, r0, r1, j, flagger && first_tile, qe);
      // the pieces (or, for a two-level merge, the group partials) in slot order
      if (tree)
        fold(c_first + s_idx, kGroup, ng, r0, r1);
      else
        fold(c_first + s_idx, 1, npc, r0, r1);
      if constexpr (D > 128) s_b = load_q<KS>(p, sg, hc, r0, r1, j, flagger && first_tile, qe);
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
        unsigned char* stK = smem + p.ring_off + warp * (32 * D);
        unsigned char* stV = stK + 8 * D * 2;
        if (p.wmode == 2) {
          constexpr int PR = D / 2;  // bf16 pairs per row
#pragma unroll 1
          for (int idx = lane; idx < 8 * PR; idx += 32) {
            const int kl = idx / PR, c = (idx % PR) * 2;
            const int key = td * 8 + kl;
            if (key >= p.L) continue;
            const long long row = paged_row(p, sg.b, sg.P + key);
            if (row < 0) continue;
            const long long src = static_cast<long long>(s_b) + key;
            const float2 xk = unpack_bf16(ld_u32(p.ke + src * p.ke_s0 + static_cast<long long>(kvh) * p.ke_s1 + c));
            const float2 xv = unpack_bf16(ld_u32(p.ve + src * p.ve_s0 + static_cast<long long>(kvh) * p.ve_s1 + c));
            unsigned char* kd = p.kw + row * p.kb_s0 + static_cast<long long>(kvh) * p.kb_s1;
            unsigned char* vd = p.vw + row * p.vb_s0 + static_cast<long long>(kvh) * p.vb_s1;
            uint32_t dk, dv;
            if constexpr (FP8) {
              const unsigned short ck = store_e4m3x2(xk.x, xk.y, p.kq);
              const unsigned short cv = store_e4m3x2(xv.x, xv.y, p.vq);
              dk = e4m3x2_to_bf16x2(ck);
              dv = e4m3x2_to_bf16x2(cv);
              if (first_tile) {
                *reinterpret_cast<unsigned short*>(kd + c) = ck;
                *reinterpret_cast<unsigned short*>(vd + c) = cv;
              }
            } else {
              dk = store_bf16x2(xk.x, xk.y, p.kq);
              dv = store_bf16x2(xv.x, xv.y, p.vq);
              if (first_tile) {
                *reinterpret_cast<uint32_t*>(kd + c * 2) = dk;
                *reinterpret_cast<uint32_t*>(vd + c * 2) = dv;
              }
            }
            *reinterpret_cast<uint32_t*>(stK + (kl * D + c) * 2) = dk;
            *reinterpret_cast<uint32_t*>(stV + (kl * D + c) * 2) = dv;
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
        if constexpr (D <= 128) {
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
              const unsigned char* vr = stV + ((key - td * 8) * D + 2 * j) * 2;
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
#include "verify_combine.cuh"

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
thread_local std::string g_err;

int fail(const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return 0;
}

// process-wide tuning overrides (0 = default)
int g_num_ctas = 0;
long long g_min_tokens = 0;
int g_max_stages = 0;
int g_max_heads = 0;
int g_tiles = 0;  // tiles per warp override (0 = default)
int g_tc = 0;     // tensor-memory stream for head_dim 256: 1 on, 0 off (the default: slower here)
int g_cs = 1;     // column-split stream for head_dim 256: 1 below kColSplitMaxWork, 2 always, 0 never
int g_sl = 1;     // stream + combine launches for head_dim 64 / 128: 1 below kSplitLaunchMaxWork, 2 always, 0 never

struct Plan {
  int gq, R, MT, MTW, HC, n_hg, nwc, threads, ek;
  int stage_bytes, nst, ring_off, head_bytes, misc_off, misc_bytes;
  size_t smem;
  int ctas_per_sm;
};

int floor_pow2(int x) {
  int r = 1;
  while (r * 2 <= x) r *= 2;
  return r;
}

// Chooses the CTA shape: HC KV heads per CTA x MT 16-row tiles per head; a
// consumer warp owns MTW tiles (two at head_dim <= 128 when a head has more
// than one tile, so its K / V fragments feed both); ring depth from the
// shared-memory budget.
bool make_plan(long long h_q, long long h_kv, long long D, long long L, bool fp8, Plan& pl,
               long long total_tokens, int tiles) {
  if (h_kv <= 0 || h_q % h_kv != 0) return fail("h_q (%lld) must be a positive multiple of h_kv (%lld)", h_q, h_kv);
  const long long R = (h_q / h_kv) * L;
  const int maxw = D > 128 ? 4 : 8;
  if (R > 16LL * maxw) return fail("packed rows (h_q/h_kv)*l_ext = %lld exceed %d for head_dim %lld", R, 16 * maxw, D);
  pl.gq = static_cast<int>(h_q / h_kv);
  pl.R = static_cast<int>(R);
  int mt = 1;
  while (16 * mt < R) mt *= 2;
  pl.MT = mt;
  // two tiles per warp pay off once there is enough prefix to stream;
  // small problems are latency bound and want more, lighter warps
  if (tiles == 0) tiles = g_tiles;
  if (tiles == 0) tiles = total_tokens >= kTwoTileMinTokens ? 2 : 1;
  pl.MTW = (D <= 128 && mt >= 2 && tiles == 2) ? 2 : 1;
  const int wph = mt / pl.MTW;  // warps per head
  int hc = 1;
  const int hc_cap = g_max_heads > 0 ? g_max_heads : maxw;
  while (hc * 2 * wph <= maxw && hc * 2 <= hc_cap && h_kv % (hc * 2) == 0) hc *= 2;
  pl.HC = hc;
  pl.n_hg = static_cast<int>(h_kv / hc);
  pl.nwc = hc * wph;
  pl.threads = pl.nwc * 32;
  pl.ek = fp8 ? 1 : 2;
  // per head: nst stages of 16 K rows + 16 V rows; per warp: the index ring,
  // the mask ring and (two-tile warps; e4m3 pools at head_dim 256) the query tiles
  pl.stage_bytes = 2 * kStageTokens * static_cast<int>(D) * pl.ek;
  const int qsm_tiles = (fp8 && D == 256) ? 1 : (pl.MTW == 2 ? 2 : 0);  // query tiles kept in shared memory
  const int fixed = kIdxRing * 128 + 128 + qsm_tiles * 16 * static_cast<int>(D) * 2;
  // CTAs per SM: as many as keep about 8 warps per SM with a ring of at
  // least 3 stages (2 if nothing better fits)
  const int kmax = pl.nwc >= 8 ? 1 : (pl.nwc >= 4 ? 2 : 4);
  const int cap = g_max_stages > 0 ? std::min(g_max_stages, kMaxStages) : kMaxStages;
  pl.nst = 0;
  for (int want = 3; want >= 2 && pl.nst == 0; --want) {
    for (int k = kmax; k >= 1; --k) {
      const int budget = std::min(kSmemPerCTAMax, kSmemPerSM / k - kReservedPerCTA);
      const int nst = std::min(cap, (budget - kCtlBytes - pl.nwc * fixed) / (pl.HC * pl.stage_bytes));
      if (nst >= std::min(want, cap)) {
        pl.nst = nst;
        pl.ctas_per_sm = k;
        break;
      }
    }
  }
  if (pl.nst < 2) return fail("stage of %d bytes does not fit shared memory", pl.stage_bytes);
  pl.head_bytes = pl.nst * pl.stage_bytes;
  pl.misc_bytes = fixed;
  pl.ring_off = kCtlBytes;
  // the ring region also holds each warp's staged drafts (32 * D bytes) after streaming
  const int rings = std::max(pl.HC * pl.head_bytes, pl.nwc * 32 * static_cast<int>(D));
  pl.misc_off = pl.ring_off + rings;
  pl.smem = static_cast<size_t>(pl.misc_off) + static_cast<size_t>(pl.nwc) * pl.misc_bytes;
  if (pl.smem > static_cast<size_t>(kSmemPerCTAMax)) return fail("shared memory plan of %zu bytes too large", pl.smem);
  return true;
}

// The tensor-memory stream (vtc_kernel) serves head_dim 256 with at most 32
// packed query rows per KV head.
bool tc_eligible(long long h_q, long long h_kv, long long D, long long L) {
  if (g_tc != 1 || D != 256 || h_kv <= 0 || h_q % h_kv != 0) return false;
  return (h_q / h_kv) * L <= 32;
}

// Plan fields of a two-launch call (tensor-memory or column-split stream,
// then the combine kernel): one KV head per segment, RM = 16 or 32 packed
// rows (MT = RM / 16 tiles).  The stream kernel sets its own launch shape.
bool make_tc_plan(long long h_q, long long h_kv, long long D, long long L, bool fp8, Plan& pl) {
  if (h_kv <= 0 || h_q % h_kv != 0) return fail("h_q (%lld) must be a positive multiple of h_kv (%lld)", h_q, h_kv);
  const long long R = (h_q / h_kv) * L;
  if (R > 32) return fail("packed rows %lld exceed 32", R);
  pl.gq = static_cast<int>(h_q / h_kv);
  pl.R = static_cast<int>(R);
  pl.MT = R <= 16 ? 1 : 2;
  pl.MTW = 1;
  pl.HC = 1;
  pl.n_hg = static_cast<int>(h_kv);
  pl.nwc = pl.MT;
  pl.threads = pl.nwc * 32;
  pl.ek = fp8 ? 1 : 2;
  pl.stage_bytes = 0;
  pl.nst = 0;
  pl.ring_off = kCtlBytes;
  pl.head_bytes = 0;
  pl.misc_bytes = 0;
  pl.misc_off = kCtlBytes + pl.nwc * 32 * static_cast<int>(D);
  pl.smem = static_cast<size_t>(pl.misc_off);
  pl.ctas_per_sm = 1;
  return true;
}

// Column-split stream (vsk_kernel<256, ., 1, false, 2>): head_dim 256 with at
// most 32 packed rows per KV head.  The workspace / epilogue plan is the
// tensor-memory one (one KV head per segment, MT = RM / 16, the epilogue in
// MT warps); the stream runs 2 MT warps per CTA, three CTAs per SM.  Lighter
// warps, more CTAs and the ticket-free combine launch shorten small calls; on
// long ones the pair exchange costs more than it saves, so by default only
// calls of at most kColSplitMaxWork prefix tokens x KV heads (from static
// shapes) take it.
bool cs_eligible(long long h_q, long long h_kv, long long D, long long L, long long total_tokens) {
  if (g_cs == 0 || D != 256 || h_kv <= 0 || h_q % h_kv != 0 || (h_q / h_kv) * L > 32) return false;
  return g_cs == 2 || total_tokens * h_kv <= kColSplitMaxWork;
}
// Stream-only vsk_kernel then the combine kernel, for head_dim 64 / 128 calls
// with at most cmb::kMaxL drafts: small and mid-size calls, where the
// one-launch kernel's tail (tickets, a two-level fold of the pieces, the
// draft block) is a chain of memory round trips that the combine launch
// shortens.  Not for the very smallest (the second launch costs more than it
// saves), nor for long batches, where the one-launch kernel's finishers hide
// its tail behind other CTAs' streaming.  Warps take two tiles (more than 16
// packed rows) from kSplitTwoTileMinTokens prefix tokens.
bool sl_eligible(long long h_q, long long h_kv, long long D, long long L, long long total_tokens) {
  if (g_sl == 0 || (D != 64 && D != 128) || h_kv <= 0 || h_q % h_kv != 0 || L > cmb::kMaxL) return false;
  if (g_sl == 2) return true;
  const long long work = total_tokens * h_kv;
  const long long cap = (h_q / h_kv) * L <= 16 ? kSplitLaunchMaxWork16 : kSplitLaunchMaxWork;
  return work >= kSplitLaunchMinWork && work <= cap;
}
struct StreamPlan {
  int threads, nst, ring_off, head_bytes, misc_off, misc_bytes, per_sm;
  size_t smem;
};
bool make_cs_stream_plan(const Plan& pl, long long D, bool fp8, StreamPlan& sp) {
  const int nwc = 2 * pl.MT;
  sp.threads = nwc * 32;
  sp.per_sm = 3;
  const int stage_bytes = 2 * kStageTokens * static_cast<int>(D) * (fp8 ? 1 : 2);
  // per warp: index ring, mask ring, query tile (e4m3 pools: 16 rows x D/2 f16), score exchange buffer (2 x 1 KB)
  sp.misc_bytes = kIdxRing * 128 + 128 + (fp8 ? 16 * static_cast<int>(D / 2) * 2 : 0) + 2048;
  const int budget = std::min(kSmemPerCTAMax, kSmemPerSM / sp.per_sm - kReservedPerCTA);
  sp.nst = std::min(kMaxStages, (budget - kCtlBytes - nwc * sp.misc_bytes) / stage_bytes);
  if (g_max_stages > 0) sp.nst = std::min(sp.nst, g_max_stages);
  if (sp.nst < 2) return fail("column-split stage of %d bytes does not fit shared memory", stage_bytes);
  sp.ring_off = kCtlBytes;
  sp.head_bytes = sp.nst * stage_bytes;
  sp.misc_off = sp.ring_off + sp.head_bytes;
  sp.smem = static_cast<size_t>(sp.misc_off) + static_cast<size_t>(nwc) * sp.misc_bytes;
  return true;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Workspace: the error word at offset 0, the partials from offset 256 up,
// and the tickets in the LAST cnt_bytes of the buffer, at least 64 KiB.  The
// tickets' place is then the same for every call on a given buffer whatever
// its shapes (up to 16,384 tickets), so the zero tickets a call leaves are the
// ones the next call finds, and no call's partials reach them.
struct WsLayout {
  size_t lse_off, o_off, cnt_bytes, total;
};

WsLayout ws_layout(long long n_cta, long long B, const Plan& pl, long long D) {
  WsLayout w;
  const long long segs = B * pl.n_hg;
  const long long slots = n_cta + segs;
  const long long rows = slots * pl.HC * 16LL * pl.MT;
  w.lse_off = 256;
  w.o_off = w.lse_off + align256(4 * static_cast<size_t>(rows));
  w.cnt_bytes = std::max(static_cast<size_t>(kTicketBytes), align256(4 * static_cast<size_t>(segs + slots)));
  w.total = align256(w.o_off + 4 * static_cast<size_t>(rows) * static_cast<size_t>(D)) + w.cnt_bytes;
  return w;
}



struct DevWs {
  void* ptr = nullptr;
  size_t bytes = 0;
};
std::mutex g_ws_mu;
std::vector<DevWs> g_ws;
std::vector<int> g_sms;

int device_sms(int dev) {
  std::lock_guard<std::mutex> lk(g_ws_mu);
  if (static_cast<int>(g_sms.size()) <= dev) g_sms.resize(dev + 1, 0);
  if (g_sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sms[dev] = n;
  }
  return g_sms[dev];
}

bool check_3d(const vsk_tensor* t, const char* name) {
  if (!t) return fail("%s is NULL", name);
  if (t->ndim != 3) return fail("%s must be 3-d (got ndim %d)", name, t->ndim);
  for (int i = 0; i < 3; ++i)
    if (t->shape[i] < 0) return fail("%s has a negative extent", name);
  if (t->shape[0] > 0 && t->shape[1] > 0 && t->shape[2] > 1 && t->stride[2] != 1)
    return fail("%s: last dimension must be contiguous", name);
  const long long n = t->shape[0] * t->shape[1] * t->shape[2];
  if (n > 0 && !t->data) return fail("%s: NULL data with %lld elements", name, n);
  return true;
}

bool check_1d(const vsk_tensor* t, const char* name) {
  if (!t) return fail("%s is NULL", name);
  if (t->ndim != 1) return fail("%s must be 1-d (got ndim %d)", name, t->ndim);
  if (t->shape[0] < 0) return fail("%s has a negative extent", name);
  if (t->shape[0] > 1 && t->stride[0] != 1) return fail("%s must be contiguous", name);
  if (t->shape[0] > 0 && !t->data) return fail("%s: NULL data", name);
  return true;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// can_handle of the "verify_splitkv.py" page plus this build's limits.
bool gate(const vsk_tensor* q, const vsk_tensor* ke, const vsk_tensor* ve, const vsk_tensor* kb,
          const vsk_tensor* vb, const vsk_tensor* qo, const vsk_tensor* kvp, const vsk_tensor* kvi,
          int is_causal, long long mle, long long sliding_window, int has_sinks, float logit_cap,
          long long xai_len) {
  // features the kernel does not implement
  if (has_sinks) return fail("attention sinks are not supported");
  if (sliding_window > 0) return fail("sliding_window_size > 0 is not supported");
  if (logit_cap > 0.f) return fail("logit_cap > 0 is not supported");
  if (xai_len > 0) return fail("xai_temperature_len > 0 is not supported");
  if (!is_causal) return fail("only causal (topk = 1) verify is supported");
  if (!check_3d(q, "q_extend") || !check_3d(ke, "k_extend") || !check_3d(ve, "v_extend") ||
      !check_3d(kb, "k_buffer") || !check_3d(vb, "v_buffer"))
    return false;
  if (!check_1d(qo, "qo_indptr") || !check_1d(kvp, "kv_indptr") || !check_1d(kvi, "kv_indices")) return false;
  const long long h_q = q->shape[1], h_kv = ke->shape[1];
  if (h_kv == 0 || h_q % h_kv != 0) return fail("h_q (%lld) is not a multiple of h_kv (%lld)", h_q, h_kv);
  if (kb->shape[1] != h_kv || vb->shape[1] != h_kv || ve->shape[1] != h_kv)
    return fail("KV head count mismatch between k_extend, v_extend and the buffers");
  const long long D = q->shape[2], Dv = ve->shape[2];
  if (ke->shape[2] != D || kb->shape[2] != D) return fail("head_dim mismatch between q, k_extend and k_buffer");
  if (vb->shape[2] != Dv) return fail("v_head_dim mismatch between v_extend and v_buffer");
  const long long bs = qo->shape[0] - 1;
  if (bs < 1) return fail("batch size must be >= 1");
  if (kvp->shape[0] != bs + 1) return fail("kv_indptr must have B+1 entries");
  if (mle < 1) return fail("max_len_extend must be >= 1");
  if (q->shape[0] != bs * mle) return fail("ragged extend: q has %lld rows, expected B*max_len_extend = %lld", q->shape[0], bs * mle);
  if (ke->shape[0] != q->shape[0] || ve->shape[0] != q->shape[0]) return fail("k_extend/v_extend rows differ from q_extend");
  if (kb->shape[0] != vb->shape[0]) return fail("k_buffer and v_buffer pools differ in size");
  // this build's limits
  if (D != Dv) return fail("head_dim (%lld) != v_head_dim (%lld) is not built", D, Dv);
  if (D != 64 && D != 128 && D != 256) return fail("head_dim %lld not in {64, 128, 256}", D);
  if (q->dtype != VSK_DTYPE_BF16 || ke->dtype != VSK_DTYPE_BF16 || ve->dtype != VSK_DTYPE_BF16)
    return fail("q_extend, k_extend and v_extend must be bf16");
  if (kb->dtype != vb->dtype || (kb->dtype != VSK_DTYPE_BF16 && kb->dtype != VSK_DTYPE_FP8E4M3))
    return fail("k_buffer and v_buffer must both be bf16 or both fp8 e4m3");
  if (qo->dtype != VSK_DTYPE_I32 || kvp->dtype != VSK_DTYPE_I32) return fail("indptr arrays must be int32");
  if (kvi->dtype != VSK_DTYPE_I32 && kvi->dtype != VSK_DTYPE_I64) return fail("kv_indices must be int32 or int64");
  const long long R = (h_q / h_kv) * mle;
  const long long maxR = D > 128 ? 64 : 128;
  if (R > maxR) return fail("(h_q/h_kv)*max_len_extend = %lld exceeds %lld", R, maxR);
  const size_t ek = kb->dtype == VSK_DTYPE_BF16 ? 2 : 1;
  for (const vsk_tensor* t : {kb, vb}) {
    if (!aligned(t->data, 16) || (t->stride[0] * ek) % 16 != 0 || (t->stride[1] * ek) % 16 != 0)
      return fail("K/V pool rows must be 16-byte aligned");
  }
  for (const vsk_tensor* t : {q, ke, ve}) {
    if (!aligned(t->data, 4) || (t->stride[0] % 2) != 0 || (t->stride[1] % 2) != 0)
      return fail("q_extend/k_extend/v_extend must be 4-byte aligned with even strides");
  }
  return true;
}

using KernelFn = void (*)(Params);

template <int D, bool FP8, int MTW>
KernelFn kernel_ptr() {
  return vsk_kernel<D, FP8, MTW>;
}

KernelFn pick_kernel(int D, bool fp8, int mtw) {
  if (mtw == 2) {
    switch (D) {
      case 64: return fp8 ? kernel_ptr<64, true, 2>() : kernel_ptr<64, false, 2>();
      case 128: return fp8 ? kernel_ptr<128, true, 2>() : kernel_ptr<128, false, 2>();
      default: return nullptr;
    }
  }
  switch (D) {
    case 64: return fp8 ? kernel_ptr<64, true, 1>() : kernel_ptr<64, false, 1>();
    case 128: return fp8 ? kernel_ptr<128, true, 1>() : kernel_ptr<128, false, 1>();
    case 256: return fp8 ? kernel_ptr<256, true, 1>() : kernel_ptr<256, false, 1>();
    default: return nullptr;
  }
}

KernelFn pick_tc_kernel(bool fp8, int rm) {
  if (rm == 16) return fp8 ? static_cast<KernelFn>(vtc_kernel<256, true, 16>) : static_cast<KernelFn>(vtc_kernel<256, false, 16>);
  return fp8 ? static_cast<KernelFn>(vtc_kernel<256, true, 32>) : static_cast<KernelFn>(vtc_kernel<256, false, 32>);
}

KernelFn pick_cs_kernel(bool fp8) {
  return fp8 ? static_cast<KernelFn>(vsk_kernel<256, true, 1, 2>) : static_cast<KernelFn>(vsk_kernel<256, false, 1, 2>);
}

KernelFn pick_so_kernel(int D, bool fp8, int mtw) {
  if (mtw == 2) {
    switch (D) {
      case 64: return fp8 ? static_cast<KernelFn>(vsk_kernel<64, true, 2, 1, true>)
                          : static_cast<KernelFn>(vsk_kernel<64, false, 2, 1, true>);
      case 128: return fp8 ? static_cast<KernelFn>(vsk_kernel<128, true, 2, 1, true>)
                           : static_cast<KernelFn>(vsk_kernel<128, false, 2, 1, true>);
      default: return nullptr;
    }
  }
  switch (D) {
    case 64: return fp8 ? static_cast<KernelFn>(vsk_kernel<64, true, 1, 1, true>)
                        : static_cast<KernelFn>(vsk_kernel<64, false, 1, 1, true>);
    case 128: return fp8 ? static_cast<KernelFn>(vsk_kernel<128, true, 1, 1, true>)
                         : static_cast<KernelFn>(vsk_kernel<128, false, 1, 1, true>);
    default: return nullptr;
  }
}

KernelFn pick_combine_kernel(int D, bool fp8) {
  switch (D) {
    case 64: return fp8 ? static_cast<KernelFn>(vsk_combine_kernel<64, true>)
                        : static_cast<KernelFn>(vsk_combine_kernel<64, false>);
    case 128: return fp8 ? static_cast<KernelFn>(vsk_combine_kernel<128, true>)
                         : static_cast<KernelFn>(vsk_combine_kernel<128, false>);
    case 256: return fp8 ? static_cast<KernelFn>(vsk_combine_kernel<256, true>)
                         : static_cast<KernelFn>(vsk_combine_kernel<256, false>);
    default: return nullptr;
  }
}

int combine_smem(int D) {
  return D == 64 ? cmb::Geo<64>::kSmem : D == 128 ? cmb::Geo<128>::kSmem : cmb::Geo<256>::kSmem;
}


// Ring entries and shared memory of vtc_kernel (e4m3 pools: an even number
// of entries, so that V rows always sit in odd entries).
template <bool FP8, int RM>
void tc_smem(int& ne, size_t& smem) {
  using G = tc::Geo<256, FP8, RM>;
  ne = std::min(tc::kMaxNE, (kSmemPerCTAMax - G::ring_off) / G::ENT);
  if (FP8) ne &= ~1;
  smem = static_cast<size_t>(G::ring_off) + static_cast<size_t>(ne) * G::ENT;
}

int prepare_kernel(KernelFn fn) {
  // the attribute is per function and context; set it before every launch
  // configuration query (cheap, idempotent)
  return cudaFuncSetAttribute(reinterpret_cast<const void*>(fn), cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSmemPerCTAMax) == cudaSuccess;
}

void* internal_workspace(int dev, size_t need, cudaStream_t stream, size_t* bytes) {
  std::lock_guard<std::mutex> lk(g_ws_mu);
  if (static_cast<int>(g_ws.size()) <= dev) g_ws.resize(dev + 1);
  DevWs& w = g_ws[dev];
  if (w.bytes >= need) {
    *bytes = w.bytes;
    return w.ptr;
  }
  if (w.ptr) {
    cudaStreamSynchronize(stream);
    cudaFree(w.ptr);
    w.ptr = nullptr;
    w.bytes = 0;
  }
  void* p = nullptr;
  if (cudaMalloc(&p, need) != cudaSuccess) return nullptr;
  if (cudaMemset(p, 0, need) != cudaSuccess) {
    cudaFree(p);
    return nullptr;
  }
  w.ptr = p;
  w.bytes = need;
  *bytes = need;
  return p;
}

// device address of the allocation-free entry point's built-in scratch
void* static_scratch(int dev);

}  // namespace vsk

using namespace vsk;

extern "C" {

int vsk_can_handle(const vsk_tensor* q_extend, const vsk_tensor* k_extend, const vsk_tensor* v_extend,
                   const vsk_tensor* k_buffer, const vsk_tensor* v_buffer, const vsk_tensor* qo_indptr,
                   const vsk_tensor* kv_indptr, const vsk_tensor* kv_indices, int is_causal,
                   int64_t max_len_extend, int64_t sliding_window_size, int has_sinks, float logit_cap,
                   int64_t xai_temperature_len) {
  g_err.clear();
  return gate(q_extend, k_extend, v_extend, k_buffer, v_buffer, qo_indptr, kv_indptr, kv_indices, is_causal,
              max_len_extend, sliding_window_size, has_sinks, logit_cap, xai_temperature_len)
             ? 1
             : 0;
}

size_t vsk_workspace_size_for_sms(int num_sms, int64_t max_bs, int64_t h_q, int64_t h_kv, int64_t head_dim,
                                  int64_t v_head_dim, int64_t max_len_extend) {
  if (num_sms <= 0 || max_bs < 1 || head_dim != v_head_dim || max_len_extend < 1) return 0;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return 0;
  const long long n_cta = static_cast<long long>(num_sms) * 4;  // bound on CTAs per SM
  size_t need = 0;
  for (int fp8 = 0; fp8 < 2; ++fp8) {
    for (int tiles = 1; tiles <= 2; ++tiles) {
      Plan pl;
      if (!make_plan(h_q, h_kv, head_dim, max_len_extend, fp8 != 0, pl, 0, tiles)) return 0;
      need = std::max(need, ws_layout(n_cta, max_bs, pl, head_dim).total);
    }
  }
  Plan tp;
  if (head_dim == 256 && (h_q / h_kv) * max_len_extend <= 32 && make_tc_plan(h_q, h_kv, head_dim, max_len_extend, false, tp))
    need = std::max(need, ws_layout(n_cta, max_bs, tp, head_dim).total);
  return need;
}

size_t vsk_workspace_size(int64_t max_bs, int64_t h_q, int64_t h_kv, int64_t head_dim, int64_t v_head_dim,
                          int64_t max_len_extend) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const int sms = device_sms(dev);
  if (sms <= 0) return 0;
  size_t need = vsk_workspace_size_for_sms(sms, max_bs, h_q, h_kv, head_dim, v_head_dim, max_len_extend);
  if (g_num_ctas > 4 * sms) {
    for (int tiles = 1; tiles <= 2; ++tiles) {
      Plan pl;
      if (make_plan(h_q, h_kv, head_dim, max_len_extend, false, pl, 0, tiles)) {
        const size_t t = ws_layout(g_num_ctas, max_bs, pl, head_dim).total;
        if (t > need) need = t;
      }
    }
    Plan tp;
    if (head_dim == 256 && h_kv > 0 && h_q % h_kv == 0 && (h_q / h_kv) * max_len_extend <= 32 &&
        make_tc_plan(h_q, h_kv, head_dim, max_len_extend, false, tp)) {
      const size_t t = ws_layout(g_num_ctas, max_bs, tp, head_dim).total;
      if (t > need) need = t;
    }
  }
  return need;
}

int vsk_workspace_init(void* workspace, size_t bytes, void* stream) {
  g_err.clear();
  if (!workspace || bytes == 0) return 1;
  const cudaError_t e = cudaMemsetAsync(workspace, 0, bytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail("cudaMemsetAsync: %s", cudaGetErrorString(e));
  return 1;
}

int vsk_read_error_flags(void* workspace, void* stream, uint32_t* flags) {
  g_err.clear();
  if (!flags) return fail("flags is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return fail("cudaStreamSynchronize: %s", cudaGetErrorString(e));
  void* ws = workspace;
  if (!ws || ws == VSK_NOALLOC_SCRATCH) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail("no CUDA device");
    if (ws == VSK_NOALLOC_SCRATCH) {
      ws = static_scratch(dev);
      if (!ws) return 0;
    } else {
      std::lock_guard<std::mutex> lk(g_ws_mu);
      if (static_cast<int>(g_ws.size()) > dev) ws = g_ws[dev].ptr;
    }
  }
  if (!ws) {
    *flags = 0;
    return 1;
  }
  e = cudaMemcpy(flags, ws, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail("cudaMemcpy: %s", cudaGetErrorString(e));
  e = cudaMemset(ws, 0, sizeof(uint32_t));
  if (e != cudaSuccess) return fail("cudaMemset: %s", cudaGetErrorString(e));
  return 1;
}

void vsk_set_tuning(int num_ctas, int min_tokens_per_cta) {
  g_num_ctas = num_ctas > 0 ? num_ctas : 0;
  g_min_tokens = min_tokens_per_cta > 0 ? min_tokens_per_cta : 0;
}

void vsk_set_tuning_tiles(int tiles_per_warp) { g_tiles = tiles_per_warp == 1 || tiles_per_warp == 2 ? tiles_per_warp : 0; }

void vsk_set_tuning_tc(int mode) { g_tc = mode == 1 ? 1 : 0; }

void vsk_set_tuning_colsplit(int mode) { g_cs = (mode == 0 || mode == 2) ? mode : 1; }

void vsk_set_tuning_split_launch(int mode) { g_sl = (mode == 0 || mode == 2) ? mode : 1; }

int vsk_launches_per_call(int64_t batch, int64_t h_q, int64_t h_kv, int64_t head_dim, int64_t max_len_extend,
                          int64_t prefix_tokens) {
  if (batch < 1 || h_kv <= 0 || h_q % h_kv != 0 || max_len_extend < 1 || prefix_tokens < 0) return 0;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return 0;
  const long long tokens = prefix_tokens / batch * batch;  // the entry points' static estimate
  return (tc_eligible(h_q, h_kv, head_dim, max_len_extend) ||
          cs_eligible(h_q, h_kv, head_dim, max_len_extend, tokens) ||
          sl_eligible(h_q, h_kv, head_dim, max_len_extend, tokens))
             ? 2
             : 1;
}

void vsk_set_tuning_shape(int max_ring_stages, int max_kv_heads_per_cta) {
  g_max_stages = max_ring_stages >= 2 ? max_ring_stages : 0;
  g_max_heads = max_kv_heads_per_cta > 0 ? max_kv_heads_per_cta : 0;
}

const char* vsk_last_error(void) { return g_err.c_str(); }

const char* vsk_version(void) { return VSK_VERSION; }

}  // extern "C"

namespace vsk {
// Everything the launches of one call need, decided from static shapes only
// (no device read): the form (one launch, or a stream then the combine
// kernel), the CTA shape, the kernels, the grid, the share floor and the
// workspace layout.  Every entry point plans a call with plan_call and
// enqueues it with enqueue_call, so the workspace a caller (or the built-in
// scratch of the allocation-free entry point) is checked against is the one
// the kernels use.
struct CallPlan {
  bool use_tc = false, use_cs = false, use_sl = false;
  Plan pl{};
  StreamPlan sp{};
  KernelFn fn = nullptr, fn_comb = nullptr;
  int threads = 0;
  size_t smem = 0;
  long long n_cta = 0, n_comb = 0, w_min = 0;
  WsLayout wl{};
  int dev = 0;
  int D = 0;
};

static int plan_call(long long B, long long h_q, long long h_kv, long long D, long long L, bool fp8,
                     long long mean_len, CallPlan& cp) {
  cp.D = static_cast<int>(D);
  cp.use_tc = tc_eligible(h_q, h_kv, D, L);
  cp.use_cs = !cp.use_tc && cs_eligible(h_q, h_kv, D, L, mean_len * B);
  cp.use_sl = !cp.use_tc && !cp.use_cs && sl_eligible(h_q, h_kv, D, L, mean_len * B);
  Plan& pl = cp.pl;
  if ((cp.use_tc || cp.use_cs)
          ? !make_tc_plan(h_q, h_kv, D, L, fp8, pl)
          : !make_plan(h_q, h_kv, D, L, fp8, pl, mean_len * B,
                       cp.use_sl && g_tiles == 0 ? (mean_len * B >= kSplitTwoTileMinTokens ? 2 : 1) : 0))
    return 0;
  if (cp.use_cs && !make_cs_stream_plan(pl, D, fp8, cp.sp)) return 0;
  cudaError_t e = cudaGetDevice(&cp.dev);
  if (e != cudaSuccess) return fail("cudaGetDevice: %s", cudaGetErrorString(e));
  const int sms = device_sms(cp.dev);
  if (sms <= 0) return fail("cannot query the SM count of device %d", cp.dev);
  // the streaming kernel (the whole call on the one-launch path; the prefix
  // stream on the two-launch paths, followed by the combine kernel)
  cp.threads = pl.threads;
  cp.smem = pl.smem;
  int per_sm = pl.ctas_per_sm;
  if (cp.use_tc) {
    const int rm = 16 * pl.MT;
    cp.fn = pick_tc_kernel(fp8, rm);
    cp.fn_comb = pick_combine_kernel(256, fp8);
    if (!prepare_kernel(cp.fn) || !prepare_kernel(cp.fn_comb)) return fail("tensor-memory kernels unavailable");
    int ne = 0;
    if (fp8)
      rm == 16 ? tc_smem<true, 16>(ne, cp.smem) : tc_smem<true, 32>(ne, cp.smem);
    else
      rm == 16 ? tc_smem<false, 16>(ne, cp.smem) : tc_smem<false, 32>(ne, cp.smem);
    if (ne < 4) return fail("tensor-memory ring of %d entries is too shallow", ne);
    pl.nst = ne;
    cp.threads = tc::kThreads;
  } else if (cp.use_cs) {
    cp.fn = pick_cs_kernel(fp8);
    cp.fn_comb = pick_combine_kernel(256, fp8);
    if (!prepare_kernel(cp.fn) || !prepare_kernel(cp.fn_comb)) return fail("column-split kernels unavailable");
    cp.threads = cp.sp.threads;
    cp.smem = cp.sp.smem;
    per_sm = cp.sp.per_sm;
  } else if (cp.use_sl) {
    cp.fn = pick_so_kernel(static_cast<int>(D), fp8, pl.MTW);
    cp.fn_comb = pick_combine_kernel(static_cast<int>(D), fp8);
    if (!cp.fn || !cp.fn_comb || !prepare_kernel(cp.fn) || !prepare_kernel(cp.fn_comb))
      return fail("stream-only kernels for head_dim %lld unavailable", D);
  } else {
    cp.fn = pick_kernel(static_cast<int>(D), fp8, pl.MTW);
    if (!cp.fn || !prepare_kernel(cp.fn)) return fail("kernel for head_dim %lld unavailable", D);
  }
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, reinterpret_cast<const void*>(cp.fn), cp.threads, cp.smem);
  if (e != cudaSuccess || occ < 1) return fail("kernel does not fit an SM (%s)", cudaGetErrorString(e));
  per_sm = std::min(occ, per_sm);
  cp.n_cta = g_num_ctas > 0 ? g_num_ctas : static_cast<long long>(sms) * per_sm;
  cp.wl = ws_layout(cp.n_cta, B, pl, D);
  if (cp.fn_comb) {
    // one combine CTA per (segment, 16-row tile, 32-column slice)
    cp.n_comb = B * pl.n_hg * pl.HC * pl.MT * (D / cmb::kCols);
    if (cp.n_comb > 0x7FFFFFFFLL) return fail("combine grid of %lld CTAs too large", cp.n_comb);
  }
  // Smallest CTA share, from static shapes only (no device read, graph
  // safe): at least 64 tokens and, for small batches where the shares get
  // short, at least the mean prefix / 24 in whole stages, which bounds the
  // pieces a segment's finisher merges.  The two-launch forms (partials
  // folded by the combine launch) do best with every CTA busy: mean prefix / 48.
  if (g_min_tokens > 0) {
    cp.w_min = g_min_tokens;
  } else {
    const long long per = (cp.use_cs || cp.use_sl) ? kPiecesPerSegmentColSplit : kPiecesPerSegment;
    const long long wp = (mean_len / per + kStageTokens - 1) / kStageTokens * kStageTokens;
    cp.w_min = std::max(kDefaultMinTokens, wp);
  }
  return 1;
}

// Fills the plan-dependent fields of p and enqueues the call's launches on
// st, with ws (ws_bytes bytes, 256-byte aligned, at least cp.wl.total) as the
// workspace.  Tickets sit in the last cp.wl.cnt_bytes of the buffer; the
// one-launch kernel leaves every ticket it draws at zero, so the last
// kTicketBytes of a buffer are zero between calls, but a call whose ticket
// region is larger (very large batches) first clears the part beyond them,
// where an earlier call may have left partials.
static int enqueue_call(Params& p, const CallPlan& cp, long long B, long long L, unsigned char* ws, size_t ws_bytes,
                        cudaStream_t st) {
  const Plan& pl = cp.pl;
  p.B = static_cast<int>(B);
  p.L = static_cast<int>(L);
  p.gq = pl.gq;
  p.R = pl.R;
  p.HC = pl.HC;
  p.MT = pl.MT;
  p.n_hg = pl.n_hg;
  p.nwc = pl.nwc;
  p.nst = pl.nst;
  p.ring_off = pl.ring_off;
  p.head_bytes = pl.head_bytes;
  p.misc_off = pl.misc_off;
  p.misc_bytes = pl.misc_bytes;
  p.w_min = cp.w_min;
  const size_t cnt_off = (ws_bytes & ~static_cast<size_t>(255)) - cp.wl.cnt_bytes;
  p.err = reinterpret_cast<unsigned*>(ws);
  p.cnt = reinterpret_cast<int*>(ws + cnt_off);
  p.nseg = B * pl.n_hg;
  p.plse = reinterpret_cast<float*>(ws + cp.wl.lse_off);
  p.po = reinterpret_cast<float*>(ws + cp.wl.o_off);
  p.n_stream = static_cast<int>(cp.n_cta);
  if (cp.use_cs) {
    p.nwc = 2 * pl.MT;
    p.nst = cp.sp.nst;
    p.ring_off = cp.sp.ring_off;
    p.head_bytes = cp.sp.head_bytes;
    p.misc_off = cp.sp.misc_off;
    p.misc_bytes = cp.sp.misc_bytes;
  }
  cudaError_t e;
  if (!cp.fn_comb && cp.wl.cnt_bytes > static_cast<size_t>(kTicketBytes)) {
    e = cudaMemsetAsync(ws + cnt_off, 0, cp.wl.cnt_bytes - kTicketBytes, st);
    if (e != cudaSuccess) return fail("cudaMemsetAsync of the ticket region: %s", cudaGetErrorString(e));
  }
  void* args[] = {&p};
  e = cudaLaunchKernel(reinterpret_cast<const void*>(cp.fn), dim3(static_cast<unsigned>(cp.n_cta)), dim3(cp.threads),
                       args, cp.smem, st);
  if (e != cudaSuccess) return fail("kernel launch failed: %s", cudaGetErrorString(e));
  if (cp.fn_comb) {
    // the share floor and n_stream let the combine kernel find the pieces the
    // stream launch wrote
    e = cudaLaunchKernel(reinterpret_cast<const void*>(cp.fn_comb), dim3(static_cast<unsigned>(cp.n_comb)),
                         dim3(cmb::kThreads), args, combine_smem(cp.D), st);
    if (e != cudaSuccess) return fail("combine kernel launch failed: %s", cudaGetErrorString(e));
  }
  return 1;
}

// Plans the call, resolves the workspace (NULL: the library-owned per-device
// buffer) and enqueues the launches.
static int launch_with_plan(Params& p, long long B, long long h_q, long long h_kv, long long D, long long L, bool fp8,
                            void* workspace, size_t workspace_bytes, void* stream, long long mean_len) {
  CallPlan cp;
  if (!plan_call(B, h_q, h_kv, D, L, fp8, mean_len, cp)) return 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  size_t ws_bytes = workspace_bytes;
  if (!ws) {
    ws = static_cast<unsigned char*>(internal_workspace(cp.dev, cp.wl.total, st, &ws_bytes));
    if (!ws) return fail("cannot allocate a %zu-byte workspace", cp.wl.total);
  } else if (workspace_bytes < cp.wl.total) {
    return fail("workspace of %zu bytes is smaller than the %zu bytes needed", workspace_bytes, cp.wl.total);
  } else if (!aligned(ws, 256)) {
    return fail("workspace must be 256-byte aligned");
  }
  return enqueue_call(p, cp, B, L, ws, ws_bytes, st);
}

// The checks and the parameter block shared by the flat entry points (causal,
// tree, fused store, allocation-free); cm / mi select tree verify (both null:
// causal drafts), ocl the fused store.  Returns the static shapes the plan
// needs.
struct CallShape {
  long long B, h_q, h_kv, D, L, mean_len;
  bool fp8;
};

static int prepare_verify(const vsk_tensor* q, const vsk_tensor* ke, const vsk_tensor* ve, const vsk_tensor* o,
                          const vsk_tensor* kb, const vsk_tensor* vb, const vsk_tensor* qo, const vsk_tensor* kvp,
                          const vsk_tensor* kvi, int is_causal, int64_t max_len_extend, float k_scale, float v_scale,
                          float sm_scale, const vsk_tensor* cm, const vsk_tensor* mi, const vsk_tensor* ocl, Params& p,
                          CallShape& cs) {
  if (!gate(q, ke, ve, kb, vb, qo, kvp, kvi, is_causal, max_len_extend, -1, 0, 0.f, -1)) return 0;
  if (!check_3d(o, "o_extend")) return 0;
  if (o->dtype != VSK_DTYPE_BF16 || o->shape[0] != q->shape[0] || o->shape[1] != q->shape[1] ||
      o->shape[2] != ve->shape[2])
    return fail("o_extend must be bf16 [B*l_ext, h_q, v_head_dim]");
  if (!aligned(o->data, 4) || (o->stride[0] % 2) != 0 || (o->stride[1] % 2) != 0)
    return fail("o_extend must be 4-byte aligned with even strides");
  if (!std::isfinite(k_scale) || !std::isfinite(v_scale)) return fail("k_scale and v_scale must be finite");

  memset(&p, 0, sizeof p);
  p.q = static_cast<const __nv_bfloat16*>(q->data);
  p.q_s0 = q->stride[0];
  p.q_s1 = q->stride[1];
  p.ke = static_cast<const __nv_bfloat16*>(ke->data);
  p.ke_s0 = ke->stride[0];
  p.ke_s1 = ke->stride[1];
  p.ve = static_cast<const __nv_bfloat16*>(ve->data);
  p.ve_s0 = ve->stride[0];
  p.ve_s1 = ve->stride[1];
  p.o = static_cast<__nv_bfloat16*>(const_cast<void*>(o->data));
  p.o_s0 = o->stride[0];
  p.o_s1 = o->stride[1];
  p.kb = static_cast<const unsigned char*>(kb->data);
  const int ek = kb->dtype == VSK_DTYPE_FP8E4M3 ? 1 : 2;
  p.kb_s0 = kb->stride[0] * ek;
  p.kb_s1 = kb->stride[1] * ek;
  p.vb = static_cast<const unsigned char*>(vb->data);
  p.vb_s0 = vb->stride[0] * ek;
  p.vb_s1 = vb->stride[1] * ek;
  p.qo = static_cast<const int*>(qo->data);
  p.kvp = static_cast<const int*>(kvp->data);
  p.kvi = kvi->data;
  p.idx64 = kvi->dtype == VSK_DTYPE_I64;
  p.n_idx = kvi->shape[0];
  p.pool = kb->shape[0];
  p.n_rows = q->shape[0];
  const long long D = q->shape[2];
  const double sm = (sm_scale > 0.f && std::isfinite(sm_scale)) ? static_cast<double>(sm_scale)
                                                                 : 1.0 / std::sqrt(static_cast<double>(D));
  const double log2e = 1.4426950408889634;
  p.scale2 = static_cast<float>(sm * static_cast<double>(k_scale) * log2e);
  p.dscale2 = static_cast<float>(sm * log2e);
  p.dvs = 1.f;
  p.v_scale = v_scale;
  p.cmask = cm ? static_cast<const unsigned char*>(cm->data) : nullptr;
  p.mindptr = mi ? mi->data : nullptr;
  p.mindptr64 = (mi && mi->dtype == VSK_DTYPE_I64) ? 1 : 0;
  p.n_mask = cm ? cm->shape[0] : 0;
  if (p.cmask == nullptr) p.mindptr = nullptr;
  if (ocl) {
    if (!check_1d(ocl, "out_cache_loc")) return 0;
    if (ocl->dtype != VSK_DTYPE_I32 && ocl->dtype != VSK_DTYPE_I64) return fail("out_cache_loc must be int32 or int64");
    if (ocl->shape[0] != q->shape[0]) return fail("out_cache_loc must have one entry per q_extend row");
    if (!(k_scale > 0.f) || !(v_scale > 0.f)) return fail("storing into the cache needs k_scale > 0 and v_scale > 0");
    p.wmode = 1;
    p.ocl = ocl->data;
    p.ocl64 = ocl->dtype == VSK_DTYPE_I64;
    p.kw = static_cast<unsigned char*>(const_cast<void*>(kb->data));
    p.vw = static_cast<unsigned char*>(const_cast<void*>(vb->data));
    p.kq = k_scale;
    p.vq = v_scale;
  }
  cs.B = qo->shape[0] - 1;
  cs.h_q = q->shape[1];
  cs.h_kv = ke->shape[1];
  cs.D = D;
  cs.L = max_len_extend;
  cs.fp8 = kb->dtype == VSK_DTYPE_FP8E4M3;
  cs.mean_len = kvi->shape[0] / cs.B;
  return 1;
}

// Shared body of the workspace entry points.
static int run_verify(const vsk_tensor* q, const vsk_tensor* ke, const vsk_tensor* ve, const vsk_tensor* o,
                      const vsk_tensor* kb, const vsk_tensor* vb, const vsk_tensor* qo, const vsk_tensor* kvp,
                      const vsk_tensor* kvi, int is_causal, int64_t max_len_extend, float k_scale, float v_scale,
                      float sm_scale, void* workspace, size_t workspace_bytes, void* stream, const vsk_tensor* cm,
                      const vsk_tensor* mi, const vsk_tensor* ocl = nullptr) {
  Params p;
  CallShape cs;
  if (!prepare_verify(q, ke, ve, o, kb, vb, qo, kvp, kvi, is_causal, max_len_extend, k_scale, v_scale, sm_scale, cm,
                      mi, ocl, p, cs))
    return 0;
  return launch_with_plan(p, cs.B, cs.h_q, cs.h_kv, cs.D, cs.L, cs.fp8, workspace, workspace_bytes, stream,
                          cs.mean_len);
}

bool check_2d(const vsk_tensor* t, const char* name) {
  if (!t) return fail("%s is NULL", name);
  if (t->ndim != 2) return fail("%s must be 2-d (got ndim %d)", name, t->ndim);
  if (t->shape[0] < 0 || t->shape[1] < 0) return fail("%s has a negative extent", name);
  if (t->shape[0] > 0 && t->shape[1] > 1 && t->stride[1] != 1) return fail("%s: rows must be contiguous", name);
  if (t->shape[0] * t->shape[1] > 0 && !t->data) return fail("%s: NULL data", name);
  return true;
}

// Drafts already written to a paged cache (the unified verify of the
// "aiter_backend.py" page): sequence b's cache position t lives in pool row
// block_table[b][t / page_size] * page_size + t % page_size, its prefix is
// positions [0, seq_lens[b]) and its drafts [seq_lens[b], seq_lens[b] + L).
static int run_paged(const vsk_tensor* q, const vsk_tensor* o, const vsk_tensor* kc, const vsk_tensor* vc,
                     const vsk_tensor* bt, const vsk_tensor* sl, int64_t page_size, int64_t mle, float k_scale,
                     float v_scale, float sm_scale, void* workspace, size_t workspace_bytes, void* stream,
                     const vsk_tensor* k_new = nullptr, const vsk_tensor* v_new = nullptr) {
  if (!check_3d(q, "q") || !check_3d(o, "o") || !check_3d(kc, "k_cache") || !check_3d(vc, "v_cache")) return 0;
  if (!check_2d(bt, "block_table") || !check_1d(sl, "seq_lens")) return 0;
  if (page_size < 1) return fail("page_size must be >= 1");
  if (mle < 1) return fail("max_len_extend must be >= 1");
  const long long bs = sl->shape[0];
  if (bs < 1) return fail("batch size must be >= 1");
  if (bt->shape[0] != bs) return fail("block_table must have one row per sequence (B = %lld)", bs);
  if (bt->shape[1] < 1) return fail("block_table has no columns");
  if (bt->shape[1] * page_size > INT_MAX) return fail("block_table columns x page_size exceeds 2^31 - 1");
  if (bt->shape[1] * page_size < mle) return fail("block_table covers fewer than max_len_extend positions");
  if (bt->dtype != VSK_DTYPE_I32 || sl->dtype != VSK_DTYPE_I32) return fail("block_table and seq_lens must be int32");
  if (q->shape[0] != bs * mle)
    return fail("ragged extend: q has %lld rows, expected B*max_len_extend = %lld", q->shape[0], bs * mle);
  const long long h_q = q->shape[1], h_kv = kc->shape[1], D = q->shape[2];
  if (h_kv == 0 || h_q % h_kv != 0) return fail("h_q (%lld) is not a multiple of h_kv (%lld)", h_q, h_kv);
  if (vc->shape[1] != h_kv) return fail("KV head count mismatch between k_cache and v_cache");
  if (kc->shape[2] != D) return fail("head_dim mismatch between q and k_cache");
  if (vc->shape[2] != D) return fail("v_head_dim (%lld) != head_dim (%lld) is not built", vc->shape[2], D);
  if (D != 64 && D != 128 && D != 256) return fail("head_dim %lld not in {64, 128, 256}", D);
  if (kc->shape[0] != vc->shape[0]) return fail("k_cache and v_cache pools differ in size");
  if (kc->shape[0] % page_size != 0) return fail("cache rows (%lld) are not a whole number of pages", kc->shape[0]);
  if (q->dtype != VSK_DTYPE_BF16) return fail("q must be bf16");
  if (kc->dtype != vc->dtype || (kc->dtype != VSK_DTYPE_BF16 && kc->dtype != VSK_DTYPE_FP8E4M3))
    return fail("k_cache and v_cache must both be bf16 or both fp8 e4m3");
  const long long R = (h_q / h_kv) * mle;
  const long long maxR = D > 128 ? 64 : 128;
  if (R > maxR) return fail("(h_q/h_kv)*max_len_extend = %lld exceeds %lld", R, maxR);
  const size_t ek = kc->dtype == VSK_DTYPE_BF16 ? 2 : 1;
  for (const vsk_tensor* t : {kc, vc}) {
    if (!aligned(t->data, 16) || (t->stride[0] * ek) % 16 != 0 || (t->stride[1] * ek) % 16 != 0)
      return fail("K/V cache rows must be 16-byte aligned");
  }
  if (o->dtype != VSK_DTYPE_BF16 || o->shape[0] != q->shape[0] || o->shape[1] != h_q || o->shape[2] != D)
    return fail("o must be bf16 [B*l_ext, h_q, head_dim]");
  for (const vsk_tensor* t : {q, o}) {
    if (!aligned(t->data, 4) || (t->stride[0] % 2) != 0 || (t->stride[1] % 2) != 0)
      return fail("q and o must be 4-byte aligned with even strides");
  }
  if (!aligned(bt->data, 4) || !aligned(sl->data, 4)) return fail("block_table and seq_lens must be 4-byte aligned");
  if (!std::isfinite(k_scale) || !std::isfinite(v_scale)) return fail("k_scale and v_scale must be finite");

  Params p;
  memset(&p, 0, sizeof p);
  p.q = static_cast<const __nv_bfloat16*>(q->data);
  p.q_s0 = q->stride[0];
  p.q_s1 = q->stride[1];
  p.o = static_cast<__nv_bfloat16*>(const_cast<void*>(o->data));
  p.o_s0 = o->stride[0];
  p.o_s1 = o->stride[1];
  p.kb = static_cast<const unsigned char*>(kc->data);
  p.kb_s0 = kc->stride[0] * static_cast<long long>(ek);
  p.kb_s1 = kc->stride[1] * static_cast<long long>(ek);
  p.vb = static_cast<const unsigned char*>(vc->data);
  p.vb_s0 = vc->stride[0] * static_cast<long long>(ek);
  p.vb_s1 = vc->stride[1] * static_cast<long long>(ek);
  p.pool = kc->shape[0];
  p.n_rows = q->shape[0];
  p.paged = 1;
  p.bt = static_cast<const int*>(bt->data);
  p.bt_s0 = bt->stride[0];
  p.bt_cols = static_cast<int>(bt->shape[1]);
  p.page = static_cast<int>(page_size);
  {
    int l = 0;
    while ((1LL << l) < page_size) ++l;
    p.pg_l = l;
    p.pg_m = static_cast<unsigned>(((1ULL << (32 + l)) + static_cast<unsigned long long>(page_size) - 1) /
                                       static_cast<unsigned long long>(page_size) -
                                   (1ULL << 32));
  }
  p.slens = static_cast<const int*>(sl->data);
  const double sm = (sm_scale > 0.f && std::isfinite(sm_scale)) ? static_cast<double>(sm_scale)
                                                                 : 1.0 / std::sqrt(static_cast<double>(D));
  const double log2e = 1.4426950408889634;
  // every cached key, drafts included, carries the cache's scales
  p.scale2 = static_cast<float>(sm * static_cast<double>(k_scale) * log2e);
  p.dscale2 = p.scale2;
  p.dvs = v_scale;
  p.v_scale = v_scale;
  if (k_new || v_new) {
    if (!check_3d(k_new, "k_new") || !check_3d(v_new, "v_new")) return 0;
    if (k_new->dtype != VSK_DTYPE_BF16 || v_new->dtype != VSK_DTYPE_BF16) return fail("k_new and v_new must be bf16");
    if (k_new->shape[0] != q->shape[0] || v_new->shape[0] != q->shape[0] || k_new->shape[1] != h_kv ||
        v_new->shape[1] != h_kv || k_new->shape[2] != D || v_new->shape[2] != D)
      return fail("k_new / v_new must be [B*l_ext, h_kv, head_dim]");
    for (const vsk_tensor* t : {k_new, v_new}) {
      if (!aligned(t->data, 4) || (t->stride[0] % 2) != 0 || (t->stride[1] % 2) != 0)
        return fail("k_new and v_new must be 4-byte aligned with even strides");
    }
    if (!(k_scale > 0.f) || !(v_scale > 0.f)) return fail("storing into the cache needs k_scale > 0 and v_scale > 0");
    p.ke = static_cast<const __nv_bfloat16*>(k_new->data);
    p.ke_s0 = k_new->stride[0];
    p.ke_s1 = k_new->stride[1];
    p.ve = static_cast<const __nv_bfloat16*>(v_new->data);
    p.ve_s0 = v_new->stride[0];
    p.ve_s1 = v_new->stride[1];
    p.wmode = 2;
    p.kw = static_cast<unsigned char*>(const_cast<void*>(kc->data));
    p.vw = static_cast<unsigned char*>(const_cast<void*>(vc->data));
    p.kq = k_scale;
    p.vq = v_scale;
  }
  // the block table bounds every sequence's length: its capacity stands in for the mean
  return launch_with_plan(p, bs, h_q, h_kv, D, mle, kc->dtype == VSK_DTYPE_FP8E4M3, workspace, workspace_bytes,
                          stream, bt->shape[1] * page_size);
}
}  // namespace vsk

extern "C" {

int verify_splitkv_paged_fwd(const vsk_tensor* q, const vsk_tensor* o, const vsk_tensor* k_cache,
                             const vsk_tensor* v_cache, const vsk_tensor* block_table, const vsk_tensor* seq_lens,
                             int64_t page_size, int64_t max_len_extend, float k_scale, float v_scale, float sm_scale,
                             void* workspace, size_t workspace_bytes, void* stream) {
  g_err.clear();
  return run_paged(q, o, k_cache, v_cache, block_table, seq_lens, page_size, max_len_extend, k_scale, v_scale,
                   sm_scale, workspace, workspace_bytes, stream);
}

int verify_splitkv_paged_write_fwd(const vsk_tensor* q, const vsk_tensor* k_new, const vsk_tensor* v_new,
                                   const vsk_tensor* o, const vsk_tensor* k_cache, const vsk_tensor* v_cache,
                                   const vsk_tensor* block_table, const vsk_tensor* seq_lens, int64_t page_size,
                                   int64_t max_len_extend, float k_scale, float v_scale, float sm_scale,
                                   void* workspace, size_t workspace_bytes, void* stream) {
  g_err.clear();
  if (!k_new || !v_new) return fail("k_new and v_new are required");
  return run_paged(q, o, k_cache, v_cache, block_table, seq_lens, page_size, max_len_extend, k_scale, v_scale,
                   sm_scale, workspace, workspace_bytes, stream, k_new, v_new);
}

int verify_splitkv_write_fwd(const vsk_tensor* q, const vsk_tensor* ke, const vsk_tensor* ve, const vsk_tensor* o,
                             const vsk_tensor* kb, const vsk_tensor* vb, const vsk_tensor* qo, const vsk_tensor* kvp,
                             const vsk_tensor* kvi, const vsk_tensor* out_cache_loc, int64_t max_len_extend,
                             float k_scale, float v_scale, float sm_scale, void* workspace, size_t workspace_bytes,
                             void* stream) {
  g_err.clear();
  if (!out_cache_loc) return fail("out_cache_loc is NULL");
  return run_verify(q, ke, ve, o, kb, vb, qo, kvp, kvi, 1, max_len_extend, k_scale, v_scale, sm_scale, workspace,
                    workspace_bytes, stream, nullptr, nullptr, out_cache_loc);
}

int verify_splitkv_fwd(const vsk_tensor* q, const vsk_tensor* ke, const vsk_tensor* ve, const vsk_tensor* o,
                       const vsk_tensor* kb, const vsk_tensor* vb, const vsk_tensor* qo, const vsk_tensor* kvp,
                       const vsk_tensor* kvi, int is_causal, int64_t max_len_extend, float k_scale, float v_scale,
                       float sm_scale, void* workspace, size_t workspace_bytes, void* stream) {
  g_err.clear();
  return run_verify(q, ke, ve, o, kb, vb, qo, kvp, kvi, is_causal, max_len_extend, k_scale, v_scale, sm_scale,
                    workspace, workspace_bytes, stream, nullptr, nullptr);
}

int verify_splitkv_tree_fwd(const vsk_tensor* q, const vsk_tensor* ke, const vsk_tensor* ve, const vsk_tensor* o,
                            const vsk_tensor* kb, const vsk_tensor* vb, const vsk_tensor* qo, const vsk_tensor* kvp,
                            const vsk_tensor* kvi, const vsk_tensor* custom_mask, const vsk_tensor* mask_indptr,
                            int64_t max_len_extend, float k_scale, float v_scale, float sm_scale, void* workspace,
                            size_t workspace_bytes, void* stream) {
  g_err.clear();
  if (!check_1d(custom_mask, "custom_mask") || !check_1d(mask_indptr, "mask_indptr")) return 0;
  if (custom_mask->dtype != VSK_DTYPE_U8) return fail("custom_mask must be uint8 (or bool)");
  if (mask_indptr->dtype != VSK_DTYPE_I32 && mask_indptr->dtype != VSK_DTYPE_I64)
    return fail("mask_indptr must be int32 or int64");
  if (!qo || mask_indptr->shape[0] != qo->shape[0]) return fail("mask_indptr must have B+1 entries");
  return run_verify(q, ke, ve, o, kb, vb, qo, kvp, kvi, 1, max_len_extend, k_scale, v_scale, sm_scale, workspace,
                    workspace_bytes, stream, custom_mask, mask_indptr);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free entry point.
//
// Some callers cannot call cudaMalloc at all: engines that hand every free
// byte of HBM to their own pool allocator at start-up and forbid stray device
// allocations (a cudaMalloc there can fail, fragment the pool, or stall every
// stream while the driver maps memory), and plugin hosts whose interface
// passes only input and output pointers with no workspace.  For them the
// scratch this kernel needs (one ticket per segment, the error word and the
// per-CTA log-sum-exp partials) lives in the array below, which the driver
// creates when the library's module is loaded on a GPU and keeps until the
// process exits.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_vsk_static_scratch[VSK_NOALLOC_SCRATCH_BYTES];

namespace vsk {

std::mutex g_static_mu;
std::vector<void*> g_static_addr;  // per device: device address of g_vsk_static_scratch

// Device address of the scratch array on device dev, which must be the
// current device.  The host-side name is only a stand-in, so the address is
// asked from the runtime once per device and cached.
void* static_scratch(int dev) {
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (static_cast<int>(g_static_addr.size()) <= dev) g_static_addr.resize(dev + 1, nullptr);
  if (!g_static_addr[dev]) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_vsk_static_scratch);
    if (e != cudaSuccess) {
      fail("cudaGetSymbolAddress of the built-in scratch failed: %s", cudaGetErrorString(e));
      return nullptr;
    }
    g_static_addr[dev] = ptr;
  }
  return g_static_addr[dev];
}

}  // namespace vsk

extern "C" int verify_splitkv_fwd_noalloc(const vsk_tensor* q, const vsk_tensor* ke, const vsk_tensor* ve,
                                          const vsk_tensor* o, const vsk_tensor* kb, const vsk_tensor* vb,
                                          const vsk_tensor* qo, const vsk_tensor* kvp, const vsk_tensor* kvi,
                                          int is_causal, int64_t max_len_extend, float k_scale, float v_scale,
                                          float sm_scale, void* stream) {
  g_err.clear();
  Params p;
  CallShape cs;
  if (!prepare_verify(q, ke, ve, o, kb, vb, qo, kvp, kvi, is_causal, max_len_extend, k_scale, v_scale, sm_scale,
                      nullptr, nullptr, nullptr, p, cs))
    return 0;
  // the same plan (form, grid, workspace layout) verify_splitkv_fwd would use
  CallPlan cp;
  if (!plan_call(cs.B, cs.h_q, cs.h_kv, cs.D, cs.L, cs.fp8, cs.mean_len, cp)) return 0;
  if (cp.wl.total > static_cast<size_t>(VSK_NOALLOC_SCRATCH_BYTES))
    return fail("this problem needs %zu bytes of scratch, more than the %d bytes built into the library for "
                "verify_splitkv_fwd_noalloc; use verify_splitkv_fwd with a caller workspace",
                cp.wl.total, VSK_NOALLOC_SCRATCH_BYTES);
  unsigned char* scratch = static_cast<unsigned char*>(static_scratch(cp.dev));
  if (!scratch) return 0;
  // The array keeps whatever the previous call left: zero the error word and
  // this call's whole ticket span (at the end of the array) before its
  // kernels run.
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(scratch, 0, 256, st);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(scratch + VSK_NOALLOC_SCRATCH_BYTES - cp.wl.cnt_bytes, 0, cp.wl.cnt_bytes, st);
  if (e != cudaSuccess) return fail("cudaMemsetAsync on the built-in scratch: %s", cudaGetErrorString(e));
  return enqueue_call(p, cp, cs.B, cs.L, scratch, VSK_NOALLOC_SCRATCH_BYTES, st);
}
