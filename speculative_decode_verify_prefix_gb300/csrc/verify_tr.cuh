// Tensor-memory form of the prefix stream for head_dim 256 with the packed
// query rows on the M side of both products (tcgen05, sm_103a).
//
// Same operation, work split and partial format as vtc_kernel (the
// "verify_splitkv.py" page, "_verify_prefix_stage1": per-split partial
// softmaxes over the gathered prefix, qk *= sm_scale * k_scale, acc *=
// v_scale); vsk_combine_kernel folds the partials, adds the draft block and
// writes the output in a second launch.  vtc_kernel puts the keys on M, so
// every tcgen05.mma there has N = 16-32 (the packed rows) and costs about as
// much as a far larger one.  Here the rows are M and the products are
//   S[64][64 keys]  = Qs[64][256] x K_tile^T     (M = 64, N = 64, TMEM)
//   O[64][256 dv]  += P[64][64 keys] x V_tile    (M = 64, N = 256, TMEM)
// which takes 8 + 4 instructions per 64-key tile for an e4m3 pool (vtc_kernel:
// 16 + 8).
//
// Rows of Qs.  An M = 64 accumulator lives in lanes 0-15 of each TMEM
// sub-partition (row 16 w + i in lane 32 w + i).  Row 16 w + j of Qs (j < 8)
// holds packed query row 8 w + j and row 16 w + 8 + j its second term: for an
// e4m3 pool each query splits exactly into two e4m3 terms (q 2^sh = hi + lo,
// the largest |q| 2^sh in [128, 256)), so both terms of a score come out of
// one kind::f8f6f4 MMA straight from the e4m3 K rows, in lanes j and j + 8 of
// sub-partition w; for a bf16 pool the second-term rows are zero.  P holds
// packed row 8 w + j in row 16 w + j (rows 16 w + 8 .. 16 w + 15 stay zero),
// so O's row of packed row 8 w + j is lane j of sub-partition w.
//
// Roles (16 warps of 128 registers, one CTA per SM):
//   warps 0-3   softmax: warp w reads sub-partition w in the 16-lane fragment
//               shape (tcgen05.ld 16x256b), which hands each thread lanes g
//               and g + 8, i.e. both terms of packed row 8 w + g, for 16 of
//               the tile's keys; the four threads of a quad share the row.
//               Online softmax in the log2 domain with a running maximum
//               raised only when a score exceeds it by more than 2^8 (O is
//               then rescaled in TMEM); P (f16 for e4m3 pools, bf16
//               otherwise) into shared memory; the partial at a piece's end.
//               They also load each piece's queries.
//   warps 4-7   e4m3 pools: widen each V tile exactly to f16 (PV's B operand);
//               bf16 pools: loaders.
//   warp 8      TMEM allocation; lane 0 issues every MMA.
//   warps 9-15  loaders (with 4-7 for bf16 pools): kv_indices / page ids,
//               16-byte cp.async gathers of the K and V rows into a ring
//               (e4m3: one slot per 64-key tile, K rows then V rows; bf16:
//               alternating K and V entries, a V entry being read in place by
//               PV), completion by cp.async.mbarrier.arrive.noinc; each warp
//               publishes its keys' validity in a tagged 8-byte word.
// Operands in shared memory use the 128-byte swizzled canonical layouts:
//   Qs (A), K tile (B)   K-major   [128-byte column block][row][128 B]
//   P (A)                K-major   [row][128 B] (64 keys of 16 bits)
//   V tile (B)           MN-major  [64-dv block][key][128 B]
// Every mbarrier wait is bounded (one second); a wait that gives up sets the
// CTA's abort flag and error bit 8, and the CTA drains, frees TMEM and exits.
// Each role keeps a small code footprint (loops rolled, one copy of the
// loader's tile code): four roles share every SM sub-partition's instruction
// cache, and fetch stalls bounded an earlier version.
#pragma once
#include "verify_kernel.cuh"

namespace vsk {
namespace tr {

constexpr int KT = 64;                     // keys per tile (N of S)
constexpr int kSmThreads = 128;            // softmax warps 0-3
constexpr int kWarpCvt0 = 4;               // widening warps 4-7 (e4m3 pools; loaders for bf16 pools)
constexpr int kWarpMma = 8;
constexpr int kThreads = 16 * 32;
// loader warps: 9-15 for e4m3 pools; 4-7 and 9-15 for bf16 pools (no widening)
template <bool FP8>
__host__ __device__ constexpr int nl() { return FP8 ? 7 : 11; }
template <bool FP8>
__device__ __forceinline__ int loader_index(int warp) {  // -1: not a loader
  return warp >= 9 ? warp - (FP8 ? 9 : 5) : (!FP8 && warp >= 4 && warp < 8 ? warp - 4 : -1);
}
// The ring: for e4m3 pools tile slots (K rows, then V rows of a 64-key tile,
// freed once QK is done and V widened); for bf16 pools separate K and V
// entries (a V entry stays until PV has read it in place), alternating.
constexpr int kMaxNE = 10;                 // ring slots (e4m3) or entries (bf16) at most
constexpr float kThr = 8.f;                // log2 headroom before the running maximum is raised
constexpr int NCS = 1;                     // accumulation chains of S
constexpr int kColO = 2 * NCS * KT;        // TMEM column of O; S buffer b, chain c at (b NCS + c) KT
constexpr int kCols = 512;
static_assert(kColO + 256 <= kCols, "TMEM columns");
// shared-memory map ([0, 256) is cta_share's)
constexpr int kBarOff = 256;
constexpr int kTmemOff = 640;
constexpr int kAbortOff = 644;
constexpr int kRedOff = 1024;              // per-warp largest |q| bits
constexpr int kMaskOff = 2048;             // [kMaskRing][kMaskWords] valid-key words: tile + 1 (high half), key bits (low)
constexpr int kMaskWords = 11;             // one per loader warp (at most 11)
constexpr int kMaskRing = 8;               // > the tiles the loaders can run ahead of the softmax
constexpr int kDataOff = 3072;
constexpr int kBFull = 0, kBEmpty = kMaxNE, kBSFull = 2 * kMaxNE, kBSEmpty = kBSFull + 2, kBPFull = kBSEmpty + 2,
              kBPEmpty = kBPFull + 2, kBV16Full = kBPEmpty + 2, kBV16Empty = kBV16Full + 2, kBQFull = kBV16Empty + 2,
              kNumBars = kBQFull + 1;
static_assert(kBarOff + 8 * kNumBars <= kTmemOff, "barriers overlap");
static_assert(kMaskOff + kMaskRing * kMaskWords * 8 <= kDataOff, "masks overlap");
static_assert(kMaxNE / 2 + 3 <= kMaskRing, "mask ring too short (bf16 entries; e4m3 slots are capped on the host)");

template <bool FP8>
struct Geo {
  static constexpr int D = 256;
  static constexpr int ROWB = D * (FP8 ? 1 : 2);  // one K (or V) row of one head
  static constexpr int CPR = ROWB / 16;           // its 16-byte chunks
  static constexpr int ENT = KT * ROWB;           // K (or V) rows of a tile
  static constexpr int TILEB = 2 * ENT;           // one e4m3 ring slot: K rows, then V rows
  static constexpr int RING_UNIT = FP8 ? TILEB : ENT;  // bytes per ring slot (e4m3) or entry (bf16)
  static constexpr int QB = 64 * ROWB;            // Qs
  static constexpr int PB = 64 * 128;             // one P buffer
  static constexpr int V16B = FP8 ? 4 * KT * 128 : 0;  // one widened V tile
  static constexpr int q_off = kDataOff;
  static constexpr int p_off = q_off + QB;
  static constexpr int v16_off = p_off + 2 * PB;
  static constexpr int ring_off = v16_off + 2 * V16B;
};

// Position in the ring: slot and lap.
struct RingPos {
  int slot;
  uint32_t lap;
  __device__ __forceinline__ void step(int n, int by = 1) {
    slot += by;
    if (slot >= n) {
      slot -= n;
      ++lap;
    }
  }
};

// Bounded mbarrier waits (as tc::mbar_wait) with a non-blocking test first:
// a phase that has already completed costs one test.
__device__ __forceinline__ bool test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, unsigned* err) {
  return test(bar, parity) || tc::mbar_wait(bar, parity, abort_flag, err);
}
__device__ __forceinline__ void wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag, unsigned* err) {
  if ((threadIdx.x & 31) == 0) wait(bar, parity, abort_flag, err);
  __syncwarp();
}

// TMEM <-> registers in the 16-lane fragment shape, 64 columns: thread t gets
// lanes t / 4 and t / 4 + 8 of the warp's sub-partition, columns 8 i + 2 (t %
// 4) and + 1 of group i: v[4 i], v[4 i + 1] (lane t / 4), v[4 i + 2], v[4 i +
// 3] (lane t / 4 + 8).
__device__ __forceinline__ void ld16x256b_x8(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void st16x256b_x8(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x256b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

// Valid keys of tile u (bit k = key k): every lane reads the loader warps'
// words (tag u + 1 in the high half, the warp's key bits in the low half),
// waiting (one second at most) until all carry the tag.
template <int NL>
__device__ __forceinline__ unsigned long long tile_mask(const volatile unsigned long long* maskq, long long u,
                                                        volatile int* abort_flag, unsigned* err) {
  const uint32_t want = static_cast<uint32_t>(u + 1);
  const volatile unsigned long long* mq = maskq + (u % kMaskRing) * kMaskWords;
  unsigned long long w[NL];
  auto read = [&]() {
    bool ok = true;
#pragma unroll
    for (int i = 0; i < NL; ++i) {
      w[i] = mq[i];
      ok &= static_cast<uint32_t>(w[i] >> 32) == want;
    }
    return ok;
  };
  bool ok = read();
  if (!__all_sync(0xffffffffu, ok)) {
    const unsigned long long t0 = tc::global_ns();
    do {
      __nanosleep(32);
      ok = read();
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      if (tc::global_ns() - t0 > 1000000000ull) {
        if ((threadIdx.x & 31) == 0) {
          *abort_flag = 1;
          atomicOr(err, kErrTimeout);
        }
        break;
      }
    } while (!__all_sync(0xffffffffu, ok));
  }
  unsigned long long m = 0;
#pragma unroll
  for (int i = 0; i < NL; ++i) m |= (w[i] & 0xFFFFFFFFull) << (KT * i / NL);
  return m;
}

}  // namespace tr

// The piece's packed query rows (row r = draft r / gq, query head kvh gq +
// r % gq; rows >= R zero) into Qs, by the 128 softmax threads (tw = 0..127).
// Returns the score scale into the log2 domain (sm_scale k_scale log2 e, for
// an e4m3 pool times 2^-sh).
template <bool FP8>
__device__ __forceinline__ float tr_load_q(const Params& p, const Seg& s, unsigned char* qs, unsigned* red_u,
                                           int tw) {
  const int a = p.qo ? __ldg(p.qo + s.b) : s.b * p.L, e = p.qo ? __ldg(p.qo + s.b + 1) : (s.b + 1) * p.L;
  const bool ok = a >= 0 && e - a == p.L && static_cast<long long>(a) + p.L <= p.n_rows;
  if (!ok && tw == 0) atomicOr(p.err, kErrBadQoIndptr);
  const int s_b = ok ? a : s.b * p.L;
  const int kvh = s.hg;
  constexpr int CH = 32;             // 8-element chunks of a 256-wide row
  constexpr int NCH = 32 * CH / 128;  // chunks per thread (32 packed rows)
  uint32_t v[NCH][4];
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    const int ci = tw + 128 * i;
    const int r = ci / CH, c = ci % CH;
    if (r < p.R) {
      const __nv_bfloat16* src = p.q + (static_cast<long long>(s_b) + r / p.gq) * p.q_s0 +
                                 static_cast<long long>(kvh * p.gq + r % p.gq) * p.q_s1 + c * 8;
#pragma unroll
      for (int w = 0; w < 4; ++w) v[i][w] = ld_u32(src + 2 * w);
    } else {
      v[i][0] = v[i][1] = v[i][2] = v[i][3] = 0u;
    }
  }
  if constexpr (!FP8) {
    // bf16 rows: 512 bytes, four 128-byte column blocks; chunk c = bytes 16c
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
      const int ci = tw + 128 * i;
      const int r = ci / CH, c = ci % CH;
      const int ar = 16 * (r >> 3) + (r & 7);
      *reinterpret_cast<uint4*>(qs + (c >> 3) * (64 * 128) + ar * 128 + (((c & 7) ^ (ar & 7)) << 4)) =
          make_uint4(v[i][0], v[i][1], v[i][2], v[i][3]);
    }
    return p.scale2;
  } else {
    // largest |q| of the piece's rows (bf16 bit patterns order like magnitudes)
    unsigned mx = 0;
#pragma unroll
    for (int i = 0; i < NCH; ++i)
#pragma unroll
      for (int w = 0; w < 4; ++w) mx = max(mx, max(v[i][w] & 0x7FFFu, (v[i][w] >> 16) & 0x7FFFu));
    mx = __reduce_max_sync(0xffffffffu, mx);
    if ((tw & 31) == 0) red_u[tw >> 5] = mx;
    named_bar_sync(1, tr::kSmThreads);
    mx = max(max(red_u[0], red_u[1]), max(red_u[2], red_u[3]));
    named_bar_sync(1, tr::kSmThreads);  // red_u is free again
    const int ex = static_cast<int>(mx >> 7) - 127;
    int sh = mx == 0 ? 0 : 7 - ex;  // the largest |q| 2^sh lies in [128, 256)
    sh = max(-120, min(120, sh));
    const float up = __int_as_float((127 + sh) << 23);
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
      const int ci = tw + 128 * i;
      const int r = ci / CH, c = ci % CH;
      uint32_t hw[2], lw[2];
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float2 f = unpack_bf16(v[i][w]);
        const float x0 = f.x * up, x1 = f.y * up;
        const unsigned short h = __nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3);
        const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(h), __NV_E4M3);
        const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hr));
        const unsigned short l =
            __nv_cvt_float2_to_fp8x2(make_float2(x0 - hf.x, x1 - hf.y), __NV_SATFINITE, __NV_E4M3);
        if (w & 1) {
          hw[w >> 1] |= static_cast<uint32_t>(h) << 16;
          lw[w >> 1] |= static_cast<uint32_t>(l) << 16;
        } else {
          hw[w >> 1] = h;
          lw[w >> 1] = l;
        }
      }
      // e4m3 rows: 256 bytes, two 128-byte column blocks; elements d = 8c ..
      // 8c + 7 sit in 16-byte chunk (d % 128) / 16 at byte d % 16
      const int d = 8 * c;
      const int ah = 16 * (r >> 3) + (r & 7), al = ah + 8;
      const int base = (d >> 7) * (64 * 128) + (d & 15);
      const int ck = (d & 127) >> 4;
      *reinterpret_cast<uint2*>(qs + base + ah * 128 + ((ck ^ (ah & 7)) << 4)) = make_uint2(hw[0], hw[1]);
      *reinterpret_cast<uint2*>(qs + base + al * 128 + ((ck ^ (al & 7)) << 4)) = make_uint2(lw[0], lw[1]);
    }
    return p.scale2 * __int_as_float((127 - sh) << 23);
  }
}

template <bool FP8, int RM>
__global__ void __launch_bounds__(tr::kThreads, 1) vtr_kernel(const __grid_constant__ Params p) {
  using namespace tc;
  using tr::KT;
  using G = tr::Geo<FP8>;
  constexpr int D = 256;
  constexpr int NL = tr::nl<FP8>();
  constexpr int ENT = G::ENT;
  extern __shared__ __align__(1024) unsigned char smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NE = p.nst;  // ring slots (e4m3) or entries (bf16)
  // the combine kernel, when launched as a programmatic dependent, may start
  // its CTAs now (its griddepcontrol.wait still waits for this whole grid)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  long long start, end, W;
  Seg seg0;
  if (!cta_share(p, smem, start, end, W, seg0)) return;  // uniform: no work
  // The 128-byte swizzled layouts need a 1024-byte aligned base (dynamic
  // shared memory of a kernel without static shared memory starts there; were
  // it not so, the CTA reports the pipeline error bit and writes nothing).
  if ((smem_u32(smem) & 1023u) != 0u) {
    if (tid == 0) atomicOr(p.err, kErrTimeout);
    return;
  }

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + tr::kBarOff);
  auto bar = [&](int i) -> uint32_t { return smem_u32(bars + i); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + tr::kAbortOff);
  volatile unsigned long long* maskq = reinterpret_cast<volatile unsigned long long*>(smem + tr::kMaskOff);
  const uint32_t q_s = smem_u32(smem + G::q_off);
  const uint32_t p_s = smem_u32(smem + G::p_off);
  const uint32_t v16_s = smem_u32(smem + G::v16_off);
  const uint32_t ring_s = smem_u32(smem + G::ring_off);

  if (tid == 0) {
    *abort_flag = 0;
    for (int i = 0; i < NE; ++i) {
      mbar_init(bar(tr::kBFull + i), NL * 32);  // every loader lane copies part of each slot / entry
      // e4m3: released by the QK products' commit and the four widening
      // warps; bf16: by the commit of the products that read the entry
      mbar_init(bar(tr::kBEmpty + i), FP8 ? 1 + 4 : 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(tr::kBSFull + b), 1);
      mbar_init(bar(tr::kBSEmpty + b), 4);
      mbar_init(bar(tr::kBPFull + b), 4);
      mbar_init(bar(tr::kBPEmpty + b), 1);
      mbar_init(bar(tr::kBV16Full + b), 4);
      mbar_init(bar(tr::kBV16Empty + b), 1);
    }
    mbar_init(bar(tr::kBQFull), 4);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // Qs and both P buffers start zero: the rows no thread writes (second-term
  // rows of a bf16 pool, P rows 16 w + 8 .. 16 w + 15) stay zero
  for (int i = tid; i < (G::QB + 2 * G::PB) / 16; i += tr::kThreads)
    *reinterpret_cast<uint4*>(smem + G::q_off + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
  if (tid < tr::kMaskRing * tr::kMaskWords) maskq[tid] = 0ull;  // tag 0: no tile
  fence_proxy_async();
  if (warp == tr::kWarpMma) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem + tr::kTmemOff)),
                 "r"(tr::kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + tr::kTmemOff);

  if (tr::loader_index<FP8>(warp) >= 0) {
    // ================================ loaders ================================
    const int lw = tr::loader_index<FP8>(warp);
    const uint64_t pol = policy_evict_first();
    constexpr int CPR = G::CPR;     // 16-byte chunks of a row: 16 (e4m3) or 32 (bf16)
    constexpr int CPL = 4;          // chunks per lane per row (64-byte runs per instruction)
    constexpr int LPT = CPR / CPL;  // lanes per row
    constexpr int TSTEP = 32 / LPT;  // rows per pass
    constexpr int TPW = (KT + NL - 1) / NL;  // tokens of a tile per loader warp, at most
    const int tlo = KT * lw / NL, cnt = KT * (lw + 1) / NL - tlo;  // this warp's tokens of a tile
    tr::RingPos pos{0, 0u};
    uint32_t tile = 0;  // tiles issued
    // one tile: its ring slot (K rows, then V rows) from the pool rows of
    // this warp's cnt tokens (lane j < cnt holds token tlo + j's row)
    auto load_tile = [&](const TileIt& it, long long raw) {
      const int t = it.tok + tlo + lane;
      const long long loc = tile_loc(p, it, tlo + lane, raw);
      const bool ok = lane < cnt && t < it.te && loc >= 0 && loc < p.pool;
      if (lane < cnt && t < it.te && !ok) atomicOr(p.err, kErrBadIndex);
      const unsigned m = __ballot_sync(0xffffffffu, ok);
      const long long head = it.s.hg;
      const unsigned char* kbase = p.kb + head * p.kb_s1;
      const unsigned char* vbase = p.vb + head * p.vb_s1;
#pragma unroll 1
      for (int kv = 0; kv < (FP8 ? 1 : 2); ++kv) {
        // e4m3: one slot for K and V; bf16: the K entry, then the V entry
        const int slot = pos.slot;
        tr::wait_warp(bar(tr::kBEmpty + slot), (pos.lap & 1u) ^ 1u, abort_flag, p.err);
        if (kv == 0 && lane == 0)
          // this warp's valid keys of the tile (token tlo + j: bit j), tagged
          maskq[(tile % tr::kMaskRing) * tr::kMaskWords + lw] = (static_cast<unsigned long long>(tile + 1) << 32) | m;
        const uint32_t d0 = ring_s + static_cast<uint32_t>(slot) * G::RING_UNIT;
#pragma unroll 1
        for (int i = 0; i < (TPW + TSTEP - 1) / TSTEP; ++i) {
          const int tl = i * TSTEP + lane / LPT;  // token among this warp's cnt
          const long long lc = __shfl_sync(0xffffffffu, loc, tl & 31);
          if (tl < cnt) {
            const bool v = (m >> tl) & 1u;
            const int tt = tlo + tl;  // token within the tile
            const unsigned char* q0 = reinterpret_cast<const unsigned char*>(p.q);
            const unsigned char* sk = v ? (kv ? vbase + lc * p.vb_s0 : kbase + lc * p.kb_s0) : q0;
            const unsigned char* sv = v && FP8 ? vbase + lc * p.vb_s0 : q0;
#pragma unroll
            for (int cj = 0; cj < CPL; ++cj) {
              const int c = lane % LPT + LPT * cj;
              const uint32_t d = (c >> 3) * (KT * 128) + tt * 128 + (((c & 7) ^ (tt & 7)) << 4);
              cp_async_16_zfill(d0 + d, v ? sk + c * 16 : sk, v, pol);
              if constexpr (FP8) cp_async_16_zfill(d0 + ENT + d, v ? sv + c * 16 : sv, v, pol);
            }
          }
        }
        cp_async_arrive_noinc(bar(tr::kBFull + slot));
        pos.step(NE);
      }
      ++tile;
    };
    // pool rows are read four tiles before their tile is copied, rotating
    // through registers (one copy of the tile code: a small instruction
    // footprint beside the other roles)
    TileIt cur;
    cur.s = seg0;
    cur.tok = static_cast<int>(start - seg0.off);
    cur.te = piece_real_end(seg0, end);
    tile_settle(p, cur, end);
    TileIt ahead = cur;
    const int jl = lane < cnt ? tlo + lane : KT;
    long long r0 = tile_raw(p, ahead, jl);
    tile_next(p, ahead, end);
    long long r1 = tile_raw(p, ahead, jl);
    tile_next(p, ahead, end);
    long long r2 = tile_raw(p, ahead, jl);
    tile_next(p, ahead, end);
    long long r3 = tile_raw(p, ahead, jl);
    tile_next(p, ahead, end);
#pragma unroll 1
    while (cur.valid) {
      load_tile(cur, r0);
      r0 = r1;
      r1 = r2;
      r2 = r3;
      r3 = tile_raw(p, ahead, jl);
      tile_next(p, ahead, end);
      tile_next(p, cur, end);
    }
    cp_async_wait<0>();
  } else if (warp == tr::kWarpMma) {
    // ============================ MMA issue (one thread) ============================
    if (lane == 0) {
      constexpr uint32_t idS = FP8 ? idesc(0, 0, 0, 0, 64, KT) : idesc(1, 1, 0, 0, 64, KT);
      constexpr uint32_t idPV = FP8 ? idesc(0, 0, 0, 1, 64, D) : idesc(1, 1, 0, 1, 64, D);
      constexpr int NKS = FP8 ? D / 32 : D / 16;  // k-steps of 32 bytes, four per 128-byte column block
      // descriptors of the operands' bases; an offset is added in 16-byte units
      const uint64_t dq0 = sdesc(q_s, 16, 1024), dk0 = sdesc(ring_s, 16, 1024), dp0 = sdesc(p_s, 16, 1024);
      const uint64_t dv0 = sdesc(FP8 ? v16_s : ring_s, KT * 128, 1024);
      // ring positions of the next QK tile and the next PV tile (bf16: its V entry)
      tr::RingPos kpos{0, 0u}, vpos{FP8 ? 0 : 1, 0u};
      long long u = 0, qp = 0;
      long long pu = -1;  // tile whose PV is pending
      bool pfirst = false;
      auto issue_pv = [&](long long w, bool first) {
        tr::wait(bar(tr::kBPFull + (w & 1)), static_cast<uint32_t>((w >> 1) & 1), abort_flag, p.err);
        const int slotV = vpos.slot;
        if constexpr (FP8)
          tr::wait(bar(tr::kBV16Full + (w & 1)), static_cast<uint32_t>((w >> 1) & 1), abort_flag, p.err);
        else
          tr::wait(bar(tr::kBFull + slotV), vpos.lap & 1u, abort_flag, p.err);
        vpos.step(NE, FP8 ? 1 : 2);
        fence_proxy_async();
        tc_fence_after();
        const uint64_t pd = dp0 + static_cast<uint64_t>(((w & 1) * G::PB) >> 4);
        const uint64_t vd = dv0 + static_cast<uint64_t>((FP8 ? (w & 1) * G::V16B : slotV * ENT) >> 4);
#pragma unroll
        for (int ks = 0; ks < KT / 16; ++ks)
          mma_f16_ss(tmem + tr::kColO, pd + static_cast<uint64_t>(ks * 2), vd + static_cast<uint64_t>(ks * 128), idPV,
                     !(first && ks == 0));
        mma_commit(bar(tr::kBPEmpty + (w & 1)));
        if constexpr (FP8)
          mma_commit(bar(tr::kBV16Empty + (w & 1)));
        else
          mma_commit(bar(tr::kBEmpty + slotV));
      };
      Seg s = seg0;
      while (seg_live(p, s, end)) {
        const int t0 = static_cast<int>(max(start, s.off) - s.off);
        const int te = piece_real_end(s, end);
        if (t0 < te) {
          // the previous piece's last PV first: its partial precedes this piece's queries
          if (pu >= 0) {
            issue_pv(pu, pfirst);
            pu = -1;
          }
          tr::wait(bar(tr::kBQFull), static_cast<uint32_t>(qp & 1), abort_flag, p.err);
          ++qp;
          for (int tok0 = t0; tok0 < te; tok0 += KT, ++u) {
            const int slotK = kpos.slot;
            tr::wait(bar(tr::kBFull + slotK), kpos.lap & 1u, abort_flag, p.err);
            kpos.step(NE, FP8 ? 1 : 2);
            tr::wait(bar(tr::kBSEmpty + (u & 1)), static_cast<uint32_t>(((u >> 1) & 1) ^ 1), abort_flag, p.err);
            fence_proxy_async();
            tc_fence_after();
            const uint64_t kd = dk0 + static_cast<uint64_t>((slotK * G::RING_UNIT) >> 4);
            const uint32_t sS = tmem + static_cast<uint32_t>((u & 1) * tr::NCS * KT);
#pragma unroll
            for (int ks = 0; ks < NKS; ++ks) {
              const uint64_t ad = dq0 + static_cast<uint64_t>(((ks >> 2) * (64 * 128) + (ks & 3) * 32) >> 4);
              const uint64_t bd = kd + static_cast<uint64_t>(((ks >> 2) * (KT * 128) + (ks & 3) * 32) >> 4);
              const uint32_t dc = sS + static_cast<uint32_t>((ks % tr::NCS) * KT);
              if constexpr (FP8)
                mma_f8_ss(dc, ad, bd, idS, ks >= tr::NCS);
              else
                mma_f16_ss(dc, ad, bd, idS, ks >= tr::NCS);
            }
            mma_commit(bar(tr::kBSFull + (u & 1)));
            mma_commit(bar(tr::kBEmpty + slotK));
            if (pu >= 0) issue_pv(pu, pfirst);
            pu = u;
            pfirst = tok0 == t0;
          }
        }
        seg_advance(p, s);
      }
      if (pu >= 0) issue_pv(pu, pfirst);
    }
    __syncwarp();
  } else if (warp >= tr::kWarpCvt0) {
    // ======================= V widening (e4m3 pools) =======================
    if constexpr (FP8) {
      const int ct = tid - tr::kWarpCvt0 * 32;
      constexpr int CPR = G::CPR;  // 16-byte chunks of an e4m3 row
      TileIt it;
      it.s = seg0;
      it.tok = static_cast<int>(start - seg0.off);
      it.te = piece_real_end(seg0, end);
      tile_settle(p, it, end);
      long long u = 0;
      tr::RingPos vpos{0, 0u};
      while (it.valid) {
        const int slotV = vpos.slot;
        tr::wait_warp(bar(tr::kBFull + slotV), vpos.lap & 1u, abort_flag, p.err);
        vpos.step(NE);
        tr::wait_warp(bar(tr::kBV16Empty + (u & 1)), static_cast<uint32_t>(((u >> 1) & 1) ^ 1), abort_flag, p.err);
        const unsigned char* raw = smem + G::ring_off + slotV * G::TILEB + ENT;
        unsigned char* v16 = smem + G::v16_off + (u & 1) * G::V16B;
#pragma unroll 2
        for (int i = 0; i < KT * CPR / 128; ++i) {
          const int ci = ct + 128 * i;
          const int tt = ci / CPR, c = ci % CPR;
          const uint4 w = *reinterpret_cast<const uint4*>(raw + (c >> 3) * (KT * 128) + tt * 128 +
                                                          (((c & 7) ^ (tt & 7)) << 4));
          // dv = 16c .. 16c + 15: 64-dv block c / 4, f16 chunks 2 (c % 4) and 2 (c % 4) + 1
          unsigned char* dst = v16 + (c >> 2) * (KT * 128) + tt * 128;
          const int ch = (c & 3) * 2;
          *reinterpret_cast<uint4*>(dst + ((ch ^ (tt & 7)) << 4)) =
              make_uint4(e4m3x2_to_f16x2(w.x & 0xFFFFu), e4m3x2_to_f16x2(w.x >> 16), e4m3x2_to_f16x2(w.y & 0xFFFFu),
                         e4m3x2_to_f16x2(w.y >> 16));
          *reinterpret_cast<uint4*>(dst + (((ch + 1) ^ (tt & 7)) << 4)) =
              make_uint4(e4m3x2_to_f16x2(w.z & 0xFFFFu), e4m3x2_to_f16x2(w.z >> 16), e4m3x2_to_f16x2(w.w & 0xFFFFu),
                         e4m3x2_to_f16x2(w.w >> 16));
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(tr::kBV16Full + (u & 1)));
          mbar_arrive(bar(tr::kBEmpty + slotV));
        }
        tile_next(p, it, end);
        ++u;
      }
    }
  } else {
    // ================================ softmax ================================
    // Scores and O are read in the 16-lane fragment shape: thread t holds
    // rows g = t / 4 and g + 8 of its sub-partition (packed row 8 w + g: its
    // two terms) at columns 8 i + 2 c, 8 i + 2 c + 1 (c = t % 4) of every
    // 8-column group i, so each thread owns 16 keys of one packed row and the
    // four threads of a quad share the row.
    const int g = lane >> 2, c4 = lane & 3;
    const int prow = 8 * warp + g;   // packed query row of this thread
    const int arow = 16 * warp + g;  // its row of P and O
    const uint32_t t_lane = static_cast<uint32_t>(warp * 32) << 16;
    const uint64_t keep = policy_evict_last();
    const float NEG_INF = -INFINITY;
    unsigned* red_u = reinterpret_cast<unsigned*>(smem + tr::kRedOff);
    Seg s = seg0;
    long long u = 0;
    while (seg_live(p, s, end)) {
      const int t0 = static_cast<int>(max(start, s.off) - s.off);
      const int te = piece_real_end(s, end);
      const long long slot_self = blockIdx.x + static_cast<long long>(s.b) * p.n_hg + s.hg;
      float* lse_p = p.plse + slot_self * RM;
      float* o_p = p.po + slot_self * RM * D;
      if (t0 >= te) {
        // no real token in this piece: an empty partial
        for (int i = tid; i < RM * D; i += tr::kSmThreads) st_keep(o_p + i, 0.f, keep);
        if (tid < RM) st_keep(lse_p + tid, NEG_INF, keep);
        seg_advance(p, s);
        continue;
      }
      const float qsc = tr_load_q<FP8>(p, s, smem + G::q_off, red_u, tid);
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(tr::kBQFull));
      float mrun = NEG_INF, lp = 0.f;
#pragma unroll 1
      for (int tok0 = t0; tok0 < te; tok0 += KT, ++u) {
        const bool first = tok0 == t0, last = tok0 + KT >= te;
        // ---- scores of tile u: this thread's 16 keys, both terms summed ----
        tr::wait_warp(bar(tr::kBSFull + (u & 1)), static_cast<uint32_t>((u >> 1) & 1), abort_flag, p.err);
        tc_fence_after();
        float x[16];
        {
          float v[32];
          tr::ld16x256b_x8(tmem + t_lane + static_cast<uint32_t>((u & 1) * tr::NCS * KT), v);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(tr::kBSEmpty + (u & 1)));
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            x[2 * i] = v[4 * i] + v[4 * i + 2];
            x[2 * i + 1] = v[4 * i + 1] + v[4 * i + 3];
          }
        }
        // tile u's valid keys: one tagged word per loader warp
        const unsigned long long mw = tr::tile_mask<NL>(maskq, u, abort_flag, p.err);
        float t4[4] = {NEG_INF, NEG_INF, NEG_INF, NEG_INF};
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float y = ((mw >> (8 * i + 2 * c4 + e)) & 1ull) ? x[2 * i + e] * qsc : NEG_INF;
            x[2 * i + e] = y;
            t4[(2 * i + e) & 3] = fmaxf(t4[(2 * i + e) & 3], y);
          }
        float tm = fmaxf(fmaxf(t4[0], t4[1]), fmaxf(t4[2], t4[3]));
        tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 1));
        tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 2));  // the row's tile maximum, alike in the quad
        if (__any_sync(0xffffffffu, tm > mrun + tr::kThr)) {
          const float mn = fmaxf(mrun, tm);
          const float al = mn == NEG_INF ? 1.f : fast_exp2(mrun - mn);
          if (!first && __any_sync(0xffffffffu, al != 1.f)) {
            // O holds earlier tiles of this piece: rescale this warp's rows
            // once the last PV is done
            tr::wait_warp(bar(tr::kBPEmpty + ((u - 1) & 1)), static_cast<uint32_t>(((u - 1) >> 1) & 1), abort_flag,
                          p.err);
            tc_fence_after();
#pragma unroll 1
            for (int cb = 0; cb < D / 64; ++cb) {
              float o[32];
              tr::ld16x256b_x8(tmem + t_lane + tr::kColO + 64 * cb, o);
#pragma unroll
              for (int k = 0; k < 32; ++k) o[k] *= al;
              tr::st16x256b_x8(tmem + t_lane + tr::kColO + 64 * cb, o);
            }
            tmem_wait_st();
          }
          lp *= al;
          mrun = mn;
        }
        // ---- probabilities of tile u into P (f16 for e4m3 pools, bf16 otherwise) ----
        const float mref = mrun == NEG_INF ? 0.f : mrun;
        uint32_t pk[8];
        float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float p0 = fast_exp2(x[2 * i] - mref), p1 = fast_exp2(x[2 * i + 1] - mref);
          l4[i & 3] += p0 + p1;
          pk[i] = FP8 ? pack_f16(p0, p1) : pack_bf16(p0, p1);
        }
        lp += (l4[0] + l4[1]) + (l4[2] + l4[3]);
        tr::wait_warp(bar(tr::kBPEmpty + (u & 1)), static_cast<uint32_t>(((u >> 1) & 1) ^ 1), abort_flag, p.err);
        {
          // keys 8 i + 2 c4, + 1: 16-byte chunk i of row arow, bytes 4 c4 .. 4 c4 + 3
          unsigned char* pr = smem + G::p_off + (u & 1) * G::PB + arow * 128 + 4 * c4;
#pragma unroll
          for (int i = 0; i < 8; ++i) *reinterpret_cast<uint32_t*>(pr + ((i ^ (arow & 7)) << 4)) = pk[i];
        }
        fence_proxy_async();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(tr::kBPFull + (u & 1)));
        if (last) {
          // ---- piece end: this warp's rows of the partial (o v_scale / l, m + log2 l) ----
          tr::wait_warp(bar(tr::kBPEmpty + (u & 1)), static_cast<uint32_t>((u >> 1) & 1), abort_flag, p.err);
          tc_fence_after();
          float l = lp + __shfl_xor_sync(0xffffffffu, lp, 1);
          l += __shfl_xor_sync(0xffffffffu, l, 2);
          const bool wr = prow < RM;
          const float inv = l > 0.f ? p.v_scale / l : 0.f;
          if (wr && c4 == 0) st_keep(lse_p + prow, l > 0.f ? mrun + log2f(l) : NEG_INF, keep);
#pragma unroll 1
          for (int cb = 0; cb < D / 64; ++cb) {
            float o[32];
            tr::ld16x256b_x8(tmem + t_lane + tr::kColO + 64 * cb, o);
            if (wr) {
#pragma unroll
              for (int i = 0; i < 8; ++i)
                st_keep2(o_p + prow * D + 64 * cb + 8 * i + 2 * c4, o[4 * i] * inv, o[4 * i + 1] * inv, keep);
            }
          }
          tc_fence_before();
        }
      }
      seg_advance(p, s);
    }
  }
  // ---- teardown: every MMA was waited for by the softmax warps ----
  tc_fence_before();
  __syncthreads();
  if (warp == tr::kWarpMma) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tr::kCols) : "memory");
  }
}

// rows-on-M tensor-memory stream, head_dim 256, rm = 16 or 32 packed rows
KernelFn kernel_tr(bool fp8, int rm);

}  // namespace vsk
