// Tensor-memory form of the prefix stream for head_dim 256 (tcgen05, sm_103a).
//
// Same operation and work split as vsk_kernel's streaming phase (the
// "verify_splitkv.py" page, "_verify_prefix_stage1": per-split partial
// softmaxes over the gathered prefix, qk *= sm_scale * k_scale, acc *=
// v_scale), with the two contractions on the 5th-generation tensor cores and
// their accumulators in tensor memory, so that no thread holds a 16 x 256
// accumulator tile in registers.  It writes the per-piece (o, log-sum-exp)
// partials in vsk_kernel's workspace format; vsk_combine_kernel then folds
// them, adds the draft block and writes the output (a second launch).
//
// One CTA per SM, one KV head per segment (heads per CTA HC = 1), 64-key tiles.
// Keys are the M dimension of both products, so the packed query rows (RM =
// 16 or 32) are N and the output is kept transposed:
//   S^T[64 keys][RM]   = K_tile[64][256]      x Q^T         (TMEM, 2 buffers; the
//                        contraction split over 4 accumulators, since dependent
//                        accumulations into one tile issue far slower than
//                        independent ones)
//   O^T[256 dv][RM]   += V_tile^T[256][64]    x P^T[64][RM] (TMEM, 2 halves of 128)
// Roles (warp specialised, all hand-offs on mbarriers with bounded waits):
//   warps 0-7  softmax, two warpgroups, each owning half of the RM packed rows
//              (warps w and w + 4 read the same TMEM lanes): thread = TMEM
//              lane = key of a tile (S) / dv (O); online softmax in the log2
//              domain whose running maximum is raised only when a score
//              exceeds it by more than 2^8 (then O is rescaled in TMEM); P^T
//              to shared memory; for an e4m3 pool also the e4m3 -> f16
//              widening of the V tile.
//   warp 8     TMEM allocation; lane 0 issues every tcgen05.mma.
//   warps 9-15 loaders: kv_indices / page ids, 16-byte cp.async gathers of the
//              K and V rows into a ring of 64-key entries, completion through
//              cp.async.mbarrier.arrive.noinc (seven warps, since the copies a
//              single warp keeps in flight are limited).
// Operands in shared memory use the 128-byte swizzled canonical layouts:
//   K tile, Q          K-major   [128-byte column block][row][128 B]
//   V tile (A = V^T)   MN-major  [64-dv block][key][128 B]   (same bytes as
//                      a K-major row store: one loader code serves both)
//   P^T (B)            MN-major  [key][128 B] (RM <= 64 rows in one block)
// For an e4m3 pool S uses kind::f8f6f4 straight from the e4m3 K rows with the
// queries split exactly into two e4m3 terms (q * 2^sh = hi + lo, max |q| 2^sh
// in [128, 256)); PV uses f16 (e4m3 V widened exactly, P in f16).

namespace tc {

constexpr int KT = 64;                     // keys per tile (M of S^T)
constexpr int NL = 7;                      // loader warps: warp i copies tokens [KT i / NL, KT (i+1) / NL) of every tile
constexpr int TPW = (KT + NL - 1) / NL;    // at most this many tokens a warp
constexpr int kSmThreads = 256;            // two softmax warpgroups
constexpr int kWarpMma = 8;
constexpr int kWarpLoad0 = 9;
constexpr int kThreads = (kWarpLoad0 + NL) * 32;  // 16 warps: 4 per SM sub-partition at 128 registers
constexpr int kMaxNE = 12;                 // ring entries at most
constexpr float kThr = 8.f;                // log2 headroom before the running maximum is raised
constexpr int NC = 4;                      // independent accumulation chains of S^T (summed by the softmax)
// shared-memory map
constexpr int kBarOff = 256;               // mbarriers, 8 B each
constexpr int kTmemOff = 544;              // TMEM base address written by tcgen05.alloc
constexpr int kAbortOff = 548;             // set when a wait gave up
constexpr int kMcntOff = 552;              // key-mask bytes published so far (release / acquire)
constexpr int kRedOff = 1024;              // [2 warpgroups][4 warps][32 rows] fp32 row reductions
constexpr int kMaskOff = 2048;             // [kMaskRing][NL] 64-bit valid-key words of the tiles
constexpr int kMaskRing = 16;              // > the tiles loaders can run ahead of the softmax
constexpr int kDataOff = 3072;             // 1024-aligned operand regions from here
// barrier indices
constexpr int kBFull = 0, kBEmpty = kMaxNE, kBSFull = 2 * kMaxNE, kBSEmpty = kBSFull + 2, kBPFull = kBSEmpty + 2,
              kBPEmpty = kBPFull + 2, kBQFull = kBPEmpty + 2, kBV16Empty = kBQFull + 1, kNumBars = kBV16Empty + 1;
static_assert(kBarOff + 8 * kNumBars <= kTmemOff, "barriers overlap");
static_assert(kMaskOff + kMaskRing * NL * 8 <= kDataOff, "masks overlap");

// Byte sizes of the regions (all multiples of 1024).
template <int D, bool FP8, int RM>
struct Geo {
  static constexpr int EK = FP8 ? 1 : 2;
  static constexpr int ROWB = D * EK;              // one K (or V) row of one head
  static constexpr int CPR = ROWB / 16;            // its 16-byte chunks
  static constexpr int ENT = KT * ROWB;            // one ring entry: K or V rows of a tile
  static constexpr int NHALF = D / 128;            // M = 128 blocks of O^T
  static constexpr int QB = RM * D * 2;            // bf16 Q, or e4m3 hi and lo
  static constexpr int PB = KT * 128;              // one P^T buffer
  static constexpr int V16B = FP8 ? (D / 64) * KT * 128 : 0;  // widened V tile
  static constexpr int q_off = kDataOff;
  static constexpr int p_off = q_off + QB;
  static constexpr int v16_off = p_off + 2 * PB;
  static constexpr int ring_off = v16_off + V16B;
  static constexpr int cols = (2 * NC + NHALF) * RM;  // TMEM columns: 2 S buffers x NC chains, O^T halves
  static constexpr int alloc_cols = cols <= 32 ? 32 : (cols <= 64 ? 64 : (cols <= 128 ? 128 : (cols <= 256 ? 256 : 512)));
};

__device__ __forceinline__ void mbar_init(uint32_t bar, int count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// try_wait with a suspend-time hint: a waiting thread sleeps (up to 0.5 ms)
// until the phase completes instead of re-polling shared memory.
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\nselp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(500000)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
// Wait for the phase of the given parity to complete, for one second at
// most; a wait that gives up sets the CTA's abort flag (every later wait then
// returns at once, so the CTA drains) and the timeout error bit.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, unsigned* err) {
  if (mbar_try(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
    if (mbar_try(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > 1000000000ull) {
      *abort_flag = 1;
      atomicOr(err, kErrTimeout);
      return false;
    }
  }
}
// The same for a whole warp: lane 0 waits (the phase's completion is then
// visible to the other lanes through __syncwarp), so 32 lanes do not all
// poll shared memory.
__device__ __forceinline__ void mbar_wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                               unsigned* err) {
  if ((threadIdx.x & 31) == 0) mbar_wait(bar, parity, abort_flag, err);
  __syncwarp();
}
__device__ __forceinline__ void red_release_add(uint32_t addr, unsigned v) {
  asm volatile("red.release.cta.shared::cta.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire(uint32_t addr) {
  unsigned v;
  asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
// Wait (one second at most, like mbar_wait) until the counter reaches n;
// lane 0 of the warp polls, the others meet it at __syncwarp.
__device__ __forceinline__ void wait_count(uint32_t addr, unsigned n, volatile int* abort_flag, unsigned* err) {
  if ((threadIdx.x & 31) == 0 && ld_acquire(addr) < n) {
    const unsigned long long t0 = global_ns();
    while (ld_acquire(addr) < n) {
      __nanosleep(64);
      if (*abort_flag) break;
      if (global_ns() - t0 > 1000000000ull) {
        *abort_flag = 1;
        atomicOr(err, kErrTimeout);
        break;
      }
    }
  }
  __syncwarp();
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ bool bar_red_or(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n.reg .pred pi, po;\nsetp.ne.u32 pi, %1, 0;\nbar.red.or.pred po, %2, %3, pi;\nselp.u32 %0, 1, 0, po;\n}\n"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// Shared-memory matrix descriptor: start, leading / stride byte offsets,
// descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFF) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor (kind::f16 / kind::f8f6f4): fp32 accumulator, operand
// formats, operand majors (1 = MN-major), N >> 3, M >> 4.
__host__ __device__ constexpr uint32_t idesc(int afmt, int bfmt, int amaj, int bmaj, int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(afmt) << 7) | (static_cast<uint32_t>(bfmt) << 10) |
         (static_cast<uint32_t>(amaj) << 15) | (static_cast<uint32_t>(bmaj) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
__device__ __forceinline__ void mma_f16_ss(uint32_t tmem, uint64_t a, uint64_t b, uint32_t id, bool acc) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem),
      "l"(a), "l"(b), "r"(id), "r"(acc ? 1 : 0));
}
__device__ __forceinline__ void mma_f8_ss(uint32_t tmem, uint64_t a, uint64_t b, uint32_t id, bool acc) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          tmem),
      "l"(a), "l"(b), "r"(id), "r"(acc ? 1 : 0));
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// TMEM <-> registers, 32 lanes x N columns of 32 bits (lane = thread of the warp).
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float (&v)[N]);
template <>
__device__ __forceinline__ void tmem_ld<8>(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
template <>
__device__ __forceinline__ void tmem_ld<16>(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
template <>
__device__ __forceinline__ void tmem_ld<32>(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
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
template <int N>
__device__ __forceinline__ void tmem_st(uint32_t taddr, const float (&v)[N]);
template <>
__device__ __forceinline__ void tmem_st<8>(uint32_t taddr, const float (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
               "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
               "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
               "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
               : "memory");
}
template <>
__device__ __forceinline__ void tmem_st<16>(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}
template <>
__device__ __forceinline__ void tmem_st<32>(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
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
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Reduce N values per lane over the 32 lanes of a warp, row by row (max or
// sum): halving exchanges leave lane l with rows whose index is l's bits (N =
// 32: row l; N = 16: row l >> 1, lanes 2i and 2i+1 alike).  Returns the row
// of v[0].
template <int N, bool MAX>
__device__ __forceinline__ int warp_rows_reduce(float (&v)[N], int lane) {
  int n = N;
  int row = 0;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    if (n >= 2) {
      const int h = n / 2;
      const bool up = (lane & off) != 0;
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        if (i < h) {
          const float send = up ? v[i] : v[i + h];
          const float keep = up ? v[i + h] : v[i];
          const float got = __shfl_xor_sync(0xffffffffu, send, off);
          v[i] = MAX ? fmaxf(keep, got) : keep + got;
        }
      }
      if (up) row += h;
      n = h;
    } else {
      const float got = __shfl_xor_sync(0xffffffffu, v[0], off);
      v[0] = MAX ? fmaxf(v[0], got) : v[0] + got;
    }
  }
  return row;
}

}  // namespace tc

// Successive 64-key tiles of this CTA's share (pieces without a real token
// are skipped): segment, first token, end of the piece's real tokens.
struct TileIt {
  Seg s;
  int tok, te;
  bool valid;
};
__device__ __forceinline__ void tile_settle(const Params& p, TileIt& it, long long end) {
  while (seg_live(p, it.s, end) && it.tok >= it.te) {
    seg_advance(p, it.s);
    it.tok = 0;
    if (seg_live(p, it.s, end)) it.te = piece_real_end(it.s, end);
  }
  it.valid = seg_live(p, it.s, end);
}
__device__ __forceinline__ void tile_next(const Params& p, TileIt& it, long long end) {
  if (!it.valid) return;
  it.tok += tc::KT;
  tile_settle(p, it, end);
}
// The loaded value that locates token tok + j of a tile: its kv_indices
// entry, or for a paged cache the page id of its block-table column; -1 past
// the piece.  No arithmetic depends on the load, so it stays in flight until
// tile_loc reads it.
__device__ __forceinline__ long long tile_raw(const Params& p, const TileIt& it, int j) {
  if (!it.valid || j >= tc::KT) return -1;
  const int t = it.tok + j;
  if (t >= it.te) return -1;
  if (p.paged) return __ldg(p.bt + static_cast<long long>(it.s.b) * p.bt_s0 + page_of(p, t));
  const long long n = it.s.kv0 + t;
  return p.idx64 ? __ldg(static_cast<const long long*>(p.kvi) + n)
                 : static_cast<long long>(__ldg(static_cast<const int*>(p.kvi) + n));
}
// Pool row of token tok + j from its tile_raw value (-1: none or invalid page).
__device__ __forceinline__ long long tile_loc(const Params& p, const TileIt& it, int j, long long raw) {
  if (!p.paged || raw < 0) return raw;
  const int t = it.tok + j;
  return raw * p.page + (t - page_of(p, t) * p.page);
}

// One warpgroup's half of the piece's query rows (packed row r = draft r / gq,
// query head kvh * gq + r % gq, for r in [wg * RH, wg * RH + RH); rows >= R are
// zero) into the B operand of S^T, K-major 128-byte swizzled: bf16 [RM][D], or
// for an e4m3 pool e4m3 hi and lo [RM][D] with q * 2^sh = hi + lo (sh chosen
// per warpgroup).  Called by the warpgroup's 128 threads (tw = 0..127);
// returns the score scale of its rows into the log2 domain (sm_scale *
// k_scale * log2 e, times 2^-sh).
template <int D, bool FP8, int RM>
__device__ __forceinline__ float tc_load_q(const Params& p, const Seg& s, unsigned char* qs, unsigned* red_u,
                                           int wg, int tw) {
  constexpr int RH = RM / 2;
  const int a = p.qo ? __ldg(p.qo + s.b) : s.b * p.L, e = p.qo ? __ldg(p.qo + s.b + 1) : (s.b + 1) * p.L;
  const bool ok = a >= 0 && e - a == p.L && static_cast<long long>(a) + p.L <= p.n_rows;
  if (!ok && wg == 0 && tw == 0) atomicOr(p.err, kErrBadQoIndptr);
  const int s_b = ok ? a : s.b * p.L;
  const int kvh = s.hg;                     // one KV head per segment
  constexpr int CH = D / 8;                 // 8-element chunks per row
  constexpr int NCH = RH * CH / 128;        // chunks per thread
  uint32_t v[NCH][4];
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    const int ci = tw + 128 * i;
    const int r = wg * RH + ci / CH, c = ci % CH;
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
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
      const int ci = tw + 128 * i;
      const int r = wg * RH + ci / CH, c = ci % CH;
      *reinterpret_cast<uint4*>(qs + (c >> 3) * (RM * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4)) =
          make_uint4(v[i][0], v[i][1], v[i][2], v[i][3]);
    }
    return p.scale2;
  } else {
    // largest |q| of these rows (bf16 bit patterns order like magnitudes)
    unsigned mx = 0;
#pragma unroll
    for (int i = 0; i < NCH; ++i)
#pragma unroll
      for (int w = 0; w < 4; ++w) mx = max(mx, max(v[i][w] & 0x7FFFu, (v[i][w] >> 16) & 0x7FFFu));
    mx = __reduce_max_sync(0xffffffffu, mx);
    if ((tw & 31) == 0) red_u[tw >> 5] = mx;
    named_bar_sync(1 + wg, 128);
    mx = max(max(red_u[0], red_u[1]), max(red_u[2], red_u[3]));
    named_bar_sync(1 + wg, 128);  // red_u is free again
    const int ex = static_cast<int>(mx >> 7) - 127;
    int sh = mx == 0 ? 0 : 7 - ex;  // the largest |q| * 2^sh lies in [128, 256)
    sh = max(-120, min(120, sh));
    const float up = __int_as_float((127 + sh) << 23);
    unsigned char* qhi = qs;
    unsigned char* qlo = qs + RM * D;
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
      const int ci = tw + 128 * i;
      const int r = wg * RH + ci / CH, c = ci % CH;
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
      // elements d = 8c .. 8c+7: 128-element column block d / 128, 16-byte
      // chunk (d % 128) / 16, byte d % 16
      const int d = 8 * c;
      const int off = (d >> 7) * (RM * 128) + r * 128 + ((((d & 127) >> 4) ^ (r & 7)) << 4) + (d & 15);
      *reinterpret_cast<uint2*>(qhi + off) = make_uint2(hw[0], hw[1]);
      *reinterpret_cast<uint2*>(qlo + off) = make_uint2(lw[0], lw[1]);
    }
    return p.scale2 * __int_as_float((127 - sh) << 23);
  }
}

template <int D, bool FP8, int RM>
__global__ void __launch_bounds__(tc::kThreads, 1) vtc_kernel(const __grid_constant__ Params p) {
  using namespace tc;
  using G = Geo<D, FP8, RM>;
  extern __shared__ __align__(1024) unsigned char smem[];
  constexpr int NHALF = G::NHALF;
  constexpr int ENT = G::ENT;
  constexpr int PB = G::PB;
  constexpr int RH = RM / 2;  // rows of one softmax warpgroup
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NE = p.nst;

  long long start, end, W;
  Seg seg0;
  if (!cta_share(p, smem, start, end, W, seg0)) return;  // uniform: no work
  // The 128-byte swizzled layouts need a 1024-byte aligned base.  Dynamic
  // shared memory of a kernel without static shared memory starts there; were
  // it not so, the CTA reports the pipeline error bit and writes nothing.
  if ((smem_u32(smem) & 1023u) != 0u) {
    if (tid == 0) atomicOr(p.err, kErrTimeout);
    return;
  }

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
  auto bar = [&](int i) -> uint32_t { return smem_u32(bars + i); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortOff);
  unsigned long long* maskq = reinterpret_cast<unsigned long long*>(smem + kMaskOff);
  const uint32_t mcnt = smem_u32(smem + kMcntOff);
  const uint32_t q_s = smem_u32(smem + G::q_off);
  const uint32_t p_s = smem_u32(smem + G::p_off);
  const uint32_t v16_s = smem_u32(smem + G::v16_off);
  const uint32_t ring_s = smem_u32(smem + G::ring_off);

  if (tid == 0) {
    *abort_flag = 0;
    *reinterpret_cast<volatile unsigned*>(smem + kMcntOff) = 0u;
    for (int i = 0; i < NE; ++i) {
      mbar_init(bar(kBFull + i), NL * 32);
      // e4m3 pools: odd entries hold V rows, released by the widening threads
      mbar_init(bar(kBEmpty + i), (FP8 && (i & 1)) ? kSmThreads : 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(kBSFull + b), 1);
      mbar_init(bar(kBSEmpty + b), kSmThreads);
      mbar_init(bar(kBPFull + b), kSmThreads);
      mbar_init(bar(kBPEmpty + b), 1);
    }
    mbar_init(bar(kBQFull), kSmThreads);
    mbar_init(bar(kBV16Empty), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kWarpMma) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem + kTmemOff)),
                 "r"(G::alloc_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kTmemOff);
  // S buffer b, chain c at column (b * NC + c) * RM; O^T halves at colO + h * RM
  const uint32_t colO = 2 * NC * RM;

  if (warp >= kWarpLoad0) {
    // ================================ loaders ================================
    const int lw = warp - kWarpLoad0;
    const uint64_t pol = policy_evict_first();
    constexpr int CPR = G::CPR;
    constexpr int LPT = CPR < 32 ? CPR : 32;  // lanes per row
    constexpr int TSTEP = 32 / LPT;          // rows per warp instruction
    constexpr int CPL = CPR / LPT;           // chunks per lane per row
    const int tlo = KT * lw / NL, cnt = KT * (lw + 1) / NL - tlo;  // this warp's tokens of a tile
    long long e = 0;  // ring entries issued
    // one tile: its two ring entries (K rows, then V rows) from the pool rows
    // of this warp's cnt tokens (lane j < cnt holds token tlo + j's row)
    auto load_tile = [&](const TileIt& it, long long raw) {
      const int t = it.tok + tlo + lane;
      const long long loc = tile_loc(p, it, tlo + lane, raw);
      const bool ok = lane < cnt && t < it.te && loc >= 0 && loc < p.pool;
      if (lane < cnt && t < it.te && !ok) atomicOr(p.err, kErrBadIndex);
      const unsigned m = __ballot_sync(0xffffffffu, ok);
      const long long head = it.s.hg;
#pragma unroll 1
      for (int kv = 0; kv < 2; ++kv, ++e) {
        const int slot = static_cast<int>(e % NE);
        mbar_wait_warp(bar(kBEmpty + slot), static_cast<uint32_t>(((e / NE) & 1) ^ 1), abort_flag, p.err);
        if (kv == 0 && lane == 0) {
          // this warp's valid keys of the tile, published for the softmax warps
          maskq[static_cast<int>((e >> 1) % kMaskRing) * NL + lw] = static_cast<unsigned long long>(m) << tlo;
          red_release_add(mcnt, 1u);
        }
        const unsigned char* base = (kv ? p.vb + head * p.vb_s1 : p.kb + head * p.kb_s1);
        const long long s0 = kv ? p.vb_s0 : p.kb_s0;
        const uint32_t dst0 = ring_s + static_cast<uint32_t>(slot) * ENT;
#pragma unroll
        for (int i = 0; i < (TPW + TSTEP - 1) / TSTEP; ++i) {
          const int tl = i * TSTEP + lane / LPT;  // token among this warp's cnt
          const long long lc = __shfl_sync(0xffffffffu, loc, tl & 31);
          if (tl < cnt) {
            const bool v = (m >> tl) & 1u;
            const int tt = tlo + tl;  // token within the tile
#pragma unroll
            for (int cj = 0; cj < CPL; ++cj) {
              const int c = lane % LPT + LPT * cj;
              const uint32_t d = dst0 + (c >> 3) * (KT * 128) + tt * 128 + (((c & 7) ^ (tt & 7)) << 4);
              const unsigned char* src = v ? base + lc * s0 + c * 16 : reinterpret_cast<const unsigned char*>(p.q);
              cp_async_16_zfill(d, src, v, pol);
            }
          }
        }
        cp_async_arrive_noinc(bar(kBFull + slot));
      }
    };
    // Pool rows are read kPF tiles before their tile is copied, into kPF
    // registers used in place (no register copy waits on a load in flight).
    constexpr int kPF = 4;
    TileIt cur;
    cur.s = seg0;
    cur.tok = static_cast<int>(start - seg0.off);
    cur.te = piece_real_end(seg0, end);
    tile_settle(p, cur, end);
    TileIt ahead = cur;
    long long rows[kPF];
#pragma unroll
    for (int k = 0; k < kPF; ++k) {
      rows[k] = tile_raw(p, ahead, lane < cnt ? tlo + lane : KT);
      tile_next(p, ahead, end);
    }
    while (cur.valid) {
#pragma unroll
      for (int k = 0; k < kPF; ++k) {
        if (cur.valid) {
          load_tile(cur, rows[k]);
          rows[k] = tile_raw(p, ahead, lane < cnt ? tlo + lane : KT);
          tile_next(p, ahead, end);
          tile_next(p, cur, end);
        }
      }
    }
    cp_async_wait<0>();
  } else if (warp == kWarpMma) {
    // ============================ MMA issue (one thread) ============================
    if (lane == 0) {
      constexpr uint32_t idS = FP8 ? idesc(0, 0, 0, 0, KT, RM) : idesc(1, 1, 0, 0, KT, RM);
      constexpr uint32_t idPV = FP8 ? idesc(0, 0, 1, 1, 128, RM) : idesc(1, 1, 1, 1, 128, RM);
      long long u = 0, qp = 0;
      long long pu = -1;  // tile whose PV is pending
      bool pfirst = false;
      auto issue_pv = [&](long long w, bool first) {
        mbar_wait(bar(kBPFull + (w & 1)), static_cast<uint32_t>((w >> 1) & 1), abort_flag, p.err);
        const long long eV = 2 * w + 1;
        const int slotV = static_cast<int>(eV % NE);
        if constexpr (!FP8) mbar_wait(bar(kBFull + slotV), static_cast<uint32_t>((eV / NE) & 1), abort_flag, p.err);
        fence_proxy_async();
        tc_fence_after();
        const uint32_t abase = FP8 ? v16_s : ring_s + static_cast<uint32_t>(slotV) * ENT;
        const uint32_t bbase = p_s + static_cast<uint32_t>(w & 1) * PB;
#pragma unroll
        for (int ks = 0; ks < KT / 16; ++ks) {
          const uint64_t bd = sdesc(bbase + 2 * ks * 1024, KT * 128, 1024);
#pragma unroll
          for (int h = 0; h < NHALF; ++h) {  // the halves are independent chains: alternate them
            const uint64_t ad = sdesc(abase + 2 * h * (KT * 128) + 2 * ks * 1024, KT * 128, 1024);
            mma_f16_ss(tmem + colO + h * RM, ad, bd, idPV, !(first && ks == 0));
          }
        }
        mma_commit(bar(kBPEmpty + (w & 1)));
        if constexpr (FP8)
          mma_commit(bar(kBV16Empty));
        else
          mma_commit(bar(kBEmpty + slotV));
      };
      Seg s = seg0;
      while (seg_live(p, s, end)) {
        const int t0 = static_cast<int>(max(start, s.off) - s.off);
        const int te = piece_real_end(s, end);
        if (t0 < te) {
          // the previous piece's last PV first: its finaliser loads this piece's Q
          if (pu >= 0) {
            issue_pv(pu, pfirst);
            pu = -1;
          }
          mbar_wait(bar(kBQFull), static_cast<uint32_t>(qp & 1), abort_flag, p.err);
          ++qp;
          for (int tok0 = t0; tok0 < te; tok0 += KT, ++u) {
            const long long eK = 2 * u;
            const int slotK = static_cast<int>(eK % NE);
            mbar_wait(bar(kBFull + slotK), static_cast<uint32_t>((eK / NE) & 1), abort_flag, p.err);
            mbar_wait(bar(kBSEmpty + (u & 1)), static_cast<uint32_t>(((u >> 1) & 1) ^ 1), abort_flag, p.err);
            fence_proxy_async();
            tc_fence_after();
            const uint32_t kbase = ring_s + static_cast<uint32_t>(slotK) * ENT;
            const uint32_t sS = tmem + static_cast<uint32_t>((u & 1) * NC * RM);
            if constexpr (FP8) {
              // chains (k-step parity, hi / lo): consecutive MMAs never share an accumulator
#pragma unroll
              for (int ks = 0; ks < D / 32; ++ks) {
                const uint64_t ad = sdesc(kbase + (ks >> 2) * (KT * 128) + (ks & 3) * 32, 16, 1024);
                const uint32_t qo = (ks >> 2) * (RM * 128) + (ks & 3) * 32;
                const uint32_t c0 = static_cast<uint32_t>((ks & 1) * 2) * RM;
                mma_f8_ss(sS + c0, ad, sdesc(q_s + qo, 16, 1024), idS, ks >= 2);
                mma_f8_ss(sS + c0 + RM, ad, sdesc(q_s + RM * D + qo, 16, 1024), idS, ks >= 2);
              }
            } else {
#pragma unroll
              for (int ks = 0; ks < D / 16; ++ks) {
                const uint64_t ad = sdesc(kbase + (ks >> 2) * (KT * 128) + (ks & 3) * 32, 16, 1024);
                const uint64_t bd = sdesc(q_s + (ks >> 2) * (RM * 128) + (ks & 3) * 32, 16, 1024);
                mma_f16_ss(sS + static_cast<uint32_t>(ks % NC) * RM, ad, bd, idS, ks >= NC);
              }
            }
            mma_commit(bar(kBSFull + (u & 1)));
            mma_commit(bar(kBEmpty + slotK));
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
  } else {
    // ================================ softmax ================================
    // warpgroup wg owns packed rows [wg * RH, wg * RH + RH); warp w4 = warp % 4
    // reads TMEM lanes [32 * w4, 32 * w4 + 32)
    const int wg = warp >> 2, w4 = warp & 3, tw = tid & 127;
    const int key = (w4 << 4) + lane;  // M = 64: lanes 0-15 of subpartition w4 hold keys 16 w4 .. 16 w4 + 15
    const bool klane = lane < 16;
    const uint32_t t_lane = static_cast<uint32_t>(w4 * 32) << 16;
    const uint64_t keep = policy_evict_last();
    const float NEG_INF = -INFINITY;
    float* red = reinterpret_cast<float*>(smem + kRedOff) + wg * 128;  // [4 warps][32]
    const int bid = 1 + wg;  // this warpgroup's named barrier
    constexpr int LPR = 32 / RH;  // lanes holding one row after a warp row reduction
    float mrun[RH], lp[RH];
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
        for (int i = tid; i < RM * D; i += kSmThreads) st_keep(o_p + i, 0.f, keep);
        if (tid < RM) st_keep(lse_p + tid, NEG_INF, keep);
        seg_advance(p, s);
        continue;
      }
      const float qsc = tc_load_q<D, FP8, RM>(p, s, smem + G::q_off, reinterpret_cast<unsigned*>(red), wg, tw);
      fence_proxy_async();
      mbar_arrive(bar(kBQFull));
#pragma unroll
      for (int r = 0; r < RH; ++r) {
        mrun[r] = NEG_INF;
        lp[r] = 0.f;
      }
#pragma unroll 1
      for (int tok0 = t0; tok0 < te; tok0 += KT, ++u) {
        const bool first = tok0 == t0, last = tok0 + KT >= te;
        // ---- scores of tile u (this warpgroup's rows; the NC chains summed) ----
        mbar_wait_warp(bar(kBSFull + (u & 1)), static_cast<uint32_t>((u >> 1) & 1), abort_flag, p.err);
        tc_fence_after();
        float x[RH];
        {
          const uint32_t sc = tmem + t_lane + static_cast<uint32_t>((u & 1) * NC * RM + wg * RH);
          tmem_ld<RH>(sc, x);
#pragma unroll
          for (int c = 1; c < NC; ++c) {
            float y[RH];
            tmem_ld<RH>(sc + c * RM, y);
#pragma unroll
            for (int r = 0; r < RH; ++r) x[r] += y[r];
          }
        }
        tc_fence_before();
        mbar_arrive(bar(kBSEmpty + (u & 1)));
        wait_count(mcnt, static_cast<unsigned>(NL * (u + 1)), abort_flag, p.err);  // tile u's key mask
        unsigned long long mw = lane < NL ? maskq[static_cast<int>(u % kMaskRing) * NL + lane] : 0ull;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) mw |= __shfl_xor_sync(0xffffffffu, mw, off);
        const bool valid = klane && ((mw >> key) & 1ull);
        bool need = false;
#pragma unroll
        for (int r = 0; r < RH; ++r) {
          x[r] = valid ? x[r] * qsc : NEG_INF;
          need |= x[r] > mrun[r] + kThr;
        }
        need = bar_red_or(bid, 128, need);
        if (need) {
          // raise the running maxima to the tile's row maxima
          float y[RH];
#pragma unroll
          for (int r = 0; r < RH; ++r) y[r] = x[r];
          const int row = warp_rows_reduce<RH, true>(y, lane);
          if (lane % LPR == 0) red[w4 * 32 + row] = y[0];
          named_bar_sync(bid, 128);
          float al[RH];
          bool moved = false;
#pragma unroll
          for (int r = 0; r < RH; ++r) {
            const float tm = fmaxf(fmaxf(red[r], red[32 + r]), fmaxf(red[64 + r], red[96 + r]));
            const float mn = fmaxf(mrun[r], tm);
            al[r] = mn == NEG_INF ? 1.f : fast_exp2(mrun[r] - mn);
            moved |= al[r] != 1.f;
            mrun[r] = mn;
          }
          named_bar_sync(bid, 128);  // the row maxima are read: red is free
          if (!first && moved) {
            // O^T holds earlier tiles of this piece: rescale this warpgroup's
            // columns once the last PV is done
            mbar_wait_warp(bar(kBPEmpty + ((u - 1) & 1)), static_cast<uint32_t>(((u - 1) >> 1) & 1), abort_flag, p.err);
            tc_fence_after();
#pragma unroll
            for (int h = 0; h < NHALF; ++h) {
              float o[RH];
              tmem_ld<RH>(tmem + t_lane + colO + h * RM + wg * RH, o);
#pragma unroll
              for (int r = 0; r < RH; ++r) o[r] *= al[r];
              tmem_st<RH>(tmem + t_lane + colO + h * RM + wg * RH, o);
            }
            tmem_wait_st();
          }
#pragma unroll
          for (int r = 0; r < RH; ++r) lp[r] *= al[r];
        }
        // ---- probabilities: P^T of tile u (f16 for e4m3 pools, bf16 otherwise) ----
        uint32_t pk[RH / 2];
#pragma unroll
        for (int r = 0; r < RH; r += 2) {
          const float m0 = mrun[r] == NEG_INF ? 0.f : mrun[r];
          const float m1 = mrun[r + 1] == NEG_INF ? 0.f : mrun[r + 1];
          const float p0 = fast_exp2(x[r] - m0), p1 = fast_exp2(x[r + 1] - m1);
          lp[r] += p0;
          lp[r + 1] += p1;
          pk[r / 2] = FP8 ? pack_f16(p0, p1) : pack_bf16(p0, p1);
        }
        mbar_wait_warp(bar(kBPEmpty + (u & 1)), static_cast<uint32_t>(((u >> 1) & 1) ^ 1), abort_flag, p.err);
        if (klane) {
          unsigned char* pr = smem + G::p_off + (u & 1) * PB + (key >> 3) * 1024 + (key & 7) * 128;
#pragma unroll
          for (int cc = 0; cc < RH / 8; ++cc) {
            const int ch = wg * (RH / 8) + cc;  // 16-byte chunk = rows 8 ch .. 8 ch + 7
            *reinterpret_cast<uint4*>(pr + ((ch ^ (key & 7)) << 4)) =
                make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
          }
        }
        if constexpr (FP8) {
          // widen tile u's e4m3 V rows to f16 (the A operand of PV), both warpgroups
          if (u > 0) mbar_wait_warp(bar(kBV16Empty), static_cast<uint32_t>((u - 1) & 1), abort_flag, p.err);
          const long long eV = 2 * u + 1;
          const int slotV = static_cast<int>(eV % NE);
          mbar_wait_warp(bar(kBFull + slotV), static_cast<uint32_t>((eV / NE) & 1), abort_flag, p.err);
          const unsigned char* raw = smem + G::ring_off + slotV * ENT;
          unsigned char* v16 = smem + G::v16_off;
          constexpr int CPR = G::CPR;  // 16-byte chunks of an e4m3 row
#pragma unroll
          for (int i = 0; i < KT * CPR / kSmThreads; ++i) {
            const int ci = tid + kSmThreads * i;
            const int tt = ci / CPR, c = ci % CPR;
            const uint4 w = *reinterpret_cast<const uint4*>(raw + (c >> 3) * (KT * 128) + tt * 128 +
                                                            (((c & 7) ^ (tt & 7)) << 4));
            // dv = 16c .. 16c+15: 64-dv block c / 4, f16 chunks 2(c % 4) and 2(c % 4) + 1
            unsigned char* dst = v16 + (c >> 2) * (KT * 128) + tt * 128;
            const int ch = (c & 3) * 2;
            *reinterpret_cast<uint4*>(dst + ((ch ^ (tt & 7)) << 4)) =
                make_uint4(e4m3x2_to_f16x2(w.x & 0xFFFFu), e4m3x2_to_f16x2(w.x >> 16), e4m3x2_to_f16x2(w.y & 0xFFFFu),
                           e4m3x2_to_f16x2(w.y >> 16));
            *reinterpret_cast<uint4*>(dst + (((ch + 1) ^ (tt & 7)) << 4)) =
                make_uint4(e4m3x2_to_f16x2(w.z & 0xFFFFu), e4m3x2_to_f16x2(w.z >> 16), e4m3x2_to_f16x2(w.w & 0xFFFFu),
                           e4m3x2_to_f16x2(w.w >> 16));
          }
          mbar_arrive(bar(kBEmpty + slotV));
        }
        fence_proxy_async();
        tc_fence_before();
        mbar_arrive(bar(kBPFull + (u & 1)));
        if (last) {
          // ---- piece end: this warpgroup's rows of the partial (o * v_scale / l, m + log2 l) ----
          mbar_wait_warp(bar(kBPEmpty + (u & 1)), static_cast<uint32_t>((u >> 1) & 1), abort_flag, p.err);
          tc_fence_after();
          float y[RH];
#pragma unroll
          for (int r = 0; r < RH; ++r) y[r] = lp[r];
          const int row = warp_rows_reduce<RH, false>(y, lane);
          if (lane % LPR == 0) red[w4 * 32 + row] = y[0];
          named_bar_sync(bid, 128);
          float inv[RH];
          float lse_mine = NEG_INF;
#pragma unroll
          for (int r = 0; r < RH; ++r) {
            const float l = (red[r] + red[32 + r]) + (red[64 + r] + red[96 + r]);
            inv[r] = l > 0.f ? p.v_scale / l : 0.f;
            if (r == tw) lse_mine = l > 0.f ? mrun[r] + log2f(l) : NEG_INF;
          }
          named_bar_sync(bid, 128);
          if (tw < RH) st_keep(lse_p + wg * RH + tw, lse_mine, keep);
#pragma unroll
          for (int h = 0; h < NHALF; ++h) {
            float o[RH];
            tmem_ld<RH>(tmem + t_lane + colO + h * RM + wg * RH, o);
            const int dv = h * 128 + tw;
#pragma unroll
            for (int r = 0; r < RH; ++r) st_keep(o_p + (wg * RH + r) * D + dv, o[r] * inv[r], keep);
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
  if (warp == kWarpMma) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(G::alloc_cols) : "memory");
  }
}
