// sparse_attn_tc.cu — CSA2 sparse attention on the 5th-generation tensor
// cores (tcgen05, TMEM accumulators): gathered FP4 main-KV rows plus the
// layer's SWA rows, all heads of one sequence (or prefill query) per pair of
// CTAs.
//
// [CSA2] wire.sakhanda.co, "DeepSeek AI выпустила DeepSeek-V4.1-Flash ...",
//        section "Сжатое разреженное внимание 2 (CSA2)": sparse attention over
//        the Top-512 main-KV entries plus each layer's own SWA KV.
// [FP4]  same page, section "FP4 KV, ограниченное повторное проигрывание и
//        другие расширения": E2M1 x E4M3 per 16 channels (exact in bf16).
// [CED]  same page, section "Каузальный энкодер-декодер: вдвое меньший
//        префилл": 128-token sliding window in every layer.
//
// One (row, layer, key split) is attended by a cluster of two CTAs that split
// the 512 head dims: CTA r holds dims 256 r .. 256 r + 255 of the queries and
// of every key (K = V), so both S = Q K^T (a sum over dims) and O = P V (whose
// columns are dims) divide between them:
//   - each CTA computes a partial S over its dims for all 64 heads;
//   - the CTAs exchange halves of it through distributed shared memory: CTA r
//     owns heads 32 r .. 32 r + 31, receives the peer's partial S of those
//     heads, adds its own and runs their online softmax;
//   - the owner writes P (bf16) of its heads into both CTAs' P buffers (and
//     the O rescale factors when a running maximum moved);
//   - each CTA accumulates O = P V for its 256 dims and all heads.
// Halving the dims per CTA is what lets a key tile be 128 keys wide: S is an
// M = 64 (heads) x N = 128 (keys) MMA, twice the keys per instruction of a
// 64-key tile at the same instruction cost, with two 64 KB key buffers.
//
// Every operand is bf16 and exact: the queries and SWA rows are bf16 inputs
// and the FP4 dequantisation (E2M1 times its E4M3 scale, <= 6 significant
// bits between 2^-10 and 2688) is exact in bf16. P is rounded to bf16; the
// softmax denominator sums the rounded values. S, O and the softmax are fp32.
//
// Warp roles (416 threads):
//   warps 0-3   softmax / exchange / O rescale; warp q reads TMEM lanes of
//               heads 16 q .. 16 q + 15 (the M = 64 accumulator layout puts
//               head h in lane 32 (h / 16) + h % 16). Warps of the quadrants
//               the CTA owns run the softmax; the others send their partial S.
//   warps 4-11  producers: row sources of tile j + 3, FP4 rows of tile j + 2
//               prefetched into registers, dequantised into one of two key
//               buffers ([dim/64][key][128 B], K-major, 128-byte swizzle);
//               SWA rows copied in with cp.async; absent rows zero.
//   warp 12     TMEM allocation and, on one thread, the MMA issue: S(t) into
//               one of two S buffers as soon as tile t is in shared memory,
//               and PV(t) once both owners' P(t) is in place.
// TMEM: S buffers at columns 0 and 128 (N = 128), O at 256..511 (N = 256
// dims), 512 columns, one CTA per SM.
//
// Split-K partials (m, l, unnormalised O; O stored [dim/4][head][4]) are
// merged by the log-sum-exp merge kernel. Every wait is bounded (wall time
// and poll count) and also returns when either CTA of the pair has given up;
// a CTA that gives up reports CSA2_ERR_TIMEOUT, tells its peer and winds down
// (the warp groups decide to stop by barrier reductions, so no warp is left at
// a barrier). Both CTAs meet at a cluster barrier before exiting, so neither
// leaves while the other may still write into its shared memory.
#include "common.cuh"
#include "tcgen05.cuh"

namespace csa2 {

constexpr int kTD = 512;                  // head dim
constexpr int kDH = 256;                  // dims per CTA of the pair
constexpr int kTT = 128;                  // keys per tile
constexpr int kTThreads = 416;            // warps 0-3 softmax, 4-11 producers, 12 MMA
constexpr int kSoftWarps = 4;
constexpr int kSoftThreads = 32 * kSoftWarps;
constexpr int kProdBase = kSoftThreads;   // first producer thread
constexpr int kProd = 256;                // producer threads
constexpr int kProdWarps = kProd / 32;
constexpr int kItems = 8;                 // FP4 items (row, 16-channel group) per producer thread and tile
constexpr int kMmaWarp = 12;
constexpr int kRing = 8;                  // row-source ring: tiles j .. j+4 may be live at once
constexpr uint32_t kOCol = 256;           // O accumulator columns 256..511
constexpr int kXsStride = 528;            // bytes per head row of the exchange buffer (512 + 16: conflict-free)

struct TcSmem {                           // offsets from a 1024-aligned base
  static constexpr int kQ = 0;                            // [4][64 heads][128 B]   32 KB
  static constexpr int kKV = kQ + 4 * 64 * 128;           // 2 x [4][128 keys][128 B]
  static constexpr int kKVBytes = 4 * kTT * 128;          // 64 KB
  static constexpr int kP = kKV + 2 * kKVBytes;           // 2 x [2][64 heads][128 B]
  static constexpr int kPBytes = 2 * 64 * 128;            // 16 KB
  static constexpr int kXS = kP + 2 * kPBytes;            // [32 heads][528 B] partial S from the peer
  static constexpr int kSrc = kXS + 32 * kXsStride;       // int64 [kRing][128]: >= 0 FP4 row, -1 absent, <= -2 SWA row
  static constexpr int kMask = kSrc + kRing * kTT * 8;    // u32 [kRing][4] valid keys
  static constexpr int kFp4 = kMask + kRing * 16;         // u32 [kRing][4] keys that are FP4 rows
  static constexpr int kAlpha = kFp4 + kRing * 16;        // float [2][64] O rescale factors of a tile
  static constexpr int kFlag = kAlpha + 2 * 64 * 4;       // u32 [2][2]: tile + 1 when owner half r rescaled
  static constexpr int kL = kFlag + 16;                   // float [64] softmax denominators
  static constexpr int kM = kL + 256;                     // float [64] running maxima (log2 domain)
  static constexpr int kBar = kM + 256;                   // mbarriers (slots below)
  static constexpr int kMisc = kBar + 24 * 8;             // [0] tmem base, [1] abort
  static constexpr int kBytes = kMisc + 64 + 1024;        // + alignment slack
};
static_assert(TcSmem::kBytes <= 232448, "shared memory of the attention kernel");
static_assert(TcSmem::kBar % 8 == 0 && TcSmem::kSrc % 8 == 0, "alignment");
// mbarrier slots
constexpr int kBarKvFull = 0;             // [2] producers -> MMA (count kProd)
constexpr int kBarKvEmpty = 2;            // [2] PV done with a key buffer (local commit)
constexpr int kBarSFull = 4;              // [2] S ready (local commit)
constexpr int kBarXsFull = 6;             // the peer's partial S is in kXS (64 remote arrives)
constexpr int kBarXsEmpty = 7;            // the peer has read our partial S (64 remote arrives)
constexpr int kBarPFull = 8;              // [2] P of all heads in place (64 local + 64 remote arrives)
constexpr int kBarPFree = 10;             // [2] PV of both CTAs done with a P buffer (multicast commits)
constexpr int kBarPvGo = 12;              // [2] P ready and O rescaled: PV may go (count 1). Two of
                                          // them: the softmax of tile j + 1 may finish before the
                                          // MMA thread has seen tile j's, and a phase must not be
                                          // overtaken before it is observed
constexpr int kBarFin = 14;               // every MMA of the CTA done (local commit)
constexpr int kBarLFull = 15;             // the peer's (l, m) of its heads are in kL / kM (32 remote arrives)

// K-major 128-byte-swizzle offset of 16-byte chunk `chunk` (0..7) of `row`
// within one 64-dim (or 64-key) block of 128-byte rows.
__device__ __forceinline__ uint32_t sw_off(int row, int chunk) {
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// E4M3 scale byte -> {s, s} as f16x2 (exact).
__device__ __forceinline__ uint32_t scale_f16x2(uint32_t sbyte) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)(sbyte | (sbyte << 8))));
  return h2;
}
// One byte of two E2M1 codes times the scale -> bf16x2 (low code -> low half).
// The fp16 product is exact (<= 6 significant bits, 2^-10 .. 2688), and so is
// its bf16 form.
__device__ __forceinline__ uint32_t e2m1x2_scaled_bf16x2(uint32_t byte, uint32_t s_h2) {
  const uint32_t h2 = e2m1x2_to_f16x2(byte);
  uint32_t p;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(p) : "r"(h2), "r"(s_h2));
  const float lo = __half2float(__ushort_as_half((unsigned short)(p & 0xFFFFu)));
  const float hi = __half2float(__ushort_as_half((unsigned short)(p >> 16)));
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// 16x32bx2.x32: lanes 0-15 of the warp's TMEM quadrant; thread t < 16 gets
// lane t, columns c..c+31, thread t >= 16 gets lane t - 16, columns c+32..c+63
__device__ __forceinline__ void tmem_ld_16x32bx2_32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32], 32;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// the matching store shape
__device__ __forceinline__ void tmem_st_16x32bx2_32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x32bx2.x32.b32 [%0], 32, {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
        "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
        "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]));
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Named barrier over `count` threads (a multiple of 32), and its OR-reduction
// form, which hands every participant the same answer.
__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ bool named_or(int id, int count, bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n barrier.cta.red.or.pred q, %2, %3, p;\n"
      " selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r) : "r"((uint32_t)v), "r"(id), "r"(count) : "memory");
  return r != 0;
}
constexpr int kNbSoft = 1, kNbProd = 2;   // named barrier ids (0 is __syncthreads)

__device__ __forceinline__ uint2 ldg_hint_u2(const void* p, uint64_t pol) {
  uint2 v;
  asm volatile("ld.global.nc.L2::cache_hint.v2.u32 {%0, %1}, [%2], %3;" : "=r"(v.x), "=r"(v.y) : "l"(p), "l"(pol));
  return v;
}
__device__ __forceinline__ uint32_t ldg_hint_u8(const void* p, uint64_t pol) {
  uint16_t v;
  asm volatile("ld.global.nc.L2::cache_hint.u8 %0, [%1], %2;" : "=h"(v) : "l"(p), "l"(pol));
  return v;
}

// Bounded wait on a local mbarrier that the peer CTA may arrive on. Gives up
// after `limit_ns` of wall time, or as soon as the abort word is set (by this
// CTA or by its peer); returns false then.
__device__ __forceinline__ bool pair_wait(uint32_t bar, uint32_t parity, const volatile uint32_t* abort_word,
                                          uint64_t limit_ns) {
  const uint64_t t0 = tc::globaltimer_ns();
  for (uint32_t i = 0; i < (1u << 24); ++i) {
    if (tc::mbar_try_wait_cluster(bar, parity)) return true;
    if ((i & 31) == 31 && (*abort_word != 0 || tc::globaltimer_ns() - t0 > limit_ns)) return false;
  }
  return false;
}

__global__ void __maxnreg__(152) k_sparse_attn_tc(
    const AttnLayers lay, int H, const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
    int64_t kv_seq_stride, int64_t n_cap, const int32_t* __restrict__ idx, int k, int64_t swa_seq_stride, int W,
    int swa_tail, int rps, const int32_t* __restrict__ swa_len, float scale_log2, int splits, int tiles_per_split,
    float* __restrict__ part_o, float* __restrict__ part_ml, int32_t* st, uint64_t wait_ns, int fault) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023) & ~1023u;
  unsigned char* sp = smem_raw + (base - raw);
  using L = TcSmem;
  float* sAlpha = reinterpret_cast<float*>(sp + L::kAlpha);
  volatile uint32_t* sFlag = reinterpret_cast<volatile uint32_t*>(sp + L::kFlag);
  float* sL = reinterpret_cast<float*>(sp + L::kL);
  float* sMx = reinterpret_cast<float*>(sp + L::kM);
  int64_t* sSrc = reinterpret_cast<int64_t*>(sp + L::kSrc);
  uint32_t* sMask = reinterpret_cast<uint32_t*>(sp + L::kMask);
  uint32_t* sFp4 = reinterpret_cast<uint32_t*>(sp + L::kFp4);
  volatile uint32_t* sMisc = reinterpret_cast<volatile uint32_t*>(sp + L::kMisc);
  auto bar = [&](int i) { return base + L::kBar + 8u * (uint32_t)i; };

  const uint32_t rank = tc::cluster_rank(), peer = rank ^ 1u;
  // the peer's view of an address of this CTA's shared memory
  auto remote = [&](uint32_t local_saddr) { return tc::mapa(local_saddr, peer); };
  const int b = blockIdx.y, split = blockIdx.x >> 1, layer = blockIdx.z;
  const __nv_bfloat16* __restrict__ q = lay.q[layer];
  const __nv_bfloat16* __restrict__ swa = lay.swa[layer];
  __nv_bfloat16* __restrict__ out = lay.out[layer];
  const int64_t unit = (int64_t)layer * gridDim.y + b;     // (layer, row) of the partials
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_tiles = (k + W + kTT - 1) / kTT;
  const int t_begin = split * tiles_per_split;
  const int t_end = min(t_begin + tiles_per_split, n_tiles);
  const int nt = max(t_end - t_begin, 0);
  const int d0 = kDH * (int)rank;                           // this CTA's first head dim
  const volatile uint32_t* abort_word = sMisc + 1;
  // give up: report, and tell both CTAs of the pair to wind down
  auto give_up = [&]() {
    report(st, CSA2_ERR_TIMEOUT);
    sMisc[1] = 1;
    tc::st_cluster_u32(remote(base + L::kMisc + 4), 1u);
  };
  auto wait = [&](int slot, uint32_t parity) { return pair_wait(bar(slot), parity, abort_word, wait_ns); };

  // ---- set-up: barriers touch no global memory and overlap the preceding
  //      kernel; both CTAs' barriers exist before either arrives remotely
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(bar(kBarKvFull + i), kProd);
      tc::mbar_init(bar(kBarKvEmpty + i), 1);
      tc::mbar_init(bar(kBarSFull + i), 1);
      tc::mbar_init(bar(kBarPFull + i), 128);
      tc::mbar_init(bar(kBarPFree + i), 2);
      tc::mbar_init(bar(kBarPvGo + i), 1);
    }
    tc::mbar_init(bar(kBarXsFull), 64);
    tc::mbar_init(bar(kBarXsEmpty), 64);
    tc::mbar_init(bar(kBarFin), 1);
    tc::mbar_init(bar(kBarLFull), 32);
    tc::fence_barrier_init();
    sMisc[1] = 0;
    for (int i = 0; i < 4; ++i) sFlag[i] = 0;
  }
  tc::cluster_sync();
  pdl_wait();
  if (warp == kMmaWarp) {
    tc::tmem_alloc(base + L::kMisc, 512);
    tc::tmem_relinquish();
  }
  const uint64_t pol_keep = l2_evict_last(), pol_stream = l2_evict_first();
  // Q rows (this CTA's 256 dims, bf16) straight into their K-major layout;
  // heads >= H are zero rows
  for (int e = tid; e < 64 * 32; e += kTThreads) {
    const int h = e >> 5, cc = e & 31;                     // chunk cc: dim block cc / 8, chunk cc % 8
    const uint32_t off = (cc >> 3) * 8192 + sw_off(h, cc & 7);
    if (h < H) cp_async16_hint(base + L::kQ + off, q + ((int64_t)b * H + h) * kTD + d0 + cc * 8, pol_stream);
    else *reinterpret_cast<uint4*>(sp + L::kQ + off) = make_uint4(0, 0, 0, 0);
  }
  cp_async_commit();
  // the SWA length is clamped without a branch, so nothing waits on its load
  const int slen_in = swa_len[b];
  // row b reads the caches of sequence b / rps; with rps > 1 the sequence's
  // SWA rows are linear and row b's window starts b % rps rows in
  const int64_t kv_row0 = (int64_t)(b / rps) * kv_seq_stride;
  const int64_t swa_row0 = (int64_t)(b / rps) * swa_seq_stride + (b % rps);
  const int slen = min(max(slen_in, 0), W);

  // Row sources of tile j (called by four whole warps: slot p of the tile).
  // Key slot s < W is SWA row s (present if s < slen); slot W + i is Top-K entry i.
  auto row_sources = [&](int j, int p) {
    const int slot = j % kRing;
    const int s = (t_begin + j) * kTT + p;
    int64_t src = -1;
    if (s < W) {
      if (s < slen) src = -2 - (swa_row0 + (swa_tail ? W - slen : 0) + s);
    } else if (s - W < k) {
      const int32_t pos = idx[(int64_t)b * k + (s - W)];
      if (pos >= 0 && pos < n_cap) src = kv_row0 + pos;
      else if (pos >= n_cap) report(st, CSA2_ERR_DEVICE_BOUNDS);
    }
    sSrc[slot * kTT + p] = src;
    const uint32_t valid = __ballot_sync(0xffffffffu, src != -1);
    const uint32_t fp4 = __ballot_sync(0xffffffffu, src >= 0);
    if ((p & 31) == 0) {
      sMask[slot * 4 + (p >> 5)] = valid;
      sFp4[slot * 4 + (p >> 5)] = fp4;
    }
  };
  if (tid < kTT) {
    for (int j = 0; j < 3 && j < nt; ++j) row_sources(j, tid);
  }
  __syncthreads();
  // the SWA rows of tile 0 travel with Q
  for (int e = tid; e < kTT * 32 && nt > 0; e += kTThreads) {
    const int rr = e >> 5, cc = e & 31;
    const int64_t s0 = sSrc[rr];
    if (s0 <= -2)
      cp_async16_hint(base + L::kKV + (cc >> 3) * 16384 + sw_off(rr, cc & 7), swa + (-2 - s0) * kTD + d0 + cc * 8,
                      pol_stream);
  }
  cp_async_commit();
  cp_async_wait<0>();
  tc::fence_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = sMisc[0];
  pdl_trigger();                              // TMEM is held: the next kernel may start launching

  // softmax owner threads (warps 2 rank, 2 rank + 1): head 16 warp + (lane & 15),
  // key columns 32 (lane >> 4) + 0..31 and 64 + 32 (lane >> 4) + 0..31 of a
  // tile; l_run sums the thread's columns, m_run is the same in both halves
  float m_run = -INFINITY, l_run = 0.f, l_tot = 0.f;

  if (warp >= kSoftWarps && warp < kMmaWarp) {
    // ================= producers =================
    const int p = tid - kProdBase, pw = p >> 5;
    // this thread's FP4 items of a tile: rows 64 (pw / 4) + 8 i + (lane & 7),
    // 16-channel group 4 (pw % 4) + (lane >> 3) of the CTA's 16, i.e. dim block
    // pw % 4 and its chunks 2 (lane >> 3), +1. Eight lanes of a store wavefront
    // write eight consecutive rows of one chunk column: distinct swizzle slots.
    const int rl = lane & 7, gl = lane >> 3, db = pw & 3, rbase = 64 * (pw >> 2) + rl;
    const int g = 4 * db + gl;                               // group within the CTA's dims
    uint2 cwA[kItems], cwB[kItems];
    uint32_t sbA[kItems], sbB[kItems];
    auto prefetch = [&](int j, uint2* cw, uint32_t* sb) {
      const int64_t* src = sSrc + (j % kRing) * kTT;
#pragma unroll
      for (int i = 0; i < kItems; ++i) {
        const int64_t s = src[rbase + 8 * i];
        cw[i] = make_uint2(0u, 0u);
        sb[i] = 0u;
        if (s >= 0) {
          cw[i] = ldg_hint_u2(codes + s * 256 + 128 * rank + g * 8, pol_keep);
          sb[i] = ldg_hint_u8(scales + s * 32 + 16 * rank + g, pol_keep);
        }
      }
    };
    // one tile: returns false when the pair stops
    auto produce = [&](int j, uint2* cw, uint32_t* sb) -> bool {
      if (named_or(kNbProd, kProd, sMisc[1] != 0)) return false;
      const int buf = j & 1, slot = j % kRing;
      const uint32_t kv = base + L::kKV + buf * L::kKVBytes;
      unsigned char* kvp = sp + L::kKV + buf * L::kKVBytes;
      if (j + 3 < nt && p < kTT) row_sources(j + 3, p);
      // the buffer is free once PV(j - 2) has finished
      if (j >= 2 && !wait(kBarKvEmpty + buf, ((j >> 1) - 1) & 1)) give_up();
      const int64_t* src = sSrc + slot * kTT;
      const uint32_t* vm = sMask + slot * 4;
      const uint32_t* fm = sFp4 + slot * 4;
      const bool any_other = (fm[0] & fm[1] & fm[2] & fm[3]) != 0xffffffffu;
      // absent rows: zero; SWA rows: bf16 straight into the key buffer (tile
      // 0's came with Q). Warp pw takes rows pw + 8 m, a lane one 16-byte chunk.
      bool copied = false;
      if (any_other) {
#pragma unroll
        for (int m = 0; m < kTT / kProdWarps; ++m) {
          const int rr = pw + 8 * m;                          // word m / 4 of the masks, bit pw + 8 (m % 4)
          const uint32_t vbit = (vm[m >> 2] >> (rr & 31)) & 1u, fbit = (fm[m >> 2] >> (rr & 31)) & 1u;
          const uint32_t off = (lane >> 3) * 16384 + sw_off(rr, lane & 7);
          if (!vbit) {
            *reinterpret_cast<uint4*>(kvp + off) = make_uint4(0, 0, 0, 0);
          } else if (!fbit && j > 0) {
            cp_async16_hint(kv + off, swa + (-2 - src[rr]) * kTD + d0 + lane * 8, pol_stream);
            copied = true;
          }
        }
      }
      cp_async_commit();
      // FP4 rows of this tile (in registers): one 16-channel group per item;
      // item i's row rbase + 8 i sits in mask word 2 (pw / 4) + i / 4
      const uint32_t f_lo = fm[2 * (pw >> 2)], f_hi = fm[2 * (pw >> 2) + 1];
#pragma unroll
      for (int i = 0; i < kItems; ++i) {
        const int rr = rbase + 8 * i;
        if (!(((i < 4 ? f_lo : f_hi) >> (rr & 31)) & 1u)) continue;
        const uint32_t sh2 = scale_f16x2(sb[i]);
        uint32_t o[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint32_t byte = ((u < 4 ? cw[i].x : cw[i].y) >> (8 * (u & 3))) & 0xFF;
          o[u] = e2m1x2_scaled_bf16x2(byte, sh2);
        }
        unsigned char* blk = kvp + db * 16384;
        *reinterpret_cast<uint4*>(blk + sw_off(rr, 2 * gl)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(blk + sw_off(rr, 2 * gl + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
      }
      if (copied) cp_async_wait<0>();
      tc::fence_async_smem();
      // fault injection (tests of the bounded waits): the last tile is never signalled
      if (!(fault == 1 && j == nt - 1)) tc::mbar_arrive(bar(kBarKvFull + buf));
      // tile j + 2's row sources were written in produce(j - 1), before this
      // call's opening barrier
      if (j + 2 < nt) prefetch(j + 2, cw, sb);
      return true;
    };
    if (nt > 0) prefetch(0, cwA, sbA);
    if (nt > 1) prefetch(1, cwB, sbB);
    for (int j = 0; j < nt; j += 2) {
      if (!produce(j, cwA, sbA)) break;
      if (j + 1 < nt && !produce(j + 1, cwB, sbB)) break;
    }
    cp_async_wait<0>();
  } else if (warp < kSoftWarps) {
    // ================= softmax / exchange / O correction =================
    const bool own = (uint32_t)(warp >> 1) == rank;
    const int h = 16 * warp + (lane & 15);                 // head of this thread's TMEM lane
    const int half = lane >> 4;
    const int hl = h - 32 * (warp >> 1);                    // row of the owner's exchange buffer
    const uint32_t xs_row = base + L::kXS + (uint32_t)hl * kXsStride + (uint32_t)half * 128;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * warp) << 16);
    for (int j = 0; j < nt; ++j) {
      if (named_or(kNbSoft, kSoftThreads, sMisc[1] != 0)) break;
      const int sbuf = j & 1;
      uint32_t r[64];                                       // columns 32 half + x, then 64 + 32 half + x
      bool ok = wait(kBarSFull + sbuf, (j >> 1) & 1);
      ok = ok && wait(kBarKvFull + sbuf, (j >> 1) & 1);    // orders the mask reads
      // tcgen05.ld / st are warp-collective: every decision that guards one is
      // made warp-uniform (a wait may run out for some lanes only)
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        tc::tc_fence_after();
        tmem_ld_16x32bx2_32(lane_base + 128u * sbuf, r);
        tmem_ld_16x32bx2_32(lane_base + 128u * sbuf + 64u, r + 32);
        tc::tmem_ld_wait();
      }
      if (!own) {
        // send this quadrant's partial S to the owner of its heads, once the
        // owner has read the previous tile's
        if (ok && j > 0) ok = wait(kBarXsEmpty, (j - 1) & 1);
        if (ok) {
          const uint32_t dst = remote(xs_row);
#pragma unroll
          for (int x = 0; x < 32; x += 4) {
            tc::st_cluster_v4(dst + 4 * x, r[x], r[x + 1], r[x + 2], r[x + 3]);
            tc::st_cluster_v4(dst + 256 + 4 * x, r[32 + x], r[33 + x], r[34 + x], r[35 + x]);
          }
          tc::mbar_arrive_cluster(remote(bar(kBarXsFull)));
        }
      } else {
        // owner: the peer's partial S of these heads, then the softmax
        if (ok) ok = wait(kBarXsFull, j & 1);
        if (ok) {
          const float4* xr = reinterpret_cast<const float4*>(sp + (xs_row - base));
#pragma unroll
          for (int x = 0; x < 8; ++x) {
            const float4 a = xr[x], c = xr[16 + x];
            r[4 * x] = __float_as_uint(__uint_as_float(r[4 * x]) + a.x);
            r[4 * x + 1] = __float_as_uint(__uint_as_float(r[4 * x + 1]) + a.y);
            r[4 * x + 2] = __float_as_uint(__uint_as_float(r[4 * x + 2]) + a.z);
            r[4 * x + 3] = __float_as_uint(__uint_as_float(r[4 * x + 3]) + a.w);
            r[32 + 4 * x] = __float_as_uint(__uint_as_float(r[32 + 4 * x]) + c.x);
            r[33 + 4 * x] = __float_as_uint(__uint_as_float(r[33 + 4 * x]) + c.y);
            r[34 + 4 * x] = __float_as_uint(__uint_as_float(r[34 + 4 * x]) + c.z);
            r[35 + 4 * x] = __float_as_uint(__uint_as_float(r[35 + 4 * x]) + c.w);
          }
          tc::mbar_arrive_cluster(remote(bar(kBarXsEmpty)));
          const uint32_t* vm = sMask + (j % kRing) * 4;
          const uint32_t v0 = vm[half], v1 = vm[2 + half];
          if ((v0 & v1) != 0xffffffffu) {
#pragma unroll
            for (int x = 0; x < 32; ++x) {
              if (!((v0 >> x) & 1u)) r[x] = __float_as_uint(-INFINITY);
              if (!((v1 >> x) & 1u)) r[32 + x] = __float_as_uint(-INFINITY);
            }
          }
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int x = 0; x < 64; ++x) m4[x & 3] = fmaxf(m4[x & 3], __uint_as_float(r[x]));
          float mh = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
          mh = fmaxf(mh, __shfl_xor_sync(0xffffffffu, mh, 16));
          // the scale is positive, so the scaled maximum is the maximum of the scaled scores
          const float mt = mh * scale_log2;
          float alpha = 1.f;
          if (mt > m_run + 8.f) {                 // raise the reference only when needed (P <= 256)
            alpha = (m_run == -INFINITY) ? 0.f : exp2f(m_run - mt);
            m_run = mt;
          }
          const float nbase = (m_run == -INFINITY) ? 0.f : -m_run;
          // both CTAs' P buffers are free once PV(j - 2) has finished in both
          if (j >= 2) ok = wait(kBarPFree + sbuf, ((j >> 1) - 1) & 1);
          if (ok) {
            float sum[4] = {0.f, 0.f, 0.f, 0.f};
            const uint32_t prow = base + L::kP + sbuf * L::kPBytes + h * 128;
            const uint32_t prow_r = remote(prow);
#pragma unroll
            for (int kb = 0; kb < 2; ++kb) {
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                uint32_t pk[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  const int x = 32 * kb + 8 * c + 2 * u;
                  const __nv_bfloat162 pv =
                      __floats2bfloat162_rn(exp2f(fmaf(__uint_as_float(r[x]), scale_log2, nbase)),
                                            exp2f(fmaf(__uint_as_float(r[x + 1]), scale_log2, nbase)));
                  const float2 f = __bfloat1622float2(pv);
                  sum[u] += f.x + f.y;
                  pk[u] = *reinterpret_cast<const uint32_t*>(&pv);
                }
                const uint32_t off = kb * 8192 + (((4 * half + c) ^ (h & 7)) << 4);
                *reinterpret_cast<uint4*>(sp + (prow - base) + off) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                tc::st_cluster_v4(prow_r + off, pk[0], pk[1], pk[2], pk[3]);
              }
            }
            l_run = l_run * alpha + ((sum[0] + sum[1]) + (sum[2] + sum[3]));
            const uint32_t a_addr = base + L::kAlpha + (uint32_t)(sbuf * 64 + h) * 4;
            if (half == 0) {
              *reinterpret_cast<float*>(sp + (a_addr - base)) = alpha;
              tc::st_cluster_u32(remote(a_addr), __float_as_uint(alpha));
            }
            if (alpha != 1.f && j > 0) {          // this half of the heads moved its reference
              const uint32_t f_addr = base + L::kFlag + (uint32_t)(sbuf * 2 + rank) * 4;
              sFlag[sbuf * 2 + rank] = (uint32_t)(j + 1);
              tc::st_cluster_u32(remote(f_addr), (uint32_t)(j + 1));
            }
            tc::fence_async_smem_cluster();
            tc::mbar_arrive(bar(kBarPFull + sbuf));
            tc::mbar_arrive_cluster(remote(bar(kBarPFull + sbuf)));
          }
        }
      }
      // every quadrant: all heads' P (and rescale factors) of this tile in place
      if (ok) ok = wait(kBarPFull + sbuf, (j >> 1) & 1);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) give_up();
      // -- rescale O when an owner half raised its reference (rare); O is
      //    free once this CTA's PV(j - 1) has finished (both CTAs' commits)
      const bool resc = __all_sync(0xffffffffu, ok && (sFlag[sbuf * 2] == (uint32_t)(j + 1) ||
                                                        sFlag[sbuf * 2 + 1] == (uint32_t)(j + 1)));
      if (resc) {
        if (__all_sync(0xffffffffu, wait(kBarPFree + ((j - 1) & 1), ((j - 1) >> 1) & 1))) {
          tc::tc_fence_after();
          const float a = sAlpha[sbuf * 64 + h];
          for (int c = 0; c < 256; c += 64) {
            uint32_t o[32];
            tmem_ld_16x32bx2_32(lane_base + kOCol + c, o);
            tc::tmem_ld_wait();
#pragma unroll
            for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * a);
            tmem_st_16x32bx2_32(lane_base + kOCol + c, o);
          }
          tmem_st_wait();
        } else {
          give_up();
        }
      }
      tc::tc_fence_before();
      named_sync(kNbSoft, kSoftThreads);
      if (tid == 0 && sMisc[1] == 0) tc::mbar_arrive(bar(kBarPvGo + sbuf));
    }
    if (own) l_tot = l_run + __shfl_xor_sync(0xffffffffu, l_run, 16);
  } else {
    // ================= MMA issue (one thread) =================
    if (lane == 0) {
      const uint32_t idesc_s = tc::instr_desc(tc::kFmtBF16, tc::kFmtBF16, 0, 0, 64, kTT);   // heads x keys
      const uint32_t idesc_o = tc::instr_desc(tc::kFmtBF16, tc::kFmtBF16, 0, 1, 64, kDH);   // heads x dims
      auto issue_s = [&](int j) {
        const uint32_t kv = base + L::kKV + (j & 1) * L::kKVBytes;
#pragma unroll 4
        for (int ks = 0; ks < kDH / 16; ++ks) {
          const uint64_t ad = tc::smem_desc(base + L::kQ + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024, tc::kSwizzle128B);
          const uint64_t bd = tc::smem_desc(kv + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024, tc::kSwizzle128B);
          tc::mma_f16(tmem + 128u * (j & 1), ad, bd, idesc_s, ks > 0 ? 1u : 0u);
        }
        tc::mma_commit(bar(kBarSFull + (j & 1)));
      };
      auto issue_pv = [&](int j) {
        const uint32_t kv = base + L::kKV + (j & 1) * L::kKVBytes;
        const uint32_t pb = base + L::kP + (j & 1) * L::kPBytes;
#pragma unroll
        for (int ks = 0; ks < kTT / 16; ++ks) {
          const uint64_t ad = tc::smem_desc(pb + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024, tc::kSwizzle128B);
          const uint64_t bd = tc::smem_desc(kv + ks * 2048, 16384, 1024, tc::kSwizzle128B);
          tc::mma_f16(tmem + kOCol, ad, bd, idesc_o, (j > 0 || ks > 0) ? 1u : 0u);
        }
        tc::mma_commit(bar(kBarKvEmpty + (j & 1)));
        tc::mma_commit_multicast(bar(kBarPFree + (j & 1)), (uint16_t)3);
      };
      // Issue S(js) once its key tile is ready (and S(js - 2)'s softmax has
      // handed over, i.e. PV(js - 2) was issued), and PV(jp) once its P is
      // ready; whichever comes first. The polls share one time bound.
      bool ok = true;
      int js = 0, jp = 0;
      uint64_t t0 = tc::globaltimer_ns();
      uint32_t polls = 0;
      while (jp < nt) {
        bool progressed = false;
        if (js < nt && js <= jp + 1 && tc::mbar_test_wait(bar(kBarKvFull + (js & 1)), (js >> 1) & 1)) {
          tc::tc_fence_after();
          issue_s(js++);
          progressed = true;
        }
        if (jp < js && tc::mbar_test_wait(bar(kBarPvGo + (jp & 1)), (jp >> 1) & 1)) {
          tc::tc_fence_after();
          issue_pv(jp++);
          progressed = true;
        }
        if (progressed) {
          t0 = tc::globaltimer_ns();
          polls = 0;
        } else if ((++polls & 255) == 0 && (sMisc[1] || tc::globaltimer_ns() - t0 > wait_ns)) {
          ok = false;
          break;
        }
      }
      if (!ok) give_up();
      // every MMA of this CTA has completed before TMEM is read or freed
      tc::mma_commit(bar(kBarFin));
      if (!tc::mbar_wait(bar(kBarFin), 0)) give_up();
    }
    __syncwarp();
  }
  __syncthreads();
  tc::tc_fence_after();
  bool have_o = nt > 0 && sMisc[1] == 0;
  if ((slen_in < 0 || slen_in > W) && split == 0 && rank == 0 && tid == 0) report(st, CSA2_ERR_DEVICE_BOUNDS);
  // (l, m) of every head: owners write theirs here and into the peer
  if (warp < kSoftWarps && (uint32_t)(warp >> 1) == rank && lane < 16) {
    const int h = 16 * warp + lane;
    const float lv = have_o ? l_tot : 0.f, mv = have_o ? m_run : -INFINITY;
    sL[h] = lv;
    sMx[h] = mv;
    tc::st_cluster_u32(remote(base + L::kL + 4u * h), __float_as_uint(lv));
    tc::st_cluster_u32(remote(base + L::kM + 4u * h), __float_as_uint(mv));
    tc::mbar_arrive_cluster(remote(bar(kBarLFull)));
  }
  if (tid == 0 && !pair_wait(bar(kBarLFull), 0, abort_word, wait_ns)) give_up();
  __syncthreads();
  have_o = have_o && sMisc[1] == 0;
  if (warp < 8) {
    // the peer may set the abort word at any time: decide per warp, once
    have_o = __all_sync(0xffffffffu, have_o);
    // ---- epilogue: warp w reads the TMEM quadrant w % 4 (heads 16 (w % 4) ..
    // + 15) and the column half w / 4 of O's 256 dims. tcgen05.ld is
    // warp-collective, so whole warps load; lanes of heads >= H only skip
    // the stores.
    const int qd = warp & 3, chalf = warp >> 2;
    const int h = 16 * qd + (lane & 15);
    const bool live = h < H;
    const uint32_t ta = tmem + ((uint32_t)(32 * qd) << 16) + kOCol + 128 * chalf;
    const float lsum = sL[h];
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
#pragma unroll 1
    for (int c = 0; c < 128; c += 64) {
      uint32_t r[32];
      if (have_o) {
        tmem_ld_16x32bx2_32(ta + c, r);
        tc::tmem_ld_wait();
      } else {
#pragma unroll
        for (int x = 0; x < 32; ++x) r[x] = 0u;
      }
      if (!live) continue;
      const int dim0 = d0 + 128 * chalf + c + 32 * (lane >> 4);
      if (splits == 1) {
        __nv_bfloat16* o = out + ((int64_t)b * H + h) * kTD + dim0;
#pragma unroll
        for (int x = 0; x < 32; x += 8) {
          uint32_t pk[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(r[x + 2 * u]) * inv,
                                                          __uint_as_float(r[x + 2 * u + 1]) * inv);
            pk[u] = *reinterpret_cast<const uint32_t*>(&v);
          }
          st_global_hint(o + x, make_uint4(pk[0], pk[1], pk[2], pk[3]), pol_stream);
        }
      } else {
        // partial O layout [unit][split][dim / 4][H][4]
        float* o = part_o + (((unit * splits + split) * (kTD / 4) + dim0 / 4) * H + h) * 4;
#pragma unroll
        for (int x = 0; x < 32; x += 4)
          *reinterpret_cast<float4*>(o + (int64_t)(x / 4) * H * 4) =
              make_float4(__uint_as_float(r[x]), __uint_as_float(r[x + 1]), __uint_as_float(r[x + 2]),
                          __uint_as_float(r[x + 3]));
      }
    }
    // (m, l) of the partials: each CTA writes the heads it owns
    if (live && splits > 1 && chalf == 0 && lane < 16 && (uint32_t)(qd >> 1) == rank) {
      const int64_t pidx = (unit * splits + split) * H + h;
      part_ml[pidx * 2 + 0] = sMx[h];
      part_ml[pidx * 2 + 1] = sL[h];
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  // neither CTA leaves while the other may still write into its shared memory
  tc::cluster_sync();
  if (warp == kMmaWarp) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

int attn_tc_init_attributes() {
  if (cudaFuncSetAttribute(k_sparse_attn_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, TcSmem::kBytes) !=
      cudaSuccess)
    return CSA2_ERR_CUDA;
  return CSA2_OK;
}

int launch_sparse_attn_tc(const AttnLayers& lay, int L, int B, int H, const uint8_t* codes, const uint8_t* scales,
                          int64_t kv_seq_stride, int64_t n_cap, const int32_t* idx, int k, int64_t swa_seq_stride,
                          int W, int swa_tail, int rps, const int32_t* swa_len, float softmax_scale, float* part_o,
                          float* part_ml, int splits, int tps, int32_t* st, uint64_t wait_ns, int fault,
                          cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * splits), (unsigned)B, (unsigned)L);
  cfg.blockDim = dim3(kTThreads);
  cfg.dynamicSmemBytes = TcSmem::kBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, k_sparse_attn_tc, lay, H, codes, scales, kv_seq_stride, n_cap, idx, k,
                                           swa_seq_stride, W, swa_tail, rps, swa_len,
                                           softmax_scale * 1.4426950408889634f, splits, tps, part_o, part_ml, st,
                                           wait_ns, fault);
  count_launch();
  return launch_status(e);
}

}  // namespace csa2
