// sparse_attn_tc.cu — CSA2 sparse attention on the 5th-generation tensor
// cores (tcgen05, TMEM accumulators): gathered FP4 main-KV rows plus the
// layer's SWA rows, all heads of one sequence (or prefill query) per CTA.
//
// [CSA2] wire.sakhanda.co, "DeepSeek AI выпустила DeepSeek-V4.1-Flash ...",
//        section "Сжатое разреженное внимание 2 (CSA2)": sparse attention over
//        the Top-512 main-KV entries plus each layer's own SWA KV.
// [FP4]  same page, section "FP4 KV, ограниченное повторное проигрывание и
//        другие расширения": E2M1 x E4M3 per 16 channels (exact in fp16).
// [CED]  same page, section "Каузальный энкодер-декодер: вдвое меньший
//        префилл": 128-token sliding window in every layer.
//
// Key slots are processed in tiles of 64 (the layer's SWA rows first, then
// the gathered rows) by a warp-specialised pipeline:
//   producers (warps 4-11): row sources from the Top-K indices three tiles
//             ahead; the FP4 rows prefetched into registers two tiles ahead,
//             then dequantised (E2M1 -> f16x2 hardware convert times the
//             E4M3 scale as a packed f16 multiply: the product, <= 6
//             significant bits in 2^-10 .. 2688, is exact in fp16) into one
//             of two key buffers in the K-major 128-byte-swizzle layout
//             [dim/64][key][128 B]. SWA rows (bf16) arrive in that layout by
//             TMA (one 2-D load per dim block of 64 rows, issued at set-up)
//             and are converted in place; a row whose largest magnitude
//             reaches 2^16 is first scaled by 2^-b (b <= 7, exact), and its
//             logits and probabilities are scaled back by 2^b in the softmax
//             (rows reaching 2^23 are reported as out of range). Below 2^-14
//             a value keeps an absolute accuracy of 2^-25; absent rows are
//             zero;
//   MMA (one thread each of warps 12 and 13): warp 12 issues
//             S(t) = Q K(t)^T with tcgen05.mma kind::f16, M = 64 heads,
//             N = 64 keys, K = 512, into one of two S buffers in TMEM, as
//             soon as tile t is ready and the softmax has read S(t - 2);
//             warp 13 issues O += P(t) V(t) as soon as P(t) is ready, so PV
//             never waits behind the issue of an S;
//   softmax (warps 0-3, two threads per head: key columns 0..31 and
//             32..63): reads S, takes the tile's per-head maximum across the
//             two halves by a shuffle, raises the running max only when a
//             tile exceeds it by more than 2^8 (probabilities stay <= 256)
//             and writes P (fp16); in the rare case of a raised max, the same
//             warps first rescale O in TMEM.
// Each query head is read from global memory and converted to fp16 (by the
// softmax and MMA warps) scaled by the power of two that puts its largest
// magnitude in [2^14, 2^15), which is exact for every bf16 row; the factor
// goes into that head's softmax scale.
// O for dims 0..255 accumulates in TMEM lanes 0..63 and dims 256..511 in
// lanes 64..127 of the same 256 columns: two MMAs with A = [P; 0] and
// A = [0; P] (zero rows leave the other half unchanged). P is stored once,
// between two zero blocks, and each MMA's A starts at a different block.
// TMEM: S at columns 0..63 and 64..127 (lanes 0-15 of each quadrant), O at
// 256..511 (512 allocated, one CTA per SM). Split-K partials (m, l,
// unnormalised O; O stored [dim/4][head][4] so the epilogue's stores and the
// merge's loads are contiguous across heads) are merged by the log-sum-exp
// merge kernel. In a layer-group call the kernel starts early (see the
// set-up): everything but the index reads and the global stores runs before
// the wait for the Top-K kernels. Every wait is bounded; after a timed-out
// wait the CTA reports CSA2_ERR_TIMEOUT and winds down (the warp groups
// decide to stop by barrier reductions, so no warp is left behind at a
// barrier).
#include <cstring>

#include "common.cuh"
#include "tcgen05.cuh"

namespace csa2 {

constexpr int kTD = 512;                  // head dim
constexpr int kTT = 64;                   // keys per tile
constexpr int kTThreads = 448;            // warps 0-3 softmax/correction, 4-11 producers, 12 S issue, 13 PV issue
constexpr int kSoftWarps = 4;
constexpr int kSoftThreads = 32 * kSoftWarps;
constexpr int kProdBase = kSoftThreads;   // first producer thread
constexpr int kProd = 256;                // producer threads
constexpr int kProdWarps = kProd / 32;
constexpr int kItems = kTT / kProdWarps;  // FP4 rows per producer thread and tile (one 16-channel group each)
constexpr int kMmaWarp = 12;             // issues S; allocates TMEM
constexpr int kPvWarp = 13;              // issues PV
static_assert(kPvWarp == kMmaWarp + 1 && kTThreads == 32 * (kPvWarp + 1), "warp roles: the last two warps issue MMAs");
constexpr int kRing = 8;                  // row-source ring: tiles j-2 .. j+3 may be live at once
constexpr uint32_t kTOcol = 256;

struct TcSmem {                           // offsets from a 1024-aligned base
  static constexpr int kQ = 0;                          // [8][64 heads][128 B]  64 KB
  static constexpr int kKV = kQ + 8 * 64 * 128;         // 2 x [8][64 keys][128 B]  128 KB
  static constexpr int kKVBytes = 8 * 64 * 128;
  static constexpr int kP = kKV + 2 * kKVBytes;         // Z | P | Z  3 x 8 KB
  static constexpr int kSrc = kP + 3 * 8192;            // int64 [kRing][64]: >= 0 FP4 row, -1 absent, <= -2 SWA row
  static constexpr int kMask = kSrc + kRing * kTT * 8;  // u32 [kRing][2] valid keys
  static constexpr int kFp4 = kMask + kRing * 8;        // u32 [kRing][2] keys that are FP4 rows
  static constexpr int kAlpha = kFp4 + kRing * 8;       // float[64]
  static constexpr int kL = kAlpha + 256;               // float[64]
  static constexpr int kM = kL + 256;                   // float[64]
  static constexpr int kQScale = kM + 256;              // float[64] 2^a of each query head
  static constexpr int kKeyB = kQScale + 256;           // u8 [kRing][64] SWA row scale exponents b
  static constexpr int kKeyFlag = kKeyB + kRing * 64;   // u32 [kRing]: some row of the tile is scaled
  static constexpr int kBar = kKeyFlag + kRing * 4;     // mbarriers (slots below)
  static constexpr int kMisc = kBar + 16 * 8;           // [0] tmem, [1..2] rescale flags, [3] abort
  static constexpr int kBytes = kMisc + 64 + 1024;      // + alignment slack
};
static_assert(TcSmem::kBytes <= 232448, "shared memory of the attention kernel");
static_assert(TcSmem::kBar % 8 == 0, "mbarrier alignment");
// mbarrier slots
constexpr int kBarKvFull = 0;             // [2] producers -> MMA (count kProd)
constexpr int kBarKvEmpty = 2;            // [2] PV done with a key buffer (tcgen05.commit)
constexpr int kBarSFull = 4;              // [2] S ready (tcgen05.commit)
constexpr int kBarPFull = 6;              // P ready (one arrive after the softmax group's barrier)
constexpr int kBarODone = 7;              // PV done (tcgen05.commit)
constexpr int kBarFin = 8;                // every MMA of the CTA done (tcgen05.commit)
constexpr int kBarQ = 9;                  // Q converted (every thread of the converting warps arrives)
constexpr int kBarSFree = 10;             // [2] S buffer read by the softmax (the PV warp arrives)
constexpr int kBarSFin = 12;
constexpr int kBarWin = 13;               // [2] window rows of key buffer i landed (TMA, expect_tx)              // every S MMA done (tcgen05.commit of the S warp)
constexpr int kQWarps = kSoftWarps + 2;   // the softmax warps and the two MMA warps convert Q

__device__ __forceinline__ uint32_t kt_off(int row, int chunk) {     // chunk = 16-byte unit of 8 dims
  return (uint32_t)((chunk >> 3) * 8192 + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

// Eight bf16 values (uint4) -> eight fp16 values, round-to-nearest, saturating.
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v) {
  uint32_t in[4] = {v.x, v.y, v.z, v.w}, o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = __uint_as_float(in[i] << 16), hi = __uint_as_float(in[i] & 0xFFFF0000u);
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(o[i]) : "f"(hi), "f"(lo));
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// The same, each value first multiplied by f (a power of two: exact), the
// two values of a pair by one fp32x2 multiply.
__device__ __forceinline__ uint4 bf16x8_to_f16x8_scaled(uint4 v, float f) {
  uint32_t in[4] = {v.x, v.y, v.z, v.w}, o[4];
  uint64_t f2;
  asm("mov.b64 %0, {%1, %1};" : "=l"(f2) : "f"(f));
#pragma unroll
  for (int i = 0; i < 4; ++i)
    asm("{\n .reg .b64 d;\n .reg .f32 a, b;\n mov.b64 d, {%1, %2};\n mul.rn.f32x2 d, d, %3;\n"
        " mov.b64 {a, b}, d;\n cvt.rn.satfinite.f16x2.f32 %0, b, a;\n}"
        : "=r"(o[i]) : "r"(in[i] << 16), "r"(in[i] & 0xFFFF0000u), "l"(f2));
  return make_uint4(o[0], o[1], o[2], o[3]);
}
// Largest magnitude bit pattern of 16 bf16 values (bit patterns of
// non-negative values order like the values).
__device__ __forceinline__ uint32_t bf16x16_max_mag(uint4 a, uint4 b) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t m = 0;                                   // two 16-bit lanes: the magnitudes' bit patterns
#pragma unroll
  for (int i = 0; i < 8; ++i) asm("max.u16x2 %0, %0, %1;" : "+r"(m) : "r"(w[i] & 0x7FFF7FFFu));
  return max(m & 0xFFFFu, m >> 16);
}
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((127 + e) << 23); }   // |e| <= 126

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
        "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
        "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]));
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
__device__ __forceinline__ uint4 ldg_hint_u4(const void* p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p), "l"(pol));
  return v;
}
__device__ __forceinline__ uint32_t ldg_hint_u8(const void* p, uint64_t pol) {
  uint16_t v;
  asm volatile("ld.global.nc.L2::cache_hint.u8 %0, [%1], %2;" : "=h"(v) : "l"(p), "l"(pol));
  return v;
}

// 2^((s0 - m) * sl) and 2^((s1 - m) * sl): the subtraction and the scaling as
// two fp32x2 operations (each lane rounds as the scalar form), then the
// hardware base-2 exponential (PTX ex2.approx.ftz: relative error about
// 2^-22, results below 2^-126 flushed to zero; P is rounded to fp16 next).
__device__ __forceinline__ void exp2_pair(uint32_t s0, uint32_t s1, uint64_t negm2, uint64_t sl2, float& p0,
                                          float& p1) {
  asm("{\n .reg .b64 d;\n .reg .f32 a, b;\n"
      " mov.b64 d, {%2, %3};\n add.rn.f32x2 d, d, %4;\n mul.rn.f32x2 d, d, %5;\n"
      " mov.b64 {a, b}, d;\n ex2.approx.ftz.f32 %0, a;\n ex2.approx.ftz.f32 %1, b;\n}"
      : "=f"(p0), "=f"(p1) : "r"(s0), "r"(s1), "l"(negm2), "l"(sl2));
}
// acc += the two fp16 values of h2, as one fp32x2 addition
__device__ __forceinline__ uint64_t add_half2(uint64_t acc, uint32_t h2) {
  asm("{\n .reg .b16 lo, hi;\n .reg .f32 a, b;\n .reg .b64 p;\n"
      " mov.b32 {lo, hi}, %1;\n cvt.f32.f16 a, lo;\n cvt.f32.f16 b, hi;\n"
      " mov.b64 p, {a, b};\n add.rn.f32x2 %0, %0, p;\n}"
      : "+l"(acc) : "r"(h2));
  return acc;
}
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ float hsum_f32x2(uint64_t a) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a));
  return lo + hi;
}

// One 2-D tensor map per layer over its SWA rows ([rows][1024 B], box 64
// rows x 128 B, 128-byte swizzle): one load of a dim block of 64 window rows
// lands in the key-buffer layout.
struct SwaMaps {
  CUtensorMap m[kMaxAttnLayers];
};

__global__ void __launch_bounds__(kTThreads, 1) k_sparse_attn_tc(
    const AttnLayers lay, const __grid_constant__ SwaMaps swa_maps, int H, const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
    int64_t kv_seq_stride, int64_t n_cap, const int32_t* __restrict__ idx, int k, int64_t swa_seq_stride, int W,
    int swa_tail, int rps, const int32_t* __restrict__ swa_len, float scale_log2, int splits, int tiles_per_split,
    float* __restrict__ part_o, float* __restrict__ part_ml, int32_t* st, uint64_t wait_ns, int fault, int early) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023) & ~1023u;
  unsigned char* sp = smem_raw + (base - raw);
  using L = TcSmem;
  float* sAlpha = reinterpret_cast<float*>(sp + L::kAlpha);
  float* sL = reinterpret_cast<float*>(sp + L::kL);
  float* sMx = reinterpret_cast<float*>(sp + L::kM);
  float* sQScale = reinterpret_cast<float*>(sp + L::kQScale);
  uint8_t* sKeyB = reinterpret_cast<uint8_t*>(sp + L::kKeyB);
  volatile uint32_t* sKeyFlag = reinterpret_cast<volatile uint32_t*>(sp + L::kKeyFlag);
  int64_t* sSrc = reinterpret_cast<int64_t*>(sp + L::kSrc);
  uint32_t* sMask = reinterpret_cast<uint32_t*>(sp + L::kMask);
  uint32_t* sFp4 = reinterpret_cast<uint32_t*>(sp + L::kFp4);
  volatile uint32_t* sMisc = reinterpret_cast<volatile uint32_t*>(sp + L::kMisc);
  auto bar = [&](int i) { return base + L::kBar + 8u * (uint32_t)i; };

  const int b = blockIdx.y, split = blockIdx.x, layer = blockIdx.z;
  const __nv_bfloat16* __restrict__ q = lay.q[layer];
  __nv_bfloat16* __restrict__ out = lay.out[layer];
  const int64_t unit = (int64_t)layer * gridDim.y + b;     // (layer, row) of the partials
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_tiles = (k + W + kTT - 1) / kTT;
  const int t_begin = split * tiles_per_split;
  const int t_end = min(t_begin + tiles_per_split, n_tiles);
  const int nt = max(t_end - t_begin, 0);

  // ---- set-up: barriers and the zero block touch no global memory and overlap
  //      the preceding kernel; then wait for it, allocate TMEM, load Q.
  //      Early launch (`early`, set when the preceding kernels of the same call
  //      write only the Top-K indices): Q, the SWA rows, swa_len and the main KV
  //      were complete before that call began, so everything but the index
  //      reads runs before the wait: Q, the SWA tiles, their S and softmax.
  //      Index reads wait (griddepcontrol.wait) in the threads that make
  //      them, and every thread waits before the first global store.
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(bar(kBarKvFull + i), kProd);
      tc::mbar_init(bar(kBarKvEmpty + i), 1);
      tc::mbar_init(bar(kBarSFull + i), 1);
    }
    tc::mbar_init(bar(kBarPFull), 1);
    tc::mbar_init(bar(kBarODone), 1);
    tc::mbar_init(bar(kBarFin), 1);
    tc::mbar_init(bar(kBarQ), 32 * kQWarps);
    tc::mbar_init(bar(kBarSFree), 1);
    tc::mbar_init(bar(kBarSFree + 1), 1);
    tc::mbar_init(bar(kBarSFin), 1);
    tc::mbar_init(bar(kBarWin), 1);
    tc::mbar_init(bar(kBarWin + 1), 1);
    tc::fence_barrier_init();
    sMisc[1] = 0;
    sMisc[2] = 0;
    sMisc[3] = 0;
    sMisc[4] = 0;                                             // window loads issued (bit per key buffer)
  }
  for (int e = tid; e < 3 * 8192 / 16; e += kTThreads)      // P, Z, P' zero
    *reinterpret_cast<uint4*>(sp + L::kP + e * 16) = make_uint4(0, 0, 0, 0);
  if (!early) pdl_wait();
  if (warp == kMmaWarp) {
    tc::tmem_alloc(base + L::kMisc, 512);
    tc::tmem_relinquish();
  }
  const uint64_t pol_keep = l2_evict_last(), pol_stream = l2_evict_first();
  // the SWA length is clamped without a branch, so nothing waits on its load
  const int slen_in = swa_len[b];
  // row b reads the caches of sequence b / rps; with rps > 1 the sequence's
  // SWA rows are linear and row b's window starts b % rps rows in
  const int64_t kv_row0 = (int64_t)(b / rps) * kv_seq_stride;
  const int64_t swa_row0 = (int64_t)(b / rps) * swa_seq_stride + (b % rps);
  const int slen = min(max(slen_in, 0), W);
  // Window tiles (local tiles 0 .. j_win - 1 hold window slots r < W): their
  // rows come by TMA, one dim block (64 rows x 128 B) per load, into the key
  // buffer of the tile, both issued here. Rows past the window or the buffer
  // are zeroed or overwritten by the producers after the load.
  const int j_win = min(max((W + kTT - 1) / kTT - t_begin, 0), 2);
  auto window_load = [&](int j) {                             // one thread
    const int buf = j & 1;
    const int64_t y = swa_row0 + (swa_tail ? W - slen : 0) + (int64_t)(t_begin + j) * kTT;
    atomicOr(const_cast<uint32_t*>(&sMisc[4]), 1u << buf);
    tc::mbar_expect_tx(bar(kBarWin + buf), 8 * 8192);
#pragma unroll
    for (int d = 0; d < 8; ++d)
      tc::tma_load_2d(base + L::kKV + buf * L::kKVBytes + d * 8192, &swa_maps.m[layer], d * 128, (int32_t)y,
                      bar(kBarWin + buf));
  };
  if (tid == 0 && j_win > 0 && nt > 0) window_load(0);
  if (tid == 0 && j_win > 1 && nt > 1) window_load(1);

  // Row sources of tile j (called by a whole warp pair: row p of the tile).
  // Key slot r < W is SWA row r (present if r < slen); slot W + i is Top-K entry i.
  auto row_sources = [&](int j, int p) {
    const int slot = j % kRing;
    const int r = (t_begin + j) * kTT + p;
    int64_t src = -1;
    if (r < W) {
      if (r < slen) src = -2 - (swa_row0 + (swa_tail ? W - slen : 0) + r);
    } else if (r - W < k) {
      const int32_t pos = idx[(int64_t)b * k + (r - W)];
      if (pos >= 0 && pos < n_cap) src = kv_row0 + pos;
      else if (pos >= n_cap) report(st, CSA2_ERR_DEVICE_BOUNDS);
    }
    sSrc[slot * kTT + p] = src;
    sKeyB[slot * kTT + p] = 0;
    if (p == 0) sKeyFlag[slot] = 0;
    const uint32_t valid = __ballot_sync(0xffffffffu, src != -1);
    const uint32_t fp4 = __ballot_sync(0xffffffffu, src >= 0);
    if ((p & 31) == 0) {
      sMask[slot * 2 + (p >> 5)] = valid;
      sFp4[slot * 2 + (p >> 5)] = fp4;
    }
  };
  // tiles 0 .. j_idx - 1 hold SWA rows only and read no index; in an early
  // launch the producers take the row sources of tiles j_idx .. 2 after the wait
  const int j_idx = early ? min(max(W / kTT - t_begin, 0), 3) : 3;
  if (tid < 64) {
    for (int j = 0; j < j_idx && j < nt; ++j) row_sources(j, tid);
  }
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = sMisc[0];
  pdl_trigger();                              // TMEM is held: the next kernel may start launching
  // Q -> fp16, one warp per head: scaled by 2^-a so that the head's largest
  // magnitude lies in [2^14, 2^15) (heads >= H and all-zero heads: a = 0).
  // The softmax warps and the two MMA warps read Q's rows from global memory
  // (four heads of a warp in flight) and write them converted, while the
  // producers start on the window tiles; S and the softmax wait on kBarQ.
  if (warp < kSoftWarps || warp >= kMmaWarp) {
    const int h_first = warp < kSoftWarps ? warp : kSoftWarps + (warp - kMmaWarp);
#pragma unroll 1
    for (int h0 = h_first; h0 < 64; h0 += 4 * kQWarps) {
      uint4 v[4][2];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int h = h0 + u * kQWarps;
        v[u][0] = make_uint4(0, 0, 0, 0);
        v[u][1] = v[u][0];
        if (h < H) {                                          // H <= 64
          const __nv_bfloat16* qrow = q + ((int64_t)b * H + h) * kTD;
          v[u][0] = ldg_hint_u4(qrow + lane * 8, pol_stream);
          v[u][1] = ldg_hint_u4(qrow + (lane + 32) * 8, pol_stream);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int h = h0 + u * kQWarps;
        if (h >= 64) break;                                   // warp-uniform
        const uint32_t mx = __reduce_max_sync(0xffffffffu, bf16x16_max_mag(v[u][0], v[u][1]));
        const int a = mx == 0 ? 0 : min(max((int)(mx >> 7) - 127 - 14, -100), 100);
        const float f = pow2f(-a);
        *reinterpret_cast<uint4*>(sp + L::kQ + kt_off(h, lane)) = bf16x8_to_f16x8_scaled(v[u][0], f);
        *reinterpret_cast<uint4*>(sp + L::kQ + kt_off(h, lane + 32)) = bf16x8_to_f16x8_scaled(v[u][1], f);
        if (lane == 0) sQScale[h] = pow2f(a);
      }
    }
    tc::fence_async_smem();
    tc::mbar_arrive(bar(kBarQ));
  }

  // softmax threads (warps 0-3): head 16 warp + (lane & 15), key columns
  // 32 (lane >> 4) .. + 31 of a tile; l_run sums the thread's column half,
  // m_run is the same in both halves, l_tot is the head's total
  float m_run = -INFINITY, l_run = 0.f, l_tot = 0.f;

  if (warp >= kSoftWarps && warp < kMmaWarp) {
    // ================= producers =================
    const int p = tid - kProdBase, pw = p >> 5;
    // this thread's FP4 items of a tile: rows 8 i + (lane & 7) (i < kItems),
    // 16-channel group 4 pw + (lane >> 3). Per item a warp writes one 64-dim
    // block of eight consecutive rows, so the eight lanes of a store
    // wavefront hit eight distinct swizzle slots. Two register sets hold
    // tiles j and j + 1 in flight (set A even tiles, set B odd ones).
    const int rl = lane & 7, g = 4 * pw + (lane >> 3);
    uint2 cwA[kItems], cwB[kItems];
    uint32_t sbA[kItems], sbB[kItems];
    auto prefetch = [&](int j, uint2* cw, uint32_t* sb) {
      const int64_t* src = sSrc + (j % kRing) * kTT;
#pragma unroll
      for (int i = 0; i < kItems; ++i) {
        const int64_t s = src[8 * i + rl];
        cw[i] = make_uint2(0u, 0u);
        sb[i] = 0u;
        if (s >= 0) {
          cw[i] = ldg_hint_u2(codes + s * 256 + g * 8, pol_keep);
          sb[i] = ldg_hint_u8(scales + s * 32 + g, pol_keep);
        }
      }
    };
    // One tile, its FP4 rows in set (cw, sb), the other set (cwo, sbo):
    // returns false when the group stops. An early launch first produces its
    // SWA-only tiles 0 .. j0 - 1 (`lite`: no index work after them); at tile
    // j0 it waits for the preceding kernel and takes the row sources of tiles
    // j0 .. j0 + 2. At tile j0, tiles j0 and j0 + 1 are prefetched. The loop
    // below inlines this code twice, once per register set (as few copies as
    // static register indexing allows: the instruction caches are a limit).
    const int j0 = early ? min(j_idx, nt) : 0;
    auto produce = [&](int j, uint2* cw, uint32_t* sb, uint2* cwo, uint32_t* sbo) -> bool {
      const bool lite = j < j0;
      if (j == j0) {
        if (early) {
          if (p < 64) {
            pdl_wait();
            for (int jj = j0; jj < j0 + 3 && jj < nt; ++jj) row_sources(jj, p);
          }
          named_sync(kNbProd, kProd);
        }
        prefetch(j, cw, sb);
        if (j + 1 < nt) prefetch(j + 1, cwo, sbo);
      }
      if (named_or(kNbProd, kProd, sMisc[3] != 0)) return false;
      const int buf = j & 1, slot = j % kRing;
      unsigned char* kvp = sp + L::kKV + buf * L::kKVBytes;
      // the buffer is free once PV(j - 2) has finished
      if (j >= 2 && !tc::mbar_wait(bar(kBarKvEmpty + buf), ((j >> 1) - 1) & 1, wait_ns)) {
        report(st, CSA2_ERR_TIMEOUT);
        sMisc[3] = 1;
      }
      // a window tile's rows land by TMA before anything else is written there
      if (j < j_win) {
        if (!tc::mbar_wait(bar(kBarWin + buf), 0, wait_ns)) {
          report(st, CSA2_ERR_TIMEOUT);
          sMisc[3] = 1;
        }
      }
      const uint64_t valid = (uint64_t)sMask[slot * 2] | ((uint64_t)sMask[slot * 2 + 1] << 32);
      const uint64_t fp4 = (uint64_t)sFp4[slot * 2] | ((uint64_t)sFp4[slot * 2 + 1] << 32);
      const uint64_t swa_rows = valid & ~fp4;
      // absent rows: zero. Warp pw takes rows pw + 8 m, a lane two 16-byte chunks.
      if (~valid != 0) {
        for (int r = pw; r < kTT; r += kProdWarps) {
          if (!((valid >> r) & 1))
            for (int c = lane; c < 64; c += 32) *reinterpret_cast<uint4*>(kvp + kt_off(r, c)) = make_uint4(0, 0, 0, 0);
        }
      }
      // FP4 rows of this tile (in registers): one 16-channel group per item
#pragma unroll
      for (int i = 0; i < kItems; ++i) {
        const int r = 8 * i + rl;
        if (!((fp4 >> r) & 1)) continue;
        uint32_t sh2;                                           // scale as f16x2 {s, s}
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(sh2) : "h"((uint16_t)(sb[i] | (sb[i] << 8))));
        uint32_t o[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint32_t byte = ((u < 4 ? cw[i].x : cw[i].y) >> (8 * (u & 3))) & 0xFF;
          const uint32_t h2 = e2m1x2_to_f16x2(byte);
          asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[u]) : "r"(h2), "r"(sh2));
        }
        *reinterpret_cast<uint4*>(kvp + kt_off(r, 2 * g)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(kvp + kt_off(r, 2 * g + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
      }
      // SWA rows: bf16 -> fp16 in place (each lane two 16-byte chunks of a
      // row). A row whose largest magnitude reaches 2^16 (beyond fp16) is
      // scaled by 2^-b first (b = its binary exponent - 15, at most 7: rows
      // reaching 2^23 saturate and are reported); b goes to the softmax
      // through kKeyB.
      if (swa_rows) {
#pragma unroll 2
        for (int r = pw; r < kTT; r += kProdWarps) {
          if (!((swa_rows >> r) & 1)) continue;                 // warp-uniform
          uint4* p0 = reinterpret_cast<uint4*>(kvp + kt_off(r, lane));
          uint4* p1 = reinterpret_cast<uint4*>(kvp + kt_off(r, lane + 32));
          const uint4 v0 = *p0, v1 = *p1;
          const int e = (int)(__reduce_max_sync(0xffffffffu, bf16x16_max_mag(v0, v1)) >> 7) - 127;
          int bsh = e >= 16 ? e - 15 : 0;
          if (bsh > 7) {
            if (lane == 0) report(st, CSA2_ERR_DEVICE_RANGE);
            bsh = 7;
          }
          if (bsh == 0) {                                       // the common case: no scale
            *p0 = bf16x8_to_f16x8(v0);
            *p1 = bf16x8_to_f16x8(v1);
          } else {
            const float f = pow2f(-bsh);
            *p0 = bf16x8_to_f16x8_scaled(v0, f);
            *p1 = bf16x8_to_f16x8_scaled(v1, f);
          }
          if (bsh != 0 && lane == 0) {
            sKeyB[slot * kTT + r] = (uint8_t)bsh;
            sKeyFlag[slot] = 1;
          }
        }
      }
      tc::fence_async_smem();
      // fault injection (tests of the bounded waits): the last tile is never signalled
      if (!(fault == 1 && j == nt - 1)) tc::mbar_arrive(bar(kBarKvFull + buf));
      if (lite) return true;
      if (j + 2 < nt) prefetch(j + 2, cw, sb);
      // the row sources of tile j + 3 last: the latency of their index loads
      // then overlaps the next tile's wait for its key buffer
      if (j + 3 < nt && p < 64) {
        pdl_wait();                                           // returns at once after the first
        row_sources(j + 3, p);
      }
      return true;
    };
    for (int j = 0; j < nt; j += 2) {
      if (!produce(j, cwA, sbA, cwB, sbB)) break;
      if (j + 1 < nt && !produce(j + 1, cwB, sbB, cwA, sbA)) break;
    }
  } else if (warp < kSoftWarps) {
    // ================= softmax / O correction =================
    // S(t) is an M = 64 accumulator: head h in TMEM lane 32 (h / 16) + h % 16.
    // Warp q reads heads 16 q .. + 15 with the 16x32bx2 shape: lanes 0-15 get
    // key columns 0..31, lanes 16-31 columns 32..63 of the same heads, so the
    // two halves of a head exchange their maxima and sums by one shuffle.
    // Warps 0-3 also rescale O (TMEM lanes 0-127) when a head raised its
    // reference.
    const int h = 16 * warp + (lane & 15);
    const int half = lane >> 4;
    if (!tc::mbar_wait(bar(kBarQ), 0, wait_ns)) { report(st, CSA2_ERR_TIMEOUT); sMisc[3] = 1; }
    const float sl = scale_log2 * sQScale[h];               // the head's query was scaled by 2^-a
    for (int j = 0; j < nt; ++j) {
      if (named_or(kNbSoft, kSoftThreads, sMisc[3] != 0)) break;
      const int sbuf = j & 1;
      uint32_t r[32];
      bool ok = tc::mbar_wait(bar(kBarSFull + sbuf), (j >> 1) & 1, wait_ns);
      ok = tc::mbar_wait(bar(kBarKvFull + sbuf), (j >> 1) & 1, wait_ns) && ok;     // orders the mask reads
      tc::tc_fence_after();
      tmem_ld_16x32bx2_32(tmem + ((uint32_t)(32 * warp) << 16) + 64u * sbuf, r);
      tc::tmem_ld_wait();
      const uint32_t vm = sMask[(j % kRing) * 2 + half];
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (vm != 0xffffffffu) {
#pragma unroll
        for (int x = 0; x < 32; ++x)
          if (!((vm >> x) & 1u)) r[x] = __float_as_uint(-INFINITY);
      }
      // SWA rows that were scaled by 2^-b: their scores times 2^b (exact)
      const bool kscaled = sKeyFlag[j % kRing] != 0;         // the same for every thread
      uint32_t bw[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (kscaled) {
        const uint32_t* bsrc = reinterpret_cast<const uint32_t*>(sKeyB + (j % kRing) * kTT + 32 * half);
#pragma unroll
        for (int i = 0; i < 8; ++i) bw[i] = bsrc[i];
#pragma unroll
        for (int x = 0; x < 32; ++x)
          r[x] = __float_as_uint(__uint_as_float(r[x]) * pow2f((int)((bw[x >> 2] >> (8 * (x & 3))) & 0xFF)));
      }
#pragma unroll
      for (int x = 0; x < 32; ++x) m4[x & 3] = fmaxf(m4[x & 3], __uint_as_float(r[x]));
      float mh = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      mh = fmaxf(mh, __shfl_xor_sync(0xffffffffu, mh, 16));
      // The running maximum m_run is kept in score units and every exponent
      // is formed as (s - m_run) * scale: the subtraction is exact near the
      // maximum, so the largest key gets exactly 1 however large the logits
      // (forming s * scale - m_run * scale instead loses the rounding error of
      // m_run * scale, which for huge logits overflows exp2). The reference is
      // raised only when a tile exceeds it by more than 8 in log2 units
      // (probabilities stay <= 256).
      float alpha = 1.f;
      if (mh > m_run && (m_run == -INFINITY || (mh - m_run) * sl > 8.f)) {
        alpha = (m_run == -INFINITY) ? 0.f : exp2f((m_run - mh) * sl);
        m_run = mh;
      }
      const float mref = (m_run == -INFINITY) ? 0.f : m_run;
      // P and O are free once PV(j - 1) has finished
      if (j > 0) ok = tc::mbar_wait(bar(kBarODone), (j - 1) & 1, wait_ns) && ok;
      if (!ok) { report(st, CSA2_ERR_TIMEOUT); sMisc[3] = 1; }
      uint64_t sum2[4] = {0ull, 0ull, 0ull, 0ull};            // pairs of fp32 partial sums
      const uint64_t negm2 = pack_f32x2(-mref, -mref), sl2 = pack_f32x2(sl, sl);
      unsigned char* prow = sp + L::kP + 8192 + h * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int x = 8 * c + 2 * u;
          float p0, p1;
          exp2_pair(r[x], r[x + 1], negm2, sl2, p0, p1);
          if (kscaled) {                      // a scaled row's value enters PV as 2^-b v: its P as 2^b P
            const int b0 = (int)((bw[x >> 2] >> (8 * (x & 3))) & 0xFF);
            const int b1 = (int)((bw[(x + 1) >> 2] >> (8 * ((x + 1) & 3))) & 0xFF);
            const __half2 pv = __floats2half2_rn(p0 * pow2f(b0), p1 * pow2f(b1));
            const float2 f = __half22float2(pv);
            float lo, hi;
            asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(sum2[u]));
            sum2[u] = pack_f32x2(lo + f.x * pow2f(-b0), hi + f.y * pow2f(-b1));
            pk[u] = *reinterpret_cast<const uint32_t*>(&pv);
          } else {
            const __half2 pv = __floats2half2_rn(p0, p1);
            pk[u] = *reinterpret_cast<const uint32_t*>(&pv);
            sum2[u] = add_half2(sum2[u], pk[u]);
          }
        }
        const uint4 v4 = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        const int sw = (((4 * half + c) ^ (h & 7)) << 4);
        if (h < H) {
          *reinterpret_cast<uint4*>(prow + sw) = v4;               // rows 0..63 of [P; Z], 64..127 of [Z; P]
        }
      }
      l_run = l_run * alpha + ((hsum_f32x2(sum2[0]) + hsum_f32x2(sum2[1])) + (hsum_f32x2(sum2[2]) + hsum_f32x2(sum2[3])));
      if (half == 0) sAlpha[h] = alpha;
      if (alpha != 1.f && j > 0) sMisc[1 + (j & 1)] = 1;
      named_sync(kNbSoft, kSoftThreads);
      // -- rescale O when some head raised its reference (rare)
      if (sMisc[1 + (j & 1)]) {
        tc::tc_fence_after();
        const float a = sAlpha[(32 * warp + lane) & 63];
        const uint32_t ta = tmem + ((uint32_t)(32 * warp) << 16) + kTOcol;
        for (int c = 0; c < 256; c += 32) {
          uint32_t o[32];
          tc::tmem_ld32(ta + c, o);
          tc::tmem_ld_wait();
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * a);
          tmem_st32(ta + c, o);
        }
        tmem_st_wait();
      }
      tc::fence_async_smem();
      tc::tc_fence_before();
      named_sync(kNbSoft, kSoftThreads);
      if (tid == 0) {
        sMisc[1 + (j & 1)] = 0;
        tc::mbar_arrive(bar(kBarPFull));
      }
    }
    l_tot = l_run + __shfl_xor_sync(0xffffffffu, l_run, 16);
  } else {
    // ================= MMA issue (lane 0 of warps 12 and 13) =================
    if (lane == 0) {
      const uint32_t idesc_s = tc::instr_desc(tc::kFmtF16, tc::kFmtF16, 0, 0, 64, kTT);   // heads: M = 64
      const uint32_t idesc_o = tc::instr_desc(tc::kFmtF16, tc::kFmtF16, 0, 1, 128, 256);
      auto issue_pv = [&](int j) {
        const uint32_t kv = base + L::kKV + (j & 1) * L::kKVBytes;
#pragma unroll
        for (int ks = 0; ks < kTT / 16; ++ks) {
          const uint64_t a0 = tc::smem_desc(base + L::kP + 8192 + ks * 32, 16, 1024, tc::kSwizzle128B);   // [P; Z]
          const uint64_t a1 = tc::smem_desc(base + L::kP + ks * 32, 16, 1024, tc::kSwizzle128B);          // [Z; P]
          const uint64_t b0 = tc::smem_desc(kv + ks * 2048, 8192, 1024, tc::kSwizzle128B);
          const uint64_t b1 = tc::smem_desc(kv + 4 * 8192 + ks * 2048, 8192, 1024, tc::kSwizzle128B);
          tc::mma_f16(tmem + kTOcol, a0, b0, idesc_o, (j > 0 || ks > 0) ? 1u : 0u);
          tc::mma_f16(tmem + kTOcol, a1, b1, idesc_o, 1u);
        }
        tc::mma_commit(bar(kBarODone));
        tc::mma_commit(bar(kBarKvEmpty + (j & 1)));
      };
      auto issue_s = [&](int j) {
        const uint32_t kv = base + L::kKV + (j & 1) * L::kKVBytes;
#pragma unroll 4
        for (int ks = 0; ks < kTD / 16; ++ks) {
          const uint32_t off = (ks >> 2) * 8192 + (ks & 3) * 32;
          const uint64_t ad = tc::smem_desc(base + L::kQ + off, 16, 1024, tc::kSwizzle128B);
          const uint64_t bd = tc::smem_desc(kv + off, 16, 1024, tc::kSwizzle128B);
          tc::mma_f16(tmem + 64u * (j & 1), ad, bd, idesc_s, ks > 0 ? 1u : 0u);
        }
        tc::mma_commit(bar(kBarSFull + (j & 1)));
      };
      // Two issuers: this warp issues S(js) as soon as its key tile is ready
      // and the softmax has read S(js - 2) from the same TMEM buffer; the PV
      // warp issues PV(jp) as soon as P(jp) is ready. PV no longer waits
      // behind the issue of a 32-instruction S.
      if (warp == kMmaWarp) {
        bool ok = tc::mbar_wait(bar(kBarQ), 0, wait_ns);
        for (int js = 0; ok && js < nt; ++js) {
          ok = tc::mbar_wait(bar(kBarKvFull + (js & 1)), (js >> 1) & 1, wait_ns);
          if (ok && js >= 2) ok = tc::mbar_wait(bar(kBarSFree + (js & 1)), ((js >> 1) - 1) & 1, wait_ns);
          if (!ok || sMisc[3]) { ok = false; break; }
          tc::tc_fence_after();
          issue_s(js);
        }
        if (!ok) { report(st, CSA2_ERR_TIMEOUT); sMisc[3] = 1; }
        // every S MMA has completed before TMEM is read or freed
        tc::mma_commit(bar(kBarSFin));
        if (!tc::mbar_wait(bar(kBarSFin), 0, wait_ns)) { report(st, CSA2_ERR_TIMEOUT); sMisc[3] = 1; }
      } else {
        bool ok = true;
        int jp = 0;
        for (; jp < nt; ++jp) {
          ok = tc::mbar_wait(bar(kBarPFull), jp & 1, wait_ns);
          if (!ok || sMisc[3]) { ok = false; break; }
          tc::tc_fence_after();
          tc::mbar_arrive(bar(kBarSFree + (jp & 1)));   // the softmax read S(jp) before P(jp) was ready
          issue_pv(jp);
        }
        if (!ok) { report(st, CSA2_ERR_TIMEOUT); sMisc[3] = 1; }
        // every PV MMA has completed before TMEM is read or freed
        tc::mma_commit(bar(kBarFin));
        if (!tc::mbar_wait(bar(kBarFin), 0, wait_ns)) { report(st, CSA2_ERR_TIMEOUT); sMisc[3] = 1; }
        if (jp < nt) sMisc[3] = 1;
      }
    }
    __syncwarp();
  }
  __syncthreads();
  tc::tc_fence_after();
  if (early) pdl_wait();                        // before the first global store
  const bool have_o = nt > 0 && sMisc[3] == 0;  // uniform: read after the barrier
  if ((slen_in < 0 || slen_in > W) && split == 0 && tid == 0) report(st, CSA2_ERR_DEVICE_BOUNDS);
  if (warp < kSoftWarps && lane < 16) {
    const int h = 16 * warp + lane;
    sL[h] = have_o ? l_tot : 0.f;
    // the partials carry the maximum in log2 units (the merge's domain)
    sMx[h] = (have_o && m_run != -INFINITY) ? m_run * (scale_log2 * sQScale[h]) : -INFINITY;
  }
  __syncthreads();
  if (warp < 8) {
    // ---- epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31 (row r holds
    // head r % 64, dims 0..255 for r < 64 and 256..511 above) and the column
    // half w / 4 of O's 256 columns. tcgen05.ld is warp-collective, so whole
    // warps load; lanes of heads >= H only skip the stores.
    const int lg = warp & 3, chalf = warp >> 2;
    const int row = 32 * lg + lane, h = row & 63;
    const bool live = h < H;
    const uint32_t ta = tmem + ((uint32_t)(32 * lg) << 16) + kTOcol + 128 * chalf;
    const float lsum = sL[h];
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    const int dbase = (row >> 6) * 256 + 128 * chalf;
#pragma unroll 1
    for (int c = 0; c < 128; c += 64) {
      uint32_t r[64];
      if (have_o) {
        tc::tmem_ld32(ta + c, r);
        tc::tmem_ld32(ta + c + 32, r + 32);
        tc::tmem_ld_wait();
      } else {
#pragma unroll
        for (int x = 0; x < 64; ++x) r[x] = 0u;
      }
      if (!live) continue;
      const int dim0 = dbase + c;
      if (splits == 1) {
        __nv_bfloat16* o = out + ((int64_t)b * H + h) * kTD + dim0;
#pragma unroll
        for (int x = 0; x < 64; x += 8) {
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
        // partial O layout [b][split][dim / 4][H][4]: a warp stores 32 heads' float4 contiguously
        float* o = part_o + (((unit * splits + split) * (kTD / 4) + dim0 / 4) * H + h) * 4;
#pragma unroll
        for (int x = 0; x < 64; x += 4)
          *reinterpret_cast<float4*>(o + (int64_t)(x / 4) * H * 4) =
              make_float4(__uint_as_float(r[x]), __uint_as_float(r[x + 1]), __uint_as_float(r[x + 2]),
                          __uint_as_float(r[x + 3]));
      }
    }
    if (live && splits > 1 && row < 64 && chalf == 0) {
      const int64_t pidx = (unit * splits + split) * H + h;
      part_ml[pidx * 2 + 0] = sMx[h];
      part_ml[pidx * 2 + 1] = sL[h];
    }
  }
  // no window load may still be in flight when the CTA exits (a group that
  // stopped early may not have waited for one)
  if (tid == 0) {
    const uint32_t issued = sMisc[4];
    for (int i = 0; i < 2; ++i)
      if ((issued >> i) & 1) (void)tc::mbar_wait(bar(kBarWin + i), 0, wait_ns);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

int attn_tc_init_attributes() {
  const cudaError_t e =
      cudaFuncSetAttribute(k_sparse_attn_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, TcSmem::kBytes);
  note_cuda_error(e);
  return e == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA;
}

int launch_sparse_attn_tc(const AttnLayers& lay, int L, int B, int H, const uint8_t* codes, const uint8_t* scales,
                          int64_t kv_seq_stride, int64_t n_cap, const int32_t* idx, int k, int64_t swa_seq_stride,
                          int W, int swa_tail, int rps, const int32_t* swa_len, float softmax_scale, float* part_o,
                          float* part_ml, int splits, int tps, int32_t* st, uint64_t wait_ns, int fault,
                          int early, cudaStream_t s) {
  dim3 grid((unsigned)splits, (unsigned)B, (unsigned)L);
  // each layer's window rows as a 2-D tensor up to the last row's window end
  SwaMaps maps;
  memset(&maps, 0, sizeof(maps));
  if (W > 0) {
    const uint64_t rows = (uint64_t)((B - 1) / rps) * (uint64_t)swa_seq_stride + (uint64_t)((B - 1) % rps) + (uint64_t)W;
    for (int l = 0; l < L; ++l)
      if (!make_tmap_rows128(&maps.m[l], lay.swa[l], rows, (uint64_t)kTD * 2, kTT)) return CSA2_ERR_CUDA;
  }
  const cudaError_t e = launch_pdl(k_sparse_attn_tc, grid, dim3(kTThreads), TcSmem::kBytes, s, lay, maps, H, codes, scales,
                                   kv_seq_stride, n_cap, idx, k, swa_seq_stride, W, swa_tail, rps, swa_len,
                                   softmax_scale * 1.4426950408889634f, splits, tps, part_o, part_ml, st, wait_ns,
                                   fault, early);
  count_launch();
  return launch_status(e);
}

}  // namespace csa2
