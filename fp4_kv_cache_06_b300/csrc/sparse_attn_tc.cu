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
// Per tile of 64 key slots (gathered rows first, then SWA rows):
//   gather  : cp.async of the 288-byte FP4 rows, prefetched one tile ahead
//             (SWA rows are converted into the key tile directly);
//   dequant : E2M1 -> f16x2 (hardware convert) times the E4M3 scale as a
//             packed f16 multiply (the product, <= 6 significant bits in
//             2^-10 .. 2688, is exact in fp16), written in the K-major
//             128-byte-swizzle layout [dim/64][key][128 B]. The tile operands
//             are fp16: Q and the SWA rows are converted from bf16 once
//             (exact for magnitudes 2^-14 .. 65504; smaller values keep
//             2^-24 absolute accuracy, larger ones saturate);
//   S = Q K^T : tcgen05.mma kind::f16, M = 128 (heads padded from <= 64),
//             N = 64 keys, K = 512 in 32 steps, fp32 in TMEM columns 0..63;
//   softmax : one thread per head reads its S row from TMEM; the running
//             max is only raised when a tile exceeds it by more than 2^8
//             (probabilities stay <= 256), so O is rescaled rarely;
//   O += P V: the same key tile read as the MN-major B operand. O for dims
//             0..255 accumulates in TMEM lanes 0..63 and dims 256..511 in
//             lanes 64..127 of the same 256 columns: two MMAs with A = [P; 0]
//             and A = [0; P] (zero rows leave the other half unchanged).
// TMEM: S at columns 0..63, O at 256..511 (512 allocated, one CTA per SM).
// Split-K partials (m, l, unnormalised O; O stored [dim/4][head][4] so the
// epilogue's stores and the merge's loads are contiguous across heads) are
// merged by the log-sum-exp merge kernel. Waits on MMA completion are bounded.
#include "common.cuh"
#include "tcgen05.cuh"

namespace csa2 {

constexpr int kTD = 512;                  // head dim
constexpr int kTT = 64;                   // keys per tile
constexpr int kTThreads = 256;
constexpr uint32_t kTScol = 0, kTOcol = 256;

struct TcSmem {                           // offsets from a 1024-aligned base
  static constexpr int kQ = 0;                          // [8][64 heads][128 B]  64 KB
  static constexpr int kKV = kQ + 8 * 64 * 128;         // [8][64 keys][128 B]   64 KB
  static constexpr int kP = kKV + 8 * 64 * 128;         // P | Z | P'  3 x 8 KB
  static constexpr int kNS = 3;                         // FP4 staging ring: prefetch two tiles ahead
  static constexpr int kStage = kP + 3 * 8192;          // kNS x (64 x 256 codes + 64 x 32 scales)
  static constexpr int kStageBytes = kTT * 288;
  static constexpr int kAlpha = kStage + kNS * kStageBytes;  // float[64]
  static constexpr int kL = kAlpha + 256;                    // float[64]
  static constexpr int kM = kL + 256;                        // float[64]
  static constexpr int kSrc = kM + 256;                      // int64[kNS][64]
  static constexpr int kKind = kSrc + kNS * kTT * 8;         // int32[kNS][64]
  static constexpr int kMask = kKind + kNS * kTT * 4;        // u32[kNS][2] valid keys, then u32[kNS][2] special rows
  static constexpr int kBar = kMask + 64;                    // 2 mbarriers
  static constexpr int kMisc = kBar + 16;                    // tmem addr, flags
  static constexpr int kBytes = kMisc + 64 + 1024;           // + alignment slack
};

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

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
        "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
        "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]));
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__global__ void __launch_bounds__(kTThreads, 1) k_sparse_attn_tc(
    const __nv_bfloat16* __restrict__ q, int H, const uint8_t* __restrict__ codes,
    const uint8_t* __restrict__ scales, int64_t kv_seq_stride, int64_t n_cap, const int32_t* __restrict__ idx,
    int k, const __nv_bfloat16* __restrict__ swa, int64_t swa_seq_stride, int W, int swa_tail,
    const int32_t* __restrict__ swa_len, float scale_log2, int splits, int tiles_per_split,
    __nv_bfloat16* __restrict__ out, float* __restrict__ part_o, float* __restrict__ part_ml, int32_t* st) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023) & ~1023u;
  unsigned char* sp = smem_raw + (base - raw);
  using L = TcSmem;
  float* sAlpha = reinterpret_cast<float*>(sp + L::kAlpha);
  float* sL = reinterpret_cast<float*>(sp + L::kL);
  float* sMx = reinterpret_cast<float*>(sp + L::kM);
  int64_t* sSrc = reinterpret_cast<int64_t*>(sp + L::kSrc);
  int32_t* sKind = reinterpret_cast<int32_t*>(sp + L::kKind);
  volatile uint32_t* sMisc = reinterpret_cast<volatile uint32_t*>(sp + L::kMisc);   // [0] tmem, [1] rescale, [2] abort
  const uint32_t bar_s = base + L::kBar, bar_o = base + L::kBar + 8;

  const int b = blockIdx.y, split = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint64_t pol_keep = l2_evict_last(), pol_stream = l2_evict_first();
  const int n_tiles = (k + W + kTT - 1) / kTT;
  const int t_begin = split * tiles_per_split;
  const int t_end = min(t_begin + tiles_per_split, n_tiles);
  // ---- set-up: barriers and the zero block touch no global memory and overlap
  //      the preceding kernel; then wait for it, allocate TMEM, load the Q tile
  //      and the row sources of the first tiles
  if (tid == 0) {
    tc::mbar_init(bar_s, 1);
    tc::mbar_init(bar_o, 1);
    tc::fence_barrier_init();
    sMisc[1] = 0;
    sMisc[2] = 0;
  }
  for (int e = tid; e < 3 * 8192 / 16; e += kTThreads)      // P, Z, P' zero
    *reinterpret_cast<uint4*>(sp + L::kP + e * 16) = make_uint4(0, 0, 0, 0);
  pdl_wait();
  if (warp == 0) {
    tc::tmem_alloc(base + L::kMisc, 512);
    tc::tmem_relinquish();
  }
  for (int e = tid; e < 64 * 64; e += kTThreads) {          // Q rows (bf16) staged in the key tile
    const int h = e >> 6, c = e & 63;
    if (h < H) cp_async16_hint(base + L::kKV + kt_off(h, c), q + ((int64_t)b * H + h) * kTD + c * 8, pol_stream);
  }
  // the SWA length is clamped without a branch, so nothing waits on its load
  // before the row-index loads are issued
  const int slen_in = swa_len[b];
  const int slen = min(max(slen_in, 0), W);

  auto row_sources = [&](int tile, int buf) {
    if (tid < kTT) {
      const int j = tile * kTT + tid;
      int64_t src = -1;
      int kind = 0;
      if (j < k) {
        const int32_t p = idx[(int64_t)b * k + j];
        if (p >= 0 && p < n_cap) src = (int64_t)b * kv_seq_stride + p;
        else if (p >= n_cap) report(st, CSA2_ERR_DEVICE_BOUNDS);
      } else if (j - k < slen) {
        src = (int64_t)b * swa_seq_stride + (swa_tail ? W - slen : 0) + (j - k);
        kind = 1;
      }
      sSrc[buf * kTT + tid] = src;
      sKind[buf * kTT + tid] = kind;
      const uint32_t valid = __ballot_sync(0xffffffffu, src >= 0);
      const uint32_t swa_or_hole = __ballot_sync(0xffffffffu, src < 0 || kind == 1);
      if ((tid & 31) == 0) {
        reinterpret_cast<uint32_t*>(sp + L::kMask)[buf * 2 + (tid >> 5)] = valid;
        reinterpret_cast<uint32_t*>(sp + L::kMask + 32)[buf * 2 + (tid >> 5)] = swa_or_hole;
      }
    }
  };
  // FP4 rows of a tile -> staging buffer (SWA rows are copied later, straight into the key tile)
  auto gather_fp4 = [&](int buf) {
    const uint32_t stg = base + L::kStage + buf * L::kStageBytes;
    for (int e = tid; e < kTT * 16; e += kTThreads) {          // 16 code chunks per row
      const int r = e >> 4, c = e & 15;
      const int64_t src = sSrc[buf * kTT + r];
      if (src >= 0 && sKind[buf * kTT + r] == 0) cp_async16_hint(stg + r * 256 + c * 16, codes + src * 256 + c * 16, pol_keep);
    }
    if (tid < kTT * 2) {                                       // 2 scale chunks per row
      const int r = tid >> 1, c = tid & 1;
      const int64_t src = sSrc[buf * kTT + r];
      if (src >= 0 && sKind[buf * kTT + r] == 0) cp_async16_hint(stg + kTT * 256 + r * 32 + c * 16, scales + src * 32 + c * 16, pol_keep);
    }
  };

  float m_run = -INFINITY, l_run = 0.f;      // softmax threads (tid < 64): head tid
  cp_async_commit();                          // Q
  if (t_begin < t_end) row_sources(t_begin, t_begin % L::kNS);
  if (t_begin + 1 < t_end) row_sources(t_begin + 1, (t_begin + 1) % L::kNS);
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = sMisc[0];
  pdl_trigger();                              // TMEM is held: the next kernel may start launching
  if (t_begin < t_end) gather_fp4(t_begin % L::kNS);
  cp_async_commit();
  if (t_begin + 1 < t_end) gather_fp4((t_begin + 1) % L::kNS);
  cp_async_commit();
  cp_async_wait<2>();                         // Q has landed (the first two tiles' rows may still fly)
  __syncthreads();
  for (int e = tid; e < 64 * 64; e += kTThreads) {          // Q -> fp16 (heads >= H: zero)
    const int h = e >> 6, c = e & 63;
    const uint32_t off = kt_off(h, c);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (h < H) v = bf16x8_to_f16x8(*reinterpret_cast<const uint4*>(sp + L::kKV + off));
    *reinterpret_cast<uint4*>(sp + L::kQ + off) = v;
  }
  __syncthreads();

  const uint32_t idesc_s = tc::instr_desc(tc::kFmtF16, tc::kFmtF16, 0, 0, 128, kTT);
  const uint32_t idesc_o = tc::instr_desc(tc::kFmtF16, tc::kFmtF16, 0, 1, 128, 256);
  int n_pv = 0;                               // PV groups committed (for the bar_o parity)
  bool ok = true;

  for (int tile = t_begin; tile < t_end; ++tile) {
    const int buf = tile % L::kNS;
    // -- the key tile is free once the previous PV has finished
    if (n_pv > 0) {
      if (!tc::mbar_wait(bar_o, (n_pv - 1) & 1)) { report(st, CSA2_ERR_TIMEOUT); ok = false; }
      tc::tc_fence_after();
    }
    // SWA rows (bf16) straight into the key tile, converted below; absent rows zero
    const uint32_t* sflags = reinterpret_cast<const uint32_t*>(sp + L::kMask + 32) + buf * 2;
    const uint64_t special = (uint64_t)sflags[0] | ((uint64_t)sflags[1] << 32);
    if (special) {
      for (int e = tid; e < kTT * 64; e += kTThreads) {
        const int r = e >> 6, c = e & 63;
        if (!((special >> r) & 1)) continue;
        const int64_t src = sSrc[buf * kTT + r];
        if (src >= 0) cp_async16(base + L::kKV + kt_off(r, c), swa + src * kTD + c * 8);
        else *reinterpret_cast<uint4*>(sp + L::kKV + kt_off(r, c)) = make_uint4(0, 0, 0, 0);
      }
      cp_async_commit();
    }
    // -- prefetch the FP4 rows two tiles ahead (left in flight)
    if (tile + 2 < t_end) row_sources(tile + 2, (tile + 2) % L::kNS);
    __syncthreads();
    if (tile + 2 < t_end) gather_fp4((tile + 2) % L::kNS);
    cp_async_commit();
    // this tile's FP4 rows (and SWA rows) have landed; the next two tiles may still fly
    if (special) cp_async_wait<1>(); else cp_async_wait<2>();
    __syncthreads();
    {
      const uint32_t* flags = reinterpret_cast<const uint32_t*>(sp + L::kMask + 32) + buf * 2;
      const uint32_t* vmask = reinterpret_cast<const uint32_t*>(sp + L::kMask) + buf * 2;
      const uint64_t swa_rows = ((uint64_t)flags[0] | ((uint64_t)flags[1] << 32)) &
                                ((uint64_t)vmask[0] | ((uint64_t)vmask[1] << 32));
      if (swa_rows) {                          // SWA rows (bf16) -> fp16 in place
        for (int e = tid; e < kTT * 64; e += kTThreads) {
          const int r = e >> 6, c = e & 63;
          if (!((swa_rows >> r) & 1)) continue;
          uint4* pv = reinterpret_cast<uint4*>(sp + L::kKV + kt_off(r, c));
          *pv = bf16x8_to_f16x8(*pv);
        }
      }
    }
    // -- dequant FP4 rows, one 16-channel group (one scale) per step: group g
    //    of row r = code bytes 8g..8g+7 -> dims 16g..16g+15 = chunks 2g, 2g+1
    {
      // thread (warp w, lane g) dequantises group g of rows w, w + 8, .., w + 56;
      // all eight rows' codes and scales are loaded before any is converted
      const unsigned char* stg = sp + L::kStage + buf * L::kStageBytes;
      const uint32_t* vmask = reinterpret_cast<const uint32_t*>(sp + L::kMask) + buf * 2;
      const uint32_t* smask = reinterpret_cast<const uint32_t*>(sp + L::kMask + 32) + buf * 2;
      const uint64_t fp4rows = ((uint64_t)vmask[0] | ((uint64_t)vmask[1] << 32)) &
                               ~((uint64_t)smask[0] | ((uint64_t)smask[1] << 32));
      constexpr int kRowsPerThread = kTT * 32 / kTThreads;
      const int g = lane;
      uint2 cw[kRowsPerThread];
      uint32_t sb[kRowsPerThread];
#pragma unroll
      for (int it = 0; it < kRowsPerThread; ++it) {
        const int r = warp + 8 * it;
        cw[it] = make_uint2(0u, 0u);
        sb[it] = 0u;
        if ((fp4rows >> r) & 1) {
          cw[it] = *reinterpret_cast<const uint2*>(stg + r * 256 + g * 8);
          sb[it] = stg[kTT * 256 + r * 32 + g];
        }
      }
#pragma unroll
      for (int it = 0; it < kRowsPerThread; ++it) {
        const int r = warp + 8 * it;
        if (!((fp4rows >> r) & 1)) continue;
        uint32_t sh2;                                           // scale as f16x2 {s, s}
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(sh2) : "h"((uint16_t)(sb[it] | (sb[it] << 8))));
        uint32_t o[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint32_t byte = ((u < 4 ? cw[it].x : cw[it].y) >> (8 * (u & 3))) & 0xFF;
          const uint32_t h2 = e2m1x2_to_f16x2(byte);
          asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[u]) : "r"(h2), "r"(sh2));
        }
        *reinterpret_cast<uint4*>(sp + L::kKV + kt_off(r, 2 * g)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(sp + L::kKV + kt_off(r, 2 * g + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
      }
    }
    tc::fence_async_smem();
    __syncthreads();
    // -- S = Q K^T
    if (tid == 0 && ok) {
      tc::tc_fence_after();
#pragma unroll 4
      for (int ks = 0; ks < kTD / 16; ++ks) {
        const uint32_t off = (ks >> 2) * 8192 + (ks & 3) * 32;
        const uint64_t ad = tc::smem_desc(base + L::kQ + off, 16, 1024, tc::kSwizzle128B);
        const uint64_t bd = tc::smem_desc(base + L::kKV + off, 16, 1024, tc::kSwizzle128B);
        tc::mma_f16(tmem + kTScol, ad, bd, idesc_s, ks > 0 ? 1u : 0u);
      }
      tc::mma_commit(bar_s);
    }
    if (!tc::mbar_wait(bar_s, (tile - t_begin) & 1, ok ? (1u << 22) : 1u)) { report(st, CSA2_ERR_TIMEOUT); ok = false; }
    tc::tc_fence_after();
    // -- softmax: thread h < 64 owns head h (TMEM lane h)
    if (warp < 2) {
      uint32_t r[64];
      tc::tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + kTScol, r);
      tc::tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + kTScol + 32, r + 32);
      tc::tmem_ld_wait();
      const int h = tid;
      const uint32_t* vm = reinterpret_cast<const uint32_t*>(sp + L::kMask) + buf * 2;
      const uint32_t vm0 = vm[0], vm1 = vm[1];
      float mt = -INFINITY;
#pragma unroll
      for (int j = 0; j < kTT; ++j) {
        const bool valid = ((j < 32 ? vm0 : vm1) >> (j & 31)) & 1u;
        const float v = valid ? __uint_as_float(r[j]) * scale_log2 : -INFINITY;
        r[j] = __float_as_uint(v);
        mt = fmaxf(mt, v);
      }
      float alpha = 1.f;
      if (mt > m_run + 8.f) {                 // raise the reference only when needed
        alpha = (m_run == -INFINITY) ? 0.f : exp2f(m_run - mt);
        m_run = mt;
      }
      const float base_m = (m_run == -INFINITY) ? 0.f : m_run;
      float sum = 0.f;
      unsigned char* prow = sp + L::kP + h * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t pk[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const __half2 pv = __floats2half2_rn(exp2f(__uint_as_float(r[8 * c + 2 * u]) - base_m),
                                               exp2f(__uint_as_float(r[8 * c + 2 * u + 1]) - base_m));
          const float2 f = __half22float2(pv);
          sum += f.x + f.y;
          pk[u] = *reinterpret_cast<const uint32_t*>(&pv);
        }
        const uint4 v4 = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        const int sw = ((c ^ (h & 7)) << 4);
        if (h < H) {
          *reinterpret_cast<uint4*>(prow + sw) = v4;               // P  (rows 0..63 of [P; Z])
          *reinterpret_cast<uint4*>(prow + 16384 + sw) = v4;       // P' (rows 64..127 of [Z; P'])
        }
      }
      l_run = l_run * alpha + sum;
      sAlpha[h] = alpha;
      if (alpha != 1.f && tile > t_begin) sMisc[1] = 1;
    }
    tc::tc_fence_before();
    __syncthreads();
    // -- rescale O when some head raised its reference (rare)
    if (sMisc[1] && warp < 4) {
      tc::tc_fence_after();
      const float a = sAlpha[(32 * warp + lane) & 63];
      const uint32_t ta = tmem + ((uint32_t)(32 * warp) << 16) + kTOcol;
      for (int c = 0; c < 256; c += 32) {
        uint32_t r[32];
        tc::tmem_ld32(ta + c, r);
        tc::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * a);
        tmem_st32(ta + c, r);
      }
      tmem_st_wait();
      tc::tc_fence_before();
    }
    __syncthreads();
    if (tid == 0) sMisc[1] = 0;
    tc::fence_async_smem();
    // -- O += P V
    if (tid == 0 && ok) {
      tc::tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < kTT / 16; ++ks) {
        const uint64_t a0 = tc::smem_desc(base + L::kP + ks * 32, 16, 1024, tc::kSwizzle128B);
        const uint64_t a1 = tc::smem_desc(base + L::kP + 8192 + ks * 32, 16, 1024, tc::kSwizzle128B);
        const uint64_t b0 = tc::smem_desc(base + L::kKV + ks * 2048, 8192, 1024, tc::kSwizzle128B);
        const uint64_t b1 = tc::smem_desc(base + L::kKV + 4 * 8192 + ks * 2048, 8192, 1024, tc::kSwizzle128B);
        tc::mma_f16(tmem + kTOcol, a0, b0, idesc_o, (tile > t_begin || ks > 0) ? 1u : 0u);
        tc::mma_f16(tmem + kTOcol, a1, b1, idesc_o, 1u);
      }
      tc::mma_commit(bar_o);
    }
    ++n_pv;
    if (__syncthreads_or(!ok)) break;          // uniform exit after a timed-out wait
  }
  cp_async_wait<0>();
  if ((slen_in < 0 || slen_in > W) && split == 0 && tid == 0) report(st, CSA2_ERR_DEVICE_BOUNDS);
  // ---- epilogue
  if (n_pv > 0) {
    if (!tc::mbar_wait(bar_o, (n_pv - 1) & 1)) report(st, CSA2_ERR_TIMEOUT);
    tc::tc_fence_after();
  }
  if (!ok) n_pv = 0;                          // a timed-out CTA writes zeros
  if (tid < 64) { sL[tid] = l_run; sMx[tid] = m_run; }
  __syncthreads();
  {
    // All eight warps: warp w reads TMEM lanes 32 (w % 4) .. + 31 (row r holds
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
      if (n_pv > 0) {
        tc::tmem_ld32(ta + c, r);
        tc::tmem_ld32(ta + c + 32, r + 32);
        tc::tmem_ld_wait();
      } else {
#pragma unroll
        for (int j = 0; j < 64; ++j) r[j] = 0u;
      }
      if (!live) continue;
      const int dim0 = dbase + c;
      if (splits == 1) {
        __nv_bfloat16* o = out + ((int64_t)b * H + h) * kTD + dim0;
#pragma unroll
        for (int j = 0; j < 64; j += 8) {
          uint32_t pk[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(r[j + 2 * u]) * inv,
                                                          __uint_as_float(r[j + 2 * u + 1]) * inv);
            pk[u] = *reinterpret_cast<const uint32_t*>(&v);
          }
          st_global_hint(o + j, make_uint4(pk[0], pk[1], pk[2], pk[3]), pol_stream);
        }
      } else {
        // partial O layout [b][split][dim / 4][H][4]: a warp stores 32 heads' float4 contiguously
        float* o = part_o + ((((int64_t)b * splits + split) * (kTD / 4) + dim0 / 4) * H + h) * 4;
#pragma unroll
        for (int j = 0; j < 64; j += 4)
          *reinterpret_cast<float4*>(o + (int64_t)(j / 4) * H * 4) =
              make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]), __uint_as_float(r[j + 2]),
                          __uint_as_float(r[j + 3]));
      }
    }
    if (live && splits > 1 && row < 64 && chalf == 0) {
      const int64_t pidx = ((int64_t)b * splits + split) * H + h;
      part_ml[pidx * 2 + 0] = sMx[h];
      part_ml[pidx * 2 + 1] = sL[h];
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
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

int launch_sparse_attn_tc(const void* q, int B, int H, const uint8_t* codes, const uint8_t* scales,
                          int64_t kv_seq_stride, int64_t n_cap, const int32_t* idx, int k, const void* swa,
                          int64_t swa_seq_stride, int W, int swa_tail, const int32_t* swa_len, float softmax_scale,
                          void* out, float* part_o, float* part_ml, int splits, int tps, int32_t* st,
                          cudaStream_t s) {
  dim3 grid((unsigned)splits, (unsigned)B);
  const cudaError_t e = launch_pdl(
      k_sparse_attn_tc, grid, dim3(kTThreads), TcSmem::kBytes, s, reinterpret_cast<const __nv_bfloat16*>(q), H,
      codes, scales, kv_seq_stride, n_cap, idx, k, reinterpret_cast<const __nv_bfloat16*>(swa), swa_seq_stride, W,
      swa_tail, swa_len, softmax_scale * 1.4426950408889634f, splits, tps, reinterpret_cast<__nv_bfloat16*>(out),
      part_o, part_ml, st);
  count_launch();
  return launch_status(e);
}

}  // namespace csa2
