// sparse_attn.cu — CSA2 decode/prefill attention over gathered FP4 main-KV
// rows plus the layer's sliding-window rows.
//
// [CSA2] wire.sakhanda.co, "DeepSeek AI выпустила DeepSeek-V4.1-Flash ...",
//        section "Сжатое разреженное внимание 2 (CSA2)": each layer attends
//        sparsely over the Top-512 main-KV entries (shared across the group in
//        Reuse mode) and keeps its own main Q and SWA KV.
// [FP4]  same page, section "FP4 KV, ограниченное повторное проигрывание и
//        другие расширения": the main KV is E2M1 with one E4M3 scale per 16
//        channels; the product of the two is exact in bf16.
// [CED]  same page, section "Каузальный энкодер-декодер: вдвое меньший
//        префилл": 128-token sliding window in every layer.
//
// Layout of the work: key slots 0..k-1 are the gathered main-KV rows idx[b][j]
// (-1 = absent), slots k..k+W-1 the SWA rows. Slots are processed in tiles of
// 64 keys; a CTA owns one sequence and a contiguous range of tiles (split-K)
// and all H heads. Per tile:
//   gather  : cp.async 16-byte copies of the 64 rows (288 B per FP4 row:
//             256 B codes + 32 B scales; 1 KB per bf16 SWA row);
//   dequant : E2M1 byte -> f16x2 by the hardware converter, times the E4M3
//             scale, stored as bf16 (exact) into an XOR-swizzled smem tile;
//   S = QK^T: mma.sync m16n8k16 bf16 -> fp32, operands by ldmatrix;
//   softmax : online (running max / sum per head, log2 domain);
//   O += PV : P rounded to bf16 in smem, V by ldmatrix.trans.
// With more than one split the CTA writes (m, l, unnormalised O) partials and
// a merge kernel combines them by log-sum-exp.
#include <stdlib.h>

#include "common.cuh"

namespace csa2 {

constexpr int kD = 512;          // main head dim
constexpr int kTile = 64;        // keys per tile
constexpr int kRowBytes = kD * 2;

__device__ __forceinline__ uint32_t swz1k(int row, int chunk) {  // 1 KB rows, 16 B chunks
  return (uint32_t)(row * kRowBytes + ((chunk ^ (row & 7)) << 4));
}
__device__ __forceinline__ uint32_t swzP(int row, int chunk) {   // 128 B rows
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

template <int MT>
struct AttnSmem {
  static constexpr int H = 16 * MT;
  static constexpr int kQ = 0;
  static constexpr int kKV = kQ + H * kRowBytes;
  static constexpr int kCodes = kKV + kTile * kRowBytes;
  static constexpr int kScales = kCodes + kTile * 256;
  static constexpr int kP = kScales + kTile * 32;
  static constexpr int kRedMax = kP + H * 128;
  static constexpr int kRedSum = kRedMax + H * 4 * 4;
  static constexpr int kM = kRedSum + H * 4 * 4;
  static constexpr int kL = kM + H * 4;
  static constexpr int kAlpha = kL + H * 4;
  static constexpr int kSrc = kAlpha + H * 4;       // int64 [kTile]
  static constexpr int kKind = kSrc + kTile * 8;    // int32 [kTile]
  static constexpr int kBytes = kKind + kTile * 4;
};

template <int MT>
__global__ void __launch_bounds__(128 * MT, 1) k_sparse_attn(
    const __nv_bfloat16* __restrict__ q, const uint8_t* __restrict__ codes,
    const uint8_t* __restrict__ scales, int64_t kv_seq_stride, int64_t n_cap,
    const int32_t* __restrict__ idx, int k, const __nv_bfloat16* __restrict__ swa,
    int64_t swa_seq_stride, int W, int swa_tail, const int32_t* __restrict__ swa_len, float scale_log2,
    int splits, int tiles_per_split, __nv_bfloat16* __restrict__ out, float* __restrict__ part_o,
    float* __restrict__ part_ml, int32_t* st) {
  using L = AttnSmem<MT>;
  constexpr int H = L::H;
  constexpr int NT = 128 * MT;
  extern __shared__ __align__(128) unsigned char smem[];
  const uint32_t sbase = smem_u32(smem);
  float* sRedMax = reinterpret_cast<float*>(smem + L::kRedMax);
  float* sRedSum = reinterpret_cast<float*>(smem + L::kRedSum);
  float* sM = reinterpret_cast<float*>(smem + L::kM);
  float* sL = reinterpret_cast<float*>(smem + L::kL);
  float* sAlpha = reinterpret_cast<float*>(smem + L::kAlpha);
  int64_t* sSrc = reinterpret_cast<int64_t*>(smem + L::kSrc);
  int32_t* sKind = reinterpret_cast<int32_t*>(smem + L::kKind);

  const int b = blockIdx.y, split = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int mt = warp >> 2, wq = warp & 3;
  const int n_tiles = (k + W + kTile - 1) / kTile;
  const int t_begin = split * tiles_per_split;
  const int t_end = min(t_begin + tiles_per_split, n_tiles);
  int slen = swa_len[b];
  if (slen > W || slen < 0) {
    if (split == 0 && tid == 0) report(st, CSA2_ERR_DEVICE_BOUNDS);
    slen = slen < 0 ? 0 : W;
  }

  // Q -> smem (swizzled)
  for (int e = tid; e < H * 64; e += NT) {
    const int r = e >> 6, c = e & 63;
    cp_async16(sbase + L::kQ + swz1k(r, c), q + ((int64_t)b * H + r) * kD + c * 8);
  }
  cp_async_commit();
  if (tid < H) { sM[tid] = -INFINITY; sL[tid] = 0.f; }

  float oacc[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;

  for (int tile = t_begin; tile < t_end; ++tile) {
    // -- row sources
    if (tid < kTile) {
      const int j = tile * kTile + tid;
      int64_t src = -1;
      int kind = 0;
      if (j < k) {
        const int32_t p = idx[(int64_t)b * k + j];
        if (p >= 0 && p < n_cap) src = (int64_t)b * kv_seq_stride + p;
        else if (p >= n_cap) report(st, CSA2_ERR_DEVICE_BOUNDS);
      } else if (j - k < slen) {
        // valid SWA rows: the first slen of the W-row window, or its last slen
        src = (int64_t)b * swa_seq_stride + (swa_tail ? W - slen : 0) + (j - k);
        kind = 1;
      }
      sSrc[tid] = src;
      sKind[tid] = kind;
    }
    __syncthreads();
    // -- gather
    for (int e = tid; e < kTile * 18; e += NT) {
      const int r = e / 18, c = e - r * 18;
      const int64_t src = sSrc[r];
      if (src >= 0 && sKind[r] == 0) {
        if (c < 16) cp_async16(sbase + L::kCodes + r * 256 + c * 16, codes + src * 256 + c * 16);
        else cp_async16(sbase + L::kScales + r * 32 + (c - 16) * 16, scales + src * 32 + (c - 16) * 16);
      }
    }
    for (int e = tid; e < kTile * 64; e += NT) {
      const int r = e >> 6, c = e & 63;
      const int64_t src = sSrc[r];
      if (src >= 0 && sKind[r] == 1) {
        cp_async16(sbase + L::kKV + swz1k(r, c), swa + src * kD + c * 8);
      } else if (src < 0) {
        *reinterpret_cast<uint4*>(smem + L::kKV + swz1k(r, c)) = make_uint4(0, 0, 0, 0);
      }
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    // -- dequant FP4 rows: chunk c of row r = channels 8c..8c+7 = code bytes 4c..4c+3
    for (int e = tid; e < kTile * 64; e += NT) {
      const int r = e >> 6, c = e & 63;
      if (sSrc[r] >= 0 && sKind[r] == 0) {
        const uint32_t cw = *reinterpret_cast<const uint32_t*>(smem + L::kCodes + r * 256 + c * 4);
        const float s = e4m3_to_f32(smem[L::kScales + r * 32 + (c >> 1)]);
        uint32_t o[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t h2 = e2m1x2_to_f16x2((cw >> (8 * u)) & 0xFF);
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
          const __nv_bfloat162 v = __floats2bfloat162_rn(f.x * s, f.y * s);
          o[u] = *reinterpret_cast<const uint32_t*>(&v);
        }
        *reinterpret_cast<uint4*>(smem + L::kKV + swz1k(r, c)) = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
    __syncthreads();
    // -- S = Q K^T for heads 16mt.., keys 16wq..16wq+15
    float sacc[2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.f;
#pragma unroll 8
    for (int ks = 0; ks < kD / 16; ++ks) {
      uint32_t a[4], bb[4];
      ldmatrix_x4(a, sbase + L::kQ + swz1k(16 * mt + (lane & 15), 2 * ks + (lane >> 4)));
      ldmatrix_x4(bb, sbase + L::kKV + swz1k(16 * wq + (lane & 7) + 8 * (lane >> 4), 2 * ks + ((lane >> 3) & 1)));
      mma_bf16_16816(sacc[0], a, bb[0], bb[1]);
      mma_bf16_16816(sacc[1], a, bb[2], bb[3]);
    }
    // -- scale, mask, tile row max
    const int h0 = 16 * mt + g, h1 = h0 + 8;
    float x[2][4];
    float rmax0 = -INFINITY, rmax1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = 16 * wq + 8 * nt + 2 * t + (e & 1);
        const float v = sSrc[key] >= 0 ? sacc[nt][e] * scale_log2 : -INFINITY;
        x[nt][e] = v;
        if (e < 2) rmax0 = fmaxf(rmax0, v); else rmax1 = fmaxf(rmax1, v);
      }
    }
    rmax0 = fmaxf(rmax0, __shfl_xor_sync(0xffffffffu, rmax0, 1));
    rmax1 = fmaxf(rmax1, __shfl_xor_sync(0xffffffffu, rmax1, 1));
    rmax0 = fmaxf(rmax0, __shfl_xor_sync(0xffffffffu, rmax0, 2));
    rmax1 = fmaxf(rmax1, __shfl_xor_sync(0xffffffffu, rmax1, 2));
    if (t == 0) { sRedMax[h0 * 4 + wq] = rmax0; sRedMax[h1 * 4 + wq] = rmax1; }
    __syncthreads();
    float mnew0 = sM[h0], mnew1 = sM[h1];
#pragma unroll
    for (int j = 0; j < 4; ++j) { mnew0 = fmaxf(mnew0, sRedMax[h0 * 4 + j]); mnew1 = fmaxf(mnew1, sRedMax[h1 * 4 + j]); }
    const float base0 = mnew0 == -INFINITY ? 0.f : mnew0;
    const float base1 = mnew1 == -INFINITY ? 0.f : mnew1;
    float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const __nv_bfloat162 p0 = __floats2bfloat162_rn(exp2f(x[nt][0] - base0), exp2f(x[nt][1] - base0));
      const __nv_bfloat162 p1 = __floats2bfloat162_rn(exp2f(x[nt][2] - base1), exp2f(x[nt][3] - base1));
      const float2 f0 = __bfloat1622float2(p0), f1 = __bfloat1622float2(p1);
      rs0 += f0.x + f0.y;
      rs1 += f1.x + f1.y;
      const int chunk = 2 * wq + nt;
      *reinterpret_cast<__nv_bfloat162*>(smem + L::kP + swzP(h0, chunk) + 4 * t) = p0;
      *reinterpret_cast<__nv_bfloat162*>(smem + L::kP + swzP(h1, chunk) + 4 * t) = p1;
    }
    rs0 += __shfl_xor_sync(0xffffffffu, rs0, 1);
    rs1 += __shfl_xor_sync(0xffffffffu, rs1, 1);
    rs0 += __shfl_xor_sync(0xffffffffu, rs0, 2);
    rs1 += __shfl_xor_sync(0xffffffffu, rs1, 2);
    if (t == 0) { sRedSum[h0 * 4 + wq] = rs0; sRedSum[h1 * 4 + wq] = rs1; }
    __syncthreads();
    if (tid < H) {
      const float mold = sM[tid];
      float mn = mold, ssum = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) { mn = fmaxf(mn, sRedMax[tid * 4 + j]); ssum += sRedSum[tid * 4 + j]; }
      const float alpha = (mold == -INFINITY) ? 0.f : exp2f(mold - mn);
      sL[tid] = sL[tid] * alpha + ssum;
      sM[tid] = mn;
      sAlpha[tid] = alpha;
    }
    __syncthreads();
    // -- O += P V for heads 16mt.., dims 128wq..128wq+127
    {
      const float al0 = sAlpha[h0], al1 = sAlpha[h1];
#pragma unroll
      for (int i = 0; i < 16; ++i) { oacc[i][0] *= al0; oacc[i][1] *= al0; oacc[i][2] *= al1; oacc[i][3] *= al1; }
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk) {
        uint32_t a[4];
        ldmatrix_x4(a, sbase + L::kP + swzP(16 * mt + (lane & 15), 2 * kk + (lane >> 4)));
#pragma unroll
        for (int pr = 0; pr < 8; ++pr) {
          uint32_t bb[4];
          ldmatrix_x4_trans(bb, sbase + L::kKV + swz1k(16 * kk + (lane & 7) + 8 * ((lane >> 3) & 1),
                                                       16 * wq + 2 * pr + (lane >> 4)));
          mma_bf16_16816(oacc[2 * pr], a, bb[0], bb[1]);
          mma_bf16_16816(oacc[2 * pr + 1], a, bb[2], bb[3]);
        }
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();  // Q copies of a CTA without tiles
  __syncthreads();

  // -- epilogue
  const int h0 = 16 * mt + g, h1 = h0 + 8;
  if (splits == 1) {
    const float l0 = sL[h0], l1 = sL[h1];
    const float i0 = l0 > 0.f ? 1.f / l0 : 0.f, i1 = l1 > 0.f ? 1.f / l1 : 0.f;
    __nv_bfloat16* o0 = out + ((int64_t)b * H + h0) * kD;
    __nv_bfloat16* o1 = out + ((int64_t)b * H + h1) * kD;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int dim = 128 * wq + 8 * i + 2 * t;
      *reinterpret_cast<__nv_bfloat162*>(o0 + dim) = __floats2bfloat162_rn(oacc[i][0] * i0, oacc[i][1] * i0);
      *reinterpret_cast<__nv_bfloat162*>(o1 + dim) = __floats2bfloat162_rn(oacc[i][2] * i1, oacc[i][3] * i1);
    }
  } else {
    const int64_t pb = ((int64_t)b * splits + split) * H;
    float* o0 = part_o + (pb + h0) * kD;
    float* o1 = part_o + (pb + h1) * kD;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int dim = 128 * wq + 8 * i + 2 * t;
      *reinterpret_cast<float2*>(o0 + dim) = make_float2(oacc[i][0], oacc[i][1]);
      *reinterpret_cast<float2*>(o1 + dim) = make_float2(oacc[i][2], oacc[i][3]);
    }
    if (tid < H) {
      part_ml[(pb + tid) * 2 + 0] = sM[tid];
      part_ml[(pb + tid) * 2 + 1] = sL[tid];
    }
  }
}

// Log-sum-exp merge of split-K partials: one CTA of 128 threads per (b, h).
__global__ void __launch_bounds__(128) k_attn_merge(const float* __restrict__ part_o,
                                                    const float* __restrict__ part_ml, int H,
                                                    int splits, __nv_bfloat16* __restrict__ out) {
  const int bh = blockIdx.x;
  const int b = bh / H, h = bh - b * H;
  float M = -INFINITY;
  for (int s = 0; s < splits; ++s) M = fmaxf(M, part_ml[(((int64_t)b * splits + s) * H + h) * 2]);
  float Lsum = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const int dim = threadIdx.x * 4;
  if (M != -INFINITY) {
    for (int s = 0; s < splits; ++s) {
      const int64_t pidx = ((int64_t)b * splits + s) * H + h;
      const float m = part_ml[pidx * 2], l = part_ml[pidx * 2 + 1];
      if (m == -INFINITY) continue;
      const float wgt = exp2f(m - M);
      Lsum += wgt * l;
      const float4 v = *reinterpret_cast<const float4*>(part_o + pidx * kD + dim);
      acc.x += wgt * v.x; acc.y += wgt * v.y; acc.z += wgt * v.z; acc.w += wgt * v.w;
    }
  }
  const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
  __nv_bfloat16* o = out + ((int64_t)b * H + h) * kD + dim;
  *reinterpret_cast<__nv_bfloat162*>(o) = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  *reinterpret_cast<__nv_bfloat162*>(o + 2) = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
}

// ---- host ------------------------------------------------------------------
static int attn_occupancy(int MT) { return MT <= 2 ? 2 : 1; }

// Split-K count. A batch that fills the machine runs unsplit (a split writes
// an fp32 partial of H x 512 per CTA and needs the merge pass). Otherwise
// minimise waves x tiles per split plus one tile-equivalent for the merge;
// ties go to fewer splits.
int attn_splits(int B, int H, int k, int W) {
  const int n_tiles = (k + W + kTile - 1) / kTile;
  const int MT = H / 16;
  const int64_t slots = (int64_t)kSMs * attn_occupancy(MT);
  if ((int64_t)B >= slots) return 1;
  int best = 1;
  int64_t best_cost = -1;
  for (int s = 1; s <= n_tiles; ++s) {
    const int tps = (n_tiles + s - 1) / s;
    const int sp = (n_tiles + tps - 1) / tps;  // splits actually holding tiles
    if (sp != s) continue;
    const int64_t waves = ((int64_t)B * s + slots - 1) / slots;
    const int64_t cost = waves * tps + (s > 1 ? 1 : 0);
    if (best_cost < 0 || cost < best_cost) { best_cost = cost; best = s; }
  }
  return best;
}

size_t attn_ws_bytes(int B, int H, int k, int W) {
  const int s1 = attn_splits(B, H, k, W), s2 = attn_splits(B, 64, k, W);
  const int s = s1 > s2 ? s1 : s2;
  if (s <= 1) return 0;
  const size_t po = (size_t)B * s * H * kD * 4;
  return ((po + 255) & ~(size_t)255) + (size_t)B * s * H * 2 * 4;
}

template <int MT>
static int launch_attn_mt(const void* q, int B, const uint8_t* codes, const uint8_t* scales,
                          int64_t kv_seq_stride, int64_t n_cap, const int32_t* idx, int k,
                          const void* swa, int64_t swa_seq_stride, int W, int swa_tail, const int32_t* swa_len,
                          float softmax_scale, void* out, void* ws, int32_t* st, cudaStream_t s) {
  constexpr int H = 16 * MT;
  const int smem = AttnSmem<MT>::kBytes;
  const int splits = attn_splits(B, H, k, W);
  const int n_tiles = (k + W + kTile - 1) / kTile;
  const int tps = (n_tiles + splits - 1) / splits;
  float* part_o = nullptr;
  float* part_ml = nullptr;
  if (splits > 1) {
    part_o = static_cast<float*>(ws);
    const size_t po = (size_t)B * splits * H * kD * 4;
    part_ml = reinterpret_cast<float*>(static_cast<char*>(ws) + ((po + 255) & ~(size_t)255));
  }
  const float scale_log2 = softmax_scale * 1.4426950408889634f;
  dim3 grid((unsigned)splits, (unsigned)B);
  k_sparse_attn<MT><<<grid, 128 * MT, smem, s>>>(
      reinterpret_cast<const __nv_bfloat16*>(q), codes, scales, kv_seq_stride, n_cap, idx, k,
      reinterpret_cast<const __nv_bfloat16*>(swa), swa_seq_stride, W, swa_tail, swa_len, scale_log2, splits, tps,
      reinterpret_cast<__nv_bfloat16*>(out), part_o, part_ml, st);
  count_launch();
  int rc = launch_status();
  if (rc != CSA2_OK || splits == 1) return rc;
  k_attn_merge<<<(unsigned)(B * H), 128, 0, s>>>(part_o, part_ml, H, splits,
                                                  reinterpret_cast<__nv_bfloat16*>(out));
  count_launch();
  return launch_status();
}

int attn_init_attributes() {
  if (cudaFuncSetAttribute(k_sparse_attn<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, AttnSmem<1>::kBytes) != cudaSuccess ||
      cudaFuncSetAttribute(k_sparse_attn<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, AttnSmem<2>::kBytes) != cudaSuccess ||
      cudaFuncSetAttribute(k_sparse_attn<3>, cudaFuncAttributeMaxDynamicSharedMemorySize, AttnSmem<3>::kBytes) != cudaSuccess ||
      cudaFuncSetAttribute(k_sparse_attn<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, AttnSmem<4>::kBytes) != cudaSuccess)
    return CSA2_ERR_CUDA;
  return CSA2_OK;
}

int launch_sparse_attn_tc(const void* q, int B, int H, const uint8_t* codes, const uint8_t* scales,
                          int64_t kv_seq_stride, int64_t n_cap, const int32_t* idx, int k, const void* swa,
                          int64_t swa_seq_stride, int W, int swa_tail, const int32_t* swa_len, float softmax_scale,
                          void* out, float* part_o, float* part_ml, int splits, int tps, int32_t* st,
                          cudaStream_t s);

// tcgen05 path: all H <= 64 heads of a sequence per CTA, one CTA per SM.
static int launch_attn_tc_split(const void* q, int B, int H, const uint8_t* codes, const uint8_t* scales,
                                int64_t kv_seq_stride, int64_t n_cap, const int32_t* idx, int k, const void* swa,
                                int64_t swa_seq_stride, int W, int swa_tail, const int32_t* swa_len,
                                float softmax_scale, void* out, void* ws, int32_t* st, cudaStream_t s) {
  const int splits = attn_splits(B, 64, k, W);
  const int n_tiles = (k + W + kTile - 1) / kTile;
  const int tps = (n_tiles + splits - 1) / splits;
  float* part_o = nullptr;
  float* part_ml = nullptr;
  if (splits > 1) {
    part_o = static_cast<float*>(ws);
    const size_t po = (size_t)B * splits * H * kD * 4;
    part_ml = reinterpret_cast<float*>(static_cast<char*>(ws) + ((po + 255) & ~(size_t)255));
  }
  int rc = launch_sparse_attn_tc(q, B, H, codes, scales, kv_seq_stride, n_cap, idx, k, swa, swa_seq_stride, W,
                                 swa_tail, swa_len, softmax_scale, out, part_o, part_ml, splits, tps, st, s);
  if (rc != CSA2_OK || splits == 1) return rc;
  k_attn_merge<<<(unsigned)(B * H), 128, 0, s>>>(part_o, part_ml, H, splits, reinterpret_cast<__nv_bfloat16*>(out));
  count_launch();
  return launch_status();
}

int launch_sparse_attn(const void* q, int B, int H, const uint8_t* codes, const uint8_t* scales,
                       int64_t kv_seq_stride, int64_t n_cap, const int32_t* idx, int k, const void* swa,
                       int64_t swa_seq_stride, int W, int swa_tail, const int32_t* swa_len, float softmax_scale,
                       void* out, void* ws, int32_t* st, cudaStream_t s) {
  if (B == 0) return CSA2_OK;
  static const bool use_mma_sync = [] {
    const char* e = getenv("CSA2_ATTN_MMA_SYNC");
    return e != nullptr && e[0] == '1';
  }();
  if (!use_mma_sync)
    return launch_attn_tc_split(q, B, H, codes, scales, kv_seq_stride, n_cap, idx, k, swa, swa_seq_stride, W,
                                swa_tail, swa_len, softmax_scale, out, ws, st, s);
  switch (H) {
    case 16: return launch_attn_mt<1>(q, B, codes, scales, kv_seq_stride, n_cap, idx, k, swa, swa_seq_stride, W, swa_tail, swa_len, softmax_scale, out, ws, st, s);
    case 32: return launch_attn_mt<2>(q, B, codes, scales, kv_seq_stride, n_cap, idx, k, swa, swa_seq_stride, W, swa_tail, swa_len, softmax_scale, out, ws, st, s);
    case 48: return launch_attn_mt<3>(q, B, codes, scales, kv_seq_stride, n_cap, idx, k, swa, swa_seq_stride, W, swa_tail, swa_len, softmax_scale, out, ws, st, s);
    case 64: return launch_attn_mt<4>(q, B, codes, scales, kv_seq_stride, n_cap, idx, k, swa, swa_seq_stride, W, swa_tail, swa_len, softmax_scale, out, ws, st, s);
    default: return CSA2_ERR_UNSUPPORTED_SHAPE;
  }
}

}  // namespace csa2
