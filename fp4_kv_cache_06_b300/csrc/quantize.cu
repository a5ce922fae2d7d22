// quantize.cu — cache writers: FP4 main-KV quantise/append, indexer-K append
// with block means, sliding-window ring append.
//
// [FP4] wire.sakhanda.co, "DeepSeek AI выпустила DeepSeek-V4.1-Flash ...",
//       section "FP4 KV, ограниченное повторное проигрывание и другие
//       расширения": main KV stored as E2M1 with one E4M3 scale per 16
//       channels and no global scale.
// [CSA2] same page, section "Сжатое разреженное внимание 2 (CSA2)": the pool
//       is built from blocks of 8 positions.
// [CED] same page, section "Каузальный энкодер-декодер: вдвое меньший
//       префилл": 128-token sliding window in every layer.
//
// All three writers are HBM-bound copies with a little arithmetic; one warp
// owns one row so every load and store is a full 16-byte vector.
#include "common.cuh"

namespace csa2 {

// One warp quantises one bf16 row of 512 channels: lane l owns group l
// (channels 16l..16l+15), i.e. one E4M3 scale and 8 bytes of codes.
__device__ __forceinline__ void quantize_row_warp(const uint4* __restrict__ xrow, uint8_t* __restrict__ crow,
                                                  uint8_t* __restrict__ srow, int lane) {
  const uint4 v0 = xrow[lane * 2];
  const uint4 v1 = xrow[lane * 2 + 1];
  const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
  float f[16];
  uint32_t sign_lo = 0, sign_hi = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    f[2 * j] = __uint_as_float(w[j] << 16);
    f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    const uint32_t s0 = (w[j] >> 15) & 1u, s1 = (w[j] >> 31) & 1u;
    if (j < 4) {
      sign_lo |= (s0 << (8 * j + 3)) | (s1 << (8 * j + 7));
    } else {
      sign_hi |= (s0 << (8 * (j - 4) + 3)) | (s1 << (8 * (j - 4) + 7));
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(f[j]));
  const uint8_t sc = cvt_e4m3(__fdiv_rn(amax, 6.0f));
  const float s = e4m3_to_f32(sc);
  uint32_t lo = 0, hi = 0;
  if (s > 0.f) {
    float m[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) m[j] = __fdiv_rn(fabsf(f[j]), s);
    lo = cvt_e2m1x8(m) | sign_lo;
    hi = cvt_e2m1x8(m + 8) | sign_hi;
  }
  *reinterpret_cast<uint2*>(crow + lane * 8) = make_uint2(lo, hi);
  srow[lane] = sc;
}

__global__ void __launch_bounds__(256) k_quantize_fp4(const uint4* __restrict__ x, int B, int64_t rows,
                                                      const int64_t* __restrict__ pos,
                                                      uint8_t* __restrict__ codes,
                                                      uint8_t* __restrict__ scales, int64_t n_cap,
                                                      int32_t* st) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t total = (int64_t)B * rows;
  for (int64_t r = (((int64_t)blockIdx.x * blockDim.x) + threadIdx.x) >> 5; r < total; r += nwarps) {
    const int b = (int)(r / rows);
    const int64_t i = r - (int64_t)b * rows;
    const int64_t p = (pos ? pos[b] : 0) + i;
    if (p < 0 || p >= n_cap) {
      if (lane == 0) report(st, CSA2_ERR_DEVICE_BOUNDS);
      continue;
    }
    const int64_t row = (int64_t)b * n_cap + p;
    quantize_row_warp(x + r * 64, codes + row * 256, scales + row * 32, lane);
  }
}

// Copy E4M3 indexer-key rows into the cache: one thread per 16-byte chunk.
__global__ void k_copy_index_rows(const uint8_t* __restrict__ k_new, int B, int64_t rows, int d_I,
                                  const int64_t* __restrict__ pos, uint8_t* __restrict__ kI,
                                  int64_t n_cap, int32_t* st) {
  const int chunks = d_I / 16;
  const int64_t total = (int64_t)B * rows * chunks;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = e / chunks;
    const int c = (int)(e - r * chunks);
    const int b = (int)(r / rows);
    const int64_t i = r - (int64_t)b * rows;
    const int64_t p = (pos ? pos[b] : 0) + i;
    if (p < 0 || p >= n_cap) {
      if (c == 0) report(st, CSA2_ERR_DEVICE_BOUNDS);
      continue;
    }
    const uint4 v = *reinterpret_cast<const uint4*>(k_new + r * d_I + c * 16);
    *reinterpret_cast<uint4*>(kI + ((int64_t)b * n_cap + p) * d_I + c * 16) = v;
  }
}

// Mean key of block j of one sequence over positions [8j, end): exact fp32
// sum of E4M3 values (at most 8 terms, magnitudes 2^-9 .. 448, so at most 21
// significant bits), IEEE division by the count, E4M3 RNE with saturation.
// One warp per block; lane l owns channels 4l..4l+3.
__device__ __forceinline__ void block_mean_warp(const uint8_t* __restrict__ kI_seq,
                                                uint8_t* __restrict__ kbar_seq, int64_t j,
                                                int64_t end, int d_I, int lane) {
  const int64_t beg = j * kBlock;
  const float cnt = (float)(end - beg);
  for (int c = lane * 4; c < d_I; c += 128) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int64_t t = beg; t < end; ++t) {
      const uint32_t v = *reinterpret_cast<const uint32_t*>(kI_seq + t * d_I + c);
#pragma unroll
      for (int u = 0; u < 4; ++u) acc[u] += e4m3_to_f32((uint8_t)(v >> (8 * u)));
    }
    const uint16_t lo = cvt_e4m3x2(__fdiv_rn(acc[0], cnt), __fdiv_rn(acc[1], cnt));
    const uint16_t hi = cvt_e4m3x2(__fdiv_rn(acc[2], cnt), __fdiv_rn(acc[3], cnt));
    *reinterpret_cast<uint32_t*>(kbar_seq + j * d_I + c) = (uint32_t)lo | ((uint32_t)hi << 16);
  }
}

// Blocks touched by an append of `rows` positions starting at pos[b]: the
// mean covers the block start through the last appended position.
__global__ void k_block_means_append(const uint8_t* __restrict__ kI, int B, int64_t rows, int d_I,
                                     const int64_t* __restrict__ pos, uint8_t* __restrict__ kbar,
                                     int64_t n_cap, int64_t touched) {
  const int b = blockIdx.y;
  const int lane = threadIdx.x & 31;
  const int64_t jj = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (jj >= touched) return;
  const int64_t p0 = pos ? pos[b] : 0;
  const int64_t last = p0 + rows - 1;
  if (p0 < 0 || last >= n_cap) return;  // the copy kernel reported it
  const int64_t j = p0 / kBlock + jj;
  if (j * kBlock > last) return;
  const int64_t end = min((j + 1) * kBlock, last + 1);
  const int64_t nbc = (n_cap + kBlock - 1) / kBlock;
  block_mean_warp(kI + (int64_t)b * n_cap * d_I, kbar + (int64_t)b * nbc * d_I, j, end, d_I, lane);
}

// Every block of positions [0, n[b]).
__global__ void k_block_means_all(const uint8_t* __restrict__ kI, int d_I,
                                  const int64_t* __restrict__ n, int64_t n_cap,
                                  uint8_t* __restrict__ kbar, int32_t* st) {
  const int b = blockIdx.y;
  const int lane = threadIdx.x & 31;
  const int64_t j = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  int64_t nb = n[b];
  if (nb > n_cap) {
    if (j == 0 && lane == 0) report(st, CSA2_ERR_DEVICE_BOUNDS);
    nb = n_cap;
  }
  if (j * kBlock >= nb) return;
  const int64_t end = min((j + 1) * kBlock, nb);
  const int64_t nbc = (n_cap + kBlock - 1) / kBlock;
  block_mean_warp(kI + (int64_t)b * n_cap * d_I, kbar + (int64_t)b * nbc * d_I, j, end, d_I, lane);
}

// One warp per sequence copies its new sliding-window row into slot pos % W.
__global__ void k_append_swa(const uint4* __restrict__ x, int B, int d, const int64_t* __restrict__ pos,
                             uint4* __restrict__ swa, int W) {
  const int b = (int)(((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= B) return;
  int64_t slot = pos[b] % W;
  if (slot < 0) slot += W;
  const int chunks = d / 8;  // bf16: 8 per 16 bytes
  for (int c = lane; c < chunks; c += 32)
    swa[((int64_t)b * W + slot) * chunks + c] = x[(int64_t)b * chunks + c];
}

// ---- one decode token into every cache, one launch ---------------------------
constexpr int kMaxStepLayers = 64;
struct StepLayers {
  const uint4* src[kMaxStepLayers];   // [B][d] bf16 new SWA rows
  uint4* dst[kMaxStepLayers];         // [B][W][d] bf16 rings
};

// One warp per task; task = b * (2 + L) + kind. pos[b] is the new token's
// position tok; `ratio` tokens make one compressed main-KV entry, which is
// complete (and appended, at entry index (tok + 1) / ratio - 1) only when
// (tok + 1) % ratio == 0. Kind 0 quantises the entry's main-KV row (and writes
// the token's visible entry count and SWA length when asked), kind 1 appends
// its indexer key and refreshes the block mean (the new key is taken from
// the input, the block's earlier keys from the cache), kind 2 + l writes
// layer l's SWA row into slot tok % W.
__global__ void __launch_bounds__(256) k_append_step(const uint4* __restrict__ kv_new,
                                                     const uint8_t* __restrict__ kI_new, StepLayers layers,
                                                     int L, int W, int B, int d_I,
                                                     const int64_t* __restrict__ pos, int ratio,
                                                     uint8_t* __restrict__ codes,
                                                     uint8_t* __restrict__ scales, uint8_t* __restrict__ kI,
                                                     uint8_t* __restrict__ kbar, int64_t n_cap,
                                                     int64_t* __restrict__ n_vis_out,
                                                     int32_t* __restrict__ swa_len_out, int32_t* st) {
  const int lane = threadIdx.x & 31;
  const int64_t task = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int per = 2 + L;
  if (task >= (int64_t)B * per) return;
  const int b = (int)(task / per), kind = (int)(task - (int64_t)b * per);
  const int64_t tok = pos[b];
  if (tok < 0) {
    if (lane == 0 && kind == 0) report(st, CSA2_ERR_DEVICE_BOUNDS);
    return;
  }
  if (kind == 0 && lane == 0) {
    if (n_vis_out) n_vis_out[b] = (tok + 1) / ratio;
    if (swa_len_out) swa_len_out[b] = (int32_t)(tok + 1 < W ? tok + 1 : W);
  }
  const int64_t p = (tok + 1) % ratio == 0 ? (tok + 1) / ratio - 1 : -1;   // entry index, or none this token
  if (kind < 2 && p >= n_cap) {
    if (lane == 0 && kind == 0) report(st, CSA2_ERR_DEVICE_BOUNDS);
    return;
  }
  if (kind == 0) {
    if (p < 0) return;
    const int64_t row = (int64_t)b * n_cap + p;
    quantize_row_warp(kv_new + (int64_t)b * 64, codes + row * 256, scales + row * 32, lane);
  } else if (kind == 1) {
    if (p < 0) return;
    const uint8_t* kseq = kI + (int64_t)b * n_cap * d_I;
    const int c = lane * 4;
    if (c < d_I) {
      const uint32_t nv = *reinterpret_cast<const uint32_t*>(kI_new + (int64_t)b * d_I + c);
      *reinterpret_cast<uint32_t*>(kI + ((int64_t)b * n_cap + p) * d_I + c) = nv;
      if (kbar != nullptr) {
        const int64_t j = p / kBlock;
        float acc[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) acc[u] = e4m3_to_f32((uint8_t)(nv >> (8 * u)));
        for (int64_t t = j * kBlock; t < p; ++t) {
          const uint32_t v = *reinterpret_cast<const uint32_t*>(kseq + t * d_I + c);
#pragma unroll
          for (int u = 0; u < 4; ++u) acc[u] += e4m3_to_f32((uint8_t)(v >> (8 * u)));
        }
        const float cnt = (float)(p - j * kBlock + 1);
        const uint16_t lo = cvt_e4m3x2(__fdiv_rn(acc[0], cnt), __fdiv_rn(acc[1], cnt));
        const uint16_t hi = cvt_e4m3x2(__fdiv_rn(acc[2], cnt), __fdiv_rn(acc[3], cnt));
        const int64_t nbc = (n_cap + kBlock - 1) / kBlock;
        *reinterpret_cast<uint32_t*>(kbar + ((int64_t)b * nbc + j) * d_I + c) = (uint32_t)lo | ((uint32_t)hi << 16);
      }
    }
  } else {
    const int l = kind - 2;
    const int64_t slot = tok % W;
    const uint4* src = layers.src[l] + (int64_t)b * 64;
    uint4* dst = layers.dst[l] + ((int64_t)b * W + slot) * 64;
    dst[lane] = src[lane];
    dst[lane + 32] = src[lane + 32];
  }
}

// ---- SWA ring <-> token order (buffer management for a restored session) ----
// A layer's ring holds token t of sequence b at slot t % W. After n[b] tokens
// the window is tokens n - c .. n - 1, c = min(n, W). to_ring = 0 (export):
// lin[b][i] = ring row of token n - c + i for i < c, zero rows after it.
// to_ring = 1 (restore): each lin[b][i], i < c, goes to its token's slot and
// swa_len_out[b] = c. One warp per (layer, sequence, row).
__global__ void __launch_bounds__(256) k_swa_ring(StepLayers layers, int L, int W, int B, int chunks,
                                                  const int64_t* __restrict__ n, int to_ring,
                                                  int32_t* __restrict__ swa_len_out) {
  const int lane = threadIdx.x & 31;
  const int64_t task = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (task >= (int64_t)L * B * W) return;
  const int l = (int)(task / ((int64_t)B * W));
  const int64_t rem = task - (int64_t)l * B * W;
  const int b = (int)(rem / W), i = (int)(rem - (int64_t)b * W);
  const int64_t nb = n[b] > 0 ? n[b] : 0;
  const int64_t c = nb < W ? nb : W;
  const int64_t slot = (nb - c + i) % W;
  const uint4* src = layers.src[l];
  uint4* dst = layers.dst[l];
  if (to_ring) {
    if (i < c)
      for (int x = lane; x < chunks; x += 32)
        dst[((int64_t)b * W + slot) * chunks + x] = src[((int64_t)b * W + i) * chunks + x];
    if (swa_len_out && l == 0 && i == 0 && lane == 0) swa_len_out[b] = (int32_t)c;
  } else {
    for (int x = lane; x < chunks; x += 32)
      dst[((int64_t)b * W + i) * chunks + x] =
          i < c ? src[((int64_t)b * W + slot) * chunks + x] : make_uint4(0u, 0u, 0u, 0u);
  }
}

// ---- host launchers -----------------------------------------------------
int launch_quantize_fp4(const void* x, int B, int64_t rows, const int64_t* pos, uint8_t* codes,
                        uint8_t* scales, int64_t n_cap, int32_t* st, cudaStream_t s) {
  const int64_t total = (int64_t)B * rows;
  const int64_t warps = total;
  int64_t blocks = (warps + 7) / 8;
  blocks = blocks < kSMs * 16 ? blocks : kSMs * 16;
  if (blocks < 1) return CSA2_OK;
  k_quantize_fp4<<<(unsigned)blocks, 256, 0, s>>>(reinterpret_cast<const uint4*>(x), B, rows, pos,
                                                  codes, scales, n_cap, st);
  count_launch();
  return launch_status();
}

int launch_append_indexer_k(const uint8_t* k_new, int B, int64_t rows, int d_I, const int64_t* pos,
                            uint8_t* kI, uint8_t* kbar, int64_t n_cap, int32_t* st,
                            cudaStream_t s) {
  const int64_t total = (int64_t)B * rows * (d_I / 16);
  if (total == 0) return CSA2_OK;
  int64_t blocks = (total + 255) / 256;
  blocks = blocks < kSMs * 16 ? blocks : kSMs * 16;
  k_copy_index_rows<<<(unsigned)blocks, 256, 0, s>>>(k_new, B, rows, d_I, pos, kI, n_cap, st);
  count_launch();
  int rc = launch_status();
  if (rc != CSA2_OK || kbar == nullptr) return rc;
  const int64_t touched = (rows + kBlock - 1) / kBlock + 1;
  dim3 grid((unsigned)((touched + 7) / 8), (unsigned)B);
  k_block_means_append<<<grid, 256, 0, s>>>(kI, B, rows, d_I, pos, kbar, n_cap, touched);
  count_launch();
  return launch_status();
}

int launch_block_means(const uint8_t* kI, int B, int d_I, const int64_t* n, int64_t n_max,
                       int64_t n_cap, uint8_t* kbar, int32_t* st, cudaStream_t s) {
  const int64_t nb = (n_max + kBlock - 1) / kBlock;
  if (nb == 0 || B == 0) return CSA2_OK;
  dim3 grid((unsigned)((nb + 7) / 8), (unsigned)B);
  k_block_means_all<<<grid, 256, 0, s>>>(kI, d_I, n, n_cap, kbar, st);
  count_launch();
  return launch_status();
}

int launch_swa_ring(const void* const* src, void* const* dst, int L, int W, int B, int d, const int64_t* n,
                    int to_ring, int32_t* swa_len_out, cudaStream_t s) {
  if (L > kMaxStepLayers) return CSA2_ERR_UNSUPPORTED_SHAPE;
  StepLayers ly;
  for (int l = 0; l < kMaxStepLayers; ++l) {
    ly.src[l] = l < L ? reinterpret_cast<const uint4*>(src[l]) : nullptr;
    ly.dst[l] = l < L ? reinterpret_cast<uint4*>(dst[l]) : nullptr;
  }
  const int64_t warps = (int64_t)L * B * W;
  if (warps == 0) return CSA2_OK;
  k_swa_ring<<<(unsigned)((warps + 7) / 8), 256, 0, s>>>(ly, L, W, B, d / 8, n, to_ring, swa_len_out);
  count_launch();
  return launch_status();
}

int launch_append_swa(const void* x, int B, int d, const int64_t* pos, void* swa, int W,
                      cudaStream_t s) {
  const int64_t threads = (int64_t)B * 32;
  k_append_swa<<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(
      reinterpret_cast<const uint4*>(x), B, d, pos, reinterpret_cast<uint4*>(swa), W);
  count_launch();
  return launch_status();
}

}  // namespace csa2

namespace csa2 {
int launch_append_step(const void* kv_new, const uint8_t* kI_new, const void* const* swa_new, void* const* swa,
                       int L, int W, int B, int d_I, const int64_t* pos, int ratio, uint8_t* codes,
                       uint8_t* scales, uint8_t* kI, uint8_t* kbar, int64_t n_cap, int64_t* n_vis_out,
                       int32_t* swa_len_out, int32_t* st, cudaStream_t s) {
  if (L > kMaxStepLayers) return CSA2_ERR_UNSUPPORTED_SHAPE;
  StepLayers ly;
  for (int l = 0; l < kMaxStepLayers; ++l) {
    ly.src[l] = l < L ? reinterpret_cast<const uint4*>(swa_new[l]) : nullptr;
    ly.dst[l] = l < L ? reinterpret_cast<uint4*>(swa[l]) : nullptr;
  }
  const int64_t warps = (int64_t)B * (2 + L);
  k_append_step<<<(unsigned)((warps + 7) / 8), 256, 0, s>>>(reinterpret_cast<const uint4*>(kv_new), kI_new, ly, L,
                                                            W > 0 ? W : 1, B, d_I, pos, ratio, codes, scales, kI,
                                                            kbar, n_cap, n_vis_out, swa_len_out, st);
  count_launch();
  return launch_status();
}
}  // namespace csa2
