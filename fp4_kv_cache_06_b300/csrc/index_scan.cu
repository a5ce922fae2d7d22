// index_scan.cu — the CSA2 indexer scan (Full, pool formation, Reindex).
//
// [CSA2] wire.sakhanda.co, "DeepSeek AI выпустила DeepSeek-V4.1-Flash ...",
//        section "Сжатое разреженное внимание 2 (CSA2)": a Full layer
//        projects indexer K and selects new Top-512 indices; a Reindex layer
//        rescores the last Full layer's indexer K with its own indexer Q; the
//        Full layer forms a pool of up to 2048 blocks of 8 positions so that
//        Reindex layers score a bounded set. The score formula is not on the
//        pages; this library computes s_t = sum_h w_h * relu(q_h . k_t) with
//        one E4M3 key per position shared by all (<= 8) heads.
//
// Design (B300): the scan streams 64 or 128 bytes per position from HBM and
// does 8 x d_I FP8 MACs per position, i.e. 8 MAC per byte. At ~6.7 TB/s
// that is ~54 TMAC/s, above what the CUDA cores can sustain in fp32 FMA, so
// the dot products run on the tensor cores: mma.sync m16n8k32 E4M3 x E4M3 ->
// fp32 with the 16 rows of an m-tile as M and the (padded) 8 indexer heads
// as N. A dot product is invariant under a common permutation of its
// channels, so each thread loads whole 16-byte vectors of its rows straight
// from global memory into A fragments (fully coalesced: a warp instruction
// covers 8 rows x 64 contiguous bytes) and the query is loaded with the same
// channel permutation into B fragments. The relu * w head sum is a
// thread-local FMA pair plus two quad shuffles. The Top-K level-0 histogram
// (12 high bits of the order-preserving score key) is accumulated in shared
// memory and flushed once per CTA.
#include "common.cuh"
#include "tcgen05.cuh"

namespace csa2 {

constexpr int kScanThreads = 256;
constexpr int kScanTilesPerIter = 4;                 // m-tiles of 16 rows per warp iteration
constexpr int kScanRowsPerWarpIter = 16 * kScanTilesPerIter;

// SRC_POOL = false: rows are positions 0..n[b)-1 of the sequence.
// SRC_POOL = true : slot s maps to position pool[b][s/8]*8 + s%8 (absent if
//                   the block id is -1 or the position >= n[b]); cand_pos is
//                   written for every slot so Top-K can skip absent ones.
template <int DI, bool SRC_POOL>
__global__ void __launch_bounds__(kScanThreads) k_index_scan(
    const uint8_t* __restrict__ qI, const float* __restrict__ w, const uint8_t* __restrict__ kI,
    int64_t kI_seq_stride, int rps, const int64_t* __restrict__ n, int len_div, int H_I, int64_t n_max,
    int64_t rows_per_cta, float* __restrict__ scores, int64_t scores_stride,
    const int32_t* __restrict__ pool, int P, int32_t* __restrict__ cand_pos,
    uint32_t* __restrict__ hist, TopkHdr* __restrict__ hdr, int topk_k, int32_t* st) {
  constexpr int CH = DI / 64;                         // 16-byte chunks per row per thread
  __shared__ uint32_t sh_hist[kHistBins];
  const int b = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;

  int64_t nb = n[b];
  nb = nb < 0 ? nb : (nb + len_div - 1) / len_div;   // len_div 8: positions -> pool blocks
  if (nb > n_max || nb < 0) {
    if (blockIdx.x == 0 && tid == 0) report(st, CSA2_ERR_DEVICE_BOUNDS);
    nb = nb < 0 ? 0 : n_max;
  }
  const int64_t limit = SRC_POOL ? (int64_t)P * kBlock : nb;
  const int64_t c0 = (int64_t)blockIdx.x * rows_per_cta;
  const int64_t c1 = min(c0 + rows_per_cta, limit);
  if (hist) {
    for (int i = tid; i < kHistBins; i += kScanThreads) sh_hist[i] = 0;
    __syncthreads();
  }

  // B fragments: head g, the thread's channel chunks {16t..16t+15, 64+16t..}
  uint32_t qf[4 * CH];
  {
    const bool live = g < H_I;
    const uint8_t* qrow = qI + ((int64_t)b * H_I + (live ? g : 0)) * DI;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const uint4 v = live ? *reinterpret_cast<const uint4*>(qrow + 64 * c + 16 * t) : make_uint4(0, 0, 0, 0);
      qf[4 * c + 0] = v.x; qf[4 * c + 1] = v.y; qf[4 * c + 2] = v.z; qf[4 * c + 3] = v.w;
    }
  }
  const float w0 = (2 * t < H_I) ? w[(int64_t)b * H_I + 2 * t] : 0.f;
  const float w1 = (2 * t + 1 < H_I) ? w[(int64_t)b * H_I + 2 * t + 1] : 0.f;
  const uint8_t* kseq = kI + (int64_t)(b / rps) * kI_seq_stride * DI;   // rps query rows per sequence
  float* srow = scores + (int64_t)b * scores_stride;

  for (int64_t base = c0 + (int64_t)warp * kScanRowsPerWarpIter; base < c1;
       base += (int64_t)(kScanThreads / 32) * kScanRowsPerWarpIter) {
    uint4 ra[kScanTilesPerIter][2][CH];
    int64_t rpos[kScanTilesPerIter][2];
#pragma unroll
    for (int u = 0; u < kScanTilesPerIter; ++u) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int64_t slot = base + u * 16 + g + 8 * hh;
        int64_t p = -1;
        if (slot < c1) {
          if (SRC_POOL) {
            const int32_t blk = pool[(int64_t)b * P + (slot >> 3)];
            const int64_t q = (int64_t)blk * kBlock + (slot & 7);
            p = (blk >= 0 && q < nb) ? q : -1;
          } else {
            p = slot;
          }
        }
        rpos[u][hh] = p;
#pragma unroll
        for (int c = 0; c < CH; ++c)
          ra[u][hh][c] = (p >= 0) ? ldg_stream(kseq + p * DI + 64 * c + 16 * t) : make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < kScanTilesPerIter; ++u) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < DI / 32; ++j) {
        const uint4& r0 = ra[u][0][j >> 1];
        const uint4& r1 = ra[u][1][j >> 1];
        const uint32_t a0 = (j & 1) ? r0.z : r0.x, a2 = (j & 1) ? r0.w : r0.y;
        const uint32_t a1 = (j & 1) ? r1.z : r1.x, a3 = (j & 1) ? r1.w : r1.y;
        mma_e4m3_16832(acc, a0, a1, a2, a3, qf[2 * j], qf[2 * j + 1]);
      }
      float s0 = w0 * fmaxf(acc[0], 0.f) + w1 * fmaxf(acc[1], 0.f);
      float s1 = w0 * fmaxf(acc[2], 0.f) + w1 * fmaxf(acc[3], 0.f);
      s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
      s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
      s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
      s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
      if (t < 2) {
        const int64_t slot = base + u * 16 + g + 8 * t;
        const float sc = t ? s1 : s0;
        const int64_t p = rpos[u][t];
        if (slot < c1) {
          if (SRC_POOL) {
            cand_pos[(int64_t)b * scores_stride + slot] = (int32_t)p;
            srow[slot] = sc;
            if (hist && p >= 0) atomicAdd(&sh_hist[score_key(sc) >> 20], 1u);
          } else {
            srow[slot] = sc;
            if (hist) atomicAdd(&sh_hist[score_key(sc) >> 20], 1u);
          }
        }
      }
    }
  }
  if (hist) topk_hist_flush(sh_hist, hist + (int64_t)b * kHistBins, hdr + b, topk_k, gridDim.x);
}

// ---- TMA-staged variant for contiguous rows of 128-byte keys ------------------
// The big Full-layer and pool-formation scans stream 16 KB tiles (128 rows x
// 128 B) through a 5-stage shared-memory ring with TMA (128-byte swizzle);
// one producer warp issues the copies, 8 consumer warps each take one
// 16-row m-tile of every tile. Bytes in flight are then set by the ring, not
// by registers. Inside an m-tile, fragment row g reads smem row sigma(g) =
// {0,4,1,5,2,6,3,7}[g] (and +8): with the swizzle this makes every 16-byte
// shared load of a quarter-warp hit 8 distinct bank groups.
// With a Top-K header the row's CTAs take tiles dynamically from the header's
// counter (zero until the compaction, which the row's last CTA restores), so
// a CTA on a slower SM simply takes fewer tiles; the producer passes each
// tile's index to the consumers in shared memory and ends with index -1.
constexpr int kTmaStages = 5;
constexpr int kTmaRows = 128;
constexpr int kTmaTile = kTmaRows * 128;          // 16 KB
constexpr int kTmaThreads = 288;                  // 8 consumer warps + 1 producer warp
// after the tiles: full and empty barriers (2 x 8 x kTmaStages bytes), then the
// stages' tile indices at +128; plus alignment slack
constexpr int kTmaSmem = kTmaStages * kTmaTile + 1024 + 256;

// R > 1: one CTA serves the R query rows of a sequence (multi-token decode):
// every key tile is read once and scored against each row's queries; these
// launches write plain scores (no histogram, static tile ranges).
template <int R>
__global__ void __launch_bounds__(kTmaThreads, 2) k_index_scan_tma(
    const __grid_constant__ CUtensorMap map_k, const uint8_t* __restrict__ qI, const float* __restrict__ w,
    int64_t kI_seq_stride, int rps, const int64_t* __restrict__ n, int len_div, int H_I, int64_t n_max, int tiles_per_cta,
    float* __restrict__ scores, int64_t scores_stride, uint32_t* __restrict__ hist, TopkHdr* __restrict__ hdr,
    int topk_k, int32_t* st, uint64_t wait_ns, int fault) {
  __shared__ uint32_t sh_hist[kHistBins];
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023) & ~1023u;
  unsigned char* sp = smem_raw + (base - raw);
  const uint32_t bar_full = base + kTmaStages * kTmaTile, bar_empty = bar_full + 8 * kTmaStages;
  volatile int64_t* sTile = reinterpret_cast<volatile int64_t*>(sp + kTmaStages * kTmaTile + 128);  // [kTmaStages]
  // R == 1: row b = blockIdx.y reads sequence b / rps; R > 1: rows
  // R * blockIdx.y .. + R - 1 all read sequence blockIdx.y
  const int b = R == 1 ? (int)blockIdx.y : (int)blockIdx.y * R;
  const int64_t seq = R == 1 ? (int64_t)(b / rps) : (int64_t)blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;

  int64_t nr[R];                                  // visible rows (or blocks) of each row
  int64_t nb = 0;                                 // the most any of them sees
#pragma unroll
  for (int r = 0; r < R; ++r) {
    int64_t v = n[b + r];
    v = v < 0 ? v : (v + len_div - 1) / len_div;
    if (v > n_max || v < 0) {
      if (blockIdx.x == 0 && tid == 0) report(st, CSA2_ERR_DEVICE_BOUNDS);
      v = v < 0 ? 0 : n_max;
    }
    nr[r] = v;
    nb = v > nb ? v : nb;
  }
  const int64_t tiles_b = (nb + kTmaRows - 1) / kTmaRows;
  const int64_t t0 = (int64_t)blockIdx.x * tiles_per_cta;
  const int64_t t1 = min(t0 + (int64_t)tiles_per_cta, tiles_b);
  const bool dynamic = R == 1 && hdr != nullptr;  // take tiles from the row's counter

  if (R == 1 && hist)
    for (int i = tid; i < kHistBins; i += kTmaThreads) sh_hist[i] = 0;
  if (tid == 0) {
    for (int i = 0; i < kTmaStages; ++i) {
      tc::mbar_init(bar_full + 8 * i, 1);
      tc::mbar_init(bar_empty + 8 * i, 8);
    }
    tc::fence_barrier_init();
  }
  __syncthreads();

  if (warp == 8) {
    if (lane == 0) {                               // producer
      tc::prefetch_tmap(&map_k);
      for (int i = 0;; ++i) {
        const int s = i % kTmaStages;
        if (!tc::mbar_wait(bar_empty + 8 * s, ((i / kTmaStages) & 1) ^ 1, wait_ns)) {
          report(st, CSA2_ERR_TIMEOUT);            // the consumers time out on the full barrier
          break;
        }
        // fault injection (tests of the bounded waits): the second stage is
        // never loaded nor signalled, so the consumers' wait on it runs out
        if (fault && i == 1) break;
        const int64_t tile = dynamic ? (int64_t)atomicAdd(&hdr[b].cnt, 1u) : t0 + i;
        if (tile >= (dynamic ? tiles_b : t1)) {
          sTile[s] = -1;                           // no more tiles: an arrive without bytes
          tc::mbar_arrive(bar_full + 8 * s);
          break;
        }
        sTile[s] = tile;
        tc::mbar_expect_tx(bar_full + 8 * s, kTmaTile);
        tc::tma_load_2d(base + s * kTmaTile, &map_k, 0,
                        (int32_t)(seq * kI_seq_stride + tile * kTmaRows), bar_full + 8 * s);
      }
    }
  } else {                                         // consumers: warp w owns m-tile w of every tile
    uint32_t qf[R][8];
    float w0[R], w1[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const bool live = g < H_I;
      const uint8_t* qrow = qI + ((int64_t)(b + r) * H_I + (live ? g : 0)) * 128;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const uint4 v = live ? *reinterpret_cast<const uint4*>(qrow + 64 * c + 16 * t) : make_uint4(0, 0, 0, 0);
        qf[r][4 * c + 0] = v.x; qf[r][4 * c + 1] = v.y; qf[r][4 * c + 2] = v.z; qf[r][4 * c + 3] = v.w;
      }
      w0[r] = (2 * t < H_I) ? w[(int64_t)(b + r) * H_I + 2 * t] : 0.f;
      w1[r] = (2 * t + 1 < H_I) ? w[(int64_t)(b + r) * H_I + 2 * t + 1] : 0.f;
    }
    const int sg = ((g & 1) << 2) | (g >> 1);       // sigma(g)
    const int r1 = warp * 16 + sg, r2 = r1 + 8;     // tile rows of fragment rows g and g+8
    for (int i = 0;; ++i) {
      const int s = i % kTmaStages;
      const bool got = tc::mbar_wait(bar_full + 8 * s, (i / kTmaStages) & 1, wait_ns);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) report(st, CSA2_ERR_TIMEOUT);
        break;
      }
      const int64_t tidx = sTile[s];               // read before the stage is released
      if (tidx < 0) break;
      const unsigned char* tile = sp + s * kTmaTile;
      uint4 a[2][2];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        a[0][c] = *reinterpret_cast<const uint4*>(tile + r1 * 128 + (((4 * c + t) ^ (r1 & 7)) << 4));
        a[1][c] = *reinterpret_cast<const uint4*>(tile + r2 * 128 + (((4 * c + t) ^ (r2 & 7)) << 4));
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(bar_empty + 8 * s);   // this warp is done with the stage
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4& x0 = a[0][j >> 1];
          const uint4& x1 = a[1][j >> 1];
          mma_e4m3_16832(acc, (j & 1) ? x0.z : x0.x, (j & 1) ? x1.z : x1.x, (j & 1) ? x0.w : x0.y,
                         (j & 1) ? x1.w : x1.y, qf[r][2 * j], qf[r][2 * j + 1]);
        }
        float s0 = w0[r] * fmaxf(acc[0], 0.f) + w1[r] * fmaxf(acc[1], 0.f);
        float s1 = w0[r] * fmaxf(acc[2], 0.f) + w1[r] * fmaxf(acc[3], 0.f);
        s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
        s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
        s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
        s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
        if (t < 2) {
          const int64_t row = tidx * kTmaRows + (t ? r2 : r1);
          const float sc = t ? s1 : s0;
          if (row < nr[r]) {
            scores[(int64_t)(b + r) * scores_stride + row] = sc;
            if (R == 1 && hist) atomicAdd(&sh_hist[score_key(sc) >> 20], 1u);
          }
        }
      }
    }
  }
  if (R == 1 && hist) topk_hist_flush(sh_hist, hist + (int64_t)b * kHistBins, hdr + b, topk_k, gridDim.x);
}

static int tma_scan_init = 0;
int scan_init_attributes() {
  for (auto kern : {k_index_scan_tma<1>, k_index_scan_tma<2>, k_index_scan_tma<4>, k_index_scan_tma<8>})
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kTmaSmem) != cudaSuccess)
      return CSA2_ERR_CUDA;
  tma_scan_init = 1;
  return CSA2_OK;
}

// rows_per_cta: a multiple of the CTA's rows per iteration, sized so the
// grid covers the machine a few times over.
static int64_t scan_rows_per_cta(int B, int64_t rows) {
  const int64_t step = (int64_t)(kScanThreads / 32) * kScanRowsPerWarpIter;  // 512
  int64_t per = 4096;
  while (per > step && (int64_t)B * ((rows + per - 1) / per) < 4 * kSMs) per /= 2;
  return per;
}

int launch_index_scan(const uint8_t* qI, const float* w, const uint8_t* kI, int64_t kI_seq_stride, int rps,
                      const int64_t* n, int len_div, int B, int H_I, int d_I, int64_t n_max, float* scores,
                      int64_t scores_stride, const int32_t* pool, int P, int32_t* cand_pos,
                      uint32_t* hist, TopkHdr* hdr, int topk_k, int32_t* st, cudaStream_t s) {
  const bool use_pool = pool != nullptr;
  const int64_t rows = use_pool ? (int64_t)P * kBlock : n_max;
  if (rows == 0 || B == 0) return CSA2_OK;
  if (!use_pool && d_I == 128 && tma_scan_init) {
    // the key rows of all sequences as one 2-D tensor [rows][128 B]
    const uint64_t total_rows = (uint64_t)((B - 1) / rps) * (uint64_t)kI_seq_stride + (uint64_t)n_max;
    CUtensorMap map;
    if (make_tmap_rows128(&map, kI, total_rows, 128, kTmaRows)) {
      const int64_t tiles = (n_max + kTmaRows - 1) / kTmaRows;
      // rows of one sequence share a CTA (plain scores) when there are 2, 4 or 8
      const int R = (hist == nullptr && (rps == 2 || rps == 4 || rps == 8)) ? rps : 1;
      const int units = B / R;                      // CTA rows of the grid
      // one wave of two CTAs per SM
      int64_t per_seq = (2 * kSMs) / units;
      if (per_seq > tiles) per_seq = tiles;
      if (per_seq < 1) per_seq = 1;
      const int tpc = (int)((tiles + per_seq - 1) / per_seq);
      per_seq = (tiles + tpc - 1) / tpc;
      dim3 grid((unsigned)per_seq, (unsigned)units);
#define CSA2_TMA_SCAN(R_)                                                                                  \
  k_index_scan_tma<R_><<<grid, kTmaThreads, kTmaSmem, s>>>(map, qI, w, kI_seq_stride, rps, n, len_div, H_I, \
                                                          n_max, tpc, scores, scores_stride, hist, hdr,     \
                                                          topk_k, st, debug_wait_ns(), debug_fault() == kFaultScan)
      if (R == 8) CSA2_TMA_SCAN(8);
      else if (R == 4) CSA2_TMA_SCAN(4);
      else if (R == 2) CSA2_TMA_SCAN(2);
      else CSA2_TMA_SCAN(1);
#undef CSA2_TMA_SCAN
      count_launch();
      return launch_status();
    }
  }
  const int64_t per = scan_rows_per_cta(B, rows);
  dim3 grid((unsigned)((rows + per - 1) / per), (unsigned)B);
#define CSA2_SCAN(DI_, POOL_)                                                                   \
  k_index_scan<DI_, POOL_><<<grid, kScanThreads, 0, s>>>(qI, w, kI, kI_seq_stride, rps, n, len_div, H_I, n_max, \
                                                         per, scores, scores_stride, pool, P,     \
                                                         cand_pos, hist, hdr, topk_k, st)
  if (d_I == 128) {
    if (use_pool) CSA2_SCAN(128, true); else CSA2_SCAN(128, false);
  } else {
    if (use_pool) CSA2_SCAN(64, true); else CSA2_SCAN(64, false);
  }
#undef CSA2_SCAN
  count_launch();
  return launch_status();
}

}  // namespace csa2
