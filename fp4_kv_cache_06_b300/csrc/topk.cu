// topk.cu — deterministic Top-K selection for the CSA2 indexer.
//
// [CSA2] wire.sakhanda.co, "DeepSeek AI выпустила DeepSeek-V4.1-Flash ...",
//        section "Сжатое разреженное внимание 2 (CSA2)": Full selects new
//        Top-512 indices; Reindex selects again among the pool; the pool
//        itself keeps the best 2048 blocks.
//
// Order: score descending, then position ascending. Each candidate becomes
// a unique 64-bit key (order-preserving score bits << 32 | ~position), so the
// k best are exactly the k largest keys and the result does not depend on
// the order in which threads or CTAs visit the candidates.
//
// Pipeline per row (three launches; the first is fused into the indexer
// scan when the scan runs just before):
//   1. histogram of the 12 high key bits (4096 bins) over the row;
//   2. compaction: every CTA derives the same threshold bin from the
//      histogram and appends the candidates at or above it (at most
//      kCandCap) to the row's candidate buffer; if more than kCandCap would
//      qualify the row is flagged and left to step 3's slow path;
//   3. one CTA per row: exact radix select of the k-th largest key over the
//      compacted candidates in shared memory (or, for a flagged row, over the
//      whole row in global memory), then a bitonic sort of the chosen
//      positions, -1 padding.
#include "common.cuh"

namespace csa2 {


// Workspace layout (all offsets 256-byte aligned):
//   hist [B][kHistBins] u32 | hdr [B] TopkHdr | cand [B][kCandCap] u64
static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
size_t topk_ws_bytes(int B) {
  return align256((size_t)B * kHistBins * 4) + align256((size_t)B * sizeof(TopkHdr)) +
         align256((size_t)B * kCandCap * 8);
}
struct TopkWs {
  uint32_t* hist;
  TopkHdr* hdr;
  uint64_t* cand;
};
static TopkWs topk_ws(void* ws, int B) {
  char* p = static_cast<char*>(ws);
  TopkWs r;
  r.hist = reinterpret_cast<uint32_t*>(p);
  p += align256((size_t)B * kHistBins * 4);
  r.hdr = reinterpret_cast<TopkHdr*>(p);
  p += align256((size_t)B * sizeof(TopkHdr));
  r.cand = reinterpret_cast<uint64_t*>(p);
  return r;
}
uint32_t* topk_ws_hist(void* ws) { return static_cast<uint32_t*>(ws); }
TopkHdr* topk_ws_hdr(void* ws, int B) { return topk_ws(ws, B).hdr; }


// Candidates of row b: the first ceil(n[b] / len_div) entries, at most n_max
// (n == NULL: every row has n_max entries).
__device__ __forceinline__ int64_t row_len(const int64_t* n, int b, int len_div, int64_t n_max) {
  if (n == nullptr) return n_max;
  int64_t v = n[b];
  v = v <= 0 ? 0 : (v + len_div - 1) / len_div;
  return v < n_max ? v : n_max;
}

// ---- step 1 (standalone form) --------------------------------------------
__global__ void __launch_bounds__(kTkThreads) k_topk_hist(const float* __restrict__ scores,
                                                          const int32_t* __restrict__ cand_pos,
                                                          int64_t stride, const int64_t* __restrict__ n,
                                                          int len_div, int64_t n_max, int64_t per,
                                                          uint32_t* __restrict__ hist, TopkHdr* __restrict__ hdr,
                                                          int k) {
  __shared__ uint32_t sh[kHistBins];
  const int b = blockIdx.y;
  for (int i = threadIdx.x; i < kHistBins; i += kTkThreads) sh[i] = 0;
  __syncthreads();
  const int64_t nb = row_len(n, b, len_div, n_max);
  const int64_t c0 = (int64_t)blockIdx.x * per, c1 = min(c0 + per, nb);
  const float* s = scores + (int64_t)b * stride;
  const int32_t* cp = cand_pos ? cand_pos + (int64_t)b * stride : nullptr;
  for (int64_t i = c0 + threadIdx.x; i < c1; i += kTkThreads) {
    if (cp && cp[i] < 0) continue;
    atomicAdd(&sh[score_key(s[i]) >> 20], 1u);
  }
  topk_hist_flush(sh, hist + (int64_t)b * kHistBins, hdr + b, k, gridDim.x);
}

// ---- step 2 ----------------------------------------------------------------
__global__ void __launch_bounds__(kTkThreads) k_topk_compact(const float* __restrict__ scores,
                                                             const int32_t* __restrict__ cand_pos,
                                                             int64_t stride, const int64_t* __restrict__ n,
                                                             int len_div, int64_t n_max, int64_t per,
                                                             TopkHdr* __restrict__ hdr,
                                                             uint64_t* __restrict__ cand) {
  const int b = blockIdx.y;
  if (hdr[b].overflow) return;
  const int vbin = hdr[b].vbin;
  const int64_t nb = row_len(n, b, len_div, n_max);
  const int64_t c0 = (int64_t)blockIdx.x * per, c1 = min(c0 + per, nb);
  const float* s = scores + (int64_t)b * stride;
  const int32_t* cp = cand_pos ? cand_pos + (int64_t)b * stride : nullptr;
  uint64_t* out = cand + (int64_t)b * kCandCap;
  const int lane = threadIdx.x & 31;
  // each thread owns 8 consecutive candidates per pass, read up front (vector
  // loads when the row is 16-byte aligned) so their latencies overlap
  const bool vec = ((reinterpret_cast<uintptr_t>(s) | (cp ? reinterpret_cast<uintptr_t>(cp) : 0)) & 15) == 0 &&
                   (c0 & 7) == 0;
  for (int64_t i0 = c0; i0 < c1; i0 += (int64_t)kTkThreads * 8) {
    const int64_t i = i0 + (int64_t)threadIdx.x * 8;
    float v[8];
    int32_t p[8];
    if (vec && i + 8 <= c1) {
      const float4 a = *reinterpret_cast<const float4*>(s + i), bq = *reinterpret_cast<const float4*>(s + i + 4);
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = bq.x; v[5] = bq.y; v[6] = bq.z; v[7] = bq.w;
      if (cp) {
        const int4 pa = *reinterpret_cast<const int4*>(cp + i), pb = *reinterpret_cast<const int4*>(cp + i + 4);
        p[0] = pa.x; p[1] = pa.y; p[2] = pa.z; p[3] = pa.w; p[4] = pb.x; p[5] = pb.y; p[6] = pb.z; p[7] = pb.w;
      } else {
#pragma unroll
        for (int u = 0; u < 8; ++u) p[u] = (int32_t)(i + u);
      }
    } else {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const bool in = i + u < c1;
        v[u] = in ? s[i + u] : 0.f;
        p[u] = in ? (cp ? cp[i + u] : (int32_t)(i + u)) : -1;
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const bool take = p[u] >= 0 && (int)(score_key(v[u]) >> 20) >= vbin;
      const uint32_t m = __ballot_sync(0xffffffffu, take);
      if (m) {
        uint32_t basei = 0;
        const int leader = __ffs(m) - 1;
        if (lane == leader) basei = atomicAdd(&hdr[b].cnt, (uint32_t)__popc(m));
        basei = __shfl_sync(0xffffffffu, basei, leader);
        if (take) {
          const uint32_t slot = basei + __popc(m & ((1u << lane) - 1u));
          if (slot < (uint32_t)kCandCap) out[slot] = cand_key(v[u], p[u]);   // always: the row did not overflow
        }
      }
    }
  }
}

// ---- step 3 ----------------------------------------------------------------
constexpr int kFinThreads = 1024;

// Key sources for the radix select.
struct SmemKeys {
  const uint64_t* keys;
  int cnt;
  __device__ int64_t size() const { return cnt; }
  __device__ bool get(int64_t i, uint64_t& key) const { key = keys[i]; return true; }
};
struct RowKeys {
  const float* s;
  const int32_t* cp;
  int64_t cnt;
  __device__ int64_t size() const { return cnt; }
  __device__ bool get(int64_t i, uint64_t& key) const {
    const int32_t p = cp ? cp[i] : (int32_t)i;
    if (p < 0) return false;
    key = cand_key(s[i], p);
    return true;
  }
};

// Exact key of the k-th largest among the source's keys (all distinct);
// requires at least k keys. MSD radix, 8 bits per pass.
template <class Src>
__device__ uint64_t radix_kth(const Src& src, int k, uint32_t* h256) {
  __shared__ uint64_t s_prefix;
  __shared__ int s_remaining;
  __shared__ unsigned long long s_and, s_or;
  const int tid = threadIdx.x;
  // bits shared by every key are fixed: skip the digits above the first difference
  if (tid == 0) { s_and = ~0ull; s_or = 0ull; }
  __syncthreads();
  {
    unsigned long long a = ~0ull, o = 0ull;
    const int64_t m = src.size();
    for (int64_t i = tid; i < m; i += kFinThreads) {
      uint64_t key;
      if (src.get(i, key)) { a &= key; o |= key; }
    }
    for (int off = 16; off > 0; off >>= 1) {
      a &= __shfl_xor_sync(0xffffffffu, a, off);
      o |= __shfl_xor_sync(0xffffffffu, o, off);
    }
    if ((tid & 31) == 0) { atomicAnd(&s_and, a); atomicOr(&s_or, o); }
  }
  __syncthreads();
  const uint64_t diff = s_and ^ s_or;                 // bits that are not common to all keys
  const int top = diff ? 63 - __clzll((long long)diff) : -1;
  int start = 56;
  while (start > 0 && start > top) start -= 8;        // first digit holding a differing bit
  uint64_t mask = start < 56 ? ~((1ull << (start + 8)) - 1) : 0ull;
  uint64_t prefix = s_and & mask;
  int remaining = k;
  for (int shift = start; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kFinThreads) h256[i] = 0;
    __syncthreads();
    const int64_t m = src.size();
    const int lane = tid & 31;
    for (int64_t i0 = 0; i0 < m; i0 += kFinThreads) {
      const int64_t i = i0 + tid;
      uint64_t key = 0;
      const bool ok = i < m && src.get(i, key) && (key & mask) == prefix;
      const uint32_t dgt = ok ? (uint32_t)((key >> shift) & 255) : 256u;
      const uint32_t peers = __match_any_sync(0xffffffffu, dgt);   // lanes holding the same digit
      if (ok && lane == __ffs(peers) - 1) atomicAdd(&h256[dgt], (uint32_t)__popc(peers));
    }
    __syncthreads();
    if (tid < 32) {
      // lane l owns digits [255-8l-7, 255-8l], counted from the top
      uint32_t loc = 0;
      for (int j = 0; j < 8; ++j) loc += h256[255 - 8 * tid - j];
      uint32_t incl = loc;
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, off);
        if (tid >= off) incl += v;
      }
      const uint32_t excl = incl - loc;
      if (excl < (uint32_t)remaining && incl >= (uint32_t)remaining) {
        uint32_t run = excl;
        for (int j = 0; j < 8; ++j) {
          const int dgt = 255 - 8 * tid - j;
          const uint32_t c = h256[dgt];
          if (run + c >= (uint32_t)remaining) {
            s_prefix = prefix | ((uint64_t)dgt << shift);
            s_remaining = remaining - (int)run;
            break;
          }
          run += c;
        }
      }
    }
    __syncthreads();
    prefix = s_prefix;
    remaining = s_remaining;
    mask |= (uint64_t)255 << shift;
    __syncthreads();
  }
  return prefix;
}

// Bitonic sort of sel[0..np) ascending (np a power of two, padded with INT_MAX).
__device__ void bitonic_sort_i32(int32_t* sel, int np) {
  for (int size = 2; size <= np; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      __syncthreads();
      for (int i = threadIdx.x; i < np / 2; i += kFinThreads) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool up = ((lo & size) == 0);
        const int32_t a = sel[lo], c = sel[hi];
        if ((a > c) == up) { sel[lo] = c; sel[hi] = a; }
      }
    }
  }
  __syncthreads();
}

template <class Src>
__device__ void select_and_write(const Src& src, int k, int64_t n_keys, int32_t* __restrict__ out,
                                 uint32_t* h256, int32_t* sel) {
  __shared__ uint32_t s_cnt;
  const int tid = threadIdx.x;
  uint64_t thr = 0;
  if (n_keys > k) thr = radix_kth(src, k, h256);
  if (tid == 0) s_cnt = 0;
  __syncthreads();
  const int64_t m = src.size();
  const int lane = tid & 31;
  for (int64_t i0 = 0; i0 < m; i0 += kFinThreads) {
    const int64_t i = i0 + tid;
    uint64_t key = 0;
    const bool take = i < m && src.get(i, key) && key >= thr;
    const uint32_t bal = __ballot_sync(0xffffffffu, take);
    uint32_t base = 0;
    if (bal) {
      if (lane == __ffs(bal) - 1) base = atomicAdd(&s_cnt, (uint32_t)__popc(bal));
      base = __shfl_sync(0xffffffffu, base, __ffs(bal) - 1);
    }
    if (take) {
      const uint32_t slot = base + __popc(bal & ((1u << lane) - 1u));
      if (slot < (uint32_t)k) sel[slot] = cand_pos_of(key);
    }
  }
  __syncthreads();
  const int cnt = (int)min(s_cnt, (uint32_t)k);
  if (k <= 512) {
    // ascending order by rank: the chosen positions are distinct, so the rank
    // of one is the number of chosen positions below it (reads broadcast)
    for (int i = tid; i < cnt; i += kFinThreads) {
      const int32_t mine = sel[i];
      int rank = 0;
      for (int j = 0; j < cnt; ++j) rank += sel[j] < mine;
      out[rank] = mine;
    }
    for (int i = cnt + tid; i < k; i += kFinThreads) out[i] = -1;
  } else {
    int np = 1;
    while (np < k) np <<= 1;
    for (int i = cnt + tid; i < np; i += kFinThreads) sel[i] = 0x7FFFFFFF;
    bitonic_sort_i32(sel, np);
    for (int i = tid; i < k; i += kFinThreads) out[i] = i < cnt ? sel[i] : -1;
  }
}

__global__ void __launch_bounds__(kFinThreads) k_topk_final(const float* __restrict__ scores,
                                                            const int32_t* __restrict__ cand_pos,
                                                            int64_t stride, const int64_t* __restrict__ n,
                                                            int len_div, int64_t n_max, int k,
                                                            const TopkHdr* __restrict__ hdr,
                                                            const uint64_t* __restrict__ cand,
                                                            int32_t* __restrict__ idx_out) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint64_t* keys = reinterpret_cast<uint64_t*>(smem);                 // kCandCap
  uint32_t* h256 = reinterpret_cast<uint32_t*>(keys + kCandCap);      // 256
  int32_t* sel = reinterpret_cast<int32_t*>(h256 + 256);              // kMaxTopK
  const int b = blockIdx.x;
  int32_t* out = idx_out + (int64_t)b * k;
  const int64_t nb = row_len(n, b, len_div, n_max);
  if (hdr[b].overflow) {
    // slow path: count the row's present candidates, then select over global memory
    __shared__ uint32_t s_valid;
    if (threadIdx.x == 0) s_valid = 0;
    __syncthreads();
    const float* s = scores + (int64_t)b * stride;
    const int32_t* cp = cand_pos ? cand_pos + (int64_t)b * stride : nullptr;
    uint32_t loc = 0;
    for (int64_t i = threadIdx.x; i < nb; i += kFinThreads) loc += (cp == nullptr || cp[i] >= 0);
    atomicAdd(&s_valid, loc);
    __syncthreads();
    RowKeys src{s, cp, nb};
    select_and_write(src, k, (int64_t)s_valid, out, h256, sel);
    return;
  }
  const int cnt = (int)min(hdr[b].cnt, (uint32_t)kCandCap);
  for (int i = threadIdx.x; i < cnt; i += kFinThreads) keys[i] = cand[(int64_t)b * kCandCap + i];
  __syncthreads();
  SmemKeys src{keys, cnt};
  select_and_write(src, k, cnt, out, h256, sel);
}

int topk_final_smem() { return kCandCap * 8 + 256 * 4 + kMaxTopK * 4; }

// ---- host ------------------------------------------------------------------
static int64_t tk_rows_per_cta(int B, int64_t rows) {
  int64_t per = 16384;
  while (per > 1024 && (int64_t)B * ((rows + per - 1) / per) < 4 * kSMs) per /= 2;
  return per;
}

// Zero the histogram and headers of B rows (before the scan or step 1).
int topk_prepare(void* ws, int B, cudaStream_t s) {
  const size_t bytes = align256((size_t)B * kHistBins * 4) + align256((size_t)B * sizeof(TopkHdr));
  if (cudaMemsetAsync(ws, 0, bytes, s) != cudaSuccess) return CSA2_ERR_CUDA;
  return CSA2_OK;
}

// Steps 1 (unless the histogram is already in the workspace), 2 and 3.
int launch_topk(const float* scores, const int32_t* cand_pos, int64_t stride, const int64_t* n,
                int len_div, int B, int64_t n_max, int k, int32_t* idx_out, void* ws, bool hist_ready,
                cudaStream_t s) {
  if (B == 0) return CSA2_OK;
  TopkWs w = topk_ws(ws, B);
  int rc;
  const int64_t per = tk_rows_per_cta(B, n_max);
  dim3 grid((unsigned)((n_max + per - 1) / per > 0 ? (n_max + per - 1) / per : 1), (unsigned)B);
  if (!hist_ready) {
    if ((rc = topk_prepare(ws, B, s)) != CSA2_OK) return rc;
    k_topk_hist<<<grid, kTkThreads, 0, s>>>(scores, cand_pos, stride, n, len_div, n_max, per, w.hist, w.hdr, k);
    count_launch();
    if ((rc = launch_status()) != CSA2_OK) return rc;
  }
  k_topk_compact<<<grid, kTkThreads, 0, s>>>(scores, cand_pos, stride, n, len_div, n_max, per, w.hdr,
                                             w.cand);
  count_launch();
  if ((rc = launch_status()) != CSA2_OK) return rc;
  k_topk_final<<<B, kFinThreads, topk_final_smem(), s>>>(scores, cand_pos, stride, n, len_div, n_max, k, w.hdr,
                                                          w.cand, idx_out);
  count_launch();
  return launch_status();
}

int topk_init_attributes() {
  if (cudaFuncSetAttribute(k_topk_final, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           topk_final_smem()) != cudaSuccess)
    return CSA2_ERR_CUDA;
  return CSA2_OK;
}

}  // namespace csa2
